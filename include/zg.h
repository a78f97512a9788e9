/*
 * zg.h -- C ABI of the sharded mixed-precision optimizer step on one GB300.
 *
 * What the library computes (ZeRO stage two over a flat parameter vector):
 * P data-parallel ranks are simulated on one GPU. Each rank r holds a bf16
 * gradient buffer G_r (already multiplied by the loss scale L) for the whole
 * flat vector of N parameters. Rank r owns the shard [r*S, min((r+1)*S, N)),
 * S = zg_shard_len(). For every index i of every shard a step
 *   1. reduce-scatters: g^_i = G_0[i] + G_1[i] + ... + G_{P-1}[i], in fp32, in
 *      rank order (Zero From Scratch, item 7: all-reduce is reduce-scatter
 *      followed by all-gather);
 *   2. unscales and averages: g_i = g^_i * fp32(1 / (L * P)) (item 6: data
 *      parallel ranks average their gradients);
 *   3. takes the global norm over all N: sumsq = sum of fp64(g_i * g_i);
 *      a non-finite sumsq skips the whole step (nothing is written, the step
 *      count stays); otherwise c = min(1, max_grad_norm / (norm + norm_eps));
 *   4. applies AdamW (decoupled weight decay) to the fp32 master weight w_i
 *      and moments m_i, v_i -- the 4 + 4 + 4 of the sixteen bytes per weight
 *      of item 1 -- in one fused pass (item 3: one read and one write per
 *      array instead of one per operation);
 *   5. writes p_i = bf16(w_i) into the one parameter buffer every rank reads:
 *      the all-gather.
 * Per element, every fp32 operation is rounded on its own in the order
 *   ga = g*c; m = b1*m + (1-b1)*ga; v = b2*v + (1-b2)*(ga*ga);
 *   mh = m/bc1; vh = v/bc2; d = sqrt(vh) + eps; w = w - (lr*wd)*w;
 *   w = w - lr*(mh/d); p = bf16_rne(w)
 * with bc1 = fp32(1 - b1^t), bc2 = fp32(1 - b2^t), b^t kept as fp64 running
 * products and each constant formed in fp64 and rounded once.
 * The optional MXFP8 path (item 14) first encodes each rank's gradient per
 * 32-element block as E4M3 codes plus one E8M0 scale byte, and the step then
 * sums decoded values instead of bf16 values.
 *
 * Citations name a page and a section: "Zero From Scratch" (When the model is
 * bigger than the machine), its outline items counted from 1 after the
 * introduction; and the review of the DeepSpeed documentation and tutorials.
 *
 * Conventions for every call:
 *   - Device pointers are plain CUDA device addresses (for example from
 *     torch), 16-byte aligned, owned by the caller and never freed here.
 *     A buffer "of n elements" must hold at least n elements; no call reads
 *     or writes an element at or past n. The shard layout pads each buffer
 *     to P * S elements; buffers that long are always large enough.
 *   - Every pointer is checked for the kind of memory behind it
 *     (cudaPointerGetAttributes) before anything is launched: it must be
 *     memory of the current device (cudaMalloc, a memory pool or managed
 *     memory), except w, m and v, which may also be pinned host memory
 *     mapped at the same address. Ordinary host memory (malloc, the stack),
 *     pinned host memory where device memory is needed, and another device's
 *     memory are refused with ZG_ERR_INVALID_ARG and a message naming the
 *     argument. The answer is remembered per pointer value, so calls that
 *     pass the same buffers again (every step) ask the driver only once; a
 *     buffer freed and its address handed out again as another kind of
 *     memory is not looked at again.
 *   - A zg_stream is a cudaStream_t (NULL: the legacy default stream). Every
 *     GPU call is stream-ordered and returns without waiting, except
 *     zg_get_info, which waits for its stream.
 *   - Return value: ZG_OK (0) or a negative ZG_ERR_* code; nothing else
 *     crosses the ABI (no exceptions). zg_strerror names a code and
 *     zg_last_error gives the calling thread's detailed message.
 *   - One context per stream at a time; contexts are independent.
 */
#ifndef ZG_H
#define ZG_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define ZG_OK 0
#define ZG_ERR_INVALID_ARG (-1)    /* a size, count, pointer or value out of range */
#define ZG_ERR_MISALIGNED (-2)     /* a pointer not 16-byte aligned */
#define ZG_ERR_NOT_BOUND (-3)      /* zg_bind has not been called on this context */
#define ZG_ERR_CUDA (-4)           /* a CUDA call or launch failed; see zg_last_error */
#define ZG_ERR_DEVICE_TIMEOUT (-5) /* a bounded device-side wait ran out (status only) */
#define ZG_ERR_STALE_NORM (-6)     /* a shard step ran without a fresh norm pass (status only) */
#define ZG_ERR_NO_MEMORY (-7)      /* host or device workspace allocation failed */
#define ZG_ERR_STATE_PARTIAL (-8)  /* a bounded wait ran out after part of w, m, v and the parameters were
                                      written (status only): restore the state from a checkpoint */

#define ZG_MAX_RANKS 16

/* Ways to run a bf16 step; all compute identical results. */
#define ZG_VARIANT_LDG 0    /* fused step with 128-bit vector loads straight from HBM (default) */
#define ZG_VARIANT_TMA 1    /* fused step, operands staged in a shared-memory ring by bulk async copies
                              (one producer warp, consumer warps; tile size chosen by P) */
#define ZG_VARIANT_STAGED 2 /* the norm pass also stores the reduced fp32 gradient; the step reads it */
#define ZG_VARIANT_SINGLE 3 /* zg_step runs the norm pass and the fused step in one cooperative launch,
                              with a grid-wide barrier between them (the same norm, decision and
                              state bits as the two launches) */

typedef struct CUstream_st *zg_stream; /* same type as cudaStream_t */
typedef struct zg_ctx zg_ctx;          /* opaque; owned by the library */

typedef struct {
    double lr, beta1, beta2, eps, weight_decay;
    double max_grad_norm; /* <= 0 turns the clip off */
    double norm_eps;      /* added to the norm in the clip ratio, e.g. 1e-6 */
    int grad_average;     /* 1: average over the P ranks; 0: plain sum */
} zg_hparams;

typedef struct {
    double sumsq;     /* global sum of squares of the unscaled, averaged gradient */
    double norm;      /* sqrt(sumsq) */
    float clip_coef;  /* c applied in the last step that ran (1 when the clip is off) */
    int found_inf;    /* 1: the last step saw a non-finite gradient and was skipped */
    int64_t step_t;   /* applied (not skipped) steps so far */
    int status;       /* ZG_OK or a device-side ZG_ERR_* code, sticky until zg_get_info */
} zg_step_info;

/* Create a context for N parameters over P simulated ranks (1 <= P <= 16,
 * 1 <= N < 2^62) on the current CUDA device. Allocates only a small device
 * workspace (64 KB of fp64 block partials for the MXFP8 norm pass from
 * codes, a 4.5 KB work array with the counters the norm and step passes hand
 * out their work with and the norm's exact fixed-point sum, and a 112-byte
 * block of step scalars).
 * Step count starts at 0. Layout: Zero From Scratch, item 17 (one flat
 * vector cut into P contiguous shards). *out is NULL on failure. */
int zg_init(int64_t n, int p, const zg_hparams *hp, zg_ctx **out);

/* Shard length S = ceil(N/P) rounded up to a multiple of 32 (one MX block);
 * rank r owns flat indices [r*S, min((r+1)*S, N)). -1 for a NULL context. */
int64_t zg_shard_len(const zg_ctx *ctx);

/* Attach the caller's optimizer state: fp32 master weights w, moments m and
 * v, and the bf16 parameter buffer (each N elements, 16-byte aligned). The
 * library keeps the pointers, never the memory. params must be device
 * memory. w, m and v may be device memory or pinned, device-accessible host
 * memory: optimizer state moved off the card (Zero From Scratch, item 11),
 * which the step kernels then read and write in place over the host link. */
int zg_bind(zg_ctx *ctx, float *w, float *m, float *v, uint16_t *params_bf16);

/* One whole step: zg_grad_norm then zg_shard_step on `stream`.
 * grad_ptrs: host array of P device pointers, each a bf16 buffer of N
 * elements (rank r's gradient times loss_scale); read during the call only.
 * loss_scale: finite and > 0. The skip decision stays on the device. */
int zg_step(zg_ctx *ctx, const uint16_t *const *grad_ptrs, float loss_scale, zg_stream stream);

/* First half of a step: the global norm (item 7's reduce-scatter, summed and
 * squared, then one scalar all-reduce, here an exact sum of per-chunk
 * partial sums rounded once to binary64, so the result does not depend on
 * how the work was spread over the GPU), the found-inf decision, the clip
 * factor and the next bias corrections, all left in device memory. Reads 2P
 * bytes per parameter. The exact sum's 64-bit digit words hold any N below
 * 2^38 (2.7e11 elements; a rank's bf16 gradient of that length would need
 * 550 GB of device memory). */
int zg_grad_norm(zg_ctx *ctx, const uint16_t *const *grad_ptrs, float loss_scale, zg_stream stream);

/* The first half of a step taken bucket by bucket, so each bucket's share of
 * the norm can be computed while later layers are still producing their
 * gradients (Zero From Scratch, item 13: sending each bucket while later
 * layers compute). The clip needs the norm of all N, so the AdamW update
 * still waits for the last bucket: that bucket's norm and the step pass are
 * the part that cannot be hidden. Buckets are contiguous flat ranges
 * [lo, hi) submitted in order on one stream: the first carries
 * ZG_BUCKET_FIRST and starts at 0, each next starts where the previous
 * ended, the last carries ZG_BUCKET_LAST and ends at N (one bucket may carry
 * both). lo must be a multiple of 8. Each bucket's sum of squares is added,
 * in submission order, to a running fp64 sum on the device; the last bucket
 * makes the same decision zg_grad_norm makes. grad_ptrs point at the start of
 * the full P buffers (not at the bucket). Out-of-order, gapped or unterminated
 * sequences are refused with ZG_ERR_INVALID_ARG before anything launches.
 * With ZG_VARIANT_STAGED each bucket also stores its part of the gradient. */
#define ZG_BUCKET_FIRST 1
#define ZG_BUCKET_LAST 2
int zg_grad_norm_bucket(zg_ctx *ctx, const uint16_t *const *grad_ptrs, int64_t lo, int64_t hi, float loss_scale,
                        int flags, zg_stream stream);

/* Second half: the fused reduce-scatter + unscale + clip + AdamW + bf16
 * all-gather over every shard, using the decision of the preceding
 * zg_grad_norm (items 3, 6, 7). Reads 2P + 12 and writes 14 bytes per
 * parameter. Call exactly once after each zg_grad_norm; a second call finds
 * the norm consumed, writes nothing and reports ZG_ERR_STALE_NORM in the
 * status. On a skipped step it writes nothing. */
int zg_shard_step(zg_ctx *ctx, const uint16_t *const *grad_ptrs, float loss_scale, zg_stream stream);

/* MXFP8-encode one rank's bf16 buffer of n elements (Zero From Scratch,
 * item 14): per block k of 32 elements [32k, 32k+32), amax = max |x|;
 * e = floor(log2 amax) - 8 clamped to [-127, 127] (e = -127 for an all-zero
 * block); scales[k] = e + 127 (E8M0); codes[i] = E4M3(x_i * 2^-e), round to
 * nearest even, magnitudes at or above 448 saturate to 448, signs kept.
 * A block holding an infinity or NaN gets scale 0xFF and codes 0x7F (NaN).
 * Elements past n count as zero in the last block's amax and get no code.
 * codes: n bytes; scales: ceil(n/32) bytes; both device memory. n >= 0. */
int zg_quant_mxfp8(const uint16_t *in, int64_t n, uint8_t *codes, uint8_t *scales, zg_stream stream);

/* Whole step from MX-encoded gradients: codes[r] (N bytes) and scales[r]
 * (ceil(N/32) bytes) are rank r's zg_quant_mxfp8 output for its N-element
 * buffer. Each rank value is decoded as E4M3(code) * 2^(scale - 127) before
 * the rank-ordered sum; the rest is zg_step. */
int zg_step_mxfp8(zg_ctx *ctx, const uint8_t *const *codes, const uint8_t *const *scales,
                  float loss_scale, zg_stream stream);

/* The two halves of zg_step_mxfp8, for separate timing. */
int zg_grad_norm_mxfp8(zg_ctx *ctx, const uint8_t *const *codes, const uint8_t *const *scales,
                       float loss_scale, zg_stream stream);
int zg_shard_step_mxfp8(zg_ctx *ctx, const uint8_t *const *codes, const uint8_t *const *scales,
                        float loss_scale, zg_stream stream);

/* The MXFP8 wire path's encode and norm pass in one launch, for gradients
 * that are all on this GPU: every rank's bf16 buffer grad_ptrs[r] (N
 * elements, 16-byte aligned device memory) is encoded into codes[r] (N
 * bytes, 16-byte aligned) and scales[r] (ceil(N/32) bytes) exactly as
 * zg_quant_mxfp8 encodes it, and the global norm, found-inf decision and
 * clip factor are taken from the same codes decoded in registers, exactly as
 * zg_grad_norm_mxfp8 decodes them (its norm agrees with that pass's to
 * rounding: the same per-element values, summed in another order). It sums
 * the squares exactly as zg_grad_norm does, so on gradients MXFP8 holds
 * exactly the two give the same bits. Follow it with zg_shard_step_mxfp8 on the same codes
 * and scales. It reads 2P and writes P(1 + 1/32) bytes per parameter, instead
 * of the P encodes plus a norm pass that reads the P(1 + 1/32) bytes back.
 * With ZG_VARIANT_STAGED it also stores the reduced gradient, as the MX norm
 * pass does. Errors as zg_grad_norm_mxfp8. */
int zg_quant_norm_mxfp8(zg_ctx *ctx, const uint16_t *const *grad_ptrs, uint8_t *const *codes,
                        uint8_t *const *scales, float loss_scale, zg_stream stream);

/* Wait for `stream`, then copy out the step scalars. Reports and clears the
 * sticky device status. This is the only device-to-host read of a step. */
int zg_get_info(zg_ctx *ctx, zg_stream stream, zg_step_info *info);

/* Resume: set the applied-step count to t (0 <= t <= 2^62); the running
 * powers b1^t and b2^t are rebuilt on the host by t multiplications from 1,
 * as an uninterrupted run forms them, so steps after a resume match an
 * uninterrupted run bit for bit. Any norm pass not yet followed by its shard
 * step is marked consumed (it predates the resume). Stream-ordered: one
 * single-thread kernel on `stream` writes the new values after the work
 * already queued there; the call does not wait, and no other stream or
 * context waits for it. Issue it on the stream that runs this context's
 * steps (or order the streams with events). */
int zg_set_step(zg_ctx *ctx, int64_t t, zg_stream stream);

/* Store the updated parameters as MXFP8 instead of bf16 (Zero From Scratch,
 * item 14: MXFP8 takes its share off stored state; bf16 parameters and
 * gradients as MXFP8 make a weight 16 - 2 * (2 - 33/32) bytes, 12 % less).
 * After this call every step encodes the new fp32 master weights block by
 * block with the rule of zg_quant_mxfp8 (E4M3 codes, one E8M0 scale per 32
 * elements, round to nearest even, saturating; a short last block counts
 * its missing elements as zero) and writes codes (N bytes, 16-byte aligned)
 * and scales (ceil(N/32) bytes), caller-owned device memory, in place of the
 * bf16 parameter buffer, which is then left untouched. The step pass moves
 * 2P + 24 + 33/32 bytes per parameter instead of 2P + 26. Both pointers NULL
 * goes back to bf16 parameters. Works with the plain and staged step
 * kernels and the MX gradient path; refused with ZG_VARIANT_TMA. */
int zg_bind_params_mxfp8(zg_ctx *ctx, uint8_t *codes, uint8_t *scales);

/* The staged variant keeps the reduce-scatter output the way a stage-two
 * rank holds it (Zero From Scratch, item 7: the reduce-scatter leaves each
 * rank its summed shard): the norm pass writes the unscaled, averaged fp32
 * gradient g_i (exactly the value the fused step would compute) into
 * `stage`, a caller-owned device buffer of N floats, 16-byte aligned, and the
 * step pass reads 4 bytes per parameter instead of the P bf16 replicas.
 * A whole step then moves 2P + 34 bytes per parameter instead of 4P + 26
 * (fewer from P = 5 on). Binding only records the pointer. */
int zg_bind_grad_stage(zg_ctx *ctx, float *stage);

/* Choose how bf16 steps run: ZG_VARIANT_LDG, ZG_VARIANT_TMA,
 * ZG_VARIANT_STAGED (which needs zg_bind_grad_stage first, else
 * ZG_ERR_NOT_BOUND) or ZG_VARIANT_SINGLE. The MX path follows
 * ZG_VARIANT_STAGED too (its norm pass stores the reduced gradient, its step
 * pass reads it) and otherwise runs its fused plain-load kernels.
 * ZG_VARIANT_SINGLE changes zg_step only (one launch for the whole step; its
 * grid-wide barrier waits at most the zg_set_wait_limit bound, with the same
 * statuses as the TMA variant's waits); zg_grad_norm and zg_shard_step called
 * on their own run the plain two-launch kernels. The TMA and one-launch
 * variants write bf16 parameters only: with MX parameters bound they are
 * refused. */
int zg_set_variant(zg_ctx *ctx, int variant);

/* Bound, in polls, on each device-side wait of the TMA variant and on the
 * grid-wide barrier of the one-launch variant (default a few million, far
 * above any healthy wait). A wait that runs out makes the
 * kernel drain its own copies, skip its remaining work and leave the step
 * uncommitted (the step count stays, the norm is consumed). The status then
 * tells the caller what state it is in: ZG_ERR_DEVICE_TIMEOUT when no CTA
 * had written anything yet (w, m, v and the parameters are untouched; run
 * the norm pass and the step again), ZG_ERR_STATE_PARTIAL when some tiles
 * had already been written (w, m, v and the parameters hold a mix of updated
 * and old values and must be restored from a checkpoint before stepping
 * again). 0 makes every first poll run out (used to test that path). */
int zg_set_wait_limit(zg_ctx *ctx, int64_t polls);

/* Stage three: parameters gathered just in time (DeepSpeed documentation
 * review, paragraph on the three stages: the parameters themselves are split,
 * gathered for each layer's computation and released afterwards; Zero From
 * Scratch, items 9 and 18, the third flag). Rank r keeps only the parameters
 * [r*S, (r+1)*S) in shards[r], a device buffer of S = zg_shard_len(ctx) bf16
 * values (the bf16 parameter vector zg_bind received is exactly these P
 * shards end to end: shards[r] = params + r*S). The call writes the flat
 * parameters [lo, hi), 0 <= lo <= hi <= N, into out[0, hi - lo): out[j] is
 * element (lo + j) mod S of shard (lo + j) / S. On one GPU this stands for the
 * all-gather every rank runs before the layer; `out` is the caller's
 * (device) working buffer, which it releases or reuses after the layer.
 * Every shards[r] and out must be 16-byte aligned device memory (else
 * ZG_ERR_MISALIGNED); NULL pointers or a range outside [0, N) give
 * ZG_ERR_INVALID_ARG; lo == hi does nothing. An lo that is a multiple of 8
 * takes the vector path (one 16-byte load and store per 8 values). Moves 4
 * bytes per gathered parameter. Stream-ordered, no allocation. */
int zg_gather_params(const zg_ctx *ctx, const uint16_t *const *shards, int64_t lo, int64_t hi, uint16_t *out,
                     zg_stream stream);

/* zg_gather_params carried out by the copy engines instead of a kernel: one
 * device-to-device cudaMemcpyAsync per shard the range crosses (at most P),
 * enqueued on `stream`. Same arguments, result and errors; it occupies no
 * SM, so it can run beside a computation that fills every SM (the layer
 * before), which a gather kernel cannot. */
int zg_gather_params_dma(const zg_ctx *ctx, const uint16_t *const *shards, int64_t lo, int64_t hi, uint16_t *out,
                         zg_stream stream);

/* The same gather from parameter shards stored as MXFP8 (Zero From Scratch,
 * item 14: MXFP8 on stored state, the layout zg_bind_params_mxfp8 writes):
 * codes[r] holds S E4M3 codes of rank r (16-byte aligned) and scales[r] its
 * S/32 E8M0 scales. Each gathered element is decoded to its exact binary32
 * value code * 2^(scale - 127) and rounded to bf16 (nearest even; this only
 * acts below 2^-126, since a decoded value has at most four significant
 * bits); a NaN code or scale gathers as 0x7FC0. An lo that is a multiple of
 * 8 takes the vector path (8 codes in, one 16-byte store out). Reads 1 + 1/32 and writes 2 bytes per gathered
 * parameter. Errors as zg_gather_params. */
int zg_gather_params_mxfp8(const zg_ctx *ctx, const uint8_t *const *codes, const uint8_t *const *scales, int64_t lo,
                           int64_t hi, uint16_t *out, zg_stream stream);

/* Measurement aid: copy `bytes` (a multiple of 16, both pointers 16-byte
 * aligned device memory) with a plain streaming copy kernel; its time gives
 * the achievable HBM bandwidth in the same run. */
int zg_probe_copy(const void *src, void *dst, int64_t bytes, zg_stream stream);

/* The norm pass for callers that cannot allocate device memory. No passage
 * of the pages corresponds to it: it exists for callers such as a process
 * whose framework allocator has reserved nearly all device memory, a
 * latency-critical loop that cannot afford the synchronisation a cudaMalloc
 * or cudaFree may imply, or a plug-in handed device buffers with no way to
 * release memory of its own. It computes what zg_grad_norm computes for the
 * same gradients (same kernel, same summation) and writes
 *   out[0] = sum of squares of the unscaled, averaged gradient,
 *   out[1] = its square root (the global norm),
 * to `out`, a caller-owned device buffer of two doubles (8-byte aligned).
 * A non-finite out[0] means some gradient is infinite or NaN.
 * grad_ptrs: host array of P device pointers to bf16 buffers of N elements
 * (16-byte aligned); 1 <= P <= 16, 1 <= N < 2^62; loss_scale finite > 0;
 * grad_average 0 or 1. Other values are rejected with ZG_ERR_INVALID_ARG or
 * ZG_ERR_MISALIGNED and a message in zg_last_error.
 * It allocates nothing: no cudaMalloc, no cudaFree, no allocating library
 * call. Its scratch is a fixed 4,736-byte array inside the library's device
 * image (a result block and the norm pass's work array); every GPU that loads
 * the library holds that array until the process exits. The first call on a device looks up the array's
 * device address (cudaGetSymbolAddress), so make that first call before any
 * stream capture; after a device reset (a new CUDA context on the device) the
 * next call looks the address up again, and should likewise come before any
 * capture. Every pointer is checked for the kind of memory behind it, asked
 * of the driver on every call (nothing is remembered). All calls on a device
 * share the array and each clears it first: calls that overlap on the GPU
 * race and must be ordered by the caller (one stream, or events). Stream-ordered; does not wait. */
int zg_grad_norm_noalloc(const uint16_t *const *grad_ptrs, int p, int64_t n, float loss_scale, int grad_average,
                         double *out, zg_stream stream);

/* Free the context and its workspace (after the stream work using it is done). */
void zg_destroy(zg_ctx *ctx);

const char *zg_strerror(int code);
const char *zg_last_error(void); /* this thread's last detailed message */
int zg_version(void);

#ifdef __cplusplus
}
#endif

#endif /* ZG_H */
