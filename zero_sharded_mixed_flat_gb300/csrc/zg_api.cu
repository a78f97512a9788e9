// zg_api.cu -- the C ABI declared in include/zg.h: argument checks, the
// small device workspace, and the launches. No kernel runs on the host and
// no call here allocates anything per step.
#include <cuda_runtime.h>
#include <math.h>
#include <stdarg.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include <map>
#include <mutex>
#include <unordered_map>
#include <utility>

#include "zg.h"
#include "zg_launch.h"

struct zg_ctx {
    int64_t n;
    int p;
    int64_t s;
    zg_hparams hp;
    zg::FinalizeK fk;
    zg::StepK k;
    float *w, *m, *v;
    uint16_t *params;
    bool bound;
    float *stage;  // caller's fp32 buffer for the staged variant, or NULL
    uint8_t *pcodes;      // MX parameter codes (written instead of bf16 params), or NULL
    uint8_t *pscales;     // their E8M0 scales
    int64_t bucket_next;  // where the next bucket of an open bucketed norm must start
    bool bucket_open;     // a bucketed norm has started and not yet seen its last bucket
    int device;
    zg::Scalars *d_sc;
    double *d_partials;
    int partials_cap;
    unsigned long long *d_work;  // the step and norm passes' work array (zg::kWorkWords words)
    zg::Scalars *h_sc;
    int variant;
    long long wait_limit;
};

namespace {

thread_local char g_err[512] = "";

int fail(int code, const char *fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
    return code;
}

int cuda_fail(cudaError_t e, const char *what)
{
    return fail(ZG_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorString(e), cudaGetErrorName(e));
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

constexpr int kPartialsCap = 8192;
constexpr long long kDefaultWaitLimit = 4000000;

int check_ctx(const zg_ctx *ctx, bool need_bound)
{
    if (!ctx) return fail(ZG_ERR_INVALID_ARG, "context is NULL");
    if (need_bound && !ctx->bound) return fail(ZG_ERR_NOT_BOUND, "zg_bind has not been called");
    return ZG_OK;
}

int check_scale(float loss_scale)
{
    if (!(loss_scale > 0.0f) || !isfinite(loss_scale))
        return fail(ZG_ERR_INVALID_ARG, "loss_scale must be finite and > 0 (got %g)", double(loss_scale));
    return ZG_OK;
}

template <class T>
int check_rank_ptrs(const zg_ctx *ctx, const T *const *ptrs, const char *what, bool need_align)
{
    if (!ptrs) return fail(ZG_ERR_INVALID_ARG, "%s array is NULL", what);
    char name[64];
    for (int r = 0; r < ctx->p; ++r) {
        if (!ptrs[r]) return fail(ZG_ERR_INVALID_ARG, "%s[%d] is NULL", what, r);
        if (need_align && !aligned16(ptrs[r])) return fail(ZG_ERR_MISALIGNED, "%s[%d] is not 16-byte aligned", what, r);
        snprintf(name, sizeof name, "%s[%d]", what, r);
        if (int rc = zg::check_memory(ptrs[r], false, name)) return rc;
    }
    return ZG_OK;
}

float inv_scale(const zg_ctx *ctx, float loss_scale)
{
    const double denom = double(loss_scale) * (ctx->hp.grad_average ? double(ctx->p) : 1.0);
    return float(1.0 / denom);
}

zg::State state_of(const zg_ctx *ctx)
{
    return zg::State{ctx->w, ctx->m, ctx->v, ctx->params, ctx->pcodes, ctx->pscales, ctx->d_work};
}

// Checks shared by the gathers: a context, a range inside [0, N) and a
// 16-byte aligned output. Returns a ZG_ERR_* code, ZG_OK to go on, or
// kNothingToDo for an empty range (which needs no pointers at all).
constexpr int kNothingToDo = 1;

int check_gather(const zg_ctx *ctx, int64_t lo, int64_t hi, const void *out)
{
    if (int rc = check_ctx(ctx, false)) return rc;
    if (lo < 0 || hi < lo || hi > ctx->n)
        return fail(ZG_ERR_INVALID_ARG, "range [%lld, %lld) is not inside [0, N = %lld)", (long long)lo,
                    (long long)hi, (long long)ctx->n);
    if (lo == hi) return kNothingToDo;
    if (!out) return fail(ZG_ERR_INVALID_ARG, "out is NULL");
    if (!aligned16(out)) return fail(ZG_ERR_MISALIGNED, "out must be 16-byte aligned");
    return zg::check_memory(out, false, "out");
}

int finish_launch(cudaError_t e, const char *what) { return e == cudaSuccess ? ZG_OK : cuda_fail(e, what); }

}  // namespace

namespace zg {

int wave_blocks(const void *kernel, int threads, size_t smem)
{
    static std::mutex mu;
    static std::map<std::pair<int, const void *>, int> cache;
    int dev = 0;
    cudaGetDevice(&dev);
    std::lock_guard<std::mutex> lock(mu);
    auto key = std::make_pair(dev, kernel);
    auto it = cache.find(key);
    if (it != cache.end()) return it->second;
    int sms = 0, per_sm = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, smem);
    int blocks = sms * per_sm;
    if (blocks < 1) blocks = 1;
    cache[key] = blocks;
    return blocks;
}

int norm_blocks_cap() { return kPartialsCap; }

// What cudaPointerGetAttributes said about a pointer the library accepted:
// its memory type and device. Kept per pointer value so repeated calls with
// the same buffers (every step) ask the driver once; only accepted pointers
// are remembered, so a refused one is looked at again on its next use.
namespace {
struct Kind {
    int type;
    int device;
};
std::mutex g_kind_mu;
std::unordered_map<uintptr_t, Kind> g_kinds;
constexpr size_t kKindCacheCap = 1 << 16;
}  // namespace

// The driver's answer for one pointer, checked against what the argument
// accepts; `a` receives the attributes.
int classify_memory(const void *p, bool host_ok, const char *what, int dev, cudaPointerAttributes &a)
{
    cudaError_t e = cudaPointerGetAttributes(&a, p);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return cuda_fail(e, what);
    }
    switch (a.type) {
    case cudaMemoryTypeDevice:
    case cudaMemoryTypeManaged:
        if (a.device != dev)
            return fail(ZG_ERR_INVALID_ARG, "%s is memory of device %d, but the current device is %d", what, a.device,
                        dev);
        break;
    case cudaMemoryTypeHost:
        if (!host_ok)
            return fail(ZG_ERR_INVALID_ARG, "%s is pinned host memory; it must be device memory", what);
        if (a.devicePointer != p)
            return fail(ZG_ERR_INVALID_ARG,
                        "%s is pinned host memory that the device does not see at the same address "
                        "(pin it mapped, e.g. cudaHostRegisterMapped)",
                        what);
        break;
    default:
        return fail(ZG_ERR_INVALID_ARG, "%s is not memory CUDA knows (ordinary host memory?); it must be %s", what,
                    host_ok ? "device memory or pinned host memory" : "device memory");
    }
    return ZG_OK;
}

int check_memory_uncached(const void *p, bool host_ok, const char *what)
{
    int dev = 0;
    const cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, what);
    cudaPointerAttributes a;
    return classify_memory(p, host_ok, what, dev, a);
}

int check_memory(const void *p, bool host_ok, const char *what)
{
    int dev = 0;
    const cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, what);
    const uintptr_t key = reinterpret_cast<uintptr_t>(p);
    {
        std::lock_guard<std::mutex> lock(g_kind_mu);
        auto it = g_kinds.find(key);
        if (it != g_kinds.end() && (it->second.type != cudaMemoryTypeHost || host_ok) &&
            (it->second.type == cudaMemoryTypeHost || it->second.device == dev))
            return ZG_OK;
    }
    cudaPointerAttributes a;
    if (int rc = classify_memory(p, host_ok, what, dev, a)) return rc;
    std::lock_guard<std::mutex> lock(g_kind_mu);
    if (g_kinds.size() >= kKindCacheCap) g_kinds.clear();
    g_kinds[key] = Kind{int(a.type), a.device};
    return ZG_OK;
}

int report_error(int code, const char *msg) { return fail(code, "%s", msg); }

// Resume at applied-step count t: the step count and the running powers, and
// the pending norm (if any) marked consumed, written in stream order.
__global__ void resume_kernel(Scalars *sc, int64_t t, double b1p, double b2p)
{
    sc->t = t;
    sc->b1p = b1p;
    sc->b2p = b2p;
    sc->step_gen = sc->norm_gen;
}

}  // namespace zg

extern "C" {

int zg_version(void) { return 100; }

const char *zg_last_error(void) { return g_err; }

const char *zg_strerror(int code)
{
    switch (code) {
    case ZG_OK: return "ok";
    case ZG_ERR_INVALID_ARG: return "invalid argument";
    case ZG_ERR_MISALIGNED: return "pointer not 16-byte aligned";
    case ZG_ERR_NOT_BOUND: return "optimizer state not bound (call zg_bind)";
    case ZG_ERR_CUDA: return "CUDA error";
    case ZG_ERR_DEVICE_TIMEOUT: return "a bounded device-side wait ran out";
    case ZG_ERR_STALE_NORM: return "shard step without a fresh norm pass";
    case ZG_ERR_NO_MEMORY: return "out of memory";
    case ZG_ERR_STATE_PARTIAL: return "a bounded device-side wait ran out after part of the state was written";
    default: return "unknown status";
    }
}

int zg_init(int64_t n, int p, const zg_hparams *hp, zg_ctx **out)
{
    if (!out) return fail(ZG_ERR_INVALID_ARG, "out is NULL");
    *out = nullptr;
    if (n < 1 || n >= (int64_t(1) << 62)) return fail(ZG_ERR_INVALID_ARG, "N must be in [1, 2^62) (got %lld)", (long long)n);
    if (p < 1 || p > ZG_MAX_RANKS) return fail(ZG_ERR_INVALID_ARG, "P must be in [1, %d] (got %d)", ZG_MAX_RANKS, p);
    if (!hp) return fail(ZG_ERR_INVALID_ARG, "hparams is NULL");
    const double vals[] = {hp->lr, hp->beta1, hp->beta2, hp->eps, hp->weight_decay, hp->max_grad_norm, hp->norm_eps};
    for (double x : vals)
        if (!isfinite(x)) return fail(ZG_ERR_INVALID_ARG, "hyperparameters must be finite");
    if (hp->lr < 0 || hp->eps < 0 || hp->norm_eps < 0) return fail(ZG_ERR_INVALID_ARG, "lr, eps and norm_eps must be >= 0");
    if (!(hp->beta1 >= 0 && hp->beta1 < 1 && hp->beta2 >= 0 && hp->beta2 < 1))
        return fail(ZG_ERR_INVALID_ARG, "betas must be in [0, 1)");
    if (hp->grad_average != 0 && hp->grad_average != 1) return fail(ZG_ERR_INVALID_ARG, "grad_average must be 0 or 1");

    zg_ctx *ctx = new (std::nothrow) zg_ctx();
    if (!ctx) return fail(ZG_ERR_NO_MEMORY, "host allocation of the context failed");
    ctx->n = n;
    ctx->p = p;
    int64_t s = (n + p - 1) / p;
    ctx->s = (s + 31) / 32 * 32;
    ctx->hp = *hp;
    ctx->fk = zg::FinalizeK{hp->beta1, hp->beta2, hp->max_grad_norm, hp->norm_eps};
    ctx->k = zg::StepK{float(hp->beta1),       float(hp->beta2), float(1.0 - hp->beta1), float(1.0 - hp->beta2),
                       float(hp->eps),         float(hp->lr),    float(hp->lr * hp->weight_decay)};
    ctx->variant = ZG_VARIANT_LDG;
    ctx->wait_limit = kDefaultWaitLimit;
    ctx->partials_cap = zg::norm_blocks_cap();
    cudaError_t e = cudaGetDevice(&ctx->device);
    if (e == cudaSuccess) e = cudaMalloc(&ctx->d_sc, sizeof(zg::Scalars));
    if (e == cudaSuccess) e = cudaMalloc(&ctx->d_partials, sizeof(double) * ctx->partials_cap);
    if (e == cudaSuccess) e = cudaMalloc(&ctx->d_work, sizeof(unsigned long long) * zg::kWorkWords);
    if (e == cudaSuccess) e = cudaMemset(ctx->d_work, 0, sizeof(unsigned long long) * zg::kWorkWords);
    if (e == cudaSuccess) e = cudaMallocHost(&ctx->h_sc, sizeof(zg::Scalars));
    if (e == cudaSuccess) {
        memset(ctx->h_sc, 0, sizeof(zg::Scalars));
        ctx->h_sc->b1p = 1.0;
        ctx->h_sc->b2p = 1.0;
        ctx->h_sc->clip = 1.0f;
        e = cudaMemcpy(ctx->d_sc, ctx->h_sc, sizeof(zg::Scalars), cudaMemcpyHostToDevice);
    }
    if (e != cudaSuccess) {
        int rc = cuda_fail(e, "zg_init workspace");
        cudaGetLastError();
        zg_destroy(ctx);
        return rc;
    }
    *out = ctx;
    return ZG_OK;
}

int64_t zg_shard_len(const zg_ctx *ctx) { return ctx ? ctx->s : -1; }

int zg_bind(zg_ctx *ctx, float *w, float *m, float *v, uint16_t *params_bf16)
{
    if (int rc = check_ctx(ctx, false)) return rc;
    if (!w || !m || !v || !params_bf16) return fail(ZG_ERR_INVALID_ARG, "state pointers must not be NULL");
    if (!aligned16(w) || !aligned16(m) || !aligned16(v) || !aligned16(params_bf16))
        return fail(ZG_ERR_MISALIGNED, "state pointers must be 16-byte aligned");
    if (int rc = zg::check_memory(w, true, "w")) return rc;
    if (int rc = zg::check_memory(m, true, "m")) return rc;
    if (int rc = zg::check_memory(v, true, "v")) return rc;
    if (int rc = zg::check_memory(params_bf16, false, "params")) return rc;
    ctx->w = w;
    ctx->m = m;
    ctx->v = v;
    ctx->params = params_bf16;
    ctx->bound = true;
    return ZG_OK;
}

int zg_bind_params_mxfp8(zg_ctx *ctx, uint8_t *codes, uint8_t *scales)
{
    if (int rc = check_ctx(ctx, false)) return rc;
    if (!codes && !scales) {
        ctx->pcodes = nullptr;
        ctx->pscales = nullptr;
        return ZG_OK;
    }
    if (!codes || !scales) return fail(ZG_ERR_INVALID_ARG, "codes and scales must both be set (or both NULL)");
    if (!aligned16(codes)) return fail(ZG_ERR_MISALIGNED, "codes must be 16-byte aligned");
    if (ctx->variant == ZG_VARIANT_TMA || ctx->variant == ZG_VARIANT_SINGLE)
        return fail(ZG_ERR_INVALID_ARG,
                    "MX parameters are written by the plain and staged step kernels, not the TMA or one-launch ones");
    if (int rc = zg::check_memory(codes, false, "codes")) return rc;
    if (int rc = zg::check_memory(scales, false, "scales")) return rc;
    ctx->pcodes = codes;
    ctx->pscales = scales;
    return ZG_OK;
}

int zg_bind_grad_stage(zg_ctx *ctx, float *stage)
{
    if (int rc = check_ctx(ctx, false)) return rc;
    if (!stage) return fail(ZG_ERR_INVALID_ARG, "stage must not be NULL");
    if (!aligned16(stage)) return fail(ZG_ERR_MISALIGNED, "stage must be 16-byte aligned");
    if (int rc = zg::check_memory(stage, false, "stage")) return rc;
    ctx->stage = stage;
    return ZG_OK;
}

int zg_grad_norm(zg_ctx *ctx, const uint16_t *const *grad_ptrs, float loss_scale, zg_stream stream)
{
    if (int rc = check_ctx(ctx, false)) return rc;
    if (int rc = check_scale(loss_scale)) return rc;
    if (int rc = check_rank_ptrs(ctx, grad_ptrs, "grad_ptrs", true)) return rc;
    return finish_launch(zg::launch_norm_bf16(ctx->p, grad_ptrs, ctx->n, inv_scale(ctx, loss_scale), ctx->d_work,
                                              ctx->d_sc, ctx->fk, stream,
                                              ctx->variant == ZG_VARIANT_STAGED ? ctx->stage : nullptr),
                         "norm pass launch");
}

int zg_grad_norm_bucket(zg_ctx *ctx, const uint16_t *const *grad_ptrs, int64_t lo, int64_t hi, float loss_scale,
                        int flags, zg_stream stream)
{
    if (int rc = check_ctx(ctx, false)) return rc;
    if (int rc = check_scale(loss_scale)) return rc;
    if (int rc = check_rank_ptrs(ctx, grad_ptrs, "grad_ptrs", true)) return rc;
    if (flags & ~(ZG_BUCKET_FIRST | ZG_BUCKET_LAST)) return fail(ZG_ERR_INVALID_ARG, "unknown bucket flags %d", flags);
    if (lo < 0 || hi <= lo || hi > ctx->n)
        return fail(ZG_ERR_INVALID_ARG, "bucket [%lld, %lld) must be a non-empty range inside [0, N)", (long long)lo,
                    (long long)hi);
    if (lo % 8) return fail(ZG_ERR_INVALID_ARG, "bucket starts must be multiples of 8 elements (got %lld)", (long long)lo);
    if (flags & ZG_BUCKET_FIRST) {
        if (lo != 0) return fail(ZG_ERR_INVALID_ARG, "the first bucket must start at 0");
    } else {
        if (!ctx->bucket_open)
            return fail(ZG_ERR_INVALID_ARG, "no bucketed norm is open (the first bucket carries ZG_BUCKET_FIRST)");
        if (lo != ctx->bucket_next)
            return fail(ZG_ERR_INVALID_ARG, "buckets must be contiguous and in order: expected start %lld, got %lld",
                        (long long)ctx->bucket_next, (long long)lo);
    }
    if ((flags & ZG_BUCKET_LAST) && hi != ctx->n) return fail(ZG_ERR_INVALID_ARG, "the last bucket must end at N");
    if (!(flags & ZG_BUCKET_LAST) && hi == ctx->n)
        return fail(ZG_ERR_INVALID_ARG, "a bucket that ends at N must carry ZG_BUCKET_LAST");
    const uint16_t *g[ZG_MAX_RANKS];
    for (int r = 0; r < ctx->p; ++r) g[r] = grad_ptrs[r] + lo;
    float *stage = ctx->variant == ZG_VARIANT_STAGED ? ctx->stage + lo : nullptr;
    const int mode = zg::kNormBucket | ((flags & ZG_BUCKET_FIRST) ? zg::kNormFirst : 0) |
                     ((flags & ZG_BUCKET_LAST) ? zg::kNormLast : 0);
    const int rc = finish_launch(zg::launch_norm_bf16(ctx->p, g, hi - lo, inv_scale(ctx, loss_scale), ctx->d_work,
                                                      ctx->d_sc, ctx->fk, stream, stage, mode),
                                 "bucket norm launch");
    if (rc == ZG_OK) {
        ctx->bucket_open = !(flags & ZG_BUCKET_LAST);
        ctx->bucket_next = hi;
    }
    return rc;
}

int zg_shard_step(zg_ctx *ctx, const uint16_t *const *grad_ptrs, float loss_scale, zg_stream stream)
{
    if (int rc = check_ctx(ctx, true)) return rc;
    if (int rc = check_scale(loss_scale)) return rc;
    if (int rc = check_rank_ptrs(ctx, grad_ptrs, "grad_ptrs", true)) return rc;
    if (ctx->variant == ZG_VARIANT_STAGED)
        return finish_launch(zg::launch_step_staged(ctx->stage, ctx->n, ctx->k, state_of(ctx), ctx->d_sc, stream),
                             "staged step pass launch");
    if (ctx->variant == ZG_VARIANT_TMA)
        return finish_launch(zg::launch_step_tma(ctx->p, grad_ptrs, ctx->n, inv_scale(ctx, loss_scale), ctx->k,
                                                 state_of(ctx), ctx->d_sc, ctx->wait_limit, stream),
                             "TMA step pass launch");
    return finish_launch(zg::launch_step_bf16(ctx->p, grad_ptrs, ctx->n, inv_scale(ctx, loss_scale), ctx->k,
                                              state_of(ctx), ctx->d_sc, stream),
                         "step pass launch");
}

int zg_step(zg_ctx *ctx, const uint16_t *const *grad_ptrs, float loss_scale, zg_stream stream)
{
    if (int rc = check_ctx(ctx, true)) return rc;
    if (ctx->variant == ZG_VARIANT_SINGLE) {
        if (int rc = check_scale(loss_scale)) return rc;
        if (int rc = check_rank_ptrs(ctx, grad_ptrs, "grad_ptrs", true)) return rc;
        return finish_launch(zg::launch_step_whole(ctx->p, grad_ptrs, ctx->n, inv_scale(ctx, loss_scale), ctx->k,
                                                   state_of(ctx), ctx->d_sc, ctx->fk, ctx->wait_limit, stream),
                             "whole-step launch");
    }
    if (int rc = zg_grad_norm(ctx, grad_ptrs, loss_scale, stream)) return rc;
    return zg_shard_step(ctx, grad_ptrs, loss_scale, stream);
}

int zg_quant_mxfp8(const uint16_t *in, int64_t n, uint8_t *codes, uint8_t *scales, zg_stream stream)
{
    if (n < 0 || n >= (int64_t(1) << 62)) return fail(ZG_ERR_INVALID_ARG, "n must be in [0, 2^62)");
    if (n == 0) return ZG_OK;
    if (!in || !codes || !scales) return fail(ZG_ERR_INVALID_ARG, "pointers must not be NULL");
    if (!aligned16(in) || !aligned16(codes)) return fail(ZG_ERR_MISALIGNED, "in and codes must be 16-byte aligned");
    if (int rc = zg::check_memory(in, false, "in")) return rc;
    if (int rc = zg::check_memory(codes, false, "codes")) return rc;
    if (int rc = zg::check_memory(scales, false, "scales")) return rc;
    return finish_launch(zg::launch_quant(in, n, codes, scales, stream), "MXFP8 encoder launch");
}

int zg_grad_norm_mxfp8(zg_ctx *ctx, const uint8_t *const *codes, const uint8_t *const *scales, float loss_scale,
                       zg_stream stream)
{
    if (int rc = check_ctx(ctx, false)) return rc;
    if (int rc = check_scale(loss_scale)) return rc;
    if (int rc = check_rank_ptrs(ctx, codes, "codes", true)) return rc;
    if (int rc = check_rank_ptrs(ctx, scales, "scales", false)) return rc;
    return finish_launch(zg::launch_norm_mx(ctx->p, codes, scales, ctx->n, inv_scale(ctx, loss_scale), ctx->d_partials,
                                            ctx->partials_cap, ctx->d_sc, ctx->fk, stream,
                                            ctx->variant == ZG_VARIANT_STAGED ? ctx->stage : nullptr),
                         "MX norm pass launch");
}

int zg_quant_norm_mxfp8(zg_ctx *ctx, const uint16_t *const *grad_ptrs, uint8_t *const *codes,
                        uint8_t *const *scales, float loss_scale, zg_stream stream)
{
    if (int rc = check_ctx(ctx, false)) return rc;
    if (int rc = check_scale(loss_scale)) return rc;
    if (int rc = check_rank_ptrs(ctx, grad_ptrs, "grad_ptrs", true)) return rc;
    if (int rc = check_rank_ptrs(ctx, codes, "codes", true)) return rc;
    if (int rc = check_rank_ptrs(ctx, scales, "scales", false)) return rc;
    return finish_launch(zg::launch_quant_norm(ctx->p, grad_ptrs, codes, scales, ctx->n, inv_scale(ctx, loss_scale),
                                               ctx->d_work, ctx->d_sc, ctx->fk, stream,
                                               ctx->variant == ZG_VARIANT_STAGED ? ctx->stage : nullptr),
                         "MX encode and norm pass launch");
}

int zg_shard_step_mxfp8(zg_ctx *ctx, const uint8_t *const *codes, const uint8_t *const *scales, float loss_scale,
                        zg_stream stream)
{
    if (int rc = check_ctx(ctx, true)) return rc;
    if (int rc = check_scale(loss_scale)) return rc;
    if (int rc = check_rank_ptrs(ctx, codes, "codes", true)) return rc;
    if (int rc = check_rank_ptrs(ctx, scales, "scales", false)) return rc;
    if (ctx->variant == ZG_VARIANT_STAGED)
        return finish_launch(zg::launch_step_staged(ctx->stage, ctx->n, ctx->k, state_of(ctx), ctx->d_sc, stream),
                             "staged step pass launch");
    return finish_launch(zg::launch_step_mx(ctx->p, codes, scales, ctx->n, inv_scale(ctx, loss_scale), ctx->k,
                                            state_of(ctx), ctx->d_sc, stream),
                         "MX step pass launch");
}

int zg_step_mxfp8(zg_ctx *ctx, const uint8_t *const *codes, const uint8_t *const *scales, float loss_scale,
                  zg_stream stream)
{
    if (int rc = check_ctx(ctx, true)) return rc;
    if (int rc = zg_grad_norm_mxfp8(ctx, codes, scales, loss_scale, stream)) return rc;
    return zg_shard_step_mxfp8(ctx, codes, scales, loss_scale, stream);
}

int zg_get_info(zg_ctx *ctx, zg_stream stream, zg_step_info *info)
{
    if (int rc = check_ctx(ctx, false)) return rc;
    if (!info) return fail(ZG_ERR_INVALID_ARG, "info is NULL");
    cudaError_t e = cudaMemcpyAsync(ctx->h_sc, ctx->d_sc, sizeof(zg::Scalars), cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return cuda_fail(e, "zg_get_info");
    const zg::Scalars &h = *ctx->h_sc;
    info->sumsq = h.sumsq;
    info->norm = h.norm;
    info->clip_coef = h.clip;
    info->found_inf = h.found_inf;
    info->step_t = h.t;
    info->status = h.status;
    if (h.status != 0) {
        e = cudaMemsetAsync(reinterpret_cast<char *>(ctx->d_sc) + offsetof(zg::Scalars, status), 0, sizeof(int), stream);
        if (e != cudaSuccess) return cuda_fail(e, "zg_get_info status reset");
    }
    return ZG_OK;
}

int zg_set_step(zg_ctx *ctx, int64_t t, zg_stream stream)
{
    if (int rc = check_ctx(ctx, false)) return rc;
    if (t < 0 || t > (int64_t(1) << 62)) return fail(ZG_ERR_INVALID_ARG, "t must be in [0, 2^62] (got %lld)", (long long)t);
    double b1p = 1.0, b2p = 1.0;
    for (int64_t i = 0; i < t; ++i) {
        b1p = b1p * ctx->hp.beta1;
        b2p = b2p * ctx->hp.beta2;
        if (b1p == 0.0 && b2p == 0.0) break;  // every further product is zero too
    }
    // one single-thread kernel on the caller's stream writes the step count,
    // the running powers and marks any pending norm consumed (it predates the
    // resume): ordered after the work already on the stream, and nothing
    // else on the device waits for it
    zg::resume_kernel<<<1, 1, 0, stream>>>(ctx->d_sc, t, b1p, b2p);
    return finish_launch(cudaGetLastError(), "zg_set_step");
}

int zg_set_variant(zg_ctx *ctx, int variant)
{
    if (int rc = check_ctx(ctx, false)) return rc;
    if (variant != ZG_VARIANT_LDG && variant != ZG_VARIANT_TMA && variant != ZG_VARIANT_STAGED &&
        variant != ZG_VARIANT_SINGLE)
        return fail(ZG_ERR_INVALID_ARG, "unknown variant %d", variant);
    if ((variant == ZG_VARIANT_TMA || variant == ZG_VARIANT_SINGLE) && ctx->pcodes)
        return fail(ZG_ERR_INVALID_ARG,
                    "the TMA and one-launch step kernels write bf16 parameters only (MX parameters are bound)");
    if (variant == ZG_VARIANT_STAGED && !ctx->stage)
        return fail(ZG_ERR_NOT_BOUND, "the staged variant needs zg_bind_grad_stage first");
    ctx->variant = variant;
    return ZG_OK;
}

int zg_set_wait_limit(zg_ctx *ctx, int64_t polls)
{
    if (int rc = check_ctx(ctx, false)) return rc;
    if (polls < 0) return fail(ZG_ERR_INVALID_ARG, "polls must be >= 0");
    ctx->wait_limit = polls;
    return ZG_OK;
}

int zg_gather_params(const zg_ctx *ctx, const uint16_t *const *shards, int64_t lo, int64_t hi, uint16_t *out,
                     zg_stream stream)
{
    if (int rc = check_gather(ctx, lo, hi, out)) return rc == kNothingToDo ? ZG_OK : rc;
    if (int rc = check_rank_ptrs(ctx, shards, "shards", true)) return rc;
    return finish_launch(zg::launch_gather(ctx->p, ctx->s, shards, lo, hi, out, stream), "parameter gather launch");
}

int zg_gather_params_dma(const zg_ctx *ctx, const uint16_t *const *shards, int64_t lo, int64_t hi, uint16_t *out,
                         zg_stream stream)
{
    if (int rc = check_gather(ctx, lo, hi, out)) return rc == kNothingToDo ? ZG_OK : rc;
    if (int rc = check_rank_ptrs(ctx, shards, "shards", true)) return rc;
    // one device-to-device copy per shard the range crosses (at most P)
    for (int64_t i = lo; i < hi;) {
        const int64_t r = i / ctx->s;
        const int64_t end = (r + 1) * ctx->s < hi ? (r + 1) * ctx->s : hi;
        const cudaError_t e = cudaMemcpyAsync(out + (i - lo), shards[r] + (i - r * ctx->s),
                                              size_t(end - i) * sizeof(uint16_t), cudaMemcpyDeviceToDevice, stream);
        if (e != cudaSuccess) return cuda_fail(e, "parameter gather copy");
        i = end;
    }
    return ZG_OK;
}

int zg_gather_params_mxfp8(const zg_ctx *ctx, const uint8_t *const *codes, const uint8_t *const *scales, int64_t lo,
                           int64_t hi, uint16_t *out, zg_stream stream)
{
    if (int rc = check_gather(ctx, lo, hi, out)) return rc == kNothingToDo ? ZG_OK : rc;
    if (int rc = check_rank_ptrs(ctx, codes, "codes", true)) return rc;
    if (int rc = check_rank_ptrs(ctx, scales, "scales", false)) return rc;
    return finish_launch(zg::launch_gather_mx(ctx->p, ctx->s, codes, scales, lo, hi, out, stream),
                         "MX parameter gather launch");
}

int zg_probe_copy(const void *src, void *dst, int64_t bytes, zg_stream stream)
{
    if (bytes < 0 || bytes % 16) return fail(ZG_ERR_INVALID_ARG, "bytes must be a non-negative multiple of 16");
    if (bytes == 0) return ZG_OK;
    if (!src || !dst) return fail(ZG_ERR_INVALID_ARG, "pointers must not be NULL");
    if (!aligned16(src) || !aligned16(dst)) return fail(ZG_ERR_MISALIGNED, "pointers must be 16-byte aligned");
    if (int rc = zg::check_memory(src, false, "src")) return rc;
    if (int rc = zg::check_memory(dst, false, "dst")) return rc;
    return finish_launch(zg::launch_copy(src, dst, bytes, stream), "copy probe launch");
}

void zg_destroy(zg_ctx *ctx)
{
    if (!ctx) return;
    if (ctx->d_sc) cudaFree(ctx->d_sc);
    if (ctx->d_partials) cudaFree(ctx->d_partials);
    if (ctx->d_work) cudaFree(ctx->d_work);
    if (ctx->h_sc) cudaFreeHost(ctx->h_sc);
    delete ctx;
}

}  // extern "C"
