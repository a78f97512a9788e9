/*
 * zg_oracle.c -- the oracle: a plain, slow CPU statement of the sharded
 * mixed-precision optimizer step over a flat parameter vector.
 *
 * TEST INFRASTRUCTURE ONLY. The test suite, the smoke check and the
 * benchmark's CPU-baseline leg are the only callers. The CUDA library never
 * loads, links or calls this file, and the two share no code, header, table
 * or constant.
 *
 * Sources (page title, then the outline item of "Zero From Scratch", counted
 * from 1 after its introduction):
 *   - Zero From Scratch, item 1 (sixteen bytes per weight): the state is bf16
 *     parameters and gradients plus fp32 master weights and two fp32 moments.
 *     That fixes the precision here: every per-element operation is one IEEE
 *     binary32 operation, rounded on its own (build with -ffp-contract=off and
 *     without fast-math), in the order written below.
 *   - Zero From Scratch, item 6 (data parallel): ranks average their gradients.
 *   - Zero From Scratch, item 7 (all-reduce = reduce-scatter + all-gather):
 *     the shard owner sums the P gradient slices; the updated bf16 parameters
 *     are then gathered to every rank.
 *   - Zero From Scratch, item 17 (flat parameter vector): one contiguous
 *     vector, cut into P contiguous shards.
 *   - Zero From Scratch, item 14 (MXFP8): E4M3 elements with one shared
 *     power-of-two scale per block of 32.
 *   - DeepSpeed documentation and tutorials (review), paragraph on the three
 *     stages: stage two shards optimizer state and gradients.
 * The pages print no optimizer formula, clip rule, loss-scale rule or MX
 * scale rule. The readings taken here (textbook AdamW with decoupled weight
 * decay; clip c = min(1, max_norm / (norm + norm_eps)); skip on a non-finite
 * norm; the OCP MX floor scale rule) are each stated at the function that
 * implements them.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    double lr, beta1, beta2, eps, weight_decay;
    double max_grad_norm; /* <= 0 turns the clip off */
    double norm_eps;      /* added to the norm in the clip ratio */
    int grad_average;     /* 1: divide the rank sum by P; 0: keep the sum */
} orc_hparams;

/* Step bookkeeping that survives across steps. */
typedef struct {
    int64_t t;       /* number of applied (not skipped) steps so far */
    double b1p, b2p; /* beta1^t and beta2^t, kept as running products */
} orc_counters;

/* Everything the norm pass decides for one step. */
typedef struct {
    double sumsq, norm;
    float clip, bc1, bc2;
    int found_inf;
    int64_t t;       /* step count after this step (unchanged on skip) */
    double b1p, b2p; /* running products after this step */
} orc_decision;

/* ------------------------------------------------------------------ */
/* Layout of the flat vector (Zero From Scratch, item 17).             */
/* ------------------------------------------------------------------ */

/* Shard length S: ceil(N / P) rounded up to a whole number of 32-element
 * blocks, so every shard starts on an MX block boundary. Rank r owns the flat
 * range [r*S, min((r+1)*S, N)); buffers are P*S long. Reading: the pages do
 * not say how a ragged N is split; padding the last shard is the plain
 * choice. */
int64_t orc_shard_len(int64_t n, int p)
{
    int64_t s = (n + p - 1) / p;
    return (s + 31) / 32 * 32;
}

/* ------------------------------------------------------------------ */
/* Number formats.                                                     */
/* ------------------------------------------------------------------ */

static float f32_from_bits(uint32_t u)
{
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

static uint32_t bits_from_f32(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return u;
}

/* bf16 is the top half of a binary32; widening is exact. */
float orc_bf16_to_f32(uint16_t h) { return f32_from_bits((uint32_t)h << 16); }

/* Narrow binary32 to bf16, round to nearest, ties to even. The two
 * candidates are the truncated pattern and the next one up in magnitude;
 * the dropped low half decides between them. A carry out of the mantissa
 * moves to the next binade, and out of the largest binade to infinity,
 * which is what rounding does. NaN stays a quiet NaN. */
uint16_t orc_f32_to_bf16(float f)
{
    uint32_t u = bits_from_f32(f);
    if ((u & 0x7fffffffu) > 0x7f800000u)
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t kept = u >> 16;
    uint32_t dropped = u & 0xffffu;
    if (dropped > 0x8000u || (dropped == 0x8000u && (kept & 1u)))
        kept += 1u;
    return (uint16_t)kept;
}

/* E4M3 (OCP FP8, "fn" variant): 1 sign bit, 4 exponent bits with bias 7,
 * 3 mantissa bits; exponent field 0 holds subnormals m/8 * 2^-6; the single
 * pattern S.1111.111 is NaN; there is no infinity; the largest finite value
 * is 1.75 * 2^8 = 448. Returns the value of one code. */
double orc_e4m3_value(uint8_t code)
{
    int sign = code >> 7;
    int ex = (code >> 3) & 0xf;
    int mant = code & 0x7;
    double mag;
    if (ex == 0xf && mant == 0x7)
        return NAN;
    if (ex == 0)
        mag = ldexp((double)mant / 8.0, -6);
    else
        mag = ldexp(1.0 + (double)mant / 8.0, ex - 7);
    return sign ? -mag : mag;
}

/* Round half to even on a non-negative double: the integer below, unless the
 * fraction is above one half, or exactly one half with an odd integer below. */
static double round_half_even(double q)
{
    double lo = floor(q);
    double frac = q - lo;
    if (frac > 0.5 || (frac == 0.5 && fmod(lo, 2.0) != 0.0))
        lo += 1.0;
    return lo;
}

/* Encode a finite value as E4M3: round to nearest, ties to even, and
 * saturate magnitudes at or above 448 to 448 (the "satfinite" behaviour; the
 * format has no infinity to overflow into). The sign is kept, so a negative
 * value that rounds to zero gives the negative-zero code 0x80. */
uint8_t orc_e4m3_encode(double y)
{
    uint8_t sign = signbit(y) ? 0x80 : 0x00;
    double a = fabs(y);
    uint8_t mag;
    if (a >= 448.0) {
        mag = 0x7e;
    } else if (a < ldexp(1.0, -6)) {
        /* subnormal binade: steps of 2^-9; a result of 8 steps is the
         * smallest normal, whose code is also 8 */
        mag = (uint8_t)round_half_even(a * 512.0);
    } else {
        int k;
        (void)frexp(a, &k); /* a = f * 2^k, f in [0.5, 1) */
        int e = k - 1;      /* floor(log2 a), in [-6, 8] */
        double q = ldexp(a, 3 - e); /* in [8, 16): 1.mmm scaled by 8 */
        int r = (int)round_half_even(q); /* 16 carries into the next binade */
        mag = (uint8_t)(((e + 7) << 3) + (r - 8));
    }
    return (uint8_t)(sign | mag);
}

/* ------------------------------------------------------------------ */
/* MXFP8 wire format (Zero From Scratch, item 14).                     */
/* ------------------------------------------------------------------ */

/* Encode one block of cnt <= 32 values (as doubles, exact). Elements past
 * cnt count as zero for the amax and get no code.
 * Scale rule (reading, the OCP MX v1.0 rule): e = floor(log2 amax) - 8, where
 * 8 is the exponent of E4M3's largest binade, clamped to [-127, 127]; the
 * scale byte is the E8M0 pattern e + 127 and code j is E4M3(x_j * 2^-e) with
 * saturation. An all-zero block takes e = -127. A block holding any infinity
 * or NaN takes scale byte 0xFF (E8M0 NaN) and NaN codes 0x7F, so it decodes
 * to NaN and trips the step's found-inf check. */
static void mx_encode_block(const double *vals, int cnt, uint8_t *codes, uint8_t *scale)
{
    const int emax_elem = 8; /* 448 = 1.75 * 2^8 */
    double amax = 0.0;
    int nonfinite = 0;
    for (int j = 0; j < cnt; ++j) {
        if (!isfinite(vals[j]))
            nonfinite = 1;
        else if (fabs(vals[j]) > amax)
            amax = fabs(vals[j]);
    }
    if (nonfinite) {
        *scale = 0xff;
        for (int j = 0; j < cnt; ++j)
            codes[j] = 0x7f;
        return;
    }
    int e;
    if (amax == 0.0) {
        e = -127;
    } else {
        int k;
        (void)frexp(amax, &k);
        e = (k - 1) - emax_elem;
        if (e < -127)
            e = -127;
        if (e > 127)
            e = 127;
    }
    *scale = (uint8_t)(e + 127);
    for (int j = 0; j < cnt; ++j)
        codes[j] = orc_e4m3_encode(ldexp(vals[j], -e)); /* the scaling is exact */
}

/* Encode one rank's bf16 buffer x[0..n) block by block (the wire format of
 * the gradients). Block k covers [32k, 32k+32); the last block may be short. */
void orc_mx_encode(const uint16_t *x, int64_t n, uint8_t *codes, uint8_t *scales)
{
    double vals[32];
    for (int64_t b = 0; b < (n + 31) / 32; ++b) {
        int64_t lo = 32 * b;
        int cnt = (int)(lo + 32 < n ? 32 : n - lo);
        for (int j = 0; j < cnt; ++j)
            vals[j] = (double)orc_bf16_to_f32(x[lo + j]);
        mx_encode_block(vals, cnt, codes + lo, scales + b);
    }
}

/* The same format for fp32 values: the master weights stored as MXFP8
 * parameters in place of bf16 (Zero From Scratch, item 14: MXFP8 on stored
 * state). Every binary32 value is exact as a double. */
void orc_mx_encode_f32(const float *x, int64_t n, uint8_t *codes, uint8_t *scales)
{
    double vals[32];
    for (int64_t b = 0; b < (n + 31) / 32; ++b) {
        int64_t lo = 32 * b;
        int cnt = (int)(lo + 32 < n ? 32 : n - lo);
        for (int j = 0; j < cnt; ++j)
            vals[j] = (double)x[lo + j];
        mx_encode_block(vals, cnt, codes + lo, scales + b);
    }
}

/* Value of one MX element: E4M3 value times the block's 2^(s - 127), as a
 * binary32. The product is exact in binary32: the smallest nonzero magnitude
 * is 2^-9 * 2^-127 = 2^-136 and the largest 448 * 2^127 does not occur for
 * finite blocks (s <= 246). A NaN scale byte or NaN code gives NaN. */
float orc_mx_decode(uint8_t code, uint8_t scale)
{
    if (scale == 0xff)
        return NAN;
    double v = orc_e4m3_value(code);
    return (float)ldexp(v, (int)scale - 127);
}

/* ------------------------------------------------------------------ */
/* The step.                                                           */
/* ------------------------------------------------------------------ */

/* Unscale factor applied to the rank sum: 1 / (L * P) when the ranks average
 * (Zero From Scratch, item 6), 1 / L when they only sum. Computed in binary64,
 * rounded once. For a power-of-two L*P it is exact, and multiplying by it is
 * then identical to dividing by L and by P in turn. */
float orc_inv_scale(float loss_scale, int p, int grad_average)
{
    double denom = (double)loss_scale * (grad_average ? (double)p : 1.0);
    return (float)(1.0 / denom);
}

/* Reduce-scatter, then unscale, for flat indices [lo, hi)
 * (Zero From Scratch, item 7). For each index the P rank values are widened
 * to binary32 and added in rank order 0..P-1, starting from +0. Output g[i-lo]. */
void orc_reduce_unscale(int p, const uint16_t *const *grads, int64_t lo, int64_t hi,
                        float inv, float *g)
{
    for (int64_t i = lo; i < hi; ++i) {
        float s = 0.0f;
        for (int r = 0; r < p; ++r)
            s = s + orc_bf16_to_f32(grads[r][i]);
        g[i - lo] = s * inv;
    }
}

/* The same, from MX codes: each rank value is decoded first. Scales are
 * indexed by the flat block i / 32 of that rank's buffer. */
void orc_mx_reduce_unscale(int p, const uint8_t *const *codes, const uint8_t *const *scales,
                           int64_t lo, int64_t hi, float inv, float *g)
{
    for (int64_t i = lo; i < hi; ++i) {
        float s = 0.0f;
        for (int r = 0; r < p; ++r)
            s = s + orc_mx_decode(codes[r][i], scales[r][i / 32]);
        g[i - lo] = s * inv;
    }
}

/* Sum of squares in index order: each square is a binary32 product, the
 * running sum is binary64. Returns the partial for g[0..n). */
double orc_sumsq(const float *g, int64_t n)
{
    double acc = 0.0;
    for (int64_t i = 0; i < n; ++i) {
        float q = g[i] * g[i];
        acc = acc + (double)q;
    }
    return acc;
}

/* Decide the step from the global sum of squares.
 * found_inf: the sum is not finite, i.e. some g_i is +-inf or NaN (or its
 * square overflowed). Then nothing changes: the step is skipped and the step
 * count stays (reading: a dynamic loss-scale update is the caller's business).
 * Otherwise t advances, the running powers take one more factor, the bias
 * corrections are 1 - beta^t rounded once to binary32, and the clip factor is
 * min(1, max_norm / (norm + norm_eps)) rounded once, or 1 with the clip off. */
void orc_decide(const orc_hparams *hp, const orc_counters *now, double sumsq, orc_decision *d)
{
    d->sumsq = sumsq;
    d->norm = sqrt(sumsq);
    d->found_inf = !isfinite(sumsq);
    d->t = now->t;
    d->b1p = now->b1p;
    d->b2p = now->b2p;
    d->clip = 1.0f;
    d->bc1 = 1.0f;
    d->bc2 = 1.0f;
    if (d->found_inf)
        return;
    d->t = now->t + 1;
    d->b1p = now->b1p * hp->beta1;
    d->b2p = now->b2p * hp->beta2;
    d->bc1 = (float)(1.0 - d->b1p);
    d->bc2 = (float)(1.0 - d->b2p);
    if (hp->max_grad_norm > 0.0) {
        double q = hp->max_grad_norm / (d->norm + hp->norm_eps);
        d->clip = (float)(q < 1.0 ? q : 1.0);
    }
}

/* AdamW on n elements (textbook form with decoupled weight decay; the pages
 * give no formula, this is the reading). Per element, in this order:
 *   ga = g * c
 *   m  = beta1 * m + (1 - beta1) * ga
 *   v  = beta2 * v + (1 - beta2) * (ga * ga)
 *   mh = m / bc1,  vh = v / bc2
 *   d  = sqrt(vh) + eps
 *   w  = w - (lr * wd) * w
 *   w  = w - lr * (mh / d)
 *   p  = bf16(w)             -- the value every rank receives (all-gather)
 * Each constant (beta1, beta2, 1 - beta1, 1 - beta2, eps, lr, lr * wd) is
 * formed in binary64 and rounded once to binary32. */
void orc_adamw(const orc_hparams *hp, const orc_decision *d, const float *g,
               float *w, float *m, float *v, uint16_t *p, int64_t n)
{
    const float b1 = (float)hp->beta1;
    const float b2 = (float)hp->beta2;
    const float omb1 = (float)(1.0 - hp->beta1);
    const float omb2 = (float)(1.0 - hp->beta2);
    const float eps = (float)hp->eps;
    const float lr = (float)hp->lr;
    const float lrwd = (float)(hp->lr * hp->weight_decay);
    for (int64_t i = 0; i < n; ++i) {
        float ga = g[i] * d->clip;
        float mi = b1 * m[i] + omb1 * ga;
        float vi = b2 * v[i] + omb2 * (ga * ga);
        float mh = mi / d->bc1;
        float vh = vi / d->bc2;
        float den = sqrtf(vh) + eps;
        float wi = w[i] - lrwd * w[i];
        wi = wi - lr * (mh / den);
        m[i] = mi;
        v[i] = vi;
        w[i] = wi;
        p[i] = orc_f32_to_bf16(wi);
    }
}

/* One whole step on the unsharded vector, as a single device would run it:
 * reduce + unscale every index, the global sum of squares in index order,
 * the decision, then AdamW everywhere unless skipped. Returns found_inf,
 * or -1 when the scratch vector cannot be allocated. */
int orc_step(int64_t n, int p, const uint16_t *const *grads, float loss_scale,
             const orc_hparams *hp, orc_counters *ctr, float *w, float *m, float *v,
             uint16_t *params, orc_decision *out)
{
    float inv = orc_inv_scale(loss_scale, p, hp->grad_average);
    float *g = (float *)malloc((size_t)(n > 0 ? n : 1) * sizeof(float));
    if (!g)
        return -1;
    orc_reduce_unscale(p, grads, 0, n, inv, g);
    double ss = orc_sumsq(g, n);
    orc_decide(hp, ctr, ss, out);
    if (!out->found_inf) {
        orc_adamw(hp, out, g, w, m, v, params, n);
        ctr->t = out->t;
        ctr->b1p = out->b1p;
        ctr->b2p = out->b2p;
    }
    free(g);
    return out->found_inf;
}

/* The same step with MX-encoded rank gradients. */
int orc_step_mx(int64_t n, int p, const uint8_t *const *codes, const uint8_t *const *scales,
                float loss_scale, const orc_hparams *hp, orc_counters *ctr, float *w,
                float *m, float *v, uint16_t *params, orc_decision *out)
{
    float inv = orc_inv_scale(loss_scale, p, hp->grad_average);
    float *g = (float *)malloc((size_t)(n > 0 ? n : 1) * sizeof(float));
    if (!g)
        return -1;
    orc_mx_reduce_unscale(p, codes, scales, 0, n, inv, g);
    double ss = orc_sumsq(g, n);
    orc_decide(hp, ctr, ss, out);
    if (!out->found_inf) {
        orc_adamw(hp, out, g, w, m, v, params, n);
        ctr->t = out->t;
        ctr->b1p = out->b1p;
        ctr->b2p = out->b2p;
    }
    free(g);
    return out->found_inf;
}

/* The same step written the ZeRO stage-two way (DeepSpeed documentation
 * review, paragraph on the stages; Zero From Scratch, items 7 and 9): each
 * rank r reduce-scatters its own shard [r*S, min((r+1)*S, N)) and forms the
 * partial sum of squares over it; one scalar all-reduce (ranks added in rank
 * order) gives the global sum; every rank makes the same decision and updates
 * only its shard of w, m, v; the bf16 shards are then all-gathered (here:
 * written into the one shared params vector). Returns found_inf, or -1. */
int orc_step_sharded(int64_t n, int p, const uint16_t *const *grads, float loss_scale,
                     const orc_hparams *hp, orc_counters *ctr, float *w, float *m, float *v,
                     uint16_t *params, orc_decision *out)
{
    float inv = orc_inv_scale(loss_scale, p, hp->grad_average);
    int64_t s = orc_shard_len(n, p);
    float *g = (float *)malloc((size_t)(s > 0 ? s : 1) * sizeof(float));
    double *partial = (double *)malloc((size_t)p * sizeof(double));
    if (!g || !partial) {
        free(g);
        free(partial);
        return -1;
    }
    for (int r = 0; r < p; ++r) {
        int64_t lo = r * s < n ? r * s : n;
        int64_t hi = (r + 1) * s < n ? (r + 1) * s : n;
        orc_reduce_unscale(p, grads, lo, hi, inv, g);
        partial[r] = orc_sumsq(g, hi - lo);
    }
    double ss = 0.0;
    for (int r = 0; r < p; ++r)
        ss = ss + partial[r];
    orc_decide(hp, ctr, ss, out);
    if (!out->found_inf) {
        for (int r = 0; r < p; ++r) {
            int64_t lo = r * s < n ? r * s : n;
            int64_t hi = (r + 1) * s < n ? (r + 1) * s : n;
            orc_reduce_unscale(p, grads, lo, hi, inv, g);
            orc_adamw(hp, out, g, w + lo, m + lo, v + lo, params + lo, hi - lo);
        }
        ctr->t = out->t;
        ctr->b1p = out->b1p;
        ctr->b2p = out->b2p;
    }
    free(g);
    free(partial);
    return out->found_inf;
}

/* Running products for a resumed run: beta^t built by t multiplications from
 * 1.0, the same sequence an uninterrupted run performs. */
void orc_counters_at(const orc_hparams *hp, int64_t t, orc_counters *ctr)
{
    ctr->t = t;
    ctr->b1p = 1.0;
    ctr->b2p = 1.0;
    for (int64_t k = 0; k < t; ++k) {
        ctr->b1p = ctr->b1p * hp->beta1;
        ctr->b2p = ctr->b2p * hp->beta2;
    }
}

/* ------------------------------------------------------------------ */
/* Stage three: parameters gathered just in time.                      */
/* ------------------------------------------------------------------ */

/* With the parameters themselves sharded (DeepSpeed documentation review,
 * paragraph on the three stages; Zero From Scratch, items 9 and 18: the
 * third flag), rank r keeps only the bf16 parameters [r*S, (r+1)*S), and a
 * layer that computes on flat indices [lo, hi) first gathers them from
 * their owners. Flat index i lives on rank i / S at offset i mod S.
 * out[i - lo] receives that element for every i in [lo, hi). */
void orc_gather(int64_t s, const uint16_t *const *shards, int64_t lo, int64_t hi, uint16_t *out)
{
    for (int64_t i = lo; i < hi; ++i) {
        int64_t r = i / s;
        int64_t k = i - r * s;
        out[i - lo] = shards[r][k];
    }
}

/* The same gather from parameter shards stored as MXFP8 (Zero From Scratch,
 * item 14: MXFP8 on stored state): each gathered element is decoded to its
 * exact binary32 value and rounded to bf16 for the layer's computation. A
 * decoded value has at most four significant bits, so the rounding changes
 * nothing above the bf16 subnormal range; NaN gathers as NaN. */
void orc_gather_mx(int64_t s, const uint8_t *const *codes, const uint8_t *const *scales,
                   int64_t lo, int64_t hi, uint16_t *out)
{
    for (int64_t i = lo; i < hi; ++i) {
        int64_t r = i / s;
        int64_t k = i - r * s;
        out[i - lo] = orc_f32_to_bf16(orc_mx_decode(codes[r][k], scales[r][k / 32]));
    }
}
