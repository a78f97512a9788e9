// Norm pass over MXFP8 rank gradients (instantiated for P = 1..16).
//
// Sixteen elements per thread per vector: one 16-byte code load and one scale
// byte per rank (the sixteen lie in one 32-element block), so the address
// arithmetic, the scale decode and the check for scale bytes the encoder never
// writes are paid once per sixteen elements. Decoding is issue-bound, not
// bandwidth-bound (8.25 bytes per parameter at P = 8), which is what this
// layout buys back. Per element: the rank-ordered fp32 sum of exact decoded
// products, times the unscale factor, squared in fp32. The squares are added
// in two-sum runs of 32 widened to fp64 over a fixed grid-stride split, not
// by the bf16 norm pass's exact chunk sum (whose butterfly per 32 vectors
// this 16-element layout would pay for in issue slots), so the two norms can
// differ in their last bits (within 1e-12).
#include "zg_launch.h"

namespace zg {

constexpr int kMxNormVec = 16;

// Resident blocks per SM: P 16-byte code loads in flight per thread fit
// three 256-thread blocks per SM up to P = 8, two above.
template <int P>
struct MxNormMinBlocks {
    static constexpr int value = P <= 8 ? 3 : 2;
};

// Rank-ordered sum of the decoded products for sixteen elements. Every
// product E4M3 * 2^(s - 127) is exact in binary32 for s <= 246, so a packed
// fused multiply-add gives the bits of the separate multiply and add; a scale
// byte in 247..254 (never written by the encoder) takes the separate
// operations, where an overflowing product reads as inf.
template <int P>
__device__ __forceinline__ void mx_reduce16(const uint4 (&c)[P], const uint32_t (&sb)[P], float (&out)[kMxNormVec])
{
    uint32_t big = 0u;
#pragma unroll
    for (int r = 0; r < P; ++r) big |= uint32_t(sb[r] - 247u < 8u);
    float2 acc[kMxNormVec / 2];
#pragma unroll
    for (int q = 0; q < kMxNormVec / 2; ++q) acc[q] = make_float2(0.0f, 0.0f);
    if (!big) {
#pragma unroll
        for (int r = 0; r < P; ++r) {
            const float scale = e8m0_value(sb[r]);
            const float2 s2 = make_float2(scale, scale);
            const uint32_t w[4] = {c[r].x, c[r].y, c[r].z, c[r].w};
#pragma unroll
            for (int q = 0; q < kMxNormVec / 2; ++q)
                acc[q] = fma_f32x2(e4m3x2_to_f32x2(uint16_t(w[q >> 1] >> (16 * (q & 1)))), s2, acc[q]);
        }
    } else {
#pragma unroll
        for (int r = 0; r < P; ++r) {
            const float scale = e8m0_value(sb[r]);
            const uint32_t w[4] = {c[r].x, c[r].y, c[r].z, c[r].w};
#pragma unroll
            for (int q = 0; q < kMxNormVec / 2; ++q) {
                const float2 f = e4m3x2_to_f32x2(uint16_t(w[q >> 1] >> (16 * (q & 1))));
                acc[q].x = __fadd_rn(acc[q].x, __fmul_rn(f.x, scale));
                acc[q].y = __fadd_rn(acc[q].y, __fmul_rn(f.y, scale));
            }
        }
    }
#pragma unroll
    for (int q = 0; q < kMxNormVec / 2; ++q) {
        out[2 * q] = acc[q].x;
        out[2 * q + 1] = acc[q].y;
    }
}

// Grid-stride over 16-element vectors; runs of two vectors (32 squares) per
// two-sum pair, each run widened to fp64. A run whose fp32 pair is not finite
// is redone with every square widened on its own, so the result is non-finite
// exactly when some square is. Same N, P and grid: bit-identical norm.
// With kStage the pass also stores the unscaled, averaged gradient g (the
// reduce-scatter output) for the staged step pass.
template <int P, bool kStage>
__global__ void __launch_bounds__(kNormThreads, MxNormMinBlocks<P>::value)
    norm_mx_kernel(MxSrc<P> src, int64_t n, float inv, double *__restrict__ partials, Scalars *sc, FinalizeK fk,
                   float *__restrict__ stage)
{
    pdl_wait();
    pdl_trigger();
    const int64_t nvec = n / kMxNormVec;
    const int64_t stride = int64_t(gridDim.x) * kNormThreads;
    const float2 inv2 = make_float2(inv, inv);
    int64_t v = int64_t(blockIdx.x) * kNormThreads + threadIdx.x;
    double acc = 0.0;
    while (v < nvec) {
        const int64_t run_start = v;
        float hi = 0.0f, lo = 0.0f;
#pragma unroll 1
        for (int k = 0; k < 2 && v < nvec; ++k, v += stride) {
            uint4 c[P];
            uint32_t sb[P];
#pragma unroll
            for (int r = 0; r < P; ++r) {
                c[r] = ld_stream(reinterpret_cast<const uint4 *>(src.c[r]) + v);
                sb[r] = src.s[r][v >> 1];
            }
            float g[kMxNormVec];
            mx_reduce16<P>(c, sb, g);
#pragma unroll
            for (int j = 0; j < kMxNormVec; j += 2) {
                const float2 gg = mul_f32x2(make_float2(g[j], g[j + 1]), inv2);
                const float2 sq = mul_f32x2(gg, gg);
                two_sum_acc(hi, lo, sq.x);
                two_sum_acc(hi, lo, sq.y);
                g[j] = gg.x;
                g[j + 1] = gg.y;
            }
            if (kStage) {  // the tail the step pass reads first keeps the default policy
                float4 *o = reinterpret_cast<float4 *>(stage) + 4 * v;
                const bool keep = v >= nvec - kStageKeepBytes / 64;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float4 x = make_float4(g[4 * q], g[4 * q + 1], g[4 * q + 2], g[4 * q + 3]);
                    if (keep)
                        o[q] = x;
                    else
                        __stcs(o + q, x);
                }
            }
        }
        if (isfinite(hi) && isfinite(lo)) {
            acc += double(hi);
            acc += double(lo);
        } else {
#pragma unroll 1
            for (int64_t u = run_start; u < v && u < nvec; u += stride) {
#pragma unroll 1
                for (int j = 0; j < kMxNormVec; ++j) {
                    const float g = __fmul_rn(src.sum1(u * kMxNormVec + j), inv);
                    acc += double(__fmul_rn(g, g));
                }
            }
        }
    }
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        for (int64_t i = nvec * kMxNormVec; i < n; ++i) {  // ragged tail, fewer than 16 elements
            const float g = __fmul_rn(src.sum1(i), inv);
            acc += double(__fmul_rn(g, g));
            if (kStage) stage[i] = g;
        }
    }
    norm_finish(acc, partials, sc, fk, kNormWhole);
}

cudaError_t launch_norm_mx(int p, const uint8_t *const *c, const uint8_t *const *s, int64_t n, float inv,
                           double *partials, int max_blocks, Scalars *sc, FinalizeK fk, cudaStream_t st, float *stage)
{
    return with_ranks(p, [&](auto rk) {
        constexpr int P = decltype(rk)::value;
        MxSrc<P> src;
        for (int r = 0; r < P; ++r) {
            src.c[r] = c[r];
            src.s[r] = s[r];
        }
        auto *kernel = stage ? &norm_mx_kernel<P, true> : &norm_mx_kernel<P, false>;
        const int64_t want = (n / kMxNormVec + kNormThreads - 1) / kNormThreads;
        int blocks = int(want < 1 ? 1 : (want < max_blocks ? want : max_blocks));
        const int wave = wave_blocks(reinterpret_cast<const void *>(kernel), kNormThreads, 0);
        if (blocks > wave) blocks = wave;
        return launch_dependent(kernel, blocks, kNormThreads, 0, st, src, n, inv, partials, sc, fk, stage);
    });
}

}  // namespace zg
