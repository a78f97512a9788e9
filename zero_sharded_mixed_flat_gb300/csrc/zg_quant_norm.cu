// The MXFP8 wire path's encode and norm pass in one pass (P = 1..16).
//
// With every rank's bf16 gradient resident on this GPU, the encode (Zero From
// Scratch, item 14: MXFP8 on the wire) and the norm pass that follows it can
// share one read: per 16-element half block, each rank's bf16 values are
// encoded exactly as zg_quant_mxfp8 encodes them (mx_encode16) and the codes
// and scale byte stored (the wire payload the step pass reads), and the same
// codes are decoded in registers and summed in rank order exactly as the MX
// norm pass sums them from the payload (packed fused multiply-adds, exact
// because each product E4M3 * 2^(s - 127) is, and the encoder never writes a
// scale byte in 247..254). The unscaled, averaged g is squared in fp32 and
// added with two-sum in runs of two vectors (32 squares) widened to fp64, as
// in the MX norm pass. This saves the P * (1 + 1/32)
// bytes per parameter the separate norm pass reads back, and P + 1 launches
// become one.
//
// Work is split in warp-wide rows of 32 consecutive half blocks (the encoder
// needs both halves of a block in neighbouring lanes); each thread's vectors
// are the MX norm pass's (vector v = row + lane, rows grid-strided), and the
// last, partial vector is read and written element by element with the
// values past N taken as zero, as the encoder takes them.
#include "zg_launch.h"

namespace zg {

constexpr int kQnVec = 16;

template <int P>
struct QuantNormMinBlocks {
    static constexpr int value = P <= 8 ? 3 : 2;
};

struct MxOut {
    uint8_t *c[kMaxRanks];
    uint8_t *s[kMaxRanks];
};

// Rank r's 16 bf16 values of vector v (values at or past n as zero).
template <int P>
__device__ __forceinline__ void load16(const Bf16Src<P> &src, int r, int64_t v, int64_t n, uint32_t (&wd)[8])
{
    const int64_t nvec_full = n / kQnVec;
    if (v < nvec_full) {
        const uint4 a = ld_stream(reinterpret_cast<const uint4 *>(src.g[r]) + 2 * v);
        const uint4 b = ld_stream(reinterpret_cast<const uint4 *>(src.g[r]) + 2 * v + 1);
        wd[0] = a.x, wd[1] = a.y, wd[2] = a.z, wd[3] = a.w;
        wd[4] = b.x, wd[5] = b.y, wd[6] = b.z, wd[7] = b.w;
    } else {
#pragma unroll
        for (int q = 0; q < 8; ++q) wd[q] = 0u;
        if (v * kQnVec < n) {
#pragma unroll
            for (int j = 0; j < kQnVec; ++j)
                if (v * kQnVec + j < n) wd[j >> 1] |= uint32_t(src.g[r][v * kQnVec + j]) << (16 * (j & 1));
        }
    }
}

template <int P, bool kStage>
__global__ void __launch_bounds__(kNormThreads, QuantNormMinBlocks<P>::value)
    quant_norm_kernel(Bf16Src<P> src, MxOut out, int64_t n, float inv, double *__restrict__ partials, Scalars *sc,
                      FinalizeK fk, float *__restrict__ stage)
{
    pdl_wait();
    pdl_trigger();
    const int64_t nvec_full = n / kQnVec;
    const int64_t nvec_all = (n + kQnVec - 1) / kQnVec;
    const int64_t stride = int64_t(gridDim.x) * kNormThreads;
    const int lane = threadIdx.x & 31;
    const float2 inv2 = make_float2(inv, inv);
    double acc = 0.0;
#pragma unroll 1
    for (int64_t row = int64_t(blockIdx.x) * kNormThreads + (threadIdx.x & ~31); row < nvec_all; row += 2 * stride) {
        float hi = 0.0f, lo = 0.0f;
#pragma unroll 1
        for (int k = 0; k < 2; ++k) {
            const int64_t base = row + k * stride;
            if (base >= nvec_all) break;  // warp-uniform
            const int64_t v = base + lane;
            const bool live = v < nvec_all;
            float2 g2[kQnVec / 2];
#pragma unroll
            for (int q = 0; q < kQnVec / 2; ++q) g2[q] = make_float2(0.0f, 0.0f);
            uint32_t cur[8], nxt[8];
            if (live) load16(src, 0, v, n, cur);
            else {
#pragma unroll
                for (int q = 0; q < 8; ++q) cur[q] = 0u;
            }
#pragma unroll
            for (int r = 0; r < P; ++r) {
                if (r + 1 < P) {  // the next rank's loads in flight while this one is encoded
                    if (live) load16(src, r + 1, v, n, nxt);
                    else {
#pragma unroll
                        for (int q = 0; q < 8; ++q) nxt[q] = 0u;
                    }
                }
                uint32_t pairs[8];
                const uint32_t sbyte = mx_encode16(cur, pairs);
                if (v < nvec_full) {
                    __stcs(reinterpret_cast<uint4 *>(out.c[r]) + v,
                           make_uint4(pairs[0] | (pairs[1] << 16), pairs[2] | (pairs[3] << 16),
                                      pairs[4] | (pairs[5] << 16), pairs[6] | (pairs[7] << 16)));
                } else if (live) {
#pragma unroll
                    for (int j = 0; j < kQnVec; ++j)
                        if (v * kQnVec + j < n) out.c[r][v * kQnVec + j] = uint8_t(pairs[j >> 1] >> (8 * (j & 1)));
                }
                if ((lane & 1) == 0 && live) out.s[r][v >> 1] = uint8_t(sbyte);
                // the decoded payload, summed in rank order
                const float scale = e8m0_value(sbyte);
                const float2 s2 = make_float2(scale, scale);
#pragma unroll
                for (int q = 0; q < kQnVec / 2; ++q) g2[q] = fma_f32x2(e4m3x2_to_f32x2(uint16_t(pairs[q])), s2, g2[q]);
                if (r + 1 < P) {
#pragma unroll
                    for (int q = 0; q < 8; ++q) cur[q] = nxt[q];
                }
            }
            // unscale, square in fp32, add every square with two-sum
#pragma unroll
            for (int q = 0; q < kQnVec / 2; ++q) {
                g2[q] = mul_f32x2(g2[q], inv2);
                const float2 sq = mul_f32x2(g2[q], g2[q]);
                two_sum_acc(hi, lo, sq.x);
                two_sum_acc(hi, lo, sq.y);
            }
            if (kStage && live) {
                // the reduce-scatter output for the staged step pass
                if (v < nvec_full) {
                    float4 *o = reinterpret_cast<float4 *>(stage) + 4 * v;
                    const bool keep = v >= nvec_full - kStageKeepBytes / 64;
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const float4 x = make_float4(g2[2 * q].x, g2[2 * q].y, g2[2 * q + 1].x, g2[2 * q + 1].y);
                        if (keep)
                            o[q] = x;
                        else
                            __stcs(o + q, x);
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < kQnVec; ++j)
                        if (v * kQnVec + j < n) stage[v * kQnVec + j] = (j & 1) ? g2[j >> 1].y : g2[j >> 1].x;
                }
            }
        }
        // the codes and scale bytes of this run are written; the non-finite
        // case below reads them back (the partner lane wrote the scale byte).
        // Vectors past the end added zeros (their squares are +0).
        __syncwarp();
        if (isfinite(hi) && isfinite(lo)) {
            acc += double(hi);
            acc += double(lo);
        } else {
            // a square that is not finite (or a run whose fp32 partial
            // overflowed): redo the run with every square widened to fp64 on
            // its own, from the payload
            MxSrc<P> mx;
#pragma unroll
            for (int r = 0; r < P; ++r) {
                mx.c[r] = out.c[r];
                mx.s[r] = out.s[r];
            }
#pragma unroll 1
            for (int k = 0; k < 2; ++k) {
                const int64_t v = row + k * stride + lane;
                if (v >= nvec_all) break;
#pragma unroll 1
                for (int j = 0; j < kQnVec; ++j) {
                    const int64_t i = v * kQnVec + j;
                    if (i >= n) break;
                    const float g = __fmul_rn(mx.sum1(i), inv);
                    acc += double(__fmul_rn(g, g));
                }
            }
        }
    }
    norm_finish(acc, partials, sc, fk, kNormWhole);
}

cudaError_t launch_quant_norm(int p, const uint16_t *const *g, uint8_t *const *codes, uint8_t *const *scales,
                              int64_t n, float inv, double *partials, int max_blocks, Scalars *sc, FinalizeK fk,
                              cudaStream_t st, float *stage)
{
    return with_ranks(p, [&](auto rk) {
        constexpr int P = decltype(rk)::value;
        Bf16Src<P> src;
        MxOut out = {};
        for (int r = 0; r < P; ++r) {
            src.g[r] = g[r];
            out.c[r] = codes[r];
            out.s[r] = scales[r];
        }
        auto *kernel = stage ? &quant_norm_kernel<P, true> : &quant_norm_kernel<P, false>;
        const int64_t nvec = (n + kQnVec - 1) / kQnVec;
        const int64_t want = (nvec + kNormThreads - 1) / kNormThreads;
        int blocks = int(want < 1 ? 1 : (want < max_blocks ? want : max_blocks));
        const int wave = wave_blocks(reinterpret_cast<const void *>(kernel), kNormThreads, 0);
        if (blocks > wave) blocks = wave;
        return launch_dependent(kernel, blocks, kNormThreads, 0, st, src, out, n, inv, partials, sc, fk, stage);
    });
}

}  // namespace zg
