// The MXFP8 wire path's encode and norm pass in one pass (P = 1..16).
//
// With every rank's bf16 gradient resident on this GPU, the encode (Zero From
// Scratch, item 14: MXFP8 on the wire) and the norm pass that follows it can
// share one read: per 8-element quarter block, each rank's bf16 values are
// encoded exactly as zg_quant_mxfp8 encodes them (mx_encode_slice, the same
// block rule over the four lanes that hold a block) and the codes and scale
// byte stored (the wire payload the step pass reads), and the same codes are
// decoded in registers and summed in rank order exactly as the MX norm pass
// and the MX step pass sum them from the payload (packed fused multiply-adds,
// exact because each product E4M3 * 2^(s - 127) is, and the encoder never
// writes a scale byte in 247..254). The unscaled, averaged g is squared in
// fp32 and summed as the bf16 norm pass sums it: warp chunks of 32 vectors
// handed out by counters, each lane's two-sum pair, the chunk's fixed
// butterfly and the exact fixed-point total (so on gradients MXFP8 holds
// exactly, the two passes give the same bits). This saves the
// P * (1 + 1/32) bytes per parameter the separate norm pass reads back, and
// P + 1 launches become one.
//
// Each thread issues all P ranks' 16-byte loads of its vector before encoding
// any (P * 16 bytes in flight per thread, four 256-thread blocks per SM up to
// P = 8). A chunk's 32 vectors sit one per lane, so a 32-element block's four
// quarters are in neighbouring lanes; the last, partial vector is read and
// written element by element with the values past N taken as zero, as the
// encoder takes them.
#include "zg_launch.h"

namespace zg {

constexpr int kQnVec = 8;  // elements per thread per vector: one 16-byte bf16 load per rank

template <int P>
struct QuantNormMinBlocks {
    static constexpr int value = P <= 8 ? 4 : 2;
};

struct MxOut {
    uint8_t *c[kMaxRanks];
    uint8_t *s[kMaxRanks];
};

template <int P, bool kStage>
__global__ void __launch_bounds__(kNormThreads, QuantNormMinBlocks<P>::value)
    quant_norm_kernel(Bf16Src<P> src, MxOut out, int64_t n, float inv, unsigned long long *work, Scalars *sc,
                      FinalizeK fk, float *__restrict__ stage)
{
    static_assert(kQnVec == kVec, "the norm pass's chunks are 32 vectors of 8");
    pdl_wait();
    pdl_trigger();
    const int64_t nvec_full = n / kQnVec;
    const int64_t nvec_all = (n + kQnVec - 1) / kQnVec;
    const int64_t nchunk = (nvec_all + 31) / 32;
    const int lane = threadIdx.x & 31;
    const int wq = threadIdx.x >> 5;
    const float2 inv2 = make_float2(inv, inv);
    unsigned long long *ctr = work + kNormCtr + wq * kWorkStride;
    int64_t ch = wq + int64_t(kWorkLanes) * blockIdx.x;
    long long word = 0;
    uint32_t flags = 0u;
#pragma unroll 1
    while (ch < nchunk) {  // warp-uniform: a chunk is 32 vectors, one per lane
        unsigned long long next = 0ull;
        if (lane == 0) next = atomicAdd(ctr, 1ull);
        const int64_t v = ch * 32 + lane;
        // every rank's values of this vector, loads issued together
        uint32_t wd[P][4];
        if (v < nvec_full) {
#pragma unroll
            for (int r = 0; r < P; ++r) {
                const uint4 x = ld_stream(reinterpret_cast<const uint4 *>(src.g[r]) + v);
                wd[r][0] = x.x, wd[r][1] = x.y, wd[r][2] = x.z, wd[r][3] = x.w;
            }
        } else {
#pragma unroll
            for (int r = 0; r < P; ++r) {
#pragma unroll
                for (int q = 0; q < 4; ++q) wd[r][q] = 0u;
                if (v < nvec_all) {
#pragma unroll
                    for (int j = 0; j < kQnVec; ++j)
                        if (v * kQnVec + j < n) wd[r][j >> 1] |= uint32_t(src.g[r][v * kQnVec + j]) << (16 * (j & 1));
                }
            }
        }
        float2 g2[kQnVec / 2];
#pragma unroll
        for (int q = 0; q < kQnVec / 2; ++q) g2[q] = make_float2(0.0f, 0.0f);
#pragma unroll
        for (int r = 0; r < P; ++r) {
            uint32_t pairs[4];
            const uint32_t sbyte = mx_encode_slice<4>(wd[r], pairs);
            if (v < nvec_full) {
                __stcs(reinterpret_cast<uint2 *>(out.c[r]) + v,
                       make_uint2(pairs[0] | (pairs[1] << 16), pairs[2] | (pairs[3] << 16)));
            } else if (v < nvec_all) {
#pragma unroll
                for (int j = 0; j < kQnVec; ++j)
                    if (v * kQnVec + j < n) out.c[r][v * kQnVec + j] = uint8_t(pairs[j >> 1] >> (8 * (j & 1)));
            }
            if ((lane & 3) == 0 && v < nvec_all) out.s[r][v >> 2] = uint8_t(sbyte);
            // the decoded payload, summed in rank order
            const float scale = e8m0_value(sbyte);
            const float2 s2 = make_float2(scale, scale);
#pragma unroll
            for (int q = 0; q < kQnVec / 2; ++q) g2[q] = fma_f32x2(e4m3x2_to_f32x2(uint16_t(pairs[q])), s2, g2[q]);
        }
        // unscale, square in fp32, the lane's two-sum pair in element order
        // (vectors past the end hold zeros: their squares are +0)
        float g[kQnVec];
        float hi = 0.0f, lo = 0.0f;
#pragma unroll
        for (int q = 0; q < kQnVec / 2; ++q) {
            g2[q] = mul_f32x2(g2[q], inv2);
            g[2 * q] = g2[q].x;
            g[2 * q + 1] = g2[q].y;
            const float2 sq = mul_f32x2(g2[q], g2[q]);
            two_sum_acc(hi, lo, sq.x);
            two_sum_acc(hi, lo, sq.y);
        }
        if (kStage && v < nvec_all) {
            // the reduce-scatter output for the staged step pass
            if (v < nvec_full) {
                float4 *o = reinterpret_cast<float4 *>(stage) + 2 * v;
                const float4 a = make_float4(g[0], g[1], g[2], g[3]);
                const float4 b = make_float4(g[4], g[5], g[6], g[7]);
                if (v >= nvec_full - kStageKeepBytes / 32) {
                    o[0] = a;
                    o[1] = b;
                } else {
                    __stcs(o, a);
                    __stcs(o + 1, b);
                }
            } else {
#pragma unroll
                for (int j = 0; j < kQnVec; ++j)
                    if (v * kQnVec + j < n) stage[v * kQnVec + j] = g[j];
            }
        }
        chunk_add(hi, lo, g, lane, word, flags);
        next = __shfl_sync(0xffffffffu, next, 0);
        ch = wq + int64_t(kWorkLanes) * (int64_t(gridDim.x) + int64_t(next));
    }
    norm_exact_finish(word, flags, work, sc, fk, kNormWhole);
}

cudaError_t launch_quant_norm(int p, const uint16_t *const *g, uint8_t *const *codes, uint8_t *const *scales,
                              int64_t n, float inv, unsigned long long *work, Scalars *sc, FinalizeK fk,
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
        // warp chunks of 32 vectors: no more blocks than give every warp one,
        // no more than one wave
        const int64_t chunks = ((n + kQnVec - 1) / kQnVec + 31) / 32;
        const int64_t want = (chunks + kNormThreads / 32 - 1) / (kNormThreads / 32);
        const int wave = wave_blocks(reinterpret_cast<const void *>(kernel), kNormThreads, 0);
        const int blocks = int(want < 1 ? 1 : (want < wave ? want : wave));
        return launch_dependent(kernel, blocks, kNormThreads, 0, st, src, out, n, inv, work, sc, fk, stage);
    });
}

}  // namespace zg
