// Fused step pass with TMA-staged operands (P = 1..16).
#include "zg_launch.h"

namespace zg {

// One warp-specialised CTA per SM. With 2048-element tiles (P >= 5) three
// ring buffers: measured on GB300 against two CTAs of two buffers and one CTA
// of four, the shape whose whole steps match or beat the plain-load kernel;
// with 4096-element tiles (P <= 4) two buffers.
#ifndef ZG_TMA_CTAS_PER_SM
#define ZG_TMA_CTAS_PER_SM 1
#endif
constexpr int kTmaCtasPerSm = ZG_TMA_CTAS_PER_SM;
#ifndef ZG_TMA_MAX_STAGES
#define ZG_TMA_MAX_STAGES 3
#endif
static_assert(ZG_TMA_MAX_STAGES >= 2 && ZG_TMA_MAX_STAGES <= 8, "the kernel holds eight barriers");

cudaError_t launch_step_tma(int p, const uint16_t *const *g, int64_t n, float inv, StepK k, State state, Scalars *sc,
                            long long wait_limit, cudaStream_t st)
{
    return with_ranks(p, [&](auto rk) {
        constexpr int P = decltype(rk)::value;
        Bf16Src<P> src;
        for (int r = 0; r < P; ++r) src.g[r] = g[r];
        constexpr int T = tma::TileFor<P>::value;
        constexpr int threads = tma::ws_threads(T);
        const tma::Layout lay = tma::Layout::of(P, T);
        const int cap = T == tma::kTileSmallP ? 2 : ZG_TMA_MAX_STAGES;
        // Ring buffers per CTA: as many (2..ZG_TMA_MAX_STAGES) as fit when kTmaCtasPerSm CTAs
        // share an SM's 228 KB; if two buffers do not fit that way, one CTA
        // per SM with as many as fit (two at P = 16).
        const int sm_bytes = 227 * 1024 - 1024;
        int stages = sm_bytes / kTmaCtasPerSm / int(lay.stage_bytes);
        if (stages < 2) stages = sm_bytes / int(lay.stage_bytes);
        stages = stages > cap ? cap : stages;
        if (stages < 2) return cudaErrorInvalidConfiguration;
        const size_t smem = size_t(stages) * lay.stage_bytes;
        auto *fn = &tma::step_kernel_tma<P, T>;
        cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
        if (e != cudaSuccess) return e;
        const int64_t covered = (n / kVec) * kVec;
        const int64_t tiles = (covered + T - 1) / T;
        const int wave = wave_blocks(reinterpret_cast<const void *>(fn), threads, smem);
        const int blocks = int(tiles < 1 ? 1 : (tiles < wave ? tiles : wave));
        return launch_dependent(fn, blocks, threads, smem, st, src, n, inv, k, state, sc, stages, wait_limit);
    });
}

}  // namespace zg
