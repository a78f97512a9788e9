// Norm pass over bf16 rank gradients (instantiated for P = 1..16).
#include "zg_launch.h"

namespace zg {

namespace {

// Warp chunks of 32 vectors, taken `per_take` at a time, one take per warp to
// start with: no more blocks than give every warp a take, and no more than
// one wave.
int grid_for(const void *kernel, int64_t n, int per_take)
{
    const int64_t chunks = ((n + kVec - 1) / kVec + 31) / 32;
    const int64_t takes = (chunks + per_take - 1) / per_take;
    const int64_t want = (takes + kNormThreads / 32 - 1) / (kNormThreads / 32);
    const int wave = wave_blocks(kernel, kNormThreads, 0);
    return int(want < 1 ? 1 : (want < wave ? want : wave));
}

}  // namespace

cudaError_t launch_norm_bf16(int p, const uint16_t *const *g, int64_t n, float inv, unsigned long long *work,
                             Scalars *sc, FinalizeK fk, cudaStream_t st, float *stage, int mode)
{
    return with_ranks(p, [&](auto rk) {
        constexpr int P = decltype(rk)::value;
        Bf16Src<P> src;
        for (int r = 0; r < P; ++r) src.g[r] = g[r];
        auto *kernel = stage ? &norm_kernel<Bf16Src<P>, true> : &norm_kernel<Bf16Src<P>, false>;
        const int blocks = grid_for(reinterpret_cast<const void *>(kernel), n, NormChunksPerTake<Bf16Src<P>>::value);
        return launch_dependent(kernel, blocks, kNormThreads, 0, st, src, n, inv, work, sc, fk, stage, mode);
    });
}

}  // namespace zg
