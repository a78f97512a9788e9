// Norm pass over bf16 rank gradients (instantiated for P = 1..16).
#include "zg_launch.h"

namespace zg {

cudaError_t launch_norm_bf16(int p, const uint16_t *const *g, int64_t n, float inv, double *partials,
                             int max_blocks, Scalars *sc, FinalizeK fk, cudaStream_t st, float *stage, int mode)
{
    return with_ranks(p, [&](auto rk) {
        constexpr int P = decltype(rk)::value;
        Bf16Src<P> src;
        for (int r = 0; r < P; ++r) src.g[r] = g[r];
        auto *kernel = stage ? &norm_kernel<Bf16Src<P>, true> : &norm_kernel<Bf16Src<P>, false>;
        const int64_t want = (n / kVec + kNormThreads - 1) / kNormThreads;
        int blocks = int(want < 1 ? 1 : (want < max_blocks ? want : max_blocks));
        const int wave = wave_blocks(reinterpret_cast<const void *>(kernel), kNormThreads, 0);
        if (blocks > wave) blocks = wave;
        return launch_dependent(kernel, blocks, kNormThreads, 0, st, src, n, inv, partials, sc, fk, stage, mode);
    });
}

}  // namespace zg
