// Norm pass over MXFP8 rank gradients (instantiated for P = 1..16).
#include "zg_launch.h"

namespace zg {

cudaError_t launch_norm_mx(int p, const uint8_t *const *c, const uint8_t *const *s, int64_t n, float inv,
                           double *partials, int max_blocks, Scalars *sc, FinalizeK fk, cudaStream_t st)
{
    return with_ranks(p, [&](auto rk) {
        constexpr int P = decltype(rk)::value;
        MxSrc<P> src;
        for (int r = 0; r < P; ++r) {
            src.c[r] = c[r];
            src.s[r] = s[r];
        }
        const void *fn = reinterpret_cast<const void *>(&norm_kernel<MxSrc<P>, false>);
        const int64_t want = (n / kVec + kNormThreads - 1) / kNormThreads;
        int blocks = int(want < 1 ? 1 : (want < max_blocks ? want : max_blocks));
        const int wave = wave_blocks(fn, kNormThreads, 0);
        if (blocks > wave) blocks = wave;
        return launch_dependent(&norm_kernel<MxSrc<P>, false>, blocks, kNormThreads, 0, st, src, n, inv, partials,
                                sc, fk, static_cast<float *>(nullptr), kNormWhole);
    });
}

}  // namespace zg
