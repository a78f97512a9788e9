// Fused step pass over MXFP8 rank gradients, plain vector loads (P = 1..16).
#include "zg_launch.h"

namespace zg {

cudaError_t launch_step_mx(int p, const uint8_t *const *c, const uint8_t *const *s, int64_t n, float inv,
                           StepK k, State state, Scalars *sc, cudaStream_t st)
{
    return with_ranks(p, [&](auto rk) {
        constexpr int P = decltype(rk)::value;
        MxSrc<P> src;
        for (int r = 0; r < P; ++r) {
            src.c[r] = c[r];
            src.s[r] = s[r];
        }
        return launch_step_kernel(src, n, inv, k, state, sc, st);
    });
}

}  // namespace zg
