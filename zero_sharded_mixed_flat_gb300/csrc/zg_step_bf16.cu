// Fused step pass over bf16 rank gradients, plain vector loads (P = 1..16).
#include "zg_launch.h"

namespace zg {

cudaError_t launch_step_bf16(int p, const uint16_t *const *g, int64_t n, float inv, StepK k, State state,
                             Scalars *sc, cudaStream_t st)
{
    return with_ranks(p, [&](auto rk) {
        constexpr int P = decltype(rk)::value;
        Bf16Src<P> src;
        for (int r = 0; r < P; ++r) src.g[r] = g[r];
        return launch_step_kernel(src, n, inv, k, state, sc, st);
    });
}

cudaError_t launch_step_staged(const float *stage, int64_t n, StepK k, State state, Scalars *sc, cudaStream_t st)
{
    StagedSrc src{stage};
    return launch_step_kernel(src, n, 1.0f, k, state, sc, st);
}

}  // namespace zg
