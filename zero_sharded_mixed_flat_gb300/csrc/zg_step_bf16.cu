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
        const void *fn = reinterpret_cast<const void *>(&step_kernel<Bf16Src<P>>);
        const int64_t want = (n / kVec + kStepThreads - 1) / kStepThreads;
        const int wave = wave_blocks(fn, kStepThreads, 0);
        const int blocks = int(want < 1 ? 1 : (want < wave ? want : wave));
        return launch_dependent(&step_kernel<Bf16Src<P>>, blocks, kStepThreads, 0, st, src, n, inv, k, state, sc);
    });
}

cudaError_t launch_step_staged(const float *stage, int64_t n, StepK k, State state, Scalars *sc, cudaStream_t st)
{
    StagedSrc src{stage};
    auto *kernel = &step_kernel<StagedSrc>;
    const int64_t want = (n / kVec + kStepThreads - 1) / kStepThreads;
    const int wave = wave_blocks(reinterpret_cast<const void *>(kernel), kStepThreads, 0);
    const int blocks = int(want < 1 ? 1 : (want < wave ? want : wave));
    return launch_dependent(kernel, blocks, kStepThreads, 0, st, src, n, 1.0f, k, state, sc);
}

}  // namespace zg
