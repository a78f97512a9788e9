// The whole bf16 step in one launch (ZG_VARIANT_SINGLE), P = 1..16.
//
// The clip needs the norm of all N before any update, so the step is two
// passes over the gradients. Here both run in one cooperative launch: each
// block takes its share of the norm pass (the same per-thread arithmetic as
// norm_kernel), writes its block partial and arrives at a grid-wide barrier;
// the last block to arrive sums the partials in index order, writes the
// decision (norm, found-inf, clip factor, next bias corrections) and releases
// the barrier; every block then reads the decision and runs its share of the
// fused step pass (the same per-thread code as step_kernel). This saves the
// kernel boundary between the passes and the finalize that the next launch
// would wait for. The norm depends on the grid, which is this kernel's own
// (three resident blocks per SM, the step pass's occupancy, against the norm
// kernel's four), so the norm can differ from the two-launch path's in its
// last fp64 bits; the state is the same bit for bit whenever the clip factor
// is.
//
// The launch is cooperative, so every block is resident and the barrier
// cannot wait on a block that has not started. Its wait is bounded all the
// same (wait_limit polls): a block whose wait runs out records
// ZG_ERR_DEVICE_TIMEOUT and skips its share of the step pass; if some other
// block had already stored results, the step reports ZG_ERR_STATE_PARTIAL.
// Every block, the last one included, polls the release at least once, so a
// limit of 0 makes every block give up before storing anything.
#include "zg_launch.h"

namespace zg {

namespace {

__device__ __forceinline__ unsigned int ld_acquire(const unsigned int *p)
{
    unsigned int v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Bounded wait for the barrier's release: the last block to arrive resets
// the arrival counter to zero (an arrived block has seen it at one or more).
__device__ __forceinline__ bool wait_release(const unsigned int *ticket, long long limit)
{
    for (long long i = 0; i < limit; ++i)
        if (ld_acquire(ticket) == 0u) return true;
    return false;
}

}  // namespace

// Resident blocks per SM: the step pass's three up to P = 8; above that the
// norm loop's P loads in flight need more registers than three allow.
template <int P>
struct WholeMinBlocks {
    static constexpr int value = P <= 8 ? ZG_STEP_MINB : 2;
};

template <int P>
__global__ void __launch_bounds__(kStepThreads, WholeMinBlocks<P>::value)
    whole_step_kernel(Bf16Src<P> src, int64_t n, float inv, StepK k, State st, Scalars *sc, FinalizeK fk,
                      double *__restrict__ partials, long long wait_limit)
{
    static_assert(kStepThreads == kNormThreads, "one block size for both passes");
    __shared__ double red[kStepThreads / 32];
    __shared__ int s_last, s_ok, s_skip;
    __shared__ float s_c, s_bc1, s_bc2;
    const int64_t v0 = int64_t(blockIdx.x) * kStepThreads + threadIdx.x;
    const int64_t stride = int64_t(gridDim.x) * kStepThreads;

    // norm pass: this block's partial, then the barrier
    const double acc = norm_thread_sum<Bf16Src<P>, false>(src, n, inv, nullptr, v0, stride);
    const double bsum = block_sum<kStepThreads>(acc, red);
    if (threadIdx.x == 0) {
        partials[blockIdx.x] = bsum;
        __threadfence();
        s_last = atomicAdd(&sc->norm_ticket, 1u) == gridDim.x - 1;
    }
    __syncthreads();
    if (s_last) {
        // the last block: every partial is written; sum them in index order
        __threadfence();
        double s = 0.0;
        for (int i = threadIdx.x; i < int(gridDim.x); i += kStepThreads) s += __ldcg(partials + i);
        const double total = block_sum<kStepThreads>(s, red);
        if (threadIdx.x == 0) {
            finalize_decision(sc, total, fk);
            __threadfence();
            atomicExch(&sc->norm_ticket, 0u);  // release
        }
    }
    if (threadIdx.x == 0) {
        s_ok = wait_release(&sc->norm_ticket, wait_limit);
        if (s_ok) {
            __threadfence();
            s_skip = __ldcg(&sc->found_inf) ? 1 : 0;
            s_c = __ldcg(&sc->clip);
            s_bc1 = __ldcg(&sc->bc1);
            s_bc2 = __ldcg(&sc->bc2);
        }
    }
    __syncthreads();

    // fused step pass
    bool stored = false;
    if (s_ok && !s_skip) {
        stored = step_thread_loop(src, n, inv, s_c, s_bc1, s_bc2, k, st, v0, stride);
        if (blockIdx.x == 0 && threadIdx.x == 0 && n % kVec) {
            step_tail(src, n, inv, s_c, s_bc1, s_bc2, k, st);
            stored = true;
        }
    }
    const int any_stored = __syncthreads_or(stored);

    // commit: the last block of the step counts the step unless it was
    // skipped or some block's wait ran out, and marks the norm consumed
    if (threadIdx.x == 0) {
        if (!s_ok) {
            sc->status = kStatusTimeout;
            atomicAdd(&sc->step_faults, 1u);
        }
        if (any_stored) atomicOr(&sc->step_faults, kFaultStored);
        __threadfence();
        if (atomicAdd(&sc->step_ticket, 1u) == gridDim.x - 1) {
            const unsigned int faults = atomicAdd(&sc->step_faults, 0u);
            const bool any_timeout = (faults & ~kFaultStored) != 0u;
            sc->step_faults = 0u;
            if (any_timeout && (faults & kFaultStored)) sc->status = kStatusPartial;
            if (!any_timeout && !s_skip) {
                sc->t = sc->t_next;
                sc->b1p = sc->b1p_next;
                sc->b2p = sc->b2p_next;
            }
            sc->step_gen = sc->norm_gen;
            sc->step_ticket = 0u;
        }
    }
}

cudaError_t launch_step_whole(int p, const uint16_t *const *g, int64_t n, float inv, StepK k, State state,
                              Scalars *sc, FinalizeK fk, double *partials, int max_blocks, long long wait_limit,
                              cudaStream_t st)
{
    return with_ranks(p, [&](auto rk) {
        constexpr int P = decltype(rk)::value;
        Bf16Src<P> src;
        for (int r = 0; r < P; ++r) src.g[r] = g[r];
        auto *kernel = &whole_step_kernel<P>;
        const int64_t want = (n / kVec + kStepThreads - 1) / kStepThreads;
        int blocks = int(want < 1 ? 1 : (want < max_blocks ? want : max_blocks));
        const int wave = wave_blocks(reinterpret_cast<const void *>(kernel), kStepThreads, 0);
        if (blocks > wave) blocks = wave;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(blocks);
        cfg.blockDim = dim3(kStepThreads);
        cfg.dynamicSmemBytes = 0;
        cfg.stream = st;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeCooperative;
        attr[0].val.cooperative = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        return cudaLaunchKernelEx(&cfg, kernel, src, n, inv, k, state, sc, fk, partials, wait_limit);
    });
}

}  // namespace zg
