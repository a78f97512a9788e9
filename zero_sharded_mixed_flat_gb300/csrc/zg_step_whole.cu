// The whole bf16 step in one launch (ZG_VARIANT_SINGLE), P = 1..16.
//
// The clip needs the norm of all N before any update, so the step is two
// passes over the gradients. Here both run in one cooperative launch: each
// block takes warp chunks of the norm pass (the norm kernel's code: chunks
// from counters, the exact fixed-point sum), adds its digits into the work
// array and arrives at a grid-wide barrier; the last block to arrive rounds
// the sum, writes the decision (norm, found-inf, clip factor, next bias
// corrections) and releases the barrier; every block then reads the decision
// and takes warp chunks of the fused step pass (the step kernel's code). This
// saves the kernel boundary between the passes. The norm is the same exact
// sum the two-launch path takes, so both give the same bits.
//
// The launch is cooperative, so every block is resident and the barrier
// cannot wait on a block that has not started. Its wait is bounded all the
// same (wait_limit polls): a block whose wait runs out records
// ZG_ERR_DEVICE_TIMEOUT and takes no step chunks; if some other block had
// already stored results, the step reports ZG_ERR_STATE_PARTIAL (the chunks
// no block took keep their old values). Every block, the last one included,
// polls the release at least once, so a limit of 0 makes every block give up
// before storing anything.
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
                      long long wait_limit)
{
    static_assert(kStepThreads == kNormThreads, "one block size for both passes");
    __shared__ int s_ok, s_skip;
    __shared__ float s_c, s_bc1, s_bc2;

    // norm pass: this block's chunks, then the barrier
    long long word = 0;
    uint32_t flags = 0u;
    norm_chunk_loop<Bf16Src<P>, false>(src, n, inv, nullptr, st.work, word, flags);
    if (norm_block_publish(word, flags, st.work, sc) && threadIdx.x == 0) {
        // the last block: every block's digits are in; round, decide, release
        norm_total_decide(st.work, sc, fk, kNormWhole);
        __threadfence();
        atomicExch(&sc->norm_ticket, 0u);  // release
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
        stored = step_chunk_loop(src, n, inv, s_c, s_bc1, s_bc2, k, st);
        if (blockIdx.x == 0 && threadIdx.x == 0 && n % kVec) {
            step_tail(src, n, inv, s_c, s_bc1, s_bc2, k, st);
            stored = true;
        }
    }
    const int any_stored = __syncthreads_or(stored);

    // commit: the last block of the step counts the step unless it was
    // skipped or some block's wait ran out, marks the norm consumed and
    // clears the step counters
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
#pragma unroll
            for (int q = 0; q < kWorkLanes; ++q) st.work[kStepCtr + q * kWorkStride] = 0ull;
            sc->step_ticket = 0u;
        }
    }
}

cudaError_t launch_step_whole(int p, const uint16_t *const *g, int64_t n, float inv, StepK k, State state,
                              Scalars *sc, FinalizeK fk, long long wait_limit, cudaStream_t st)
{
    return with_ranks(p, [&](auto rk) {
        constexpr int P = decltype(rk)::value;
        Bf16Src<P> src;
        for (int r = 0; r < P; ++r) src.g[r] = g[r];
        auto *kernel = &whole_step_kernel<P>;
        // warp chunks of 32 vectors: no more blocks than give every warp one,
        // no more than one wave (cooperative: all resident)
        const int64_t chunks = ((n + kVec - 1) / kVec + 31) / 32;
        const int64_t want = (chunks + kStepThreads / 32 - 1) / (kStepThreads / 32);
        const int wave = wave_blocks(reinterpret_cast<const void *>(kernel), kStepThreads, 0);
        const int blocks = int(want < 1 ? 1 : (want < wave ? want : wave));
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
        return cudaLaunchKernelEx(&cfg, kernel, src, n, inv, k, state, sc, fk, wait_limit);
    });
}

}  // namespace zg
