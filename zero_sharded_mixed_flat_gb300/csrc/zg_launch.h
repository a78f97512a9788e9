// zg_launch.h -- host-side launchers shared by the C-ABI (internal).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "zg_kernels.cuh"

namespace zg {

// Grid for a grid-stride kernel: enough blocks for the work, at most one
// full wave of resident blocks (SM count x blocks per SM).
int wave_blocks(const void *kernel, int threads, size_t smem);

// With `stage` non-null the pass also writes the unscaled fp32 gradient there.
cudaError_t launch_norm_bf16(int p, const uint16_t *const *g, int64_t n, float inv, unsigned long long *work,
                             Scalars *sc, FinalizeK fk, cudaStream_t st, float *stage = nullptr,
                             int mode = kNormWhole);
// With `stage` non-null the pass also writes the unscaled fp32 gradient there.
cudaError_t launch_norm_mx(int p, const uint8_t *const *c, const uint8_t *const *s, int64_t n, float inv,
                           double *partials, int max_blocks, Scalars *sc, FinalizeK fk, cudaStream_t st,
                           float *stage = nullptr);
// Encode every rank's bf16 gradient to MXFP8 (codes, scales) and take the
// norm pass from the decoded values, in one launch.
cudaError_t launch_quant_norm(int p, const uint16_t *const *g, uint8_t *const *codes, uint8_t *const *scales,
                              int64_t n, float inv, unsigned long long *work, Scalars *sc, FinalizeK fk,
                              cudaStream_t st, float *stage = nullptr);
cudaError_t launch_step_bf16(int p, const uint16_t *const *g, int64_t n, float inv, StepK k, State state,
                             Scalars *sc, cudaStream_t st);
cudaError_t launch_step_staged(const float *stage, int64_t n, StepK k, State state, Scalars *sc, cudaStream_t st);
cudaError_t launch_step_tma(int p, const uint16_t *const *g, int64_t n, float inv, StepK k, State state,
                            Scalars *sc, long long wait_limit, cudaStream_t st);
// The whole bf16 step (norm pass, grid barrier, step pass) in one cooperative
// launch; partials holds at least max_blocks doubles.
cudaError_t launch_step_whole(int p, const uint16_t *const *g, int64_t n, float inv, StepK k, State state,
                              Scalars *sc, FinalizeK fk, long long wait_limit, cudaStream_t st);
cudaError_t launch_step_mx(int p, const uint8_t *const *c, const uint8_t *const *s, int64_t n, float inv,
                           StepK k, State state, Scalars *sc, cudaStream_t st);
cudaError_t launch_quant(const uint16_t *in, int64_t n, uint8_t *codes, uint8_t *scales, cudaStream_t st);
cudaError_t launch_copy(const void *src, void *dst, int64_t bytes, cudaStream_t st);
// Stage three: gather parameters [lo, hi) from P shards of S elements each.
cudaError_t launch_gather(int p, int64_t s, const uint16_t *const *shards, int64_t lo, int64_t hi, uint16_t *out,
                          cudaStream_t st);
cudaError_t launch_gather_mx(int p, int64_t s, const uint8_t *const *codes, const uint8_t *const *scales, int64_t lo,
                             int64_t hi, uint16_t *out, cudaStream_t st);

// Launch the step pass for one gradient source: grid = enough blocks for the
// 8-element vectors, at most one wave; the MX-parameter instantiation when
// the state carries MX parameter buffers.
template <class Src>
cudaError_t launch_step_kernel(const Src &src, int64_t n, float inv, StepK k, State state, Scalars *sc,
                               cudaStream_t st)
{
    auto *kernel = state.pcodes ? &step_kernel<Src, true> : &step_kernel<Src, false>;
    const int64_t want = (n / kVec + kStepThreads - 1) / kStepThreads;
    const int wave = wave_blocks(reinterpret_cast<const void *>(kernel), kStepThreads, 0);
    const int blocks = int(want < 1 ? 1 : (want < wave ? want : wave));
    return launch_dependent(kernel, blocks, kStepThreads, 0, st, src, n, inv, k, state, sc);
}

// Largest grid any norm launch may use (sizes the partials array).
int norm_blocks_cap();

// Record `msg` as the calling thread's last error text (zg_last_error) and
// return `code`.
int report_error(int code, const char *msg);

// ZG_OK when `p` is memory of the current device (device or managed), or,
// with `host_ok`, pinned host memory mapped at the same address; otherwise a
// ZG_ERR_* code with a message naming `what`. Nothing is launched.
int check_memory(const void *p, bool host_ok, const char *what);
// The same check without remembering the answer (no host allocation).
int check_memory_uncached(const void *p, bool host_ok, const char *what);

}  // namespace zg
