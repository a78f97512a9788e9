// zg_noalloc.cu -- the norm pass for callers that cannot allocate device memory.
//
// zg_grad_norm keeps its work array (chunk counters and the exact sum of
// squares) and its result in a workspace that zg_init allocates with
// cudaMalloc. Some callers cannot do that: a process
// whose framework allocator has already reserved nearly all device memory
// (a raw cudaMalloc then fails, or fragments memory the allocator counts on),
// a latency-critical loop that cannot afford the device synchronisation a
// cudaMalloc or cudaFree may imply, or a plug-in that is given device buffers
// but no hook to release memory of its own. zg_grad_norm_noalloc runs the
// same norm kernel with its scratch in a fixed array compiled into this
// library, so it allocates nothing: the caller passes the gradients and a
// 16-byte result buffer, and the library touches no other memory.
//
// The array (kScratchBytes, under 5 KB) is part of the library's device
// image: every GPU that loads the library holds it until the process exits.
// Every call on a device shares it. Each call clears it on its stream before
// launching (the result block, the block counter and the work array must
// start at zero; a completed launch leaves them so, but an earlier call that
// did not complete might not have). Calls that overlap on the
// GPU (on different streams, or from different threads without ordering)
// race on the array and give wrong results.
//
// The array's device address is looked up (cudaGetSymbolAddress) on the first
// call in each CUDA context of a device and kept, with that context's id, in
// a fixed table. A device reset (cudaDeviceReset) or a released and recreated
// primary context loads the library's device image again, possibly at
// another address; the next call sees a different context id and looks the
// address up again, so it never hands the kernel the old one.
#include <cuda.h>  // CUcontext and CUresult only: the two driver calls are found at run time
#include <cuda_runtime.h>
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdio.h>

#include <mutex>

#include "zg.h"
#include "zg_launch.h"

namespace {

constexpr size_t kResultBytes = 256;  // the scalar block (result + counter), padded to keep the work array aligned
constexpr size_t kScratchBytes = kResultBytes + zg::kWorkWords * sizeof(unsigned long long);  // 4,736 bytes
static_assert(sizeof(zg::Scalars) <= kResultBytes, "the scalar block must fit in front of the work array");
static_assert(offsetof(zg::Scalars, sumsq) == 0 && offsetof(zg::Scalars, norm) == sizeof(double),
              "the result copy takes sumsq and norm as the first 16 bytes");

static __device__ __align__(256) unsigned char zg_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mu;
void *g_scratch_addr[kMaxDevices];               // device address of the array, per device
unsigned long long g_scratch_ctx[kMaxDevices];   // id of the context that address belongs to
int g_wave[kMaxDevices][ZG_MAX_RANKS + 1];       // resident blocks in one wave, per device and P

typedef CUresult (*CtxGetCurrentFn)(CUcontext *);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long *);
CtxGetCurrentFn g_ctx_get_current;
CtxGetIdFn g_ctx_get_id;

// The driver's cuCtxGetCurrent and cuCtxGetId, found through the runtime
// (the library does not link the driver library itself). Called with
// g_setup_mu held.
cudaError_t driver_entry_points()
{
    if (g_ctx_get_current && g_ctx_get_id) return cudaSuccess;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    void *fn = nullptr;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess) return e;
    if (q != cudaDriverEntryPointSuccess || !fn) return cudaErrorSymbolNotFound;
    g_ctx_get_current = reinterpret_cast<CtxGetCurrentFn>(fn);
    fn = nullptr;
    e = cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess) return e;
    if (q != cudaDriverEntryPointSuccess || !fn) return cudaErrorSymbolNotFound;
    g_ctx_get_id = reinterpret_cast<CtxGetIdFn>(fn);
    return cudaSuccess;
}

// Id of the calling thread's current context, 0 when none is current yet.
unsigned long long current_context_id()
{
    CUcontext c = nullptr;
    unsigned long long id = 0;
    if (g_ctx_get_current(&c) != CUDA_SUCCESS || !c) return 0;
    if (g_ctx_get_id(c, &id) != CUDA_SUCCESS) return 0;
    return id;
}

// The device address of the array on `dev` (the current device): looked up
// by the first call in each context of the device, then reused while that
// context stays current.
cudaError_t scratch_on(int dev, void **addr)
{
    std::lock_guard<std::mutex> lock(g_setup_mu);
    cudaError_t e = driver_entry_points();
    if (e != cudaSuccess) return e;
    const unsigned long long id = current_context_id();
    if (!g_scratch_addr[dev] || id == 0 || id != g_scratch_ctx[dev]) {
        void *ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, zg_noalloc_scratch);  // also makes the device's primary context current
        if (e != cudaSuccess) return e;
        const unsigned long long now = current_context_id();
        if (now == 0) return cudaErrorDeviceUninitialized;  // no context became current
        g_scratch_addr[dev] = ptr;
        g_scratch_ctx[dev] = now;
    }
    *addr = g_scratch_addr[dev];
    return cudaSuccess;
}

template <int P>
cudaError_t wave_of(int dev, int *blocks)
{
    std::lock_guard<std::mutex> lock(g_setup_mu);
    if (!g_wave[dev][P]) {
        int sms = 0, per_sm = 0;
        cudaError_t e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e == cudaSuccess)
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                &per_sm, reinterpret_cast<const void *>(&zg::norm_kernel<zg::Bf16Src<P>>), zg::kNormThreads, 0);
        if (e != cudaSuccess) return e;
        g_wave[dev][P] = sms * per_sm > 0 ? sms * per_sm : 1;
    }
    *blocks = g_wave[dev][P];
    return cudaSuccess;
}

int bad(int code, const char *what) { return zg::report_error(code, what); }

}  // namespace

extern "C" int zg_grad_norm_noalloc(const uint16_t *const *grad_ptrs, int p, int64_t n, float loss_scale,
                                    int grad_average, double *out, zg_stream stream)
{
    char msg[200];
    if (p < 1 || p > ZG_MAX_RANKS) {
        snprintf(msg, sizeof msg, "P must be in [1, %d] (got %d)", ZG_MAX_RANKS, p);
        return bad(ZG_ERR_INVALID_ARG, msg);
    }
    if (n < 1 || n >= (int64_t(1) << 62)) {
        snprintf(msg, sizeof msg, "N must be in [1, 2^62) (got %lld)", (long long)n);
        return bad(ZG_ERR_INVALID_ARG, msg);
    }
    if (!(loss_scale > 0.0f) || !isfinite(loss_scale)) return bad(ZG_ERR_INVALID_ARG, "loss_scale must be finite and > 0");
    if (grad_average != 0 && grad_average != 1) return bad(ZG_ERR_INVALID_ARG, "grad_average must be 0 or 1");
    if (!grad_ptrs) return bad(ZG_ERR_INVALID_ARG, "grad_ptrs is NULL");
    for (int r = 0; r < p; ++r) {
        if (!grad_ptrs[r]) return bad(ZG_ERR_INVALID_ARG, "a gradient pointer is NULL");
        if (reinterpret_cast<uintptr_t>(grad_ptrs[r]) & 15u)
            return bad(ZG_ERR_MISALIGNED, "gradient pointers must be 16-byte aligned");
    }
    if (!out) return bad(ZG_ERR_INVALID_ARG, "out is NULL");
    if (reinterpret_cast<uintptr_t>(out) & 7u) return bad(ZG_ERR_MISALIGNED, "out must be 8-byte aligned");
    // the kind of memory behind every pointer, asked of the driver each call
    // (nothing is remembered, so nothing is allocated on the host either)
    for (int r = 0; r < p; ++r) {
        snprintf(msg, sizeof msg, "grad_ptrs[%d]", r);
        if (int rc = zg::check_memory_uncached(grad_ptrs[r], false, msg)) return rc;
    }
    if (int rc = zg::check_memory_uncached(out, false, "out")) return rc;

    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return bad(ZG_ERR_CUDA, cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices) return bad(ZG_ERR_INVALID_ARG, "device ordinal beyond the 64 this entry point tracks");
    void *scratch = nullptr;
    e = scratch_on(dev, &scratch);
    if (e != cudaSuccess) {
        snprintf(msg, sizeof msg, "cudaGetSymbolAddress of the static scratch failed: %s", cudaGetErrorString(e));
        return bad(ZG_ERR_CUDA, msg);
    }
    zg::Scalars *sc = static_cast<zg::Scalars *>(scratch);
    auto *work = reinterpret_cast<unsigned long long *>(static_cast<unsigned char *>(scratch) + kResultBytes);
    const float inv = float(1.0 / (double(loss_scale) * (grad_average ? double(p) : 1.0)));
    const zg::FinalizeK fk{0.9, 0.999, 0.0, 0.0};  // clip off; only sumsq and norm are returned

    e = zg::with_ranks(p, [&](auto rk) {
        constexpr int P = decltype(rk)::value;
        int wave = 0;
        cudaError_t err = wave_of<P>(dev, &wave);
        if (err != cudaSuccess) return err;
        // warp chunks of 32 vectors taken a few at a time: no more blocks than
        // give every warp a take, no more than one wave (the sum does not
        // depend on the grid)
        constexpr int kPerTake = zg::NormChunksPerTake<zg::Bf16Src<P>>::value;
        const int64_t chunks = ((n + zg::kVec - 1) / zg::kVec + 31) / 32;
        const int64_t takes = (chunks + kPerTake - 1) / kPerTake;
        const int64_t want = (takes + zg::kNormThreads / 32 - 1) / (zg::kNormThreads / 32);
        int64_t blocks = want < 1 ? 1 : want;
        if (blocks > wave) blocks = wave;
        zg::Bf16Src<P> src;
        for (int r = 0; r < P; ++r) src.g[r] = grad_ptrs[r];
        err = cudaMemsetAsync(scratch, 0, kScratchBytes, stream);  // result block, counter and work array start at zero
        if (err != cudaSuccess) return err;
        zg::norm_kernel<zg::Bf16Src<P>><<<int(blocks), zg::kNormThreads, 0, stream>>>(src, n, inv, work, sc, fk);
        err = cudaGetLastError();
        if (err != cudaSuccess) return err;
        return cudaMemcpyAsync(out, sc, 2 * sizeof(double), cudaMemcpyDeviceToDevice, stream);
    });
    if (e != cudaSuccess) return bad(ZG_ERR_CUDA, cudaGetErrorString(e));
    return ZG_OK;
}
