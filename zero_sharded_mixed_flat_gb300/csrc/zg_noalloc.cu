// zg_noalloc.cu -- the norm pass for callers that cannot allocate device memory.
//
// zg_grad_norm keeps its block partials and result in a workspace that
// zg_init allocates with cudaMalloc. Some callers cannot do that: a process
// whose framework allocator has already reserved nearly all device memory
// (a raw cudaMalloc then fails, or fragments memory the allocator counts on),
// a latency-critical loop that cannot afford the device synchronisation a
// cudaMalloc or cudaFree may imply, or a plug-in that is given device buffers
// but no hook to release memory of its own. zg_grad_norm_noalloc runs the
// same norm kernel with its scratch in a fixed array compiled into this
// library, so it allocates nothing: the caller passes the gradients and a
// 16-byte result buffer, and the library touches no other memory.
//
// The array (kScratchBytes, about 33 KB) is part of the library's device
// image: every GPU that loads the library holds it until the process exits.
// Every call on a device shares it and it keeps the last call's contents, so
// each call clears the part that must start at zero (the result block and the
// block counter) on its stream before launching. Calls that overlap on the
// GPU (on different streams, or from different threads without ordering)
// race on the array and give wrong results.
#include <cuda_runtime.h>
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdio.h>

#include <mutex>

#include "zg.h"
#include "zg_launch.h"

namespace {

constexpr int kNoAllocBlocks = 4096;  // block partials the scratch holds; launches never use more
constexpr size_t kResultBytes = 256;  // the scalar block (result + counter), padded to keep partials aligned
constexpr size_t kScratchBytes = kResultBytes + kNoAllocBlocks * sizeof(double);  // 33,024 bytes
static_assert(sizeof(zg::Scalars) <= kResultBytes, "the scalar block must fit in front of the partials");
static_assert(offsetof(zg::Scalars, sumsq) == 0 && offsetof(zg::Scalars, norm) == sizeof(double),
              "the result copy takes sumsq and norm as the first 16 bytes");

static __device__ __align__(256) unsigned char zg_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mu;
void *g_scratch_addr[kMaxDevices];          // device address of the array, per device, once set up
int g_wave[kMaxDevices][ZG_MAX_RANKS + 1];  // resident blocks in one wave, per device and P

// The device address of the array on `dev` (the current device). Looked up
// once per device; the first call on a device does it.
cudaError_t scratch_on(int dev, void **addr)
{
    std::lock_guard<std::mutex> lock(g_setup_mu);
    if (!g_scratch_addr[dev]) {
        void *ptr = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&ptr, zg_noalloc_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_addr[dev] = ptr;
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
    double *partials = reinterpret_cast<double *>(static_cast<unsigned char *>(scratch) + kResultBytes);
    const float inv = float(1.0 / (double(loss_scale) * (grad_average ? double(p) : 1.0)));
    const zg::FinalizeK fk{0.9, 0.999, 0.0, 0.0};  // clip off; only sumsq and norm are returned

    e = zg::with_ranks(p, [&](auto rk) {
        constexpr int P = decltype(rk)::value;
        int wave = 0;
        cudaError_t err = wave_of<P>(dev, &wave);
        if (err != cudaSuccess) return err;
        const int64_t want = (n / zg::kVec + zg::kNormThreads - 1) / zg::kNormThreads;
        int64_t blocks = want < 1 ? 1 : want;
        if (blocks > wave) blocks = wave;
        if (blocks > kNoAllocBlocks) blocks = kNoAllocBlocks;  // the scratch bounds the grid, not N
        zg::Bf16Src<P> src;
        for (int r = 0; r < P; ++r) src.g[r] = grad_ptrs[r];
        err = cudaMemsetAsync(sc, 0, kResultBytes, stream);  // result block and block counter start at zero
        if (err != cudaSuccess) return err;
        zg::norm_kernel<zg::Bf16Src<P>><<<int(blocks), zg::kNormThreads, 0, stream>>>(src, n, inv, partials, sc, fk);
        err = cudaGetLastError();
        if (err != cudaSuccess) return err;
        return cudaMemcpyAsync(out, sc, 2 * sizeof(double), cudaMemcpyDeviceToDevice, stream);
    });
    if (e != cudaSuccess) return bad(ZG_ERR_CUDA, cudaGetErrorString(e));
    return ZG_OK;
}
