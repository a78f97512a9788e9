// MXFP8 encoder and the HBM copy probe.
#include "zg_launch.h"

namespace zg {

// ------------------------------------------------------------------ MXFP8 encoder

constexpr int kQuantThreads = 256;
constexpr int kQuantVec = 16;  // elements per thread: two 16-byte bf16 loads, one 16-byte code store

// Two lanes share one 32-element block (16 elements each), encoded by
// mx_encode16.
__global__ void __launch_bounds__(kQuantThreads)
    quant_kernel(const uint16_t *__restrict__ in, int64_t n, uint8_t *__restrict__ codes,
                 uint8_t *__restrict__ scales)
{
    const int64_t nvec_full = n / kQuantVec;
    const int64_t nvec_all = (n + kQuantVec - 1) / kQuantVec;
    const int lane = threadIdx.x & 31;
    const int64_t stride = int64_t(gridDim.x) * kQuantThreads;
#pragma unroll 1
    for (int64_t base = int64_t(blockIdx.x) * kQuantThreads + (threadIdx.x & ~31); base < nvec_all;
         base += stride) {
        const int64_t v = base + lane;
        uint32_t wd[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
        if (v < nvec_full) {
            const uint4 a = ld_stream(reinterpret_cast<const uint4 *>(in) + 2 * v);
            const uint4 b = ld_stream(reinterpret_cast<const uint4 *>(in) + 2 * v + 1);
            wd[0] = a.x, wd[1] = a.y, wd[2] = a.z, wd[3] = a.w;
            wd[4] = b.x, wd[5] = b.y, wd[6] = b.z, wd[7] = b.w;
        } else if (v < nvec_all) {
#pragma unroll
            for (int j = 0; j < kQuantVec; ++j)
                if (v * kQuantVec + j < n) wd[j >> 1] |= uint32_t(in[v * kQuantVec + j]) << (16 * (j & 1));
        }
        uint32_t pairs[8];
        const uint32_t sbyte = mx_encode16(wd, pairs);
        if (v < nvec_full) {
            __stcs(reinterpret_cast<uint4 *>(codes) + v,
                   make_uint4(pairs[0] | (pairs[1] << 16), pairs[2] | (pairs[3] << 16), pairs[4] | (pairs[5] << 16),
                              pairs[6] | (pairs[7] << 16)));
        } else if (v < nvec_all) {
#pragma unroll
            for (int j = 0; j < kQuantVec; ++j)
                if (v * kQuantVec + j < n) codes[v * kQuantVec + j] = uint8_t(pairs[j >> 1] >> (8 * (j & 1)));
        }
        if ((lane & 1) == 0 && v < nvec_all) scales[v >> 1] = uint8_t(sbyte);
    }
}

// ------------------------------------------------------------------ probe

// Plain streaming copy, 16 bytes per thread per iteration: the achievable
// HBM bandwidth measured in the same process as the step.
__global__ void __launch_bounds__(256) copy_kernel(const uint4 *__restrict__ src, uint4 *__restrict__ dst, int64_t n16)
{
    const int64_t stride = int64_t(gridDim.x) * blockDim.x;
#pragma unroll 4
    for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n16; i += stride)
        __stcs(dst + i, __ldcs(src + i));
}

cudaError_t launch_quant(const uint16_t *in, int64_t n, uint8_t *codes, uint8_t *scales, cudaStream_t st)
{
    if (n == 0) return cudaSuccess;
    const void *fn = reinterpret_cast<const void *>(&quant_kernel);
    const int64_t nvec = (n + kQuantVec - 1) / kQuantVec;
    const int64_t want = (nvec + kQuantThreads - 1) / kQuantThreads;
    const int wave = wave_blocks(fn, kQuantThreads, 0);
    const int blocks = int(want < wave ? want : wave);
    quant_kernel<<<blocks, kQuantThreads, 0, st>>>(in, n, codes, scales);
    return cudaGetLastError();
}

cudaError_t launch_copy(const void *src, void *dst, int64_t bytes, cudaStream_t st)
{
    if (bytes == 0) return cudaSuccess;
    const void *fn = reinterpret_cast<const void *>(&copy_kernel);
    const int64_t n16 = bytes / 16;
    const int64_t want = (n16 + 255) / 256;
    const int wave = wave_blocks(fn, 256, 0);
    const int blocks = int(want < wave ? want : wave);
    copy_kernel<<<blocks, 256, 0, st>>>(static_cast<const uint4 *>(src), static_cast<uint4 *>(dst), n16);
    return cudaGetLastError();
}

}  // namespace zg
