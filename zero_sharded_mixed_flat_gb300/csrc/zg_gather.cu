// zg_gather.cu -- stage three: parameter shards gathered just in time.
//
// With the parameters themselves sharded (DeepSpeed documentation review,
// paragraph on the three stages; Zero From Scratch, items 9 and 18), rank r
// keeps only the parameters [r*S, (r+1)*S), and a layer gathers the flat
// range it computes on, [lo, hi), from the owners right before it runs. On one
// GPU the P shards are P device buffers and the gather is an HBM-bound copy
// (2 bytes read + 2 written per bf16 parameter), or a decode of MXFP8 shards
// (1 + 1/32 read + 2 written). The output is stored with the default cache
// policy so that the layer's computation finds it in L2; the shards are read
// with the streaming (evict-first) policy.
#include "zg_launch.h"

namespace zg {

constexpr int kGatherThreads = 256;
constexpr int kGatherUnroll = 4;    // independent bf16 vectors in flight per thread
constexpr int kGatherUnrollMx = 4;  // independent MX vectors in flight per thread
constexpr int kMxVec = 8;           // MX elements per thread per vector: one 8-byte code load, one 16-byte store

// Owner of flat index i: rank floor(i / s). The binary32 estimate i * (1/s)
// carries a relative error below 2^-22 and i / s < 16, so it is within 2^-18
// of the quotient: off by at most one, and one correction each way makes it
// exact.
struct Owner {
    int64_t s;
    int p;
    float inv_s;

    __device__ __forceinline__ int rank(int64_t i) const
    {
        int r = int(float(i) * inv_s);
        r = r > p - 1 ? p - 1 : r;
        if (int64_t(r) * s > i)
            --r;
        else if (int64_t(r + 1) * s <= i)
            ++r;
        return r;
    }
};

// a[r] for a rank known only at run time, as a chain of selects over the
// kernel-parameter table (a dynamic index would copy the table to local
// memory).
template <class T>
__device__ __forceinline__ T pick(const T (&a)[kMaxRanks], int r)
{
    T x = a[0];
#pragma unroll
    for (int k = 1; k < kMaxRanks; ++k) x = r == k ? a[k] : x;
    return x;
}

struct Bf16Shards {
    const uint16_t *p[kMaxRanks];
};

struct MxShards {
    const uint8_t *c[kMaxRanks];
    const uint8_t *s[kMaxRanks];
};

// One MX element to bf16: its exact binary32 value rounded to nearest even;
// NaN (a NaN code or a NaN scale) gathers as the quiet NaN 0x7FC0.
__device__ __forceinline__ uint32_t mx_to_bf16(float x)
{
    return x != x ? 0x7fc0u : uint32_t(__bfloat16_as_ushort(__float2bfloat16_rn(x)));
}

// 8 codes of one block at one scale byte to 8 bf16 values (4 words, element
// 2k in the low half). A NaN scale or any NaN code (0x7F / 0xFF, which the
// encoder writes only into blocks with a NaN scale) sends the vector down the
// element-wise path, which maps NaN to 0x7FC0.
__device__ __forceinline__ uint4 mx8_to_bf16(uint2 c, uint32_t sbyte)
{
    const uint32_t cw[2] = {c.x, c.y};
    uint32_t nan = sbyte == 0xffu;
#pragma unroll
    for (int q = 0; q < 2; ++q) nan |= __vcmpeq4(cw[q] & 0x7f7f7f7fu, 0x7f7f7f7fu);
    const float scale = e8m0_value(sbyte);
    uint32_t w[4];
    if (!nan) {
        const float2 s2 = make_float2(scale, scale);
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            const float2 a = mul_f32x2(e4m3x2_to_f32x2(uint16_t(cw[q])), s2);
            const float2 b = mul_f32x2(e4m3x2_to_f32x2(uint16_t(cw[q] >> 16)), s2);
            w[2 * q] = pack_bf16x2(a.x, a.y);
            w[2 * q + 1] = pack_bf16x2(b.x, b.y);
        }
    } else {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float2 f = e4m3x2_to_f32x2(uint16_t(cw[q >> 1] >> (16 * (q & 1))));
            w[q] = mx_to_bf16(__fmul_rn(f.x, scale)) | (mx_to_bf16(__fmul_rn(f.y, scale)) << 16);
        }
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// The owning shard of the index a thread is at. A thread's indices only grow
// (grid-stride loops), so it looks its owner up again only when it leaves
// the flat range [start, next) of the current one: at most P times.
struct Cursor {
    int64_t start = 0, next = 0;
    int r = 0;

    __device__ __forceinline__ bool locate(const Owner &own, int64_t i)
    {
        if (i >= start && i < next) return false;
        r = own.rank(i);
        start = int64_t(r) * own.s;
        next = start + own.s;
        return true;
    }
};

// bf16 shards -> out[0, n) = parameters [lo, lo + n). With lo a multiple of 8
// every 8-element vector lies inside one shard (S is a multiple of 32) and
// moves as one 16-byte load and store; otherwise element by element.
__global__ void __launch_bounds__(kGatherThreads)
    gather_kernel(Bf16Shards sh, Owner own, int64_t lo, int64_t n, uint16_t *__restrict__ out)
{
    const int64_t stride = int64_t(gridDim.x) * kGatherThreads;
    const int64_t tid = int64_t(blockIdx.x) * kGatherThreads + threadIdx.x;
    Cursor cur;
    const uint16_t *base = nullptr;
    int64_t done = 0;
    if ((lo & (kVec - 1)) == 0) {
        const int64_t nvec = n / kVec;
#pragma unroll 1
        for (int64_t v0 = tid; v0 < nvec; v0 += kGatherUnroll * stride) {
            uint4 x[kGatherUnroll];
#pragma unroll
            for (int u = 0; u < kGatherUnroll; ++u) {
                const int64_t v = v0 + u * stride;
                if (v < nvec) {
                    const int64_t i = lo + v * kVec;
                    if (cur.locate(own, i)) base = pick(sh.p, cur.r);
                    x[u] = ld_stream(reinterpret_cast<const uint4 *>(base + (i - cur.start)));
                }
            }
#pragma unroll
            for (int u = 0; u < kGatherUnroll; ++u) {
                const int64_t v = v0 + u * stride;
                if (v < nvec) reinterpret_cast<uint4 *>(out)[v] = x[u];
            }
        }
        done = nvec * kVec;
    }
#pragma unroll 1
    for (int64_t j = done + tid; j < n; j += stride) {
        const int64_t i = lo + j;
        if (cur.locate(own, i)) base = pick(sh.p, cur.r);
        out[j] = base[i - cur.start];
    }
}

// MX shards -> bf16 out[0, n). With lo a multiple of 8 each thread decodes
// 8 codes of one 32-element block (one 8-byte load, one scale byte shared by
// four lanes) into one 16-byte store, so a warp's loads and stores each
// cover one contiguous span (256 and 512 bytes); otherwise element by
// element.
__global__ void __launch_bounds__(kGatherThreads)
    gather_mx_kernel(MxShards sh, Owner own, int64_t lo, int64_t n, uint16_t *__restrict__ out)
{
    const int64_t stride = int64_t(gridDim.x) * kGatherThreads;
    const int64_t tid = int64_t(blockIdx.x) * kGatherThreads + threadIdx.x;
    Cursor cur;
    const uint8_t *cbase = nullptr, *sbase = nullptr;
    int64_t done = 0;
    if ((lo & (kMxVec - 1)) == 0) {
        const int64_t nvec = n / kMxVec;
#pragma unroll 1
        for (int64_t v0 = tid; v0 < nvec; v0 += kGatherUnrollMx * stride) {
            uint2 c[kGatherUnrollMx];
            uint32_t sb[kGatherUnrollMx];
#pragma unroll
            for (int u = 0; u < kGatherUnrollMx; ++u) {
                const int64_t v = v0 + u * stride;
                if (v < nvec) {
                    const int64_t i = lo + v * kMxVec;
                    if (cur.locate(own, i)) {
                        cbase = pick(sh.c, cur.r);
                        sbase = pick(sh.s, cur.r);
                    }
                    const int64_t k = i - cur.start;
                    c[u] = ld_stream(reinterpret_cast<const uint2 *>(cbase + k));
                    sb[u] = sbase[k >> 5];
                }
            }
#pragma unroll
            for (int u = 0; u < kGatherUnrollMx; ++u) {
                const int64_t v = v0 + u * stride;
                if (v < nvec) reinterpret_cast<uint4 *>(out)[v] = mx8_to_bf16(c[u], sb[u]);
            }
        }
        done = nvec * kMxVec;
    }
#pragma unroll 1
    for (int64_t j = done + tid; j < n; j += stride) {
        const int64_t i = lo + j;
        if (cur.locate(own, i)) {
            cbase = pick(sh.c, cur.r);
            sbase = pick(sh.s, cur.r);
        }
        const int64_t k = i - cur.start;
        const float x = __fmul_rn(e4m3x2_to_f32x2(uint16_t(cbase[k])).x, e8m0_value(sbase[k >> 5]));
        out[j] = uint16_t(mx_to_bf16(x));
    }
}

namespace {

template <class Kernel>
int gather_blocks(Kernel *kernel, int64_t units)
{
    const int64_t want = (units + kGatherThreads - 1) / kGatherThreads;
    const int wave = wave_blocks(reinterpret_cast<const void *>(kernel), kGatherThreads, 0);
    return int(want < 1 ? 1 : (want < wave ? want : wave));
}

Owner owner_of(int p, int64_t s) { return Owner{s, p, float(1.0 / double(s))}; }

}  // namespace

cudaError_t launch_gather(int p, int64_t s, const uint16_t *const *shards, int64_t lo, int64_t hi, uint16_t *out,
                          cudaStream_t st)
{
    const int64_t n = hi - lo;
    if (n <= 0) return cudaSuccess;
    Bf16Shards sh{};
    for (int r = 0; r < p; ++r) sh.p[r] = shards[r];
    const int64_t units = (lo % kVec) == 0 ? (n + kVec - 1) / kVec : n;
    gather_kernel<<<gather_blocks(&gather_kernel, units), kGatherThreads, 0, st>>>(sh, owner_of(p, s), lo, n, out);
    return cudaGetLastError();
}

cudaError_t launch_gather_mx(int p, int64_t s, const uint8_t *const *codes, const uint8_t *const *scales, int64_t lo,
                             int64_t hi, uint16_t *out, cudaStream_t st)
{
    const int64_t n = hi - lo;
    if (n <= 0) return cudaSuccess;
    MxShards sh{};
    for (int r = 0; r < p; ++r) {
        sh.c[r] = codes[r];
        sh.s[r] = scales[r];
    }
    const int64_t units = (lo % kMxVec) == 0 ? (n + kMxVec - 1) / kMxVec : n;
    gather_mx_kernel<<<gather_blocks(&gather_mx_kernel, units), kGatherThreads, 0, st>>>(sh, owner_of(p, s), lo, n,
                                                                                          out);
    return cudaGetLastError();
}

}  // namespace zg
