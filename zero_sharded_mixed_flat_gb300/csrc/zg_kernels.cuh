// zg_kernels.cuh -- device code of the sharded mixed-precision optimizer step.
//
// Memory-bound throughout (about 20 fp32 operations against 2P + 26 bytes
// per parameter), so no tensor cores: the design goal is one coalesced
// 128-bit read and write per array per element and enough bytes in flight
// per SM to keep HBM3e busy.
//
// Numerics: every per-element operation uses a correctly rounded intrinsic
// (__fadd_rn, __fmul_rn, __fdiv_rn, __fsqrt_rn), which the compiler never
// fuses into an FMA, in the order the step is defined:
//   g  = (G_0 + G_1 + ... + G_{P-1}) * inv        (reduce-scatter + unscale)
//   ga = g * c; m = b1*m + (1-b1)*ga; v = b2*v + (1-b2)*(ga*ga)
//   mh = m/bc1; vh = v/bc2; d = sqrt(vh) + eps
//   w = w - (lr*wd)*w; w = w - lr*(mh/d); p = bf16_rne(w)
// (Zero From Scratch, items 3, 6 and 7; the AdamW form is the textbook one
// with decoupled weight decay, the pages print no formula.) The one fused
// multiply-add is in the MXFP8 decode, where each product E4M3 * 2^(s - 127)
// is exact, so fusing it with the rank sum changes no bit (MxSrc::reduce).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <type_traits>
#include <utility>

namespace zg {

constexpr int kMaxRanks = 16;
constexpr int kVec = 8;  // elements per thread per iteration: one 16-byte bf16 load

// Device-resident step scalars. The norm pass writes the "pending" decision;
// the step pass consumes it and commits the step count. The host reads the
// block only in zg_get_info, so a skipped step never needs a host round trip.
struct Scalars {
    double sumsq;
    double norm;
    double b1p_next;
    double b2p_next;
    int64_t t_next;
    float clip;
    float bc1;
    float bc2;
    int found_inf;
    int64_t t;
    double b1p;
    double b2p;
    unsigned int norm_ticket;  // norm-pass blocks finished in the current launch
    unsigned int step_ticket;  // step-pass blocks finished in the current launch
    unsigned int norm_gen;     // bumped by every norm finalize
    unsigned int step_gen;     // = norm_gen once a step pass consumed that norm
    int status;                // sticky device status (ZG_OK or ZG_ERR_*)
    unsigned int step_faults;  // CTAs of the current step launch whose wait ran out
    double bucket_acc;         // running sum of squares over the buckets submitted so far
};
static_assert(sizeof(Scalars) == 112, "the host copies this block back; keep its size in step");

// How a norm launch ends: kNormWhole finalizes its own total; a bucket
// launch (kNormBucket) adds its total to bucket_acc in submission order,
// restarting the sum on kNormFirst and finalizing on kNormLast.
constexpr int kNormWhole = 0;
constexpr int kNormFirst = 1;
constexpr int kNormLast = 2;
constexpr int kNormBucket = 4;

struct FinalizeK {
    double beta1, beta2, max_grad_norm, norm_eps;
};

// Per-step fp32 constants, each formed in fp64 on the host and rounded once.
struct StepK {
    float b1, b2, omb1, omb2, eps, lr, lrwd;
};

struct State {
    float *w, *m, *v;
    uint16_t *p;        // bf16 parameters (written unless MX parameters are bound)
    uint8_t *pcodes;    // MXFP8 parameters: E4M3 codes, one per element, or null
    uint8_t *pscales;   // and their E8M0 scales, one per 32 elements
    unsigned long long *work;  // the work array below (kWorkWords words, zero between launches)
};

// The work array, a small device array that is zero between launches (the
// last block of each launch clears what it used). The fused step pass and the
// norm pass each hand out their vectors in warp chunks from kWorkLanes
// counters, each counter in its own 256-byte line; the norm pass also adds
// its exact sum of squares into kAccDigits words and records non-finite
// squares in one flag word.
constexpr int kWorkLanes = 8;
constexpr int kWorkStride = 32;  // 64-bit words from one counter to the next
constexpr int kStepCtr = 0;                              // the step pass's counters
constexpr int kNormCtr = kStepCtr + kWorkLanes * kWorkStride;  // the norm pass's counters
constexpr int kAccDigits = 12;                           // base-2^32 digits of the norm's fixed-point sum
constexpr int kNormAcc = kNormCtr + kWorkLanes * kWorkStride;
constexpr int kNormFlags = kNormAcc + 16;                // bit 0: an infinite square, bit 1: a NaN one
constexpr int kWorkWords = kNormFlags + kWorkStride;

constexpr int kStatusTimeout = -5;     // ZG_ERR_DEVICE_TIMEOUT
constexpr int kStatusStaleNorm = -6;   // ZG_ERR_STALE_NORM
constexpr int kStatusPartial = -8;     // ZG_ERR_STATE_PARTIAL

// step_faults: the low 31 bits count the CTAs of the current step launch
// whose wait ran out; the top bit is set once any CTA has stored results.
constexpr unsigned int kFaultStored = 0x80000000u;

// ------------------------------------------------------------------ loads

// Streaming loads. ZG_LOAD_HINT picks the cache policy: 0 = evict-first
// (ld.global.cs), 1 = read-only non-coherent path (ld.global.nc), 2 = plain.
#ifndef ZG_LOAD_HINT
#define ZG_LOAD_HINT 0
#endif
template <class T>
__device__ __forceinline__ T ld_hint(const T *p)
{
#if ZG_LOAD_HINT == 0
    return __ldcs(p);
#elif ZG_LOAD_HINT == 1
    return __ldg(p);
#else
    return *p;
#endif
}
__device__ __forceinline__ uint4 ld_stream(const uint4 *p) { return ld_hint(p); }

// A 16-byte load that asks L2 to keep the line (evict-last policy): the norm
// pass reads the gradients this way when the step pass is to find the last
// ones it touched still in L2.
__device__ __forceinline__ uint4 ld_keep_l2(const uint4 *p)
{
    uint64_t pol;
    asm("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    uint4 r;
    asm volatile("ld.global.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p), "l"(pol));
    return r;
}

// The step pass walks the vectors from the end, where the norm pass
// finished: its first reads find the norm pass's last gradient lines still in
// L2, and the dependent launch overlaps on warm data. Measured on GB300: whole
// step +5 % at N = 2^24, +4 % at N = 1.2e8 (P = 8). Asking L2 to keep the
// norm pass's loads (evict-last) measured no gain and stays off.
#ifndef ZG_NORM_KEEP_L2
#define ZG_NORM_KEEP_L2 0
#endif
#ifndef ZG_STEP_REVERSE
#define ZG_STEP_REVERSE 1
#endif
__device__ __forceinline__ uint2 ld_stream(const uint2 *p) { return ld_hint(p); }
__device__ __forceinline__ float4 ld_stream(const float4 *p) { return __ldcs(p); }
__device__ __forceinline__ void st_stream(float4 *p, float4 v) { __stcs(p, v); }
__device__ __forceinline__ void st_stream(uint4 *p, uint4 v) { __stcs(p, v); }

// Programmatic dependent launch. A kernel launched with programmatic stream
// serialisation may start while the kernel before it on the stream is still
// running; pdl_wait() blocks until that kernel has completed and its writes
// are visible (a no-op for an ordinary launch), and pdl_trigger() lets the
// next kernel on the stream start launching its blocks.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Pull a line into L2 ahead of its load.
__device__ __forceinline__ void prefetch_l2(const void *p) { asm volatile("prefetch.global.L2 [%0];" ::"l"(p)); }

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Two binary32 values to packed bf16 (lo in bits 0..15), round to nearest even.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}

// Two binary32 operations per instruction (Blackwell's packed fp32 pipe),
// each lane rounded to nearest even exactly as its scalar form would be.
__device__ __forceinline__ float2 mul_f32x2(float2 a, float2 b)
{
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;"
        : "=l"(d)
        : "l"(*reinterpret_cast<const uint64_t *>(&a)), "l"(*reinterpret_cast<const uint64_t *>(&b)));
    return *reinterpret_cast<const float2 *>(&d);
}

__device__ __forceinline__ float2 fma_f32x2(float2 a, float2 b, float2 c)
{
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;"
        : "=l"(d)
        : "l"(*reinterpret_cast<const uint64_t *>(&a)), "l"(*reinterpret_cast<const uint64_t *>(&b)),
          "l"(*reinterpret_cast<const uint64_t *>(&c)));
    return *reinterpret_cast<const float2 *>(&d);
}

// ------------------------------------------------------------------ MXFP8

// E8M0 scale byte to its value 2^(s - 127) as a binary32; 0 gives the
// subnormal 2^-127 and 0xFF is NaN.
__device__ __forceinline__ float e8m0_value(uint32_t s)
{
    if (s == 0xffu) return __uint_as_float(0x7fc00000u);
    return __uint_as_float(s == 0u ? 0x00400000u : (s << 23));
}

// Two E4M3 codes (element 2k in the low byte) to two binary32 values, exact.
__device__ __forceinline__ float2 e4m3x2_to_f32x2(uint16_t codes)
{
    uint32_t h2;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(codes));
    return __half22float2(*reinterpret_cast<__half2 *>(&h2));
}

// Two binary32 values to E4M3 codes, round to nearest even, saturating at
// +-448; `lo` goes to the low byte.
__device__ __forceinline__ uint32_t f32x2_to_e4m3x2(float lo, float hi)
{
    uint16_t d;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(d) : "f"(hi), "f"(lo));
    return d;
}

// ------------------------------------------------------------------ MXFP8 encoder core

// A slice of one 32-element MX block, 2W bf16 values (wd: element 2k in the
// low half of word k; values past the end of the data loaded as zero),
// encoded by the 16 / W neighbouring lanes that hold the block's slices
// (W = 8: two lanes of sixteen values, W = 4: four lanes of eight), so every
// lane of the warp must call this together. The block amax is a max over the
// |x| bit patterns (non-negative bf16 order like unsigned integers), taken on
// 16-bit pairs and combined across the lanes with xor shuffles. E8M0 byte
// from the amax exponent field E: e = max(E - 135, -127), byte = e + 127; a
// block holding inf or NaN gets byte 0xFF and codes 0x7F. x * 2^-e is exact
// wherever the E4M3 rounding can see it, so the packed multiply gives the
// codes of the scalar one. Returns the scale byte; pairs[q] holds the codes
// of elements 2q and 2q + 1 (low byte first).
template <int W>
__device__ __forceinline__ uint32_t mx_encode_slice(const uint32_t (&wd)[W], uint32_t (&pairs)[W])
{
    static_assert(W == 4 || W == 8, "a block is split over two or four lanes");
    uint32_t m2 = 0u;
#pragma unroll
    for (int q = 0; q < W; ++q) m2 = __vmaxu2(m2, wd[q] & 0x7fff7fffu);
    uint32_t amax = max(m2 & 0xffffu, m2 >> 16);
#pragma unroll
    for (int off = 1; off < 16 / W; off <<= 1) amax = max(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    const bool bad = amax >= 0x7f80u;
    const uint32_t ex = amax >> 7;
    const uint32_t sbyte = bad ? 0xffu : (ex > 8u ? ex - 8u : 0u);
    const float to_unit = __uint_as_float((254u - (bad ? 0u : sbyte)) << 23);  // 2^-e
    const float2 u2 = make_float2(to_unit, to_unit);
#pragma unroll
    for (int q = 0; q < W; ++q) {
        const float2 y = mul_f32x2(make_float2(bf16_lo(wd[q]), bf16_hi(wd[q])), u2);
        pairs[q] = bad ? 0x7f7fu : f32x2_to_e4m3x2(y.x, y.y);
    }
    return sbyte;
}

__device__ __forceinline__ uint32_t mx_encode16(const uint32_t (&wd)[8], uint32_t (&pairs)[8])
{
    return mx_encode_slice<8>(wd, pairs);
}

// ------------------------------------------------------------------ gradient sources
//
// A source yields, for a vector of 8 consecutive flat indices, the
// rank-ordered fp32 sum of the P rank values (the reduce-scatter of one
// shard element), starting from +0.

template <int P>
struct Bf16Src {
    static constexpr int kRanks = P;
    const uint16_t *g[P];

    struct Raw {
        uint4 x[P];
    };

    __device__ __forceinline__ void prefetch(int64_t vec) const
    {
#pragma unroll
        for (int r = 0; r < P; ++r) prefetch_l2(g[r] + vec * kVec);
    }

    // Issue the P 16-byte loads of one vector.
    __device__ __forceinline__ void load(int64_t vec, Raw &raw) const
    {
#pragma unroll
        for (int r = 0; r < P; ++r) raw.x[r] = ld_stream(reinterpret_cast<const uint4 *>(g[r]) + vec);
    }

    // The norm pass's loads (kept in L2 when the step pass reuses them).
    __device__ __forceinline__ void load_norm(int64_t vec, Raw &raw) const
    {
#if ZG_NORM_KEEP_L2
#pragma unroll
        for (int r = 0; r < P; ++r) raw.x[r] = ld_keep_l2(reinterpret_cast<const uint4 *>(g[r]) + vec);
#else
        load(vec, raw);
#endif
    }

    // Rank-ordered fp32 sums of a loaded vector.
    __device__ __forceinline__ void reduce(const Raw &raw, float (&out)[kVec]) const
    {
#pragma unroll
        for (int j = 0; j < kVec; ++j) out[j] = 0.0f;
#pragma unroll
        for (int r = 0; r < P; ++r) {
            const uint32_t w4[4] = {raw.x[r].x, raw.x[r].y, raw.x[r].z, raw.x[r].w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                out[2 * q] = __fadd_rn(out[2 * q], bf16_lo(w4[q]));
                out[2 * q + 1] = __fadd_rn(out[2 * q + 1], bf16_hi(w4[q]));
            }
        }
    }

    __device__ __forceinline__ float sum1(int64_t i) const
    {
        float s = 0.0f;
#pragma unroll
        for (int r = 0; r < P; ++r) s = __fadd_rn(s, __uint_as_float(uint32_t(g[r][i]) << 16));
        return s;
    }
};

template <int P>
struct MxSrc {
    static constexpr int kRanks = P;
    const uint8_t *c[P];  // E4M3 codes, one byte per element
    const uint8_t *s[P];  // E8M0 scales, one byte per 32 elements

    struct Raw {
        uint2 x[P];
        uint32_t sc[P];
    };

    __device__ __forceinline__ void prefetch(int64_t vec) const
    {
#pragma unroll
        for (int r = 0; r < P; ++r) prefetch_l2(c[r] + vec * kVec);
    }

    __device__ __forceinline__ void load(int64_t vec, Raw &raw) const
    {
#pragma unroll
        for (int r = 0; r < P; ++r) {
            raw.x[r] = ld_stream(reinterpret_cast<const uint2 *>(c[r]) + vec);
            raw.sc[r] = s[r][vec >> 2];
        }
    }

    // Each decoded product E4M3 * 2^(s - 127) is exact in binary32 while
    // s <= 246 (the largest scale byte the encoder writes for finite data),
    // so one fused multiply-add per element yields exactly the bits of the
    // separate multiply and add, and the packed form takes two elements per
    // instruction. A vector with a scale byte in 247..254 (which the encoder
    // never writes) keeps the separate operations, where a product that
    // overflows must read as inf before it is added.
    __device__ __forceinline__ void reduce(const Raw &raw, float (&out)[kVec]) const
    {
        uint32_t big = 0u;
#pragma unroll
        for (int r = 0; r < P; ++r) big |= uint32_t(raw.sc[r] - 247u < 8u);
        if (!big) {
            float2 acc[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) acc[q] = make_float2(0.0f, 0.0f);
#pragma unroll
            for (int r = 0; r < P; ++r) {
                const float scale = e8m0_value(raw.sc[r]);
                const float2 s2 = make_float2(scale, scale);
                const uint32_t w2[2] = {raw.x[r].x, raw.x[r].y};
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    acc[q] = fma_f32x2(e4m3x2_to_f32x2(uint16_t(w2[q >> 1] >> (16 * (q & 1)))), s2, acc[q]);
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                out[2 * q] = acc[q].x;
                out[2 * q + 1] = acc[q].y;
            }
            return;
        }
#pragma unroll
        for (int j = 0; j < kVec; ++j) out[j] = 0.0f;
#pragma unroll
        for (int r = 0; r < P; ++r) {
            const float scale = e8m0_value(raw.sc[r]);
            const uint32_t w2[2] = {raw.x[r].x, raw.x[r].y};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float2 f = e4m3x2_to_f32x2(uint16_t(w2[q >> 1] >> (16 * (q & 1))));
                out[2 * q] = __fadd_rn(out[2 * q], __fmul_rn(f.x, scale));
                out[2 * q + 1] = __fadd_rn(out[2 * q + 1], __fmul_rn(f.y, scale));
            }
        }
    }

    __device__ __forceinline__ float sum1(int64_t i) const
    {
        float s = 0.0f;
#pragma unroll
        for (int r = 0; r < P; ++r) {
            const float2 f = e4m3x2_to_f32x2(uint16_t(c[r][i]));
            s = __fadd_rn(s, __fmul_rn(f.x, e8m0_value(this->s[r][i >> 5])));
        }
        return s;
    }
};

// The reduce-scatter output kept from the norm pass: the unscaled, averaged
// fp32 shard gradient g, 4 bytes per parameter (used with inv = 1).
struct StagedSrc {
    static constexpr int kRanks = 1;
    const float *g;

    struct Raw {
        float4 a, b;
    };

    __device__ __forceinline__ void prefetch(int64_t vec) const { prefetch_l2(g + vec * kVec); }

    __device__ __forceinline__ void load(int64_t vec, Raw &raw) const
    {
        const float4 *p = reinterpret_cast<const float4 *>(g) + 2 * vec;
        raw.a = __ldcs(p);
        raw.b = __ldcs(p + 1);
    }

    __device__ __forceinline__ void reduce(const Raw &raw, float (&out)[kVec]) const
    {
        out[0] = raw.a.x, out[1] = raw.a.y, out[2] = raw.a.z, out[3] = raw.a.w;
        out[4] = raw.b.x, out[5] = raw.b.y, out[6] = raw.b.z, out[7] = raw.b.w;
    }

    __device__ __forceinline__ float sum1(int64_t i) const { return g[i]; }
};

// ------------------------------------------------------------------ reductions

// Error-free accumulation of x into the unevaluated pair hi + lo (Knuth's
// two-sum): the norm keeps about 48 bits per thread without fp64 arithmetic,
// which GB300 runs at a small fraction of its fp32 rate.
__device__ __forceinline__ void two_sum_acc(float &hi, float &lo, float x)
{
    const float s = __fadd_rn(hi, x);
    const float bp = __fsub_rn(s, hi);
    const float e = __fadd_rn(__fsub_rn(hi, __fsub_rn(s, bp)), __fsub_rn(x, bp));
    hi = s;
    lo = __fadd_rn(lo, e);
}

// Deterministic block sum of one double per thread; the result is valid in
// thread 0. Fixed butterfly within warps, then warp 0 over the warp sums.
template <int THREADS>
__device__ __forceinline__ double block_sum(double x, double *smem)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
    __syncthreads();  // earlier readers of smem are done
    if (lane == 0) smem[warp] = x;
    __syncthreads();
    if (warp == 0) {
        x = lane < THREADS / 32 ? smem[lane] : 0.0;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
    }
    return x;
}

// ------------------------------------------------------------------ AdamW element

__device__ __forceinline__ void adamw(float g, float c, float bc1, float bc2, const StepK &k,
                                      float &w, float &m, float &v)
{
    const float ga = __fmul_rn(g, c);
    const float mi = __fadd_rn(__fmul_rn(k.b1, m), __fmul_rn(k.omb1, ga));
    const float vi = __fadd_rn(__fmul_rn(k.b2, v), __fmul_rn(k.omb2, __fmul_rn(ga, ga)));
    const float mh = __fdiv_rn(mi, bc1);
    const float vh = __fdiv_rn(vi, bc2);
    const float den = __fadd_rn(__fsqrt_rn(vh), k.eps);
    float wi = __fsub_rn(w, __fmul_rn(k.lrwd, w));
    wi = __fsub_rn(wi, __fmul_rn(k.lr, __fdiv_rn(mh, den)));
    m = mi;
    v = vi;
    w = wi;
}

// ------------------------------------------------------------------ norm pass

constexpr int kNormThreads = 256;

// Resident blocks per SM the compiler must allow (caps registers per
// thread): four 256-thread blocks while the P loads of a vector fit in 64
// registers without spilling (P = 5..8), three where a lane loads several
// chunks' vectors at once (P < 5, see NormChunksPerTake), two above P = 8.
template <class Src>
struct NormMinBlocks {
#ifdef ZG_NORM_MINB
    static constexpr int value = ZG_NORM_MINB;
#else
    static constexpr int value = Src::kRanks > 8 ? 2 : (Src::kRanks >= 5 ? 4 : 3);
#endif
};
// The tail of the staged gradient written with the default store policy (see
// norm_kernel); the rest uses evict-first stores.
#ifndef ZG_STAGE_KEEP_MB
#define ZG_STAGE_KEEP_MB 96
#endif
constexpr int64_t kStageKeepBytes = int64_t(ZG_STAGE_KEEP_MB) << 20;

// Finalize: runs once, in the last block of the norm pass (thread 0), given
// the step count and running powers the step passes left in `sc`.
__device__ __forceinline__ void finalize_decision(Scalars *sc, double sumsq, const FinalizeK &fk, int64_t t,
                                                  double b1p, double b2p)
{
    const int bad = !isfinite(sumsq);
    sc->sumsq = sumsq;
    sc->norm = sqrt(sumsq);
    sc->found_inf = bad;
    if (bad) {
        sc->t_next = t;
        sc->b1p_next = b1p;
        sc->b2p_next = b2p;
        sc->clip = 1.0f;
        sc->bc1 = 1.0f;
        sc->bc2 = 1.0f;
    } else {
        const double b1n = b1p * fk.beta1, b2n = b2p * fk.beta2;
        sc->t_next = t + 1;
        sc->b1p_next = b1n;
        sc->b2p_next = b2n;
        sc->bc1 = float(1.0 - b1n);
        sc->bc2 = float(1.0 - b2n);
        if (fk.max_grad_norm > 0.0) {
            const double q = fk.max_grad_norm / (sc->norm + fk.norm_eps);
            sc->clip = float(q < 1.0 ? q : 1.0);
        } else {
            sc->clip = 1.0f;
        }
    }
    sc->norm_gen = sc->norm_gen + 1u;
}

__device__ __forceinline__ void finalize_decision(Scalars *sc, double sumsq, const FinalizeK &fk)
{
    finalize_decision(sc, sumsq, fk, sc->t, sc->b1p, sc->b2p);
}

// The end of every norm pass: the block's fixed-tree sum of the threads'
// fp64 partials goes to partials[blockIdx.x]; the last block to finish (an
// atomic ticket) sums the block partials in index order and writes the
// decision (or, for a bucket, adds to the running bucket sum).
__device__ __forceinline__ void norm_finish(double acc, double *__restrict__ partials, Scalars *sc,
                                            const FinalizeK &fk, int mode)
{
    __shared__ double red[kNormThreads / 32];
    __shared__ int am_last;
    const double bsum = block_sum<kNormThreads>(acc, red);
    if (threadIdx.x == 0) {
        partials[blockIdx.x] = bsum;
        __threadfence();
        const unsigned int ticket = atomicAdd(&sc->norm_ticket, 1u);
        am_last = (ticket == gridDim.x - 1);
    }
    __syncthreads();
    if (!am_last) return;
    __threadfence();
    double s = 0.0;
    for (int i = threadIdx.x; i < int(gridDim.x); i += kNormThreads) s += __ldcg(partials + i);
    const double total = block_sum<kNormThreads>(s, red);
    if (threadIdx.x == 0) {
        if (!(mode & kNormBucket)) {
            finalize_decision(sc, total, fk);
        } else {
            const double run = (mode & kNormFirst) ? total : sc->bucket_acc + total;
            sc->bucket_acc = run;
            if (mode & kNormLast) finalize_decision(sc, run, fk);
        }
        sc->norm_ticket = 0u;
    }
}

// ------------------------------------------------------------------ exact, order-free norm sum
//
// The norm pass hands out its vectors in warp chunks, like the step pass, so
// which warp sums which chunk changes from launch to launch; the norm must
// not. A chunk is 32 consecutive vectors (one per lane): each lane adds its
// eight squares with two-sum into a binary32 pair (hi, lo), and the warp
// combines the 32 pairs in a fixed butterfly of pair additions (two-sum of
// the high parts, the low parts and the error added, renormalised), which
// leaves the chunk's sum as one pair (H, L) in every lane. H and L are
// binary32 values, integer multiples of 2^-149, and are added EXACTLY into a
// fixed-point accumulator that counts units of 2^-149 in kAccDigits base-2^32
// digits held one per lane (a 64-bit word per digit, so signed contributions
// and carries wait until the end). Integer addition does not care about
// order: the total is the exact sum of the chunk pairs, the same whichever
// warps took the chunks and whatever the grid. A chunk whose pair is not
// finite (a square that is inf or NaN, or a binary32 sum that overflowed)
// adds its finite squares one by one, exactly, and flags the others. The
// chunks are defined on g padded with zeros to whole vectors, so any pass
// that forms the same g (the fused MX encode-and-norm pass from decoded
// codes, when those hold the gradients exactly) gets the same bits.
// Blocks add their warps' words into the work array; the last block to
// finish turns the words into the correctly rounded binary64 sum of squares
// (non-finite when a square was: NaN before inf) and makes the decision.

__device__ __forceinline__ void two_sum(float a, float b, float &s, float &e)
{
    s = __fadd_rn(a, b);
    const float bp = __fsub_rn(s, a);
    e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bp)), __fsub_rn(b, bp));
}

// (h, l) + (oh, ol) as binary32 pairs; the same bits whichever operand comes
// first (two-sum's error term is exact, and each addition is commutative).
__device__ __forceinline__ void pair_add(float &h, float &l, float oh, float ol)
{
    float s, e;
    two_sum(h, oh, s, e);
    const float t = __fadd_rn(__fadd_rn(l, ol), e);
    h = __fadd_rn(s, t);
    l = __fsub_rn(t, __fsub_rn(h, s));
}

// Adds x * 2^149 (x a finite binary32 value of either sign, so an integer) to
// the digits held one per lane: x = m * 2^(max(E, 1) - 150) for the biased
// exponent E and the significand m, so x * 2^149 = m << (max(E, 1) - 1),
// which touches two digits.
__device__ __forceinline__ void acc_add(long long &word, float x, int lane)
{
    const uint32_t b = __float_as_uint(x);
    const uint32_t e = (b >> 23) & 0xffu;
    const uint32_t sh = (e ? e : 1u) - 1u;
    const uint64_t v = uint64_t((b & 0x7fffffu) | (e ? 0x800000u : 0u)) << (sh & 31u);
    const int k = int(sh >> 5);
    const long long add = lane == k ? (long long)(v & 0xffffffffull) : (lane == k + 1 ? (long long)(v >> 32) : 0ll);
    word += (b >> 31) ? -add : add;
}

// The accumulated digits as the correctly rounded binary64 value of their
// sum times 2^-149 (the sum is non-negative). One thread.
__device__ __forceinline__ double acc_to_double(const long long (&w)[kAccDigits])
{
    uint32_t d[kAccDigits];
    long long carry = 0;
#pragma unroll
    for (int i = 0; i < kAccDigits; ++i) {
        const long long t = w[i] + carry;
        d[i] = uint32_t(t);
        carry = t >> 32;  // floor division by 2^32
    }
    int top = -1;
#pragma unroll
    for (int i = 0; i < kAccDigits; ++i)
        if (d[i] != 0u) top = i;
    if (top < 0) return 0.0;
    // the 96 bits from the top digit down, shifted to put the leading one at
    // bit 95; the high 64 of them, with every lower bit folded into a sticky
    // bit 0 (below the rounding position), round as the whole would
    uint32_t a = 0u, b = 0u, c = 0u;
    bool sticky = false;
#pragma unroll
    for (int i = 0; i < kAccDigits; ++i) {  // constant indices: the digits stay in registers
        a = i == top ? d[i] : a;
        b = i == top - 1 ? d[i] : b;
        c = i == top - 2 ? d[i] : c;
        sticky |= i < top - 2 && d[i] != 0u;
    }
    const int lz = __clz(a);
    const uint64_t ab = (uint64_t(a) << 32) | b;
    uint64_t y = lz ? (ab << lz) | (uint64_t(c) >> (32 - lz)) : ab;
    const uint32_t rest = lz ? (c << lz) : c;
    if (rest != 0u || sticky) y |= 1ull;
    const int k = 32 * (top - 1) - lz - 149;  // y * 2^k, with -212 <= k <= 171
    return __ull2double_rn(y) * __longlong_as_double((long long)(k + 1023) << 52);
}

// One chunk's contribution: each lane holds its vector's eight g values and
// the two-sum pair (hi, lo) of their squares in element order. The warp's
// 32 pairs are combined by a fixed butterfly (xor distances 16, 8, 4, 2, 1)
// into the chunk pair, added exactly to the digits; if a lane's pair or the
// chunk pair is not finite, every square is added on its own instead and
// the non-finite ones are flagged. Warp-uniform; every lane must take part.
__device__ __forceinline__ void chunk_add(float hi, float lo, const float (&g)[kVec], int lane, long long &word,
                                          uint32_t &flags)
{
    if (__all_sync(0xffffffffu, isfinite(hi) && isfinite(lo))) {
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
            pair_add(hi, lo, __shfl_xor_sync(0xffffffffu, hi, off), __shfl_xor_sync(0xffffffffu, lo, off));
        if (isfinite(hi) && isfinite(lo)) {  // the same in every lane
            acc_add(word, hi, lane);
            acc_add(word, lo, lane);
            return;
        }
    }
    // rare: every square on its own, broadcast from its lane
#pragma unroll 1
    for (int from = 0; from < 32; ++from) {
#pragma unroll
        for (int j = 0; j < kVec; ++j) {
            const float x = __shfl_sync(0xffffffffu, __fmul_rn(g[j], g[j]), from);
            if (isfinite(x))
                acc_add(word, x, lane);
            else
                flags |= isnan(x) ? 2u : 1u;
        }
    }
}

// Chunks a warp takes at a time in the norm pass: with few ranks a vector
// is few bytes, so a lane loads one vector of each of U consecutive chunks
// before summing any (U * P * 16 bytes in flight per lane: U = 4 at P = 1
// and 2, 2 at P = 3 and 4, else 1). The chunks, and so the sum, do not
// change with U.
template <class Src>
struct NormChunksPerTake {
    static constexpr int value = Src::kRanks >= 5 ? 1 : (Src::kRanks >= 3 ? 2 : 4);
};

// The staged variant's store of vector v's g (the reduce-scatter output the
// step pass reads). Its last kStageKeepBytes (the part the step pass,
// walking from the end, reads first) get the default store policy so they
// can still be in L2; the rest streams out. The partial last vector is
// stored element by element; vectors past it store nothing.
__device__ __forceinline__ void norm_stage_store(float *__restrict__ stage, int64_t n, int64_t nfull, int64_t v,
                                                 const float (&gh)[kVec])
{
    if (v < nfull) {
        float4 *o = reinterpret_cast<float4 *>(stage) + 2 * v;
        const float4 a = make_float4(gh[0], gh[1], gh[2], gh[3]);
        const float4 b = make_float4(gh[4], gh[5], gh[6], gh[7]);
        if (v >= nfull - kStageKeepBytes / 32) {
            o[0] = a;
            o[1] = b;
        } else {
            __stcs(o, a);
            __stcs(o + 1, b);
        }
    } else if (v * kVec < n) {
#pragma unroll
        for (int j = 0; j < kVec; ++j)
            if (v * kVec + j < n) stage[v * kVec + j] = gh[j];
    }
}

// g of chunk `ch` at this lane (its vector, zeros past N), from the loaded
// raw vector when the vector is whole.
template <class Src>
__device__ __forceinline__ void chunk_g(const Src &src, int64_t n, float inv, int64_t ch, int lane,
                                        const typename Src::Raw &raw, float (&gh)[kVec])
{
    const int64_t v = ch * 32 + lane;
    if (v < n / kVec) {
        src.reduce(raw, gh);
    } else {
#pragma unroll
        for (int j = 0; j < kVec; ++j) gh[j] = v * kVec + j < n ? src.sum1(v * kVec + j) : 0.0f;
    }
#pragma unroll
    for (int j = 0; j < kVec; ++j) gh[j] = __fmul_rn(gh[j], inv);
}

// One warp's share of the norm pass over warp chunks (see above), adding
// into this lane's digit `word` and non-finite flags. The vectors are those
// of g padded with zeros to a multiple of 8 elements: the last, partial one
// is read element by element. Work is handed out in takes of U chunks, whose
// butterflies run side by side; each chunk is added exactly as chunk_add
// adds it (the same decision between its pair and its squares one by one).
template <class Src, bool kStage>
__device__ __forceinline__ void norm_chunk_loop(const Src &src, int64_t n, float inv, float *__restrict__ stage,
                                                unsigned long long *work, long long &word, uint32_t &flags)
{
    constexpr int U = NormChunksPerTake<Src>::value;
    const int64_t nfull = n / kVec;
    const int64_t nvec = (n + kVec - 1) / kVec;
    const int64_t nchunk = (nvec + 31) / 32;
    const int64_t ntake = (nchunk + U - 1) / U;
    const int lane = threadIdx.x & 31;
    const int q = threadIdx.x >> 5;
    unsigned long long *ctr = work + kNormCtr + q * kWorkStride;
    int64_t tk = q + int64_t(kWorkLanes) * blockIdx.x;
    if constexpr (U == 1) {
#pragma unroll 1
        while (tk < ntake) {  // warp-uniform
            unsigned long long next = 0ull;
            if (lane == 0) next = atomicAdd(ctr, 1ull);
            const int64_t v = tk * 32 + lane;
            typename Src::Raw raw;
            if (v < nfull) src.load_norm(v, raw);
            float gh[kVec];
            chunk_g(src, n, inv, tk, lane, raw, gh);
            float hi = 0.0f, lo = 0.0f;
#pragma unroll
            for (int j = 0; j < kVec; ++j) two_sum_acc(hi, lo, __fmul_rn(gh[j], gh[j]));
            if (kStage) norm_stage_store(stage, n, nfull, v, gh);
            chunk_add(hi, lo, gh, lane, word, flags);
            next = __shfl_sync(0xffffffffu, next, 0);
            tk = q + int64_t(kWorkLanes) * (int64_t(gridDim.x) + int64_t(next));
        }
    } else {
#pragma unroll 1
        while (tk < ntake) {  // warp-uniform
            unsigned long long next = 0ull;
            if (lane == 0) next = atomicAdd(ctr, 1ull);
            typename Src::Raw raw[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t v = (tk * U + u) * 32 + lane;
                if (v < nfull) src.load_norm(v, raw[u]);
            }
            float hi[U], lo[U];
            uint32_t fast = 0u;  // chunks whose lanes' pairs are all finite
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t ch = tk * U + u;  // chunks past the end are all zeros
                const int64_t v = ch * 32 + lane;
                float gh[kVec];
                chunk_g(src, n, inv, ch, lane, raw[u], gh);
                hi[u] = 0.0f;
                lo[u] = 0.0f;
#pragma unroll
                for (int j = 0; j < kVec; ++j) two_sum_acc(hi[u], lo[u], __fmul_rn(gh[j], gh[j]));
                if (kStage) norm_stage_store(stage, n, nfull, v, gh);
                fast |= uint32_t(__all_sync(0xffffffffu, isfinite(hi[u]) && isfinite(lo[u]))) << u;
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
#pragma unroll
                for (int u = 0; u < U; ++u)
                    pair_add(hi[u], lo[u], __shfl_xor_sync(0xffffffffu, hi[u], off),
                             __shfl_xor_sync(0xffffffffu, lo[u], off));
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                if (((fast >> u) & 1u) && isfinite(hi[u]) && isfinite(lo[u])) {  // the same in every lane
                    acc_add(word, hi[u], lane);
                    acc_add(word, lo[u], lane);
                } else {
                    // rare: every square on its own, broadcast from its lane (g
                    // loaded again, so the raw vectors need not stay in registers)
                    float gh[kVec];
                    typename Src::Raw again;
                    const int64_t v = (tk * U + u) * 32 + lane;
                    if (v < nfull) src.load_norm(v, again);
                    chunk_g(src, n, inv, tk * U + u, lane, again, gh);
#pragma unroll 1
                    for (int from = 0; from < 32; ++from) {
#pragma unroll
                        for (int j = 0; j < kVec; ++j) {
                            const float x = __shfl_sync(0xffffffffu, __fmul_rn(gh[j], gh[j]), from);
                            if (isfinite(x))
                                acc_add(word, x, lane);
                            else
                                flags |= isnan(x) ? 2u : 1u;
                        }
                    }
                }
            }
            next = __shfl_sync(0xffffffffu, next, 0);
            tk = q + int64_t(kWorkLanes) * (int64_t(gridDim.x) + int64_t(next));
        }
    }
}

// The end of a block's share of the norm: its digits and flags go into the
// work array, then an atomic ticket. True (in every thread) in the last
// block to finish.
__device__ __forceinline__ bool norm_block_publish(long long word, uint32_t flags, unsigned long long *work,
                                                   Scalars *sc)
{
    __shared__ long long s_acc[kNormThreads / 32][kAccDigits];
    __shared__ uint32_t s_flags;
    __shared__ int am_last;
    const int lane = threadIdx.x & 31, q = threadIdx.x >> 5;
    if (threadIdx.x == 0) s_flags = 0u;
    __syncthreads();
    if (lane < kAccDigits) s_acc[q][lane] = word;
    if (lane == 0 && flags) atomicOr(&s_flags, flags);
    __syncthreads();
    if (threadIdx.x < kAccDigits) {
        long long t = 0;
#pragma unroll
        for (int w = 0; w < kNormThreads / 32; ++w) t += s_acc[w][threadIdx.x];
        if (t) atomicAdd(work + kNormAcc + threadIdx.x, (unsigned long long)t);
    } else if (threadIdx.x == kAccDigits && s_flags) {
        atomicOr(reinterpret_cast<unsigned int *>(work + kNormFlags), s_flags);
    }
    if (threadIdx.x <= kAccDigits) __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
        const unsigned int ticket = atomicAdd(&sc->norm_ticket, 1u);
        am_last = (ticket == gridDim.x - 1);
    }
    __syncthreads();
    return am_last != 0;
}

// The last block's thread 0: takes the words (and clears them, the flags and
// the norm counters for the next launch), rounds the sum to binary64 and
// writes the decision (or, for a bucket, adds to the running bucket sum).
// The caller resets the ticket.
__device__ __forceinline__ void norm_total_decide(unsigned long long *work, Scalars *sc, const FinalizeK &fk,
                                                  int mode)
{
    __threadfence();
    // what the decision needs besides the sum, read while the words are fetched
    const int64_t t = sc->t;
    const double b1p = sc->b1p, b2p = sc->b2p, bucket_acc = sc->bucket_acc;
    long long w[kAccDigits];
#pragma unroll
    for (int i = 0; i < kAccDigits; ++i) w[i] = (long long)atomicExch(work + kNormAcc + i, 0ull);
    const unsigned int fl = atomicExch(reinterpret_cast<unsigned int *>(work + kNormFlags), 0u);
#pragma unroll
    for (int i = 0; i < kWorkLanes; ++i) work[kNormCtr + i * kWorkStride] = 0ull;
    double total = acc_to_double(w);
    if (fl & 2u)
        total = __longlong_as_double(0x7ff8000000000000ll);  // NaN
    else if (fl & 1u)
        total = __longlong_as_double(0x7ff0000000000000ll);  // +inf
    if (!(mode & kNormBucket)) {
        finalize_decision(sc, total, fk, t, b1p, b2p);
    } else {
        const double run = (mode & kNormFirst) ? total : bucket_acc + total;
        sc->bucket_acc = run;
        if (mode & kNormLast) finalize_decision(sc, run, fk, t, b1p, b2p);
    }
}

__device__ __forceinline__ void norm_exact_finish(long long word, uint32_t flags, unsigned long long *work,
                                                  Scalars *sc, const FinalizeK &fk, int mode)
{
    if (!norm_block_publish(word, flags, work, sc) || threadIdx.x != 0) return;
    norm_total_decide(work, sc, fk, mode);
    sc->norm_ticket = 0u;
}

// The norm pass: warp chunks, the exact sum above. Same gradients, N and P:
// bit-identical norm, run after run and on any grid.
template <class Src, bool kStage = false>
__global__ void __launch_bounds__(kNormThreads, NormMinBlocks<Src>::value)
    norm_kernel(Src src, int64_t n, float inv, unsigned long long *work, Scalars *sc, FinalizeK fk,
                float *__restrict__ stage = nullptr, int mode = kNormWhole)
{
    static_assert(kNormThreads / 32 == kWorkLanes && kAccDigits <= 32, "one counter per warp, one digit per lane");
    pdl_wait();     // the gradients may come from the kernel just before
    pdl_trigger();  // the step pass may start its blocks as ours retire
    long long word = 0;
    uint32_t flags = 0u;
    norm_chunk_loop<Src, kStage>(src, n, inv, stage, work, word, flags);
    norm_exact_finish(word, flags, work, sc, fk, mode);
}

// ------------------------------------------------------------------ fused step pass

constexpr int kStepThreads = 256;

// Resident 256-thread blocks per SM the compiler must allow. Three (up to
// 85 registers per thread) measured best on GB300: at two the SM holds too
// few loads in flight, at four the 64-register cap costs instruction-level
// parallelism (sweeps at N = 2^24 and 1.2e8, P = 4 and 8).
#ifndef ZG_STEP_MINB
#define ZG_STEP_MINB 3
#endif
template <class Src>
struct StepMinBlocks {
    static constexpr int value = ZG_STEP_MINB;
};

// Vectors whose loads a thread issues before computing any of them. The
// fused sources already put 2P + 24 bytes per vector in flight; the staged
// fp32 gradient only 32 + 24, so each thread takes two vectors at a time
// (at two resident blocks per SM to keep the registers).
#ifndef ZG_STAGED_UNROLL
#define ZG_STAGED_UNROLL 2
#endif
template <class Src>
struct StepUnroll {
    static constexpr int value = 1;
};
template <>
struct StepUnroll<StagedSrc> {
    static constexpr int value = ZG_STAGED_UNROLL;
};
template <int P>
struct StepMinBlocks<MxSrc<P>> {  // P > 8 MX operands need more than 85 registers
    static constexpr int value = P <= 8 ? ZG_STEP_MINB : 2;
};
template <>
struct StepMinBlocks<StagedSrc> {
    static constexpr int value = ZG_STAGED_UNROLL > 1 ? 2 : ZG_STEP_MINB;
};

// The last block of a step pass commits the step count (unless skipped) and
// marks the norm consumed, so a repeated step pass cannot apply twice.
__device__ __forceinline__ void step_epilogue(Scalars *sc, int skip, unsigned long long *work = nullptr)
{
    __syncthreads();
    if (threadIdx.x != 0) return;
    __threadfence();
    const unsigned int ticket = atomicAdd(&sc->step_ticket, 1u);
    if (ticket != gridDim.x - 1) return;
    if (work) {  // every warp has taken its last chunk: clear the counters for the next launch
#pragma unroll
        for (int q = 0; q < kWorkLanes; ++q) work[kStepCtr + q * kWorkStride] = 0ull;
    }
    if (skip == 2) {
        sc->status = kStatusStaleNorm;
    } else {
        if (skip == 0) {
            sc->t = sc->t_next;
            sc->b1p = sc->b1p_next;
            sc->b2p = sc->b2p_next;
        }
        sc->step_gen = sc->norm_gen;
    }
    sc->step_ticket = 0u;
}

// Read the decision once per block: skip = 0 run, 1 found inf, 2 stale norm.
__device__ __forceinline__ int step_prologue(const Scalars *sc, float &c, float &bc1, float &bc2)
{
    __shared__ int s_skip;
    __shared__ float s_c, s_bc1, s_bc2;
    if (threadIdx.x == 0) {
        const int stale = sc->step_gen == sc->norm_gen;
        s_skip = stale ? 2 : (sc->found_inf ? 1 : 0);
        s_c = sc->clip;
        s_bc1 = sc->bc1;
        s_bc2 = sc->bc2;
    }
    __syncthreads();
    c = s_c;
    bc1 = s_bc1;
    bc2 = s_bc2;
    return s_skip;
}

// One vector's operands: the gradient source's raw loads and w, m, v.
template <class Src>
struct VecData {
    typename Src::Raw raw;
    float4 w[2], m[2], v[2];
};

template <class Src>
__device__ __forceinline__ void step_load(const Src &src, int64_t vec, const State &st, VecData<Src> &d)
{
    src.load(vec, d.raw);
    const float4 *w4 = reinterpret_cast<const float4 *>(st.w) + 2 * vec;
    const float4 *m4 = reinterpret_cast<const float4 *>(st.m) + 2 * vec;
    const float4 *v4 = reinterpret_cast<const float4 *>(st.v) + 2 * vec;
    d.w[0] = ld_stream(w4), d.w[1] = ld_stream(w4 + 1);
    d.m[0] = ld_stream(m4), d.m[1] = ld_stream(m4 + 1);
    d.v[0] = ld_stream(v4), d.v[1] = ld_stream(v4 + 1);
}

template <class Src>
__device__ __forceinline__ void step_compute(const Src &src, const VecData<Src> &d, float inv, float c, float bc1,
                                             float bc2, const StepK &k, float (&w)[kVec], float (&m)[kVec],
                                             float (&v)[kVec])
{
    float gh[kVec];
    src.reduce(d.raw, gh);
    w[0] = d.w[0].x, w[1] = d.w[0].y, w[2] = d.w[0].z, w[3] = d.w[0].w;
    w[4] = d.w[1].x, w[5] = d.w[1].y, w[6] = d.w[1].z, w[7] = d.w[1].w;
    m[0] = d.m[0].x, m[1] = d.m[0].y, m[2] = d.m[0].z, m[3] = d.m[0].w;
    m[4] = d.m[1].x, m[5] = d.m[1].y, m[6] = d.m[1].z, m[7] = d.m[1].w;
    v[0] = d.v[0].x, v[1] = d.v[0].y, v[2] = d.v[0].z, v[3] = d.v[0].w;
    v[4] = d.v[1].x, v[5] = d.v[1].y, v[6] = d.v[1].z, v[7] = d.v[1].w;
#pragma unroll
    for (int j = 0; j < kVec; ++j) adamw(__fmul_rn(gh[j], inv), c, bc1, bc2, k, w[j], m[j], v[j]);
}

__device__ __forceinline__ void store_state(int64_t vec, const State &st, const float (&w)[kVec],
                                            const float (&m)[kVec], const float (&v)[kVec])
{
    float4 *w4 = reinterpret_cast<float4 *>(st.w) + 2 * vec;
    float4 *m4 = reinterpret_cast<float4 *>(st.m) + 2 * vec;
    float4 *v4 = reinterpret_cast<float4 *>(st.v) + 2 * vec;
    st_stream(w4, make_float4(w[0], w[1], w[2], w[3]));
    st_stream(w4 + 1, make_float4(w[4], w[5], w[6], w[7]));
    st_stream(m4, make_float4(m[0], m[1], m[2], m[3]));
    st_stream(m4 + 1, make_float4(m[4], m[5], m[6], m[7]));
    st_stream(v4, make_float4(v[0], v[1], v[2], v[3]));
    st_stream(v4 + 1, make_float4(v[4], v[5], v[6], v[7]));
}

template <class Src>
__device__ __forceinline__ void step_compute_store(const Src &src, int64_t vec, const VecData<Src> &d, float inv,
                                                   float c, float bc1, float bc2, const StepK &k, const State &st)
{
    float w[kVec], m[kVec], v[kVec];
    step_compute(src, d, inv, c, bc1, bc2, k, w, m, v);
    store_state(vec, st, w, m, v);
    st_stream(reinterpret_cast<uint4 *>(st.p) + vec,
              make_uint4(pack_bf16x2(w[0], w[1]), pack_bf16x2(w[2], w[3]), pack_bf16x2(w[4], w[5]),
                         pack_bf16x2(w[6], w[7])));
}

// ------------------------------------------------------------------ MXFP8 parameters
//
// The updated master weights stored as MXFP8 instead of bf16 (Zero From
// Scratch, item 14: MXFP8 takes its share off stored state). Same block rule
// as the gradient encoder, on fp32 values: amax over the |w| bit patterns,
// E8M0 byte = max(E - 8, 0) from the amax exponent field E, codes =
// E4M3(w * 2^-e) with round-to-nearest-even and saturation (the scaling is
// exact whenever the code is not zero); a block with inf or NaN gets scale
// 0xFF and codes 0x7F.

__device__ __forceinline__ uint32_t mx_block_byte(uint32_t amax_bits, bool &bad)
{
    bad = amax_bits >= 0x7f800000u;
    const uint32_t ex = amax_bits >> 23;
    return bad ? 0xffu : (ex > 8u ? ex - 8u : 0u);
}

__device__ __forceinline__ float mx_to_unit(uint32_t sbyte, bool bad)
{
    return __uint_as_float((254u - (bad ? 0u : sbyte)) << 23);  // 2^-e
}

// Four consecutive lanes hold one 32-element block (8 values each): combine
// their amax, then write this lane's 8 codes and (first lane) the scale.
__device__ __forceinline__ void mx_store_group(int64_t vec, bool active, const float (&w)[kVec], const State &st)
{
    uint32_t amax = 0u;
    if (active) {
#pragma unroll
        for (int j = 0; j < kVec; ++j) amax = max(amax, __float_as_uint(w[j]) & 0x7fffffffu);
    }
    amax = max(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = max(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    bool bad;
    const uint32_t sbyte = mx_block_byte(amax, bad);
    const float to_unit = mx_to_unit(sbyte, bad);
    if (!active) return;
    uint32_t pairs[4];
#pragma unroll
    for (int q = 0; q < 4; ++q)
        pairs[q] = bad ? 0x7f7fu : f32x2_to_e4m3x2(__fmul_rn(w[2 * q], to_unit), __fmul_rn(w[2 * q + 1], to_unit));
    __stcs(reinterpret_cast<uint2 *>(st.pcodes) + vec, make_uint2(pairs[0] | (pairs[1] << 16), pairs[2] | (pairs[3] << 16)));
    if ((threadIdx.x & 3) == 0) st.pscales[vec >> 2] = uint8_t(sbyte);
}

// The elements past the last whole 32-block, with MX parameters: update
// them one by one, then encode the short block (missing elements count as
// zero in its amax). One thread.
template <class Src>
__device__ __forceinline__ void step_tail_mx(const Src &src, int64_t n, float inv, float c, float bc1, float bc2,
                                             const StepK &k, const State &st)
{
    const int64_t lo = (n / 32) * 32;
    if (lo == n) return;
    uint32_t amax = 0u;
    for (int64_t i = lo; i < n; ++i) {
        float w = st.w[i], m = st.m[i], v = st.v[i];
        adamw(__fmul_rn(src.sum1(i), inv), c, bc1, bc2, k, w, m, v);
        st.w[i] = w;
        st.m[i] = m;
        st.v[i] = v;
        amax = max(amax, __float_as_uint(w) & 0x7fffffffu);
    }
    bool bad;
    const uint32_t sbyte = mx_block_byte(amax, bad);
    const float to_unit = mx_to_unit(sbyte, bad);
    for (int64_t i = lo; i < n; ++i)
        st.pcodes[i] = bad ? uint8_t(0x7f) : uint8_t(f32x2_to_e4m3x2(__fmul_rn(st.w[i], to_unit), 0.0f));
    st.pscales[lo / 32] = uint8_t(sbyte);
}

template <class Src>
__device__ __forceinline__ void step_tail(const Src &src, int64_t n, float inv, float c, float bc1, float bc2,
                                          const StepK &k, const State &st)
{
    for (int64_t i = (n / kVec) * kVec; i < n; ++i) {
        float w = st.w[i], m = st.m[i], v = st.v[i];
        adamw(__fmul_rn(src.sum1(i), inv), c, bc1, bc2, k, w, m, v);
        st.w[i] = w;
        st.m[i] = m;
        st.v[i] = v;
        st.p[i] = __bfloat16_as_ushort(__float2bfloat16_rn(w));
    }
}

// One warp's share of the fused step pass, split dynamically. The vectors
// form chunks of 32 * U (U per lane, lane-consecutive); chunk q + 8j belongs
// to counter q (the warp's index in its block). A warp's first chunk is fixed
// (j = its block index, so the first wave covers the same vectors a
// grid-stride split would), the following ones come from its counter
// (j = grid + the counter's next value), fetched while the current chunk's
// loads are in flight. Warps whose loads return sooner take more chunks, so
// the launch ends together: with a fixed grid-stride split the blocks of one
// launch finished up to 10 us apart at N = 2^24 (GB300, one launch about
// 95 us), as some SMs get their memory traffic served sooner than others.
// Every element gets the same arithmetic either way, so the results are
// bit-identical to the fixed split. Indices are mirrored when ZG_STEP_REVERSE
// walks from the end. True when the warp stored anything.
template <class Src>
__device__ __forceinline__ bool step_chunk_loop(const Src &src, int64_t n, float inv, float c, float bc1, float bc2,
                                                const StepK &k, const State &st)
{
    constexpr int U = StepUnroll<Src>::value;
    constexpr int64_t kChunk = 32 * U;
    static_assert(kStepThreads / 32 == kWorkLanes, "one counter per warp of a block");
    const int64_t nvec = n / kVec;
    const int64_t nchunk = (nvec + kChunk - 1) / kChunk;
    const int lane = threadIdx.x & 31;
    const int q = threadIdx.x >> 5;
    unsigned long long *ctr = st.work + kStepCtr + q * kWorkStride;
    int64_t ch = q + int64_t(kWorkLanes) * blockIdx.x;
    bool any = false;
#pragma unroll 1
    while (ch < nchunk) {  // warp-uniform
        unsigned long long next = 0ull;
        if (lane == 0) next = atomicAdd(ctr, 1ull);
        VecData<Src> d[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t vv = ch * kChunk + u * 32 + lane;
            if (vv < nvec) step_load(src, ZG_STEP_REVERSE ? nvec - 1 - vv : vv, st, d[u]);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t vv = ch * kChunk + u * 32 + lane;
            if (vv < nvec)
                step_compute_store(src, ZG_STEP_REVERSE ? nvec - 1 - vv : vv, d[u], inv, c, bc1, bc2, k, st);
        }
        any = true;
        next = __shfl_sync(0xffffffffu, next, 0);
        ch = q + int64_t(kWorkLanes) * (int64_t(gridDim.x) + int64_t(next));
    }
    return any;
}

// Fused reduce-scatter + unscale + clip + AdamW + bf16 all-gather, one pass,
// plain 128-bit loads and stores over 8-element vectors in warp chunks.
template <class Src, bool kMxOut = false>
__global__ void __launch_bounds__(kStepThreads, StepMinBlocks<Src>::value)
    step_kernel(Src src, int64_t n, float inv, StepK k, State st, Scalars *sc)
{
    // Launched as a dependent of the norm pass: warm L2 with this thread's
    // first vector (inputs the norm pass does not write), then wait for the
    // norm pass's decision before reading it.
    {
        const int64_t nv = kMxOut ? (n / 32) * 4 : n / kVec;  // vectors the main loop walks
        int64_t v0 = int64_t(blockIdx.x) * kStepThreads + threadIdx.x;
        if (ZG_STEP_REVERSE) v0 = nv - 1 - v0;
        if (v0 >= 0 && v0 < nv) {
            src.prefetch(v0);
            prefetch_l2(st.w + v0 * kVec);
            prefetch_l2(st.m + v0 * kVec);
            prefetch_l2(st.v + v0 * kVec);
        }
    }
    pdl_wait();
    pdl_trigger();
    float c, bc1, bc2;
    const int skip = step_prologue(sc, c, bc1, bc2);
    if (skip == 0 && kMxOut) {
        // whole 32-blocks in warp chunks of 32 vectors (one per lane), handed
        // out as in step_chunk_loop, so four neighbouring lanes share a block.
        // Walked from the end like the plain loop: mirroring the index keeps
        // each four-lane group on one whole block (nvec and the chunk starts
        // are multiples of 4), only in reverse lane order.
        const int64_t nvec = (n / 32) * 4;
        const int64_t nchunk = (nvec + 31) / 32;
        const int lane = threadIdx.x & 31;
        const int q = threadIdx.x >> 5;
        unsigned long long *ctr = st.work + kStepCtr + q * kWorkStride;
        int64_t ch = q + int64_t(kWorkLanes) * blockIdx.x;
#pragma unroll 1
        while (ch < nchunk) {  // warp-uniform
            unsigned long long next = 0ull;
            if (lane == 0) next = atomicAdd(ctr, 1ull);
            const int64_t base = ch * 32;
            const bool active = base + lane < nvec;
            const int64_t v = ZG_STEP_REVERSE ? nvec - 1 - (base + lane) : base + lane;
            float w[kVec] = {}, m[kVec], vv[kVec];
            if (active) {
                VecData<Src> d;
                step_load(src, v, st, d);
                step_compute(src, d, inv, c, bc1, bc2, k, w, m, vv);
                store_state(v, st, w, m, vv);
            }
            mx_store_group(v, active, w, st);
            next = __shfl_sync(0xffffffffu, next, 0);
            ch = q + int64_t(kWorkLanes) * (int64_t(gridDim.x) + int64_t(next));
        }
        if (blockIdx.x == 0 && threadIdx.x == 0) step_tail_mx(src, n, inv, c, bc1, bc2, k, st);
    } else if (skip == 0) {
        step_chunk_loop(src, n, inv, c, bc1, bc2, k, st);
        if (blockIdx.x == 0 && threadIdx.x == 0) step_tail(src, n, inv, c, bc1, bc2, k, st);
    }
    step_epilogue(sc, skip, st.work);
}

// ------------------------------------------------------------------ launch

#ifndef ZG_PDL
#define ZG_PDL 1
#endif

// Launch with programmatic stream serialisation, so the kernel's blocks can
// start while the previous kernel on the stream finishes (each kernel waits
// with pdl_wait() before touching that kernel's results).
template <class... Params, class... Args>
cudaError_t launch_dependent(void (*kernel)(Params...), int blocks, int threads, size_t smem, cudaStream_t st,
                             Args &&...args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(blocks);
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = ZG_PDL;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// ------------------------------------------------------------------ rank dispatch

template <class F>
cudaError_t with_ranks(int p, F &&f)
{
    switch (p) {
#define ZG_CASE(P) \
    case P: return f(std::integral_constant<int, P>{});
        ZG_CASE(1) ZG_CASE(2) ZG_CASE(3) ZG_CASE(4) ZG_CASE(5) ZG_CASE(6) ZG_CASE(7) ZG_CASE(8)
        ZG_CASE(9) ZG_CASE(10) ZG_CASE(11) ZG_CASE(12) ZG_CASE(13) ZG_CASE(14) ZG_CASE(15) ZG_CASE(16)
#undef ZG_CASE
    }
    return cudaErrorInvalidValue;
}

}  // namespace zg

// ------------------------------------------------------------------ TMA-staged step pass
//
// The same fused step, with the operands of each tile (4096 elements up to
// P = 4, 2048 from P = 5) staged
// in shared memory by 1-D bulk asynchronous copies (cp.async.bulk, global to
// this CTA's shared memory, completion counted in bytes on an mbarrier): P
// bf16 gradient slices and the fp32 w, m, v. The CTA is warp-specialised:
// one producer warp walks the CTA's tiles through a ring of `stages`
// buffers, and the consumer warps (8 elements per thread per tile) read a
// buffer into registers, release it and compute. Each buffer has a "full"
// barrier (the producer's expect_tx arrival plus the copied bytes) and an
// "empty" barrier (one arrival per consumer warp), so no block-wide barrier
// sits in the tile loop and the producer refills a buffer as soon as the
// last warp has read it. Results go straight from registers to HBM with
// 128-bit streaming stores.
//
// Every wait is bounded (`wait_limit` polls) and gives up early once another
// thread of the CTA has recorded a timeout. A wait that runs out records the
// timeout, the CTA waits (bounded again) for the copies it already issued,
// skips the rest of its work and returns; the step is then not committed.

namespace zg {
namespace tma {

// Elements per tile, by rank count: up to P = 4 a tile holds few gradient
// bytes, so tiles are 4096 elements (sixteen consumer warps, two buffers);
// from P = 5 on, 2048 elements (eight consumer warps, three buffers; two at
// P = 16). Measured on GB300, each choice is the faster one where it is used.
constexpr int kTileSmallP = 4096;
constexpr int kTileLargeP = 2048;
template <int P>
struct TileFor {
    static constexpr int value = P <= 4 ? kTileSmallP : kTileLargeP;
};
#ifndef ZG_TMA_REVERSE
#define ZG_TMA_REVERSE ZG_STEP_REVERSE
#endif
constexpr long long kDrainLimit = 1LL << 22;

__device__ __forceinline__ uint32_t smem_addr(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

// Make the barrier initialisation visible to the bulk-copy (async) proxy.
__device__ __forceinline__ void fence_barrier_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

// Bounded wait: true when the phase completed within `limit` polls. A
// limit of 0 gives up without polling.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, long long limit)
{
    for (long long i = 0; i < limit; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}

struct Layout {
    int p;
    uint32_t grad_bytes;   // per rank per full tile
    uint32_t stage_bytes;  // P gradient slices + w, m, v
    __host__ __device__ static Layout of(int p, int tile)
    {
        Layout l;
        l.p = p;
        l.grad_bytes = uint32_t(tile) * 2;
        l.stage_bytes = p * l.grad_bytes + 3 * uint32_t(tile) * 4;
        return l;
    }
};

// Threads of a CTA for a tile size: one consumer thread per 8 elements, plus
// the producer warp.
constexpr int ws_threads(int tile) { return tile / kVec + 32; }
#ifndef ZG_TMA_WS_MINB
#define ZG_TMA_WS_MINB 1
#endif

__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// Bounded wait that also gives up once another thread of the CTA has
// recorded a timeout (checked every 256 polls).
__device__ __forceinline__ bool mbar_wait_or_abort(uint64_t *bar, uint32_t parity, long long limit,
                                                   const volatile int *abort)
{
    for (long long i = 0; i < limit; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 255) == 255 && *abort) return false;
    }
    return false;
}

template <int P, int TILE>
__global__ void __launch_bounds__(ws_threads(TILE), ZG_TMA_WS_MINB)
    step_kernel_tma(Bf16Src<P> src, int64_t n, float inv, StepK k, State st, Scalars *sc, int stages,
                    long long wait_limit)
{
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ __align__(8) uint64_t full[8];
    __shared__ __align__(8) uint64_t empty[8];
    __shared__ int s_timeout;
    __shared__ int s_stored;  // some consumer of this CTA has written results
    __shared__ long long s_issued;
    __shared__ long long s_tile[8];  // the tile each buffer holds, -1 after the last

    pdl_wait();
    pdl_trigger();
    float c, bc1, bc2;
    int skip = step_prologue(sc, c, bc1, bc2);
    constexpr int kTile = TILE;
    constexpr int kConsumers = TILE / kVec;  // 8 elements per consumer thread per tile
    const Layout lay = Layout::of(P, TILE);
    const int64_t nvec = n / kVec;
    const int64_t covered = nvec * kVec;  // elements the tiles cover; the rest is the scalar tail
    const int64_t ntiles = (covered + kTile - 1) / kTile;

    if (threadIdx.x == 0) {
        s_timeout = 0;
        s_stored = 0;
        s_issued = 0;
        for (int s = 0; s < stages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kConsumers / 32);
        }
        fence_barrier_init();
    }
    __syncthreads();

    auto stage_ptr = [&](int s) { return smem + size_t(s) * lay.stage_bytes; };
    // first element of tile t; the tiles are walked from the end, like the
    // plain kernel's vectors, where the norm pass finished
    auto tile_start = [&](int64_t t) { return (ZG_TMA_REVERSE ? ntiles - 1 - t : t) * kTile; };
    const volatile int *abort = &s_timeout;
    const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;

    if (skip == 0 && warp == kConsumers / 32) {
        // producer: one lane issues every copy of this CTA's tiles in order.
        // The CTA's first tile is its index; each further one comes from a
        // counter (grid + its next value), so CTAs whose copies land sooner
        // take more tiles and the launch ends together. After the last tile
        // the next buffer gets the index -1 and a plain arrival.
        if (lane == 0) {
            int64_t j = 0;
            int64_t t = blockIdx.x;
            for (;; ++j) {
                const int s = int(j % stages);
                if (j >= stages &&
                    !mbar_wait_or_abort(&empty[s], uint32_t(((j / stages) - 1) & 1), wait_limit, abort)) {
                    atomicExch(&s_timeout, 1);
                    break;
                }
                if (t >= ntiles) {
                    s_tile[s] = -1;
                    mbar_arrive(&full[s]);
                    break;
                }
                s_tile[s] = t;
                const int64_t t0 = tile_start(t);
                const int64_t len = covered - t0 < kTile ? covered - t0 : kTile;
                unsigned char *buf = stage_ptr(s);
                const uint32_t gb = uint32_t(len * 2), fb = uint32_t(len * 4);
                mbar_expect_tx(&full[s], P * gb + 3 * fb);
#pragma unroll
                for (int r = 0; r < P; ++r) bulk_g2s(buf + r * lay.grad_bytes, src.g[r] + t0, gb, &full[s]);
                float *f = reinterpret_cast<float *>(buf + P * lay.grad_bytes);
                bulk_g2s(f, st.w + t0, fb, &full[s]);
                bulk_g2s(f + kTile, st.m + t0, fb, &full[s]);
                bulk_g2s(f + 2 * kTile, st.v + t0, fb, &full[s]);
                t = int64_t(gridDim.x) + int64_t(atomicAdd(st.work + kStepCtr, 1ull));
            }
            s_issued = j;  // buffers with copies in flight or landed (not the -1 one)
        }
    } else if (skip == 0) {
        for (int64_t j = 0;; ++j) {
            const int s = int(j % stages);
            // one decision per warp, so no lane leaves while the others sync
            const bool ok = __all_sync(0xffffffffu, mbar_wait_or_abort(&full[s], uint32_t((j / stages) & 1),
                                                                        wait_limit, abort));
            if (!ok) {
                if (lane == 0) atomicExch(&s_timeout, 1);
                break;
            }
            const long long tile = *reinterpret_cast<volatile long long *>(&s_tile[s]);
            if (tile < 0) break;  // the producer has no more tiles
            const int64_t t0 = tile_start(tile);
            const int64_t len = covered - t0 < kTile ? covered - t0 : kTile;
            const int e = threadIdx.x * kVec;
            const bool active = e < len;
            float gh[kVec], w[kVec], m[kVec], v[kVec];
            if (active) {
                const unsigned char *buf = stage_ptr(s);
#pragma unroll
                for (int q = 0; q < kVec; ++q) gh[q] = 0.0f;
#pragma unroll
                for (int r = 0; r < P; ++r) {
                    const uint4 x = *reinterpret_cast<const uint4 *>(buf + r * lay.grad_bytes + e * 2);
                    const uint32_t w4[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        gh[2 * q] = __fadd_rn(gh[2 * q], bf16_lo(w4[q]));
                        gh[2 * q + 1] = __fadd_rn(gh[2 * q + 1], bf16_hi(w4[q]));
                    }
                }
                const float *f = reinterpret_cast<const float *>(buf + P * lay.grad_bytes);
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const float4 a = *reinterpret_cast<const float4 *>(f + e + 4 * h);
                    const float4 b = *reinterpret_cast<const float4 *>(f + kTile + e + 4 * h);
                    const float4 d = *reinterpret_cast<const float4 *>(f + 2 * kTile + e + 4 * h);
                    w[4 * h] = a.x, w[4 * h + 1] = a.y, w[4 * h + 2] = a.z, w[4 * h + 3] = a.w;
                    m[4 * h] = b.x, m[4 * h + 1] = b.y, m[4 * h + 2] = b.z, m[4 * h + 3] = b.w;
                    v[4 * h] = d.x, v[4 * h + 1] = d.y, v[4 * h + 2] = d.z, v[4 * h + 3] = d.w;
                }
            }
            // the warp's reads of buffer s are done: release it before computing
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
            if (__any_sync(0xffffffffu, active) && lane == 0) s_stored = 1;
            if (active) {
#pragma unroll
                for (int q = 0; q < kVec; ++q) adamw(__fmul_rn(gh[q], inv), c, bc1, bc2, k, w[q], m[q], v[q]);
                const int64_t gi = t0 + e;
                float4 *w4 = reinterpret_cast<float4 *>(st.w + gi);
                float4 *m4 = reinterpret_cast<float4 *>(st.m + gi);
                float4 *v4 = reinterpret_cast<float4 *>(st.v + gi);
                st_stream(w4, make_float4(w[0], w[1], w[2], w[3]));
                st_stream(w4 + 1, make_float4(w[4], w[5], w[6], w[7]));
                st_stream(m4, make_float4(m[0], m[1], m[2], m[3]));
                st_stream(m4 + 1, make_float4(m[4], m[5], m[6], m[7]));
                st_stream(v4, make_float4(v[0], v[1], v[2], v[3]));
                st_stream(v4 + 1, make_float4(v[4], v[5], v[6], v[7]));
                st_stream(reinterpret_cast<uint4 *>(st.p + gi),
                          make_uint4(pack_bf16x2(w[0], w[1]), pack_bf16x2(w[2], w[3]), pack_bf16x2(w[4], w[5]),
                                     pack_bf16x2(w[6], w[7])));
            }
        }
    }
    __syncthreads();

    if (s_timeout) {
        // Drain: wait (bounded) for the copies still in flight, the last
        // `stages` tiles issued at most, so no bulk copy lands after the CTA
        // is gone.
        if (threadIdx.x == 0) {
            const int64_t issued = s_issued;
            for (int64_t j = issued > stages ? issued - stages : 0; j < issued; ++j)
                mbar_wait(&full[int(j % stages)], uint32_t((j / stages) & 1), kDrainLimit);
            sc->status = kStatusTimeout;
            atomicAdd(&sc->step_faults, 1u);
        }
        skip = 3;
    } else if (skip == 0 && blockIdx.x == 0 && threadIdx.x == 0) {
        step_tail(src, n, inv, c, bc1, bc2, k, st);
        if (n % kVec) s_stored = 1;
    }
    __syncthreads();
    // commit (or not) exactly like the plain kernel; a timeout leaves the
    // step uncommitted and the norm consumed. A timeout in any CTA after some
    // CTA has stored results leaves the state half updated: that is reported
    // as its own status, since the step cannot simply be run again.
    if (threadIdx.x == 0) {
        if (s_stored) atomicOr(&sc->step_faults, kFaultStored);
        __threadfence();
        const unsigned int ticket = atomicAdd(&sc->step_ticket, 1u);
        if (ticket == gridDim.x - 1) {
            const unsigned int faults = atomicAdd(&sc->step_faults, 0u);
            const int any_timeout = (faults & ~kFaultStored) != 0u;
            sc->step_faults = 0u;
            if (any_timeout && (faults & kFaultStored)) sc->status = kStatusPartial;
            if (skip == 2) {
                sc->status = kStatusStaleNorm;
            } else {
                if (skip == 0 && !any_timeout) {
                    sc->t = sc->t_next;
                    sc->b1p = sc->b1p_next;
                    sc->b2p = sc->b2p_next;
                }
                sc->step_gen = sc->norm_gen;
            }
            st.work[kStepCtr] = 0ull;  // every producer has taken its last tile
            sc->step_ticket = 0u;
        }
    }
}

}  // namespace tma
}  // namespace zg
