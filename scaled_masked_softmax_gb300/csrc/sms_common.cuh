// Device helpers shared by the libsms kernels: dtype traits, 16-byte vector
// I/O with cache hints, group reductions, exp2, and bounded mbarrier / bulk-copy
// (TMA) primitives written as inline PTX for sm_103a.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "sms.h"
#include "sms_fastdiv.h"

namespace sms {

constexpr float kLog2e = 1.4426950408889634f;
__device__ __forceinline__ float neg_inf() { return __int_as_float(0xff800000); }

// --------------------------------------------------------------- dtypes ---
// Every kernel moves rows as 16-byte vectors: 4 fp32 or 8 fp16/bf16 elements.
template <typename T> struct Dt;
template <> struct Dt<float> { static constexpr int VEC = 4; };
template <> struct Dt<__half> { static constexpr int VEC = 8; };
template <> struct Dt<__nv_bfloat16> { static constexpr int VEC = 8; };

template <typename T> __device__ __forceinline__ float to_f32(T v);
template <> __device__ __forceinline__ float to_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ float to_f32<__half>(__half v) { return __half2float(v); }
template <> __device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 v) { return __bfloat162float(v); }

// fp32 -> storage type, round to nearest even.
template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ __half from_f32<__half>(float v) { return __float2half_rn(v); }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) { return __float2bfloat16_rn(v); }

// Unpack one 16-byte vector into VEC floats / pack VEC floats into one vector.
template <typename T> __device__ __forceinline__ void unpack(const uint4 &v, float *f);
template <> __device__ __forceinline__ void unpack<float>(const uint4 &v, float *f)
{
    f[0] = __uint_as_float(v.x); f[1] = __uint_as_float(v.y);
    f[2] = __uint_as_float(v.z); f[3] = __uint_as_float(v.w);
}
template <> __device__ __forceinline__ void unpack<__half>(const uint4 &v, float *f)
{
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        __half2 h = *reinterpret_cast<const __half2 *>(&w[i]);
        float2 t = __half22float2(h);
        f[2 * i] = t.x; f[2 * i + 1] = t.y;
    }
}
template <> __device__ __forceinline__ void unpack<__nv_bfloat16>(const uint4 &v, float *f)
{
    // bf16 is the high half of an fp32: widening is a 16-bit shift
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}

template <typename T> __device__ __forceinline__ uint4 pack(const float *f);
template <> __device__ __forceinline__ uint4 pack<float>(const float *f)
{
    return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]), __float_as_uint(f[3]));
}
template <> __device__ __forceinline__ uint4 pack<__half>(const float *f)
{
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        __half2 h = __floats2half2_rn(f[2 * i], f[2 * i + 1]);
        w[i] = *reinterpret_cast<uint32_t *>(&h);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}
template <> __device__ __forceinline__ uint4 pack<__nv_bfloat16>(const float *f)
{
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        __nv_bfloat162 h = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
        w[i] = *reinterpret_cast<uint32_t *>(&h);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// Elements S .. S+VEC-1 of the 2*VEC elements held by two consecutive 16-byte
// vectors (lo, hi): realigns a row that starts mid-vector relative to another.
template <int VEC, int S> __device__ __forceinline__ uint4 window_fixed(const uint4 &lo, const uint4 &hi)
{
    const uint32_t w[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
    uint32_t o[4];
    if constexpr (VEC == 4) {  // 32-bit elements: a shift of S words
#pragma unroll
        for (int i = 0; i < 4; ++i) o[i] = w[(i + S) & 7];
    } else {  // 16-bit elements: S/2 words, then half a word when S is odd
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t a = w[(i + S / 2) & 7], b = w[(i + S / 2 + 1) & 7];
            o[i] = (S & 1) ? __funnelshift_r(a, b, 16) : a;
        }
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

template <int VEC> __device__ __forceinline__ uint4 window(const uint4 &lo, const uint4 &hi, int s)
{
    switch (s) {
    case 0: return lo;
    case 1: return window_fixed<VEC, 1>(lo, hi);
    case 2: return window_fixed<VEC, 2>(lo, hi);
    case 3: return window_fixed<VEC, 3>(lo, hi);
    case 4: return window_fixed<VEC, 4 % VEC>(lo, hi);
    case 5: return window_fixed<VEC, 5 % VEC>(lo, hi);
    case 6: return window_fixed<VEC, 6 % VEC>(lo, hi);
    default: return window_fixed<VEC, 7 % VEC>(lo, hi);
    }
}

// ------------------------------------------------------ global memory I/O ---
// Scores and gradients are read exactly once: stream them past L1 and mark
// them first to leave L2.  The broadcast mask is re-read by every head of a
// batch, so it keeps the default L2 priority.
__device__ __forceinline__ uint4 ld_stream(const void *p) { return __ldcs(reinterpret_cast<const uint4 *>(p)); }
__device__ __forceinline__ uint4 ld_keep(const void *p) { return __ldg(reinterpret_cast<const uint4 *>(p)); }
__device__ __forceinline__ void st_stream(void *p, const uint4 &v) { __stcs(reinterpret_cast<uint4 *>(p), v); }

// ---------------------------------------------------------- mask elements ---
// A mask is additive (element type M == T, added to x*scale) or boolean (M ==
// uint8_t, one byte per element, nonzero = the key is masked and its score is
// -inf).  MaskIO<T, M> moves the mask elements under one 16-byte x vector
// (VEC elements): one 16-byte load for an additive mask, VEC bytes in .x (and
// .y) for a boolean one.  A boolean element becomes the additive value 0 or
// -inf, so x*scale + m is computed by the same instruction either way and a
// boolean mask gives bit for bit the result of its additive -inf twin.
template <typename T, typename M> struct MaskIO;

template <typename T> struct MaskIO<T, T> {
    static constexpr int VEC = Dt<T>::VEC;
    static __device__ __forceinline__ uint4 ld(const T *p) { return ld_keep(p); }
    static __device__ __forceinline__ void unpack_m(const uint4 &v, float *f) { unpack<T>(v, f); }
    template <int S> static __device__ __forceinline__ uint4 win(const uint4 &lo, const uint4 &hi)
    {
        return window_fixed<VEC, S>(lo, hi);
    }
    static __device__ __forceinline__ uint4 win_rt(const uint4 &lo, const uint4 &hi, int s)
    {
        return window<VEC>(lo, hi, s);
    }
    static __device__ __forceinline__ float elem(const T *p) { return to_f32<T>(*p); }
};

template <typename T> struct MaskIO<T, uint8_t> {
    static constexpr int VEC = Dt<T>::VEC;
    static __device__ __forceinline__ uint4 ld(const uint8_t *p)
    {
        if constexpr (VEC == 4) {
            return make_uint4(__ldg(reinterpret_cast<const unsigned int *>(p)), 0u, 0u, 0u);
        } else {
            const uint2 v = __ldg(reinterpret_cast<const uint2 *>(p));
            return make_uint4(v.x, v.y, 0u, 0u);
        }
    }
    static __device__ __forceinline__ void unpack_m(const uint4 &v, float *f)
    {
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
            const uint32_t w = e < 4 ? v.x : v.y;
            f[e] = ((w >> (8 * (e & 3))) & 0xffu) ? neg_inf() : 0.f;
        }
    }
    // Bytes S .. S+VEC-1 of the 2*VEC bytes held by two consecutive VEC-byte
    // groups (lo, hi).
    template <int S> static __device__ __forceinline__ uint4 win(const uint4 &lo, const uint4 &hi)
    {
        if constexpr (S == 0) return lo;
        if constexpr (VEC == 4) {
            return make_uint4(__funnelshift_r(lo.x, hi.x, 8 * S), 0u, 0u, 0u);
        } else {
            const uint32_t w[4] = {lo.x, lo.y, hi.x, hi.y};
            constexpr int q = S / 4, b = 8 * (S % 4);
            return make_uint4(__funnelshift_r(w[q], w[q + 1], b), __funnelshift_r(w[q + 1], w[q + 2], b), 0u, 0u);
        }
    }
    static __device__ __forceinline__ uint4 win_rt(const uint4 &lo, const uint4 &hi, int s)
    {
        switch (s) {
        case 0: return lo;
        case 1: return win<1>(lo, hi);
        case 2: return win<2>(lo, hi);
        case 3: return win<3>(lo, hi);
        case 4: return win<4 % VEC>(lo, hi);
        case 5: return win<5 % VEC>(lo, hi);
        case 6: return win<6 % VEC>(lo, hi);
        default: return win<7 % VEC>(lo, hi);
        }
    }
    static __device__ __forceinline__ float elem(const uint8_t *p) { return *p ? neg_inf() : 0.f; }
};
// ------------------------------------------------------------ arithmetic ---
// 2^x on the special-function unit (PTX ex2.approx, subnormal results flushed
// to zero; 2^-inf = +0).
__device__ __forceinline__ float ex2(float x)
{
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

// Reductions over aligned groups of G lanes (G a power of two, <= 32).
template <int G> __device__ __forceinline__ float group_max(float v)
{
#pragma unroll
    for (int o = G / 2; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
template <int G> __device__ __forceinline__ float group_sum(float v)
{
#pragma unroll
    for (int o = G / 2; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// ------------------------------------------- mbarrier + bulk async copies ---
// Every wait is bounded by wall time (globaltimer); on expiry the caller gets
// `false` and must record the failure and unwind without touching the stage.
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s

__device__ __forceinline__ uint64_t global_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" :: "r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}"
                 :: "r"(smem_u32(bar)), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
    return ok != 0;
}

// Wait for the phase with the given parity to complete; false on timeout or
// when *abort becomes nonzero (another thread already gave up).
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity, volatile int *abort,
                                                  uint64_t limit_ns = kWaitLimitNs)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort) return false;
        if (global_ns() - t0 > limit_ns) return false;
    }
}

// 1-D bulk copy global -> shared (the TMA unit), completion signalled on `bar`
// as transaction bytes.  dst, src and bytes must be multiples of 16.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;"
        :: "r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy) : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ uint64_t policy_evict_last()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ uint64_t policy_evict_normal()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// Named barrier over the first `threads` threads of the CTA (id != 0).
__device__ __forceinline__ void named_sync(int id, int threads)
{
    asm volatile("bar.sync %0, %1;" :: "r"(id), "r"(threads) : "memory");
}

// ------------------------------------------------------------ row index ---
// Row r of the [rows, cols] view is query position q of head h of batch b:
// r = (b * heads + h) * cols + q.
__device__ __forceinline__ void split_row(int64_t r, int64_t cols, int64_t heads, const FastDiv &dc,
                                          const FastDiv &dh, int64_t &q, int64_t &h, int64_t &b)
{
    if (r <= 0xffffffffll) {
        const uint32_t rr = (uint32_t)r;
        const uint32_t rc = dc.div(rr);
        q = rr - rc * (uint32_t)cols;
        const uint32_t bb = dh.div(rc);
        h = rc - bb * (uint32_t)heads;
        b = bb;
    } else {
        const int64_t rc = r / cols;
        q = r - rc * cols;
        b = rc / heads;
        h = rc - b * heads;
    }
}

__device__ __forceinline__ int64_t row_q(int64_t r, int64_t cols, const FastDiv &dc)
{
    if (r <= 0xffffffffll) {
        const uint32_t rr = (uint32_t)r;
        return rr - dc.div(rr) * (uint32_t)cols;
    }
    return r % cols;
}

// Elements a row reads: `limit` (q + 1 under the causal flag, else cols),
// further cut to the first lengths[b] keys when per-batch key lengths are
// given (a length outside [0, cols] is clamped).  0 is a live row with no
// kept key: its output is all zero.
__device__ __forceinline__ int key_limit(const int32_t *lengths, int64_t b, int64_t cols, int limit)
{
    if (!lengths) return limit;
    const int L = min(max(__ldg(lengths + b), 0), (int)cols);
    return min(limit, L);
}

// Records the first failure code in the library's device error word (its
// address is passed to every kernel that waits on a barrier).
__device__ __forceinline__ void report_error(int *err, int code)
{
    if (err) atomicCAS(err, 0, code);
}

}  // namespace sms
