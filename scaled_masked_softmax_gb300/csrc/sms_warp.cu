// Register-resident row kernels: a group of G lanes (a whole warp for rows of
// 128+ elements, a part of one for shorter rows) owns one row, holds it in
// registers as NV 16-byte vectors per lane, and reduces with warp shuffles.
//
// Prior art: the warp-per-row kernel of the second article (pnsm.cn/news/1983787,
// §2.2 granularity table and §3.2 kernel) made three global passes over the row
// with four rows per block.  Here the row is read from HBM exactly once,
// kept in registers between the max, exp/sum and normalise steps, exp is
// evaluated once per element, and the causal positions j > q are never read.
//
// Element mapping.  Rows are walked in 16-byte vectors aligned to the tensor
// (not to the row): vector vi of a row covers row elements
// vi*VEC - xoff .. vi*VEC - xoff + VEC - 1 where xoff = (row*cols) mod VEC, so a
// row that starts mid-vector (cols not a multiple of VEC) still moves with
// 16-byte loads; the partial head and tail vectors are stored element-wise.
#include "sms_common.cuh"
#include "sms_internal.h"

namespace sms {
namespace {

constexpr int kThreads = 256;  // 8 warps per CTA

template <typename T, int G, int NV, bool ALIGNED>
__global__ void __launch_bounds__(kThreads) fwd_warp_kernel(const FwdArgs a)
{
    constexpr int VEC = Dt<T>::VEC;
    constexpr int RPW = 32 / G;  // rows per warp
    const int lane = threadIdx.x & 31;
    const int gl = lane & (G - 1);
    const int64_t row = ((int64_t)blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5)) * RPW + lane / G;
    const bool live = row < a.rows;
    const int64_t r = live ? row : a.rows - 1;  // dead lanes still join the shuffles
    const int64_t cols = a.cols;
    int64_t q = 0, h = 0, b = 0;
    if (a.causal || a.mask) split_row(r, cols, a.heads, a.dcols, a.dheads, q, h, b);
    const int limit = a.causal ? (int)(q + 1) : (int)cols;  // elements that are read
    const int64_t x0 = r * cols;
    const int xoff = ALIGNED ? 0 : (int)(x0 & (VEC - 1));
    const T *xs = reinterpret_cast<const T *>(a.x) + (x0 - xoff);

    const T *ms = nullptr;
    int64_t m0 = 0;
    bool mvec = ALIGNED;
    if (a.mask) {
        m0 = b * a.msb + h * a.msh + q * cols;
        ms = reinterpret_cast<const T *>(a.mask) + m0;
        if (!ALIGNED) mvec = ((m0 - xoff) & (VEC - 1)) == 0;
    }

    float s[NV][VEC];
    float mx = neg_inf();
#pragma unroll
    for (int k = 0; k < NV; ++k) {
        const int vi = k * G + gl;
        const int j0 = vi * VEC - xoff;
        float xv[VEC], mv[VEC];
#pragma unroll
        for (int e = 0; e < VEC; ++e) { xv[e] = 0.f; mv[e] = 0.f; }
        const bool any = j0 < limit;
        if (any) {
            const int64_t g = x0 - xoff + (int64_t)vi * VEC;
            if (ALIGNED || g + VEC <= a.x_total) {
                unpack<T>(ld_stream(xs + vi * VEC), xv);
            } else {
#pragma unroll
                for (int e = 0; e < VEC; ++e)
                    if (g + e < a.x_total) xv[e] = to_f32<T>(xs[vi * VEC + e]);
            }
            if (ms) {
                if (mvec && (ALIGNED || m0 + j0 + VEC <= a.mask_total)) {
                    unpack<T>(ld_keep(ms + j0), mv);
                } else {
#pragma unroll
                    for (int e = 0; e < VEC; ++e) {
                        const int j = j0 + e;
                        if (j >= 0 && j < limit) mv[e] = to_f32<T>(ms[j]);
                    }
                }
            }
        }
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
            const int j = j0 + e;
            const bool valid = any && j >= 0 && j < limit;
            s[k][e] = valid ? fmaf(xv[e], a.scale, mv[e]) : neg_inf();
            mx = fmaxf(mx, s[k][e]);
        }
    }

    mx = group_max<G>(mx);
    const float mref = (mx == neg_inf()) ? 0.f : mx;  // fully masked row: every term becomes 0
    float sum = 0.f;
#pragma unroll
    for (int k = 0; k < NV; ++k)
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
            const float t = ex2((s[k][e] - mref) * kLog2e);
            s[k][e] = t;
            sum += t;
        }
    sum = group_sum<G>(sum);
    const float inv = sum > 0.f ? __frcp_rn(sum) : 0.f;
    if (!live) return;

    T *ys = reinterpret_cast<T *>(a.y) + (x0 - xoff);
#pragma unroll
    for (int k = 0; k < NV; ++k) {
        const int vi = k * G + gl;
        const int j0 = vi * VEC - xoff;
        if (j0 >= cols) continue;
        float o[VEC];
#pragma unroll
        for (int e = 0; e < VEC; ++e) o[e] = s[k][e] * inv;
        if (ALIGNED || (j0 >= 0 && j0 + VEC <= cols)) {
            st_stream(ys + vi * VEC, pack<T>(o));
        } else {
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
                const int j = j0 + e;
                if (j >= 0 && j < cols) ys[vi * VEC + e] = from_f32<T>(o[e]);
            }
        }
    }
}

template <typename T, int G, int NV, bool ALIGNED>
__global__ void __launch_bounds__(kThreads) bwd_warp_kernel(const BwdArgs a)
{
    constexpr int VEC = Dt<T>::VEC;
    constexpr int RPW = 32 / G;
    const int lane = threadIdx.x & 31;
    const int gl = lane & (G - 1);
    const int64_t row = ((int64_t)blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5)) * RPW + lane / G;
    const bool live = row < a.rows;
    const int64_t r = live ? row : a.rows - 1;
    const int64_t cols = a.cols;
    const int limit = a.causal ? (int)(row_q(r, cols, a.dcols) + 1) : (int)cols;
    const int64_t x0 = r * cols;
    const int xoff = ALIGNED ? 0 : (int)(x0 & (VEC - 1));
    const T *ys = reinterpret_cast<const T *>(a.y) + (x0 - xoff);
    const T *gs = reinterpret_cast<const T *>(a.dy) + (x0 - xoff);

    float yv[NV][VEC], gv[NV][VEC];
    float dot = 0.f;
#pragma unroll
    for (int k = 0; k < NV; ++k) {
        const int vi = k * G + gl;
        const int j0 = vi * VEC - xoff;
#pragma unroll
        for (int e = 0; e < VEC; ++e) { yv[k][e] = 0.f; gv[k][e] = 0.f; }
        if (j0 < limit) {
            const int64_t g = x0 - xoff + (int64_t)vi * VEC;
            float tv[VEC], tg[VEC];
            if (ALIGNED || g + VEC <= a.total) {
                unpack<T>(ld_stream(ys + vi * VEC), tv);
                unpack<T>(ld_stream(gs + vi * VEC), tg);
            } else {
#pragma unroll
                for (int e = 0; e < VEC; ++e) {
                    const bool in = g + e < a.total;
                    tv[e] = in ? to_f32<T>(ys[vi * VEC + e]) : 0.f;
                    tg[e] = in ? to_f32<T>(gs[vi * VEC + e]) : 0.f;
                }
            }
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
                const int j = j0 + e;
                const bool valid = j >= 0 && j < limit;
                yv[k][e] = valid ? tv[e] : 0.f;
                gv[k][e] = valid ? tg[e] : 0.f;
                dot = fmaf(yv[k][e], gv[k][e], dot);
            }
        }
    }
    dot = group_sum<G>(dot);
    if (!live) return;

    T *dxs = reinterpret_cast<T *>(a.dx) + (x0 - xoff);
#pragma unroll
    for (int k = 0; k < NV; ++k) {
        const int vi = k * G + gl;
        const int j0 = vi * VEC - xoff;
        if (j0 >= cols) continue;
        float o[VEC];
#pragma unroll
        for (int e = 0; e < VEC; ++e)  // y == 0 (masked) gives exactly +0
            o[e] = (yv[k][e] == 0.f) ? 0.f : (gv[k][e] - dot) * yv[k][e] * a.scale;
        if (ALIGNED || (j0 >= 0 && j0 + VEC <= cols)) {
            st_stream(dxs + vi * VEC, pack<T>(o));
        } else {
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
                const int j = j0 + e;
                if (j >= 0 && j < cols) dxs[vi * VEC + e] = from_f32<T>(o[e]);
            }
        }
    }
}

template <typename T, int G, int NV, bool ALIGNED, bool BWD, typename Args>
cudaError_t launch_one(const Args &a, cudaStream_t st)
{
    constexpr int rows_per_cta = (kThreads / 32) * (32 / G);
    const int64_t blocks = (a.rows + rows_per_cta - 1) / rows_per_cta;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks);
    cfg.blockDim = dim3(kThreads);
    cfg.stream = st;
    if constexpr (BWD)
        return cudaLaunchKernelEx(&cfg, bwd_warp_kernel<T, G, NV, ALIGNED>, a);
    else
        return cudaLaunchKernelEx(&cfg, fwd_warp_kernel<T, G, NV, ALIGNED>, a);
}

// Lane-group / vectors-per-lane shapes, smallest first.  Capacity = G*NV
// vectors; a lane holds at most 64 fp32 values.
template <typename T, bool ALIGNED, bool BWD, typename Args>
cudaError_t launch_t(const Args &a, cudaStream_t st)
{
    constexpr int VEC = Dt<T>::VEC;
    const int64_t need = (a.cols + VEC - 1) / VEC + (ALIGNED ? 0 : 1);
#define SMS_TRY(G, NV) \
    if (need <= (G) * (NV)) return launch_one<T, G, NV, ALIGNED, BWD>(a, st);
    SMS_TRY(4, 1) SMS_TRY(8, 1) SMS_TRY(16, 1) SMS_TRY(32, 1) SMS_TRY(32, 2) SMS_TRY(32, 3) SMS_TRY(32, 4)
    SMS_TRY(32, 6) SMS_TRY(32, 8)
    if constexpr (VEC == 4) { SMS_TRY(32, 12) SMS_TRY(32, 16) }
#undef SMS_TRY
    return cudaErrorNotSupported;
}

template <bool BWD, typename Args>
cudaError_t dispatch(const Args &a, int dtype, bool aligned, cudaStream_t st)
{
    switch (dtype) {
    case kF32:
        return aligned ? launch_t<float, true, BWD>(a, st) : launch_t<float, false, BWD>(a, st);
    case kF16:
        return aligned ? launch_t<__half, true, BWD>(a, st) : launch_t<__half, false, BWD>(a, st);
    case kBF16:
        return aligned ? launch_t<__nv_bfloat16, true, BWD>(a, st) : launch_t<__nv_bfloat16, false, BWD>(a, st);
    default:
        return cudaErrorInvalidValue;
    }
}

}  // namespace

bool warp_fits(int64_t cols, int dtype, bool aligned)
{
    const int vec = vec_elems(dtype);
    const int64_t need = (cols + vec - 1) / vec + (aligned ? 0 : 1);
    const int64_t cap = vec == 4 ? 32 * 16 : 32 * 8;
    return need <= cap;
}

cudaError_t launch_fwd_warp(const FwdArgs &a, int dtype, bool aligned, cudaStream_t st)
{
    return dispatch<false>(a, dtype, aligned, st);
}

cudaError_t launch_bwd_warp(const BwdArgs &a, int dtype, bool aligned, cudaStream_t st)
{
    return dispatch<true>(a, dtype, aligned, st);
}

}  // namespace sms
