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

// One lane group (G lanes: part of a warp, a warp, or W = G/32 warps) handles
// RPG consecutive rows at once: every raw 16-byte load of all RPG rows is
// issued before any arithmetic, so each lane keeps RPG*NV vectors in flight.
// Groups of one warp or less reduce with shuffles alone; multi-warp groups
// merge per-warp (max, sum) pairs through shared memory with one barrier.
template <typename T, int G, int NV, int RPG, bool ALIGNED>
__global__ void __launch_bounds__(kThreads, 2) fwd_warp_kernel(const FwdArgs a)
{
    constexpr int VEC = Dt<T>::VEC;
    constexpr int GPC = kThreads / G;         // groups per CTA
    constexpr int W = G > 32 ? G / 32 : 1;    // warps per group
    const int gl = threadIdx.x % G;           // lane within the group
    const int gi = threadIdx.x / G;           // group within the CTA
    const int64_t row0 = ((int64_t)blockIdx.x * GPC + gi) * RPG;
    const int64_t cols = a.cols;

    int64_t x0[RPG];
    int xoff[RPG], limit[RPG];
    const T *ms[RPG];
    bool mvec[RPG], live[RPG];
    uint4 xr[RPG][NV], mr[RPG][NV];

#pragma unroll
    for (int i = 0; i < RPG; ++i) {
        live[i] = row0 + i < a.rows;
        const int64_t r = live[i] ? row0 + i : a.rows - 1;  // dead rows still join the shuffles
        int64_t q = 0, h = 0, b = 0;
        if (a.causal || a.mask) split_row(r, cols, a.heads, a.dcols, a.dheads, q, h, b);
        limit[i] = a.causal ? (int)(q + 1) : (int)cols;
        x0[i] = r * cols;
        xoff[i] = ALIGNED ? 0 : (int)(x0[i] & (VEC - 1));
        ms[i] = nullptr;
        mvec[i] = ALIGNED;
        if (a.mask) {
            const int64_t m0 = b * a.msb + h * a.msh + q * cols;
            ms[i] = reinterpret_cast<const T *>(a.mask) + m0;
            if (!ALIGNED) mvec[i] = ((m0 - xoff[i]) & (VEC - 1)) == 0 && m0 - xoff[i] + (int64_t)G * NV * VEC <= a.mask_total;
        }
    }
    // issue every full-vector load first
#pragma unroll
    for (int i = 0; i < RPG; ++i) {
        const T *xs = reinterpret_cast<const T *>(a.x) + (x0[i] - xoff[i]);
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int vi = k * G + gl;
            const int j0 = vi * VEC - xoff[i];
            xr[i][k] = make_uint4(0, 0, 0, 0);
            mr[i][k] = make_uint4(0, 0, 0, 0);
            if (j0 < limit[i]) {
                if (ALIGNED || x0[i] - xoff[i] + (int64_t)(vi + 1) * VEC <= a.x_total) xr[i][k] = ld_stream(xs + vi * VEC);
                if (ms[i] && mvec[i]) mr[i][k] = ld_keep(ms[i] + j0);
            }
        }
    }

    float s[RPG][NV][VEC];
    float mx[RPG];
#pragma unroll
    for (int i = 0; i < RPG; ++i) {
        mx[i] = neg_inf();
        const T *xs = reinterpret_cast<const T *>(a.x) + (x0[i] - xoff[i]);
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int vi = k * G + gl;
            const int j0 = vi * VEC - xoff[i];
            float xv[VEC], mv[VEC];
            unpack<T>(xr[i][k], xv);
            unpack<T>(mr[i][k], mv);
            if (!ALIGNED && j0 < limit[i]) {
                const int64_t g = x0[i] - xoff[i] + (int64_t)vi * VEC;
                if (g + VEC > a.x_total) {  // last partial vector of the tensor
#pragma unroll
                    for (int e = 0; e < VEC; ++e) xv[e] = g + e < a.x_total ? to_f32<T>(xs[vi * VEC + e]) : 0.f;
                }
                if (ms[i] && !mvec[i]) {  // mask row not aligned like the x row: element loads
#pragma unroll
                    for (int e = 0; e < VEC; ++e) {
                        const int j = j0 + e;
                        mv[e] = (j >= 0 && j < limit[i]) ? to_f32<T>(ms[i][j]) : 0.f;
                    }
                }
            }
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
                const int j = j0 + e;
                const bool valid = j >= 0 && j < limit[i];
                s[i][k][e] = valid ? fmaf(xv[e], a.scale, mv[e]) : neg_inf();
                mx[i] = fmaxf(mx[i], s[i][k][e]);
            }
        }
    }
    float fac[RPG];  // y = e * fac, e the exponentials kept in s
    if constexpr (G <= 32) {
        float sum[RPG];
#pragma unroll
        for (int i = 0; i < RPG; ++i) {
            mx[i] = group_max<G>(mx[i]);
            const float mref = (mx[i] == neg_inf()) ? 0.f : mx[i];  // fully masked row: every term becomes 0
            sum[i] = 0.f;
#pragma unroll
            for (int k = 0; k < NV; ++k)
#pragma unroll
                for (int e = 0; e < VEC; ++e) {
                    const float t = ex2((s[i][k][e] - mref) * kLog2e);
                    s[i][k][e] = t;
                    sum[i] += t;
                }
        }
#pragma unroll
        for (int i = 0; i < RPG; ++i) {
            sum[i] = group_sum<G>(sum[i]);
            fac[i] = sum[i] > 0.f ? __frcp_rn(sum[i]) : 0.f;
        }
    } else {
        // each lane exponentiates against its own max; warps merge (max, sum)
        // pairs, the group's warps merge theirs through shared memory
        __shared__ float red_m[GPC][RPG][W], red_l[GPC][RPG][W];
        const int wg = gl >> 5, lane = threadIdx.x & 31;
        float lt[RPG];
#pragma unroll
        for (int i = 0; i < RPG; ++i) {
            const float mtr = (mx[i] == neg_inf()) ? 0.f : mx[i];
            lt[i] = 0.f;
#pragma unroll
            for (int k = 0; k < NV; ++k)
#pragma unroll
                for (int e = 0; e < VEC; ++e) {
                    const float t = ex2((s[i][k][e] - mtr) * kLog2e);
                    s[i][k][e] = t;
                    lt[i] += t;
                }
            const float mw = group_max<32>(mx[i]);
            const float mwr = (mw == neg_inf()) ? 0.f : mw;
            const float lw = group_sum<32>(mx[i] == neg_inf() ? 0.f : lt[i] * ex2((mx[i] - mwr) * kLog2e));
            if (lane == 0) {
                red_m[gi][i][wg] = mw;
                red_l[gi][i][wg] = lw;
            }
        }
        __syncthreads();
#pragma unroll
        for (int i = 0; i < RPG; ++i) {
            float M = neg_inf();
#pragma unroll
            for (int w = 0; w < W; ++w) M = fmaxf(M, red_m[gi][i][w]);
            const float Mr = (M == neg_inf()) ? 0.f : M;
            float tot = 0.f;
#pragma unroll
            for (int w = 0; w < W; ++w) {
                const float m2 = red_m[gi][i][w];
                tot += (m2 == neg_inf()) ? 0.f : red_l[gi][i][w] * ex2((m2 - Mr) * kLog2e);
            }
            const float inv = tot > 0.f ? __frcp_rn(tot) : 0.f;
            fac[i] = (mx[i] == neg_inf()) ? 0.f : ex2((mx[i] - Mr) * kLog2e) * inv;
        }
    }
#pragma unroll
    for (int i = 0; i < RPG; ++i) {
        if (!live[i]) continue;
        T *ys = reinterpret_cast<T *>(a.y) + (x0[i] - xoff[i]);
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int vi = k * G + gl;
            const int j0 = vi * VEC - xoff[i];
            if (j0 >= cols) continue;
            float o[VEC];
#pragma unroll
            for (int e = 0; e < VEC; ++e) o[e] = s[i][k][e] * fac[i];
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
}

template <typename T, int G, int NV, int RPG, bool ALIGNED>
__global__ void __launch_bounds__(kThreads, 2) bwd_warp_kernel(const BwdArgs a)
{
    constexpr int VEC = Dt<T>::VEC;
    constexpr int GPC = kThreads / G;
    constexpr int W = G > 32 ? G / 32 : 1;
    const int gl = threadIdx.x % G;
    const int gi = threadIdx.x / G;
    const int64_t row0 = ((int64_t)blockIdx.x * GPC + gi) * RPG;
    const int64_t cols = a.cols;

    int64_t x0[RPG];
    int xoff[RPG], limit[RPG];
    bool live[RPG];
    uint4 yr[RPG][NV], gr[RPG][NV];
#pragma unroll
    for (int i = 0; i < RPG; ++i) {
        live[i] = row0 + i < a.rows;
        const int64_t r = live[i] ? row0 + i : a.rows - 1;
        limit[i] = a.causal ? (int)(row_q(r, cols, a.dcols) + 1) : (int)cols;
        x0[i] = r * cols;
        xoff[i] = ALIGNED ? 0 : (int)(x0[i] & (VEC - 1));
    }
#pragma unroll
    for (int i = 0; i < RPG; ++i) {
        const T *ys = reinterpret_cast<const T *>(a.y) + (x0[i] - xoff[i]);
        const T *gs = reinterpret_cast<const T *>(a.dy) + (x0[i] - xoff[i]);
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int vi = k * G + gl;
            const int j0 = vi * VEC - xoff[i];
            yr[i][k] = make_uint4(0, 0, 0, 0);
            gr[i][k] = make_uint4(0, 0, 0, 0);
            if (j0 < limit[i] && (ALIGNED || x0[i] - xoff[i] + (int64_t)(vi + 1) * VEC <= a.total)) {
                yr[i][k] = ld_stream(ys + vi * VEC);
                gr[i][k] = ld_stream(gs + vi * VEC);
            }
        }
    }
    float dot[RPG];
#pragma unroll
    for (int i = 0; i < RPG; ++i) {
        dot[i] = 0.f;
        const T *ys = reinterpret_cast<const T *>(a.y) + (x0[i] - xoff[i]);
        const T *gs = reinterpret_cast<const T *>(a.dy) + (x0[i] - xoff[i]);
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int vi = k * G + gl;
            const int j0 = vi * VEC - xoff[i];
            if (!ALIGNED && j0 < limit[i]) {
                const int64_t g = x0[i] - xoff[i] + (int64_t)vi * VEC;
                if (g + VEC > a.total) {  // last partial vector of the tensor
                    float tv[VEC], tg[VEC];
#pragma unroll
                    for (int e = 0; e < VEC; ++e) {
                        const bool in = g + e < a.total;
                        tv[e] = in ? to_f32<T>(ys[vi * VEC + e]) : 0.f;
                        tg[e] = in ? to_f32<T>(gs[vi * VEC + e]) : 0.f;
                    }
                    yr[i][k] = pack<T>(tv);
                    gr[i][k] = pack<T>(tg);
                }
            }
            float yv[VEC], gv[VEC];
            unpack<T>(yr[i][k], yv);
            unpack<T>(gr[i][k], gv);
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
                const int j = j0 + e;
                if (j >= 0 && j < limit[i]) dot[i] = fmaf(yv[e], gv[e], dot[i]);
            }
        }
    }
    if constexpr (G <= 32) {
#pragma unroll
        for (int i = 0; i < RPG; ++i) dot[i] = group_sum<G>(dot[i]);
    } else {
        __shared__ float red[GPC][RPG][W];
        const int wg = gl >> 5, lane = threadIdx.x & 31;
#pragma unroll
        for (int i = 0; i < RPG; ++i) {
            const float d = group_sum<32>(dot[i]);
            if (lane == 0) red[gi][i][wg] = d;
        }
        __syncthreads();
#pragma unroll
        for (int i = 0; i < RPG; ++i) {
            dot[i] = 0.f;
#pragma unroll
            for (int w = 0; w < W; ++w) dot[i] += red[gi][i][w];
        }
    }
#pragma unroll
    for (int i = 0; i < RPG; ++i) {
        if (!live[i]) continue;
        T *dxs = reinterpret_cast<T *>(a.dx) + (x0[i] - xoff[i]);
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int vi = k * G + gl;
            const int j0 = vi * VEC - xoff[i];
            if (j0 >= cols) continue;
            float yv[VEC], gv[VEC], o[VEC];
            unpack<T>(yr[i][k], yv);
            unpack<T>(gr[i][k], gv);
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
                const int j = j0 + e;
                const bool valid = j >= 0 && j < limit[i];  // y == 0 (masked) gives exactly +0
                o[e] = (!valid || yv[e] == 0.f) ? 0.f : (gv[e] - dot[i]) * yv[e] * a.scale;
            }
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
}

template <typename T, int G, int NV, int RPG, bool ALIGNED, bool BWD, typename Args>
cudaError_t launch_one(const Args &a, cudaStream_t st)
{
    constexpr int rows_per_cta = (kThreads / G) * RPG;
    const int64_t blocks = (a.rows + rows_per_cta - 1) / rows_per_cta;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks);
    cfg.blockDim = dim3(kThreads);
    cfg.stream = st;
    if constexpr (BWD)
        return cudaLaunchKernelEx(&cfg, bwd_warp_kernel<T, G, NV, RPG, ALIGNED>, a);
    else
        return cudaLaunchKernelEx(&cfg, fwd_warp_kernel<T, G, NV, RPG, ALIGNED>, a);
}

// (lanes per row, vectors per lane per row, rows per lane group), smallest
// capacity first.  Capacity = G*NV vectors; each lane keeps RPG*NV vectors
// per input stream in flight: up to 8 for fp32 rows and 4 for 16-bit rows
// (32 fp32 values either way).
template <typename T, bool ALIGNED, bool BWD, typename Args>
cudaError_t launch_t(const Args &a, cudaStream_t st)
{
    constexpr int VEC = Dt<T>::VEC;
    const int64_t need = (a.cols + VEC - 1) / VEC + (ALIGNED ? 0 : 1);
    // rows that may start mid-vector carry more bookkeeping: half the rows per group
#define SMS_TRY(G, NV, RPG) \
    if (need <= (G) * (NV)) return launch_one<T, G, NV, (ALIGNED || (RPG) == 1 ? (RPG) : (RPG) / 2), ALIGNED, BWD>(a, st);
    if constexpr (VEC == 4) {
        SMS_TRY(4, 1, 8) SMS_TRY(8, 1, 8) SMS_TRY(16, 1, 8) SMS_TRY(32, 1, 8) SMS_TRY(32, 2, 4) SMS_TRY(32, 3, 2)
        SMS_TRY(32, 4, 2) SMS_TRY(32, 6, 1) SMS_TRY(32, 8, 1) SMS_TRY(64, 8, 1) SMS_TRY(128, 8, 1)
        SMS_TRY(256, 6, 1) SMS_TRY(256, 8, 1)
    } else {
        SMS_TRY(4, 1, 4) SMS_TRY(8, 1, 4) SMS_TRY(16, 1, 4) SMS_TRY(32, 1, 4) SMS_TRY(32, 2, 2) SMS_TRY(32, 3, 1)
        SMS_TRY(32, 4, 1) SMS_TRY(64, 4, 1) SMS_TRY(128, 4, 1) SMS_TRY(256, 3, 1) SMS_TRY(256, 4, 1)
    }
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

bool warp_fits(int64_t cols, int dtype, bool aligned, bool bwd)
{
    const int vec = vec_elems(dtype);
    const int64_t need = (cols + vec - 1) / vec + (aligned ? 0 : 1);
    (void)bwd;
    const int64_t cap = vec == 4 ? 256 * 8 : 256 * 4;  // widest shapes: 256 lanes x 8 (fp32) / 4 (16-bit) vectors
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
