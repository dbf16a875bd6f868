// Register-resident kernels for causal rows, processed in balanced pairs.
//
// Under the causal flag row q reads only q+1 of its S elements (the page
// "用CUDA自定义融合Softmax算子并封装进PyTorch", §1.2 and §3.1: positions j > q are
// masked), so one-row-per-group kernels leave on average half of their lanes
// and half of their memory parallelism idle.  Here a lane group takes rows q
// and S-1-q of the same head together: their read prefixes hold
// (q+1) + (S-q) = S+1 elements, so every group streams one full row's worth
// of loads.  The group's lanes walk the concatenation of both prefixes as
// 16-byte vectors (all loads first), reduce each row separately, store the
// two prefixes, then fill the causal suffixes with zeros (stores only).
//
// The backward (dx = (dy - sum dy*y) * y * scale) uses the same pairing: with
// the causal hint y is 0 beyond the diagonal, so only the prefixes are read.
#include "sms_common.cuh"
#include "sms_internal.h"

namespace sms {
namespace {

constexpr int kThreads = 256;

// Rows of pair u: head hb = u / P, position q = u mod P with P = ceil(S/2);
// r1 = hb*S + q and r2 = hb*S + S-1-q (r2 == r1 for the middle row of an odd
// S: that unit has one row).  Rows at or beyond `rows` are dead.
struct PairRow {
    int64_t r;     // row index (valid when live)
    int64_t x0;    // r * cols
    int64_t m0;    // mask row start
    int xoff;      // x0 mod VEC
    int limit;     // elements read: q + 1
    int nread;     // vectors holding elements < limit
    int nrow;      // vectors holding row elements
    bool live;
};

template <int VEC>
__device__ __forceinline__ PairRow pair_row(int64_t r, int64_t q, int64_t rows, int64_t cols, int64_t mrow0,
                                            bool live)
{
    PairRow p;
    p.live = live && r < rows;
    p.r = r;
    p.x0 = r * cols;
    p.xoff = (int)(p.x0 & (VEC - 1));
    p.limit = p.live ? (int)(q + 1) : 0;
    p.nread = p.live ? (p.xoff + p.limit + VEC - 1) / VEC : 0;
    p.nrow = (int)((p.xoff + cols + VEC - 1) / VEC);
    p.m0 = mrow0;
    return p;
}

template <int VEC>
__device__ __forceinline__ void pair_rows(int64_t u, int64_t rows, int64_t cols, int64_t heads, const FastDiv &dh,
                                          int64_t msb, int64_t msh, PairRow &A, PairRow &B)
{
    const int64_t P = (cols + 1) / 2;
    const int64_t hb = u / P;  // head index over all batches (one division per group)
    const int64_t q = u - hb * P;
    const int64_t q2 = cols - 1 - q;
    int64_t h = 0, b = 0;
    if (hb <= 0xffffffffll) {
        const uint32_t bb = dh.div((uint32_t)hb);
        b = bb;
        h = hb - (int64_t)bb * heads;
    } else {
        b = hb / heads;
        h = hb - b * heads;
    }
    const int64_t mb = b * msb + h * msh;
    A = pair_row<VEC>(hb * cols + q, q, rows, cols, mb + q * cols, true);
    B = pair_row<VEC>(hb * cols + q2, q2, rows, cols, mb + q2 * cols, q2 != q);
}

// Zero the causal suffix of a row: vectors [nread, nrow), whole vectors as
// 16-byte stores, the partial tail vector element-wise.
template <typename T, int G>
__device__ __forceinline__ void zero_suffix(T *base, const PairRow &p, int64_t cols, int gl)
{
    constexpr int VEC = Dt<T>::VEC;
    if (!p.live) return;
    T *row = base + (p.x0 - p.xoff);
    for (int v = p.nread + gl; v < p.nrow; v += G) {
        const int j0 = v * VEC - p.xoff;
        if (j0 >= 0 && j0 + VEC <= cols) {
            st_stream(row + v * VEC, make_uint4(0, 0, 0, 0));
        } else {
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
                const int j = j0 + e;
                if (j >= 0 && j < cols) row[v * VEC + e] = from_f32<T>(0.f);
            }
        }
    }
}

template <typename T, int G, int NV>
__global__ void __launch_bounds__(kThreads, 2) fwd_pair_kernel(const FwdArgs a, int64_t units)
{
    constexpr int VEC = Dt<T>::VEC;
    constexpr int GPC = kThreads / G;
    constexpr int W = G > 32 ? G / 32 : 1;
    const int gl = threadIdx.x % G;
    const int gi = threadIdx.x / G;
    const int64_t u = (int64_t)blockIdx.x * GPC + gi;
    const int64_t cols = a.cols;
    PairRow R[2];
    pair_rows<VEC>(u < units ? u : 0, a.rows, cols, a.heads, a.dheads, a.msb, a.msh, R[0], R[1]);
    if (u >= units) { R[0].live = R[1].live = false; R[0].limit = R[1].limit = 0; R[0].nread = R[1].nread = 0; }
    const int n0 = R[0].nread, ntot = R[0].nread + R[1].nread;

    // mask realignment per row (see the warp kernels): D = m0 - xoff
    int msh[2];
    int64_t mA[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int64_t D = R[i].m0 - R[i].xoff;
        msh[i] = (int)(D & (VEC - 1));
        mA[i] = D - msh[i];
    }

    uint4 xr[NV], mr[NV], mr2[NV];
#pragma unroll
    for (int k = 0; k < NV; ++k) {
        const int c = k * G + gl;
        const int sel = c >= n0;
        const int vi = sel ? c - n0 : c;
        xr[k] = mr[k] = mr2[k] = make_uint4(0, 0, 0, 0);
        if (c < ntot) {
            const int64_t xb = sel ? R[1].x0 - R[1].xoff : R[0].x0 - R[0].xoff;
            if (xb + (int64_t)(vi + 1) * VEC <= a.x_total)
                xr[k] = ld_stream(reinterpret_cast<const T *>(a.x) + xb + (int64_t)vi * VEC);
            if (a.mask) {
                const int sh = sel ? msh[1] : msh[0];
                const int64_t mb = (sel ? mA[1] : mA[0]) + (int64_t)vi * VEC;
                if (mb >= 0 && mb + (sh ? 2 : 1) * VEC <= a.mask_total) {
                    mr[k] = ld_keep(reinterpret_cast<const T *>(a.mask) + mb);
                    if (sh) mr2[k] = ld_keep(reinterpret_cast<const T *>(a.mask) + mb + VEC);
                }
            }
        }
    }

    float s[NV][VEC];
    float mx[2] = {neg_inf(), neg_inf()};
#pragma unroll
    for (int k = 0; k < NV; ++k) {
        const int c = k * G + gl;
        const int sel = c >= n0;
        const int vi = sel ? c - n0 : c;
        const int pxoff = sel ? R[1].xoff : R[0].xoff, plimit = sel ? R[1].limit : R[0].limit;
        const int64_t px0 = sel ? R[1].x0 : R[0].x0, pm0 = sel ? R[1].m0 : R[0].m0;
        const int j0 = vi * VEC - pxoff;
        float xv[VEC], mv[VEC];
        unpack<T>(xr[k], xv);
#pragma unroll
        for (int e = 0; e < VEC; ++e) mv[e] = 0.f;
        const bool act = c < ntot;
        if (act) {
            const int64_t xb = px0 - pxoff;
            if (xb + (int64_t)(vi + 1) * VEC > a.x_total) {  // last partial vector of the tensor
                const T *xs = reinterpret_cast<const T *>(a.x) + xb;
#pragma unroll
                for (int e = 0; e < VEC; ++e)
                    xv[e] = xb + vi * VEC + e < a.x_total ? to_f32<T>(xs[vi * VEC + e]) : 0.f;
            }
            if (a.mask) {
                const int sh = sel ? msh[1] : msh[0];
                const int64_t mb = (sel ? mA[1] : mA[0]) + (int64_t)vi * VEC;
                if (mb >= 0 && mb + (sh ? 2 : 1) * VEC <= a.mask_total) {
                    unpack<T>(window<VEC>(mr[k], mr2[k], sh), mv);
                } else {
                    const T *ms = reinterpret_cast<const T *>(a.mask) + pm0;
#pragma unroll
                    for (int e = 0; e < VEC; ++e) {
                        const int j = j0 + e;
                        mv[e] = (j >= 0 && j < plimit) ? to_f32<T>(ms[j]) : 0.f;
                    }
                }
            }
        }
        float m = neg_inf();
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
            const int j = j0 + e;
            s[k][e] = (act && j >= 0 && j < plimit) ? fmaf(xv[e], a.scale, mv[e]) : neg_inf();
            m = fmaxf(m, s[k][e]);
        }
        if (sel) mx[1] = fmaxf(mx[1], m); else mx[0] = fmaxf(mx[0], m);
    }

    // each lane exponentiates against its own per-row max, then the group
    // merges (max, sum) pairs of both rows
    float lt[2] = {0.f, 0.f};
    const float c0 = (mx[0] == neg_inf()) ? 0.f : -mx[0] * kLog2e;
    const float c1 = (mx[1] == neg_inf()) ? 0.f : -mx[1] * kLog2e;
#pragma unroll
    for (int k = 0; k < NV; ++k) {
        const int c = k * G + gl;
        const int sel = c >= n0;
        float l = 0.f;
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
            const float t = ex2(fmaf(s[k][e], kLog2e, sel ? c1 : c0));
            s[k][e] = t;
            l += t;
        }
        if (sel) lt[1] += l; else lt[0] += l;
    }
    float fac[2];
    if constexpr (G <= 32) {
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const float mw = group_max<G>(mx[i]);
            const float mwr = (mw == neg_inf()) ? 0.f : mw;
            const float tot = group_sum<G>(mx[i] == neg_inf() ? 0.f : lt[i] * ex2((mx[i] - mwr) * kLog2e));
            const float inv = tot > 0.f ? __frcp_rn(tot) : 0.f;
            fac[i] = (mx[i] == neg_inf()) ? 0.f : ex2((mx[i] - mwr) * kLog2e) * inv;
        }
    } else {
        __shared__ float red_m[GPC][2][W], red_l[GPC][2][W];
        const int wg = gl >> 5, lane = threadIdx.x & 31;
#pragma unroll
        for (int i = 0; i < 2; ++i) {
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
        for (int i = 0; i < 2; ++i) {
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

    T *yb = reinterpret_cast<T *>(a.y);
#pragma unroll
    for (int k = 0; k < NV; ++k) {
        const int c = k * G + gl;
        if (c >= ntot) continue;
        const int sel = c >= n0;
        const int vi = sel ? c - n0 : c;
        const int pxoff = sel ? R[1].xoff : R[0].xoff;
        const int64_t px0 = sel ? R[1].x0 : R[0].x0;
        const int j0 = vi * VEC - pxoff;
        const float f = sel ? fac[1] : fac[0];
        float o[VEC];
#pragma unroll
        for (int e = 0; e < VEC; ++e) o[e] = s[k][e] * f;
        T *row = yb + (px0 - pxoff);
        if (j0 >= 0 && j0 + VEC <= cols) {
            st_stream(row + vi * VEC, pack<T>(o));
        } else {
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
                const int j = j0 + e;
                if (j >= 0 && j < cols) row[vi * VEC + e] = from_f32<T>(o[e]);
            }
        }
    }
    zero_suffix<T, G>(yb, R[0], cols, gl);
    zero_suffix<T, G>(yb, R[1], cols, gl);
}

template <typename T, int G, int NV>
__global__ void __launch_bounds__(kThreads, 2) bwd_pair_kernel(const BwdArgs a, int64_t units)
{
    constexpr int VEC = Dt<T>::VEC;
    constexpr int GPC = kThreads / G;
    constexpr int W = G > 32 ? G / 32 : 1;
    const int gl = threadIdx.x % G;
    const int gi = threadIdx.x / G;
    const int64_t u = (int64_t)blockIdx.x * GPC + gi;
    const int64_t cols = a.cols;
    PairRow R[2];
    const FastDiv one;  // positions only: the head split is not needed
    pair_rows<VEC>(u < units ? u : 0, a.rows, cols, 1, one, 0, 0, R[0], R[1]);
    if (u >= units) { R[0].live = R[1].live = false; R[0].limit = R[1].limit = 0; R[0].nread = R[1].nread = 0; }
    const int n0 = R[0].nread, ntot = R[0].nread + R[1].nread;

    uint4 yr[NV], gr[NV];
#pragma unroll
    for (int k = 0; k < NV; ++k) {
        const int c = k * G + gl;
        const int sel = c >= n0;
        const int vi = sel ? c - n0 : c;
        yr[k] = gr[k] = make_uint4(0, 0, 0, 0);
        if (c < ntot) {
            const int64_t xb = sel ? R[1].x0 - R[1].xoff : R[0].x0 - R[0].xoff;
            if (xb + (int64_t)(vi + 1) * VEC <= a.total) {
                yr[k] = ld_stream(reinterpret_cast<const T *>(a.y) + xb + (int64_t)vi * VEC);
                gr[k] = ld_stream(reinterpret_cast<const T *>(a.dy) + xb + (int64_t)vi * VEC);
            }
        }
    }
    float dot[2] = {0.f, 0.f};
#pragma unroll
    for (int k = 0; k < NV; ++k) {
        const int c = k * G + gl;
        if (c >= ntot) continue;
        const int sel = c >= n0;
        const int vi = sel ? c - n0 : c;
        const int pxoff = sel ? R[1].xoff : R[0].xoff, plimit = sel ? R[1].limit : R[0].limit;
        const int j0 = vi * VEC - pxoff;
        const int64_t xb = (sel ? R[1].x0 : R[0].x0) - pxoff;
        if (xb + (int64_t)(vi + 1) * VEC > a.total) {  // last partial vector of the tensor
            float tv[VEC], tg[VEC];
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
                const bool in = xb + vi * VEC + e < a.total;
                tv[e] = in ? to_f32<T>(reinterpret_cast<const T *>(a.y)[xb + vi * VEC + e]) : 0.f;
                tg[e] = in ? to_f32<T>(reinterpret_cast<const T *>(a.dy)[xb + vi * VEC + e]) : 0.f;
            }
            yr[k] = pack<T>(tv);
            gr[k] = pack<T>(tg);
        }
        float yv[VEC], gv[VEC];
        unpack<T>(yr[k], yv);
        unpack<T>(gr[k], gv);
        float d = 0.f;
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
            const int j = j0 + e;
            if (j >= 0 && j < plimit) d = fmaf(yv[e], gv[e], d);
        }
        if (sel) dot[1] += d; else dot[0] += d;
    }
    if constexpr (G <= 32) {
        dot[0] = group_sum<G>(dot[0]);
        dot[1] = group_sum<G>(dot[1]);
    } else {
        __shared__ float red[GPC][2][W];
        const int wg = gl >> 5, lane = threadIdx.x & 31;
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const float d = group_sum<32>(dot[i]);
            if (lane == 0) red[gi][i][wg] = d;
        }
        __syncthreads();
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            dot[i] = 0.f;
#pragma unroll
            for (int w = 0; w < W; ++w) dot[i] += red[gi][i][w];
        }
    }
    T *db = reinterpret_cast<T *>(a.dx);
#pragma unroll
    for (int k = 0; k < NV; ++k) {
        const int c = k * G + gl;
        if (c >= ntot) continue;
        const int sel = c >= n0;
        const int vi = sel ? c - n0 : c;
        const int pxoff = sel ? R[1].xoff : R[0].xoff, plimit = sel ? R[1].limit : R[0].limit;
        const int64_t px0 = sel ? R[1].x0 : R[0].x0;
        const int j0 = vi * VEC - pxoff;
        const float d = sel ? dot[1] : dot[0];
        float yv[VEC], gv[VEC], o[VEC];
        unpack<T>(yr[k], yv);
        unpack<T>(gr[k], gv);
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
            const int j = j0 + e;
            const bool valid = j >= 0 && j < plimit;  // y == 0 (masked) gives exactly +0
            o[e] = (!valid || yv[e] == 0.f) ? 0.f : (gv[e] - d) * yv[e] * a.scale;
        }
        T *row = db + (px0 - pxoff);
        if (j0 >= 0 && j0 + VEC <= cols) {
            st_stream(row + vi * VEC, pack<T>(o));
        } else {
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
                const int j = j0 + e;
                if (j >= 0 && j < cols) row[vi * VEC + e] = from_f32<T>(o[e]);
            }
        }
    }
    zero_suffix<T, G>(db, R[0], cols, gl);
    zero_suffix<T, G>(db, R[1], cols, gl);
}

template <typename T, int G, int NV, bool BWD, typename Args>
cudaError_t launch_one(const Args &a, int64_t units, cudaStream_t st)
{
    constexpr int per_cta = kThreads / G;
    const int64_t blocks = (units + per_cta - 1) / per_cta;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks);
    cfg.blockDim = dim3(kThreads);
    cfg.stream = st;
    if constexpr (BWD)
        return cudaLaunchKernelEx(&cfg, bwd_pair_kernel<T, G, NV>, a, units);
    else
        return cudaLaunchKernelEx(&cfg, fwd_pair_kernel<T, G, NV>, a, units);
}

// Vectors a pair can span: the two prefixes hold S+1 elements; each prefix
// adds at most one vector when rows start mid-vector, and the two partial end
// vectors at most one more.
inline int64_t pair_need(int64_t cols, int vec) { return (cols + 1 + vec - 1) / vec + (cols % vec ? 3 : 1); }

template <typename T, bool BWD, typename Args>
cudaError_t launch_t(const Args &a, cudaStream_t st)
{
    constexpr int VEC = Dt<T>::VEC;
    const int64_t need = pair_need(a.cols, VEC);
    const int64_t units = ((a.rows + a.cols - 1) / a.cols) * ((a.cols + 1) / 2);
#define SMS_TRY(G, NV) \
    if (need <= (G) * (NV)) return launch_one<T, G, NV, BWD>(a, units, st);
    SMS_TRY(4, 4) SMS_TRY(8, 4) SMS_TRY(16, 4) SMS_TRY(32, 4) SMS_TRY(64, 4) SMS_TRY(64, 5) SMS_TRY(128, 4)
    SMS_TRY(128, 5) SMS_TRY(256, 4) SMS_TRY(256, 5)
#undef SMS_TRY
    return cudaErrorNotSupported;
}

template <bool BWD, typename Args>
cudaError_t dispatch(const Args &a, int dtype, cudaStream_t st)
{
    switch (dtype) {
    case kF32: return launch_t<float, BWD>(a, st);
    case kF16: return launch_t<__half, BWD>(a, st);
    case kBF16: return launch_t<__nv_bfloat16, BWD>(a, st);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace

bool pair_fits(int64_t cols, int dtype) { return pair_need(cols, vec_elems(dtype)) <= 256 * 5; }

cudaError_t launch_fwd_pair(const FwdArgs &a, int dtype, cudaStream_t st) { return dispatch<false>(a, dtype, st); }

cudaError_t launch_bwd_pair(const BwdArgs &a, int dtype, cudaStream_t st) { return dispatch<true>(a, dtype, st); }

}  // namespace sms
