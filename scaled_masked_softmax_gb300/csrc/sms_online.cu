// Streaming two-pass kernels for rows of any length.
//
// Forward: pass 1 streams the row once and keeps a running (max m, sum l)
// pair per thread with the online-softmax update of the page
// "从GEMM到Transformer：手写CUDA算子优化的完整路线与性能调优实践" §2.2
//     m' = max(m, v);  l' = l * exp(m - m') + exp(v - m')
// (applied here once per 16-byte vector: the vector's own max first, then one
// rescale), merges the pairs across the CTA with the same rule, and pass 2
// re-reads the row (largely from L2: pass 1 leaves it at normal L2 priority)
// and writes y = exp(s - m) / l.  Backward: pass 1 accumulates
// dot = sum dy*y, pass 2 re-reads y and dy and writes dx.
//
// One CTA owns one row at a time (persistent grid, rows strided by the grid),
// each thread keeps U vectors in flight per iteration.
#include "sms_common.cuh"
#include "sms_internal.h"

namespace sms {
namespace {

constexpr int kNT = 512;
constexpr int kNW = kNT / 32;
constexpr int kU = 4;

struct OnlineRow {
    int64_t x0;
    int xoff;
    int limit;
    int nv_read;
    int nv_row;
};

template <int VEC>
__device__ __forceinline__ OnlineRow online_geom(int64_t r, int64_t cols, int causal, int64_t q,
                                                 const int32_t *lengths, int64_t b)
{
    OnlineRow g;
    g.x0 = r * cols;
    g.xoff = (int)(g.x0 & (VEC - 1));
    g.limit = key_limit(lengths, b, cols, causal ? (int)(q + 1) : (int)cols);
    g.nv_read = (g.xoff + g.limit + VEC - 1) / VEC;
    g.nv_row = (int)((g.xoff + cols + VEC - 1) / VEC);
    return g;
}

// Scores of vector vi of the row (-inf outside [0, limit)).
template <typename T, typename M, bool KEEP>
__device__ __forceinline__ void load_scores(const FwdArgs &a, const OnlineRow &g, const T *xs, const M *ms,
                                            int64_t m0, bool mvec, int vi, float *s)
{
    constexpr int VEC = Dt<T>::VEC;
    using MIO = MaskIO<T, M>;
    const int j0 = vi * VEC - g.xoff;
    float xv[VEC], mv[VEC];
#pragma unroll
    for (int e = 0; e < VEC; ++e) { xv[e] = 0.f; mv[e] = 0.f; }
    const int64_t gidx = g.x0 - g.xoff + (int64_t)vi * VEC;
    if (gidx + VEC <= a.x_total) {
        unpack<T>(KEEP ? ld_keep(xs + vi * VEC) : ld_stream(xs + vi * VEC), xv);
    } else {
#pragma unroll
        for (int e = 0; e < VEC; ++e)
            if (gidx + e < a.x_total) xv[e] = to_f32<T>(xs[vi * VEC + e]);
    }
    if (ms) {
        if (mvec && m0 + j0 + VEC <= a.mask_total) {
            MIO::unpack_m(MIO::ld(ms + j0), mv);
        } else {
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
                const int j = j0 + e;
                if (j >= 0 && j < g.limit) mv[e] = MIO::elem(ms + j);
            }
        }
    }
#pragma unroll
    for (int e = 0; e < VEC; ++e) {
        const int j = j0 + e;
        s[e] = (j >= 0 && j < g.limit) ? fmaf(xv[e], a.scale, mv[e]) : neg_inf();
    }
}

// Merge two (max, sum) pairs: the sums are rescaled to the larger max.
__device__ __forceinline__ void merge_ml(float &m, float &l, float m2, float l2)
{
    const float M = fmaxf(m, m2);
    const float a = (m == neg_inf()) ? 0.f : l * ex2((m - M) * kLog2e);
    const float b = (m2 == neg_inf()) ? 0.f : l2 * ex2((m2 - M) * kLog2e);
    m = M;
    l = a + b;
}

template <typename T, typename M>
__global__ void __launch_bounds__(kNT) fwd_online_kernel(const FwdArgs a)
{
    constexpr int VEC = Dt<T>::VEC;
    __shared__ float red_m[2][kNW], red_l[2][kNW];
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    int rp = 0;
    for (int64_t r = blockIdx.x; r < a.rows; r += gridDim.x, rp ^= 1) {
        int64_t q, hh, bb;
        split_row(r, a.cols, a.heads, a.dcols, a.dheads, q, hh, bb);
        const OnlineRow g = online_geom<VEC>(r, a.cols, a.causal, q, a.lengths, bb);
        const T *xs = reinterpret_cast<const T *>(a.x) + (g.x0 - g.xoff);
        const M *ms = nullptr;
        int64_t m0 = 0;
        bool mvec = false;
        if (a.mask) {
            m0 = bb * a.msb + hh * a.msh + q * a.cols;
            ms = reinterpret_cast<const M *>(a.mask) + m0;
            mvec = ((m0 - g.xoff) & (VEC - 1)) == 0;
        }

        // pass 1: running (max, sum)
        float m = neg_inf(), l = 0.f;
        for (int base = 0; base < g.nv_read; base += kNT * kU) {
            float s[kU][VEC];
            float vmax = neg_inf();
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                const int vi = base + u * kNT + t;
                if (vi < g.nv_read) {
                    load_scores<T, M, true>(a, g, xs, ms, m0, mvec, vi, s[u]);
                } else {
#pragma unroll
                    for (int e = 0; e < VEC; ++e) s[u][e] = neg_inf();
                }
#pragma unroll
                for (int e = 0; e < VEC; ++e) vmax = fmaxf(vmax, s[u][e]);
            }
            if (vmax > m) {
                l = (m == neg_inf()) ? 0.f : l * ex2((m - vmax) * kLog2e);
                m = vmax;
            }
            if (m != neg_inf()) {
#pragma unroll
                for (int u = 0; u < kU; ++u)
#pragma unroll
                    for (int e = 0; e < VEC; ++e) l += ex2((s[u][e] - m) * kLog2e);
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
            const float l2 = __shfl_xor_sync(0xffffffffu, l, o);
            merge_ml(m, l, m2, l2);
        }
        if (lane == 0) { red_m[rp][warp] = m; red_l[rp][warp] = l; }
        __syncthreads();
        m = red_m[rp][0];
        l = red_l[rp][0];
#pragma unroll
        for (int w = 1; w < kNW; ++w) merge_ml(m, l, red_m[rp][w], red_l[rp][w]);
        const float mref = (m == neg_inf()) ? 0.f : m;
        const float inv = l > 0.f ? __frcp_rn(l) : 0.f;

        // pass 2: re-read, normalise, store
        T *ys = reinterpret_cast<T *>(a.y) + (g.x0 - g.xoff);
        for (int base = 0; base < g.nv_row; base += kNT * kU) {
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                const int vi = base + u * kNT + t;
                if (vi >= g.nv_row) continue;
                float s[VEC];
                if (vi < g.nv_read) {
                    load_scores<T, M, false>(a, g, xs, ms, m0, mvec, vi, s);
                } else {
#pragma unroll
                    for (int e = 0; e < VEC; ++e) s[e] = neg_inf();
                }
                float o[VEC];
#pragma unroll
                for (int e = 0; e < VEC; ++e) o[e] = ex2((s[e] - mref) * kLog2e) * inv;
                const int j0 = vi * VEC - g.xoff;
                if (j0 >= 0 && j0 + VEC <= a.cols) {
                    st_stream(ys + vi * VEC, pack<T>(o));
                } else {
#pragma unroll
                    for (int e = 0; e < VEC; ++e) {
                        const int j = j0 + e;
                        if (j >= 0 && j < a.cols) ys[vi * VEC + e] = from_f32<T>(o[e]);
                    }
                }
            }
        }
    }
}

// y and dy of vector vi (0 outside [0, limit)).
template <typename T, bool KEEP>
__device__ __forceinline__ void load_pair(const BwdArgs &a, const OnlineRow &g, const T *ys, const T *gs, int vi,
                                          float *yv, float *gv)
{
    constexpr int VEC = Dt<T>::VEC;
    const int j0 = vi * VEC - g.xoff;
    float ty[VEC], tg[VEC];
    const int64_t gidx = g.x0 - g.xoff + (int64_t)vi * VEC;
    if (gidx + VEC <= a.total) {
        unpack<T>(KEEP ? ld_keep(ys + vi * VEC) : ld_stream(ys + vi * VEC), ty);
        unpack<T>(KEEP ? ld_keep(gs + vi * VEC) : ld_stream(gs + vi * VEC), tg);
    } else {
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
            const bool in = gidx + e < a.total;
            ty[e] = in ? to_f32<T>(ys[vi * VEC + e]) : 0.f;
            tg[e] = in ? to_f32<T>(gs[vi * VEC + e]) : 0.f;
        }
    }
#pragma unroll
    for (int e = 0; e < VEC; ++e) {
        const int j = j0 + e;
        const bool valid = j >= 0 && j < g.limit;
        yv[e] = valid ? ty[e] : 0.f;
        gv[e] = valid ? tg[e] : 0.f;
    }
}

template <typename T>
__global__ void __launch_bounds__(kNT) bwd_online_kernel(const BwdArgs a)
{
    constexpr int VEC = Dt<T>::VEC;
    __shared__ float red[2][kNW];
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    int rp = 0;
    for (int64_t r = blockIdx.x; r < a.rows; r += gridDim.x, rp ^= 1) {
        int64_t q = 0, hh = 0, bb = 0;
        if (a.lengths) split_row(r, a.cols, a.heads, a.dcols, a.dheads, q, hh, bb);
        else q = row_q(r, a.cols, a.dcols);
        const OnlineRow g = online_geom<VEC>(r, a.cols, a.causal, q, a.lengths, bb);
        const T *ys = reinterpret_cast<const T *>(a.y) + (g.x0 - g.xoff);
        const T *gs = reinterpret_cast<const T *>(a.dy) + (g.x0 - g.xoff);
        float dot = 0.f;
        for (int base = 0; base < g.nv_read; base += kNT * kU) {
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                const int vi = base + u * kNT + t;
                if (vi >= g.nv_read) continue;
                float yv[VEC], gv[VEC];
                load_pair<T, true>(a, g, ys, gs, vi, yv, gv);
#pragma unroll
                for (int e = 0; e < VEC; ++e) dot = fmaf(yv[e], gv[e], dot);
            }
        }
        dot = group_sum<32>(dot);
        if (lane == 0) red[rp][warp] = dot;
        __syncthreads();
        dot = 0.f;
#pragma unroll
        for (int w = 0; w < kNW; ++w) dot += red[rp][w];

        T *ds = reinterpret_cast<T *>(a.dx) + (g.x0 - g.xoff);
        for (int base = 0; base < g.nv_row; base += kNT * kU) {
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                const int vi = base + u * kNT + t;
                if (vi >= g.nv_row) continue;
                float yv[VEC], gv[VEC];
                if (vi < g.nv_read) {
                    load_pair<T, false>(a, g, ys, gs, vi, yv, gv);
                } else {
#pragma unroll
                    for (int e = 0; e < VEC; ++e) { yv[e] = 0.f; gv[e] = 0.f; }
                }
                float o[VEC];
#pragma unroll
                for (int e = 0; e < VEC; ++e) o[e] = (yv[e] == 0.f) ? 0.f : (gv[e] - dot) * yv[e] * a.scale;
                const int j0 = vi * VEC - g.xoff;
                if (j0 >= 0 && j0 + VEC <= a.cols) {
                    st_stream(ds + vi * VEC, pack<T>(o));
                } else {
#pragma unroll
                    for (int e = 0; e < VEC; ++e) {
                        const int j = j0 + e;
                        if (j >= 0 && j < a.cols) ds[vi * VEC + e] = from_f32<T>(o[e]);
                    }
                }
            }
        }
    }
}

template <typename Args, typename K>
cudaError_t launch_persistent(K kern, const Args &a, cudaStream_t st)
{
    const int64_t grid = persistent_grid(2, a.rows);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kNT);
    cfg.stream = st;
    return cudaLaunchKernelEx(&cfg, kern, a);
}

}  // namespace

cudaError_t launch_fwd_online(const FwdArgs &a, int dtype, cudaStream_t st)
{
    switch (dtype) {
    case kF32:
        return a.mask_bool ? launch_persistent(fwd_online_kernel<float, uint8_t>, a, st)
                           : launch_persistent(fwd_online_kernel<float, float>, a, st);
    case kF16:
        return a.mask_bool ? launch_persistent(fwd_online_kernel<__half, uint8_t>, a, st)
                           : launch_persistent(fwd_online_kernel<__half, __half>, a, st);
    case kBF16:
        return a.mask_bool ? launch_persistent(fwd_online_kernel<__nv_bfloat16, uint8_t>, a, st)
                           : launch_persistent(fwd_online_kernel<__nv_bfloat16, __nv_bfloat16>, a, st);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_bwd_online(const BwdArgs &a, int dtype, cudaStream_t st)
{
    switch (dtype) {
    case kF32: return launch_persistent(bwd_online_kernel<float>, a, st);
    case kF16: return launch_persistent(bwd_online_kernel<__half>, a, st);
    case kBF16: return launch_persistent(bwd_online_kernel<__nv_bfloat16>, a, st);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace sms
