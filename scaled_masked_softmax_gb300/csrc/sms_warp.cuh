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
#pragma once

#include <type_traits>

#include "sms_rowmath.cuh"

namespace sms {
namespace {

constexpr int kThreads = 256;  // 8 warps per CTA

// Positions of the RPG consecutive rows row0 .. row0+RPG-1 of a lane group:
// the first is split with the invariant-divisor division, the others follow
// by stepping one row (q+1, wrapping into the next head and batch).  Rows at
// or beyond `rows` get limit 0: they read and write nothing.  With per-batch
// key lengths the limit is cut to the row's batch length.
template <int RPG>
__device__ __forceinline__ void group_rows(int64_t row0, int64_t rows, int64_t cols, int64_t heads, bool causal,
                                           bool need_pos, const FastDiv &dc, const FastDiv &dh, int64_t msb,
                                           int64_t msh, const int32_t *lengths, int (&limit)[RPG],
                                           int64_t (&m0)[RPG])
{
    int64_t q = 0, h = 0, b = 0;
    if (need_pos && row0 < rows) split_row(row0, cols, heads, dc, dh, q, h, b);
#pragma unroll
    for (int i = 0; i < RPG; ++i) {
        if (i > 0 && need_pos) {
            if (++q == cols) {
                q = 0;
                if (++h == heads) { h = 0; ++b; }
            }
        }
        const bool live = row0 + i < rows;
        limit[i] = live ? key_limit(lengths, b, cols, causal ? (int)(q + 1) : (int)cols) : 0;
        m0[i] = b * msb + h * msh + q * cols;
    }
}

// One lane group (G lanes: part of a warp, a warp, or W = G/32 warps) handles
// RPG consecutive rows at once: every raw 16-byte load of all RPG rows is
// issued before any arithmetic, so each lane keeps RPG*NV vectors in flight.
// Groups of one warp or less reduce with shuffles alone; multi-warp groups
// merge per-warp (max, sum) pairs through shared memory with one barrier.
template <typename T, int G, int NV, int RPG, bool ALIGNED, typename M>
__global__ void __launch_bounds__(kThreads, 2) fwd_warp_kernel(const FwdArgs a)
{
    constexpr int VEC = Dt<T>::VEC;
    using MIO = MaskIO<T, M>;
    constexpr int GPC = kThreads / G;         // groups per CTA
    constexpr int W = G > 32 ? G / 32 : 1;    // warps per group
    const int gl = threadIdx.x % G;           // lane within the group
    const int gi = threadIdx.x / G;           // group within the CTA
    const int64_t row0 = ((int64_t)blockIdx.x * GPC + gi) * RPG;
    const int64_t cols = a.cols;

    int limit[RPG];
    int64_t m0[RPG];
    group_rows<RPG>(row0, a.rows, cols, a.heads, a.causal, a.causal || a.mask || a.lengths, a.dcols, a.dheads, a.msb,
                    a.msh, a.lengths, limit, m0);
    // The mask row of row i starts D = m0 - xoff elements into the x-aligned
    // vector grid: its elements for x vector vi sit at A + vi*VEC + sh ..,
    // A = D - sh aligned, sh = D mod VEC.  sh == 0: one 16-byte load per
    // vector; otherwise two neighbouring aligned loads and a register shift.
    int xoff[RPG], msh[RPG];
    int64_t mA[RPG];
    uint4 xr[RPG][NV], mr[RPG][NV];
    uint4 mr2[ALIGNED ? 1 : RPG][ALIGNED ? 1 : NV];
#pragma unroll
    for (int i = 0; i < RPG; ++i) {
        const int64_t x0 = (row0 + i) * cols;
        xoff[i] = ALIGNED ? 0 : (int)(x0 & (VEC - 1));
        const int64_t D = m0[i] - xoff[i];
        msh[i] = ALIGNED ? 0 : (int)(D & (VEC - 1));
        mA[i] = D - msh[i];
    }
    // issue every full-vector load first
#pragma unroll
    for (int i = 0; i < RPG; ++i) {
        const int64_t xb = (row0 + i) * cols - xoff[i];  // aligned start of the row's vectors
        const T *xs = reinterpret_cast<const T *>(a.x) + xb;
        const M *mk = reinterpret_cast<const M *>(a.mask);
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int vi = k * G + gl;
            const int j0 = vi * VEC - xoff[i];
            xr[i][k] = make_uint4(0, 0, 0, 0);
            mr[i][k] = make_uint4(0, 0, 0, 0);
            if constexpr (!ALIGNED) mr2[i][k] = make_uint4(0, 0, 0, 0);
            if (j0 < limit[i]) {
                if (ALIGNED || xb + (int64_t)(vi + 1) * VEC <= a.x_total) xr[i][k] = ld_stream(xs + vi * VEC);
                if (a.mask) {
                    const int64_t mb = mA[i] + (int64_t)vi * VEC;  // first aligned mask vector
                    if (ALIGNED) {
                        mr[i][k] = MIO::ld(mk + mb);
                    } else if (mb >= 0 && mb + (msh[i] ? 2 : 1) * VEC <= a.mask_total) {
                        mr[i][k] = MIO::ld(mk + mb);
                        if (msh[i]) mr2[i][k] = MIO::ld(mk + mb + VEC);
                    }
                }
            }
        }
    }

    float s[RPG][NV][VEC];
    float mx[RPG];
#pragma unroll
    for (int i = 0; i < RPG; ++i) {
        mx[i] = neg_inf();
        const int64_t xb = (row0 + i) * cols - xoff[i];
        const T *xs = reinterpret_cast<const T *>(a.x) + xb;
        const M *ms = reinterpret_cast<const M *>(a.mask) + m0[i];
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int vi = k * G + gl;
            const int j0 = vi * VEC - xoff[i];
            float xv[VEC], mv[VEC];
            unpack<T>(xr[i][k], xv);
            if constexpr (ALIGNED) {
                MIO::unpack_m(mr[i][k], mv);
            } else {
#pragma unroll
                for (int e = 0; e < VEC; ++e) mv[e] = 0.f;
                if (j0 < limit[i]) {
                    if (xb + (int64_t)(vi + 1) * VEC > a.x_total) {  // last partial vector of the tensor
#pragma unroll
                        for (int e = 0; e < VEC; ++e)
                            xv[e] = xb + vi * VEC + e < a.x_total ? to_f32<T>(xs[vi * VEC + e]) : 0.f;
                    }
                    if (a.mask) {
                        const int64_t mb = mA[i] + (int64_t)vi * VEC;
                        if (mb >= 0 && mb + (msh[i] ? 2 : 1) * VEC <= a.mask_total) {
                            MIO::unpack_m(MIO::win_rt(mr[i][k], mr2[i][k], msh[i]), mv);
                        } else {  // mask vectors at the ends of the mask buffer: element loads
#pragma unroll
                            for (int e = 0; e < VEC; ++e) {
                                const int j = j0 + e;
                                mv[e] = (j >= 0 && j < limit[i]) ? MIO::elem(ms + j) : 0.f;
                            }
                        }
                    }
                }
            }
            if (j0 >= 0 && j0 + VEC <= limit[i]) {  // interior vector: every element is read
#pragma unroll
                for (int e = 0; e < VEC; ++e) {
                    s[i][k][e] = fmaf(xv[e], a.scale, mv[e]);
                    mx[i] = fmaxf(mx[i], s[i][k][e]);
                }
            } else {
#pragma unroll
                for (int e = 0; e < VEC; ++e) {
                    const int j = j0 + e;
                    s[i][k][e] = (j >= 0 && j < limit[i]) ? fmaf(xv[e], a.scale, mv[e]) : neg_inf();
                    mx[i] = fmaxf(mx[i], s[i][k][e]);
                }
            }
        }
    }

    // exp(s - m) = 2^(s*log2e - m*log2e): one FMA per element; the rounding
    // of m*log2e is common to the whole row and cancels in the normalisation
    float fac[RPG];  // y = e * fac, e the exponentials kept in s
    if constexpr (G <= 32) {
        float sum[RPG];
#pragma unroll
        for (int i = 0; i < RPG; ++i) {
            mx[i] = group_max<G>(mx[i]);
            const float c = (mx[i] == neg_inf()) ? 0.f : -mx[i] * kLog2e;  // fully masked row: every term 0
            sum[i] = 0.f;
#pragma unroll
            for (int k = 0; k < NV; ++k)
#pragma unroll
                for (int e = 0; e < VEC; ++e) {
                    const float t = ex2(fmaf(s[i][k][e], kLog2e, c));
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
#pragma unroll
        for (int i = 0; i < RPG; ++i) {
            const float c = (mx[i] == neg_inf()) ? 0.f : -mx[i] * kLog2e;
            float lt = 0.f;
#pragma unroll
            for (int k = 0; k < NV; ++k)
#pragma unroll
                for (int e = 0; e < VEC; ++e) {
                    const float t = ex2(fmaf(s[i][k][e], kLog2e, c));
                    s[i][k][e] = t;
                    lt += t;
                }
            const float mw = group_max<32>(mx[i]);
            const float mwr = (mw == neg_inf()) ? 0.f : mw;
            const float lw = group_sum<32>(mx[i] == neg_inf() ? 0.f : lt * ex2((mx[i] - mwr) * kLog2e));
            if (lane == 0) {
                red_m[gi][i][wg] = mw;
                red_l[gi][i][wg] = lw;
            }
        }
        __syncthreads();
#pragma unroll
        for (int i = 0; i < RPG; ++i) {
            float mg = neg_inf();
#pragma unroll
            for (int w = 0; w < W; ++w) mg = fmaxf(mg, red_m[gi][i][w]);
            const float Mr = (mg == neg_inf()) ? 0.f : mg;
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
        if (row0 + i >= a.rows) continue;
        T *ys = reinterpret_cast<T *>(a.y) + ((row0 + i) * cols - xoff[i]);
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

    int limit[RPG];
    int64_t unused_m0[RPG];
    group_rows<RPG>(row0, a.rows, cols, a.heads, a.causal, a.causal || a.lengths, a.dcols, a.dheads, 0, 0, a.lengths,
                    limit, unused_m0);
    int xoff[RPG];
    uint4 yr[RPG][NV], gr[RPG][NV];
#pragma unroll
    for (int i = 0; i < RPG; ++i) xoff[i] = ALIGNED ? 0 : (int)(((row0 + i) * cols) & (VEC - 1));
#pragma unroll
    for (int i = 0; i < RPG; ++i) {
        const int64_t xb = (row0 + i) * cols - xoff[i];
        const T *ys = reinterpret_cast<const T *>(a.y) + xb;
        const T *gs = reinterpret_cast<const T *>(a.dy) + xb;
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int vi = k * G + gl;
            const int j0 = vi * VEC - xoff[i];
            yr[i][k] = make_uint4(0, 0, 0, 0);
            gr[i][k] = make_uint4(0, 0, 0, 0);
            if (j0 < limit[i] && (ALIGNED || xb + (int64_t)(vi + 1) * VEC <= a.total)) {
                yr[i][k] = ld_stream(ys + vi * VEC);
                gr[i][k] = ld_stream(gs + vi * VEC);
            }
        }
    }
    float dot[RPG];
#pragma unroll
    for (int i = 0; i < RPG; ++i) {
        dot[i] = 0.f;
        const int64_t xb = (row0 + i) * cols - xoff[i];
        const T *ys = reinterpret_cast<const T *>(a.y) + xb;
        const T *gs = reinterpret_cast<const T *>(a.dy) + xb;
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int vi = k * G + gl;
            const int j0 = vi * VEC - xoff[i];
            if (!ALIGNED && j0 < limit[i] && xb + (int64_t)(vi + 1) * VEC > a.total) {  // last partial vector
                float tv[VEC], tg[VEC];
#pragma unroll
                for (int e = 0; e < VEC; ++e) {
                    const bool in = xb + vi * VEC + e < a.total;
                    tv[e] = in ? to_f32<T>(ys[vi * VEC + e]) : 0.f;
                    tg[e] = in ? to_f32<T>(gs[vi * VEC + e]) : 0.f;
                }
                yr[i][k] = pack<T>(tv);
                gr[i][k] = pack<T>(tg);
            }
            float yv[VEC], gv[VEC];
            unpack<T>(yr[i][k], yv);
            unpack<T>(gr[i][k], gv);
            if (j0 >= 0 && j0 + VEC <= limit[i]) {  // interior vector
#pragma unroll
                for (int e = 0; e < VEC; ++e) dot[i] = fmaf(yv[e], gv[e], dot[i]);
            } else {
#pragma unroll
                for (int e = 0; e < VEC; ++e) {
                    const int j = j0 + e;
                    if (j >= 0 && j < limit[i]) dot[i] = fmaf(yv[e], gv[e], dot[i]);
                }
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
        if (row0 + i >= a.rows) continue;
        T *dxs = reinterpret_cast<T *>(a.dx) + ((row0 + i) * cols - xoff[i]);
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

// Row at place n of the launch order under the mask-reuse order (ReuseOrder):
// the super-block, then the region of tiles, then (block k, query q) inside
// the tile, blocks in order and queries in order within a block.
__device__ __forceinline__ int64_t reuse_row(const FwdArgs &a, int64_t n)
{
    const ReuseOrder &o = a.reuse;
    if (n >= o.rows) return n;  // natural order (o.rows == 0 when the order is off)
    constexpr uint32_t T = kReuseTile;
    const uint32_t S = (uint32_t)a.cols, nn = (uint32_t)n;
    const uint32_t sb = o.d_sb.div(nn);
    uint32_t loc = nn - sb * o.sb, k, q;
    if (loc < o.pa) {  // A: kf + 1 blocks of T rows per tile
        const uint32_t t = o.d_a.div(loc);
        const uint32_t j = loc - t * ((o.kf + 1) * T);
        k = j / T;
        q = t * T + j % T;
    } else if ((loc -= o.pa) < o.pb) {  // B: kf blocks of wb rows, then the last block's rem_b
        if (loc < o.kf * o.wb) {
            k = loc / o.wb;
            q = o.ta * T + (loc - k * o.wb);
        } else {
            k = o.kf;
            q = o.ta * T + (loc - o.kf * o.wb);
        }
    } else if ((loc -= o.pb) < o.pc) {  // C, whole tiles: kf blocks of T rows
        const uint32_t t = o.d_c.div(loc);
        const uint32_t j = loc - t * (o.kf * T);
        k = j / T;
        q = o.base_c + t * T + j % T;
    } else {  // C, the final narrower tile
        loc -= o.pc;
        const uint32_t w = S - o.base_c - o.nc * T;
        k = loc / w;
        q = o.base_c + o.nc * T + (loc - k * w);
    }
    return (int64_t)sb * o.sb + (int64_t)k * S + q;
}

// Misaligned rows on whole warps take the contiguous lane mapping (each warp
// a run of consecutive vectors); with an additive mask they also take their
// second aligned mask vector from the neighbouring lane by shuffle instead of
// a second load per slot (4*NV fewer registers).  A byte mask's second vector
// is one or two words, and the shuffles cost it 3-4 points: it keeps the
// second load, on the same mapping, so that a boolean mask and its additive
// -inf form give the same bits.  Measured on GB300, with the CTAs per SM
// the freed registers allow (fwd_min_ctas): 16-bit rows gain at every lane
// count from 32; fp32 rows gain from 128 lanes (S=2049 73% -> 76%, S=3333
// 73% -> 74%, S=4099 71% -> 77%) and lose 0.5-2 points at 64 lanes, which
// keep the old form.
template <typename T, int G, int NV, bool ALIGNED> __host__ __device__ constexpr bool fwd_contiguous()
{
    return !ALIGNED && G >= 32 && (sizeof(T) == 2 || G >= 128);
}
template <typename T, typename M, int G, int NV, bool ALIGNED> __host__ __device__ constexpr bool fwd_shuffled()
{
    return fwd_contiguous<T, G, NV, ALIGNED>() && std::is_same<T, M>::value;
}

// One row per lane group: the shared row math of sms_rowmath.cuh (one
// switch per row realigns a misaligned mask, bounds are tested once per row,
// paired elements use the packed fp32x2 forms).  CTAs per SM it is compiled
// for: the shuffled shapes of at most 5 vectors per lane take four, at 64
// registers (fp32 S=4099, 256 x 5, no spill: +6 points; the 16-bit 32, 64
// and 128 x 5 shapes spill 212-284 B and still gain 4-5 points over three
// CTAs at S = 1100, 2049, 2500 and 4099), those of 6 or 7 take three, at 80
// (spilling 40-600 B, against two CTAs: f16 S=1500 57% -> 69%, S=1700
// 59% -> 69%, S=3333 59% -> 66%).  Otherwise fp32 rows
// are held in at most 80 registers, three CTAs per multiprocessor: measured
// faster than two CTAs with more registers (S=4099: 66% against 43% of the
// copy rate; S=1024: +5%); not for misaligned fp32 rows of 6 or 8 vectors per
// lane (they would spill).  The 16-bit forms take three CTAs at 5 vectors per
// lane (the misaligned ones gained 9-11 points over two CTAs at S=2049, 2500
// and 4099); at 4, 6 or 8 vectors two CTAs measured no worse.
template <typename T, typename M, int G, int NV, bool ALIGNED> constexpr int fwd_min_ctas()
{
    if (fwd_shuffled<T, M, G, NV, ALIGNED>() && NV <= 5) return 4;
    if (fwd_shuffled<T, M, G, NV, ALIGNED>() && NV <= 7) return 3;
    return (Dt<T>::VEC == 4 && (ALIGNED || NV <= 5)) ? 3 : (NV == 5 ? 3 : 2);
}

template <typename T, int G, int NV, bool ALIGNED, typename M>
__global__ void __launch_bounds__(kThreads, fwd_min_ctas<T, M, G, NV, ALIGNED>()) fwd_row_kernel(const FwdArgs a)
{
    using namespace rowmath;
    constexpr int GPC = kThreads / G;
    constexpr int W = G > 32 ? G / 32 : 1;
    __shared__ float red_m[GPC][W], red_l[GPC][W];
    const int gl = threadIdx.x % G;
    const int gi = threadIdx.x / G;
    const int64_t n = (int64_t)blockIdx.x * GPC + gi;
    // the mask-reuse order is only ever set up for fp32 rows of 4096 or more
    // columns (sms_abi.cu); other shapes leave its arithmetic out
    constexpr bool REUSE = sizeof(T) == 4 && G * NV * Dt<T>::VEC >= 4096;
    const RowPos p = fwd_pos<Dt<T>::VEC, ALIGNED>(a, REUSE ? reuse_row(a, n) : n);
    constexpr bool SHUF = fwd_shuffled<T, M, G, NV, ALIGNED>(), CONTIG = fwd_contiguous<T, G, NV, ALIGNED>();
    FwdBuf<NV, ALIGNED, SHUF> B;
    fwd_issue<T, G, NV, ALIGNED, M, SHUF, CONTIG>(a, p, gl, B);
    fwd_finish<T, G, NV, ALIGNED, M, SHUF, CONTIG>(a, p, gl, gi, B, red_m, red_l);
}

template <typename T, int G, int NV, bool ALIGNED>
__global__ void __launch_bounds__(kThreads, 2) bwd_row_kernel(const BwdArgs a)
{
    using namespace rowmath;
    constexpr int GPC = kThreads / G;
    constexpr int W = G > 32 ? G / 32 : 1;
    __shared__ float red[GPC][W];
    const int gl = threadIdx.x % G;
    const int gi = threadIdx.x / G;
    const BRowPos p = bwd_pos<Dt<T>::VEC, ALIGNED>(a, (int64_t)blockIdx.x * GPC + gi);
    BwdBuf<NV> B;
    bwd_issue<T, G, NV, ALIGNED>(a, p, gl, B);
    bwd_finish<T, G, NV, ALIGNED>(a, p, gl, gi, B, red);
}

template <typename T, int G, int NV, int RPG, bool ALIGNED, bool BWD, typename M, typename Args>
cudaError_t launch_one(const Args &a, cudaStream_t st)
{
    constexpr int rows_per_cta = (kThreads / G) * RPG;
    const int64_t blocks = (a.rows + rows_per_cta - 1) / rows_per_cta;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks);
    cfg.blockDim = dim3(kThreads);
    cfg.stream = st;
    if constexpr (RPG == 1) {
        if constexpr (BWD)
            return cudaLaunchKernelEx(&cfg, bwd_row_kernel<T, G, NV, ALIGNED>, a);
        else
            return cudaLaunchKernelEx(&cfg, fwd_row_kernel<T, G, NV, ALIGNED, M>, a);
    } else {
        if constexpr (BWD)
            return cudaLaunchKernelEx(&cfg, bwd_warp_kernel<T, G, NV, RPG, ALIGNED>, a);
        else
            return cudaLaunchKernelEx(&cfg, fwd_warp_kernel<T, G, NV, RPG, ALIGNED, M>, a);
    }
}

// (lanes per row, vectors per lane per row, rows per lane group), smallest
// capacity first.  Between the power-of-two lane counts, rows take 5, 6 or 7
// vectors per lane on fewer lanes instead of twice the lanes half idle
// (S = 1025 .. 1792 and 2049 .. 3584, often misaligned): measured +10 to +30
// points there (f16 S=1025: 30% -> 59%, S=3500: 48% -> 62%; fp32 S=1100:
// 64% -> 90%, S=3500: 84% -> 95% of the copy rate).  128 lanes x 7 is left out
// of the 16-bit list: 256 x 4 measured faster for those rows (S=7000).  Capacity = G*NV vectors.  Each lane keeps RPG*NV vectors
// per input stream in flight: 4 (5 for rows just past a power of two) for
// every backward and 16-bit forward shape, up to 8 for the fp32 forward (its
// mask stream is served by L2).  More vectors per lane stop fitting the 128
// registers that keep two CTAs per SM, and loads then serialise.  Short rows
// use few lanes with several vectors each: fewer shuffle rounds per row.
// Aligned 16-bit forward rows beyond 256*5 vectors take 6 or 8 vectors per
// lane (no realignment registers are needed there): measured faster than the
// staged CTA path at those widths, slower than 4-5 vectors below them.
template <typename T, bool ALIGNED, bool BWD, typename M, typename Args>
cudaError_t launch_t(const Args &a, cudaStream_t st)
{
    constexpr int VEC = Dt<T>::VEC;
    const int64_t need = (a.cols + VEC - 1) / VEC + (ALIGNED ? 0 : 1);
    // rows that may start mid-vector carry more bookkeeping: half the rows per group
#define SMS_TRY(G, NV, RPG) \
    if (need <= (G) * (NV)) return launch_one<T, G, NV, (ALIGNED || (RPG) == 1 ? (RPG) : (RPG) / 2), ALIGNED, BWD, M>(a, st);
    if constexpr (VEC == 4 && !BWD) {
        SMS_TRY(4, 1, 8) SMS_TRY(4, 2, 4) SMS_TRY(8, 2, 4) SMS_TRY(8, 4, 2) SMS_TRY(16, 4, 2) SMS_TRY(32, 4, 2)
        SMS_TRY(32, 8, 1) SMS_TRY(64, 5, 1) SMS_TRY(64, 6, 1) SMS_TRY(64, 7, 1) SMS_TRY(128, 4, 1) SMS_TRY(128, 5, 1)
        SMS_TRY(128, 6, 1) SMS_TRY(128, 7, 1) SMS_TRY(256, 4, 1) SMS_TRY(256, 5, 1)
        SMS_TRY(256, 6, 1) SMS_TRY(256, 8, 1)
    } else {
        SMS_TRY(4, 1, 4) SMS_TRY(4, 2, 2) SMS_TRY(4, 4, 1) SMS_TRY(8, 4, 1) SMS_TRY(16, 4, 1) SMS_TRY(32, 4, 1)
        SMS_TRY(32, 5, 1) SMS_TRY(32, 6, 1) SMS_TRY(32, 7, 1) SMS_TRY(64, 4, 1) SMS_TRY(64, 5, 1) SMS_TRY(64, 6, 1)
        SMS_TRY(64, 7, 1) SMS_TRY(128, 4, 1) SMS_TRY(128, 5, 1) SMS_TRY(128, 6, 1) SMS_TRY(256, 4, 1)
        SMS_TRY(256, 5, 1)
        if constexpr (!BWD && ALIGNED) { SMS_TRY(256, 6, 1) SMS_TRY(256, 8, 1) }
    }
#undef SMS_TRY
    return cudaErrorNotSupported;
}

// MASKB: the forward's mask is boolean (one byte per element), else additive
// with the dtype of x (the backward reads no mask).
template <bool BWD, bool MASKB, typename Args>
cudaError_t dispatch(const Args &a, int dtype, bool aligned, cudaStream_t st)
{
    switch (dtype) {
    case kF32: {
        using M = std::conditional_t<MASKB, uint8_t, float>;
        return aligned ? launch_t<float, true, BWD, M>(a, st) : launch_t<float, false, BWD, M>(a, st);
    }
    case kF16: {
        using M = std::conditional_t<MASKB, uint8_t, __half>;
        return aligned ? launch_t<__half, true, BWD, M>(a, st) : launch_t<__half, false, BWD, M>(a, st);
    }
    case kBF16: {
        using M = std::conditional_t<MASKB, uint8_t, __nv_bfloat16>;
        return aligned ? launch_t<__nv_bfloat16, true, BWD, M>(a, st) : launch_t<__nv_bfloat16, false, BWD, M>(a, st);
    }
    default:
        return cudaErrorInvalidValue;
    }
}

}  // namespace
}  // namespace sms
