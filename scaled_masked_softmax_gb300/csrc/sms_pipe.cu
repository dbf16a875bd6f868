// Pipelined lane-group kernels: the register-resident row kernels with their
// loads moved off the register file.
//
// A lane group (G lanes: part of a warp, a warp, or several) owns a unit of
// RPG consecutive rows, each lane the same NV 16-byte vectors per row as in
// the register-resident kernels.  Persistent CTAs walk a strided sequence of
// units; every thread streams its own vectors of the next K-1 units into a
// private ring of K shared-memory stages with cp.async (asynchronous 16-byte
// copies, completion per thread through commit groups), so the bytes in
// flight per SM are bounded by shared memory (about 190 KB) rather than by
// registers.  A thread reads back exactly the vectors it copied, so no barrier
// is needed for the data; groups wider than a warp still merge their partial
// (max, sum) pairs (forward) or dot products (backward) through one named
// barrier per unit.  The broadcast mask of the forward is not staged: it is
// read with ordinary loads (served by L2) while the row waits.
//
// The arithmetic is that of the register-resident kernels: s = x*scale + m,
// exp(s - max) evaluated once per element as 2^(s*log2e - max*log2e), one
// normalisation, stores rounded once to the output type; backward
// dx = (dy - sum dy*y) * y * scale.
#include "sms_common.cuh"
#include "sms_internal.h"

#include <atomic>

namespace sms {
namespace {

constexpr int kNT = 512;                   // threads per CTA (16 warps), one CTA per SM
constexpr int kStageBudget = 192 * 1024;   // shared memory for the rings

// Position (q, h, b) of a row, advanced by a fixed number of rows with
// carries instead of divisions.
struct Cursor {
    int64_t r, q, h, b;
};

__device__ __forceinline__ void cursor_split(Cursor &c, int64_t r, int64_t cols, int64_t heads, const FastDiv &dc,
                                             const FastDiv &dh)
{
    c.r = r;
    split_row(r, cols, heads, dc, dh, c.q, c.h, c.b);
}

// Advance by D = dq + cols * (dh + heads * db) rows.
__device__ __forceinline__ void cursor_step(Cursor &c, int64_t D, int64_t dq, int64_t dhh, int64_t db, int64_t cols,
                                            int64_t heads)
{
    c.r += D;
    c.q += dq;
    int64_t carry = 0;
    if (c.q >= cols) { c.q -= cols; carry = 1; }
    c.h += dhh + carry;
    carry = 0;
    if (c.h >= heads) { c.h -= heads; carry = 1; }
    c.b += db + carry;
}

// Next row (q + 1, wrapping into the next head and batch).
__device__ __forceinline__ void cursor_next(Cursor &c, int64_t cols, int64_t heads)
{
    ++c.r;
    if (++c.q == cols) {
        c.q = 0;
        if (++c.h == heads) { c.h = 0; ++c.b; }
    }
}

template <typename T, int NV, int RPG, int STREAMS>
struct PipeGeo {
    static constexpr int SLOTS = RPG * NV;                         // vectors per thread per unit per stream
    static constexpr int STAGE = STREAMS * SLOTS * kNT;            // uint4 per stage
    static constexpr int K = kStageBudget / (STAGE * 16) < 8 ? kStageBudget / (STAGE * 16) : 8;
    static constexpr int SMEM = K * STAGE * 16;
    static_assert(K >= 2, "a ring needs two stages");
};

// ------------------------------------------------------------------ forward

// Issue this thread's cp.async copies of the x vectors of the unit whose first
// row is at cursor c0 into ring stage `stage`.
template <typename T, int G, int NV, int RPG, bool ALIGNED, int SLOTS>
__device__ __forceinline__ void fwd_issue(const FwdArgs &a, const Cursor &c0, int stage, bool need_pos, int gl, int tid,
                                          uint4 *sbuf, uint64_t pol)
{
    constexpr int VEC = Dt<T>::VEC;
    Cursor c = c0;
#pragma unroll
    for (int i = 0; i < RPG; ++i) {
        if (i > 0) {
            if (need_pos) cursor_next(c, a.cols, a.heads); else ++c.r;
        }
        if (c.r < a.rows) {
            const int limit = a.causal ? (int)(c.q + 1) : (int)a.cols;
            const int64_t x0 = c.r * a.cols;
            const int xoff = ALIGNED ? 0 : (int)(x0 & (VEC - 1));
            const int64_t xb = x0 - xoff;
#pragma unroll
            for (int k = 0; k < NV; ++k) {
                const int vi = k * G + gl;
                if (vi * VEC - xoff < limit && (ALIGNED || xb + (int64_t)(vi + 1) * VEC <= a.x_total))
                    cp_async16(&sbuf[((size_t)stage * SLOTS + i * NV + k) * kNT + tid],
                               reinterpret_cast<const T *>(a.x) + xb + (int64_t)vi * VEC, pol);
            }
        }
    }
}

template <typename T, int G, int NV, int RPG, bool ALIGNED>
__global__ void __launch_bounds__(kNT, 1) fwd_pipe_kernel(const FwdArgs a, int64_t units)
{
    using PG = PipeGeo<T, NV, RPG, 1>;
    constexpr int VEC = Dt<T>::VEC;
    constexpr int K = PG::K;
    constexpr int GPC = kNT / G;
    constexpr int W = G > 32 ? G / 32 : 1;
    extern __shared__ __align__(16) uint4 sbuf[];
    const int tid = threadIdx.x;
    const int gl = tid % G, gi = tid / G;
    const int64_t cols = a.cols, heads = a.heads;
    const int64_t NG = (int64_t)gridDim.x * GPC;
    const int64_t gid = (int64_t)blockIdx.x * GPC + gi;
    // iterations: the unit count of the warp's first group, so every lane of a
    // warp runs the same loop (the shuffles are warp-wide); a group past its
    // last unit has rows >= rows and reads and writes nothing
    const int64_t gid_w = (int64_t)blockIdx.x * GPC + ((tid & ~31) / G);
    const int64_t n_units = units > gid_w ? (units - gid_w + NG - 1) / NG : 0;
    const bool need_pos = a.causal || a.mask;
    const uint64_t pol = policy_evict_first();

    // stride between a group's units, split once: D = NG*RPG rows
    const int64_t D = NG * RPG;
    int64_t dq = 0, dhh = 0, db = 0;
    if (need_pos) split_row(D, cols, heads, a.dcols, a.dheads, dq, dhh, db);

    Cursor ci, cc;  // issue cursor (K-1 units ahead) and compute cursor
    if (need_pos) {
        cursor_split(cc, gid * RPG, cols, heads, a.dcols, a.dheads);
    } else {
        cc.r = gid * RPG;
        cc.q = cc.h = cc.b = 0;
    }
    ci = cc;

    // prologue: K-1 units in flight
#pragma unroll
    for (int p = 0; p < K - 1; ++p) {
        if (p < n_units) fwd_issue<T, G, NV, RPG, ALIGNED, PG::SLOTS>(a, ci, p, need_pos, gl, tid, sbuf, pol);
        cp_async_commit();
        if (need_pos) cursor_step(ci, D, dq, dhh, db, cols, heads); else ci.r += D;
    }

    for (int64_t it = 0; it < n_units; ++it) {
        if (it + K - 1 < n_units)
            fwd_issue<T, G, NV, RPG, ALIGNED, PG::SLOTS>(a, ci, (int)((it + K - 1) % K), need_pos, gl, tid, sbuf, pol);
        cp_async_commit();
        if (need_pos) cursor_step(ci, D, dq, dhh, db, cols, heads); else ci.r += D;
        const int stage = (int)(it % K);

        // positions of this unit's rows; the mask loads go out before the wait
        int limit[RPG], xoff[RPG], msh[RPG];
        int64_t x0[RPG], m0[RPG], mA[RPG];
        bool live[RPG];
        uint4 mr[RPG][NV], mr2[ALIGNED ? 1 : RPG][ALIGNED ? 1 : NV];
        {
            Cursor c = cc;
#pragma unroll
            for (int i = 0; i < RPG; ++i) {
                if (i > 0) {
                    if (need_pos) cursor_next(c, cols, heads); else ++c.r;
                }
                live[i] = c.r < a.rows;
                limit[i] = live[i] ? (a.causal ? (int)(c.q + 1) : (int)cols) : 0;
                x0[i] = c.r * cols;
                xoff[i] = ALIGNED ? 0 : (int)(x0[i] & (VEC - 1));
                m0[i] = c.b * a.msb + c.h * a.msh + c.q * cols;
                const int64_t Dm = m0[i] - xoff[i];
                msh[i] = ALIGNED ? 0 : (int)(Dm & (VEC - 1));
                mA[i] = Dm - msh[i];
            }
        }
#pragma unroll
        for (int i = 0; i < RPG; ++i)
#pragma unroll
            for (int k = 0; k < NV; ++k) {
                const int vi = k * G + gl;
                mr[i][k] = make_uint4(0, 0, 0, 0);
                if constexpr (!ALIGNED) mr2[i][k] = make_uint4(0, 0, 0, 0);
                if (a.mask && vi * VEC - xoff[i] < limit[i]) {
                    const int64_t mb = mA[i] + (int64_t)vi * VEC;
                    const T *mk = reinterpret_cast<const T *>(a.mask);
                    if constexpr (ALIGNED) {
                        mr[i][k] = ld_keep(mk + mb);
                    } else {
                        if (mb >= 0 && mb + (msh[i] ? 2 : 1) * VEC <= a.mask_total) {
                            mr[i][k] = ld_keep(mk + mb);
                            if (msh[i]) mr2[i][k] = ld_keep(mk + mb + VEC);
                        }
                    }
                }
            }
        cp_async_wait<K - 1>();  // this thread's copies of unit `it` have landed

        float s[RPG][NV][VEC];
        float mx[RPG];
#pragma unroll
        for (int i = 0; i < RPG; ++i) {
            mx[i] = neg_inf();
            const int64_t xb = x0[i] - xoff[i];
#pragma unroll
            for (int k = 0; k < NV; ++k) {
                const int vi = k * G + gl;
                const int j0 = vi * VEC - xoff[i];
                float xv[VEC], mv[VEC];
#pragma unroll
                for (int e = 0; e < VEC; ++e) { xv[e] = 0.f; mv[e] = 0.f; }
                if (j0 < limit[i]) {
                    if (ALIGNED || xb + (int64_t)(vi + 1) * VEC <= a.x_total) {
                        unpack<T>(sbuf[((size_t)stage * PG::SLOTS + i * NV + k) * kNT + tid], xv);
                    } else {  // last partial vector of the tensor: not staged
                        const T *xs = reinterpret_cast<const T *>(a.x) + xb;
#pragma unroll
                        for (int e = 0; e < VEC; ++e)
                            xv[e] = xb + vi * VEC + e < a.x_total ? to_f32<T>(xs[vi * VEC + e]) : 0.f;
                    }
                    if (a.mask) {
                        if constexpr (ALIGNED) {
                            unpack<T>(mr[i][k], mv);
                        } else {
                            const int64_t mb = mA[i] + (int64_t)vi * VEC;
                            if (mb >= 0 && mb + (msh[i] ? 2 : 1) * VEC <= a.mask_total) {
                                unpack<T>(window<VEC>(mr[i][k], mr2[i][k], msh[i]), mv);
                            } else {
                                const T *ms = reinterpret_cast<const T *>(a.mask) + m0[i];
#pragma unroll
                                for (int e = 0; e < VEC; ++e) {
                                    const int j = j0 + e;
                                    mv[e] = (j >= 0 && j < limit[i]) ? to_f32<T>(ms[j]) : 0.f;
                                }
                            }
                        }
                    }
                }
                if (j0 >= 0 && j0 + VEC <= limit[i]) {  // interior vector
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

        // exp(s - m) = 2^(s*log2e - m*log2e); the rounding of m*log2e is common
        // to the row and cancels in the normalisation
        float fac[RPG];
        __syncwarp();  // every lane of the warp takes part in the shuffles below
        if constexpr (G <= 32) {
#pragma unroll
            for (int i = 0; i < RPG; ++i) {
                mx[i] = group_max<G>(mx[i]);
                const float c = (mx[i] == neg_inf()) ? 0.f : -mx[i] * kLog2e;
                float sum = 0.f;
#pragma unroll
                for (int k = 0; k < NV; ++k)
#pragma unroll
                    for (int e = 0; e < VEC; ++e) {
                        const float t = ex2(fmaf(s[i][k][e], kLog2e, c));
                        s[i][k][e] = t;
                        sum += t;
                    }
                sum = group_sum<G>(sum);
                fac[i] = sum > 0.f ? __frcp_rn(sum) : 0.f;
            }
        } else {
            __shared__ float red_m[2][GPC][RPG][W], red_l[2][GPC][RPG][W];
            const int wg = gl >> 5, lane = tid & 31, rp = (int)(it & 1);
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
                    red_m[rp][gi][i][wg] = mw;
                    red_l[rp][gi][i][wg] = lw;
                }
            }
            named_sync(1 + gi, G);
#pragma unroll
            for (int i = 0; i < RPG; ++i) {
                float M = neg_inf();
#pragma unroll
                for (int w = 0; w < W; ++w) M = fmaxf(M, red_m[rp][gi][i][w]);
                const float Mr = (M == neg_inf()) ? 0.f : M;
                float tot = 0.f;
#pragma unroll
                for (int w = 0; w < W; ++w) {
                    const float m2 = red_m[rp][gi][i][w];
                    tot += (m2 == neg_inf()) ? 0.f : red_l[rp][gi][i][w] * ex2((m2 - Mr) * kLog2e);
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
        if (need_pos) cursor_step(cc, D, dq, dhh, db, cols, heads); else cc.r += D;
    }
    cp_async_wait<0>();
}

// ----------------------------------------------------------------- backward

// Issue this thread's cp.async copies of the y and dy vectors of a unit.
template <typename T, int G, int NV, int RPG, bool ALIGNED, int SLOTS>
__device__ __forceinline__ void bwd_issue(const BwdArgs &a, const Cursor &c0, int stage, bool need_pos, int gl, int tid,
                                          uint4 *sbuf, uint64_t pol)
{
    constexpr int VEC = Dt<T>::VEC;
    Cursor c = c0;
#pragma unroll
    for (int i = 0; i < RPG; ++i) {
        if (i > 0) {
            if (need_pos) cursor_next(c, a.cols, 1); else ++c.r;
        }
        if (c.r < a.rows) {
            const int limit = a.causal ? (int)(c.q + 1) : (int)a.cols;
            const int64_t x0 = c.r * a.cols;
            const int xoff = ALIGNED ? 0 : (int)(x0 & (VEC - 1));
            const int64_t xb = x0 - xoff;
#pragma unroll
            for (int k = 0; k < NV; ++k) {
                const int vi = k * G + gl;
                if (vi * VEC - xoff < limit && (ALIGNED || xb + (int64_t)(vi + 1) * VEC <= a.total)) {
                    const size_t s0 = (((size_t)stage * 2 + 0) * SLOTS + i * NV + k) * kNT + tid;
                    const size_t s1 = (((size_t)stage * 2 + 1) * SLOTS + i * NV + k) * kNT + tid;
                    cp_async16(&sbuf[s0], reinterpret_cast<const T *>(a.y) + xb + (int64_t)vi * VEC, pol);
                    cp_async16(&sbuf[s1], reinterpret_cast<const T *>(a.dy) + xb + (int64_t)vi * VEC, pol);
                }
            }
        }
    }
}

template <typename T, int G, int NV, int RPG, bool ALIGNED>
__global__ void __launch_bounds__(kNT, 1) bwd_pipe_kernel(const BwdArgs a, int64_t units)
{
    using PG = PipeGeo<T, NV, RPG, 2>;
    constexpr int VEC = Dt<T>::VEC;
    constexpr int K = PG::K;
    constexpr int GPC = kNT / G;
    constexpr int W = G > 32 ? G / 32 : 1;
    extern __shared__ __align__(16) uint4 sbuf[];
    const int tid = threadIdx.x;
    const int gl = tid % G, gi = tid / G;
    const int64_t cols = a.cols;
    const int64_t NG = (int64_t)gridDim.x * GPC;
    const int64_t gid = (int64_t)blockIdx.x * GPC + gi;
    const int64_t gid_w = (int64_t)blockIdx.x * GPC + ((tid & ~31) / G);  // see the forward
    const int64_t n_units = units > gid_w ? (units - gid_w + NG - 1) / NG : 0;
    const bool need_pos = a.causal;
    const uint64_t pol = policy_evict_first();
    const FastDiv one;

    const int64_t D = NG * RPG;
    int64_t dq = 0, dhh = 0, db = 0;
    if (need_pos) split_row(D, cols, 1, a.dcols, one, dq, dhh, db);
    Cursor ci, cc;
    if (need_pos) {
        cursor_split(cc, gid * RPG, cols, 1, a.dcols, one);
    } else {
        cc.r = gid * RPG;
        cc.q = cc.h = cc.b = 0;
    }
    ci = cc;

    auto slot_idx = [](int stage, int stream, int i, int k, int t) -> size_t {
        return (((size_t)stage * 2 + stream) * PG::SLOTS + i * NV + k) * kNT + t;
    };

#pragma unroll
    for (int p = 0; p < K - 1; ++p) {
        if (p < n_units) bwd_issue<T, G, NV, RPG, ALIGNED, PG::SLOTS>(a, ci, p, need_pos, gl, tid, sbuf, pol);
        cp_async_commit();
        if (need_pos) cursor_step(ci, D, dq, dhh, db, cols, 1); else ci.r += D;
    }

    for (int64_t it = 0; it < n_units; ++it) {
        if (it + K - 1 < n_units)
            bwd_issue<T, G, NV, RPG, ALIGNED, PG::SLOTS>(a, ci, (int)((it + K - 1) % K), need_pos, gl, tid, sbuf, pol);
        cp_async_commit();
        if (need_pos) cursor_step(ci, D, dq, dhh, db, cols, 1); else ci.r += D;
        const int stage = (int)(it % K);

        int limit[RPG], xoff[RPG];
        int64_t x0[RPG];
        bool live[RPG];
        {
            Cursor c = cc;
#pragma unroll
            for (int i = 0; i < RPG; ++i) {
                if (i > 0) {
                    if (need_pos) cursor_next(c, cols, 1); else ++c.r;
                }
                live[i] = c.r < a.rows;
                limit[i] = live[i] ? (a.causal ? (int)(c.q + 1) : (int)cols) : 0;
                x0[i] = c.r * cols;
                xoff[i] = ALIGNED ? 0 : (int)(x0[i] & (VEC - 1));
            }
        }
        cp_async_wait<K - 1>();

        uint4 yr[RPG][NV], gr[RPG][NV];
        float dot[RPG];
#pragma unroll
        for (int i = 0; i < RPG; ++i) {
            dot[i] = 0.f;
            const int64_t xb = x0[i] - xoff[i];
#pragma unroll
            for (int k = 0; k < NV; ++k) {
                const int vi = k * G + gl;
                const int j0 = vi * VEC - xoff[i];
                yr[i][k] = gr[i][k] = make_uint4(0, 0, 0, 0);
                if (j0 < limit[i]) {
                    if (ALIGNED || xb + (int64_t)(vi + 1) * VEC <= a.total) {
                        yr[i][k] = sbuf[slot_idx(stage, 0, i, k, tid)];
                        gr[i][k] = sbuf[slot_idx(stage, 1, i, k, tid)];
                    } else {  // last partial vector of the tensor: not staged
                        float tv[VEC], tg[VEC];
#pragma unroll
                        for (int e = 0; e < VEC; ++e) {
                            const bool in = xb + vi * VEC + e < a.total;
                            tv[e] = in ? to_f32<T>(reinterpret_cast<const T *>(a.y)[xb + vi * VEC + e]) : 0.f;
                            tg[e] = in ? to_f32<T>(reinterpret_cast<const T *>(a.dy)[xb + vi * VEC + e]) : 0.f;
                        }
                        yr[i][k] = pack<T>(tv);
                        gr[i][k] = pack<T>(tg);
                    }
                }
                float yv[VEC], gv[VEC];
                unpack<T>(yr[i][k], yv);
                unpack<T>(gr[i][k], gv);
                if (j0 >= 0 && j0 + VEC <= limit[i]) {
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
        __syncwarp();  // every lane of the warp takes part in the shuffles below
        if constexpr (G <= 32) {
#pragma unroll
            for (int i = 0; i < RPG; ++i) dot[i] = group_sum<G>(dot[i]);
        } else {
            __shared__ float red[2][GPC][RPG][W];
            const int wg = gl >> 5, lane = tid & 31, rp = (int)(it & 1);
#pragma unroll
            for (int i = 0; i < RPG; ++i) {
                const float d = group_sum<32>(dot[i]);
                if (lane == 0) red[rp][gi][i][wg] = d;
            }
            named_sync(1 + gi, G);
#pragma unroll
            for (int i = 0; i < RPG; ++i) {
                dot[i] = 0.f;
#pragma unroll
                for (int w = 0; w < W; ++w) dot[i] += red[rp][gi][i][w];
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
        if (need_pos) cursor_step(cc, D, dq, dhh, db, cols, 1); else cc.r += D;
    }
    cp_async_wait<0>();
}

// ------------------------------------------------------------------- launch

template <typename T, int G, int NV, int RPG, bool ALIGNED, bool BWD, typename Args>
cudaError_t launch_one(const Args &a, cudaStream_t st)
{
    constexpr int smem = PipeGeo<T, NV, RPG, BWD ? 2 : 1>::SMEM;
    static std::atomic<int> attr_done[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    auto kern = [] {
        if constexpr (BWD) return bwd_pipe_kernel<T, G, NV, RPG, ALIGNED>;
        else return fwd_pipe_kernel<T, G, NV, RPG, ALIGNED>;
    }();
    if (!attr_done[dev & 63].load(std::memory_order_acquire)) {  // idempotent: a race only repeats the call
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        attr_done[dev & 63].store(1, std::memory_order_release);
    }
    const int64_t units = (a.rows + RPG - 1) / RPG;
    // persistent: one CTA per SM, no more CTAs than have a unit at all
    const int64_t grid = persistent_grid(1, (units + kNT / G - 1) / (kNT / G));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kNT);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    return cudaLaunchKernelEx(&cfg, kern, a, units);
}

// Lane shapes as in the register-resident kernels (capacity G*NV vectors);
// the shared-memory ring, not registers, now bounds the bytes in flight.
template <typename T, bool ALIGNED, bool BWD, typename Args>
cudaError_t launch_t(const Args &a, cudaStream_t st)
{
    constexpr int VEC = Dt<T>::VEC;
    const int64_t need = (a.cols + VEC - 1) / VEC + (ALIGNED ? 0 : 1);
#define SMS_TRY(G, NV, RPG) \
    if (need <= (G) * (NV)) return launch_one<T, G, NV, RPG, ALIGNED, BWD>(a, st);
    SMS_TRY(4, 1, 4) SMS_TRY(4, 2, 2) SMS_TRY(4, 4, 1) SMS_TRY(8, 4, 1) SMS_TRY(16, 4, 1) SMS_TRY(32, 4, 1)
    SMS_TRY(64, 4, 1) SMS_TRY(64, 5, 1) SMS_TRY(128, 4, 1) SMS_TRY(128, 5, 1) SMS_TRY(256, 4, 1)
    SMS_TRY(256, 5, 1) SMS_TRY(512, 4, 1) SMS_TRY(512, 5, 1)
#undef SMS_TRY
    return cudaErrorNotSupported;
}

template <bool BWD, typename Args>
cudaError_t dispatch(const Args &a, int dtype, bool aligned, cudaStream_t st)
{
    switch (dtype) {
    case kF32: return aligned ? launch_t<float, true, BWD>(a, st) : launch_t<float, false, BWD>(a, st);
    case kF16: return aligned ? launch_t<__half, true, BWD>(a, st) : launch_t<__half, false, BWD>(a, st);
    case kBF16:
        return aligned ? launch_t<__nv_bfloat16, true, BWD>(a, st) : launch_t<__nv_bfloat16, false, BWD>(a, st);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace

bool pipe_fits(int64_t cols, int dtype, bool aligned)
{
    const int vec = vec_elems(dtype);
    return (cols + vec - 1) / vec + (aligned ? 0 : 1) <= 512 * 5;
}

cudaError_t launch_fwd_pipe(const FwdArgs &a, int dtype, bool aligned, cudaStream_t st)
{
    return dispatch<false>(a, dtype, aligned, st);
}

cudaError_t launch_bwd_pipe(const BwdArgs &a, int dtype, bool aligned, cudaStream_t st)
{
    return dispatch<true>(a, dtype, aligned, st);
}

}  // namespace sms
