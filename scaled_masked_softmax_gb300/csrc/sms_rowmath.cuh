// One row of the fused scaled, masked softmax held in registers by a group of
// G lanes: where the row sits, the issue of its 16-byte loads, and the
// reduction / normalisation / store (forward) or dot / gradient / store
// (backward).  Used by the persistent kernels in sms_stream.cu.
//
// The operation is the one of the page "用CUDA自定义融合Softmax算子并封装进PyTorch":
//   forward  s_j = x_j*scale + mask_j (§1.2, §2.2), s_j = -inf for j > q under
//            the causal flag (§3.1), y_j = exp(s_j - max s) / sum exp(s - max s)
//            (§2.1); a row with no finite score gives y = 0;
//   backward dx_j = (dy_j - sum_k dy_k y_k) * y_j * scale (§3.3).
//
// Arithmetic (all fp32, Blackwell instruction forms):
//   * paired elements go through the packed fp32x2 FMA / add / multiply
//     (__ffma2_rn, __fadd2_rn, __fmul2_rn: each half rounded as the scalar op);
//   * the running max takes two new scores per three-input max.f32;
//   * exp(s - m) = 2^(s*log2e - m*log2e), one FMA and one ex2.approx per
//     element; the rounding of m*log2e is common to the row and cancels in the
//     normalisation;
//   * the backward's row dot uses the mixed-precision fma.rn.f32.{f16,bf16}
//     for 16-bit data (the product of two 16-bit values is exact in fp32, so
//     this equals widening both and one fp32 FMA);
//   * dx = fma(y, (dy - dot)*scale, +0): an exact-zero product (y == 0)
//     comes out as +0.
#pragma once

#include "sms_common.cuh"
#include "sms_internal.h"

namespace sms {
namespace rowmath {

__device__ __forceinline__ float max3(float a, float b, float c)
{
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

template <typename T> __device__ __forceinline__ float dot_vec(const uint4 &y, const uint4 &g, float acc);
template <> __device__ __forceinline__ float dot_vec<float>(const uint4 &y, const uint4 &g, float acc)
{
    float2 a = make_float2(0.f, 0.f);
    a = __ffma2_rn(make_float2(__uint_as_float(y.x), __uint_as_float(y.y)),
                   make_float2(__uint_as_float(g.x), __uint_as_float(g.y)), a);
    a = __ffma2_rn(make_float2(__uint_as_float(y.z), __uint_as_float(y.w)),
                   make_float2(__uint_as_float(g.z), __uint_as_float(g.w)), a);
    return acc + (a.x + a.y);
}
template <> __device__ __forceinline__ float dot_vec<__half>(const uint4 &y, const uint4 &g, float acc)
{
    const uint32_t yw[4] = {y.x, y.y, y.z, y.w}, gw[4] = {g.x, g.y, g.z, g.w};
    float lo = 0.f, hi = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        asm("{\n\t.reg .b16 yl, yh, gl, gh;\n\t"
            "mov.b32 {yl, yh}, %2;\n\tmov.b32 {gl, gh}, %3;\n\t"
            "fma.rn.f32.f16 %0, yl, gl, %0;\n\tfma.rn.f32.f16 %1, yh, gh, %1;\n\t}"
            : "+f"(lo), "+f"(hi) : "r"(yw[i]), "r"(gw[i]));
    }
    return acc + (lo + hi);
}
template <> __device__ __forceinline__ float dot_vec<__nv_bfloat16>(const uint4 &y, const uint4 &g, float acc)
{
    const uint32_t yw[4] = {y.x, y.y, y.z, y.w}, gw[4] = {g.x, g.y, g.z, g.w};
    float lo = 0.f, hi = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        asm("{\n\t.reg .b16 yl, yh, gl, gh;\n\t"
            "mov.b32 {yl, yh}, %2;\n\tmov.b32 {gl, gh}, %3;\n\t"
            "fma.rn.f32.bf16 %0, yl, gl, %0;\n\tfma.rn.f32.bf16 %1, yh, gh, %1;\n\t}"
            : "+f"(lo), "+f"(hi) : "r"(yw[i]), "r"(gw[i]));
    }
    return acc + (lo + hi);
}

// ------------------------------------------------------------- forward ---

// Where one row's vectors and mask vectors sit (every lane of the group
// computes the same values).  Rows are walked in 16-byte vectors aligned to
// the tensor: vector vi covers row elements vi*VEC - xoff .. + VEC-1.
struct RowPos {
    int64_t xb;   // flat index of the row's first vector
    int64_t mA;   // flat mask index of the first aligned mask vector of the row
    int xoff;     // row start mod VEC
    int msh;      // mask elements to shift by (mask row misaligned relative to x)
    int limit;    // elements read: q + 1 under causal, cols otherwise, cut to the key length; 0 for a dead row
    bool live;    // r < rows (a live row with limit 0 still writes its zeros)
    bool fast;    // every vector read lies inside x and the mask: no per-vector bounds tests
};

template <int VEC, bool ALIGNED>
__device__ __forceinline__ RowPos fwd_pos(const FwdArgs &a, int64_t r)
{
    RowPos p;
    const bool live = r < a.rows;
    const int64_t x0 = r * a.cols;
    p.xoff = (ALIGNED || !live) ? 0 : (int)(x0 & (VEC - 1));  // dead row: no vector has j0 < limit = 0
    p.xb = x0 - p.xoff;
    int64_t q = 0, h = 0, b = 0;
    if (live && (a.causal || a.mask || a.lengths)) split_row(r, a.cols, a.heads, a.dcols, a.dheads, q, h, b);
    p.live = live;
    p.limit = live ? key_limit(a.lengths, b, a.cols, a.causal ? (int)(q + 1) : (int)a.cols) : 0;
    const int64_t D = b * a.msb + h * a.msh + q * a.cols - p.xoff;
    p.msh = ALIGNED ? 0 : (int)(D & (VEC - 1));
    p.mA = D - p.msh;
    if (ALIGNED) {
        p.fast = true;
    } else {
        const int64_t nv = (p.xoff + p.limit + VEC - 1) / VEC;  // vectors the row reads
        const bool xin = p.xb + nv * VEC <= a.x_total;
        const bool min_ = !a.mask || (p.mA >= 0 && p.mA + (nv + (p.msh ? 1 : 0)) * VEC <= a.mask_total);
        p.fast = xin && min_;
    }
    return p;
}

// Misaligned rows on groups of 32 or more lanes may take the contiguous lane
// mapping (CONTIG, see vec_index) and, with an additive mask, the shuffled
// realignment (SHUF): the second aligned mask vector of a slot is then not
// loaded but taken from the neighbouring lane (realign_shfl), and m2[0] is the
// one vector past the end of the warp's run, loaded by the warp's last lane.
template <int NV, bool ALIGNED, bool SHUF = false> struct FwdBuf {
    uint4 x[NV], m[NV], m2[(ALIGNED || SHUF) ? 1 : NV];
};

// Row vector held by lane gl of the group in slot k.  Slot-major (vector
// k*G + gl) except with CONTIG, where each warp of the group holds a
// contiguous run of 32*NV vectors (slot k of lane l: vector k*32 + l of the
// run), so the vector after a lane's own sits in lane l+1 or, for lane 31, in
// lane 0's next slot.  Both forms read 512 contiguous bytes per warp and slot.
template <int G, int NV, bool CONTIG>
__device__ __forceinline__ int vec_index(int k, int gl)
{
    if constexpr (CONTIG && G > 32) return (gl >> 5) * (32 * NV) + k * 32 + (gl & 31);
    else return k * G + gl;
}

// Issue every 16-byte load of row p: x, then the mask (two aligned mask
// vectors per x vector when the mask row is misaligned relative to x).  The
// per-vector bounds tests of rows at the ends of the buffers live in their
// own loop: one warp-uniform branch per row keeps them out of the common path.
template <typename T, int G, int NV, bool ALIGNED, typename M = T, bool SHUF = false, bool CONTIG = SHUF>
__device__ __forceinline__ void fwd_issue(const FwdArgs &a, const RowPos &p, int gl, FwdBuf<NV, ALIGNED, SHUF> &B)
{
    constexpr int VEC = Dt<T>::VEC;
    using MIO = MaskIO<T, M>;
    const T *xs = reinterpret_cast<const T *>(a.x) + p.xb;
    const M *mk = reinterpret_cast<const M *>(a.mask) + p.mA;
    static_assert(!SHUF || (!ALIGNED && G >= 32 && CONTIG), "shuffled realignment: misaligned rows, whole warps");
    static_assert(!CONTIG || (!ALIGNED && G >= 32), "contiguous mapping: misaligned rows, whole warps");
#pragma unroll
    for (int k = 0; k < NV; ++k) {
        B.x[k] = make_uint4(0, 0, 0, 0);
        B.m[k] = make_uint4(0, 0, 0, 0);
        if constexpr (!ALIGNED && !SHUF) B.m2[k] = make_uint4(0, 0, 0, 0);
    }
    if constexpr (SHUF) B.m2[0] = make_uint4(0, 0, 0, 0);
    if constexpr (SHUF) {
        if (!p.fast) {  // a row at an end of x or of the mask buffer: the mask is read element-wise later
#pragma unroll
            for (int k = 0; k < NV; ++k) {
                const int vi = vec_index<G, NV, CONTIG>(k, gl);
                if (vi * VEC - p.xoff < p.limit && p.xb + (int64_t)(vi + 1) * VEC <= a.x_total)
                    B.x[k] = ld_stream(xs + vi * VEC);
            }
            return;
        }
        // a misaligned mask row also needs the aligned mask vector after the
        // row's last x vector: mask vectors are read one vector further
        const int mlim = p.limit + (p.msh ? VEC : 0);
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int vi = vec_index<G, NV, CONTIG>(k, gl);
            const int j0 = vi * VEC - p.xoff;
            if (j0 < p.limit) B.x[k] = ld_stream(xs + vi * VEC);
            if (a.mask && j0 < mlim) B.m[k] = MIO::ld(mk + vi * VEC);
            if (k == NV - 1 && (gl & 31) == 31 && a.mask && p.msh && j0 < p.limit)
                B.m2[0] = MIO::ld(mk + vi * VEC + VEC);  // the vector after the warp's run
        }
        return;
    }
    if (ALIGNED || p.fast) {
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int vi = vec_index<G, NV, CONTIG>(k, gl);
            if (vi * VEC - p.xoff < p.limit) {
                B.x[k] = ld_stream(xs + vi * VEC);
                if (a.mask) {
                    B.m[k] = MIO::ld(mk + vi * VEC);
                    if constexpr (!ALIGNED) {
                        if (p.msh) B.m2[k] = MIO::ld(mk + vi * VEC + VEC);
                    }
                }
            }
        }
    } else if constexpr (!ALIGNED) {  // a row at an end of x or of the mask buffer
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int vi = vec_index<G, NV, CONTIG>(k, gl);
            if (vi * VEC - p.xoff < p.limit) {
                if (p.xb + (int64_t)(vi + 1) * VEC <= a.x_total) B.x[k] = ld_stream(xs + vi * VEC);
                if (a.mask) {
                    const int64_t mb = p.mA + (int64_t)vi * VEC;
                    if (mb >= 0 && mb + (p.msh ? 2 : 1) * VEC <= a.mask_total) {
                        B.m[k] = MIO::ld(mk + vi * VEC);
                        if (p.msh) B.m2[k] = MIO::ld(mk + vi * VEC + VEC);
                    }
                }
            }
        }
    }
}

// Realign all NV mask vectors by the row's shift: one switch per row.
template <typename MIO, int NV, int S>
__device__ __forceinline__ void realign_fixed(uint4 (&m)[NV], const uint4 (&m2)[NV])
{
#pragma unroll
    for (int k = 0; k < NV; ++k) m[k] = MIO::template win<S>(m[k], m2[k]);
}
template <typename MIO, int NV>
__device__ __forceinline__ void realign(uint4 (&m)[NV], const uint4 (&m2)[NV], int s)
{
    constexpr int VEC = MIO::VEC;
    switch (s) {
    case 0: break;
    case 1: realign_fixed<MIO, NV, 1>(m, m2); break;
    case 2: realign_fixed<MIO, NV, 2>(m, m2); break;
    case 3: realign_fixed<MIO, NV, 3>(m, m2); break;
    case 4: realign_fixed<MIO, NV, 4 % VEC>(m, m2); break;
    case 5: realign_fixed<MIO, NV, 5 % VEC>(m, m2); break;
    case 6: realign_fixed<MIO, NV, 6 % VEC>(m, m2); break;
    default: realign_fixed<MIO, NV, 7 % VEC>(m, m2); break;
    }
}

// Realignment by shuffles (FwdBuf SHUF): slot k of warp lane l takes the
// window S elements into (its own aligned mask vector, the next one), the
// next one coming from lane l+1's slot k, or for lane 31 from lane 0's slot
// k+1 (from the loaded m2[0] in the last slot).  Slots are done in order, so
// slot k+1 is still raw when lane 0 hands it over.  Whole warps only.
template <typename MIO, int NV, int S>
__device__ __forceinline__ void realign_shfl_fixed(uint4 (&m)[NV], const uint4 &ext, int lane)
{
    const int src = (lane + 1) & 31;
#pragma unroll
    for (int k = 0; k < NV; ++k) {
        const uint4 v = (k + 1 < NV && lane == 0) ? m[k + 1] : m[k];
        uint4 nx;
        nx.x = __shfl_sync(0xffffffffu, v.x, src);
        nx.y = __shfl_sync(0xffffffffu, v.y, src);
        nx.z = __shfl_sync(0xffffffffu, v.z, src);
        nx.w = __shfl_sync(0xffffffffu, v.w, src);
        if (k == NV - 1 && lane == 31) nx = ext;
        m[k] = MIO::template win<S>(m[k], nx);
    }
}
template <typename MIO, int NV>
__device__ __forceinline__ void realign_shfl(uint4 (&m)[NV], const uint4 &ext, int s, int lane)
{
    constexpr int VEC = MIO::VEC;
    switch (s) {
    case 0: break;
    case 1: realign_shfl_fixed<MIO, NV, 1>(m, ext, lane); break;
    case 2: realign_shfl_fixed<MIO, NV, 2>(m, ext, lane); break;
    case 3: realign_shfl_fixed<MIO, NV, 3>(m, ext, lane); break;
    case 4: realign_shfl_fixed<MIO, NV, 4 % VEC>(m, ext, lane); break;
    case 5: realign_shfl_fixed<MIO, NV, 5 % VEC>(m, ext, lane); break;
    case 6: realign_shfl_fixed<MIO, NV, 6 % VEC>(m, ext, lane); break;
    default: realign_shfl_fixed<MIO, NV, 7 % VEC>(m, ext, lane); break;
    }
}

// Scores s = x*scale + mask of one vector (-inf outside [0, limit)), folded
// into the running max.
template <int VEC>
__device__ __forceinline__ void score_vec(const float (&xv)[VEC], const float (&mv)[VEC], float scale, int j0,
                                          int limit, float (&s)[VEC], float &mx)
{
    if (j0 >= 0 && j0 + VEC <= limit) {  // interior vector: every element is read
        const float2 sc = make_float2(scale, scale);
#pragma unroll
        for (int e = 0; e < VEC; e += 2) {
            const float2 t = __ffma2_rn(make_float2(xv[e], xv[e + 1]), sc, make_float2(mv[e], mv[e + 1]));
            s[e] = t.x;
            s[e + 1] = t.y;
            mx = max3(mx, t.x, t.y);
        }
    } else {
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
            const int j = j0 + e;
            s[e] = (j >= 0 && j < limit) ? fmaf(xv[e], scale, mv[e]) : neg_inf();
            mx = fmaxf(mx, s[e]);
        }
    }
}

// Scores of vector slot k on the common path: every vector read lies inside
// x and the mask, and the mask is already realigned.
template <typename T, int G, int NV, bool ALIGNED, typename M = T, bool SHUF = false, bool CONTIG = SHUF>
__device__ __forceinline__ void fwd_scores(const FwdArgs &a, const RowPos &p, int gl, int k,
                                           const FwdBuf<NV, ALIGNED, SHUF> &B, float (&s)[Dt<T>::VEC], float &mx)
{
    constexpr int VEC = Dt<T>::VEC;
    float xv[VEC], mv[VEC];
    unpack<T>(B.x[k], xv);
    if (a.mask) {
        MaskIO<T, M>::unpack_m(B.m[k], mv);
    } else {
#pragma unroll
        for (int e = 0; e < VEC; ++e) mv[e] = 0.f;
    }
    score_vec<VEC>(xv, mv, a.scale, vec_index<G, NV, CONTIG>(k, gl) * VEC - p.xoff, p.limit, s, mx);
}

// Scores of vector slot k of a row at an end of x or of the mask buffer:
// partial vectors are read element by element.
template <typename T, int G, int NV, typename M = T, bool SHUF = false, bool CONTIG = SHUF>
__device__ __forceinline__ void fwd_scores_edge(const FwdArgs &a, const RowPos &p, int gl, int k,
                                                const FwdBuf<NV, false, SHUF> &B, float (&s)[Dt<T>::VEC], float &mx)
{
    constexpr int VEC = Dt<T>::VEC;
    using MIO = MaskIO<T, M>;
    const int vi = vec_index<G, NV, CONTIG>(k, gl);
    const int j0 = vi * VEC - p.xoff;
    float xv[VEC], mv[VEC];
    unpack<T>(B.x[k], xv);
#pragma unroll
    for (int e = 0; e < VEC; ++e) mv[e] = 0.f;
    const T *xs = reinterpret_cast<const T *>(a.x) + p.xb;
    const M *ms = reinterpret_cast<const M *>(a.mask) + p.mA + p.msh;  // ms[vi*VEC + e]: element j0 + e
    if (j0 < p.limit) {
        if (p.xb + (int64_t)(vi + 1) * VEC > a.x_total) {  // last partial vector of the tensor
#pragma unroll
            for (int e = 0; e < VEC; ++e)
                xv[e] = p.xb + vi * VEC + e < a.x_total ? to_f32<T>(xs[vi * VEC + e]) : 0.f;
        }
        if (a.mask) {
            const int64_t mb = p.mA + (int64_t)vi * VEC;
            if (!SHUF && mb >= 0 && mb + (p.msh ? 2 : 1) * VEC <= a.mask_total) {
                MIO::unpack_m(MIO::win_rt(B.m[k], B.m2[SHUF ? 0 : k], p.msh), mv);
            } else {  // mask vectors at the ends of the mask buffer: element loads
#pragma unroll
                for (int e = 0; e < VEC; ++e) {
                    const int j = j0 + e;
                    mv[e] = (j >= 0 && j < p.limit) ? MIO::elem(ms + vi * VEC + e) : 0.f;
                }
            }
        }
    }
    score_vec<VEC>(xv, mv, a.scale, j0, p.limit, s, mx);
}

// exp of every score against the offset c = -m*log2e (in place); returns the
// lane's partial sum.  LIVE: only the first `nslot` vector slots hold scores
// (nslot is uniform over the lane group; the other slots are left untouched).
template <int NV, int VEC, bool LIVE = false>
__device__ __forceinline__ float exp_sum(float (&s)[NV][VEC], float c, int nslot = NV)
{
    const float2 l2 = make_float2(kLog2e, kLog2e), c2 = make_float2(c, c);
    float2 acc = make_float2(0.f, 0.f);
#pragma unroll
    for (int k = 0; k < NV; ++k) {
        if (LIVE && k >= nslot) break;
#pragma unroll
        for (int e = 0; e < VEC; e += 2) {
            float2 t = __ffma2_rn(make_float2(s[k][e], s[k][e + 1]), l2, c2);
            t.x = ex2(t.x);
            t.y = ex2(t.y);
            s[k][e] = t.x;
            s[k][e + 1] = t.y;
            acc = __fadd2_rn(acc, t);
        }
    }
    return acc.x + acc.y;
}

// Group barrier of a multi-warp lane group: the whole CTA (bar == 0, every
// thread of the CTA calls it equally often) or named barrier `bar` over the
// G threads of the group.
template <int G> __device__ __forceinline__ void group_barrier(int bar)
{
    if (bar == 0) __syncthreads();
    else named_sync(bar, G);
}

// From the scores s (the lane's running max mx) to the exponentials (in s)
// and the row's normalisation factor, merged over the group of G lanes.
// LIVE: only the first nslot slots hold scores (see exp_sum).
template <int G, int NV, int VEC, bool LIVE = false>
__device__ __forceinline__ float fwd_norm(float (&s)[NV][VEC], float mx, int gl, int gi,
                                          float (*red_m)[G > 32 ? G / 32 : 1], float (*red_l)[G > 32 ? G / 32 : 1],
                                          int bar, int nslot = NV)
{
    constexpr int W = G > 32 ? G / 32 : 1;
    if constexpr (G <= 32) {
        mx = group_max<G>(mx);
        const float c = (mx == neg_inf()) ? 0.f : -mx * kLog2e;  // fully masked row: every term 0
        const float sum = group_sum<G>(exp_sum<NV, VEC, LIVE>(s, c, nslot));
        return sum > 0.f ? __frcp_rn(sum) : 0.f;
    } else {
        // each lane exponentiates against its own max; warps merge (max, sum)
        // pairs, the group's warps merge theirs through shared memory
        const int wg = gl >> 5, lane = threadIdx.x & 31;
        const float c = (mx == neg_inf()) ? 0.f : -mx * kLog2e;
        const float lt = exp_sum<NV, VEC, LIVE>(s, c, nslot);
        const float mw = group_max<32>(mx);
        const float mwr = (mw == neg_inf()) ? 0.f : mw;
        const float lw = group_sum<32>(mx == neg_inf() ? 0.f : lt * ex2((mx - mwr) * kLog2e));
        if (lane == 0) {
            red_m[gi][wg] = mw;
            red_l[gi][wg] = lw;
        }
        group_barrier<G>(bar);
        float mg = neg_inf();
#pragma unroll
        for (int w = 0; w < W; ++w) mg = fmaxf(mg, red_m[gi][w]);
        const float Mr = (mg == neg_inf()) ? 0.f : mg;
        float tot = 0.f;
#pragma unroll
        for (int w = 0; w < W; ++w) {
            const float m2 = red_m[gi][w];
            tot += (m2 == neg_inf()) ? 0.f : red_l[gi][w] * ex2((m2 - Mr) * kLog2e);
        }
        const float inv = tot > 0.f ? __frcp_rn(tot) : 0.f;
        return (mx == neg_inf()) ? 0.f : ex2((mx - Mr) * kLog2e) * inv;
    }
}

// Scores, exponentials and the row's normalisation factor: s holds the
// exponentials on return.  red_m / red_l: this call's shared slots
// [group][warp] (multi-warp groups only).
template <typename T, int G, int NV, bool ALIGNED, typename M = T, bool SHUF = false, bool CONTIG = SHUF>
__device__ __forceinline__ float fwd_reduce(const FwdArgs &a, const RowPos &p, int gl, int gi,
                                            FwdBuf<NV, ALIGNED, SHUF> &B, float (&s)[NV][Dt<T>::VEC],
                                            float (*red_m)[G > 32 ? G / 32 : 1], float (*red_l)[G > 32 ? G / 32 : 1],
                                            int bar)
{
    constexpr int VEC = Dt<T>::VEC;
    float mx = neg_inf();
    if (ALIGNED || p.fast) {
        if constexpr (SHUF) {
            if (a.mask) realign_shfl<MaskIO<T, M>, NV>(B.m, B.m2[0], p.msh, threadIdx.x & 31);
        } else if constexpr (!ALIGNED) {
            if (a.mask) realign<MaskIO<T, M>, NV>(B.m, B.m2, p.msh);
        }
#pragma unroll
        for (int k = 0; k < NV; ++k) fwd_scores<T, G, NV, ALIGNED, M, SHUF, CONTIG>(a, p, gl, k, B, s[k], mx);
    } else if constexpr (!ALIGNED) {
#pragma unroll
        for (int k = 0; k < NV; ++k) fwd_scores_edge<T, G, NV, M, SHUF, CONTIG>(a, p, gl, k, B, s[k], mx);
    }

    return fwd_norm<G, NV, VEC>(s, mx, gl, gi, red_m, red_l, bar);
}

// y = e * fac for every element the lane holds.
template <typename T, int G, int NV, bool ALIGNED, bool CONTIG = false>
__device__ __forceinline__ void fwd_store(const FwdArgs &a, const RowPos &p, int gl, const float (&s)[NV][Dt<T>::VEC],
                                          float fac)
{
    constexpr int VEC = Dt<T>::VEC;
    if (!p.live) return;
    T *ys = reinterpret_cast<T *>(a.y) + p.xb;
    const int64_t cols = a.cols;
    const float2 f2 = make_float2(fac, fac);
#pragma unroll
    for (int k = 0; k < NV; ++k) {
        const int vi = vec_index<G, NV, CONTIG>(k, gl);
        const int j0 = vi * VEC - p.xoff;
        if (j0 >= cols) continue;
        float o[VEC];
#pragma unroll
        for (int e = 0; e < VEC; e += 2) {
            const float2 t = __fmul2_rn(make_float2(s[k][e], s[k][e + 1]), f2);
            o[e] = t.x;
            o[e + 1] = t.y;
        }
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

// Reduce, normalise and store row p from its loaded buffer (every thread of
// the CTA calls this equally often when G > 32 and bar == 0).
template <typename T, int G, int NV, bool ALIGNED, typename M = T, bool SHUF = false, bool CONTIG = SHUF>
__device__ __forceinline__ void fwd_finish(const FwdArgs &a, const RowPos &p, int gl, int gi,
                                           FwdBuf<NV, ALIGNED, SHUF> &B, float (*red_m)[G > 32 ? G / 32 : 1],
                                           float (*red_l)[G > 32 ? G / 32 : 1], int bar = 0)
{
    float s[NV][Dt<T>::VEC];
    const float fac = fwd_reduce<T, G, NV, ALIGNED, M, SHUF, CONTIG>(a, p, gl, gi, B, s, red_m, red_l, bar);
    fwd_store<T, G, NV, ALIGNED, CONTIG>(a, p, gl, s, fac);
}

// ------------------------------------------------------------ backward ---

struct BRowPos {
    int64_t xb;
    int xoff;
    int limit;   // elements read: q + 1 under the causal hint, cols otherwise, cut to the key length; 0 for a dead row
    bool live;   // r < rows
    bool fast;   // every vector read lies inside the tensors
};

template <int VEC, bool ALIGNED>
__device__ __forceinline__ BRowPos bwd_pos(const BwdArgs &a, int64_t r)
{
    BRowPos p;
    const bool live = r < a.rows;
    const int64_t x0 = r * a.cols;
    p.xoff = (ALIGNED || !live) ? 0 : (int)(x0 & (VEC - 1));
    p.xb = x0 - p.xoff;
    int64_t q = 0, h = 0, b = 0;
    if (live && a.lengths) split_row(r, a.cols, a.heads, a.dcols, a.dheads, q, h, b);
    else if (live && a.causal) q = row_q(r, a.cols, a.dcols);
    p.live = live;
    p.limit = live ? key_limit(a.lengths, b, a.cols, a.causal ? (int)(q + 1) : (int)a.cols) : 0;
    const int64_t nv = (p.xoff + p.limit + VEC - 1) / VEC;
    p.fast = ALIGNED || p.xb + nv * VEC <= a.total;
    return p;
}

template <int NV> struct BwdBuf {
    uint4 y[NV], g[NV];
};

template <typename T, int G, int NV, bool ALIGNED>
__device__ __forceinline__ void bwd_issue(const BwdArgs &a, const BRowPos &p, int gl, BwdBuf<NV> &B)
{
    constexpr int VEC = Dt<T>::VEC;
    const T *ys = reinterpret_cast<const T *>(a.y) + p.xb;
    const T *gs = reinterpret_cast<const T *>(a.dy) + p.xb;
#pragma unroll
    for (int k = 0; k < NV; ++k) {
        const int vi = k * G + gl;
        const int j0 = vi * VEC - p.xoff;
        B.y[k] = make_uint4(0, 0, 0, 0);
        B.g[k] = make_uint4(0, 0, 0, 0);
        if (j0 < p.limit && (p.fast || p.xb + (int64_t)(vi + 1) * VEC <= a.total)) {
            B.y[k] = ld_stream(ys + vi * VEC);
            B.g[k] = ld_stream(gs + vi * VEC);
        }
    }
}

// Vectors of the row that are not wholly inside [0, limit) (row ends and the
// causal diagonal) are handled element by element; on a row at the very end
// of the tensors, a partial last vector is read element-wise.
template <typename T, int G, int NV, bool ALIGNED>
__device__ __forceinline__ void bwd_edge(const BwdArgs &a, const BRowPos &p, int vi, float (&yv)[Dt<T>::VEC],
                                         float (&gv)[Dt<T>::VEC], const BwdBuf<NV> &B, int k)
{
    constexpr int VEC = Dt<T>::VEC;
    unpack<T>(B.y[k], yv);
    unpack<T>(B.g[k], gv);
    if (!p.fast && vi * VEC - p.xoff < p.limit && p.xb + (int64_t)(vi + 1) * VEC > a.total) {
        const T *ys = reinterpret_cast<const T *>(a.y) + p.xb;
        const T *gs = reinterpret_cast<const T *>(a.dy) + p.xb;
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
            const bool in = p.xb + vi * VEC + e < a.total;
            yv[e] = in ? to_f32<T>(ys[vi * VEC + e]) : 0.f;
            gv[e] = in ? to_f32<T>(gs[vi * VEC + e]) : 0.f;
        }
    }
}

// Row dot contribution of vector slot k: packed for interior vectors,
// element-wise (within [0, limit)) for the others.
template <typename T, int VEC>
__device__ __forceinline__ float dot_slot(const uint4 &y, const uint4 &g, int j0, int limit, float dot)
{
    if (j0 >= 0 && j0 + VEC <= limit) return dot_vec<T>(y, g, dot);
    if (j0 < limit) {
        float yv[VEC], gv[VEC];
        unpack<T>(y, yv);
        unpack<T>(g, gv);
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
            const int j = j0 + e;
            if (j >= 0 && j < limit) dot = fmaf(yv[e], gv[e], dot);
        }
    }
    return dot;
}

// The row dot sum_j y_j dy_j over the group (with the barrier rule of fwd_reduce).
template <typename T, int G, int NV, bool ALIGNED>
__device__ __forceinline__ float bwd_reduce(const BwdArgs &a, const BRowPos &p, int gl, int gi, const BwdBuf<NV> &B,
                                            float (*red)[G > 32 ? G / 32 : 1], int bar)
{
    constexpr int VEC = Dt<T>::VEC;
    constexpr int W = G > 32 ? G / 32 : 1;
    float dot = 0.f;
    if (ALIGNED || p.fast) {
#pragma unroll
        for (int k = 0; k < NV; ++k) dot = dot_slot<T, VEC>(B.y[k], B.g[k], (k * G + gl) * VEC - p.xoff, p.limit, dot);
    } else if constexpr (!ALIGNED) {  // a row at the end of the tensors: partial last vector
#pragma unroll
        for (int k = 0; k < NV; ++k) {
            const int vi = k * G + gl;
            const int j0 = vi * VEC - p.xoff;
            if (j0 < p.limit) {
                float yv[VEC], gv[VEC];
                bwd_edge<T, G, NV, ALIGNED>(a, p, vi, yv, gv, B, k);
#pragma unroll
                for (int e = 0; e < VEC; ++e) {
                    const int j = j0 + e;
                    if (j >= 0 && j < p.limit) dot = fmaf(yv[e], gv[e], dot);
                }
            }
        }
    }
    if constexpr (G <= 32) {
        return group_sum<G>(dot);
    } else {
        const int wg = gl >> 5, lane = threadIdx.x & 31;
        const float d = group_sum<32>(dot);
        if (lane == 0) red[gi][wg] = d;
        group_barrier<G>(bar);
        dot = 0.f;
#pragma unroll
        for (int w = 0; w < W; ++w) dot += red[gi][w];
        return dot;
    }
}

// dx of one vector: packed for interior vectors; element-wise for the rest
// (+0 beyond [0, limit) and where y == 0).
template <typename T, int VEC>
__device__ __forceinline__ void dx_vec(const float (&yv)[VEC], const float (&gv)[VEC], int j0, int limit, float dot,
                                       float scale, float (&o)[VEC])
{
    if (j0 >= 0 && j0 + VEC <= limit) {
        const float2 nd = make_float2(-dot, -dot), sc = make_float2(scale, scale), z = make_float2(0.f, 0.f);
#pragma unroll
        for (int e = 0; e < VEC; e += 2) {
            const float2 w = __fmul2_rn(__fadd2_rn(make_float2(gv[e], gv[e + 1]), nd), sc);
            const float2 t = __ffma2_rn(make_float2(yv[e], yv[e + 1]), w, z);  // y == 0 gives +0
            o[e] = t.x;
            o[e + 1] = t.y;
        }
    } else {
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
            const int j = j0 + e;
            const bool valid = j >= 0 && j < limit;  // beyond the diagonal (or y == 0): +0
            o[e] = (!valid || yv[e] == 0.f) ? 0.f : (gv[e] - dot) * scale * yv[e];
        }
    }
}

// dx = (dy - dot) * scale * y for every element the lane holds.
template <typename T, int G, int NV, bool ALIGNED>
__device__ __forceinline__ void bwd_store(const BwdArgs &a, const BRowPos &p, int gl, const BwdBuf<NV> &B, float dot)
{
    constexpr int VEC = Dt<T>::VEC;
    if (!p.live) return;
    T *dxs = reinterpret_cast<T *>(a.dx) + p.xb;
    const int64_t cols = a.cols;
    const bool fast = ALIGNED || p.fast;
#pragma unroll
    for (int k = 0; k < NV; ++k) {
        const int vi = k * G + gl;
        const int j0 = vi * VEC - p.xoff;
        if (j0 >= cols) continue;
        float yv[VEC], gv[VEC], o[VEC];
        if (fast) {
            unpack<T>(B.y[k], yv);
            unpack<T>(B.g[k], gv);
        } else if constexpr (!ALIGNED) {
            bwd_edge<T, G, NV, ALIGNED>(a, p, vi, yv, gv, B, k);
        }
        dx_vec<T, VEC>(yv, gv, j0, p.limit, dot, a.scale, o);
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

template <typename T, int G, int NV, bool ALIGNED>
__device__ __forceinline__ void bwd_finish(const BwdArgs &a, const BRowPos &p, int gl, int gi, BwdBuf<NV> &B,
                                           float (*red)[G > 32 ? G / 32 : 1], int bar = 0)
{
    const float dot = bwd_reduce<T, G, NV, ALIGNED>(a, p, gl, gi, B, red, bar);
    bwd_store<T, G, NV, ALIGNED>(a, p, gl, B, dot);
}

}  // namespace rowmath
}  // namespace sms
