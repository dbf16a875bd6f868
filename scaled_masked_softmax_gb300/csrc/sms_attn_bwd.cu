// Fused attention backward on the 5th-generation tensor cores: the gradient
// of O = softmax(Q K^T * scale + mask, causal) V by the chain rule through
// the three steps (the forward's §4.4 / §2.2 fusion, differentiated with
// the softmax Jacobian of "用CUDA自定义融合Softmax算子并封装进PyTorch" §3.3):
//     P     = exp(Q K^T * scale + mask - lse)     (recomputed, never stored)
//     dV    = P^T dO,          dP = dO V^T
//     delta = rowsum(dO * O)   (= rowsum(P * dP))
//     dS    = scale * P * (dP - delta)
//     dQ    = dS K,            dK = dS^T Q
//
// Three kernels on the caller's stream:
//   1. attn_bwd_pre: delta per query row into the workspace, and the fp32 dQ
//      accumulator in the workspace cleared;
//   2. attn_bwd_kernel: one CTA per (batch, head, block of 128 keys) walks the
//      query blocks (those at or after its keys under causal).  Per block:
//        S^T = K Q^T and dP^T = V dO^T on tcgen05 into TMEM (keys in lanes);
//        256 threads (two per key) form P^T and dS^T as 16-bit values in
//        shared memory in the MMA's swizzled layout;
//        dV += P^T dO and dK += dS^T Q accumulate in TMEM; dQ_blk = dS K goes
//        to TMEM (reusing the dP^T columns); the same threads, now one query
//        row each, copy it into shared memory (the P^T / dS^T area, which the
//        products have finished with), and one thread hands the tile to the
//        TMA unit as bulk adds into the fp32 accumulator (two groups, in the
//        order the next block's stores reuse the area), which run while the
//        next block is computed.
//      At the end dK and dV leave TMEM once, rounded to the 16-bit dtype;
//   3. attn_bwd_post: dQ = the accumulator rounded to the 16-bit dtype.
// Roles: warp 0 one lane issues the TMA loads (K and V once; dO and Q of each
// query block through a ring of tile slots, so that they arrive a block
// ahead), warp 1 one lane the MMAs (and owns TMEM), warps 2..9 the
// element-wise work.  The next block's S^T product is issued before this
// block's dQ has left TMEM (they use different columns), so it overlaps the
// dQ copy.  Every mbarrier wait is bounded (2 s) as in the forward.
#include <cuda.h>

#include <atomic>
#include <type_traits>

#include "sms_attn.h"
#include "sms_attn_mask.cuh"
#include "sms_common.cuh"
#include "sms_internal.h"
#include "sms_tc.cuh"

namespace sms {

cudaError_t attn_tensor_map(CUtensorMap *m, const void *base, int dtype, int BH, int S, int D);

namespace {

constexpr int kBM = 128;          // keys per CTA (the MMA's M for S^T, dP^T, dV, dK)
constexpr int kBN = kAttnBwdQueryBlock;  // queries per block (128)
constexpr int kThreads = 320;     // warps 0 (TMA), 1 (MMA), 2..9 (element-wise: two warps per TMEM lane quarter)
constexpr int kMath = 256;
constexpr int kHeadGroup = 4;     // heads whose CTAs are scheduled together
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAtom = 16384;

template <int D> struct BwdCfg {
    // dO and Q tiles of the query blocks in order (dO(n), Q(n), dO(n+1), ...)
    // through a ring of NSLOT slots
    static constexpr int NSLOT = D == 128 ? 3 : 4;
    static constexpr uint32_t TILE = (D / 64) * kAtom;    // 128 x D
    static constexpr uint32_t SQ = 2 * kAtom;             // 128 x 128 (P^T, dS^T)
    static constexpr uint32_t OFF_K = 0;
    static constexpr uint32_t OFF_V = OFF_K + TILE;
    static constexpr uint32_t OFF_R = OFF_V + TILE;
    static constexpr uint32_t OFF_P = OFF_R + NSLOT * TILE;
    static constexpr uint32_t OFF_DS = OFF_P + SQ;
    static constexpr uint32_t OFF_LSE = OFF_DS + SQ;       // 128 floats: lse * log2e (+inf: fully masked)
    static constexpr uint32_t OFF_DEL = OFF_LSE + 512;     // 128 floats: delta
    static constexpr uint32_t OFF_BAR = OFF_DEL + 512;
    static constexpr uint32_t BAR_BYTES = 512;
    static constexpr uint32_t SMEM = OFF_BAR + BAR_BYTES + 1024;
    static constexpr uint32_t COL_S = 0, COL_DP = 128, COL_DV = 256, COL_DK = 256 + D, COL_DQ = 128;
    // one block's dQ in fp32, staged over P^T and dS^T: element (query r, column c)
    // at byte ((c / 4) * 128 + r) * 16 + (c % 4) * 4, the accumulator's tile layout.
    // Piece p (columns 32p .. 32p+31, 16 KB at p * 16 KB) overlays atom p % 2 of
    // P^T (p < 2) or dS^T (p >= 2)
    static constexpr uint32_t DQ_BYTES = kBN * D * 4;
    static constexpr int DQ_PIECES = D / 32;
    static_assert(DQ_BYTES <= 2 * SQ && OFF_DS == OFF_P + SQ, "dQ staging area");
    static_assert(SMEM <= 232448, "shared memory per CTA");
};

struct BwdBars {
    uint64_t kv_full;
    uint64_t r_full[4], r_empty[4];
    uint64_t s_full, ds_full, dq_full, dq_free, stage_free[2];
    uint64_t mma_drain;
    uint32_t tmem_base;
    int abort;
};

template <typename T> struct AbFmt;
template <> struct AbFmt<__half> { static constexpr int v = 0; };
template <> struct AbFmt<__nv_bfloat16> { static constexpr int v = 1; };

__device__ __forceinline__ bool wait_or_flag(uint64_t *bar, uint32_t parity, BwdBars &b, int *err)
{
    if (mbar_wait_bounded(bar, parity, &b.abort)) return true;
    *reinterpret_cast<volatile int *>(&b.abort) = 1;
    report_error(err, SMS_DEVERR_ATTN_WAIT);
    return false;
}

__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, BwdBars &b, int *err)
{
    const bool w = wait_or_flag(bar, parity, b, err);
    return __all_sync(0xffffffffu, w);
}

__device__ __forceinline__ void drain_wait(uint64_t *bar, uint32_t parity)
{
    if (mbar_try_wait(bar, parity)) return;
    const uint64_t t0 = global_ns();
    while (!mbar_try_wait(bar, parity))
        if (global_ns() - t0 > kWaitLimitNs) return;
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi, __half *)
{
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}
__device__ __forceinline__ uint32_t pack2(float lo, float hi, __nv_bfloat16 *)
{
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}

// Mask elements of key j for the 32 queries i0 .. i0+31 (element (i, j) at
// mbase + i*S), packed: a byte mask four per word, an additive 16-bit mask
// two per word.  Queries at or beyond S (and keys beyond S) read nothing and
// count as kept.  Loaded before the block's scores are ready, so that the
// loads' latency passes while the tensor cores compute them.
template <typename T, int MK>
__device__ __forceinline__ void mask_col_load(const AttnArgs &a, int64_t mbase, int i0, bool key_ok,
                                              uint32_t (&w)[MaskWords<MK>::n])
{
#pragma unroll
    for (int k = 0; k < MaskWords<MK>::n; ++k) w[k] = 0u;
    if constexpr (MK != 0) {
        if (!key_ok) return;
        // all 32 loads first (rows past S clamped to the last row and dropped below), so that they
        // are in flight together: element by element behind a bounds test they went one at a time
        using E = std::conditional_t<MK == 1, uint16_t, uint8_t>;
        const E *col = reinterpret_cast<const E *>(a.mask) + mbase;
        uint32_t v[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) v[e] = __ldg(col + (int64_t)min(i0 + e, a.S - 1) * a.S);
#pragma unroll
        for (int e = 0; e < 32; ++e) {
            const uint32_t x = (i0 + e < a.S) ? v[e] : 0u;
            if constexpr (MK == 1) w[e >> 1] |= x << (16 * (e & 1));
            else w[e >> 2] |= x << (8 * (e & 3));
        }
    }
}

// P^T and dS^T of one 32-query chunk c for this thread's key j (TMEM lane):
// sv / dv hold S^T and dP^T of queries c*32 .. c*32+31, s_lse their lse in
// log2 units (+inf: no kept key), s_dsc their delta * scale; pk / dk get the
// results as 16-bit pairs in query order.  PR: the chunk may hold positions
// that are masked out by position (causal diagonal, keys or queries past S).
template <typename T, int MK, bool PR>
__device__ __forceinline__ void p_ds_chunk(const AttnArgs &a, const uint32_t (&sv)[32], const uint32_t (&dv)[32],
                                           const float (&m2)[32], const float *s_lse, const float *s_dsc, int c,
                                           int i0, int j, bool key_ok, float sl2, uint32_t (&pk)[16],
                                           uint32_t (&dk)[16])
{
    const float4 *l4 = reinterpret_cast<const float4 *>(s_lse + c * 32);
    const float4 *g4 = reinterpret_cast<const float4 *>(s_dsc + c * 32);
#pragma unroll
    for (int e4 = 0; e4 < 8; ++e4) {
        const float4 L = l4[e4], G = g4[e4];
        const float lq[4] = {L.x, L.y, L.z, L.w}, gq[4] = {G.x, G.y, G.z, G.w};
        float p[4], ds[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int e = 4 * e4 + u;
            // log2 of P: S * scale * log2e + mask - lse (one rounding without a mask)
            float x = MK == 0 ? fmaf(__uint_as_float(sv[e]), sl2, -lq[u])
                              : fmaf(__uint_as_float(sv[e]), sl2, m2[e]) - lq[u];
            if constexpr (PR) {
                const int i = i0 + c * 32 + e;
                if (!key_ok || i >= a.S || (a.causal && j > i)) x = neg_inf();
            }
            p[u] = ex2(x);
            ds[u] = p[u] * fmaf(__uint_as_float(dv[e]), a.scale, -gq[u]);  // scale * P * (dP - delta)
        }
        pk[2 * e4] = pack2(p[0], p[1], static_cast<T *>(nullptr));
        pk[2 * e4 + 1] = pack2(p[2], p[3], static_cast<T *>(nullptr));
        dk[2 * e4] = pack2(ds[0], ds[1], static_cast<T *>(nullptr));
        dk[2 * e4 + 1] = pack2(ds[2], ds[3], static_cast<T *>(nullptr));
    }
}

template <typename T, int D, int MK>
__global__ void __launch_bounds__(kThreads, 1)
attn_bwd_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                const __grid_constant__ CUtensorMap tmv, const __grid_constant__ CUtensorMap tmdo, const AttnArgs a)
{
    using C = BwdCfg<D>;
    constexpr int NS = C::NSLOT;
    constexpr int FMT = AbFmt<T>::v;
    constexpr uint32_t IDESC_SQ = tc::idesc_f16(FMT, 0, kBM, kBN);          // S^T, dP^T: K-major A and B
    constexpr uint32_t IDESC_ACC = tc::idesc_f16(FMT, 1, kBM, D);           // dV, dK: K-major A, MN-major B
    constexpr uint32_t IDESC_DQ = tc::idesc_f16(FMT, 1, kBN, D, 1);         // dQ: MN-major A and B

    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw = static_cast<uint32_t>(__cvta_generic_to_shared(smem_raw));
    unsigned char *smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    BwdBars &b = *reinterpret_cast<BwdBars *>(smem + C::OFF_BAR);
    const uint32_t s_base = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
    float *s_lse = reinterpret_cast<float *>(smem + C::OFF_LSE);
    float *s_dsc = reinterpret_cast<float *>(smem + C::OFF_DEL);  // delta * scale per query of the block

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int BH = a.B * a.H;
    const int nkb = (a.S + kBM - 1) / kBM;
    // CTAs in groups of kHeadGroup heads, so that the CTAs running at one time
    // share few heads: the group's fp32 dQ accumulator, Q and dO stay in L2.
    // Inside a group, key blocks in order (under causal, key block 0 sees every
    // query block and the last only its own: heaviest first), then heads.
    const int grp = (int)(blockIdx.x / (unsigned)(kHeadGroup * nkb));
    const int gsz = min(kHeadGroup, BH - grp * kHeadGroup);
    const int rk = (int)(blockIdx.x - (unsigned)(grp * kHeadGroup * nkb));
    const int kb = a.causal ? rk / gsz : nkb - 1 - rk / gsz;
    const int bh = grp * kHeadGroup + rk % gsz;
    const int j0 = kb * kBM;
    const int nqb = (a.S + kBN - 1) / kBN;
    const int qb0 = a.causal ? j0 / kBN : 0;  // query blocks before the keys see none of them
    const int npair = nqb - qb0;

    if (threadIdx.x == 0) {
        mbar_init(&b.kv_full, 1);
        for (int s = 0; s < NS; ++s) {
            mbar_init(&b.r_full[s], 1);
            mbar_init(&b.r_empty[s], 1);
        }
        mbar_init(&b.s_full, 1);
        mbar_init(&b.ds_full, kMath / 32);   // one arrival per element-wise warp
        mbar_init(&b.dq_full, 1);
        mbar_init(&b.dq_free, kMath / 32);
        mbar_init(&b.stage_free[0], 1);
        mbar_init(&b.stage_free[1], 1);
        mbar_init(&b.mma_drain, 1);
        b.abort = 0;
        fence_mbar_init();
    }
    if (warp == 1) tc::tmem_alloc(&b.tmem_base, kTmemCols);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = b.tmem_base;

    if (warp == 0) {
        // ------------------------------------------------------ TMA loads ---
        if (lane == 0) {
            tc::prefetch_tmap(&tmq);
            tc::prefetch_tmap(&tmk);
            tc::prefetch_tmap(&tmv);
            tc::prefetch_tmap(&tmdo);
            mbar_arrive_expect_tx(&b.kv_full, 2 * C::TILE);
#pragma unroll
            for (int at = 0; at < D / 64; ++at) {
                tc::tma_load_3d(smem + C::OFF_K + at * kAtom, &tmk, at * 64, j0, bh, &b.kv_full);
                tc::tma_load_3d(smem + C::OFF_V + at * kAtom, &tmv, at * 64, j0, bh, &b.kv_full);
            }
            // tile u: dO (u even) or Q (u odd) of query block qb0 + u / 2, into slot u % NS
            int armed = 0;
            for (int u = 0; u < 2 * npair; ++u) {
                const int sl = u % NS, i0 = (qb0 + (u >> 1)) * kBN;
                if (u >= NS && !wait_or_flag(&b.r_empty[sl], (uint32_t)((u / NS - 1) & 1), b, a.err)) break;
                if (*reinterpret_cast<volatile int *>(&b.abort)) break;
                const CUtensorMap *m = (u & 1) ? &tmq : &tmdo;
                mbar_arrive_expect_tx(&b.r_full[sl], C::TILE);
#pragma unroll
                for (int at = 0; at < D / 64; ++at)
                    tc::tma_load_3d(smem + C::OFF_R + sl * C::TILE + at * kAtom, m, at * 64, i0, bh, &b.r_full[sl]);
                armed = u + 1;
            }
            drain_wait(&b.kv_full, 0);
            for (int u = (armed > NS ? armed - NS : 0); u < armed; ++u) drain_wait(&b.r_full[u % NS], (uint32_t)((u / NS) & 1));
        }
    } else if (warp == 1) {
        // ----------------------------------------------------------- MMAs ---
        if (lane == 0) {
            bool ok = wait_or_flag(&b.kv_full, 0, b, a.err);
            const uint32_t k_addr = s_base + C::OFF_K, v_addr = s_base + C::OFF_V;
            const uint32_t p_addr = s_base + C::OFF_P, ds_addr = s_base + C::OFF_DS;
            for (int n = 0; ok && n < npair; ++n) {
                const int ud = 2 * n, uq = 2 * n + 1;  // ring tiles of dO(n) and Q(n)
                const int sd = ud % NS, sq = uq % NS;
                const uint32_t q_addr = s_base + C::OFF_R + sq * C::TILE, do_addr = s_base + C::OFF_R + sd * C::TILE;
                // S^T: its columns were read out before the previous ds_full
                if (!wait_or_flag(&b.r_full[sq], (uint32_t)((uq / NS) & 1), b, a.err)) { ok = false; break; }
                tc::fence_after_sync();
#pragma unroll
                for (int k = 0; k < D / 16; ++k) {
                    const uint32_t ko = (k / 4) * kAtom + (k % 4) * 32;
                    tc::mma_f16(tmem + C::COL_S, tc::desc_sw128(k_addr + ko, 16, 1024), tc::desc_sw128(q_addr + ko, 16, 1024),
                                IDESC_SQ, k > 0 ? 1u : 0u);
                }
                // dP^T shares its columns with the previous block's dQ: drained first
                if (!wait_or_flag(&b.r_full[sd], (uint32_t)((ud / NS) & 1), b, a.err)) { ok = false; break; }
                if (n >= 1 && !wait_or_flag(&b.dq_free, (uint32_t)((n - 1) & 1), b, a.err)) { ok = false; break; }
                tc::fence_after_sync();
#pragma unroll
                for (int k = 0; k < D / 16; ++k) {
                    const uint32_t ko = (k / 4) * kAtom + (k % 4) * 32;
                    tc::mma_f16(tmem + C::COL_DP, tc::desc_sw128(v_addr + ko, 16, 1024),
                                tc::desc_sw128(do_addr + ko, 16, 1024), IDESC_SQ, k > 0 ? 1u : 0u);
                }
                tc::commit(&b.s_full);
                if (!wait_or_flag(&b.ds_full, (uint32_t)(n & 1), b, a.err)) { ok = false; break; }
                tc::fence_after_sync();
                // K-major slice k of P^T / dS^T at (k / 4) * kAtom + (k % 4) * 32; MN-major slice of dO / Q at k * 2048
#pragma unroll
                for (int k = 0; k < kBN / 16; ++k)
                    tc::mma_f16(tmem + C::COL_DV, tc::desc_sw128(p_addr + (k / 4) * kAtom + (k % 4) * 32, 16, 1024),
                                tc::desc_sw128(do_addr + k * 2048, kAtom, 1024), IDESC_ACC, (n > 0 || k > 0) ? 1u : 0u);
                tc::commit(&b.r_empty[sd]);
#pragma unroll
                for (int k = 0; k < kBN / 16; ++k)
                    tc::mma_f16(tmem + C::COL_DK, tc::desc_sw128(ds_addr + (k / 4) * kAtom + (k % 4) * 32, 16, 1024),
                                tc::desc_sw128(q_addr + k * 2048, kAtom, 1024), IDESC_ACC, (n > 0 || k > 0) ? 1u : 0u);
                tc::commit(&b.r_empty[sq]);
#pragma unroll
                for (int k = 0; k < kBM / 16; ++k) {
                    // dQ = dS K: A = dS (queries x keys) read MN-major from dS^T, B = K MN-major
                    tc::mma_f16(tmem + C::COL_DQ, tc::desc_sw128(ds_addr + k * 2048, kAtom, 1024),
                                tc::desc_sw128(k_addr + k * 2048, kAtom, 1024), IDESC_DQ, k > 0 ? 1u : 0u);
                }
                tc::commit(&b.dq_full);
            }
            tc::commit(&b.mma_drain);
            drain_wait(&b.mma_drain, 0);
        }
    } else {
        // --------------------------------------------- element-wise work ---
        // two warps per TMEM lane quarter: `half` takes half of the columns
        // (queries of S^T / dP^T, head-dim columns of dQ, dK, dV)
        const int quarter = warp & 3;
        const int half = (warp - 2) >> 2;
        const int mt = threadIdx.x - 64;   // 0 .. 255
        const int t = quarter * 32 + lane;  // TMEM lane: key j0 + t (S^T, dP^T, dV, dK) or query i0 + t (dQ)
        const int j = j0 + t;
        const bool key_ok = j < a.S;
        const uint32_t tl = tmem + ((uint32_t)(quarter * 32) << 16);
        const float sl2 = a.scale * kLog2e;
        const int bidx = bh / a.H, hidx = bh - bidx * a.H;
        const int64_t mbase = (int64_t)bidx * a.msb + (int64_t)hidx * a.msh + j;
        const int64_t row0 = (int64_t)bh * a.S;
        bool ok = true;
        // lse and delta of a query block: loaded one block ahead by threads
        // mt < 128 (one query each), so the global loads are off the block's path
        float lse_n = 0.f, del_n = 0.f;
        auto fetch = [&](int n) {
            const int i = (qb0 + n) * kBN + mt;
            lse_n = neg_inf();
            del_n = 0.f;
            if (mt < kBN && n < npair && i < a.S) {
                lse_n = a.lse_in[row0 + i];
                del_n = a.delta[row0 + i];
            }
        };
        fetch(0);
        for (int n = 0; n < npair; ++n) {
            const int i0 = (qb0 + n) * kBN;
            // this block's lse (log2 units; +inf where the row has no kept key, or beyond S) and delta
            // (every thread finished reading the previous block's at the dQ barrier below)
            if (mt < kBN) {
                s_lse[mt] = (lse_n == neg_inf()) ? __int_as_float(0x7f800000) : lse_n * kLog2e;
                s_dsc[mt] = del_n * a.scale;
            }
            named_sync(1, kMath);
            fetch(n + 1);
            const bool pred = !key_ok || (i0 + kBN > a.S) || (a.causal && j0 + kBM - 1 > i0);
            // this block's mask elements (both chunks), fetched while S^T and dP^T are computed
            uint32_t mw[kBN / 64][MaskWords<MK>::n];
#pragma unroll
            for (int cc = 0; cc < kBN / 64; ++cc) mask_col_load<T, MK>(a, mbase, i0 + (cc * 2 + half) * 32, key_ok, mw[cc]);
            if (!warp_wait(&b.s_full, (uint32_t)(n & 1), b, a.err)) { ok = false; break; }
            tc::fence_after_sync();
            bool staged = true;
#pragma unroll
            for (int cc = 0; cc < kBN / 64; ++cc) {
                // chunk cc of both warps of a lane quarter covers queries 64cc .. 64cc+63: atom cc
                // of P^T and of dS^T, the ones the dQ pieces of bulk group cc overlay
                const int c = cc * 2 + half;
                float m2[32];
                mask_terms<T, MK>(mw[cc], m2);
                uint32_t sv[32], dv[32];
                tc::tmem_ld32(tl + C::COL_S + c * 32, sv);
                tc::tmem_ld32(tl + C::COL_DP + c * 32, dv);
                tc::tmem_wait_ld();
                uint32_t pk[16], dk[16];
                // a chunk in which no lane of the warp has a masked element (most blocks of a key-padding
                // mask) takes the unmasked body
                if (MK == 0 || mask_none<MK>(mw[cc])) {
                    if (pred) p_ds_chunk<T, 0, true>(a, sv, dv, m2, s_lse, s_dsc, c, i0, j, key_ok, sl2, pk, dk);
                    else p_ds_chunk<T, 0, false>(a, sv, dv, m2, s_lse, s_dsc, c, i0, j, key_ok, sl2, pk, dk);
                } else {
                    if (pred) p_ds_chunk<T, MK, true>(a, sv, dv, m2, s_lse, s_dsc, c, i0, j, key_ok, sl2, pk, dk);
                    else p_ds_chunk<T, MK, false>(a, sv, dv, m2, s_lse, s_dsc, c, i0, j, key_ok, sl2, pk, dk);
                }
                if (n > 0) {
                    // the previous block's dQ pieces over atom cc have been read by their bulk adds
                    // (group cc) before the stores here; the waits overlap the chunks' arithmetic
                    if (mt == 0) {
                        if (cc == 0) tc::bulk_wait_read_but_last();
                        else tc::bulk_wait_read();
                        mbar_arrive(&b.stage_free[cc]);
                    }
                    __syncwarp();
                    if (!warp_wait(&b.stage_free[cc], (uint32_t)((n - 1) & 1), b, a.err)) { staged = false; break; }
                }
                unsigned char *pa = smem + C::OFF_P + (c / 2) * kAtom;
                unsigned char *da = smem + C::OFF_DS + (c / 2) * kAtom;
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    const uint32_t off = tc::sw128_off((uint32_t)t, (uint32_t)((c & 1) * 4 + q4));
                    *reinterpret_cast<uint4 *>(pa + off) = make_uint4(pk[4 * q4], pk[4 * q4 + 1], pk[4 * q4 + 2], pk[4 * q4 + 3]);
                    *reinterpret_cast<uint4 *>(da + off) = make_uint4(dk[4 * q4], dk[4 * q4 + 1], dk[4 * q4 + 2], dk[4 * q4 + 3]);
                }
            }
            if (!staged) { ok = false; break; }
            tc::fence_before_sync();
            tc::fence_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&b.ds_full);
            // this block's dQ (lane t = query i0 + t) out of TMEM, staged in shared memory in the
            // accumulator's tile layout (a warp's 32 queries fill 512 contiguous bytes per 4 columns)
            if (!warp_wait(&b.dq_full, (uint32_t)(n & 1), b, a.err)) { ok = false; break; }
            tc::fence_after_sync();
            uint32_t v[D / 64][32];
#pragma unroll
            for (int cc = 0; cc < D / 64; ++cc) tc::tmem_ld32(tl + C::COL_DQ + (half * (D / 64) + cc) * 32, v[cc]);
            tc::tmem_wait_ld();
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&b.dq_free);
#pragma unroll
            for (int cc = 0; cc < D / 64; ++cc) {
                const int c = half * (D / 64) + cc;  // this warp's 32-column chunks of dQ
#pragma unroll
                for (int g = 0; g < 8; ++g)
                    *reinterpret_cast<uint4 *>(smem + C::OFF_P + ((c * 8 + g) * kBN + t) * 16) =
                        make_uint4(v[cc][4 * g], v[cc][4 * g + 1], v[cc][4 * g + 2], v[cc][4 * g + 3]);
            }
            tc::fence_async_smem();
            named_sync(2, kMath);
            // the tile added into the accumulator by the TMA unit: the pieces over atom 0 of
            // P^T / dS^T as one bulk group, then those over atom 1 (the next block writes atom 0 first)
            if (mt == 0) {
                float *g = a.dq_acc + ((int64_t)bh * nqb + qb0 + n) * (kBN * D);
#pragma unroll
                for (int grp = 0; grp < 2; ++grp) {
#pragma unroll
                    for (int p = grp; p < C::DQ_PIECES; p += 2)
                        tc::bulk_reduce_add_f32(g + p * (kBN * 32), s_base + C::OFF_P + p * kAtom, kAtom);
                    tc::bulk_commit();
                }
            }
        }
        // the last bulk adds have finished before the CTA's shared memory is released
        if (mt == 0) tc::bulk_wait_all();
        if (ok) {
            // dK and dV of this CTA's keys (the last dq_full covered every MMA)
            tc::fence_after_sync();
            T *dkr = reinterpret_cast<T *>(a.dk) + (row0 + j) * D;
            T *dvr = reinterpret_cast<T *>(a.dv) + (row0 + j) * D;
#pragma unroll
            for (int cc = 0; cc < D / 64; ++cc) {
                const int c = half * (D / 64) + cc;
                uint32_t kv[32], vv[32];
                tc::tmem_ld32(tl + C::COL_DK + c * 32, kv);
                tc::tmem_ld32(tl + C::COL_DV + c * 32, vv);
                tc::tmem_wait_ld();
                if (key_ok) {
#pragma unroll
                    for (int w = 0; w < 4; ++w) {
                        float fk[8], fv[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            fk[e] = __uint_as_float(kv[8 * w + e]);
                            fv[e] = __uint_as_float(vv[8 * w + e]);
                        }
                        st_stream(dkr + c * 32 + 8 * w, pack<T>(fk));
                        st_stream(dvr + c * 32 + 8 * w, pack<T>(fv));
                    }
                }
            }
        }
    }

    tc::fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, kTmemCols);
    }
}

// The dQ accumulator cleared (D floats per warp, acc_rows warps), and
// delta[r] = sum_d dO[r, d] * O[r, d] (fp32) by warp r for each of the `rows`
// query rows.
template <typename T, int D>
__global__ void __launch_bounds__(256) attn_bwd_pre(const AttnArgs a, int64_t rows, int64_t acc_rows)
{
    const int64_t r = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (r >= acc_rows) return;
    float4 *acc = reinterpret_cast<float4 *>(a.dq_acc + r * D);
    for (int e = lane; e < D / 4; e += 32) acc[e] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (r >= rows) return;
    const T *o = reinterpret_cast<const T *>(a.o_in) + r * D;
    const T *g = reinterpret_cast<const T *>(a.dout) + r * D;
    float s = 0.f;
#pragma unroll
    for (int e = lane; e < D; e += 32) s = fmaf(to_f32<T>(o[e]), to_f32<T>(g[e]), s);
    s = group_sum<32>(s);
    if (lane == 0) a.delta[r] = s;
}

// dQ = the fp32 accumulator rounded to T: each thread 8 columns of one query
// row, a warp 4 rows x 8 column groups (64-byte runs read from the tile
// layout, 128-byte runs written to dQ's rows).
template <typename T, int D>
__global__ void __launch_bounds__(256) attn_bwd_post(const AttnArgs a, int64_t units)
{
    const int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (g >= units) return;
    constexpr int per_tile = kBN * D / 8;
    const int64_t tile = g / per_tile;
    const int w = (int)(g - tile * per_tile), wi = w >> 5, lane = w & 31;
    const int r = (wi / (D / 64)) * 4 + (lane & 3);       // query within the block
    const int cg = (wi % (D / 64)) * 8 + (lane >> 2);     // 8-column group
    const int nqb = (a.S + kBN - 1) / kBN;
    const int64_t bh = tile / nqb;
    const int i = (int)(tile - bh * nqb) * kBN + r;
    if (i >= a.S) return;
    const float4 *acc = reinterpret_cast<const float4 *>(a.dq_acc) + tile * (kBN * D / 4);
    const float4 u = acc[(2 * cg) * kBN + r], v = acc[(2 * cg + 1) * kBN + r];
    const float f[8] = {u.x, u.y, u.z, u.w, v.x, v.y, v.z, v.w};
    st_stream(reinterpret_cast<T *>(a.dq) + (bh * a.S + i) * D + cg * 8, pack<T>(f));
}

template <typename T, int D, int MK>
cudaError_t launch_main(const AttnArgs &a, const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                        const CUtensorMap &tdo, cudaStream_t st)
{
    auto kern = attn_bwd_kernel<T, D, MK>;
    constexpr uint32_t smem = BwdCfg<D>::SMEM;
    static_assert(sizeof(BwdBars) <= BwdCfg<D>::BAR_BYTES, "barrier area");
    static thread_local bool attr_done[64];  // per device and host thread: the shared-memory limit has been raised
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (!attr_done[dev & 63]) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        attr_done[dev & 63] = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(((a.S + kBM - 1) / kBM) * a.B * a.H));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    return cudaLaunchKernelEx(&cfg, kern, tq, tk, tv, tdo, a);
}

template <typename T, int D>
cudaError_t launch_all(const AttnArgs &a, const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                       const CUtensorMap &tdo, cudaStream_t st, const char **step)
{
    const int64_t rows = (int64_t)a.B * a.H * a.S;
    const int64_t acc_rows = attn_bwd_acc_rows(a.B, a.H, a.S);
    *step = "delta kernel";
    attn_bwd_pre<T, D><<<(unsigned)((acc_rows + 7) / 8), 256, 0, st>>>(a, rows, acc_rows);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    *step = "main backward kernel";
    if (!a.mask) e = launch_main<T, D, 0>(a, tq, tk, tv, tdo, st);
    else if (a.mask_bool) e = launch_main<T, D, 2>(a, tq, tk, tv, tdo, st);
    else e = launch_main<T, D, 1>(a, tq, tk, tv, tdo, st);
    if (e != cudaSuccess) return e;
    *step = "dQ kernel";
    const int64_t units = acc_rows * D / 8;
    attn_bwd_post<T, D><<<(unsigned)((units + 255) / 256), 256, 0, st>>>(a, units);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_bwd(const AttnArgs &a, cudaStream_t st, const char **step)
{
    const char *dummy = nullptr;
    if (!step) step = &dummy;
    alignas(64) CUtensorMap tq, tk, tv, tdo;  // the encoder needs 64-byte aligned maps
    cudaError_t e;
    const int BH = a.B * a.H;
    *step = "tensor map of q";
    if ((e = attn_tensor_map(&tq, a.q, a.dtype, BH, a.S, a.D)) != cudaSuccess) return e;
    *step = "tensor map of k";
    if ((e = attn_tensor_map(&tk, a.k, a.dtype, BH, a.S, a.D)) != cudaSuccess) return e;
    *step = "tensor map of v";
    if ((e = attn_tensor_map(&tv, a.v, a.dtype, BH, a.S, a.D)) != cudaSuccess) return e;
    *step = "tensor map of d_o";
    if ((e = attn_tensor_map(&tdo, a.dout, a.dtype, BH, a.S, a.D)) != cudaSuccess) return e;
    if (a.dtype == kBF16)
        return a.D == 128 ? launch_all<__nv_bfloat16, 128>(a, tq, tk, tv, tdo, st, step)
                          : launch_all<__nv_bfloat16, 64>(a, tq, tk, tv, tdo, st, step);
    return a.D == 128 ? launch_all<__half, 128>(a, tq, tk, tv, tdo, st, step)
                      : launch_all<__half, 64>(a, tq, tk, tv, tdo, st, step);
}

}  // namespace sms
