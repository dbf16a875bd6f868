// Fused attention forward on the 5th-generation tensor cores:
//     O = softmax(Q K^T * scale + mask, causal) V,   lse = log sum exp per row
// without materialising the [S, S] score tensor (the fusion the second
// article, pnsm.cn/news/1983787, names in §4.4, with the streaming softmax
// of "从GEMM到Transformer：手写CUDA算子优化的完整路线与性能调优实践" §2.2).
//
// One CTA owns two tiles of 128 query rows of one (batch, head) and walks the
// key blocks of 128 keys:
//   * warp 0: lane 0 the TMA loads (cp.async.bulk.tensor, 128-byte swizzle)
//     of both Q tiles once and of the K blocks into a ring of slots, lane 1
//     those of the V blocks into their own ring (V slots free up later);
//   * warp 1, one lane: the MMAs, S_t(j) = Q_t K_j^T into tile t's TMEM score
//     columns, then O_t += P_t(j) V_j into its TMEM output columns; warp 1
//     also owns the TMEM allocation (512 columns: per tile 128 for S, D for O);
//   * warps 2..5 (tile 0) and 6..9 (tile 1), one query row per thread (the
//     row is the warp's TMEM lane quarter): read S_t(j) from TMEM in one go
//     and release the columns, apply scale, mask and the causal rule, keep the
//     running max m and sum l of the online softmax (m' = max(m, max_j s),
//     l' = l * 2^(m - m') + sum 2^(s - m')), write P = 2^(s - m) as 16-bit
//     values into shared memory in the MMA's swizzled layout, and rescale O in
//     TMEM when m grows by more than 8 (log2 units; in between the
//     exponentials stay below 2^8, so most blocks skip it); at the end O / l
//     is stored and lse = (m + log2 l) ln 2.
// The scores of block j+1 are issued before the products of block j, so the
// tensor cores compute one tile's work while the other tile's softmax runs
// (the two tiles' softmax phases alternate).  At D = 128 the tiles share one P
// buffer, taking turns with it, which leaves room for two V slots.
//
// Every mbarrier wait is bounded (2 s).  A role whose wait gives up records
// an error in the device word and stops; before the CTA leaves, the TMA lane
// waits (bounded) for every load it issued, the MMA lane for every MMA it
// issued, and warp 1 frees the TMEM.
#include <cuda.h>

#include <atomic>

#include "sms_attn.h"
#include "sms_attn_mask.cuh"
#include "sms_common.cuh"
#include "sms_internal.h"
#include "sms_tc.cuh"

namespace sms {
namespace {

constexpr int kBM = 128;          // query rows per tile (the MMA's M); a CTA owns two tiles
constexpr int kBN = 128;          // keys per block
constexpr int kThreads = 320;     // warps 0 (TMA), 1 (MMA), 2..5 (softmax, tile 0), 6..9 (softmax, tile 1)
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAtom = 16384;  // 128 rows x 128 bytes

template <int D> struct FwdCfg {
    // D = 128: one P buffer for both tiles (they take turns with it, see the
    // softmax below), which leaves room for two V slots.  A single V slot made
    // V_{j+1} wait for the last product with V_j and then the whole load.
    static constexpr bool SHARED_P = D == 128;
    static constexpr int NK = D == 128 ? 2 : 3;        // K slots
    static constexpr int NV = D == 128 ? 2 : 3;        // V slots
    static constexpr uint32_t TILE = (D / 64) * kAtom;  // one 128 x D tile (Q, K or V)
    static constexpr uint32_t PBUF = (kBN / 64) * kAtom;
    static constexpr uint32_t OFF_Q = 0;                // two Q tiles
    static constexpr uint32_t OFF_K = OFF_Q + 2 * TILE;
    static constexpr uint32_t OFF_V = OFF_K + NK * TILE;
    static constexpr uint32_t OFF_P = OFF_V + NV * TILE;  // P buffer(s)
    static constexpr uint32_t OFF_BAR = OFF_P + (SHARED_P ? 1 : 2) * PBUF;
    static constexpr uint32_t BAR_BYTES = 512;
    static constexpr uint32_t SMEM = OFF_BAR + BAR_BYTES + 1024;  // + alignment slack
    // TMEM columns of tile t: scores at t*256, output accumulator at t*256 + 128
    static constexpr uint32_t COL_S = 0, COL_O = kBN, TILE_COLS = 256;
};

struct FwdBars {
    uint64_t q_full;
    uint64_t k_full[3], k_empty[3], v_full[3], v_empty[3];
    uint64_t s_full[2], s_free[2];   // per tile
    uint64_t p_full[2], pv_done[2];  // per tile
    uint64_t mma_drain;
    uint32_t tmem_base;
    int abort;
};

template <typename T> struct AbFmt;
template <> struct AbFmt<__half> { static constexpr int v = 0; };
template <> struct AbFmt<__nv_bfloat16> { static constexpr int v = 1; };

__device__ __forceinline__ float rowmath_max3(float a, float b, float c)
{
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// Bounded wait on phase `parity`; on failure the CTA is flagged and the
// device word gets the code.
__device__ __forceinline__ bool wait_or_flag(uint64_t *bar, uint32_t parity, FwdBars &b, int *err)
{
    if (mbar_wait_bounded(bar, parity, &b.abort)) return true;
    *reinterpret_cast<volatile int *>(&b.abort) = 1;
    report_error(err, SMS_DEVERR_ATTN_WAIT);
    return false;
}

// Wait (bounded, whatever the abort flag says) for the copies or MMAs this
// thread itself issued, before the CTA may leave.
__device__ __forceinline__ void drain_wait(uint64_t *bar, uint32_t parity)
{
    if (mbar_try_wait(bar, parity)) return;
    const uint64_t t0 = global_ns();
    while (!mbar_try_wait(bar, parity))
        if (global_ns() - t0 > kWaitLimitNs) return;
}

// Warp-uniform bounded wait: every lane waits, the warp goes on only if all did.
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, FwdBars &b, int *err)
{
    const bool w = wait_or_flag(bar, parity, b, err);
    return __all_sync(0xffffffffu, w);
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

// The 32 mask elements of columns c0 .. c0+31 of one query row, packed
// (MaskWords): 16-byte loads where the chunk is whole and aligned, element
// loads otherwise.  Columns at or beyond S read nothing and count as kept.
template <typename T, int MK>
__device__ __forceinline__ void mask_chunk_load(const AttnArgs &a, int64_t mrow, int c0, bool row_ok,
                                                uint32_t (&w)[MaskWords<MK>::n])
{
#pragma unroll
    for (int k = 0; k < MaskWords<MK>::n; ++k) w[k] = 0u;
    if constexpr (MK != 0) {
        if (!row_ok) return;
        const int64_t base = mrow + c0;
        const int S = a.S;
        constexpr int EB = MK == 1 ? 2 : 1;  // bytes per element
        const unsigned char *mp = reinterpret_cast<const unsigned char *>(a.mask) + base * EB;
        const bool vec = (c0 + 32 <= S) && ((reinterpret_cast<uintptr_t>(mp) & 15u) == 0);
        if (vec) {
#pragma unroll
            for (int v = 0; v < 2 * EB; ++v) {
                const uint4 q = ld_keep(reinterpret_cast<const T *>(mp + 16 * v));
                w[4 * v] = q.x;
                w[4 * v + 1] = q.y;
                w[4 * v + 2] = q.z;
                w[4 * v + 3] = q.w;
            }
        } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) {
                if (c0 + e < S) {
                    if constexpr (MK == 1) w[e >> 1] |= (uint32_t)reinterpret_cast<const uint16_t *>(mp)[e] << (16 * (e & 1));
                    else w[e >> 2] |= (uint32_t)mp[e] << (8 * (e & 3));
                }
            }
        }
    }
}

// One bit per element of a packed byte-mask chunk (MaskWords<2>: 8 words of 4
// bytes): bit e set when element e is nonzero (masked).  Per word the bytes
// become 0x00 / 0xff and a multiply by 2^21 + 2^14 + 2^7 + 1 moves their top
// bits to bits 28 .. 31 (the other partial products stay below bit 24).
__device__ __forceinline__ uint32_t mask_bits(const uint32_t (&w)[8])
{
    uint32_t bits = 0u;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const uint32_t m = __vcmpne4(w[k], 0u) & 0x80808080u;
        bits |= ((m * 0x00204081u) >> 28) << (4 * k);
    }
    return bits;
}

// Scores of 32 keys col0 .. col0+31 for query row i with a byte mask given as
// bits (bit e set: key col0 + e masked): as score_chunk, masked keys -inf.
template <bool PR>
__device__ __forceinline__ float score_chunk_bits(const AttnArgs &a, float (&s)[32], uint32_t bits, int col0, int i,
                                                  float sl2, float mx)
{
#pragma unroll
    for (int e = 0; e < 32; e += 2) {
        float s0 = ((bits >> e) & 1u) ? neg_inf() : s[e] * sl2;
        float s1 = ((bits >> (e + 1)) & 1u) ? neg_inf() : s[e + 1] * sl2;
        if constexpr (PR) {
            const int col = col0 + e;
            if (col >= a.S || (a.causal && col > i)) s0 = neg_inf();
            if (col + 1 >= a.S || (a.causal && col + 1 > i)) s1 = neg_inf();
        }
        s[e] = s0;
        s[e + 1] = s1;
        mx = rowmath_max3(mx, s0, s1);
    }
    return mx;
}

// Scores of 32 keys col0 .. col0+31 for query row i, in place, in log2 units:
// S * scale * log2e (+ the mask terms m2 when MT); with PR, keys past S or
// (causal) after i get -inf.  Returns the running maximum updated with them.
template <bool PR, bool MT>
__device__ __forceinline__ float score_chunk(const AttnArgs &a, float (&s)[32], const float (&m2)[32], int col0, int i,
                                             float sl2, float mx)
{
#pragma unroll
    for (int e = 0; e < 32; e += 2) {
        float s0 = MT ? fmaf(s[e], sl2, m2[e]) : s[e] * sl2;
        float s1 = MT ? fmaf(s[e + 1], sl2, m2[e + 1]) : s[e + 1] * sl2;
        if constexpr (PR) {
            const int col = col0 + e;
            if (col >= a.S || (a.causal && col > i)) s0 = neg_inf();
            if (col + 1 >= a.S || (a.causal && col + 1 > i)) s1 = neg_inf();
        }
        s[e] = s0;
        s[e + 1] = s1;
        mx = rowmath_max3(mx, s0, s1);
    }
    return mx;
}

template <typename T, int D, int MK>
__global__ void __launch_bounds__(kThreads, 1)
attn_fwd_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                const __grid_constant__ CUtensorMap tmv, const AttnArgs a)
{
    using C = FwdCfg<D>;
    constexpr int NK = C::NK, NV = C::NV;
    constexpr uint32_t IDESC_QK = tc::idesc_f16(AbFmt<T>::v, 0, kBM, kBN);
    constexpr uint32_t IDESC_PV = tc::idesc_f16(AbFmt<T>::v, 1, kBM, D);

    extern __shared__ unsigned char smem_raw[];
    // 1024-byte alignment of the shared-memory address (the swizzle atoms)
    const uint32_t raw = static_cast<uint32_t>(__cvta_generic_to_shared(smem_raw));
    unsigned char *smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    FwdBars &b = *reinterpret_cast<FwdBars *>(smem + C::OFF_BAR);
    const uint32_t s_base = static_cast<uint32_t>(__cvta_generic_to_shared(smem));

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int BH = a.B * a.H;
    const int npair = (a.S + 2 * kBM - 1) / (2 * kBM);
    const int pr = npair - 1 - (int)(blockIdx.x / (unsigned)BH);  // heaviest causal pairs first, every head
    const int bh = (int)(blockIdx.x % (unsigned)BH);
    const int q0 = pr * 2 * kBM;  // tile t covers query rows q0 + t*128 .. + 127
    const int nkv_all = (a.S + kBN - 1) / kBN;
    int nt[2];  // key blocks tile t reads
#pragma unroll
    for (int t = 0; t < 2; ++t)
        nt[t] = a.causal ? min(nkv_all, (q0 + t * kBM + kBM - 1) / kBN + 1) : nkv_all;
    const int nmax = max(nt[0], nt[1]);

    if (threadIdx.x == 0) {
        mbar_init(&b.q_full, 1);
        for (int s = 0; s < 3; ++s) {
            mbar_init(&b.k_full[s], 1);
            mbar_init(&b.k_empty[s], 1);
            mbar_init(&b.v_full[s], 1);
            mbar_init(&b.v_empty[s], 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&b.s_full[s], 1);
            mbar_init(&b.s_free[s], kBM);
            mbar_init(&b.p_full[s], kBM);
            mbar_init(&b.pv_done[s], 1);
        }
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
        // lane 0: both Q tiles, then the K blocks; lane 1: the V blocks (their
        // slots free up later than the K slots, so they get their own lane)
        if (lane == 0) {
            tc::prefetch_tmap(&tmq);
            tc::prefetch_tmap(&tmk);
            mbar_arrive_expect_tx(&b.q_full, 2 * C::TILE);
#pragma unroll
            for (int t = 0; t < 2; ++t)
#pragma unroll
                for (int at = 0; at < D / 64; ++at)
                    tc::tma_load_3d(smem + C::OFF_Q + t * C::TILE + at * kAtom, &tmq, at * 64, q0 + t * kBM, bh,
                                    &b.q_full);
            int armed = 0;
            for (int j = 0; j < nmax; ++j) {
                const int st = j % NK;
                if (j >= NK && !wait_or_flag(&b.k_empty[st], (uint32_t)((j / NK - 1) & 1), b, a.err)) break;
                if (*reinterpret_cast<volatile int *>(&b.abort)) break;
                mbar_arrive_expect_tx(&b.k_full[st], C::TILE);
#pragma unroll
                for (int at = 0; at < D / 64; ++at)
                    tc::tma_load_3d(smem + C::OFF_K + st * C::TILE + at * kAtom, &tmk, at * 64, j * kBN, bh, &b.k_full[st]);
                armed = j + 1;
            }
            drain_wait(&b.q_full, 0);
            for (int j = (armed > NK ? armed - NK : 0); j < armed; ++j) drain_wait(&b.k_full[j % NK], (uint32_t)((j / NK) & 1));
        } else if (lane == 1) {
            tc::prefetch_tmap(&tmv);
            int armed = 0;
            for (int j = 0; j < nmax; ++j) {
                const int st = j % NV;
                if (j >= NV && !wait_or_flag(&b.v_empty[st], (uint32_t)((j / NV - 1) & 1), b, a.err)) break;
                if (*reinterpret_cast<volatile int *>(&b.abort)) break;
                mbar_arrive_expect_tx(&b.v_full[st], C::TILE);
#pragma unroll
                for (int at = 0; at < D / 64; ++at)
                    tc::tma_load_3d(smem + C::OFF_V + st * C::TILE + at * kAtom, &tmv, at * 64, j * kBN, bh, &b.v_full[st]);
                armed = j + 1;
            }
            for (int j = (armed > NV ? armed - NV : 0); j < armed; ++j) drain_wait(&b.v_full[j % NV], (uint32_t)((j / NV) & 1));
        }
    } else if (warp == 1) {
        // ----------------------------------------------------------- MMAs ---
        // Per key block j and tile t: S_t(j) = Q_t K_j^T into tile t's score
        // columns, P_t(j) V_j into its output columns.  The scores run one block
        // ahead: while one tile's softmax works, the tensor cores compute the
        // other tile's scores and products.
        if (lane == 0) {
            bool ok = wait_or_flag(&b.q_full, 0, b, a.err);
            auto qk = [&](int t, int j) -> bool {
                const int st = j % NK;
                if (!wait_or_flag(&b.k_full[st], (uint32_t)((j / NK) & 1), b, a.err)) return false;
                if (j >= 1 && !wait_or_flag(&b.s_free[t], (uint32_t)((j - 1) & 1), b, a.err)) return false;
                tc::fence_after_sync();
                const uint32_t q_addr = s_base + C::OFF_Q + t * C::TILE, k_addr = s_base + C::OFF_K + st * C::TILE;
#pragma unroll
                for (int k = 0; k < D / 16; ++k) {
                    const uint32_t ko = (k / 4) * kAtom + (k % 4) * 32;
                    tc::mma_f16(tmem + t * C::TILE_COLS + C::COL_S, tc::desc_sw128(q_addr + ko, 16, 1024),
                                tc::desc_sw128(k_addr + ko, 16, 1024), IDESC_QK, k > 0 ? 1u : 0u);
                }
                tc::commit(&b.s_full[t]);
                if (t == 1 || j >= nt[1]) tc::commit(&b.k_empty[st]);  // the last tile that reads K_j
                return true;
            };
            auto pv = [&](int t, int j) -> bool {
                const int st = j % NV;
                if (!wait_or_flag(&b.p_full[t], (uint32_t)(j & 1), b, a.err)) return false;
                if (!wait_or_flag(&b.v_full[st], (uint32_t)((j / NV) & 1), b, a.err)) return false;
                tc::fence_after_sync();
                const uint32_t p_addr = s_base + C::OFF_P + (C::SHARED_P ? 0 : t * C::PBUF), v_addr = s_base + C::OFF_V + st * C::TILE;
#pragma unroll
                for (int k = 0; k < kBN / 16; ++k) {
                    const uint64_t da = tc::desc_sw128(p_addr + (k / 4) * kAtom + (k % 4) * 32, 16, 1024);
                    const uint64_t db = tc::desc_sw128(v_addr + k * 2048, kAtom, 1024);
                    tc::mma_f16(tmem + t * C::TILE_COLS + C::COL_O, da, db, IDESC_PV, (j > 0 || k > 0) ? 1u : 0u);
                }
                tc::commit(&b.pv_done[t]);
                if (t == 1 || j >= nt[1]) tc::commit(&b.v_empty[st]);  // the last tile that reads V_j
                return true;
            };
            for (int t = 0; ok && t < 2; ++t)
                if (nt[t] > 0 && !qk(t, 0)) ok = false;
            for (int j = 0; ok && j < nmax; ++j) {
                for (int t = 0; t < 2; ++t) {
                    if (j + 1 < nt[t] && !qk(t, j + 1)) { ok = false; break; }
                    if (j < nt[t] && !pv(t, j)) { ok = false; break; }
                }
            }
            // leave no MMA in flight
            tc::commit(&b.mma_drain);
            drain_wait(&b.mma_drain, 0);
        }
    } else {
        // -------------------------------------------------------- softmax ---
        const int t = (warp - 2) >> 2;       // tile of this warp group
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;   // query row within the tile = TMEM lane
        const int i = q0 + t * kBM + r;
        const bool row_ok = i < a.S;
        const uint32_t tl = tmem + ((uint32_t)(quarter * 32) << 16) + t * C::TILE_COLS;
        const float sl2 = a.scale * kLog2e;
        const int bidx = bh / a.H, hidx = bh - bidx * a.H;
        const int64_t mrow = (int64_t)bidx * a.msb + (int64_t)hidx * a.msh + (int64_t)i * a.S;
        const int n = nt[t];
        const int qt0 = q0 + t * kBM;
        float m_run = neg_inf(), l = 0.f;
        bool ok = true;
        unsigned char *pbuf = smem + C::OFF_P + (C::SHARED_P ? 0 : t * C::PBUF);
        for (int j = 0; j < n; ++j) {
            const int j0 = j * kBN;
            // per-element rules only where a block crosses the diagonal or the end of the keys
            const bool pred = (j0 + kBN > a.S) || (a.causal && j0 + kBN - 1 > qt0);
            // this block's mask elements, fetched while the scores are computed: a byte mask whole,
            // compressed to one bit per key (mbits[c] bit e: key j0 + 32c + e masked); an additive
            // mask's first 32 keys (its others in place: more words held ahead spilled the scores)
            uint32_t mw[MaskWords<MK>::n];
            uint32_t mbits[MK == 2 ? kBN / 32 : 1];
            if constexpr (MK == 2) {
                const uint8_t *mp = reinterpret_cast<const uint8_t *>(a.mask) + mrow + j0;
                if (row_ok && j0 + kBN <= a.S && (reinterpret_cast<uintptr_t>(mp) & 15u) == 0) {
                    // the whole 128-byte row segment: eight 16-byte loads in flight together
                    uint4 q[kBN / 16];
#pragma unroll
                    for (int v = 0; v < kBN / 16; ++v) q[v] = ld_keep(reinterpret_cast<const T *>(mp + 16 * v));
#pragma unroll
                    for (int c = 0; c < kBN / 32; ++c) {
                        const uint32_t w8[8] = {q[2 * c].x, q[2 * c].y, q[2 * c].z, q[2 * c].w,
                                                q[2 * c + 1].x, q[2 * c + 1].y, q[2 * c + 1].z, q[2 * c + 1].w};
                        mbits[c] = mask_bits(w8);
                    }
                } else {  // a row past S, the ragged end of the keys, or a row that is not 16-byte aligned
#pragma unroll
                    for (int c = 0; c < kBN / 32; ++c) {
                        mask_chunk_load<T, MK>(a, mrow, j0 + c * 32, row_ok, mw);
                        mbits[c] = mask_bits(mw);
                    }
                }
            } else {
                mask_chunk_load<T, MK>(a, mrow, j0, row_ok, mw);
            }
            if (!warp_wait(&b.s_full[t], (uint32_t)(j & 1), b, a.err)) { ok = false; break; }
            tc::fence_after_sync();
            // the whole block row in registers, then the score columns go back to the MMA
            float sv[kBN];
#pragma unroll
            for (int c = 0; c < kBN / 32; ++c) tc::tmem_ld32(tl + C::COL_S + c * 32, *reinterpret_cast<uint32_t(*)[32]>(sv + 32 * c));
            tc::tmem_wait_ld();
            tc::fence_before_sync();
            mbar_arrive(&b.s_free[t]);
            float mx = neg_inf();
#pragma unroll
            for (int c = 0; c < kBN / 32; ++c) {
                if (MK == 1 && c > 0) mask_chunk_load<T, MK>(a, mrow, j0 + c * 32, row_ok, mw);
                float(&sc)[32] = *reinterpret_cast<float(*)[32]>(sv + 32 * c);
                // no lane of the warp with a masked key in these 32 (most blocks of a key-padding mask):
                // the unmasked body, no mask terms to decode
                if constexpr (MK == 2) {
                    if (__all_sync(0xffffffffu, mbits[c] == 0u)) {
                        mx = pred ? score_chunk<true, false>(a, sc, sc, j0 + c * 32, i, sl2, mx)
                                  : score_chunk<false, false>(a, sc, sc, j0 + c * 32, i, sl2, mx);
                    } else {
                        mx = pred ? score_chunk_bits<true>(a, sc, mbits[c], j0 + c * 32, i, sl2, mx)
                                  : score_chunk_bits<false>(a, sc, mbits[c], j0 + c * 32, i, sl2, mx);
                    }
                } else if (MK == 0 || mask_none<MK>(mw)) {
                    mx = pred ? score_chunk<true, false>(a, sc, sc, j0 + c * 32, i, sl2, mx)
                              : score_chunk<false, false>(a, sc, sc, j0 + c * 32, i, sl2, mx);
                } else {
                    float m2[32];
                    mask_terms<T, MK>(mw, m2);
                    mx = pred ? score_chunk<true, true>(a, sc, m2, j0 + c * 32, i, sl2, mx)
                              : score_chunk<false, true>(a, sc, m2, j0 + c * 32, i, sl2, mx);
                }
            }
            const float m_new = fmaxf(m_run, mx);
            const bool resc = m_new > m_run + 8.f;  // false while both are -inf
            const float m_use = resc ? m_new : m_run;
            const float alpha = resc ? ex2(m_run - m_new) : 1.f;  // 0 when m_run is -inf
            const float moff = (m_use == neg_inf()) ? 0.f : m_use;
            float lsum = 0.f;
#pragma unroll
            for (int e = 0; e < kBN; ++e) {
                sv[e] = ex2(sv[e] - moff);
                lsum += sv[e];
            }
            l = l * alpha + lsum;
            // P of block j - 1 has been consumed (this tile's P buffer is free)
            // and O holds every block before j once that P V is done
            // with the shared P buffer (taken P_0(j), P_1(j), P_0(j+1), ...) also the other tile's
            // product that last read it: tile 1 writes block j once P_0(j) V_j is done (tile 0 has
            // blocks 0 .. nt[0]-1), tile 0 once P_1(j-1) V_{j-1} is.  One wait site for both.
            bool waited = true;
#pragma unroll 1
            for (int w = 0; w < (C::SHARED_P ? 2 : 1); ++w) {
                int wt = t, wj = j - 1;
                if (w == 1) {
                    wt = 1 - t;
                    wj = t == 1 ? (j < nt[0] ? j : -1) : j - 1;
                }
                if (wj >= 0 && !warp_wait(&b.pv_done[wt], (uint32_t)(wj & 1), b, a.err)) { waited = false; break; }
            }
            if (!waited) { ok = false; break; }
            tc::fence_after_sync();
#pragma unroll
            for (int c = 0; c < kBN / 32; ++c) {
                unsigned char *atom = pbuf + (c / 2) * kAtom;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    uint32_t w[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u)
                        w[u] = pack2(sv[32 * c + 8 * q + 2 * u], sv[32 * c + 8 * q + 2 * u + 1], static_cast<T *>(nullptr));
                    const uint32_t off = tc::sw128_off((uint32_t)r, (uint32_t)((c & 1) * 4 + q));
                    *reinterpret_cast<uint4 *>(atom + off) = make_uint4(w[0], w[1], w[2], w[3]);
                }
            }
            if (j >= 1 && __any_sync(0xffffffffu, resc)) {  // the running max grew: rescale O
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t o[32];
                    tc::tmem_ld32(tl + C::COL_O + c * 32, o);
                    tc::tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                    tc::tmem_st32(tl + C::COL_O + c * 32, o);
                }
                tc::tmem_wait_st();
            }
            tc::fence_async_smem();
            tc::fence_before_sync();
            mbar_arrive(&b.p_full[t]);
            m_run = m_use;
        }
        // epilogue: O / l, lse
        if (ok && n > 0) ok = warp_wait(&b.pv_done[t], (uint32_t)((n - 1) & 1), b, a.err);
        if (ok && n > 0) {
            tc::fence_after_sync();
            const float inv = l > 0.f ? 1.f / l : 0.f;
            T *orow = reinterpret_cast<T *>(a.o) + ((int64_t)bh * a.S + i) * D;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                uint32_t o[32];
                tc::tmem_ld32(tl + C::COL_O + c * 32, o);
                tc::tmem_wait_ld();
                if (row_ok) {
#pragma unroll
                    for (int v = 0; v < 4; ++v) {
                        float f[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) f[e] = __uint_as_float(o[8 * v + e]) * inv;
                        st_stream(orow + c * 32 + 8 * v, pack<T>(f));
                    }
                }
            }
            if (row_ok && a.lse)
                a.lse[(int64_t)bh * a.S + i] = l > 0.f ? (m_run + log2f(l)) * 0.6931471805599453f : neg_inf();
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

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link
// against libcuda).
using EncodeFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                              const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                              CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeFn encode_fn()
{
    static EncodeFn fn = [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            p = nullptr;
        return reinterpret_cast<EncodeFn>(p);
    }();
    return fn;
}

}  // namespace

// The tensor-map encoder is a driver call: it needs the device's context
// current in the calling thread, which the runtime only makes current on a
// thread's first call that needs it (a host thread that has launched nothing
// yet, such as an autograd worker, has none).  cudaSetDevice makes it current.
cudaError_t context_current()
{
    static thread_local int done = -1;  // the device this thread made current
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (done == dev) return cudaSuccess;
    e = cudaSetDevice(dev);
    if (e == cudaSuccess) done = dev;
    return e;
}

// [B*H, S, D] 16-bit tensor, boxes of 64 x 128 x 1, 128-byte swizzle; rows
// beyond S of a head read as zeros.
cudaError_t attn_tensor_map(CUtensorMap *m, const void *base, int dtype, int BH, int S, int D)
{
    EncodeFn fn = encode_fn();
    if (!fn) return cudaErrorNotSupported;
    const cudaError_t ce = context_current();
    if (ce != cudaSuccess) return ce;
    const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)S, (cuuint64_t)BH};
    const cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)S * D * 2};
    const cuuint32_t box[3] = {64, 128, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = fn(m, dtype == kBF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
                          const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

namespace {

template <typename T, int D, int MK>
cudaError_t launch_fwd(const AttnArgs &a, const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                       cudaStream_t st)
{
    auto kern = attn_fwd_kernel<T, D, MK>;
    constexpr uint32_t smem = FwdCfg<D>::SMEM;
    static_assert(sizeof(FwdBars) <= FwdCfg<D>::BAR_BYTES, "barrier area");
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
    cfg.gridDim = dim3((unsigned)(((a.S + 2 * kBM - 1) / (2 * kBM)) * a.B * a.H));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    return cudaLaunchKernelEx(&cfg, kern, tq, tk, tv, a);
}

template <typename T, int D>
cudaError_t launch_fwd_mk(const AttnArgs &a, const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                          cudaStream_t st)
{
    if (!a.mask) return launch_fwd<T, D, 0>(a, tq, tk, tv, st);
    if (a.mask_bool) return launch_fwd<T, D, 2>(a, tq, tk, tv, st);
    return launch_fwd<T, D, 1>(a, tq, tk, tv, st);
}

}  // namespace

cudaError_t launch_attn_fwd(const AttnArgs &a, cudaStream_t st, const char **step)
{
    const char *dummy = nullptr;
    if (!step) step = &dummy;
    alignas(64) CUtensorMap tq, tk, tv;  // the encoder needs 64-byte aligned maps
    cudaError_t e;
    const int BH = a.B * a.H;
    *step = "tensor map of q";
    if ((e = attn_tensor_map(&tq, a.q, a.dtype, BH, a.S, a.D)) != cudaSuccess) return e;
    *step = "tensor map of k";
    if ((e = attn_tensor_map(&tk, a.k, a.dtype, BH, a.S, a.D)) != cudaSuccess) return e;
    *step = "tensor map of v";
    if ((e = attn_tensor_map(&tv, a.v, a.dtype, BH, a.S, a.D)) != cudaSuccess) return e;
    *step = "forward kernel";
    if (a.dtype == kBF16) {
        return a.D == 128 ? launch_fwd_mk<__nv_bfloat16, 128>(a, tq, tk, tv, st)
                          : launch_fwd_mk<__nv_bfloat16, 64>(a, tq, tk, tv, st);
    }
    return a.D == 128 ? launch_fwd_mk<__half, 128>(a, tq, tk, tv, st) : launch_fwd_mk<__half, 64>(a, tq, tk, tv, st);
}

}  // namespace sms
