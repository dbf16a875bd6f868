// Warp-per-row kernels fed by per-warp rings of bulk copies (the TMA unit):
// the kernel template and its launchers.  Instantiated per dtype and
// direction in sms_ring_{fwd_f32,fwd_f16,fwd_bf16,bwd}.cu (compiled in
// parallel); sms_ring.cu dispatches.
//
// In the register-resident kernels the bytes a multiprocessor keeps in flight
// are bounded by registers: a lane can only have as many 16-byte loads
// outstanding as it has registers to land them in, so rows that read little
// (16-bit data, causal prefixes) leave HBM under-used.  Here every warp owns
// K shared-memory stages and one of its lanes issues the bulk copies of its
// next rows (x and the mask, or y and dy) with cp.async.bulk, completion
// counted by one mbarrier per stage.  The warp waits for its oldest stage,
// moves that row into registers, hands the stage straight back to the copy
// engine for the row K ahead, and then reduces, normalises and stores the row
// as the register kernels do (sms_rowmath.cuh).  In-flight bytes are bounded
// by shared memory (up to K rows per warp), not by registers, and the per-row
// work of issuing copies is spread over all warps (no producer warp).
//
// Rows that a bulk copy cannot take whole (a partial 16-byte vector at the
// end of x, or a mask row whose aligned span leaves the mask buffer) skip the
// copy and are read from global memory by the lanes themselves.
//
// Every mbarrier wait is bounded (2 s); a warp whose wait gives up records
// an error in the device word, stops taking rows, waits (bounded) for the
// copies it still has in flight and leaves.
#pragma once

#include <atomic>

#include <type_traits>

#include "sms_rowmath.cuh"

namespace sms {
namespace {

using namespace rowmath;

constexpr int kRingBudget = 200 * 1024;  // shared memory per CTA (one CTA per multiprocessor)
constexpr int kRingHdr = 2048;            // barriers, abort words and reduction slots

// Stage layout: A = x (or y) vectors, B = mask (or dy) vectors; B holds one
// extra vector for the realignment window of a misaligned mask row.
// MB: the stage has a B area (a forward with a mask, or any backward).
template <int G, int NV, bool MB> struct RingGeo {
    static constexpr int A_BYTES = 16 * G * NV;
    static constexpr int B_OFF = A_BYTES;
    static constexpr int B_BYTES = MB ? 16 * (G * NV + 1) : 0;
    static constexpr int STAGE = (A_BYTES + B_BYTES + 127) / 128 * 128;
};

// Lane groups (of G lanes, one row each) per CTA: as many rings of K stages
// as the shared-memory budget holds, at most 16 warps.
template <int G, int NV, int K, bool MB> constexpr int ring_groups()
{
    constexpr int byb = (kRingBudget - kRingHdr) / (K * RingGeo<G, NV, MB>::STAGE);
    constexpr int byw = 16 / (G / 32);
    return byb < 1 ? 1 : (byb > byw ? byw : byb);
}

template <int G, int NV, int K, bool MB> constexpr int ring_smem()
{
    return kRingHdr + ring_groups<G, NV, K, MB>() * K * RingGeo<G, NV, MB>::STAGE;
}

// Header: per group K full barriers, an abort word, and double-buffered
// reduction slots for multi-warp groups.
template <int K> struct RingHdr {
    uint64_t full[16][K];
    uint64_t stall;                    // test control: a barrier nothing ever arrives at
    int abort[16];
    float red_m[2][16], red_l[2][16];  // [row parity][group * W + warp]
};

__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Position of row r and whether it travels by bulk copy.
struct RingRow {
    int64_t xb, mA;
    int msh, nv;  // nv: vectors the row reads
    bool copy;
};

template <typename T, bool ALIGNED>
__device__ __forceinline__ RingRow ring_row(const FwdArgs &fa, int64_t r)
{
    constexpr int VEC = Dt<T>::VEC;
    const RowPos p = fwd_pos<VEC, ALIGNED>(fa, r);
    RingRow w;
    w.xb = p.xb; w.mA = p.mA; w.msh = p.msh;
    w.nv = (p.xoff + p.limit + VEC - 1) / VEC;
    w.copy = p.fast && p.limit > 0;
    return w;
}

template <typename T, bool ALIGNED>
__device__ __forceinline__ RingRow ring_row(const BwdArgs &ba, int64_t r)
{
    constexpr int VEC = Dt<T>::VEC;
    const BRowPos p = bwd_pos<VEC, ALIGNED>(ba, r);
    RingRow w;
    w.xb = p.xb; w.mA = p.xb; w.msh = 0;
    w.nv = (p.xoff + p.limit + VEC - 1) / VEC;
    w.copy = p.fast && p.limit > 0;
    return w;
}

// The group's issuing lane: arm the stage's barrier and issue the row's copies.
template <typename T, int G, int NV, bool MB, bool ALIGNED, bool BWD>
__device__ __forceinline__ void ring_issue(const FwdArgs &fa, const BwdArgs &ba, int64_t r, unsigned char *st,
                                           uint64_t *bar, uint64_t polA, uint64_t polB)
{
    RingRow w;
    if constexpr (BWD) w = ring_row<T, ALIGNED>(ba, r);
    else w = ring_row<T, ALIGNED>(fa, r);
    uint32_t bytesA = 0, bytesB = 0;
    if (w.copy) {
        bytesA = (uint32_t)w.nv * 16u;
        if (BWD) bytesB = bytesA;
        else if (MB) bytesB = (uint32_t)(w.nv + (w.msh ? 1 : 0)) * 16u;
    }
    mbar_arrive_expect_tx(bar, bytesA + bytesB);
    if (bytesA) {
        const T *srcA = reinterpret_cast<const T *>(BWD ? ba.y : fa.x) + w.xb;
        bulk_g2s(st, srcA, bytesA, bar, polA);
    }
    if (bytesB) {
        const T *srcB = BWD ? reinterpret_cast<const T *>(ba.dy) + w.xb : reinterpret_cast<const T *>(fa.mask) + w.mA;
        bulk_g2s(st + RingGeo<G, NV, MB>::B_OFF, srcB, bytesB, bar, polB);
    }
}

// One row per group of G = 32*WG lanes.  MB: the stages carry the mask (or
// dy); a forward without MB reads its mask, if any, from global memory, with
// M its element type (T: additive, uint8_t: boolean; staged masks are additive).
template <typename T, int G, int NV, int K, bool MB, bool ALIGNED, bool BWD, typename M>
__global__ void __launch_bounds__(ring_groups<G, NV, K, MB>() * G, 1) ring_kernel(const FwdArgs fa, const BwdArgs ba)
{
    static_assert(!MB || BWD || std::is_same<M, T>::value, "a staged mask is additive");
    constexpr int VEC = Dt<T>::VEC;
    constexpr int GPC = ring_groups<G, NV, K, MB>();
    constexpr int W = G / 32;
    using Geo = RingGeo<G, NV, MB>;
    static_assert(sizeof(RingHdr<K>) <= kRingHdr, "ring header");
    extern __shared__ __align__(128) unsigned char smem[];
    RingHdr<K> &h = *reinterpret_cast<RingHdr<K> *>(smem);
    const int gi = threadIdx.x / G, gl = threadIdx.x % G, lane = threadIdx.x & 31;
    const bool issuer = gl == 0;
    uint64_t *bars = h.full[gi];
    unsigned char *ring = smem + kRingHdr + (size_t)gi * K * Geo::STAGE;
    const int bar_id = 1 + gi;  // named barrier of the group (multi-warp groups)

    const int64_t rows = BWD ? ba.rows : fa.rows;
    int *err = BWD ? ba.err : fa.err;
    const int64_t ng = (int64_t)gridDim.x * GPC;
    const int64_t r0 = (int64_t)blockIdx.x * GPC + gi;

    const uint32_t stall_ns = BWD ? ba.stall_ns : fa.stall_ns;
    if (issuer) {
        for (int s = 0; s < K; ++s) mbar_init(&bars[s], 1);
        h.abort[gi] = 0;
        if (gi == 0) mbar_init(&h.stall, 1);
        fence_mbar_init();
    }
    if (stall_ns) __syncthreads();  // the stall barrier is initialised before any group waits on it
    if constexpr (W > 1) named_sync(bar_id, G);
    else __syncwarp();
    volatile int *abort_flag = &h.abort[gi];

    const uint64_t polA = policy_evict_first();
    const uint64_t polB = BWD ? polA : policy_evict_normal();

    // prologue: the group's first K rows
    if (issuer) {
        for (int s = 0; s < K; ++s) {
            const int64_t r = r0 + s * ng;
            if (r >= rows) break;
            ring_issue<T, G, NV, MB, ALIGNED, BWD>(fa, ba, r, ring + s * Geo::STAGE, &bars[s], polA, polB);
        }
    }

    int64_t i = 0;
    bool failed = false;
    for (int64_t r = r0; r < rows; r += ng, ++i) {
        const int s = (int)(i % K);
        const uint32_t par = (uint32_t)((i / K) & 1);
        unsigned char *st = ring + s * Geo::STAGE;
        // a warp whose wait gave up reads nothing, flags the group, and still
        // takes part in the group barrier; the group then leaves together
        // (test control: the first wait is one on the stall barrier, which never completes)
        const bool ok = __all_sync(0xffffffffu, (stall_ns && i == 0)
                                                    ? mbar_wait_bounded(&h.stall, 0, abort_flag, stall_ns)
                                                    : mbar_wait_bounded(&bars[s], par, abort_flag));
        if (!ok && lane == 0) {
            *abort_flag = 1;
            report_error(err, SMS_DEVERR_RING_WAIT);
        }
        const int64_t rn = r + K * ng;  // the row this stage takes next
        const int rp = (int)(i & 1);   // reduction slots of this row
        if constexpr (BWD) {
            const BRowPos p = bwd_pos<VEC, ALIGNED>(ba, r);
            BwdBuf<NV> B;
            if (ok && p.fast && p.limit > 0) {
                const uint4 *A4 = reinterpret_cast<const uint4 *>(st);
                const uint4 *B4 = reinterpret_cast<const uint4 *>(st + Geo::B_OFF);
#pragma unroll
                for (int k = 0; k < NV; ++k) {
                    const int vi = k * G + gl;
                    B.y[k] = make_uint4(0, 0, 0, 0);
                    B.g[k] = make_uint4(0, 0, 0, 0);
                    if (vi * VEC - p.xoff < p.limit) {
                        B.y[k] = A4[vi];
                        B.g[k] = B4[vi];
                    }
                }
            } else {
                bwd_issue<T, G, NV, ALIGNED>(ba, p, gl, B);
            }
            fence_proxy_async_smem();
            if constexpr (W == 1) {
                __syncwarp();
                if (issuer && rn < rows && !*abort_flag)
                    ring_issue<T, G, NV, MB, ALIGNED, BWD>(fa, ba, rn, st, &bars[s], polA, polB);
            }
            const float dot = bwd_reduce<T, G, NV, ALIGNED>(ba, p, gl, gi, B, reinterpret_cast<float(*)[W]>(h.red_m[rp]),
                                                            bar_id);
            if (W == 1 ? !ok : *abort_flag != 0) { failed = true; break; }  // group-uniform: after the barrier
            if constexpr (W > 1) {
                if (issuer && rn < rows) ring_issue<T, G, NV, MB, ALIGNED, BWD>(fa, ba, rn, st, &bars[s], polA, polB);
            }
            bwd_store<T, G, NV, ALIGNED>(ba, p, gl, B, dot);
        } else if constexpr (ALIGNED) {
            // Only the vector slots that hold kept elements (j < limit: the
            // causal prefix, the key length) are read, scored and
            // exponentiated; slot k is live for the whole group when
            // k < nslot.  The rest of the row is stored as zeros.  A row
            // whose wait gave up reads nothing (nslot = 0).
            const RowPos p = fwd_pos<VEC, true>(fa, r);
            const int nvl = ok ? (p.limit + VEC - 1) / VEC : 0;  // vectors holding kept elements
            const int nslot = (nvl + G - 1) / G;
            const uint4 *A4 = reinterpret_cast<const uint4 *>(st);
            const uint4 *M4 = reinterpret_cast<const uint4 *>(st + Geo::B_OFF);
            uint4 mreg[MB ? 1 : NV];
            if constexpr (!MB) {
                if (fa.mask) {  // a mask shared by many rows: read through L2 by the lanes, all loads first
                    const M *mk = reinterpret_cast<const M *>(fa.mask) + p.mA;
#pragma unroll
                    for (int k = 0; k < NV; ++k) {
                        if (k >= nslot) break;
                        const int vi = k * G + gl;
                        mreg[k] = vi < nvl ? MaskIO<T, M>::ld(mk + vi * VEC) : make_uint4(0, 0, 0, 0);
                    }
                }
            }
            float sc[NV][VEC];
            float mx = neg_inf();
#pragma unroll
            for (int k = 0; k < NV; ++k) {
                if (k >= nslot) break;
                const int vi = k * G + gl;
                float xv[VEC], mv[VEC];
                unpack<T>(A4[vi], xv);  // beyond nvl: stale stage bytes, every score there is -inf
                if (fa.mask) {
                    MaskIO<T, M>::unpack_m(MB ? M4[vi] : mreg[MB ? 0 : k], mv);
                } else {
#pragma unroll
                    for (int e = 0; e < VEC; ++e) mv[e] = 0.f;
                }
                score_vec<VEC>(xv, mv, fa.scale, vi * VEC, p.limit, sc[k], mx);
            }
            fence_proxy_async_smem();
            if constexpr (W == 1) {
                __syncwarp();
                if (issuer && rn < rows && !*abort_flag)
                    ring_issue<T, G, NV, MB, ALIGNED, BWD>(fa, ba, rn, st, &bars[s], polA, polB);
            }
            const float fac = fwd_norm<G, NV, VEC, true>(sc, mx, gl, gi, reinterpret_cast<float(*)[W]>(h.red_m[rp]),
                                                         reinterpret_cast<float(*)[W]>(h.red_l[rp]), bar_id, nslot);
            if (W == 1 ? !ok : *abort_flag != 0) { failed = true; break; }  // group-uniform: after the barrier
            if constexpr (W > 1) {
                if (issuer && rn < rows) ring_issue<T, G, NV, MB, ALIGNED, BWD>(fa, ba, rn, st, &bars[s], polA, polB);
            }
            T *ys = reinterpret_cast<T *>(fa.y) + p.xb;
            const int nvrow = (int)(fa.cols / VEC);
            const float2 f2 = make_float2(fac, fac);
#pragma unroll
            for (int k = 0; k < NV; ++k) {
                const int vi = k * G + gl;
                if (k * G >= nvrow) break;
                if (vi >= nvrow) continue;
                uint4 v = make_uint4(0, 0, 0, 0);
                if (k < nslot) {
                    float o[VEC];
#pragma unroll
                    for (int e = 0; e < VEC; e += 2) {
                        const float2 t = __fmul2_rn(make_float2(sc[k][e], sc[k][e + 1]), f2);
                        o[e] = t.x;
                        o[e + 1] = t.y;
                    }
                    v = pack<T>(o);
                }
                st_stream(ys + vi * VEC, v);
            }
        } else {
            const RowPos p = fwd_pos<VEC, ALIGNED>(fa, r);
            FwdBuf<NV, ALIGNED> B;
            if (ok && p.fast && p.limit > 0) {
                const uint4 *A4 = reinterpret_cast<const uint4 *>(st);
                const uint4 *M4 = reinterpret_cast<const uint4 *>(st + Geo::B_OFF);
                const M *mk = reinterpret_cast<const M *>(fa.mask) + p.mA;
#pragma unroll
                for (int k = 0; k < NV; ++k) {
                    const int vi = k * G + gl;
                    B.x[k] = make_uint4(0, 0, 0, 0);
                    B.m[k] = make_uint4(0, 0, 0, 0);
                    if constexpr (!ALIGNED) B.m2[k] = make_uint4(0, 0, 0, 0);
                    if (vi * VEC - p.xoff < p.limit) {
                        B.x[k] = A4[vi];
                        if constexpr (MB) {
                            B.m[k] = M4[vi];
                            if constexpr (!ALIGNED) {
                                if (p.msh) B.m2[k] = M4[vi + 1];
                            }
                        } else if (fa.mask) {  // a mask shared by many rows: read through L2 by the lanes
                            B.m[k] = MaskIO<T, M>::ld(mk + vi * VEC);
                            if constexpr (!ALIGNED) {
                                if (p.msh) B.m2[k] = MaskIO<T, M>::ld(mk + vi * VEC + VEC);
                            }
                        }
                    }
                }
            } else {
                fwd_issue<T, G, NV, ALIGNED, M>(fa, p, gl, B);
            }
            fence_proxy_async_smem();
            if constexpr (W == 1) {
                __syncwarp();
                if (issuer && rn < rows && !*abort_flag)
                    ring_issue<T, G, NV, MB, ALIGNED, BWD>(fa, ba, rn, st, &bars[s], polA, polB);
            }
            float sc[NV][VEC];
            const float fac = fwd_reduce<T, G, NV, ALIGNED, M>(fa, p, gl, gi, B, sc, reinterpret_cast<float(*)[W]>(h.red_m[rp]),
                                                            reinterpret_cast<float(*)[W]>(h.red_l[rp]), bar_id);
            if (W == 1 ? !ok : *abort_flag != 0) { failed = true; break; }  // group-uniform: after the barrier
            if constexpr (W > 1) {
                if (issuer && rn < rows) ring_issue<T, G, NV, MB, ALIGNED, BWD>(fa, ba, rn, st, &bars[s], polA, polB);
            }
            fwd_store<T, G, NV, ALIGNED>(fa, p, gl, sc, fac);
        }
    }
    if (failed && issuer) {
        // stop with no copy in flight: wait (bounded) for the failed stage and
        // every stage armed after it
        for (int64_t j = i; j < i + K; ++j) {
            const int64_t r = r0 + j * ng;
            if (r >= rows) break;
            const int s = (int)(j % K);
            const uint32_t par = (uint32_t)((j / K) & 1);
            if (!mbar_try_wait(&bars[s], par)) {
                const uint64_t t0 = global_ns();
                while (!mbar_try_wait(&bars[s], par))
                    if (global_ns() - t0 > kWaitLimitNs) break;
            }
        }
    }
}

template <typename T, int G, int NV, int K, bool MB, bool ALIGNED, bool BWD, typename M>
cudaError_t launch_ring(const FwdArgs &fa, const BwdArgs &ba, cudaStream_t st)
{
    constexpr int smem = ring_smem<G, NV, K, MB>();
    constexpr int GPC = ring_groups<G, NV, K, MB>();
    auto kern = ring_kernel<T, G, NV, K, MB, ALIGNED, BWD, M>;
    static thread_local bool attr_done[64];  // per device and host thread: the shared-memory limit has been raised
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (!attr_done[dev & 63]) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        attr_done[dev & 63] = true;
    }
    const int64_t rows = BWD ? ba.rows : fa.rows;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)persistent_grid(1, (rows + GPC - 1) / GPC));
    cfg.blockDim = dim3(GPC * G);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    return cudaLaunchKernelEx(&cfg, kern, fa, ba);
}

constexpr int kStages = 3;

// Rows of up to 2048 vectors: one warp with 1, 2, 4 or 8 vectors per lane,
// then groups of 2 to 8 warps with 6 or 8 (the 6-vector groups keep rows
// just past a power of two, 4099 say, from doubling their stage and group).
template <typename T, bool MB, bool ALIGNED, bool BWD, typename M = T>
cudaError_t launch_t(const FwdArgs &fa, const BwdArgs &ba, cudaStream_t st)
{
    constexpr int VEC = Dt<T>::VEC;
    const int64_t cols = BWD ? ba.cols : fa.cols;
    const int64_t need = (cols + VEC - 1) / VEC + (ALIGNED ? 0 : 1);
#define SMS_RING(G, NV) \
    if (need <= (G) * (NV)) return launch_ring<T, G, NV, kStages, MB, ALIGNED, BWD, M>(fa, ba, st);
    SMS_RING(32, 1) SMS_RING(32, 2) SMS_RING(32, 4) SMS_RING(32, 8) SMS_RING(64, 8) SMS_RING(96, 6)
    SMS_RING(128, 8) SMS_RING(192, 6) SMS_RING(256, 8)
#undef SMS_RING
    return cudaErrorNotSupported;
}

// A mask at least a quarter the size of x is read about once per use (rows
// of different heads or batches do not share it): it travels through the
// stages with x.  A smaller mask is shared by many rows and is served by L2;
// the lanes read it directly and the stages hold x alone (twice the groups).
// A boolean mask (a quarter or half of x's bytes per element) is always read
// by the lanes.
inline bool stage_mask(const FwdArgs &fa) { return fa.mask && !fa.mask_bool && fa.mask_total * 4 >= fa.x_total; }

template <typename T, bool BWD>
cudaError_t launch_dt(const FwdArgs &fa, const BwdArgs &ba, bool aligned, cudaStream_t st)
{
    if constexpr (BWD) {
        return aligned ? launch_t<T, true, true, true>(fa, ba, st) : launch_t<T, true, false, true>(fa, ba, st);
    } else {
        if (fa.mask_bool)
            return aligned ? launch_t<T, false, true, false, uint8_t>(fa, ba, st)
                           : launch_t<T, false, false, false, uint8_t>(fa, ba, st);
        if (stage_mask(fa))
            return aligned ? launch_t<T, true, true, false>(fa, ba, st) : launch_t<T, true, false, false>(fa, ba, st);
        return aligned ? launch_t<T, false, true, false>(fa, ba, st) : launch_t<T, false, false, false>(fa, ba, st);
    }
}

}  // namespace

// One translation unit per dtype (forward) and one for the backward.
cudaError_t ring_fwd_f32(const FwdArgs &a, bool aligned, cudaStream_t st);
cudaError_t ring_fwd_f16(const FwdArgs &a, bool aligned, cudaStream_t st);
cudaError_t ring_fwd_bf16(const FwdArgs &a, bool aligned, cudaStream_t st);
cudaError_t ring_bwd_any(const BwdArgs &a, int dtype, bool aligned, cudaStream_t st);

}  // namespace sms
