// Persistent staged kernels: rows are streamed into shared memory by the bulk
// copy (TMA) engine and reduced by groups of warps, for rows too wide for the
// register-resident warp kernels.
//
// Prior art: the page "用CUDA自定义融合Softmax算子并封装进PyTorch" (§2.3 one block per
// row, §3.1 shared-memory row cache, §3.2 tree reductions) launched one
// 128-thread block per row, cached the scaled row in shared memory and reduced
// with log2(128) barrier rounds.  On sm_103a the idea is arranged differently:
//   * a CTA holds R independent consumer groups of WG warps; group g takes
//     every R-th row of the CTA's row sequence, so R rows are reduced at once;
//   * one producer lane feeds every group's ring of K shared-memory stages
//     with cp.async.bulk, running up to K rows (or row chunks) ahead of the
//     group, so HBM reads for later rows overlap the reductions and stores of
//     the current ones;
//   * a stage holds CH register slots of the group (a whole row when
//     CH == SLOTS, else a chunk of it) and starts with a 64-byte descriptor
//     the producer writes (row start, alignment, causal limit, mask span), so
//     consumers do no index arithmetic;
//   * each consumer thread pulls its vectors into registers and releases the
//     stage at once; the forward merges per-thread (max, sum) pairs so a row
//     needs one group barrier (none when WG == 1); exp is evaluated once per
//     element; causal positions j > q are never copied.
// Rows of any start alignment are handled: stages hold 16-byte vectors
// aligned to the tensor (x or y) and, separately, to the mask; elements a bulk
// copy cannot cover (a partial vector at the very end of a tensor) are read
// directly from global memory.
//
// Every mbarrier wait is bounded (2 s).  A warp whose wait gives up skips the
// stage, marks its group aborted, the group leaves at its next barrier, and
// the producer waits (bounded) for every copy it issued before exiting.
#pragma once

#include <atomic>
#include <type_traits>

#include "sms_common.cuh"
#include "sms_internal.h"

namespace sms {
namespace tile {
namespace {  // internal linkage: no launch state is shared with another copy of the library

constexpr int kMaxK = 16;                  // ring stages per group (upper bound)
constexpr int kSmemBudget = 200 * 1024;    // one CTA per SM

// Written by the producer at the head of every stage.
struct __align__(16) ChunkDesc {
    int64_t x0;      // flat element index of the row start
    int64_t m0;      // mask row start (elements)
    int32_t mrel;    // stage index of mask element j is j + mrel
    int32_t mcnt;    // mask elements held by the stage
    int32_t mvec;    // mask row aligned like the x row: 16-byte stage reads
    int32_t pad0;
    int32_t cx_hi;   // one past the last row vector (row-relative) held by the stage
    int32_t xoff;    // x0 mod VEC
    int32_t limit;   // elements read: q+1 under causal, else cols, cut to the key length
    int32_t nv_read; // vectors holding elements < limit
    int32_t nv_row;  // vectors holding row elements
    int32_t nchunks; // stages the row occupies
    int32_t pad1, pad2;
};
static_assert(sizeof(ChunkDesc) == 64, "descriptor is one 64-byte slot");

template <int WG, int R, int SLOTS, int CH> struct Geo {
    static constexpr int GT = WG * 32;          // threads per consumer group
    static constexpr int CT = R * GT;           // consumer threads
    static constexpr int THREADS = CT + 32;     // + one producer warp
    static constexpr int PV = CH * GT;          // 16-byte vectors of x (or y) per stage
    static constexpr int NCH = SLOTS / CH;      // stages of a full-width row
    static constexpr int A_OFF = 64;            // after the descriptor
    static constexpr int B_OFF = 64 + 16 * PV;  // mask (or dy) area: PV + 1 vectors
    static constexpr int STAGE = 64 + 16 * (2 * PV + 1);
    static_assert(SLOTS % CH == 0, "a stage holds whole slots");
};

template <int WG, int R> struct Hdr {
    uint64_t full[R][kMaxK];
    uint64_t empty[R][kMaxK];
    float red_max[R][2][WG];  // double buffered by row parity
    float red_sum[R][2][WG];
    int abort;                // any thread gave up (producer or consumer)
    int cons_abort[R];        // a warp of group g gave up (read after the group barrier)
};

template <int WG, int R> __host__ __device__ constexpr int hdr_bytes()
{
    return (int)((sizeof(Hdr<WG, R>) + 127) / 128 * 128);
}

template <int WG, int R, int SLOTS, int CH> __host__ __device__ constexpr int ring_k()
{
    return (kSmemBudget - hdr_bytes<WG, R>()) / (R * Geo<WG, R, SLOTS, CH>::STAGE) < kMaxK
               ? (kSmemBudget - hdr_bytes<WG, R>()) / (R * Geo<WG, R, SLOTS, CH>::STAGE)
               : kMaxK;
}

template <int WG, int R, int SLOTS, int CH> __host__ __device__ constexpr int smem_bytes()
{
    return hdr_bytes<WG, R>() + R * ring_k<WG, R, SLOTS, CH>() * Geo<WG, R, SLOTS, CH>::STAGE;
}

// M: the mask element type of the forward (T: additive; uint8_t: one byte per
// element, nonzero = masked).  Mask rows are staged in 16-byte vectors of
// their own alignment either way: MEPV elements per vector.
template <typename T, int WG, int R, int SLOTS, int CH, bool BWD, typename M>
__global__ void __launch_bounds__(Geo<WG, R, SLOTS, CH>::THREADS, 1)
    tile_kernel(const FwdArgs fa, const BwdArgs ba)
{
    using G = Geo<WG, R, SLOTS, CH>;
    constexpr int K = ring_k<WG, R, SLOTS, CH>();
    static_assert(K >= 2, "each group needs at least two stages");
    constexpr int VEC = Dt<T>::VEC;
    constexpr int MEPV = 16 / (int)sizeof(M);  // mask elements per 16-byte vector
    constexpr bool MBOOL = !std::is_same<M, T>::value;
    constexpr int GT = G::GT;
    extern __shared__ __align__(128) unsigned char smem[];
    Hdr<WG, R> &h = *reinterpret_cast<Hdr<WG, R> *>(smem);
    unsigned char *stages = smem + hdr_bytes<WG, R>();

    const int64_t rows = BWD ? ba.rows : fa.rows;
    const int64_t cols = BWD ? ba.cols : fa.cols;
    const int64_t total = BWD ? ba.total : fa.x_total;
    const int causal = BWD ? ba.causal : fa.causal;
    const void *srcA = BWD ? ba.y : fa.x;
    const void *srcB = BWD ? ba.dy : fa.mask;
    int *err = BWD ? ba.err : fa.err;
    const int64_t full_vecs = total / VEC;  // vectors lying wholly inside the tensor

    if (threadIdx.x == 0) {
        for (int g = 0; g < R; ++g) {
            for (int s = 0; s < K; ++s) {
                mbar_init(&h.full[g][s], 1);
                mbar_init(&h.empty[g][s], WG);
            }
            h.cons_abort[g] = 0;
        }
        h.abort = 0;
        fence_mbar_init();
    }
    __syncthreads();

    volatile int *abort_flag = &h.abort;

    if (threadIdx.x >= G::CT) {
        // ------------------------------------------------------- producer ---
        if (threadIdx.x != G::CT) return;
        const uint64_t polA = policy_evict_first();
        const uint64_t polB = BWD ? polA : policy_evict_normal();
        uint32_t issued[R], parity[R], ph[R];  // per group: stages ever issued / parity of last issue / ring phase
        int stage[R];
#pragma unroll
        for (int g = 0; g < R; ++g) { issued[g] = 0; parity[g] = 0; ph[g] = 0; stage[g] = 0; }
        bool ok = true;
        int64_t r = blockIdx.x;
        while (r < rows && ok) {
#pragma unroll
            for (int g = 0; g < R; ++g) {  // rows go to the groups in turn
                if (r < rows && ok) {
                    int64_t q = 0, hh = 0, bb = 0;
                    const int32_t *lengths = BWD ? ba.lengths : fa.lengths;
                    if (BWD) {
                        if (lengths) split_row(r, cols, ba.heads, ba.dcols, ba.dheads, q, hh, bb);
                        else if (causal) q = row_q(r, cols, ba.dcols);
                    } else if (causal || srcB || lengths) {
                        split_row(r, cols, fa.heads, fa.dcols, fa.dheads, q, hh, bb);
                    }
                    ChunkDesc d;
                    d.x0 = r * cols;
                    d.xoff = (int)(d.x0 & (VEC - 1));
                    const int64_t gbase = (d.x0 - d.xoff) / VEC;
                    d.limit = key_limit(lengths, bb, cols, causal ? (int)(q + 1) : (int)cols);
                    d.nv_read = (d.xoff + d.limit + VEC - 1) / VEC;
                    d.nv_row = (int)((d.xoff + cols + VEC - 1) / VEC);
                    // at least one stage per row, also for a row with no kept key:
                    // its consumers wait for exactly one stage
                    d.nchunks = max(1, (d.nv_read + G::PV - 1) / G::PV);
                    d.m0 = (!BWD && srcB) ? bb * fa.msb + hh * fa.msh + q * cols : 0;
                    d.mvec = ((d.m0 - d.xoff) & (VEC - 1)) == 0;
                    d.pad0 = d.pad1 = d.pad2 = 0;
                    for (int c = 0; c < d.nchunks; ++c) {
                        if (!mbar_wait_bounded(&h.empty[g][stage[g]], ph[g] ^ 1u, abort_flag)) {
                            *abort_flag = 1;
                            report_error(err, SMS_DEVERR_CTA_PRODUCER_WAIT);
                            ok = false;
                            break;
                        }
                        const int vlo = c * G::PV;
                        const int vhi = min(d.nv_read, vlo + G::PV);
                        d.cx_hi = (int)min((int64_t)vhi, full_vecs - gbase);
                        const uint32_t bytesA = d.cx_hi > vlo ? (uint32_t)(d.cx_hi - vlo) * 16u : 0u;
                        uint32_t bytesB = 0;
                        int64_t b_src = 0;
                        d.mrel = 0;
                        d.mcnt = 0;
                        if (BWD) {
                            bytesB = bytesA;
                            b_src = gbase + vlo;
                        } else if (srcB) {
                            const int64_t jlo = max(0, vlo * VEC - d.xoff);
                            const int64_t jhi = min((int64_t)d.limit, (int64_t)vhi * VEC - d.xoff);
                            const int64_t mv_lo = (d.m0 + jlo) / MEPV;
                            const int64_t cm_hi = min((d.m0 + jhi + MEPV - 1) / MEPV, fa.mask_total / MEPV);
                            d.mrel = (int)(d.m0 - mv_lo * MEPV);
                            d.mcnt = cm_hi > mv_lo ? (int)(cm_hi - mv_lo) * MEPV : 0;
                            bytesB = cm_hi > mv_lo ? (uint32_t)(cm_hi - mv_lo) * 16u : 0u;
                            b_src = mv_lo;
                        }
                        unsigned char *st = stages + (size_t)(g * K + stage[g]) * G::STAGE;
                        *reinterpret_cast<ChunkDesc *>(st) = d;  // visible to consumers through the barrier
                        uint64_t *fb = &h.full[g][stage[g]];
                        mbar_arrive_expect_tx(fb, bytesA + bytesB);
                        if (bytesA)
                            bulk_g2s(st + G::A_OFF, reinterpret_cast<const uint4 *>(srcA) + gbase + vlo, bytesA, fb,
                                     polA);
                        if (bytesB)
                            bulk_g2s(st + G::B_OFF, reinterpret_cast<const uint4 *>(srcB) + b_src, bytesB, fb, polB);
                        issued[g] |= 1u << stage[g];
                        parity[g] = (parity[g] & ~(1u << stage[g])) | (ph[g] << stage[g]);
                        if (++stage[g] == K) { stage[g] = 0; ph[g] ^= 1u; }
                    }
                    r += gridDim.x;
                }
            }
        }
        // never leave with copies in flight: wait for the last issue of every stage
#pragma unroll
        for (int g = 0; g < R; ++g)
            for (int s = 0; s < K; ++s)
                if (issued[g] & (1u << s)) {
                    const uint32_t p = (parity[g] >> s) & 1u;
                    if (!mbar_try_wait(&h.full[g][s], p)) {
                        const uint64_t t0 = global_ns();
                        while (!mbar_try_wait(&h.full[g][s], p))
                            if (global_ns() - t0 > kWaitLimitNs) { report_error(err, SMS_DEVERR_CTA_PRODUCER_WAIT); break; }
                    }
                }
        return;
    }

    // ---------------------------------------------------------- consumers ---
    const int g = threadIdx.x / GT;   // consumer group
    const int tg = threadIdx.x % GT;  // thread within the group
    const int lane = threadIdx.x & 31, wg = tg >> 5;
    int stage = 0;
    uint32_t ph = 0;
    int rp = 0;  // row parity: selects the reduction buffer
    const int64_t n_cta = rows > blockIdx.x ? (rows - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
    const int64_t my_rows = n_cta > g ? (n_cta - g + R - 1) / R : 0;

    for (int64_t it = 0; it < my_rows; ++it, rp ^= 1) {
        // forward: scores s as fp32; backward: y and dy kept as the raw 16-byte
        // vectors (half the registers for fp16/bf16), widened again for dx
        float va[BWD ? 1 : SLOTS][VEC];
        uint4 ra[BWD ? SLOTS : 1], rb[BWD ? SLOTS : 1];
        float acc = BWD ? 0.f : neg_inf();  // backward: dot; forward: running max
        int64_t x0 = 0;
        int xoff = 0, limit = 0, nv_row = 0, nchunks = 1;
        bool row_ok = true, ok = true;
        const unsigned char *st = stages;

#pragma unroll
        for (int k = 0; k < SLOTS; ++k) {
            const int c = k / CH, kk = k % CH;
            if (BWD) {
                ra[k] = make_uint4(0, 0, 0, 0);
                rb[k] = make_uint4(0, 0, 0, 0);
            } else {
#pragma unroll
                for (int e = 0; e < VEC; ++e) va[k][e] = neg_inf();
            }
            if (c < nchunks) {
                if (kk == 0) {
                    // warp-uniform outcome: a warp whose wait failed skips the
                    // stage (its descriptor may be stale)
                    ok = __all_sync(0xffffffffu, mbar_wait_bounded(&h.full[g][stage], ph, abort_flag));
                    if (!ok) {
                        row_ok = false;
                        if (lane == 0) {
                            *abort_flag = 1;
                            h.cons_abort[g] = 1;
                            report_error(err, SMS_DEVERR_CTA_CONSUMER_WAIT);
                        }
                    }
                    st = stages + (size_t)(g * K + stage) * G::STAGE;
                }
                const ChunkDesc &d = *reinterpret_cast<const ChunkDesc *>(st);
                if (k == 0 && ok) {
                    x0 = d.x0;
                    xoff = d.xoff;
                    limit = d.limit;
                    nv_row = d.nv_row;
                    nchunks = min(max(d.nchunks, 1), G::NCH);
                }
                const int vi = k * GT + tg;   // vector of the row
                const int lv = kk * GT + tg;  // vector within the stage
                const int j0 = vi * VEC - xoff;
                if (ok && vi < d.nv_read) {
                    const T *arow = reinterpret_cast<const T *>(srcA) + (x0 - xoff);
                    const int64_t gv = (x0 - xoff) / VEC + vi;
                    float a[VEC], b[VEC];
                    const bool staged = vi < d.cx_hi;  // else: last partial vector of the tensor
                    if (BWD) {
                        const T *brow = reinterpret_cast<const T *>(srcB) + (x0 - xoff);
                        if (staged) {
                            ra[k] = reinterpret_cast<const uint4 *>(st + G::A_OFF)[lv];
                            rb[k] = reinterpret_cast<const uint4 *>(st + G::B_OFF)[lv];
                        } else {
#pragma unroll
                            for (int e = 0; e < VEC; ++e) {
                                const bool in = gv * VEC + e < total;
                                a[e] = in ? to_f32<T>(arow[vi * VEC + e]) : 0.f;
                                b[e] = in ? to_f32<T>(brow[vi * VEC + e]) : 0.f;
                            }
                            ra[k] = pack<T>(a);
                            rb[k] = pack<T>(b);
                        }
                        unpack<T>(ra[k], a);
                        unpack<T>(rb[k], b);
#pragma unroll
                        for (int e = 0; e < VEC; ++e) {
                            const int j = j0 + e;
                            if (j >= 0 && j < limit) acc = fmaf(a[e], b[e], acc);
                        }
                    } else {
                        if (staged) {
                            unpack<T>(reinterpret_cast<const uint4 *>(st + G::A_OFF)[lv], a);
                        } else {
#pragma unroll
                            for (int e = 0; e < VEC; ++e)
                                a[e] = gv * VEC + e < total ? to_f32<T>(arow[vi * VEC + e]) : 0.f;
                        }
#pragma unroll
                        for (int e = 0; e < VEC; ++e) b[e] = 0.f;
                        if (srcB) {
                            using MIO = MaskIO<T, M>;
                            const M *msm = reinterpret_cast<const M *>(st + G::B_OFF);
                            const int jj = j0 + d.mrel;  // stage index of element j0
                            if (d.mvec && jj >= 0 && jj + VEC <= d.mcnt) {
                                if constexpr (MBOOL) {  // VEC bytes: one 4- or 8-byte shared load
                                    uint4 w = make_uint4(0, 0, 0, 0);
                                    if constexpr (VEC == 4) {
                                        w.x = *reinterpret_cast<const uint32_t *>(msm + jj);
                                    } else {
                                        const uint2 v = *reinterpret_cast<const uint2 *>(msm + jj);
                                        w.x = v.x;
                                        w.y = v.y;
                                    }
                                    MIO::unpack_m(w, b);
                                } else {
                                    unpack<T>(*reinterpret_cast<const uint4 *>(msm + jj), b);
                                }
                            } else {
                                const M *mrow = reinterpret_cast<const M *>(srcB) + d.m0;
#pragma unroll
                                for (int e = 0; e < VEC; ++e) {
                                    const int j = j0 + e;
                                    if (j >= 0 && j < limit) {
                                        const int idx = j + d.mrel;
                                        b[e] = idx < d.mcnt ? MIO::elem(msm + idx) : MIO::elem(mrow + j);
                                    }
                                }
                            }
                        }
#pragma unroll
                        for (int e = 0; e < VEC; ++e) {
                            const int j = j0 + e;
                            va[k][e] = (j >= 0 && j < limit) ? fmaf(a[e], fa.scale, b[e]) : neg_inf();
                            acc = fmaxf(acc, va[k][e]);
                        }
                    }
                }
                if (kk == CH - 1) {  // last slot of the stage: release it
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&h.empty[g][stage]);
                    if (++stage == K) { stage = 0; ph ^= 1u; }
                }
            }
        }

        if (BWD) {
            float dot = group_sum<32>(acc);
            if constexpr (WG > 1) {
                if (lane == 0) h.red_sum[g][rp][wg] = dot;
                named_sync(1 + g, GT);
                if (h.cons_abort[g]) break;  // uniform within the group
                dot = 0.f;
#pragma unroll
                for (int w = 0; w < WG; ++w) dot += h.red_sum[g][rp][w];
            } else {
                if (!row_ok) break;  // warp-uniform
            }
            T *orow = reinterpret_cast<T *>(ba.dx) + (x0 - xoff);
#pragma unroll
            for (int k = 0; k < SLOTS; ++k) {
                const int vi = k * GT + tg;
                const int j0 = vi * VEC - xoff;
                if (vi >= nv_row) continue;
                float yv[VEC], gv[VEC], o[VEC];
                unpack<T>(ra[k], yv);
                unpack<T>(rb[k], gv);
#pragma unroll
                for (int e = 0; e < VEC; ++e) {
                    const int j = j0 + e;
                    const bool valid = j >= 0 && j < limit;  // y == 0 (masked) gives exactly +0
                    o[e] = (!valid || yv[e] == 0.f) ? 0.f : (gv[e] - dot) * yv[e] * ba.scale;
                }
                if (j0 >= 0 && j0 + VEC <= cols) {
                    st_stream(orow + vi * VEC, pack<T>(o));
                } else {
#pragma unroll
                    for (int e = 0; e < VEC; ++e) {
                        const int j = j0 + e;
                        if (j >= 0 && j < cols) orow[vi * VEC + e] = from_f32<T>(o[e]);
                    }
                }
            }
        } else {
            // each thread exponentiates against its own max; warps merge
            // (max, sum) pairs; groups of several warps merge through one barrier
            const float mt = acc;
            const float mtr = (mt == neg_inf()) ? 0.f : mt;
            float lt = 0.f;
#pragma unroll
            for (int k = 0; k < SLOTS; ++k)
#pragma unroll
                for (int e = 0; e < VEC; ++e) {
                    const float v = ex2((va[k][e] - mtr) * kLog2e);
                    va[k][e] = v;
                    lt += v;
                }
            const float mw = group_max<32>(mt);
            const float mwr = (mw == neg_inf()) ? 0.f : mw;
            float M = mw;
            float tot = group_sum<32>(mt == neg_inf() ? 0.f : lt * ex2((mt - mwr) * kLog2e));
            if constexpr (WG > 1) {
                if (lane == 0) {
                    h.red_max[g][rp][wg] = mw;
                    h.red_sum[g][rp][wg] = tot;
                }
                named_sync(1 + g, GT);
                if (h.cons_abort[g]) break;  // uniform within the group
                M = neg_inf();
#pragma unroll
                for (int w = 0; w < WG; ++w) M = fmaxf(M, h.red_max[g][rp][w]);
                const float Mr = (M == neg_inf()) ? 0.f : M;
                tot = 0.f;
#pragma unroll
                for (int w = 0; w < WG; ++w) {
                    const float m2 = h.red_max[g][rp][w];
                    tot += (m2 == neg_inf()) ? 0.f : h.red_sum[g][rp][w] * ex2((m2 - Mr) * kLog2e);
                }
            } else {
                if (!row_ok) break;  // warp-uniform
            }
            const float Mr = (M == neg_inf()) ? 0.f : M;
            const float inv = tot > 0.f ? __frcp_rn(tot) : 0.f;
            const float f = (mt == neg_inf()) ? 0.f : ex2((mt - Mr) * kLog2e) * inv;  // this thread's factor
            T *orow = reinterpret_cast<T *>(fa.y) + (x0 - xoff);
#pragma unroll
            for (int k = 0; k < SLOTS; ++k) {
                const int vi = k * GT + tg;
                const int j0 = vi * VEC - xoff;
                if (vi >= nv_row) continue;
                float o[VEC];
#pragma unroll
                for (int e = 0; e < VEC; ++e) o[e] = va[k][e] * f;
                if (j0 >= 0 && j0 + VEC <= cols) {
                    st_stream(orow + vi * VEC, pack<T>(o));
                } else {
#pragma unroll
                    for (int e = 0; e < VEC; ++e) {
                        const int j = j0 + e;
                        if (j >= 0 && j < cols) orow[vi * VEC + e] = from_f32<T>(o[e]);
                    }
                }
            }
        }
    }
}

template <typename T, int WG, int R, int SLOTS, int CH, bool BWD, typename M>
cudaError_t launch_tile(const FwdArgs &fa, const BwdArgs &ba, cudaStream_t st)
{
    constexpr int smem = smem_bytes<WG, R, SLOTS, CH>();
    auto kern = tile_kernel<T, WG, R, SLOTS, CH, BWD, M>;
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
    const int64_t grid = persistent_grid(1, rows);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(Geo<WG, R, SLOTS, CH>::THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    return cudaLaunchKernelEx(&cfg, kern, fa, ba);
}

// 16-byte vectors a row spans (one more when rows may start mid-vector).
inline int64_t row_vectors(int64_t cols, int dtype, bool aligned)
{
    const int vec = vec_elems(dtype);
    return (cols + vec - 1) / vec + (aligned ? 0 : 1);
}

// Shapes, smallest capacity first (capacity = WG*32*SLOTS vectors):
//   WG=1  R=8 : 1, 2, 4, 8 slots, whole rows per stage
//   WG=2  R=4 : 4, 8 slots, whole rows
//   WG=4  R=2 : 4, 8 slots, whole rows
//   WG=8  R=1 : 4, 8 slots, whole rows
//   WG=16 R=1 : 4, 8 slots, rows in 2 or 4 chunks
// SLOTS is capped at 4 for the 16-bit forward (8 fp32 scores per slot) and 8
// elsewhere, which keeps every thread within 32 fp32 values per slot set.
template <typename T, bool BWD, typename M = T>
cudaError_t launch_t(const FwdArgs &fa, const BwdArgs &ba, int64_t vecs, cudaStream_t st)
{
    constexpr bool S8 = BWD || Dt<T>::VEC == 4;  // 8 slots allowed
#define SMS_TILE(WG, R, SL, CH) \
    if (vecs <= (int64_t)(WG) * 32 * (SL)) return launch_tile<T, WG, R, SL, CH, BWD, M>(fa, ba, st);
    SMS_TILE(1, 8, 1, 1) SMS_TILE(1, 8, 2, 2) SMS_TILE(1, 8, 4, 4)
    if constexpr (S8) { SMS_TILE(1, 8, 8, 8) }
    SMS_TILE(2, 4, 4, 4)
    if constexpr (S8) { SMS_TILE(2, 4, 8, 8) }
    SMS_TILE(4, 2, 4, 4)
    if constexpr (S8) { SMS_TILE(4, 2, 8, 8) }
    SMS_TILE(8, 1, 4, 4)
    if constexpr (S8) { SMS_TILE(8, 1, 8, 8) }
    SMS_TILE(16, 1, 4, 2)
    if constexpr (S8) { SMS_TILE(16, 1, 8, 2) }
#undef SMS_TILE
    return cudaErrorNotSupported;
}

inline int64_t tile_capacity(int dtype, bool bwd) { return 16 * 32 * ((bwd || vec_elems(dtype) == 4) ? 8 : 4); }

template <bool BWD>
cudaError_t dispatch(const FwdArgs &fa, const BwdArgs &ba, int64_t cols, int dtype, bool aligned, cudaStream_t st)
{
    const int64_t vecs = row_vectors(cols, dtype, aligned);
    const bool mb = !BWD && fa.mask && fa.mask_bool;
    switch (dtype) {
    case kF32: return mb ? launch_t<float, BWD, uint8_t>(fa, ba, vecs, st) : launch_t<float, BWD>(fa, ba, vecs, st);
    case kF16: return mb ? launch_t<__half, BWD, uint8_t>(fa, ba, vecs, st) : launch_t<__half, BWD>(fa, ba, vecs, st);
    case kBF16:
        return mb ? launch_t<__nv_bfloat16, BWD, uint8_t>(fa, ba, vecs, st)
                  : launch_t<__nv_bfloat16, BWD>(fa, ba, vecs, st);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace
}  // namespace tile
}  // namespace sms
