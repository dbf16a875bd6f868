// Persistent CTA-per-row kernels with bulk-copy (TMA) staging, for rows too
// wide for one warp's registers.
//
// Prior art: the page "用CUDA自定义融合Softmax算子并封装进PyTorch" (§2.3 one block per
// row, §3.1 shared-memory row cache, §3.2 tree reductions) launched one
// 128-thread block per row, cached the whole scaled row in shared memory and
// reduced with log2(128) barrier rounds.  On sm_103a the same "CTA owns a row"
// idea is arranged differently:
//   * one producer lane streams rows into a ring of shared-memory stages with
//     cp.async.bulk (the TMA unit), running ahead of the consumers by up to
//     the whole ring, so HBM reads for the next rows overlap the reductions
//     and stores of the current one;
//   * the producer also writes a 64-byte descriptor into every stage (row
//     start, alignment, causal limit, mask span, ...): consumer threads do no
//     index arithmetic of their own;
//   * NT consumer threads pull each stage into registers (the row stays in
//     registers, not shared memory) and release the stage at once;
//   * reductions are warp shuffles plus one shared exchange across warps;
//   * exp is evaluated once per element, and causal positions j > q are never
//     copied.
// Rows of any start alignment are handled: stages hold 16-byte vectors
// aligned to the tensor (x) and, separately, to the mask; elements the bulk
// copies cannot cover (a partial vector at the very end of a tensor) are read
// directly from global memory.
//
// Every mbarrier wait is bounded (2 s); a consumer that gives up marks the CTA
// aborted, all consumers leave together at the next row boundary, and the
// producer waits (bounded) for its in-flight copies before exiting.
#include "sms_common.cuh"
#include "sms_internal.h"

#include <mutex>

namespace sms {
namespace {

constexpr int kMaxStages = 32;

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
    int32_t limit;   // elements read: q+1 under causal, else cols
    int32_t nv_read; // vectors holding elements < limit
    int32_t nv_row;  // vectors holding row elements
    int32_t nchunks; // stages the row occupies
    int32_t pad1, pad2;
};
static_assert(sizeof(ChunkDesc) == 64, "descriptor is one 64-byte slot");

template <int NT> struct Geo {
    static constexpr int NW = NT / 32;
    static constexpr int THREADS = NT + 32;                 // + one producer warp
    static constexpr int SV = NT;                           // 16-byte vectors of x (or y) per stage
    static constexpr int A_OFF = 64;                        // after the descriptor
    static constexpr int B_OFF = 64 + 16 * SV;              // mask (or dy) area, SV + 1 vectors
    static constexpr int STAGE = 64 + 16 * (2 * SV + 1);
};

template <int NT> struct Hdr {
    uint64_t full[kMaxStages];
    uint64_t empty[kMaxStages];
    float red_max[2][Geo<NT>::NW];  // double buffered by row parity: one barrier per row
    float red_sum[2][Geo<NT>::NW];
    int abort;                      // any thread gave up (producer or consumer)
    int cons_abort;                 // a consumer gave up (read only after a consumer barrier)
};
template <int NT> __host__ __device__ constexpr int hdr_bytes() { return (int)((sizeof(Hdr<NT>) + 127) / 128 * 128); }

// CTAs resident per SM: 512 / NT (shared memory is split the same way)
template <int NT> __host__ __device__ constexpr int ctas_per_sm() { return NT >= 512 ? 1 : 512 / NT; }

template <typename T, int NT, int SLOTS, bool BWD>
__global__ void __launch_bounds__(Geo<NT>::THREADS, ctas_per_sm<NT>())
    cta_kernel(const FwdArgs fa, const BwdArgs ba, int nstage)
{
    using G = Geo<NT>;
    constexpr int VEC = Dt<T>::VEC;
    constexpr int SV = G::SV;
    extern __shared__ __align__(128) unsigned char smem[];
    Hdr<NT> &h = *reinterpret_cast<Hdr<NT> *>(smem);
    unsigned char *stages = smem + hdr_bytes<NT>();

    const int64_t rows = BWD ? ba.rows : fa.rows;
    const int64_t cols = BWD ? ba.cols : fa.cols;
    const int64_t total = BWD ? ba.total : fa.x_total;
    const int causal = BWD ? ba.causal : fa.causal;
    const void *srcA = BWD ? ba.y : fa.x;
    const void *srcB = BWD ? ba.dy : fa.mask;
    int *err = BWD ? ba.err : fa.err;
    const int64_t full_vecs = total / VEC;  // vectors lying wholly inside the tensor

    if (threadIdx.x == 0) {
        for (int s = 0; s < nstage; ++s) {
            mbar_init(&h.full[s], 1);
            mbar_init(&h.empty[s], G::NW);
        }
        h.abort = 0;
        h.cons_abort = 0;
        fence_mbar_init();
    }
    __syncthreads();

    volatile int *abort_flag = &h.abort;

    if (threadIdx.x >= NT) {
        // ------------------------------------------------------- producer ---
        if (threadIdx.x != NT) return;
        const uint64_t polA = policy_evict_first();
        const uint64_t polB = BWD ? polA : policy_evict_normal();
        uint32_t issued = 0, parity = 0;  // per stage: ever issued / parity of its last issue
        int stage = 0;
        uint32_t ph = 0;
        bool ok = true;
        for (int64_t r = blockIdx.x; r < rows && ok; r += gridDim.x) {
            int64_t q = 0, hh = 0, bb = 0;
            if (BWD) {
                if (causal) q = row_q(r, cols, ba.dcols);
            } else if (causal || srcB) {
                split_row(r, cols, fa.heads, fa.dcols, fa.dheads, q, hh, bb);
            }
            ChunkDesc d;
            d.x0 = r * cols;
            d.xoff = (int)(d.x0 & (VEC - 1));
            const int64_t gbase = (d.x0 - d.xoff) / VEC;
            d.limit = causal ? (int)(q + 1) : (int)cols;
            d.nv_read = (d.xoff + d.limit + VEC - 1) / VEC;
            d.nv_row = (int)((d.xoff + cols + VEC - 1) / VEC);
            d.nchunks = (d.nv_read + SV - 1) / SV;
            d.m0 = (!BWD && srcB) ? bb * fa.msb + hh * fa.msh + q * cols : 0;
            d.mvec = ((d.m0 - d.xoff) & (VEC - 1)) == 0;
            d.pad0 = d.pad1 = d.pad2 = 0;
            for (int c = 0; c < d.nchunks; ++c) {
                if (!mbar_wait_bounded(&h.empty[stage], ph ^ 1u, abort_flag)) {
                    *abort_flag = 1;
                    report_error(err, 2);
                    ok = false;
                    break;
                }
                const int vlo = c * SV;
                const int vhi = min(d.nv_read, vlo + SV);
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
                    const int64_t mv_lo = (d.m0 + jlo) / VEC;
                    const int64_t cm_hi = min((d.m0 + jhi + VEC - 1) / VEC, fa.mask_total / VEC);
                    d.mrel = (int)(d.m0 - mv_lo * VEC);
                    d.mcnt = cm_hi > mv_lo ? (int)(cm_hi - mv_lo) * VEC : 0;
                    bytesB = cm_hi > mv_lo ? (uint32_t)(cm_hi - mv_lo) * 16u : 0u;
                    b_src = mv_lo;
                }
                unsigned char *st = stages + (size_t)stage * G::STAGE;
                *reinterpret_cast<ChunkDesc *>(st) = d;  // visible to consumers through the barrier
                mbar_arrive_expect_tx(&h.full[stage], bytesA + bytesB);
                if (bytesA)
                    bulk_g2s(st + G::A_OFF, reinterpret_cast<const uint4 *>(srcA) + gbase + vlo, bytesA,
                             &h.full[stage], polA);
                if (bytesB)
                    bulk_g2s(st + G::B_OFF, reinterpret_cast<const uint4 *>(srcB) + b_src, bytesB, &h.full[stage],
                             polB);
                issued |= 1u << stage;
                parity = (parity & ~(1u << stage)) | (ph << stage);
                if (++stage == nstage) { stage = 0; ph ^= 1u; }
            }
        }
        // never leave with copies in flight: wait for the last issue of every stage
        for (int s = 0; s < nstage; ++s)
            if (issued & (1u << s)) {
                const uint32_t p = (parity >> s) & 1u;
                if (!mbar_try_wait(&h.full[s], p)) {
                    const uint64_t t0 = global_ns();
                    while (!mbar_try_wait(&h.full[s], p))
                        if (global_ns() - t0 > kWaitLimitNs) { report_error(err, 2); break; }
                }
            }
        return;
    }

    // ---------------------------------------------------------- consumers ---
    const int t = threadIdx.x;
    const int lane = t & 31, warp = t >> 5;
    int stage = 0;
    uint32_t ph = 0;
    int rp = 0;  // row parity: selects the reduction buffer
    const int64_t my_rows = rows > blockIdx.x ? (rows - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;

    for (int64_t it = 0; it < my_rows; ++it, rp ^= 1) {
        // forward: scores s as fp32; backward: y and dy kept as the raw 16-byte
        // vectors (half the registers for fp16/bf16), widened again for dx
        float va[BWD ? 1 : SLOTS][VEC];
        uint4 ra[BWD ? SLOTS : 1], rb[BWD ? SLOTS : 1];
        float acc = BWD ? 0.f : neg_inf();  // backward: dot; forward: running max
        int64_t x0 = 0;
        int xoff = 0, limit = 0, nv_row = 0, nchunks = 1;

#pragma unroll
        for (int k = 0; k < SLOTS; ++k) {
            if (BWD) {
                ra[k] = make_uint4(0, 0, 0, 0);
                rb[k] = make_uint4(0, 0, 0, 0);
            } else {
#pragma unroll
                for (int e = 0; e < VEC; ++e) va[k][e] = neg_inf();
            }
            if (k < nchunks) {
                // warp-uniform outcome: a warp whose wait failed skips the stage
                // (its descriptor may be stale) and the CTA leaves at the barrier
                const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(&h.full[stage], ph, abort_flag));
                if (!ok && lane == 0) {
                    *abort_flag = 1;
                    h.cons_abort = 1;
                    report_error(err, 1);
                }
                const unsigned char *st = stages + (size_t)stage * G::STAGE;
                const ChunkDesc &d = *reinterpret_cast<const ChunkDesc *>(st);
                if (k == 0 && ok) {
                    x0 = d.x0;
                    xoff = d.xoff;
                    limit = d.limit;
                    nv_row = d.nv_row;
                    nchunks = min(max(d.nchunks, 1), SLOTS);
                }
                const int vi = k * SV + t;
                const int j0 = vi * VEC - xoff;
                if (ok && vi < d.nv_read) {
                    const T *arow = reinterpret_cast<const T *>(srcA) + (x0 - xoff);
                    const int64_t gv = (x0 - xoff) / VEC + vi;
                    float a[VEC], b[VEC];
                    const bool staged = vi < d.cx_hi;  // else: last partial vector of the tensor
                    if (BWD) {
                        const T *brow = reinterpret_cast<const T *>(srcB) + (x0 - xoff);
                        if (staged) {
                            ra[k] = reinterpret_cast<const uint4 *>(st + G::A_OFF)[t];
                            rb[k] = reinterpret_cast<const uint4 *>(st + G::B_OFF)[t];
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
                            unpack<T>(reinterpret_cast<const uint4 *>(st + G::A_OFF)[t], a);
                        } else {
#pragma unroll
                            for (int e = 0; e < VEC; ++e)
                                a[e] = gv * VEC + e < total ? to_f32<T>(arow[vi * VEC + e]) : 0.f;
                        }
#pragma unroll
                        for (int e = 0; e < VEC; ++e) b[e] = 0.f;
                        if (srcB) {
                            const T *msm = reinterpret_cast<const T *>(st + G::B_OFF);
                            const int jj = j0 + d.mrel;  // stage index of element j0
                            if (d.mvec && jj >= 0 && jj + VEC <= d.mcnt) {
                                unpack<T>(*reinterpret_cast<const uint4 *>(msm + jj), b);
                            } else {
                                const T *mrow = reinterpret_cast<const T *>(srcB) + d.m0;
#pragma unroll
                                for (int e = 0; e < VEC; ++e) {
                                    const int j = j0 + e;
                                    if (j >= 0 && j < limit) {
                                        const int idx = j + d.mrel;
                                        b[e] = idx < d.mcnt ? to_f32<T>(msm[idx]) : to_f32<T>(mrow[j]);
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
                __syncwarp();
                if (lane == 0) mbar_arrive(&h.empty[stage]);
                if (++stage == nstage) { stage = 0; ph ^= 1u; }
            }
        }

        if (BWD) {
            acc = group_sum<32>(acc);
            if (lane == 0) h.red_sum[rp][warp] = acc;
            named_sync(1, NT);  // one barrier per row
            if (h.cons_abort) break;  // uniform: every consumer reads the same value here
            float dot = 0.f;
#pragma unroll
            for (int w = 0; w < G::NW; ++w) dot += h.red_sum[rp][w];
            T *orow = reinterpret_cast<T *>(ba.dx) + (x0 - xoff);
#pragma unroll
            for (int k = 0; k < SLOTS; ++k) {
                const int vi = k * SV + t;
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
            // one barrier per row: each thread exponentiates against its own
            // max, warps merge (max, sum) pairs, the CTA merges the warps' pairs
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
            const float lw = group_sum<32>(mt == neg_inf() ? 0.f : lt * ex2((mt - mwr) * kLog2e));
            if (lane == 0) {
                h.red_max[rp][warp] = mw;
                h.red_sum[rp][warp] = lw;
            }
            named_sync(1, NT);
            if (h.cons_abort) break;  // uniform: every consumer reads the same value here
            float M = neg_inf();
#pragma unroll
            for (int w = 0; w < G::NW; ++w) M = fmaxf(M, h.red_max[rp][w]);
            const float Mr = (M == neg_inf()) ? 0.f : M;
            float tot = 0.f;
#pragma unroll
            for (int w = 0; w < G::NW; ++w) {
                const float m2 = h.red_max[rp][w];
                tot += (m2 == neg_inf()) ? 0.f : h.red_sum[rp][w] * ex2((m2 - Mr) * kLog2e);
            }
            const float inv = tot > 0.f ? __frcp_rn(tot) : 0.f;
            const float f = (mt == neg_inf()) ? 0.f : ex2((mt - Mr) * kLog2e) * inv;  // this thread's factor
            T *orow = reinterpret_cast<T *>(fa.y) + (x0 - xoff);
#pragma unroll
            for (int k = 0; k < SLOTS; ++k) {
                const int vi = k * SV + t;
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

// ~200 KB of shared memory per SM, split over the resident CTAs.
template <int NT> constexpr int smem_target() { return 200 * 1024 / ctas_per_sm<NT>(); }
template <int NT> constexpr int n_stages()
{
    return (smem_target<NT>() - hdr_bytes<NT>()) / Geo<NT>::STAGE < kMaxStages
               ? (smem_target<NT>() - hdr_bytes<NT>()) / Geo<NT>::STAGE
               : kMaxStages;
}

template <typename T, int NT, int SLOTS, bool BWD>
cudaError_t launch_one(const FwdArgs &fa, const BwdArgs &ba, cudaStream_t st)
{
    constexpr int nstage = n_stages<NT>();
    constexpr int smem = hdr_bytes<NT>() + nstage * Geo<NT>::STAGE;
    auto kern = cta_kernel<T, NT, SLOTS, BWD>;
    static std::once_flag once[64];
    static cudaError_t attr_status[64];
    static int per_sm[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::call_once(once[dev & 63], [&] {
        cudaError_t s = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        int n = 1;
        if (s == cudaSuccess) s = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, Geo<NT>::THREADS, smem);
        attr_status[dev & 63] = s;
        per_sm[dev & 63] = n > 0 ? n : 1;
    });
    if (attr_status[dev & 63] != cudaSuccess) return attr_status[dev & 63];
    const int64_t rows = BWD ? ba.rows : fa.rows;
    int64_t grid = (int64_t)sm_count() * per_sm[dev & 63];
    if (grid > rows) grid = rows;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(Geo<NT>::THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    return cudaLaunchKernelEx(&cfg, kern, fa, ba, nstage);
}

// 16-byte vectors a row spans (one more when rows may start mid-vector).
inline int64_t row_vectors(int64_t cols, int dtype, bool aligned)
{
    const int vec = vec_elems(dtype);
    return (cols + vec - 1) / vec + (aligned ? 0 : 1);
}

// Consumer threads: the smallest of 128 / 256 / 512 that keeps a row within
// `slots` register slots (16-byte vectors per thread); smaller CTAs run more
// rows per SM at once (4 / 2 / 1 CTAs per SM).  The 16-bit forward holds 8
// fp32 scores per slot, so it aims at 4 slots.
inline int pick_nt(int64_t vecs, int slots)
{
    return vecs <= slots * 128 ? 128 : (vecs <= slots * 256 ? 256 : 512);
}

template <typename T, bool BWD, int NT>
cudaError_t launch_nt(const FwdArgs &fa, const BwdArgs &ba, int64_t vecs, cudaStream_t st)
{
    const int64_t s = (vecs + NT - 1) / NT;
    if (s <= 1) return launch_one<T, NT, 1, BWD>(fa, ba, st);
    if (s <= 2) return launch_one<T, NT, 2, BWD>(fa, ba, st);
    if (s <= 4) return launch_one<T, NT, 4, BWD>(fa, ba, st);
    if (s <= 8) return launch_one<T, NT, 8, BWD>(fa, ba, st);
    if constexpr (NT == 512 && !BWD && Dt<T>::VEC == 4) {
        if (s <= 16) return launch_one<T, NT, 16, BWD>(fa, ba, st);
    }
    return cudaErrorNotSupported;
}

template <typename T, bool BWD>
cudaError_t launch_t(const FwdArgs &fa, const BwdArgs &ba, int64_t cols, int dtype, bool aligned, cudaStream_t st)
{
    const int64_t vecs = row_vectors(cols, dtype, aligned);
    const int nt = pick_nt(vecs, (!BWD && Dt<T>::VEC == 8) ? 4 : 8);
    if (nt == 128) return launch_nt<T, BWD, 128>(fa, ba, vecs, st);
    if (nt == 256) return launch_nt<T, BWD, 256>(fa, ba, vecs, st);
    return launch_nt<T, BWD, 512>(fa, ba, vecs, st);
}

template <bool BWD>
cudaError_t dispatch(const FwdArgs &fa, const BwdArgs &ba, int64_t cols, int dtype, bool aligned, cudaStream_t st)
{
    switch (dtype) {
    case kF32: return launch_t<float, BWD>(fa, ba, cols, dtype, aligned, st);
    case kF16: return launch_t<__half, BWD>(fa, ba, cols, dtype, aligned, st);
    case kBF16: return launch_t<__nv_bfloat16, BWD>(fa, ba, cols, dtype, aligned, st);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace

// Forward keeps fp32 scores: up to 16 slots (64 values) for fp32 rows, 8 for
// 16-bit rows (64 values); backward keeps raw vectors: 8 slots.
bool cta_fits(int64_t cols, int dtype, bool aligned)
{
    return row_vectors(cols, dtype, aligned) <= 512 * (vec_elems(dtype) == 4 ? 16 : 8);
}

bool cta_fits_bwd(int64_t cols, int dtype, bool aligned) { return row_vectors(cols, dtype, aligned) <= 512 * 8; }

cudaError_t launch_fwd_cta(const FwdArgs &a, int dtype, bool aligned, cudaStream_t st)
{
    BwdArgs none = {};
    return dispatch<false>(a, none, a.cols, dtype, aligned, st);
}

cudaError_t launch_bwd_cta(const BwdArgs &a, int dtype, bool aligned, cudaStream_t st)
{
    FwdArgs none = {};
    return dispatch<true>(none, a, a.cols, dtype, aligned, st);
}

}  // namespace sms
