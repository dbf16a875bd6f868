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
//   * NT consumer threads pull each stage into registers (the row stays in
//     registers, not shared memory) and release the stage at once;
//   * reductions are warp shuffles plus one 16-entry shared exchange;
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

constexpr int kNT = 512;                    // consumer threads (16 warps)
constexpr int kNW = kNT / 32;
constexpr int kThreads = kNT + 32;          // + one producer warp
constexpr int kSV = kNT;                    // 16-byte vectors of x (or y) per stage
constexpr int kStageBytes = 16 * (2 * kSV + 1);  // x/y area + mask/dy area (+1 vector of slack)
constexpr int kMaxStages = 16;
constexpr int kSmemTarget = 200 * 1024;

struct Hdr {
    uint64_t full[kMaxStages];
    uint64_t empty[kMaxStages];
    float red_max[kNW];
    float red_sum[2][kNW];  // double buffered by row parity (one barrier per row in backward)
    int abort;       // any thread gave up (producer or consumer)
    int cons_abort;  // a consumer gave up (read only after a consumer barrier)
};
constexpr int kHdrBytes = (int)((sizeof(Hdr) + 127) / 128 * 128);

// Geometry of one row, computed identically by producer and consumers.
struct Row {
    int64_t x0;     // flat element index of the row start
    int64_t gbase;  // tensor vector index of the aligned row start
    int xoff;       // x0 mod VEC
    int limit;      // elements read (q+1 under causal, else cols)
    int nv_read;    // vectors holding elements < limit
    int nv_row;     // vectors holding row elements
    int nchunks;    // stages used by the row
    int64_t m0;     // mask row start (forward)
};

template <int VEC>
__device__ __forceinline__ Row row_geom(int64_t r, int64_t cols, int causal)
{
    Row g;
    g.x0 = r * cols;
    g.xoff = (int)(g.x0 & (VEC - 1));
    g.gbase = (g.x0 - g.xoff) / VEC;
    const int64_t q = r % cols;
    g.limit = causal ? (int)(q + 1) : (int)cols;
    g.nv_read = (g.xoff + g.limit + VEC - 1) / VEC;
    g.nv_row = (int)((g.xoff + cols + VEC - 1) / VEC);
    g.nchunks = (g.nv_read + kSV - 1) / kSV;
    g.m0 = 0;
    return g;
}

// Mask vectors of chunk c: [mv_lo, cm_hi) are in the stage (tensor vector indices).
template <int VEC>
__device__ __forceinline__ void mask_span(const Row &g, int c, int64_t mask_total, int64_t &mv_lo, int64_t &cm_hi)
{
    const int vlo = c * kSV;
    const int vhi = min(g.nv_read, vlo + kSV);
    const int64_t jlo = max(0, vlo * VEC - g.xoff);
    const int64_t jhi = min((int64_t)g.limit, (int64_t)vhi * VEC - g.xoff);
    mv_lo = (g.m0 + jlo) / VEC;
    const int64_t mv_hi = (g.m0 + jhi + VEC - 1) / VEC;
    cm_hi = min(mv_hi, mask_total / VEC);
}

template <typename T, int SLOTS, bool BWD>
__global__ void __launch_bounds__(kThreads, 1) cta_kernel(const FwdArgs fa, const BwdArgs ba, int nstage)
{
    constexpr int VEC = Dt<T>::VEC;
    extern __shared__ __align__(128) unsigned char smem[];
    Hdr &h = *reinterpret_cast<Hdr *>(smem);
    unsigned char *stages = smem + kHdrBytes;

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
            mbar_init(&h.empty[s], kNW);
        }
        h.abort = 0;
        h.cons_abort = 0;
        fence_mbar_init();
    }
    __syncthreads();

    volatile int *abort_flag = &h.abort;

    if (threadIdx.x >= kNT) {
        // ------------------------------------------------------- producer ---
        if (threadIdx.x != kNT) return;
        const uint64_t polA = policy_evict_first();
        const uint64_t polB = BWD ? polA : policy_evict_normal();
        uint32_t issued = 0, parity = 0;  // per stage: ever issued / parity of its last issue
        int stage = 0;
        uint32_t ph = 0;
        bool ok = true;
        for (int64_t r = blockIdx.x; r < rows && ok; r += gridDim.x) {
            Row g = row_geom<VEC>(r, cols, causal);
            if (!BWD && srcB) {
                const int64_t hh = (r / cols) % fa.heads, bb = r / (cols * fa.heads);
                g.m0 = bb * fa.msb + hh * fa.msh + (r % cols) * cols;
            }
            for (int c = 0; c < g.nchunks; ++c) {
                if (!mbar_wait_bounded(&h.empty[stage], ph ^ 1u, abort_flag)) {
                    *abort_flag = 1;
                    report_error(err, 2);
                    ok = false;
                    break;
                }
                const int vlo = c * kSV;
                const int vhi = min(g.nv_read, vlo + kSV);
                const int64_t cx_hi = min((int64_t)vhi, full_vecs - g.gbase);
                const uint32_t bytesA = cx_hi > vlo ? (uint32_t)(cx_hi - vlo) * 16u : 0u;
                uint32_t bytesB = 0;
                int64_t b_src = 0;
                if (BWD) {
                    bytesB = bytesA;
                    b_src = g.gbase + vlo;
                } else if (srcB) {
                    int64_t mv_lo, cm_hi;
                    mask_span<VEC>(g, c, fa.mask_total, mv_lo, cm_hi);
                    bytesB = cm_hi > mv_lo ? (uint32_t)(cm_hi - mv_lo) * 16u : 0u;
                    b_src = mv_lo;
                }
                unsigned char *st = stages + (size_t)stage * kStageBytes;
                mbar_arrive_expect_tx(&h.full[stage], bytesA + bytesB);
                if (bytesA)
                    bulk_g2s(st, reinterpret_cast<const uint4 *>(srcA) + g.gbase + vlo, bytesA, &h.full[stage], polA);
                if (bytesB)
                    bulk_g2s(st + 16 * kSV, reinterpret_cast<const uint4 *>(srcB) + b_src, bytesB, &h.full[stage], polB);
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

    for (int64_t r = blockIdx.x; r < rows; r += gridDim.x, rp ^= 1) {
        Row g = row_geom<VEC>(r, cols, causal);
        const T *mrow = nullptr;
        bool mvec = false;
        if (!BWD && srcB) {
            const int64_t hh = (r / cols) % fa.heads, bb = r / (cols * fa.heads);
            g.m0 = bb * fa.msb + hh * fa.msh + (r % cols) * cols;
            mrow = reinterpret_cast<const T *>(srcB) + g.m0;
            mvec = ((g.m0 - g.xoff) & (VEC - 1)) == 0;
        }
        const T *arow = reinterpret_cast<const T *>(srcA) + (g.x0 - g.xoff);  // aligned
        const T *brow = BWD ? reinterpret_cast<const T *>(srcB) + (g.x0 - g.xoff) : nullptr;

        // forward: scores s as fp32; backward: y and dy kept as the raw 16-byte
        // vectors (half the registers for fp16/bf16), widened again for dx
        float va[BWD ? 1 : SLOTS][VEC];
        uint4 ra[BWD ? SLOTS : 1], rb[BWD ? SLOTS : 1];
        float acc = BWD ? 0.f : neg_inf();  // backward: dot; forward: running max

#pragma unroll
        for (int k = 0; k < SLOTS; ++k) {
            if (BWD) {
                ra[k] = make_uint4(0, 0, 0, 0);
                rb[k] = make_uint4(0, 0, 0, 0);
            } else {
#pragma unroll
                for (int e = 0; e < VEC; ++e) va[k][e] = neg_inf();
            }
            if (k < g.nchunks) {
                if (!mbar_wait_bounded(&h.full[stage], ph, abort_flag)) {
                    *abort_flag = 1;
                    h.cons_abort = 1;
                    report_error(err, 1);
                }
                const unsigned char *st = stages + (size_t)stage * kStageBytes;
                const int vi = k * kSV + t;
                const int j0 = vi * VEC - g.xoff;
                if (vi < g.nv_read) {
                    const int64_t gv = g.gbase + vi;
                    float a[VEC], b[VEC];
                    if (BWD) {
                        if (gv < full_vecs) {
                            ra[k] = reinterpret_cast<const uint4 *>(st)[t];
                            rb[k] = reinterpret_cast<const uint4 *>(st + 16 * kSV)[t];
                        } else {  // last partial vector of the tensor: not in the stage
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
                            if (j >= 0 && j < g.limit) acc = fmaf(a[e], b[e], acc);
                        }
                    } else {
                        if (gv < full_vecs) {
                            unpack<T>(reinterpret_cast<const uint4 *>(st)[t], a);
                        } else {  // last partial vector of the tensor: not in the stage
#pragma unroll
                            for (int e = 0; e < VEC; ++e)
                                a[e] = gv * VEC + e < total ? to_f32<T>(arow[vi * VEC + e]) : 0.f;
                        }
#pragma unroll
                        for (int e = 0; e < VEC; ++e) b[e] = 0.f;
                        if (mrow) {
                            int64_t mv_lo, cm_hi;
                            mask_span<VEC>(g, k, fa.mask_total, mv_lo, cm_hi);
                            const T *msm = reinterpret_cast<const T *>(st + 16 * kSV);
                            const int64_t mvi = (g.m0 - g.xoff) / VEC + vi;  // valid when mvec
                            if (mvec && mvi >= mv_lo && mvi < cm_hi) {
                                unpack<T>(reinterpret_cast<const uint4 *>(msm)[mvi - mv_lo], b);
                            } else {
#pragma unroll
                                for (int e = 0; e < VEC; ++e) {
                                    const int j = j0 + e;
                                    if (j >= 0 && j < g.limit) {
                                        const int64_t f = g.m0 + j;
                                        b[e] = f < cm_hi * VEC ? to_f32<T>(msm[f - mv_lo * VEC]) : to_f32<T>(mrow[j]);
                                    }
                                }
                            }
                        }
#pragma unroll
                        for (int e = 0; e < VEC; ++e) {
                            const int j = j0 + e;
                            va[k][e] = (j >= 0 && j < g.limit) ? fmaf(a[e], fa.scale, b[e]) : neg_inf();
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
            named_sync(1, kNT);
            if (h.cons_abort) break;  // uniform: every consumer reads the same value here
            float dot = 0.f;
#pragma unroll
            for (int w = 0; w < kNW; ++w) dot += h.red_sum[rp][w];
            T *orow = reinterpret_cast<T *>(ba.dx) + (g.x0 - g.xoff);
#pragma unroll
            for (int k = 0; k < SLOTS; ++k) {
                const int vi = k * kSV + t;
                const int j0 = vi * VEC - g.xoff;
                if (vi >= g.nv_row) continue;
                float yv[VEC], gv[VEC], o[VEC];
                unpack<T>(ra[k], yv);
                unpack<T>(rb[k], gv);
#pragma unroll
                for (int e = 0; e < VEC; ++e) {
                    const int j = j0 + e;
                    const bool valid = j >= 0 && j < g.limit;  // y == 0 (masked) gives exactly +0
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
            acc = group_max<32>(acc);
            if (lane == 0) h.red_max[warp] = acc;
            named_sync(1, kNT);
            if (h.cons_abort) break;  // uniform: every consumer reads the same value here
            float mx = neg_inf();
#pragma unroll
            for (int w = 0; w < kNW; ++w) mx = fmaxf(mx, h.red_max[w]);
            const float mref = (mx == neg_inf()) ? 0.f : mx;
            float sum = 0.f;
#pragma unroll
            for (int k = 0; k < SLOTS; ++k)
#pragma unroll
                for (int e = 0; e < VEC; ++e) {
                    const float v = ex2((va[k][e] - mref) * kLog2e);
                    va[k][e] = v;
                    sum += v;
                }
            sum = group_sum<32>(sum);
            if (lane == 0) h.red_sum[rp][warp] = sum;
            named_sync(1, kNT);
            float tot = 0.f;
#pragma unroll
            for (int w = 0; w < kNW; ++w) tot += h.red_sum[rp][w];
            const float inv = tot > 0.f ? __frcp_rn(tot) : 0.f;
            T *orow = reinterpret_cast<T *>(fa.y) + (g.x0 - g.xoff);
#pragma unroll
            for (int k = 0; k < SLOTS; ++k) {
                const int vi = k * kSV + t;
                const int j0 = vi * VEC - g.xoff;
                if (vi >= g.nv_row) continue;
                float o[VEC];
#pragma unroll
                for (int e = 0; e < VEC; ++e) o[e] = va[k][e] * inv;
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

int stages_for_budget() { return (kSmemTarget - kHdrBytes) / kStageBytes; }

template <typename T, int SLOTS, bool BWD>
cudaError_t launch_one(const FwdArgs &fa, const BwdArgs &ba, cudaStream_t st)
{
    const int nstage = stages_for_budget() < kMaxStages ? stages_for_budget() : kMaxStages;
    const int smem = kHdrBytes + nstage * kStageBytes;
    auto kern = cta_kernel<T, SLOTS, BWD>;
    static std::once_flag once[64];
    int dev = 0;
    cudaGetDevice(&dev);
    cudaError_t attr = cudaSuccess;
    std::call_once(once[dev & 63], [&] {
        attr = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    });
    if (attr != cudaSuccess) return attr;
    const int64_t rows = BWD ? ba.rows : fa.rows;
    int64_t grid = (int64_t)sm_count();
    if (grid > rows) grid = rows;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    return cudaLaunchKernelEx(&cfg, kern, fa, ba, nstage);
}

// Register slots (16-byte vectors per consumer thread) needed for a row.
inline int64_t slots_needed(int64_t cols, int dtype)
{
    const int vec = vec_elems(dtype);
    const int64_t vecs = (cols + vec - 1) / vec + 1;  // +1: a row may start mid-vector
    return (vecs + kNT - 1) / kNT;
}

template <typename T, bool BWD>
cudaError_t launch_t(const FwdArgs &fa, const BwdArgs &ba, int64_t cols, int dtype, cudaStream_t st)
{
    const int64_t s = slots_needed(cols, dtype);
    if (s <= 1) return launch_one<T, 1, BWD>(fa, ba, st);
    if (s <= 2) return launch_one<T, 2, BWD>(fa, ba, st);
    if (s <= 4) return launch_one<T, 4, BWD>(fa, ba, st);
    if (s <= 8) return launch_one<T, 8, BWD>(fa, ba, st);
    if constexpr (!BWD && Dt<T>::VEC == 4) {
        if (s <= 16) return launch_one<T, 16, BWD>(fa, ba, st);
    }
    return cudaErrorNotSupported;
}

template <bool BWD>
cudaError_t dispatch(const FwdArgs &fa, const BwdArgs &ba, int64_t cols, int dtype, cudaStream_t st)
{
    switch (dtype) {
    case kF32: return launch_t<float, BWD>(fa, ba, cols, dtype, st);
    case kF16: return launch_t<__half, BWD>(fa, ba, cols, dtype, st);
    case kBF16: return launch_t<__nv_bfloat16, BWD>(fa, ba, cols, dtype, st);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace

// Forward keeps fp32 scores: 16 slots (64 values) for fp32 rows, 8 for 16-bit
// rows (64 values); backward keeps raw vectors: 8 slots.
bool cta_fits(int64_t cols, int dtype) { return slots_needed(cols, dtype) <= (vec_elems(dtype) == 4 ? 16 : 8); }

bool cta_fits_bwd(int64_t cols, int dtype) { return slots_needed(cols, dtype) <= 8; }

cudaError_t launch_fwd_cta(const FwdArgs &a, int dtype, cudaStream_t st)
{
    BwdArgs none = {};
    return dispatch<false>(a, none, a.cols, dtype, st);
}

cudaError_t launch_bwd_cta(const BwdArgs &a, int dtype, cudaStream_t st)
{
    FwdArgs none = {};
    return dispatch<true>(none, a, a.cols, dtype, st);
}

}  // namespace sms
