// Persistent register-resident row kernels with a one-row software prefetch.
//
// The one-shot lane-group kernels (sms_warp.cu) issue a row's loads, wait, and
// then spend the reductions, the exponentials and the stores with no load of
// their own in flight; HBM is kept busy only by the other resident groups that
// happen to be in their load phase.  Here each lane group walks a strided
// sequence of rows (persistent CTAs) and issues the loads of its next row
// before it computes the current one, so every group keeps one row's worth
// of 16-byte loads in flight through its whole life.  Register cost: two row
// buffers.  Row positions are re-derived per row with the invariant-divisor
// division (no per-CTA start-up).
//
// The per-row work (positions, loads, reductions, stores, and the operation's
// definition with its page citations) is in sms_rowmath.cuh.
//
// Barriers: every CTA runs the same number of iterations (the loop is driven
// by the CTA's first row), so the multi-warp groups' __syncthreads are
// reached uniformly; the shared reduction slots alternate between two halves
// so a fast warp never overwrites slots another warp is still reading.
#include <type_traits>

#include "sms_rowmath.cuh"

namespace sms {
namespace {

constexpr int kThreads = 256;

using namespace rowmath;

template <typename T, int G, int NV, bool ALIGNED, typename M>
__global__ void __launch_bounds__(kThreads, 2) fwd_stream_kernel(const FwdArgs a)
{
    constexpr int VEC = Dt<T>::VEC;
    constexpr int GPC = kThreads / G;
    constexpr int W = G > 32 ? G / 32 : 1;
    __shared__ float red_m[2][GPC][W], red_l[2][GPC][W];
    const int gl = threadIdx.x % G;
    const int gi = threadIdx.x / G;
    const int64_t stride = (int64_t)gridDim.x * GPC;
    int64_t base = (int64_t)blockIdx.x * GPC;  // the CTA's first row: drives the (CTA-uniform) loop
    FwdBuf<NV, ALIGNED> A, B;
    RowPos pa = fwd_pos<VEC, ALIGNED>(a, base + gi), pb;
    fwd_issue<T, G, NV, ALIGNED, M>(a, pa, gl, A);
    while (true) {
        const bool more1 = base + stride < a.rows;
        if (more1) {
            pb = fwd_pos<VEC, ALIGNED>(a, base + stride + gi);
            fwd_issue<T, G, NV, ALIGNED, M>(a, pb, gl, B);
        }
        fwd_finish<T, G, NV, ALIGNED, M>(a, pa, gl, gi, A, red_m[0], red_l[0]);
        if (!more1) break;
        base += stride;
        const bool more2 = base + stride < a.rows;
        if (more2) {
            pa = fwd_pos<VEC, ALIGNED>(a, base + stride + gi);
            fwd_issue<T, G, NV, ALIGNED, M>(a, pa, gl, A);
        }
        fwd_finish<T, G, NV, ALIGNED, M>(a, pb, gl, gi, B, red_m[1], red_l[1]);
        if (!more2) break;
        base += stride;
    }
}

template <typename T, int G, int NV, bool ALIGNED>
__global__ void __launch_bounds__(kThreads, 2) bwd_stream_kernel(const BwdArgs a)
{
    constexpr int VEC = Dt<T>::VEC;
    constexpr int GPC = kThreads / G;
    constexpr int W = G > 32 ? G / 32 : 1;
    __shared__ float red[2][GPC][W];
    const int gl = threadIdx.x % G;
    const int gi = threadIdx.x / G;
    const int64_t stride = (int64_t)gridDim.x * GPC;
    int64_t base = (int64_t)blockIdx.x * GPC;
    BwdBuf<NV> A, B;
    BRowPos pa = bwd_pos<VEC, ALIGNED>(a, base + gi), pb;
    bwd_issue<T, G, NV, ALIGNED>(a, pa, gl, A);
    while (true) {
        const bool more1 = base + stride < a.rows;
        if (more1) {
            pb = bwd_pos<VEC, ALIGNED>(a, base + stride + gi);
            bwd_issue<T, G, NV, ALIGNED>(a, pb, gl, B);
        }
        bwd_finish<T, G, NV, ALIGNED>(a, pa, gl, gi, A, red[0]);
        if (!more1) break;
        base += stride;
        const bool more2 = base + stride < a.rows;
        if (more2) {
            pa = bwd_pos<VEC, ALIGNED>(a, base + stride + gi);
            bwd_issue<T, G, NV, ALIGNED>(a, pa, gl, A);
        }
        bwd_finish<T, G, NV, ALIGNED>(a, pb, gl, gi, B, red[1]);
        if (!more2) break;
        base += stride;
    }
}

// ------------------------------------------------------------- launch ---

// Resident CTAs per multiprocessor of a kernel (asked once per instantiation;
// at least the 2 its launch bounds guarantee).
template <typename K>
int resident_ctas(K kern)
{
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, 0) != cudaSuccess || per_sm < 2) {
        cudaGetLastError();
        per_sm = 2;
    }
    return per_sm;
}

template <typename T, int G, int NV, bool ALIGNED, bool BWD, typename M, typename Args>
cudaError_t launch_one(const Args &a, cudaStream_t st)
{
    constexpr int GPC = kThreads / G;
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(kThreads);
    cfg.stream = st;
    const int64_t useful = (a.rows + GPC - 1) / GPC;
    if constexpr (BWD) {
        static const int per_sm = resident_ctas(bwd_stream_kernel<T, G, NV, ALIGNED>);
        cfg.gridDim = dim3((unsigned)persistent_grid(per_sm, useful));
        return cudaLaunchKernelEx(&cfg, bwd_stream_kernel<T, G, NV, ALIGNED>, a);
    } else {
        static const int per_sm = resident_ctas(fwd_stream_kernel<T, G, NV, ALIGNED, M>);
        cfg.gridDim = dim3((unsigned)persistent_grid(per_sm, useful));
        return cudaLaunchKernelEx(&cfg, fwd_stream_kernel<T, G, NV, ALIGNED, M>, a);
    }
}

// (lanes per row, vectors per lane), smallest capacity first; one row per
// group, two row buffers per lane.
template <typename T, bool ALIGNED, bool BWD, typename M, typename Args>
cudaError_t launch_t(const Args &a, cudaStream_t st)
{
    constexpr int VEC = Dt<T>::VEC;
    if constexpr (!BWD && !ALIGNED) {
        // two row buffers plus the mask realignment registers do not fit 128
        // registers: rows that start mid-vector stay with the one-shot kernels
        return cudaErrorNotSupported;
    } else {
        const int64_t need = (a.cols + VEC - 1) / VEC + (ALIGNED ? 0 : 1);
#define SMS_TRY(G, NV) \
    if (need <= (G) * (NV)) return launch_one<T, G, NV, ALIGNED, BWD, M>(a, st);
        SMS_TRY(4, 4) SMS_TRY(8, 4) SMS_TRY(16, 4) SMS_TRY(32, 4) SMS_TRY(64, 4) SMS_TRY(128, 4) SMS_TRY(256, 4)
#undef SMS_TRY
        return cudaErrorNotSupported;
    }
}

// MASKB: the forward's mask is boolean (one byte per element), else additive.
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

bool stream_fits(int64_t cols, int dtype, bool aligned, bool bwd)
{
    const int vec = vec_elems(dtype);
    return (bwd || aligned) && (cols + vec - 1) / vec + (aligned ? 0 : 1) <= 256 * 4;
}

cudaError_t launch_fwd_stream(const FwdArgs &a, int dtype, bool aligned, cudaStream_t st)
{
    return a.mask_bool ? dispatch<false, true>(a, dtype, aligned, st) : dispatch<false, false>(a, dtype, aligned, st);
}

cudaError_t launch_bwd_stream(const BwdArgs &a, int dtype, bool aligned, cudaStream_t st)
{
    return dispatch<true, false>(a, dtype, aligned, st);
}

}  // namespace sms
