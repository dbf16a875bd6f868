// Register-resident row kernels (templates in sms_warp.cuh): the additive-mask
// forward and the backward.  The boolean-mask forward is instantiated in
// sms_warp_bool.cu, compiled in parallel.
#include "sms_warp.cuh"

namespace sms {

bool warp_fits(int64_t cols, int dtype, bool aligned, bool bwd)
{
    const int vec = vec_elems(dtype);
    const int64_t need = (cols + vec - 1) / vec + (aligned ? 0 : 1);
    const int64_t cap = (!bwd && (vec == 4 || aligned)) ? 256 * 8 : 256 * 5;  // widest shapes (see launch_t)
    return need <= cap;
}

cudaError_t launch_fwd_warp(const FwdArgs &a, int dtype, bool aligned, cudaStream_t st)
{
    if (a.mask_bool) return launch_fwd_warp_bool(a, dtype, aligned, st);
    return dispatch<false, false>(a, dtype, aligned, st);
}

cudaError_t launch_bwd_warp(const BwdArgs &a, int dtype, bool aligned, cudaStream_t st)
{
    return dispatch<true, false>(a, dtype, aligned, st);
}

}  // namespace sms
