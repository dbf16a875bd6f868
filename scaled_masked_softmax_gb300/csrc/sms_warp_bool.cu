// Register-resident forward kernels for a boolean mask (one byte per element,
// nonzero = masked key), the boolean form of the mask on the page
// "用CUDA自定义融合Softmax算子并封装进PyTorch" §2.2, read in-kernel instead of
// being converted to an additive tensor first.  Same lane shapes and row
// routine as the additive forward (sms_warp.cuh); only the mask loads differ:
// VEC bytes under each 16-byte x vector, widened to 0 / -inf in registers.
#include "sms_warp.cuh"

namespace sms {

cudaError_t launch_fwd_warp_bool(const FwdArgs &a, int dtype, bool aligned, cudaStream_t st)
{
    return dispatch<false, true>(a, dtype, aligned, st);
}

}  // namespace sms
