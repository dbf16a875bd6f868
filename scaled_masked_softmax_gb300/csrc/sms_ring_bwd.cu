// Backward ring kernels for every dtype.
#include "sms_ring.cuh"

namespace sms {

cudaError_t ring_bwd_any(const BwdArgs &a, int dtype, bool aligned, cudaStream_t st)
{
    switch (dtype) {
    case kF32: return launch_dt<float, true>(FwdArgs{}, a, aligned, st);
    case kF16: return launch_dt<__half, true>(FwdArgs{}, a, aligned, st);
    case kBF16: return launch_dt<__nv_bfloat16, true>(FwdArgs{}, a, aligned, st);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace sms
