// Forward ring kernels for float rows (every mask kind and alignment).
#include "sms_ring.cuh"

namespace sms {

cudaError_t ring_fwd_f32(const FwdArgs &a, bool aligned, cudaStream_t st)
{
    return launch_dt<float, false>(a, BwdArgs{}, aligned, st);
}

}  // namespace sms
