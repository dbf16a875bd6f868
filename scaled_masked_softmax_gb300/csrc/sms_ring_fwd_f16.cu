// Forward ring kernels for __half rows (every mask kind and alignment).
#include "sms_ring.cuh"

namespace sms {

cudaError_t ring_fwd_f16(const FwdArgs &a, bool aligned, cudaStream_t st)
{
    return launch_dt<__half, false>(a, BwdArgs{}, aligned, st);
}

}  // namespace sms
