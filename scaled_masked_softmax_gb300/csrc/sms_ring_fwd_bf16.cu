// Forward ring kernels for __nv_bfloat16 rows (every mask kind and alignment).
#include "sms_ring.cuh"

namespace sms {

cudaError_t ring_fwd_bf16(const FwdArgs &a, bool aligned, cudaStream_t st)
{
    return launch_dt<__nv_bfloat16, false>(a, BwdArgs{}, aligned, st);
}

}  // namespace sms
