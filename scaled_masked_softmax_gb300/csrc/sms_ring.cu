// Kernel-family entry points of the bulk-copy ring path (kernels in
// sms_ring.cuh, instantiated in sms_ring_fwd_{f32,f16,bf16}.cu and
// sms_ring_bwd.cu).
#include "sms_ring.cuh"

namespace sms {

bool ring_fits(int64_t cols, int dtype, bool aligned)
{
    const int vec = vec_elems(dtype);
    return (cols + vec - 1) / vec + (aligned ? 0 : 1) <= 2048;
}

cudaError_t launch_fwd_ring(const FwdArgs &a, int dtype, bool aligned, cudaStream_t st)
{
    switch (dtype) {
    case kF32: return ring_fwd_f32(a, aligned, st);
    case kF16: return ring_fwd_f16(a, aligned, st);
    case kBF16: return ring_fwd_bf16(a, aligned, st);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_bwd_ring(const BwdArgs &a, int dtype, bool aligned, cudaStream_t st)
{
    return ring_bwd_any(a, dtype, aligned, st);
}

}  // namespace sms
