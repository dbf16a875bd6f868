// Attention backward for callers that cannot allocate device memory: the same
// kernels as sms_attention_backward, with the scratch taken from a
// fixed-size array in this library's device image instead of a
// caller-supplied workspace (see sms_attention_backward_static in sms.h).
#include <atomic>
#include <cstdio>
#include <mutex>

#include "sms.h"
#include "sms_attn.h"
#include "sms_internal.h"

namespace sms {
namespace {

// The scratch of every call: the fp32 dQ accumulator, then one fp32 per query
// row.  Every GPU that loads the library holds it until the process exits.
constexpr int64_t kStaticScratchBytes = SMS_ATTN_STATIC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_attn_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::once_flag g_once[kMaxDevices];
void *g_addr[kMaxDevices];
cudaError_t g_status[kMaxDevices];

// Device address of the array on the current device, looked up once per
// device with that device current (host code only sees a stand-in symbol).
cudaError_t scratch_address(void **p)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::call_once(g_once[dev], [dev] {
        void *a = nullptr;
        g_status[dev] = cudaGetSymbolAddress(&a, g_attn_scratch);
        g_addr[dev] = a;
    });
    *p = g_addr[dev];
    return g_status[dev];
}

}  // namespace
}  // namespace sms

extern "C" int sms_attention_backward_static(const void *q, const void *k, const void *v, const void *o,
                                             const void *d_o, const float *lse, const void *mask, int64_t mask_numel,
                                             int64_t mask_stride_b, int64_t mask_stride_h, int mask_is_bool,
                                             void *dq, void *dk, void *dv, int64_t batch, int64_t heads, int64_t seq,
                                             int64_t head_dim, float scale, int is_causal, int dtype, void *stream)
{
    using namespace sms;
    const int64_t need = sms_attention_backward_workspace(batch, heads, seq, head_dim);
    if (need > kStaticScratchBytes) {
        char buf[200];
        snprintf(buf, sizeof(buf),
                 "sms_attention_backward_static: the problem needs %lld bytes of scratch, above the %lld of the "
                 "library's static array; use sms_attention_backward with a workspace",
                 (long long)need, (long long)kStaticScratchBytes);
        return set_last_error(SMS_ERR_INVALID_ARG, buf);
    }
    void *scratch = nullptr;
    if (need > 0) {
        const cudaError_t e = scratch_address(&scratch);
        if (e != cudaSuccess || !scratch) {
            cudaGetLastError();
            return set_last_error(SMS_ERR_CUDA, "sms_attention_backward_static: cudaGetSymbolAddress of the static "
                                                "scratch failed");
        }
    }
    return sms_attention_backward(q, k, v, o, d_o, lse, mask, mask_numel, mask_stride_b, mask_stride_h, mask_is_bool,
                                  dq, dk, dv, scratch, kStaticScratchBytes, batch, heads, seq, head_dim, scale,
                                  is_causal, dtype, stream);
}
