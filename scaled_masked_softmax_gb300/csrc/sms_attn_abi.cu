// C ABI of the fused attention step (include/sms.h: sms_attention_forward,
// sms_attention_backward, sms_attention_backward_workspace): host-side
// validation, then the tensor-core kernels of sms_attn_fwd.cu /
// sms_attn_bwd.cu.
#include <cmath>
#include <cstdio>

#include "sms.h"
#include "sms_attn.h"
#include "sms_internal.h"

namespace sms {
namespace {

bool al16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool overlap(const void *a, int64_t na, const void *b, int64_t nb)
{
    if (!a || !b || na <= 0 || nb <= 0) return false;
    const uintptr_t pa = reinterpret_cast<uintptr_t>(a), pb = reinterpret_cast<uintptr_t>(b);
    return pa < pb + (uintptr_t)nb && pb < pa + (uintptr_t)na;
}

int fail(int status, const char *who, const char *what)
{
    char buf[256];
    snprintf(buf, sizeof(buf), "%s: %s", who, what);
    return set_last_error(status, buf);
}

// Shape, dtype, pointer and mask checks shared by the forward and the backward.
int check_common(const char *who, const void *q, const void *k, const void *v, const void *mask, int64_t mask_numel,
                 int64_t msb, int64_t msh, int mask_is_bool, int64_t B, int64_t H, int64_t S, int64_t D, float scale,
                 int dtype, bool &empty)
{
    empty = false;
    if (dtype != SMS_F16 && dtype != SMS_BF16)
        return fail(dtype == SMS_F32 ? SMS_ERR_UNSUPPORTED : SMS_ERR_INVALID_ARG, who,
                    "dtype must be SMS_F16 or SMS_BF16 (the tensor-core path)");
    if (B < 0 || H < 0 || S < 0) return fail(SMS_ERR_INVALID_ARG, who, "batch, heads and seq must be >= 0");
    if (!attn_head_dim_ok((int)D) || D != (int64_t)(int)D)
        return fail(SMS_ERR_UNSUPPORTED, who, "head_dim must be 64 or 128");
    if (B == 0 || H == 0 || S == 0) {
        empty = true;
        return SMS_OK;
    }
    if (S > (1 << 24) || B * H > (1 << 24) || B * H * ((S + 127) / 128) > 0x7fffffffll)
        return fail(SMS_ERR_INVALID_ARG, who, "problem too large (seq <= 2^24, batch*heads <= 2^24)");
    if (!std::isfinite(scale)) return fail(SMS_ERR_INVALID_ARG, who, "scale must be finite");
    if (!q || !k || !v) return fail(SMS_ERR_INVALID_ARG, who, "q, k and v must not be NULL");
    if (!al16(q) || !al16(k) || !al16(v)) return fail(SMS_ERR_INVALID_ARG, who, "q, k and v must be 16-byte aligned");
    if (mask) {
        if (msb < 0 || msh < 0) return fail(SMS_ERR_INVALID_ARG, who, "mask strides must be >= 0");
        if (!al16(mask)) return fail(SMS_ERR_INVALID_ARG, who, "mask must be 16-byte aligned");
        const double ext = (double)(B - 1) * (double)msb + (double)(H - 1) * (double)msh + (double)S * (double)S;
        if (mask_numel < 0 || ext > (double)mask_numel)
            return fail(SMS_ERR_INVALID_ARG, who, "the mask rows reach beyond mask_numel");
    }
    (void)mask_is_bool;
    return SMS_OK;
}

int launch_result(cudaError_t e, const char *who, const char *step)
{
    if (e == cudaSuccess) {
        count_launch();
        return SMS_OK;
    }
    cudaGetLastError();
    char buf[200];
    snprintf(buf, sizeof(buf), "%s failed: %s (%s)", step ? step : "launch", cudaGetErrorString(e),
             cudaGetErrorName(e));
    return fail(e == cudaErrorNotSupported ? SMS_ERR_UNSUPPORTED : SMS_ERR_CUDA, who, buf);
}

}  // namespace
}  // namespace sms

using namespace sms;

extern "C" {

int sms_attention_forward(const void *q, const void *k, const void *v, const void *mask, int64_t mask_numel,
                          int64_t mask_stride_b, int64_t mask_stride_h, int mask_is_bool, void *o, float *lse,
                          int64_t batch, int64_t heads, int64_t seq, int64_t head_dim, float scale, int is_causal,
                          int dtype, void *stream)
{
    const char *who = "sms_attention_forward";
    clear_last_error();
    bool empty = false;
    int rc = check_common(who, q, k, v, mask, mask_numel, mask_stride_b, mask_stride_h, mask_is_bool, batch, heads,
                          seq, head_dim, scale, dtype, empty);
    if (rc != SMS_OK || empty) return rc;
    if (!o || !al16(o)) return fail(SMS_ERR_INVALID_ARG, who, "o must be a 16-byte aligned, non-NULL pointer");
    if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) return fail(SMS_ERR_INVALID_ARG, who, "lse must be 4-byte aligned");
    const int64_t nt = batch * heads * seq * head_dim * 2;
    const int64_t nm = mask ? mask_numel * (mask_is_bool ? 1 : 2) : 0;
    if (overlap(o, nt, q, nt) || overlap(o, nt, k, nt) || overlap(o, nt, v, nt) || overlap(o, nt, mask, nm))
        return fail(SMS_ERR_INVALID_ARG, who, "o overlaps an input");
    const int64_t nl = batch * heads * seq * 4;
    if (lse && (overlap(lse, nl, o, nt) || overlap(lse, nl, q, nt) || overlap(lse, nl, k, nt) ||
                overlap(lse, nl, v, nt) || overlap(lse, nl, mask, nm)))
        return fail(SMS_ERR_INVALID_ARG, who, "lse overlaps another buffer");
    int *err = nullptr;
    cudaError_t e = device_error_word(&err);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(SMS_ERR_CUDA, who, "device query failed");
    }
    AttnArgs a = {};
    a.q = q; a.k = k; a.v = v;
    a.mask = mask; a.mask_total = mask ? mask_numel : 0; a.msb = mask_stride_b; a.msh = mask_stride_h;
    a.mask_bool = (mask && mask_is_bool) ? 1 : 0;
    a.B = (int)batch; a.H = (int)heads; a.S = (int)seq; a.D = (int)head_dim;
    a.scale = scale; a.causal = is_causal ? 1 : 0; a.dtype = dtype; a.err = err;
    a.o = o; a.lse = lse;
    const char *step = nullptr;
    const cudaError_t e2 = launch_attn_fwd(a, static_cast<cudaStream_t>(stream), &step);
    return launch_result(e2, who, step);
}

int64_t sms_attention_backward_workspace(int64_t batch, int64_t heads, int64_t seq, int64_t head_dim)
{
    if (batch < 0 || heads < 0 || seq < 0 || head_dim < 0) return -1;
    // fp32 dQ accumulator in whole query blocks, then fp32 delta per query row
    return attn_bwd_acc_rows(batch, heads, seq) * head_dim * 4 + batch * heads * seq * 4;
}

int sms_attention_backward(const void *q, const void *k, const void *v, const void *o, const void *d_o,
                           const float *lse, const void *mask, int64_t mask_numel, int64_t mask_stride_b,
                           int64_t mask_stride_h, int mask_is_bool, void *dq, void *dk, void *dv, void *workspace,
                           int64_t workspace_bytes, int64_t batch, int64_t heads, int64_t seq, int64_t head_dim,
                           float scale, int is_causal, int dtype, void *stream)
{
    const char *who = "sms_attention_backward";
    clear_last_error();
    bool empty = false;
    int rc = check_common(who, q, k, v, mask, mask_numel, mask_stride_b, mask_stride_h, mask_is_bool, batch, heads,
                          seq, head_dim, scale, dtype, empty);
    if (rc != SMS_OK || empty) return rc;
    if (!o || !d_o || !al16(o) || !al16(d_o)) return fail(SMS_ERR_INVALID_ARG, who, "o and d_o must be 16-byte aligned, non-NULL");
    if (!lse || (reinterpret_cast<uintptr_t>(lse) & 3u)) return fail(SMS_ERR_INVALID_ARG, who, "lse must be a 4-byte aligned, non-NULL pointer");
    if (!dq || !dk || !dv || !al16(dq) || !al16(dk) || !al16(dv))
        return fail(SMS_ERR_INVALID_ARG, who, "dq, dk and dv must be 16-byte aligned, non-NULL");
    const int64_t need = sms_attention_backward_workspace(batch, heads, seq, head_dim);
    if (!workspace || !al16(workspace) || workspace_bytes < need)
        return fail(SMS_ERR_INVALID_ARG, who, "workspace must be 16-byte aligned with at least "
                                              "sms_attention_backward_workspace() bytes");
    const int64_t nt = batch * heads * seq * head_dim * 2, nl = batch * heads * seq * 4;
    const int64_t nm = mask ? mask_numel * (mask_is_bool ? 1 : 2) : 0;
    const void *ins[] = {q, k, v, o, d_o};
    void *outs[] = {dq, dk, dv};
    for (void *w : outs) {
        for (const void *x : ins)
            if (overlap(w, nt, x, nt)) return fail(SMS_ERR_INVALID_ARG, who, "a gradient overlaps an input");
        if (overlap(w, nt, lse, nl) || overlap(w, nt, mask, nm) || overlap(w, nt, workspace, need))
            return fail(SMS_ERR_INVALID_ARG, who, "a gradient overlaps lse, the mask or the workspace");
    }
    if (overlap(dq, nt, dk, nt) || overlap(dq, nt, dv, nt) || overlap(dk, nt, dv, nt))
        return fail(SMS_ERR_INVALID_ARG, who, "dq, dk and dv overlap");
    for (const void *x : ins)
        if (overlap(workspace, need, x, nt)) return fail(SMS_ERR_INVALID_ARG, who, "the workspace overlaps an input");
    if (overlap(workspace, need, lse, nl) || overlap(workspace, need, mask, nm))
        return fail(SMS_ERR_INVALID_ARG, who, "the workspace overlaps lse or the mask");
    int *err = nullptr;
    cudaError_t e = device_error_word(&err);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(SMS_ERR_CUDA, who, "device query failed");
    }
    AttnArgs a = {};
    a.q = q; a.k = k; a.v = v;
    a.mask = mask; a.mask_total = mask ? mask_numel : 0; a.msb = mask_stride_b; a.msh = mask_stride_h;
    a.mask_bool = (mask && mask_is_bool) ? 1 : 0;
    a.B = (int)batch; a.H = (int)heads; a.S = (int)seq; a.D = (int)head_dim;
    a.scale = scale; a.causal = is_causal ? 1 : 0; a.dtype = dtype; a.err = err;
    a.o_in = o; a.dout = d_o; a.lse_in = lse;
    a.dq = dq; a.dk = dk; a.dv = dv;
    a.dq_acc = static_cast<float *>(workspace);
    a.delta = reinterpret_cast<float *>(static_cast<char *>(workspace) + attn_bwd_acc_rows(batch, heads, seq) * head_dim * 4);
    const char *step = nullptr;
    e = launch_attn_bwd(a, static_cast<cudaStream_t>(stream), &step);
    if (e == cudaSuccess) {  // three kernels: delta, the main pass, dQ
        count_launch();
        count_launch();
    }
    return launch_result(e, who, step);
}

}  // extern "C"
