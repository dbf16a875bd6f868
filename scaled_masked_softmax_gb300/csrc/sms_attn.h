// Host-side interface of the fused attention kernels (sms_attn_fwd.cu,
// sms_attn_bwd.cu) used by the C ABI (sms_attn_abi.cu).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace sms {

// Problem description shared by the forward and the backward.  Q, K, V, O
// (and dO, dQ, dK, dV) are dense [B, H, S, D] tensors of one 16-bit dtype;
// the mask follows the softmax's rule: query row i of head (b, h) reads the
// S mask elements from b*msb + h*msh + i*S.
struct AttnArgs {
    const void *q, *k, *v;
    const void *mask;      // nullptr: none
    int64_t mask_total;    // elements in the mask buffer
    int64_t msb, msh;
    int mask_bool;         // 1: one byte per element, nonzero = masked; 0: additive, dtype of q
    int B, H, S, D;
    float scale;           // multiplier of Q K^T
    int causal;
    int dtype;             // kF16 or kBF16
    int *err;              // device error word
    // forward
    void *o;               // [B, H, S, D]
    float *lse;            // [B, H, S]: log of each row's softmax denominator (natural log, -inf for a
                           // fully masked row), or nullptr
    // backward
    const void *o_in, *dout;
    const float *lse_in;
    void *dq, *dk, *dv;
    float *dq_acc;         // fp32 scratch of attn_bwd_acc_rows() x D (zeroed by the backward before use): one
                           // tile per (batch, head, block of kAttnBwdQueryBlock queries), element (r, c) of a
                           // tile at float ((c / 4) * kAttnBwdQueryBlock + r) * 4 + c % 4
    float *delta;          // [B, H, S] fp32 scratch: rowsum(dO * O)
};

// Queries per block of the backward; its dQ accumulator holds whole blocks.
constexpr int kAttnBwdQueryBlock = 128;
inline int64_t attn_bwd_acc_rows(int64_t B, int64_t H, int64_t S)
{
    return B * H * ((S + kAttnBwdQueryBlock - 1) / kAttnBwdQueryBlock) * kAttnBwdQueryBlock;
}

// Head dimensions the tensor-core kernels take.
inline bool attn_head_dim_ok(int d) { return d == 64 || d == 128; }

// `step` (optional) names the step that failed: a tensor map or a kernel launch.
cudaError_t launch_attn_fwd(const AttnArgs &a, cudaStream_t st, const char **step = nullptr);
cudaError_t launch_attn_bwd(const AttnArgs &a, cudaStream_t st, const char **step = nullptr);

}  // namespace sms
