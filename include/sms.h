/*
 * sms.h - C ABI of libsms, the GB300 (sm_103a) fused ScaledMaskSoftmax library.
 *
 * The operation is defined on the page "用CUDA自定义融合Softmax算子并封装进PyTorch"
 * (lmnt.cn/news/346102):
 *   forward  (§1.2 formula, §2.1 max-subtracted form, §2.2 additive mask plus
 *             causal flag, §3.1 kernel: causal applied after the mask add)
 *       s_j = x_j * scale + mask_j ;  s_j = -inf if is_causal and j > q
 *       y_j = exp(s_j - max_k s_k) / sum_k exp(s_k - max_k s_k)
 *   backward (§3.3 Jacobian derivation)
 *       dot = sum_j dy_j * y_j ;  dx_j = (dy_j - dot) * y_j * scale
 * A row whose every score is -inf yields y = 0 (the second article,
 * pnsm.cn/news/1983787, §4.2 table and §4.3 pitfall 1: never divide such a
 * row; the all-zero choice is taken).
 *
 * Layout.  Every tensor is a dense row-major [rows, cols] view of the
 * [B, H, S_q, S_k] score tensor with cols = S_k and rows = B*H*S_q (the page's
 * §4.2 "rows = numel / size(-1)" view).  Row r has query position q = r mod cols
 * (the page's §3.1 kernel: S_q = S_k), head h = (r / cols) mod heads and batch
 * b = r / (cols * heads).  rows need not be a multiple of cols.
 *
 * Mask.  The additive mask has the dtype of x.  Row r reads the `cols`
 * contiguous mask elements starting at
 *       b * mask_stride_b + h * mask_stride_h + q * cols
 * so [S,S] is (0, 0), [B,1,S,S] is (S*S, 0) and [B,H,S,S] is (H*S*S, S*S)
 * (the second article's §2.1 input contract).  mask == NULL means no mask
 * (the page's §2.2: an empty mask means none); then the strides, heads and
 * mask_numel are ignored.  The mask is not scaled: only x is.
 *
 * Numerics.  Inputs are widened to fp32, every step runs in fp32, and the
 * result is rounded once to the output dtype (round to nearest even) - the
 * page's §6.3 advice.  Masked and causal positions are written as exact 0.
 *
 * Ownership and streams.  The caller owns every buffer; they are device
 * pointers (cudaMalloc / PyTorch allocations) on the current device.  The
 * library allocates nothing, never synchronises, and enqueues its kernels on
 * `stream` (a cudaStream_t passed as void*, NULL = legacy default stream), so
 * the caller must pass the stream its tensors are used on (the second
 * article's §4.3 pitfall 3).  Calls are asynchronous: a SMS_OK return means the
 * launch was accepted.
 *
 * Graphs.  Every launch goes on `stream`, so calls can be captured into a CUDA
 * graph (the second article's §1.1 and §4.4 on launch overhead).  Make one
 * eager call per shape and kernel family before capturing, from the host
 * thread that captures: it does that kernel's one-time set-up (the shared-
 * memory limit of the kernel, once per device and host thread; the occupancy
 * query and the device error word's address, once per device), which must
 * not happen during a capture.
 *
 * Alignment.  x, y, mask, dy and dx must be 16-byte aligned (every CUDA / PyTorch
 * allocation is); rows may start at any element.
 *
 * Errors.  Functions return an sms_status; nothing is thrown across the ABI and
 * no CUDA error is left pending by a rejected call.  Arguments are validated on
 * the host before any launch:
 *   SMS_ERR_INVALID_ARG  NULL x/y (dy/dx), rows < 0, cols <= 0, heads <= 0,
 *                        unknown dtype, non-finite scale, an unaligned pointer,
 *                        negative mask strides, a mask extent beyond mask_numel,
 *                        element counts beyond 2^60, or an output that overlaps
 *                        an input without being the same buffer.
 *   SMS_ERR_UNSUPPORTED  a forced path that cannot take the shape.
 *   SMS_ERR_CUDA         the launch failed (cudaGetLastError after the launch).
 * sms_last_error() gives a one-line description of the last failure on the
 * calling host thread.
 */
#ifndef SMS_H
#define SMS_H

#include <stdint.h>

/* Only the entry points below are exported; everything else in the library
 * is hidden, so two copies of libsms in one process share no state. */
#if defined(__GNUC__)
#define SMS_API __attribute__((visibility("default")))
#else
#define SMS_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { SMS_F32 = 0, SMS_F16 = 1, SMS_BF16 = 2 } sms_dtype;

typedef enum {
    SMS_OK = 0,
    SMS_ERR_INVALID_ARG = 1,
    SMS_ERR_UNSUPPORTED = 2,
    SMS_ERR_CUDA = 3
} sms_status;

/* Kernel families; SMS_PATH_AUTO lets the dispatcher choose by row width. */
typedef enum {
    SMS_PATH_AUTO = 0,
    SMS_PATH_WARP = 1,   /* rows held in registers by a warp (or part of one)          */
    SMS_PATH_CTA = 2,    /* persistent CTA per row, rows staged by bulk (TMA) copies   */
    SMS_PATH_ONLINE = 3, /* streaming two pass: online max/sum, then re-read and write */
    SMS_PATH_STREAM = 4, /* persistent lane groups, rows in registers, next row prefetched */
    SMS_PATH_RING = 5    /* a warp per row, fed by its own ring of bulk (TMA) copies       */
} sms_path;

/*
 * Forward.  y[r, j] = softmax_j(x[r, :] * scale + mask_row(r)) with the causal
 * override, for r < rows, j < cols (see the top of this file).
 *   x, y           [rows, cols] device buffers of `dtype`; y may equal x (in place)
 *   mask           NULL or the additive mask (device, `dtype`), mask_numel elements
 *   mask_stride_b  elements between batches of the mask (0 = broadcast)
 *   mask_stride_h  elements between heads of the mask (0 = broadcast)
 *   heads          H of the [B,H,S,S] view (>= 1); only used to locate mask rows
 *   scale          multiplier of x (finite), typically 1/sqrt(d_k)
 *   is_causal      nonzero: positions j > q are masked
 *   stream         cudaStream_t
 * rows == 0 (with cols >= 1) is a valid no-op; the pointers may then be NULL.
 */
SMS_API int sms_forward(const void *x, const void *mask, int64_t mask_numel, int64_t mask_stride_b,
                int64_t mask_stride_h, int64_t heads, void *y, int64_t rows, int64_t cols, float scale,
                int is_causal, int dtype, void *stream);

/*
 * Forward with a boolean mask.  The page "用CUDA自定义融合Softmax算子并封装进PyTorch"
 * §2.2 starts from a boolean mask (true = the key is masked) and turns it into
 * the additive one as mask * (-inf) before the kernel; the second article
 * (pnsm.cn/news/1983787, §2.3) has the operator read a 0/1 mask itself and
 * use -inf where it is 1.  Here the kernel reads the boolean mask, one byte
 * per element:
 *       s_j = -inf if mask_row(r)[j] != 0, else x_j * scale
 *       s_j = -inf if is_causal and j > q;  y as in sms_forward
 * which is bit for bit sms_forward with the additive mask holding -inf where
 * the byte is nonzero and 0 elsewhere, at a quarter (fp32) or half (fp16,
 * bf16) of that mask's bytes.  A row with every key masked gives y = 0.
 *   mask      device array of mask_numel bytes (torch.bool / uint8 storage),
 *             16-byte aligned, not NULL; any nonzero byte masks its key
 *   mask_stride_b, mask_stride_h, heads
 *             as in sms_forward, in elements (= bytes) of the mask
 *   other arguments as sms_forward; y may equal x and must not overlap the mask.
 * The backward is sms_backward (the mask only shapes y).
 * Every kernel family reads the boolean mask (the staged CTA family stages
 * its bytes with the scores), and the dispatcher chooses as for sms_forward.
 * Errors as sms_forward, plus SMS_ERR_INVALID_ARG for a NULL mask (rows > 0).
 */
SMS_API int sms_forward_bool(const void *x, const uint8_t *mask, int64_t mask_numel, int64_t mask_stride_b,
                             int64_t mask_stride_h, int64_t heads, void *y, int64_t rows, int64_t cols, float scale,
                             int is_causal, int dtype, void *stream);

/*
 * Backward.  dx[r, j] = (dy[r, j] - sum_k dy[r, k] * y[r, k]) * y[r, j] * scale.
 *   y              forward output [rows, cols] (device, `dtype`)
 *   dy             upstream gradient [rows, cols] (device, `dtype`)
 *   dx             result [rows, cols] (device, `dtype`); may equal dy (in place)
 *   is_causal_hint nonzero promises that y[r, j] == 0 for every j > q (true for a
 *                  forward run with is_causal); the kernels then skip reading y
 *                  and dy there and write dx = +0.  For finite dy the result equals
 *                  the unhinted one up to the rounding of the row sum's
 *                  summation order; positions with y == 0 are +0 either way.
 * rows == 0 (with cols >= 1) is a valid no-op; the pointers may then be NULL.
 */
SMS_API int sms_backward(const void *y, const void *dy, void *dx, int64_t rows, int64_t cols, float scale,
                 int is_causal_hint, int dtype, void *stream);

/*
 * Key-padding forward with per-batch lengths.  The second article
 * (pnsm.cn/news/1983787) lists key-padding masks among the masks to fuse
 * (§2.1 input contract, §4.4 and §5 on fusing several mask kinds), and the
 * page "用CUDA自定义融合Softmax算子并封装进PyTorch" §2.2 defines a padded key as
 * one whose score is -inf.  Here the padding is given by lengths instead of an
 * additive [B,1,S,S] tensor: row r of batch b = r / (heads * cols) keeps the
 * keys j < L_b, L_b = lengths[b] clamped to [0, cols]:
 *       s_j = x_j * scale            for j < L_b,   s_j = -inf  for j >= L_b
 *       s_j = -inf if is_causal and j > q;  y as in sms_forward
 * which equals sms_forward with a [B,1,S,S] mask holding 0 for j < L_b and
 * -inf beyond.  A row with no kept key (L_b = 0) gives y = 0.  x is never
 * read at j >= L_b, and no mask tensor is read at all.
 *   lengths  device int32 array, 4-byte aligned, at least
 *            ceil(rows / (heads * cols)) entries (one per batch); the caller
 *            keeps it unchanged until the kernel has run
 *   heads    H of the [B,H,S,S] view (>= 1): locates b
 *   other arguments as sms_forward (x, y, rows, cols, scale, is_causal, dtype,
 *   stream); y may equal x, and must not overlap lengths.
 * Errors as sms_forward, plus SMS_ERR_INVALID_ARG for a NULL or unaligned
 * lengths pointer.
 */
SMS_API int sms_forward_lengths(const void *x, const int32_t *lengths, int64_t heads, void *y, int64_t rows,
                                int64_t cols, float scale, int is_causal, int dtype, void *stream);

/*
 * Backward of sms_forward_lengths: sms_backward with a key-length hint.  The
 * caller promises y[r, j] == 0 for j >= L_b (true for a forward run with the
 * same lengths); the kernels skip reading y and dy there and write dx = +0,
 * as under is_causal_hint (which may be combined with it).  The result equals
 * sms_backward's up to the rounding of the row sum's summation order.
 * lengths and heads as in sms_forward_lengths; dx must not overlap lengths.
 */
SMS_API int sms_backward_lengths(const void *y, const void *dy, void *dx, const int32_t *lengths, int64_t heads,
                                 int64_t rows, int64_t cols, float scale, int is_causal_hint, int dtype,
                                 void *stream);

/*
 * Fused attention forward on the tensor cores: the step the second article
 * (pnsm.cn/news/1983787) names as next in §4.4 and the page
 * "从GEMM到Transformer：手写CUDA算子优化的完整路线与性能调优实践" computes in §2.2
 * (scores, softmax and the product with V in one kernel, with the streaming
 * max / sum of that section, so the [S, S] score tensor is never stored):
 *       O[b,h] = softmax_j(Q[b,h] K[b,h]^T * scale + mask_row, causal) V[b,h]
 * with the softmax of sms_forward (the mask is not scaled; j > i is masked
 * under is_causal; a row with every key masked gives O = 0).
 *   q, k, v, o     dense [batch, heads, seq, head_dim] device buffers of `dtype`
 *                  (SMS_F16 or SMS_BF16), 16-byte aligned; o must not overlap
 *                  an input
 *   mask           NULL, or a mask in the layout of sms_forward: query row i of
 *                  head (b, h) reads the seq elements from
 *                  b*mask_stride_b + h*mask_stride_h + i*seq; additive of
 *                  `dtype` (mask_is_bool = 0) or one byte per element with
 *                  nonzero = masked (mask_is_bool = 1); mask_numel elements
 *   lse            NULL, or [batch, heads, seq] fp32: per query row the natural
 *                  log of the softmax denominator, log sum_j exp(s_j) (-inf for
 *                  a row with every key masked), which the backward reads
 *   head_dim       64 or 128
 *   scale          multiplier of Q K^T (finite), typically 1/sqrt(head_dim)
 * Arithmetic: Q K^T and P V on tcgen05.mma with fp32 accumulation in tensor
 * memory; the softmax in fp32; P is rounded to `dtype` before P V; O is
 * rounded once to `dtype`.  batch * heads * seq == 0 is a valid no-op.
 * Errors: SMS_ERR_UNSUPPORTED for SMS_F32 or another head_dim;
 * SMS_ERR_INVALID_ARG for NULL or unaligned pointers, negative sizes or
 * strides, a mask extent beyond mask_numel, overlapping outputs, a
 * non-finite scale; SMS_ERR_CUDA when the launch fails.  A bounded wait that
 * gives up inside the kernel sets SMS_DEVERR_ATTN_WAIT (sms_device_error).
 */
SMS_API int sms_attention_forward(const void *q, const void *k, const void *v, const void *mask, int64_t mask_numel,
                                  int64_t mask_stride_b, int64_t mask_stride_h, int mask_is_bool, void *o,
                                  float *lse, int64_t batch, int64_t heads, int64_t seq, int64_t head_dim,
                                  float scale, int is_causal, int dtype, void *stream);

/*
 * Backward of sms_attention_forward: dQ, dK and dV of sum(dO * O), by the
 * chain rule through the three steps (the softmax Jacobian of the page
 * "用CUDA自定义融合Softmax算子并封装进PyTorch" §3.3 in the middle):
 *       P = softmax(...) recomputed from q, k, the mask and lse;
 *       dV = P^T dO,  dP = dO V^T,  dS = scale * P * (dP - rowsum(dO * O)),
 *       dQ = dS K,    dK = dS^T Q.
 *   q, k, v, mask, scale, is_causal, sizes, dtype   as given to the forward
 *   o, lse          the forward's outputs
 *   d_o             the upstream gradient [batch, heads, seq, head_dim]
 *   dq, dk, dv      results, same shape and dtype; none may overlap another
 *                   buffer
 *   workspace       caller-owned device scratch of at least
 *                   sms_attention_backward_workspace() bytes, 16-byte aligned
 *                   (an fp32 dQ accumulator padded to whole blocks of 128
 *                   queries, and an fp32 value per query row);
 *                   its contents on entry do not matter, and it must not be
 *                   used by anything else until the call's kernels are done
 * Three kernels are enqueued on `stream`.  Arithmetic: the five products on
 * tcgen05.mma with fp32 accumulation; P and dS are rounded to `dtype` as MMA
 * operands; dQ accumulates in fp32 across key blocks; every gradient is
 * rounded once to `dtype`.  Errors as sms_attention_forward, plus
 * SMS_ERR_INVALID_ARG for a missing or small workspace.
 */
SMS_API int sms_attention_backward(const void *q, const void *k, const void *v, const void *o, const void *d_o,
                                   const float *lse, const void *mask, int64_t mask_numel, int64_t mask_stride_b,
                                   int64_t mask_stride_h, int mask_is_bool, void *dq, void *dk, void *dv,
                                   void *workspace, int64_t workspace_bytes, int64_t batch, int64_t heads,
                                   int64_t seq, int64_t head_dim, float scale, int is_causal, int dtype,
                                   void *stream);

/* Bytes of workspace sms_attention_backward needs (-1 for a negative size). */
SMS_API int64_t sms_attention_backward_workspace(int64_t batch, int64_t heads, int64_t seq, int64_t head_dim);

/*
 * sms_attention_backward for callers that cannot allocate device memory: a
 * process whose memory is owned by a framework or pool it cannot call into,
 * code that runs where an allocation could block or fail at the wrong time
 * (inside a captured region, an interrupt-like callback, a real-time loop), or
 * a plain C caller with no allocator at hand.  The source pages have no
 * counterpart: this is an addition of the library.
 * Same arguments, kernels and results as sms_attention_backward, without the
 * workspace: the scratch (the fp32 dQ accumulator and one fp32 per query row,
 * sms_attention_backward_workspace() bytes) lives in one array of
 * SMS_ATTN_STATIC_SCRATCH_BYTES inside the library's device image, which
 * every GPU that loads the library holds until the process exits.
 *   - A problem needing more scratch than that is refused with
 *     SMS_ERR_INVALID_ARG before anything is launched (use the workspace entry
 *     point for it).
 *   - No call allocates: not the library, not the CUDA runtime on its behalf.
 *   - The first call on a device looks up the array's device address there
 *     (cudaGetSymbolAddress, with that device current); make that first call
 *     before any stream capture on that device.
 *   - Every call uses the same array and leaves its contents behind; the
 *     kernels clear the accumulator themselves before use.  Calls whose
 *     kernels overlap on the GPU (other streams, other host threads) race on
 *     the array: order them on one stream.
 */
#define SMS_ATTN_STATIC_SCRATCH_BYTES (32ll << 20)
SMS_API int sms_attention_backward_static(const void *q, const void *k, const void *v, const void *o,
                                          const void *d_o, const float *lse, const void *mask, int64_t mask_numel,
                                          int64_t mask_stride_b, int64_t mask_stride_h, int mask_is_bool, void *dq,
                                          void *dk, void *dv, int64_t batch, int64_t heads, int64_t seq,
                                          int64_t head_dim, float scale, int is_causal, int dtype, void *stream);

/* Static description of a status code. */
SMS_API const char *sms_status_string(int status);

/* One-line description of the last failure on this host thread ("" if none). */
SMS_API const char *sms_last_error(void);

/*
 * Force every later call in this process onto one kernel family (testing and
 * benchmarking); SMS_PATH_AUTO restores the dispatcher.  Returns the previous
 * setting, or -1 for an unknown path.  Process-wide, not thread-safe.
 */
SMS_API int sms_set_forced_path(int path);

/*
 * Cap the CTAs of the persistent kernel families (SMS_PATH_STREAM, SMS_PATH_RING,
 * SMS_PATH_CTA, SMS_PATH_ONLINE)
 * at `ctas` (0 = as many as the device holds, the default): each CTA then
 * walks more rows, which lets small tests cover multi-row pipelines.
 * Returns the previous cap, or -1 for a negative argument.  Process-wide.
 */
SMS_API int sms_set_grid_limit(int ctas);

/*
 * Test control of the bounded-wait abort path (process-wide; 0 = off, the
 * default).  With ns > 0, every lane group of the SMS_PATH_RING kernels makes
 * its first wait one on a barrier that nothing ever arrives at, bounded at ns
 * nanoseconds instead of 2 s: the wait gives up, the kernel records
 * SMS_DEVERR_RING_WAIT, waits (bounded at 2 s) for the bulk copies it has in
 * flight and returns without finishing its rows.  Returns the previous value,
 * or -1 for ns outside [0, 1e9].
 */
SMS_API int64_t sms_set_test_stall(int64_t ns);

/* The family the dispatcher would pick for this forward (or backward) shape of non-causal rows. */
SMS_API int sms_select_path(int64_t rows, int64_t cols, int dtype, int is_backward);

/* The family taken by the last successful call on this host thread. */
SMS_API int sms_last_path(void);

/*
 * Number of kernel launches made by successful calls since load, process-wide
 * (each sms_forward / sms_backward enqueues exactly one kernel when rows > 0).
 */
SMS_API int64_t sms_launch_count(void);

/* Values of the device error word (sms_device_error): which bounded wait of a
 * kernel fed by bulk (TMA) copies gave up.  The first failure is kept. */
typedef enum {
    SMS_DEVERR_NONE = 0,
    SMS_DEVERR_CTA_CONSUMER_WAIT = 1, /* SMS_PATH_CTA: a consumer group waited for a staged row  */
    SMS_DEVERR_CTA_PRODUCER_WAIT = 2, /* SMS_PATH_CTA: the producer waited for a free stage      */
    SMS_DEVERR_RING_WAIT = 3,         /* SMS_PATH_RING: a lane group waited for its own copies   */
    SMS_DEVERR_ATTN_WAIT = 4          /* fused attention: a role waited for a copy, an MMA or a peer */
} sms_device_error_code;

/*
 * Reads (and clears) the device-side error word of the current device after
 * synchronising `stream`.  Nonzero (an sms_device_error_code) means a kernel
 * gave up on a bounded wait (2 s) for its own bulk copies; it then stopped
 * taking rows, waited (bounded) for the copies it had in flight and left, so
 * its output is incomplete but the context stays usable.  Returns -1 if the
 * read itself failed.
 */
SMS_API int sms_device_error(void *stream);

/* ABI version: 100 * major + minor. */
SMS_API int sms_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SMS_H */
