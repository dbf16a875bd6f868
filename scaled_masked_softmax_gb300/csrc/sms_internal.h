// Host-side interface between the C ABI (sms_abi.cu) and the kernel families.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "sms_fastdiv.h"

namespace sms {

// dtype codes, equal to sms_dtype in include/sms.h
enum { kF32 = 0, kF16 = 1, kBF16 = 2 };

inline int vec_elems(int dtype) { return dtype == kF32 ? 4 : 8; }
inline int elem_bytes(int dtype) { return dtype == kF32 ? 4 : 2; }

// Mask-reuse row order.  Rows r = k*cols + q of a super-block (the rows that
// share one [cols, cols] mask: every head of every batch when the mask has
// no batch or head stride, the heads of one batch when it has only a batch
// stride) read mask row q.  In the natural order the super-block's blocks
// k read the whole mask one after another, and a mask too large for L2 is
// fetched from HBM once per block.  Reordered, the rows go in tiles of
// kReuseTile query positions, each tile walking every block (the last block
// as far as its `rem` rows reach), so the reads of a mask row come close
// together.  Place n of a super-block maps to (k, q) by three regions of
// tiles: A, tiles the last block covers (kf + 1 blocks of kReuseTile rows);
// B, the one tile it covers in part (or the narrower last tile); C, tiles it
// does not reach (kf blocks each; the final tile may be narrower).
constexpr uint32_t kReuseTile = 64;
struct ReuseOrder {
    int64_t rows;              // places reordered (whole super-blocks); 0: natural order
    uint32_t sb;               // rows per super-block
    uint32_t kf;               // blocks of the super-block before its last one (>= 1)
    uint32_t ta, wb, rem_b;    // region B: tile ta, its width, the last block's rows in it
    uint32_t pa, pb;           // places in regions A and B
    uint32_t base_c, nc, pc;   // region C: first query position, whole tiles, places in them
    FastDiv d_sb, d_a, d_c;    // division by sb, (kf + 1) * kReuseTile and kf * kReuseTile
};

struct FwdArgs {
    const void *x;
    const void *mask;      // nullptr: no mask
    void *y;
    int64_t rows, cols;
    int64_t x_total;       // rows * cols
    int64_t mask_total;    // elements in the mask buffer
    int64_t msb, msh, heads;
    float scale;
    int causal;
    int *err;              // device error word
    FastDiv dcols, dheads; // division by cols and by heads
    const int32_t *lengths;  // per-batch key lengths (device), nullptr: none
    int mask_bool;         // 1: the mask holds one byte per element (nonzero = masked), 0: additive, dtype of x
    uint32_t stall_ns;     // test control (sms_set_test_stall): >0 makes a ring group's first wait one on a
                           // barrier nothing arrives at, bounded at this many ns
    ReuseOrder reuse;      // row order of the register row kernels (fwd_row_kernel)
};

struct BwdArgs {
    const void *y;
    const void *dy;
    void *dx;
    int64_t rows, cols;
    int64_t total;         // rows * cols
    float scale;
    int causal;            // the causal hint: y == 0 beyond the diagonal
    int *err;
    FastDiv dcols;         // division by cols
    const int32_t *lengths;  // key-length hint: y == 0 at j >= lengths[b]; nullptr: none
    int64_t heads;         // heads of the [B,H,S,S] view (locates b for the lengths)
    FastDiv dheads;        // division by heads
    uint32_t stall_ns;     // test control, as in FwdArgs
};

// "aligned" means every row (and every mask row) starts on a 16-byte boundary:
// cols and both mask strides are multiples of the 16-byte vector width.
// A boolean mask (FwdArgs::mask_bool) is taken by every forward family but
// the staged CTA one.

// warp-per-row (or a power-of-two part of a warp per row), rows in registers
bool warp_fits(int64_t cols, int dtype, bool aligned, bool bwd);
cudaError_t launch_fwd_warp(const FwdArgs &a, int dtype, bool aligned, cudaStream_t st);  // either mask kind
cudaError_t launch_fwd_warp_bool(const FwdArgs &a, int dtype, bool aligned, cudaStream_t st);
cudaError_t launch_bwd_warp(const BwdArgs &a, int dtype, bool aligned, cudaStream_t st);


// persistent lane groups walking rows with a one-row register prefetch
bool stream_fits(int64_t cols, int dtype, bool aligned, bool bwd);  // forward: aligned rows only
cudaError_t launch_fwd_stream(const FwdArgs &a, int dtype, bool aligned, cudaStream_t st);
cudaError_t launch_bwd_stream(const BwdArgs &a, int dtype, bool aligned, cudaStream_t st);

// a warp per row, each warp feeding itself through a ring of bulk copies (TMA)
bool ring_fits(int64_t cols, int dtype, bool aligned);
cudaError_t launch_fwd_ring(const FwdArgs &a, int dtype, bool aligned, cudaStream_t st);
cudaError_t launch_bwd_ring(const BwdArgs &a, int dtype, bool aligned, cudaStream_t st);

// persistent CTA per row, bulk-copy (TMA) staging ring, rows in registers
bool cta_fits(int64_t cols, int dtype, bool aligned);      // forward
bool cta_fits_bwd(int64_t cols, int dtype, bool aligned);  // backward (y and dy both held)
cudaError_t launch_fwd_cta(const FwdArgs &a, int dtype, bool aligned, cudaStream_t st);
cudaError_t launch_bwd_cta(const BwdArgs &a, int dtype, bool aligned, cudaStream_t st);

// streaming two pass, any row length (either mask kind)
cudaError_t launch_fwd_online(const FwdArgs &a, int dtype, cudaStream_t st);
cudaError_t launch_bwd_online(const BwdArgs &a, int dtype, cudaStream_t st);

// multiprocessor count of the current device (cached per device)
int sm_count();

// Shared with the attention entry points (sms_attn_abi.cu): the calling
// thread's last-error text, the process-wide launch counter, and the current
// device's error word.
int set_last_error(int status, const char *msg);
void clear_last_error();
void count_launch();
cudaError_t device_error_word(int **err);

// The test control of sms_set_test_stall (0: off).
uint32_t test_stall_ns();

// CTAs for a persistent kernel: `per_sm` per multiprocessor, at most `useful`,
// at most the limit set by sms_set_grid_limit
int64_t persistent_grid(int per_sm, int64_t useful);

}  // namespace sms
