/*
 * fp64 CPU oracle for the fused ScaledMaskSoftmax forward and backward.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the independent definition that the
 * CUDA library is checked against.  Only the test suite, the smoke check and
 * the CPU-baseline / reference arm of the benchmark may load it; the product
 * path never does.  It shares no code, header, table or helper with the CUDA
 * sources: it decodes fp16 / bf16 bit patterns with its own routines and does
 * all arithmetic in IEEE binary64.
 *
 * Source pages (cited as page title + section):
 *   [P2] "用CUDA自定义融合Softmax算子并封装进PyTorch" (lmnt.cn/news/346102)
 *   [P3] "ScaledMaskSoftmax 自定义算子" article (pnsm.cn/news/1983787.html)
 *
 * What is computed (the plain definition, no blocking or reordering):
 *   forward  [P2 §1.2 formula, §2.1 stable form, §2.2 mask + causal flag]
 *     s_j = x_j * scale + mask_j                  (mask is added after scaling,
 *                                                  and is not itself scaled)
 *     s_j = -inf  if is_causal and j > q,  q = row mod cols   [P2 §3.1 kernel]
 *     M   = max_j s_j
 *     y_j = exp(s_j - M) / sum_k exp(s_k - M)
 *     A row whose every s_j is -inf gives y = 0 everywhere: [P3 §4.2 table /
 *     §4.3 pitfall 1] says such a row must not be divided and should come out
 *     uniform or all zero; the all-zero reading is taken.
 *   backward [P2 §3.3 Jacobian derivation]
 *     dot  = sum_j dy_j * y_j
 *     dx_j = (dy_j - dot) * y_j * scale           (the mask gets no gradient)
 *
 * Boolean mask (mask_kind 1): one byte per element; a nonzero byte masks its
 * key, s_j = -inf, and a zero byte leaves s_j = x_j * scale.  [P2 §2.2] names
 * this form: the kernel overrides the true positions with -inf.  Same
 * broadcast as the additive mask.
 *
 * Key lengths (optional): row r of batch b keeps only the keys j < L_b,
 * L_b = lengths[b] clamped to [0, cols]; s_j = -inf for j >= L_b.  This is the
 * key-padding mask of [P3 §2.1] written as lengths; [P2 §2.2] makes a padded
 * key's score -inf.  It is applied with the causal override, after the mask.
 *
 * Mask broadcasting: row r = ((b*heads) + h)*cols + q of the [rows, cols] view
 * reads the additive mask row starting at element
 *     b*mask_stride_b + h*mask_stride_h + q*cols
 * so an [S,S] mask has strides (0,0), [B,1,S,S] has (S*S, 0) and [B,H,S,S]
 * has (H*S*S, S*S)  [P3 §2.1 input contract; P2 §3.1 full-shape indexing].
 *
 * Every function here is pinned by the non-GPU tests (closed forms, library
 * softmax on special cases, invariants, finite differences).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORC_F32 = 0, ORC_F16 = 1, ORC_BF16 = 2, ORC_F64 = 3 };

/* IEEE 754 binary16: sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
static double decode_f16(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);               /* subnormal: f * 2^-10 * 2^-14 */
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + f), e - 25);   /* (1 + f/2^10) * 2^(e-15) */
    return sign ? -v : v;
}

/* bfloat16: the high half of a binary32 - sign, 8 exponent bits (bias 127),
 * 7 fraction bits. */
static double decode_bf16(uint16_t b)
{
    int sign = (b >> 15) & 1;
    int e = (b >> 7) & 0xff;
    int f = b & 0x7f;
    double v;
    if (e == 0)
        v = ldexp((double)f, -133);              /* subnormal: f * 2^-7 * 2^-126 */
    else if (e == 255)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(128 + f), e - 134);   /* (1 + f/2^7) * 2^(e-127) */
    return sign ? -v : v;
}

/* Element i of a buffer holding values of the given dtype, widened to fp64. */
static double load_elem(const void *p, int64_t i, int dtype)
{
    switch (dtype) {
    case ORC_F32: {
        float f;
        memcpy(&f, (const char *)p + 4 * i, 4);
        return (double)f;
    }
    case ORC_F16: {
        uint16_t h;
        memcpy(&h, (const char *)p + 2 * i, 2);
        return decode_f16(h);
    }
    case ORC_BF16: {
        uint16_t b;
        memcpy(&b, (const char *)p + 2 * i, 2);
        return decode_bf16(b);
    }
    default: {
        double d;
        memcpy(&d, (const char *)p + 8 * i, 8);
        return d;
    }
    }
}

static int dtype_ok(int dtype) { return dtype >= ORC_F32 && dtype <= ORC_F64; }

/* Exposed so that the tests can pin the decoders over every bit pattern. */
double oracle_decode(const void *p, int64_t i, int dtype) { return load_elem(p, i, dtype); }

/* Every element of an array widened to binary64 with the decoders above. */
int oracle_decode_array(const void *p, int64_t n, int dtype, double *out)
{
    if (!dtype_ok(dtype) || n < 0 || (n > 0 && (!p || !out))) return 1;
    for (int64_t i = 0; i < n; ++i) out[i] = load_elem(p, i, dtype);
    return 0;
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_num_threads(int n)
{
#ifdef _OPENMP
    if (n > 0)
        omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/*
 * Forward over n_rows rows.
 *   x_rows    n_rows x cols values of `dtype`, row-major (the rows to evaluate)
 *   row_index logical row id of each of those rows in the [rows, cols] view
 *             (fixes q, b, h); NULL means 0..n_rows-1
 *   mask      NULL for no mask, else additive mask values of `dtype`
 *             (mask_kind 0) or one byte per element, nonzero = masked (mask_kind 1)
 *   lengths   NULL, or the per-batch key lengths (int32, one per batch b)
 *   y         n_rows x cols fp64 output
 * Returns 0, or -1 for an argument it cannot interpret.
 */
int oracle_forward(const void *x_rows, int64_t n_rows, const int64_t *row_index, int64_t cols,
                   const void *mask, int64_t mask_stride_b, int64_t mask_stride_h, int64_t heads,
                   const int32_t *lengths, int mask_kind, double scale, int is_causal, int dtype, double *y)
{
    if (!x_rows || !y || n_rows < 0 || cols <= 0 || heads <= 0 || !dtype_ok(dtype) || mask_kind < 0 || mask_kind > 1)
        return -1;
    int64_t i;
#pragma omp parallel for schedule(dynamic, 16)
    for (i = 0; i < n_rows; i++) {
        int64_t r = row_index ? row_index[i] : i;
        int64_t q = r % cols;
        int64_t h = (r / cols) % heads;
        int64_t b = r / (cols * heads);
        double *s = y + i * cols; /* the output row holds the scores first */
        int64_t j;
        int64_t kept = cols; /* keys j < kept survive the key-length mask */
        if (lengths) {
            kept = lengths[b];
            if (kept < 0)
                kept = 0;
            if (kept > cols)
                kept = cols;
        }

        for (j = 0; j < cols; j++) {
            double v = load_elem(x_rows, i * cols + j, dtype) * scale;
            if (mask) {
                int64_t mi = b * mask_stride_b + h * mask_stride_h + q * cols + j;
                if (mask_kind == 1) {
                    if (((const uint8_t *)mask)[mi] != 0)
                        v = -INFINITY;
                } else {
                    v += load_elem(mask, mi, dtype);
                }
            }
            if (is_causal && j > q)
                v = -INFINITY;
            if (j >= kept)
                v = -INFINITY;
            s[j] = v;
        }

        double m = -INFINITY;
        for (j = 0; j < cols; j++)
            if (s[j] > m)
                m = s[j];

        if (m == -INFINITY) { /* every position masked: all-zero row */
            for (j = 0; j < cols; j++)
                s[j] = 0.0;
            continue;
        }

        double sum = 0.0;
        for (j = 0; j < cols; j++) {
            s[j] = exp(s[j] - m);
            sum += s[j];
        }
        for (j = 0; j < cols; j++)
            s[j] = s[j] / sum;
    }
    return 0;
}

/*
 * Backward over n_rows rows: dx = (dy - sum(dy*y)) * y * scale.
 *   y_rows  n_rows x cols values of y_dtype (the forward output kept for backward)
 *   dy_rows n_rows x cols values of dy_dtype
 *   dx      n_rows x cols fp64 output
 */
int oracle_backward(const void *y_rows, int y_dtype, const void *dy_rows, int dy_dtype,
                    int64_t n_rows, int64_t cols, double scale, double *dx)
{
    if (!y_rows || !dy_rows || !dx || n_rows < 0 || cols <= 0 || !dtype_ok(y_dtype) ||
        !dtype_ok(dy_dtype))
        return -1;
    int64_t i;
#pragma omp parallel for schedule(dynamic, 16)
    for (i = 0; i < n_rows; i++) {
        int64_t j;
        double dot = 0.0;
        for (j = 0; j < cols; j++)
            dot += load_elem(dy_rows, i * cols + j, dy_dtype) * load_elem(y_rows, i * cols + j, y_dtype);
        for (j = 0; j < cols; j++) {
            double yv = load_elem(y_rows, i * cols + j, y_dtype);
            double dyv = load_elem(dy_rows, i * cols + j, dy_dtype);
            dx[i * cols + j] = (dyv - dot) * yv * scale;
        }
    }
    return 0;
}
