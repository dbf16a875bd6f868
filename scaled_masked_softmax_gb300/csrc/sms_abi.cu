// C ABI of libsms: host-side argument validation, kernel-family dispatch,
// status reporting.  See include/sms.h for the contract of every entry point.
#include "sms.h"
#include "sms_internal.h"

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

namespace sms {

// Error word written by kernels whose bounded waits expire (one per device;
// its address is looked up once per device and passed to the kernels).
__device__ int g_device_error = 0;

namespace {

thread_local char t_err[256] = "";
thread_local int t_last_path = SMS_PATH_AUTO;
std::atomic<int> g_forced{SMS_PATH_AUTO};
std::atomic<int> g_grid_limit{0};
std::atomic<int64_t> g_launches{0};
std::atomic<uint32_t> g_stall_ns{0};

constexpr int kMaxDevices = 64;
std::once_flag g_dev_once[kMaxDevices];
int g_dev_sms[kMaxDevices];
int *g_dev_err[kMaxDevices];
cudaError_t g_dev_status[kMaxDevices];

int fail(int status, const char *fmt, ...) __attribute__((format(printf, 2, 3)));
int fail(int status, const char *fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(t_err, sizeof(t_err), fmt, ap);
    va_end(ap);
    return status;
}

// Per-device facts, looked up once with that device current.
cudaError_t device_info(int &dev, int &sms, int *&err)
{
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::call_once(g_dev_once[dev], [dev] {
        int n = 0;
        cudaError_t s = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        void *p = nullptr;
        if (s == cudaSuccess) s = cudaGetSymbolAddress(&p, g_device_error);
        g_dev_sms[dev] = n;
        g_dev_err[dev] = static_cast<int *>(p);
        g_dev_status[dev] = s;
    });
    sms = g_dev_sms[dev];
    err = g_dev_err[dev];
    return g_dev_status[dev];
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// [a, a+na) and [b, b+nb) share a byte (both non-empty).
bool overlap(const void *a, int64_t na, const void *b, int64_t nb)
{
    const uintptr_t pa = reinterpret_cast<uintptr_t>(a), pb = reinterpret_cast<uintptr_t>(b);
    return pa < pb + (uintptr_t)nb && pb < pa + (uintptr_t)na;
}

// Largest mask element any row touches, plus one (see sms.h for the row rule).
int64_t mask_extent(int64_t rows, int64_t cols, int64_t heads, int64_t sb, int64_t sh)
{
    auto off = [&](int64_t r) {
        return (r / (cols * heads)) * sb + ((r / cols) % heads) * sh + (r % cols) * cols;
    };
    const int64_t last = rows - 1;
    int64_t m = off(last);
    const int64_t b = last / (cols * heads), h = (last / cols) % heads;
    if (h > 0) m = std::max(m, off((b * heads + h) * cols - 1));
    if (b > 0) m = std::max(m, off(b * heads * cols - 1));
    return m + cols;
}

const char *cuda_msg(cudaError_t e) { return cudaGetErrorString(e); }

int launch_status(cudaError_t e, const char *what)
{
    if (e == cudaSuccess) {
        g_launches.fetch_add(1, std::memory_order_relaxed);
        return SMS_OK;
    }
    cudaGetLastError();  // leave no error pending from this launch
    if (e == cudaErrorNotSupported) return fail(SMS_ERR_UNSUPPORTED, "%s: shape not supported by the path", what);
    return fail(SMS_ERR_CUDA, "%s: launch failed: %s", what, cuda_msg(e));
}

constexpr int64_t kMaxCols = (int64_t)1 << 30;
constexpr int64_t kMaxElems = (int64_t)1 << 60;

int pick_path(int forced, int64_t cols, int dtype, bool aligned, bool bwd, bool causal)
{
    if (forced != SMS_PATH_AUTO) return forced;
    // By measurement on GB300 (per-family sweeps over the benchmark shapes):
    //  * causal forward rows read a variable prefix; the per-warp bulk-copy
    //    rings keep enough of them in flight (registers do not): ring;
    //  * short aligned fp32 forward rows: the persistent prefetching groups;
    //  * otherwise register-resident lane groups while a row fits them
    //    (misaligned 16-bit backward rows too: 65-75% of the copy rate at
    //    S = 2049 .. 3333 against 43-57% on the rings);
    //  * 16-bit backward rows too wide for registers: ring, then the staged
    //    CTA path while a row fits its registers; beyond that, stream twice.
    if (!bwd && causal && aligned && ring_fits(cols, dtype, aligned)) return SMS_PATH_RING;
    if (!bwd && dtype == SMS_F32 && aligned && cols <= 512) return SMS_PATH_STREAM;
    if (warp_fits(cols, dtype, aligned, bwd)) return SMS_PATH_WARP;
    if (bwd && dtype != SMS_F32 && ring_fits(cols, dtype, aligned)) return SMS_PATH_RING;
    if (bwd ? cta_fits_bwd(cols, dtype, aligned) : cta_fits(cols, dtype, aligned)) return SMS_PATH_CTA;
    return SMS_PATH_ONLINE;
}

}  // namespace

int set_last_error(int status, const char *msg)
{
    snprintf(t_err, sizeof(t_err), "%s", msg);
    return status;
}

void clear_last_error() { t_err[0] = '\0'; }

void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

uint32_t test_stall_ns() { return g_stall_ns.load(std::memory_order_relaxed); }

cudaError_t device_error_word(int **err)
{
    int dev = 0, n = 0;
    return device_info(dev, n, *err);
}

int sm_count()
{
    int dev = 0, n = 0;
    int *err = nullptr;
    if (device_info(dev, n, err) != cudaSuccess || n <= 0) return 148;
    return n;
}

int64_t persistent_grid(int per_sm, int64_t useful)
{
    int64_t g = (int64_t)sm_count() * (per_sm > 0 ? per_sm : 1);
    const int lim = g_grid_limit.load();
    if (lim > 0 && g > lim) g = lim;
    if (g > useful) g = useful;
    return g > 0 ? g : 1;
}

}  // namespace sms

using namespace sms;

extern "C" {

int sms_version(void) { return 100; }

const char *sms_status_string(int status)
{
    switch (status) {
    case SMS_OK: return "ok";
    case SMS_ERR_INVALID_ARG: return "invalid argument";
    case SMS_ERR_UNSUPPORTED: return "unsupported by the selected path";
    case SMS_ERR_CUDA: return "CUDA error";
    default: return "unknown status";
    }
}

const char *sms_last_error(void) { return t_err; }

int sms_set_forced_path(int path)
{
    if (path < SMS_PATH_AUTO || path > SMS_PATH_RING) return -1;
    return g_forced.exchange(path);
}

int sms_last_path(void) { return t_last_path; }

int sms_set_grid_limit(int ctas)
{
    if (ctas < 0) return -1;
    return g_grid_limit.exchange(ctas);
}

int64_t sms_launch_count(void) { return g_launches.load(); }

int64_t sms_set_test_stall(int64_t ns)
{
    if (ns < 0 || ns > 1000000000ll) return -1;
    return g_stall_ns.exchange((uint32_t)ns);
}

int sms_select_path(int64_t rows, int64_t cols, int dtype, int is_backward)
{
    (void)rows;
    if (cols <= 0 || dtype < SMS_F32 || dtype > SMS_BF16) return -1;
    const bool aligned = cols % vec_elems(dtype) == 0;
    return pick_path(SMS_PATH_AUTO, cols, dtype, aligned, is_backward != 0, false);
}

}  // extern "C"

namespace {

// The mask-reuse order (ReuseOrder) of rows sharing a [cols, cols] mask with
// no head stride: one super-block of every row when the mask has no batch
// stride either (its last block may be partial), else one per batch of
// `heads` whole blocks (a partial last batch keeps the natural order).
ReuseOrder reuse_order(int64_t rows, int64_t cols, int64_t heads, int64_t mask_stride_b)
{
    ReuseOrder o{};
    const int64_t T = kReuseTile;
    int64_t sb, kf, rem;
    if (mask_stride_b == 0) {
        sb = rows;
        kf = (rows - 1) / cols;
        rem = rows - kf * cols;
    } else {
        sb = heads * cols;
        kf = heads - 1;
        rem = cols;
    }
    if (kf < 1 || rows > 0xffffffffll || rows / sb < 1) return o;  // places are 32-bit in the kernel
    o.rows = rows / sb * sb;
    o.sb = (uint32_t)sb;
    o.kf = (uint32_t)kf;
    const int64_t ta = rem / T, wb = std::min<int64_t>(T, cols - ta * T), rem_b = rem - ta * T;
    o.ta = (uint32_t)ta;
    o.wb = (uint32_t)wb;
    o.rem_b = (uint32_t)rem_b;
    o.pa = (uint32_t)((kf + 1) * T * ta);
    o.pb = (uint32_t)(ta * T < cols ? kf * wb + rem_b : 0);
    o.base_c = (uint32_t)(ta * T + (ta * T < cols ? wb : 0));
    o.nc = (uint32_t)((cols - o.base_c) / T);
    o.pc = (uint32_t)(kf * T * o.nc);
    o.d_sb = FastDiv((uint32_t)sb);
    o.d_a = FastDiv((uint32_t)((kf + 1) * T));
    o.d_c = FastDiv((uint32_t)(kf * T));
    return o;
}

// Validation and dispatch shared by sms_forward, sms_forward_bool and
// sms_forward_lengths (`who` names the entry point in error messages;
// mask_bool: the mask holds one byte per element).
int forward_impl(const char *who, const void *x, const void *mask, int64_t mask_numel, int64_t mask_stride_b,
                 int64_t mask_stride_h, int64_t heads, const int32_t *lengths, void *y, int64_t rows, int64_t cols,
                 float scale, int is_causal, int dtype, void *stream, bool mask_bool = false)
{
    t_err[0] = '\0';
    if (dtype < SMS_F32 || dtype > SMS_BF16) return fail(SMS_ERR_INVALID_ARG, "%s: unknown dtype %d", who, dtype);
    if (rows < 0) return fail(SMS_ERR_INVALID_ARG, "%s: rows < 0", who);
    if (rows == 0 && cols > 0) {  // empty problem: nothing is read, pointers may be NULL
        t_last_path = SMS_PATH_AUTO;
        return SMS_OK;
    }
    if (!x || !y) return fail(SMS_ERR_INVALID_ARG, "%s: x and y must not be NULL", who);
    if (cols <= 0 || cols > kMaxCols) return fail(SMS_ERR_INVALID_ARG, "%s: cols must be in [1, 2^30]", who);
    if (rows > 0 && rows > kMaxElems / cols) return fail(SMS_ERR_INVALID_ARG, "%s: rows*cols too large", who);
    if (!std::isfinite(scale)) return fail(SMS_ERR_INVALID_ARG, "%s: scale must be finite", who);
    if (!aligned16(x) || !aligned16(y)) return fail(SMS_ERR_INVALID_ARG, "%s: x and y must be 16-byte aligned", who);
    const int eb = elem_bytes(dtype);
    const int64_t total = rows * cols;
    if (x != y && overlap(x, total * eb, y, total * eb))
        return fail(SMS_ERR_INVALID_ARG, "%s: y partially overlaps x", who);
    if (mask || lengths) {
        if (heads <= 0 || heads > ((int64_t)1 << 31)) return fail(SMS_ERR_INVALID_ARG, "%s: heads must be in [1, 2^31]", who);
    }
    if (lengths) {
        if (reinterpret_cast<uintptr_t>(lengths) & 3u)
            return fail(SMS_ERR_INVALID_ARG, "%s: lengths must be 4-byte aligned", who);
        const int64_t nb = (rows + cols * heads - 1) / (cols * heads);  // batches: entries read from lengths
        if (overlap(lengths, nb * 4, y, total * eb)) return fail(SMS_ERR_INVALID_ARG, "%s: y overlaps lengths", who);
    }
    if (mask) {
        if (mask_stride_b < 0 || mask_stride_h < 0)
            return fail(SMS_ERR_INVALID_ARG, "%s: mask strides must be >= 0", who);
        if (!aligned16(mask)) return fail(SMS_ERR_INVALID_ARG, "%s: mask must be 16-byte aligned", who);
        if (mask_numel < 0 || mask_numel > kMaxElems) return fail(SMS_ERR_INVALID_ARG, "%s: bad mask_numel", who);
        if (rows > 0) {
            // guard the extent arithmetic against overflow before evaluating it
            const double est = (double)(rows / (cols * heads) + 1) * (double)mask_stride_b +
                               (double)heads * (double)mask_stride_h + (double)cols * (double)cols;
            if (est > 4e18) return fail(SMS_ERR_INVALID_ARG, "%s: mask strides too large", who);
            const int64_t ext = mask_extent(rows, cols, heads, mask_stride_b, mask_stride_h);
            if (ext > mask_numel)
                return fail(SMS_ERR_INVALID_ARG, "%s: rows reach mask element %lld but mask_numel is %lld", who,
                            (long long)ext - 1, (long long)mask_numel);
            if (overlap(mask, mask_numel * (mask_bool ? 1 : eb), y, total * eb))
                return fail(SMS_ERR_INVALID_ARG, "%s: y overlaps the mask", who);
        }
    } else if (!lengths && heads <= 0) {
        heads = 1;
    }
    if (rows == 0) {
        t_last_path = SMS_PATH_AUTO;
        return SMS_OK;
    }

    const int vec = vec_elems(dtype);
    const bool aligned = cols % vec == 0 && (!mask || (mask_stride_b % vec == 0 && mask_stride_h % vec == 0));
    const int path = pick_path(g_forced.load(), cols, dtype, aligned, false, is_causal != 0);

    int dev = 0, nsm = 0;
    int *err = nullptr;
    cudaError_t e = device_info(dev, nsm, err);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(SMS_ERR_CUDA, "%s: device query failed: %s", who, cuda_msg(e));
    }

    FwdArgs a;
    a.x = x; a.mask = mask; a.y = y;
    a.rows = rows; a.cols = cols; a.x_total = total;
    a.mask_total = mask ? mask_numel : 0;
    a.msb = mask ? mask_stride_b : 0; a.msh = mask ? mask_stride_h : 0; a.heads = heads;
    a.scale = scale; a.causal = is_causal ? 1 : 0; a.err = err;
    a.dcols = FastDiv((uint32_t)cols);
    a.dheads = FastDiv((uint32_t)heads);
    a.lengths = lengths;
    a.mask_bool = (mask && mask_bool) ? 1 : 0;
    a.stall_ns = test_stall_ns();
    // mask-reuse row order: fp32 rows whose per-block mask (cols x cols) is
    // at least 64 MB.  Measured on GB300 (fp32 S=4099, a 67 MB mask read
    // about four times in the natural order: 71% -> 83% of the copy rate).
    // Below that size enough of the mask stays in L2 in the natural order and
    // the order's index arithmetic costs more than it saves (fp32 S=2049 and
    // S=3333: -4 to -5 points), and 16-bit rows, bound by issue, lost 1-4
    // points at every size.
    a.reuse = ReuseOrder{};
    if (mask && mask_stride_h == 0 && eb == 4 &&
        (double)cols * (double)cols * (mask_bool ? 1 : eb) >= (double)(64 << 20))
        a.reuse = reuse_order(rows, cols, heads, mask_stride_b);

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    switch (path) {
    case SMS_PATH_WARP:
        if (!warp_fits(cols, dtype, aligned, false)) return fail(SMS_ERR_UNSUPPORTED, "%s: row too wide for the warp path", who);
        e = launch_fwd_warp(a, dtype, aligned, st);
        break;
    case SMS_PATH_RING:
        if (!ring_fits(cols, dtype, aligned)) return fail(SMS_ERR_UNSUPPORTED, "%s: row too wide for the ring path", who);
        e = launch_fwd_ring(a, dtype, aligned, st);
        break;
    case SMS_PATH_STREAM:
        if (!stream_fits(cols, dtype, aligned, false))
            return fail(SMS_ERR_UNSUPPORTED, "%s: row too wide for the stream path", who);
        e = launch_fwd_stream(a, dtype, aligned, st);
        break;
    case SMS_PATH_CTA:
        if (!cta_fits(cols, dtype, aligned)) return fail(SMS_ERR_UNSUPPORTED, "%s: row too wide for the CTA path", who);
        e = launch_fwd_cta(a, dtype, aligned, st);
        break;
    default:
        e = launch_fwd_online(a, dtype, st);
        break;
    }
    const int rc = launch_status(e, who);
    if (rc == SMS_OK) t_last_path = path;
    return rc;
}

// Validation and dispatch shared by sms_backward and sms_backward_lengths.
int backward_impl(const char *who, const void *y, const void *dy, void *dx, const int32_t *lengths, int64_t heads,
                  int64_t rows, int64_t cols, float scale, int is_causal_hint, int dtype, void *stream)
{
    t_err[0] = '\0';
    if (dtype < SMS_F32 || dtype > SMS_BF16) return fail(SMS_ERR_INVALID_ARG, "%s: unknown dtype %d", who, dtype);
    if (rows < 0) return fail(SMS_ERR_INVALID_ARG, "%s: rows < 0", who);
    if (rows == 0 && cols > 0) {  // empty problem: nothing is read, pointers may be NULL
        t_last_path = SMS_PATH_AUTO;
        return SMS_OK;
    }
    if (!y || !dy || !dx) return fail(SMS_ERR_INVALID_ARG, "%s: y, dy and dx must not be NULL", who);
    if (cols <= 0 || cols > kMaxCols) return fail(SMS_ERR_INVALID_ARG, "%s: cols must be in [1, 2^30]", who);
    if (rows > 0 && rows > kMaxElems / cols) return fail(SMS_ERR_INVALID_ARG, "%s: rows*cols too large", who);
    if (!std::isfinite(scale)) return fail(SMS_ERR_INVALID_ARG, "%s: scale must be finite", who);
    if (!aligned16(y) || !aligned16(dy) || !aligned16(dx))
        return fail(SMS_ERR_INVALID_ARG, "%s: y, dy and dx must be 16-byte aligned", who);
    const int eb = elem_bytes(dtype);
    const int64_t total = rows * cols;
    if (overlap(dx, total * eb, y, total * eb)) return fail(SMS_ERR_INVALID_ARG, "%s: dx overlaps y", who);
    if (dx != dy && overlap(dx, total * eb, dy, total * eb))
        return fail(SMS_ERR_INVALID_ARG, "%s: dx partially overlaps dy", who);
    if (lengths) {
        if (heads <= 0 || heads > ((int64_t)1 << 31)) return fail(SMS_ERR_INVALID_ARG, "%s: heads must be in [1, 2^31]", who);
        if (reinterpret_cast<uintptr_t>(lengths) & 3u)
            return fail(SMS_ERR_INVALID_ARG, "%s: lengths must be 4-byte aligned", who);
        const int64_t nb = (rows + cols * heads - 1) / (cols * heads);
        if (overlap(lengths, nb * 4, dx, total * eb)) return fail(SMS_ERR_INVALID_ARG, "%s: dx overlaps lengths", who);
    } else {
        heads = 1;
    }
    if (rows == 0) {
        t_last_path = SMS_PATH_AUTO;
        return SMS_OK;
    }

    int dev = 0, nsm = 0;
    int *err = nullptr;
    cudaError_t e = device_info(dev, nsm, err);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(SMS_ERR_CUDA, "%s: device query failed: %s", who, cuda_msg(e));
    }

    const bool aligned = cols % vec_elems(dtype) == 0;
    BwdArgs a;
    a.y = y; a.dy = dy; a.dx = dx;
    a.rows = rows; a.cols = cols; a.total = total;
    a.scale = scale; a.causal = is_causal_hint ? 1 : 0; a.err = err;
    a.dcols = FastDiv((uint32_t)cols);
    a.lengths = lengths;
    a.heads = heads;
    a.dheads = FastDiv((uint32_t)heads);
    a.stall_ns = test_stall_ns();

    const int path = pick_path(g_forced.load(), cols, dtype, aligned, true, a.causal != 0);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    switch (path) {
    case SMS_PATH_WARP:
        if (!warp_fits(cols, dtype, aligned, true)) return fail(SMS_ERR_UNSUPPORTED, "%s: row too wide for the warp path", who);
        e = launch_bwd_warp(a, dtype, aligned, st);
        break;
    case SMS_PATH_RING:
        if (!ring_fits(cols, dtype, aligned)) return fail(SMS_ERR_UNSUPPORTED, "%s: row too wide for the ring path", who);
        e = launch_bwd_ring(a, dtype, aligned, st);
        break;
    case SMS_PATH_STREAM:
        if (!stream_fits(cols, dtype, aligned, true))
            return fail(SMS_ERR_UNSUPPORTED, "%s: row too wide for the stream path", who);
        e = launch_bwd_stream(a, dtype, aligned, st);
        break;
    case SMS_PATH_CTA:
        if (!cta_fits_bwd(cols, dtype, aligned)) return fail(SMS_ERR_UNSUPPORTED, "%s: row too wide for the CTA path", who);
        e = launch_bwd_cta(a, dtype, aligned, st);
        break;
    default:
        e = launch_bwd_online(a, dtype, st);
        break;
    }
    const int rc = launch_status(e, who);
    if (rc == SMS_OK) t_last_path = path;
    return rc;
}

}  // namespace

extern "C" {

int sms_forward(const void *x, const void *mask, int64_t mask_numel, int64_t mask_stride_b, int64_t mask_stride_h,
                int64_t heads, void *y, int64_t rows, int64_t cols, float scale, int is_causal, int dtype,
                void *stream)
{
    return forward_impl("sms_forward", x, mask, mask_numel, mask_stride_b, mask_stride_h, heads, nullptr, y, rows,
                        cols, scale, is_causal, dtype, stream);
}

int sms_forward_bool(const void *x, const uint8_t *mask, int64_t mask_numel, int64_t mask_stride_b,
                     int64_t mask_stride_h, int64_t heads, void *y, int64_t rows, int64_t cols, float scale,
                     int is_causal, int dtype, void *stream)
{
    if (!mask && rows != 0) {
        t_err[0] = '\0';
        return fail(SMS_ERR_INVALID_ARG, "sms_forward_bool: mask must not be NULL");
    }
    return forward_impl("sms_forward_bool", x, mask, mask_numel, mask_stride_b, mask_stride_h, heads, nullptr, y,
                        rows, cols, scale, is_causal, dtype, stream, true);
}

int sms_forward_lengths(const void *x, const int32_t *lengths, int64_t heads, void *y, int64_t rows, int64_t cols,
                        float scale, int is_causal, int dtype, void *stream)
{
    if (!lengths) {
        t_err[0] = '\0';
        return fail(SMS_ERR_INVALID_ARG, "sms_forward_lengths: lengths must not be NULL");
    }
    return forward_impl("sms_forward_lengths", x, nullptr, 0, 0, 0, heads, lengths, y, rows, cols, scale, is_causal,
                        dtype, stream);
}

int sms_backward(const void *y, const void *dy, void *dx, int64_t rows, int64_t cols, float scale,
                 int is_causal_hint, int dtype, void *stream)
{
    return backward_impl("sms_backward", y, dy, dx, nullptr, 1, rows, cols, scale, is_causal_hint, dtype, stream);
}

int sms_backward_lengths(const void *y, const void *dy, void *dx, const int32_t *lengths, int64_t heads, int64_t rows,
                         int64_t cols, float scale, int is_causal_hint, int dtype, void *stream)
{
    if (!lengths) {
        t_err[0] = '\0';
        return fail(SMS_ERR_INVALID_ARG, "sms_backward_lengths: lengths must not be NULL");
    }
    return backward_impl("sms_backward_lengths", y, dy, dx, lengths, heads, rows, cols, scale, is_causal_hint, dtype,
                         stream);
}

int sms_device_error(void *stream)
{
    int dev = 0, nsm = 0;
    int *err = nullptr;
    if (device_info(dev, nsm, err) != cudaSuccess || !err) {
        cudaGetLastError();
        return -1;
    }
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int v = 0;
    const int zero = 0;
    if (cudaMemcpyAsync(&v, err, sizeof(int), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
        cudaMemcpyAsync(err, &zero, sizeof(int), cudaMemcpyHostToDevice, st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess) {
        cudaGetLastError();
        return -1;
    }
    return v;
}

}  // extern "C"
