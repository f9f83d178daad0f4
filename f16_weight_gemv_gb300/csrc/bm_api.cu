// bm_api.cu -- the C ABI of include/bm.h: argument validation, path selection
// and dispatch to the kernels.  Every check happens on the host before any
// launch, so a non-zero status other than BM_ERR_CUDA means nothing ran.
#include "../../include/bm.h"
#include "bm_internal.h"

#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <algorithm>
#include <atomic>
#include <mutex>

namespace bm {

static thread_local char g_last_error[512];

int fail(int status, const char *fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
    va_end(ap);
    return status;
}

static void clear_error() { g_last_error[0] = 0; }

namespace {
constexpr int kMaxDevices = 64;
DeviceInfo g_dev[kMaxDevices];
std::once_flag g_once[kMaxDevices];
int g_dev_status[kMaxDevices];
std::atomic<int> g_pdl{0};
std::atomic<int> g_exact_cols{2};  // bm_set_exact_sgemm_cols
std::atomic<int> g_stream_k{-1};   // bm_set_stream_k
unsigned int *g_err_addr[kMaxDevices];
std::once_flag g_err_once[kMaxDevices];
}  // namespace

// BM_OK, or BM_ERR_TIMEOUT once a kernel gave up a bounded wait; one per device.
__device__ unsigned int g_device_error;

unsigned int *device_error_word()
{
    int d = -1;
    if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= kMaxDevices) return nullptr;
    std::call_once(g_err_once[d], [d] {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_device_error) == cudaSuccess) g_err_addr[d] = static_cast<unsigned int *>(p);
    });
    return g_err_addr[d];
}

bool pdl_enabled() { return g_pdl.load(std::memory_order_relaxed) != 0; }
int stream_k_mode() { return g_stream_k.load(std::memory_order_relaxed); }

int read_device_error(cudaStream_t s)
{
    cudaError_t e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return fail(BM_ERR_CUDA, "stream synchronize failed: %s", cudaGetErrorString(e));
    unsigned int *w = device_error_word();
    if (!w) return fail(BM_ERR_CUDA, "device error word unavailable");
    unsigned int v = 0, zero = 0;
    e = cudaMemcpy(&v, w, sizeof v, cudaMemcpyDeviceToHost);
    if (e == cudaSuccess) e = cudaMemcpy(w, &zero, sizeof zero, cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return fail(BM_ERR_CUDA, "reading the device error word failed: %s", cudaGetErrorString(e));
    if (v == BM_ERR_INVALID_ARG) return fail((int)v, "a kernel met an invalid argument on the device (an id out of range)");
    if (v != 0) return fail((int)v, "a kernel gave up a bounded wait");
    return BM_OK;
}

bool current_device(DeviceInfo *info, int *status)
{
    int d = -1;
    cudaError_t e = cudaGetDevice(&d);
    if (e != cudaSuccess || d < 0 || d >= kMaxDevices) {
        *status = fail(BM_ERR_CUDA, "cudaGetDevice failed: %s", cudaGetErrorString(e));
        return false;
    }
    std::call_once(g_once[d], [d] {
        DeviceInfo &di = g_dev[d];
        int st = BM_OK;
        if (cudaDeviceGetAttribute(&di.major, cudaDevAttrComputeCapabilityMajor, d) != cudaSuccess ||
            cudaDeviceGetAttribute(&di.minor, cudaDevAttrComputeCapabilityMinor, d) != cudaSuccess ||
            cudaDeviceGetAttribute(&di.sm_count, cudaDevAttrMultiProcessorCount, d) != cudaSuccess ||
            cudaDeviceGetAttribute(&di.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, d) !=
                cudaSuccess ||
            cudaDeviceGetAttribute(&di.smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, d) != cudaSuccess ||
            cudaDeviceGetAttribute(&di.smem_reserved, cudaDevAttrReservedSharedMemoryPerBlock, d) != cudaSuccess)
            st = BM_ERR_CUDA;
        else if (di.major != 10 || di.minor != 3)
            st = BM_ERR_UNSUPPORTED_DEVICE;
        g_dev_status[d] = st;
    });
    if (g_dev_status[d] == BM_ERR_CUDA) {
        *status = fail(BM_ERR_CUDA, "cannot query device %d", d);
        return false;
    }
    if (g_dev_status[d] == BM_ERR_UNSUPPORTED_DEVICE) {
        *status = fail(BM_ERR_UNSUPPORTED_DEVICE,
                       "device %d is compute capability %d.%d; this library is built for sm_103a only", d,
                       g_dev[d].major, g_dev[d].minor);
        return false;
    }
    *info = g_dev[d];
    return true;
}

}  // namespace bm

using namespace bm;

namespace {

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// [a, a+na) and [b, b+nb) in bytes overlap.
bool overlap(const void *a, int64_t na, const void *b, int64_t nb)
{
    uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return na > 0 && nb > 0 && x < y + (uintptr_t)nb && y < x + (uintptr_t)na;
}

// rows * k * 2 bytes must fit an int64 and the products' index arithmetic.
bool sizes_ok(int64_t rows, int64_t k) { return rows >= 0 && k >= 1 && rows <= (INT64_MAX / 4) / k; }

int check_matrix_args(const char *fn, const uint16_t *W, int64_t rows, int64_t k, const uint16_t *X,
                      int64_t ncols, const float *Y)
{
    if (k < 1 || k > BM_MAX_K) return fail(BM_ERR_INVALID_ARG, "%s: k = %lld outside 1..%d", fn, (long long)k, BM_MAX_K);
    if (rows < 0 || ncols < 0) return fail(BM_ERR_INVALID_ARG, "%s: negative size", fn);
    if (!sizes_ok(rows, k) || !sizes_ok(ncols, k) || (rows > 0 && ncols > INT64_MAX / 8 / rows))
        return fail(BM_ERR_INVALID_ARG, "%s: sizes overflow", fn);
    if (rows == 0 || ncols == 0) return BM_OK;
    if (!W || !X || !Y) return fail(BM_ERR_INVALID_ARG, "%s: null pointer", fn);
    if (!aligned(W, 16) || !aligned(X, 16))
        return fail(BM_ERR_ALIGNMENT, "%s: W and the activation must be 16-byte aligned", fn);
    if (!aligned(Y, 4)) return fail(BM_ERR_ALIGNMENT, "%s: the output must be 4-byte aligned", fn);
    if (overlap(Y, rows * ncols * 4, W, rows * k * 2) || overlap(Y, rows * ncols * 4, X, ncols * k * 2))
        return fail(BM_ERR_INVALID_ARG, "%s: the output overlaps an input", fn);
    return BM_OK;
}

int product(const char *fn, const uint16_t *W, int64_t rows, int64_t k, const uint16_t *X, int64_t ncols,
            float *Y, bm_stream_t stream)
{
    int st = check_matrix_args(fn, W, rows, k, X, ncols, Y);
    if (st != BM_OK || rows == 0 || ncols == 0) return st;
    DeviceInfo dev;
    if (!current_device(&dev, &st)) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (bm_takes_sgemm(rows, k, ncols))
        return ncols <= g_exact_cols.load(std::memory_order_relaxed)
                   ? launch_sgemm_stream(W, rows, k, X, ncols, Y, s, dev)
                   : launch_gemm_tc(W, rows, k, X, ncols, Y, s, dev);
    VecdotJob job{};
    job.W[0] = W;
    job.y[0] = Y;
    job.rows[0] = rows;
    job.nmat = 1;
    job.k = k;
    job.X = X;
    job.ncols = ncols;
    return ncols == 1 ? launch_vecdot_1col(job, s, dev) : launch_vecdot_ncol(job, s, dev);
}

}  // namespace

extern "C" {

int bm_f16_get_rows(const uint16_t *E, int64_t vocab, int64_t hidden, const int32_t *ids, int64_t n, float *out,
                    bm_stream_t stream)
{
    clear_error();
    if (n < 0 || vocab < 0 || hidden < 0) return fail(BM_ERR_INVALID_ARG, "bm_f16_get_rows: negative size");
    if (n == 0) return BM_OK;
    if (vocab < 1 || hidden < 1) return fail(BM_ERR_INVALID_ARG, "bm_f16_get_rows: empty table");
    if (vocab > INT32_MAX || hidden > INT64_MAX / 8 / vocab || n > INT64_MAX / 8 / hidden)
        return fail(BM_ERR_INVALID_ARG, "bm_f16_get_rows: sizes overflow");
    if (!E || !ids || !out) return fail(BM_ERR_INVALID_ARG, "bm_f16_get_rows: null pointer");
    if (!aligned(E, 16) || !aligned(ids, 16))
        return fail(BM_ERR_ALIGNMENT, "bm_f16_get_rows: the table and the ids must be 16-byte aligned");
    if (!aligned(out, 4)) return fail(BM_ERR_ALIGNMENT, "bm_f16_get_rows: the output must be 4-byte aligned");
    if (overlap(out, n * hidden * 4, E, vocab * hidden * 2) || overlap(out, n * hidden * 4, ids, n * 4))
        return fail(BM_ERR_INVALID_ARG, "bm_f16_get_rows: the output overlaps an input");
    DeviceInfo dev;
    int st = BM_OK;
    if (!current_device(&dev, &st)) return st;
    return launch_get_rows(E, vocab, hidden, ids, n, out, reinterpret_cast<cudaStream_t>(stream), dev);
}

int bm_takes_sgemm(int64_t rows, int64_t k, int64_t ncols)
{
    return ncols >= 2 && rows % 4 == 0 && k % 8 == 0;
}

int bm_to_f16(const float *x, uint16_t *h, int64_t n, bm_stream_t stream)
{
    clear_error();
    if (n < 0 || n > INT64_MAX / 8) return fail(BM_ERR_INVALID_ARG, "bm_to_f16: bad n = %lld", (long long)n);
    if (n == 0) return BM_OK;
    if (!x || !h) return fail(BM_ERR_INVALID_ARG, "bm_to_f16: null pointer");
    if (!aligned(x, 16) || !aligned(h, 16))
        return fail(BM_ERR_ALIGNMENT, "bm_to_f16: x and h must be 16-byte aligned");
    if (overlap(x, n * 4, h, n * 2)) return fail(BM_ERR_INVALID_ARG, "bm_to_f16: h overlaps x");
    int st;
    DeviceInfo dev;
    if (!current_device(&dev, &st)) return st;
    return launch_to_f16(x, h, n, reinterpret_cast<cudaStream_t>(stream), dev);
}

int bm_f16_mad(uint16_t *acc, const uint16_t *v, float w, int64_t n, bm_stream_t stream)
{
    clear_error();
    if (n < 0 || n > INT64_MAX / 8) return fail(BM_ERR_INVALID_ARG, "bm_f16_mad: bad n = %lld", (long long)n);
    if (n == 0) return BM_OK;
    if (!acc || !v) return fail(BM_ERR_INVALID_ARG, "bm_f16_mad: null pointer");
    if (!aligned(acc, 2) || !aligned(v, 2)) return fail(BM_ERR_ALIGNMENT, "bm_f16_mad: acc and v must be 2-byte aligned");
    if (static_cast<const void *>(v) != static_cast<const void *>(acc) && overlap(v, n * 2, acc, n * 2))
        return fail(BM_ERR_INVALID_ARG, "bm_f16_mad: v overlaps acc (only v == acc may share memory)");
    int st;
    DeviceInfo dev;
    if (!current_device(&dev, &st)) return st;
    return launch_f16_accum(true, acc, v, w, n, reinterpret_cast<cudaStream_t>(stream), dev);
}

int bm_f16_scale(uint16_t *acc, float s, int64_t n, bm_stream_t stream)
{
    clear_error();
    if (n < 0 || n > INT64_MAX / 8) return fail(BM_ERR_INVALID_ARG, "bm_f16_scale: bad n = %lld", (long long)n);
    if (n == 0) return BM_OK;
    if (!acc) return fail(BM_ERR_INVALID_ARG, "bm_f16_scale: null pointer");
    if (!aligned(acc, 2)) return fail(BM_ERR_ALIGNMENT, "bm_f16_scale: acc must be 2-byte aligned");
    int st;
    DeviceInfo dev;
    if (!current_device(&dev, &st)) return st;
    return launch_f16_accum(false, acc, nullptr, s, n, reinterpret_cast<cudaStream_t>(stream), dev);
}

int bm_f16_matvec(const uint16_t *W, int64_t rows, int64_t k, const uint16_t *x, float *y, bm_stream_t stream)
{
    clear_error();
    int st = check_matrix_args("bm_f16_matvec", W, rows, k, x, 1, y);
    if (st != BM_OK || rows == 0) return st;
    DeviceInfo dev;
    if (!current_device(&dev, &st)) return st;
    VecdotJob job{};
    job.W[0] = W;
    job.y[0] = y;
    job.rows[0] = rows;
    job.nmat = 1;
    job.k = k;
    job.X = x;
    job.ncols = 1;
    return launch_vecdot_1col(job, reinterpret_cast<cudaStream_t>(stream), dev);
}

int bm_f16_matvec_multi(int nmat, const uint16_t *const *W, const int64_t *rows, int64_t k, const uint16_t *x,
                        float *const *y, bm_stream_t stream)
{
    clear_error();
    if (nmat < 1 || nmat > 4) return fail(BM_ERR_INVALID_ARG, "bm_f16_matvec_multi: nmat = %d outside 1..4", nmat);
    if (!W || !rows || !y) return fail(BM_ERR_INVALID_ARG, "bm_f16_matvec_multi: null host array");
    VecdotJob job{};
    job.nmat = 0;
    job.k = k;
    job.X = x;
    job.ncols = 1;
    for (int m = 0; m < nmat; m++) {
        int st = check_matrix_args("bm_f16_matvec_multi", W[m], rows[m], k, x, 1, y[m]);
        if (st != BM_OK) return st;
        for (int q = 0; q < m; q++)
            if (overlap(y[m], rows[m] * 4, y[q], rows[q] * 4) || overlap(y[m], rows[m] * 4, W[q], rows[q] * k * 2) ||
                overlap(y[q], rows[q] * 4, W[m], rows[m] * k * 2))
                return fail(BM_ERR_INVALID_ARG, "bm_f16_matvec_multi: output %d overlaps an input or output", m);
        if (rows[m] == 0) continue;  // empty matrices take no row groups
        job.W[job.nmat] = W[m];
        job.y[job.nmat] = y[m];
        job.rows[job.nmat] = rows[m];
        job.nmat++;
    }
    if (job.nmat == 0) return BM_OK;
    int st;
    DeviceInfo dev;
    if (!current_device(&dev, &st)) return st;
    return launch_vecdot_1col(job, reinterpret_cast<cudaStream_t>(stream), dev);
}

namespace {

// bm_f16_matvec_act and bm_f16_matvec_norm: the f32 activation, optionally normalised
// (nrm non-null), rounded to f16 and multiplied by up to four matrices.
int act_products(const char *fn, int nmat, const uint16_t *const *W, const int64_t *rows, int64_t k, const float *x,
                 const ActNorm *nrm, uint16_t *h, float *const *y, bm_stream_t stream)
{
    if (nmat < 1 || nmat > 4) return fail(BM_ERR_INVALID_ARG, "%s: nmat = %d outside 1..4", fn, nmat);
    if (!W || !rows || !y) return fail(BM_ERR_INVALID_ARG, "%s: null host array", fn);
    if (k < 1 || k > BM_MAX_K) return fail(BM_ERR_INVALID_ARG, "%s: k = %lld outside 1..%d", fn, (long long)k, BM_MAX_K);
    if (!x) return fail(BM_ERR_INVALID_ARG, "%s: null activation", fn);
    if (!aligned(x, 16) || (h && !aligned(h, 16)))
        return fail(BM_ERR_ALIGNMENT, "%s: x and h must be 16-byte aligned", fn);
    if (h && overlap(h, k * 2, x, k * 4)) return fail(BM_ERR_INVALID_ARG, "%s: h overlaps x", fn);
    float *n_out = nrm ? nrm->n_out : nullptr;
    if (nrm) {
        if (!nrm->g) return fail(BM_ERR_INVALID_ARG, "%s: null norm weight", fn);
        if (!aligned(nrm->g, 16) || (n_out && !aligned(n_out, 16)))
            return fail(BM_ERR_ALIGNMENT, "%s: g and n_out must be 16-byte aligned", fn);
        if (n_out && (overlap(n_out, k * 4, x, k * 4) || overlap(n_out, k * 4, nrm->g, k * 4) ||
                      (h && overlap(n_out, k * 4, h, k * 2))))
            return fail(BM_ERR_INVALID_ARG, "%s: n_out overlaps x, g or h", fn);
        if (h && overlap(h, k * 2, nrm->g, k * 4)) return fail(BM_ERR_INVALID_ARG, "%s: h overlaps g", fn);
    }
    VecdotJob job{};
    job.k = k;
    job.ncols = 1;
    for (int m = 0; m < nmat; m++) {
        // the products' checks, with the activation standing in as X (same size in bytes or larger)
        int st = check_matrix_args(fn, W[m], rows[m], k, reinterpret_cast<const uint16_t *>(x), 1, y[m]);
        if (st != BM_OK) return st;
        if (overlap(y[m], rows[m] * 4, x, k * 4) || (h && (overlap(h, k * 2, y[m], rows[m] * 4) ||
                                                          overlap(h, k * 2, W[m], rows[m] * k * 2))))
            return fail(BM_ERR_INVALID_ARG, "%s: output %d overlaps an input or output", fn, m);
        if (nrm && (overlap(y[m], rows[m] * 4, nrm->g, k * 4) ||
                    (n_out && (overlap(n_out, k * 4, y[m], rows[m] * 4) ||
                               overlap(n_out, k * 4, W[m], rows[m] * k * 2)))))
            return fail(BM_ERR_INVALID_ARG, "%s: output %d overlaps an input or output", fn, m);
        for (int q = 0; q < m; q++)
            if (overlap(y[m], rows[m] * 4, y[q], rows[q] * 4) || overlap(y[m], rows[m] * 4, W[q], rows[q] * k * 2) ||
                overlap(y[q], rows[q] * 4, W[m], rows[m] * k * 2))
                return fail(BM_ERR_INVALID_ARG, "%s: output %d overlaps an input or output", fn, m);
        if (rows[m] == 0) continue;
        job.W[job.nmat] = W[m];
        job.y[job.nmat] = y[m];
        job.rows[job.nmat] = rows[m];
        job.nmat++;
    }
    if (job.nmat > 0 && k % 8 != 0 && !h) return fail(BM_ERR_INVALID_ARG, "%s: k %% 8 != 0 needs the h buffer", fn);
    int st;
    DeviceInfo dev;
    if (!current_device(&dev, &st)) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (job.nmat == 0) {
        if (nrm) return (h || n_out) ? launch_rms_norm(x, nrm->g, 1, k, nrm->eps, n_out, h, s, dev) : BM_OK;
        return h ? launch_to_f16(x, h, k, s, dev) : BM_OK;
    }
    if (k % 8 == 0) return launch_gemv_stream(job, x, h, s, dev, nrm);
    // rows that are not 16-byte aligned: round into h, then the lane-per-chain kernel
    st = nrm ? launch_rms_norm(x, nrm->g, 1, k, nrm->eps, n_out, h, s, dev) : launch_to_f16(x, h, k, s, dev);
    if (st != BM_OK) return st;
    job.X = h;
    return launch_vecdot_1col(job, s, dev);
}

}  // namespace

int bm_f16_matvec_act(int nmat, const uint16_t *const *W, const int64_t *rows, int64_t k, const float *x,
                      uint16_t *h, float *const *y, bm_stream_t stream)
{
    clear_error();
    return act_products("bm_f16_matvec_act", nmat, W, rows, k, x, nullptr, h, y, stream);
}

int bm_f16_matvec_norm(int nmat, const uint16_t *const *W, const int64_t *rows, int64_t k, const float *x,
                       const float *g, float eps, float *n_out, uint16_t *h, float *const *y, bm_stream_t stream)
{
    clear_error();
    ActNorm nrm;
    nrm.g = g;
    nrm.eps = eps;
    nrm.n_out = n_out;
    return act_products("bm_f16_matvec_norm", nmat, W, rows, k, x, &nrm, h, y, stream);
}

int bm_step_create(const bm_matvec_call *calls, int ncalls, bm_step **step)
{
    clear_error();
    if (!step) return fail(BM_ERR_INVALID_ARG, "bm_step_create: null step");
    *step = nullptr;
    if (!calls || ncalls < 1 || ncalls > 65535)
        return fail(BM_ERR_INVALID_ARG, "bm_step_create: ncalls = %d outside 1..65535 (or null calls)", ncalls);
    for (int i = 0; i < ncalls; i++) {
        const bm_matvec_call &c = calls[i];
        if (c.nmat < 1 || c.nmat > 4)
            return fail(BM_ERR_INVALID_ARG, "bm_step_create: call %d: nmat = %d outside 1..4", i, c.nmat);
        if (c.k < 8 || c.k > BM_MAX_K || c.k % 8 != 0)
            return fail(BM_ERR_INVALID_ARG, "bm_step_create: call %d: k = %lld (need 8 <= k <= %d, k %% 8 == 0)", i,
                        (long long)c.k, BM_MAX_K);
        if (!c.x) return fail(BM_ERR_INVALID_ARG, "bm_step_create: call %d: null activation", i);
        if (!aligned(c.x, 16)) return fail(BM_ERR_ALIGNMENT, "bm_step_create: call %d: x must be 16-byte aligned", i);
        for (int m = 0; m < c.nmat; m++) {
            if (c.rows[m] > 0x7fffffffLL)
                return fail(BM_ERR_INVALID_ARG, "bm_step_create: call %d: rows must be below 2^31", i);
            int st = check_matrix_args("bm_step_create", c.W[m], c.rows[m], c.k,
                                       reinterpret_cast<const uint16_t *>(c.x), 1, c.y[m]);
            if (st != BM_OK) return st;
            if (c.rows[m] == 0) continue;
            if (overlap(c.y[m], c.rows[m] * 4, c.x, c.k * 4))
                return fail(BM_ERR_INVALID_ARG, "bm_step_create: call %d: output %d overlaps the activation", i, m);
            for (int q = 0; q < m; q++)
                if (c.rows[q] > 0 && (overlap(c.y[m], c.rows[m] * 4, c.y[q], c.rows[q] * 4) ||
                                      overlap(c.y[m], c.rows[m] * 4, c.W[q], c.rows[q] * c.k * 2) ||
                                      overlap(c.y[q], c.rows[q] * 4, c.W[m], c.rows[m] * c.k * 2)))
                    return fail(BM_ERR_INVALID_ARG, "bm_step_create: call %d: output %d overlaps an input or output",
                                i, m);
        }
    }
    // no call writes into any call's weights (the weights of later calls stream early)
    for (int i = 0; i < ncalls; i++)
        for (int m = 0; m < calls[i].nmat; m++) {
            if (calls[i].rows[m] == 0) continue;
            for (int j = 0; j < ncalls; j++)
                for (int q = 0; q < calls[j].nmat; q++)
                    if (calls[j].rows[q] > 0 && overlap(calls[i].y[m], calls[i].rows[m] * 4, calls[j].W[q],
                                                        calls[j].rows[q] * calls[j].k * 2))
                        return fail(BM_ERR_INVALID_ARG, "bm_step_create: call %d writes into call %d's weights", i, j);
        }
    int st;
    DeviceInfo dev;
    if (!current_device(&dev, &st)) return st;
    void *h = nullptr;
    st = step_create(calls, ncalls, dev, &h);
    if (st != BM_OK) return st;
    *step = static_cast<bm_step *>(h);
    return BM_OK;
}

int bm_step_run(const bm_step *step, bm_stream_t stream)
{
    clear_error();
    if (!step) return fail(BM_ERR_INVALID_ARG, "bm_step_run: null step");
    return step_run(const_cast<bm_step *>(step), reinterpret_cast<cudaStream_t>(stream));
}

int bm_step_destroy(bm_step *step)
{
    clear_error();
    step_destroy(step);
    return BM_OK;
}

int bm_rms_norm_mul(const float *x, const float *g, int64_t nrows, int64_t k, float eps, float *out, uint16_t *h,
                    bm_stream_t stream)
{
    clear_error();
    if (nrows < 0 || k < 1 || k > BM_MAX_K)
        return fail(BM_ERR_INVALID_ARG, "bm_rms_norm_mul: nrows = %lld, k = %lld (need nrows >= 0, 1 <= k <= %d)",
                    (long long)nrows, (long long)k, BM_MAX_K);
    if (nrows > (INT64_MAX / 4) / k) return fail(BM_ERR_INVALID_ARG, "bm_rms_norm_mul: nrows * k too large");
    if (!x || !g) return fail(BM_ERR_INVALID_ARG, "bm_rms_norm_mul: null x or g");
    if (!out && !h) return fail(BM_ERR_INVALID_ARG, "bm_rms_norm_mul: neither out nor h given");
    if (!aligned(x, 4) || !aligned(g, 4) || (out && !aligned(out, 4)) || (h && !aligned(h, 2)))
        return fail(BM_ERR_ALIGNMENT, "bm_rms_norm_mul: x, g, out must be 4-byte aligned and h 2-byte aligned");
    const int64_t n = nrows * k;
    if (out && out != x && overlap(out, n * 4, x, n * 4))
        return fail(BM_ERR_INVALID_ARG, "bm_rms_norm_mul: out overlaps x without being x");
    if ((out && overlap(out, n * 4, g, k * 4)) || (h && (overlap(h, n * 2, x, n * 4) || overlap(h, n * 2, g, k * 4) ||
                                                         (out && overlap(h, n * 2, out, n * 4)))))
        return fail(BM_ERR_INVALID_ARG, "bm_rms_norm_mul: an output overlaps an input or the other output");
    if (nrows == 0) return BM_OK;
    int st;
    DeviceInfo dev;
    if (!current_device(&dev, &st)) return st;
    return launch_rms_norm(x, g, nrows, k, eps, out, h, reinterpret_cast<cudaStream_t>(stream), dev);
}

int bm_f16_matmul(const uint16_t *W, int64_t rows, int64_t k, const uint16_t *X, int64_t ncols, float *Y,
                  bm_stream_t stream)
{
    clear_error();
    return product("bm_f16_matmul", W, rows, k, X, ncols, Y, stream);
}

int bm_f16_matmul_multi(int nmat, const uint16_t *const *W, const int64_t *rows, int64_t k, const uint16_t *X,
                        int64_t ncols, float *const *Y, bm_stream_t stream)
{
    clear_error();
    if (nmat < 1 || nmat > 4) return fail(BM_ERR_INVALID_ARG, "bm_f16_matmul_multi: nmat = %d outside 1..4", nmat);
    if (!W || !rows || !Y) return fail(BM_ERR_INVALID_ARG, "bm_f16_matmul_multi: null host array");
    for (int m = 0; m < nmat; m++) {
        int st = check_matrix_args("bm_f16_matmul_multi", W[m], rows[m], k, X, ncols, Y[m]);
        if (st != BM_OK) return st;
        for (int q = 0; q < m; q++)
            if (overlap(Y[m], rows[m] * ncols * 4, Y[q], rows[q] * ncols * 4) ||
                overlap(Y[m], rows[m] * ncols * 4, W[q], rows[q] * k * 2) ||
                overlap(Y[q], rows[q] * ncols * 4, W[m], rows[m] * k * 2))
                return fail(BM_ERR_INVALID_ARG, "bm_f16_matmul_multi: output %d overlaps an input or output", m);
    }
    if (ncols == 0) return BM_OK;
    // The matrices whose own shape takes the tensor-core path share one launch; any other
    // matrix (vec_dot, or tinyBLAS's bits on the CUDA-core kernel) is its own product.
    const int exact_cols = g_exact_cols.load(std::memory_order_relaxed);
    const uint16_t *tw[4];
    int64_t trows[4];
    float *ty[4];
    int nt = 0;
    for (int m = 0; m < nmat; m++) {
        if (rows[m] == 0) continue;
        if (bm_takes_sgemm(rows[m], k, ncols) && ncols > exact_cols) {
            tw[nt] = W[m];
            trows[nt] = rows[m];
            ty[nt] = Y[m];
            nt++;
            continue;
        }
        int st = product("bm_f16_matmul_multi", W[m], rows[m], k, X, ncols, Y[m], stream);
        if (st != BM_OK) return st;
    }
    if (nt == 0) return BM_OK;
    int st;
    DeviceInfo dev;
    if (!current_device(&dev, &st)) return st;
    return launch_gemm_tc_multi(nt, tw, trows, k, X, ncols, ty, reinterpret_cast<cudaStream_t>(stream), dev);
}

int bm_f16_matmul_noalloc(const uint16_t *W, int64_t rows, int64_t k, const uint16_t *X, int64_t ncols, float *Y,
                          bm_stream_t stream)
{
    clear_error();
    int st = check_matrix_args("bm_f16_matmul_noalloc", W, rows, k, X, ncols, Y);
    if (st != BM_OK || rows == 0 || ncols == 0) return st;
    DeviceInfo dev;
    if (!current_device(&dev, &st)) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // the CUDA-core kernels use no scratch memory
    if (bm_takes_sgemm(rows, k, ncols))
        return ncols <= g_exact_cols.load(std::memory_order_relaxed)
                   ? launch_sgemm_stream(W, rows, k, X, ncols, Y, s, dev)
                   : launch_gemm_tc_noalloc(W, rows, k, X, ncols, Y, s, dev);
    VecdotJob job{};
    job.W[0] = W;
    job.y[0] = Y;
    job.rows[0] = rows;
    job.nmat = 1;
    job.k = k;
    job.X = X;
    job.ncols = ncols;
    return ncols == 1 ? launch_vecdot_1col(job, s, dev) : launch_vecdot_ncol(job, s, dev);
}

int bm_f16_logits(const uint16_t *E, int64_t vocab, int64_t hidden, const uint16_t *X, int64_t ncols, float *Y,
                  bm_stream_t stream)
{
    clear_error();
    return product("bm_f16_logits", E, vocab, hidden, X, ncols, Y, stream);
}

int bm_set_pdl(int enable)
{
    clear_error();
    return g_pdl.exchange(enable ? 1 : 0);
}

int bm_set_exact_sgemm_cols(int ncols)
{
    clear_error();
    return g_exact_cols.exchange(std::max(0, std::min(ncols, kSgemmStreamMaxCols)));
}

int bm_set_stream_k(int mode)
{
    clear_error();
    return g_stream_k.exchange(mode < 0 ? -1 : mode > 0 ? 1 : 0);
}

int bm_tc_plan(int64_t rows, int64_t k, int64_t ncols, int noalloc, int64_t *info)
{
    clear_error();
    if (!info) return fail(BM_ERR_INVALID_ARG, "bm_tc_plan: null info");
    if (k < 1 || k > BM_MAX_K || rows < 1 || !bm_takes_sgemm(rows, k, ncols))
        return fail(BM_ERR_INVALID_ARG, "bm_tc_plan: %lld x %lld x %lld is not a tensor-core product",
                    (long long)rows, (long long)k, (long long)ncols);
    if (!sizes_ok(rows, k) || !sizes_ok(ncols, k) || ncols > INT64_MAX / 8 / rows)
        return fail(BM_ERR_INVALID_ARG, "bm_tc_plan: sizes overflow");
    int st;
    DeviceInfo dev;
    if (!current_device(&dev, &st)) return st;
    return plan_info_gemm_tc(rows, k, ncols, noalloc != 0, dev, info);
}

int bm_device_status(bm_stream_t stream)
{
    clear_error();
    return read_device_error(reinterpret_cast<cudaStream_t>(stream));
}

int bm_selftest_wait_timeout(const uint16_t *W, const uint16_t *X, float *Y, bm_stream_t stream)
{
    clear_error();
    int st = check_matrix_args("bm_selftest_wait_timeout", W, 128, 64, X, 16, Y);
    if (st != BM_OK) return st;
    DeviceInfo dev;
    if (!current_device(&dev, &st)) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // Clear any earlier give-up first, so the status read below is this run's.
    st = read_device_error(s);
    if (st != BM_OK && st != BM_ERR_TIMEOUT) return st;
    st = launch_gemm_tc_withheld(W, 128, 64, X, 16, Y, s, dev, 20ull * 1000 * 1000);
    if (st != BM_OK) return st;
    st = read_device_error(s);
    if (st == BM_OK) return fail(BM_ERR_CUDA, "bm_selftest_wait_timeout: the withheld wait did not give up");
    return st;
}

const char *bm_status_string(int status)
{
    switch (status) {
    case BM_OK: return "ok";
    case BM_ERR_INVALID_ARG: return "invalid argument";
    case BM_ERR_ALIGNMENT: return "misaligned pointer";
    case BM_ERR_UNSUPPORTED_DEVICE: return "unsupported device (needs sm_103)";
    case BM_ERR_CUDA: return "CUDA error";
    case BM_ERR_TIMEOUT: return "device-side bounded wait gave up";
    default: return "unknown status";
    }
}

const char *bm_last_error(void) { return g_last_error; }

}  // extern "C"
