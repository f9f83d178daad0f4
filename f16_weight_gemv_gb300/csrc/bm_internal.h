// bm_internal.h -- shared declarations of the CUDA library behind include/bm.h.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/bm.h"

namespace bm {

// Per-device facts read once.
struct DeviceInfo {
    int major = 0, minor = 0;
    int sm_count = 0;
    int max_smem_optin = 0;  // bytes of dynamic shared memory a block may opt into
    int smem_per_sm = 0;     // bytes of shared memory of one SM
    int smem_reserved = 0;   // bytes of it the system reserves for each resident block
};

// Fills *info for the current device; returns false (and sets the last error)
// when the device cannot be queried or is not compute capability 10.3.
bool current_device(DeviceInfo *info, int *status);

// Records a reason for the calling host thread and returns `status`.
int fail(int status, const char *fmt, ...);

// Device address of this library's error word on the current device (kernels
// that give up a bounded wait write BM_ERR_TIMEOUT there), or null on failure.
unsigned int *device_error_word();

// Whether products are launched with programmatic dependent launch (bm_set_pdl).
bool pdl_enabled();
int stream_k_mode();  // bm_set_stream_k: -1 by the time model, 0 never, 1 always

// Up to four matrices that share one activation (the fused Q/K/V or gate/up
// products), or one matrix with several activation columns.
struct VecdotJob {
    const uint16_t *W[4];
    float *y[4];
    int64_t rows[4];
    int64_t gbeg[5];  // first row group of matrix m; gbeg[nmat] = total groups
    int nmat;
    int64_t k;
    const uint16_t *X;  // activation column(s), [ncols][k]
    int64_t ncols;
};

// Launchers (each returns a bm_status; nothing is launched for empty jobs).
int launch_to_f16(const float *x, uint16_t *h, int64_t n, cudaStream_t s, const DeviceInfo &dev);
// bm_f16_mad (mad = true: acc = f16(fma(v, w, acc))) and bm_f16_scale (acc = f16(acc * w)).
int launch_f16_accum(bool mad, uint16_t *acc, const uint16_t *v, float w, int64_t n, cudaStream_t s,
                     const DeviceInfo &dev);
// One column, any k; uses the 16-byte fast kernel when k % 8 == 0.
int launch_vecdot_1col(const VecdotJob &job, cudaStream_t s, const DeviceInfo &dev);
// The rms_norm then mul that may precede the rounding of an f32 activation.
struct ActNorm {
    const float *g = nullptr;  // norm weight, f32[k], 16-byte aligned
    float eps = 0.0f;
    float *n_out = nullptr;    // optional: the normalised row, f32[k], 16-byte aligned
};
// One column, k % 8 == 0: rows streamed through shared memory by TMA.  With
// x_f32 non-null the activation is read in f32 and rounded in the kernel
// (job.X is then unused), after rms_norm then mul when nrm is non-null; h_out, if
// non-null, receives the rounded activation.
int launch_gemv_stream(const VecdotJob &job, const float *x_f32, uint16_t *h_out, cudaStream_t s,
                       const DeviceInfo &dev, const ActNorm *nrm = nullptr);
// One column, rows not 16-byte aligned (k % 8 != 0): each row's k-slices streamed by
// 1-D bulk copies of their 16-byte-aligned windows (job.X 16-byte aligned).
int launch_gemv_bulk(const VecdotJob &job, cudaStream_t s, const DeviceInfo &dev);
// rms_norm then mul of nrows rows of k values (out and/or h; out may equal x).
int launch_rms_norm(const float *x, const float *g, int64_t nrows, int64_t k, float eps, float *out, uint16_t *h,
                    cudaStream_t s, const DeviceInfo &dev);
// ncols >= 1 columns of one matrix, any k, Y[c*rows + r], bit-exact vec_dot.
int launch_vecdot_ncol(const VecdotJob &job, cudaStream_t s, const DeviceInfo &dev);
// Most columns taken by the CUDA-core tinyBLAS kernel (launch_sgemm_stream); wider
// bm_takes_sgemm products go to the tensor cores.
constexpr int kSgemmStreamMaxCols = 8;
// bm_takes_sgemm shapes with 2..kSgemmStreamMaxCols columns: tinyBLAS's sgemm_dot per
// element, bit for bit, on the CUDA cores, weights streamed through shared memory by TMA.
int launch_sgemm_stream(const uint16_t *W, int64_t rows, int64_t k, const uint16_t *X, int64_t ncols, float *Y,
                        cudaStream_t s, const DeviceInfo &dev);
// launch_sgemm_stream's products on the one-column kernel's streaming (k_sgemm_ring.cu):
// same bits; taken when sgemm_ring_applies (X 16-byte aligned and small enough to stage
// whole in shared memory).
bool sgemm_ring_applies(const uint16_t *X, int64_t ncols, int64_t k, const DeviceInfo &dev);
int launch_sgemm_ring(const uint16_t *W, int64_t rows, int64_t k, const uint16_t *X, int64_t ncols, float *Y,
                      cudaStream_t s, const DeviceInfo &dev);
// Tensor-core product for bm_takes_sgemm shapes (rows % 4 == 0, k % 8 == 0, ncols >= 2).
int launch_gemm_tc(const uint16_t *W, int64_t rows, int64_t k, const uint16_t *X, int64_t ncols,
                   float *Y, cudaStream_t s, const DeviceInfo &dev);
// Up to four bm_takes_sgemm products sharing the activation X in one tensor-core launch:
// Y[m] = W[m] (rows[m] x k) times X (ncols x k), each laid out [ncols][rows[m]].
int launch_gemm_tc_multi(int nmat, const uint16_t *const *W, const int64_t *rows, int64_t k, const uint16_t *X,
                         int64_t ncols, float *const *Y, cudaStream_t s, const DeviceInfo &dev);
// As launch_gemm_tc, with the split-k workspace in a static device array instead of
// a stream-ordered allocation (no allocation of any kind).
int launch_gemm_tc_noalloc(const uint16_t *W, int64_t rows, int64_t k, const uint16_t *X, int64_t ncols,
                           float *Y, cudaStream_t s, const DeviceInfo &dev);
// The plan the tensor-core product takes for one rows x k x ncols product on the current
// device (noalloc: bm_f16_matmul_noalloc's plan): info[0..5] = row tiles per unit (MT),
// tile columns, k-splits, balanced k ranges (0/1), scratch bytes, CTAs.
int plan_info_gemm_tc(int64_t rows, int64_t k, int64_t ncols, bool noalloc, const DeviceInfo &dev, int64_t *info);
// Self-test of the bounded waits: a 128 x 64 x 16 product whose producer never
// fills its only stage, so the MMA issuer gives up after `timeout_ns`.
int launch_gemm_tc_withheld(const uint16_t *W, int64_t rows, int64_t k, const uint16_t *X, int64_t ncols,
                            float *Y, cudaStream_t s, const DeviceInfo &dev, unsigned long long timeout_ns);
// Rows of an f16 table widened to f32 (ids checked on the device).
int launch_get_rows(const uint16_t *E, int64_t vocab, int64_t hidden, const int32_t *ids, int64_t n, float *out,
                    cudaStream_t s, const DeviceInfo &dev);
// A recorded decode step (bm_step_create / bm_step_run / bm_step_destroy); the calls are
// validated by the caller.
int step_create(const bm_matvec_call *calls, int ncalls, const DeviceInfo &dev, void **out);
int step_run(void *step, cudaStream_t s);
void step_destroy(void *step);
// Waits for `s` and reads/clears the device error word of the tensor-core kernels.
int read_device_error(cudaStream_t s);

}  // namespace bm
