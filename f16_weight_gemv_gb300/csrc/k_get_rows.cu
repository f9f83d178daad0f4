// k_get_rows.cu -- rows of an f16 table widened to f32, exactly: the token
// embedding lookup of the page "docs/modules/f16.md" (Technical usage,
// `dequantize_row`: F16 bytes widened to f32, as get_rows does; `widen` is
// exact).  out[i][j] = (float) E[ids[i]][j].
//
// HBM-bound gather: 6 bytes per element (2 read, 4 written).  With hidden % 8 == 0
// and a 16-byte aligned output each thread moves 16-byte chunks (8 f16 in, two
// 16-byte f32 stores out); otherwise one element per thread.  An id outside
// [0, vocab) leaves its output row untouched and records BM_ERR_INVALID_ARG in the
// device error word (bm_device_status).
#include "../../include/bm.h"
#include "bm_device.cuh"
#include "bm_internal.h"

#include <cuda_fp16.h>

namespace bm {
namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ float widen(uint16_t h) { return __half2float(__ushort_as_half(h)); }

__device__ __forceinline__ bool valid_id(int32_t id, int64_t vocab, unsigned int *err)
{
    if (id >= 0 && (int64_t)id < vocab) return true;
    atomicCAS(err, 0u, (unsigned)BM_ERR_INVALID_ARG);
    return false;
}

__global__ void __launch_bounds__(kThreads) k_get_rows_vec(const uint16_t *__restrict__ E, int64_t vocab,
                                                           int64_t hidden, const int32_t *__restrict__ ids, int64_t n,
                                                           float *__restrict__ out, unsigned int *err)
{
    dev::pdl_trigger();
    dev::pdl_wait();  // ids (and the table) may be the previous kernel's output
    const int64_t cpr = hidden >> 3;  // 16-byte chunks per row
    const int64_t total = n * cpr;
    for (int64_t c = (int64_t)blockIdx.x * kThreads + threadIdx.x; c < total; c += (int64_t)gridDim.x * kThreads) {
        const int64_t i = c / cpr, j = c - i * cpr;
        const int32_t id = __ldg(ids + i);
        if (!valid_id(id, vocab, err)) continue;
        const uint4 h = __ldg(reinterpret_cast<const uint4 *>(E + id * hidden) + j);
        const __half2 *p = reinterpret_cast<const __half2 *>(&h);
        const float2 a = __half22float2(p[0]), b = __half22float2(p[1]), q = __half22float2(p[2]),
                     d = __half22float2(p[3]);
        float4 *o = reinterpret_cast<float4 *>(out + i * hidden) + 2 * j;
        o[0] = make_float4(a.x, a.y, b.x, b.y);
        o[1] = make_float4(q.x, q.y, d.x, d.y);
    }
}

__global__ void __launch_bounds__(kThreads) k_get_rows_scalar(const uint16_t *__restrict__ E, int64_t vocab,
                                                              int64_t hidden, const int32_t *__restrict__ ids,
                                                              int64_t n, float *__restrict__ out, unsigned int *err)
{
    dev::pdl_trigger();
    dev::pdl_wait();
    const int64_t total = n * hidden;
    for (int64_t e = (int64_t)blockIdx.x * kThreads + threadIdx.x; e < total; e += (int64_t)gridDim.x * kThreads) {
        const int64_t i = e / hidden, j = e - i * hidden;
        const int32_t id = __ldg(ids + i);
        if (!valid_id(id, vocab, err)) continue;
        out[e] = widen(E[id * hidden + j]);
    }
}

}  // namespace

int launch_get_rows(const uint16_t *E, int64_t vocab, int64_t hidden, const int32_t *ids, int64_t n, float *out,
                    cudaStream_t s, const DeviceInfo &dev)
{
    unsigned int *err = device_error_word();
    if (!err) return fail(BM_ERR_CUDA, "bm_f16_get_rows: device error word unavailable");
    const bool vec = hidden % 8 == 0 && (reinterpret_cast<uintptr_t>(out) & 15) == 0;
    const int64_t work = vec ? n * (hidden >> 3) : n * hidden;
    int64_t blocks = (work + kThreads - 1) / kThreads;
    const int64_t cap = (int64_t)dev.sm_count * 8;  // 8 resident blocks of 256 threads per SM
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)blocks);
    cfg.blockDim = dim3(kThreads);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_enabled() ? 1 : 0;
    cudaError_t e = vec ? cudaLaunchKernelEx(&cfg, k_get_rows_vec, E, vocab, hidden, ids, n, out, err)
                        : cudaLaunchKernelEx(&cfg, k_get_rows_scalar, E, vocab, hidden, ids, n, out, err);
    if (e != cudaSuccess) return fail(BM_ERR_CUDA, "bm_f16_get_rows: launch failed: %s", cudaGetErrorString(e));
    return BM_OK;
}

}  // namespace bm
