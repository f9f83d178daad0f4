// k_rms_norm.cu -- rms_norm then mul of whole rows (page "docs/modules/forward.md",
// Technical usage, "Other public pieces"; Design notes, step three: the first RMS
// norm with its weight gives attn_norm-0), optionally rounded to f16 for the
// products that follow (page "docs/modules/f16.md", Design notes, "Activation").
//
// One CTA of kNormThreads threads per row (grid-stride over rows).  The steps
// are those of bm_norm.cuh (the sum of squares exact in a 128-bit integer, the
// mean by integer steps), shared with the fused front end of k_gemv_stream, so
// the two give the same bits.  A row of up to 4096 values is read once into
// registers for the sum; rows of 1025..4096 values also take their outputs from
// there (with the norm weight's chunks loaded together), shorter ones read x once
// more, longer ones three times (largest square, exact sum, scaled values; the
// later reads hit L1/L2).  Outputs are written once.
//
// In place (out == x) is safe: every thread has finished reading the row for the
// sum before the block barrier, and the second pass reads and writes each element
// in the same thread.
#include "../../include/bm.h"
#include "bm_device.cuh"
#include "bm_internal.h"
#include "bm_norm.cuh"

#include <cuda_fp16.h>

namespace bm {
namespace {

using norm::kNormThreads;

__device__ __forceinline__ uint32_t pack_rn(float lo, float hi)
{
    __half2 p = __floats2half2_rn(lo, hi);  // lo -> low 16 bits
    return *reinterpret_cast<uint32_t *>(&p);
}

__device__ __forceinline__ uint16_t to_f16(float v)
{
    __half r = __float2half_rn(v);
    return *reinterpret_cast<uint16_t *>(&r);
}

// vec: x, g and out 16-byte aligned, h 8-byte aligned and k % 4 == 0, so that every
// row keeps that alignment.  HOLD (rows of 1025..4096 values, several chunks a thread):
// the outputs come from the chunks held for the sum, with the norm weight's chunks
// loaded together, instead of a second pass of serial round trips; it takes more
// registers, which rows of one chunk a thread would pay for in occupancy.
template <bool HOLD>
__global__ void __launch_bounds__(kNormThreads) k_rms_norm(const float *x, const float *__restrict__ g, int64_t nrows,
                                                           int64_t k, norm::Recip rk, float eps, float *out,
                                                           uint16_t *h, int vec)
{
    __shared__ norm::Scratch sh;
    dev::pdl_trigger();
    dev::pdl_wait();  // x may be the previous kernel's output
    const int t = threadIdx.x;
    for (int64_t r = blockIdx.x; r < nrows; r += gridDim.x) {
        const float *xr = x + r * k;
        float scale;
        if (HOLD) {
            // the row's chunks held in registers: one read of x; after the reduction the norm
            // weight's chunks, all four loads in flight together, and the outputs from the
            // registers
            const int64_t n4 = k >> 2;
            float4 v[4], w[4];
#pragma unroll
            for (int i = 0; i < 4; i++) {
                const int64_t c = t + i * kNormThreads;
                v[i] = c < n4 ? reinterpret_cast<const float4 *>(xr)[c] : make_float4(0.f, 0.f, 0.f, 0.f);
            }
            scale = norm::row_scale_held(v, (int)n4, rk, eps, t, sh, [] { __syncthreads(); });
            __syncthreads();  // sh is refilled by the next row
#pragma unroll
            for (int i = 0; i < 4; i++) {
                const int64_t c = t + i * kNormThreads;
                w[i] = c < n4 ? __ldg(reinterpret_cast<const float4 *>(g) + c) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
            float4 *o4 = out ? reinterpret_cast<float4 *>(out + r * k) : nullptr;
            uint2 *h4 = h ? reinterpret_cast<uint2 *>(h + r * k) : nullptr;
#pragma unroll
            for (int i = 0; i < 4; i++) {
                const int64_t c = t + i * kNormThreads;
                if (c < n4) {
                    const float4 o = make_float4(norm::apply(v[i].x, scale, w[i].x), norm::apply(v[i].y, scale, w[i].y),
                                                 norm::apply(v[i].z, scale, w[i].z), norm::apply(v[i].w, scale, w[i].w));
                    if (o4) o4[c] = o;
                    if (h4) h4[c] = make_uint2(pack_rn(o.x, o.y), pack_rn(o.z, o.w));
                }
            }
            continue;
        } else if (vec && k <= 4 * 4 * kNormThreads) {  // the row's chunks held in registers for the sum
            const int64_t n4 = k >> 2;
            float4 v[4];
#pragma unroll
            for (int i = 0; i < 4; i++) {
                const int64_t c = t + i * kNormThreads;
                v[i] = c < n4 ? reinterpret_cast<const float4 *>(xr)[c] : make_float4(0.f, 0.f, 0.f, 0.f);
            }
            scale = norm::row_scale_held(v, (int)n4, rk, eps, t, sh, [] { __syncthreads(); });
        } else {
            scale = norm::row_scale(xr, k, rk, eps, vec != 0, t, sh, [] { __syncthreads(); });
        }
        __syncthreads();  // sh is refilled by the next row
        if (vec) {
            const float4 *x4 = reinterpret_cast<const float4 *>(xr);
            const float4 *g4 = reinterpret_cast<const float4 *>(g);
            float4 *o4 = out ? reinterpret_cast<float4 *>(out + r * k) : nullptr;
            uint2 *h4 = h ? reinterpret_cast<uint2 *>(h + r * k) : nullptr;
            for (int64_t c = t; c < (k >> 2); c += kNormThreads) {
                const float4 v = x4[c], w = __ldg(g4 + c);
                const float4 o = make_float4(norm::apply(v.x, scale, w.x), norm::apply(v.y, scale, w.y),
                                             norm::apply(v.z, scale, w.z), norm::apply(v.w, scale, w.w));
                if (o4) o4[c] = o;
                if (h4) h4[c] = make_uint2(pack_rn(o.x, o.y), pack_rn(o.z, o.w));
            }
        } else {
            for (int64_t i = t; i < k; i += kNormThreads) {
                const float o = norm::apply(xr[i], scale, __ldg(g + i));
                if (out) out[r * k + i] = o;
                if (h) h[r * k + i] = to_f16(o);
            }
        }
    }
}

}  // namespace

int launch_rms_norm(const float *x, const float *g, int64_t nrows, int64_t k, float eps, float *out, uint16_t *h,
                    cudaStream_t s, const DeviceInfo &dev)
{
    if (nrows == 0) return BM_OK;
    const auto a16 = [](const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; };
    const bool vec = k % 4 == 0 && a16(x) && a16(g) && (!out || a16(out)) &&
                     (!h || (reinterpret_cast<uintptr_t>(h) & 7) == 0);
    int64_t blocks = nrows;
    const int64_t cap = (int64_t)dev.sm_count * 8;  // 8 resident blocks of 256 threads per SM
    if (blocks > cap) blocks = cap;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)blocks);
    cfg.blockDim = dim3(kNormThreads);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_enabled() ? 1 : 0;
    const bool hold = vec && k > 4 * kNormThreads && k <= 4 * 4 * kNormThreads;
    cudaError_t e = hold ? cudaLaunchKernelEx(&cfg, k_rms_norm<true>, x, g, nrows, k, norm::reciprocal_of(k), eps, out, h, 1)
                         : cudaLaunchKernelEx(&cfg, k_rms_norm<false>, x, g, nrows, k, norm::reciprocal_of(k), eps, out, h,
                                              vec ? 1 : 0);
    if (e != cudaSuccess) return fail(BM_ERR_CUDA, "rms_norm: launch failed: %s", cudaGetErrorString(e));
    return BM_OK;
}

}  // namespace bm
