// k_f16_accum.cu -- the f16 accumulator helpers of the attention side (page
// "docs/modules/f16.md", Technical usage: `mad` is ggml_vec_mad_f16, flash
// attention's V accumulator; `scale` is ggml_vec_scale_f16), in place on an f16
// vector:
//   mad:   acc[i] = f16(fma(widen(v[i]), w, widen(acc[i])))
//   scale: acc[i] = f16(widen(acc[i]) * s)
// The product and sum of mad round once in f32 (__fmaf_rn), the product of scale is
// one f32 multiply (__fmul_rn: never fused with anything), and the f32 result goes to
// f16 nearest-even (__float2half_rn); widening f16 to f32 is exact.
//
// HBM-bound elementwise kernels: mad moves 6 bytes per element (acc and v read, acc
// written), scale 4.  With 16-byte aligned vectors each thread handles 8 elements per
// trip (16-byte loads and stores), the n % 8 end one element per thread of the first
// block; otherwise one element per thread.  v may be acc itself.
#include "../../include/bm.h"
#include "bm_device.cuh"
#include "bm_internal.h"

#include <cuda_fp16.h>

namespace bm {
namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ float widen(uint16_t h) { return __half2float(__ushort_as_half(h)); }

__device__ __forceinline__ uint16_t to_f16(float x) { return __half_as_ushort(__float2half_rn(x)); }

template <bool kMad>
__device__ __forceinline__ uint16_t step(uint16_t a, uint16_t v, float w)
{
    return kMad ? to_f16(__fmaf_rn(widen(v), w, widen(a))) : to_f16(__fmul_rn(widen(a), w));
}

template <bool kMad>
__global__ void __launch_bounds__(kThreads) k_f16_accum(uint16_t *acc, const uint16_t *v, float w, int64_t n, int vec)
{
    // acc (and v) may be the previous kernel's output
    dev::pdl_trigger();
    dev::pdl_wait();
    const int64_t stride = (int64_t)gridDim.x * kThreads;
    const int64_t t0 = (int64_t)blockIdx.x * kThreads + threadIdx.x;
    if (vec) {
        const int64_t nv = n >> 3;
        uint4 *av = reinterpret_cast<uint4 *>(acc);
        const uint4 *vv = reinterpret_cast<const uint4 *>(v);
        for (int64_t q = t0; q < nv; q += stride) {
            uint4 a = av[q];
            uint4 b = kMad ? vv[q] : make_uint4(0, 0, 0, 0);
            uint32_t *pa = reinterpret_cast<uint32_t *>(&a);
            const uint32_t *pb = reinterpret_cast<const uint32_t *>(&b);
#pragma unroll
            for (int e = 0; e < 4; e++) {
                const uint16_t lo = step<kMad>((uint16_t)(pa[e] & 0xffffu), (uint16_t)(pb[e] & 0xffffu), w);
                const uint16_t hi = step<kMad>((uint16_t)(pa[e] >> 16), (uint16_t)(pb[e] >> 16), w);
                pa[e] = (uint32_t)lo | ((uint32_t)hi << 16);
            }
            av[q] = a;
        }
        if (blockIdx.x == 0 && threadIdx.x < (n & 7)) {
            const int64_t i = (nv << 3) + threadIdx.x;
            acc[i] = step<kMad>(acc[i], kMad ? v[i] : (uint16_t)0, w);
        }
    } else {
        for (int64_t i = t0; i < n; i += stride) acc[i] = step<kMad>(acc[i], kMad ? v[i] : (uint16_t)0, w);
    }
}

}  // namespace

int launch_f16_accum(bool mad, uint16_t *acc, const uint16_t *v, float w, int64_t n, cudaStream_t s,
                     const DeviceInfo &dev)
{
    const auto a16 = [](const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; };
    const bool vec = a16(acc) && (!mad || a16(v));
    const int64_t work = vec ? (n >> 3) : n;
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
    cudaError_t e = mad ? cudaLaunchKernelEx(&cfg, k_f16_accum<true>, acc, v, w, n, vec ? 1 : 0)
                        : cudaLaunchKernelEx(&cfg, k_f16_accum<false>, acc, v, w, n, vec ? 1 : 0);
    if (e != cudaSuccess)
        return fail(BM_ERR_CUDA, "%s: launch failed: %s", mad ? "bm_f16_mad" : "bm_f16_scale", cudaGetErrorString(e));
    return BM_OK;
}

}  // namespace bm
