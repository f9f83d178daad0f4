// k_to_f16.cu -- the activation rounding of the page "docs/modules/f16.md"
// (Design notes, "Activation"): every f32 activation value is rounded to f16,
// to nearest with ties to even, before any product.
//
// HBM-bound elementwise kernel: 6 bytes per element (4 read, 2 written).
// Each thread converts 8 values per trip: two 16-byte loads, one 16-byte store.
// cvt.rn.f16x2.f32 rounds to nearest even, keeps f16 subnormals and sends
// |x| >= 65520 to infinity, which is the IEEE binary16 conversion.
#include "../../include/bm.h"
#include "bm_device.cuh"
#include "bm_internal.h"

#include <cuda_fp16.h>

namespace bm {
namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ uint32_t pack_rn(float lo, float hi)
{
    __half2 p = __floats2half2_rn(lo, hi);  // lo -> low 16 bits
    return *reinterpret_cast<uint32_t *>(&p);
}

__global__ void __launch_bounds__(kThreads) k_to_f16(const float *__restrict__ x, uint16_t *__restrict__ h, int64_t n)
{
    // Under programmatic dependent launch: let the next kernel be scheduled now, and
    // touch x and h only once the kernel ahead of this one has finished.
    dev::pdl_trigger();
    dev::pdl_wait();
    const int64_t nv = n >> 3;
    const int64_t stride = (int64_t)gridDim.x * kThreads;
    const float4 *xv = reinterpret_cast<const float4 *>(x);
    uint4 *hv = reinterpret_cast<uint4 *>(h);
    for (int64_t v = (int64_t)blockIdx.x * kThreads + threadIdx.x; v < nv; v += stride) {
        float4 a = __ldcs(xv + 2 * v);
        float4 b = __ldcs(xv + 2 * v + 1);
        uint4 o;
        o.x = pack_rn(a.x, a.y);
        o.y = pack_rn(a.z, a.w);
        o.z = pack_rn(b.x, b.y);
        o.w = pack_rn(b.z, b.w);
        hv[v] = o;
    }
    // the n % 8 ragged end, one element per thread of the first block
    if (blockIdx.x == 0 && threadIdx.x < (n & 7)) {
        int64_t i = (nv << 3) + threadIdx.x;
        __half r = __float2half_rn(x[i]);
        h[i] = *reinterpret_cast<uint16_t *>(&r);
    }
}

}  // namespace

int launch_to_f16(const float *x, uint16_t *h, int64_t n, cudaStream_t s, const DeviceInfo &dev)
{
    int64_t nv = n >> 3;
    int64_t blocks = (nv + kThreads - 1) / kThreads;
    int64_t cap = (int64_t)dev.sm_count * 8;  // 8 resident blocks of 256 threads per SM
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
    cudaError_t e = cudaLaunchKernelEx(&cfg, k_to_f16, x, h, n);
    if (e != cudaSuccess) return fail(BM_ERR_CUDA, "bm_to_f16: launch failed: %s", cudaGetErrorString(e));
    return BM_OK;
}

}  // namespace bm
