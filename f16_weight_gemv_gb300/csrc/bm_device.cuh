// bm_device.cuh -- device-side building blocks shared by the kernels:
// mbarrier waits bounded by the global timer, 1-D bulk copies (TMA),
// programmatic-dependent-launch controls.
#pragma once

#include <cstdint>

namespace bm {
namespace dev {

constexpr unsigned kTimeoutStatus = 5;  // BM_ERR_TIMEOUT

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long now_ns()
{
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count));
}

// Makes initialised barriers visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_barrier_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// As mbar_try_wait, but the thread may be suspended in hardware for up to
// `hint_ns` nanoseconds waiting for the phase (it resumes as soon as the phase
// completes), so a waiting warp does not spin on the issue slots.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity, uint32_t hint_ns)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}

// Waits for the phase of parity `parity` to complete.  Gives up when the CTA's
// abort flag is raised, or after `timeout_ns`, in which case it raises the
// flag and records the give-up in the device error word.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                          unsigned long long timeout_ns, unsigned int *err_word)
{
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = now_ns();
    while (true) {
        if (mbar_try_wait_sleep(bar, parity, 20000u)) return true;
        if (*abort_flag) return false;
        if (now_ns() - t0 > timeout_ns) {
            *abort_flag = 1;
            atomicExch(err_word, kTimeoutStatus);
            return false;
        }
    }
}

// mbar_wait for all 32 lanes of a warp, with one answer for the whole warp (a lane
// that gave up makes every lane give up, so later warp-collective steps stay uniform).
__device__ __forceinline__ bool mbar_wait_warp(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                               unsigned long long timeout_ns, unsigned int *err_word)
{
    const bool ok = mbar_wait(bar, parity, abort_flag, timeout_ns, err_word);
    return __all_sync(0xffffffffu, ok);
}

// Bounded drain used on the abort path: waits for a phase without raising anything.
__device__ __forceinline__ void mbar_drain(uint32_t bar, uint32_t parity, unsigned long long timeout_ns)
{
    const unsigned long long t0 = now_ns();
    while (!mbar_try_wait(bar, parity) && now_ns() - t0 < timeout_ns) {
    }
}

// 1-D bulk copy global -> shared, completing `bytes` on mbarrier `bar`.
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     dst),
                 "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}

// Programmatic dependent launch.  Without a programmatic launch both are no-ops
// in effect: the grid only starts once the previous work on the stream is done.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

}  // namespace dev
}  // namespace bm
