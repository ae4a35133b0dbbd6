// Device helpers shared by the library's kernels: Q2_K / q8_1 constants,
// inline PTX for bulk asynchronous copies, mbarriers with bounded waits,
// and the integer dot products.  sm_103a only.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace q2k {

constexpr int kBlockBytes = 84;   // one Q2_K super-block (engram_v41.rs, ENGRAM_ROW_BYTES)
constexpr int kBlockWeights = 256;
constexpr int kQ8Bytes = 36;      // q8_1 block: fp16 d, fp16 s, int8 q[32]
constexpr int kQ8Values = 32;

// Library error word (bit 0: a bounded wait gave up).  One per module;
// q2k_device_error() reads every module's word.
#define Q2K_ERR_BIT_WAIT_TIMEOUT 1

// ---- shared-memory address / PTX wrappers ----------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void* p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Make mbarrier initialisation visible to the async (bulk copy) proxy.
__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(bar)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile(
        "{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(bar),
        "r"(bytes)
        : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Non-blocking test of the phase with the given parity.
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wait for the phase with the given parity to complete, giving up after
// about two seconds of wall time.  Returns false on give-up; `abort_flag`
// (shared memory, may be null) lets another warp cut the wait short.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  const volatile int* abort_flag)
{
    if (mbar_try_wait(bar, parity))
        return true;
    uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity))
            return true;
        if ((it & 63u) == 0) {
            if (abort_flag && *abort_flag)
                return false;
            if (global_timer_ns() - t0 > 2000000000ull)
                return false;
        }
    }
}

// 1-D bulk copy global -> shared (TMA engine), completion counted on `bar`
// in bytes.  dst, src and bytes must be multiples of 16.
__device__ __forceinline__ void bulk_copy_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                              uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

// L2 cache policies for bulk copies: weights are streamed once (evict
// first), activations are reused by every CTA (evict last).
__device__ __forceinline__ uint64_t l2_policy_evict_first()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t l2_policy_evict_last()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// 1-D bulk copy global -> shared with an L2 cache policy.
__device__ __forceinline__ void bulk_copy_g2s_hint(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar,
                                                   uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
            dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(policy)
        : "memory");
}

__device__ __forceinline__ uint32_t lds32(const uint8_t* p)
{
    return *reinterpret_cast<const uint32_t*>(p);
}

__device__ __forceinline__ uint32_t ldg32_nc(const void* p)
{
    uint32_t v;
    asm volatile("ld.global.nc.u32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}

// ---- integer dot products ---------------------------------------------------

// sum of four u8*s8 products + c
__device__ __forceinline__ int dp4a_us(uint32_t a_u8x4, uint32_t b_s8x4, int c)
{
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a_u8x4), "r"(b_s8x4), "r"(c));
    return d;
}

// a.s16[0]*b.u8[0] + a.s16[1]*b.u8[1] + c   (bytes 0,1 of b)
__device__ __forceinline__ int dp2a_lo_su(uint32_t a_s16x2, uint32_t b_u8x4, int c)
{
    int d;
    asm("dp2a.lo.s32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a_s16x2), "r"(b_u8x4), "r"(c));
    return d;
}

// a.s16[0]*b.u8[2] + a.s16[1]*b.u8[3] + c   (bytes 2,3 of b)
__device__ __forceinline__ int dp2a_hi_su(uint32_t a_s16x2, uint32_t b_u8x4, int c)
{
    int d;
    asm("dp2a.hi.s32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a_s16x2), "r"(b_u8x4), "r"(c));
    return d;
}

// Byte j (0..3) of v, a value 0..255, as float: the byte is placed under
// the exponent of 2^23 and 2^23 is subtracted (exact).
template <int J>
__device__ __forceinline__ float byte_as_float(uint32_t v)
{
    constexpr uint32_t sel = J | (4u << 4) | (4u << 8) | (7u << 12);
    return __int_as_float(__byte_perm(v, 0x4B000000u, sel)) - 8388608.0f;
}

__device__ __forceinline__ float half_lo_f(uint32_t v)
{
    return __half2float(__ushort_as_half(static_cast<unsigned short>(v & 0xFFFFu)));
}

__device__ __forceinline__ float half_hi_f(uint32_t v)
{
    return __half2float(__ushort_as_half(static_cast<unsigned short>(v >> 16)));
}

__device__ __forceinline__ float bf16_bits_f(uint16_t b)
{
    return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

// Programmatic dependent launch.  Every kernel of the library is launched as
// a programmatic dependent of the previous kernel in its stream, so its
// launch and setup overlap that kernel's tail.  A kernel lets its own
// dependents be scheduled at entry and calls pdl_wait() before its first
// access to global memory (the previous grid may still be writing it); the
// wait returns at once when the kernel was launched normally.
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, Args&&... args)
{
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

}  // namespace q2k
