// device_common.cuh - sm_103a device helpers shared by the flush kernels:
// mbarrier + cp.async.bulk staging (the Blackwell bulk-copy engine), bounded
// waits, and the library's device error word.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_fp16.h>

#include "vq.h"

namespace vq {

constexpr unsigned FULL_MASK = 0xffffffffu;

// Upper bound on the wall-clock time of one mbarrier wait (nanoseconds of
// %globaltimer).  A copy that has not landed by then never will; the kernel
// records VQ_DEVERR_WAIT_TIMEOUT and returns instead of spinning.
constexpr uint64_t MBAR_TIMEOUT_NS = 2000000000ull;

// One device error word per translation unit; each .cu exposes a host reader.
#define VQ_DEFINE_ERROR_WORD(name) static __device__ unsigned int name = 0u

// Sign-flip mask of one fp16 pair: bit 0 of `two` flips the low half (bit 15),
// bit 1 the high half (bit 31).  Used for the randomised-sign rotation.
__host__ __device__ __forceinline__ uint32_t half2_sign_mask(uint32_t two)
{
    return ((two & 1u) << 15) | ((two & 2u) << 30);
}

// The two sign bits of coordinates c, c + 1 (c even) from sign words s[4].
__host__ __device__ __forceinline__ uint32_t sign_pair(const uint32_t *s, int c)
{
    return (s[c >> 5] >> (c & 31)) & 3u;
}

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

// Make barrier initialisation visible to the async (bulk-copy) proxy.
__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Order this thread's generic-proxy shared-memory accesses before later
// async-proxy accesses (a bulk copy overwriting a buffer that was just read).
__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t globaltimer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Bounded wait for phase `parity` of `bar`.  Returns false if it gave up.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
        if (mbar_try_wait(bar, parity)) return true;
        if (globaltimer_ns() - t0 > MBAR_TIMEOUT_NS) return false;
    }
}

// 1-D bulk copy global -> shared, completion signalled on `bar` (tx bytes).
// Both addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void *dst_smem, const void *src_gmem, uint32_t bytes,
                                         uint64_t *bar, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst_smem)),
        "l"(src_gmem), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// Tiled tensor copies global -> shared (TMA), completion on `bar`.  The
// innermost coordinate times the element size must be a multiple of 16 bytes;
// the box lands in shared memory as the tensor map's layout (and swizzle)
// dictates, out-of-range elements zero-filled, and always counts its full
// size in bytes on the barrier.
__device__ __forceinline__ void tma_load_2d(void *dst_smem, const CUtensorMap *map, int c0, int c1,
                                            uint64_t *bar, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst_smem)),
        "l"(map), "r"(c0), "r"(c1), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void tma_load_3d(void *dst_smem, const CUtensorMap *map, int c0, int c1, int c2,
                                            uint64_t *bar, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_u32(dst_smem)),
        "l"(map), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// Byte offset of 16-byte chunk `c` of 128-byte line `line` in a box written
// with the 128-byte swizzle (buffer aligned to 1024 bytes).
__device__ __forceinline__ uint32_t swz128(int line, int c)
{
    return (uint32_t)(line * 128 + ((c ^ (line & 7)) << 4));
}

// Shared memory base rounded up to 1024 bytes (the 128-byte swizzle pattern is
// taken from address bits 7-9); launches request 1024 extra bytes.
__device__ __forceinline__ unsigned char *smem_1k(unsigned char *p)
{
    const uint32_t a = smem_u32(p);
    return p + (((a + 1023u) & ~1023u) - a);
}

// L2 policy for data read exactly once (streamed input).
__device__ __forceinline__ uint64_t l2_policy_evict_first()
{
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// fp32 sum of an fp16 value and an fp32 value with one rounding (the fp16
// operand is read directly, without a separate conversion).
__device__ __forceinline__ float add_f16_f32(__half a, float c)
{
    float r;
    asm("add.rn.f32.f16 %0, %1, %2;" : "=f"(r) : "h"(__half_as_ushort(a)), "f"(c));
    return r;
}

// Error-free transformations (Knuth TwoSum, Dekker Fast2Sum) for the
// extended-precision recompute paths.
__device__ __forceinline__ void two_sum(float a, float b, float &s, float &e)
{
    s = __fadd_rn(a, b);
    float bb = __fsub_rn(s, a);
    e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}

__device__ __forceinline__ void fast_two_sum(float a, float b, float &s, float &e)
{
    s = __fadd_rn(a, b);
    e = __fsub_rn(b, __fsub_rn(s, a));
}

}  // namespace vq
