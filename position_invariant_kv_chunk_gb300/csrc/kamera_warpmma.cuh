// kamera_warpmma.cuh -- helpers shared by the attention kernels (sm_103a):
// 8x8 matrix loads from shared memory, the m16n8k16 bf16 MMA with fp32
// accumulation, bf16 hi + lo splits of fp32 values (about 16 significant bits
// as a pair), and the time-bounded wait on a tile buffer's mbarrier.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>

#include "kamera_common.cuh"
#include "kamera_ptx.cuh"

namespace kamera {
namespace wmma16 {

__device__ __forceinline__ void ldsm_x4(uint32_t a, uint32_t (&r)[4])
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(a)
                 : "memory");
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t a, uint32_t (&r)[4])
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(a)
                 : "memory");
}
__device__ __forceinline__ void ldsm_x2(uint32_t a, uint32_t (&r)[2])
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0, %1}, [%2];"
                 : "=r"(r[0]), "=r"(r[1])
                 : "r"(a)
                 : "memory");
}
__device__ __forceinline__ void ldsm_x2_t(uint32_t a, uint32_t (&r)[2])
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0, %1}, [%2];"
                 : "=r"(r[0]), "=r"(r[1])
                 : "r"(a)
                 : "memory");
}
// D += A B: A 16x16 (row-major fragments), B 16x8 (column fragments), fp32 D.
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1)
{
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// (x, y) as bf16 pairs hi and lo with hi + lo = (x, y) to about 2^-16 relative.
__device__ __forceinline__ void split_hl(float x, float y, uint32_t& hi, uint32_t& lo)
{
    hi = pack_bf16x2(x, y);
    lo = pack_bf16x2(x - bf16lo(hi), y - bf16hi(hi));
}
__device__ __forceinline__ void split1(float v, __nv_bfloat16& hi, __nv_bfloat16& lo)
{
    hi = __float2bfloat16_rn(v);
    lo = __float2bfloat16_rn(v - __bfloat162float(hi));
}

// Bounded wait on an mbarrier phase.  On expiry the call reports
// KAMERA_DEVERR_TIMEOUT, every later wait of the CTA returns at once (the abort
// flag), and the kernel runs its barriers to the end (its output is then
// undefined).
__device__ __forceinline__ bool tile_wait(uint32_t bar, uint32_t parity, volatile int32_t* abort, int32_t* err,
                                          uint64_t limit)
{
    if (ptx::mbar_try_wait(bar, parity))
        return true;
    const uint64_t t0 = ptx::globaltimer();
    for (uint32_t it = 1;; ++it) {
        if (ptx::mbar_try_wait(bar, parity))
            return true;
        if ((it & 63u) == 0) {
            if (*abort)
                return false;
            if (ptx::globaltimer() - t0 > limit) {
                *abort = 1;
                raise_err(err, KAMERA_DEVERR_TIMEOUT);
                return false;
            }
        }
    }
}

}  // namespace wmma16
}  // namespace kamera
