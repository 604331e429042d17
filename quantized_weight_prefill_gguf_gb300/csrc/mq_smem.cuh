// mq_smem.cuh -- shared-memory readers for block bytes at their real
// (2-byte-aligned) offsets: blocks of 210 (Q6_K) or 34 (Q8_0) bytes are only
// 2-byte aligned, so wider fields are assembled from aligned words.
#pragma once

#include <cstdint>

namespace mq {

__device__ __forceinline__ uint32_t lds_u32(uint32_t saddr)
{
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(saddr));
    return v;
}

__device__ __forceinline__ uint32_t lds_u16(uint32_t saddr)
{
    unsigned short v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(saddr));
    return v;
}

__device__ __forceinline__ int lds_s8(uint32_t saddr)
{
    short v;
    asm volatile("ld.shared.s8 %0, [%1];" : "=h"(v) : "r"(saddr));
    return v;
}

// 32 bytes starting at a 2-byte-aligned shared address, as 8 little-endian
// words: nine aligned word loads and a funnel shift by 0 or 16 bits.
__device__ __forceinline__ void lds_32B_a2(uint32_t saddr, uint32_t (&w)[8])
{
    const uint32_t base = saddr & ~3u;
    const uint32_t sh = (saddr & 3u) * 8u;
    uint32_t t[9];
#pragma unroll
    for (int i = 0; i < 9; ++i)
        t[i] = lds_u32(base + 4 * i);
#pragma unroll
    for (int i = 0; i < 8; ++i)
        w[i] = __funnelshift_r(t[i], t[i + 1], sh);
}

// 16 bytes starting at a 2-byte-aligned shared address, as 4 words.
__device__ __forceinline__ void lds_16B_a2(uint32_t saddr, uint32_t (&w)[4])
{
    const uint32_t base = saddr & ~3u;
    const uint32_t sh = (saddr & 3u) * 8u;
    uint32_t t[5];
#pragma unroll
    for (int i = 0; i < 5; ++i)
        t[i] = lds_u32(base + 4 * i);
#pragma unroll
    for (int i = 0; i < 4; ++i)
        w[i] = __funnelshift_r(t[i], t[i + 1], sh);
}

}  // namespace mq
