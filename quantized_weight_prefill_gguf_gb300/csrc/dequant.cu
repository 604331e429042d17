// dequant.cu -- standalone sm_103a block decoders Q4_K / Q6_K / Q8_0 -> f16.
//
// The f16 cache is filled by these kernels once, at registration ("05 · 8p —
// Persistent f16 weight cache + fused dequant-in-GEMM", section 3.1: decode
// at load, keep the f16 copy resident).  The work is a streaming pass: read
// each block once, write 2 bytes per element once, so HBM bandwidth bounds
// it (algorithmic bytes per element: 0.5625+2, 0.8203+2, 1.0625+2).
//
// Data movement.  Q6_K (210 B) and Q8_0 (34 B) blocks are only 2-byte
// aligned, so a wide load at a block-relative offset can be misaligned (the
// page's Q5_0 crash, "05 · 8p", section 2: alignment is stride*g + offset mod
// width).  Here a CTA never loads at block-relative offsets: it copies a
// span of G whole blocks, which starts on a 16-byte boundary because
// G*bytes is a multiple of 16, with 16-byte vector loads into shared memory,
// and decodes from there with 2-byte shared loads.  The last partial span
// stops its vector loads at the stream's end and finishes with byte loads,
// so nothing past the stream is read.
//
// Output: element (n,k) of the flat stream (flat index n*K+k) goes to
// out[n*ldo + k], eight elements (16 bytes) per store.  K % 8 == 0 keeps a
// group of eight inside one row.
#include <cstdint>
#include <cuda_runtime.h>

#include "mq_decode.cuh"
#include "mq_internal.h"
#include "mq_ptx.cuh"

namespace mq {
namespace {

template <int T> struct Fmt;
template <> struct Fmt<8> { static constexpr int QK = 32, BB = 34, G = 256; };    // span 8704 B
template <> struct Fmt<12> { static constexpr int QK = 256, BB = 144, G = 64; };  // span 9216 B
template <> struct Fmt<14> { static constexpr int QK = 256, BB = 210, G = 64; };  // span 13440 B

constexpr int kThreads = 256;

__device__ __forceinline__ uint32_t lds_u16(const uint8_t *p)
{
    return *reinterpret_cast<const uint16_t *>(p);
}

// Little-endian 32-bit word from two 2-byte-aligned shared loads.
__device__ __forceinline__ uint32_t lds_u32_a2(const uint8_t *p)
{
    return lds_u16(p) | (lds_u16(p + 2) << 16);
}

__device__ __forceinline__ void store8(__half *out, int64_t flat, int64_t K, int64_t ldo, uint4 v)
{
    __half *dst;
    if (ldo == K) {
        dst = out + flat;
    } else {
        const int64_t n = flat / K;
        dst = out + n * ldo + (flat - n * K);
    }
    stg_v4(dst, v);
}

template <int T>
__global__ void __launch_bounds__(kThreads) k_dequant(const uint8_t *__restrict__ q, int64_t nblocks,
                                                      __half *__restrict__ out, int64_t K, int64_t ldo)
{
    using F = Fmt<T>;
    __shared__ __align__(16) uint8_t sm[F::G * F::BB];

    const int64_t b0 = static_cast<int64_t>(blockIdx.x) * F::G;
    const int nb = static_cast<int>(nblocks - b0 < F::G ? nblocks - b0 : F::G);
    const uint8_t *src = q + b0 * F::BB;
    const int bytes = nb * F::BB;
    const int n16 = bytes >> 4;
    for (int i = threadIdx.x; i < n16; i += kThreads)
        *reinterpret_cast<uint4 *>(sm + 16 * i) = ldg_nc_v4(src + 16 * i);
    for (int i = (n16 << 4) + threadIdx.x; i < bytes; i += kThreads)
        sm[i] = src[i];
    __syncthreads();

    if constexpr (T == 12) {
        // 16 items per block: qs bytes [32p+i0, 32p+i0+8) feed elements
        // 64p+i0.. (low nibbles, sub-block 2p) and 64p+32+i0.. (high, 2p+1).
        for (int it = threadIdx.x; it < nb * 16; it += kThreads) {
            const int blk = it >> 4, sub = it & 15;
            const int p = sub >> 2, i0 = (sub & 3) * 8;
            const uint8_t *b = sm + blk * F::BB;          // 16-byte aligned
            const uint32_t h = *reinterpret_cast<const uint32_t *>(b);
            const float d = f16_bits_to_f32(h), dmin = f16_bits_to_f32(h >> 16);
            const uint32_t s0 = *reinterpret_cast<const uint32_t *>(b + 4);
            const uint32_t s1 = *reinterpret_cast<const uint32_t *>(b + 8);
            const uint32_t s2 = *reinterpret_cast<const uint32_t *>(b + 12);
            const uint2 qw = *reinterpret_cast<const uint2 *>(b + 16 + 32 * p + i0);
            int sc, m;
            q4k_scale_min(s0, s1, s2, 2 * p, sc, m);
            const uint4 lo = q4k_eight(__fmul_rn(d, (float)sc), __fmul_rn(dmin, (float)m), qw.x, qw.y, 0);
            q4k_scale_min(s0, s1, s2, 2 * p + 1, sc, m);
            const uint4 hi = q4k_eight(__fmul_rn(d, (float)sc), __fmul_rn(dmin, (float)m), qw.x, qw.y, 4);
            const int64_t f = (b0 + blk) * F::QK + 64 * p + i0;
            store8(out, f, K, ldo, lo);
            store8(out, f + 32, K, ldo, hi);
        }
    } else if constexpr (T == 14) {
        // 8 items per block: half h, l0 in {0,8,16,24}: ql bytes 64h+l0..
        // and 64h+32+l0.., qh bytes 32h+l0.. feed the four quarters t of the
        // half, elements 128h + 32t + l0 .. +8 with scale sc[8h + 2t + l0/16].
        for (int it = threadIdx.x; it < nb * 8; it += kThreads) {
            const int blk = it >> 3, sub = it & 7;
            const int hh = sub >> 2, l0 = (sub & 3) * 8;
            const uint8_t *b = sm + blk * F::BB;          // 2-byte aligned
            const uint8_t *ql = b + 64 * hh + l0;
            const uint8_t *qh = b + 128 + 32 * hh + l0;
            const uint32_t la0 = lds_u32_a2(ql), la1 = lds_u32_a2(ql + 4);
            const uint32_t lb0 = lds_u32_a2(ql + 32), lb1 = lds_u32_a2(ql + 36);
            const uint32_t h0 = lds_u32_a2(qh), h1 = lds_u32_a2(qh + 4);
            const float d = f16_bits_to_f32(lds_u16(b + 208));
            const int8_t *sc = reinterpret_cast<const int8_t *>(b + 192 + 8 * hh + (l0 >> 4));
            const int64_t f = (b0 + blk) * F::QK + 128 * hh + l0;
            store8(out, f, K, ldo, q6k_eight(__fmul_rn(d, (float)sc[0]), la0, la1, 0, h0, h1, 0));
            store8(out, f + 32, K, ldo, q6k_eight(__fmul_rn(d, (float)sc[2]), lb0, lb1, 0, h0, h1, 2));
            store8(out, f + 64, K, ldo, q6k_eight(__fmul_rn(d, (float)sc[4]), la0, la1, 4, h0, h1, 4));
            store8(out, f + 96, K, ldo, q6k_eight(__fmul_rn(d, (float)sc[6]), lb0, lb1, 4, h0, h1, 6));
        }
    } else {
        // 4 items per block: quants 8c..8c+7.
        for (int it = threadIdx.x; it < nb * 4; it += kThreads) {
            const int blk = it >> 2, c = it & 3;
            const uint8_t *b = sm + blk * F::BB;          // 2-byte aligned
            const uint32_t d16 = lds_u16(b);
            const uint32_t w0 = lds_u32_a2(b + 2 + 8 * c), w1 = lds_u32_a2(b + 6 + 8 * c);
            store8(out, (b0 + blk) * F::QK + 8 * c, K, ldo, q80_eight(d16, w0, w1));
        }
    }
}

template <int T>
cudaError_t launch_t(const void *q, int64_t nblocks, __half *out, int64_t K, int64_t ldo, cudaStream_t s)
{
    const int64_t grid = (nblocks + Fmt<T>::G - 1) / Fmt<T>::G;
    if (grid > 0x7FFFFFFF)
        return cudaErrorInvalidValue;
    k_dequant<T><<<static_cast<unsigned>(grid), kThreads, 0, s>>>(static_cast<const uint8_t *>(q), nblocks, out,
                                                                  K, ldo);
    note_launch();
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_dequant(int type, const void *q, int64_t nblocks, __half *out, int64_t K, int64_t ldo,
                           cudaStream_t s)
{
    if (nblocks <= 0)
        return cudaSuccess;
    switch (type) {
    case 8: return launch_t<8>(q, nblocks, out, K, ldo, s);
    case 12: return launch_t<12>(q, nblocks, out, K, ldo, s);
    case 14: return launch_t<14>(q, nblocks, out, K, ldo, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace mq
