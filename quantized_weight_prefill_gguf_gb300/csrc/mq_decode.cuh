// mq_decode.cuh -- per-element decode arithmetic of the three GGUF block
// formats, shared by the standalone decoders (the f16 cache is built with
// them) and by the fused GEMM's on-chip decoder, so both paths produce the
// same f16 bits ("05 · 8p — Persistent f16 weight cache + fused
// dequant-in-GEMM", section 3.3 Pitfalls: the same rounding path).
//
// Exactness, which lets the kernels use FMA and 8-at-a-time packing:
//  * d, dmin are f16 (11 significant bits), Q4_K scales/mins 6 bits, nibbles
//    4 bits: A = d*sc (<= 17 bits), A*q (<= 21 bits) and B = dmin*m (<= 17
//    bits) are exact in f32.  fmaf(A, q, -B) therefore equals
//    RN32(RN32(A*q) - B): one f32 rounding, at the subtraction, as in the
//    block definition d*sc*q - dmin*m.
//  * Q6_K: |sc*q6| <= 128*32 = 4096, so d*sc*q6 has <= 23 significant bits
//    and (d*sc)*q6 is exact in f32.  Q8_0: d*q <= 18 bits, exact.
//  * The only remaining rounding is f32 -> f16, round to nearest even
//    (cvt.rn.f16x2.f32), which keeps subnormals and signed zeros.  For Q8_0,
//    where d*q is exact, that single rounding is done by an f16 multiply.
#pragma once

#include <cstdint>
#include <cuda_fp16.h>

namespace mq {

// Integer 0..2^23-1 held in the low bits of `v` -> exact f32, without I2F:
// 0x4B000000 is 2^23, so the bit pattern 0x4B000000|v is 2^23 + v.
__device__ __forceinline__ float small_uint_to_f32(uint32_t v)
{
    return __int_as_float(0x4B000000u | v) - 8388608.0f;
}

__device__ __forceinline__ float f16_bits_to_f32(uint32_t bits16)
{
    return __half2float(__ushort_as_half(static_cast<unsigned short>(bits16 & 0xFFFFu)));
}

// Q4_K 6-bit scale and min of sub-block s from the 12 packed bytes, given as
// three little-endian words s0 = bytes 0..3, s1 = 4..7, s2 = 8..11:
//   s < 4 : sc = byte[s] & 63,                    m = byte[s+4] & 63
//   s >= 4: sc = (byte[s+4] & 15) | (byte[s-4] >> 6) << 4
//           m  = (byte[s+4] >> 4) | (byte[s]   >> 6) << 4
__device__ __forceinline__ void q4k_scale_min(uint32_t s0, uint32_t s1, uint32_t s2, int s, int &sc, int &m)
{
    if (s < 4) {
        sc = (s0 >> (8 * s)) & 63;
        m = (s1 >> (8 * s)) & 63;
    } else {
        const int j = s - 4;
        const uint32_t b8 = (s2 >> (8 * j)) & 0xFF;
        sc = (b8 & 15) | (((s0 >> (8 * j + 6)) & 3) << 4);
        m = (b8 >> 4) | (((s1 >> (8 * j + 6)) & 3) << 4);
    }
}

// ---- packed helpers.  Two f32 lanes travel in one 64-bit register so the
// sm_100-family paired instructions (add/mul/fma .rn.f32x2) do two elements
// per instruction; each lane rounds exactly like its scalar form.

__device__ __forceinline__ uint64_t f32x2(float lo, float hi)
{
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}

// Bytes j and j+1 of v (each 0..255) -> two f32 values 2^23 + byte: the byte
// permute places the byte under exponent byte 0x4B (0x4B0000bb).
__device__ __forceinline__ uint64_t magic_pair(uint32_t v, int j)
{
    const uint32_t a = __byte_perm(v, 0x4B000000u, 0x7540u | j);
    const uint32_t b = __byte_perm(v, 0x4B000000u, 0x7540u | (j + 1));
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(a), "r"(b));
    return r;
}

__device__ __forceinline__ uint64_t add_f32x2(uint64_t a, uint64_t b)
{
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

__device__ __forceinline__ uint64_t mul_f32x2(uint64_t a, uint64_t b)
{
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

__device__ __forceinline__ uint64_t fma_f32x2(uint64_t a, uint64_t b, uint64_t c)
{
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

__device__ __forceinline__ void unpack_f32x2(uint64_t v, float &lo, float &hi)
{
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}

// Two f32 lanes -> f16x2 (lane 0 in the low half), round to nearest even.
__device__ __forceinline__ uint32_t cvt_f16x2(uint64_t v)
{
    float lo, hi;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// Eight outputs y_j = RN16(RN32(a * c_j - b)) where c_j is byte j of (v0, v1)
// (bytes 0..3 of v0 first), given a2 = {a, a} and nb2 = {-b, -b}: the byte
// permute puts c_j under the exponent of 2^23, 2^23 is subtracted exactly,
// then one packed FMA and one packed f32 -> f16 conversion per two outputs.
// Exact whenever a * c_j is exact in f32.
__device__ __forceinline__ uint4 fma_bytes_eight(uint64_t a2, uint64_t nb2, uint32_t v0, uint32_t v1)
{
    const uint64_t m2 = f32x2(-8388608.0f, -8388608.0f);
    return make_uint4(cvt_f16x2(fma_f32x2(a2, add_f32x2(magic_pair(v0, 0), m2), nb2)),
                      cvt_f16x2(fma_f32x2(a2, add_f32x2(magic_pair(v0, 2), m2), nb2)),
                      cvt_f16x2(fma_f32x2(a2, add_f32x2(magic_pair(v1, 0), m2), nb2)),
                      cvt_f16x2(fma_f32x2(a2, add_f32x2(magic_pair(v1, 2), m2), nb2)));
}

// Eight Q4_K outputs of one sub-block: nibbles taken from the 8 bytes held in
// w0 (bytes 0..3) and w1 (bytes 4..7), low nibbles if sh == 0, high if 4.
// A = d*sc, B = dmin*m.  Output element j comes from byte j.
// q = (2^23 + q) - 2^23 exactly, then y = RN16(fma(A, q, -B)).
__device__ __forceinline__ uint4 q4k_eight(float A, float B, uint32_t w0, uint32_t w1, int sh)
{
    const uint32_t v0 = (w0 >> sh) & 0x0F0F0F0Fu, v1 = (w1 >> sh) & 0x0F0F0F0Fu;
    const uint64_t a2 = f32x2(A, A), nb2 = f32x2(-B, -B), m2 = f32x2(-8388608.0f, -8388608.0f);
    return make_uint4(cvt_f16x2(fma_f32x2(a2, add_f32x2(magic_pair(v0, 0), m2), nb2)),
                      cvt_f16x2(fma_f32x2(a2, add_f32x2(magic_pair(v0, 2), m2), nb2)),
                      cvt_f16x2(fma_f32x2(a2, add_f32x2(magic_pair(v1, 0), m2), nb2)),
                      cvt_f16x2(fma_f32x2(a2, add_f32x2(magic_pair(v1, 2), m2), nb2)));
}

// Core of the Q6_K decode: v0, v1 hold the eight unsigned 6-bit values
// (value + 32 of the block definition) one per byte.
__device__ __forceinline__ uint4 q6k_core(float A, uint32_t v0, uint32_t v1)
{
    const uint64_t a2 = f32x2(A, A), m2 = f32x2(-8388640.0f, -8388640.0f);   // -(2^23 + 32)
    return make_uint4(cvt_f16x2(mul_f32x2(a2, add_f32x2(magic_pair(v0, 0), m2))),
                      cvt_f16x2(mul_f32x2(a2, add_f32x2(magic_pair(v0, 2), m2))),
                      cvt_f16x2(mul_f32x2(a2, add_f32x2(magic_pair(v1, 0), m2))),
                      cvt_f16x2(mul_f32x2(a2, add_f32x2(magic_pair(v1, 2), m2))));
}

// Eight Q6_K outputs: low 4 bits from the nibbles of ql bytes (l0 = bytes
// 0..3, l1 = 4..7; shift lsh 0 or 4), high 2 bits from bits hsh..hsh+1 of
// qh bytes (h0, h1).  q6 = value - 32, y = RN16(A * q6) with A = d*sc.
__device__ __forceinline__ uint4 q6k_eight(float A, uint32_t l0, uint32_t l1, int lsh, uint32_t h0, uint32_t h1,
                                           int hsh)
{
    const uint32_t v0 = ((l0 >> lsh) & 0x0F0F0F0Fu) | (((h0 >> hsh) & 0x03030303u) << 4);
    const uint32_t v1 = ((l1 >> lsh) & 0x0F0F0F0Fu) | (((h1 >> hsh) & 0x03030303u) << 4);
    return q6k_core(A, v0, v1);
}

// The 6-bit values of q6k_eight with shift amounts that vary per thread:
// lsh = 0 or 4 as there; hrot = (hsh + 28) & 31 rotates bits hsh, hsh+1 of
// every qh byte onto bits 4, 5 of the same byte (a rotation by 28 is a left
// shift by 4; bits that wrap around land outside the 0x30 mask).
__device__ __forceinline__ uint32_t q6k_bytes(uint32_t l, int lsh, uint32_t h, int hrot)
{
    return ((l >> lsh) & 0x0F0F0F0Fu) | (__funnelshift_r(h, h, hrot) & 0x30303030u);
}

// Eight Q8_0 outputs from 8 int8 quants (w0 bytes 0..3, w1 bytes 4..7) and
// the block's f16 scale bits d16.  d*q is exact in f32, so RN16(RN32(d*q))
// is RN16(d*q), which the f16x2 multiply computes directly: bytes q+128 are
// placed under the f16 exponent of 1024 (0x64nn = 1024 + nn), 1152 is
// subtracted exactly, and the f16 product with d rounds once.
__device__ __forceinline__ uint32_t q80_pair(uint32_t v, int j, uint32_t d2)
{
    const uint32_t h = __byte_perm(v, 0x64646464u, 0x5040u | j | ((j + 1) << 8));
    uint32_t q, y;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(q) : "r"(h), "r"(0x64806480u));   // 1152 = 0x6480
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(y) : "r"(q), "r"(d2));
    return y;
}

__device__ __forceinline__ uint4 q80_eight(uint32_t d16, uint32_t w0, uint32_t w1)
{
    const uint32_t d2 = (d16 & 0xFFFFu) * 0x10001u;
    const uint32_t v0 = w0 ^ 0x80808080u, v1 = w1 ^ 0x80808080u;
    return make_uint4(q80_pair(v0, 0, d2), q80_pair(v0, 2, d2), q80_pair(v1, 0, d2), q80_pair(v1, 2, d2));
}

// Eight outputs y_j = RN16(d * (c_j - bias)) from bytes c_j of (v0, v1)
// (bytes 0..3 of v0 first): the byte permute puts c_j under the f16
// exponent of 1024 (0x64nn = 1024 + nn), subtracting 1024 + bias (given as
// f16x2 bits in bias2) is exact, and one f16 multiply by d rounds once.
// d * (c_j - bias) is exact in f32 whenever |c_j - bias| < 2^13 (d has 11
// significant bits), so this equals RN16(RN32(d * q)).
__device__ __forceinline__ uint32_t f16_bias_pair(uint32_t v, int j, uint32_t bias2, uint32_t d2)
{
    const uint32_t h = __byte_perm(v, 0x64646464u, 0x5040u | j | ((j + 1) << 8));
    uint32_t q, y;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(q) : "r"(h), "r"(bias2));
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(y) : "r"(q), "r"(d2));
    return y;
}

__device__ __forceinline__ uint4 f16_bias_eight(uint32_t d16, uint32_t v0, uint32_t v1, uint32_t bias2)
{
    const uint32_t d2 = (d16 & 0xFFFFu) * 0x10001u;
    return make_uint4(f16_bias_pair(v0, 0, bias2, d2), f16_bias_pair(v0, 2, bias2, d2),
                      f16_bias_pair(v1, 0, bias2, d2), f16_bias_pair(v1, 2, bias2, d2));
}

// Bits 0..3 of x spread to bit 4 of bytes 0..3 (0x10 per set bit): the
// multiply moves bit i to bit 8i, the mask keeps those, the shift lifts
// them to bit 4.  Used for Q5_0 / Q5_1's qh bit plane (the fifth bit of
// four consecutive elements).
__device__ __forceinline__ uint32_t spread4_bit4(uint32_t x)
{
    return (((x & 0xFu) * 0x00204081u) & 0x01010101u) << 4;
}

}  // namespace mq
