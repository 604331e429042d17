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
//    (cvt.rn.f16x2.f32), which keeps subnormals and signed zeros.
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

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi)
{
    __half2 h = __floats2half2_rn(lo, hi);   // .x (low 16 bits) = lo
    return *reinterpret_cast<uint32_t *>(&h);
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

// Eight Q4_K outputs of one sub-block: nibbles taken from the 8 bytes held in
// w0 (bytes 0..3) and w1 (bytes 4..7), low nibbles if sh == 0, high if 4.
// A = d*sc, B = dmin*m.  Output element j comes from byte j.
__device__ __forceinline__ uint4 q4k_eight(float A, float B, uint32_t w0, uint32_t w1, int sh)
{
    float v[8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        v[j] = fmaf(A, small_uint_to_f32((w0 >> (8 * j + sh)) & 15u), -B);
        v[4 + j] = fmaf(A, small_uint_to_f32((w1 >> (8 * j + sh)) & 15u), -B);
    }
    return make_uint4(pack_f16x2(v[0], v[1]), pack_f16x2(v[2], v[3]), pack_f16x2(v[4], v[5]),
                      pack_f16x2(v[6], v[7]));
}

// Eight Q6_K outputs: low 4 bits from the nibbles of ql bytes (l0 = bytes
// 0..3, l1 = 4..7; shift lsh 0 or 4), high 2 bits from bits hsh..hsh+1 of
// qh bytes (h0, h1).  q6 = value - 32, y = RN16(A * q6) with A = d*sc.
__device__ __forceinline__ uint4 q6k_eight(float A, uint32_t l0, uint32_t l1, int lsh, uint32_t h0, uint32_t h1,
                                           int hsh)
{
    float v[8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint32_t a = ((l0 >> (8 * j + lsh)) & 15u) | (((h0 >> (8 * j + hsh)) & 3u) << 4);
        const uint32_t b = ((l1 >> (8 * j + lsh)) & 15u) | (((h1 >> (8 * j + hsh)) & 3u) << 4);
        v[j] = __fmul_rn(A, small_uint_to_f32(a) - 32.0f);
        v[4 + j] = __fmul_rn(A, small_uint_to_f32(b) - 32.0f);
    }
    return make_uint4(pack_f16x2(v[0], v[1]), pack_f16x2(v[2], v[3]), pack_f16x2(v[4], v[5]),
                      pack_f16x2(v[6], v[7]));
}

// Eight Q8_0 outputs from 8 int8 quants (w0 bytes 0..3, w1 bytes 4..7).
// y = RN16(d * q).  (q ^ 0x80) is q + 128 as an unsigned byte.
__device__ __forceinline__ uint4 q80_eight(float d, uint32_t w0, uint32_t w1)
{
    float v[8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        v[j] = __fmul_rn(d, small_uint_to_f32(((w0 >> (8 * j)) & 0xFFu) ^ 0x80u) - 128.0f);
        v[4 + j] = __fmul_rn(d, small_uint_to_f32(((w1 >> (8 * j)) & 0xFFu) ^ 0x80u) - 128.0f);
    }
    return make_uint4(pack_f16x2(v[0], v[1]), pack_f16x2(v[2], v[3]), pack_f16x2(v[4], v[5]),
                      pack_f16x2(v[6], v[7]));
}

}  // namespace mq
