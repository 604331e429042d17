// dequant.cu -- standalone sm_103a decoders -> f16: the block formats Q4_0,
// Q5_0, Q5_1, Q8_0, Q4_K, Q5_K, Q6_K, and the float weights F32 / F16 / BF16
// (a conversion; the f16 copy then carries the row padding below).
//
// The f16 cache is filled by these kernels once, at registration ("05 · 8p —
// Persistent f16 weight cache + fused dequant-in-GEMM", section 3.1: decode
// at load, keep the f16 copy resident).  The work is a streaming pass: read
// each block once, write 2 bytes per element once, so HBM bandwidth bounds
// it (algorithmic bytes per element: block bytes / block length + 2, e.g.
// Q4_K 0.5625+2, Q6_K 0.8203+2, Q8_0 1.0625+2; F32 4+2, F16 and BF16 2+2).
//
// Float weights ("ggml-cuda: GEMM weight row padding + one-time K-padded f16
// dequant for prefill", Summary: pad a float weight's rows by one 128-byte
// line when its row size is a multiple of 2048 bytes, so consecutive rows do
// not collide in the same cache sets) are converted into the same K-padded
// f16 layout the block formats decode into.
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
// Work split.  A CTA owns a span of G whole blocks.  Each warp decodes
// kPasses groups of blocks; in a group the 32 lanes cover whole blocks and
// every lane produces 16 elements from one scale computation, written as two
// 16-byte stores.  The lanes are paired so that the two lanes of a pair
// write the two halves of one 32-byte sector in the same store instruction:
// a store instruction of the warp writes 16 complete sectors.
//
// Output: element (n,k) of the flat stream (flat index n*K+k) goes to
// out[n*ldo + k].  Three addressing cases, uniform per launch: ldo == K (the
// flat index is the address); K a multiple of the block length (a block lies
// in one row, its row comes from one multiply-high division per block); any
// other K (K % 8 == 0 keeps a group of eight inside one row; one division
// per group of eight).
#include <cstdint>
#include <cuda_runtime.h>

#include "mq_decode.cuh"
#include "mq_internal.h"
#include "mq_launch.cuh"
#include "mq_ptx.cuh"

namespace mq {
namespace {

template <int T> struct Fmt;
// QK elements per block, BB bytes per block, BPG blocks per lane group, G
// blocks per CTA span (G * BB is a multiple of 16).
template <> struct Fmt<2> { static constexpr int QK = 32, BB = 18, BPG = 16, G = 256; };    // Q4_0, span 4608 B
template <> struct Fmt<6> { static constexpr int QK = 32, BB = 22, BPG = 16, G = 256; };    // Q5_0, span 5632 B
template <> struct Fmt<7> { static constexpr int QK = 32, BB = 24, BPG = 16, G = 256; };    // Q5_1, span 6144 B
template <> struct Fmt<8> { static constexpr int QK = 32, BB = 34, BPG = 16, G = 256; };    // Q8_0, span 8704 B
template <> struct Fmt<12> { static constexpr int QK = 256, BB = 144, BPG = 2, G = 32; };   // Q4_K, span 4608 B
template <> struct Fmt<13> { static constexpr int QK = 256, BB = 176, BPG = 2, G = 32; };   // Q5_K, span 5632 B
template <> struct Fmt<14> { static constexpr int QK = 256, BB = 210, BPG = 2, G = 32; };   // Q6_K, span 6720 B

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

// Row/column of a block index: q = x / d by multiply-high with
// m = floor((2^32 - 1) / d), which undershoots the quotient by at most 2 for
// x < 2^32, then at most two corrections.
struct BlockRows {
    uint32_t bpr, m;
};

__device__ __forceinline__ void block_row(uint32_t x, BlockRows br, uint32_t &q, uint32_t &r)
{
    q = __umulhi(x, br.m);
    r = x - q * br.bpr;
    if (r >= br.bpr) { ++q; r -= br.bpr; }
    if (r >= br.bpr) { ++q; r -= br.bpr; }
}

// Eight consecutive bytes of the staged span at a 2-byte-aligned offset, as
// two little-endian words: three aligned word loads and a funnel shift.
// May read up to 4 bytes past the eight (the span buffer is padded).
__device__ __forceinline__ uint2 lds8_a2(const uint8_t *sm, int off)
{
    const uint32_t *w = reinterpret_cast<const uint32_t *>(sm) + (off >> 2);
    const uint32_t sh = static_cast<uint32_t>(off & 2) * 8u;
    const uint32_t t0 = w[0], t1 = w[1], t2 = w[2];
    return make_uint2(__funnelshift_r(t0, t1, sh), __funnelshift_r(t1, t2, sh));
}

__device__ __forceinline__ uint32_t lds_u16(const uint8_t *sm, int off)
{
    return *reinterpret_cast<const uint16_t *>(sm + off);
}

// Destination of element e of block bi.  mode 0: ldo == K; mode 1: K is a
// multiple of QK; mode 2: general (e and e+7 in the same row).
template <int QK>
__device__ __forceinline__ __half *dest(__half *out, uint32_t bi, int e, int mode, int64_t K, int64_t ldo,
                                        BlockRows br)
{
    if (mode == 0)
        return out + static_cast<int64_t>(bi) * QK + e;
    if (mode == 1) {
        uint32_t n, c;
        block_row(bi, br, n, c);
        return out + static_cast<int64_t>(n) * ldo + static_cast<int64_t>(c) * QK + e;
    }
    const int64_t f = static_cast<int64_t>(bi) * QK + e;
    const int64_t n = f / K;
    return out + n * ldo + (f - n * K);
}

template <int T>
__global__ void __launch_bounds__(kThreads) k_dequant(const uint8_t *__restrict__ q, int64_t nblocks,
                                                      __half *__restrict__ out, int64_t K, int64_t ldo, int mode,
                                                      BlockRows br)
{
    using F = Fmt<T>;
    constexpr int kPasses = F::G / (kWarps * F::BPG);
    __shared__ __align__(16) uint8_t sm[F::G * F::BB + 16];

    const int64_t b0 = static_cast<int64_t>(blockIdx.x) * F::G;
    const int nb = static_cast<int>(nblocks - b0 < F::G ? nblocks - b0 : F::G);
    const uint8_t *src = q + b0 * F::BB;
    const int bytes = nb * F::BB;
    const int n16 = bytes >> 4;
    for (int i = threadIdx.x; i < n16; i += kThreads)
        *reinterpret_cast<uint4 *>(sm + 16 * i) = ldg_nc_v4(src + 16 * i);
    for (int i = (n16 << 4) + threadIdx.x; i < bytes; i += kThreads)
        sm[i] = src[i];
    grid_dep_launch();
    grid_dep_wait();   // the output may be read by the previous kernel on the stream
    __syncthreads();

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if constexpr (T == 12 || T == 13) {
        // Lane pair (2j, 2j+1) of a 16-lane half owns sub-block s = j of one
        // block: 32 elements with one (scale, min); lane h = 0/1 of the pair
        // takes elements 32s + 8h + {0..7} and 32s + 16 + 8h + {0..7}, whose
        // nibbles sit in qs bytes 32(s/2) + 8h and +16 (low nibbles for even
        // s, high for odd).
        const int l = lane & 15, sub = l >> 1, h = l & 1;
        const int nsh = (sub & 1) * 4;
        const int bsel = (sub & 3) * 8;                 // byte j = s mod 4 of the scale words
        const bool upper = sub >= 4;
        // Q5_K: qs starts at byte 48 and the fifth bit of position i of
        // sub-block s is bit s of qh[i] (qh at byte 16), rotated onto bit 4.
        const int qoff = (T == 12 ? 16 : 48) + 32 * (sub >> 1) + 8 * h;
        const int qhoff = 16 + 8 * h;
        const int hrot = (sub + 28) & 31;
        const int eoff = 32 * sub + 8 * h;
#pragma unroll
        for (int ps = 0; ps < kPasses; ++ps) {
            const int blk = (warp * kPasses + ps) * F::BPG + (lane >> 4);
            if (blk < nb) {
                const uint8_t *b = sm + blk * F::BB;    // 16-byte aligned
                const uint4 hd = *reinterpret_cast<const uint4 *>(b);
                const uint2 w0 = *reinterpret_cast<const uint2 *>(b + qoff);
                const uint2 w1 = *reinterpret_cast<const uint2 *>(b + qoff + 16);
                // 6-bit scale and min of sub-block s from the 12 scale bytes
                // (words hd.y, hd.z, hd.w): for s < 4 the low 6 bits of
                // bytes s and s+4; for s >= 4 the nibbles of byte s+4 with
                // the top two bits of bytes s-4 and s on top.
                const uint32_t a = (hd.y >> bsel) & 0xFFu, bm = (hd.z >> bsel) & 0xFFu, c = (hd.w >> bsel) & 0xFFu;
                const uint32_t sc = upper ? ((c & 15u) | ((a >> 2) & 0x30u)) : (a & 63u);
                const uint32_t mn = upper ? ((c >> 4) | ((bm >> 2) & 0x30u)) : (bm & 63u);
                const float A = __fmul_rn(f16_bits_to_f32(hd.x), small_uint_to_f32(sc));
                const float B = __fmul_rn(f16_bits_to_f32(hd.x >> 16), small_uint_to_f32(mn));
                uint4 y0, y1;
                if constexpr (T == 12) {
                    y0 = q4k_eight(A, B, w0.x, w0.y, nsh);
                    y1 = q4k_eight(A, B, w1.x, w1.y, nsh);
                } else {
                    const uint2 h0 = *reinterpret_cast<const uint2 *>(b + qhoff);
                    const uint2 h1 = *reinterpret_cast<const uint2 *>(b + qhoff + 16);
                    const uint64_t a2 = f32x2(A, A), nb2 = f32x2(-B, -B);
                    y0 = fma_bytes_eight(a2, nb2,
                                         ((w0.x >> nsh) & 0x0F0F0F0Fu) | (__funnelshift_r(h0.x, h0.x, hrot) & 0x10101010u),
                                         ((w0.y >> nsh) & 0x0F0F0F0Fu) | (__funnelshift_r(h0.y, h0.y, hrot) & 0x10101010u));
                    y1 = fma_bytes_eight(a2, nb2,
                                         ((w1.x >> nsh) & 0x0F0F0F0Fu) | (__funnelshift_r(h1.x, h1.x, hrot) & 0x10101010u),
                                         ((w1.y >> nsh) & 0x0F0F0F0Fu) | (__funnelshift_r(h1.y, h1.y, hrot) & 0x10101010u));
                }
                const uint32_t bi = static_cast<uint32_t>(b0 + blk);
                stg_v4(dest<F::QK>(out, bi, eoff, mode, K, ldo, br), y0);
                stg_v4(dest<F::QK>(out, bi, eoff + 16, mode, K, ldo, br), y1);
            }
        }
    } else if constexpr (T == 14) {
        // Lane pair j of a 16-lane half owns the 32 elements 128hh + 32t + l
        // (l = 0..31) with hh = j/4, t = j%4; lane h of the pair takes l in
        // 8h + {0..7} (scale byte 8hh + 2t) and 16 + 8h + {0..7} (scale
        // byte 8hh + 2t + 1).  Low nibbles: ql bytes 64hh + 32(t%2) + l,
        // shifted by 4(t/2); high bits: qh bytes 32hh + l, bits 2t, 2t+1.
        const int l = lane & 15, grp = l >> 1, h = l & 1;
        const int hh = grp >> 2, t = grp & 3;
        const int lsh = (t >> 1) * 4, hrot = (2 * t + 28) & 31;
        const int qloff = 64 * hh + 32 * (t & 1) + 8 * h;
        const int qhoff = 128 + 32 * hh + 8 * h;
        const int scoff = 192 + 8 * hh + 2 * t;
        const int eoff = 128 * hh + 32 * t + 8 * h;
#pragma unroll
        for (int ps = 0; ps < kPasses; ++ps) {
            const int blk = (warp * kPasses + ps) * F::BPG + (lane >> 4);
            if (blk < nb) {
                const int bo = blk * F::BB;             // 2-byte aligned
                const uint2 l0 = lds8_a2(sm, bo + qloff), l1 = lds8_a2(sm, bo + qloff + 16);
                const uint2 h0 = lds8_a2(sm, bo + qhoff), h1 = lds8_a2(sm, bo + qhoff + 16);
                const float d = f16_bits_to_f32(lds_u16(sm, bo + 208));
                // Two int8 scales: biased to 0..255 by flipping the sign bit,
                // converted exactly with the 2^23 trick, unbiased, times d.
                const uint64_t s2 = add_f32x2(magic_pair(lds_u16(sm, bo + scoff) ^ 0x8080u, 0),
                                              f32x2(-8388736.0f, -8388736.0f));   // -(2^23 + 128)
                float A0, A1;
                asm("mov.b64 {%0, %1}, %2;" : "=f"(A0), "=f"(A1) : "l"(mul_f32x2(s2, f32x2(d, d))));
                const uint4 y0 = q6k_core(A0, q6k_bytes(l0.x, lsh, h0.x, hrot), q6k_bytes(l0.y, lsh, h0.y, hrot));
                const uint4 y1 = q6k_core(A1, q6k_bytes(l1.x, lsh, h1.x, hrot), q6k_bytes(l1.y, lsh, h1.y, hrot));
                const uint32_t bi = static_cast<uint32_t>(b0 + blk);
                stg_v4(dest<F::QK>(out, bi, eoff, mode, K, ldo, br), y0);
                stg_v4(dest<F::QK>(out, bi, eoff + 16, mode, K, ldo, br), y1);
            }
        }
    } else if constexpr (T == 2 || T == 6 || T == 7) {
        // Q4_0 / Q5_0 / Q5_1.  Lane pair j owns block j of the group; lane h
        // takes elements 8h + {0..7} (low nibbles of qs[8h..8h+7]) and
        // 16 + 8h + {0..7} (high nibbles of the same bytes).  Q5_0 / Q5_1 add
        // bit e of the 32-bit qh plane as the fifth bit of element e.
        constexpr int kQh = T == 6 ? 2 : 4;                    // qh offset (Q5_0, Q5_1)
        constexpr int kQs = T == 2 ? 2 : (T == 6 ? 6 : 8);     // qs offset
        const int h = lane & 1;
#pragma unroll
        for (int ps = 0; ps < kPasses; ++ps) {
            const int blk = (warp * kPasses + ps) * F::BPG + (lane >> 1);
            if (blk < nb) {
                const int bo = blk * F::BB;              // 2-byte aligned (Q5_1: 8-byte)
                const uint32_t d16 = lds_u16(sm, bo);
                const uint2 w = lds8_a2(sm, bo + kQs + 8 * h);
                uint32_t l0 = w.x & 0x0F0F0F0Fu, l1 = w.y & 0x0F0F0F0Fu;
                uint32_t u0 = (w.x >> 4) & 0x0F0F0F0Fu, u1 = (w.y >> 4) & 0x0F0F0F0Fu;
                if constexpr (T != 2) {
                    const uint32_t qh = lds_u16(sm, bo + kQh) | (lds_u16(sm, bo + kQh + 2) << 16);
                    const uint32_t lo_bits = qh >> (8 * h), hi_bits = qh >> (16 + 8 * h);
                    l0 |= spread4_bit4(lo_bits);
                    l1 |= spread4_bit4(lo_bits >> 4);
                    u0 |= spread4_bit4(hi_bits);
                    u1 |= spread4_bit4(hi_bits >> 4);
                }
                uint4 y0, y1;
                if constexpr (T == 7) {
                    // y = RN16(RN32(d * q5 + m))
                    const float d = f16_bits_to_f32(d16), m = f16_bits_to_f32(lds_u16(sm, bo + 2));
                    const uint64_t a2 = f32x2(d, d), m2 = f32x2(m, m);
                    y0 = fma_bytes_eight(a2, m2, l0, l1);
                    y1 = fma_bytes_eight(a2, m2, u0, u1);
                } else {
                    // y = RN16(d * (q - 8)) (Q4_0), RN16(d * (q5 - 16)) (Q5_0)
                    constexpr uint32_t kBias = T == 2 ? 0x64086408u : 0x64106410u;   // f16 1032 / 1040
                    y0 = f16_bias_eight(d16, l0, l1, kBias);
                    y1 = f16_bias_eight(d16, u0, u1, kBias);
                }
                const uint32_t bi = static_cast<uint32_t>(b0 + blk);
                stg_v4(dest<F::QK>(out, bi, 8 * h, mode, K, ldo, br), y0);
                stg_v4(dest<F::QK>(out, bi, 16 + 8 * h, mode, K, ldo, br), y1);
            }
        }
    } else {
        // Lane pair j owns block j of the group; lane h takes quants 8h +
        // {0..7} and 16 + 8h + {0..7}.
        const int h = lane & 1;
#pragma unroll
        for (int ps = 0; ps < kPasses; ++ps) {
            const int blk = (warp * kPasses + ps) * F::BPG + (lane >> 1);
            if (blk < nb) {
                const int bo = blk * F::BB;             // 2-byte aligned
                const uint32_t d16 = lds_u16(sm, bo);
                const uint2 w0 = lds8_a2(sm, bo + 2 + 8 * h), w1 = lds8_a2(sm, bo + 18 + 8 * h);
                const uint32_t bi = static_cast<uint32_t>(b0 + blk);
                stg_v4(dest<F::QK>(out, bi, 8 * h, mode, K, ldo, br), q80_eight(d16, w0.x, w0.y));
                stg_v4(dest<F::QK>(out, bi, 16 + 8 * h, mode, K, ldo, br), q80_eight(d16, w1.x, w1.y));
            }
        }
    }
}

// Float weights: F32 (type 0), F16 (1), BF16 (30).  One f16 per element,
// round to nearest even (F16 is copied bit for bit; a BF16 value widens
// exactly to f32 first).  Piece v is elements 8v .. 8v+7 of the flat stream
// (K % 8 == 0, so the eight share a row), stored as one 16-byte write;
// consecutive threads take consecutive pieces on both sides.  Each thread
// has kConvPieces pieces, kConvThreads apart, with all loads in flight
// before the first store.
constexpr int kConvThreads = 256;
constexpr int kConvPieces = 4;

template <int T>
__device__ __forceinline__ uint4 convert_piece(const uint8_t *src)
{
    if constexpr (T == 1) {
        return ldg_nc_v4(src);
    } else if constexpr (T == 30) {
        const uint4 b = ldg_nc_v4(src);
        const uint32_t w[4] = {b.x, b.y, b.z, b.w};
        uint32_t r[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
            r[i] = cvt_f16x2(f32x2(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xFFFF0000u)));
        return make_uint4(r[0], r[1], r[2], r[3]);
    } else {
        const uint4 a = ldg_nc_v4(src), b = ldg_nc_v4(src + 16);
        return make_uint4(cvt_f16x2(f32x2(__uint_as_float(a.x), __uint_as_float(a.y))),
                          cvt_f16x2(f32x2(__uint_as_float(a.z), __uint_as_float(a.w))),
                          cvt_f16x2(f32x2(__uint_as_float(b.x), __uint_as_float(b.y))),
                          cvt_f16x2(f32x2(__uint_as_float(b.z), __uint_as_float(b.w))));
    }
}

template <int T>
__global__ void __launch_bounds__(kConvThreads) k_convert(const uint8_t *__restrict__ q, uint32_t npieces,
                                                         __half *__restrict__ out, int64_t ldo, int mode,
                                                         BlockRows pr)
{
    constexpr int kSrcBytes = T == 0 ? 32 : 16;
    const uint32_t v0 = blockIdx.x * (kConvThreads * kConvPieces) + threadIdx.x;
    uint4 y[kConvPieces];
#pragma unroll
    for (int i = 0; i < kConvPieces; ++i) {
        const uint32_t v = v0 + i * kConvThreads;
        if (v < npieces)
            y[i] = convert_piece<T>(q + static_cast<int64_t>(v) * kSrcBytes);
    }
    grid_dep_launch();
    grid_dep_wait();   // the output may be read by the previous kernel on the stream
#pragma unroll
    for (int i = 0; i < kConvPieces; ++i) {
        const uint32_t v = v0 + i * kConvThreads;
        if (v < npieces) {
            __half *dst;
            if (mode == 0) {
                dst = out + static_cast<int64_t>(v) * 8;
            } else {
                uint32_t n, c;
                block_row(v, pr, n, c);
                dst = out + static_cast<int64_t>(n) * ldo + static_cast<int64_t>(c) * 8;
            }
            stg_v4(dst, y[i]);
        }
    }
}

template <int T>
cudaError_t launch_convert(const void *q, int64_t nelem, __half *out, int64_t K, int64_t ldo, cudaStream_t s)
{
    const int64_t npieces = nelem / 8;
    if (npieces > 0xFFFFFFFFLL - kConvThreads * kConvPieces || K % 8 != 0)
        return cudaErrorInvalidValue;
    const int64_t per_cta = kConvThreads * kConvPieces;
    BlockRows pr{1u, 0xFFFFFFFFu};
    int mode = 0;
    if (ldo != K) {
        mode = 1;
        pr.bpr = static_cast<uint32_t>(K / 8);
        pr.m = 0xFFFFFFFFu / pr.bpr;
    }
    const cudaError_t e =
        launch_kernel(k_convert<T>, dim3(static_cast<unsigned>((npieces + per_cta - 1) / per_cta)),
                      dim3(kConvThreads), 0, s, static_cast<const uint8_t *>(q), static_cast<uint32_t>(npieces),
                      out, ldo, mode, pr);
    note_launch();
    return e;
}

template <int T>
cudaError_t launch_t(const void *q, int64_t nblocks, __half *out, int64_t K, int64_t ldo, cudaStream_t s)
{
    using F = Fmt<T>;
    if (nblocks > 0x7FFFFFFF)   // block indices are 32-bit in the kernel
        return cudaErrorInvalidValue;
    const int64_t grid = (nblocks + F::G - 1) / F::G;
    BlockRows br{1u, 0xFFFFFFFFu};
    int mode = 2;
    if (ldo == K) {
        mode = 0;
    } else if (K % F::QK == 0) {
        mode = 1;
        br.bpr = static_cast<uint32_t>(K / F::QK);
        br.m = 0xFFFFFFFFu / br.bpr;
    }
    const cudaError_t e = launch_kernel(k_dequant<T>, dim3(static_cast<unsigned>(grid)), dim3(kThreads), 0, s,
                                        static_cast<const uint8_t *>(q), nblocks, out, K, ldo, mode, br);
    note_launch();
    return e;
}

}  // namespace

namespace {

// The binary32 bit patterns first + i (i < 2 * pairs) through the decoders'
// own f32 -> f16 step (cvt_f16x2: two values, round to nearest even):
// out[i] holds the f16 bits of pattern first + 2i (low half) and
// first + 2i + 1 (high half).  Test hook for that rounding step.
__global__ void k_debug_cvt_f16(uint32_t first, uint32_t pairs, uint32_t *__restrict__ out)
{
    grid_dep_wait();
    const uint32_t stride = gridDim.x * blockDim.x;
    for (uint32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < pairs; i += stride) {
        const uint32_t b = first + 2u * i;
        out[i] = cvt_f16x2(f32x2(__uint_as_float(b), __uint_as_float(b + 1u)));
    }
}

}  // namespace

cudaError_t launch_debug_cvt_f16(uint32_t first, int64_t count, uint16_t *out, cudaStream_t s)
{
    const uint32_t pairs = static_cast<uint32_t>(count / 2);
    const cudaError_t e = launch_kernel(k_debug_cvt_f16, dim3(1216), dim3(256), 0, s, first, pairs,
                                        reinterpret_cast<uint32_t *>(out));
    note_launch();
    return e;
}

cudaError_t launch_dequant(int type, const void *q, int64_t nblocks, __half *out, int64_t K, int64_t ldo,
                           cudaStream_t s)
{
    if (nblocks <= 0)
        return cudaSuccess;
    switch (type) {
    case 0: return launch_convert<0>(q, nblocks, out, K, ldo, s);
    case 1: return launch_convert<1>(q, nblocks, out, K, ldo, s);
    case 30: return launch_convert<30>(q, nblocks, out, K, ldo, s);
    case 2: return launch_t<2>(q, nblocks, out, K, ldo, s);
    case 6: return launch_t<6>(q, nblocks, out, K, ldo, s);
    case 7: return launch_t<7>(q, nblocks, out, K, ldo, s);
    case 8: return launch_t<8>(q, nblocks, out, K, ldo, s);
    case 12: return launch_t<12>(q, nblocks, out, K, ldo, s);
    case 13: return launch_t<13>(q, nblocks, out, K, ldo, s);
    case 14: return launch_t<14>(q, nblocks, out, K, ldo, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace mq
