// fused.cu -- fused dequant-in-GEMM on the tcgen05 tensor cores (sm_103a).
//
//   Y[m, n] = sum_k X[m, k] * W[n, k],  W decoded on chip from its raw blocks
//
// ("05 · 8p — Persistent f16 weight cache + fused dequant-in-GEMM",
// section 2: B tiles are staged in shared memory as quantized bytes and
// expanded to f16 right before the MMA; no extra VRAM.  Section 3.2, third
// site: the fused GEMM body.  Section 3.3: its decode must round exactly as
// the standalone decoder does -- both use mq_decode.cuh.)
//
// Tile geometry and schedule are those of the cached GEMM (mq_tile.cuh):
// 128 weight rows (MMA M) x BN tokens (MMA N) per tile, persistent CTAs,
// split-K tail.  What changes is where the 128x64 f16 weight operand comes
// from.  Three rings decouple the roles:
//   raw ring  (shared memory) 256 K elements of raw blocks for the tile's rows,
//   A ring    (tensor memory) the decoded f16 weight operand of one raw
//             chunk: 128 rows (TMEM lanes) x 256 K (128 columns, 2 f16 per
//             column); tcgen05.mma reads its A operand straight from TMEM,
//             so the decoded operand never passes through shared memory,
//   X ring    (shared memory) the BN x 256 activations of a chunk (TMA,
//             128-byte swizzle, four 64-wide K boxes).
// Warp roles (512 threads):
//   warp 0      raw producer.  Weights whose rows start on block boundaries
//               (K % 256 == 0) are read with 2-D TMA: the row stride RB is a
//               multiple of 16 bytes for every g-th row (g in {1,2,4,8}), so
//               g tensor maps, one per class of rows mod g with its base
//               aligned down to 16 bytes, fetch a chunk of all 128 rows in g
//               copies; the decoders read the bytes at their real offsets.
//               Other weights (rows starting inside a block) take one 1-D
//               bulk copy per row of the 16-byte-aligned byte range.  Q6_K
//               (210 B) and Q8_0 (34 B) blocks are only 2-byte aligned; in
//               both cases every global access stays 16-byte aligned.
//   warps 1, 3  MMA issuers (one thread each; warp 1 also owns the TMEM
//               allocation): per chunk one wait, M=128 x N=BN x K=16 MMAs
//               with A in TMEM, one commit.  With two issuers (BN <= 64),
//               on different sub-partitions, each takes two of the chunk's
//               four K steps into its own partial accumulator: the issue of
//               an MMA is a short chain of dependent instructions competing
//               with the decode warps for issue slots, and one thread alone
//               leaves the tensor pipe idle between MMAs.
//   warp 2      activation producer (TMA, lane 0): the BN x 256 activations
//               of a chunk (four 64-wide boxes) into the chunk slot's X
//               stage; lane 1 announces each slot's landed activations.
//   warps 4-7   epilogue (TMEM -> Y / split-K workspace; sums the partial
//               accumulators in a fixed order).
//   warps 8-15  decoders: each thread turns the raw elements of one weight
//               row into f16 and stores them with tcgen05.st into its row's
//               TMEM lane -- at tiles of up to 32 tokens (all formats but
//               Q6_K) as two groups of four warps on alternate chunks, four
//               K steps (256 elements) per thread; otherwise all eight warps
//               on every chunk, two K steps (128 elements) per thread.  Eight
//               warps keep the integer pipe busy; more of them take issue
//               slots from the MMA issuers (measured: ~86 cycles per MMA next
//               to 8 busy warps, ~220 next to 30).
// Chunk slots: A stage s (TMEM) and X stage s (shared memory) form one slot;
// `ready[s]` completes when the warps that decode the chunk have written A
// and a second thread of warp 2 has seen the slot's activations land;
// `done[s]` (an MMA commit) frees both.
#include <cstdint>
#include <cuda_runtime.h>

#include "mq_decode.cuh"
#include "mq_internal.h"
#include "mq_launch.cuh"
#include "mq_ptx.cuh"
#include "mq_smem.cuh"
#include "mq_tile.cuh"

namespace mq {
namespace {

constexpr int kDecodeWarp0 = 8;
constexpr int kDecodeWarps = 8;                         // 8 or 16
constexpr int kThreadsF = (kDecodeWarp0 + kDecodeWarps) * 32;

// Decoder groups: with two, the decoder warps split into two groups of four
// (one warp per TMEM lane quarter) that take alternate chunks, each thread
// decoding all four K steps of its row; with one, all eight decode every
// chunk, two K steps per thread.  Measured back to back (rotating copies of
// an 18944 x 3584 weight, and the 3584 x 18944 Q6_K one): at tiles of up to 32
// tokens two groups are 2-6 % faster for every format but Q6_K (Q4_K at
// M = 32: 18.30 -> 17.56 us; Q5_K 21.69 -> 20.44; Q5_0 18.96 -> 17.82); at
// 128-token tiles and for Q6_K they are as fast or slower (Q6_K down, M = 32:
// 23.8 -> 25.3 us).
__host__ __device__ constexpr int decoder_groups(int qt, int bn)
{
    return (bn <= 32 && qt != 14) ? 2 : 1;
}
constexpr int kChunkSteps = 4;               // K steps (of 64) per raw stage: 256 K elements
constexpr int kMaxRaw = 8, kMaxStages = 3;
// MMA issuers: two (warps 1 and 3, on different SM sub-partitions) each
// taking half of every chunk's K steps into its own partial accumulator
// while BN <= 64, one at BN = 128.  An issuing thread shares its sub-partition's issue slots
// with the decode warps, and the issue of one tcgen05.mma is a short chain
// of dependent instructions, so one thread alone cannot keep the tensor pipe
// busy while the decoders run.
//
// TMEM: two accumulator slots (double buffering across units) of
// kIssuers partial accumulators of BN columns each, then the A stages of
// 128 columns each (one raw chunk of 256 K elements, two f16 per column):
// three stages from column 128 for BN <= 32, two from column 256 above.
constexpr int kTmemCols = 512;
constexpr int kAStageCols = 128;
constexpr int kSmemLimit = 227 * 1024;
constexpr int kBarBytes = 512;

__host__ __device__ constexpr int issuers_for(int bn)
{
    return bn <= 64 ? 2 : 1;
}

__host__ __device__ constexpr int a_stages_for(int bn)
{
    return bn <= 32 ? 3 : 2;
}

__host__ __device__ constexpr uint32_t a_col0_for(int bn)
{
    return bn <= 32 ? 128u : 256u;
}

template <int QT> struct QF;
template <> struct QF<2> { static constexpr int QK = 32, BB = 18; };     // Q4_0
template <> struct QF<6> { static constexpr int QK = 32, BB = 22; };     // Q5_0
template <> struct QF<7> { static constexpr int QK = 32, BB = 24; };     // Q5_1
template <> struct QF<8> { static constexpr int QK = 32, BB = 34; };     // Q8_0
template <> struct QF<12> { static constexpr int QK = 256, BB = 144; };  // Q4_K
template <> struct QF<13> { static constexpr int QK = 256, BB = 176; };  // Q5_K
template <> struct QF<14> { static constexpr int QK = 256, BB = 210; };  // Q6_K

// Whole 32-element blocks of Q4_0 / Q5_0 / Q5_1 at a 2-byte-aligned shared
// address, into out[0..3] (8 f16 each, elements 0..31 in order): element e
// is the low nibble of qs[e] (e < 16) or the high nibble of qs[e-16], with
// bit e of the 32-bit qh plane as fifth bit for Q5_0 / Q5_1.
template <int QT>
__device__ __forceinline__ void small_block32(uint32_t blk, uint4 (&out)[4])
{
    constexpr int kQs = QT == 2 ? 2 : (QT == 6 ? 6 : 8);
    uint32_t q[4];
    lds_16B_a2(blk + kQs, q);
    uint32_t v[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        v[i] = q[i] & 0x0F0F0F0Fu;             // elements 4i .. 4i+3
        v[4 + i] = (q[i] >> 4) & 0x0F0F0F0Fu;  // elements 16+4i .. 16+4i+3
    }
    if constexpr (QT != 2) {
        constexpr int kQh = QT == 6 ? 2 : 4;
        const uint32_t qh = lds_u16(blk + kQh) | (lds_u16(blk + kQh + 2) << 16);
#pragma unroll
        for (int i = 0; i < 8; ++i)
            v[i] |= spread4_bit4(qh >> (4 * i));
    }
    const uint32_t d16 = lds_u16(blk);
    if constexpr (QT == 7) {
        const float d = f16_bits_to_f32(d16), m = f16_bits_to_f32(lds_u16(blk + 2));
        const uint64_t a2 = f32x2(d, d), m2 = f32x2(m, m);
#pragma unroll
        for (int i = 0; i < 4; ++i)
            out[i] = fma_bytes_eight(a2, m2, v[2 * i], v[2 * i + 1]);
    } else {
        constexpr uint32_t kBias = QT == 2 ? 0x64086408u : 0x64106410u;   // f16 1032 (q - 8) / 1040 (q - 16)
#pragma unroll
        for (int i = 0; i < 4; ++i)
            out[i] = f16_bias_eight(d16, v[2 * i], v[2 * i + 1], kBias);
    }
}

// Q4_K / Q5_K: (d*sc, -dmin*m) of sub-blocks 2j and 2j+1 from the block
// header (d | dmin, scale bytes 0..3, 4..7, 8..11): the block format's
// packing rule applied four bytes at a time, then the byte pair 2(j%2).
__device__ __forceinline__ void kquant_pair_scales(uint4 hdr, int j, float &A0, float &A1, float &nB0, float &nB1)
{
    uint32_t scw, mnw;
    if (j < 2) {
        scw = hdr.y & 0x3F3F3F3Fu;
        mnw = hdr.z & 0x3F3F3F3Fu;
    } else {
        scw = (hdr.w & 0x0F0F0F0Fu) | ((hdr.y >> 2) & 0x30303030u);
        mnw = ((hdr.w >> 4) & 0x0F0F0F0Fu) | ((hdr.z >> 2) & 0x30303030u);
    }
    const int bsel = 2 * (j & 1);
    const uint64_t m2 = f32x2(-8388608.0f, -8388608.0f);
    const float d = f16_bits_to_f32(hdr.x), dmin = f16_bits_to_f32(hdr.x >> 16);
    unpack_f32x2(mul_f32x2(add_f32x2(magic_pair(scw, bsel), m2), f32x2(d, d)), A0, A1);
    unpack_f32x2(mul_f32x2(add_f32x2(magic_pair(mnw, bsel), m2), f32x2(-dmin, -dmin)), nB0, nB1);
}

// Q5_K sub-block s (elements 32s .. 32s+31) of the 16-byte-aligned block at
// b, given that sub-block's d*sc (A) and -(dmin*m) (nB): nibble (low for
// even s, high for odd) of qs[32(s/2) + i] plus bit s of qh[i] as fifth bit.
__device__ __forceinline__ void q5k_sub32(uint32_t b, int s, float A, float nB, uint4 (&out)[4])
{
    const uint4 q0 = lds_v4(b + 48 + 32 * (s >> 1)), q1 = lds_v4(b + 64 + 32 * (s >> 1));
    const uint4 h0 = lds_v4(b + 16), h1 = lds_v4(b + 32);
    const int nsh = 4 * (s & 1);
    const int hrot = (s + 28) & 31;   // rotate bit s of every byte onto bit 4
    const uint64_t a2 = f32x2(A, A), nb2 = f32x2(nB, nB);
    const uint32_t qw[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
    const uint32_t hw[8] = {h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
    uint32_t v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
        v[i] = ((qw[i] >> nsh) & 0x0F0F0F0Fu) | (__funnelshift_r(hw[i], hw[i], hrot) & 0x10101010u);
#pragma unroll
    for (int i = 0; i < 4; ++i)
        out[i] = fma_bytes_eight(a2, nb2, v[2 * i], v[2 * i + 1]);
}

struct RowSpan {
    int64_t s0;       // 16-byte-aligned start of the copied range in the stream
    uint32_t bytes;   // multiple of 16
};

// Bulk-copy path: byte range of the stream holding flat elements
// [n*K + kc0, n*K + kc0 + len), widened to 16-byte boundaries.  The stream's
// length is a multiple of 16 (checked on the host), so the widened end
// never passes it.
template <int QT>
__device__ __forceinline__ RowSpan row_span(int64_t n, int64_t K, int64_t kc0, int64_t len)
{
    using F = QF<QT>;
    const int64_t e0 = n * K + kc0, e1 = e0 + len;
    const int64_t b0 = (e0 / F::QK) * F::BB;
    const int64_t b1 = ((e1 + F::QK - 1) / F::QK) * F::BB;
    RowSpan r;
    r.s0 = b0 & ~static_cast<int64_t>(15);
    r.bytes = static_cast<uint32_t>(((b1 + 15) & ~static_cast<int64_t>(15)) - r.s0);
    return r;
}

// Decode 32 consecutive elements starting at element o of the block at
// shared address b into out[0..3] (8 f16 each).
template <int QT>
__device__ __forceinline__ void decode32(uint32_t b, int o, uint4 (&out)[4]);

template <>
__device__ __forceinline__ void decode32<12>(uint32_t b, int o, uint4 (&out)[4])
{
    // Q4_K: b is 16-byte aligned (144-byte blocks, copies start on a block).
    const uint4 hdr = lds_v4(b);   // d | dmin, scale bytes 0..3, 4..7, 8..11
    const float d = f16_bits_to_f32(hdr.x), dmin = f16_bits_to_f32(hdr.x >> 16);
    const int p = o >> 6, hi = (o >> 5) & 1;
    int sc, m;
    q4k_scale_min(hdr.y, hdr.z, hdr.w, 2 * p + hi, sc, m);
    const float A = __fmul_rn(d, static_cast<float>(sc)), B = __fmul_rn(dmin, static_cast<float>(m));
    const uint4 q0 = lds_v4(b + 16 + 32 * p), q1 = lds_v4(b + 32 + 32 * p);
    const int sh = 4 * hi;
    out[0] = q4k_eight(A, B, q0.x, q0.y, sh);
    out[1] = q4k_eight(A, B, q0.z, q0.w, sh);
    out[2] = q4k_eight(A, B, q1.x, q1.y, sh);
    out[3] = q4k_eight(A, B, q1.z, q1.w, sh);
}

template <>
__device__ __forceinline__ void decode32<14>(uint32_t b, int o, uint4 (&out)[4])
{
    // Q6_K: b is 2-byte aligned.  Elements o .. o+31 are quarter t of half hh.
    const int hh = o >> 7, t = (o >> 5) & 3;
    uint32_t lq[8], hq[8];
    lds_32B_a2(b + 64 * hh + ((t & 1) ? 32 : 0), lq);
    lds_32B_a2(b + 128 + 32 * hh, hq);
    const int lsh = (t & 2) ? 4 : 0, hsh = 2 * t;
    const float d = f16_bits_to_f32(lds_u16(b + 208));
    const float A0 = __fmul_rn(d, static_cast<float>(lds_s8(b + 192 + (o >> 4))));
    const float A1 = __fmul_rn(d, static_cast<float>(lds_s8(b + 193 + (o >> 4))));
    out[0] = q6k_eight(A0, lq[0], lq[1], lsh, hq[0], hq[1], hsh);
    out[1] = q6k_eight(A0, lq[2], lq[3], lsh, hq[2], hq[3], hsh);
    out[2] = q6k_eight(A1, lq[4], lq[5], lsh, hq[4], hq[5], hsh);
    out[3] = q6k_eight(A1, lq[6], lq[7], lsh, hq[6], hq[7], hsh);
}

template <>
__device__ __forceinline__ void decode32<8>(uint32_t b, int o, uint4 (&out)[4])
{
    // Q8_0: one whole 34-byte block (o == 0), 2-byte aligned.
    (void)o;
    const uint32_t d16 = lds_u16(b);
    uint32_t q[8];
    lds_32B_a2(b + 2, q);
#pragma unroll
    for (int j = 0; j < 4; ++j)
        out[j] = q80_eight(d16, q[2 * j], q[2 * j + 1]);
}

template <>
__device__ __forceinline__ void decode32<2>(uint32_t b, int o, uint4 (&out)[4])
{
    (void)o;   // Q4_0: one whole block (o == 0), 2-byte aligned
    small_block32<2>(b, out);
}

template <>
__device__ __forceinline__ void decode32<6>(uint32_t b, int o, uint4 (&out)[4])
{
    (void)o;   // Q5_0
    small_block32<6>(b, out);
}

template <>
__device__ __forceinline__ void decode32<7>(uint32_t b, int o, uint4 (&out)[4])
{
    (void)o;   // Q5_1
    small_block32<7>(b, out);
}

template <>
__device__ __forceinline__ void decode32<13>(uint32_t b, int o, uint4 (&out)[4])
{
    // Q5_K: b is 16-byte aligned; elements o .. o+31 are sub-block o/32.
    const uint4 hdr = lds_v4(b);
    const int s = o >> 5;
    float A0, A1, nB0, nB1;
    kquant_pair_scales(hdr, s >> 1, A0, A1, nB0, nB1);
    q5k_sub32(b, s, (s & 1) ? A1 : A0, (s & 1) ? nB1 : nB0, out);
}

// Block-aligned weights (K % 256 == 0): one raw chunk of a row is 256
// consecutive elements starting on a block boundary -- one Q4_K or Q6_K
// block, or eight Q8_0 blocks -- at `b` (the row's slot plus its leading
// misalignment).  decode_step decodes the 64 elements of K step j of the
// chunk (j = 0..3; elements 64j + 32h .. +31 for halves h = 0, 1) and stores
// each half into TMEM columns col + 16h .. +15 (two f16 per column).
// tcgen05.st is .sync.aligned: j is the same for all lanes of a warp and the
// stores sit outside any lane-dependent branch.  Rows past the weight's end
// decode whatever their slot holds: the MMA keeps weight rows apart (row r
// of A only feeds row r of the accumulator) and the epilogue never stores
// rows past N, so those values cannot reach Y.

// int8 held in the low byte of v -> exact f32 (sign flipped to a 0..255
// bias, 2^23 trick, bias removed).
__device__ __forceinline__ float s8_to_f32(uint32_t v)
{
    return __int_as_float(0x4B000000u | ((v ^ 0x80u) & 0xFFu)) - 8388736.0f;   // 2^23 + 128
}

template <int QT>
__device__ __forceinline__ void decode_step(uint32_t b, int j, uint32_t col);

template <>
__device__ __forceinline__ void decode_step<12>(uint32_t b, int j, uint32_t col)
{
    // Q4_K, b 16-byte aligned.  Step j is group p = j: qs bytes 32j .. +31,
    // low nibbles for sub-block 2j (half 0), high nibbles for 2j+1 (half 1).
    const uint4 hdr = lds_v4(b);   // d | dmin, scale bytes 0..3, 4..7, 8..11
    const uint4 q0 = lds_v4(b + 16 + 32 * j), q1 = lds_v4(b + 32 + 32 * j);
    float A0, A1, nB0, nB1;   // d*sc and -(dmin*m) of the two sub-blocks, exact
    kquant_pair_scales(hdr, j, A0, A1, nB0, nB1);
    {
        const uint64_t a2 = f32x2(A0, A0), nb2 = f32x2(nB0, nB0);
        uint4 out[4];
        out[0] = fma_bytes_eight(a2, nb2, q0.x & 0x0F0F0F0Fu, q0.y & 0x0F0F0F0Fu);
        out[1] = fma_bytes_eight(a2, nb2, q0.z & 0x0F0F0F0Fu, q0.w & 0x0F0F0F0Fu);
        out[2] = fma_bytes_eight(a2, nb2, q1.x & 0x0F0F0F0Fu, q1.y & 0x0F0F0F0Fu);
        out[3] = fma_bytes_eight(a2, nb2, q1.z & 0x0F0F0F0Fu, q1.w & 0x0F0F0F0Fu);
        __syncwarp();
        tmem_st_32x32b_x16(col, out);
    }
    {
        // High nibbles stay in place (bytes 16q); A/16 is exact (a power-of-two
        // scaling of a normal f32), so (A/16)*(16q) = A*q as for the low half.
        const float a16 = A1 * 0.0625f;
        const uint64_t a2 = f32x2(a16, a16), nb2 = f32x2(nB1, nB1);
        uint4 out[4];
        out[0] = fma_bytes_eight(a2, nb2, q0.x & 0xF0F0F0F0u, q0.y & 0xF0F0F0F0u);
        out[1] = fma_bytes_eight(a2, nb2, q0.z & 0xF0F0F0F0u, q0.w & 0xF0F0F0F0u);
        out[2] = fma_bytes_eight(a2, nb2, q1.x & 0xF0F0F0F0u, q1.y & 0xF0F0F0F0u);
        out[3] = fma_bytes_eight(a2, nb2, q1.z & 0xF0F0F0F0u, q1.w & 0xF0F0F0F0u);
        __syncwarp();
        tmem_st_32x32b_x16(col + 16, out);
    }
}

template <>
__device__ __forceinline__ void decode_step<13>(uint32_t b, int j, uint32_t col)
{
    // Q5_K, b 16-byte aligned: sub-blocks 2j (half 0) and 2j+1 (half 1).
    const uint4 hdr = lds_v4(b);
    float A0, A1, nB0, nB1;
    kquant_pair_scales(hdr, j, A0, A1, nB0, nB1);
    uint4 out[4];
    q5k_sub32(b, 2 * j, A0, nB0, out);
    __syncwarp();
    tmem_st_32x32b_x16(col, out);
    q5k_sub32(b, 2 * j + 1, A1, nB1, out);
    __syncwarp();
    tmem_st_32x32b_x16(col + 16, out);
}

template <>
__device__ __forceinline__ void decode_step<14>(uint32_t b, int j, uint32_t col)
{
    // Q6_K, b 2-byte aligned.  Step j lies in block half hh = j/2; its half h
    // is quarter t = 2(j%2) + h: low bits from ql bytes 64hh + 32h .. +31
    // (low nibbles for even j, high for odd), high bits from qh bytes
    // 128 + 32hh .. +31 (bits 2t, 2t+1), scales sc[4j + 2h] and sc[4j + 2h + 1].
    const int hh = j >> 1, odd = j & 1;
    const float d = f16_bits_to_f32(lds_u16(b + 208));
    uint32_t hq[8];
    lds_32B_a2(b + 128 + 32 * hh, hq);
    const uint32_t scw = lds_u16(b + 192 + 4 * j) | (lds_u16(b + 194 + 4 * j) << 16);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        uint32_t lq[8];
        lds_32B_a2(b + 64 * hh + 32 * h, lq);
        const int lsh = 4 * odd, hsh = 2 * (2 * odd + h);
        const float A0 = __fmul_rn(d, s8_to_f32(scw >> (16 * h)));
        const float A1 = __fmul_rn(d, s8_to_f32(scw >> (16 * h + 8)));
        uint4 out[4];
        out[0] = q6k_eight(A0, lq[0], lq[1], lsh, hq[0], hq[1], hsh);
        out[1] = q6k_eight(A0, lq[2], lq[3], lsh, hq[2], hq[3], hsh);
        out[2] = q6k_eight(A1, lq[4], lq[5], lsh, hq[4], hq[5], hsh);
        out[3] = q6k_eight(A1, lq[6], lq[7], lsh, hq[6], hq[7], hsh);
        __syncwarp();
        tmem_st_32x32b_x16(col + 16 * h, out);
    }
}

template <>
__device__ __forceinline__ void decode_step<8>(uint32_t b, int j, uint32_t col)
{
    // Q8_0: half h of step j is the whole block 2j + h (34 bytes, 2-byte aligned).
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const uint32_t blk = b + 34 * (2 * j + h);
        const uint32_t d16 = lds_u16(blk);
        uint32_t q[8];
        lds_32B_a2(blk + 2, q);
        uint4 out[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
            out[i] = q80_eight(d16, q[2 * i], q[2 * i + 1]);
        __syncwarp();
        tmem_st_32x32b_x16(col + 16 * h, out);
    }
}

// Q4_0 / Q5_0 / Q5_1: a 256-element chunk is eight blocks; half h of step j
// is the whole block 2j + h.
#define MQ_SMALL_STEP(QT_)                                                              \
    template <>                                                                         \
    __device__ __forceinline__ void decode_step<QT_>(uint32_t b, int j, uint32_t col)   \
    {                                                                                   \
        _Pragma("unroll") for (int h = 0; h < 2; ++h)                                   \
        {                                                                               \
            uint4 out[4];                                                               \
            small_block32<QT_>(b + QF<QT_>::BB * (2 * j + h), out);                     \
            __syncwarp();                                                               \
            tmem_st_32x32b_x16(col + 16 * h, out);                                      \
        }                                                                               \
    }
MQ_SMALL_STEP(2)
MQ_SMALL_STEP(6)
MQ_SMALL_STEP(7)
#undef MQ_SMALL_STEP

template <int BN, int QT, bool TMA_RAW>
__global__ void __launch_bounds__(kThreadsF, 1)
    k_gemm_fused(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ RawMapsG maps, const GemmArgs a)
{
    using F = QF<QT>;
    constexpr int kXSub = BN * kBK * 2;               // one 64-wide K step of activations
    constexpr int kXBytes = kChunkSteps * kXSub;      // one X stage: a whole 256-element chunk
    constexpr int kNAcc = 2;                          // accumulators at TMEM columns [0, 2*BN)
    constexpr int S = a_stages_for(BN);               // A and X stages (one ring of chunk slots)
    static_assert(BN <= 128, "fused tiles stop at 128 tokens");
    constexpr int kIssuers = issuers_for(BN);
    constexpr int kGroups = decoder_groups(QT, BN);
    constexpr uint32_t kACol0 = a_col0_for(BN);
    static_assert(kNAcc * kIssuers * BN <= static_cast<int>(kACol0) && kACol0 + S * kAStageCols <= kTmemCols,
                  "TMEM budget");
    const int R = a.raw_stages, RS = a.raw_rs;

    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t *sX = base;
    uint8_t *sR = sX + S * kXBytes;
    uint64_t *bars = reinterpret_cast<uint64_t *>(sR + static_cast<size_t>(R) * kTileRows * RS);
    uint64_t *raw_full = bars;                // raw chunk landed (TMA bytes)
    uint64_t *raw_empty = raw_full + kMaxRaw; // raw chunk decoded (decoder warps)
    uint64_t *x_full = raw_empty + kMaxRaw;   // activation chunk landed (TMA bytes)
    uint64_t *ready = x_full + kMaxStages;    // A stage decoded and its X stage landed
    uint64_t *done = ready + kMaxStages;      // MMAs of the chunk slot finished (commit)
    uint64_t *tfull = done + kMaxStages;
    uint64_t *tempty = tfull + 2;
    uint64_t *drain = tempty + 2;             // one per issuer
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 2);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = TMA_RAW ? a.raw_g : 1;
    const int rows_per_class = kTileRows / g;

    if (threadIdx.x == 0) {
        for (int r = 0; r < R; ++r) {
            mbar_init(&raw_full[r], 1);
            mbar_init(&raw_empty[r], kDecodeWarps / kGroups);
        }
        for (int s = 0; s < S; ++s) {
            mbar_init(&x_full[s], 1);
            mbar_init(&ready[s], kDecodeWarps / kGroups + 1);
            mbar_init(&done[s], kIssuers);
        }
        for (int i = 0; i < kNAcc; ++i) {
            mbar_init(&tfull[i], kIssuers);
            mbar_init(&tempty[i], 4);
        }
        mbar_init(&drain[0], 1);
        mbar_init(&drain[1], 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    if (warp == 2 && lane == 0) {
        prefetch_tensormap(&tm_x);
        if (TMA_RAW)
            for (int gm = 0; gm < a.groups; ++gm)
                for (int c = 0; c < g; ++c)
                    prefetch_tensormap(&maps.w[gm].m[c]);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    grid_dep_launch();

    if (warp == 0) {
        // ---------------- raw producer (the raw blocks do not depend on the
        // previous kernel on the stream: no grid_dep_wait here)
        int r = 0;
        uint32_t rphase = 0;
        uint32_t issued = 0, iparity = 0;
        bool ok = a.stall_producer == 0;
        for (int u = blockIdx.x; ok && u < a.units; u += gridDim.x) {
            const UnitInfo ui = unit_info(a, u);
            const int nt = ui.tile / a.m_tiles;
            const int gm = group_of(a, nt);   // member of a group; rows counted inside it
            const int64_t n0 = static_cast<int64_t>(nt - a.g_tile0[gm]) * kTileRows;
            for (int kb = ui.kb0; kb < ui.kb1; kb += kChunkSteps) {
                const int steps = ui.kb1 - kb < kChunkSteps ? ui.kb1 - kb : kChunkSteps;
                bool w = true;
                if (lane == 0)
                    w = mbar_wait_bounded(&raw_empty[r], rphase ^ 1u, abort_flag, a.status);
                if (!__shfl_sync(0xFFFFFFFFu, w, 0)) {
                    ok = false;
                    break;
                }
                uint8_t *slot = sR + static_cast<size_t>(r) * kTileRows * RS;
                if (TMA_RAW) {
                    if (lane == 0) {
                        mbar_arrive_expect_tx(&raw_full[r], static_cast<uint32_t>(kTileRows * RS));
                        // byte offset of the chunk inside a row
                        const int64_t ob = static_cast<int64_t>(kb) * kBK / F::QK * F::BB;
                        for (int c = 0; c < g; ++c) {
                            const int mis = static_cast<int>((c * a.raw_rb) & 15);
                            const int x0 = static_cast<int>(((mis + ob) & ~static_cast<int64_t>(15)) >> 1);
                            tma_load_2d(slot + static_cast<size_t>(c) * rows_per_class * RS, &maps.w[gm].m[c],
                                        &raw_full[r], x0, static_cast<int32_t>(n0 / g));
                        }
                    }
                } else {
                    RowSpan sp[4];
                    uint32_t total = 0;
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int64_t n = n0 + lane + 32 * i;
                        if (n < a.g_N[gm]) {
                            sp[i] = row_span<QT>(n, a.K, static_cast<int64_t>(kb) * kBK,
                                                 static_cast<int64_t>(steps) * kBK);
                            total += sp[i].bytes;
                        } else {
                            sp[i].s0 = 0;
                            sp[i].bytes = 0;
                        }
                    }
#pragma unroll
                    for (int off = 16; off > 0; off >>= 1)
                        total += __shfl_xor_sync(0xFFFFFFFFu, total, off);
                    if (lane == 0)
                        mbar_arrive_expect_tx(&raw_full[r], total);
                    __syncwarp();
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        if (sp[i].bytes)
                            bulk_load(slot + static_cast<size_t>(lane + 32 * i) * RS, a.g_wq[gm] + sp[i].s0, sp[i].bytes,
                                      &raw_full[r]);
                }
                issued |= 1u << r;
                iparity = (iparity & ~(1u << r)) | (rphase << r);
                if (++r == R) {
                    r = 0;
                    rphase ^= 1u;
                }
            }
        }
        if (!ok && lane == 0) {
            volatile int no_abort = 0;
            for (int i = 0; i < R; ++i)
                if (issued & (1u << i))
                    mbar_wait_bounded(&raw_full[i], (iparity >> i) & 1u, &no_abort, a.status);
        }
    } else if (warp == 1 || warp == 3) {
        const int t = warp == 1 ? 0 : 1;   // issuer index
        if (lane == 0 && t < kIssuers) {
            // ---------------- MMA issuer t: A from TMEM, B (activations) from
            // shared memory.  Issuer t takes K steps [kSteps*t, kSteps*(t+1))
            // of every chunk (kSteps = 4 / kIssuers) into its own partial
            // accumulator and commits `done` once per chunk (the barrier
            // completes with one commit per issuer).
            constexpr uint32_t idesc = idesc_f16_f32(kTileRows, BN);
            constexpr int kSteps = kChunkSteps / kIssuers;
            int s = 0;
            uint32_t ph = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            for (int u = blockIdx.x; ok && u < a.units; u += gridDim.x) {
                const UnitInfo ui = unit_info(a, u);
                if (!mbar_wait_bounded(&tempty[acc], acc_phase ^ 1u, abort_flag, a.status))
                    break;
                const uint32_t d_tmem = tmem + static_cast<uint32_t>((acc * kIssuers + t) * BN);
                for (int kb = ui.kb0; kb < ui.kb1; kb += kChunkSteps) {
                    const int steps = ui.kb1 - kb < kChunkSteps ? ui.kb1 - kb : kChunkSteps;
                    if (!mbar_wait_bounded(&ready[s], ph, abort_flag, a.status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_tmem = tmem + kACol0 + static_cast<uint32_t>(s * kAStageCols);
                    const uint64_t b_desc = sdesc_k_sw128(smem_u32(sX + s * kXBytes));
                    const uint32_t acc_in = kb > ui.kb0 ? 1u : 0u;
                    const int st0 = kSteps * t;
                    if (steps == kChunkSteps) {
#pragma unroll
                        for (int k = 0; k < kSteps * (kBK / 16); ++k) {
                            const int kk = st0 * (kBK / 16) + k;
                            umma_f16_ta(d_tmem, a_tmem + static_cast<uint32_t>(kk * 8),
                                        b_desc + static_cast<uint64_t>(((kk >> 2) * kXSub + 32 * (kk & 3)) >> 4), idesc,
                                        k > 0 ? 1u : acc_in);
                        }
                    } else {
                        const int st1 = steps < st0 + kSteps ? steps : st0 + kSteps;
                        for (int kk = st0 * (kBK / 16); kk < st1 * (kBK / 16); ++kk)
                            umma_f16_ta(d_tmem, a_tmem + static_cast<uint32_t>(kk * 8),
                                        b_desc + static_cast<uint64_t>(((kk >> 2) * kXSub + 32 * (kk & 3)) >> 4), idesc,
                                        kk > st0 * (kBK / 16) ? 1u : acc_in);
                    }
                    umma_commit(&done[s]);
                    if (++s == S) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
                if (!ok)
                    break;
                umma_commit(&tfull[acc]);
                if (++acc == kNAcc) {
                    acc = 0;
                    acc_phase ^= 1u;
                }
            }
            umma_commit(&drain[t]);
            volatile int no_abort = 0;
            mbar_wait_bounded(&drain[t], 0, &no_abort, a.status);
        }
    } else if (warp == 2) {
        if (lane == 0) {
            // ---------------- activation-tile producer: chunk slot s is free
            // again once the MMAs that read it are done.  The activations may
            // come from the previous kernel on the stream; Y is written only
            // after MMAs that read them, so this wait also orders the stores.
            grid_dep_wait();
            int s = 0;
            uint32_t ph = 0;
            uint32_t issued = 0, iparity = 0;
            bool ok = true;
            for (int u = blockIdx.x; ok && u < a.units; u += gridDim.x) {
                const UnitInfo ui = unit_info(a, u);
                const int m0 = (ui.tile % a.m_tiles) * BN;
                for (int kb = ui.kb0; kb < ui.kb1; kb += kChunkSteps) {
                    const int steps = ui.kb1 - kb < kChunkSteps ? ui.kb1 - kb : kChunkSteps;
                    if (!mbar_wait_bounded(&done[s], ph ^ 1u, abort_flag, a.status)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&x_full[s], static_cast<uint32_t>(steps * kXSub));
                    for (int st = 0; st < steps; ++st)
                        tma_load_2d(sX + s * kXBytes + st * kXSub, &tm_x, &x_full[s], (kb + st) * kBK, m0);
                    issued |= 1u << s;
                    iparity = (iparity & ~(1u << s)) | (ph << s);
                    if (++s == S) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
            if (!ok) {
                volatile int no_abort = 0;
                for (int i = 0; i < S; ++i)
                    if (issued & (1u << i))
                        mbar_wait_bounded(&x_full[i], (iparity >> i) & 1u, &no_abort, a.status);
            }
        } else if (lane == 1) {
            // ---------------- announcer: in chunk order, once a slot's
            // activations have landed, the one extra arrival `ready` waits
            // for (the decoders never wait for X themselves).
            int s = 0;
            uint32_t ph = 0;
            bool ok = true;
            for (int u = blockIdx.x; ok && u < a.units; u += gridDim.x) {
                const UnitInfo ui = unit_info(a, u);
                for (int kb = ui.kb0; kb < ui.kb1; kb += kChunkSteps) {
                    if (!mbar_wait_bounded(&x_full[s], ph, abort_flag, a.status)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive(&ready[s]);
                    if (++s == S) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
        }
    } else if (warp >= 4 && warp < 8) {
        // ---------------- epilogue: warps 4..7 own TMEM lane quarters 0..3
        epilogue_role<BN, kNAcc, kIssuers>(a, tmem, tfull, tempty, abort_flag, warp, lane, kChunkSteps / kIssuers);
    } else if (warp >= kDecodeWarp0) {
        // ---------------- decoders: warp w holds weight rows 32*(w%4) .. +31
        // (the TMEM lanes it may access); group grp = dw / kWG decodes the
        // chunks c with c % kGroups == grp, and in them kSPT K steps from
        // j0 = kSPT*((dw % kWG)/4): thread (row, j0) writes the f16 of its row
        // for those steps into TMEM lane `row`, columns 32*j0 .. of the
        // chunk's A stage.
        const int dw = warp - kDecodeWarp0;
        const int row = (warp & 3) * 32 + lane;
        constexpr int kWG = kDecodeWarps / kGroups;   // warps decoding one chunk
        constexpr int kSPT = kChunkSteps * 4 / kWG;   // K steps per thread per chunk
        const int j0 = kSPT * ((dw % kWG) >> 2);
        const int grp = dw / kWG;
        int cc = 0;
        const uint32_t lane_base = static_cast<uint32_t>(row & ~31) << 16;
        // shared-memory row of this weight row inside a raw stage
        const int srow = TMA_RAW ? (row % g) * rows_per_class + row / g : row;
        const uint32_t raw_row0 = smem_u32(sR) + static_cast<uint32_t>(srow * RS);
        const uint32_t slot_bytes = static_cast<uint32_t>(kTileRows * RS);
        const uint32_t a_col0 = tmem + lane_base + kACol0 + static_cast<uint32_t>(32 * j0);
        // bytes of one 256-element chunk inside a row (K % 256 == 0)
        constexpr uint32_t kChunkRowBytes = kChunkSteps * kBK / F::QK * F::BB;
        int r = 0, s = 0;
        uint32_t rph = 0, ph = 0;
        bool ok = true;
        for (int u = blockIdx.x; ok && u < a.units; u += gridDim.x) {
            const UnitInfo ui = unit_info(a, u);
            const int nt = ui.tile / a.m_tiles;
            const int gm = group_of(a, nt);
            const int64_t n = static_cast<int64_t>(nt - a.g_tile0[gm]) * kTileRows + row;   // row inside member gm
            const bool valid = n < a.g_N[gm];
            // Tensor-map path: the slot row of a chunk starts at the 16-byte
            // boundary at or below the chunk's first byte, so the chunk sits
            // lead = (mis + ob) % 16 bytes into it, where mis is the row's
            // misalignment in its class map and ob the chunk's offset in the
            // row.  Rows past N read their zero-filled slot.
            uint32_t mis = 0, ob = 0;
            if (TMA_RAW) {
                mis = valid ? static_cast<uint32_t>(((n % g) * a.raw_rb) & 15) : 0u;
                ob = static_cast<uint32_t>(ui.kb0 / kChunkSteps) * kChunkRowBytes;
            }
            for (int kb = ui.kb0; ok && kb < ui.kb1; kb += kChunkSteps) {
                const int steps = ui.kb1 - kb < kChunkSteps ? ui.kb1 - kb : kChunkSteps;
                if (kGroups > 1 && (cc++ % kGroups) != grp) {   // the other group's chunk
                    if (TMA_RAW)
                        ob += kChunkRowBytes;
                    if (++s == S) {
                        s = 0;
                        ph ^= 1u;
                    }
                    if (++r == R) {
                        r = 0;
                        rph ^= 1u;
                    }
                    continue;
                }
                if (!__all_sync(0xFFFFFFFFu, mbar_wait_bounded(&raw_full[r], rph, abort_flag, a.status) &&
                                                 mbar_wait_bounded(&done[s], ph ^ 1u, abort_flag, a.status))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t raw_row = raw_row0 + static_cast<uint32_t>(r) * slot_bytes;
                const uint32_t a_col = a_col0 + static_cast<uint32_t>(s * kAStageCols);
                if (TMA_RAW && steps == kChunkSteps) {
                    const uint32_t blk = raw_row + ((mis + ob) & 15u);
#pragma unroll
                    for (int jj = 0; jj < kSPT; ++jj)
                        decode_step<QT>(blk, j0 + jj, a_col + 32 * jj);
                    ob += kChunkRowBytes;
                } else {
                    // Bulk-copy path: the slot row holds the stream from the
                    // 16-byte boundary at or below the chunk's first block.
                    const int64_t s0 =
                        valid ? row_span<QT>(n, a.K, static_cast<int64_t>(kb) * kBK, static_cast<int64_t>(steps) * kBK).s0
                              : 0;
#pragma unroll 1
                    for (int j = j0; j < j0 + kSPT && j < steps; ++j) {
#pragma unroll 1
                        for (int h = 0; h < 2; ++h) {
                            uint4 out[4] = {make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0),
                                            make_uint4(0, 0, 0, 0)};
                            if (valid) {
                                const int64_t es = n * a.K + static_cast<int64_t>(kb + j) * kBK + 32 * h;
                                const int64_t blk = es / F::QK;
                                const int o = static_cast<int>(es - blk * F::QK);
                                decode32<QT>(raw_row + static_cast<uint32_t>(blk * F::BB - s0), o, out);
                            }
                            __syncwarp();
                            tmem_st_32x32b_x16(a_col + static_cast<uint32_t>(32 * (j - j0) + 16 * h), out);
                        }
                    }
                }
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&raw_empty[r]);
                    mbar_arrive(&ready[s]);
                }
                if (++s == S) {
                    s = 0;
                    ph ^= 1u;
                }
                if (++r == R) {
                    r = 0;
                    rph ^= 1u;
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

struct FusedLayout {
    int rs, x_stages, raw_stages, smem;
};

int qk_of(int qt) { return (qt == 12 || qt == 13 || qt == 14) ? 256 : 32; }
int bb_of(int qt)
{
    switch (qt) {
    case 2: return 18;
    case 6: return 22;
    case 7: return 24;
    case 8: return 34;
    case 12: return 144;
    case 13: return 176;
    default: return 210;
    }
}

// Row pitch of a raw stage: at least `bytes`, an odd multiple of 16.  The
// 32 lanes of a decoder warp read the same offset of 32 consecutive slot
// rows; an odd number of 16-byte units per row puts the 8 lanes of each
// 16-byte load phase on 8 distinct bank quads (no conflict) and spreads
// 4-byte loads over 8 banks (4-way at worst).  An even count can put a
// whole warp on 2 banks (a 192-byte pitch: 16-way).
int odd16(int bytes)
{
    const int u = (bytes + 15) / 16;
    return 16 * (u | 1);
}

// Bytes per row of a raw stage on the tensor-map path (the box width): one
// 256-element chunk plus the leading misalignment (only Q6_K chunks start
// off a 16-byte boundary, by up to 14 bytes), padded to an odd multiple of
// 16.  Box bytes past the chunk are the row's next bytes or the map's zero
// fill, and are not decoded.
int tma_rs_of(int qt)
{
    const int chunk = 256 / qk_of(qt) * bb_of(qt);
    return odd16(chunk + (qt == 14 ? 14 : 0));
}

// Shared-memory plan: per-row raw slot size and the depth of the raw ring
// within 227 KB (the f16 weight operand lives in TMEM; the activation ring
// has one slot per A stage).  The raw ring takes what is left, up to 8
// chunks: under load a raw chunk takes ~3 us from issue to arrival, and the
// chunks in flight per SM set the stream rate.
FusedLayout fused_layout(int qt, int bn, bool tma_raw)
{
    FusedLayout L{};
    if (tma_raw) {
        L.rs = tma_rs_of(qt);
    } else {
        // A 256-element chunk of a row whose start is a multiple of 64
        // elements touches 256/QK blocks (QK = 32) or up to 2 (QK = 256);
        // the first block may sit up to 14 bytes into its 16-byte line.
        const int span = (qk_of(qt) == 32) ? 8 : 2;
        const int mis = (bb_of(qt) % 16 == 0) ? 0 : 14;
        L.rs = odd16(span * bb_of(qt) + mis);
    }
    const int xb = kChunkSteps * bn * kBK * 2;   // one chunk of activations
    const int raw = kTileRows * L.rs;
    const int budget = kSmemLimit - 1024 - kBarBytes;
    L.x_stages = a_stages_for(bn);
    L.raw_stages = kMaxRaw;
    while (L.x_stages * xb + L.raw_stages * raw > budget) {
        if (L.raw_stages == 1)
            return FusedLayout{};
        --L.raw_stages;   // one stage only for wide raw slots (rows starting inside blocks) at BN = 128
    }
    L.smem = 1024 + L.x_stages * xb + L.raw_stages * raw + kBarBytes;
    return L;
}

template <int BN, int QT, bool TMA_RAW>
cudaError_t launch_f(const CUtensorMap &tx, const RawMapsG &maps, const GemmArgs &a0, const GemmPlan &p,
                     cudaStream_t s)
{
    const FusedLayout L = fused_layout(QT, BN, TMA_RAW);
    if (L.smem == 0)
        return cudaErrorInvalidConfiguration;
    GemmArgs a = a0;
    a.raw_rs = L.rs;
    a.a_stages = L.x_stages;
    a.x_stages = L.x_stages;
    a.raw_stages = L.raw_stages;
    static bool attr_done[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 0 || dev >= 64 || !attr_done[dev]) {
        e = cudaFuncSetAttribute(k_gemm_fused<BN, QT, TMA_RAW>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kSmemLimit);
        if (e != cudaSuccess)
            return e;
        if (dev >= 0 && dev < 64)
            attr_done[dev] = true;
    }
    e = launch_kernel(k_gemm_fused<BN, QT, TMA_RAW>, dim3(p.grid), dim3(kThreadsF), L.smem, s, tx, maps, a);
    note_launch();
    return e;
}

template <int QT, bool TMA_RAW>
cudaError_t launch_q(const CUtensorMap &tx, const RawMapsG &maps, const GemmArgs &a, const GemmPlan &p,
                     cudaStream_t s)
{
    switch (p.bn) {
    case 128: return launch_f<128, QT, TMA_RAW>(tx, maps, a, p, s);
    case 64: return launch_f<64, QT, TMA_RAW>(tx, maps, a, p, s);
    case 32: return launch_f<32, QT, TMA_RAW>(tx, maps, a, p, s);
    case 16: return launch_f<16, QT, TMA_RAW>(tx, maps, a, p, s);
    default: return cudaErrorInvalidValue;
    }
}

typedef CUresult (*PFN_encodeTiledF)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                     const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                     CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

PFN_encodeTiledF encoder()
{
    static PFN_encodeTiledF fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_encodeTiledF>(p);
    }
    return fn;
}

}  // namespace

int encode_raw_maps(RawMaps *maps, const void *qdata, int type, int64_t N, int64_t K)
{
    if (K % 256 != 0 || (type != 2 && type != 6 && type != 7 && type != 8 && type != 12 && type != 13 && type != 14))
        return 0;
    PFN_encodeTiledF fn = encoder();
    if (!fn)
        return 0;
    const int64_t rb = K / qk_of(type) * bb_of(type);
    int g = 1;
    while ((g * rb) % 16 != 0)
        g *= 2;                                   // rb is even, so g <= 8
    const int box_bytes = tma_rs_of(type);
    for (int c = 0; c < g; ++c) {
        const int64_t rows = (N - c + g - 1) / g;   // rows n = c, c+g, ... < N
        if (rows <= 0) {
            maps->m[c] = maps->m[0];
            continue;
        }
        const int64_t mis = (c * rb) % 16;
        const uint8_t *base = static_cast<const uint8_t *>(qdata) + c * rb - mis;
        const cuuint64_t dims[2] = {static_cast<cuuint64_t>((rb + mis) / 2), static_cast<cuuint64_t>(rows)};
        const cuuint64_t strides[1] = {static_cast<cuuint64_t>(g * rb)};
        const cuuint32_t box[2] = {static_cast<cuuint32_t>(box_bytes / 2), static_cast<cuuint32_t>(kTileRows / g)};
        const cuuint32_t estr[2] = {1, 1};
        if (fn(&maps->m[c], CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<uint8_t *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return 0;
    }
    return g;
}

cudaError_t launch_gemm_fused(const CUtensorMap &tx, const RawMapsG &maps, const GemmArgs &a, const GemmPlan &p,
                              cudaStream_t s)
{
    if (a.K % kBK != 0 || p.kb_align != kChunkSteps)
        return cudaErrorInvalidValue;
    const bool tma = a.raw_g > 0;
    switch (a.qtype) {
    case 2: return tma ? launch_q<2, true>(tx, maps, a, p, s) : launch_q<2, false>(tx, maps, a, p, s);
    case 6: return tma ? launch_q<6, true>(tx, maps, a, p, s) : launch_q<6, false>(tx, maps, a, p, s);
    case 7: return tma ? launch_q<7, true>(tx, maps, a, p, s) : launch_q<7, false>(tx, maps, a, p, s);
    case 8: return tma ? launch_q<8, true>(tx, maps, a, p, s) : launch_q<8, false>(tx, maps, a, p, s);
    case 13: return tma ? launch_q<13, true>(tx, maps, a, p, s) : launch_q<13, false>(tx, maps, a, p, s);
    case 12: return tma ? launch_q<12, true>(tx, maps, a, p, s) : launch_q<12, false>(tx, maps, a, p, s);
    case 14: return tma ? launch_q<14, true>(tx, maps, a, p, s) : launch_q<14, false>(tx, maps, a, p, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace mq
