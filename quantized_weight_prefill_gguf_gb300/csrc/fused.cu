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
//   warp 1      TMEM allocation and the MMA issuer (one thread): per raw
//               chunk one wait for its A stage and X stage, then sixteen
//               unrolled M=128 x N=BN x K=16 MMAs with A in TMEM.  This
//               thread shares its SM sub-partition with decode warps, so it
//               spends as few instructions per MMA as possible.
//   warp 2      activation producer (TMA): the BN x 256 activations of a
//               chunk (four 64-wide boxes) per stage, up to x_stages ahead.
//   warps 4-7   epilogue (TMEM -> Y / split-K workspace).
//   warps 8-15  decoders: thread (row, half) turns 32 raw elements of one
//               weight row per K step into 16 packed f16 words and stores
//               them with tcgen05.st into its row's TMEM lane; one barrier
//               round trip per 256-element chunk.
#include <cstdint>
#include <cuda_runtime.h>

#include "mq_decode.cuh"
#include "mq_internal.h"
#include "mq_ptx.cuh"
#include "mq_smem.cuh"
#include "mq_tile.cuh"

namespace mq {
namespace {

constexpr int kThreadsF = 512;
constexpr int kDecodeWarp0 = 8;
constexpr int kDecodeWarps = 8;
constexpr int kChunkSteps = 4;               // K steps (of 64) per raw stage: 256 K elements
constexpr int kMaxX = 4, kMaxRaw = 4;
// TMEM: accumulators in columns [0, 256), two A stages of 128 columns (one
// raw chunk of 256 K elements, two f16 per column) in [256, 512).
constexpr int kTmemCols = 512;
constexpr uint32_t kACol0 = 256;
constexpr int kAStages = 2;
constexpr int kAStageCols = 128;
constexpr int kSmemLimit = 227 * 1024;
constexpr int kBarBytes = 512;

template <int QT> struct QF;
template <> struct QF<8> { static constexpr int QK = 32, BB = 34; };
template <> struct QF<12> { static constexpr int QK = 256, BB = 144; };
template <> struct QF<14> { static constexpr int QK = 256, BB = 210; };

// Shared-memory bytes per row of a raw stage on the tensor-map path: one
// 256-element chunk plus up to 14 bytes of leading misalignment, rounded to
// 16 (Q4_K chunks are always aligned).
template <int QT> constexpr int tma_row_bytes()
{
    return QT == 12 ? 144 : (QT == 14 ? 224 : 272);
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

// Block-aligned weights (K % 256 == 0): one raw chunk of a row is 256
// consecutive elements starting on a block boundary -- one Q4_K or Q6_K
// block, or eight Q8_0 blocks -- at `b` (the row's slot plus its leading
// misalignment).  These decode the thread's 4 x 32 elements of the chunk
// (K step st covers elements 64*st + 32*half .. +31) fully unrolled and store
// each group of 32 into TMEM columns col + 32*st .. +15.  Rows past the
// weight's end (valid == false) store zeros.  tcgen05.st is .sync.aligned:
// every lane of the warp must reach the same store, so the stores sit
// outside any lane-dependent branch.

__device__ __forceinline__ void store_step(uint32_t taddr, uint4 (&out)[4], bool valid)
{
    if (!valid) {
#pragma unroll
        for (int j = 0; j < 4; ++j)
            out[j] = make_uint4(0, 0, 0, 0);
    }
    __syncwarp();
    tmem_st_32x32b_x16(taddr, out);
}

template <int QT>
__device__ __forceinline__ void decode_chunk(uint32_t b, int half, uint32_t col, bool valid);

template <>
__device__ __forceinline__ void decode_chunk<12>(uint32_t b, int half, uint32_t col, bool valid)
{
    // Q4_K, b 16-byte aligned.  Step st is group p = st: sub-block 2*st+half,
    // nibbles (low for half 0, high for half 1) of qs bytes 32*st .. +31.
    const uint4 hdr = lds_v4(b);
    const float d = f16_bits_to_f32(hdr.x), dmin = f16_bits_to_f32(hdr.x >> 16);
    const int sh = 4 * half;
#pragma unroll
    for (int st = 0; st < 4; ++st) {
        int sc, m;
        q4k_scale_min(hdr.y, hdr.z, hdr.w, 2 * st + half, sc, m);
        const float A = __fmul_rn(d, static_cast<float>(sc)), B = __fmul_rn(dmin, static_cast<float>(m));
        const uint4 q0 = lds_v4(b + 16 + 32 * st), q1 = lds_v4(b + 32 + 32 * st);
        uint4 out[4];
        out[0] = q4k_eight(A, B, q0.x, q0.y, sh);
        out[1] = q4k_eight(A, B, q0.z, q0.w, sh);
        out[2] = q4k_eight(A, B, q1.x, q1.y, sh);
        out[3] = q4k_eight(A, B, q1.z, q1.w, sh);
        store_step(col + 32 * st, out, valid);
    }
}

template <>
__device__ __forceinline__ void decode_chunk<14>(uint32_t b, int half, uint32_t col, bool valid)
{
    // Q6_K, b 2-byte aligned.  Step st covers quarter t = (2*st+half) & 3 of
    // block half hh = st >> 1: low bits from ql bytes 64*hh + 32*half .. +31
    // (low nibble for even st, high for odd), high bits from qh bytes
    // 32*hh .. +31 (bits 2t), scales sc[4*st + 2*half], sc[4*st + 2*half + 1].
    const float d = f16_bits_to_f32(lds_u16(b + 208));
    uint32_t lq[2][8], hq[2][8];
    lds_32B_a2(b + 32 * half, lq[0]);
    lds_32B_a2(b + 64 + 32 * half, lq[1]);
    lds_32B_a2(b + 128, hq[0]);
    lds_32B_a2(b + 160, hq[1]);
#pragma unroll
    for (int st = 0; st < 4; ++st) {
        const int hh = st >> 1, t = (2 * st + half) & 3;
        const int lsh = (st & 1) ? 4 : 0, hsh = 2 * t;
        const int si = 4 * st + 2 * half;
        const float A0 = __fmul_rn(d, static_cast<float>(lds_s8(b + 192 + si)));
        const float A1 = __fmul_rn(d, static_cast<float>(lds_s8(b + 193 + si)));
        uint4 out[4];
        out[0] = q6k_eight(A0, lq[hh][0], lq[hh][1], lsh, hq[hh][0], hq[hh][1], hsh);
        out[1] = q6k_eight(A0, lq[hh][2], lq[hh][3], lsh, hq[hh][2], hq[hh][3], hsh);
        out[2] = q6k_eight(A1, lq[hh][4], lq[hh][5], lsh, hq[hh][4], hq[hh][5], hsh);
        out[3] = q6k_eight(A1, lq[hh][6], lq[hh][7], lsh, hq[hh][6], hq[hh][7], hsh);
        store_step(col + 32 * st, out, valid);
    }
}

template <>
__device__ __forceinline__ void decode_chunk<8>(uint32_t b, int half, uint32_t col, bool valid)
{
    // Q8_0: step st is the whole block 2*st + half (34 bytes, 2-byte aligned).
#pragma unroll
    for (int st = 0; st < 4; ++st) {
        const uint32_t blk = b + 34 * (2 * st + half);
        const uint32_t d16 = lds_u16(blk);
        uint32_t q[8];
        lds_32B_a2(blk + 2, q);
        uint4 out[4];
#pragma unroll
        for (int j = 0; j < 4; ++j)
            out[j] = q80_eight(d16, q[2 * j], q[2 * j + 1]);
        store_step(col + 32 * st, out, valid);
    }
}

template <int BN, int QT, bool TMA_RAW>
__global__ void __launch_bounds__(kThreadsF, 1)
    k_gemm_fused(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ RawMaps maps, const GemmArgs a)
{
    using F = QF<QT>;
    constexpr int kXSub = BN * kBK * 2;               // one 64-wide K step of activations
    constexpr int kXBytes = kChunkSteps * kXSub;      // one X stage: a whole 256-element chunk
    constexpr int kNAcc = 2;                          // accumulators at TMEM columns [0, 2*BN)
    static_assert(BN <= 128, "fused tiles stop at 128 tokens");
    const int SX = a.x_stages, R = a.raw_stages, RS = a.raw_rs;

    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t *sX = base;
    uint8_t *sR = sX + SX * kXBytes;
    uint64_t *bars = reinterpret_cast<uint64_t *>(sR + static_cast<size_t>(R) * kTileRows * RS);
    uint64_t *raw_full = bars;
    uint64_t *raw_empty = raw_full + kMaxRaw;
    uint64_t *x_full = raw_empty + kMaxRaw;
    uint64_t *x_empty = x_full + kMaxX;
    uint64_t *a_full = x_empty + kMaxX;
    uint64_t *a_empty = a_full + kAStages;
    uint64_t *tfull = a_empty + kAStages;
    uint64_t *tempty = tfull + 2;
    uint64_t *drain = tempty + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = TMA_RAW ? a.raw_g : 1;
    const int rows_per_class = kTileRows / g;

    if (threadIdx.x == 0) {
        for (int r = 0; r < R; ++r) {
            mbar_init(&raw_full[r], 1);
            mbar_init(&raw_empty[r], kDecodeWarps);
        }
        for (int s = 0; s < SX; ++s) {
            mbar_init(&x_full[s], 1);
            mbar_init(&x_empty[s], 1);
        }
        for (int s = 0; s < kAStages; ++s) {
            mbar_init(&a_full[s], kDecodeWarps);
            mbar_init(&a_empty[s], 1);
        }
        for (int i = 0; i < kNAcc; ++i) {
            mbar_init(&tfull[i], 1);
            mbar_init(&tempty[i], 4);
        }
        mbar_init(drain, 1);
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
            for (int c = 0; c < g; ++c)
                prefetch_tensormap(&maps.m[c]);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ---------------- raw producer
        int r = 0;
        uint32_t rphase = 0;
        uint32_t issued = 0, iparity = 0;
        bool ok = a.stall_producer == 0;
        for (int u = blockIdx.x; ok && u < a.units; u += gridDim.x) {
            const UnitInfo ui = unit_info(a, u);
            const int64_t n0 = static_cast<int64_t>(ui.tile / a.m_tiles) * kTileRows;
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
                            tma_load_2d(slot + static_cast<size_t>(c) * rows_per_class * RS, &maps.m[c],
                                        &raw_full[r], x0, static_cast<int32_t>(n0 / g));
                        }
                    }
                } else {
                    RowSpan sp[4];
                    uint32_t total = 0;
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int64_t n = n0 + lane + 32 * i;
                        if (n < a.N) {
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
                            bulk_load(slot + static_cast<size_t>(lane + 32 * i) * RS, a.wq + sp[i].s0, sp[i].bytes,
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
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------- MMA issuer: A from TMEM, B (activations) from shared memory
            constexpr uint32_t idesc = idesc_f16_f32(kTileRows, BN);
            int sa = 0, sx = 0;
            uint32_t pa = 0, px = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            for (int u = blockIdx.x; ok && u < a.units; u += gridDim.x) {
                const UnitInfo ui = unit_info(a, u);
                if (!mbar_wait_bounded(&tempty[acc], acc_phase ^ 1u, abort_flag, a.status))
                    break;
                tc_fence_after();
                const uint32_t d_tmem = tmem + static_cast<uint32_t>(acc * BN);
                for (int kb = ui.kb0; ok && kb < ui.kb1; kb += kChunkSteps) {
                    const int steps = ui.kb1 - kb < kChunkSteps ? ui.kb1 - kb : kChunkSteps;
                    if (!mbar_wait_bounded(&a_full[sa], pa, abort_flag, a.status) ||
                        !mbar_wait_bounded(&x_full[sx], px, abort_flag, a.status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_tmem = tmem + kACol0 + static_cast<uint32_t>(sa * kAStageCols);
                    const uint64_t b_desc = sdesc_k_sw128(smem_u32(sX + sx * kXBytes));
                    const uint32_t acc_in = kb > ui.kb0 ? 1u : 0u;
                    if (steps == kChunkSteps) {
#pragma unroll
                        for (int st = 0; st < kChunkSteps; ++st)
#pragma unroll
                            for (int k = 0; k < kBK / 16; ++k)
                                umma_f16_ta(d_tmem, a_tmem + static_cast<uint32_t>(st * 32 + k * 8),
                                            b_desc + static_cast<uint64_t>((st * kXSub + 32 * k) >> 4), idesc,
                                            (st > 0 || k > 0) ? 1u : acc_in);
                    } else {
                        for (int st = 0; st < steps; ++st)
#pragma unroll
                            for (int k = 0; k < kBK / 16; ++k)
                                umma_f16_ta(d_tmem, a_tmem + static_cast<uint32_t>(st * 32 + k * 8),
                                            b_desc + static_cast<uint64_t>((st * kXSub + 32 * k) >> 4), idesc,
                                            (st > 0 || k > 0) ? 1u : acc_in);
                    }
                    umma_commit(&a_empty[sa]);
                    umma_commit(&x_empty[sx]);
                    if (++sa == kAStages) {
                        sa = 0;
                        pa ^= 1u;
                    }
                    if (++sx == SX) {
                        sx = 0;
                        px ^= 1u;
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
            umma_commit(drain);
            volatile int no_abort = 0;
            mbar_wait_bounded(drain, 0, &no_abort, a.status);
        }
    } else if (warp == 2) {
        if (lane == 0) {
            // ---------------- activation-tile producer
            int s = 0;
            uint32_t ph = 0;
            uint32_t issued = 0, iparity = 0;
            bool ok = true;
            for (int u = blockIdx.x; ok && u < a.units; u += gridDim.x) {
                const UnitInfo ui = unit_info(a, u);
                const int m0 = (ui.tile % a.m_tiles) * BN;
                for (int kb = ui.kb0; kb < ui.kb1; kb += kChunkSteps) {
                    const int steps = ui.kb1 - kb < kChunkSteps ? ui.kb1 - kb : kChunkSteps;
                    if (!mbar_wait_bounded(&x_empty[s], ph ^ 1u, abort_flag, a.status)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&x_full[s], static_cast<uint32_t>(steps * kXSub));
                    for (int st = 0; st < steps; ++st)
                        tma_load_2d(sX + s * kXBytes + st * kXSub, &tm_x, &x_full[s], (kb + st) * kBK, m0);
                    issued |= 1u << s;
                    iparity = (iparity & ~(1u << s)) | (ph << s);
                    if (++s == SX) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
            if (!ok) {
                volatile int no_abort = 0;
                for (int i = 0; i < SX; ++i)
                    if (issued & (1u << i))
                        mbar_wait_bounded(&x_full[i], (iparity >> i) & 1u, &no_abort, a.status);
            }
        }
    } else if (warp >= 4 && warp < 8) {
        // ---------------- epilogue: warps 4..7 own TMEM lane quarters 0..3
        epilogue_role<BN, kNAcc>(a, tmem, tfull, tempty, abort_flag, warp, lane);
    } else if (warp >= kDecodeWarp0) {
        // ---------------- decoders: thread (row, half) writes, for each 64-wide
        // K step of a raw chunk, 32 f16 of its row into TMEM lane `row`,
        // columns (step*32 + half*16) .. +15 of the chunk's A stage.  Warp w
        // holds rows 32*(w%4) .. +31, the TMEM lanes it may access.
        const int dt = threadIdx.x - kDecodeWarp0 * 32;
        const int row = dt & (kTileRows - 1);
        const int half = dt >> 7;
        const uint32_t lane_base = static_cast<uint32_t>(row & ~31) << 16;
        // shared-memory row of this weight row inside a raw stage
        const int srow = TMA_RAW ? (row % g) * rows_per_class + row / g : row;
        int r = 0, sa = 0;
        uint32_t rph = 0, pa = 0;
        bool ok = true;
        for (int u = blockIdx.x; ok && u < a.units; u += gridDim.x) {
            const UnitInfo ui = unit_info(a, u);
            const int64_t n = static_cast<int64_t>(ui.tile / a.m_tiles) * kTileRows + row;
            const bool valid = n < a.N;
            for (int kb = ui.kb0; ok && kb < ui.kb1; kb += kChunkSteps) {
                const int steps = ui.kb1 - kb < kChunkSteps ? ui.kb1 - kb : kChunkSteps;
                if (!__all_sync(0xFFFFFFFFu, mbar_wait_bounded(&raw_full[r], rph, abort_flag, a.status) &&
                                                 mbar_wait_bounded(&a_empty[sa], pa ^ 1u, abort_flag, a.status))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                // Byte position in the stream that shared-memory byte 0 of
                // this row's raw slot holds.
                int64_t s0 = 0;
                if (TMA_RAW) {
                    const int64_t ob = static_cast<int64_t>(kb) * kBK / F::QK * F::BB;
                    const int64_t mis = ((n % g) * a.raw_rb) & 15;
                    s0 = n * a.raw_rb - mis + ((mis + ob) & ~static_cast<int64_t>(15));
                } else if (valid) {
                    s0 = row_span<QT>(n, a.K, static_cast<int64_t>(kb) * kBK, static_cast<int64_t>(steps) * kBK).s0;
                }
                const uint32_t raw_row =
                    smem_u32(sR + static_cast<size_t>(r) * kTileRows * RS + static_cast<size_t>(srow) * RS);
                const uint32_t a_col = tmem + lane_base + kACol0 + static_cast<uint32_t>(sa * kAStageCols + half * 16);
                if (TMA_RAW && steps == kChunkSteps) {
                    // The chunk's first block sits (mis + ob) % 16 bytes into
                    // the slot.  Rows past N read their (zero-filled) slot and
                    // store zeros.
                    const uint32_t lead = valid ? static_cast<uint32_t>(n * a.raw_rb +
                                                                        static_cast<int64_t>(kb) * kBK / F::QK * F::BB - s0)
                                                : 0u;
                    decode_chunk<QT>(raw_row + lead, half, a_col, valid);
                } else for (int st = 0; st < steps; ++st) {
                    uint4 out[4] = {make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0),
                                    make_uint4(0, 0, 0, 0)};
                    if (valid) {
                        const int64_t es = n * a.K + static_cast<int64_t>(kb + st) * kBK + 32 * half;
                        const int64_t blk = es / F::QK;
                        const int o = static_cast<int>(es - blk * F::QK);
                        decode32<QT>(raw_row + static_cast<uint32_t>(blk * F::BB - s0), o, out);
                    }
                    __syncwarp();
                    tmem_st_32x32b_x16(a_col + static_cast<uint32_t>(st * 32), out);
                }
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&a_full[sa]);
                    mbar_arrive(&raw_empty[r]);
                }
                if (++sa == kAStages) {
                    sa = 0;
                    pa ^= 1u;
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

int qk_of(int qt) { return qt == 8 ? 32 : 256; }
int bb_of(int qt) { return qt == 8 ? 34 : (qt == 12 ? 144 : 210); }

// Shared-memory plan: per-row raw slot size and the depth of the raw and
// activation rings within 227 KB (the f16 weight operand lives in TMEM).
// Preferred depths: raw 4 chunks (1024 K elements ahead), activations
// 4/4/3/2 chunks for BN = 16/32/64/128; the larger ring gives way first.
FusedLayout fused_layout(int qt, int bn, bool tma_raw)
{
    FusedLayout L{};
    if (tma_raw) {
        L.rs = qt == 12 ? 144 : (qt == 14 ? 224 : 272);
    } else {
        // A 256-element chunk of a row whose start is a multiple of 64
        // elements touches 256/QK blocks (QK = 32) or up to 2 (QK = 256);
        // the first block may sit up to 14 bytes into its 16-byte line.
        const int span = (qk_of(qt) == 32) ? 8 : 2;
        const int mis = (bb_of(qt) % 16 == 0) ? 0 : 14;
        L.rs = (span * bb_of(qt) + mis + 15) / 16 * 16;
    }
    const int xb = kChunkSteps * bn * kBK * 2;   // one chunk of activations
    const int raw = kTileRows * L.rs;
    const int budget = kSmemLimit - 1024 - kBarBytes;
    L.x_stages = bn <= 32 ? 4 : (bn <= 64 ? 3 : 2);
    L.raw_stages = kMaxRaw;
    auto total = [&] { return L.x_stages * xb + L.raw_stages * raw; };
    while (total() > budget) {
        if (L.raw_stages > 2 && L.raw_stages * raw >= L.x_stages * xb)
            --L.raw_stages;
        else if (L.x_stages > 2)
            --L.x_stages;
        else if (L.raw_stages > 2)
            --L.raw_stages;
        else if (L.x_stages > 1)
            --L.x_stages;   // wide raw slots (rows starting inside blocks) at BN = 128
        else
            return FusedLayout{};
    }
    L.smem = 1024 + total() + kBarBytes;
    return L;
}

template <int BN, int QT, bool TMA_RAW>
cudaError_t launch_f(const CUtensorMap &tx, const RawMaps &maps, const GemmArgs &a0, const GemmPlan &p,
                     cudaStream_t s)
{
    const FusedLayout L = fused_layout(QT, BN, TMA_RAW);
    if (L.smem == 0)
        return cudaErrorInvalidConfiguration;
    GemmArgs a = a0;
    a.raw_rs = L.rs;
    a.a_stages = kAStages;
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
    k_gemm_fused<BN, QT, TMA_RAW><<<p.grid, kThreadsF, L.smem, s>>>(tx, maps, a);
    note_launch();
    return cudaGetLastError();
}

template <int QT, bool TMA_RAW>
cudaError_t launch_q(const CUtensorMap &tx, const RawMaps &maps, const GemmArgs &a, const GemmPlan &p,
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
    if (K % 256 != 0 || (type != 8 && type != 12 && type != 14))
        return 0;
    PFN_encodeTiledF fn = encoder();
    if (!fn)
        return 0;
    const int64_t rb = K / qk_of(type) * bb_of(type);
    int g = 1;
    while ((g * rb) % 16 != 0)
        g *= 2;                                   // rb is even, so g <= 8
    const int box_bytes = type == 12 ? 144 : (type == 14 ? 224 : 272);
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

cudaError_t launch_gemm_fused(const CUtensorMap &tx, const RawMaps &maps, const GemmArgs &a, const GemmPlan &p,
                              cudaStream_t s)
{
    if (a.K % kBK != 0 || p.kb_align != kChunkSteps)
        return cudaErrorInvalidValue;
    const bool tma = a.raw_g > 0;
    switch (a.qtype) {
    case 8: return tma ? launch_q<8, true>(tx, maps, a, p, s) : launch_q<8, false>(tx, maps, a, p, s);
    case 12: return tma ? launch_q<12, true>(tx, maps, a, p, s) : launch_q<12, false>(tx, maps, a, p, s);
    case 14: return tma ? launch_q<14, true>(tx, maps, a, p, s) : launch_q<14, false>(tx, maps, a, p, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace mq
