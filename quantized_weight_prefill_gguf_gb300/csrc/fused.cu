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
// from.  Warp roles (512 threads):
//   warp 0      raw producer: for each weight row of the tile, one 1-D bulk
//               copy (cp.async.bulk) of the 16-byte-aligned byte range that
//               holds the row's blocks for 256 K elements, into a ring of
//               raw stages.  Q6_K (210 B) and Q8_0 (34 B) blocks are only
//               2-byte aligned; copying the aligned superset keeps every
//               global access aligned, and the decoders read the bytes at
//               their real offsets from shared memory.
//   warp 1      TMEM allocation and the MMA issuer (one thread).
//   warp 2      TMA producer of the activation tile (BN x 64, 128-byte swizzle).
//   warps 4-7   epilogue (TMEM -> Y / split-K workspace).
//   warps 8-15  decoders: thread (row, half) turns 32 raw elements of one
//               weight row into four 16-byte f16 chunks, stored in the
//               128-byte-swizzled K-major layout the MMA descriptor reads,
//               then fences the generic->async proxy and arrives.
// The raw ring runs up to 4 x 256 K elements ahead of the MMA, which is what
// keeps enough bytes in flight at small M, where this kernel is bound by
// HBM and by the decode ALU rather than by the tensor cores.
#include <cstdint>
#include <cuda_runtime.h>

#include "mq_decode.cuh"
#include "mq_internal.h"
#include "mq_ptx.cuh"
#include "mq_tile.cuh"

namespace mq {
namespace {

constexpr int kThreadsF = 512;
constexpr int kDecodeWarp0 = 8;
constexpr int kDecodeWarps = 8;
constexpr int kChunkSteps = 4;               // K steps (of 64) per raw stage: 256 K elements
constexpr int kMaxStages = 4;
constexpr int kMaxRaw = 4;
constexpr int kSmemLimit = 227 * 1024;

template <int QT> struct QF;
template <> struct QF<8> { static constexpr int QK = 32, BB = 34; };
template <> struct QF<12> { static constexpr int QK = 256, BB = 144; };
template <> struct QF<14> { static constexpr int QK = 256, BB = 210; };

struct RowSpan {
    int64_t s0;       // 16-byte-aligned start of the copied range in the stream
    uint32_t bytes;   // multiple of 16
};

// Byte range of the stream holding flat elements [n*K + kc0, n*K + kc0 + len),
// widened to 16-byte boundaries.  The stream's length is a multiple of 16
// (checked on the host), so the widened end never passes it.
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

// Decode 32 consecutive elements starting at element o of the block at
// shared address b into out[0..3] (8 f16 each).
template <int QT>
__device__ __forceinline__ void decode32(uint32_t b, int o, uint4 (&out)[4]);

template <>
__device__ __forceinline__ void decode32<12>(uint32_t b, int o, uint4 (&out)[4])
{
    // Q4_K: b is 16-byte aligned (blocks are 144 B and copies start on a block).
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
    const float d = f16_bits_to_f32(lds_u16(b));
    uint32_t q[8];
    lds_32B_a2(b + 2, q);
#pragma unroll
    for (int j = 0; j < 4; ++j)
        out[j] = q80_eight(d, q[2 * j], q[2 * j + 1]);
}

template <int BN, int QT>
__global__ void __launch_bounds__(kThreadsF, 1)
    k_gemm_fused(const __grid_constant__ CUtensorMap tm_x, const GemmArgs a)
{
    using F = QF<QT>;
    constexpr int kXBytes = BN * kBK * 2;
    constexpr int kTmemCols = 2 * BN;
    const int S = a.stages, R = a.raw_stages, RS = a.raw_rs;

    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t *sA = base;
    uint8_t *sX = sA + S * kABytes;
    uint8_t *sR = sX + S * kXBytes;
    uint64_t *bars = reinterpret_cast<uint64_t *>(sR + static_cast<size_t>(R) * kTileRows * RS);
    uint64_t *raw_full = bars;
    uint64_t *raw_empty = bars + kMaxRaw;
    uint64_t *x_full = raw_empty + kMaxRaw;
    uint64_t *a_full = x_full + kMaxStages;
    uint64_t *s_empty = a_full + kMaxStages;
    uint64_t *tfull = s_empty + kMaxStages;
    uint64_t *tempty = tfull + 2;
    uint64_t *drain = tempty + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int r = 0; r < R; ++r) {
            mbar_init(&raw_full[r], 1);
            mbar_init(&raw_empty[r], kDecodeWarps);
        }
        for (int s = 0; s < S; ++s) {
            mbar_init(&x_full[s], 1);
            mbar_init(&a_full[s], kDecodeWarps);
            mbar_init(&s_empty[s], 1);
        }
        for (int i = 0; i < 2; ++i) {
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
    if (warp == 2 && lane == 0)
        prefetch_tensormap(&tm_x);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ---------------- raw producer (whole warp: 4 rows per lane)
        int r = 0;
        uint32_t rphase = 0;
        uint32_t issued = 0, iparity = 0;
        bool ok = true;
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
                RowSpan sp[4];
                uint32_t total = 0;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int64_t n = n0 + lane + 32 * i;
                    if (n < a.N) {
                        sp[i] = row_span<QT>(n, a.K, static_cast<int64_t>(kb) * kBK, static_cast<int64_t>(steps) * kBK);
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
                uint8_t *slot = sR + static_cast<size_t>(r) * kTileRows * RS;
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    if (sp[i].bytes)
                        bulk_load(slot + static_cast<size_t>(lane + 32 * i) * RS, a.wq + sp[i].s0, sp[i].bytes,
                                  &raw_full[r]);
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
            // ---------------- MMA issuer
            constexpr uint32_t idesc = idesc_f16_f32(kTileRows, BN);
            int s = 0;
            uint32_t ph = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            for (int u = blockIdx.x; ok && u < a.units; u += gridDim.x) {
                const UnitInfo ui = unit_info(a, u);
                if (!mbar_wait_bounded(&tempty[acc], acc_phase ^ 1u, abort_flag, a.status))
                    break;
                tc_fence_after();
                const uint32_t d_tmem = tmem + static_cast<uint32_t>(acc * BN);
                for (int kb = ui.kb0; kb < ui.kb1; ++kb) {
                    if (!mbar_wait_bounded(&x_full[s], ph, abort_flag, a.status) ||
                        !mbar_wait_bounded(&a_full[s], ph, abort_flag, a.status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_addr = smem_u32(sA + s * kABytes);
                    const uint32_t b_addr = smem_u32(sX + s * kXBytes);
#pragma unroll
                    for (int k = 0; k < kBK / 16; ++k)
                        umma_f16(d_tmem, sdesc_k_sw128(a_addr + 32 * k), sdesc_k_sw128(b_addr + 32 * k), idesc,
                                 (kb > ui.kb0 || k > 0) ? 1u : 0u);
                    umma_commit(&s_empty[s]);
                    if (++s == S) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
                if (!ok)
                    break;
                umma_commit(&tfull[acc]);
                if (++acc == 2) {
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
                for (int kb = ui.kb0; kb < ui.kb1; ++kb) {
                    if (!mbar_wait_bounded(&s_empty[s], ph ^ 1u, abort_flag, a.status)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&x_full[s], kXBytes);
                    tma_load_2d(sX + s * kXBytes, &tm_x, &x_full[s], kb * kBK, m0);
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
        }
    } else if (warp >= 4 && warp < 8) {
        // ---------------- epilogue: warps 4..7 own TMEM lane quarters 0..3
        epilogue_role<BN>(a, tmem, tfull, tempty, abort_flag, warp, lane);
    } else if (warp >= kDecodeWarp0) {
        // ---------------- decoders
        const int dt = threadIdx.x - kDecodeWarp0 * 32;
        const int row = dt & (kTileRows - 1);
        const int half = dt >> 7;
        int s = 0, r = 0;
        uint32_t ph = 0, rph = 0;
        bool ok = true;
        for (int u = blockIdx.x; ok && u < a.units; u += gridDim.x) {
            const UnitInfo ui = unit_info(a, u);
            const int64_t n = static_cast<int64_t>(ui.tile / a.m_tiles) * kTileRows + row;
            const bool valid = n < a.N;
            for (int kb = ui.kb0; ok && kb < ui.kb1; kb += kChunkSteps) {
                const int steps = ui.kb1 - kb < kChunkSteps ? ui.kb1 - kb : kChunkSteps;
                if (!__all_sync(0xFFFFFFFFu, mbar_wait_bounded(&raw_full[r], rph, abort_flag, a.status))) {
                    ok = false;
                    break;
                }
                RowSpan sp{0, 0};
                if (valid)
                    sp = row_span<QT>(n, a.K, static_cast<int64_t>(kb) * kBK, static_cast<int64_t>(steps) * kBK);
                const uint32_t raw_row = smem_u32(sR + static_cast<size_t>(r) * kTileRows * RS + static_cast<size_t>(row) * RS);
                for (int st = 0; st < steps; ++st) {
                    if (!__all_sync(0xFFFFFFFFu, mbar_wait_bounded(&s_empty[s], ph ^ 1u, abort_flag, a.status))) {
                        ok = false;
                        break;
                    }
                    uint4 out[4] = {make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0),
                                    make_uint4(0, 0, 0, 0)};
                    if (valid) {
                        const int64_t es = n * a.K + static_cast<int64_t>(kb + st) * kBK + 32 * half;
                        const int64_t blk = es / F::QK;
                        const int o = static_cast<int>(es - blk * F::QK);
                        decode32<QT>(raw_row + static_cast<uint32_t>(blk * F::BB - sp.s0), o, out);
                    }
                    const uint32_t a_row = smem_u32(sA + s * kABytes) + (row >> 3) * 1024 + (row & 7) * 128;
#pragma unroll
                    for (int c4 = 0; c4 < 4; ++c4) {
                        const int c = 4 * half + c4;
                        sts_v4(a_row + ((c ^ (row & 7)) << 4), out[c4]);
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive(&a_full[s]);
                    if (++s == S) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&raw_empty[r]);
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
    int rs, stages, raw_stages, smem;
};

// Shared-memory plan: per-row raw slot size, f16 operand stages and raw
// stages that fit in 227 KB.
FusedLayout fused_layout(int qt, int64_t K, int bn)
{
    int qk = 0, bb = 0;
    switch (qt) {
    case 8: qk = 32; bb = 34; break;
    case 12: qk = 256; bb = 144; break;
    default: qk = 256; bb = 210; break;
    }
    // Blocks a 256-element chunk of one row can touch: chunks start on
    // multiples of 64 elements of the flat stream, so with K % 256 == 0 a
    // chunk is exactly 256/QK blocks; otherwise a 256-element block can be
    // straddled.  Misalignment of the first block inside its 16-byte line is
    // 0 for 144-byte blocks and at most 14 bytes otherwise.
    const int span = (qk == 32) ? 8 : ((K % 256 == 0) ? 1 : 2);
    const int mis = (bb % 16 == 0) ? 0 : 14;
    FusedLayout L{};
    L.rs = (span * bb + mis + 15) / 16 * 16;
    const int stage = kABytes + bn * kBK * 2;
    const int raw = kTileRows * L.rs;
    const int budget = kSmemLimit - 1024 - 256;
    L.stages = kMaxStages;
    while (L.stages > 2 && L.stages * stage + 2 * raw > budget)
        --L.stages;
    L.raw_stages = (budget - L.stages * stage) / raw;
    if (L.raw_stages > kMaxRaw)
        L.raw_stages = kMaxRaw;
    L.smem = 1024 + L.stages * stage + L.raw_stages * raw + 256;
    return L;
}

template <int BN, int QT>
cudaError_t launch_f(const CUtensorMap &tx, const GemmArgs &a0, const GemmPlan &p, cudaStream_t s)
{
    const FusedLayout L = fused_layout(QT, a0.K, BN);
    if (L.raw_stages < 2)
        return cudaErrorInvalidConfiguration;
    GemmArgs a = a0;
    a.raw_rs = L.rs;
    a.stages = L.stages;
    a.raw_stages = L.raw_stages;
    static bool attr_done[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 0 || dev >= 64 || !attr_done[dev]) {
        e = cudaFuncSetAttribute(k_gemm_fused<BN, QT>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit);
        if (e != cudaSuccess)
            return e;
        if (dev >= 0 && dev < 64)
            attr_done[dev] = true;
    }
    k_gemm_fused<BN, QT><<<p.grid, kThreadsF, L.smem, s>>>(tx, a);
    note_launch();
    return cudaGetLastError();
}

template <int QT>
cudaError_t launch_q(const CUtensorMap &tx, const GemmArgs &a, const GemmPlan &p, cudaStream_t s)
{
    switch (p.bn) {
    case 256: return launch_f<256, QT>(tx, a, p, s);
    case 128: return launch_f<128, QT>(tx, a, p, s);
    case 64: return launch_f<64, QT>(tx, a, p, s);
    case 32: return launch_f<32, QT>(tx, a, p, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_gemm_fused(const CUtensorMap &tx, const GemmArgs &a, const GemmPlan &p, cudaStream_t s)
{
    if (a.K % kBK != 0 || p.kb_align != kChunkSteps)
        return cudaErrorInvalidValue;
    switch (a.qtype) {
    case 8: return launch_q<8>(tx, a, p, s);
    case 12: return launch_q<12>(tx, a, p, s);
    case 14: return launch_q<14>(tx, a, p, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace mq
