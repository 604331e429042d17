// gemm.cu -- cached-path GEMM on the 5th-generation tensor cores (sm_103a),
// its split-K reduction, and the work planner shared with the fused path.
//
//   Y[m, n] = sum_k X[m, k] * Wc[n, k]      X f16 [M,K], Wc f16 [N,ldk], Y f32
//
// ("05 · 8p — Persistent f16 weight cache + fused dequant-in-GEMM",
// section 2: the GEMM reads only the resident f16 copy; "Eager GPU Offload
// Without A Compute Graph", section "Storage and transfer reuse": f16
// inputs with f32 output, split-K with a fixed-order reduction when the
// output grid underfills the GPU.)
//
// Design (one CTA per SM, persistent):
//  * The weight rows are the MMA's M side (128 rows per tile) and the tokens
//    its N side (BN = 32..256 per tile).  This "swap-AB" orientation puts a
//    token's outputs for 32 consecutive weight rows in 32 consecutive TMEM
//    lanes, so each epilogue store instruction writes 128 contiguous bytes of
//    a Y row.
//  * Warp 0: TMA producer.  Per 64-wide K step it loads the 128x64 weight
//    tile and the BNx64 activation tile (128-byte swizzle, zero fill past the
//    edges) into one of STAGES shared-memory stages.
//  * Warp 1: allocates TMEM (2 x BN f32 columns: two accumulators) and one
//    thread issues tcgen05.mma (M=128, N=BN, K=16; four per K step),
//    committing each stage back to the producer and each finished tile to
//    the epilogue.
//  * Warps 2-5: epilogue.  tcgen05.ld 32 lanes x 32 columns, then plain
//    coalesced stores to Y (or to the split-K workspace).  Two accumulators
//    let the epilogue of tile i overlap the main loop of tile i+1.
//  * Every pipeline wait is bounded (mq_ptx.cuh); on a timeout all roles stop
//    and the CTA still frees its TMEM.
#include <algorithm>
#include <cstdint>
#include <cuda_runtime.h>

#include "mq_internal.h"
#include "mq_ptx.cuh"

namespace mq {

namespace {

constexpr int kBK = 64;                       // K elements per stage (one 128-byte swizzle row)
constexpr int kTileRows = 128;                // weight rows per tile (MMA M)
constexpr int kABytes = kTileRows * kBK * 2;  // 16 KB
constexpr int kThreads = 192;

template <int BN> struct Cfg {
    static constexpr int kBBytes = BN * kBK * 2;
    static constexpr int kStages = BN >= 256 ? 4 : (BN >= 128 ? 6 : 8);
    static constexpr int kTmemCols = 2 * BN;   // two accumulators
    static constexpr int kSmem = 1024 + kStages * (kABytes + kBBytes) + 256;
};

struct UnitInfo {
    int tile, kb0, kb1, part, slot;
};

__device__ __forceinline__ UnitInfo unit_info(const GemmArgs &a, int u)
{
    UnitInfo r;
    if (u < a.full_tiles) {
        r.tile = u;
        r.kb0 = 0;
        r.kb1 = a.kblocks;
        r.part = -1;
        r.slot = 0;
    } else {
        const int v = u - a.full_tiles;
        r.slot = v / a.split;
        r.part = v - r.slot * a.split;
        r.tile = a.full_tiles + r.slot;
        r.kb0 = static_cast<int>(static_cast<int64_t>(r.part) * a.kblocks / a.split);
        r.kb1 = static_cast<int>(static_cast<int64_t>(r.part + 1) * a.kblocks / a.split);
    }
    return r;
}

template <int BN>
__global__ void __launch_bounds__(kThreads, 1)
    k_gemm_cached(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_x,
                  const GemmArgs a)
{
    using C = Cfg<BN>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t *sA = base;
    uint8_t *sB = base + C::kStages * kABytes;
    uint64_t *full = reinterpret_cast<uint64_t *>(sB + C::kStages * C::kBBytes);
    uint64_t *empty = full + C::kStages;
    uint64_t *tfull = empty + C::kStages;
    uint64_t *tempty = tfull + 2;
    uint64_t *drain = tempty + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
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
        tmem_alloc(tmem_slot, C::kTmemCols);
        tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tensormap(&tm_w);
        prefetch_tensormap(&tm_x);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer
            int stage = 0;
            uint32_t phase = 0;
            uint32_t issued = 0, issue_parity = 0;   // per-stage: load in flight, its phase parity
            bool ok = true;
            for (int u = blockIdx.x; ok && u < a.units; u += gridDim.x) {
                const UnitInfo ui = unit_info(a, u);
                const int n0 = (ui.tile / a.m_tiles) * kTileRows;
                const int m0 = (ui.tile % a.m_tiles) * BN;
                for (int kb = ui.kb0; kb < ui.kb1; ++kb) {
                    if (!mbar_wait_bounded(&empty[stage], phase ^ 1u, abort_flag, a.status)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&full[stage], kABytes + C::kBBytes);
                    tma_load_2d(sA + stage * kABytes, &tm_w, &full[stage], kb * kBK, n0);
                    tma_load_2d(sB + stage * C::kBBytes, &tm_x, &full[stage], kb * kBK, m0);
                    issued |= 1u << stage;
                    issue_parity = (issue_parity & ~(1u << stage)) | (phase << stage);
                    if (++stage == C::kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok) {
                // Let every load this thread issued land before the CTA's
                // shared memory can be handed to anyone else.
                volatile int no_abort = 0;
                for (int s = 0; s < C::kStages; ++s)
                    if (issued & (1u << s))
                        mbar_wait_bounded(&full[s], (issue_parity >> s) & 1u, &no_abort, a.status);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------- MMA issuer
            constexpr uint32_t idesc = idesc_f16_f32(kTileRows, BN);
            int stage = 0;
            uint32_t phase = 0;
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
                    if (!mbar_wait_bounded(&full[stage], phase, abort_flag, a.status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_addr = smem_u32(sA + stage * kABytes);
                    const uint32_t b_addr = smem_u32(sB + stage * C::kBBytes);
#pragma unroll
                    for (int k = 0; k < kBK / 16; ++k)
                        umma_f16(d_tmem, sdesc_k_sw128(a_addr + 32 * k), sdesc_k_sw128(b_addr + 32 * k), idesc,
                                 (kb > ui.kb0 || k > 0) ? 1u : 0u);
                    umma_commit(&empty[stage]);
                    if (++stage == C::kStages) {
                        stage = 0;
                        phase ^= 1u;
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
            // Every MMA this thread issued has finished before TMEM can be
            // freed, also when a wait gave up midway.
            umma_commit(drain);
            volatile int no_abort = 0;
            mbar_wait_bounded(drain, 0, &no_abort, a.status);
        }
    } else {
        // ---------------- epilogue: warps 2..5 own TMEM lane quarters 2,3,0,1
        const int q = warp & 3;
        const int row = q * 32 + lane;
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int u = blockIdx.x; u < a.units; u += gridDim.x) {
            const UnitInfo ui = unit_info(a, u);
            const bool ok = mbar_wait_bounded(&tfull[acc], acc_phase, abort_flag, a.status);
            if (!__all_sync(0xFFFFFFFFu, ok))
                break;
            tc_fence_after();
            const int64_t n = static_cast<int64_t>(ui.tile / a.m_tiles) * kTileRows + row;
            const int64_t m0 = static_cast<int64_t>(ui.tile % a.m_tiles) * BN;
#pragma unroll 1
            for (int c = 0; c < BN; c += 32) {
                uint32_t r[32];
                tmem_ld_32x32b_x32(tmem + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * BN + c),
                                   r);
                tmem_ld_wait();
                if (ui.part < 0) {
                    if (n < a.N) {
                        float *yp = a.y + (m0 + c) * a.N + n;
                        const int64_t rem = a.M - (m0 + c);
                        const int lim = rem < 32 ? static_cast<int>(rem) : 32;
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            if (j < lim)
                                yp[static_cast<int64_t>(j) * a.N] = __uint_as_float(r[j]);
                    }
                } else {
                    float *wp = a.ws + ((static_cast<int64_t>(ui.slot) * a.split + ui.part) * BN + c) * kTileRows + row;
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        wp[j * kTileRows] = __uint_as_float(r[j]);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&tempty[acc]);
            if (++acc == 2) {
                acc = 0;
                acc_phase ^= 1u;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, C::kTmemCols);
    }
}

// Fixed-order split-K reduction: Y = sum over p = 0..split-1 of the partial
// planes, p ascending, for the split tiles.  One CTA per split tile.
__global__ void __launch_bounds__(256) k_splitk_reduce(const GemmArgs a, int bn)
{
    const int slot = blockIdx.x;
    const int tile = a.full_tiles + slot;
    const int64_t n0 = static_cast<int64_t>(tile / a.m_tiles) * kTileRows;
    const int64_t m0 = static_cast<int64_t>(tile % a.m_tiles) * bn;
    const int64_t plane = static_cast<int64_t>(bn) * kTileRows;
    const float *base = a.ws + static_cast<int64_t>(slot) * a.split * plane;
    for (int e = threadIdx.x; e < bn * kTileRows; e += blockDim.x) {
        const int col = e >> 7, row = e & 127;
        const int64_t m = m0 + col, n = n0 + row;
        if (m < a.M && n < a.N) {
            float acc = base[e];
            for (int p = 1; p < a.split; ++p)
                acc = __fadd_rn(acc, base[p * plane + e]);
            a.y[m * a.N + n] = acc;
        }
    }
}

template <int BN>
cudaError_t launch_bn(const CUtensorMap &tw, const CUtensorMap &tx, const GemmArgs &a, const GemmPlan &p,
                      cudaStream_t s)
{
    using C = Cfg<BN>;
    static bool attr_done[64] = {};   // the attribute is set once per device
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 0 || dev >= 64 || !attr_done[dev]) {
        e = cudaFuncSetAttribute(k_gemm_cached<BN>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
        if (e != cudaSuccess)
            return e;
        if (dev >= 0 && dev < 64)
            attr_done[dev] = true;
    }
    k_gemm_cached<BN><<<p.grid, kThreads, C::kSmem, s>>>(tw, tx, a);
    note_launch();
    return cudaGetLastError();
}

}  // namespace

GemmPlan plan_gemm(int64_t M, int64_t N, int64_t K, int sms, bool fused, int64_t ws_available)
{
    (void)fused;
    GemmPlan p{};
    p.bn = M > 128 ? 256 : (M > 64 ? 128 : (M > 32 ? 64 : 32));
    const int64_t m_tiles = (M + p.bn - 1) / p.bn;
    const int64_t n_tiles = (N + kTileRows - 1) / kTileRows;
    const int64_t kblocks = (K + kBK - 1) / kBK;
    p.tiles = static_cast<int>(m_tiles * n_tiles);
    p.split = 1;
    p.full_tiles = p.tiles;
    // Split-K tail: the tiles of the last, partial wave are split so that
    // the wave fills the SMs; each part keeps at least 4 K steps.
    const int tail = p.tiles % sms;
    if (tail != 0) {
        int s = sms / tail;
        s = static_cast<int>(std::min<int64_t>(s, std::max<int64_t>(1, kblocks / 4)));
        s = std::min(s, 8);
        if (s >= 2) {
            const int64_t bytes = static_cast<int64_t>(tail) * s * p.bn * kTileRows * 4;
            if (bytes <= ws_available) {
                p.split = s;
                p.full_tiles = p.tiles - tail;
                p.ws_bytes = bytes;
            }
        }
    }
    p.units = p.full_tiles + (p.tiles - p.full_tiles) * p.split;
    p.grid = std::min(p.units, sms);
    return p;
}

int64_t plan_ws_bytes_wanted(int64_t M, int64_t N, int64_t K, int sms)
{
    return plan_gemm(M, N, K, sms, false, INT64_MAX).ws_bytes;
}

cudaError_t launch_gemm_cached(const CUtensorMap &tw, const CUtensorMap &tx, const GemmArgs &a, const GemmPlan &p,
                               cudaStream_t s)
{
    switch (p.bn) {
    case 256: return launch_bn<256>(tw, tx, a, p, s);
    case 128: return launch_bn<128>(tw, tx, a, p, s);
    case 64: return launch_bn<64>(tw, tx, a, p, s);
    case 32: return launch_bn<32>(tw, tx, a, p, s);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_splitk_reduce(const GemmArgs &a, const GemmPlan &p, cudaStream_t s)
{
    const int slots = p.tiles - p.full_tiles;
    if (slots <= 0 || p.split <= 1)
        return cudaSuccess;
    k_splitk_reduce<<<slots, 256, 0, s>>>(a, p.bn);
    note_launch();
    return cudaGetLastError();
}

}  // namespace mq
