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
//
// The 8-bit variant (k_gemm_e4m3) is the same kernel on e4m3 operands: a
// stage is still one 128-byte swizzle row per operand row, now 128 K
// elements, and each of its four MMAs (kind::f8f6f4, K = 32) advances 32
// bytes as for f16; the epilogue scales by the weight row's and the token's
// quantization scales.
//
// CTA pairs (PAIR): two CTAs of a cluster take adjacent 128-row weight
// tiles of the same token tile.  Each loads its own weight tile and half of
// the token tile, multicast into both CTAs' shared memory, so a stage costs
// an SM 16 + BN*64 bytes of L2 reads instead of 16 + 2*BN*64 KB.  A
// stage's "empty" barrier then counts both CTAs' MMA commits: neither
// producer refills a stage its peer may still be reading.
#include <algorithm>
#include <cstdint>
#include <cuda_runtime.h>

#include "mq_internal.h"
#include "mq_launch.cuh"
#include "mq_ptx.cuh"
#include "mq_tile.cuh"

namespace mq {

namespace {

constexpr int kThreads = 192;

template <int BN> struct Cfg {
    static constexpr int kBBytes = BN * kBK * 2;
    static constexpr int kStages = BN >= 256 ? 4 : (BN >= 128 ? 6 : 8);
    static constexpr int kTmemCols = 2 * BN;   // two accumulators
    static constexpr int kSmem = 1024 + kStages * (kABytes + kBBytes) + kYStageBytes + 256;
};

// The kernel body: F8 selects e4m3 operands (K step kBK8, kind::f8f6f4,
// scaled epilogue) over f16 (K step kBK, kind::f16); PAIR runs the CTA as
// one of a cluster pair (tm_x's box is then BN/2 tokens high).
template <int BN, bool F8, bool PAIR>
__device__ __forceinline__ void gemm_body(const WMaps &tm_w, const CUtensorMap &tm_x, const GemmArgs &a)
{
    using C = Cfg<BN>;
    constexpr int kStep = F8 ? kBK8 : kBK;   // K elements per stage (128 bytes per row either way)
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t *sA = base;
    uint8_t *sB = base + C::kStages * kABytes;
    float *sY = reinterpret_cast<float *>(sB + C::kStages * C::kBBytes);   // staged output boxes
    uint64_t *full = reinterpret_cast<uint64_t *>(sB + C::kStages * C::kBBytes + kYStageBytes);
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
            mbar_init(&empty[s], PAIR ? 2 : 1);
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
        for (int g = 0; g < a.groups; ++g)
            prefetch_tensormap(&tm_w.m[g]);
        prefetch_tensormap(&tm_x);
    }
    tc_fence_before();
    if constexpr (PAIR)
        cluster_sync();   // the peer's barriers exist before any multicast reaches them
    else
        __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    grid_dep_launch();
    const UnitWalk wk = unit_walk(a);

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer.  The weight tiles of the first
            // kStages K steps do not depend on the previous kernel on the
            // stream, so they are requested before grid_dep_wait(); the
            // activation tiles (and everything after) follow it.
            int stage = 0;
            uint32_t phase = 0;
            uint32_t issued = 0, issue_parity = 0;   // per-stage: load in flight, its phase parity
            bool ok = a.stall_producer == 0;
            int pre = 0;
            for (int u = wk.first; ok && pre < C::kStages && u < a.units; u += wk.stride) {
                const UnitInfo ui = unit_info(a, u, wk.rank);
                int nt, mt;
                tile_coords(a, ui.tile, nt, mt);
                const int g = group_of(a, nt);
                const int n0 = (nt - a.g_tile0[g]) * kTileRows;
                for (int kb = ui.kb0; kb < ui.kb1 && pre < C::kStages; ++kb, ++pre) {
                    mbar_arrive_expect_tx(&full[pre], kABytes + C::kBBytes);
                    tma_load_2d(sA + pre * kABytes, &tm_w.m[g], &full[pre], kb * kStep, n0);
                    issued |= 1u << pre;
                }
            }
            grid_dep_wait();
            int step = 0;
            // the token rows this CTA loads: all BN, or its half of the pair's
            const int b_off = PAIR ? wk.rank * (BN / 2) : 0;
            uint8_t *sB_own = sB + b_off * 128;
            for (int u = wk.first; ok && u < a.units; u += wk.stride) {
                const UnitInfo ui = unit_info(a, u, wk.rank);
                int nt, mt;
                tile_coords(a, ui.tile, nt, mt);
                const int g = group_of(a, nt);
                const CUtensorMap *tmw = &tm_w.m[g];
                const int n0 = (nt - a.g_tile0[g]) * kTileRows;   // row inside member g
                const int m0 = mt * BN + b_off;
                for (int kb = ui.kb0; kb < ui.kb1; ++kb, ++step) {
                    if (step < pre) {
                        // weight tile already requested (stage == step, phase 0)
                        if constexpr (PAIR)
                            tma_load_2d_mc(sB_own + stage * C::kBBytes, &tm_x, &full[stage], kb * kStep, m0, 0x3);
                        else
                            tma_load_2d(sB + stage * C::kBBytes, &tm_x, &full[stage], kb * kStep, m0);
                        if (++stage == C::kStages) {
                            stage = 0;
                            phase ^= 1u;
                        }
                        continue;
                    }
                    if (!mbar_wait_bounded(&empty[stage], phase ^ 1u, abort_flag, a.status)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&full[stage], kABytes + C::kBBytes);
                    tma_load_2d(sA + stage * kABytes, tmw, &full[stage], kb * kStep, n0);
                    if constexpr (PAIR)
                        tma_load_2d_mc(sB_own + stage * C::kBBytes, &tm_x, &full[stage], kb * kStep, m0, 0x3);
                    else
                        tma_load_2d(sB + stage * C::kBBytes, &tm_x, &full[stage], kb * kStep, m0);
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
            // ---------------- MMA issuer.  Descriptors are precomputed, so
            // only adds sit between consecutive MMAs of a stage.  (Waiting
            // for the next stage before the current stage's last MMA was
            // measured slower: it delays the commit that frees the stage.)
            constexpr uint32_t idesc = F8 ? idesc_e4m3_f32(kTileRows, BN) : idesc_f16_f32(kTileRows, BN);
            const uint64_t a_desc0 = sdesc_k_sw128(smem_u32(sA));
            const uint64_t b_desc0 = sdesc_k_sw128(smem_u32(sB));
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            for (int u = wk.first; ok && u < a.units; u += wk.stride) {
                const UnitInfo ui = unit_info(a, u, wk.rank);
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
                    // descriptor start fields are 16-byte units (14 bits): shared
                    // addresses stay below 256 KB, so adding the stage offset
                    // never carries out of the field
                    const uint64_t ad = a_desc0 + static_cast<uint64_t>((stage * kABytes) >> 4);
                    const uint64_t bd = b_desc0 + static_cast<uint64_t>((stage * C::kBBytes) >> 4);
#pragma unroll
                    for (int k = 0; k < 4; ++k) {   // four MMAs of 32 bytes of K each
                        if constexpr (F8)
                            umma_e4m3(d_tmem, ad + 2 * k, bd + 2 * k, idesc, (kb > ui.kb0 || k > 0) ? 1u : 0u);
                        else
                            umma_f16(d_tmem, ad + 2 * k, bd + 2 * k, idesc, (kb > ui.kb0 || k > 0) ? 1u : 0u);
                    }
                    if constexpr (PAIR)
                        umma_commit_mc(&empty[stage], 0x3);   // frees the stage in both CTAs
                    else
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
        epilogue_role<BN, 2, 1, F8, true>(a, tmem, tfull, tempty, abort_flag, warp, lane, 1, -1, tm_w.y, sY);
    }

    tc_fence_before();
    if constexpr (PAIR)
        cluster_sync();   // no CTA leaves while its peer may still write into it
    else
        __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, C::kTmemCols);
    }
}

// ---------------------------------------------------------------- 2-SM MMAs
// A CTA pair computes a 256 x BN tile with tcgen05.mma.cta_group::2: each
// CTA stages its own 128 weight rows and half of the BN tokens (32 KB per
// K step at BN = 256 instead of 48 KB), so the same shared memory holds six
// K steps instead of four and each byte in flight covers half again as much
// MMA time (the single-CTA kernel's loads could not hide the L2 latency: its
// tensor pipe idled 30 % of the time; the 7B gate GEMM goes 174 -> 165 us).  The
// even CTA issues the MMAs; each D half lands in its own CTA's TMEM.
// Barriers: the even CTA's producer expects both CTAs' bytes of a stage on
// its own `full`, and the odd CTA's TMA copies complete there directly
// (`cp.async.bulk.tensor ... .cta_group::2` takes the peer's barrier), so the
// MMA issuer waits on one barrier per stage; the MMA commits arrive on
// `empty` and `tfull` of both CTAs; both CTAs' epilogues release the
// accumulator on the even CTA's `tempty`.
constexpr int kTwoSmAccs = 2;   // accumulators in TMEM (kTwoSmAccs * BN columns)

// Six stages of one K step (32 KB per CTA, 192 KB).  What the single
// MMA-issuing thread spends per stage decides the depth: a clock64 trace of
// the 7B gate GEMM (515 cycles of MMA work per K step, 4 x 128.8) showed it
// busy ~613 cycles per stage when the odd CTA relayed its arrivals to a
// second barrier (two waits, four MMAs, the commit, the loop), so the
// pipeline ran at the issuer's pace.  Two K steps per stage (three 64 KB
// stages) halved that cost but left a freed stage only two stages' MMA time
// (~2060 cycles) to refill, against a load latency of 1580 cycles median and
// 3140 at p90: the issuer then stalled on data.  With the odd CTA's copies
// completing on the even CTA's barrier the issuer waits once per stage and
// keeps up with one K step per stage, and five stages of slack (~2575
// cycles) hide most of the latency: the 7B gate GEMM takes 159 us (161 with
// two K steps per stage, 164.8 relayed with one), the e4m3 one 85.5 us.
// A seventh stage (225.5 KB) gains 0.5 % on the gate GEMM alone but leaves
// the SM too little shared memory for the next kernel (the e4m3 step's
// activation quantization) to start beside the GEMM's tail, which cost that
// step 28 us.  (An L2 prefetch of the weight tiles a few K steps ahead made
// the loop slower: 163 -> 170 us.)
constexpr int kTwoSmSlots = 6;   // 32 KB K-step slots of shared memory per CTA
constexpr int kTwoSmSub = 1;     // K steps per pipeline stage
template <int BN, bool F8 = false> struct Cfg2 {
    static constexpr int kHalfB = (BN / 2) * 128;   // this CTA's half of one K step's tokens
    static constexpr int kSub = kTwoSmSub;
    static constexpr int kStages = kTwoSmSlots / kSub;
    static constexpr int kStageA = kSub * kABytes;
    static constexpr int kStageB = kSub * kHalfB;
    static constexpr int kTmemCols = kTwoSmAccs * BN;
    static constexpr int kSmem = 1024 + kStages * (kStageA + kStageB) + kYStageBytes + 512;
};

template <int BN, bool F8>
__device__ __forceinline__ void gemm_body_2sm(const WMaps &tm_w, const CUtensorMap &tm_x, const GemmArgs &a)
{
    using C = Cfg2<BN, F8>;
    constexpr int kStep = F8 ? kBK8 : kBK;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t *sA = base;
    uint8_t *sB = base + C::kStages * C::kStageA;
    float *sY = reinterpret_cast<float *>(sB + C::kStages * C::kStageB);   // staged output boxes
    uint64_t *full = reinterpret_cast<uint64_t *>(sB + C::kStages * C::kStageB + kYStageBytes);
    uint64_t *empty = full + C::kStages;
    uint64_t *tfull = empty + C::kStages;
    uint64_t *tempty = tfull + 2;
    uint64_t *drain = tempty + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(&full[s], 1);   // the even CTA's producer; both CTAs' bytes
            mbar_init(&empty[s], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&tfull[i], 1);
            mbar_init(&tempty[i], 8);   // four epilogue warps in each CTA
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc_pair(tmem_slot, C::kTmemCols);
        tmem_relinquish_pair();
    }
    if (warp == 0 && lane == 0) {
        for (int g = 0; g < a.groups; ++g)
            prefetch_tensormap(&tm_w.m[g]);
        prefetch_tensormap(&tm_x);
    }
    tc_fence_before();
    cluster_sync();   // barriers and TMEM of both CTAs exist before either uses the other's
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    grid_dep_launch();
    const UnitWalk wk = unit_walk(a);

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer: own weight rows, own half of the tokens
            int stage = 0;
            uint32_t phase = 0;
            uint32_t issued = 0, issue_parity = 0;
            bool ok = a.stall_producer == 0;
            // The even CTA expects both CTAs' bytes of a stage on its own
            // `full`; the odd CTA's copies complete there (.cta_group::2).
            const bool odd = rank == 1;
            const uint32_t full_even = mapa_shared(&full[0], 0);
            constexpr uint32_t kStageTx = 2u * (kABytes + C::kHalfB);
            auto load = [&](void *dst, const CUtensorMap *map, int st, int c0, int c1) {
                if (odd)
                    tma_load_2d_pair(dst, map, full_even + static_cast<uint32_t>(st) * 8u, c0, c1);
                else
                    tma_load_2d(dst, map, &full[st], c0, c1);
            };
            int pre = 0;
            for (int u = wk.first; ok && pre < C::kStages && u < a.units; u += wk.stride) {
                const UnitInfo ui = unit_info(a, u, wk.rank);
                int nt, mt;
                tile_coords(a, ui.tile, nt, mt);
                const int g = group_of(a, nt);
                const int n0 = (nt - a.g_tile0[g]) * kTileRows;
                for (int kb = ui.kb0; kb < ui.kb1 && pre < C::kStages; kb += C::kSub, ++pre) {
                    const int ns = min(C::kSub, ui.kb1 - kb);
                    if (!odd)
                        mbar_arrive_expect_tx(&full[pre], ns * kStageTx);
                    for (int j = 0; j < ns; ++j)
                        load(sA + pre * C::kStageA + j * kABytes, &tm_w.m[g], pre, (kb + j) * kStep, n0);
                    issued |= 1u << pre;
                }
            }
            grid_dep_wait();
            int step = 0;
            for (int u = wk.first; ok && u < a.units; u += wk.stride) {
                const UnitInfo ui = unit_info(a, u, wk.rank);
                int nt, mt;
                tile_coords(a, ui.tile, nt, mt);
                const int g = group_of(a, nt);
                const CUtensorMap *tmw = &tm_w.m[g];
                const int n0 = (nt - a.g_tile0[g]) * kTileRows;
                const int m0 = mt * BN + static_cast<int>(rank) * (BN / 2);
                for (int kb = ui.kb0; kb < ui.kb1; kb += C::kSub, ++step) {
                    const int ns = min(C::kSub, ui.kb1 - kb);
                    if (step < pre) {
                        for (int j = 0; j < ns; ++j)
                            load(sB + stage * C::kStageB + j * C::kHalfB, &tm_x, stage, (kb + j) * kStep, m0);
                        if (++stage == C::kStages) {
                            stage = 0;
                            phase ^= 1u;
                        }
                        continue;
                    }
                    if (!mbar_wait_bounded(&empty[stage], phase ^ 1u, abort_flag, a.status)) {
                        ok = false;
                        break;
                    }
                    if (!odd)
                        mbar_arrive_expect_tx(&full[stage], ns * kStageTx);
                    for (int j = 0; j < ns; ++j) {
                        load(sA + stage * C::kStageA + j * kABytes, tmw, stage, (kb + j) * kStep, n0);
                        load(sB + stage * C::kStageB + j * C::kHalfB, &tm_x, stage, (kb + j) * kStep, m0);
                    }
                    issued |= 1u << stage;
                    issue_parity = (issue_parity & ~(1u << stage)) | (phase << stage);
                    if (++stage == C::kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok) {
                volatile int no_abort = 0;
                if (odd) {
                    // This CTA's copies complete on the even CTA's barriers, which
                    // it cannot wait on: give any still in flight 200 us to land
                    // (the even CTA's own drain, before the final cluster barrier,
                    // covers every stage both CTAs issued).
                    if (issued) {
                        const uint64_t t0 = globaltimer_ns();
                        while (globaltimer_ns() - t0 < 200000ull)
                            __nanosleep(1000);
                    }
                } else {
                    for (int s = 0; s < C::kStages; ++s)
                        if (issued & (1u << s))
                            mbar_wait_bounded(&full[s], (issue_parity >> s) & 1u, &no_abort, a.status);
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && rank == 0) {
            // ---------------- MMA issuer (even CTA): M = 256 across the pair
            constexpr uint32_t idesc = F8 ? idesc_e4m3_f32(2 * kTileRows, BN) : idesc_f16_f32(2 * kTileRows, BN);
            const uint64_t a_desc0 = sdesc_k_sw128(smem_u32(sA));
            const uint64_t b_desc0 = sdesc_k_sw128(smem_u32(sB));
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            for (int u = wk.first; ok && u < a.units; u += wk.stride) {
                const UnitInfo ui = unit_info(a, u, wk.rank);
                if (!mbar_wait_bounded(&tempty[acc], acc_phase ^ 1u, abort_flag, a.status))
                    break;
                tc_fence_after();
                const uint32_t d_tmem = tmem + static_cast<uint32_t>(acc * BN);
                for (int kb = ui.kb0; kb < ui.kb1; kb += C::kSub) {
                    const int ns = min(C::kSub, ui.kb1 - kb);
                    if (!mbar_wait_bounded(&full[stage], phase, abort_flag, a.status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int j = 0; j < C::kSub; ++j) {
                        if (j >= ns)
                            break;
                        const uint64_t ad = a_desc0 + static_cast<uint64_t>((stage * C::kStageA + j * kABytes) >> 4);
                        const uint64_t bd = b_desc0 + static_cast<uint64_t>((stage * C::kStageB + j * C::kHalfB) >> 4);
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const uint32_t accum = (kb > ui.kb0 || j > 0 || k > 0) ? 1u : 0u;
                            if constexpr (F8)
                                umma_e4m3_pair(d_tmem, ad + 2 * k, bd + 2 * k, idesc, accum);
                            else
                                umma_f16_pair(d_tmem, ad + 2 * k, bd + 2 * k, idesc, accum);
                        }
                    }
                    umma_commit_pair_mc(&empty[stage], 0x3);
                    if (++stage == C::kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok)
                    break;
                umma_commit_pair_mc(&tfull[acc], 0x3);
                if (++acc == kTwoSmAccs) {
                    acc = 0;
                    acc_phase ^= 1u;
                }
            }
            umma_commit_pair_mc(drain, 0x1);
            volatile int no_abort = 0;
            mbar_wait_bounded(drain, 0, &no_abort, a.status);
        }
    } else {
        // ---------------- epilogue: warps 2..5, this CTA's 128 rows of D
        epilogue_role<BN, kTwoSmAccs, 1, F8, true>(a, tmem, tfull, tempty, abort_flag, warp, lane, 1, 0, tm_w.y, sY);
    }

    tc_fence_before();
    cluster_sync();   // no CTA leaves (or frees TMEM) while its peer may still reach into it
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem, C::kTmemCols);
    }
}

template <int BN>
__global__ void __launch_bounds__(kThreads, 1)
    k_gemm_cached(const __grid_constant__ WMaps tm_w, const __grid_constant__ CUtensorMap tm_x, const GemmArgs a)
{
    gemm_body<BN, false, false>(tm_w, tm_x, a);
}

template <int BN>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    k_gemm_cached_pair(const __grid_constant__ WMaps tm_w, const __grid_constant__ CUtensorMap tm_x, const GemmArgs a)
{
    gemm_body<BN, false, true>(tm_w, tm_x, a);
}

template <int BN>
__global__ void __launch_bounds__(kThreads, 1)
    k_gemm_e4m3(const __grid_constant__ WMaps tm_w, const __grid_constant__ CUtensorMap tm_x, const GemmArgs a)
{
    gemm_body<BN, true, false>(tm_w, tm_x, a);
}

template <int BN>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    k_gemm_e4m3_pair(const __grid_constant__ WMaps tm_w, const __grid_constant__ CUtensorMap tm_x, const GemmArgs a)
{
    gemm_body<BN, true, true>(tm_w, tm_x, a);
}

template <int BN>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    k_gemm_cached_2sm(const __grid_constant__ WMaps tm_w, const __grid_constant__ CUtensorMap tm_x, const GemmArgs a)
{
    gemm_body_2sm<BN, false>(tm_w, tm_x, a);
}

template <int BN>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    k_gemm_e4m3_2sm(const __grid_constant__ WMaps tm_w, const __grid_constant__ CUtensorMap tm_x, const GemmArgs a)
{
    gemm_body_2sm<BN, true>(tm_w, tm_x, a);
}

template <bool F8>
cudaError_t launch_2sm(const WMaps &tw, const CUtensorMap &tx, const GemmArgs &a, const GemmPlan &p, cudaStream_t s)
{
    using C = Cfg2<256, F8>;
    auto *kern = F8 ? k_gemm_e4m3_2sm<256> : k_gemm_cached_2sm<256>;
    static bool attr_done[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 0 || dev >= 64 || !attr_done[dev]) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
        if (e != cudaSuccess)
            return e;
        if (dev >= 0 && dev < 64)
            attr_done[dev] = true;
    }
    e = launch_kernel(kern, dim3(p.grid), dim3(kThreads), C::kSmem, s, tw, tx, a);
    note_launch();
    return e;
}

template <int BN, bool F8, bool PAIR>
constexpr auto gemm_kernel()
{
    if constexpr (PAIR)
        return F8 ? k_gemm_e4m3_pair<BN> : k_gemm_cached_pair<BN>;
    else
        return F8 ? k_gemm_e4m3<BN> : k_gemm_cached<BN>;
}

// Fixed-order split-K reduction: Y = sum over p = 0..split-1 of the partial
// planes, p ascending, for the split tiles.  Grid (bn/8, slots): each thread
// owns 4 consecutive weight rows of one token column, loads all split
// partials first (so their latencies overlap) and adds them in order.
constexpr int kMaxSplit = 8;

__global__ void __launch_bounds__(256) k_splitk_reduce(const GemmArgs a, int bn)
{
    grid_dep_launch();
    grid_dep_wait();   // the partial planes come from the GEMM kernel just before
    const int slot = blockIdx.y;
    const int tile = a.full_tiles + slot;
    const int64_t plane = static_cast<int64_t>(bn) * kTileRows;
    const int e = (blockIdx.x * 256 + threadIdx.x) * 4;
    if (e >= plane)
        return;
    const int col = e >> 7, row = e & 127;
    int nt, mt;
    tile_coords(a, tile, nt, mt);
    const int g = group_of(a, nt);
    const int64_t Ng = a.g_N[g];
    const int64_t m = static_cast<int64_t>(mt) * bn + col;
    const int64_t n = static_cast<int64_t>(nt - a.g_tile0[g]) * kTileRows + row;   // row inside member g
    if (m >= a.M || n >= Ng)
        return;
    const float4 *base = reinterpret_cast<const float4 *>(a.ws + static_cast<int64_t>(slot) * a.split * plane + e);
    float4 v[kMaxSplit];
#pragma unroll
    for (int p = 0; p < kMaxSplit; ++p)
        if (p < a.split)
            v[p] = __ldcs(base + p * (plane / 4));
    float4 acc = v[0];
#pragma unroll
    for (int p = 1; p < kMaxSplit; ++p)
        if (p < a.split) {
            acc.x = __fadd_rn(acc.x, v[p].x);
            acc.y = __fadd_rn(acc.y, v[p].y);
            acc.z = __fadd_rn(acc.z, v[p].z);
            acc.w = __fadd_rn(acc.w, v[p].w);
        }
    float *yp = a.g_y[g] + m * Ng + n;
    if ((Ng & 3) == 0 && n + 3 < Ng) {
        *reinterpret_cast<float4 *>(yp) = acc;
    } else {
        const float r[4] = {acc.x, acc.y, acc.z, acc.w};
        for (int i = 0; i < 4 && n + i < Ng; ++i)
            yp[i] = r[i];
    }
}

template <int BN, bool F8, bool PAIR>
cudaError_t launch_bn(const WMaps &tw, const CUtensorMap &tx, const GemmArgs &a, const GemmPlan &p, cudaStream_t s)
{
    using C = Cfg<BN>;
    auto *kern = gemm_kernel<BN, F8, PAIR>();
    static bool attr_done[64] = {};   // the attribute is set once per device (per instantiation)
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 0 || dev >= 64 || !attr_done[dev]) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
        if (e != cudaSuccess)
            return e;
        if (dev >= 0 && dev < 64)
            attr_done[dev] = true;
    }
    e = launch_kernel(kern, dim3(p.grid), dim3(kThreads), C::kSmem, s, tw, tx, a);
    note_launch();
    return e;
}

}  // namespace

GemmPlan plan_gemm(int64_t M, int64_t N, int64_t K, int sms, bool fused, int64_t ws_available, int bn_override,
                   int kstep, int pair_clusters)
{
    GemmPlan p{};
    // The fused path keeps a whole 256-element K chunk of activations per
    // stage, so its tiles stop at 128 tokens; at M <= 16 it uses the
    // narrowest MMA (N = 16), which halves the accumulator traffic per MMA.
    if (fused)
        p.bn = M > 64 ? 128 : (M > 32 ? 64 : (M > 16 ? 32 : 16));
    else
        p.bn = M > 128 ? 256 : (M > 64 ? 128 : (M > 32 ? 64 : 32));
    if (!fused && bn_override > 0)
        p.bn = bn_override;
    // The fused path stages raw weight bytes 256 K-elements (4 K steps) at a
    // time, so its split boundaries fall on multiples of 4 K steps.
    p.kb_align = fused ? 4 : 1;
    const int64_t m_tiles = (M + p.bn - 1) / p.bn;
    const int64_t n_tiles = (N + kTileRows - 1) / kTileRows;
    const int64_t kblocks = (K + kstep - 1) / kstep;
    const int64_t groups = (kblocks + p.kb_align - 1) / p.kb_align;
    // Work items: tiles on `slots` SMs, or pair tiles (two CTA tiles each,
    // the second a phantom past N when the weight-row tiles are odd) on
    // `slots` resident clusters.
    p.pair = (!fused && pair_clusters > 0) ? 1 : 0;
    const int per = p.pair ? 2 : 1;
    const int slots = p.pair ? pair_clusters : sms;
    const int items = static_cast<int>(m_tiles * (p.pair ? (n_tiles + 1) / 2 : n_tiles));
    int full_items = items;
    p.split = 1;
    // Split-K tail: the items of the last, partial wave are split so that
    // the wave fills the SMs; each part keeps at least 4 K steps.
    const int tail = items % slots;
    if (tail != 0) {
        int s = slots / tail;
        const int64_t max_parts = fused ? groups : std::max<int64_t>(1, kblocks / 4);
        s = static_cast<int>(std::min<int64_t>(s, max_parts));
        s = std::min(s, kMaxSplit);
        if (s >= 2) {
            const int64_t bytes = static_cast<int64_t>(tail) * per * s * p.bn * kTileRows * 4;
            if (bytes <= ws_available) {
                p.split = s;
                full_items = items - tail;
                p.ws_bytes = bytes;
            }
        }
    }
    p.tiles = items * per;
    p.full_tiles = full_items * per;
    p.units = full_items + (items - full_items) * p.split;
    p.grid = std::min(p.units, slots) * per;
    return p;
}

int64_t schedule_units(const GemmPlan &p, int64_t M, int64_t N, int64_t K, int kstep, int32_t *out, int64_t cap)
{
    GemmArgs a{};
    a.M = M;
    a.N = N;
    a.K = K;
    a.m_tiles = static_cast<int>((M + p.bn - 1) / p.bn);
    a.kblocks = static_cast<int>((K + kstep - 1) / kstep);
    a.full_tiles = p.full_tiles;
    a.split = p.split;
    a.units = p.units;
    a.kb_align = p.kb_align;
    a.pair = p.pair;
    int64_t n = 0;
    for (int cta = 0; cta < p.grid; ++cta) {
        const UnitWalk wk = unit_walk_of(a, cta, p.grid);
        for (int u = wk.first; u < a.units; u += wk.stride, ++n) {
            if (n >= cap)
                continue;
            const UnitInfo ui = unit_info(a, u, wk.rank);
            int nt, mt;
            tile_coords(a, ui.tile, nt, mt);
            int32_t *r = out + 8 * n;
            r[0] = cta;
            r[1] = ui.tile;
            r[2] = nt;
            r[3] = mt;
            r[4] = ui.kb0;
            r[5] = ui.kb1;
            r[6] = ui.part;
            r[7] = ui.slot;
        }
    }
    return n;
}

int64_t plan_ws_bytes_wanted(int64_t M, int64_t N, int64_t K, int sms, bool fused, int bn_override, int kstep,
                             int pair_clusters)
{
    return plan_gemm(M, N, K, sms, fused, INT64_MAX, bn_override, kstep, pair_clusters).ws_bytes;
}

cudaError_t launch_gemm_cached(const WMaps &tw, const CUtensorMap &tx, const GemmArgs &a, const GemmPlan &p,
                               cudaStream_t s)
{
    if (p.two_sm && p.pair && p.bn == 256)
        return launch_2sm<false>(tw, tx, a, p, s);
    if (p.pair) {
        switch (p.bn) {
        case 256: return launch_bn<256, false, true>(tw, tx, a, p, s);
        case 128: return launch_bn<128, false, true>(tw, tx, a, p, s);
        case 64: return launch_bn<64, false, true>(tw, tx, a, p, s);
        default: return cudaErrorInvalidValue;
        }
    }
    switch (p.bn) {
    case 256: return launch_bn<256, false, false>(tw, tx, a, p, s);
    case 128: return launch_bn<128, false, false>(tw, tx, a, p, s);
    case 64: return launch_bn<64, false, false>(tw, tx, a, p, s);
    case 32: return launch_bn<32, false, false>(tw, tx, a, p, s);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_gemm_e4m3(const WMaps &tw, const CUtensorMap &tx, const GemmArgs &a, const GemmPlan &p,
                             cudaStream_t s)
{
    if (p.two_sm && p.pair && p.bn == 256)
        return launch_2sm<true>(tw, tx, a, p, s);
    if (p.pair) {
        switch (p.bn) {
        case 256: return launch_bn<256, true, true>(tw, tx, a, p, s);
        case 128: return launch_bn<128, true, true>(tw, tx, a, p, s);
        case 64: return launch_bn<64, true, true>(tw, tx, a, p, s);
        default: return cudaErrorInvalidValue;
        }
    }
    switch (p.bn) {
    case 256: return launch_bn<256, true, false>(tw, tx, a, p, s);
    case 128: return launch_bn<128, true, false>(tw, tx, a, p, s);
    case 64: return launch_bn<64, true, false>(tw, tx, a, p, s);
    case 32: return launch_bn<32, true, false>(tw, tx, a, p, s);
    default: return cudaErrorInvalidValue;
    }
}

// Clusters of two that can be resident at once, per device and kernel
// (cached after the first query).
template <int BN, bool F8, bool TWO_SM>
int pair_clusters_bn()
{
    static int cached[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return 0;
    if (cached[dev] != 0)
        return cached[dev] > 0 ? cached[dev] : 0;
    const int smem = TWO_SM ? Cfg2<BN, F8>::kSmem : Cfg<BN>::kSmem;
    auto *kern = TWO_SM ? (F8 ? k_gemm_e4m3_2sm<BN> : k_gemm_cached_2sm<BN>) : gemm_kernel<BN, F8, true>();
    int n = 0;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) == cudaSuccess) {
        cudaLaunchConfig_t cfg{};
        cfg.gridDim = dim3(2);
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = smem;
        if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess)
            n = 0;
    }
    cudaGetLastError();
    cached[dev] = n > 0 ? n : -1;
    return n > 0 ? n : 0;
}

int pair_clusters_for(int bn, bool e4m3, bool two_sm)
{
    switch (bn) {
    case 256:
        if (two_sm)
            return e4m3 ? pair_clusters_bn<256, true, true>() : pair_clusters_bn<256, false, true>();
        return e4m3 ? pair_clusters_bn<256, true, false>() : pair_clusters_bn<256, false, false>();
    case 128: return e4m3 ? pair_clusters_bn<128, true, false>() : pair_clusters_bn<128, false, false>();
    case 64: return e4m3 ? pair_clusters_bn<64, true, false>() : pair_clusters_bn<64, false, false>();
    default: return 0;
    }
}

cudaError_t launch_splitk_reduce(const GemmArgs &a, const GemmPlan &p, cudaStream_t s)
{
    const int slots = p.tiles - p.full_tiles;
    if (slots <= 0 || p.split <= 1)
        return cudaSuccess;
    if (p.split > kMaxSplit || a.groups < 1 || a.groups > kMaxGroup)
        return cudaErrorInvalidValue;
    const cudaError_t e = launch_kernel(k_splitk_reduce, dim3(p.bn / 8, slots), dim3(256), 0, s, a, p.bn);
    note_launch();
    return e;
}

}  // namespace mq
