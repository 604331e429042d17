// mq_tile.cuh -- what the cached and the fused GEMM kernels share: tile
// geometry, the unit (tile x K-range) schedule, and the epilogue role that
// drains TMEM accumulators into Y or into the split-K workspace.
#pragma once

#include <cstdint>

#include "mq_internal.h"
#include "mq_ptx.cuh"

namespace mq {

constexpr int kBK = kKStepF16;                // K elements per MMA stage (one 128-byte swizzle row of f16)
constexpr int kBK8 = kKStepE4m3;              // the same 128-byte row of 8-bit operands
constexpr int kTileRows = 128;                // weight rows per tile (the MMA's M)
constexpr int kABytes = kTileRows * kBK * 2;  // 16 KB f16 weight tile per stage

struct UnitInfo {
    int tile, kb0, kb1, part, slot;
};

// Weight-row tile nt and token tile mt of tile t.  Single CTAs: t = nt *
// m_tiles + mt.  CTA pairs (a.pair): pair-major numbering, t = 2p + r for
// pair tile p = (nt / 2) * m_tiles + mt and r = nt % 2, so the two CTAs of a
// cluster take tiles 2p and 2p+1 -- adjacent weight rows, the same tokens.
__host__ __device__ inline void tile_coords(const GemmArgs &a, int t, int &nt, int &mt)
{
    if (a.pair) {
        const int p = t >> 1;
        nt = 2 * (p / a.m_tiles) + (t & 1);
        mt = p % a.m_tiles;
    } else {
        nt = t / a.m_tiles;
        mt = t % a.m_tiles;
    }
}

// Unit u of the schedule: tiles [0, full_tiles) take all of K; after them,
// each remaining tile is `split` consecutive units over K-ranges whose
// boundaries are multiples of kb_align K steps (tile_coords places a tile).
// With CTA pairs, u counts pair units and rank r (0 or 1) picks the pair's
// tile: the two CTAs of a cluster run the same K-ranges in step.
__host__ __device__ inline UnitInfo unit_info(const GemmArgs &a, int u, int r = 0)
{
    UnitInfo ui;
    const int full = a.pair ? a.full_tiles >> 1 : a.full_tiles;
    if (u < full) {
        ui.tile = a.pair ? 2 * u + r : u;
        ui.kb0 = 0;
        ui.kb1 = a.kblocks;
        ui.part = -1;
        ui.slot = 0;
    } else {
        const int v = u - full;
        const int s = v / a.split;
        ui.part = v - s * a.split;
        ui.slot = a.pair ? 2 * s + r : s;
        ui.tile = a.full_tiles + ui.slot;
        const int groups = (a.kblocks + a.kb_align - 1) / a.kb_align;
        const int g0 = static_cast<int>(static_cast<int64_t>(ui.part) * groups / a.split);
        const int g1 = static_cast<int>(static_cast<int64_t>(ui.part + 1) * groups / a.split);
        ui.kb0 = g0 * a.kb_align;
        ui.kb1 = g1 * a.kb_align < a.kblocks ? g1 * a.kb_align : a.kblocks;
    }
    return ui;
}

// This CTA's walk over the units: first unit, stride, and pair rank.
struct UnitWalk {
    int first, stride, rank;
};

__host__ __device__ inline UnitWalk unit_walk_of(const GemmArgs &a, int cta, int grid)
{
    if (a.pair)
        return UnitWalk{cta >> 1, grid >> 1, cta & 1};
    return UnitWalk{cta, grid, 0};
}

__device__ __forceinline__ UnitWalk unit_walk(const GemmArgs &a)
{
    return unit_walk_of(a, static_cast<int>(blockIdx.x), static_cast<int>(gridDim.x));
}

// Epilogue role, run by four warps whose (warp index % 4) are 0..3: warp w
// may only read TMEM lanes 32*(w%4) .. +31, which hold weight rows
// 32*(w%4) .. +31 of the tile.  For each unit it waits for the accumulator,
// reads it 32 columns (tokens) at a time and stores: Y[m, n] for a whole
// tile, the partial plane ws[slot][part][col][row] for a split unit.  In
// both cases the 32 lanes of a store instruction write 32 consecutive
// floats.  Then it hands the accumulator back to the MMA warp.
//
// TMEM layout: NACC accumulator slots (double buffering across units), each
// made of NPART partial accumulators of BN columns, slot a part p at column
// (a*NPART + p)*BN.  Partial accumulators come from MMA issuers that each
// take kb_split of every kb_split*NPART consecutive K steps; part 1 exists
// when the unit has more than kb_split K steps, and the parts are added
// here in part order (0 + 1).
//
// SCALED (the 8-bit path): every accumulator value is multiplied by its
// weight row's scale and then by its token's scale, RN32(RN32(acc * sw) *
// sx), before it is stored (partial planes too: the scaling is linear).
//
// tempty_rank >= 0 (2-SM MMAs): the accumulator is handed back on the
// tempty barrier of CTA tempty_rank of the cluster (the MMA-issuing CTA),
// which counts the epilogue warps of both CTAs.
//
// TMA_Y with a.y_tma set: whole-tile outputs leave through TMA stores
// instead of st.global.  The four epilogue warps stage a box of the tile's
// 128 weight rows x kYRows tokens in shared memory as [token][row] (a warp's
// writes hit 32 consecutive words) and one thread (lane 0 of the warp with
// q = 0) stores it through member g's map ymaps[g] (f32 [M, N_g], box
// kYRows x 128), which clips rows past N_g and tokens past M.  Two boxes
// alternate, so a box is rewritten only after the store issued two boxes
// earlier has read it; the storing thread waits for all its stores before
// the role returns.  The warps meet on named barrier 1 (128 threads) twice
// per box; every condition that skips a box or leaves the unit loop is the
// same for all four warps (they wait on the same accumulator phase, which
// cannot advance before all four have released it, and the box position
// depends only on the unit and the column), so no warp waits there alone.
// With plain stores the 2-SM GEMM's tensor pipe was busy 85 % of its active
// cycles: on the 7B gate|up GEMM (2048 x 37888 x 3584) a timing copy without
// the output stores took 297 us against 320 us with them -- stores
// overlapping the next tile's main loop starved the MMAs.  Per-warp boxes of
// 32 rows brought it to 309 us and one 128-row box per kYRows tokens (four
// times fewer store operations) a little further.
constexpr int kYRows = kYBoxRows;   // tokens per staged output box
constexpr int kYBufs = 2;           // staged boxes, used in turn
constexpr int kYStageBytes = kYBufs * kTileRows * kYRows * 4;

template <int BN, int NACC = 2, int NPART = 1, bool SCALED = false, bool TMA_Y = false>
__device__ __forceinline__ void epilogue_role(const GemmArgs &a, uint32_t tmem, uint64_t *tfull, uint64_t *tempty,
                                              volatile int *abort_flag, int warp, int lane, int kb_split = 1,
                                              int tempty_rank = -1, const CUtensorMap *ymaps = nullptr,
                                              float *ystage = nullptr)
{
    const int q = warp & 3;
    const int row = q * 32 + lane;
    int acc = 0;
    uint32_t acc_phase = 0;
    int ybuf = 0;   // TMA_Y: the staged box written next
    const UnitWalk wk = unit_walk(a);
    for (int u = wk.first; u < a.units; u += wk.stride) {
        const UnitInfo ui = unit_info(a, u, wk.rank);
        const bool ok = mbar_wait_bounded(&tfull[acc], acc_phase, abort_flag, a.status);
        if (!__all_sync(0xFFFFFFFFu, ok))
            break;
        tc_fence_after();
        int nt, mt;
        tile_coords(a, ui.tile, nt, mt);
        const int g = group_of(a, nt);
        const int64_t Ng = a.g_N[g];
        const int64_t n = static_cast<int64_t>(nt - a.g_tile0[g]) * kTileRows + row;   // row inside member g
        const int64_t m0 = static_cast<int64_t>(mt) * BN;
        const bool two = NPART == 2 && ui.kb1 - ui.kb0 > kb_split;
        float wscale = 0.0f;
        if constexpr (SCALED)
            wscale = n < Ng ? a.g_wscale[g][n] : 0.0f;
        constexpr int kCols = BN < 32 ? BN : 32;   // columns per TMEM load
#pragma unroll 1
        for (int c = 0; c < BN; c += kCols) {
            if (m0 + c >= a.M)   // the rest of the tile's columns are past the last token: nothing
                break;           // reads them (the reduce skips them too); same for all four warps
            uint32_t r[32];
            const uint32_t taddr = tmem + (static_cast<uint32_t>(q * 32) << 16) +
                                   static_cast<uint32_t>(acc * NPART * BN + c);
            if constexpr (kCols == 32) {
                tmem_ld_32x32b_x32(taddr, r);
            } else {
                uint32_t (&r16)[16] = *reinterpret_cast<uint32_t (*)[16]>(r);
                tmem_ld_32x32b_x16(taddr, r16);
            }
            if constexpr (NPART == 2) {
                if (two) {
                    uint32_t r2[32];
                    if constexpr (kCols == 32) {
                        tmem_ld_32x32b_x32(taddr + BN, r2);
                    } else {
                        uint32_t (&r16)[16] = *reinterpret_cast<uint32_t (*)[16]>(r2);
                        tmem_ld_32x32b_x16(taddr + BN, r16);
                    }
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < kCols; ++j)
                        r[j] = __float_as_uint(__fadd_rn(__uint_as_float(r[j]), __uint_as_float(r2[j])));
                }
            }
            tmem_ld_wait();
            if constexpr (SCALED) {
                // lane j fetches token m0+c+j's scale; every lane takes it by shuffle
                const int64_t mj = m0 + c + lane;
                const float xs_lane = (lane < kCols && mj < a.M) ? a.x_scale[mj] : 0.0f;
#pragma unroll
                for (int j = 0; j < kCols; ++j) {
                    const float xs = __shfl_sync(0xFFFFFFFFu, xs_lane, j);
                    r[j] = __float_as_uint(__fmul_rn(__fmul_rn(__uint_as_float(r[j]), wscale), xs));
                }
            }
            if (TMA_Y && kCols == 32 && ui.part < 0 && a.y_tma) {
                const int64_t nt0 = n - row;   // the tile's first weight row in member g
                const bool storer = q == 0 && lane == 0;
#pragma unroll
                for (int h = 0; h < 32 / kYRows; ++h) {
                    const int64_t mh = m0 + c + h * kYRows;
                    if (mh >= a.M)   // box entirely past the last token: nothing to store
                        continue;
                    float *box = ystage + ybuf * (kTileRows * kYRows);
                    if (storer)
                        bulk_wait_group_read<kYBufs - 1>();
                    named_barrier_sync(1, 128);
#pragma unroll
                    for (int j = 0; j < kYRows; ++j)
                        box[j * kTileRows + row] = __uint_as_float(r[h * kYRows + j]);
                    fence_proxy_async_smem();
                    named_barrier_sync(1, 128);
                    if (storer) {
                        tma_store_2d(&ymaps[g], box, static_cast<int32_t>(nt0), static_cast<int32_t>(mh));
                        bulk_commit_group();
                    }
                    ybuf = ybuf + 1 == kYBufs ? 0 : ybuf + 1;
                }
            } else if (ui.part < 0) {
                if (n < Ng) {
                    float *yp = a.g_y[g] + (m0 + c) * Ng + n;
                    const int64_t rem = a.M - (m0 + c);
                    const int lim = rem < kCols ? static_cast<int>(rem) : kCols;
#pragma unroll
                    for (int j = 0; j < kCols; ++j)
                        if (j < lim)
                            yp[static_cast<int64_t>(j) * Ng] = __uint_as_float(r[j]);
                }
            } else {
                float *wp = a.ws + ((static_cast<int64_t>(ui.slot) * a.split + ui.part) * BN + c) * kTileRows + row;
#pragma unroll
                for (int j = 0; j < kCols; ++j)
                    wp[j * kTileRows] = __uint_as_float(r[j]);
            }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
            if (tempty_rank >= 0)
                mbar_arrive_cluster(mapa_shared(&tempty[acc], static_cast<uint32_t>(tempty_rank)));
            else
                mbar_arrive(&tempty[acc]);
        }
        if (++acc == NACC) {
            acc = 0;
            acc_phase ^= 1u;
        }
    }
    if constexpr (TMA_Y) {
        if (lane == 0)
            bulk_wait_group<0>();   // every staged box read and written before the CTA's memory goes
        __syncwarp();
    }
}

}  // namespace mq
