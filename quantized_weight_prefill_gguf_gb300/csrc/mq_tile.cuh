// mq_tile.cuh -- what the cached and the fused GEMM kernels share: tile
// geometry, the unit (tile x K-range) schedule, and the epilogue role that
// drains TMEM accumulators into Y or into the split-K workspace.
#pragma once

#include <cstdint>

#include "mq_internal.h"
#include "mq_ptx.cuh"

namespace mq {

constexpr int kBK = 64;                       // K elements per MMA stage (one 128-byte swizzle row of f16)
constexpr int kBK8 = kKStepE4m3;              // the same 128-byte row of 8-bit operands
constexpr int kTileRows = 128;                // weight rows per tile (the MMA's M)
constexpr int kABytes = kTileRows * kBK * 2;  // 16 KB f16 weight tile per stage

struct UnitInfo {
    int tile, kb0, kb1, part, slot;
};

// Unit u of the schedule: tiles [0, full_tiles) take all of K; after them,
// each remaining tile is `split` consecutive units over K-ranges whose
// boundaries are multiples of kb_align K steps.  Tile t covers weight rows
// (t / m_tiles)*128 .. +127 and tokens (t % m_tiles)*BN .. +BN-1.
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
        const int groups = (a.kblocks + a.kb_align - 1) / a.kb_align;
        const int g0 = static_cast<int>(static_cast<int64_t>(r.part) * groups / a.split);
        const int g1 = static_cast<int>(static_cast<int64_t>(r.part + 1) * groups / a.split);
        r.kb0 = g0 * a.kb_align;
        r.kb1 = g1 * a.kb_align < a.kblocks ? g1 * a.kb_align : a.kblocks;
    }
    return r;
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
template <int BN, int NACC = 2, int NPART = 1, bool SCALED = false>
__device__ __forceinline__ void epilogue_role(const GemmArgs &a, uint32_t tmem, uint64_t *tfull, uint64_t *tempty,
                                              volatile int *abort_flag, int warp, int lane, int kb_split = 1)
{
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
        const int nt = ui.tile / a.m_tiles;
        const int g = group_of(a, nt);
        const int64_t Ng = a.g_N[g];
        const int64_t n = static_cast<int64_t>(nt - a.g_tile0[g]) * kTileRows + row;   // row inside member g
        const int64_t m0 = static_cast<int64_t>(ui.tile % a.m_tiles) * BN;
        const bool two = NPART == 2 && ui.kb1 - ui.kb0 > kb_split;
        float wscale = 0.0f;
        if constexpr (SCALED)
            wscale = n < Ng ? a.g_wscale[g][n] : 0.0f;
        constexpr int kCols = BN < 32 ? BN : 32;   // columns per TMEM load
#pragma unroll 1
        for (int c = 0; c < BN; c += kCols) {
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
            if (ui.part < 0) {
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
        if (lane == 0)
            mbar_arrive(&tempty[acc]);
        if (++acc == NACC) {
            acc = 0;
            acc_phase ^= 1u;
        }
    }
}

}  // namespace mq
