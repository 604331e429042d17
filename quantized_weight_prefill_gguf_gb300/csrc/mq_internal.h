// mq_internal.h -- host-side interface between the C ABI (api.cpp) and the
// kernel translation units.  Not installed; no torch types anywhere.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

struct mq_weight;   // the C ABI's handle type (include/mq.h)

namespace mq {

// Counts every kernel launch the library makes (reported by mq_launch_count).
void note_launch();

// ---------------------------------------------------------------- decoders
cudaError_t launch_dequant(int type, const void *q, int64_t nblocks, __half *out, int64_t K, int64_t ldo,
                           cudaStream_t s);

// The decoders' f32 -> f16 rounding step on the binary32 patterns
// first .. first + count - 1 (count even, first even): out[i] = f16 bits of
// pattern first + i.
cudaError_t launch_debug_cvt_f16(uint32_t first, int64_t count, uint16_t *out, cudaStream_t s);

// ---------------------------------------------------------------- GEMMs
// Work decomposition of one GEMM: the output is cut into tiles of 128
// weight rows (MMA M) x BN tokens (MMA N); tiles [0, full_tiles) run over
// all of K in one unit, the remaining tiles are split into `split` K-ranges
// whose f32 partial planes go to the workspace and are summed in fixed
// order p = 0..split-1 by the reduce kernel.
// A grouped call runs several weights that share K and X in one launch, as
// one weight stacked along N: member g owns n-tiles [g_tile0[g],
// g_tile0[g+1]) (every member's N is a multiple of the 128-row tile, so a
// tile never straddles two members), and its outputs go to g_y[g] [M, g_N[g]].
// A single weight is the group of one (g_y[0] = y, g_N[0] = N).
constexpr int kMaxGroup = 4;

// K elements per pipeline stage of the GEMMs: one 128-byte swizzle row of
// f16 (64) or of 8-bit e4m3 (128) operands.
constexpr int kKStepF16 = 64;
constexpr int kKStepE4m3 = 128;

struct GemmArgs {
    float *y;            // [M, N] f32 output
    float *ws;           // split-K partial planes: [slot][part][BN][128]
    unsigned *status;    // device status word
    const uint8_t *wq;   // raw quantized stream of member 0 (fused path)
    int64_t M, N, K;
    int m_tiles, n_tiles;
    int kblocks;         // ceil(K / 64)
    int full_tiles;
    int split;
    int units;
    int kb_align;        // split boundaries are multiples of this many K steps
    int qtype;           // fused path: GGUF type id
    int raw_rs;          // fused path: shared-memory bytes per weight row of a raw stage
    int raw_stages;      // fused path: raw stages in the ring
    int a_stages;        // fused path: f16 weight-operand stages in the ring
    int x_stages;        // fused path: activation-tile stages in the ring
    int raw_g;           // fused path: tensor maps over rows (row classes mod g); 0 = per-row bulk copies
    int64_t raw_rb;      // fused path: bytes per weight row (when rows start on block boundaries)
    int stall_producer;  // failure-injection hook: the weight producer issues nothing, so the
                         // consumers' bounded waits run out (tests of the timeout path)
    int pair;                       // CTAs run in clusters of two (see tile_coords)
    int y_tma;                      // cached/e4m3 GEMMs: whole-tile outputs leave by TMA stores
                                    // through WMaps::y (set only when every member's map exists)
    const float *x_scale;           // 8-bit path: per-token scale of X [M]
    const float *g_wscale[kMaxGroup];  // 8-bit path: per-row scale of each member's weight
    int groups;                     // members of the group (1 for a single weight)
    int g_tile0[kMaxGroup + 1];     // first n-tile of each member; g_tile0[groups] = n_tiles
    float *g_y[kMaxGroup];          // member outputs
    const uint8_t *g_wq[kMaxGroup]; // fused path: member raw streams
    int64_t g_N[kMaxGroup];         // member row counts
};

// Member of the group that owns n-tile nt.
__host__ __device__ inline int group_of(const GemmArgs &a, int nt)
{
    int g = 0;
    while (g + 1 < a.groups && nt >= a.g_tile0[g + 1])
        ++g;
    return g;
}

// Tokens per output box that the cached/e4m3 epilogue stores by TMA.
constexpr int kYBoxRows = 16;

// Tensor maps of the members of a group (one for a single weight): the
// f16 weight caches (m) and, for GEMMs launched with y_tma, the f32 outputs
// (y: [M, N_g], box 16 tokens x 128 rows, no swizzle).
struct WMaps {
    CUtensorMap m[kMaxGroup];
    CUtensorMap y[kMaxGroup];
};

// Raw-weight tensor maps of a weight whose rows start on block boundaries
// (K % 256 == 0): row n is RB = K/QK*bytes bytes long.  When RB is not a
// multiple of 16 (Q6_K), only every g-th row starts 16-byte aligned, so map
// c (c < g) covers the rows n = c + g*i with row stride g*RB and a base
// aligned down by (c*RB) % 16.  Elements are u16; a box is one 256-element
// chunk (plus the misalignment) of 128/g rows.
constexpr int kMaxRawMaps = 8;
struct RawMaps {
    CUtensorMap m[kMaxRawMaps];
};

// Raw-block tensor maps of the members of a fused group (one for a single
// weight); every member has the same type and K, so the same row classes.
struct RawMapsG {
    RawMaps w[kMaxGroup];
};

struct GemmPlan {
    int bn;              // tokens per tile (MMA N)
    int pair;            // 1: CTAs in clusters of two sharing the token tile
    int two_sm;          // with pair and bn = 256: 2-SM MMAs (M = 256 across the pair)
    int kb_align;        // split boundaries in K steps (4 for the fused path)
    int split;
    int full_tiles;
    int tiles;
    int units;
    int grid;
    int64_t ws_bytes;
};

// Choose tile width, split-K and grid for an M x N x K problem on `sms` SMs.
// bn_override > 0 forces the cached path's tile width (32, 64, 128 or 256).
// kstep: K elements per pipeline stage (64 for f16 operands, 128 for 8-bit).
// pair_clusters > 0: plan for CTA pairs (clusters of two sharing the token
// tile), at most pair_clusters of them resident; tiles, units and grid then
// count pair-major tiles, pair units and CTAs.
GemmPlan plan_gemm(int64_t M, int64_t N, int64_t K, int sms, bool fused, int64_t ws_available,
                   int bn_override = 0, int kstep = 64, int pair_clusters = 0);

// Workspace bytes the plan would use with an unlimited workspace.
int64_t plan_ws_bytes_wanted(int64_t M, int64_t N, int64_t K, int sms, bool fused, int bn_override = 0,
                             int kstep = 64, int pair_clusters = 0);

// The units every CTA of a planned launch runs, computed with the kernels'
// own schedule code: 8 ints per unit (cta, tile, nt, mt, kb0, kb1, part,
// slot), at most cap units written; returns the number of units.
int64_t schedule_units(const GemmPlan &p, int64_t M, int64_t N, int64_t K, int kstep, int32_t *out, int64_t cap);

// Clusters of two cached-GEMM CTAs (tile width bn, f16 or e4m3 operands,
// multicast pairs or 2-SM MMAs) that can be resident at once on the current
// device (0 if none).
int pair_clusters_for(int bn, bool e4m3, bool two_sm);

// Cached path: tm_w.m[g] maps member g's f16 cache [N_g, ldk_g] (box 64 x
// 128), tm_x maps X [M, K] (box 64 x bn).  All 128-byte swizzled.
cudaError_t launch_gemm_cached(const WMaps &tm_w, const CUtensorMap &tm_x, const GemmArgs &a,
                               const GemmPlan &p, cudaStream_t s);

// 8-bit path: the same GEMM on e4m3 operands (tm_w.m[g] maps member g's
// e4m3 copy [N_g, ldk8_g], box 128 x 128; tm_x maps X8 [M, K], box 128 x
// bn; 128-byte swizzle), Y = acc * g_wscale[g][n] * x_scale[m].
cudaError_t launch_gemm_e4m3(const WMaps &tm_w, const CUtensorMap &tm_x, const GemmArgs &a,
                             const GemmPlan &p, cudaStream_t s);

// Row-wise e4m3 quantization of an f16 matrix [rows, K] (row stride ld):
// codes into dst (row stride ldo bytes) and one f32 scale per row.
// K % 16 == 0, ld % 8 == 0, ldo % 16 == 0.
cudaError_t launch_quant_e4m3(const __half *src, int64_t rows, int64_t K, int64_t ld, uint8_t *dst, int64_t ldo,
                              float *scales, cudaStream_t s);

// Fused path: tm_x as above; the weight is read from a.wq, through `maps`
// when a.raw_g > 0.
cudaError_t launch_gemm_fused(const CUtensorMap &tm_x, const RawMapsG &maps, const GemmArgs &a, const GemmPlan &p,
                              cudaStream_t s);

// Build the raw-weight tensor maps of a block-aligned weight; returns g (0
// when the weight does not qualify: K % 256 != 0).
int encode_raw_maps(RawMaps *maps, const void *qdata, int type, int64_t N, int64_t K);

// Fixed-order sum of the split-K partial planes into Y.
cudaError_t launch_splitk_reduce(const GemmArgs &a, const GemmPlan &p, cudaStream_t s);

// The cached GEMM into caller-provided split-K scratch and status word,
// allocating nothing; MQ_ERR_SHAPE when the plan needs more than
// scratch_bytes.  Used by mq_gemm_noalloc.
int gemm_cached_into_scratch(const void *x, ::mq_weight *w, float *y, int64_t M, cudaStream_t s, float *scratch,
                             int64_t scratch_bytes, unsigned *status);

// Record `code` with a detail message (what, and the CUDA error if any) for
// mq_last_error_detail(); returns code.
int set_error(int code, const char *what, cudaError_t e);

// Read and clear the status word of mq_gemm_noalloc calls on the current
// device (0 when that entry point was never set up there).
unsigned noalloc_take_status();

// ---------------------------------------------------------------- tensor maps
// Encode a 2-D f16 row-major [rows, cols] tensor map with row stride `ld`
// elements, a box of box_cols x box_rows and 128-byte swizzle.
CUresult encode_f16_2d(CUtensorMap *map, const void *base, int64_t rows, int64_t cols, int64_t ld,
                       int box_cols, int box_rows);

// The same for a byte matrix (e4m3 codes): ld in bytes.
// Output map of a cached/e4m3 GEMM: f32 Y [rows = M, cols = N], row stride
// ld floats, box box_rows x 128.  Needs a 16-byte aligned base and ld % 4 == 0.
CUresult encode_f32_out_2d(CUtensorMap *map, void *base, int64_t rows, int64_t cols, int64_t ld, int box_rows);

// Fill maps.y and set a.y_tma for the members' outputs a.g_y / a.g_N (M
// tokens) when every output allows a TMA store (16-byte aligned base, N % 4
// == 0) and MQ_TMA_Y is not 0; otherwise a.y_tma = 0 (plain stores).
void set_output_maps(WMaps &maps, GemmArgs &a);

CUresult encode_u8_2d(CUtensorMap *map, const void *base, int64_t rows, int64_t cols, int64_t ld,
                      int box_cols, int box_rows);

}  // namespace mq
