/*
 * mq.h -- C ABI of the GB300 (sm_103a) quantized-weight prefill GEMM library.
 *
 * Computes the prefill matmul Y[M,N] = X[M,K] . W[N,K]^T where X is f16
 * activations, W is a GGUF weight (the block formats Q4_0, Q5_0, Q5_1, Q8_0,
 * Q4_K, Q5_K, Q6_K, or the float types F32 / F16 / BF16) and Y is f32.  Two
 * ways, both from the pages:
 *
 *   cached  W is decoded once, at registration, into a persistent f16 copy
 *           that a tensor-core GEMM then reads ("05 · 8p — Persistent f16
 *           weight cache + fused dequant-in-GEMM", sections 1-2; "ggml-cuda:
 *           GEMM weight row padding + one-time K-padded f16 dequant for
 *           prefill", Summary: the load-time K-padded f16 shadow).
 *   fused   the GEMM stages the raw quantized blocks on chip and decodes them
 *           to f16 right before the MMA ("05 · 8p", section 2, fused
 *           dequant-in-GEMM; section 3.2, third site).
 *
 * and an M gate that picks one per call ("ggml-cuda: GEMM weight row
 * padding ...", Summary: the token-count threshold GGML_PREFILL_DEQUANT).
 *
 * Conventions for every function below:
 *  - Return value: MQ_OK (0) or a negative MQ_ERR_* code.  No call aborts the
 *    process and no call falls back to the CPU.  mq_last_error_detail()
 *    names the argument and the reason of the last failure on this thread.
 *  - Pointers named x, y, qdata, out_f16 are DEVICE pointers owned by the
 *    caller; they must stay valid until the stream work that uses them has
 *    completed.  `stream` is a cudaStream_t (NULL = legacy default stream).
 *  - All device work is enqueued on `stream` in call order; no function
 *    except mq_stream_status() and mq_release_weight() synchronizes.
 *  - Layouts are row-major: X[M,K] with row stride K elements, Y[M,N] with
 *    row stride N elements.
 *  - Decoded weights match the block definitions bit for bit: each value is
 *    computed in f32 as d*sc*q - dmin*m (Q4_K), d*sc*q (Q6_K) or d*q (Q8_0)
 *    and rounded once to nearest-even f16 (the dequant kernel of "05 · 8p",
 *    section 3.2: f32 product, then __float2half).  The cached and the fused
 *    paths decode to identical f16 values (section 3.3 Pitfalls: the same
 *    rounding path).  The other formats follow the same rule (their value
 *    definitions are given with mq_type below).
 *
 * Environment switches (read on every call unless noted; tuning and
 * diagnostics only, never needed for correct results):
 *   MQ_M_GATE=n   mq_gemm_auto's token threshold (default 129: the fused path
 *                 up to M = 128, the measured crossover).
 *   MQ_PAIR=0     cached / e4m3 GEMMs without CTA pairs (default on: two CTAs
 *                 of a cluster share each token tile).
 *   MQ_2SM=0      256-token tiles as multicast CTA pairs instead of 2-SM MMAs
 *                 (tcgen05.mma.cta_group::2, the default).
 *   MQ_TMA_Y=0    cached / e4m3 GEMMs store whole output tiles with plain
 *                 stores instead of TMA stores of staged boxes (default on
 *                 where Y is 16-byte aligned and N % 4 == 0).
 *   MQ_SPLITK=0   no split-K tail (default on).
 *   MQ_BN=32|64|128|256   force the cached GEMM's token-tile width.
 *   MQ_PDL=0      launch without programmatic dependent launch (default on;
 *                 read once, at the first launch).
 *   MQ_KPAD=0|1   cache row padding never / always (default: the 2048-byte
 *                 rule; the MQ_REG_* flags take precedence).
 *   MQ_RAW_TMA=0  the fused path reads raw blocks by per-row bulk copies even
 *                 when row tensor maps apply (at registration).
 *   MQ_LOG=1      one line per registration and GEMM plan on stderr (read
 *                 once).
 * Test-only failure injection (leave unset): MQ_FAULT_ALLOC=1 makes
 * registration's cache allocation fail (MQ_ERR_OOM); MQ_INJECT_PRODUCER_STALL=1
 * stops a GEMM's weight producer so its bounded waits time out (the kernel
 * exits cleanly and mq_stream_status() reports MQ_ERR_DEVICE).
 */
#ifndef MQ_H
#define MQ_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* GGUF type ids of the supported weight types.  The pages name the types;
 * field layouts are the GGUF convention ("05 · 8p — Persistent f16 weight
 * cache + fused dequant-in-GEMM", sections 1-2 give Q5_0's fields and the
 * block sizes).  The float types are the ones whose rows "ggml-cuda: GEMM
 * weight row padding + one-time K-padded f16 dequant for prefill", Summary,
 * pads (F16 / BF16 / F32): a block of one element, its f16 value the
 * element rounded to nearest even (a NaN stays a NaN, payload not kept). */
typedef enum {
    MQ_TYPE_F32 = 0,    /* 4-byte IEEE binary32, row-major [N, K]                     */
    MQ_TYPE_F16 = 1,    /* 2-byte IEEE binary16, row-major [N, K]                     */
    MQ_TYPE_Q4_0 = 2,   /* 32 elements in 18 bytes: f16 d, 16 B of 4-bit quants (q - 8) */
    MQ_TYPE_Q5_0 = 6,   /* 32 elements in 22 bytes: f16 d, 4 B fifth-bit plane, 16 B of
                           low 4 bits (q - 16); 2-byte aligned blocks                   */
    MQ_TYPE_Q5_1 = 7,   /* 32 elements in 24 bytes: f16 d, f16 m, 4 B fifth-bit plane,
                           16 B of low 4 bits (d*q + m)                                */
    MQ_TYPE_Q8_0 = 8,   /* 32 elements in 34 bytes: f16 d, int8 q[32]                 */
    MQ_TYPE_Q4_K = 12,  /* 256 elements in 144 bytes: f16 d, f16 dmin, 12 B of 6-bit
                           scales/mins, 128 B of 4-bit quants                          */
    MQ_TYPE_Q5_K = 13,  /* 256 elements in 176 bytes: as Q4_K plus 32 B of fifth bits
                           (bit s of byte i belongs to sub-block s, position i)        */
    MQ_TYPE_Q6_K = 14,  /* 256 elements in 210 bytes: 128 B low nibbles, 64 B high
                           2-bit fields, 16 int8 scales, f16 d                          */
    MQ_TYPE_BF16 = 30   /* 2-byte bfloat16 (the top half of a binary32), [N, K]      */
} mq_type;

/* Status codes. */
#define MQ_OK                    0
#define MQ_ERR_INVALID          -1  /* null pointer, unknown or released handle, bad flag  */
#define MQ_ERR_UNSUPPORTED_TYPE -2  /* type id is not one of the mq_type weight types       */
#define MQ_ERR_SHAPE            -3  /* a size precondition does not hold                   */
#define MQ_ERR_ALIGN            -4  /* a pointer is not 16-byte aligned                    */
#define MQ_ERR_NO_CACHE         -5  /* mq_gemm on a handle registered with MQ_REG_NO_CACHE */
#define MQ_ERR_OOM              -6  /* device allocation failed                            */
#define MQ_ERR_CUDA             -7  /* a CUDA runtime/driver call failed (detail has it)   */
#define MQ_ERR_DEVICE           -8  /* a kernel flagged a device-side error (timeout)      */
#define MQ_ERR_NO_DEVICE        -9  /* no usable sm_103 device / kernel image              */

/* Registration flags. */
#define MQ_REG_NO_CACHE 0x1u  /* build no f16 cache: only fused calls on this handle     */
#define MQ_REG_NO_KPAD  0x2u  /* cache row stride ldk = K even when 2K % 2048 == 0       */
#define MQ_REG_KPAD     0x4u  /* force ldk = K + 64                                      */
#define MQ_REG_E4M3     0x8u  /* also build the e4m3 copy read by mq_gemm_e4m3           */

typedef struct mq_weight *mq_handle;

/*
 * mq_register_weight -- take a quantized weight and (unless MQ_REG_NO_CACHE)
 * decode it once into a persistent f16 cache.
 *
 * Passage: "05 · 8p", section 3.1 (dequantize at load in the warm pass, the
 * f16 copy stays resident) and section 2 (weights are immutable after load,
 * so the pointer can key the cache); "ggml-cuda: GEMM weight row padding ...",
 * Summary (the shadow is K-padded by one 128-byte line only when its f16 row
 * size is a multiple of 2048 bytes; allocation failure is reported at load,
 * Known limitation).
 *
 *  type   block format.
 *  qdata  device pointer to ONE flat stream of N*K/QK consecutive blocks;
 *         element (n,k) is flat element n*K+k (rows may start inside a
 *         block when K % QK != 0).  16-byte aligned.  Caller-owned: it must
 *         stay valid and UNCHANGED for the lifetime of the handle, because
 *         fused calls read it on every call.
 *  N, K   weight rows (output features) and columns (input features).
 *         Requires N >= 1, K >= 8, K % 8 == 0, N*K % QK == 0.
 *  flags  MQ_REG_* bits.
 *  stream decode kernels are enqueued here; the cache is ready when this
 *         stream's work up to this call has completed.
 *  out    receives the handle.
 *
 * Cache layout: f16 [N, ldk] row-major, ldk = K + 64 if (2K) % 2048 == 0
 * (K % 1024 == 0) else K; the pad columns hold +0.0.  The cache is
 * library-owned and freed by mq_release_weight().
 *
 * Float weights (F32 / F16 / BF16; qdata is then the row-major [N, K]
 * matrix): the cache is the weight converted to f16 with the same row
 * padding.  An F16 weight whose rows need no padding (ldk == K, or
 * MQ_REG_NO_KPAD, or MQ_REG_NO_CACHE) is read in place: no copy is made,
 * mq_weight_info() returns qdata as the cache, and release frees nothing.
 * F32 and BF16 always get the f16 copy (MQ_REG_NO_CACHE is MQ_ERR_INVALID).
 * mq_gemm_fused() on a float weight runs the cached GEMM (there is nothing
 * to decode on chip).
 * Errors: MQ_ERR_UNSUPPORTED_TYPE, MQ_ERR_SHAPE, MQ_ERR_ALIGN, MQ_ERR_INVALID,
 * MQ_ERR_OOM (nothing is left allocated), MQ_ERR_CUDA.
 */
int mq_register_weight(mq_type type, const void *qdata, int64_t N, int64_t K,
                       uint32_t flags, void *stream, mq_handle *out);

/* Free the handle and its f16 cache (synchronizes the device first so no
 * enqueued call still reads it).  Never touches qdata.  Errors: MQ_ERR_INVALID. */
int mq_release_weight(mq_handle w);

/* Query a handle.  Any output pointer may be NULL.  *f16_cache is NULL for a
 * MQ_REG_NO_CACHE handle.  Errors: MQ_ERR_INVALID. */
int mq_weight_info(mq_handle w, int64_t *N, int64_t *K, int64_t *ldk,
                   const void **f16_cache);

/*
 * mq_dequantize -- decode a flat block stream into f16 W[N,K] with row
 * stride ldo (>= K, ldo % 8 == 0).  Columns [K, ldo) are left untouched.
 * This is the decoder the cache is built with, exposed on its own.
 * Passage: "05 · 8p", section 3.2, second site (the dequant kernel; 2-byte
 * aligned blocks are read without wider misaligned loads).
 * qdata and out_f16 are device pointers, 16-byte aligned.
 * Errors: MQ_ERR_UNSUPPORTED_TYPE, MQ_ERR_SHAPE, MQ_ERR_ALIGN, MQ_ERR_INVALID,
 * MQ_ERR_CUDA.
 */
int mq_dequantize(mq_type type, const void *qdata, int64_t N, int64_t K,
                  void *out_f16, int64_t ldo, void *stream);

/*
 * mq_gemm -- cached path: Y[M,N] = X[M,K] . Wc[:, :K]^T with the f16 cache,
 * f16 x f16 products accumulated in f32 on the tensor cores ("05 · 8p",
 * section 2, persistent f16 cache; "Eager GPU Offload Without A Compute
 * Graph", section "Storage and transfer reuse": f16 inputs, f32 output; when
 * the output grid underfills the GPU, K is split and the partial planes are
 * reduced in a fixed order on the same stream).
 *  x  device f16 [M,K], 16-byte aligned.   y  device f32 [M,N], 16-byte aligned.
 *  M  number of tokens, M >= 1.
 * Results are bitwise reproducible from call to call for the same M.
 * Errors: MQ_ERR_INVALID, MQ_ERR_NO_CACHE, MQ_ERR_SHAPE, MQ_ERR_ALIGN,
 * MQ_ERR_OOM (split-K workspace), MQ_ERR_CUDA.
 */
int mq_gemm(const void *x, mq_handle w, float *y, int64_t M, void *stream);

/*
 * mq_gemm_fused -- fused path: same Y, decoding the raw blocks of qdata on
 * chip into the f16 MMA operand ("05 · 8p", section 2: B tiles staged as
 * quantized bytes and dequantized before the MMA; zero extra VRAM).  The
 * on-chip decode produces the same f16 values as the cache.
 * Extra preconditions: K % 64 == 0 (a 64-element K chunk never straddles a
 * block); when K % 256 != 0 (rows start inside blocks) the stream length
 * (N*K/QK blocks times the block bytes) must also be a multiple of 16 bytes.
 * Errors as mq_gemm, minus MQ_ERR_NO_CACHE.
 */
int mq_gemm_fused(const void *x, mq_handle w, float *y, int64_t M, void *stream);

/*
 * mq_gemm_grouped -- the cached GEMM for `count` (1..4) weights that share K
 * and the activations X, in one launch: y[g][M, N_g] = X . W_g^T for every
 * member g.  ("Eager GPU Offload Without A Compute Graph", section "Storage
 * and transfer reuse": a shared-input batch runs several weight matrices on
 * the same activation rows without replicating them; here they also share
 * one persistent tile schedule, so small members such as the k and v
 * projections fill the GPU together with q instead of each needing split-K.)
 *
 * Arguments: x as for mq_gemm; w[0..count) handles registered with an f16
 * cache, all with the same K and on the same device; y[0..count) caller-owned
 * f32 outputs, y[g] of M x N_g, row-major, 16-byte aligned.  The members'
 * outputs equal what mq_gemm computes for each, up to f32 summation order
 * (a member may be split over K differently).  When every N_g is a multiple
 * of 128 the call is one GEMM launch (plus one split-K reduction when the
 * tile grid's last wave is split); otherwise the members run one after
 * another with mq_gemm.
 * Errors: MQ_ERR_INVALID (w or y NULL, count out of range, stale handle,
 * members on different devices), MQ_ERR_NO_CACHE, MQ_ERR_SHAPE (K differs,
 * bad M), MQ_ERR_ALIGN, and the errors of mq_gemm.  Nothing is launched when
 * an argument check fails.
 */
int mq_gemm_grouped(const void *x, const mq_handle *w, int count, float *const *y, int64_t M, void *stream);

/*
 * mq_gemm_fused_grouped -- the fused path for `count` (1..4) weights that
 * share K and X, in one launch: y[g][M, N_g] = X . W_g^T, every member's raw
 * blocks decoded on chip as in mq_gemm_fused (the same f16 values as the
 * cache).  The shared-input batch of mq_gemm_grouped ("Eager GPU Offload
 * Without A Compute Graph", section "Storage and transfer reuse") on the
 * raw-block path: at small M, where each fused launch pays a fixed ramp-up
 * of its weight stream, q|k|v or gate|up then pay it once.
 *
 * Arguments: as mq_gemm_grouped, but the handles need no f16 cache
 * (MQ_REG_NO_CACHE is fine) and all members have the same block format.
 * One launch when every N_g is a multiple of 128 (plus one split-K
 * reduction when the last wave is split); otherwise the members run one
 * after another with mq_gemm_fused.  Float weights (F32/F16/BF16) have
 * nothing to decode: the call is then mq_gemm_grouped.  The outputs equal
 * what mq_gemm_fused computes for each member, up to f32 summation order.
 * Errors: MQ_ERR_INVALID (w or y NULL, count out of range, stale handle,
 * members on different devices or of different types), MQ_ERR_SHAPE (K
 * differs, bad M, the fused path's K and stream-length conditions),
 * MQ_ERR_ALIGN, MQ_ERR_OOM (split-K workspace), MQ_ERR_CUDA.  Nothing is
 * launched when an argument check fails.
 */
int mq_gemm_fused_grouped(const void *x, const mq_handle *w, int count, float *const *y, int64_t M, void *stream);

/*
 * mq_gemm_auto_grouped -- the M gate of mq_gemm_auto for a group: below the
 * gate (mq_get_m_gate()), when every member can take the fused path (one
 * block format, the fused path's K and stream-length conditions), the call
 * is mq_gemm_fused_grouped; at and above it mq_gemm_grouped.  A member
 * registered without an f16 cache sends the whole group to
 * mq_gemm_fused_grouped.  Arguments, results and errors: those of the call
 * it makes.
 */
int mq_gemm_auto_grouped(const void *x, const mq_handle *w, int count, float *const *y, int64_t M, void *stream);

/*
 * mq_gemm_auto -- M gate: fused when M < gate (and the handle allows it),
 * cached otherwise ("ggml-cuda: GEMM weight row padding ...", Summary: the
 * f16 path is a large-batch win; the threshold is a token count per call).
 * The gate is mq_get_m_gate(); environment variable MQ_M_GATE overrides it.
 * Default 129: measured on GB300, calls back to back over weights larger than
 * L2, the fused path is faster up to M = 128 and the cached path from M = 129
 * on the 7B gate, down and o shapes, the Q8_0 pair and the Llama-3.1-8B gate
 * (the fused path's token tiles stop at 128, so past that it decodes each
 * weight tile once per token tile).
 */
int mq_gemm_auto(const void *x, mq_handle w, float *y, int64_t M, void *stream);

/*
 * mq_gemm_scratch -- per-call dequant: decode the weight's raw blocks into
 * the caller's f16 scratch, then run the cached GEMM on it, both on
 * `stream`.  Same Y as mq_gemm (the scratch holds the values the cache
 * would).  Works on any handle, with or without a cache.
 * Passage: "05 · 8p", the time-vs-memory triangle and its per-call mode
 * (the weight is re-dequantized into an f16 scratch on every call and the
 * GEMM reads the scratch; it saves the resident copy and costs one decode
 * pass per call).
 *
 *  scratch        device memory, 16-byte aligned, caller-owned, at least
 *                 2*N*ldk bytes (ldk from mq_weight_info); its contents on
 *                 return are the decoded weight in the cache layout (pad
 *                 columns not written).  Calls that overlap on the device
 *                 must not share one scratch.
 *  scratch_bytes  its size.
 * Errors: as mq_gemm (minus MQ_ERR_NO_CACHE), MQ_ERR_INVALID (scratch NULL),
 * MQ_ERR_ALIGN, MQ_ERR_SHAPE (scratch_bytes < 2*N*ldk).
 */
int mq_gemm_scratch(const void *x, mq_handle w, float *y, int64_t M, void *scratch,
                    int64_t scratch_bytes, void *stream);

/*
 * The 8-bit variant.  Passage: "Eager GPU Offload Without A Compute Graph",
 * section "F16 and GGUF quantized linears" (the activation-quantized MMQ
 * path: quantize each activation tile once to an 8-bit layout with scales,
 * run the MMA on 8-bit operands; a separate numeric contract).  On this GPU
 * the 8-bit operands are e4m3 floats (OCP: bias 7, 3 mantissa bits, largest
 * finite 448) with one binary32 scale per row:
 *
 *     amax = max |v| over the row,  s = RN32(amax / 448),
 *     code = e4m3_rn_satfinite(RN32(v * RN32(448 / amax)))
 *
 * (s = 1 and all codes 0 for an all-zero row), and
 *
 *     Y[m, n] = RN32(RN32(acc[m, n] * sw[n]) * sx[m]),
 *     acc = sum_k x8[m, k] * w8[n, k] with f32 accumulation.
 *
 * The result differs from mq_gemm's by the quantization error (a few
 * percent, relative); it is a separate contract, checked against the exact
 * product of the quantized operands.  Inputs must be finite.
 *
 * mq_quantize_e4m3 -- quantize rows of an f16 matrix.
 *  x       f16 [rows, K], row stride ld (ld >= K, ld % 8 == 0), device,
 *          16-byte aligned.
 *  dst     e4m3 codes [rows, K], row stride ldo bytes (ldo >= K, ldo % 16
 *          == 0), device, 16-byte aligned; columns past K are not written.
 *  scales  f32 [rows], device, 4-byte aligned.
 *  K % 16 == 0.  Errors: MQ_ERR_INVALID, MQ_ERR_SHAPE, MQ_ERR_ALIGN,
 *  MQ_ERR_CUDA.
 */
int mq_quantize_e4m3(const void *x, int64_t rows, int64_t K, int64_t ld, void *dst, int64_t ldo,
                     float *scales, void *stream);

/*
 * mq_gemm_e4m3 -- Y = (x8 . w8^T) * sw[n] * sx[m] (see above) on the weight's
 * e4m3 copy (registered with MQ_REG_E4M3: the f16 cache quantized per row,
 * rows padded by 128 bytes when K % 2048 == 0).
 *  x8       e4m3 codes [M, K], row stride K (from mq_quantize_e4m3 with
 *           ldo = K), device, 16-byte aligned.
 *  x_scale  f32 [M], device.
 *  y        f32 [M, N].
 * Same stream, workspace and split-K behaviour as mq_gemm.  Errors:
 * MQ_ERR_INVALID, MQ_ERR_NO_CACHE (no e4m3 copy), MQ_ERR_SHAPE,
 * MQ_ERR_ALIGN, MQ_ERR_OOM (split-K workspace), MQ_ERR_CUDA.
 */
int mq_gemm_e4m3(const void *x8, const float *x_scale, mq_handle w, float *y, int64_t M, void *stream);

/* mq_gemm_e4m3 for `count` (1..4) weights sharing K and the quantized X:
 * y[g] = the member-g product, one launch when every N is a multiple of 128
 * (else one after another), as mq_gemm_grouped.  Errors: those of
 * mq_gemm_grouped, MQ_ERR_NO_CACHE for a member without an e4m3 copy. */
int mq_gemm_e4m3_grouped(const void *x8, const float *x_scale, const mq_handle *w, int count, float *const *y,
                         int64_t M, void *stream);

/* The weight's e4m3 copy: row stride ldk8 (bytes), codes [N, ldk8] and
 * scales [N] (NULL without MQ_REG_E4M3).  Any output may be NULL.
 * Errors: MQ_ERR_INVALID. */
int mq_weight_e4m3_info(mq_handle w, int64_t *ldk8, const void **codes, const float **scales);

/*
 * mq_debug_schedule -- the work plan of one GEMM launch, for tests and
 * tuning; host only, launches nothing, needs no device.
 *  M, N, K, sms   the problem and the SM count to plan for.
 *  path           0 cached f16, 1 fused, 2 e4m3.
 *  pair_clusters  > 0: plan CTA pairs with this many resident clusters
 *                 (ignored for the fused path); 0: single CTAs.
 *  plan_out       9 values: tile width, pair flag, split, full tiles,
 *                 tiles, units, grid, split-K workspace bytes, split
 *                 alignment in K steps.
 *  units          receives up to cap units, 8 int32 each: CTA, tile,
 *                 weight-row tile, token tile, first and end K step, split
 *                 part (-1: whole K), workspace slot.
 *  count          the number of units the CTAs run (may exceed cap).
 * The kernels' own schedule code computes it.  Errors: MQ_ERR_INVALID.
 */
int mq_debug_schedule(int64_t M, int64_t N, int64_t K, int sms, int path, int pair_clusters, int64_t *plan_out,
                      int32_t *units, int64_t cap, int64_t *count);

/*
 * mq_debug_cvt_f16 -- test hook for the decoders' last step, the f32 -> f16
 * rounding (round to nearest even, subnormals kept, sign of zero kept:
 * "05 · 8p — Persistent f16 weight cache + fused dequant-in-GEMM",
 * section 3.3 Pitfalls, the fused and cached decodes must round through the
 * same path).  Writes to out[i] (device, uint16, count elements) the f16
 * bits that the decoders' own packed conversion gives for the binary32 bit
 * pattern first + i.  first and count must be even and first + count <=
 * 2^32; out 4-byte aligned.  Stream-ordered.  Errors: MQ_ERR_INVALID,
 * MQ_ERR_SHAPE, MQ_ERR_ALIGN, MQ_ERR_CUDA.
 */
int mq_debug_cvt_f16(uint32_t first, int64_t count, void *out, void *stream);

/*
 * mq_gemm_noalloc -- the cached GEMM, same arguments as mq_gemm, for
 * callers that cannot allocate device memory: engines and serving runtimes
 * whose own pool reserves the device's memory up front and forbids any
 * other allocation, and latency-critical paths that must not risk the
 * implicit device synchronization a cudaMalloc or cudaFree can cause.
 * mq_gemm may grow its split-K scratch with cudaMalloc on first use; this
 * entry point never calls cudaMalloc, cudaFree or any allocating routine.
 * No page describes it: the pages have no counterpart, it is this library's
 * own addition.
 *
 * Result: within the GEMM tolerance of mq_gemm, not bit for bit.  It runs
 * the single-CTA plan (no CTA pairs, no 2-SM MMAs) with its split-K tail
 * bounded by the scratch below, so its summation order can differ; the
 * tuning switches MQ_SPLITK, MQ_BN, MQ_PAIR and MQ_2SM do not apply to it
 * (MQ_TMA_Y does: the output path is the same kernel's).
 *
 * Its split-K scratch is one 16 MiB file-scope device array, which every GPU
 * that loads this library holds until the process exits.  A call whose split
 * plan needs more than 16 MiB fails with MQ_ERR_SHAPE and says so (at
 * M = 2048 that is the case for a 3584-row weight, for example).  The first
 * call on each device does a one-time set-up: it looks up the array's device
 * address (with that device current).  Make that first call before any
 * stream capture.  All calls share the array, so calls that overlap on the
 * GPU (different streams, or graphs replayed concurrently) race and must be
 * serialized by the caller.  Every call writes all the scratch it reads
 * before reading it, so nothing needs clearing between calls.  Device-side
 * timeouts of these calls are reported by mq_stream_status (whose own first
 * call on a device does allocate).
 * Errors: as mq_gemm, plus MQ_ERR_SHAPE when the scratch is too small.
 */
int mq_gemm_noalloc(const void *x, mq_handle w, float *y, int64_t M, void *stream);

/* Current M gate and a setter (value >= 1). */
int64_t mq_get_m_gate(void);
int mq_set_m_gate(int64_t m);

/*
 * mq_reserve_workspace -- grow the library's split-K workspace to at least
 * `bytes` on the current device (never shrinks).  Call it before capturing
 * mq_gemm* into a CUDA graph: inside a capture the library never allocates
 * and, if the workspace is too small, it runs without split-K instead.
 * The workspace serves one stream at a time: calls on different streams
 * that overlap on the device must not share it.  Errors: MQ_ERR_OOM.
 */
int mq_reserve_workspace(int64_t bytes);

/*
 * mq_stream_status -- synchronize `stream`, then read and clear the
 * library's device status word.  MQ_ERR_DEVICE if a kernel gave up on a
 * bounded wait (every pipeline wait in the library's kernels has a time
 * limit, after which the kernel records the error and exits cleanly instead
 * of hanging); MQ_ERR_CUDA if the CUDA context reports an error (sticky
 * errors are reported, not cleared: "Eager GPU Offload Without A Compute
 * Graph", section "Ordering and unavoidable synchronization" -- a deferred
 * device error found at the host boundary is fatal).
 */
int mq_stream_status(void *stream);

/* Number of kernel launches the library has made since load (all kinds). */
int64_t mq_launch_count(void);

/*
 * Launch tracing.  While enabled, every mq_gemm / mq_gemm_fused call (and the
 * decode of mq_register_weight) records CUDA events on the caller's stream
 * around its main kernel and around its split-K reduce, so the device time
 * of each kernel can be read back.  No page prints this; it is the library's
 * own measurement hook.  Calls made while the stream is being captured into
 * a CUDA graph are not traced.  At most 1 << 16 calls are kept.
 */
typedef struct {
    int32_t kind;      /* MQ_TRACE_* */
    int32_t type;      /* GGUF type id of the weight */
    int64_t M, N, K;
    float ms_main;     /* device time of the GEMM or decode kernel */
    float ms_aux;      /* device time of the split-K reduce (0 if none) */
} mq_trace_record;

#define MQ_TRACE_GEMM_CACHED 1
#define MQ_TRACE_GEMM_FUSED  2
#define MQ_TRACE_DECODE      3

/* Enable (clears earlier records) or disable recording. */
int mq_trace_enable(int on);
/* Number of records kept since the last enable. */
int64_t mq_trace_count(void);
/* Read record i (synchronizes its events).  Errors: MQ_ERR_INVALID, MQ_ERR_CUDA. */
int mq_trace_read(int64_t i, mq_trace_record *out);

/* Static description of a status code. */
const char *mq_error_string(int status);

/* Detail of the last failure on the calling thread (argument and reason). */
const char *mq_last_error_detail(void);

/* Library version: major*10000 + minor*100 + patch. */
int mq_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MQ_H */
