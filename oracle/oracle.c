/*
 * oracle.c -- plain, slow, obviously-correct CPU oracle for the GGUF
 * quantized-weight prefill GEMM  Y[M,N] = X[M,K] . W[N,K]^T.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this library.  The product path
 * (the CUDA library) shares no code, header, table or helper with it.
 *
 * What it computes, and the passage each part follows:
 *
 *  O1  binary16 <-> binary32 conversion, written from the IEEE 754 binary16
 *      definition: round-to-nearest-even, gradual underflow, signed zeros.
 *      The pages round every dequantized value through __float2half, which
 *      is round-to-nearest-even ("05 · 8p — Persistent f16 weight cache +
 *      fused dequant-in-GEMM", section 3.3 Pitfalls: the same rounding path).
 *
 *  O2  Block decoders Q8_0 / Q4_K / Q6_K -> binary16.  The pages name the
 *      types and their bytes per weight only ("05 · 8p", section 1); the
 *      block sizes 34 / 144 / 210 bytes and the field layout follow the
 *      GGUF format convention (a reading: no page prints the layout).
 *      Also Q4_0 / Q5_0 / Q5_1 / Q5_K (18 / 22 / 24 / 176 bytes): the pages
 *      give Q5_0's fields (f16 d, 4-byte qh bit plane, 16 nibble bytes;
 *      "05 · 8p", section 2) and Q5_1's size, and name Q4_0 and Q5_K's
 *      bit-transposed qh ("79 · Phase-8 coverage & first-measurement
 *      batch", section 3.4); the rest of each layout is the GGUF convention.
 *      Arithmetic is binary32 in the fixed order d*sc*q - dmin*m, then one
 *      round-to-nearest to binary16, as the dequant kernel shown in
 *      "05 · 8p", section 3.2 does (f32 product, then __float2half).
 *      The weight is one flat stream of N*K elements in consecutive blocks;
 *      element (n,k) is flat index n*K+k, so a row may start inside a block.
 *
 *  O2f Float weights F32 / F16 / BF16 (GGUF ids 0 / 1 / 30), the types whose
 *      rows "ggml-cuda: GEMM weight row padding + one-time K-padded f16
 *      dequant for prefill" pads (Summary): one element per "block" (4 / 2
 *      / 2 bytes, little-endian), y = RN16(value).  An F16 element is its
 *      own value; a BF16 element is the upper half of a binary32 whose lower
 *      half is zero, widened exactly and then rounded as an F32 element is.
 *
 *  O5  The 8-bit variant (the MMQ idea of "Eager GPU Offload Without A
 *      Compute Graph", section "F16 and GGUF quantized linears": quantize
 *      the activations once per call, run the MMA on 8-bit operands, scale
 *      afterwards; with e4m3 floats in place of int8).  e4m3 is the OCP
 *      8-bit float: sign, 4 exponent bits (bias 7), 3 mantissa bits, no
 *      infinities, the all-ones code the only NaN (largest finite 448),
 *      subnormals m * 2^-9.  A row of f16 values gets one binary32 scale
 *      s = RN32(amax / 448) and codes e4m3(RN32(v * RN32(448 / amax)))
 *      (s = 1 for an all-zero row); rounding to e4m3 is to nearest even on
 *      the exact value, finite values past 448 clamp to 448.  The variant's
 *      product is Y[m,n] = (sum_k x8[m,k] * w8[n,k]) * sw[n] * sx[m], here
 *      in f64.  Inputs are assumed finite.
 *
 *  O4  GEMM with f64 accumulation in k order: Y[m,n] = sum_k X[m,k]*W[n,k]
 *      for f16 X and the f16 dequantized W, the product the pages check
 *      their kernels against ("Eager GPU Offload Without A Compute Graph",
 *      section "F16 and GGUF quantized linears": an explicitly dequantized
 *      reference).
 *
 * Build: gcc -O2 -ffp-contract=off -fno-fast-math -fopenmp -shared -fPIC.
 * Contraction stays off so every binary32 product and difference is
 * rounded exactly where the C source says.
 */
#include <stdint.h>
#include <stddef.h>
#include <stdlib.h>
#include <string.h>
#include <math.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------ */
/* O1: binary16 <-> binary32                                          */
/* ------------------------------------------------------------------ */

/* binary16 -> binary32, exact: a normal value is (1024+m) * 2^(e-25), a
 * subnormal one m * 2^-24. */
float oracle_f16_to_f32(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int m = h & 0x3ff;
    double v;
    if (e == 0x1f) {
        if (m != 0) return sign ? -NAN : NAN;
        v = INFINITY;
    } else if (e == 0) {
        v = ldexp((double)m, -24);
    } else {
        v = ldexp((double)(m + 1024), e - 25);
    }
    return (float)(sign ? -v : v);
}

/* binary32 -> binary16, round to nearest, ties to even.
 * The binary32 value is sig * 2^(e-23) with sig its 24-bit significand
 * (implicit bit included for normals).  The binary16 quantum at that
 * magnitude is 2^(max(e,-14)-10), so 13 + max(-14-e, 0) low bits of sig
 * are rounded away, leaving q.  A normal result encodes as
 * ((e+15)<<10) + (q-1024): a carry out of the significand lands in the
 * exponent field by itself.  A subnormal result encodes as q (q == 1024 is
 * the smallest normal).  Encodings >= 0x7c00 overflow to infinity.  NaNs
 * stay NaNs (quiet bit set, top payload bits kept). */
uint16_t oracle_f32_to_f16(float f)
{
    uint32_t x;
    memcpy(&x, &f, 4);
    uint16_t sign = (uint16_t)((x >> 16) & 0x8000u);
    int ex = (int)((x >> 23) & 0xff);
    uint32_t man = x & 0x7fffffu;

    if (ex == 0xff)
        return man ? (uint16_t)(sign | 0x7e00u | (man >> 13)) : (uint16_t)(sign | 0x7c00u);

    uint64_t sig = ex ? (man | 0x800000u) : man;
    int e = ex ? ex - 127 : -126;
    if (e >= 16)
        return (uint16_t)(sign | 0x7c00u);

    int shift = 13 + (e < -14 ? -14 - e : 0);
    uint64_t q = 0;
    if (shift < 40) {
        uint64_t rem = sig & ((1ull << shift) - 1);
        uint64_t half = 1ull << (shift - 1);
        q = sig >> shift;
        if (rem > half || (rem == half && (q & 1)))
            q++;
    }
    uint32_t enc = (e < -14) ? (uint32_t)q
                             : (uint32_t)((e + 15) << 10) + (uint32_t)(q - 1024);
    if (enc >= 0x7c00u)
        enc = 0x7c00u;
    return (uint16_t)(sign | enc);
}

/* ------------------------------------------------------------------ */
/* O2: block decoders                                                 */
/* ------------------------------------------------------------------ */

enum { T_F32 = 0, T_F16 = 1, T_Q4_0 = 2, T_Q5_0 = 6, T_Q5_1 = 7, T_Q8_0 = 8, T_Q4_K = 12, T_Q5_K = 13,
       T_Q6_K = 14, T_BF16 = 30 };

static uint16_t rd_u16le(const uint8_t *p) { return (uint16_t)(p[0] | (p[1] << 8)); }

/* Q8_0, 34 bytes: d (f16) at byte 0, q[32] (int8) at byte 2.
 * y_e = RN16(d * q_e). */
static void decode_q8_0_block(const uint8_t *b, uint16_t *y)
{
    float d = oracle_f16_to_f32(rd_u16le(b));
    for (int e = 0; e < 32; e++) {
        float q = (float)(int8_t)b[2 + e];
        y[e] = oracle_f32_to_f16(d * q);
    }
}

/* Q4_K 6-bit scale and min of sub-block s (0..7) from the 12 packed bytes S:
 *   s <  4: sc = S[s] & 63,                         m = S[s+4] & 63
 *   s >= 4: sc = (S[s+4] & 15) | (S[s-4] >> 6) << 4, m = (S[s+4] >> 4) | (S[s] >> 6) << 4 */
static void q4k_scale_min(const uint8_t *S, int s, int *sc, int *m)
{
    if (s < 4) {
        *sc = S[s] & 63;
        *m = S[s + 4] & 63;
    } else {
        *sc = (S[s + 4] & 15) | ((S[s - 4] >> 6) << 4);
        *m = (S[s + 4] >> 4) | ((S[s] >> 6) << 4);
    }
}

/* Q4_K, 144 bytes: d (f16) at 0, dmin (f16) at 2, S[12] at 4, qs[128] at 16.
 * Group p = 0..3 covers elements 64p .. 64p+63: element 64p+i (i < 32) is
 * the low nibble of qs[32p+i] and belongs to sub-block 2p; element
 * 64p+32+i is the high nibble of the same byte, sub-block 2p+1.
 *   y = RN16( RN32( RN32(RN32(d*sc)*q) - RN32(dmin*m) ) ) */
static void decode_q4_K_block(const uint8_t *b, uint16_t *y)
{
    float d = oracle_f16_to_f32(rd_u16le(b));
    float dmin = oracle_f16_to_f32(rd_u16le(b + 2));
    const uint8_t *S = b + 4;
    const uint8_t *qs = b + 16;
    for (int e = 0; e < 256; e++) {
        int p = e / 64;
        int hi = (e % 64) >= 32;
        int i = e % 32;
        int s = 2 * p + hi;
        int q = hi ? (qs[32 * p + i] >> 4) : (qs[32 * p + i] & 15);
        int sc, m;
        q4k_scale_min(S, s, &sc, &m);
        float a = (d * (float)sc) * (float)q;
        float c = dmin * (float)m;
        y[e] = oracle_f32_to_f16(a - c);
    }
}

/* Q6_K, 210 bytes: ql[128] at 0, qh[64] at 128, sc[16] (int8) at 192,
 * d (f16) at 208.  Half h (0,1) covers elements 128h .. 128h+127 and reads
 * L = ql + 64h, H = qh + 32h.  For l = 0..31:
 *   element 128h + l      : (L[l]    & 15) | ((H[l] >> 0) & 3) << 4
 *   element 128h + l + 32 : (L[l+32] & 15) | ((H[l] >> 2) & 3) << 4
 *   element 128h + l + 64 : (L[l]    >> 4) | ((H[l] >> 4) & 3) << 4
 *   element 128h + l + 96 : (L[l+32] >> 4) | ((H[l] >> 6) & 3) << 4
 * q6 = value - 32, its scale is sc[e/16], and
 *   y = RN16( RN32(RN32(d*sc)*q6) ) */
static void decode_q6_K_block(const uint8_t *b, uint16_t *y)
{
    const uint8_t *ql = b;
    const uint8_t *qh = b + 128;
    const int8_t *sc = (const int8_t *)(b + 192);
    float d = oracle_f16_to_f32(rd_u16le(b + 208));
    for (int e = 0; e < 256; e++) {
        int h = e / 128;
        int r = e % 128;
        int quarter = r / 32;
        int l = r % 32;
        const uint8_t *L = ql + 64 * h;
        const uint8_t *H = qh + 32 * h;
        int lo, hb;
        switch (quarter) {
        case 0:  lo = L[l] & 15;       hb = (H[l] >> 0) & 3; break;
        case 1:  lo = L[l + 32] & 15;  hb = (H[l] >> 2) & 3; break;
        case 2:  lo = L[l] >> 4;       hb = (H[l] >> 4) & 3; break;
        default: lo = L[l + 32] >> 4;  hb = (H[l] >> 6) & 3; break;
        }
        int q6 = (lo | (hb << 4)) - 32;
        float s = (float)sc[e / 16];
        y[e] = oracle_f32_to_f16((d * s) * (float)q6);
    }
}

/* Q4_0, 18 bytes: d (f16) at 0, qs[16] at 2.  Element j (0..15) is the low
 * nibble of qs[j], element j+16 the high nibble; both offset by -8.
 *   y = RN16(d * (nibble - 8)) */
static void decode_q4_0_block(const uint8_t *b, uint16_t *y)
{
    float d = oracle_f16_to_f32(rd_u16le(b));
    const uint8_t *qs = b + 2;
    for (int e = 0; e < 32; e++) {
        int nib = e < 16 ? (qs[e] & 15) : (qs[e - 16] >> 4);
        y[e] = oracle_f32_to_f16(d * (float)(nib - 8));
    }
}

/* The 5-bit value of element e (0..31) of a Q5_0 / Q5_1 block: nibble as
 * in Q4_0 (qs[e] low, qs[e-16] high), fifth bit = bit e of the 32-bit
 * little-endian bit plane qh ("05 · 8p", section 2: a 4-byte qh bit plane
 * after the f16 d, then 16 nibble bytes). */
static int q5_value(const uint8_t *qh, const uint8_t *qs, int e)
{
    uint32_t h = (uint32_t)qh[0] | ((uint32_t)qh[1] << 8) | ((uint32_t)qh[2] << 16) | ((uint32_t)qh[3] << 24);
    int nib = e < 16 ? (qs[e] & 15) : (qs[e - 16] >> 4);
    return nib | (int)(((h >> e) & 1u) << 4);
}

/* Q5_0, 22 bytes: d (f16) at 0, qh[4] at 2, qs[16] at 6.
 *   y = RN16(d * (q5 - 16)) */
static void decode_q5_0_block(const uint8_t *b, uint16_t *y)
{
    float d = oracle_f16_to_f32(rd_u16le(b));
    for (int e = 0; e < 32; e++)
        y[e] = oracle_f32_to_f16(d * (float)(q5_value(b + 2, b + 6, e) - 16));
}

/* Q5_1, 24 bytes: d (f16) at 0, m (f16) at 2, qh[4] at 4, qs[16] at 8.
 *   y = RN16( RN32(RN32(d * q5) + m) ) */
static void decode_q5_1_block(const uint8_t *b, uint16_t *y)
{
    float d = oracle_f16_to_f32(rd_u16le(b));
    float m = oracle_f16_to_f32(rd_u16le(b + 2));
    for (int e = 0; e < 32; e++) {
        float dq = d * (float)q5_value(b + 4, b + 8, e);
        y[e] = oracle_f32_to_f16(dq + m);
    }
}

/* Q5_K, 176 bytes: d (f16) at 0, dmin (f16) at 2, S[12] at 4 (packed as in
 * Q4_K), qh[32] at 16, qs[128] at 48.  Group p = 0..3 covers elements
 * 64p .. 64p+63: element 64p+i (i < 32) is the low nibble of qs[32p+i]
 * with fifth bit = bit 2p of qh[i], sub-block 2p; element 64p+32+i is the
 * high nibble of the same byte with fifth bit = bit 2p+1 of qh[i], sub-block
 * 2p+1 (qh is bit-transposed: bit s of byte i belongs to sub-block s).
 *   y = RN16( RN32( RN32(RN32(d*sc)*q) - RN32(dmin*m) ) ) */
static void decode_q5_K_block(const uint8_t *b, uint16_t *y)
{
    float d = oracle_f16_to_f32(rd_u16le(b));
    float dmin = oracle_f16_to_f32(rd_u16le(b + 2));
    const uint8_t *S = b + 4;
    const uint8_t *qh = b + 16;
    const uint8_t *qs = b + 48;
    for (int e = 0; e < 256; e++) {
        int grp = e / 64;            /* group p */
        int upper = (e % 64) >= 32;  /* high nibbles */
        int pos = e % 32;
        int sub = 2 * grp + upper;
        int nib = upper ? (qs[32 * grp + pos] >> 4) : (qs[32 * grp + pos] & 15);
        int q5 = nib | (((qh[pos] >> sub) & 1) << 4);
        int scale, mn;
        q4k_scale_min(S, sub, &scale, &mn);
        float prod = (d * (float)scale) * (float)q5;
        float off = dmin * (float)mn;
        y[e] = oracle_f32_to_f16(prod - off);
    }
}

/* O2f: one float element -> binary16 bits. */
static uint16_t decode_f32_elem(const uint8_t *b)
{
    uint32_t x = (uint32_t)b[0] | ((uint32_t)b[1] << 8) | ((uint32_t)b[2] << 16) | ((uint32_t)b[3] << 24);
    float f;
    memcpy(&f, &x, 4);
    return oracle_f32_to_f16(f);
}

static uint16_t decode_bf16_elem(const uint8_t *b)
{
    uint32_t x = (uint32_t)rd_u16le(b) << 16;
    float f;
    memcpy(&f, &x, 4);
    return oracle_f32_to_f16(f);
}

/* Elements per block (QK) and bytes per block for a GGUF type id. */
int oracle_block_size(int type, int *qk, int *bytes)
{
    switch (type) {
    case T_F32:  *qk = 1;   *bytes = 4;   return 0;
    case T_F16:  *qk = 1;   *bytes = 2;   return 0;
    case T_BF16: *qk = 1;   *bytes = 2;   return 0;
    case T_Q4_0: *qk = 32;  *bytes = 18;  return 0;
    case T_Q5_0: *qk = 32;  *bytes = 22;  return 0;
    case T_Q5_1: *qk = 32;  *bytes = 24;  return 0;
    case T_Q8_0: *qk = 32;  *bytes = 34;  return 0;
    case T_Q4_K: *qk = 256; *bytes = 144; return 0;
    case T_Q5_K: *qk = 256; *bytes = 176; return 0;
    case T_Q6_K: *qk = 256; *bytes = 210; return 0;
    default: return -1;
    }
}

/* Decode nblocks consecutive blocks of one flat stream into nblocks*QK
 * binary16 values (raw bits) in stream order.  For a weight W[N,K] stored
 * as one stream, out is W row-major with row stride K. */
int oracle_decode(int type, const uint8_t *q, int64_t nblocks, uint16_t *out)
{
    int qk, bb;
    if (oracle_block_size(type, &qk, &bb))
        return -1;
    #pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < nblocks; i++) {
        const uint8_t *b = q + i * bb;
        uint16_t *y = out + i * qk;
        switch (type) {
        case T_F32:  y[0] = decode_f32_elem(b); break;
        case T_F16:  y[0] = rd_u16le(b); break;
        case T_BF16: y[0] = decode_bf16_elem(b); break;
        case T_Q4_0: decode_q4_0_block(b, y); break;
        case T_Q5_0: decode_q5_0_block(b, y); break;
        case T_Q5_1: decode_q5_1_block(b, y); break;
        case T_Q8_0: decode_q8_0_block(b, y); break;
        case T_Q4_K: decode_q4_K_block(b, y); break;
        case T_Q5_K: decode_q5_K_block(b, y); break;
        default:     decode_q6_K_block(b, y); break;
        }
    }
    return 0;
}

/* ------------------------------------------------------------------ */
/* O4: GEMM with f64 accumulation                                     */
/* ------------------------------------------------------------------ */

static void widen_row(const uint16_t *src, int64_t K, double *dst)
{
    for (int64_t k = 0; k < K; k++)
        dst[k] = (double)oracle_f16_to_f32(src[k]);
}

static double dot_f64(const double *x, const double *w, int64_t K)
{
    double acc = 0.0;
    for (int64_t k = 0; k < K; k++)
        acc += x[k] * w[k];
    return acc;
}

/* Y[m*N + n] = sum_{k=0}^{K-1} X[m*K + k] * W[n*K + k], X [M,K] and W [N,K]
 * as f16 bits, every product and partial sum in double, k increasing. */
int oracle_gemm_f64(const uint16_t *X, int64_t M, int64_t K,
                    const uint16_t *W, int64_t N, double *Y)
{
    double *xd = (double *)malloc((size_t)(M * K > 0 ? M * K : 1) * sizeof(double));
    if (!xd)
        return -2;
    #pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; m++)
        widen_row(X + m * K, K, xd + m * K);

    int err = 0;
    #pragma omp parallel
    {
        double *wd = (double *)malloc((size_t)(K > 0 ? K : 1) * sizeof(double));
        if (!wd) {
            #pragma omp atomic write
            err = 1;
        }
        #pragma omp for schedule(dynamic, 4)
        for (int64_t n = 0; n < N; n++) {
            if (!wd)
                continue;
            widen_row(W + n * K, K, wd);
            for (int64_t m = 0; m < M; m++)
                Y[m * N + n] = dot_f64(xd + m * K, wd, K);
        }
        free(wd);
    }
    free(xd);
    return err ? -2 : 0;
}

/* The same sum for `count` chosen (m, n) pairs only: out[i] is Y[mi[i], ni[i]].
 * Lets a test check a full-size GEMM at sampled outputs. */
int oracle_gemm_f64_sampled(const uint16_t *X, int64_t K, const uint16_t *W,
                            const int64_t *mi, const int64_t *ni, int64_t count,
                            double *out)
{
    int err = 0;
    #pragma omp parallel
    {
        double *xd = (double *)malloc((size_t)(K > 0 ? K : 1) * sizeof(double));
        double *wd = (double *)malloc((size_t)(K > 0 ? K : 1) * sizeof(double));
        if (!xd || !wd) {
            #pragma omp atomic write
            err = 1;
        }
        #pragma omp for schedule(dynamic, 16)
        for (int64_t i = 0; i < count; i++) {
            if (!xd || !wd)
                continue;
            widen_row(X + mi[i] * K, K, xd);
            widen_row(W + ni[i] * K, K, wd);
            out[i] = dot_f64(xd, wd, K);
        }
        free(xd);
        free(wd);
    }
    return err ? -2 : 0;
}

/* ------------------------------------------------------------------ */
/* O5: e4m3 codes, row quantization, the 8-bit GEMM                   */
/* ------------------------------------------------------------------ */

/* Nearest integer to u >= 0, ties to even (u is exact in double). */
static double round_half_even(double u)
{
    double r = floor(u);
    double frac = u - r;
    if (frac > 0.5 || (frac == 0.5 && fmod(r, 2.0) != 0.0))
        r += 1.0;
    return r;
}

uint8_t oracle_f32_to_e4m3(float f)
{
    if (isnan(f))
        return 0x7F;
    const uint8_t sign = signbit(f) ? 0x80 : 0x00;
    const double a = fabs((double)f);
    if (a == 0.0)
        return sign;
    if (a < ldexp(1.0, -6)) {
        /* subnormal range: units of 2^-9; a count of 8 is the smallest
         * normal 2^-6, whose code is 0x08 as well */
        return (uint8_t)(sign | (uint8_t)round_half_even(a * 512.0));
    }
    int e;
    double m = frexp(a, &e); /* a = m * 2^e, m in [0.5, 1) */
    m *= 2.0;
    e -= 1;                  /* a = m * 2^e, m in [1, 2) */
    double q = round_half_even(m * 8.0); /* significand in eighths: 8 .. 16 */
    if (q == 16.0) {
        q = 8.0;
        e += 1;
    }
    if (e > 8 || (e == 8 && q > 14.0))
        return (uint8_t)(sign | 0x7E); /* clamp to 448 */
    return (uint8_t)(sign | (uint8_t)(((e + 7) << 3) | ((int)q - 8)));
}

double oracle_e4m3_to_f64(uint8_t b)
{
    const int e = (b >> 3) & 15, m = b & 7;
    if (e == 15 && m == 7)
        return NAN;
    const double v = e ? ldexp((double)(8 + m), e - 10) : ldexp((double)m, -9);
    return (b & 0x80) ? -v : v;
}

int oracle_quantize_e4m3_rows(const uint16_t *src, int64_t rows, int64_t K, int64_t ld, uint8_t *dst,
                              float *scales)
{
    #pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; r++) {
        const uint16_t *row = src + r * ld;
        float amax = 0.0f;
        for (int64_t k = 0; k < K; k++) {
            float v = fabsf(oracle_f16_to_f32(row[k]));
            if (v > amax)
                amax = v;
        }
        float s = 1.0f, inv = 1.0f;
        if (amax > 0.0f) {
            s = amax / 448.0f;
            inv = 448.0f / amax;
        }
        for (int64_t k = 0; k < K; k++) {
            float t = oracle_f16_to_f32(row[k]) * inv;
            dst[r * K + k] = oracle_f32_to_e4m3(t);
        }
        scales[r] = s;
    }
    return 0;
}

/* Y[m,n] = (sum_k x8[m,k] * w8[n,k]) * sw[n] * sx[m]: each product of two
 * e4m3 values is exact in double, the sum is taken in k order. */
static double e4m3_dot_f64(const uint8_t *x, const uint8_t *w, int64_t K)
{
    double sum = 0.0;
    for (int64_t k = 0; k < K; k++)
        sum += oracle_e4m3_to_f64(x[k]) * oracle_e4m3_to_f64(w[k]);
    return sum;
}

int oracle_gemm_e4m3_f64(const uint8_t *X8, const float *sx, int64_t M, int64_t K, const uint8_t *W8,
                         const float *sw, int64_t N, double *Y)
{
    #pragma omp parallel for collapse(2) schedule(static)
    for (int64_t m = 0; m < M; m++)
        for (int64_t n = 0; n < N; n++)
            Y[m * N + n] = e4m3_dot_f64(X8 + m * K, W8 + n * K, K) * (double)sw[n] * (double)sx[m];
    return 0;
}

int oracle_gemm_e4m3_f64_sampled(const uint8_t *X8, const float *sx, int64_t K, const uint8_t *W8,
                                 const float *sw, const int64_t *mi, const int64_t *ni, int64_t count,
                                 double *out)
{
    #pragma omp parallel for schedule(dynamic, 16)
    for (int64_t i = 0; i < count; i++)
        out[i] = e4m3_dot_f64(X8 + mi[i] * K, W8 + ni[i] * K, K) * (double)sw[ni[i]] * (double)sx[mi[i]];
    return 0;
}

/* Number of OpenMP threads a parallel region of this library uses. */
int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Element-wise array forms of O1, for tests and input preparation. */
void oracle_f32_to_f16_n(const float *src, int64_t n, uint16_t *dst)
{
    #pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; i++)
        dst[i] = oracle_f32_to_f16(src[i]);
}

void oracle_f16_to_f32_n(const uint16_t *src, int64_t n, float *dst)
{
    #pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; i++)
        dst[i] = oracle_f16_to_f32(src[i]);
}
