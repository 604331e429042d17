/*
 * encode.c -- block ENCODERS (fields -> bytes) for Q8_0 / Q4_K / Q6_K.
 *
 * TEST INFRASTRUCTURE ONLY, like the rest of this directory.  Tests build
 * blocks with chosen field values (a scale, a min, one nibble) through these
 * functions and check what the decoders in oracle.c return.  The encoders
 * are written as the inverse of the GGUF field layout (the pages name the
 * types only: "05 · 8p — Persistent f16 weight cache + fused
 * dequant-in-GEMM", section 1), independently of the decoders: no code is
 * shared between the two directions.
 */
#include <stdint.h>
#include <string.h>

static void wr_u16le(uint8_t *p, uint16_t v) { p[0] = (uint8_t)(v & 0xff); p[1] = (uint8_t)(v >> 8); }

/* Q8_0: d at byte 0, q[e] at byte 2+e. */
void oracle_pack_q8_0(uint16_t d, const int8_t *q, uint8_t *out)
{
    wr_u16le(out, d);
    for (int e = 0; e < 32; e++)
        out[2 + e] = (uint8_t)q[e];
}

/* Q4_K: d at 0, dmin at 2, 12 scale bytes at 4, 128 nibble bytes at 16.
 * Scale bytes, for j = 0..3:
 *   byte j     : sc[j] (6 bits)  | top 2 bits of sc[j+4] in bits 6..7
 *   byte j + 4 : m[j]  (6 bits)  | top 2 bits of m[j+4]  in bits 6..7
 *   byte j + 8 : low 4 bits of sc[j+4] | low 4 bits of m[j+4] << 4
 * Nibbles: value of element 64p+i (i<32) goes in the low half of byte
 * 32p+i, element 64p+32+i in its high half. */
void oracle_pack_q4_K(uint16_t d, uint16_t dmin, const uint8_t *sc, const uint8_t *m,
                      const uint8_t *q, uint8_t *out)
{
    memset(out, 0, 144);
    wr_u16le(out, d);
    wr_u16le(out + 2, dmin);
    uint8_t *S = out + 4;
    for (int j = 0; j < 4; j++) {
        S[j] = (uint8_t)((sc[j] & 63) | ((sc[j + 4] >> 4) << 6));
        S[j + 4] = (uint8_t)((m[j] & 63) | ((m[j + 4] >> 4) << 6));
        S[j + 8] = (uint8_t)((sc[j + 4] & 15) | ((m[j + 4] & 15) << 4));
    }
    uint8_t *qs = out + 16;
    for (int p = 0; p < 4; p++)
        for (int i = 0; i < 32; i++)
            qs[32 * p + i] = (uint8_t)((q[64 * p + i] & 15) | ((q[64 * p + 32 + i] & 15) << 4));
}

/* Q6_K: 128 low-nibble bytes at 0, 64 high-bit bytes at 128, 16 int8 scales
 * at 192, d at 208.  Element e holds v = q6[e] + 32 (0..63): its low 4 bits
 * go into a nibble of ql and its top 2 bits into a 2-bit field of qh.  For
 * half h, quarter t (0..3) and l (0..31), e = 128h + 32t + l:
 *   t = 0: low nibble of ql[64h+l],     qh[32h+l] bits 0..1
 *   t = 1: low nibble of ql[64h+l+32],  qh[32h+l] bits 2..3
 *   t = 2: high nibble of ql[64h+l],    qh[32h+l] bits 4..5
 *   t = 3: high nibble of ql[64h+l+32], qh[32h+l] bits 6..7 */
void oracle_pack_q6_K(uint16_t d, const int8_t *sc, const int8_t *q6, uint8_t *out)
{
    memset(out, 0, 210);
    uint8_t *ql = out;
    uint8_t *qh = out + 128;
    for (int h = 0; h < 2; h++)
        for (int t = 0; t < 4; t++)
            for (int l = 0; l < 32; l++) {
                int v = q6[128 * h + 32 * t + l] + 32;
                int lo = v & 15, hi = (v >> 4) & 3;
                int qli = 64 * h + l + ((t & 1) ? 32 : 0);
                ql[qli] |= (uint8_t)((t & 2) ? lo << 4 : lo);
                qh[32 * h + l] |= (uint8_t)(hi << (2 * t));
            }
    for (int j = 0; j < 16; j++)
        out[192 + j] = (uint8_t)sc[j];
    wr_u16le(out + 208, d);
}
