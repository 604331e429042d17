/* Exhaustive pin of the oracle's binary16 conversion: every one of the 2^32
 * binary32 inputs is narrowed by the oracle and by the C compiler's own
 * _Float16 conversion (libgcc's soft-float routine on x86-64, the FCVT
 * instruction on aarch64), and every one of the 2^16 binary16 inputs is
 * widened by both.  NaN inputs must give a NaN of the same sign. */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

uint16_t oracle_f32_to_f16(float f);
float oracle_f16_to_f32(uint16_t h);

int main(void)
{
    long long bad = 0;
    #pragma omp parallel for reduction(+:bad) schedule(static, 1 << 20)
    for (long long i = 0; i < (1LL << 32); i++) {
        uint32_t u = (uint32_t)i;
        float f;
        memcpy(&f, &u, 4);
        uint16_t o = oracle_f32_to_f16(f);
        if (f != f) {
            int ok = ((o >> 10) & 0x1f) == 0x1f && (o & 0x3ff) != 0 && (o >> 15) == (u >> 31);
            bad += !ok;
        } else {
            _Float16 h = (_Float16)f;
            uint16_t r;
            memcpy(&r, &h, 2);
            bad += (o != r);
        }
    }
    long long bad16 = 0;
    for (int i = 0; i < 65536; i++) {
        uint16_t b = (uint16_t)i;
        _Float16 h;
        memcpy(&h, &b, 2);
        float r = (float)h, o = oracle_f16_to_f32(b);
        if (r != r) {
            bad16 += !(o != o);
        } else {
            uint32_t rb, ob;
            memcpy(&rb, &r, 4);
            memcpy(&ob, &o, 4);
            bad16 += (rb != ob);
        }
    }
    printf("narrow_mismatches=%lld widen_mismatches=%lld\n", bad, bad16);
    return (bad || bad16) ? 1 : 0;
}
