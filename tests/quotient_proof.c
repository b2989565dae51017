/*
 * Exhaustive check, over every input the quantisers can see, that the
 * division the CUDA quantisers use equals IEEE binary32 division.
 *
 * The quantisers need fp32(x / s) for BF16 x with |x| <= amax, where amax is
 * the group's BF16 amax and s = fp32(amax / 448).  For a normal s they form
 * it with Markstein's correction step (P. Markstein, "Computation of
 * elementary functions on the IBM RISC System/6000 processor", IBM J. Res.
 * Dev. 34(1), 1990): with r = RN(1/s),
 *     q0 = RN(x * r);  rem = fma(-q0, s, x);  q1 = copysign(RN(rem * r + q0), x)
 * (one fma; the copysign gives the quotient x's sign, as IEEE division by a
 * positive s does, which matters for x = -0 where +0 + -0 rounds to +0).
 * The kernels take this path only for groups with amax >= 2^-90 (BF16 bit
 * pattern >= 0x1280); smaller groups use IEEE division.  This program runs the
 * sequence for every BF16 amax in [2^-90, max finite] and every BF16 x with
 * |x| <= amax, both signs and both zeros, and compares q1 with x / s bit for
 * bit.  Quotients below 2^-11 in magnitude encode to a
 * signed zero in E4M3, so where both sides are that small only the sign bits
 * must agree; such pairs are counted separately.
 *
 * The kernels apply the copysign to the E4M3 code instead (x's sign bit is
 * OR-ed into the byte converted from the unsigned result RN(rem * r + q0)).
 * That gives the same byte iff the unsigned result already carries x's sign
 * or is +0; every pair where it is neither is counted as a sign violation.
 *
 * Output: one line "pairs=<n> mismatches=<m> tiny_differences=<t>
 * sign_violations=<v> ...".  Exit status 0 iff m == 0 and v == 0.
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

static float bf(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

static uint32_t bits(float f)
{
    uint32_t u;
    memcpy(&u, &f, 4);
    return u;
}

int main(int argc, char **argv)
{
    /* optional stride over amax patterns, for a quicker partial run */
    unsigned stride = (argc > 1) ? (unsigned)atoi(argv[1]) : 1u;
    if (stride == 0)
        stride = 1;
    unsigned long long pairs = 0, mism = 0, tiny = 0, sign_viol = 0;
    for (uint32_t ha = 0x1280; ha <= 0x7F7F; ha += stride) {   /* amax >= 2^-90 */
        const float amax = bf((uint16_t)ha);
        const float s = amax / 448.0f;
        /* RN(1/s): binary64 quotient rounded once to binary32 is the correctly
         * rounded binary32 quotient (53 >= 2*24 + 2). */
        const float r = (float)(1.0 / (double)s);
        for (uint32_t i = 0; i <= 2 * ha + 1; ++i) {
            const uint32_t hx = (i >> 1) | ((i & 1u) << 15);     /* +x, then -x */
            const float x = bf((uint16_t)hx);
            const float ref = x / s;
            const float q0 = x * r;
            const float rem = fmaf(-q0, s, x);
            const float qr = fmaf(rem, r, q0);
            const float q1 = copysignf(qr, x);
            pairs++;
            if ((bits(qr) >> 31) != (bits(x) >> 31) && bits(qr) != 0u) {
                if (sign_viol < 10)
                    fprintf(stderr, "sign violation amax=%a x=%a unsigned=%a\n", amax, x, qr);
                sign_viol++;
            }
            if (bits(q1) != bits(ref)) {
                if (fabsf(ref) < 0x1p-11f && fabsf(q1) < 0x1p-11f &&
                    (bits(ref) >> 31) == (bits(q1) >> 31))
                    tiny++;
                else {
                    if (mism < 10)
                        fprintf(stderr, "mismatch amax=%a x=%a ref=%a got=%a\n", amax, x, ref, q1);
                    mism++;
                }
            }
        }
    }
    printf("pairs=%llu mismatches=%llu tiny_differences=%llu sign_violations=%llu stride=%u\n", pairs, mism,
           tiny, sign_viol, stride);
    return (mism == 0 && sign_viol == 0) ? 0 : 1;
}
