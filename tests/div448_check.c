/*
 * div448_check.c -- checks, on the CPU, the division by 448 with one
 * correction step that the fp8 kernels use for a group's scale:
 *   q0 = RN(m * c), r = fma(-q0, 448, m), q = fma(r, c, q0), c = RN(1/448),
 * against the correctly rounded quotient RN(m / 448), for every fp32 m in
 * the binades [2^e, 2^(e+1)) with first <= e <= last (arguments; the test
 * suite covers -100..127, i.e. every m in [2^-100, 2^128)).
 *
 * Reference: (float)((double)m / 448).  It is RN(m / 448): m / 448 =
 * M * 2^k / 7 for an integer significand M; if 7 divides M the quotient is
 * exact in both formats, otherwise its binary expansion repeats with
 * period 3 and never holds the 29 equal bits after the 24th that would
 * make the double result a float rounding midpoint, so the second rounding
 * cannot go wrong.
 *
 * Prints "checked N bad B"; exits 1 on any mismatch.
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#if !defined(FLT_EVAL_METHOD) && defined(__FLT_EVAL_METHOD__)
#define FLT_EVAL_METHOD __FLT_EVAL_METHOD__
#endif
#if FLT_EVAL_METHOD != 0
#error "float arithmetic must be evaluated in float"
#endif

static float from_bits(uint32_t u)
{
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

int main(int argc, char** argv)
{
    if (argc != 3)
        return 2;
    const int first = atoi(argv[1]), last = atoi(argv[2]);
    const float c = 0x1.24924ap-9f;
    if (c != (float)(1.0 / 448.0)) {
        printf("constant is not RN(1/448)\n");
        return 1;
    }
    long checked = 0, bad = 0;
    for (int k = first; k <= last; ++k) {
        const uint32_t e = (uint32_t)(k + 127);
        for (uint32_t frac = 0; frac < (1u << 23); ++frac) {
            const float m = from_bits((e << 23) | frac);
            const float q0 = m * c;
            const float r = fmaf(-q0, 448.0f, m);
            const float q = fmaf(r, c, q0);
            const float ref = (float)((double)m / 448.0);
            ++checked;
            if (q != ref) {
                if (bad < 5)
                    printf("m=%a q=%a ref=%a\n", m, q, ref);
                ++bad;
            }
        }
    }
    printf("checked %ld bad %ld\n", checked, bad);
    return bad ? 1 : 0;
}
