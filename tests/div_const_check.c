/*
 * div_const_check.c -- checks, on the CPU, the division by a constant d
 * with one correction step that the kernels use for a row's or a group's
 * scale (d = 127 for int8, 448 for fp8 e4m3, 6 for fp4 e2m1):
 *   q0 = RN(m * c), r = fma(-q0, d, m), q = fma(r, c, q0), c = RN(1/d),
 * against the correctly rounded quotient RN(m / d), for every fp32 m in
 * the binades [2^e, 2^(e+1)) with first <= e <= last (arguments: d first
 * last; the test suite covers -100..127, i.e. every m in [2^-100, 2^128)).
 *
 * Reference: (float)((double)m / d).  It is RN(m / d): m / d = M * 2^k / D
 * for an integer significand M and the odd part D of d (7, 127 or 3).  If
 * D divides M the quotient is exact in both formats; otherwise its binary
 * expansion is periodic with period p = the order of 2 modulo D (3, 7 or
 * 2), each period being the p-bit pattern of r (2^p - 1) / D for a residue
 * 0 < r < D, neither all zeros nor all ones, so no run of equal bits is
 * 2p long.  The double result is a float rounding midpoint only if the 29
 * bits after the 24th are all equal; 2p <= 14 < 29, so the second rounding
 * cannot go wrong.
 *
 * The constants c are the literals the kernels use; each is checked to be
 * RN(1/d).  Prints "checked N bad B"; exits 1 on any mismatch.
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
    if (argc != 4)
        return 2;
    const int d_int = atoi(argv[1]), first = atoi(argv[2]), last = atoi(argv[3]);
    float c;
    switch (d_int) {
    case 448: c = 0x1.24924ap-9f; break;
    case 127: c = 0x1.020408p-7f; break;
    case 6: c = 0x1.555556p-3f; break;
    default: return 2;
    }
    const float d = (float)d_int;
    if (c != (float)(1.0 / (double)d_int)) {
        printf("constant is not RN(1/%d)\n", d_int);
        return 1;
    }
    long checked = 0, bad = 0;
    for (int k = first; k <= last; ++k) {
        const uint32_t e = (uint32_t)(k + 127);
        for (uint32_t frac = 0; frac < (1u << 23); ++frac) {
            const float m = from_bits((e << 23) | frac);
            const float q0 = m * c;
            const float r = fmaf(-q0, d, m);
            const float q = fmaf(r, c, q0);
            const float ref = (float)((double)m / (double)d_int);
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
