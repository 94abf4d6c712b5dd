/*
 * log1p_series_check.c -- checks, on the CPU, the log1p(u) for u in [0, 1]
 * that the LSE merge kernel uses:
 *   s = RN(u / RN(2 + u)), z = RN(s * s),
 *   p = Horner over z of RN(1/17), RN(1/15), ..., RN(1/3) with fused
 *       multiply-adds,
 *   log1p(u) ~ fma(RN(RN(2 s) * z), p, RN(2 s))
 * (2 atanh(s) by its series, truncated after s^16 / 17: below 2^-28 of the
 * value for s <= 1/3).  These are the kernel's fp32 operations one for one,
 * so the bits are the kernel's; each result is compared with log1p in
 * double for every fp32 u in [first, last] (bit patterns, arguments).
 * Prints "checked N worst W bad B" (W: the largest relative error, in units
 * of 2^-24, over normal u) and exits 1 if any result is off by more than
 * 3 x 2^-24 relative plus 2^-148 absolute (subnormal u, where s = u / 2 is
 * subnormal too, lose relative precision; u = 0 gives 0).
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

static float log1p_unit(float u)
{
    const float c[8] = {0x1.555556p-2f, 0x1.99999ap-3f, 0x1.24924ap-3f, 0x1.c71c72p-4f,
                        0x1.745d18p-4f, 0x1.3b13b2p-4f, 0x1.111112p-4f, 0x1.e1e1e2p-5f};
    const float t = 2.0f + u;
    const float s = u / t;
    const float z = s * s;
    float p = c[7];
    for (int k = 6; k >= 0; --k)
        p = fmaf(p, z, c[k]);
    const float two_s = 2.0f * s;
    return fmaf(two_s * z, p, two_s);
}

int main(int argc, char** argv)
{
    if (argc != 3)
        return 2;
    const uint32_t first = (uint32_t)strtoul(argv[1], NULL, 0), last = (uint32_t)strtoul(argv[2], NULL, 0);
    long checked = 0, bad = 0;
    double worst = 0.0;
    for (uint64_t b = first; b <= last; ++b) {
        const float u = from_bits((uint32_t)b);
        const float got = log1p_unit(u);
        const double ref = log1p((double)u);
        ++checked;
        if (ref == 0.0) {
            if (got != 0.0f)
                ++bad;
            continue;
        }
        const double err = fabs((double)got - ref);
        const double rel = err / ref / 0x1p-24;
        if (u >= 0x1p-126f && rel > worst)
            worst = rel;
        if (err > 3.0 * 0x1p-24 * ref + 0x1p-148) {
            if (bad < 5)
                printf("u=%a got=%a ref=%a rel=%g\n", u, got, ref, rel);
            ++bad;
        }
    }
    printf("checked %ld worst %.4f bad %ld\n", checked, worst, bad);
    return bad ? 1 : 0;
}
