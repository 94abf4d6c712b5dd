/*
 * log1p_series_check.c -- checks, on the CPU, the log1p(u) for u in [0, 1]
 * that the LSE merge kernel uses:
 *   t = RN(2 + u), s = u / t by a reciprocal approximation and one
 *       correction step, z = RN(s * s),
 *   p = Horner over z of RN(1/13), RN(1/11), ..., RN(1/3) with fused
 *       multiply-adds,
 *   log1p(u) ~ fma(RN(RN(2 s) * z), p, RN(2 s))
 * (2 atanh(s) by its series, truncated after s^12 / 13: below
 * (1/9)^7 / 15 < 2^-26 of the value for s <= 1/3).  The kernel's quotient is RN(u / t) except where
 * u / t lies within 1.5 x 2^-46 (relative) of a rounding midpoint, where it
 * may be the other neighbour (the correction step leaves the value before
 * its last rounding that close to u / t; the reciprocal instruction itself
 * cannot run here).  So s takes RN(u / t), and also the other neighbour
 * wherever u / t is within 2^-44 of a midpoint (and both neighbours for
 * subnormal quotients, where only an absolute bound holds); the rest are
 * the kernel's fp32 operations one for one.  Each result is compared with
 * log1p in double for every fp32 u in [first, last] (bit patterns,
 * arguments).  Prints "checked N worst W bad B alt A" (W: the largest
 * relative error, in units of 2^-24, over u >= 2^-125, where the quotient
 * is normal; A: arguments where a second quotient was tried) and exits 1 if
 * any result is off by more than 3 x 2^-24 relative plus 2^-146 absolute
 * (for u below 2^-125 the quotient is subnormal and only the absolute term
 * holds; u = 0 gives 0).  Over [0, 1]: worst 2.9476, 16,777,578 arguments
 * with a second quotient, none off.
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

static float series_from(float s)
{
    const float c[6] = {0x1.555556p-2f, 0x1.99999ap-3f, 0x1.24924ap-3f, 0x1.c71c72p-4f,
                        0x1.745d18p-4f, 0x1.3b13b2p-4f};
    const float z = s * s;
    float p = c[5];
    for (int k = 4; k >= 0; --k)
        p = fmaf(p, z, c[k]);
    const float two_s = 2.0f * s;
    return fmaf(two_s * z, p, two_s);
}

/* The quotients the kernel may produce for u / t: n of them in q[]. */
static int quotients(float u, float t, float q[3])
{
    const float s = u / t;
    const double x = (double)u / (double)t;
    int n = 0;
    q[n++] = s;
    if (u == 0.0f)
        return n; /* q0 = 0 and a zero remainder: exactly 0 */
    if (s < 0x1p-126f) {
        if (s > 0.0f)
            q[n++] = nextafterf(s, 0.0f);
        q[n++] = nextafterf(s, 1.0f);
        return n;
    }
    const float other = (double)s < x ? nextafterf(s, 1.0f) : nextafterf(s, 0.0f);
    const double mid = 0.5 * ((double)s + (double)other);
    if (fabs(x - mid) <= 0x1p-44 * x)
        q[n++] = other;
    return n;
}

int main(int argc, char** argv)
{
    if (argc != 3)
        return 2;
    const uint32_t first = (uint32_t)strtoul(argv[1], NULL, 0), last = (uint32_t)strtoul(argv[2], NULL, 0);
    long checked = 0, bad = 0, alt = 0;
    double worst = 0.0;
    for (uint64_t b = first; b <= last; ++b) {
        const float u = from_bits((uint32_t)b);
        const float t = 2.0f + u;
        float q[3];
        const int n = quotients(u, t, q);
        const double ref = log1p((double)u);
        ++checked;
        alt += n > 1;
        for (int i = 0; i < n; ++i) {
            const float got = series_from(q[i]);
            if (ref == 0.0) {
                if (got != 0.0f)
                    ++bad;
                continue;
            }
            const double err = fabs((double)got - ref);
            const double rel = err / ref / 0x1p-24;
            if (u >= 0x1p-125f && rel > worst)
                worst = rel;
            if (err > 3.0 * 0x1p-24 * ref + 0x1p-146) {
                if (bad < 5)
                    printf("u=%a s=%a got=%a ref=%a rel=%g\n", u, q[i], got, ref, rel);
                ++bad;
            }
        }
    }
    printf("checked %ld worst %.4f bad %ld alt %ld\n", checked, worst, bad, alt);
    return bad ? 1 : 0;
}
