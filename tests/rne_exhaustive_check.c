/* Exhaustive check of the oracle's fp32 -> bf16 conversions over a range of
 * fp32 bit patterns, against a value-based computation in double precision:
 * take the two bf16 values that bracket |f| (the one nearer zero and the one
 * a bf16 ulp further out, with the ulp taken from the exponent), compare the
 * two distances exactly in double, and break ties by the even last bit (RNE)
 * or away from zero.  Truncation must give the nearer-to-zero neighbour.
 * Usage: rne_exhaustive_check FIRST COUNT; prints mismatch counts. */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

uint16_t oracle_bf16_rne(float f);
uint16_t oracle_bf16_trunc(float f);
uint16_t oracle_bf16_ties_away(float f);

static double bf16_magnitude(uint16_t b)
{
    uint32_t u = (uint32_t)(b & 0x7FFFu) << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

int main(int argc, char** argv)
{
    if (argc != 3)
        return 2;
    uint64_t first = strtoull(argv[1], NULL, 0);
    uint64_t count = strtoull(argv[2], NULL, 0);
    uint64_t bad_rne = 0, bad_trunc = 0, bad_away = 0, checked = 0;
    for (uint64_t i = 0; i < count; ++i) {
        uint32_t u = (uint32_t)(first + i);
        float f;
        memcpy(&f, &u, 4);
        uint16_t sign = (uint16_t)((u >> 16) & 0x8000u);
        uint16_t got_rne = oracle_bf16_rne(f);
        uint16_t got_trunc = oracle_bf16_trunc(f);
        uint16_t got_away = oracle_bf16_ties_away(f);
        if (isnan(f)) {
            /* NaN in, quiet NaN of the same sign out */
            if ((got_rne & 0x7F80u) != 0x7F80u || !(got_rne & 0x7Fu) || (got_rne & 0x8000u) != sign)
                ++bad_rne;
            continue;
        }
        ++checked;
        double a = fabs((double)f);
        uint16_t below = (uint16_t)((u >> 16) & 0x7FFFu);       /* bf16 with |.| <= a */
        unsigned expo = (below >> 7) & 0xFFu;
        double ulp = ldexp(1.0, (expo == 0 ? 1 : (int)expo) - 127 - 7);
        double v_lo = bf16_magnitude(below);
        uint16_t exp_rne, exp_away, exp_trunc = (uint16_t)(below | sign);
        if (isinf(f)) {
            exp_rne = exp_away = (uint16_t)(0x7F80u | sign);
        } else {
            double v_hi = v_lo + ulp;           /* next bf16 outward (2^128 past the top) */
            double d_lo = a - v_lo, d_hi = v_hi - a;
            uint16_t up = (uint16_t)((below + 1u) | sign), dn = (uint16_t)(below | sign);
            if (d_lo < d_hi) exp_rne = exp_away = dn;
            else if (d_lo > d_hi) exp_rne = exp_away = up;
            else { exp_rne = (below & 1u) ? up : dn; exp_away = up; }
        }
        bad_rne += got_rne != exp_rne;
        bad_trunc += got_trunc != exp_trunc;
        bad_away += got_away != exp_away;
    }
    printf("checked %llu rne_bad %llu trunc_bad %llu away_bad %llu\n",
           (unsigned long long)checked, (unsigned long long)bad_rne,
           (unsigned long long)bad_trunc, (unsigned long long)bad_away);
    return (bad_rne || bad_trunc || bad_away) ? 1 : 0;
}
