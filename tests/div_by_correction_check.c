/* Checks, on the host's IEEE binary32 arithmetic, the quotient that the
 * attention backward forms for a = p / l: y = RN(1 / l), q = RN(p y), then
 * twice r = p - l q and q = q + r y, each with one rounding (fmaf).  Claimed:
 * the result equals the correctly rounded p / l whenever l is in [2^-30, 2^30)
 * and p is +0 or in [2^-90, 2^90) (Markstein's theorem once the first
 * correction has made q faithful).  Compared bit for bit with IEEE division:
 *   - every significand of p in [1, 2) against a set of l significands
 *     (the sequence commutes with scaling p or l by a power of two inside
 *     the ranges, so one binade of each covers the rest);
 *   - p and l at the ends of their ranges, every exponent of p;
 *   - random pairs over the whole admitted ranges.
 * Prints the number of pairs checked and of mismatches; exit status 1 on any
 * mismatch.  Build with -ffp-contract=off so nothing else is fused. */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

static float f_of(uint32_t b)
{
    float f;
    memcpy(&f, &b, 4);
    return f;
}

static uint32_t b_of(float f)
{
    uint32_t b;
    memcpy(&b, &f, 4);
    return b;
}

static float by_correction(float p, float l)
{
    const float y = 1.0f / l;
    float q = p * y;
    q = fmaf(fmaf(-l, q, p), y, q);
    return fmaf(fmaf(-l, q, p), y, q);
}

static uint64_t checked, bad;

static void check(float p, float l)
{
    const float want = p / l, got = by_correction(p, l);
    ++checked;
    if (b_of(want) != b_of(got)) {
        if (bad < 10)
            printf("mismatch p=%a l=%a want=%a got=%a\n", p, l, want, got);
        ++bad;
    }
}

static uint64_t s = 0x9E3779B97F4A7C15ull;

static uint32_t rnd(void)   /* splitmix64 */
{
    uint64_t z = (s += 0x9E3779B97F4A7C15ull);
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return (uint32_t)((z ^ (z >> 31)) >> 32);
}

int main(void)
{
    /* l significands: the ends of the binade, halves, and random ones */
    uint32_t lm[24] = {0, 1, 2, 0x7fffff, 0x7ffffe, 0x400000, 0x3fffff, 0x400001, 0x555555, 0x2aaaab};
    for (int i = 10; i < 24; ++i)
        lm[i] = rnd() & 0x7fffff;
    for (int i = 0; i < 24; ++i) {
        const float l = f_of(0x3f800000u | lm[i]);   /* [1, 2) */
        for (uint32_t m = 0; m < (1u << 23); ++m)
            check(f_of(0x3f800000u | m), l);
    }
    /* ends of the ranges, every exponent of p */
    const uint32_t l_end[] = {0x30800000u, 0x30800001u, 0x30ffffffu, 0x4e7fffffu, 0x4e7ffffeu,
                              0x4e000000u, 0x3f800000u, 0x3f800001u, 0x3fffffffu};
    for (unsigned i = 0; i < sizeof l_end / sizeof l_end[0]; ++i) {
        const float l = f_of(l_end[i]);
        check(0.0f, l);
        for (uint32_t e = 0x25; e < 0xd9; ++e)
            for (int k = 0; k < 2048; ++k) {
                const uint32_t m = k < 4 ? (uint32_t[]){0, 1, 0x7fffff, 0x7ffffe}[k] : rnd() & 0x7fffff;
                check(f_of((e << 23) | m), l);
            }
    }
    /* random pairs over the admitted ranges */
    for (int k = 0; k < 20000000; ++k) {
        const uint32_t pb = 0x12800000u + rnd() % (0x6C800000u - 0x12800000u);
        const uint32_t lb = 0x30800000u + rnd() % 0x1E000000u;
        check(f_of(pb), f_of(lb));
    }
    printf("checked %llu mismatches %llu\n", (unsigned long long)checked, (unsigned long long)bad);
    return bad != 0;
}
