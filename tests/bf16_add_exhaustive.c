/* Exhaustive check, over every pair of bf16 bit patterns, that rounding the
 * binary32 sum of the two widened operands to bf16 (round to nearest, ties to
 * even) gives the correctly rounded bf16 sum.  The per-hop bf16 summation of
 * the ring reduce-scatter relies on this: each hop adds in fp32 and rounds to
 * bf16 once ("bf16 communication", DeepSpeed issue 8364; IEEE 754-2008
 * section 4.3.1, roundTiesToEven).
 *
 * Route 1 is that two-step rule, with the binary32 add done by the host FPU
 * (no fast-math, no contraction, no flush of subnormals).
 * Route 2 is independent: it decodes both operands into integer significands
 * and exponents, forms the exact sum as a 64-bit integer times a power of two,
 * and rounds that once to 8 significant bits.
 *
 * Usage: bf16_add_exhaustive [a_lo a_hi]   (a in [a_lo, a_hi), every b)
 * Prints "pairs=<n> mismatches=<m> first=<a>,<b>".
 *        bf16_add_exhaustive --dump a ...     route 2 for each listed a and
 * every b, as raw little-endian uint16 on stdout (65536 per a, b ascending).
 * Built with -DROUTE1_TRUNCATES, route 1 drops the 16 low bits instead of
 * rounding, a planted mistake the check must catch.
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

static uint16_t route1(uint16_t a, uint16_t b) {
    uint32_t ua = (uint32_t)a << 16, ub = (uint32_t)b << 16, us;
    float fa, fb, fs;
    memcpy(&fa, &ua, 4);
    memcpy(&fb, &ub, 4);
    fs = fa + fb;
    memcpy(&us, &fs, 4);
    if ((us & 0x7FFFFFFFu) > 0x7F800000u) return 0x7FC0;
#ifdef ROUTE1_TRUNCATES
    return (uint16_t)(us >> 16);
#else
    uint32_t half_up = 0x7FFFu + ((us >> 16) & 1u);
    return (uint16_t)((us + half_up) >> 16);
#endif
}

/* value = sign * M * 2^E, M < 256 */
typedef struct { int neg; int64_t M; int E; } dec;

static dec decode(uint16_t h) {
    dec d;
    int e = (h >> 7) & 0xFF, f = h & 0x7F;
    d.neg = h >> 15;
    if (e == 0) { d.M = f; d.E = -133; }
    else { d.M = f | 0x80; d.E = e - 134; }
    return d;
}

static int bitlen(uint64_t x) {
    int n = 0;
    while (x) { ++n; x >>= 1; }
    return n;
}

static uint16_t route2(uint16_t a, uint16_t b) {
    int ea = (a >> 7) & 0xFF, eb = (b >> 7) & 0xFF;
    int nan_a = ea == 255 && (a & 0x7F), nan_b = eb == 255 && (b & 0x7F);
    int inf_a = ea == 255 && !(a & 0x7F), inf_b = eb == 255 && !(b & 0x7F);
    if (nan_a || nan_b) return 0x7FC0;
    if (inf_a && inf_b) return ((a ^ b) & 0x8000) ? 0x7FC0 : a;
    if (inf_a) return a;
    if (inf_b) return b;
    dec x = decode(a), y = decode(b);
    uint16_t x_bits = a;
    if (x.E < y.E) { dec t = x; x = y; y = t; x_bits = b; }
    int gap = x.E - y.E;
    /* y is then below 2^-32 of x's unit in the last place: the sum rounds to x */
    if (gap > 40) return x_bits;
    int64_t S = (x.neg ? -x.M : x.M) * ((int64_t)1 << gap) + (y.neg ? -y.M : y.M);
    int E = y.E;
    if (S == 0) return (x.neg && y.neg) ? 0x8000 : 0x0000;
    int neg = S < 0;
    uint64_t A = (uint64_t)(neg ? -S : S);
    int k = bitlen(A) - 8;
    if (E + k < -133) k = -133 - E;
    uint64_t q;
    if (k <= 0) {
        q = A << (-k);
    } else {
        q = A >> k;
        uint64_t rem = A & ((1ull << k) - 1), half = 1ull << (k - 1);
        if (rem > half || (rem == half && (q & 1))) ++q;
        if (q == 256) { q = 128; ++k; }
    }
    int U = E + k;
    uint16_t sign = (uint16_t)(neg << 15);
    if (q >= 128) {
        int e = U + 134;
        if (e >= 255) return sign | 0x7F80;
        return sign | (uint16_t)(e << 7) | (uint16_t)(q - 128);
    }
    return sign | (uint16_t)q;   /* subnormal: U == -133 */
}

int main(int argc, char** argv) {
    if (argc >= 2 && strcmp(argv[1], "--dump") == 0) {
        static uint16_t row[65536];
        for (int i = 2; i < argc; ++i) {
            long a = atol(argv[i]);
            if (a < 0 || a > 65535) return 2;
            for (long b = 0; b < 65536; ++b) {
                uint16_t r = route2((uint16_t)a, (uint16_t)b);
                unsigned char* p = (unsigned char*)&row[b];
                p[0] = (unsigned char)(r & 0xFF);
                p[1] = (unsigned char)(r >> 8);
            }
            if (fwrite(row, 2, 65536, stdout) != 65536) return 3;
        }
        return 0;
    }
    long lo = 0, hi = 65536;
    if (argc == 3) { lo = atol(argv[1]); hi = atol(argv[2]); }
    if (lo < 0 || hi > 65536 || lo > hi) return 2;
    unsigned long long pairs = 0, bad = 0;
    long first = -1;
#pragma omp parallel for schedule(dynamic, 64) reduction(+ : pairs, bad)
    for (long a = lo; a < hi; ++a) {
        for (long b = 0; b < 65536; ++b) {
            ++pairs;
            if (route1((uint16_t)a, (uint16_t)b) != route2((uint16_t)a, (uint16_t)b)) {
                ++bad;
#pragma omp critical
                if (first < 0) first = a * 65536 + b;
            }
        }
    }
    printf("pairs=%llu mismatches=%llu first=%ld,%ld\n", pairs, bad,
           first < 0 ? -1 : first / 65536, first < 0 ? -1 : first % 65536);
    return 0;
}
