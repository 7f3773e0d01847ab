/* Division by L = 3 and 15 as the flush kernel computes the scale:
 *   q = RN(x * c) with c = RN(1 / L), r = fma(-q, L, x), s = fma(r, c, q),
 * checked against the IEEE quotient RN(x / L) for every non-negative finite
 * fp32 x (subnormals included). Built with -ffp-contract=off so that every
 * multiply, fma and division rounds on its own. Prints "ok" and exits 0 when
 * every x agrees; otherwise prints the first mismatches and exits 1.
 * Test infrastructure for tests/test_guard_band.py. */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#define END 0x7f800000u /* +inf: every finite x >= 0 lies below */

typedef struct {
    uint32_t lo, hi;
    float L;
    unsigned long long bad;
    uint32_t first_bad;
} Range;

static float as_float(uint32_t u) {
    float x;
    memcpy(&x, &u, sizeof x);
    return x;
}

static void* run(void* arg) {
    Range* r = (Range*)arg;
    const float L = r->L, c = 1.0f / L;
    for (uint32_t u = r->lo; u < r->hi; ++u) {
        const float x = as_float(u);
        const float ref = x / L;
        const float q = x * c;
        const float rem = fmaf(-q, L, x);
        const float s = fmaf(rem, c, q);
        if (memcmp(&s, &ref, sizeof s) != 0) {
            if (r->bad == 0) r->first_bad = u;
            r->bad++;
        }
    }
    return NULL;
}

int main(int argc, char** argv) {
    int nt = argc > 1 ? atoi(argv[1]) : 1;
    if (nt < 1) nt = 1;
    if (nt > 256) nt = 256;
    const float Ls[2] = {3.0f, 15.0f};
    int fail = 0;
    for (int li = 0; li < 2; ++li) {
        pthread_t th[256];
        Range rg[256];
        for (int t = 0; t < nt; ++t) {
            rg[t].lo = (uint32_t)((unsigned long long)END * t / nt);
            rg[t].hi = (uint32_t)((unsigned long long)END * (t + 1) / nt);
            rg[t].L = Ls[li];
            rg[t].bad = 0;
            rg[t].first_bad = 0;
            pthread_create(&th[t], NULL, run, &rg[t]);
        }
        unsigned long long bad = 0;
        for (int t = 0; t < nt; ++t) {
            pthread_join(th[t], NULL);
            if (rg[t].bad) {
                printf("L=%g first mismatch at x=%a\n", Ls[li], as_float(rg[t].first_bad));
                bad += rg[t].bad;
            }
        }
        printf("L=%g: %u values, %llu mismatches\n", Ls[li], END, bad);
        if (bad) fail = 1;
    }
    if (!fail) printf("ok\n");
    return fail;
}
