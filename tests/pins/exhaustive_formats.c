/*
 * Exhaustive pins for the oracle's element encoders (test helper, CPU only).
 *
 * E2M1: every binary32 bit pattern (NaN excluded) is encoded by the oracle's
 * round-to-nearest-even encoder and by an independent brute-force argmin over
 * the eight magnitudes {0, .5, 1, 1.5, 2, 3, 4, 6} (ties to the even code,
 * i.e. mantissa bit 0; values at or beyond 6 saturate; the sign is kept).
 *
 * E4M3: every binary32 pattern in [0, 1024), the negatives of the smallest
 * patterns, and a sweep of larger values is encoded by the oracle and by a
 * nearest-neighbour search in the sorted table of the 127 finite
 * non-negative E4M3FN values, built from the format definition (bias 7,
 * subnormal step 2^-9, largest 448); ties go to the even code; values at or
 * above 448 saturate to 448.
 *
 * Usage: exhaustive_formats <threads>   -> prints "e2m1 <checked> <bad>" and
 *                                          "e4m3 <checked> <bad>"
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "../../oracle/nvfp4_oracle.h"

static const double GRID[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};
static double E4M3[127];

static uint8_t bf_e2m1(float y) {
  int neg = signbit(y) != 0;
  double a = fabs((double)y);
  int best = 7;
  if (a < 6.0) {
    double bestd = INFINITY;
    for (int i = 0; i < 8; ++i) {
      double d = fabs(a - GRID[i]);
      if (d < bestd || (d == bestd && (i & 1) == 0)) { bestd = d; best = i; }
    }
  }
  return (uint8_t)((neg ? 8 : 0) | best);
}

static uint8_t bf_e4m3(float t) {
  double a = fabs((double)t);
  int best = 126;
  if (a < 448.0) {
    int lo = 0, hi = 126;
    while (hi - lo > 1) {
      int mid = (lo + hi) / 2;
      if (E4M3[mid] <= a) lo = mid; else hi = mid;
    }
    double dl = a - E4M3[lo], dh = E4M3[hi] - a;
    if (E4M3[lo] == a) best = lo;
    else if (dl < dh) best = lo;
    else if (dh < dl) best = hi;
    else best = (lo & 1) == 0 ? lo : hi;
  }
  return (uint8_t)((signbit(t) ? 0x80 : 0) | best);
}

typedef struct { uint64_t lo, hi; uint64_t checked, bad; int which; } job_t;

static void* run(void* p) {
  job_t* j = (job_t*)p;
  for (uint64_t b = j->lo; b < j->hi; ++b) {
    uint32_t u = (uint32_t)b;
    float f;
    memcpy(&f, &u, 4);
    if (isnan(f)) continue;
    j->checked++;
    uint8_t got = j->which == 0 ? orc_e2m1_rne(f) : orc_e4m3_rne_sat(f);
    uint8_t exp = j->which == 0 ? bf_e2m1(f) : bf_e4m3(f);
    if (got != exp) {
      if (j->bad < 4) fprintf(stderr, "%s mismatch %08x\n", j->which ? "e4m3" : "e2m1", u);
      j->bad++;
    }
  }
  return NULL;
}

static void sweep(int which, uint64_t lo, uint64_t hi, int nt, uint64_t* checked, uint64_t* bad) {
  pthread_t th[64];
  job_t jobs[64];
  uint64_t span = (hi - lo + nt - 1) / nt;
  for (int t = 0; t < nt; ++t) {
    jobs[t].lo = lo + span * t < hi ? lo + span * t : hi;
    jobs[t].hi = jobs[t].lo + span < hi ? jobs[t].lo + span : hi;
    jobs[t].checked = jobs[t].bad = 0;
    jobs[t].which = which;
    pthread_create(&th[t], NULL, run, &jobs[t]);
  }
  for (int t = 0; t < nt; ++t) {
    pthread_join(th[t], NULL);
    *checked += jobs[t].checked;
    *bad += jobs[t].bad;
  }
}

int main(int argc, char** argv) {
  int nt = argc > 1 ? atoi(argv[1]) : 8;
  if (nt < 1) nt = 1;
  if (nt > 64) nt = 64;
  for (int c = 0; c < 127; ++c) {
    int e = c >> 3, m = c & 7;
    E4M3[c] = (e == 0) ? ldexp((double)m, -9) : ldexp((double)(8 + m), e - 10);
  }
  uint64_t checked = 0, bad = 0;
  sweep(0, 0, 1ull << 32, nt, &checked, &bad);
  printf("e2m1 %llu %llu\n", (unsigned long long)checked, (unsigned long long)bad);
  checked = bad = 0;
  sweep(1, 0, 0x44800000ull, nt, &checked, &bad);
  sweep(1, 0x80000000ull, 0x80000000ull + 0x00800000ull, nt, &checked, &bad);
  for (uint64_t b = 0x44800000ull; b <= 0x7F800000ull; b += 4096) {
    uint32_t u = (uint32_t)b;
    float f;
    memcpy(&f, &u, 4);
    checked++;
    if (orc_e4m3_rne_sat(f) != bf_e4m3(f)) bad++;
  }
  printf("e4m3 %llu %llu\n", (unsigned long long)checked, (unsigned long long)bad);
  return 0;
}
