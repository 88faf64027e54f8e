/* The affine encoder's division-free quotient, checked against IEEE division.
 *
 * For a bf16 scale s (8-bit significand) and a binary32 d, the encoder kernel forms
 *   y = RN(1/s), e0 = 1 - s y (exact by FMA), yek = RN(y e0) / K, yk = y / K,
 *   p = RN(d yek), u = RN(d yk + p)
 * and takes u K as RN(d / s).  This program checks that identity for every bf16 significand of s
 * in [1, 2) and every binary32 d in [2^-4, 2^7) (K = 16 and 4: 4- and 2-bit codes), and on every
 * STRIDE-th d for s at the ends of the exponent range the encoder uses without rescaling
 * ([2^-100, 2^100]).  Plain C, binary32 arithmetic with round to nearest (no contraction, fmaf for
 * the fused operations).  Prints the number of mismatches; exit status 0 when there are none.
 *
 *   usage: quotient_check [STRIDE]        (default 97) */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

static float from_bits(uint32_t u) { float x; memcpy(&x, &u, 4); return x; }
static uint32_t to_bits(float x) { uint32_t u; memcpy(&u, &x, 4); return u; }

typedef struct { int mant, expo; uint32_t stride; long long bad, n; } Job;

static void *run(void *arg) {
  Job *j = (Job *)arg;
  volatile float sv = ldexpf(1.0f + (float)j->mant / 128.0f, j->expo);
  const float s = sv;
  volatile float yv = 1.0f / s;
  const float y = yv;
  const float e0 = fmaf(-s, y, 1.0f);
  volatile float yev = y * e0;
  const float ye = yev;
  for (int kk = 0; kk < 2; ++kk) {
    const float K = kk ? 4.0f : 16.0f;
    volatile float ykv = y / K, yekv = ye / K;
    const float yk = ykv, yek = yekv;
    const uint32_t lo = to_bits(ldexpf(1.0f, j->expo - 4)), hi = to_bits(ldexpf(1.0f, j->expo + 7));
    for (uint32_t b = lo; b < hi; b += j->stride) {
      const float d = from_bits(b);
      volatile float p = d * yek;
      const float u = fmaf(d, yk, p);
      volatile float t = d / s;
      j->n++;
      if (u * K != t) {
        if (j->bad < 3) fprintf(stderr, "s=%a d=%a K=%g: %a, IEEE %a\n", s, d, K, u * K, t);
        j->bad++;
      }
    }
  }
  return NULL;
}

int main(int argc, char **argv) {
  const uint32_t stride = argc > 1 ? (uint32_t)strtoul(argv[1], NULL, 10) : 97u;
  enum { NJ = 128 * 3 };
  static Job jobs[NJ];
  static pthread_t th[NJ];
  for (int i = 0; i < NJ; ++i) {
    const int which = i / 128;  /* 0: s in [1, 2), every d; 1, 2: the range ends, every stride-th d */
    jobs[i].mant = i % 128;
    jobs[i].expo = which == 0 ? 0 : (which == 1 ? -100 : 99);
    jobs[i].stride = which == 0 ? 1u : stride;
  }
  for (int i = 0; i < NJ; ++i) pthread_create(&th[i], NULL, run, &jobs[i]);
  long long bad = 0, n = 0;
  for (int i = 0; i < NJ; ++i) {
    pthread_join(th[i], NULL);
    bad += jobs[i].bad;
    n += jobs[i].n;
  }
  printf("%lld mismatches in %lld quotients\n", bad, n);
  return bad != 0;
}
