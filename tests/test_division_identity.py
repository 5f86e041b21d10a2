"""The quantise kernels divide by a block scale s with one IEEE reciprocal r = RN(1/s) per
scale and, per element, y = RN(x r), e = fma(-y, s, x), q = fma(e, r, y) (Markstein, IBM J.
Res. Dev. 34(1), 1990).  The INT8 and E4M3 codes are bit-exact only if q equals the IEEE
quotient RN(x / s).  This checks that on the CPU (C, hardware FMA, no contraction): every
code boundary (x / s within 4 ulp of k + 1/2, |k| <= 128) and random x, for sampled scale
significands; the result does not depend on the binade of s or x."""
import os
import subprocess
import tempfile

C_SRC = r"""
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>
static float f_of(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }
static uint32_t u_of(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }
static int check(float x, float s, float r) {
  float y = x * r, e = fmaf(-y, s, x), q = fmaf(e, r, y);
  volatile float ref = x / s;
  return u_of(q) != u_of(ref);
}
int main(void) {
  unsigned long long bad = 0, total = 0;
  uint32_t seed = 2024;
  for (int t = 0; t < 40000; ++t) {
    seed = seed * 1664525u + 1013904223u;
    uint32_t m = t < 2048 ? (uint32_t)(0x7FFFFF - t) : (t < 4096 ? (uint32_t)(t - 2048) : (seed >> 9));
    float s = f_of(0x3F800000u | m);
    volatile float one = 1.0f;
    float r = one / s;
    for (int k = -128; k <= 128; ++k) {
      uint32_t u0 = u_of((float)(((double)k + 0.5) * (double)s));
      for (int d = -4; d <= 4; ++d) { bad += check(f_of(u0 + d), s, r); total++; }
    }
    for (int i = 0; i < 64; ++i) {
      seed = seed * 1664525u + 1013904223u;
      float x = ((float)(seed >> 8) / 16777216.0f * 2.0f - 1.0f) * 448.0f * s;
      bad += check(x, s, r); total++;
    }
  }
  printf("%llu %llu\n", total, bad);
  return 0;
}
"""


def test_markstein_division_matches_ieee():
    with tempfile.TemporaryDirectory() as tmp:
        src, exe = os.path.join(tmp, "div.c"), os.path.join(tmp, "div")
        open(src, "w").write(C_SRC)
        subprocess.run(["gcc", "-O2", "-ffp-contract=off", "-o", exe, src, "-lm"], check=True)
        total, bad = map(int, subprocess.run([exe], capture_output=True, text=True, check=True).stdout.split())
    assert total > 90_000_000 and bad == 0
