"""Host brute-force check of the append kernel's division-free code rule (no GPU).

The append kernel computes codes q = clamp(rint(fl32(fl32(x - z) / s)), 0, L)
(Quanto steps 1-2 on the page "KV Cache量化技术介绍": scale, zero point,
rounding to the integer grid) without dividing: y = fl32(fl32(x - z) * r) with
r the hardware reciprocal of s (within one ulp of 1/s), rounded to an integer
by adding 1.5 * 2^23; an element whose y lies within the tie guard of a
half-integer is recomputed by the exact rule (the residual of the tie from
one fma, compared with half an ulp of the tie times s). This test restates
those steps in C, for each of the three reciprocals a one-ulp approximation
can return, and compares the codes with the binary32 division on every fp16
element of many groups (every value between the group's minimum and maximum
where there are few enough) plus planted exact ties (x - z = (k + 1/2) s with
s a power of two). The GPU parity tests check the kernel itself; this check
shows that its arithmetic rule has no counterexample.
"""
import os
import shutil
import subprocess
import tempfile

import pytest

PROGRAM = r"""
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

static float h2f(uint16_t h) {                 /* exact binary16 -> binary32 */
  const int sgn = h >> 15, e = (h >> 10) & 31, m = h & 1023;
  float v;
  if (e == 0) v = ldexpf((float)m, -24);
  else v = ldexpf((float)(1024 + m), e - 25);
  return sgn ? -v : v;
}
static float tab[0x7C00];                      /* every finite binary16 >= 0, ascending */
static uint16_t half_up(float x) {             /* smallest binary16 >= x (x >= 0) */
  int lo = 0, hi = 0x7C00;
  while (lo < hi) { int mid = (lo + hi) / 2; if (tab[mid] >= x) hi = mid; else lo = mid + 1; }
  return (uint16_t)lo;
}
static int is_half(double v, uint16_t* out) {  /* v an exact binary16 value? */
  const uint16_t sgn = v < 0 ? 0x8000 : 0;
  const double a = fabs(v);
  int lo = 0, hi = 0x7C00;
  while (lo < hi) { int mid = (lo + hi) / 2; if ((double)tab[mid] >= a) hi = mid; else lo = mid + 1; }
  if (lo < 0x7C00 && (double)tab[lo] == a) { *out = (uint16_t)(lo | sgn); return 1; }
  return 0;
}

static uint64_t st = 0x9E3779B97F4A7C15ull;   /* splitmix64 */
static uint64_t rnd(void) {
  uint64_t z = (st += 0x9E3779B97F4A7C15ull);
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

/* the division the codes are defined by */
static uint32_t code_div(float x, float z, float s, int L) {
  if (!(s > 0.0f)) return 0;
  volatile float d = x - z;
  volatile float y = d / s;
  float q = rintf(y);
  if (q < 0.0f) q = 0.0f;
  if (q > (float)L) q = (float)L;
  return (uint32_t)q;
}

/* the kernel's exact rule for an element near a tie ("near": the width's guard) */
static uint32_t code_exact(float x, float z, float s, float r, int L, float guard) {
  if (!(s > 0.0f)) return 0;
  volatile float d = x - z;
  volatile float y = d * r;
  if (y > (float)L + 0.75f) return (uint32_t)L;
  if (!(y > -0.75f)) return 0;
  const float fl = floorf(y), h = fl + 0.5f;
  float q;
  if (fabsf(y - h) > guard) {
    q = rintf(y);
  } else {
    const float rho = fmaf(-h, s, d);
    const int e = ilogbf(h);
    const float hs = s * ldexpf(1.0f, e - 24);
    if (rho > hs) q = fl + 1.0f;
    else if (rho < -hs) q = fl;
    else q = (((int)fl) & 1) ? fl + 1.0f : fl;
  }
  q = fminf(fmaxf(q, 0.0f), (float)L);
  return (uint32_t)q;
}

/* the kernel's fast path: y = (x - z) * r rounded by the 1.5 * 2^23 addition,
   the code the low bits of the sum; near a tie, the exact rule */
static uint32_t code_kernel(float x, float z, float s, float r, int bits, float guard, int* took_exact) {
  const int L = (1 << bits) - 1;
  if (!(s > 0.0f)) return 0;
  volatile float d = x - z;
  volatile float y = d * r;
  volatile float m = y + 12582912.0f;
  volatile float back = m - 12582912.0f;
  const float t = fmaf(back, -1.0f, y);
  if (fabsf(t) > 0.5f - guard) { *took_exact = 1; return code_exact(x, z, s, r, L, guard); }
  uint32_t mb;
  memcpy(&mb, (const void*)&m, 4);
  return mb & (uint32_t)L;
}

static long checked = 0, ties = 0, exact_path = 0, bad = 0;

static void check(uint16_t xh, float z, float s, int bits) {
  const int L = (1 << bits) - 1;
  const float guard = bits <= 4 ? 1e-5f : 1e-4f;
  const float x = h2f(xh);
  const uint32_t want = code_div(x, z, s, L);
  const float r0 = 1.0f / s;
  const float rs[3] = {r0, nextafterf(r0, 0.0f), nextafterf(r0, INFINITY)};
  for (int i = 0; i < 3; ++i) {
    int ex = 0;
    const uint32_t got = code_kernel(x, z, s, rs[i], bits, guard, &ex);
    exact_path += ex;
    ++checked;
    if (got != want) {
      if (bad < 10) fprintf(stderr, "mismatch bits=%d x=%a z=%a s=%a r=%a got=%u want=%u\n", bits, x, z, s, rs[i], got, want);
      ++bad;
    }
  }
}

static uint16_t rand_half(int emin, int emax) {  /* random finite binary16, exponent field in [emin, emax] */
  const int e = emin + (int)(rnd() % (uint64_t)(emax - emin + 1));
  return (uint16_t)(((rnd() & 1) << 15) | (e << 10) | (rnd() & 1023));
}

int main(int argc, char** argv) {
  const long groups = argc > 1 ? atol(argv[1]) : 4000;
  for (int i = 0; i < 0x7C00; ++i) tab[i] = h2f((uint16_t)i);
  const int widths[4] = {2, 3, 4, 8};
  for (int wi = 0; wi < 4; ++wi) {
    const int bits = widths[wi], L = (1 << bits) - 1;
    for (long g = 0; g < groups; ++g) {
      float z, M;
      int tie_group = (g % 3) == 0;
      if (tie_group) {
        /* s = 2^e exactly and z a multiple of s/2: every half-integer of the grid is an fp16 value */
        const int e = -12 + (int)(rnd() % 14);
        const double S = ldexp(1.0, e);
        const long k = (long)(rnd() % 512) - 256;
        uint16_t zh, mh;
        if (!is_half(k * S, &zh) || !is_half(k * S + L * S, &mh)) continue;
        z = h2f(zh); M = h2f(mh);
      } else {
        uint16_t a = rand_half(1, 29), b = rand_half(1, 29);
        if ((rnd() & 3) == 0) {   /* a narrow group near a */
          const float fa = h2f(a);
          uint16_t bb;
          if (!is_half((double)fa + fabs((double)fa) * ldexp(1.0, -(int)(rnd() % 9)) * (double)(rnd() % 8 + 1), &bb)) continue;
          b = bb;
        }
        float fa = h2f(a), fb = h2f(b);
        z = fminf(fa, fb); M = fmaxf(fa, fb);
        if (z == M) continue;
      }
      if (z == 0.0f) z = 0.0f;   /* -0 stored as +0 */
      volatile float span = M - z;
      volatile float q = span / (float)L;
      const uint16_t sh = half_up(q);
      if (sh >= 0x7C00) continue;
      const float s = h2f(sh);
      if (!(s > 0.0f)) continue;
      /* every fp16 value in [z, M] when there are few, else a sample */
      uint16_t zb, mb;
      if (!is_half(z, &zb) || !is_half(M, &mb)) continue;
      long cnt = 0;
      const int zneg = z < 0, mneg = M < 0;
      const long zi = zneg ? -(long)(zb & 0x7FFF) : (long)zb, mi = mneg ? -(long)(mb & 0x7FFF) : (long)mb;
      /* signed index space: -(bits of |x|) for negatives, bits for positives (monotone) */
      if (mi - zi <= 2048) {
        for (long v = zi; v <= mi; ++v) {
          const uint16_t xh = v < 0 ? (uint16_t)(0x8000 | (uint16_t)(-v)) : (uint16_t)v;
          check(xh, z, s, bits); ++cnt;
        }
      } else {
        for (int t = 0; t < 2048; ++t) {
          const long v = zi + (long)(rnd() % (uint64_t)(mi - zi + 1));
          const uint16_t xh = v < 0 ? (uint16_t)(0x8000 | (uint16_t)(-v)) : (uint16_t)v;
          check(xh, z, s, bits); ++cnt;
        }
      }
      /* planted ties: x - z = (k + 1/2) s exactly */
      for (int k = 0; k < L; ++k) {
        uint16_t xh;
        const double X = (double)z + ((double)k + 0.5) * (double)s;
        if (!is_half(X, &xh)) continue;
        volatile float d = h2f(xh) - z;
        if ((double)d != X - (double)z) continue;
        volatile float y = d / s;
        if ((double)y != (double)k + 0.5) continue;
        ++ties;
        check(xh, z, s, bits);
      }
    }
  }
  printf("checked=%ld ties=%ld exact_path=%ld bad=%ld\n", checked, ties, exact_path, bad);
  return bad != 0;
}
"""


def _compiler():
    for cc in (os.environ.get("CC"), "gcc", "cc"):
        if cc and shutil.which(cc):
            return shutil.which(cc)
    return None


def test_division_free_code_rule_matches_division():
    cc = _compiler()
    if cc is None:
        pytest.skip("no C compiler")
    with tempfile.TemporaryDirectory() as d:
        src, exe = os.path.join(d, "exact_code_check.c"), os.path.join(d, "exact_code_check")
        with open(src, "w") as f:
            f.write(PROGRAM)
        # binary32 steps exactly as written: no contraction, no excess precision
        subprocess.run([cc, "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", src, "-o", exe, "-lm"],
                       check=True, capture_output=True, text=True)
        r = subprocess.run([exe, "6000"], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    stats = dict(kv.split("=") for kv in r.stdout.split())
    assert int(stats["bad"]) == 0
    assert int(stats["checked"]) > 5_000_000
    assert int(stats["ties"]) > 20_000            # exact half-integer quotients were planted and met
    assert int(stats["exact_path"]) > 60_000      # and the near-tie path ran for them
