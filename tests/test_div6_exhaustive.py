"""The NVFP4 staging kernel forms the block scale E4M3(bmax / 6) from a
branch-free quotient: q0 = bmax * RN(1/6), r = fma(-q0, 6, bmax),
q = fma(r, RN(1/6), q0) (Markstein's correction step), with infinities passed
through.  Check, over every non-negative fp32 input and NaN, that q is the
IEEE quotient, or that both are below 2^-126, where any round-to-nearest
E4M3 encoding gives code 0 (its smallest step is 2^-9)."""
import os
import shutil
import subprocess

import pytest

SRC = r"""
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>
int main(void) {
  const float zh = (float)(1.0 / 6.0);
  long bad = 0, sub = 0;
#pragma omp parallel for reduction(+ : bad, sub) schedule(static, 1 << 20)
  for (int64_t i = 0; i <= 0x7FFFFFFF; ++i) {
    const uint32_t u = (uint32_t)i;
    float x;
    memcpy(&x, &u, 4);
    const float ref = x / 6.0f;
    const float q0 = x * zh;
    const float r = fmaf(-q0, 6.0f, x);
    float q = fmaf(r, zh, q0);
    if (isinf(x)) q = x;
    uint32_t a, b;
    memcpy(&a, &q, 4);
    memcpy(&b, &ref, 4);
    if (a == b || (isnan(q) && isnan(ref))) continue;
    if (fabsf(ref) < 0x1p-126f && fabsf(q) < 0x1p-126f) ++sub; else ++bad;
  }
  printf("%ld %ld\n", bad, sub);
  return 0;
}
"""


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_div6_matches_ieee_for_e4m3(tmp_path):
    c = tmp_path / "div6.c"
    c.write_text(SRC)
    exe = tmp_path / "div6"
    # no contraction: every product and fma is rounded exactly as written
    subprocess.run(["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-o", str(exe), str(c), "-lm"],
                   check=True)
    env = dict(os.environ, OMP_NUM_THREADS=str(min(16, os.cpu_count() or 1)))
    bad, sub = map(int, subprocess.run([str(exe)], check=True, capture_output=True, text=True,
                                       env=env).stdout.split())
    assert bad == 0
    assert 0 < sub < 1 << 22  # the subnormal quotients only
