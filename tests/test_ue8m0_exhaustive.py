"""The CUDA kernels form the UE8M0 exponent of a 1x128 group without a
division: with b the fp32 bits of a = max(amax, 1e-4), the exponent is
expfield(b) - 8 plus one when the mantissa field exceeds 0x600000 (the
mantissa of 448 = 1.75 * 2^8), clamped to [1, 254], and 254 for an infinite
amax.  The page's recipe (prepare_megamoe, _quantize_fp8_groups) divides:
s = a / 448 in fp32, then the exponent field of s plus one when its mantissa is
not zero, clamped to [1, 254].

The w13 epilogue feeds this form arbitrary fp32 amax values (the SiLU-and-mul
products), not only bf16 ones, so it is checked here over every non-negative
fp32 value: all 2^31 - 2^23 finite patterns and +inf.  NaN is left undefined
(the pages do not define NaN inputs)."""
import os
import shutil
import subprocess

import pytest

SRC = r"""
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

static uint32_t bits_of(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }

/* the page's form: divide, round the power of two up, clamp */
static uint32_t page_form(float amax) {
  const float a = fmaxf(amax, 1.0e-4f);
  const float s = a / 448.0f;
  const uint32_t b = bits_of(s);
  uint32_t e = ((b >> 23) & 0xFFu) + ((b & 0x7FFFFFu) != 0u ? 1u : 0u);
  if (e < 1u) e = 1u;
  if (e > 254u) e = 254u;
  return e;
}

/* the kernels' division-free form (ue8m0_exponent in csrc/common.cuh) */
static uint32_t kernel_form(float amax) {
  const uint32_t b = bits_of(fmaxf(amax, 1.0e-4f));
  uint32_t e = ((b >> 23) & 0xFFu) - 8u + ((b & 0x7FFFFFu) > 0x600000u ? 1u : 0u);
  if (e < 1u) e = 1u;
  if (e > 254u) e = 254u;
  return b >= 0x7F800000u ? 254u : e;
}

int main(void) {
  long bad = 0, checked = 0;
  unsigned long first_bad = 0;
#pragma omp parallel for reduction(+ : bad, checked) schedule(static, 1 << 20)
  for (int64_t i = 0; i <= 0x7F800000; ++i) {
    const uint32_t u = (uint32_t)i;
    float x;
    memcpy(&x, &u, 4);
    ++checked;
    if (page_form(x) != kernel_form(x)) {
      ++bad;
#pragma omp critical
      if (first_bad == 0) first_bad = u;
    }
  }
  printf("%ld %ld %lu\n", bad, checked, first_bad);
  return 0;
}
"""


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_ue8m0_division_free_form_matches_page_over_all_fp32(tmp_path):
    c = tmp_path / "ue8m0.c"
    c.write_text(SRC)
    exe = tmp_path / "ue8m0"
    subprocess.run(["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-o", str(exe), str(c), "-lm"],
                   check=True)
    env = dict(os.environ, OMP_NUM_THREADS=str(min(16, os.cpu_count() or 1)))
    bad, checked, first = map(int, subprocess.run([str(exe)], check=True, capture_output=True,
                                                  text=True, env=env).stdout.split())
    assert checked == 0x7F800001
    assert bad == 0, f"{bad} amax values differ, first bits {first:#010x}"
