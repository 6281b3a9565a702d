"""Pins of the oracle's NVFP4 staging (N1 E2M1 codec, N2 token rows).

* E2M1 values: the code table of the OCP MX specification (golden file).
* E2M1 rounding: brute force over a dense grid against the nearest table
  value with ties to the even code, saturating at 6.
* Rows: x_scale = amax / 2688 in fp32; dequantisation q * s * x_scale is
  within a quarter of the block's magnitude (half the widest E2M1 gap plus
  the E4M3 rounding of the scale); rows whose values are E2M1 grid values
  times one power of two come back with exactly those codes; zero rows and
  the nibble / scale-byte order.
"""
import os

import numpy as np
import pytest

from tests._util import bf16_bits
import torch

GOLD = os.path.join(os.path.dirname(__file__), "golden", "e2m1_values.txt")


def _table():
    rows = [l.split() for l in open(GOLD) if l.strip() and not l.startswith("#")]
    return {int(c): float(v) for c, v in rows}


def test_e2m1_values_match_spec(orc):
    for c, v in _table().items():
        got = orc.e2m1_decode(c)
        assert got == v and np.signbit(got) == np.signbit(v), (c, got, v)


def test_e2m1_rounding_brute_force(orc):
    tab = _table()
    mags = np.array([tab[c] for c in range(8)])
    for a in np.concatenate([np.linspace(0, 7, 2801), [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]]):
        for sgn in (1.0, -1.0):
            v = np.float32(sgn * a)
            code = orc.e2m1_encode(float(v))
            if a >= 6:
                want = 7
            else:
                d = np.abs(mags - a)
                best = np.flatnonzero(d == d.min())
                want = int(best[0] if len(best) == 1 else best[best % 2 == 0][0])
            assert code & 7 == want, (v, code, want)
            assert (code >> 3) == (1 if np.signbit(v) else 0)


def _dequant(orc, res, K):
    tab = np.array([orc.e2m1_decode(c) for c in range(16)], np.float64)
    x = res["x"].astype(np.int64)
    codes = np.stack([x & 0xF, x >> 4], axis=-1).reshape(x.shape[0], K)
    sbytes = res["x_sf"].view(np.uint8)[:, :K // 16]
    s = np.array([orc.e4m3_decode(int(b)) for b in sbytes.ravel()]).reshape(sbytes.shape)
    return tab[codes] * np.repeat(s, 16, axis=1) * res["x_scales"].astype(np.float64)[:, None], \
        codes, sbytes


def test_rows_scale_and_error_bound(orc):
    rng = np.random.default_rng(9)
    T, K = 40, 512
    x = rng.standard_normal((T, K)).astype(np.float32) * np.exp(rng.uniform(-8, 8, (T, 1))).astype(np.float32)
    x[3] = 0.0                        # all-zero row
    x[5, :16] = 0.0                   # an all-zero block
    x[7, 100] = 1e4 * np.abs(x[7]).max()  # one large outlier dwarfs the rest
    bits = bf16_bits(torch.from_numpy(x).to(torch.bfloat16))
    xb = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    res = orc.nvfp4_rows(bits)
    amax = np.abs(xb).max(axis=1).astype(np.float32)
    assert np.array_equal(res["x_scales"], amax / np.float32(2688.0))
    deq, codes, sb = _dequant(orc, res, K)
    bmax = np.abs(xb).reshape(T, K // 16, 16).max(axis=2)
    bound = np.repeat(0.26 * bmax, 16, axis=1) + 1e-30
    assert np.all(np.abs(deq - xb) <= bound)
    assert np.all(codes[3] == 0) and np.all(sb[3] == 0) and res["x_scales"][3] == 0
    assert np.all(codes[5, :16] == 0)
    # the largest element of a row always gets the largest code of its block
    for t in range(T):
        if amax[t] > 0:
            i = int(np.argmax(np.abs(xb[t])))
            assert codes[t, i] & 7 == 7


def test_grid_rows_round_trip(orc):
    tab = _table()
    rng = np.random.default_rng(4)
    T, K = 8, 256
    grid = np.array([tab[c] for c in range(16)], np.float32)
    for t in range(T):
        want = rng.integers(0, 16, size=K)
        want[rng.integers(0, K)] = 7  # the row amax is 6 * 2^j
        for b in range(K // 16):
            want[b * 16] = 7 if rng.random() < 0.5 else 15  # every block reaches |6|
        xv = grid[want] * np.float32(2.0 ** int(rng.integers(-20, 20)))
        bits = bf16_bits(torch.from_numpy(xv[None]).to(torch.bfloat16))
        res = orc.nvfp4_rows(bits)
        _, codes, sb = _dequant(orc, res, K)
        # zero codes keep their sign bit; compare magnitudes and signs of nonzeros
        nz = (want & 7) != 0
        assert np.array_equal(codes[0][nz], want[nz])
        assert np.all(codes[0][~nz] & 7 == 0)
        assert np.all(sb[0] == 0x7E)  # every block scale is 448 = 2688 / 6
