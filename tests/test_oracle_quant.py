"""Pins of the oracle's S1-S4 (e4m3 code, UE8M0 group scale, quantise, pack).

Each pin checks the oracle against something other than itself: the OCP E4M3
definition (hand-worked codes), PyTorch's own float8_e4m3fn cast (a library
routine) over every bf16 pattern, the UE8M0 closed form in exact rational
arithmetic, hand-worked exponents, and the dequantisation error bound.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                rows.append(line.split())
    return rows


def _f32(x):
    return float(np.float32(x))


# ---------------------------------------------------------------- S1 e4m3
def test_e4m3_decode_table_definition(orc):
    t = orc.e4m3_decode_table()
    assert t[0x00] == 0.0 and math.copysign(1, t[0x80]) < 0
    assert t[0x01] == 2.0 ** -9 and t[0x07] == 7 * 2.0 ** -9
    assert t[0x08] == 2.0 ** -6 and t[0x38] == 1.0 and t[0x7E] == 448.0
    assert np.isnan(t[0x7F]) and np.isnan(t[0xFF])
    assert t[0xFE] == -448.0
    finite = t[:0x7F]
    assert np.all(np.diff(finite) > 0), "codes 0x00..0x7E must increase"
    assert np.array_equal(t[0x80:0xFF], -t[0x00:0x7F])


def test_e4m3_golden_codes(orc):
    for val, code in _read_golden("e4m3_codes.txt"):
        assert orc.e4m3_encode(_f32(float(val))) == int(code, 16), val


@pytest.mark.parametrize("scale", [1.0, 2.0 ** -3, 2.0 ** 5, 2.0 ** -20, 3.0 / 7.0])
def test_e4m3_exhaustive_vs_torch(orc, scale):
    """All 65536 bf16 patterns times a scale, against torch's float8_e4m3fn cast.

    torch turns magnitudes >= 464 into NaN where the page's cast saturates, so
    the comparison covers |v| < 464 and the saturation is pinned separately.
    """
    bits = np.arange(65536, dtype=np.uint32) << 16
    v = bits.view(np.float32) * np.float32(scale)
    keep = np.isfinite(v) & (np.abs(v) < 464.0)
    v = v[keep]
    ours = orc.e4m3_encode_array(v)
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    bad = np.nonzero(ours != ref)[0]
    assert bad.size == 0, [(float(v[i]), hex(ours[i]), hex(ref[i])) for i in bad[:5]]


def test_e4m3_saturates(orc):
    for v in [448.0, 464.0, 479.0, 480.0, 1e6, 3.0e38]:
        assert orc.e4m3_encode(v) == 0x7E
        assert orc.e4m3_encode(-v) == 0xFE


# ---------------------------------------------------------------- S2 UE8M0
def _closed_form_exponent(amax_f32: float) -> int:
    """127 + ceil(log2(max(amax, 1e-4) / 448)) in exact rational arithmetic."""
    floor = Fraction(_f32(1e-4))
    a = max(Fraction(amax_f32), floor)
    q = a / 448
    n = q.numerator.bit_length() - q.denominator.bit_length()
    while Fraction(2) ** n < q:
        n += 1
    while Fraction(2) ** (n - 1) >= q:
        n -= 1
    return min(max(n + 127, 1), 254)


def test_ue8m0_golden(orc):
    for amax, e in _read_golden("ue8m0_exponents.txt"):
        code, qs = orc.group_scale(_f32(float(amax)), True)
        assert code == int(e), amax
        assert qs == 2.0 ** (int(e) - 127)
        assert _closed_form_exponent(_f32(float(amax))) == int(e)


def test_ue8m0_closed_form_all_bf16(orc):
    """The bit trick equals the exact closed form for every finite bf16 amax."""
    bits = (np.arange(0, 0x7F80, dtype=np.uint32) << 16)
    vals = bits.view(np.float32)
    seen = set()
    for a in vals[::1]:
        a = float(a)
        code, qs = orc.group_scale(a, True)
        exp = _closed_form_exponent(a)
        assert code == exp, (a, code, exp)
        assert 105 <= code <= 247
        seen.add(code)
    assert min(seen) == 105 and max(seen) == 247


def test_ue8m0_clamp_and_fp32_mode(orc):
    # the clamp only bites for fp32 amax far outside bf16-reachable values
    code, _ = orc.group_scale(3.0e38, True)
    assert code == 247
    code, qs = orc.group_scale(_f32(3.0), False)
    assert qs == _f32(np.float32(3.0) / np.float32(448.0))
    assert code == np.array([qs], np.float32).view(np.uint32)[0]
    code, qs = orc.group_scale(0.0, False)
    assert qs == _f32(np.float32(1e-4) / np.float32(448.0))


# ---------------------------------------------------------------- S3/S4 staging
def _bf16_bits(t):
    return t.view(torch.int16).numpy().view(np.uint16)


def _bf16_vals(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32)


def _unpack(words, G):
    w = words.astype(np.uint32)
    return np.stack([(w[:, g // 4] >> (8 * (g % 4))) & 0xFF for g in range(G)], axis=1)


def test_quantise_error_bound_and_range(orc):
    from moe_expert_layer_prepare_gb300 import synthetic as syn
    T, K = 64, 1024
    hid = syn.make_hidden(T, K, 7, outlier_frac=0.01, zero_group_frac=0.05)
    bits = _bf16_bits(hid)
    ids = np.zeros((T, 1), np.int32)
    st = orc.prepare_inputs(bits, ids, np.ones((T, 1), np.float32))
    G = K // 128
    exps = _unpack(st["x_sf"], G)
    table = orc.e4m3_decode_table().astype(np.float64)
    x = _bf16_vals(bits).astype(np.float64).reshape(T, G, 128)
    q = table[st["x"]].reshape(T, G, 128)
    qs = np.ldexp(1.0, exps.astype(np.int64) - 127)[:, :, None]
    assert not np.any(st["x"] == 0x7F) and not np.any(st["x"] == 0xFF)
    # no element needs saturation: |x / qs| <= 448
    assert np.all(np.abs(x / qs) <= 448.0)
    amax = np.maximum(np.abs(x).max(axis=2, keepdims=True), np.float32(1e-4))
    assert np.all(qs < 2 * amax / 448.0) and np.all(qs >= amax / 448.0)
    err = np.abs(x - q * qs)
    bound = np.maximum(np.abs(x) * 2.0 ** -4, qs * 2.0 ** -10)
    assert np.all(err <= bound)
    # all-zero groups take the floor: exponent 105 and +0 codes
    zero_groups = np.all(x == 0, axis=2)
    assert zero_groups.any()
    assert np.all(exps[zero_groups] == 105)
    assert np.all(st["x"].reshape(T, G, 128)[zero_groups] == 0)


def test_quantise_worked_group(orc):
    # a group whose amax is 448: exponent 127, 448 -> 0x7E, 1 -> 0x38
    v = np.zeros((1, 128), np.float32)
    v[0, 0] = 448.0
    v[0, 1] = 1.0
    v[0, 2] = -3.5
    bits = _bf16_bits(torch.from_numpy(v).to(torch.bfloat16))
    st = orc.prepare_inputs(bits, np.zeros((1, 1), np.int32), np.ones((1, 1), np.float32))
    assert st["x_sf"][0, 0] == 127
    assert st["x"][0, 0] == 0x7E and st["x"][0, 1] == 0x38 and st["x"][0, 2] == 0xC6
    assert np.all(st["x"][0, 3:] == 0)


def test_pack_bytes_order(orc):
    """Exponent of group g is byte g%4 of word g/4; unused bytes are zero."""
    K = 128 * 6  # G = 6 -> 2 words, the second half-filled
    v = np.zeros((1, K), np.float32)
    scales = [1.0, 2.0, 4.0, 8.0, 16.0, 32.0]
    for g, s in enumerate(scales):
        v[0, g * 128] = 448.0 * s
    bits = _bf16_bits(torch.from_numpy(v).to(torch.bfloat16))
    st = orc.prepare_inputs(bits, np.zeros((1, 1), np.int32), np.ones((1, 1), np.float32))
    w = st["x_sf"][0].astype(np.uint32)
    assert w[0] == (127 | 128 << 8 | 129 << 16 | 130 << 24)
    assert w[1] == (131 | 132 << 8)
    # G = 2: upper bytes of the single word stay zero
    st2 = orc.prepare_inputs(bits[:, :256], np.zeros((1, 1), np.int32),
                             np.ones((1, 1), np.float32))
    assert st2["x_sf"].shape == (1, 1) and st2["x_sf"][0, 0] == (127 | 128 << 8)


def test_fp32_scale_mode(orc):
    from moe_expert_layer_prepare_gb300 import synthetic as syn
    hid = syn.make_hidden(8, 256, 3)
    bits = _bf16_bits(hid)
    st = orc.prepare_inputs(bits, np.zeros((8, 1), np.int32), np.ones((8, 1), np.float32),
                            sf_mode=2)
    x = _bf16_vals(bits).reshape(8, 2, 128)
    amax = np.maximum(np.abs(x).max(axis=2), np.float32(1e-4)).astype(np.float32)
    assert np.array_equal(st["x_sf"], (amax / np.float32(448.0)).astype(np.float32))


def test_shape_error(orc):
    with pytest.raises(ValueError):
        orc.prepare_inputs(np.zeros((2, 100), np.uint16), np.zeros((2, 1), np.int32),
                           np.ones((2, 1), np.float32))
