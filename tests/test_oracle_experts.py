"""Pins of the oracle's S7 (w13 GEMM, SiLU-and-mul, requant, w2 GEMM) and S8.

Special cases with closed-form results, a float64 numpy matmul of the
dequantised operands (a library routine), and an independent brute-force
per-token loop: y_t = sum_j w_j * down_e(requant(silu(gate_e(x_t)) * up_e(x_t))).
"""
import numpy as np
import pytest
import torch

from moe_expert_layer_prepare_gb300 import synthetic as syn


def _bf16_bits(t):
    return t.view(torch.int16).numpy().view(np.uint16)


def _bf16_vals(bits):
    return (np.asarray(bits).astype(np.uint32) << 16).view(np.float32)


def _unpack(words, G):
    w = np.asarray(words).astype(np.uint32)
    return np.stack([(w[..., g // 4] >> (8 * (g % 4))) & 0xFF for g in range(G)], axis=-1)


def _deq_weights(table, q, s):
    """fp64 dequantised [E, R, C] from codes and 128x128 block scales."""
    v = table[q].astype(np.float64)
    return v * np.repeat(np.repeat(s.astype(np.float64), 128, axis=1), 128, axis=2)


def _deq_rows(table, q, sf_words):
    G = q.shape[1] // 128
    e = _unpack(sf_words, G).astype(np.int64)
    return table[q].astype(np.float64) * np.repeat(np.ldexp(1.0, e - 127), 128, axis=1)


# --------------------------------------------------------------- special cases
def test_unit_scales_all_ones(orc):
    """q == 1.0 everywhere with unit scales: h = K, y = silu(K) * K, out = N * y."""
    E, M, K, N = 2, 4, 256, 512
    x_b = np.full((E * M, K), 0x38, np.uint8)
    a_sf = np.full((E * M, 1), 127 | 127 << 8, np.int32)
    w13 = np.full((E, 2 * N, K), 0x38, np.uint8)
    w13_s = np.ones((E, 2 * N // 128, K // 128), np.float32)
    w2 = np.full((E, K, N), 0x38, np.uint8)
    w2_s = np.ones((E, K // 128, N // 128), np.float32)
    rows = np.array([0, 3, 5], np.int64)
    h, y_q, y_sf = orc.w13_rows(rows, M, K, N, x_b, a_sf, w13, w13_s, want_h=True)
    assert np.all(_bf16_vals(h[rows]) == 256.0)
    # y = 256 * 256 = 65536 -> scale 2^8 (exponent 135), code of 256 = 0x78
    assert np.all(y_q[rows] == 0x78)
    assert np.all(_unpack(y_sf[rows], N // 128) == 135)
    # untouched rows stay zero
    assert np.all(y_q[[1, 2, 4, 6, 7]] == 0)
    out_b = orc.w2_rows(rows, M, K, N, y_q, y_sf, w2, w2_s)
    assert np.all(_bf16_vals(out_b[rows]) == float(N * 65536))


def test_one_hot_input_selects_weight_column(orc):
    E, M, K, N = 2, 2, 256, 256
    table = orc.e4m3_decode_table()
    w13, w13_s = syn.make_block_fp8_weights(E, 2 * N, K, 21)
    w13, w13_s = w13.numpy(), w13_s.numpy()
    x_b = np.zeros((E * M, K), np.uint8)
    k0 = 137
    x_b[:, k0] = 0x38
    a_sf = np.full((E * M, 1), 127 | 127 << 8, np.int32)
    rows = np.arange(E * M, dtype=np.int64)
    h, _, _ = orc.w13_rows(rows, M, K, N, x_b, a_sf, w13, w13_s, want_h=True)
    for r in rows:
        e = r // M
        exact = table[w13[e, :, k0]].astype(np.float64) * w13_s[e, :, k0 // 128].astype(
            np.float64).repeat(128)
        got = _bf16_vals(h[r]).astype(np.float64)
        # bf16 rounding of one exact product: within half a bf16 ulp
        assert np.all(np.abs(got - exact) <= np.abs(exact) * 2.0 ** -8 + 1e-30)


def test_silu_zero_gate_and_large_gate(orc):
    E, M, K, N = 1, 2, 128, 128
    x_b = np.zeros((E * M, K), np.uint8)
    x_b[:, 0] = 0x38                     # x = e_0
    a_sf = np.full((E * M, 1), 127, np.int32)
    w13 = np.zeros((E, 2 * N, K), np.uint8)
    w13_s = np.ones((E, 2, 1), np.float32)
    # row 0: gate = 0 -> y = 0 ; up column = 3.0
    w13[0, N:, 0] = 0x44                 # 3.0
    rows = np.array([0], np.int64)
    h, y_q, y_sf = orc.w13_rows(rows, M, K, N, x_b, a_sf, w13, w13_s, want_h=True)
    assert np.all(_bf16_vals(h[0, :N]) == 0.0)
    table = orc.e4m3_decode_table()
    assert np.all(table[y_q[0]] == 0.0)
    assert _unpack(y_sf[0:1], 1)[0, 0] == 105
    # gate = 96 (silu(96) == 96 in fp64), up = 3 -> y = 288 -> scale 1, code(288)
    w13[0, :N, 0] = 0x6C                 # 1.5 * 2^6 = 96
    h, y_q, y_sf = orc.w13_rows(rows, M, K, N, x_b, a_sf, w13, w13_s, want_h=True)
    assert np.all(_bf16_vals(h[0, :N]) == 96.0)
    assert _unpack(y_sf[0:1], 1)[0, 0] == 127
    assert np.all(table[y_q[0]] == 288.0)


# ---------------------------------------------------------- library matmul
def test_gemms_vs_numpy_float64(orc):
    E, M, K, N = 3, 8, 512, 256
    table = orc.e4m3_decode_table()
    rng = np.random.default_rng(9)
    hid = syn.make_hidden(E * M, K, 13)
    st = orc.prepare_inputs(_bf16_bits(hid), np.zeros((E * M, 1), np.int32),
                            np.ones((E * M, 1), np.float32))
    x_b, a_sf = st["x"], st["x_sf"]
    w13, w13_s = (t.numpy() for t in syn.make_block_fp8_weights(E, 2 * N, K, 31))
    w2, w2_s = (t.numpy() for t in syn.make_block_fp8_weights(E, K, N, 32))
    # a random subset of rows; the others must stay untouched
    rows = np.sort(rng.choice(E * M, size=14, replace=False)).astype(np.int64)
    h, y_q, y_sf = orc.w13_rows(rows, M, K, N, x_b, a_sf, w13, w13_s, want_h=True)
    out_b = orc.w2_rows(rows, M, K, N, y_q, y_sf, w2, w2_s)
    A = _deq_rows(table, x_b, a_sf)
    W13 = _deq_weights(table, w13, w13_s)
    W2 = _deq_weights(table, w2, w2_s)
    Y = _deq_rows(table, y_q, y_sf)
    for r in rows:
        e = r // M
        ref_h = W13[e] @ A[r]
        got_h = _bf16_vals(h[r]).astype(np.float64)
        assert np.all(np.abs(got_h - ref_h) <= np.abs(ref_h) * 2.0 ** -8 + 1e-12)
        ref_o = W2[e] @ Y[r]
        got_o = _bf16_vals(out_b[r]).astype(np.float64)
        assert np.all(np.abs(got_o - ref_o) <= np.abs(ref_o) * 2.0 ** -8 + 1e-12)
    others = np.setdiff1d(np.arange(E * M), rows)
    assert np.all(h[others] == 0) and np.all(out_b[others] == 0)
    # a transposed weight would break the check above; so would swapping gate/up:
    g = _bf16_vals(h[rows[0], :N]).astype(np.float64)
    u = _bf16_vals(h[rows[0], N:]).astype(np.float64)
    silu = g / (1 + np.exp(-g))
    y = silu * u
    Yr = Y[rows[0]]
    assert np.linalg.norm(Yr - y) <= 0.08 * np.linalg.norm(y)


# ------------------------------------------------------------------ S8 reduce
def test_reduce_gather_and_convex(orc):
    T, K, M = 6, 256, 8
    E = 3
    rng = np.random.default_rng(3)
    ob = _bf16_bits(torch.from_numpy(rng.standard_normal((E * M, K), dtype=np.float32))
                    .to(torch.bfloat16))
    ids = np.array([[0], [1], [2], [-1], [1], [0]], np.int64)
    slot = np.array([[0], [3], [7], [-1], [2], [-1]], np.int32)
    w = np.ones((T, 1), np.float32)
    out = orc.topk_reduce(ob, ids, slot, w, M)
    assert np.array_equal(out[0], ob[0 * M + 0])
    assert np.array_equal(out[1], ob[1 * M + 3])
    assert np.array_equal(out[2], ob[2 * M + 7])
    assert np.all(out[3] == 0) and np.all(out[5] == 0)
    # identical expert outputs with weights 0.25 + 0.75 -> the same row
    ob2 = ob.copy()
    ob2[1 * M + 5] = ob2[0 * M + 2]
    ids2 = np.array([[0, 1]], np.int64)
    slot2 = np.array([[2, 5]], np.int32)
    out2 = orc.topk_reduce(ob2, ids2, slot2, np.array([[0.25, 0.75]], np.float32), M)
    assert np.array_equal(out2[0], ob2[2])
    del rng


def test_reduce_token_bound(orc):
    """moe_fused_mul_sum's num_valid_tokens: rows below the bound are the
    unbounded reduce's, rows at or past it are not written; a bound at or past
    T, or none, is the plain reduce; a bound of 0 writes nothing."""
    T, K, M, E, k = 9, 128, 4, 3, 2
    rng = np.random.default_rng(8)
    ob = _bf16_bits(torch.from_numpy(rng.standard_normal((E * M, K), dtype=np.float32))
                    .to(torch.bfloat16))
    ids = rng.integers(0, E, size=(T, k)).astype(np.int64)
    slot = rng.integers(0, M, size=(T, k)).astype(np.int32)
    w = rng.random((T, k)).astype(np.float32)
    full = orc.topk_reduce(ob, ids, slot, w, M)
    for bound in (0, 1, 5, T, T + 3):
        got = orc.topk_reduce(ob, ids, slot, w, M, num_valid=bound, fill=0xFFFF)
        n = min(bound, T)
        assert np.array_equal(got[:n], full[:n])
        assert np.all(got[n:] == 0xFFFF)
    # the contiguous layout (rows in route_slot) obeys the same bound
    rows = (ids * M + slot).astype(np.int32)
    got = orc.topk_reduce(ob, None, rows, w, M, num_valid=4, fill=0xFFFF)
    assert np.array_equal(got[:4], full[:4]) and np.all(got[4:] == 0xFFFF)


# ------------------------------------------------------- brute force, tiny
def _requant_closed_form(y):
    """Independent requant of one fp32 vector in 128-groups (torch cast)."""
    y = y.astype(np.float32)
    out = np.empty_like(y, dtype=np.float64)
    floor = float(np.float32(1e-4))
    for g in range(y.size // 128):
        seg = y[g * 128:(g + 1) * 128]
        a = max(float(np.abs(seg).max()), floor)
        n = -200
        while 448.0 * 2.0 ** n < a:
            n += 1
        qs = 2.0 ** n
        scaled = torch.from_numpy((seg.astype(np.float64) / qs).astype(np.float32))
        q = scaled.to(torch.float8_e4m3fn).to(torch.float64).numpy()
        out[g * 128:(g + 1) * 128] = q * qs
    return out


def _bf16_round(v):
    return torch.from_numpy(np.asarray(v, np.float64)).to(torch.float32).to(
        torch.bfloat16).to(torch.float64).numpy()


def test_brute_force_per_token_tiny(orc):
    wl = syn.make_workload("tiny")
    c = wl["cfg"]
    T, K, N, E, k, M = c["T"], c["K"], c["N"], c["E"], c["top_k"], c["M_max"]
    table = orc.e4m3_decode_table()
    bits = _bf16_bits(wl["hidden"])
    w13, w13_s, w2, w2_s = (wl[n].numpy() for n in ("w13", "w13_s", "w2", "w2_s"))
    res = orc.forward(bits, wl["topk_ids"].numpy(), wl["topk_weights"].numpy(), w13, w13_s,
                      w2, w2_s, E, M, N)
    assert res["dispatch"]["status"] == 0
    st = res["staging"]
    Xq = _deq_rows(table, st["x"], st["x_sf"])
    W13 = _deq_weights(table, w13, w13_s)
    W2 = _deq_weights(table, w2, w2_s)
    Xraw = _bf16_vals(bits).astype(np.float64)
    brute = np.zeros((T, K))
    unquant = np.zeros((T, K))
    for t in range(T):
        for j in range(k):
            e = st["ids"][t, j]
            wt = float(st["weights"][t, j])
            h = _bf16_round(W13[e] @ Xq[t])
            y = (h[:N] / (1 + np.exp(-h[:N]))) * h[N:]
            o = _bf16_round(W2[e] @ _requant_closed_form(y))
            brute[t] += wt * o
            hu = W13[e] @ Xraw[t]
            unquant[t] += wt * (W2[e] @ ((hu[:N] / (1 + np.exp(-hu[:N]))) * hu[N:]))
    got = _bf16_vals(res["out"]).astype(np.float64)
    ref = _bf16_round(brute)
    rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    assert rel < 2e-3, rel
    assert np.mean(got == ref) > 0.95
    # against the unquantised math: within the quantisation error
    rel_u = np.linalg.norm(got - unquant) / np.linalg.norm(unquant)
    assert rel_u < 0.1, rel_u


@pytest.mark.parametrize("mistake", ["transpose_w2_scale", "swap_gate_up"])
def test_brute_force_detects_planted_mistakes(orc, mistake):
    """A planted mistake on the oracle's inputs changes the tiny output visibly."""
    wl = syn.make_workload("tiny")
    c = wl["cfg"]
    bits = _bf16_bits(wl["hidden"])
    args = [wl[n].numpy() for n in ("w13", "w13_s", "w2", "w2_s")]
    base = orc.forward(bits, wl["topk_ids"].numpy(), wl["topk_weights"].numpy(), *args,
                       c["E"], c["M_max"], c["N"])["out"]
    w13, w13_s, w2, w2_s = [a.copy() for a in args]
    if mistake == "transpose_w2_scale":
        w2_s = np.ascontiguousarray(np.flip(w2_s, axis=2))
    else:
        N = c["N"]
        w13 = np.concatenate([w13[:, N:], w13[:, :N]], axis=1)
        w13_s = np.concatenate([w13_s[:, N // 128:], w13_s[:, :N // 128]], axis=1)
    bad = orc.forward(bits, wl["topk_ids"].numpy(), wl["topk_weights"].numpy(), w13, w13_s,
                      w2, w2_s, c["E"], c["M_max"], c["N"])["out"]
    a = _bf16_vals(base).astype(np.float64)
    b = _bf16_vals(bad).astype(np.float64)
    assert np.linalg.norm(a - b) > 0.05 * np.linalg.norm(a)


def test_fp32_activation_scales_match_ue8m0_when_powers_of_two(orc):
    """The fp32 a1q_scale path dequantises with the fp32 scale itself; fed
    the UE8M0 scales 2^(e-127) as fp32 it must reproduce the packed-exponent
    rows bit for bit (the two modes differ only in how the scale is held)."""
    from moe_expert_layer_prepare_gb300 import synthetic as syn
    from tests._util import bf16_bits
    T, K, N, E = 12, 384, 256, 2
    hid = syn.make_hidden(T, K, 77, outlier_frac=0.05)
    st = orc.prepare_inputs(bf16_bits(hid), np.zeros((T, 1), np.int32),
                            np.ones((T, 1), np.float32))
    words = st["x_sf"]
    G = K // 128
    exps = np.array([[(int(words[t, g // 4]) >> (8 * (g % 4))) & 0xFF for g in range(G)]
                     for t in range(T)], np.uint32)
    scales = (exps << 23).view(np.float32)  # 2^(e - 127)
    w13, w13_s = syn.make_block_fp8_weights(E, 2 * N, K, 78)
    rows = np.arange(T)
    packed = orc.w13_rows(rows, T, K, N, st["x"], words, w13.numpy(), w13_s.numpy(), want_h=True)
    fp32 = orc.w13_rows(rows, T, K, N, st["x"], scales, w13.numpy(), w13_s.numpy(), want_h=True)
    for a, b in zip(packed, fp32):
        assert np.array_equal(a, b)
    # a scale that is not a power of two changes the result in proportion
    scaled = orc.w13_rows(rows, T, K, N, st["x"], scales * np.float32(1.5), w13.numpy(),
                          w13_s.numpy(), want_h=True)
    from tests._util import bf16_vals
    h1, h15 = bf16_vals(packed[0]).astype(np.float64), bf16_vals(scaled[0]).astype(np.float64)
    assert np.all(np.abs(h15 - 1.5 * h1) <= 2.0 ** -7 * np.abs(1.5 * h1) + 1e-30)
