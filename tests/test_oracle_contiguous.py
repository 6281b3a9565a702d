"""Pins of the oracle's contiguous layout (S6b) against its batched layout (S6).

The two layouts hold the same routed rows in different places: the row of
route (t, j) in the contiguous layout must be the first row of its expert plus
the slot the batched dispatch gives it, the experts' row ranges must tile
[0, R) in expert order, and the GEMM rows and the reduce must give identical
results whichever layout holds the data.
"""
import numpy as np
import pytest

from moe_expert_layer_prepare_gb300 import synthetic as syn
from tests._util import bf16_bits


def _staged(orc, T, K, E, k, seed, zipf=None, pad=0.0):
    hid = syn.make_hidden(T, K, seed)
    ids, w, p = syn.make_routing(T, E, k, seed + 1, zipf_s=zipf, padding_frac=pad)
    st = orc.prepare_inputs(bf16_bits(hid), ids.numpy(), w.numpy(), is_padding=p.numpy())
    return st


@pytest.mark.parametrize("T,K,E,k,zipf,pad", [(40, 256, 4, 2, None, 0.1),
                                               (300, 384, 16, 4, 1.1, 0.05)])
def test_rows_are_offsets_plus_batched_slots(orc, T, K, E, k, zipf, pad):
    st = _staged(orc, T, K, E, k, T + E, zipf, pad)
    c = orc.dispatch_contiguous(st["ids"], st["x"], st["x_sf"], E)
    b = orc.dispatch(st["ids"], st["x"], st["x_sf"], E, T * k)
    assert c["status"] == 0 and b["status"] == 0
    n = b["expert_num_tokens"]
    assert np.array_equal(c["expert_num_tokens"], n)
    assert np.array_equal(c["expert_offsets"], np.concatenate([[0], np.cumsum(n)]))
    routed = st["ids"] >= 0
    want = np.where(routed, c["expert_offsets"][np.maximum(st["ids"], 0)] + b["route_slot"], -1)
    assert np.array_equal(c["route_row"], want)
    # each routed row appears once and holds its token's bytes and exponents
    rows = c["route_row"][routed]
    assert sorted(rows.tolist()) == list(range(int(routed.sum())))
    t_of = np.nonzero(routed)[0]
    assert np.array_equal(c["x_c"][rows], st["x"][t_of])
    assert np.array_equal(c["sf_c"][rows], st["x_sf"][t_of])
    # the expert of each row follows the offsets
    for e in range(E):
        lo, hi = c["expert_offsets"][e], c["expert_offsets"][e + 1]
        assert np.all(c["row_expert"][lo:hi] == e)


def test_gemm_rows_and_reduce_agree_across_layouts(orc):
    T, K, N, E, k = 24, 256, 256, 3, 2
    st = _staged(orc, T, K, E, k, 11)
    w13, w13_s = syn.make_block_fp8_weights(E, 2 * N, K, 12)
    w2, w2_s = syn.make_block_fp8_weights(E, K, N, 13)
    c = orc.dispatch_contiguous(st["ids"], st["x"], st["x_sf"], E)
    M = T  # batched capacity
    b = orc.dispatch(st["ids"], st["x"], st["x_sf"], E, M)
    R = int(c["expert_offsets"][-1])
    crows = np.arange(R)
    h_c, yq_c, ysf_c = orc.w13_rows(crows, 1, K, N, c["x_c"], c["sf_c"], w13.numpy(),
                                    w13_s.numpy(), want_h=True, row_expert=c["row_expert"])
    brows = orc.valid_rows(b["expert_num_tokens"], M)
    h_b, yq_b, ysf_b = orc.w13_rows(brows, M, K, N, b["x_b"], b["sf_b"], w13.numpy(),
                                    w13_s.numpy(), want_h=True)
    # batched row of each contiguous row
    routed = st["ids"] >= 0
    crow = c["route_row"][routed]
    brow = (st["ids"][routed] * M + b["route_slot"][routed]).astype(np.int64)
    assert np.array_equal(h_c[crow], h_b[brow])
    assert np.array_equal(yq_c[crow], yq_b[brow]) and np.array_equal(ysf_c[crow], ysf_b[brow])
    o_c = orc.w2_rows(crows, 1, K, N, yq_c, ysf_c, w2.numpy(), w2_s.numpy(),
                      row_expert=c["row_expert"])
    o_b = orc.w2_rows(brows, M, K, N, yq_b, ysf_b, w2.numpy(), w2_s.numpy())
    assert np.array_equal(o_c[crow], o_b[brow])
    out_c = orc.topk_reduce(o_c, None, c["route_row"], st["weights"], 1)
    out_b = orc.topk_reduce(o_b, st["ids"], b["route_slot"], st["weights"], M)
    assert np.array_equal(out_c, out_b)
