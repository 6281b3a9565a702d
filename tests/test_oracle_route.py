"""Pins of the oracle's S5 (top-k repack, padding, EPLB) and S6 (dispatch).

Invariants that follow from _store_topk / _eplb_kernel_args /
prepare_megamoe_inputs (vllm.model_executor.layers.fused_moe.prepare_megamoe)
and from the batched layout of BatchedHummingGroupedExperts
(vllm.model_executor.layers.fused_moe.experts.fused_humming_moe).
"""
import numpy as np
import pytest
import torch

from moe_expert_layer_prepare_gb300 import synthetic as syn


def _stage(orc, T=48, K=256, E=16, k=4, pad_frac=0.1, eplb=None, seed=5, **kw):
    hid = syn.make_hidden(T, K, seed)
    ids, w, pad = syn.make_routing(T, E, k, seed + 1, padding_frac=pad_frac)
    bits = hid.view(torch.int16).numpy().view(np.uint16)
    st = orc.prepare_inputs(bits, ids.numpy(), w.numpy(), is_padding=pad.numpy(),
                            **(eplb or {}), **kw)
    return ids.numpy(), w.numpy(), pad.numpy(), st


def test_repack_identity_and_padding(orc):
    ids, w, pad, st = _stage(orc)
    assert pad.any() and not pad.all()
    real = pad == 0
    assert st["ids"].dtype == np.int64 and st["weights"].dtype == np.float32
    assert np.array_equal(st["ids"][real], ids[real].astype(np.int64))
    assert np.array_equal(st["weights"][real], w[real])
    assert np.all(st["ids"][~real] == -1)
    assert np.all(st["weights"][~real] == 0.0)


def test_repack_int64_ids_input(orc):
    ids, w, pad, st = _stage(orc)
    hid = syn.make_hidden(48, 256, 5)
    bits = hid.view(torch.int16).numpy().view(np.uint16)
    st64 = orc.prepare_inputs(bits, ids.astype(np.int64), w, is_padding=pad)
    assert np.array_equal(st64["ids"], st["ids"])


def test_eplb_identity_map(orc):
    E = 16
    l2p = np.arange(E, dtype=np.int32)[:, None]
    rc = np.ones(E, np.int32)
    ids, w, pad, st = _stage(orc, eplb=dict(l2p=l2p, replica_count=rc, num_physical=E,
                                            record_enabled=True))
    real = pad == 0
    assert np.array_equal(st["ids"][real], ids[real])
    # every routed (non-padding) pair is counted once
    assert st["load"].sum() == real.sum() * ids.shape[1]
    assert np.array_equal(st["load"], np.bincount(ids[real].ravel(), minlength=E))


def test_eplb_replicas(orc):
    E = 32
    l2p, rc, nphys = syn.make_eplb(E, 11, two=6, three=3)
    l2p, rc = l2p.numpy(), rc.numpy()
    assert nphys == E + 6 + 2 * 3
    T, k = 64, 4
    ids, w, pad, st = _stage(orc, T=T, E=E, k=k,
                             eplb=dict(l2p=l2p, replica_count=rc, num_physical=nphys,
                                       record_enabled=True, num_unpadded=40))
    for t in range(T):
        for j in range(k):
            if pad[t]:
                assert st["ids"][t, j] == -1
                continue
            lid = ids[t, j]
            phys = st["ids"][t, j]
            # the physical id lies in the logical expert's replica row,
            # at the position the token index selects
            assert phys in l2p[lid, :rc[lid]]
            assert phys == l2p[lid, t % rc[lid]]
    # load: recorded only for non-padding tokens below num_unpadded
    rec = np.zeros(nphys, np.int64)
    for t in range(40):
        if not pad[t]:
            for j in range(k):
                rec[st["ids"][t, j]] += 1
    assert np.array_equal(st["load"], rec)
    assert st["load"].sum() == (pad[:40] == 0).sum() * k


def test_eplb_record_disabled(orc):
    l2p, rc, nphys = syn.make_eplb(16, 3, two=2, three=1)
    _, _, _, st = _stage(orc, eplb=dict(l2p=l2p.numpy(), replica_count=rc.numpy(),
                                        num_physical=nphys, record_enabled=False))
    assert st["load"].sum() == 0


def test_dispatch_invariants(orc):
    E, M_max = 16, 48
    ids, w, pad, st = _stage(orc, E=E)
    d = orc.dispatch(st["ids"], st["x"], st["x_sf"], E, M_max)
    assert d["status"] == 0
    n = d["expert_num_tokens"]
    R = int((st["ids"] >= 0).sum())
    assert n.sum() == R
    slot = d["route_slot"]
    assert np.all((slot >= 0) == (st["ids"] >= 0))
    for e in range(E):
        sel = st["ids"] == e
        s = slot[sel]
        # unique slots 0..n_e-1, increasing in (token, k) order
        assert np.array_equal(s, np.arange(n[e]))
    T, k = st["ids"].shape
    for t in range(T):
        for j in range(k):
            e = st["ids"][t, j]
            if e < 0:
                continue
            r = e * M_max + slot[t, j]
            assert np.array_equal(d["x_b"][r], st["x"][t])
            assert np.array_equal(d["sf_b"][r], st["x_sf"][t])


def test_dispatch_capacity_overflow(orc):
    T, k, E, M_max = 10, 1, 2, 4
    ids = np.zeros((T, k), np.int64)  # every token to expert 0
    x = np.arange(T * 128, dtype=np.uint8).reshape(T, 128)
    sf = np.zeros((T, 1), np.int32)
    d = orc.dispatch(ids, x, sf, E, M_max)
    assert d["status"] == 1
    assert d["expert_num_tokens"][0] == M_max
    assert np.array_equal(d["route_slot"][:M_max, 0], np.arange(M_max))
    assert np.all(d["route_slot"][M_max:, 0] == -1)


@pytest.mark.parametrize("name", ["tiny", "deepseek_decode"])
def test_synthetic_routing_shape(name):
    c = syn.CONFIGS[name]
    ids, w, pad = syn.make_routing(c["T"], c["E"], c["top_k"], syn.seed_of(name, 1),
                                   zipf_s=c["zipf_s"], padding_frac=c["padding_frac"])
    ids = ids.numpy()
    # each token picks distinct experts; weights renormalised to 1
    for row in ids:
        assert len(set(row.tolist())) == c["top_k"]
    assert np.allclose(w.numpy().sum(axis=1), 1.0, atol=1e-6)
    if c["zipf_s"]:
        counts = np.bincount(ids.ravel(), minlength=c["E"])
        assert (counts == 0).sum() > c["E"] // 4, "Zipf routing leaves many experts empty"
        assert pad.numpy().sum() >= 1
