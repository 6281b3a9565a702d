"""GPU parity of moe_topk_reduce against the oracle (S8)."""
import numpy as np
import pytest
import torch

from moe_expert_layer_prepare_gb300 import binding as B
from tests._util import bf16_bits, bf16_vals, need_cuda

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def cuda():
    need_cuda()
    from moe_expert_layer_prepare_gb300 import build
    build.build()
    B.load()
    return torch.device("cuda")


# k = 9 and 40 cross the groups of 8 routes read together and, for 40, the 32
# routes resolved one per lane; contig passes topk_idx NULL (slot = row).
@pytest.mark.parametrize("T,k,E,M,K,contig", [(5, 1, 2, 4, 8, False),
                                              (77, 8, 16, 64, 7168, False),
                                              (300, 2, 8, 128, 4104, False),
                                              (61, 9, 4, 32, 520, False),
                                              (19, 40, 8, 16, 264, False),
                                              (45, 40, 8, 16, 1032, True),
                                              (90, 8, 4, 64, 2048, True)])
def test_reduce_vs_oracle(cuda, orc, T, k, E, M, K, contig):
    rng = np.random.default_rng(T + K)
    out_b = torch.from_numpy(rng.standard_normal((E, M, K), dtype=np.float32)).to(torch.bfloat16)
    if contig:
        # rows of the flat [E*M, K] buffer; -1 marks an unrouted slot
        slots = rng.integers(-1, E * M, size=(T, k)).astype(np.int32)
        ids = np.where(slots >= 0, 0, -1).astype(np.int64)  # for the bound below
        rows_all = np.maximum(slots, 0).astype(np.int64)
    else:
        ids = rng.integers(-1, E, size=(T, k)).astype(np.int64)
        slots = rng.integers(-1, M, size=(T, k)).astype(np.int32)
        rows_all = np.maximum(ids, 0) * M + np.maximum(slots, 0)
    w = rng.random((T, k)).astype(np.float32)
    dev = torch.device("cuda")
    out = torch.full((T, K), 3.0, dtype=torch.bfloat16, device=dev)
    B.moe_topk_reduce(out_b.to(dev), None if contig else torch.from_numpy(ids).to(dev),
                      torch.from_numpy(slots).to(dev), torch.from_numpy(w).to(dev), out)
    torch.cuda.synchronize()
    ref = orc.topk_reduce(bf16_bits(out_b).reshape(E * M, K), None if contig else ids, slots,
                          w, M)
    got = bf16_vals(bf16_bits(out)).astype(np.float64)
    rv = bf16_vals(ref).astype(np.float64)
    # fp32 sum vs the oracle's fp64 sum: one bf16 rounding of the result plus
    # the fp32 accumulation error, which near cancellation is bounded by the
    # magnitude of the terms rather than of the result
    ob = bf16_vals(bf16_bits(out_b).reshape(E * M, K)).astype(np.float64)
    mag = np.zeros((T, K))
    for j in range(k):
        ok = (ids[:, j] >= 0) & (slots[:, j] >= 0)
        rows = np.where(ok, rows_all[:, j], 0)
        mag += np.where(ok[:, None], np.abs(w[:, j:j + 1]) * np.abs(ob[rows]), 0.0)
    bound = np.abs(rv) * 2.0 ** -7 + mag * k * 2.0 ** -23
    assert np.all(np.abs(got - rv) <= bound)
    none = np.all((ids < 0) | (slots < 0), axis=1)
    assert np.all(got[none] == 0)
    if k == 1:
        wt = np.where((ids[:, 0] >= 0) & (slots[:, 0] >= 0), w[:, 0], 0)
        assert np.all(wt >= 0)


def test_reduce_gather_exact(cuda):
    E, M, K, T = 4, 16, 512, 40
    rng = np.random.default_rng(1)
    out_b = torch.from_numpy(rng.standard_normal((E, M, K), dtype=np.float32)).to(torch.bfloat16)
    ids = rng.integers(0, E, size=(T, 1)).astype(np.int64)
    slots = rng.integers(0, M, size=(T, 1)).astype(np.int32)
    dev = torch.device("cuda")
    out = torch.empty((T, K), dtype=torch.bfloat16, device=dev)
    B.moe_topk_reduce(out_b.to(dev), torch.from_numpy(ids).to(dev),
                      torch.from_numpy(slots).to(dev),
                      torch.ones((T, 1), dtype=torch.float32, device=dev), out)
    torch.cuda.synchronize()
    exp = out_b[torch.from_numpy(ids[:, 0]), torch.from_numpy(slots[:, 0].astype(np.int64))]
    assert torch.equal(out.cpu(), exp)


@pytest.mark.parametrize("contig", [False, True])
def test_reduce_token_bound(cuda, orc, contig):
    """num_valid_tokens (a device scalar): rows below it match the oracle's
    bounded S8, rows at or past it keep their previous contents."""
    T, k, E, M, K = 77, 8, 16, 64, 7168
    rng = np.random.default_rng(91 + contig)
    out_b = torch.from_numpy(rng.standard_normal((E, M, K), dtype=np.float32)).to(torch.bfloat16)
    ids = rng.integers(0, E, size=(T, k)).astype(np.int64)
    slots = rng.integers(-1, M, size=(T, k)).astype(np.int32)
    if contig:
        slots = np.where(slots >= 0, ids * M + slots, -1).astype(np.int32)
    w = rng.random((T, k)).astype(np.float32)
    dev = torch.device("cuda")
    args = (out_b.to(dev), None if contig else torch.from_numpy(ids).to(dev),
            torch.from_numpy(slots).to(dev), torch.from_numpy(w).to(dev))
    ob = bf16_bits(out_b).reshape(E * M, K)
    nv = torch.zeros(1, dtype=torch.int32, device=dev)
    for bound in (0, 1, 13, T, 200, -5):
        nv.fill_(bound)
        out = torch.full((T, K), -1, dtype=torch.int16, device=dev).view(torch.bfloat16)
        B.moe_topk_reduce(*args, out, num_valid_tokens=nv)
        torch.cuda.synchronize()
        ref = orc.topk_reduce(ob, None if contig else ids, slots, w, M,
                              num_valid=max(bound, 0), fill=0xFFFF)
        got = bf16_bits(out)
        n = min(max(bound, 0), T)
        assert np.all(got[n:] == 0xFFFF), f"bound {bound}: rows past it were written"
        rv = bf16_vals(ref[:n]).astype(np.float64)
        gv = bf16_vals(got[:n]).astype(np.float64)
        assert np.all(np.abs(gv - rv) <= np.abs(rv) * 2.0 ** -7 + 1e-3), f"bound {bound}"


def test_reduce_token_bound_in_a_graph(cuda, orc):
    """One reduce captured in a CUDA graph for the largest batch serves a
    smaller one by updating the device scalar before each replay."""
    T, k, E, M, K = 64, 4, 8, 32, 1024
    rng = np.random.default_rng(5)
    dev = torch.device("cuda")
    out_b = torch.from_numpy(rng.standard_normal((E, M, K), dtype=np.float32)).to(
        torch.bfloat16).to(dev)
    ids = torch.from_numpy(rng.integers(0, E, size=(T, k)).astype(np.int64)).to(dev)
    slots = torch.from_numpy(rng.integers(0, M, size=(T, k)).astype(np.int32)).to(dev)
    w = torch.from_numpy(rng.random((T, k)).astype(np.float32)).to(dev)
    out = torch.zeros((T, K), dtype=torch.bfloat16, device=dev)
    nv = torch.full((1,), T, dtype=torch.int32, device=dev)
    B.moe_topk_reduce(out_b, ids, slots, w, out, num_valid_tokens=nv)  # warm-up
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        B.moe_topk_reduce(out_b, ids, slots, w, out, num_valid_tokens=nv)
    full = orc.topk_reduce(bf16_bits(out_b).reshape(E * M, K), ids.cpu().numpy(),
                           slots.cpu().numpy(), w.cpu().numpy(), M)
    for bound in (T, 10, 0, 33):
        out.view(torch.int16).fill_(-1)
        nv.fill_(bound)
        g.replay()
        torch.cuda.synchronize()
        got = bf16_bits(out)
        assert np.all(got[bound:] == 0xFFFF)
        gv = bf16_vals(got[:bound]).astype(np.float64)
        rv = bf16_vals(full[:bound]).astype(np.float64)
        assert np.all(np.abs(gv - rv) <= np.abs(rv) * 2.0 ** -7 + 1e-3)
