"""GPU parity of the contiguous layout (expert_offsets) against the oracle.

Staging writes each expert's routes into consecutive rows; both GEMMs and the
reduce address rows by expert_offsets.  Checks: offsets, counts, rows and the
dispatched bytes bit-exact; h (gate_up_output) and the outputs within the FP
tolerance; the requant of the GPU's own h by the oracle's S2-S3; rows past
the last route untouched.
"""
import numpy as np
import pytest
import torch

from moe_expert_layer_prepare_gb300 import binding as B
from moe_expert_layer_prepare_gb300 import synthetic as syn
from tests._util import (assert_codes_close, assert_fp_close, bf16_bits, bf16_vals,
                         need_cuda, oracle_sampled_forward, unpack_exponents)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def cuda():
    need_cuda()
    from moe_expert_layer_prepare_gb300 import build
    build.build()
    B.load()
    return torch.device("cuda")


def _workload(T, K, N, E, k, seed, zipf=None, pad=0.03):
    wl = dict(cfg=dict(T=T, K=K, N=N, E=E, top_k=k))
    wl["hidden"] = syn.make_hidden(T, K, seed)
    wl["topk_ids"], wl["topk_weights"], wl["is_padding"] = syn.make_routing(
        T, E, k, seed + 1, zipf_s=zipf, padding_frac=pad)
    wl["w13"], wl["w13_s"] = syn.make_block_fp8_weights(E, 2 * N, K, seed + 2)
    wl["w2"], wl["w2_s"] = syn.make_block_fp8_weights(E, K, N, seed + 3)
    return wl


@pytest.mark.parametrize("T,K,N,E,k,zipf", [
    (32, 256, 512, 4, 2, None),      # tiny
    (300, 512, 256, 8, 4, 1.1),      # hot experts span several 128-row tiles
    (16, 2048, 1024, 2, 1, None),    # few tiles: split-K w2
    (128, 7168, 2048, 256, 8, 1.1),  # DeepSeek-V3-shaped decode routing
])
def test_contiguous_full_path(cuda, orc, T, K, N, E, k, zipf):
    wl = _workload(T, K, N, E, k, 1000 + T + E, zipf)
    dev = cuda
    to = lambda t: t.to(dev)  # noqa: E731
    layer = B.MoeLayer(T, K, N, E, k, None, to(wl["w13"]), to(wl["w13_s"]), to(wl["w2"]),
                       to(wl["w2_s"]), device=dev, contiguous=True)
    rows_cap = E * layer.M_max
    layer.out_b.view(torch.int16).fill_(-1)
    h = torch.zeros((rows_cap, 2 * N), dtype=torch.bfloat16, device=dev)
    layer.prepare(to(wl["hidden"]), to(wl["topk_ids"]), to(wl["topk_weights"]),
                  to(wl["is_padding"]))
    layer.experts(gate_up_dump=h)
    layer.reduce()
    torch.cuda.synchronize()
    assert int(layer.status.item()) == 0

    st = orc.prepare_inputs(bf16_bits(wl["hidden"]), wl["topk_ids"].numpy(),
                            wl["topk_weights"].numpy(), is_padding=wl["is_padding"].numpy())
    c = orc.dispatch_contiguous(st["ids"], st["x"], st["x_sf"], E)
    assert c["status"] == 0
    assert np.array_equal(layer.expert_offsets.cpu().numpy(), c["expert_offsets"])
    assert np.array_equal(layer.expert_num_tokens.cpu().numpy(), c["expert_num_tokens"])
    assert np.array_equal(layer.route_slot.cpu().numpy(), c["route_row"])
    R = int(c["expert_offsets"][-1])
    rows = np.arange(R)
    assert np.array_equal(layer.x_b.cpu().numpy()[:R], c["x_c"][:R])
    assert np.array_equal(layer.sf_b.cpu().numpy()[:R], c["sf_c"][:R])
    args = [wl[n].numpy() for n in ("w13", "w13_s", "w2", "w2_s")]
    h_ref, _, _ = orc.w13_rows(rows, 1, K, N, c["x_c"], c["sf_c"], args[0], args[1],
                               want_h=True, row_expert=c["row_expert"])
    hg = bf16_vals(bf16_bits(h))[:R]
    assert_fp_close(hg, bf16_vals(h_ref)[:R], "gate_up_output (contiguous)")
    # requant of the GPU's own h
    q_gpu, sf_gpu = layer.inter()
    yq_ref, ysf_ref = orc.silu_requant_rows(rows, N, bf16_bits(h))
    Gn = N // 128
    eg = unpack_exponents(sf_gpu.cpu().numpy()[:R], Gn)
    er = unpack_exponents(ysf_ref[:R], Gn)
    assert np.mean(eg == er) > 0.999
    assert np.all(np.abs(eg.astype(int) - er.astype(int)) <= 1)
    assert_codes_close(q_gpu.cpu().numpy()[:R], yq_ref[:R], orc.e4m3_decode_table(),
                       "requant codes (contiguous)")
    # w2 from the GPU's own requantised rows (isolates the GEMM), then the reduce
    ob_ref = orc.w2_rows(rows, 1, K, N, q_gpu.cpu().numpy(), sf_gpu.cpu().numpy(), args[2],
                         args[3], row_expert=c["row_expert"])
    ob = bf16_bits(layer.out_b).reshape(rows_cap, K)
    assert_fp_close(bf16_vals(ob)[:R], bf16_vals(ob_ref)[:R], "down_output (contiguous)")
    assert np.all(ob[R:] == 0xFFFF), "rows past the last route were written"
    out_ref = orc.topk_reduce(ob_ref, None, c["route_row"], st["weights"], 1)
    assert_fp_close(bf16_vals(bf16_bits(layer.out)), bf16_vals(out_ref), "output (contiguous)")


def test_contiguous_prefill_full_size(cuda, orc):
    """DeepSeek-V3-shaped prefill (T=8192, E=256, top-8) in the contiguous
    layout: offsets bit-exact, sampled tokens' outputs against the oracle."""
    wl = syn.make_workload("deepseek_prefill", weights_device=cuda)
    c = wl["cfg"]
    T, K, N, E, k = c["T"], c["K"], c["N"], c["E"], c["top_k"]
    layer = B.MoeLayer(T, K, N, E, k, None, wl["w13"], wl["w13_s"], wl["w2"], wl["w2_s"],
                       device=cuda, contiguous=True)
    out = layer.forward(wl["hidden"].to(cuda), wl["topk_ids"].to(cuda),
                        wl["topk_weights"].to(cuda), wl["is_padding"].to(cuda))
    torch.cuda.synchronize()
    assert int(layer.status.item()) == 0
    ids = wl["topk_ids"].numpy().astype(np.int64)
    counts = np.bincount(ids.ravel(), minlength=E)
    assert np.array_equal(layer.expert_offsets.cpu().numpy(),
                          np.concatenate([[0], np.cumsum(counts)]).astype(np.int32))
    rng = np.random.default_rng(3)
    tokens = np.sort(rng.choice(T, 24, replace=False))
    ref = oracle_sampled_forward(orc, wl, tokens)
    got = bf16_vals(bf16_bits(out))[tokens]
    assert_fp_close(got, bf16_vals(ref["out"]), "prefill output (contiguous, sampled)")
