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
                         coverage_tokens, need_cuda, oracle_sampled_forward, unpack_exponents)

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
    layout: offsets and rows bit-exact; for a deterministic token sample whose
    routes reach every m-tile index, the tile boundaries 127/128/255/256 and
    the ragged last tile of the most-loaded expert: h, the requantised w2
    input, the expert outputs and the token outputs against the oracle."""
    wl = syn.make_workload("deepseek_prefill", weights_device=cuda)
    c = wl["cfg"]
    T, K, N, E, k = c["T"], c["K"], c["N"], c["E"], c["top_k"]
    layer = B.MoeLayer(T, K, N, E, k, None, wl["w13"], wl["w13_s"], wl["w2"], wl["w2_s"],
                       device=cuda, contiguous=True)
    h = torch.zeros((E * layer.M_max, 2 * N), dtype=torch.bfloat16, device=cuda)
    layer.prepare(wl["hidden"].to(cuda), wl["topk_ids"].to(cuda), wl["topk_weights"].to(cuda),
                  wl["is_padding"].to(cuda))
    layer.experts(gate_up_dump=h)
    layer.reduce()
    torch.cuda.synchronize()
    assert int(layer.status.item()) == 0
    ids = wl["topk_ids"].numpy().astype(np.int64)
    counts = np.bincount(ids.ravel(), minlength=E)
    offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    assert np.array_equal(layer.expert_offsets.cpu().numpy(), offs)
    st = orc.prepare_inputs(np.zeros((T, 128), np.uint16), wl["topk_ids"].numpy(),
                            wl["topk_weights"].numpy(), is_padding=wl["is_padding"].numpy())
    d = orc.dispatch(st["ids"], np.zeros((T, 128), np.uint8), np.zeros((T, 1), np.int32), E,
                     c["M_max"], copy_rows=False)
    rows_gpu = layer.route_slot.cpu().numpy()
    assert np.array_equal(rows_gpu, np.where(d["route_slot"] >= 0,
                                             offs[np.maximum(st["ids"], 0)] + d["route_slot"], -1))
    tokens = coverage_tokens(st["ids"], d["route_slot"], 64, seed=7)
    ref = oracle_sampled_forward(orc, wl, tokens, want_h=True)
    g_rows = [int(offs[e]) + s for (i, j, e, s) in ref["routes"]]
    slots = np.array([s for (i, j, e, s) in ref["routes"]])
    assert {127, 128, 255, 256} <= set(slots.tolist())
    assert len(np.unique(slots // 128)) == (int(counts.max()) + 127) // 128
    idx = torch.as_tensor(g_rows, dtype=torch.int64, device=cuda)
    cr = np.array([ref["crow_of"][(i, j)] for (i, j, e, s) in ref["routes"]])
    h_bits = bf16_bits(h[idx])
    assert_fp_close(bf16_vals(h_bits), bf16_vals(ref["h"][cr]), "prefill h rows (contiguous)")
    ob = bf16_vals(bf16_bits(layer.out_b.view(-1, K)[idx]))
    assert_fp_close(ob, bf16_vals(ref["out_b"][cr]), "prefill out_b rows (contiguous)")
    q_gpu, sf_gpu = layer.inter()
    yq_ref, ysf_ref = orc.silu_requant_rows(np.arange(len(g_rows)), N, h_bits)
    eg = unpack_exponents(sf_gpu[idx].cpu().numpy(), N // 128)
    er = unpack_exponents(ysf_ref, N // 128)
    assert np.mean(eg == er) > 0.999
    assert np.all(np.abs(eg.astype(int) - er.astype(int)) <= 1)
    assert_codes_close(q_gpu[idx].cpu().numpy(), yq_ref, orc.e4m3_decode_table(),
                       "prefill requant codes (contiguous)")
    got = bf16_vals(bf16_bits(layer.out))[tokens]
    assert_fp_close(got, bf16_vals(ref["out"]), "prefill output (contiguous, sampled)")
