"""GPU parity of the fp32 activation-scale path (the a1q_scale [M, K/128]
fp32 contract) against the oracle: staging and dispatch of fp32 scales
bit-exact, the w13 GEMM dequantising with them within the FP tolerance,
the requantised w2 input and the final output as on the UE8M0 path."""
import numpy as np
import pytest
import torch

from moe_expert_layer_prepare_gb300 import binding as B
from moe_expert_layer_prepare_gb300 import synthetic as syn
from tests._util import (assert_codes_close, assert_fp_close, bf16_bits, bf16_vals,
                         need_cuda, unpack_exponents)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def cuda():
    need_cuda()
    from moe_expert_layer_prepare_gb300 import build
    build.build()
    B.load()
    return torch.device("cuda")


@pytest.mark.parametrize("T,K,N,E,k,M_max,contig", [
    (32, 256, 512, 4, 2, 32, False),
    (200, 896, 384, 8, 4, 160, False),   # G = 7 (no packing), several tiles, padding
    (128, 7168, 2048, 64, 8, 64, True),  # DeepSeek-V3 hidden size, contiguous rows
])
def test_fp32_scales_full_path(cuda, orc, T, K, N, E, k, M_max, contig):
    seed = 500 + T
    hid = syn.make_hidden(T, K, seed, outlier_frac=0.01, zero_group_frac=0.02)
    ids, w, pad = syn.make_routing(T, E, k, seed + 1, padding_frac=0.03)
    w13, w13_s = syn.make_block_fp8_weights(E, 2 * N, K, seed + 2)
    w2, w2_s = syn.make_block_fp8_weights(E, K, N, seed + 3)
    dev = cuda
    layer = B.MoeLayer(T, K, N, E, k, M_max, w13.to(dev), w13_s.to(dev), w2.to(dev),
                       w2_s.to(dev), device=dev, contiguous=contig, fp32_scales=True)
    M = layer.M_max
    h = torch.zeros((E * M, 2 * N), dtype=torch.bfloat16, device=dev)
    layer.out_b.view(torch.int16).fill_(-1)
    layer.prepare(hid.to(dev), ids.to(dev), w.to(dev), pad.to(dev))
    layer.experts(gate_up_dump=h)
    layer.reduce()
    torch.cuda.synchronize()
    assert int(layer.status.item()) == 0

    st = orc.prepare_inputs(bf16_bits(hid), ids.numpy(), w.numpy(), is_padding=pad.numpy(),
                            sf_mode=2)
    assert np.array_equal(layer.x_sf.cpu().numpy().view(np.int32), st["x_sf"].view(np.int32))
    if contig:
        d = orc.dispatch_contiguous(st["ids"], st["x"], st["x_sf"], E)
        rows, row_expert, slots = np.arange(int(d["expert_offsets"][-1])), d["row_expert"], \
            d["route_row"]
        xb_ref, sfb_ref = d["x_c"], d["sf_c"]
    else:
        d = orc.dispatch(st["ids"], st["x"], st["x_sf"], E, M)
        assert d["status"] == 0
        rows, row_expert, slots = orc.valid_rows(d["expert_num_tokens"], M), None, d["route_slot"]
        xb_ref, sfb_ref = d["x_b"], d["sf_b"]
    assert np.array_equal(layer.route_slot.cpu().numpy(), slots)
    assert np.array_equal(layer.x_b.cpu().numpy()[rows], xb_ref[rows])
    assert np.array_equal(layer.sf_b.cpu().numpy()[rows].view(np.int32),
                          sfb_ref[rows].view(np.int32))
    mm = 1 if contig else M
    h_ref, _, _ = orc.w13_rows(rows, mm, K, N, xb_ref, sfb_ref, w13.numpy(), w13_s.numpy(),
                               want_h=True, row_expert=row_expert)
    assert_fp_close(bf16_vals(bf16_bits(h))[rows], bf16_vals(h_ref)[rows], "h (fp32 scales)")
    q_gpu, sf_gpu = layer.inter()
    yq_ref, ysf_ref = orc.silu_requant_rows(rows, N, bf16_bits(h))
    Gn = N // 128
    eg = unpack_exponents(sf_gpu.cpu().numpy()[rows], Gn)
    er = unpack_exponents(ysf_ref[rows], Gn)
    assert np.all(np.abs(eg.astype(int) - er.astype(int)) <= 1) and np.mean(eg == er) > 0.999
    assert_codes_close(q_gpu.cpu().numpy()[rows], yq_ref[rows], orc.e4m3_decode_table(),
                       "requant codes (fp32 scales)")
    ob_ref = orc.w2_rows(rows, mm, K, N, q_gpu.cpu().numpy(), sf_gpu.cpu().numpy(), w2.numpy(),
                         w2_s.numpy(), row_expert=row_expert)
    ob = bf16_bits(layer.out_b).reshape(E * M, K)
    assert_fp_close(bf16_vals(ob)[rows], bf16_vals(ob_ref)[rows], "down_output (fp32 scales)")
    out_ref = orc.topk_reduce(ob_ref, None if contig else st["ids"], slots, st["weights"], mm)
    assert_fp_close(bf16_vals(bf16_bits(layer.out)), bf16_vals(out_ref), "output (fp32 scales)")
