"""moe_prepare_inputs_noalloc gives the same results as moe_prepare_inputs.

The allocation-free entry point exists for callers that cannot allocate
device memory themselves: a plugin that is handed only its input and output
buffers, code running under a CUDA graph capture whose framework forbids
allocation, or a service held to a fixed device-memory budget.  Instead of a
caller-provided workspace, its dispatch scratch is a fixed array inside the
library.

The new entry point is called through the C ABI twice in a row, on two
different batches (so the second call finds the first call's leftovers in the
shared array), and each result is compared with the regular entry point's on
the same batch.  Everything the staging produces is integer or byte data
(fp8 codes, packed exponents, ids, slots, counts, fp32 copies of the weights),
so the comparison is exact, as in the other staging tests.
"""
import ctypes

import pytest
import torch

from moe_expert_layer_prepare_gb300 import binding as B
from moe_expert_layer_prepare_gb300 import synthetic as syn

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from moe_expert_layer_prepare_gb300 import build
    build.build()
    B.load()
    return torch.device("cuda")


def _stage(entry, hid, ids, w, pad, E, M_max):
    dev = torch.device("cuda")
    T, K = hid.shape
    k = ids.shape[1]
    W = (K // 128 + 3) // 4
    out = dict(
        x=torch.full((T, K), 0x11, dtype=torch.uint8, device=dev),
        x_sf=torch.full((T, W), -3, dtype=torch.int32, device=dev),
        ids=torch.full((T, k), 99, dtype=torch.int64, device=dev),
        w=torch.full((T, k), 5.0, dtype=torch.float32, device=dev),
        x_b=torch.full((E * M_max, K), 0x22, dtype=torch.uint8, device=dev),
        sf_b=torch.full((E * M_max, W), -5, dtype=torch.int32, device=dev),
        ent=torch.full((E,), -1, dtype=torch.int32, device=dev),
        slot=torch.full((T, k), -7, dtype=torch.int32, device=dev),
        status=torch.zeros(1, dtype=torch.int32, device=dev),
    )
    disp = dict(num_experts=E, max_tokens_per_expert=M_max, x_b=out["x_b"], sf_b=out["sf_b"],
                expert_num_tokens=out["ent"], route_slot=out["slot"])
    if entry == "regular":
        disp["workspace"] = torch.empty(B.prepare_workspace_size(T, k, E), dtype=torch.uint8,
                                        device=dev)
        fn = B.moe_prepare_inputs
    else:
        fn = B.moe_prepare_inputs_noalloc
    fn(hid.to(dev), ids.to(dev), w.to(dev), out["x"], out["x_sf"], out["ids"], out["w"],
       is_padding=pad.to(dev), dispatch=disp, device_status=out["status"])
    torch.cuda.synchronize()
    return {n: t.cpu() for n, t in out.items()}


BATCHES = [
    # T, K, k, E, M_max, Zipf, padding: a DeepSeek-shaped decode batch, then a
    # smaller batch over fewer experts spanning three route blocks
    (128, 7168, 8, 256, 128, 1.1, 0.02, 11),
    (300, 384, 8, 64, 300, None, 0.1, 12),
]


def test_noalloc_matches_regular_twice(cuda):
    for (T, K, k, E, M_max, zipf, pad_frac, seed) in BATCHES:
        hid = syn.make_hidden(T, K, seed)
        ids, w, pad = syn.make_routing(T, E, k, seed + 1, zipf_s=zipf, padding_frac=pad_frac)
        got = _stage("noalloc", hid, ids, w, pad, E, M_max)
        ref = _stage("regular", hid, ids, w, pad, E, M_max)
        assert int(got["status"].item()) == 0 and int(ref["status"].item()) == 0
        for name in ref:
            assert torch.equal(got[name], ref[name]), f"{name} differs (T={T}, E={E})"
        assert int(ref["ent"].sum().item()) == int((ref["slot"] >= 0).sum().item())


def test_noalloc_rejects_oversize(cuda):
    """A problem whose dispatch scratch exceeds the fixed array is refused on
    the host before anything is enqueued (no pointer is dereferenced)."""
    lib = B.load()
    a = B.PrepareArgs()
    fake = 0x10000
    a.num_tokens, a.hidden_size, a.top_k = 1 << 22, 256, 8
    a.hidden, a.hidden_stride0 = fake, 256
    a.topk_ids, a.topk_ids_stride0, a.topk_ids_stride1 = fake, 8, 1
    a.topk_weights, a.topk_weights_stride0, a.topk_weights_stride1 = fake, 8, 1
    a.x, a.x_stride0 = fake, 256
    a.x_sf, a.sf_mode, a.x_sf_stride0, a.x_sf_stride1 = fake, B.MOE_SF_UE8M0_PACKED, 1, 1
    a.topk_idx_out, a.topk_idx_out_stride0, a.topk_idx_out_stride1 = fake, 8, 1
    a.topk_weights_out, a.topk_weights_out_stride0, a.topk_weights_out_stride1 = fake, 8, 1
    a.num_experts, a.max_tokens_per_expert = 256, 1 << 16
    a.x_b, a.sf_b, a.expert_num_tokens, a.route_slot = fake, fake, fake, fake
    st = lib.moe_prepare_inputs_noalloc(ctypes.byref(a), None)
    assert st == 5
    assert "fixed scratch" in lib.moe_last_error().decode()


# The largest top-8 problem over 256 experts whose dispatch scratch fits the
# fixed array: 104,832 tokens need 4,193,536 of its 4,194,304 bytes; one token
# (eight routes) more needs 4,194,816.
NEAR_LIMIT_T = 104832


def test_noalloc_near_the_limit(cuda):
    """A problem that fills the fixed array to its last block: the top of the
    array is used and the result still equals the regular entry point's."""
    k, E, K = 8, 256, 128
    assert B.prepare_workspace_size(NEAR_LIMIT_T, k, E) <= 4 << 20
    assert B.prepare_workspace_size(NEAR_LIMIT_T + 1, k, E) > 4 << 20
    hid = syn.make_hidden(NEAR_LIMIT_T, K, 21)
    ids, w, pad = syn.make_routing(NEAR_LIMIT_T, E, k, 22, padding_frac=0.01)
    M_max = 4096  # every expert's count (about 3,300 routes each) fits
    got = _stage("noalloc", hid, ids, w, pad, E, M_max)
    ref = _stage("regular", hid, ids, w, pad, E, M_max)
    assert int(got["status"].item()) == 0 and int(ref["status"].item()) == 0
    for name in ref:
        assert torch.equal(got[name], ref[name]), f"{name} differs at the scratch limit"
    assert int(ref["ent"].max().item()) < M_max


def test_noalloc_refuses_one_token_past_the_limit(cuda):
    """Eight routes past the boundary are refused on the host."""
    lib = B.load()
    a = B.PrepareArgs()
    fake = 0x10000
    T, k, K = NEAR_LIMIT_T + 1, 8, 128
    a.num_tokens, a.hidden_size, a.top_k = T, K, k
    a.hidden, a.hidden_stride0 = fake, K
    a.topk_ids, a.topk_ids_stride0, a.topk_ids_stride1 = fake, k, 1
    a.topk_weights, a.topk_weights_stride0, a.topk_weights_stride1 = fake, k, 1
    a.x, a.x_stride0 = fake, K
    a.x_sf, a.sf_mode, a.x_sf_stride0, a.x_sf_stride1 = fake, B.MOE_SF_UE8M0_PACKED, 1, 1
    a.topk_idx_out, a.topk_idx_out_stride0, a.topk_idx_out_stride1 = fake, k, 1
    a.topk_weights_out, a.topk_weights_out_stride0, a.topk_weights_out_stride1 = fake, k, 1
    a.num_experts, a.max_tokens_per_expert = 256, 4096
    a.x_b, a.sf_b, a.expert_num_tokens, a.route_slot = fake, fake, fake, fake
    assert lib.moe_prepare_inputs_noalloc(ctypes.byref(a), None) == 5
    assert "fixed scratch" in lib.moe_last_error().decode()
