"""Failure detection of the GEMM's bounded pipeline waits, without a fault.

A test-only build of the library (build.build_test_variant("timeout"))
shortens the wait limit to 5 ms and has CTA 0 withhold one stage of its
first w13 work unit: it issues neither the expected-bytes arrival nor a copy
for that stage, so its full barrier is never completed -- a flag that nothing
sets -- and no copy is left in flight.  The MMA warp's bounded wait on it
runs out; the CTA then sets MOE_DEV_TIMEOUT in the status word, drains the
copies and MMAs it did issue, frees its tensor memory and returns.  The test
checks the status bit, that the call returned promptly, and that the context
is still usable: the regular library then runs the same problem in the same
process and matches the oracle.
"""
import ctypes
import time

import numpy as np
import pytest
import torch

from moe_expert_layer_prepare_gb300 import binding as B
from moe_expert_layer_prepare_gb300 import synthetic as syn
from tests._util import assert_fp_close, bf16_bits, bf16_vals, need_cuda

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def libs():
    need_cuda()
    from moe_expert_layer_prepare_gb300 import build
    build.build()
    regular = B.load()
    test_lib = B.configure(ctypes.CDLL(build.build_test_variant("timeout")))
    return regular, test_lib


def _w13(lib, layer, status):
    """The w13 stage of `layer` through the given copy of the library."""
    saved = B._lib
    B._lib = lib
    try:
        B.moe_batched_experts(layer.out_b, layer.x_b, layer.sf_b, layer.w13, layer.w13_s,
                              layer.w2, layer.w2_s, layer.expert_num_tokens, layer.ws13,
                              layer.ws2, valid_shape_m=layer.valid_shape_m,
                              stages=B.MOE_STAGE_W13, device_status=status)
    finally:
        B._lib = saved


def test_wait_timeout_sets_status_and_context_survives(libs, orc):
    regular, test_lib = libs
    dev = torch.device("cuda")
    # eight K slabs, so that the withheld third stage lies inside CTA 0's first unit
    T, K, N, E, k, M = 64, 1024, 256, 4, 2, 64
    hid = syn.make_hidden(T, K, 71)
    ids, w, pad = syn.make_routing(T, E, k, 72)
    w13, w13_s = syn.make_block_fp8_weights(E, 2 * N, K, 73)
    w2, w2_s = syn.make_block_fp8_weights(E, K, N, 74)
    layer = B.MoeLayer(T, K, N, E, k, M, w13.to(dev), w13_s.to(dev), w2.to(dev), w2_s.to(dev),
                       device=dev)
    layer.prepare(hid.to(dev), ids.to(dev), w.to(dev), pad.to(dev))
    torch.cuda.synchronize()
    assert int(layer.status.item()) == 0

    status = torch.zeros(1, dtype=torch.int32, device=dev)
    t0 = time.perf_counter()
    _w13(test_lib, layer, status)
    torch.cuda.synchronize()          # the launch returns: no hang, no fault
    elapsed = time.perf_counter() - t0
    assert int(status.item()) & B.MOE_DEV_TIMEOUT, "the withheld stage's wait did not expire"
    assert elapsed < 5.0

    # the context is intact: the regular library runs the whole path again and
    # matches the oracle on every token
    out = layer.forward(hid.to(dev), ids.to(dev), w.to(dev), pad.to(dev))
    torch.cuda.synchronize()
    assert int(layer.status.item()) == 0
    ref = orc.forward(bf16_bits(hid), ids.numpy(), w.numpy(),
                      *(t.numpy() for t in (w13, w13_s, w2, w2_s)), E, M, N,
                      is_padding=pad.numpy())
    assert_fp_close(bf16_vals(bf16_bits(out)), bf16_vals(ref["out"]), "output after a timeout")
    assert np.array_equal(layer.route_slot.cpu().numpy(), ref["dispatch"]["route_slot"])
