"""The C-ABI library loads, exports every declared entry point, and rejects bad
arguments on the host before anything is enqueued (no GPU needed: every case
below returns before the first CUDA call)."""
import ctypes
import os
import re

import pytest

from moe_expert_layer_prepare_gb300 import binding as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from moe_expert_layer_prepare_gb300 import build
    build.build()
    return B.load()


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "moe_prep.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^[A-Za-z_][\w \*]*?\b(moe_\w+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_exports_every_declared_symbol(lib):
    names = _declared_functions()
    for must in ["moe_prepare_inputs", "moe_batched_experts", "moe_topk_reduce",
                 "moe_abi_version", "moe_last_error", "moe_prepare_workspace_size",
                 "moe_batched_experts_workspace_size", "moe_prepare_nvfp4_inputs"]:
        assert must in names
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/moe_prep.h but not exported"
    assert lib.moe_abi_version() == 3


FAKE = 0x10000  # never dereferenced: every call below fails its checks first


def _prep_args(**kw):
    a = B.PrepareArgs()
    a.num_tokens, a.hidden_size, a.top_k = 8, 256, 2
    a.hidden, a.hidden_stride0 = FAKE, 256
    a.topk_ids, a.topk_ids_stride0, a.topk_ids_stride1 = FAKE, 2, 1
    a.topk_weights, a.topk_weights_stride0, a.topk_weights_stride1 = FAKE, 2, 1
    a.x, a.x_stride0 = FAKE, 256
    a.x_sf, a.sf_mode, a.x_sf_stride0, a.x_sf_stride1 = FAKE, B.MOE_SF_UE8M0_PACKED, 1, 1
    a.topk_idx_out, a.topk_idx_out_stride0, a.topk_idx_out_stride1 = FAKE, 2, 1
    a.topk_weights_out, a.topk_weights_out_stride0, a.topk_weights_out_stride1 = FAKE, 2, 1
    for k, v in kw.items():
        setattr(a, k, v)
    return a


def _prep(lib, a):
    st = lib.moe_prepare_inputs(ctypes.byref(a), None)
    return st, lib.moe_last_error().decode()


def test_prepare_rejects(lib):
    st, msg = _prep(lib, _prep_args(hidden_size=100, hidden_stride0=100, x_stride0=100))
    assert st == 2 and "128" in msg
    st, _ = _prep(lib, _prep_args(x_sf=None))
    assert st == 1
    st, _ = _prep(lib, _prep_args(sf_mode=B.MOE_SF_NONE))
    assert st == 1  # x_sf given but no quantisation
    st, _ = _prep(lib, _prep_args(top_k=0))
    assert st == 2
    st, _ = _prep(lib, _prep_args(hidden=FAKE + 8))
    assert st == 4
    st, _ = _prep(lib, _prep_args(sf_mode=7))
    assert st == 1
    st, _ = _prep(lib, _prep_args(topk_ids_dtype=5))
    assert st == 1
    st, _ = _prep(lib, _prep_args(logical_to_physical=FAKE))
    assert st == 1  # EPLB without replica counts
    # dispatch: needs packed UE8M0 scales, enough workspace
    d = dict(x_b=FAKE, sf_b=FAKE, expert_num_tokens=FAKE, route_slot=FAKE, num_experts=4,
             max_tokens_per_expert=8, workspace=FAKE, workspace_bytes=16)
    st, msg = _prep(lib, _prep_args(**d))
    assert st == 5 and "workspace" in msg
    st, _ = _prep(lib, _prep_args(sf_mode=B.MOE_SF_NONE, x_sf=None, **d))
    assert st == 3  # dispatch needs quantised scales (UE8M0 or fp32)
    st, msg = _prep(lib, _prep_args(sf_mode=B.MOE_SF_FP32, **d))
    assert st == 5 and "workspace" in msg  # fp32 scales pass the mode check
    st, _ = _prep(lib, _prep_args(num_experts=2000, **{k: v for k, v in d.items()
                                                         if k != "num_experts"}))
    assert st == 2
    # shared-expert scale pages: both or neither, UE8M0 only, enough rows
    st, _ = _prep(lib, _prep_args(shared_x_sf=FAKE))
    assert st == 1
    st, _ = _prep(lib, _prep_args(shared_block_m=128))
    assert st == 1
    sh = dict(shared_x_sf=FAKE, shared_block_m=200, shared_x_sf_stride0=2,
              shared_x_sf_stride1=1)
    st, _ = _prep(lib, _prep_args(sf_mode=B.MOE_SF_FP32, shared_x_sf_rows=256, **sh))
    assert st == 3
    st, msg = _prep(lib, _prep_args(shared_x_sf_rows=255, **sh))
    assert st == 2 and "256" in msg  # ceil(T/200) pages of 256 rows
    st, _ = _prep(lib, _prep_args(shared_block_m=-4, shared_x_sf=FAKE))
    assert st == 1
    # T == 0 is a no-op
    st, _ = _prep(lib, _prep_args(num_tokens=0))
    assert st == 0


def _exp_args(**kw):
    a = B.ExpertsArgs()
    a.num_experts, a.max_tokens_per_expert, a.hidden_size, a.intermediate_size = 4, 32, 256, 512
    a.activation, a.stages = B.MOE_ACT_SILU, B.MOE_STAGE_ALL
    a.output = a.hidden = a.a_scale = a.w13 = a.w13_scale = a.w2 = a.w2_scale = FAKE
    a.expert_num_tokens = FAKE
    a.a_scale_mode = B.MOE_SF_UE8M0_PACKED
    a.workspace13, a.workspace13_bytes = FAKE, 1
    a.workspace2, a.workspace2_bytes = FAKE, 1
    for k, v in kw.items():
        setattr(a, k, v)
    return a


def test_experts_rejects(lib):
    run = lambda a: lib.moe_batched_experts(ctypes.byref(a), None)  # noqa: E731
    assert run(_exp_args(hidden_size=200)) == 2
    assert run(_exp_args(intermediate_size=100)) == 2
    assert run(_exp_args(activation=3)) == 3
    assert run(_exp_args(a_scale_mode=B.MOE_SF_NONE)) == 3
    assert run(_exp_args(a_scale_mode=B.MOE_SF_FP32)) == 5  # fp32 scales accepted
    assert run(_exp_args(stages=B.MOE_STAGE_W2)) == 1     # w2 alone needs inter_q/inter_sf
    assert run(_exp_args(w13=FAKE + 4)) == 4
    assert run(_exp_args()) == 5                          # workspace13 too small
    assert "workspace13" in lib.moe_last_error().decode()
    assert run(_exp_args(num_experts=0)) == 1


def test_reduce_rejects(lib):
    f = lib.moe_topk_reduce
    assert f(FAKE, 4, 8, 100, FAKE, FAKE, FAKE, 4, 2, None, FAKE, None) == 2
    assert f(None, 4, 8, 256, FAKE, FAKE, FAKE, 4, 2, None, FAKE, None) == 1
    assert f(FAKE + 2, 4, 8, 256, FAKE, FAKE, FAKE, 4, 2, None, FAKE, None) == 4
    assert f(FAKE, 4, 8, 256, FAKE, FAKE, FAKE, 0, 2, FAKE, FAKE, None) == 0


def test_workspace_sizes(lib):
    s = lib.moe_prepare_workspace_size(8192, 8, 256)
    assert s >= 256 + 64 * 256 * 4 + 65536 * 4
    s13 = lib.moe_batched_experts_workspace_size(256, 1024, 7168, 2048, 65536, 13)
    assert s13 >= 256 * 1024 * 2048 + 256 * 1024 * 4 * 4
    s2 = lib.moe_batched_experts_workspace_size(8, 64, 4096, 14336, 128, 2)
    assert s2 > 0


def test_nvfp4_rejects(lib):
    def args(**kw):
        a = B.Nvfp4Args()
        a.num_tokens, a.hidden_size, a.top_k = 8, 256, 2
        a.hidden, a.hidden_stride0 = FAKE, 256
        a.topk_ids, a.topk_ids_stride0, a.topk_ids_stride1 = FAKE, 2, 1
        a.topk_weights, a.topk_weights_stride0, a.topk_weights_stride1 = FAKE, 2, 1
        a.x, a.x_stride0, a.x_sf, a.x_sf_stride0, a.x_scales = FAKE, 128, FAKE, 4, FAKE
        a.topk_idx_out, a.topk_idx_out_stride0, a.topk_idx_out_stride1 = FAKE, 2, 1
        a.topk_weights_out, a.topk_weights_out_stride0, a.topk_weights_out_stride1 = FAKE, 2, 1
        for k, v in kw.items():
            setattr(a, k, v)
        return a
    run = lambda a: lib.moe_prepare_nvfp4_inputs(ctypes.byref(a), None)  # noqa: E731
    assert run(args(hidden_size=192, hidden_stride0=192, x_stride0=96, x_sf_stride0=3)) == 2
    assert run(args(x_scales=None)) == 1
    assert run(args(w2_global_scale=FAKE)) == 1            # without l2_alpha
    assert run(args(l2_alpha=FAKE, w2_global_scale=FAKE)) == 1  # no local experts
    assert run(args(hidden=FAKE + 8)) == 4
    assert run(args(x=FAKE + 2)) == 4
    assert run(args(x_sf_stride0=3)) == 2                  # K/64 = 4 words per row
    assert run(args(top_k=0)) == 2
    assert run(args(num_tokens=0)) == 0                    # nothing to do
    # the MXFP8 shared input: shared_x_sf and shared_block_m exactly for fp8
    fp8 = dict(shared_x=FAKE, shared_x_stride0=256, shared_x_dtype=B.MOE_SHARED_FP8)
    assert run(args(**fp8)) == 1                           # no shared_x_sf
    assert run(args(**fp8, shared_x_sf=FAKE, shared_x_sf_stride0=2, shared_x_sf_stride1=1,
                    shared_x_sf_rows=128)) == 1            # no shared_block_m
    assert run(args(shared_x=FAKE, shared_x_stride0=256, shared_x_sf=FAKE,
                    shared_block_m=64, shared_x_sf_rows=128)) == 1  # bf16 shared_x with pages
    assert run(args(**fp8, shared_x_sf=FAKE, shared_x_sf_stride0=2, shared_x_sf_stride1=1,
                    shared_x_sf_rows=100, shared_block_m=64)) == 2  # needs 128 rows
    assert run(args(**dict(fp8, shared_x_dtype=7))) == 1  # bad dtype
    assert run(args(shared_x=FAKE, shared_x_stride0=256, shared_x_dtype=B.MOE_SHARED_FP8,
                    shared_x_sf=FAKE + 0, shared_x_sf_stride0=2, shared_x_sf_stride1=1,
                    shared_x_sf_rows=128, shared_block_m=64, hidden=FAKE + 8)) == 4
