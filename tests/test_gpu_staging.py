"""GPU parity of moe_prepare_inputs (staging, top-k repack, EPLB, dispatch)
against the oracle: bit-exact bytes, exponents, ids, weights, slots, counts."""
import numpy as np
import pytest
import torch

from moe_expert_layer_prepare_gb300 import binding as B
from moe_expert_layer_prepare_gb300 import synthetic as syn
from tests._util import bf16_bits, need_cuda, u8

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def cuda():
    need_cuda()
    from moe_expert_layer_prepare_gb300 import build
    build.build()
    B.load()
    return torch.device("cuda")


def _gpu_stage(hidden, ids, w, pad=None, sf_mode=B.MOE_SF_UE8M0_PACKED, eplb=None,
               dispatch=None):
    dev = torch.device("cuda")
    T, K = hidden.shape
    k = ids.shape[1]
    G = K // 128
    h = hidden.to(dev)
    x = torch.full((T, K), 0xAA, dtype=torch.uint8, device=dev) if sf_mode else \
        torch.zeros((T, K), dtype=torch.bfloat16, device=dev)
    if sf_mode == B.MOE_SF_UE8M0_PACKED:
        x_sf = torch.full((T, (G + 3) // 4), -1, dtype=torch.int32, device=dev)
    elif sf_mode == B.MOE_SF_FP32:
        x_sf = torch.full((T, G), -1.0, dtype=torch.float32, device=dev)
    else:
        x_sf = None
    ids_out = torch.full((T, k), 77, dtype=torch.int64, device=dev)
    w_out = torch.full((T, k), 7.0, dtype=torch.float32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    B.moe_prepare_inputs(h, ids.to(dev), w.to(dev), x, x_sf, ids_out, w_out,
                         is_padding=None if pad is None else pad.to(dev), sf_mode=sf_mode,
                         eplb=eplb, dispatch=dispatch, device_status=status)
    torch.cuda.synchronize()
    return x, x_sf, ids_out.cpu().numpy(), w_out.cpu().numpy(), int(status.item())


CASES = [
    # T, K, k, ids dtype, weights dtype, padding, sf mode
    (37, 640, 3, torch.int32, torch.float32, True, B.MOE_SF_UE8M0_PACKED),
    (64, 256, 2, torch.int64, torch.bfloat16, False, B.MOE_SF_UE8M0_PACKED),
    (200, 7168, 8, torch.int32, torch.float32, True, B.MOE_SF_UE8M0_PACKED),
    (33, 1024, 4, torch.int32, torch.float32, True, B.MOE_SF_FP32),
    (16, 384, 1, torch.int32, torch.float32, False, B.MOE_SF_NONE),
    # from 1024 tokens the rows stream through shared memory (one row buffer
    # per warp): every sf mode, both id and weight dtypes, a ragged last word
    (1500, 1152, 4, torch.int32, torch.float32, True, B.MOE_SF_UE8M0_PACKED),
    (1100, 640, 3, torch.int64, torch.bfloat16, False, B.MOE_SF_FP32),
    (1030, 384, 1, torch.int32, torch.float32, True, B.MOE_SF_NONE),
    (2048, 8192, 2, torch.int32, torch.float32, False, B.MOE_SF_UE8M0_PACKED),
]


@pytest.mark.parametrize("T,K,k,idt,wdt,use_pad,sf_mode", CASES)
def test_staging_token_order(cuda, orc, T, K, k, idt, wdt, use_pad, sf_mode):
    hid = syn.make_hidden(T, K, 100 + T, outlier_frac=0.01, zero_group_frac=0.05)
    ids, w, pad = syn.make_routing(T, 64, k, 200 + T, padding_frac=0.2 if use_pad else 0.0)
    ids, w = ids.to(idt), w.to(wdt)
    x, x_sf, ids_out, w_out, st = _gpu_stage(hid, ids, w, pad if use_pad else None,
                                             sf_mode=sf_mode)
    assert st == 0
    ref = orc.prepare_inputs(bf16_bits(hid), ids.numpy(), w.to(torch.float32).numpy(),
                             is_padding=pad.numpy() if use_pad else None,
                             sf_mode=sf_mode if sf_mode else 1)
    assert np.array_equal(ids_out, ref["ids"])
    assert np.array_equal(w_out.view(np.uint32), ref["weights"].view(np.uint32))
    if sf_mode == B.MOE_SF_NONE:
        assert torch.equal(x.cpu(), hid)
        return
    xb = u8(x)
    bad = np.nonzero(xb != ref["x"])
    assert bad[0].size == 0, f"{bad[0].size} fp8 bytes differ, first at {bad[0][0]},{bad[1][0]}"
    if sf_mode == B.MOE_SF_UE8M0_PACKED:
        assert np.array_equal(x_sf.cpu().numpy(), ref["x_sf"])
    else:
        assert np.array_equal(x_sf.cpu().numpy().view(np.uint32), ref["x_sf"].view(np.uint32))


def test_staging_eplb_record(cuda, orc):
    T, K, k, E = 300, 512, 8, 64
    hid = syn.make_hidden(T, K, 5)
    ids, w, pad = syn.make_routing(T, E, k, 6, padding_frac=0.05)
    l2p, rc, nphys = syn.make_eplb(E, 7, two=8, three=4)
    dev = torch.device("cuda")
    load = torch.zeros(nphys, dtype=torch.int32, device=dev)
    eplb = dict(logical_to_physical=l2p.to(dev), logical_replica_count=rc.to(dev),
                expert_load=load, should_record=torch.ones(1, dtype=torch.uint8, device=dev),
                num_unpadded_tokens=torch.tensor([250], dtype=torch.int32, device=dev))
    x, x_sf, ids_out, w_out, st = _gpu_stage(hid, ids, w, pad, eplb=eplb)
    assert st == 0
    ref = orc.prepare_inputs(bf16_bits(hid), ids.numpy(), w.numpy(), is_padding=pad.numpy(),
                             l2p=l2p.numpy(), replica_count=rc.numpy(), num_physical=nphys,
                             record_enabled=True, num_unpadded=250)
    assert np.array_equal(ids_out, ref["ids"])
    assert np.array_equal(load.cpu().numpy(), ref["load"])
    # recording off: no load
    load.zero_()
    eplb["should_record"] = torch.zeros(1, dtype=torch.uint8, device=dev)
    _gpu_stage(hid, ids, w, pad, eplb=eplb)
    assert int(load.sum().item()) == 0


def test_staging_stress_full_size(cuda, orc):
    """staging_stress (16384 x 7168, EPLB 256 -> 288) in the bench's launch
    configuration; the oracle checks every routing output, the EPLB load and
    every quantised byte and packed exponent word of all 16384 rows."""
    wl = syn.make_workload("staging_stress")
    c = wl["cfg"]
    T, K, k = c["T"], c["K"], c["top_k"]
    dev = torch.device("cuda")
    load = torch.zeros(wl["num_physical"], dtype=torch.int32, device=dev)
    eplb = dict(logical_to_physical=wl["l2p"].to(dev),
                logical_replica_count=wl["replica_count"].to(dev), expert_load=load,
                should_record=torch.ones(1, dtype=torch.uint8, device=dev),
                num_unpadded_tokens=torch.tensor([T], dtype=torch.int32, device=dev))
    x, x_sf, ids_out, w_out, st = _gpu_stage(wl["hidden"], wl["topk_ids"], wl["topk_weights"],
                                             None, eplb=eplb)
    assert st == 0
    ref = orc.prepare_inputs(bf16_bits(wl["hidden"]), wl["topk_ids"].numpy(),
                             wl["topk_weights"].numpy(), l2p=wl["l2p"].numpy(),
                             replica_count=wl["replica_count"].numpy(),
                             num_physical=wl["num_physical"], record_enabled=True)
    assert np.array_equal(ids_out, ref["ids"])
    assert np.array_equal(w_out, ref["weights"])
    assert np.array_equal(load.cpu().numpy(), ref["load"])
    xa = x.cpu().numpy()
    bad = np.nonzero(xa != ref["x"])
    assert bad[0].size == 0, f"{bad[0].size} fp8 bytes differ, first at {bad[0][0]},{bad[1][0]}"
    assert np.array_equal(x_sf.cpu().numpy(), ref["x_sf"])
    # the workload's all-zero groups take the amax floor: exponent 105, +0 codes
    G = K // 128
    e = np.stack([(ref["x_sf"][:, g // 4].astype(np.uint32) >> (8 * (g % 4))) & 0xFF
                  for g in range(G)], axis=1)
    zero = ~bf16_bits(wl["hidden"]).reshape(T, G, 128).any(axis=2)
    assert zero.any() and np.all(e[zero] == 105)


def _dispatch_case(T, K, k, E, M_max, zipf=None, pad_frac=0.0, seed=0):
    hid = syn.make_hidden(T, K, seed)
    ids, w, pad = syn.make_routing(T, E, k, seed + 1, zipf_s=zipf, padding_frac=pad_frac)
    return hid, ids, w, pad


@pytest.mark.parametrize("T,K,k,E,M_max,zipf,pad_frac", [
    (32, 256, 2, 4, 32, None, 0.0),           # tiny
    (128, 7168, 8, 256, 128, 1.1, 0.02),      # deepseek decode routing
    (300, 384, 8, 64, 300, None, 0.1),        # 3 route blocks, ragged
    (8192, 256, 8, 256, 1024, None, 0.0),     # deepseek prefill routing (narrow K)
    (120, 256, 8, 1024, 8, None, 0.0),        # the most experts, one-launch path
    (600, 256, 8, 1024, 32, None, 0.05),      # the most experts, routing kernel
])
def test_dispatch(cuda, orc, T, K, k, E, M_max, zipf, pad_frac):
    hid, ids, w, pad = _dispatch_case(T, K, k, E, M_max, zipf, pad_frac, seed=T + E)
    dev = torch.device("cuda")
    G = K // 128
    Wd = (G + 3) // 4
    x_b = torch.full((E * M_max, K), 0x5A, dtype=torch.uint8, device=dev)
    sf_b = torch.full((E * M_max, Wd), -7, dtype=torch.int32, device=dev)
    ent = torch.full((E,), -1, dtype=torch.int32, device=dev)
    slot = torch.full((T, k), -9, dtype=torch.int32, device=dev)
    ws = torch.empty(B.prepare_workspace_size(T, k, E), dtype=torch.uint8, device=dev)
    disp = dict(num_experts=E, max_tokens_per_expert=M_max, x_b=x_b, sf_b=sf_b,
                expert_num_tokens=ent, route_slot=slot, workspace=ws)
    x, x_sf, ids_out, w_out, st = _gpu_stage(hid, ids, w, pad, dispatch=disp)
    assert st == 0
    ref = orc.prepare_inputs(bf16_bits(hid), ids.numpy(), w.numpy(), is_padding=pad.numpy())
    d = orc.dispatch(ref["ids"], ref["x"], ref["x_sf"], E, M_max)
    assert d["status"] == 0
    assert np.array_equal(ent.cpu().numpy(), d["expert_num_tokens"])
    assert np.array_equal(slot.cpu().numpy(), d["route_slot"])
    n = d["expert_num_tokens"]
    xb = x_b.cpu().numpy().reshape(E, M_max, K)
    sfb = sf_b.cpu().numpy().reshape(E, M_max, Wd)
    rxb = d["x_b"].reshape(E, M_max, K)
    rsf = d["sf_b"].reshape(E, M_max, Wd)
    for e in range(E):
        assert np.array_equal(xb[e, :n[e]], rxb[e, :n[e]])
        assert np.array_equal(sfb[e, :n[e]], rsf[e, :n[e]])
        # rows past the expert's count are not written
        assert np.all(xb[e, n[e]:] == 0x5A)
    # the same call twice gives the same result (deterministic, counters reset)
    slot2 = slot.clone()
    _gpu_stage(hid, ids, w, pad, dispatch=disp)
    assert torch.equal(slot, slot2)


def test_dispatch_capacity(cuda, orc):
    T, K, k, E, M_max = 64, 128, 2, 4, 8
    hid, ids, w, pad = _dispatch_case(T, K, k, E, M_max, seed=3)
    dev = torch.device("cuda")
    x_b = torch.zeros((E * M_max, K), dtype=torch.uint8, device=dev)
    sf_b = torch.zeros((E * M_max, 1), dtype=torch.int32, device=dev)
    ent = torch.zeros(E, dtype=torch.int32, device=dev)
    slot = torch.zeros((T, k), dtype=torch.int32, device=dev)
    ws = torch.empty(B.prepare_workspace_size(T, k, E), dtype=torch.uint8, device=dev)
    disp = dict(num_experts=E, max_tokens_per_expert=M_max, x_b=x_b, sf_b=sf_b,
                expert_num_tokens=ent, route_slot=slot, workspace=ws)
    _, _, _, _, st = _gpu_stage(hid, ids, w, None, dispatch=disp)
    assert st & B.MOE_DEV_CAPACITY
    ref = orc.prepare_inputs(bf16_bits(hid), ids.numpy(), w.numpy())
    d = orc.dispatch(ref["ids"], ref["x"], ref["x_sf"], E, M_max)
    assert d["status"] == 1
    assert np.array_equal(ent.cpu().numpy(), d["expert_num_tokens"])
    assert np.array_equal(slot.cpu().numpy(), d["route_slot"])


def test_empty_batch_is_noop(cuda):
    dev = torch.device("cuda")
    x = torch.zeros((0, 256), dtype=torch.uint8, device=dev)
    B.moe_prepare_inputs(torch.zeros((0, 256), dtype=torch.bfloat16, device=dev),
                         torch.zeros((0, 2), dtype=torch.int32, device=dev),
                         torch.zeros((0, 2), dtype=torch.float32, device=dev), x,
                         torch.zeros((0, 1), dtype=torch.int32, device=dev),
                         torch.zeros((0, 2), dtype=torch.int64, device=dev),
                         torch.zeros((0, 2), dtype=torch.float32, device=dev))
    torch.cuda.synchronize()


def _shared_pages(hidden, ids, w, block_m, dispatch=None, fill=0xEE, extra_rows=5):
    dev = torch.device("cuda")
    T, K = hidden.shape
    G = K // 128
    padded = (block_m + 127) // 128 * 128
    rows = (T + block_m - 1) // block_m * padded + extra_rows
    shared = torch.full((rows, G), fill, dtype=torch.uint8, device=dev)
    x = torch.empty((T, K), dtype=torch.uint8, device=dev)
    x_sf = torch.empty((T, (G + 3) // 4), dtype=torch.int32, device=dev)
    k = ids.shape[1]
    ids_out = torch.empty((T, k), dtype=torch.int64, device=dev)
    w_out = torch.empty((T, k), dtype=torch.float32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    B.moe_prepare_inputs(hidden.to(dev), ids.to(dev), w.to(dev), x, x_sf, ids_out, w_out,
                         dispatch=dispatch, device_status=status, shared_x_sf=shared,
                         shared_block_m=block_m)
    torch.cuda.synchronize()
    return shared.cpu().numpy(), x_sf.cpu().numpy(), int(status.item())


@pytest.mark.parametrize("T,K,block_m", [
    (300, 896, 200),    # G = 7: ragged last word; partial pages
    (300, 896, 1),      # one token per block
    (257, 256, 128),    # whole pages plus one token
    (1000, 7168, 256),  # DeepSeek-V3 hidden size
    (64, 4096, 64),     # block smaller than a page
    (3000, 7168, 512),  # a long batch: rows streamed through shared memory
])
def test_shared_scale_pages(cuda, orc, T, K, block_m):
    """Shared-expert scale pages: every token's exponent bytes at its page
    row, bit-exact with the oracle; rows no token maps to stay untouched."""
    hid = syn.make_hidden(T, K, 7 + T, outlier_frac=0.01, zero_group_frac=0.05)
    ids, w, _ = syn.make_routing(T, 8, 2, 8 + T)
    shared, x_sf, st = _shared_pages(hid, ids, w, block_m)
    assert st == 0
    ref = orc.prepare_inputs(bf16_bits(hid), ids.numpy(), w.numpy())
    assert np.array_equal(x_sf, ref["x_sf"])
    want = orc.shared_sf(ref["x_sf"], K, block_m, rows=shared.shape[0], fill=0xEE)
    assert np.array_equal(shared, want)


def test_shared_scale_pages_with_dispatch(cuda, orc):
    """The pages are written in token order also when the rows are dispatched."""
    T, K, k, E, M_max = 128, 7168, 8, 256, 128
    hid, ids, w, pad = _dispatch_case(T, K, k, E, M_max, 1.1, 0.0, seed=3)
    dev = torch.device("cuda")
    Wd = (K // 128 + 3) // 4
    disp = dict(num_experts=E, max_tokens_per_expert=M_max,
                x_b=torch.empty((E * M_max, K), dtype=torch.uint8, device=dev),
                sf_b=torch.empty((E * M_max, Wd), dtype=torch.int32, device=dev),
                expert_num_tokens=torch.empty((E,), dtype=torch.int32, device=dev),
                route_slot=torch.empty((T, k), dtype=torch.int32, device=dev),
                workspace=torch.empty(B.prepare_workspace_size(T, k, E), dtype=torch.uint8,
                                      device=dev))
    shared, x_sf, st = _shared_pages(hid, ids, w, 96, dispatch=disp)
    assert st == 0
    ref = orc.prepare_inputs(bf16_bits(hid), ids.numpy(), w.numpy())
    want = orc.shared_sf(ref["x_sf"], K, 96, rows=shared.shape[0], fill=0xEE)
    assert np.array_equal(shared, want)


@pytest.mark.parametrize("T,K,k,idt,wdt,sf_mode,contiguous", [
    # up to 1024 routes: routing and quantisation in one launch
    (96, 640, 8, torch.int64, torch.bfloat16, B.MOE_SF_FP32, False),
    (128, 1152, 8, torch.int32, torch.float32, B.MOE_SF_UE8M0_PACKED, True),
    (1, 256, 3, torch.int32, torch.float32, B.MOE_SF_UE8M0_PACKED, False),
    (1024, 256, 1, torch.int32, torch.float32, B.MOE_SF_UE8M0_PACKED, True),
    # beyond: the routing kernel, then the quantisation
    (129, 640, 8, torch.int64, torch.bfloat16, B.MOE_SF_FP32, False),
    (300, 1152, 8, torch.int32, torch.float32, B.MOE_SF_UE8M0_PACKED, True),
])
def test_dispatch_with_eplb_both_paths(cuda, orc, T, K, k, idt, wdt, sf_mode, contiguous):
    """Dispatch with EPLB replicas (load recorded, a tail of padded tokens
    not counted), padding rows, either scale format and either layout, on
    both sides of the one-launch limit: every output bit-exact with the
    oracle."""
    E_log = 32
    hid = syn.make_hidden(T, K, 40 + T, outlier_frac=0.01, zero_group_frac=0.05)
    ids, w, pad = syn.make_routing(T, E_log, k, 41 + T, zipf_s=1.1, padding_frac=0.05)
    ids, w = ids.to(idt), w.to(wdt)
    l2p, rc, nphys = syn.make_eplb(E_log, 42, two=6, three=3)
    dev = torch.device("cuda")
    unpadded = max(T - 3, 1)
    load = torch.zeros(nphys, dtype=torch.int32, device=dev)
    eplb = dict(logical_to_physical=l2p.to(dev), logical_replica_count=rc.to(dev),
                expert_load=load, should_record=torch.ones(1, dtype=torch.uint8, device=dev),
                num_unpadded_tokens=torch.tensor([unpadded], dtype=torch.int32, device=dev))
    E = nphys
    M_max = (T * k + E - 1) // E if contiguous else max(8, (T * k) // E)
    G = K // 128
    Wd = G if sf_mode == B.MOE_SF_FP32 else (G + 3) // 4
    sf_dt = torch.float32 if sf_mode == B.MOE_SF_FP32 else torch.int32
    rows_cap = E * M_max
    x_b = torch.full((rows_cap, K), 0x5A, dtype=torch.uint8, device=dev)
    sf_b = torch.full((rows_cap, Wd), -7, dtype=sf_dt, device=dev)
    ent = torch.full((E,), -1, dtype=torch.int32, device=dev)
    slot = torch.full((T, k), -9, dtype=torch.int32, device=dev)
    ws = torch.empty(B.prepare_workspace_size(T, k, E), dtype=torch.uint8, device=dev)
    disp = dict(num_experts=E, max_tokens_per_expert=M_max, x_b=x_b, sf_b=sf_b,
                expert_num_tokens=ent, route_slot=slot, workspace=ws)
    offs = None
    if contiguous:
        offs = torch.full((E + 1,), -1, dtype=torch.int32, device=dev)
        disp["expert_offsets"] = offs
    x, x_sf, ids_out, w_out, st = _gpu_stage(hid, ids, w, pad, sf_mode=sf_mode, eplb=eplb,
                                             dispatch=disp)
    ref = orc.prepare_inputs(bf16_bits(hid), ids.numpy(), w.to(torch.float32).numpy(),
                             is_padding=pad.numpy(), sf_mode=sf_mode, l2p=l2p.numpy(),
                             replica_count=rc.numpy(), num_physical=nphys,
                             record_enabled=True, num_unpadded=unpadded)
    assert np.array_equal(ids_out, ref["ids"])
    assert np.array_equal(w_out.view(np.uint32), ref["weights"].view(np.uint32))
    assert np.array_equal(load.cpu().numpy(), ref["load"])
    assert np.array_equal(u8(x), ref["x"])
    sfw = x_sf.cpu().numpy()
    assert np.array_equal(sfw.view(np.uint32), ref["x_sf"].view(np.uint32))
    if contiguous:
        d = orc.dispatch_contiguous(ref["ids"], ref["x"], ref["x_sf"], E)
        assert np.array_equal(offs.cpu().numpy(), d["expert_offsets"])
        assert np.array_equal(slot.cpu().numpy(), d["route_row"])
        n_rows = int(d["expert_offsets"][-1])
        xr, sfr = d["x_c"][:n_rows], d["sf_c"][:n_rows]
        assert np.all(x_b.cpu().numpy()[n_rows:] == 0x5A)
    else:
        d = orc.dispatch(ref["ids"], ref["x"], ref["x_sf"], E, M_max)
        assert np.array_equal(slot.cpu().numpy(), d["route_slot"])
        rows = orc.valid_rows(d["expert_num_tokens"], M_max)
        n_rows = len(rows)
        xr, sfr = d["x_b"][rows], d["sf_b"][rows]
    assert st == d["status"]
    assert np.array_equal(ent.cpu().numpy(), d["expert_num_tokens"])
    got_x = x_b.cpu().numpy()
    got_sf = sf_b.cpu().numpy()
    if contiguous:
        got_x, got_sf = got_x[:n_rows], got_sf[:n_rows]
    else:
        got_x, got_sf = got_x[rows], got_sf[rows]
    assert np.array_equal(got_x, xr)
    assert np.array_equal(got_sf.view(np.uint32), np.asarray(sfr).view(np.uint32))


@pytest.mark.parametrize("T,k,E", [
    (100, 8, 1000),   # one launch: each scan thread owns four experts, the last three
    (60, 4, 300),     # one launch: two experts a thread, most threads idle
])
def test_small_dispatch_contiguous_many_experts(cuda, orc, T, k, E):
    """The one-launch dispatch in the contiguous layout with more experts than
    scan threads: offsets, rows, copied rows and scales bit-exact."""
    K = 256
    hid = syn.make_hidden(T, K, 70 + E)
    ids, w, pad = syn.make_routing(T, E, k, 71 + E, padding_frac=0.05)
    dev = torch.device("cuda")
    M_max = (T * k + E - 1) // E
    rows_cap = E * M_max
    Wd = (K // 128 + 3) // 4
    x_b = torch.full((rows_cap, K), 0x5A, dtype=torch.uint8, device=dev)
    sf_b = torch.full((rows_cap, Wd), -7, dtype=torch.int32, device=dev)
    ent = torch.full((E,), -1, dtype=torch.int32, device=dev)
    slot = torch.full((T, k), -9, dtype=torch.int32, device=dev)
    offs = torch.full((E + 1,), -1, dtype=torch.int32, device=dev)
    ws = torch.empty(B.prepare_workspace_size(T, k, E), dtype=torch.uint8, device=dev)
    disp = dict(num_experts=E, max_tokens_per_expert=M_max, x_b=x_b, sf_b=sf_b,
                expert_num_tokens=ent, route_slot=slot, workspace=ws, expert_offsets=offs)
    _, _, _, _, st = _gpu_stage(hid, ids, w, pad, dispatch=disp)
    assert st == 0
    ref = orc.prepare_inputs(bf16_bits(hid), ids.numpy(), w.numpy(), is_padding=pad.numpy())
    d = orc.dispatch_contiguous(ref["ids"], ref["x"], ref["x_sf"], E)
    assert d["status"] == 0
    assert np.array_equal(offs.cpu().numpy(), d["expert_offsets"])
    assert np.array_equal(ent.cpu().numpy(), d["expert_num_tokens"])
    assert np.array_equal(slot.cpu().numpy(), d["route_row"])
    n = int(d["expert_offsets"][-1])
    assert np.array_equal(x_b.cpu().numpy()[:n], d["x_c"][:n])
    assert np.array_equal(sf_b.cpu().numpy()[:n], d["sf_c"][:n])
    assert np.all(x_b.cpu().numpy()[n:] == 0x5A)
