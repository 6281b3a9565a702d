"""GPU parity of moe_prepare_nvfp4_inputs against the oracle: E2M1 codes,
E4M3 block scales and per-token fp32 scales bit-exact; routing outputs and
the EPLB load as in the fp8 staging; the bf16 shared copy, the MXFP8 shared
input (fp8 codes of the 1x128 UE8M0 staging, exponent bytes in the
shared-expert pages) and l2_alpha."""
import numpy as np
import pytest
import torch

from moe_expert_layer_prepare_gb300 import binding as B
from moe_expert_layer_prepare_gb300 import synthetic as syn
from tests._util import bf16_bits, need_cuda

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def cuda():
    need_cuda()
    from moe_expert_layer_prepare_gb300 import build
    build.build()
    B.load()
    return torch.device("cuda")


def _hidden(T, K, seed):
    h = syn.make_hidden(T, K, seed, outlier_frac=0.01, zero_group_frac=0.05).float()
    rng = np.random.default_rng(seed)
    scale = torch.from_numpy(np.exp(rng.uniform(-12, 12, (T, 1))).astype(np.float32))
    h = h * scale
    if T > 3:
        h[2] = 0.0                          # all-zero row
        h[3, :16] = 1e-30 * h[3, :16]       # a block far below its row's scale
    return h.to(torch.bfloat16)


def _codes_equal(got, want, orc):
    bad = np.argwhere(got != want)
    if len(bad):
        r, c = bad[0]
        lo = [orc.e2m1_decode(int(v) & 0xF) for v in (got[r, c], want[r, c])]
        hi = [orc.e2m1_decode(int(v) >> 4) for v in (got[r, c], want[r, c])]
        raise AssertionError(f"{len(bad)} code bytes differ; first at row {r} byte {c}: "
                             f"gpu {got[r, c]:#04x} oracle {want[r, c]:#04x} "
                             f"(low nibble {lo}, high nibble {hi})")


def _run(hid, ids, w, pad=None, eplb=None, shared=False, n_local=0, shared_block_m=None):
    dev = torch.device("cuda")
    T, K = hid.shape
    k = ids.shape[1]
    sx_sf = None
    if shared_block_m is not None:  # the MXFP8 shared input with its scale pages
        rows = -(-T // shared_block_m) * (-(-shared_block_m // 128) * 128)
        sx_sf = torch.full((rows, K // 128), 0xEE, dtype=torch.uint8, device=dev)
    x = torch.full((T, K // 2), 0xAB, dtype=torch.uint8, device=dev)
    x_sf = torch.full((T, K // 64), -1, dtype=torch.int32, device=dev)
    xs = torch.full((T,), -1.0, dtype=torch.float32, device=dev)
    io = torch.full((T, k), 7, dtype=torch.int64, device=dev)
    wo = torch.full((T, k), 7.0, dtype=torch.float32, device=dev)
    sx = torch.zeros((T, K), dtype=torch.bfloat16, device=dev) if shared else None
    if shared_block_m is not None:
        sx = torch.full((T, K), 0x5A, dtype=torch.uint8, device=dev)
    w2gs = l2a = None
    if n_local:
        w2gs = torch.rand(n_local, device=dev) * 3
        l2a = torch.full((n_local,), -1.0, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    B.moe_prepare_nvfp4_inputs(hid.to(dev), ids.to(dev), w.to(dev), x, x_sf, xs, io, wo,
                               is_padding=None if pad is None else pad.to(dev), shared_x=sx,
                               eplb=eplb, w2_global_scale=w2gs, l2_alpha=l2a,
                               l2_activation_scale=0.37, device_status=st, shared_x_sf=sx_sf,
                               shared_block_m=shared_block_m)
    torch.cuda.synchronize()
    return dict(x=x.cpu().numpy(), x_sf=x_sf.cpu().numpy(), xs=xs.cpu().numpy(),
                ids=io.cpu().numpy(), w=wo.cpu().numpy(), shared=sx, w2gs=w2gs, l2a=l2a,
                shared_sf=None if sx_sf is None else sx_sf.cpu().numpy(),
                status=int(st.item()))


# 16-value blocks per lane held in registers: 4 (K <= 2048), 8 (<= 4096),
# 14 (<= 7168), 16 (<= 8192); K = 9216 streams the row twice
@pytest.mark.parametrize("T,K,k", [(37, 640, 3), (64, 256, 2), (200, 7168, 8), (16, 384, 1),
                                   (24, 4096, 2), (12, 8192, 4), (9, 9216, 2)])
def test_nvfp4_rows_bit_exact(cuda, orc, T, K, k):
    hid = _hidden(T, K, 40 + T)
    ids, w, pad = syn.make_routing(T, 16, k, 41 + T, padding_frac=0.1)
    g = _run(hid, ids, w, pad, shared=True, n_local=5)
    assert g["status"] == 0
    ref = orc.nvfp4_rows(bf16_bits(hid))
    assert np.array_equal(g["xs"].view(np.int32), ref["x_scales"].view(np.int32))
    assert np.array_equal(g["x_sf"], ref["x_sf"])
    _codes_equal(g["x"], ref["x"], orc)
    rr = orc.prepare_inputs(bf16_bits(hid), ids.numpy(), w.numpy(), is_padding=pad.numpy())
    assert np.array_equal(g["ids"], rr["ids"]) and np.array_equal(g["w"], rr["weights"])
    assert torch.equal(g["shared"].cpu(), hid)
    assert torch.equal(g["l2a"], g["w2gs"] * np.float32(0.37))


def test_nvfp4_staging_stress_full_size(cuda, orc):
    """16384 x 7168 with EPLB recording, in one launch: every routing output
    and the load exactly, and the codes, block scales and row scales of all
    16384 rows."""
    wl = syn.make_workload("staging_stress")
    c = wl["cfg"]
    T, K = c["T"], c["K"]
    dev = torch.device("cuda")
    load = torch.zeros(wl["num_physical"], dtype=torch.int32, device=dev)
    eplb = dict(logical_to_physical=wl["l2p"].to(dev),
                logical_replica_count=wl["replica_count"].to(dev), expert_load=load,
                should_record=torch.ones(1, dtype=torch.uint8, device=dev),
                num_unpadded_tokens=torch.tensor([T], dtype=torch.int32, device=dev))
    g = _run(wl["hidden"], wl["topk_ids"], wl["topk_weights"], eplb=eplb)
    assert g["status"] == 0
    rr = orc.prepare_inputs(np.zeros((T, 128), np.uint16), wl["topk_ids"].numpy(),
                            wl["topk_weights"].numpy(), l2p=wl["l2p"].numpy(),
                            replica_count=wl["replica_count"].numpy(),
                            num_physical=wl["num_physical"], record_enabled=True)
    assert np.array_equal(g["ids"], rr["ids"]) and np.array_equal(g["w"], rr["weights"])
    assert np.array_equal(load.cpu().numpy(), rr["load"])
    ref = orc.nvfp4_rows(bf16_bits(wl["hidden"]))
    _codes_equal(g["x"], ref["x"], orc)
    assert np.array_equal(g["x_sf"], ref["x_sf"])
    assert np.array_equal(g["xs"].view(np.int32), ref["x_scales"].view(np.int32))


# the MXFP8 shared input in both kernel paths (rows held in registers, and
# K = 9216 streamed twice) and with page blocks of 1, partial and several pages
@pytest.mark.parametrize("T,K,block_m", [(200, 7168, 128), (37, 640, 48), (150, 9216, 64),
                                         (300, 256, 256), (16, 384, 1)])
def test_nvfp4_shared_mxfp8(cuda, orc, T, K, block_m):
    """The fp8 shared input equals the oracle's 1x128 UE8M0 staging of the
    same rows (S1-S3), and its exponent bytes sit at the rows of the
    shared-expert pages (S4b); the NVFP4 outputs are unchanged by it."""
    hid = _hidden(T, K, 60 + T)
    ids, w, pad = syn.make_routing(T, 16, 4, 61 + T, padding_frac=0.1)
    g = _run(hid, ids, w, pad, shared_block_m=block_m)
    assert g["status"] == 0
    ref = orc.prepare_inputs(bf16_bits(hid), ids.numpy(), w.numpy(), is_padding=pad.numpy())
    got = g["shared"].cpu().numpy()
    bad = np.argwhere(got != ref["x"])
    assert bad.size == 0, f"{len(bad)} fp8 bytes of the shared input differ, first {bad[0]}"
    pages = orc.shared_sf(ref["x_sf"], K, block_m, rows=g["shared_sf"].shape[0])
    assert np.array_equal(g["shared_sf"], pages)
    rn = orc.nvfp4_rows(bf16_bits(hid))
    _codes_equal(g["x"], rn["x"], orc)
    assert np.array_equal(g["x_sf"], rn["x_sf"])
    assert np.array_equal(g["xs"].view(np.int32), rn["x_scales"].view(np.int32))
    assert np.array_equal(g["ids"], ref["ids"]) and np.array_equal(g["w"], ref["weights"])


def test_nvfp4_shared_mxfp8_staging_stress(cuda, orc):
    """staging_stress (16384 x 7168) with the MXFP8 shared input: every byte
    of the fp8 rows and of the scale pages, in one launch."""
    wl = syn.make_workload("staging_stress")
    T, K = wl["cfg"]["T"], wl["cfg"]["K"]
    g = _run(wl["hidden"], wl["topk_ids"], wl["topk_weights"], shared_block_m=128)
    assert g["status"] == 0
    ref = orc.prepare_inputs(bf16_bits(wl["hidden"]), wl["topk_ids"].numpy(),
                             wl["topk_weights"].numpy())
    assert np.array_equal(g["shared"].cpu().numpy(), ref["x"])
    assert np.array_equal(g["shared_sf"], orc.shared_sf(ref["x_sf"], K, 128))


def test_nvfp4_l2_alpha_without_tokens(cuda):
    dev = torch.device("cuda")
    e = torch.empty((0, 2), dtype=torch.int32, device=dev)
    ew = torch.empty((0, 2), dtype=torch.float32, device=dev)
    w2gs = torch.tensor([1.5, 2.0, 0.25], device=dev)
    l2a = torch.zeros(3, device=dev)
    B.moe_prepare_nvfp4_inputs(torch.empty((0, 256), dtype=torch.bfloat16, device=dev), e, ew,
                               torch.empty((0, 128), dtype=torch.uint8, device=dev),
                               torch.empty((0, 4), dtype=torch.int32, device=dev),
                               torch.empty(0, device=dev),
                               torch.empty((0, 2), dtype=torch.int64, device=dev), ew.clone(),
                               w2_global_scale=w2gs, l2_alpha=l2a, l2_activation_scale=4.0)
    torch.cuda.synchronize()
    assert l2a.cpu().tolist() == [6.0, 8.0, 1.0]
