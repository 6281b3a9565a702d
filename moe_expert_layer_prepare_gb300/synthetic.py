"""Seeded synthetic inputs for the MoE expert layer workloads.

This module only draws random numbers and lays them out; it holds none of the
staging, GEMM or reduce arithmetic.  Both the CUDA path and the CPU oracle are
fed from here so that they see identical bytes.

Workloads (shapes of public models only; all values synthetic):

=================  =====  =====  =====  ===  =====  =====
name               T      K      N      E    top-k  M_max
=================  =====  =====  =====  ===  =====  =====
tiny               32     256    512    4    2      32
mixtral_decode     64     4096   14336  8    2      64
deepseek_decode    128    7168   2048   256  8      128
deepseek_prefill   8192   7168   2048   256  8      1024
staging_stress     16384  7168   --     256  8      --   (EPLB 256 -> 288)
=================  =====  =====  =====  ===  =====  =====

Recipes:

* hidden: N(0, 1) rounded to bf16.  staging_stress also multiplies 1% of the
  elements by 50 and zeroes 0.5% of the 1x128 groups.
* routing: logits N(0, 1) (deepseek_decode adds a Zipf(1.1) bias
  ``-1.1 * log(rank)`` over a seeded permutation of the experts), softmax,
  top-k, weights renormalised to sum 1.  deepseek_decode flags 2% of the
  tokens as padding (seeded Bernoulli).
* expert weights: N(0, 0.02) fp32, per 128x128 block ``scale = amax / 448``
  (fp32), fp8 e4m3 codes from PyTorch's ``float8_e4m3fn`` cast of ``w / scale``.
  This is the checkpoint format (static 128x128 block FP8), not a step of the
  path.
* EPLB (staging_stress): 16 logical experts get 2 replicas and 8 get 3 (288
  physical slots); physical ids are a seeded permutation of 0..287; the
  logical->physical table is padded with -1 to width 3.
"""
from __future__ import annotations

import numpy as np
import torch

CONFIGS = {
    "tiny": dict(index=1, T=32, K=256, N=512, E=4, top_k=2, M_max=32,
                 zipf_s=None, padding_frac=0.0),
    "mixtral_decode": dict(index=2, T=64, K=4096, N=14336, E=8, top_k=2, M_max=64,
                           zipf_s=None, padding_frac=0.0),
    "deepseek_decode": dict(index=3, T=128, K=7168, N=2048, E=256, top_k=8, M_max=128,
                            zipf_s=1.1, padding_frac=0.02),
    "deepseek_prefill": dict(index=4, T=8192, K=7168, N=2048, E=256, top_k=8, M_max=1024,
                             zipf_s=None, padding_frac=0.0),
    # profiling stand-in for deepseek_prefill: the same per-expert load
    # (~256 rows per expert) and shapes over 32 experts, small enough for a
    # full counter capture
    "deepseek_prefill_e32": dict(index=6, T=1024, K=7168, N=2048, E=32, top_k=8, M_max=1024,
                                 zipf_s=None, padding_frac=0.0),
    "staging_stress": dict(index=5, T=16384, K=7168, N=None, E=256, top_k=8, M_max=None,
                           zipf_s=None, padding_frac=0.0, outlier_frac=0.01,
                           outlier_scale=50.0, zero_group_frac=0.005,
                           eplb=dict(two=16, three=8)),
}


def seed_of(name: str, stream: int) -> int:
    """Seed of one random stream of a workload: 1000 + index, then spawned."""
    base = 1000 + CONFIGS[name]["index"] if name in CONFIGS else int(name)
    ss = np.random.SeedSequence([base, stream])
    return int(ss.generate_state(1, dtype=np.uint32)[0])


def make_hidden(T: int, K: int, seed: int, outlier_frac: float = 0.0,
                outlier_scale: float = 50.0, zero_group_frac: float = 0.0) -> torch.Tensor:
    """bf16 [T, K] on the CPU."""
    rng = np.random.default_rng(seed)
    h = rng.standard_normal((T, K), dtype=np.float32)
    if outlier_frac > 0:
        mask = rng.random((T, K), dtype=np.float32) < outlier_frac
        h[mask] *= np.float32(outlier_scale)
    if zero_group_frac > 0 and K % 128 == 0:
        g = h.reshape(T, K // 128, 128)
        zmask = rng.random((T, K // 128)) < zero_group_frac
        g[zmask] = 0.0
    return torch.from_numpy(h).to(torch.bfloat16)


def make_routing(T: int, E: int, top_k: int, seed: int, zipf_s: float | None = None,
                 padding_frac: float = 0.0):
    """Router outputs: ids int32 [T, k], weights fp32 [T, k], is_padding uint8 [T]."""
    rng = np.random.default_rng(seed)
    logits = rng.standard_normal((T, E))
    if zipf_s is not None:
        rank = np.empty(E, np.int64)
        rank[rng.permutation(E)] = np.arange(1, E + 1)
        logits = logits + (-zipf_s) * np.log(rank.astype(np.float64))[None, :]
    logits = logits - logits.max(axis=1, keepdims=True)
    p = np.exp(logits)
    p /= p.sum(axis=1, keepdims=True)
    ids = np.argsort(-p, axis=1, kind="stable")[:, :top_k]
    w = np.take_along_axis(p, ids, axis=1)
    w = w / w.sum(axis=1, keepdims=True)
    pad = (rng.random(T) < padding_frac).astype(np.uint8) if padding_frac > 0 else \
        np.zeros(T, np.uint8)
    return (torch.from_numpy(ids.astype(np.int32)), torch.from_numpy(w.astype(np.float32)),
            torch.from_numpy(pad))


def make_block_fp8_weights(E: int, rows: int, cols: int, seed: int, device="cpu",
                           std: float = 0.02, experts=None):
    """Static 128x128 block-FP8 expert weights.

    Returns (codes uint8 [E, rows, cols], scales fp32 [E, rows/128, cols/128]) on
    `device`.  Each expert is drawn from its own generator so that any expert
    can be produced alone: with ``experts`` (a list of expert ids) only those
    are drawn, stacked in that order, identical to the same experts of the full
    set on the same device.
    """
    assert rows % 128 == 0 and cols % 128 == 0
    ids = list(range(E)) if experts is None else [int(e) for e in experts]
    q = torch.empty((len(ids), rows, cols), dtype=torch.uint8, device=device)
    s = torch.empty((len(ids), rows // 128, cols // 128), dtype=torch.float32, device=device)
    for i, e in enumerate(ids):
        g = torch.Generator(device=device)
        g.manual_seed(int(seed) * 100003 + e)
        w = torch.randn((rows, cols), generator=g, device=device, dtype=torch.float32) * std
        blocks = w.view(rows // 128, 128, cols // 128, 128)
        amax = blocks.abs().amax(dim=(1, 3)).clamp_min(1e-12)
        sc = amax / 448.0
        scaled = (blocks / sc[:, None, :, None]).clamp_(-448.0, 448.0)
        q[i] = scaled.reshape(rows, cols).to(torch.float8_e4m3fn).view(torch.uint8)
        s[i] = sc
    return q, s


def make_eplb(num_logical: int, seed: int, two: int = 16, three: int = 8):
    """EPLB replica table: l2p int32 [num_logical, 3] (-1 padded), counts int32."""
    rng = np.random.default_rng(seed)
    counts = np.ones(num_logical, np.int32)
    chosen = rng.permutation(num_logical)
    counts[chosen[:two]] = 2
    counts[chosen[two:two + three]] = 3
    num_physical = int(counts.sum())
    phys = rng.permutation(num_physical).astype(np.int32)
    l2p = np.full((num_logical, 3), -1, np.int32)
    pos = 0
    for e in range(num_logical):
        l2p[e, :counts[e]] = phys[pos:pos + counts[e]]
        pos += counts[e]
    return torch.from_numpy(l2p), torch.from_numpy(counts), num_physical


def make_workload(name: str, weights_device="cpu", with_weights: bool = True,
                  T: int | None = None):
    """All inputs of one workload (optionally with fewer tokens, same recipe)."""
    c = dict(CONFIGS[name])
    if T is not None:
        c["T"] = T
    out = dict(name=name, cfg=c)
    out["hidden"] = make_hidden(c["T"], c["K"], seed_of(name, 0),
                                outlier_frac=c.get("outlier_frac", 0.0),
                                outlier_scale=c.get("outlier_scale", 50.0),
                                zero_group_frac=c.get("zero_group_frac", 0.0))
    ids, w, pad = make_routing(c["T"], c["E"], c["top_k"], seed_of(name, 1),
                               zipf_s=c["zipf_s"], padding_frac=c["padding_frac"])
    out.update(topk_ids=ids, topk_weights=w, is_padding=pad)
    if c.get("eplb"):
        l2p, rc, nphys = make_eplb(c["E"], seed_of(name, 4), **c["eplb"])
        out.update(l2p=l2p, replica_count=rc, num_physical=nphys)
    if with_weights and c.get("N"):
        out["w13"], out["w13_s"] = make_block_fp8_weights(c["E"], 2 * c["N"], c["K"],
                                                          seed_of(name, 2), weights_device)
        out["w2"], out["w2_s"] = make_block_fp8_weights(c["E"], c["K"], c["N"],
                                                        seed_of(name, 3), weights_device)
    return out
