"""Helpers shared by the tests (comparison, bf16 views, sub-problem builders)."""
import numpy as np
import pytest
import torch


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def bf16_vals(bits) -> np.ndarray:
    return (np.asarray(bits).astype(np.uint32) << 16).view(np.float32)


def u8(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.uint8).numpy()


def unpack_exponents(words, G):
    w = np.asarray(words).astype(np.uint32)
    return np.stack([(w[..., g // 4] >> (8 * (g % 4))) & 0xFF for g in range(G)], axis=-1)


def assert_fp_close(got, ref, what=""):
    """FP output tolerance: normwise relative error <= 1e-2 and elementwise
    |delta| <= 3e-2 * (|ref| + rms(ref))."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    nref = np.linalg.norm(ref)
    rel = np.linalg.norm(got - ref) / max(nref, 1e-30)
    rms = nref / np.sqrt(max(ref.size, 1))
    bound = 3e-2 * (np.abs(ref) + rms)
    bad = np.abs(got - ref) > bound
    assert rel <= 1e-2, f"{what}: normwise relative error {rel:.3e}"
    assert not bad.any(), (f"{what}: {bad.sum()} elements off, worst "
                           f"{np.max(np.abs(got - ref) - bound):.3e}")
    return rel


def assert_codes_close(got_codes, ref_codes, table, what="", max_frac=1e-3):
    """fp8 codes that come from an fp32 value computed with a different exp:
    nearly all identical; the rest one representable step apart."""
    g = np.asarray(got_codes).astype(np.int64).ravel()
    r = np.asarray(ref_codes).astype(np.int64).ravel()
    diff = g != r
    if diff.any():
        gv = table[g[diff]].astype(np.float64)
        rv = table[r[diff]].astype(np.float64)
        # adjacent codes: same sign side, |code distance| 1 in magnitude order
        mag_g = np.where(g[diff] >= 128, -(g[diff] - 128), g[diff])
        mag_r = np.where(r[diff] >= 128, -(r[diff] - 128), r[diff])
        assert np.all(np.abs(mag_g - mag_r) <= 1) or np.all(np.abs(gv - rv) <=
                                                              np.abs(rv) * 0.126 + 1e-30), what
    frac = diff.mean() if diff.size else 0.0
    assert frac <= max_frac, f"{what}: {diff.sum()} of {diff.size} codes differ"
    return int(diff.sum())


def need_cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def routes_of_tokens(ids, slots, tokens, M_max):
    """Global batched rows (e*M_max + slot) used by the given tokens' routes."""
    rows = []
    for t in tokens:
        for j in range(ids.shape[1]):
            e, s = int(ids[t, j]), int(slots[t, j])
            if e >= 0 and s >= 0:
                rows.append(e * M_max + s)
    return np.array(sorted(set(rows)), np.int64)


def compact_experts(rows, M_max, *arrays_per_expert):
    """Re-index a set of global rows onto a compact expert list.

    Returns (new_rows, M_max, [compact arrays]) where every array in
    ``arrays_per_expert`` is indexed [E, ...] and sliced to the used experts.
    """
    experts = np.unique(rows // M_max)
    remap = {int(e): i for i, e in enumerate(experts)}
    new_rows = np.array([remap[int(r // M_max)] * M_max + int(r % M_max) for r in rows], np.int64)
    out = [np.ascontiguousarray(a[experts]) for a in arrays_per_expert]
    return new_rows, experts, out


def oracle_sampled_forward(orc, wl, tokens, want_h=False):
    """Oracle S1-S8 for a sample of tokens of a full-size workload."""
    def weights_of(experts):
        sel = torch.as_tensor(np.asarray(experts, np.int64))
        return tuple(np.ascontiguousarray(wl[n][sel.to(wl[n].device)].cpu().numpy())
                     for n in ("w13", "w13_s", "w2", "w2_s"))
    c = wl["cfg"]
    return orc.sampled_forward(bf16_bits(wl["hidden"]), wl["topk_ids"].cpu().numpy(),
                               wl["topk_weights"].cpu().numpy(),
                               wl["is_padding"].cpu().numpy(), c["E"], c["M_max"], c["N"],
                               tokens, weights_of, want_h=want_h)


def coverage_tokens(ids, slots, n_target, seed, tile=128):
    """A deterministic token sample whose routes reach every m-tile index.

    ids / slots: [T, k] expert ids and within-expert slots (-1 = unrouted).
    Picks, in order: on the most-loaded expert its first slot, the tile
    boundaries 127/128/255/256, the first row of its last (ragged) tile and
    its last slot; on the least-loaded expert its first and last slot; for
    every m-tile index some expert that has that tile, its first and last
    row in it; then the last slot of a few random experts; then random
    tokens up to n_target.  Returns sorted unique token indices.
    """
    ids = np.asarray(ids)
    slots = np.asarray(slots)
    T, k = ids.shape
    E = int(ids.max()) + 1
    counts = np.zeros(E, np.int64)
    owner = {}
    for t in range(T):
        for j in range(k):
            e, s = int(ids[t, j]), int(slots[t, j])
            if e >= 0 and s >= 0:
                owner[(e, s)] = t
                counts[e] = max(counts[e], s + 1)
    picks = []

    def take(e, s):
        if 0 <= s < counts[e] and (e, s) in owner:
            picks.append(owner[(e, s)])

    heavy = int(np.argmax(counts))
    n = int(counts[heavy])
    for s in (0, tile - 1, tile, 2 * tile - 1, 2 * tile, ((n - 1) // tile) * tile, n - 1):
        take(heavy, s)
    live = np.nonzero(counts > 0)[0]
    light = int(live[np.argmin(counts[live])])
    take(light, 0)
    take(light, int(counts[light]) - 1)
    for mt in range(int((counts.max() + tile - 1) // tile)):
        have = np.nonzero(counts > mt * tile)[0]
        if have.size:
            e = int(have[len(have) // 2])
            take(e, mt * tile)
            take(e, min(int(counts[e]), (mt + 1) * tile) - 1)
    rng = np.random.default_rng(seed)
    for e in rng.choice(live, size=min(6, live.size), replace=False):
        take(int(e), int(counts[e]) - 1)
    chosen = list(dict.fromkeys(picks))
    rest = np.setdiff1d(np.arange(T), chosen)
    need = max(0, n_target - len(chosen))
    if need and rest.size:
        chosen += list(rng.choice(rest, size=min(need, rest.size), replace=False))
    return np.array(sorted(set(int(t) for t in chosen)), np.int64)
