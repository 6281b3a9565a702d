"""CPU oracle for the batched grouped-masked block-FP8 MoE expert forward.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` may import this package.  The
product path (``moe_expert_layer_prepare_gb300``) never imports it, and the two
share no code: this file only marshals numpy arrays into the plain C oracle in
``moe_oracle.c``, which restates the pages' steps S1-S8:

* vllm.model_executor.layers.fused_moe.prepare_megamoe -- ``_quantize_fp8_groups``
  (S1 e4m3, S2 group scale, S3 quantise), ``_pack_bytes`` (S4),
  ``_store_topk`` / ``_eplb_kernel_args`` / ``prepare_megamoe_inputs`` (S5).
* vllm.model_executor.layers.fused_moe.experts.fused_humming_moe --
  ``BatchedHummingGroupedExperts.apply`` and ``HummingExpertsBase.get_buffer_metas``
  (S6 batched layout, S7 GEMMs + SiLU-and-mul + requant), ``moe_fused_mul_sum`` /
  ``TopKWeightAndReduceDelegate`` (S8 weighted reduce).

Parity unpinned: the slot order inside an expert is the dispatch's choice (the
oracle takes (token, k) order); last-ulp differences between the CUDA ``expf``
and the C library ``exp`` are covered by tolerance only.
"""
from __future__ import annotations

import ctypes
import os
import platform
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", f"liboracle_{platform.machine()}.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle (gcc, -O2, OpenMP, no fast-math, no FP contraction)."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-fopenmp",
           "-ffp-contract=off", "-fno-fast-math", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        i64, i32, f32, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_float, ctypes.c_void_p
        lib.orc_abi_version.restype = i32
        lib.orc_num_threads.restype = i32
        lib.orc_e4m3_encode.restype = ctypes.c_uint8
        lib.orc_e4m3_encode.argtypes = [f32]
        lib.orc_e4m3_decode.restype = f32
        lib.orc_e4m3_decode.argtypes = [ctypes.c_uint8]
        lib.orc_bf16_from_f64.restype = ctypes.c_uint16
        lib.orc_bf16_from_f64.argtypes = [ctypes.c_double]
        lib.orc_group_scale.restype = None
        lib.orc_group_scale.argtypes = [f32, i32, ctypes.POINTER(ctypes.c_uint32),
                                        ctypes.POINTER(f32)]
        lib.orc_prepare_inputs.restype = i32
        lib.orc_prepare_inputs.argtypes = [i64, i64, i64, vp, vp, i32, vp, vp, i32, vp, vp,
                                           vp, vp, vp, i64, i64, vp, vp, i64, i32, i64]
        lib.orc_e2m1_encode.restype = ctypes.c_uint8
        lib.orc_e2m1_encode.argtypes = [f32]
        lib.orc_e2m1_decode.restype = f32
        lib.orc_e2m1_decode.argtypes = [ctypes.c_uint8]
        lib.orc_nvfp4_rows.restype = None
        lib.orc_nvfp4_rows.argtypes = [i64, i64, vp, vp, vp, vp]
        lib.orc_shared_sf_row.restype = i64
        lib.orc_shared_sf_row.argtypes = [i64, i64]
        lib.orc_shared_sf.restype = None
        lib.orc_shared_sf.argtypes = [i64, i64, vp, i64, vp, i64, i64]
        lib.orc_dispatch_contiguous.restype = i32
        lib.orc_dispatch_contiguous.argtypes = [i64, i64, i64, vp, vp, vp, i64, i64, vp, vp, vp,
                                                vp, vp]
        lib.orc_dispatch.restype = i32
        lib.orc_dispatch.argtypes = [i64, i64, i64, vp, vp, vp, i64, i64, i64, vp, vp, vp, vp]
        lib.orc_w13_rows.restype = None
        lib.orc_w13_rows.argtypes = [i64, vp, i64, i64, i64, vp, vp, vp, vp, vp, vp, vp, vp, i32]
        lib.orc_silu_requant_rows.restype = None
        lib.orc_silu_requant_rows.argtypes = [i64, vp, i64, vp, vp, vp]
        lib.orc_w2_rows.restype = None
        lib.orc_w2_rows.argtypes = [i64, vp, i64, i64, i64, vp, vp, vp, vp, vp, vp]
        lib.orc_topk_reduce.restype = None
        lib.orc_topk_reduce.argtypes = [i64, i64, i64, i64, vp, vp, vp, vp, vp, i64]
        _lib = lib
        return lib


def _p(a):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def _sf_words(a):
    """Scale rows as 4-byte words: packed UE8M0 int32 as is, fp32 bit patterns."""
    a = np.asarray(a)
    if a.dtype == np.float32:
        return np.ascontiguousarray(a).view(np.int32)
    return _c(a, np.int32)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def num_threads() -> int:
    return _load().orc_num_threads()


# --------------------------------------------------------------------------- S1
def e4m3_encode(v: float) -> int:
    return int(_load().orc_e4m3_encode(float(v)))


def e4m3_decode(code: int) -> float:
    return float(_load().orc_e4m3_decode(int(code) & 0xFF))


def e4m3_decode_table() -> np.ndarray:
    """fp32 value of each of the 256 codes (NaN for 0x7F / 0xFF)."""
    return np.array([e4m3_decode(c) for c in range(256)], dtype=np.float32)


def e4m3_encode_array(v: np.ndarray) -> np.ndarray:
    lib = _load()
    flat = np.asarray(v, dtype=np.float32).ravel()
    return np.array([lib.orc_e4m3_encode(float(x)) for x in flat], dtype=np.uint8).reshape(
        np.shape(v))


def bf16_from_f64(v: float) -> int:
    return int(_load().orc_bf16_from_f64(float(v)))


# --------------------------------------------------------------------------- S2
def group_scale(amax: float, ue8m0: bool = True):
    """Return (code, qs): UE8M0 exponent byte (or fp32 bits) and the quant scale."""
    code = ctypes.c_uint32()
    qs = ctypes.c_float()
    _load().orc_group_scale(float(amax), 1 if ue8m0 else 0, ctypes.byref(code), ctypes.byref(qs))
    return int(code.value), float(qs.value)


# ----------------------------------------------------------------------- S1-S5
def prepare_inputs(hidden_bf16_bits, topk_ids, topk_weights, is_padding=None, sf_mode=1,
                   l2p=None, replica_count=None, num_physical=0, record_enabled=False,
                   num_unpadded=None):
    """Token-order staging.  Returns dict(x, x_sf, ids, weights, load)."""
    lib = _load()
    hidden = _c(hidden_bf16_bits, np.uint16)
    T, K = hidden.shape
    ids_is_64 = np.asarray(topk_ids).dtype == np.int64
    ids = _c(topk_ids, np.int64 if ids_is_64 else np.int32)
    top_k = ids.shape[1] if ids.ndim == 2 else 0
    w = _c(topk_weights, np.float32)
    pad = None if is_padding is None else _c(is_padding, np.uint8)
    G = K // 128
    x = np.zeros((T, K), np.uint8)
    x_sf = (np.zeros((T, (G + 3) // 4), np.int32) if sf_mode == 1
            else np.zeros((T, G), np.float32))
    ids_out = np.zeros((T, top_k), np.int64)
    w_out = np.zeros((T, top_k), np.float32)
    l2p_c = None if l2p is None else _c(l2p, np.int32)
    rc = None if replica_count is None else _c(replica_count, np.int32)
    load = np.zeros(max(int(num_physical), 1), np.int32) if l2p is not None else None
    st = lib.orc_prepare_inputs(
        T, K, top_k, _p(hidden), _p(ids), int(ids_is_64), _p(w), _p(pad), int(sf_mode),
        _p(x), _p(x_sf), _p(ids_out), _p(w_out), _p(l2p_c),
        0 if l2p_c is None else l2p_c.shape[0], 0 if l2p_c is None else l2p_c.shape[1],
        _p(rc), _p(load), int(num_physical), int(bool(record_enabled)),
        T if num_unpadded is None else int(num_unpadded))
    if st != 0:
        raise ValueError(f"oracle staging rejected the shapes (status {st})")
    return dict(x=x, x_sf=x_sf, ids=ids_out, weights=w_out,
                load=None if load is None else load[:int(num_physical)])


# --------------------------------------------------------------------------- S6
def e2m1_encode(v: float) -> int:
    return int(_load().orc_e2m1_encode(float(v)))


def e2m1_decode(code: int) -> float:
    return float(_load().orc_e2m1_decode(int(code)))


def nvfp4_rows(hidden_bf16_bits):
    """NVFP4 staging of token rows (N2).  Returns dict(x [T, K/2] uint8,
    x_sf [T, K/64] int32 of packed E4M3 block scales, x_scales [T] fp32)."""
    lib = _load()
    hidden = _c(hidden_bf16_bits, np.uint16)
    T, K = hidden.shape
    x = np.zeros((T, K // 2), np.uint8)
    x_sf = np.zeros((T, (K // 16 + 3) // 4), np.int32)
    xs = np.zeros(T, np.float32)
    lib.orc_nvfp4_rows(T, K, _p(hidden), _p(x), _p(x_sf), _p(xs))
    return dict(x=x, x_sf=x_sf, x_scales=xs)


def shared_sf_row(t: int, block_m: int) -> int:
    """Row of token t in the shared-expert scale pages (S4b)."""
    return int(_load().orc_shared_sf_row(int(t), int(block_m)))


def shared_sf(x_sf_words, K: int, block_m: int, rows: int | None = None, fill: int = 0xEE):
    """Shared-expert scale pages of token-order packed exponents (S4b).

    Returns uint8 [rows, K/128]; rows that no token maps to keep ``fill``.
    """
    lib = _load()
    words = _c(x_sf_words, np.int32)
    T = words.shape[0]
    G = K // 128
    padded = (block_m + 127) // 128 * 128
    need = (T + block_m - 1) // block_m * padded
    rows = need if rows is None else rows
    out = np.full((rows, G), fill, np.uint8)
    lib.orc_shared_sf(T, G, _p(words), int(block_m), _p(out), G, 1)
    return out


def dispatch(ids, x, x_sf_words, E, M_max, copy_rows=True):
    """Batched layout.  Returns dict(expert_num_tokens, route_slot, x_b, sf_b, status)."""
    lib = _load()
    ids = _c(ids, np.int64)
    T, top_k = ids.shape
    x = _c(x, np.uint8)
    K = x.shape[1]
    sfw = _sf_words(x_sf_words)
    W = sfw.shape[1]
    ent = np.zeros(E, np.int32)
    slot = np.zeros((T, top_k), np.int32)
    x_b = np.zeros((E * M_max, K), np.uint8) if copy_rows else None
    sf_b = np.zeros((E * M_max, W), np.int32) if copy_rows else None
    st = lib.orc_dispatch(T, top_k, K, _p(ids), _p(x), _p(sfw), W, E, M_max, _p(ent), _p(slot),
                          _p(x_b), _p(sf_b))
    if sf_b is not None and np.asarray(x_sf_words).dtype == np.float32:
        sf_b = sf_b.view(np.float32)
    return dict(expert_num_tokens=ent, route_slot=slot, x_b=x_b, sf_b=sf_b, status=int(st))


def dispatch_contiguous(ids, x, x_sf_words, E):
    """Contiguous layout (S6b).  Returns dict(expert_offsets, expert_num_tokens,
    route_row, x_c, sf_c, row_expert, status); x_c / sf_c have T*k rows."""
    lib = _load()
    ids = _c(ids, np.int64)
    T, top_k = ids.shape
    x = _c(x, np.uint8)
    K = x.shape[1]
    sfw = _sf_words(x_sf_words)
    W = sfw.shape[1]
    offs = np.zeros(E + 1, np.int32)
    ent = np.zeros(E, np.int32)
    row = np.zeros((T, top_k), np.int32)
    x_c = np.zeros((max(T * top_k, 1), K), np.uint8)
    sf_c = np.zeros((max(T * top_k, 1), W), np.int32)
    st = lib.orc_dispatch_contiguous(T, top_k, K, _p(ids), _p(x), _p(sfw), W, E, _p(offs),
                                     _p(ent), _p(row), _p(x_c), _p(sf_c))
    if np.asarray(x_sf_words).dtype == np.float32:
        sf_c = sf_c.view(np.float32)
    row_expert = np.repeat(np.arange(E, dtype=np.int64), ent)
    return dict(expert_offsets=offs, expert_num_tokens=ent, route_row=row, x_c=x_c, sf_c=sf_c,
                row_expert=row_expert, status=int(st))


# --------------------------------------------------------------------------- S7
def valid_rows(expert_num_tokens, M_max):
    ent = np.asarray(expert_num_tokens)
    return np.concatenate([np.arange(n, dtype=np.int64) + e * M_max
                           for e, n in enumerate(ent)] + [np.zeros(0, np.int64)])


def w13_rows(rows, M_max, K, N, x_b, a_sf, w13, w13_s, want_h=False, row_expert=None):
    """(a_sf: packed UE8M0 int32 words, or fp32 scales [rows, K/128])"""
    return _w13_rows(rows, M_max, K, N, x_b, a_sf, w13, w13_s, want_h, row_expert)


def _w13_rows(rows, M_max, K, N, x_b, a_sf, w13, w13_s, want_h, row_expert):
    """w13 GEMM + SiLU-and-mul + requant for the given global rows.

    Returns (h, y_q, y_sf) as full-size arrays [E*M_max, .]; only `rows` are set.
    row_expert: expert of each row (contiguous layout); None = row // M_max.
    """
    lib = _load()
    rows = _c(rows, np.int64)
    x_b = _c(x_b, np.uint8)
    R = x_b.shape[0]
    a_fp32 = int(np.asarray(a_sf).dtype == np.float32)
    a_sf = _sf_words(a_sf)
    w13 = _c(w13, np.uint8)
    w13_s = _c(w13_s, np.float32)
    Gn = N // 128
    h = np.zeros((R, 2 * N), np.uint16) if want_h else None
    y_q = np.zeros((R, N), np.uint8)
    y_sf = np.zeros((R, (Gn + 3) // 4), np.int32)
    re = None if row_expert is None else _c(row_expert, np.int64)
    lib.orc_w13_rows(rows.size, _p(rows), M_max, K, N, _p(x_b), _p(a_sf), _p(w13), _p(w13_s),
                     _p(h), _p(y_q), _p(y_sf), _p(re), a_fp32)
    return h, y_q, y_sf


def silu_requant_rows(rows, N, h_bits):
    """SiLU-and-mul + 1x128 UE8M0 requant of given bf16 h rows [R, 2N]."""
    lib = _load()
    rows = _c(rows, np.int64)
    h = _c(h_bits, np.uint16)
    R = h.shape[0]
    y_q = np.zeros((R, N), np.uint8)
    y_sf = np.zeros((R, (N // 128 + 3) // 4), np.int32)
    lib.orc_silu_requant_rows(rows.size, _p(rows), N, _p(h), _p(y_q), _p(y_sf))
    return y_q, y_sf


def w2_rows(rows, M_max, K, N, y_q, y_sf, w2, w2_s, row_expert=None):
    """w2 GEMM for the given global rows; returns bf16 bits [E*M_max, K].

    row_expert: expert of each row (contiguous layout); None = row // M_max.
    """
    lib = _load()
    rows = _c(rows, np.int64)
    y_q = _c(y_q, np.uint8)
    y_sf = _c(y_sf, np.int32)
    w2 = _c(w2, np.uint8)
    w2_s = _c(w2_s, np.float32)
    out_b = np.zeros((y_q.shape[0], K), np.uint16)
    re = None if row_expert is None else _c(row_expert, np.int64)
    lib.orc_w2_rows(rows.size, _p(rows), M_max, K, N, _p(y_q), _p(y_sf), _p(w2), _p(w2_s),
                    _p(out_b), _p(re))
    return out_b


# --------------------------------------------------------------------------- S8
def topk_reduce(out_b_bits, ids, route_slot, weights, M_max, num_valid=None, fill=0):
    """S8.  ids None: route_slot holds the rows (contiguous layout).

    num_valid: rows t >= num_valid are not written (they keep ``fill``);
    None = every token."""
    lib = _load()
    out_b = _c(out_b_bits, np.uint16)
    ids = None if ids is None else _c(ids, np.int64)
    slot = _c(route_slot, np.int32)
    w = _c(weights, np.float32)
    T, top_k = slot.shape
    K = out_b.shape[-1]
    out = np.full((T, K), fill, np.uint16)
    lib.orc_topk_reduce(T, top_k, K, M_max, _p(out_b), _p(ids), _p(slot), _p(w), _p(out),
                        -1 if num_valid is None else int(num_valid))
    return out


# ----------------------------------------------------------------- whole path
def forward(hidden_bf16_bits, topk_ids, topk_weights, w13, w13_s, w2, w2_s, E, M_max, N,
            is_padding=None, eplb=None, rows=None, want_h=False):
    """S1-S8 end to end.  `rows` (global batched rows) restricts S7; default all."""
    K = hidden_bf16_bits.shape[1]
    eplb = eplb or {}
    st = prepare_inputs(hidden_bf16_bits, topk_ids, topk_weights, is_padding=is_padding,
                        sf_mode=1, **eplb)
    d = dispatch(st["ids"], st["x"], st["x_sf"], E, M_max)
    if rows is None:
        rows = valid_rows(d["expert_num_tokens"], M_max)
    h, y_q, y_sf = w13_rows(rows, M_max, K, N, d["x_b"], d["sf_b"], w13, w13_s, want_h=want_h)
    out_b = w2_rows(rows, M_max, K, N, y_q, y_sf, w2, w2_s)
    out = topk_reduce(out_b, st["ids"], d["route_slot"], st["weights"], M_max)
    return dict(staging=st, dispatch=d, rows=rows, h=h, y_q=y_q, y_sf=y_sf, out_b=out_b,
                out=out)


def sampled_forward(hidden_bits, topk_ids, topk_weights, is_padding, E, M_max, N, tokens,
                    weights_of, want_h=False, timings=None):
    """S1-S8 for a sample of tokens of a full-size workload.

    Routing and dispatch run over every token (so the slots are the full
    problem's); quantisation and the expert GEMMs run only for the sampled
    tokens' routes, on a compact copy of the experts they touch, fetched with
    ``weights_of(experts) -> (w13, w13_s, w2, w2_s)``.  ``timings`` (a dict)
    receives the wall time of the arithmetic and the FLOPs it covered.
    """
    import time
    T, K = hidden_bits.shape
    k = topk_ids.shape[1]
    tokens = np.asarray(tokens, np.int64)
    st_all = prepare_inputs(np.zeros((T, 128), np.uint16), topk_ids, topk_weights,
                            is_padding=is_padding)
    d = dispatch(st_all["ids"], np.zeros((T, 128), np.uint8), np.zeros((T, 1), np.int32),
                 E, M_max, copy_rows=False)
    routes = []
    for i, t in enumerate(tokens):
        for j in range(k):
            e, s = int(st_all["ids"][t, j]), int(d["route_slot"][t, j])
            if e >= 0 and s >= 0:
                routes.append((i, j, e, s))
    experts = sorted({r[2] for r in routes})
    w13, w13_s, w2, w2_s = weights_of(experts) if experts else (None,) * 4
    t0 = time.perf_counter()
    st = prepare_inputs(hidden_bits[tokens], topk_ids[tokens], topk_weights[tokens],
                        is_padding=None if is_padding is None else is_padding[tokens])
    cidx = {e: n for n, e in enumerate(experts)}
    counts = {}
    for r in routes:
        counts[r[2]] = counts.get(r[2], 0) + 1
    Mc = max([1] + list(counts.values()))
    W = st["x_sf"].shape[1]
    nE = max(len(experts), 1)
    x_b = np.zeros((nE * Mc, K), np.uint8)
    sf_b = np.zeros((nE * Mc, W), np.int32)
    cids = np.full((len(tokens), k), -1, np.int64)
    cslot = np.full((len(tokens), k), -1, np.int32)
    crow_of = {}
    per = {}
    for (i, j, e, s) in routes:
        n = per.get(e, 0)
        per[e] = n + 1
        r = cidx[e] * Mc + n
        x_b[r] = st["x"][i]
        sf_b[r] = st["x_sf"][i]
        cids[i, j] = cidx[e]
        cslot[i, j] = n
        crow_of[(i, j)] = r
    rows = np.array(sorted(crow_of.values()), np.int64)
    if rows.size:
        h, y_q, y_sf = w13_rows(rows, Mc, K, N, x_b, sf_b, w13, w13_s, want_h=want_h)
        out_b = w2_rows(rows, Mc, K, N, y_q, y_sf, w2, w2_s)
    else:
        h = y_q = y_sf = None
        out_b = np.zeros((nE * Mc, K), np.uint16)
    out = topk_reduce(out_b, cids, cslot, st["weights"], Mc)
    if timings is not None:
        timings["seconds"] = time.perf_counter() - t0
        timings["flops"] = 6.0 * N * K * len(routes)
        timings["routes"] = len(routes)
    return dict(out=out, routes=routes, crow_of=crow_of, h=h, y_q=y_q, y_sf=y_sf, out_b=out_b,
                dispatch=d, ids=st_all["ids"], staging=st)
