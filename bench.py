#!/usr/bin/env python
"""Benchmark of the batched grouped-masked block-FP8 MoE expert layer on GB300.

One step = the whole path over one batch of synthetic input:
moe_prepare_inputs (staging + dispatch) -> moe_batched_experts (w13 GEMM with
fused SiLU-and-mul requant, w2 GEMM) -> moe_topk_reduce.  The headline
workload is the largest single-GPU configuration, the DeepSeek-V3-shaped
prefill layer (T=8192, K=7168, N=2048, E=256, top-8, M_max=1024); the same
JSON line carries a ``per_config`` block with the Mixtral-8x7B-shaped decode,
the DeepSeek-V3-shaped decode and the staging-only stress workload (fp8 and
NVFP4 staging), each with its own time, roofline, end-to-end figure and clocks.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--config NAME] [--no-per-config]

Prints one JSON line.  `value` is TFLOP/s over valid (routed) rows; the
staging-only workload reports GB/s instead.  Multi-GPU runs (torchrun) are
independent replicas (weak scaling, no collective on the data path).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE expert-layer TFLOP/s (valid rows) & staging GB/s, % of FP8/HBM roofline, 1 GB300"
FP8_OVER_BF16 = 2.0  # nominal dense fp8 / bf16 tensor ratio (4.5 / 2.25 PFLOP/s)
FLUSH_BYTES = 512 << 20  # > 129 MB L2
L2_NOTE = "inputs larger than L2 and a 512 MB L2 flush before every step"
HEADLINE = "deepseek_prefill"
# the other workloads measured in the same run: (workload, staging format)
PER_CONFIG = [("mixtral_decode", "fp8"), ("deepseek_decode", "fp8"),
              ("staging_stress", "fp8"), ("staging_stress", "nvfp4")]


# DRAM traffic per launch (dram__bytes_read.sum + dram__bytes_write.sum) of the
# dominant kernel, from one ncu capture of the committed source; each entry
# keeps the SHA-256 prefix of the code (comments excluded) of the kernel's
# source file together with the shared device header, and is reported only
# while both are unchanged.  The
# prefill entry is captured on deepseek_prefill_e32 (same rows per expert, 1/8
# of the experts) and scaled by 8.
GEMM_SRC = "moe_expert_layer_prepare_gb300/csrc/experts_gemm.cu"
STAGING_SRC = "moe_expert_layer_prepare_gb300/csrc/staging.cu"
COMMON_SRC = "moe_expert_layer_prepare_gb300/csrc/common.cuh"
NCU_TRAFFIC = {
    ("mixtral_decode", "grouped_gemm_kernel<W13>"): (945.67e6, GEMM_SRC, "ee740f19ec2b65ed"),
    ("deepseek_decode", "grouped_gemm_kernel<W13>"): (2023.44e6, GEMM_SRC, "ee740f19ec2b65ed"),
    ("deepseek_prefill", "grouped_gemm_kernel<W13>"): (8 * 1159.99e6, GEMM_SRC,
                                                       "ee740f19ec2b65ed"),
    ("staging_stress", "quant_ring_kernel<UE8M0,repack>"): (316.96e6, STAGING_SRC,
                                                            "77a3e2abe55e3692"),
    ("staging_stress", "nvfp4_ring_kernel"): (279.43e6, STAGING_SRC, "77a3e2abe55e3692"),
}


def _code_of(text):
    """The C++ code of a source file without its comments and blank space:
    a comment edit leaves the kernels, and so their counters, as they were."""
    import re
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def source_key(src):
    """SHA-256 prefix of the code of a kernel source file and of the shared
    device header (comments and white space excluded)."""
    h = hashlib.sha256()
    for f in (src, COMMON_SRC):
        with open(os.path.join(ROOT, f), encoding="utf-8") as fh:
            h.update(_code_of(fh.read()).encode())
    return h.hexdigest()[:16]


def ncu_traffic(workload, kernel):
    ent = NCU_TRAFFIC.get((workload, kernel))
    if ent is None:
        return None
    nbytes, src, sha = ent
    return int(nbytes) if source_key(src) == sha else None


def parse(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default=HEADLINE)
    ap.add_argument("--no-per-config", action="store_true",
                    help="measure the --config workload only")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--soak-seconds", type=float, default=1.0)
    ap.add_argument("--stage-format", default="fp8", choices=["fp8", "nvfp4"],
                    help="staging_stress: 1x128 UE8M0 fp8 staging or NVFP4 token staging")
    ap.add_argument("--layout", default="batched", choices=["batched", "contiguous"],
                    help="expert row layout: [E, M_max] slots or expert_offsets")
    ap.add_argument("--act-scales", default="ue8m0", choices=["ue8m0", "fp32"],
                    help="expert layers: 1x128 activation scales as packed UE8M0 or fp32")
    ap.add_argument("--shared-block-m", type=int, default=0,
                    help="staging_stress: also write the shared-expert scale pages of this "
                         "block size (NVFP4: the MXFP8 shared input, fp8 rows + pages)")
    return ap.parse_args(argv)


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        if args.impl == "ours":
            torch.cuda.set_device(local)
        dist.init_process_group("nccl" if args.impl == "ours" else "gloo")
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(world, v):
    if world <= 1:
        return v
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return dict(hbm=d["hbm_gbs"], bf16=d["bf16_tflops"],
                    bf16_sus=d.get("bf16_tflops_sustained", d["bf16_tflops"]), src="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sus=1700.0, src="fallback")


# ----------------------------------------------------------------- clocks
class ClockSampler:
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.proc = None
        self.idx = device_index
        try:
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            self.sel = ["-i", uuid if uuid.startswith("GPU-") else "GPU-" + uuid]
        except Exception:
            self.sel = ["-i", str(device_index)]

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", *self.sel, f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return dict(sm_mhz=None, sm_max_mhz=None, reasons=["nvidia-smi unavailable"])
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out = ""
        rows = [r.split(",") for r in out.strip().splitlines() if r.count(",") >= 8]
        if not rows:
            return dict(sm_mhz=None, sm_max_mhz=None, reasons=["no samples"], samples=0)
        sm = [float(r[1]) for r in rows if r[1].strip().replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].strip().replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4)
                          if r[5 + i].strip().lower() == "active"})
        pw = [float(r[3]) for r in rows if r[3].strip().replace(".", "").isdigit()]
        return dict(sm_mhz=statistics.median(sm) if sm else None,
                    sm_max_mhz=max(mx) if mx else None, reasons=reasons, samples=len(rows),
                    power_w_max=max(pw) if pw else None)


# ----------------------------------------------------------------- workload
def build_workload(name, device, with_weights=True):
    from moe_expert_layer_prepare_gb300 import synthetic as syn
    return syn.make_workload(name, weights_device=device, with_weights=with_weights)


def routing_counts(wl):
    c = wl["cfg"]
    ids = wl["topk_ids"].cpu().numpy()
    pad = wl["is_padding"].cpu().numpy().astype(bool)
    routed = ids[~pad]
    return int(routed.size), int(np.unique(routed).size)


def algorithmic(wl, fp32_scales=False):
    """Valid-row FLOPs and algorithmic bytes per kernel.

    FLOPs count routed rows only (6*N*K per route: 4*N*K in w13, 2*N*K in w2).
    Bytes count each kernel's compulsory traffic: the weights and block scales
    of the experts with at least one route, the routed activation rows and
    scales read, and the outputs written.
    """
    c = wl["cfg"]
    T, K, N, E, k = c["T"], c["K"], c["N"], c["E"], c["top_k"]
    R, A = routing_counts(wl)
    G, Gn = K // 128, N // 128
    Wa, Wy = (G + 3) // 4, (Gn + 3) // 4
    Sa = 4 * G if fp32_scales else 4 * Wa  # one row's activation scale bytes
    w13_bytes = A * (2 * N * K + (2 * N // 128) * G * 4) + R * (K + Sa) + R * (N + Gn) + 4 * E
    w2_bytes = A * (K * N + (K // 128) * Gn * 4) + R * (N + 4 * Wy) + R * K * 2 + 4 * E
    stage_bytes = T * K * 2 + T * k * 8 + T + T * K + T * Sa + T * k * 8 + T * k * 4 + \
        R * (K + Sa) + R * 4 + E * 4
    reduce_bytes = R * K * 2 + T * K * 2 + T * k * (8 + 4 + 4)
    return dict(R=R, A=A, flops=6.0 * N * K * R, w13_bytes=w13_bytes, w2_bytes=w2_bytes,
                stage_bytes=stage_bytes, reduce_bytes=reduce_bytes,
                w13_flops=4.0 * N * K * R, w2_flops=2.0 * N * K * R)


def kernels_per_step(c):
    """Library kernels one expert-layer step launches: a batch of at most 1024
    routes (and fewer than 1024 tokens) stages and dispatches in one launch,
    a longer one routes first and then quantises; then w13, w2, reduce."""
    R = c["T"] * c["top_k"]
    small = R <= 1024 and c["T"] < 1024 and c["E"] * c["M_max"] < (1 << 31)
    return (1 if small else 2) + 3


def config_of(name, wl, layout, stage_format, world, args=None):
    """The `config` object of a JSON line; both arms build it here, so that a
    workload is named identically whichever arm measured it.  Options that
    change the work (fp32 activation scales, shared-expert pages) are named
    in it when set."""
    c = wl["cfg"]
    if c.get("N") is None:
        out = dict(workload=name, format=stage_format, T=c["T"], K=c["K"], top_k=c["top_k"],
                   experts_logical=c["E"], experts_physical=wl["num_physical"], l2=L2_NOTE,
                   parallelism=f"replicas x{world}")
        if args is not None and args.shared_block_m > 0:
            out["shared_block_m"] = args.shared_block_m
        return out
    R, A = routing_counts(wl)
    M_max = max(1, -(-(c["T"] * c["top_k"]) // c["E"])) if layout == "contiguous" else c["M_max"]
    out = dict(workload=name, T=c["T"], K=c["K"], N=c["N"], E=c["E"], top_k=c["top_k"],
               M_max=M_max, layout=layout, routed_rows=R, active_experts=A, l2=L2_NOTE,
               parallelism=f"replicas x{world}")
    if args is not None and args.act_scales != "ue8m0":
        out["act_scales"] = args.act_scales
    return out


def median(xs):
    return float(np.median(np.asarray(xs, dtype=np.float64)))


# ----------------------------------------------------------------- oracle legs
def _weights_fetcher(wl, cfg_name):
    """weights_of(experts) for the oracle: the experts' weights as host arrays,
    from the resident workload tensors when present, else drawn on demand
    (each expert from its own seeded generator, as in the full set)."""
    from moe_expert_layer_prepare_gb300 import synthetic as syn
    c = wl["cfg"]

    def weights_of(experts):
        if "w13" in wl:
            sel = torch.as_tensor(np.asarray(experts, np.int64))
            return tuple(np.ascontiguousarray(wl[n][sel.to(wl[n].device)].cpu().numpy())
                         for n in ("w13", "w13_s", "w2", "w2_s"))
        dev = "cuda" if torch.cuda.is_available() else "cpu"
        w13, w13_s = syn.make_block_fp8_weights(c["E"], 2 * c["N"], c["K"],
                                                syn.seed_of(cfg_name, 2), dev, experts=experts)
        w2, w2_s = syn.make_block_fp8_weights(c["E"], c["K"], c["N"], syn.seed_of(cfg_name, 3),
                                              dev, experts=experts)
        return tuple(np.ascontiguousarray(t.cpu().numpy()) for t in (w13, w13_s, w2, w2_s))
    return weights_of


def run_oracle_sample(wl, cfg_name, n_tok, seed=0):
    import oracle
    oracle.build()
    c = wl["cfg"]
    rng = np.random.default_rng(seed)
    pad = wl["is_padding"].cpu().numpy()
    cand = np.nonzero(pad == 0)[0]
    tokens = np.sort(rng.choice(cand, size=min(n_tok, cand.size), replace=False))
    bits = wl["hidden"].view(torch.int16).numpy().view(np.uint16)
    tm = {}
    oracle.sampled_forward(bits, wl["topk_ids"].numpy(), wl["topk_weights"].numpy(), pad,
                           c["E"], c["M_max"], c["N"], tokens, _weights_fetcher(wl, cfg_name),
                           timings=tm)
    return tm, oracle.num_threads(), len(tokens)


def run_oracle_staging(wl, n_tok):
    """Oracle staging (quantise + repack + EPLB record) of the first n_tok tokens."""
    import oracle
    oracle.build()
    c = wl["cfg"]
    n = max(1, min(int(n_tok), c["T"]))
    bits = wl["hidden"][:n].view(torch.int16).numpy().view(np.uint16)
    t0 = time.perf_counter()
    oracle.prepare_inputs(bits, wl["topk_ids"][:n].numpy(), wl["topk_weights"][:n].numpy(),
                          None, 1, wl["l2p"].numpy(), wl["replica_count"].numpy(),
                          wl["num_physical"], True, n)
    secs = time.perf_counter() - t0
    return secs, oracle.num_threads(), n


def run_oracle_nvfp4(wl, n_tok):
    import oracle
    oracle.build()
    K = wl["cfg"]["K"]
    n = max(1, min(int(n_tok), wl["cfg"]["T"]))
    bits = wl["hidden"][:n].view(torch.int16).numpy().view(np.uint16)
    t0 = time.perf_counter()
    oracle.nvfp4_rows(bits)
    return time.perf_counter() - t0, oracle.num_threads(), n


def staging_bytes(T, K, k, wl, nvfp4=False, shared_pages=False):
    G = K // 128
    b = T * K * 2 + T * k * 4 * 2 + T * K + T * 4 * ((G + 3) // 4) + T * k * 12 + \
        wl["l2p"].numel() * 4 + wl["replica_count"].numel() * 4
    if nvfp4:  # codes K/2 + E4M3 scales K/16 + fp32 scale, instead of K + K/32
        b += T * (K // 2 + K // 16 + 4) - T * (K + 4 * ((G + 3) // 4))
    if shared_pages:  # one exponent byte per group; NVFP4 also writes the fp8 rows
        b += T * G + (T * K if nvfp4 else 0)
    return b


def oracle_tokens_for(wl, seconds):
    """Token sample size for about `seconds` of oracle wall time (estimate)."""
    c = wl["cfg"]
    per_route = 6.0 * c["N"] * c["K"]
    import oracle
    thr = max(oracle.num_threads(), 1)
    rate = 4.0e8 * thr  # oracle fp64 FLOP/s per thread (measured: ~5e8 on Grace cores)
    routes = max(1, int(seconds * rate / per_route))
    return max(1, routes // max(c["top_k"], 1))


# ----------------------------------------------------------------- ours
def timed_steps(step, K, s, nev, flush, world):
    """K steps, each bracketed by `nev` events (step(evs) records them), an L2
    flush before every step outside the events.  Returns [K, nev-1] ms."""
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(nev)] for _ in range(K)]
    barrier(world)
    torch.cuda.synchronize()
    for i in range(K):
        flush.zero_()
        step(evs[i])
    torch.cuda.synchronize()
    barrier(world)
    return np.array([[evs[i][j].elapsed_time(evs[i][j + 1]) for j in range(nev - 1)]
                     for i in range(K)])


def soak(step, flush, seconds):
    t_end = time.time() + seconds
    while time.time() < t_end:
        for _ in range(10):
            flush.zero_()
            step(None)
        torch.cuda.synchronize()


def bench_experts(name, args, world, dev, peaks, flush, want_cpu):
    """The whole path on one expert-layer workload."""
    from moe_expert_layer_prepare_gb300 import binding as B
    wl = build_workload(name, dev)
    c = wl["cfg"]
    s = torch.cuda.current_stream()
    fp32_scales = args.act_scales == "fp32"
    alg = algorithmic(wl, fp32_scales=fp32_scales)
    layer = B.MoeLayer(c["T"], c["K"], c["N"], c["E"], c["top_k"], c["M_max"], wl["w13"],
                       wl["w13_s"], wl["w2"], wl["w2_s"], device=dev,
                       contiguous=args.layout == "contiguous", fp32_scales=fp32_scales)
    hid, ids, wts, pad = (wl["hidden"].to(dev), wl["topk_ids"].to(dev),
                          wl["topk_weights"].to(dev), wl["is_padding"].to(dev))
    inter_q, inter_sf = layer.inter()

    def step(evs):
        if evs:
            evs[0].record(s)
        layer.prepare(hid, ids, wts, pad)
        if evs:
            evs[1].record(s)
        B.moe_batched_experts(layer.out_b, layer.x_b, layer.sf_b, layer.w13, layer.w13_s,
                              layer.w2, layer.w2_s, layer.expert_num_tokens, layer.ws13,
                              layer.ws2, valid_shape_m=layer.valid_shape_m,
                              stages=B.MOE_STAGE_W13, device_status=layer.status,
                              expert_offsets=layer.expert_offsets)
        if evs:
            evs[2].record(s)
        B.moe_batched_experts(layer.out_b, None, None, layer.w13, layer.w13_s, layer.w2,
                              layer.w2_s, layer.expert_num_tokens, layer.ws13, layer.ws2,
                              valid_shape_m=layer.valid_shape_m, inter_q=inter_q,
                              inter_sf=inter_sf, stages=B.MOE_STAGE_W2,
                              device_status=layer.status, expert_offsets=layer.expert_offsets)
        if evs:
            evs[3].record(s)
        layer.reduce()
        if evs:
            evs[4].record(s)

    for _ in range(max(args.warmup, 3)):
        step(None)
    torch.cuda.synchronize()
    assert int(layer.status.item()) == 0, "device status set during warm-up"
    clocks = ClockSampler(dev.index)
    clocks.start()
    soak(step, flush, args.soak_seconds)
    K = args.steps

    def whole_step(evs):
        if evs:
            evs[0].record(s)
        step(None)
        if evs:
            evs[1].record(s)

    # the step is timed whole (events around it only, so that nothing breaks
    # the chaining of its kernels); a second pass with events between the
    # calls gives the per-kernel breakdown and the dominant kernel's duration
    step_ms = timed_steps(whole_step, K, s, 2, flush, world)[:, 0]
    stage_ms = timed_steps(step, K, s, 5, flush, world)
    ck = clocks.stop()
    ms = max_over_ranks(world, median(step_ms))
    value = world * alg["flops"] / (ms * 1e-3) / 1e12
    med = np.median(stage_ms, axis=0)
    w13_gbs = alg["w13_bytes"] / (med[1] * 1e-3) / 1e9
    w13_tfs = alg["w13_flops"] / (med[1] * 1e-3) / 1e12
    if name == "deepseek_prefill":
        # tensor-bound: the w13 GEMM against the fp8 burst peak (it runs for
        # ~2 ms at a time near the boost clock); the fraction of the sustained
        # figure (a seconds-long GEMM loop at a lower clock) is kept beside it
        burst = peaks["bf16"] * FP8_OVER_BF16
        sus = peaks["bf16_sus"] * FP8_OVER_BF16
        roof = dict(bound="tensor", achieved=round(w13_tfs, 2), peak=round(burst, 1),
                    unit="TFLOP/s", frac=round(w13_tfs / burst, 4),
                    traffic=ncu_traffic(name, "grouped_gemm_kernel<W13>"),
                    kernel="grouped_gemm_kernel<W13>",
                    peak_source=f"{peaks['src']} bf16 burst x {FP8_OVER_BF16} (fp8/bf16 nominal)",
                    frac_of_sustained=round(w13_tfs / sus, 4), sustained_peak=round(sus, 1))
    else:
        roof = dict(bound="hbm", achieved=round(w13_gbs, 1), peak=peaks["hbm"], unit="GB/s",
                    frac=round(w13_gbs / peaks["hbm"], 4),
                    traffic=ncu_traffic(name, "grouped_gemm_kernel<W13>"),
                    kernel="grouped_gemm_kernel<W13>", peak_source=f"{peaks['src']} hbm_gbs")

    # end to end through the public API with pinned host buffers
    hh = wl["hidden"].pin_memory()
    ih = wl["topk_ids"].pin_memory()
    wh = wl["topk_weights"].pin_memory()
    ph = wl["is_padding"].pin_memory()
    oh = torch.empty((c["T"], c["K"]), dtype=torch.bfloat16).pin_memory()
    for _ in range(3):
        layer.forward_host(hh, ih, wh, ph, oh)
    torch.cuda.synchronize()

    def e2e_step(evs):
        if evs:
            evs[0].record(s)
        layer.forward_host(hh, ih, wh, ph, oh)
        if evs:
            evs[1].record(s)

    e2e = timed_steps(e2e_step, K, s, 2, flush, world)[:, 0]
    e2e_ms = max_over_ranks(world, median(e2e))
    h2d = hh.numel() * 2 + ih.numel() * ih.element_size() + wh.numel() * 4 + ph.numel()
    d2h = oh.numel() * 2
    assert int(layer.status.item()) == 0, "device status set during the timed steps"
    out = dict(value=round(value, 3), unit="TFLOP/s", ms_per_step=round(ms, 4),
               dtype="fp8e4m3 (fp32 accumulate)",
               config=config_of(name, wl, args.layout, "fp8", world, args), roofline=roof,
               stages_ms=dict(prepare=round(med[0], 4), w13=round(med[1], 4),
                              w2=round(med[2], 4), reduce=round(med[3], 4),
                              note="separate pass, events between the calls",
                              # what staging + reduce add to the chained step:
                              # the whole step less the two GEMMs' own times
                              prepare_reduce_in_step=round(ms - med[1] - med[2], 4)),
               stages_gbs=dict(prepare=round(alg["stage_bytes"] / med[0] / 1e6, 1),
                               w13=round(w13_gbs, 1),
                               w2=round(alg["w2_bytes"] / med[2] / 1e6, 1),
                               reduce=round(alg["reduce_bytes"] / med[3] / 1e6, 1)),
               stages_tflops=dict(w13=round(w13_tfs, 2),
                                  w2=round(alg["w2_flops"] / med[2] / 1e9, 2)),
               e2e=dict(value=round(world * alg["flops"] / (e2e_ms * 1e-3) / 1e12, 3),
                        unit="TFLOP/s", h2d_bytes_per_step=int(h2d), d2h_bytes_per_step=int(d2h),
                        ms_per_step=round(e2e_ms, 4)),
               gpu_launches=kernels_per_step(c) * K, clocks=ck)
    if want_cpu:
        n_tok = oracle_tokens_for(wl, 15.0)
        tm, thr, ntok = run_oracle_sample(wl, name, n_tok)
        out["cpu_baseline"] = dict(value=round(tm["flops"] / tm["seconds"] / 1e12, 6),
                                   unit="TFLOP/s", cores=thr, kind="oracle",
                                   sample=f"{ntok} tokens ({tm['routes']} routes) of {name}, "
                                          f"{tm['seconds']:.1f} s")
    del layer
    return out


def bench_staging(args, world, dev, peaks, flush, want_cpu, fmt):
    """staging_stress: moe_prepare_inputs (or its NVFP4 form) alone, with EPLB."""
    from moe_expert_layer_prepare_gb300 import binding as B
    wl = build_workload("staging_stress", dev)
    c = wl["cfg"]
    T, K, k = c["T"], c["K"], c["top_k"]
    G = K // 128
    nvfp4 = fmt == "nvfp4"
    hid = wl["hidden"].to(dev)
    ids, wts = wl["topk_ids"].to(dev), wl["topk_weights"].to(dev)
    if nvfp4:
        x = torch.empty((T, K // 2), dtype=torch.uint8, device=dev)
        x_sf = torch.empty((T, K // 64), dtype=torch.int32, device=dev)
        x_scales = torch.empty(T, dtype=torch.float32, device=dev)
    else:
        x = torch.empty((T, K), dtype=torch.uint8, device=dev)
        x_sf = torch.empty((T, (G + 3) // 4), dtype=torch.int32, device=dev)
    io = torch.empty((T, k), dtype=torch.int64, device=dev)
    wo = torch.empty((T, k), dtype=torch.float32, device=dev)
    load = torch.zeros(wl["num_physical"], dtype=torch.int32, device=dev)
    eplb = dict(logical_to_physical=wl["l2p"].to(dev), logical_replica_count=wl["replica_count"]
                .to(dev), expert_load=load, should_record=torch.ones(1, dtype=torch.uint8,
                                                                        device=dev),
                num_unpadded_tokens=torch.tensor([T], dtype=torch.int32, device=dev))
    s = torch.cuda.current_stream()
    # optional shared-expert pages (and, for NVFP4, the MXFP8 shared input)
    bm = args.shared_block_m
    pages = shared_q = None
    if bm > 0:
        rows = (T + bm - 1) // bm * ((bm + 127) // 128 * 128)
        pages = torch.empty((rows, G), dtype=torch.uint8, device=dev)
        if nvfp4:
            shared_q = torch.empty((T, K), dtype=torch.uint8, device=dev)

    def run():
        if nvfp4:
            B.moe_prepare_nvfp4_inputs(hid, ids, wts, x, x_sf, x_scales, io, wo, eplb=eplb,
                                       shared_x=shared_q, shared_x_sf=pages,
                                       shared_block_m=bm if bm > 0 else None)
        else:
            B.moe_prepare_inputs(hid, ids, wts, x, x_sf, io, wo, eplb=eplb, shared_x_sf=pages,
                                 shared_block_m=bm if bm > 0 else None)

    def step(evs):
        if evs:
            evs[0].record(s)
        run()
        if evs:
            evs[1].record(s)

    for _ in range(max(args.warmup, 3)):
        step(None)
    clocks = ClockSampler(dev.index)
    clocks.start()
    soak(step, flush, args.soak_seconds)
    Ks = args.steps
    t = timed_steps(step, Ks, s, 2, flush, world)[:, 0]
    ck = clocks.stop()
    ms = max_over_ranks(world, median(t))
    nbytes = staging_bytes(T, K, k, wl, nvfp4, shared_pages=bm > 0)
    gbs = world * nbytes / (ms * 1e-3) / 1e9
    kern = "nvfp4_ring_kernel" if nvfp4 else "quant_ring_kernel<UE8M0,repack>"
    out = dict(value=round(gbs, 1), unit="GB/s", ms_per_step=round(ms, 4),
               dtype="bf16->e2m1 (e4m3/16, fp32/token)" if nvfp4 else
               "bf16->fp8e4m3 (fp32 scale math)",
               config=config_of("staging_stress", wl, "batched", fmt, world, args),
               roofline=dict(bound="hbm", achieved=round(gbs / world, 1), peak=peaks["hbm"],
                             unit="GB/s", frac=round(gbs / world / peaks["hbm"], 4),
                             traffic=ncu_traffic("staging_stress", kern), kernel=kern,
                             peak_source=f"{peaks['src']} hbm_gbs"),
               gpu_launches=Ks, clocks=ck)
    # end to end: pinned host inputs in, staged outputs back to the host
    hh, ih, wh = (wl["hidden"].pin_memory(), wl["topk_ids"].pin_memory(),
                  wl["topk_weights"].pin_memory())
    xh = torch.empty(x.shape, dtype=x.dtype).pin_memory()
    sfh = torch.empty(x_sf.shape, dtype=x_sf.dtype).pin_memory()
    xsh = torch.empty(T, dtype=torch.float32).pin_memory() if nvfp4 else None
    ioh = torch.empty((T, k), dtype=torch.int64).pin_memory()
    woh = torch.empty((T, k), dtype=torch.float32).pin_memory()

    def e2e_step(evs):
        if evs:
            evs[0].record(s)
        hid.copy_(hh, non_blocking=True)
        ids.copy_(ih, non_blocking=True)
        wts.copy_(wh, non_blocking=True)
        run()
        xh.copy_(x, non_blocking=True)
        sfh.copy_(x_sf, non_blocking=True)
        if nvfp4:
            xsh.copy_(x_scales, non_blocking=True)
        ioh.copy_(io, non_blocking=True)
        woh.copy_(wo, non_blocking=True)
        if evs:
            evs[1].record(s)

    for _ in range(3):
        e2e_step(None)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(world, median(timed_steps(e2e_step, Ks, s, 2, flush, world)[:, 0]))
    h2d = hh.numel() * 2 + ih.numel() * ih.element_size() + wh.numel() * 4
    d2h = xh.numel() + sfh.numel() * 4 + ioh.numel() * 8 + woh.numel() * 4 + \
        (T * 4 if nvfp4 else 0)
    out["e2e"] = dict(value=round(world * nbytes / (e2e_ms * 1e-3) / 1e9, 1), unit="GB/s",
                      h2d_bytes_per_step=int(h2d), d2h_bytes_per_step=int(d2h),
                      ms_per_step=round(e2e_ms, 4))
    if want_cpu:
        if nvfp4:
            secs, thr, n = run_oracle_nvfp4(wl, 2048)
            nb = n * (K * 2 + K // 2 + K // 16 + 4)
            what = "NVFP4 rows"
        else:
            secs, thr, n = run_oracle_staging(wl, 2048)
            nb = staging_bytes(n, K, k, wl)
            what = "staging"
        out["cpu_baseline"] = dict(value=round(nb / secs / 1e9, 4), unit="GB/s", cores=thr,
                                   kind="oracle",
                                   sample=f"{what} of the first {n} tokens of staging_stress, "
                                          f"{secs:.1f} s")
    return out


def bench_one(name, fmt, args, world, dev, peaks, flush, want_cpu):
    from moe_expert_layer_prepare_gb300 import synthetic as syn
    if syn.CONFIGS[name].get("N") is None:
        r = bench_staging(args, world, dev, peaks, flush, want_cpu, fmt)
    else:
        r = bench_experts(name, args, world, dev, peaks, flush, want_cpu)
    torch.cuda.empty_cache()
    return r


def bench_ours(args, world, rank, local):
    from moe_expert_layer_prepare_gb300 import binding as B
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    B.load()
    peaks = load_peaks()
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    want_cpu = world == 1 and rank == 0 and not args.no_cpu_baseline
    head = bench_one(args.config, args.stage_format, args, world, dev, peaks, flush, want_cpu)
    out = dict(metric=METRIC, value=head.pop("value"), unit=head.pop("unit"), n_gpus=world,
               steps=args.steps, warmup=args.warmup, ms_per_step=head.pop("ms_per_step"),
               higher_is_better=True, scaling="weak", vs_baseline=None, dtype=head.pop("dtype"),
               data="synthetic", config=head.pop("config"))
    out.update(head)
    if not args.no_per_config:
        per = {}
        for name, fmt in PER_CONFIG:
            if name == args.config and fmt == args.stage_format:
                continue
            key = name if name != "staging_stress" else f"staging_stress_{fmt}"
            r = bench_one(name, fmt, args, world, dev, peaks, flush, False)
            r.pop("gpu_launches", None)
            per[key] = r
        out["per_config"] = per
    return out


# ----------------------------------------------------------------- reference
def bench_reference(args, world, rank):
    """The oracle as it stands on the host cores: each step a bounded sample."""
    if rank != 0:
        return None
    from moe_expert_layer_prepare_gb300 import synthetic as syn
    staging = syn.CONFIGS[args.config].get("N") is None
    # expert weights are drawn only for the experts a sample touches
    wl = build_workload(args.config, "cpu", with_weights=False)
    c = wl["cfg"]
    # each step is a bounded sample so that the whole run stays near 90 s
    per_step_s = max(0.05, min(2.0, 90.0 / max(args.steps + args.warmup, 1)))
    config = config_of(args.config, wl, args.layout, args.stage_format, world, args)
    if staging:
        return bench_reference_staging(args, world, wl, per_step_s, config)
    n_tok = oracle_tokens_for(wl, per_step_s)
    for _ in range(max(args.warmup, 0)):
        run_oracle_sample(wl, args.config, n_tok, seed=1)
    secs, flops = [], []
    thr = ntok = 0
    for i in range(args.steps):
        tm, thr, ntok = run_oracle_sample(wl, args.config, n_tok, seed=100 + i)
        secs.append(tm["seconds"])
        flops.append(tm["flops"])
    value = sum(flops) / sum(secs) / 1e12
    return dict(metric=METRIC, value=round(value, 6), unit="TFLOP/s", n_gpus=world,
                steps=args.steps, warmup=args.warmup, ms_per_step=round(1e3 * median(secs), 3),
                higher_is_better=True, scaling="weak", vs_baseline=None, dtype="fp64 (oracle)",
                data="synthetic", impl="reference", config=config,
                cpu_baseline=dict(kind="oracle", cores=thr, value=round(value, 6),
                                  sample=f"{ntok} tokens per step of {args.config}"),
                e2e=dict(value=round(value, 6), unit="TFLOP/s", h2d_bytes_per_step=0,
                         d2h_bytes_per_step=0))


def bench_reference_staging(args, world, wl, per_step_s, config):
    c = wl["cfg"]
    T, K, k = c["T"], c["K"], c["top_k"]
    nvfp4 = args.stage_format == "nvfp4"
    n_tok = max(1, int(per_step_s * 7000))  # oracle staging runs ~7000 tokens/s (8 threads)
    fn = run_oracle_nvfp4 if nvfp4 else run_oracle_staging
    for _ in range(max(args.warmup, 0)):
        fn(wl, n_tok)
    secs, nbytes = [], []
    thr = n = 0
    for _ in range(args.steps):
        sec, thr, n = fn(wl, n_tok)
        secs.append(sec)
        nbytes.append(n * (K * 2 + K // 2 + K // 16 + 4) if nvfp4 else
                      staging_bytes(n, K, k, wl))
    value = sum(nbytes) / sum(secs) / 1e9
    return dict(metric=METRIC, value=round(value, 4), unit="GB/s", n_gpus=world,
                steps=args.steps, warmup=args.warmup, ms_per_step=round(1e3 * median(secs), 3),
                higher_is_better=True, scaling="weak", vs_baseline=None,
                dtype="fp32 group math (oracle)", data="synthetic", impl="reference",
                config=config,
                cpu_baseline=dict(kind="oracle", cores=thr, value=round(value, 4),
                                  sample=f"first {n} tokens per step of staging_stress"),
                e2e=dict(value=round(value, 4), unit="GB/s", h2d_bytes_per_step=0,
                         d2h_bytes_per_step=0))


def main():
    args = parse()
    world, rank, local = dist_setup(args)
    if args.impl == "reference":
        out = bench_reference(args, world, rank)
    else:
        out = bench_ours(args, world, rank, local)
    if rank == 0 and out is not None:
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
