"""Benchmark of the MoE layer hot path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

One step = one pass of the whole layer over one batch of tokens:
route (logits + top-K + weights) -> permute -> grouped FFN (GEMM1 + SwiGLU,
GEMM2) -> combine, each through its C-ABI entry point, with CUDA events on the
launching stream between the stages.  `value` is tokens/s over the K timed
steps (inputs resident in HBM); `e2e` repeats the layer through the public
moe_layer_forward call with the token batch copied in from pinned host memory
and the output copied back inside the timed region.

The default workload is the largest configuration that fits one GPU: the
DeepSeek-V3-shaped layer at N=16384 tokens (D=7168, E=256, K=8,
D_ffn=2048, SwiGLU, sigmoid then renormalise over the top-8) with router
logits biased by the log of a Zipf(1.2) popularity, so that a few hot experts
own most rows and a long tail of experts owns a few each.  The other
workloads (synth.WORKLOADS: Mixtral-shaped and DeepSeek-V3-shaped prefill,
the Qwen3-shaped decode sweep, the tiny case) can be selected with
--workload.  Inputs are
seeded synthetic tensors (random-init weights).  Where the inputs (all expert
weights and the 8 token batches) exceed twice the L2 size, the expert weights
are streamed once per step and the token batch rotates over 8 distinct
tensors; smaller inputs (the tiny workload) are flushed out of L2 before each
timed step by writing a buffer of twice the L2 size between the steps' own
CUDA-event intervals.

Multi-GPU: the layer shards by tokens as independent replicas (one process per
GPU, each with its own batch and weights, no collective on the data path);
`value` is the sum over ranks, timed as the max over ranks.

--impl reference times the fp64 CPU oracle (the correctness reference) on the
host cores, on bounded token samples of the same workload.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from mixture_experts_layer_02_gb300 import synth  # noqa: E402

FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ----------------------------------------------------------------------------
# environment helpers
# ----------------------------------------------------------------------------
def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = os.environ.get("MOE_BENCH_BACKEND") or ("nccl" if torch.cuda.is_available() else "gloo")
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v: float, world: int) -> float:
    if world == 1:
        return v
    import torch.distributed as dist
    dev = torch.device("cuda") if dist.get_backend() == "nccl" else torch.device("cpu")
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,utilization.gpu,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, device_index: int, period_ms: int = 100):
        self.lines = []
        self.proc = None
        try:
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            ident = uuid if uuid.startswith("GPU-") else f"GPU-{uuid}"
        except Exception:
            ident = str(device_index)
        cmd = ["nvidia-smi", f"--id={ident}", f"--query-gpu={self.FIELDS}",
               "--format=csv,noheader,nounits", "-lms", str(period_ms)]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (FileNotFoundError, OSError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=2)

    def summary(self, t0=None, t1=None) -> dict:
        rows = []
        for ts, line in self.lines:
            if (t0 is not None and ts < t0) or (t1 is not None and ts > t1):
                continue
            parts = [p.strip() for p in line.split(",")]
            if len(parts) != 9:
                continue
            try:
                sm, smax, util = float(parts[0]), float(parts[1]), float(parts[3])
            except ValueError:
                continue
            rows.append((sm, smax, util, parts[5:]))
        load = [r for r in rows if r[2] >= 50] or rows
        if not load:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        reasons = sorted({name for r in load for name, v in zip(self.REASONS, r[3])
                          if v.lower().startswith("active")})
        return {"sm_mhz": statistics.median(r[0] for r in load), "sm_max_mhz": max(r[1] for r in load),
                "reasons": reasons, "samples": len(load)}


# ----------------------------------------------------------------------------
# algorithmic work of one step (what the method must do, no padding)
# ----------------------------------------------------------------------------
def work_model(wl, offsets, padded_rows=None, e4m3=False, fused=False):
    """Algorithmic work of one step.  In the padded paradigm the FFN runs on
    every row of the E*capacity buffer (its padding is part of the method).
    With e4m3 experts: weights and permuted tokens are one byte per value plus
    one fp32 scale per row; h is written in bf16, re-read and written again as
    e4m3 codes (its per-row scale needs the whole row) before GEMM2 reads it."""
    A = wl.N * wl.K if padded_rows is None else padded_rows
    counts = [offsets[e + 1] - offsets[e] for e in range(wl.E)]
    touched = sum(1 for c in counts if c > 0)
    nmat = 3 if wl.act == synth.ACT_SWIGLU else 2
    ffn_flop = A * wl.D * wl.Dff * (6 if wl.act == synth.ACT_SWIGLU else 4)
    if e4m3:
        ffn_w_bytes = touched * (nmat * wl.D * wl.Dff + ((nmat - 1) * wl.Dff + wl.D) * 4)
        ffn_act_bytes = (A * wl.D + A * 4                      # xq_perm + token scales
                         + 2 * A * wl.Dff * 2                  # h written, read by the quantiser
                         + 2 * A * wl.Dff + 2 * A * 4          # hq written and read, its scales
                         + A * wl.D * 2)                       # y_perm
        permute_bytes = (wl.N * wl.D * 2 + wl.N * wl.D + wl.N * 4   # token quantisation
                         + wl.N * wl.D + A * wl.D + A * 12)         # permutation of the codes
    else:
        ffn_w_bytes = touched * nmat * wl.D * wl.Dff * 2
        ffn_act_bytes = A * wl.D * 2 + 2 * A * wl.Dff * 2 + A * wl.D * 2
        permute_bytes = wl.N * wl.D * 2 + A * wl.D * 2 + A * 12
    if fused and padded_rows is None:
        # index-only permutation (ids in, offsets / perm_src / inv_perm out); the
        # rows are read by GEMM1 (counted in the FFN's x_perm read)
        permute_bytes = wl.N * wl.K * 4 + A * 8 + (wl.N * wl.D * 2 + wl.N * wl.D + wl.N * 4 if e4m3 else 0)
    # the whole layer in one launch (decode batches): x, W_gate, the touched
    # experts' weights and out, plus every intermediate it writes once
    # (ids and weights, offsets, perm_src / inv_perm, x_perm, h, y_perm)
    layer_bytes = (wl.N * wl.D * 2 + wl.E * wl.D * 2 + wl.N * wl.K * 8 + (wl.E + 1) * 4 + A * 8
                   + ffn_w_bytes + A * wl.Dff * 2 + A * wl.D * 2 + wl.N * wl.D * 2)
    if e4m3:  # token codes and scales, their permuted copy, h's codes and scales
        layer_bytes += wl.N * wl.D + wl.N * 4 + A * wl.D + A * wl.Dff + A * 4
    else:     # x_perm
        layer_bytes += A * wl.D * 2
    return dict(
        layer_bytes=layer_bytes,
        rows=A, touched_experts=touched, max_expert_share=max(counts) / A if A else 0.0,
        empty_experts=wl.E - touched,
        ffn_flop=ffn_flop, ffn_bytes=ffn_w_bytes + ffn_act_bytes,
        gemm1_flop=A * wl.D * wl.Dff * (4 if wl.act == synth.ACT_SWIGLU else 2),
        gemm2_flop=2 * A * wl.D * wl.Dff,
        route_bytes=wl.N * wl.D * 2 + wl.E * wl.D * 2 + wl.N * wl.K * 8,
        route_flop=2 * wl.N * wl.D * wl.E,
        permute_bytes=permute_bytes,
        combine_bytes=A * wl.D * 2 + wl.N * wl.D * 2 + A * 8,
    )


GEMM_SOURCES = ("grouped_gemm.cuh", "grouped_gemm_2sm.cuh", "grouped_gemm_swap.cuh", "gemm_common.cuh",
                "device.cuh", "quant.cu", "ffn_fused_decode.cu")
# the one-launch decode layer (entries keyed "<workload>:layer")
LAYER_SOURCES = ("layer_decode.cu", "route_common.cuh", "device.cuh", "common.h")


def tensor_digest(t):
    """sha256 of a tensor's bytes: all of them up to 256 MiB, else 64 slices of
    1 MiB at evenly spaced offsets (the method is recorded beside the hash)."""
    import hashlib
    b = t.detach().contiguous().view(-1).view(torch.uint8)
    n = b.numel()
    h = hashlib.sha256()
    if n <= (256 << 20):
        h.update(b.cpu().numpy().tobytes())
        how = "all bytes"
    else:
        sl = 1 << 20
        for i in range(64):
            o = (n - sl) * i // 63
            h.update(b[o:o + sl].cpu().numpy().tobytes())
        how = "64 slices of 1 MiB at evenly spaced offsets"
    return {"sha256": h.hexdigest(), "bytes": n, "hashed": how, "shape": list(t.shape), "dtype": str(t.dtype)}


def kernel_sources_sha(sources=GEMM_SOURCES) -> str:
    """Hash of kernel sources (by default the grouped-FFN kernels') with
    comments and blank lines removed: any change to their code changes it, an
    edited comment does not."""
    import hashlib
    import re
    h = hashlib.sha256()
    for name in sorted(sources):
        text = open(os.path.join(ROOT, "mixture_experts_layer_02_gb300", "csrc", name), encoding="utf-8").read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        lines = [ln.rstrip() for ln in text.splitlines() if ln.strip()]
        h.update(("\n".join(lines) + "\n").encode())
    return h.hexdigest()[:16]


def load_traffic(workload: str, e4m3: bool = False, algorithmic_bytes: float = 0.0):
    """(DRAM bytes of one grouped-FFN call -- its GEMM launches, and the h
    quantisation for e4m3 -- or, for "<workload>:layer", of one launch of the
    one-launch decode layer, from the committed ncu summaries, how they were
    obtained), or (None, None) once the code of any of those kernels changed
    since.  A workload too large to capture under DRAM counters carries the
    ratio DRAM bytes / algorithmic bytes measured on a smaller case of the same
    kernels, applied to this call's algorithmic bytes."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(p):
        return None, None
    ent = json.load(open(p)).get(f"{workload}:e4m3" if e4m3 else workload)
    srcs = LAYER_SOURCES if workload.endswith(":layer") else GEMM_SOURCES
    if not ent or ent.get("kernel_sha") != kernel_sources_sha(srcs):
        return None, None
    if "ffn_bytes_per_call" in ent:
        return ent["ffn_bytes_per_call"], ent.get("source")
    if "layer_bytes_per_call" in ent:
        return ent["layer_bytes_per_call"], ent.get("source")
    if "traffic_per_algorithmic_byte" in ent and algorithmic_bytes > 0:
        return ent["traffic_per_algorithmic_byte"] * algorithmic_bytes, ent.get("source")
    return None, None


# ----------------------------------------------------------------------------
# our arm
# ----------------------------------------------------------------------------
def l2_flush_needed(wl, e4m3: bool, l2_size: int) -> bool:
    """Inputs that fit in L2 (all expert weights plus the 8 token batches below
    twice the L2 size) are flushed out of it before every timed step."""
    esize = 1 if e4m3 else 2
    input_bytes = (wl.E * (3 if wl.act == synth.ACT_SWIGLU else 2) * wl.D * wl.Dff * esize + 8 * wl.N * wl.D * 2 +
                   wl.E * wl.D * 2)
    return input_bytes < 2 * l2_size


def bench_config(wl, args, world: int, flush: bool) -> dict:
    """The workload description both arms print (the reference arm times the
    oracle on this same configuration)."""
    e4m3 = args.precision == "e4m3"
    padded = args.paradigm == "padded"
    cfg = dict(wl.describe(), parallelism=f"replicas{world}" if world > 1 else "single-gpu",
               experts="e4m3 codes, per-row power-of-two scales, bf16 router" if e4m3 else "bf16",
               l2=("L2 flushed before every timed step (a buffer of twice the L2 size written "
                   "outside the step's interval): the layer's inputs fit in L2"
                   if flush else
                   "inputs larger than L2: expert weights streamed every step; x rotates "
                   "over 8 distinct batches"),
               seed=args.seed)
    cfg["permute"] = ("row copy + unfused GEMM1" if not args.fused or padded else
                      "fused into GEMM1: index-only permute, GEMM1 gathers the token rows")
    if e4m3:
        cfg["stage_note"] = "permute stage includes the token quantisation"
    if padded:
        cfg["paradigm"] = f"padded, capacity factor {args.capacity_factor}"
    return cfg


def run_ours(args, world, rank, local):
    from mixture_experts_layer_02_gb300 import build, moe
    build.build()
    moe.load()
    wl = synth.WORKLOADS[args.workload]
    dev = torch.device("cuda", torch.cuda.current_device())
    stream = torch.cuda.current_stream()
    seed = args.seed + rank
    inp = synth.make_inputs(wl, seed=seed, device=dev)
    xs = [synth.make_tokens(wl, seed=seed, device=dev, step=i) for i in range(8)]
    N, D, E, K, Dff = wl.N, wl.D, wl.E, wl.K, wl.Dff
    A = N * K
    ws = moe.workspace("layer", N, D, E, K, Dff, device=dev)
    mid = moe.layer_intermediates(ws, N, D, E, K, Dff)
    ws_perm = moe.workspace("permute", N=N, E=E, device=dev)
    ws_route = moe.workspace("route", N, D, E, K, device=dev)
    ws_ffn = moe.workspace("ffn", A, D, E, 1, Dff, device=dev)
    ws_small = moe.workspace("combine", device=dev)
    out = torch.empty((N, D), dtype=torch.bfloat16, device=dev)
    w1, w3, w2 = inp["w1"], inp["w3"], inp["w2"]

    padded = args.paradigm == "padded"
    e4m3 = args.precision == "e4m3"
    # --fused: the permutation fused into GEMM1 (index-only permute + gathered
    # operand rows); the default is the row copy + unfused GEMM1, as
    # moe_layer_forward runs it unless MOE_GATHER=1
    fused = args.fused
    if fused:
        os.environ["MOE_GATHER"] = "1"   # the e2e leg's moe_layer_forward likewise
    if e4m3:
        # FP8 expert weights are prepared once (offline), as a deployment would
        qw = moe.quantize_experts_e4m3(w1, w3, w2)
        if args.no_cpu_baseline:  # the bf16 experts are needed only by the oracle leg
            torch.cuda.synchronize()
            w1 = w3 = w2 = inp["w1"] = inp["w3"] = inp["w2"] = None
            torch.cuda.empty_cache()
        ws8 = moe.workspace("layer_e4m3", N, D, E, K, Dff, device=dev)
        mid8 = moe.layer_e4m3_intermediates(ws8, N, D, E, K, Dff)
        torch.cuda.synchronize()
    if padded:
        cap = moe.capacity(N, E, K, args.capacity_factor)
        R = E * cap
        ws_layer_p = moe.workspace_padded("layer", N, D, E, K, Dff, cap, device=dev)
        pmid = moe.layer_padded_intermediates(ws_layer_p, N, D, E, K, Dff, cap)
        ws_perm = moe.workspace_padded("permute", N=N, E=E, cap=cap, device=dev)
        ws_ffn = moe.workspace("ffn", max(R, 1), D, E, 1, Dff, device=dev)

    def step_padded(x, ev=None):
        if ev is not None:
            ev[0].record(stream)
        moe.moe_route(x, inp["w_gate"], inp["bias"], K, wl.mode, pmid["topk_ids"], pmid["topk_w"], ws=ws_route)
        if ev is not None:
            ev[1].record(stream)
        moe.moe_permute_padded(x, pmid["topk_ids"], E, cap, pmid["expert_offsets"], pmid["kept"], pmid["slot"],
                               pmid["x_pad"], ws=ws_perm)
        if ev is not None:
            ev[2].record(stream)
        if R > 0:
            moe.moe_grouped_ffn(pmid["x_pad"], pmid["expert_offsets"], w1, w3, w2, wl.act, pmid["h"],
                                pmid["y_pad"], ws=ws_ffn)
        if ev is not None:
            ev[3].record(stream)
        moe.moe_combine_padded(pmid["y_pad"], pmid["slot"], pmid["topk_w"], E, cap, out, ws=ws_small)
        if ev is not None:
            ev[4].record(stream)

    def step_e4m3(x, ev=None):
        m = mid8
        if ev is not None:
            ev[0].record(stream)
        moe.moe_route(x, inp["w_gate"], inp["bias"], K, wl.mode, m["topk_ids"], m["topk_w"], ws=ws_route)
        if ev is not None:
            ev[1].record(stream)
        moe.moe_quantize_e4m3(x, m["xq"], m["x_scale"])
        if fused:
            moe.moe_permute_indices(m["topk_ids"], E, m["expert_offsets"], m["perm_src"], m["inv_perm"],
                                    ws=ws_perm)
        else:
            moe.moe_permute_e4m3(m["xq"], m["topk_ids"], E, m["expert_offsets"], m["perm_src"], m["inv_perm"],
                                 m["xq_perm"], ws=ws_perm)
        if ev is not None:
            ev[2].record(stream)
        if fused:
            moe.moe_grouped_ffn_e4m3_gathered(m["xq"], m["x_scale"], m["perm_src"], m["expert_offsets"], qw["w1q"],
                                              qw["s1"], qw["w3q"], qw["s3"], qw["w2q"], qw["s2"], wl.act, m["h"],
                                              m["hq"], m["h_scale"], m["y_perm"], ws=ws_ffn)
        else:
            moe.moe_grouped_ffn_e4m3(m["xq_perm"], m["x_scale"], m["perm_src"], m["expert_offsets"], qw["w1q"],
                                     qw["s1"], qw["w3q"], qw["s3"], qw["w2q"], qw["s2"], wl.act, m["h"], m["hq"],
                                     m["h_scale"], m["y_perm"], ws=ws_ffn)
        if ev is not None:
            ev[3].record(stream)
        moe.moe_combine(m["y_perm"], m["inv_perm"], m["topk_w"], out, ws=ws_small)
        if ev is not None:
            ev[4].record(stream)

    # decode-sized batches (up to 8 tokens) route and permute through one
    # call, whose top-K and permutation run in one launch (as
    # moe_layer_forward does)
    route_permute = (not fused) and N <= 8 and N * K <= 256
    # small decode batches: moe_layer_forward runs the whole layer as one
    # cooperative launch, and the step times exactly that call
    one_launch = (not (padded or fused)) and (
        moe.layer_launches_e4m3(N, D, E, K, Dff, wl.act) == 1 if e4m3 else
        moe.layer_launches(N, D, E, K, Dff, wl.act) == 1)
    ws_rp = moe.workspace("route_permute", N, D, E, K, device=dev) if route_permute else None

    def step_one_launch(x, ev=None):
        if ev is not None:
            ev[0].record(stream)
        if e4m3:
            moe.moe_layer_forward_e4m3(x, inp["w_gate"], inp["bias"], qw, K, wl.mode, wl.act, out=out, ws=ws8)
        else:
            moe.moe_layer_forward(x, inp["w_gate"], inp["bias"], w1, w3, w2, K, wl.mode, wl.act, out=out, ws=ws)
        if ev is not None:
            for j in range(1, 5):
                ev[j].record(stream)

    def step(x, ev=None):
        if padded:
            return step_padded(x, ev)
        if one_launch:
            return step_one_launch(x, ev)
        if e4m3:
            return step_e4m3(x, ev)
        if ev is not None:
            ev[0].record(stream)
        if route_permute:
            moe.moe_route_permute(x, inp["w_gate"], inp["bias"], K, wl.mode, mid["topk_ids"], mid["topk_w"],
                                  mid["expert_offsets"], mid["perm_src"], mid["inv_perm"], mid["x_perm"], ws=ws_rp)
            if ev is not None:
                ev[1].record(stream)
                ev[2].record(stream)
        else:
            moe.moe_route(x, inp["w_gate"], inp["bias"], K, wl.mode, mid["topk_ids"], mid["topk_w"],
                          ws=ws_route)
            if ev is not None:
                ev[1].record(stream)
        if route_permute:
            pass
        elif fused:  # indices only; GEMM1 gathers the token rows
            moe.moe_permute_indices(mid["topk_ids"], E, mid["expert_offsets"], mid["perm_src"], mid["inv_perm"],
                                    ws=ws_perm)
        else:
            moe.moe_permute(x, mid["topk_ids"], E, mid["expert_offsets"], mid["perm_src"], mid["inv_perm"],
                            mid["x_perm"], ws=ws_perm)
        if ev is not None and not route_permute:
            ev[2].record(stream)
        if fused:
            moe.moe_grouped_ffn_gathered(x, mid["perm_src"], mid["expert_offsets"], w1, w3, w2, wl.act, mid["h"],
                                         mid["y_perm"], ws=ws_ffn)
        else:
            moe.moe_grouped_ffn(mid["x_perm"], mid["expert_offsets"], w1, w3, w2, wl.act, mid["h"],
                                mid["y_perm"], ws=ws_ffn)
        if ev is not None:
            ev[3].record(stream)
        moe.moe_combine(mid["y_perm"], mid["inv_perm"], mid["topk_w"], out, ws=ws_small)
        if ev is not None:
            ev[4].record(stream)

    for i in range(args.warmup):
        step(xs[i % len(xs)])
    torch.cuda.synchronize()

    # One CUDA graph per token batch: a replay launches the step's 7 kernels
    # with no host work in between (what a serving loop would run).
    graphs = []
    if not args.no_graph:
        try:
            cap_stream = torch.cuda.Stream()
            for x in xs:
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=cap_stream):
                    step(x)
                graphs.append(g)
            # every graph's first replay uploads it to the device: do that for
            # all of them before the warm-up steps, never inside the timed region
            for g in graphs:
                g.replay()
            torch.cuda.synchronize()
            for i in range(args.warmup):
                graphs[i % len(graphs)].replay()
            torch.cuda.synchronize()
        except Exception as exc:  # capture unsupported: time direct launches instead
            print(f"# CUDA graph capture failed ({exc}); timing direct launches", file=sys.stderr)
            graphs = []

    # Inputs that fit in L2 (all expert weights plus the 8 token batches below
    # twice the L2 size) are flushed out of it before every timed step by
    # writing a buffer of twice the L2 size, outside the step's interval.
    l2_size = torch.cuda.get_device_properties(dev).L2_cache_size
    flush_buf = (torch.empty(2 * l2_size, dtype=torch.uint8, device=dev)
                 if l2_flush_needed(wl, e4m3, l2_size) else None)

    sampler = ClockSampler(dev.index) if not args.no_clocks else None

    def preload():
        """Keep the GPU busy for --preload-s before a timed leg, so that every
        leg (graph replays, direct launches, end to end) starts from the same
        sustained, power-capped state and its clock record is under load.
        Returns the wall time the preload began (the start of the leg's clock
        window)."""
        t = time.time()
        while time.time() - t < args.preload_s:
            if graphs:
                graphs[0].replay()
            else:
                step(xs[0])
            torch.cuda.synchronize()
        return t

    legs = {}  # wall-clock windows (preload start, leg end) of the three timed legs
    t_load = preload()

    def hold_gpu(seconds):
        """Queue a spin kernel so the host can enqueue ahead of the GPU."""
        torch.cuda._sleep(int(seconds * 2.2e9))
        ev = torch.cuda.Event()
        ev.record(stream)
        return ev

    # ---- timed region: K steps (graph replays; direct launches without graphs)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(args.steps)]
    e_start, e_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e_step = [torch.cuda.Event(enable_timing=True) for _ in range(max(args.steps - 1, 0))]
    # each step's own interval, with the L2 flush (when needed) between intervals
    e_a = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    e_b = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    t_wall0 = time.time()
    if graphs and flush_buf is not None:
        for i in range(args.steps):
            flush_buf.zero_()  # evict the previous step's inputs from L2, outside the interval
            e_a[i].record(stream)
            graphs[i % len(graphs)].replay()
            e_b[i].record(stream)
    elif graphs:
        e_start.record(stream)
        for i in range(args.steps):
            if i > 0:
                e_step[i - 1].record(stream)  # step boundaries: per-step median and min
            graphs[i % len(graphs)].replay()
        e_end.record(stream)
    else:
        held = hold_gpu(max(0.005, args.steps * 5e-4))
        for i in range(args.steps):
            if flush_buf is not None:
                flush_buf.zero_()
            step(xs[i % len(xs)], evs[i])
    torch.cuda.synchronize()
    barrier(world)
    t_wall1 = time.time()
    legs["value"] = (t_load, t_wall1)
    if graphs and flush_buf is not None:
        per_step = [e_a[i].elapsed_time(e_b[i]) for i in range(args.steps)]
    elif graphs:
        bounds = [e_start] + e_step + [e_end]
        per_step = [bounds[i].elapsed_time(bounds[i + 1]) for i in range(args.steps)]
    else:
        per_step = [e[0].elapsed_time(e[4]) for e in evs]
    if flush_buf is not None:
        total_ms = sum(per_step)  # the flushes between the steps are not part of the work
    else:
        total_ms = e_start.elapsed_time(e_end) if graphs else evs[0][0].elapsed_time(evs[-1][4])
    total_ms = max_over_ranks(total_ms, world)

    # ---- per-stage breakdown: the same steps launched directly, with CUDA
    # events between the stages, the host queueing every step before the GPU
    # starts the first one (so no event interval contains host time)
    host_ahead = True
    if graphs:
        t_d = preload()
        held = hold_gpu(max(0.005, args.steps * 5e-4))
        for i in range(args.steps):
            if flush_buf is not None:
                flush_buf.zero_()
            step(xs[i % len(xs)], evs[i])
        host_ahead = not held.query()
        torch.cuda.synchronize()
        legs["direct"] = (t_d, time.time())
    else:
        host_ahead = None
        legs["direct"] = legs["value"]
    stage_ms = [statistics.mean(e[j].elapsed_time(e[j + 1]) for e in evs) for j in range(4)]
    direct_ms = evs[0][0].elapsed_time(evs[-1][4]) / args.steps
    dev_status = max(moe.read_device_error(w) for w in (ws_small, ws_perm, ws_route, ws_ffn, ws) + ((ws8,) if e4m3 else ()))
    # fingerprints of the inputs and of the last timed step's output (batch
    # (steps-1) mod 8), taken before the end-to-end leg reuses the buffers
    digests = {"inputs": {k: tensor_digest(v) for k, v in inp.items() if v is not None},
               "token_batches": [tensor_digest(x)["sha256"] for x in xs],
               "output": dict(tensor_digest(out), batch=(args.steps - 1) % len(xs))}
    if e4m3:
        digests["e4m3_experts"] = {k: tensor_digest(v) for k, v in qw.items() if v is not None}
    offsets = (pmid if padded else (mid8 if e4m3 else mid))["expert_offsets"].cpu().tolist()
    dropped = int((pmid["slot"] < 0).sum().item()) if padded else 0

    # ---- end to end through the public API, host buffers, copies inside.
    # Every step copies its token batch in from pinned host memory and its
    # output back; copies run on their own streams, double-buffered, so step
    # i's output copy and step i+1's input copy overlap step i+1's compute
    # (the way a serving loop would run it).
    x_host = [xs[i].cpu().pin_memory() for i in range(2)]
    out_host = [torch.empty((N, D), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    x_dev = [torch.empty_like(xs[0]) for _ in range(2)]
    out_dev = [torch.empty((N, D), dtype=torch.bfloat16, device=dev) for _ in range(2)]
    ws_layer = moe.workspace("layer_e4m3" if e4m3 else "layer", N, D, E, K, Dff, device=dev)
    h2d, d2h = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_comp = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    for b in range(2):  # buffers start free
        ev_comp[b].record(stream)
        ev_out[b].record(stream)

    def e2e_step(i):
        b = i % 2
        with torch.cuda.stream(h2d):
            h2d.wait_event(ev_comp[b])                 # x_dev[b] no longer read
            x_dev[b].copy_(x_host[b], non_blocking=True)
            ev_in[b].record(h2d)
        stream.wait_event(ev_in[b])
        stream.wait_event(ev_out[b])                   # out_dev[b] copied out
        if padded:
            moe.moe_layer_forward_padded(x_dev[b], inp["w_gate"], inp["bias"], w1, w3, w2, K, wl.mode, wl.act,
                                         cap, out=out_dev[b], ws=ws_layer_p)
        elif e4m3:
            moe.moe_layer_forward_e4m3(x_dev[b], inp["w_gate"], inp["bias"], qw, K, wl.mode, wl.act,
                                       out=out_dev[b], ws=ws_layer)
        else:
            moe.moe_layer_forward(x_dev[b], inp["w_gate"], inp["bias"], w1, w3, w2, K, wl.mode, wl.act,
                                  out=out_dev[b], ws=ws_layer)
        ev_comp[b].record(stream)
        with torch.cuda.stream(d2h):
            d2h.wait_event(ev_comp[b])
            out_host[b].copy_(out_dev[b], non_blocking=True)
            ev_out[b].record(d2h)

    for i in range(args.warmup):
        e2e_step(i)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_e = preload()
    barrier(world)
    torch.cuda.synchronize()
    e0.record(h2d)
    for i in range(args.steps):
        e2e_step(i)
    d2h.wait_stream(h2d)
    d2h.wait_stream(stream)
    e1.record(d2h)
    torch.cuda.synchronize()
    barrier(world)
    legs["e2e"] = (t_e, time.time())
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world)
    dev_status = max(dev_status, moe.read_device_error(ws_layer))
    clocks = None
    leg_clocks = {}
    if sampler is not None:
        sampler.stop()
        clocks = sampler.summary(t0=t_load)
        leg_clocks = {k: sampler.summary(t0=a, t1=b) for k, (a, b) in legs.items()}

    if rank != 0:
        return None

    wm = work_model(wl, offsets, padded_rows=(E * cap) if padded else None, e4m3=e4m3, fused=fused)
    peaks, peak_src = load_peaks()
    ms_step = total_ms / args.steps
    tokens_per_s = N * world * args.steps / (total_ms / 1e3)
    hbm = peaks["hbm_gbs"]
    if one_launch:
        # the step is one kernel: its duration is the timed region's mean step
        layer_s = ms_step / 1e3
        achieved = wm["layer_bytes"] / layer_s / 1e9
        traffic, traffic_src = load_traffic(wl.name + (":e4m3" if e4m3 else "") + ":layer", False, wm["layer_bytes"])
        roof = {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                "traffic": traffic, "peak_source": f"{peak_src} HBM copy",
                "kernel": "layer_decode_kernel (moe_layer_forward: the whole layer in one cooperative launch)",
                "algorithmic_bytes_per_call": wm["layer_bytes"],
                "algorithmic_flop_per_call": wm["ffn_flop"] + wm["route_flop"],
                "duration_from": "mean step of the timed region (one launch per step)",
                "traffic_source": traffic_src, "gbs": achieved,
                "tflops": (wm["ffn_flop"] + wm["route_flop"]) / layer_s / 1e12}
        stages = {"layer": {"ms": stage_ms[0], "gbs": wm["layer_bytes"] / stage_ms[0] / 1e6,
                            "hbm_frac": wm["layer_bytes"] / stage_ms[0] / 1e6 / hbm,
                            "includes": "route, permute, grouped FFN and combine in one launch"}}
    else:
        ffn_s = stage_ms[2] / 1e3
        ai = wm["ffn_flop"] / wm["ffn_bytes"]
        # e4m3 tensor peak: the measured bf16 peak times the nominal e4m3/bf16 ratio (4.5 / 2.25)
        tratio = 2.0 if e4m3 else 1.0
        ridge = tratio * peaks["bf16_tflops_sustained"] * 1e12 / (peaks["hbm_gbs"] * 1e9)
        traffic, traffic_src = (None, None) if (padded or fused) else load_traffic(wl.name, e4m3, wm["ffn_bytes"])
        if ai >= ridge:
            achieved = wm["ffn_flop"] / ffn_s / 1e12
            peak = tratio * peaks["bf16_tflops_sustained"]
            roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                    "frac": achieved / peak, "traffic": traffic,
                    "peak_source": (f"{peak_src} bf16 sustained (seconds-long loop) x 2 (nominal e4m3/bf16)"
                                    if e4m3 else f"{peak_src} bf16 sustained (seconds-long loop)"),
                    "frac_of_burst_peak": achieved / (tratio * peaks["bf16_tflops"])}
        else:
            achieved = wm["ffn_bytes"] / ffn_s / 1e9
            peak = peaks["hbm_gbs"]
            roof = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                    "frac": achieved / peak, "traffic": traffic, "peak_source": f"{peak_src} HBM copy"}
        roof.update({
            "kernel": ("grouped GEMMs on e4m3 (moe_grouped_ffn_e4m3: GEMM1+SwiGLU, h quantisation, GEMM2)"
                       if e4m3 else "grouped_gemm_kernel (moe_grouped_ffn: GEMM1+SwiGLU and GEMM2 launches)"),
            "algorithmic_flop_per_call": wm["ffn_flop"], "algorithmic_bytes_per_call": wm["ffn_bytes"],
            "arith_intensity": ai, "ridge": ridge, "traffic_source": traffic_src,
            "tflops": wm["ffn_flop"] / ffn_s / 1e12, "gbs": wm["ffn_bytes"] / ffn_s / 1e9,
        })
        rp = route_permute and not (padded or e4m3)
        route_bytes = wm["route_bytes"] + (wm["permute_bytes"] if rp else 0)
        stages = {
            "route": {"ms": stage_ms[0], "gbs": route_bytes / stage_ms[0] / 1e6,
                      "hbm_frac": route_bytes / stage_ms[0] / 1e6 / hbm,
                      "tflops": wm["route_flop"] / stage_ms[0] / 1e9,
                      **({"includes": "permute (moe_route_permute: top-K and permutation in one launch)"} if rp else {})},
            "permute": ({"ms": 0.0, "fused_into": "route"} if rp else
                        {"ms": stage_ms[1], "gbs": wm["permute_bytes"] / stage_ms[1] / 1e6,
                         "hbm_frac": wm["permute_bytes"] / stage_ms[1] / 1e6 / hbm}),
            "grouped_ffn": {"ms": stage_ms[2], "tflops": roof["tflops"], "gbs": roof["gbs"]},
            "combine": {"ms": stage_ms[3], "gbs": wm["combine_bytes"] / stage_ms[3] / 1e6,
                        "hbm_frac": wm["combine_bytes"] / stage_ms[3] / 1e6 / hbm},
        }
    e2e_tps = N * world * args.steps / (e2e_ms / 1e3)
    res = {
        "metric": "MoE-layer tokens/s on 1 GB300; grouped-FFN % of BF16 peak / % of HBM BW",
        "value": tokens_per_s, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "e4m3" if e4m3 else "bf16", "data": "synthetic",
        "config": bench_config(wl, args, world, flush_buf is not None),
        "roofline": roof,
        "stages": stages,
        "routing": dict({k: wm[k] for k in ("rows", "touched_experts", "empty_experts", "max_expert_share")},
                        **({"paradigm": "padded", "capacity": cap, "dropped_assignments": dropped}
                           if padded else {"paradigm": "contiguous"})),
        "e2e": {"value": e2e_tps, "unit": "tokens/s", "h2d_bytes_per_step": N * D * 2,
                "d2h_bytes_per_step": N * D * 2,
                "api": "moe_layer_forward_e4m3" if e4m3 else "moe_layer_forward",
                "ms_per_step": e2e_ms / args.steps,
                "copies": "pinned host buffers, H2D and D2H on their own streams, double-buffered"},
        "gpu_launches": (moe.layer_launches_e4m3(N, D, E, K, Dff, wl.act) if e4m3 else
                         moe.layer_launches(N, D, E, K, Dff, wl.act, cap if padded else -1)) * args.steps,
        "timing": {"value_from": ("CUDA graph replays of the step" if graphs else "direct launches") +
                                 ("; the sum of each step's own interval, L2 flushed between steps"
                                  if flush_buf is not None else ""),
                   "stages_from": "direct launches with events between stages, host queued ahead "
                                  "of the GPU", "host_ahead": host_ahead,
                   "direct_ms_per_step": direct_ms,
                   "e2e_ms_per_step": e2e_ms / args.steps,
                   "legs_order": "value (graph replays), then direct launches, then e2e; each leg "
                                 f"preceded by {args.preload_s:g} s of the same load",
                   "leg_clocks": {k: {"sm_mhz": v.get("sm_mhz"), "samples": v.get("samples"),
                                      "reasons": v.get("reasons")} for k, v in leg_clocks.items()},
                   "step_ms": {"median": statistics.median(per_step), "min": min(per_step),
                               "max": max(per_step), "of": len(per_step)}},
        "digests": digests,
        "clocks": clocks,
        "device_status": dev_status,
        "wall_s_timed": t_wall1 - t_wall0,
    }
    return res, inp, wl


# ----------------------------------------------------------------------------
# oracle timing (cpu_baseline and the reference arm)
# ----------------------------------------------------------------------------
def host_inputs(inp):
    import numpy as np
    out = {}
    for k, v in inp.items():
        if v is None:
            out[k] = None
        elif v.dtype == torch.bfloat16:
            out[k] = v.contiguous().cpu().view(torch.int16).numpy().view(np.uint16)
        else:
            out[k] = v.cpu().numpy().astype(np.float64)
    return out


def oracle_tokens(h, wl, n, offset=0):
    from oracle import oracle as O
    x = h["x"][offset:offset + n]
    O.layer(x, h["w_gate"], h["bias"], h["w1"], h["w3"], h["w2"], wl.K, wl.mode, wl.act)


class OracleE4m3:
    """The oracle's FP8 layer on a token sample: routing, per-token e4m3 x,
    the FP8 FFN over the experts the sample touches, combine.  Weight rows are
    quantised by the oracle once per expert (offline, outside the timing)."""

    def __init__(self, h, wl):
        self.h, self.wl, self.q = h, wl, {}

    def prepare(self, x):
        from oracle import oracle as O
        wl, h = self.wl, self.h
        ids = O.select(O.logits(x, h["w_gate"], h["bias"]), wl.K)
        for e in sorted(set(ids.ravel().tolist()) - set(self.q)):
            w3 = O.quant_rows_e4m3(h["w3"][e]) if h["w3"] is not None else (None, None)
            self.q[e] = (O.quant_rows_e4m3(h["w1"][e]), w3, O.quant_rows_e4m3(h["w2"][e]))

    def __call__(self, x):
        import numpy as np
        from oracle import oracle as O
        wl, h = self.wl, self.h
        L = O.logits(x, h["w_gate"], h["bias"])
        r = O.route_from_logits(L, wl.K, wl.mode, wl.E)
        xq, sx = O.quant_rows_e4m3(x)
        off = r["offsets"]
        touched = [e for e in range(wl.E) if off[e + 1] > off[e]]
        off_c = np.concatenate([[0], np.cumsum([off[e + 1] - off[e] for e in touched])]).astype(np.int32)
        sw = wl.act == synth.ACT_SWIGLU
        st = lambda i, j: np.stack([self.q[e][i][j] for e in touched])
        g = O.grouped_ffn_e4m3(xq[r["perm_src"]], sx[r["perm_src"]], off_c, st(0, 0), st(0, 1),
                               st(1, 0) if sw else None, st(1, 1) if sw else None, st(2, 0), st(2, 1), wl.act)
        return O.combine(g["y"], r["inv_perm"], r["w"])


def time_oracle_sample(h, wl, target_s, e4m3=False):
    """Time the oracle on a token sample sized for about target_s seconds."""
    from oracle import oracle as O
    n0 = max(1, min(wl.N, -(-2 * O.default_threads() // wl.K)))   # >= 2 rows per thread
    if e4m3:
        run = OracleE4m3(h, wl)
        run.prepare(h["x"][:n0])
        t = time.perf_counter()
        run(h["x"][:n0])
        dt0 = max(time.perf_counter() - t, 1e-3)
        n = int(max(1, min(wl.N, n0 * target_s / dt0)))
        run.prepare(h["x"][:n])
        t = time.perf_counter()
        run(h["x"][:n])
        return n, time.perf_counter() - t, O.default_threads()
    t = time.perf_counter()
    oracle_tokens(h, wl, n0)
    dt0 = max(time.perf_counter() - t, 1e-3)
    n = int(max(1, min(wl.N, n0 * target_s / dt0)))
    t = time.perf_counter()
    oracle_tokens(h, wl, n, offset=0)
    dt = time.perf_counter() - t
    return n, dt, O.default_threads()


def run_reference(args, world, rank):
    if rank != 0:
        return
    from oracle import oracle as O
    O.build()
    wl = synth.WORKLOADS[args.workload]
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    h = host_inputs(synth.make_inputs(wl, seed=args.seed, device=dev))
    l2 = torch.cuda.get_device_properties(0).L2_cache_size if torch.cuda.is_available() else 0
    config = bench_config(wl, args, world, l2_flush_needed(wl, False, l2))
    per_step = max(0.5, min(5.0, 150.0 / max(1, args.steps + args.warmup)))
    n, dt, cores = time_oracle_sample(h, wl, per_step)
    for i in range(args.warmup):
        oracle_tokens(h, wl, n, offset=(i * n) % max(1, wl.N - n + 1))
    t0 = time.perf_counter()
    for i in range(args.steps):
        oracle_tokens(h, wl, n, offset=(i * n) % max(1, wl.N - n + 1))
    t = time.perf_counter() - t0
    v = n * args.steps / t
    sample = f"{n} tokens of the {wl.name} workload per step (full route over all E experts, " \
             f"FFN of the K chosen experts, combine), fp64"
    res = {
        "metric": "MoE-layer tokens/s on 1 GB300; grouped-FFN % of BF16 peak / % of HBM BW",
        "value": v, "unit": "tokens/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": t / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config,
        "impl": "reference",
        "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(res), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="dsv3_zipf", choices=sorted(synth.WORKLOADS),
                    help="default: the DeepSeek-V3-shaped layer at 16384 tokens with Zipf(1.2)-skewed routing, "
                         "the largest configuration on one GPU")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--no-graph", action="store_true")
    ap.add_argument("--paradigm", default="contiguous", choices=["contiguous", "padded"],
                    help="contiguous segments (default) or fixed capacity per expert")
    ap.add_argument("--capacity-factor", type=float, default=1.5)
    ap.add_argument("--fused", action="store_true",
                    help="fuse the permutation into GEMM1 (gathered operand rows) instead of the row copy")
    ap.add_argument("--precision", default="bf16", choices=["bf16", "e4m3"],
                    help="expert GEMM operands: bf16 (default) or e4m3 codes with per-row scales")
    ap.add_argument("--preload-s", type=float, default=1.0)
    ap.add_argument("--cpu-target-s", type=float, default=15.0)
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.precision == "e4m3" and args.paradigm == "padded":
        ap.error("--precision e4m3 runs the contiguous paradigm")
    if args.precision == "e4m3" and args.impl == "reference":
        ap.error("the reference arm times the bf16 oracle")
    world, rank, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, world, rank)
        return
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU for --impl ours")
    r = run_ours(args, world, rank, local)
    if rank == 0 and r is not None:
        res, inp, wl = r
        if world == 1 and not args.no_cpu_baseline:
            h = host_inputs(inp)
            del inp
            e4m3 = args.precision == "e4m3"
            n, dt, cores = time_oracle_sample(h, wl, args.cpu_target_s, e4m3=e4m3)
            res["cpu_baseline"] = {
                "value": n / dt, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                "sample": f"{n} of {wl.N} tokens of the same workload through the fp64 oracle "
                          f"(route over all E, {'e4m3 ' if e4m3 else ''}FFN of the K chosen experts, "
                          f"combine), {dt:.1f} s"}
        else:
            res["cpu_baseline"] = None
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
