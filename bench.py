"""Benchmark of the fused dynamic multi-LoRA linear layer on GB300.

One step = one pass of the whole hot path over one batch: the segment build
(bucket sort of lora_id_map + work lists) and the fused layer
y = x W^T + bias + scale * (x A_id^T) B_id^T, both through the C ABI.

Default workload: the decode step (M=32 tokens, K=N=4096, 20 adapters of
rank 16/32/64, 10% base-only tokens), seeded synthetic data.  Prints ONE JSON
line on rank 0.  Under torchrun each rank runs its own replica on its own GPU
(independent batches, no collective on the data path): weak scaling.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--config decode|tiny|prefill|qkv|mlp_down] [--no-sweep] [--no-cpu]

--impl reference times the CPU fp64 oracle (the reference arm of this
project): rank 0 only, each step a bounded element sample of the workload.
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from segmented_gemm_gb300 import workloads  # noqa: E402

L2_BYTES = 129 * 1024 * 1024
# nominal peaks of a GB300, printed beside the measured ones (the fractions
# that the roofline reports are of the measured peaks)
NOMINAL_HBM_GBS = 7900.0
NOMINAL_BF16_TFLOPS = 2250.0
MAX_SETS = None          # --max-sets: cap the rotating input sets (small profiler captures)
METRIC = "multi-LoRA linear tokens/s; % of HBM / bf16 tensor roofline, M=32..8192"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
CONFIG_TEXT = {
    "tiny": "tiny: M=64, K=256, N=256, 4 adapters ranks {8,8,16,16}, ids uniform over {-1..3}",
    "decode": "decode step: M=32 tokens, K=4096, N=4096, 20 adapters ranks U{16,32,64}, 10% base-only",
    "prefill": "prefill: M=1024 from 16 requests (contiguous runs), K=N=4096, 40 adapters, 5% base-only requests",
    "qkv": "merged QKV: M=2048, K=4096, N=6144, 8 adapters rank 64, Zipf(1.1) ids shuffled, 20% base-only",
    "mlp_down": "MLP down: M=8192, K=12288, N=4096, 32 adapters U{16,32,64}, Zipf(1.1) requests, 20% base-only",
}
# extra sweep lines beside the configurations above
SWEEP_EXTRA = {
    "qkv_sliced": "merged QKV with one adapter pair per slice: the qkv config's M, K and ids, output slices "
                  "4096 | 1024 | 1024, 8 adapters of rank 16 per slice",
    "decode_e4m3": "the decode step with its adapters stored as e4m3 codes (one byte per element) and one "
                   "dequant factor per adapter and factor; the same x, W, bias and ids",
    "decode_all_base": "the decode step with every id -1 (no LoRA token): the bare weight stream of the decode "
                       "kernel; the same x, W, bias and pool",
}


def make_workload(name):
    if name == "decode_e4m3":
        return workloads.to_e4m3(workloads.make_config("decode"))
    if name == "decode_all_base":
        base = workloads.make_config("decode")
        return dataclasses.replace(base, ids=torch.full_like(base.ids, -1))
    if name == "qkv_sliced":
        base = workloads.make_config("qkv")
        return workloads.make_sliced(base.M, base.K, [4096, 1024, 1024], [16] * 8, seed=1237, ids=base.ids.clone())
    return workloads.make_config(name)


def log(*a):
    print(*a, file=sys.stderr, flush=True)


# ---------------------------------------------------------------------------
# algorithmic work of one step (counts only)
# ---------------------------------------------------------------------------

def algorithmic_work(wl):
    """Bytes: W, x, y, bias, ids and the A_i / B_i of distinct adapters
    present at true rank.  Flops: 2MKN + sum over LoRA tokens 2 r (K + N);
    with S output slices each adapter has S pairs: 2 r (S K + N)."""
    ids = wl.ids
    S = len(wl.slices) if getattr(wl, "slices", None) else 1
    present = sorted(set(int(i) for i in ids.tolist() if 0 <= i < wl.num_adapters))
    adapter_elems = sum(wl.ranks[i] * (S * wl.K + wl.N) for i in present)
    adapter_bytes = adapter_elems * (1 if getattr(wl, "A8", None) is not None else 2)   # e4m3: one byte each
    nbytes = 2 * (wl.N * wl.K + wl.M * wl.K + wl.M * wl.N + (wl.N if wl.bias is not None else 0)) \
        + adapter_bytes + 4 * wl.M
    lora_flops = sum(2 * wl.ranks[int(i)] * (S * wl.K + wl.N) for i in ids.tolist() if 0 <= i < wl.num_adapters)
    flops = 2 * wl.M * wl.K * wl.N + lora_flops
    return nbytes, flops, len(present)


def dominant_kernel(wl):
    """The kernel lora_linear's automatic schedule choice launches for this
    shape (the same rule as the library's dispatch)."""
    if wl.M <= 64 and wl.K % 64 == 0:
        return "lora_cluster_kernel"
    if wl.M <= 128:
        return "lora_splitk_kernel"
    return "lora_tc_kernel"


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(p))
        return {k: float(d[k]) for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained")}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


# The source file each timed kernel is compiled from; a summary taken on an
# older copy of that file's code, or of the headers every kernel includes, is
# stale (comments do not count).
KERNEL_SOURCES = {   # the sources each kernel is compiled from (besides internal.h and ptx.cuh)
    "lora_cluster_kernel": ("fused_cluster.cu", "seg_build_body.cuh"),
    "lora_tc_kernel": ("fused_tc.cu",),
    "lora_splitk_kernel": ("fused_splitk.cu",),
    "seg_build_kernel": ("seg_build.cu", "seg_build_body.cuh"),
    "moe_pair_kernel": ("moe_pair.cu", "moe_pair.h"),
}


def code_only(src: str) -> str:
    """C/CUDA source without its comments and blank lines: an edit of a
    comment leaves a kernel's measurements standing."""
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if c in "\"'":                      # a string or character literal, kept whole
            j = i + 1
            while j < n and src[j] != c:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):
            i = src.find("\n", i)
            i = n if i < 0 else i
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    lines = (ln.rstrip() for ln in "".join(out).split("\n"))
    return "\n".join(ln for ln in lines if ln.strip())


def kernel_source_hash(kernel: str):
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "segmented_gemm_gb300", "csrc")
    for f in KERNEL_SOURCES[kernel] + ("internal.h", "ptx.cuh"):
        h.update(code_only(open(os.path.join(csrc, f)).read()).encode())
    return h.hexdigest()[:16]


def profiled_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current kernel sources (else None)."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.md")
    if not os.path.exists(path):
        return None
    txt = open(path).read()
    m = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", txt)
    h = re.search(r"source_hash:\s*([0-9a-f]+)", txt)
    if not m or not h or h.group(1) != kernel_source_hash(kernel):
        return None
    return float(m.group(1))


# ---------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.t0 = self.t1 = None
        ident = []
        try:
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            ident = ["--id=" + (uuid if uuid.startswith("GPU-") else "GPU-" + uuid)]
        except Exception:
            ident = []
        self.cmd = ["nvidia-smi", *ident, "--query-gpu=timestamp," + self.FIELDS,
                    "--format=csv,noheader,nounits", "-lms", "50"]

    def start(self):
        try:
            self.proc = subprocess.Popen(self.cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.3)

    def mark(self, which):
        setattr(self, which, time.time())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.1)
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        rows = []
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                ts += float("0." + parts[0].split(".")[1]) if "." in parts[0] else 0.0
                rows.append(dict(ts=ts, sm=float(parts[1]), smmax=float(parts[2]), power=float(parts[3]),
                                 active=parts[4], hw=parts[5], hwt=parts[6], swt=parts[7], pcap=parts[8]))
            except (ValueError, IndexError):
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        pmax = max(r["power"] for r in rows)
        window = "timed region"
        load = []
        if self.t0 is not None and self.t1 is not None:
            load = [r for r in rows if self.t0 - 0.06 <= r["ts"] <= self.t1 + 0.06]
        if not load:   # timed region shorter than the sampling interval: samples under load
            window = "under load around the timed region"
            load = [r for r in rows if r["power"] >= 0.5 * pmax] or rows
        reasons = set()
        for r in load:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                              ("swt", "sw_thermal_slowdown"), ("pcap", "sw_power_cap")):
                if r[key].lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in load), "sm_max_mhz": max(r["smmax"] for r in load),
                "reasons": sorted(reasons), "samples": len(load), "window": window,
                "power_w_max": max(r["power"] for r in load)}


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

class InputSet:
    def __init__(self, wl, L, device):
        self.x = wl.x.to(device)
        self.W = wl.W.to(device)
        self.bias = None if wl.bias is None else wl.bias.to(device)
        self.ids = wl.ids.to(device)
        if getattr(wl, "slices", None):
            self.pool = L.build_pool_sliced(wl.A_s, wl.B_s, wl.K, wl.slices, device)
        elif getattr(wl, "A8", None) is not None:
            self.pool = L.build_pool_e4m3(wl.A8, wl.B8, wl.deq, wl.K, wl.N, device, widened=wl.M > 64)
        else:
            self.pool = L.build_pool(wl.A, wl.B, wl.K, wl.N, device)
        self.y = torch.empty(wl.M, wl.N, dtype=torch.bfloat16, device=device)
        self.ws = L.Workspace(wl.M, wl.N, wl.num_adapters, device)
        self.segs = None

    def nbytes(self):
        p = self.pool
        t = [self.x, self.W, self.y, self.ids, p.a_pool, p.b_pool] + ([self.bias] if self.bias is not None else [])
        return sum(a.numel() * a.element_size() for a in t)


def build_sets(wl, L, device, min_bytes=4 * L2_BYTES, max_sets=16):
    max_sets = MAX_SETS or max_sets
    first = InputSet(wl, L, device)
    n = 1 if first.nbytes() >= min_bytes else min(max_sets, math.ceil(min_bytes / first.nbytes()))
    sets = [first] + [InputSet(wl, L, device) for _ in range(n - 1)]
    return sets


def graph_of(fn, n_steps, stream):
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(g, stream=stream):
            for i in range(n_steps):
                fn(i)
    return g


def time_steps(fn, steps, warmup, stream, chunk=None, sampler=None, dist_barrier=None):
    """Replay `fn(i)` for exactly `steps` steps inside CUDA graphs, timed with
    CUDA events on `stream`.  Returns total milliseconds."""
    chunk = chunk or min(steps, 200)
    for i in range(warmup):
        with torch.cuda.stream(stream):
            fn(i)
    torch.cuda.synchronize()
    full, rem = divmod(steps, chunk)
    g_full = graph_of(fn, chunk, stream) if full else None
    g_rem = graph_of(fn, rem, stream) if rem else None
    for g in (g_full, g_rem):          # graph warm-up
        if g is not None:
            g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if dist_barrier:
        dist_barrier()
    torch.cuda.synchronize()
    if sampler:
        sampler.mark("t0")
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(full):
            g_full.replay()
        if g_rem is not None:
            g_rem.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    if sampler:
        sampler.mark("t1")
    if dist_barrier:
        dist_barrier()
    return e0.elapsed_time(e1)


def time_isolated(fn, reps, stream):
    """Device time of single calls after an idle gap: each call is bracketed
    by CUDA events on `stream` after a device synchronize, so nothing
    overlaps it (no programmatic launch, no neighbouring call).  Median in ms."""
    ts = []
    for i in range(reps):
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            fn(i)
            e1.record(stream)
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1))
    return statistics.median(ts)


def run_config(name, L, device, steps, warmup, stream, sampler=None, dist_barrier=None, e2e=True,
               static_weights=True, compare_plain=False):
    """Time one configuration.  static_weights: the weights are loaded once
    and never written by a kernel during the steps, so each call may start
    streaming them before the previous call has finished
    (LORA_FLAG_STATIC_WEIGHTS).  compare_plain: also time both legs without
    the flag."""
    wl = make_workload(name)
    nbytes, flops, n_present = algorithmic_work(wl)
    sets = build_sets(wl, L, device)
    ns = len(sets)
    sw = static_weights

    def full_step(i):
        s = sets[i % ns]
        L.lora_linear(s.x, s.W, s.bias, s.ids, s.pool, wl.scale, s.ws, y=s.y, static_weights=sw)

    for s in sets:                          # prebuilt tables for the kernel-only timing
        s.segs = L.lora_build_segments(s.ids, s.pool, s.ws)

    def kernel_step(i):
        s = sets[i % ns]
        L.lora_linear(s.x, s.W, s.bias, s.ids, s.pool, wl.scale, s.ws, y=s.y, segs=s.segs, static_weights=sw)

    # the fused kernel alone (segment tables prebuilt): dominant-kernel duration
    kern_ms = time_steps(kernel_step, steps, warmup, stream) / steps
    iso_kern_ms = time_isolated(kernel_step, 200, stream)

    # reference: the base GEMM alone (x W^T + bias, no LoRA term) by cuBLAS
    # through PyTorch, on the same rotating inputs, timed the same way
    def base_step(i):
        s = sets[i % ns]
        if s.bias is not None:
            torch.addmm(s.bias, s.x, s.W.t(), out=s.y)
        else:
            torch.mm(s.x, s.W.t(), out=s.y)

    base_ms = time_steps(base_step, steps, warmup, stream) / steps
    plain = None
    if compare_plain:
        sw = False
        plain = {"kernel_us": round(time_steps(kernel_step, steps, warmup, stream) / steps * 1e3, 3)}
    for s in sets:                          # the timed step also rebuilds its table
        s.segs = None
    if compare_plain:
        plain["ms_per_step"] = round(time_steps(full_step, steps, warmup, stream) / steps, 6)
        sw = static_weights
    if sampler:
        sampler.start()
    total_ms = time_steps(full_step, steps, warmup, stream, sampler=sampler, dist_barrier=dist_barrier)
    clocks = sampler.stop() if sampler else None
    iso_step_ms = time_isolated(full_step, 200, stream)
    status = L.lora_get_status(sets[0].ws)
    res = dict(name=name, wl=wl, ms_per_step=total_ms / steps, kernel_ms=kern_ms, bytes=nbytes, flops=flops,
               n_present=n_present, n_sets=ns, set_bytes=sets[0].nbytes(), status=status, clocks=clocks,
               plain=plain, iso_kernel_ms=iso_kern_ms, iso_step_ms=iso_step_ms, base_ms=base_ms)
    if e2e:
        res["e2e"] = run_e2e(wl, sets, L, device, min(steps, 5000), max(3, min(warmup, 50)), stream)
    return res


SWEEP_LINES = ("prefill", "qkv", "mlp_down", "qkv_sliced", "decode_e4m3", "decode_all_base", "attention_block_prefill",
               "moe_experts")

LAYER_SHAPES = (("q", 4096, 4096), ("k", 4096, 1024), ("v", 4096, 1024), ("o", 4096, 4096))


def run_layer_step(L, device, steps, warmup, stream):
    """Four LoRA projections of one attention block (q, k, v, o: other N,
    the same adapters) on the prefill config's ids, as one step: all four in
    one launch (lora_linear_layers: a segment build, then one tiled launch
    whose work list spans the layers); or four lora_linear calls with one
    segment table built for the step; or four calls each building its own."""
    base = workloads.make_config("prefill")
    layers = [workloads.make_custom(base.M, K, N, base.ranks, seed=2000 + j, ids=base.ids.clone())
              for j, (_, K, N) in enumerate(LAYER_SHAPES)]
    nsets = 2
    sets = [[InputSet(wl, L, device) for wl in layers] for _ in range(nsets)]
    wss = [L.Workspace(base.M, max(n for _, _, n in LAYER_SHAPES), base.num_adapters, device) for _ in range(nsets)]
    flops = sum(algorithmic_work(wl)[1] for wl in layers)

    def shared(i):
        st, ws = sets[i % nsets], wss[i % nsets]
        segs = L.lora_build_segments(st[0].ids, st[0].pool, ws)
        for wl, s in zip(layers, st):
            L.lora_linear(s.x, s.W, s.bias, s.ids, s.pool, wl.scale, ws, y=s.y, segs=segs)

    def separate(i):
        st, ws = sets[i % nsets], wss[i % nsets]
        for wl, s in zip(layers, st):
            L.lora_linear(s.x, s.W, s.bias, s.ids, s.pool, wl.scale, ws, y=s.y)

    lwss = [L.LayersWorkspace(base.M, max(n for _, _, n in LAYER_SHAPES), base.num_adapters, len(LAYER_SHAPES),
                              device) for _ in range(nsets)]

    def one_launch(i):
        st, ws = sets[i % nsets], lwss[i % nsets]
        L.lora_linear_layers([(s.x, s.W, s.bias, s.pool, wl.scale, s.y) for wl, s in zip(layers, st)],
                             st[0].ids, ws)

    ms_one = time_steps(one_launch, steps, warmup, stream) / steps
    ms_shared = time_steps(shared, steps, warmup, stream) / steps
    ms_sep = time_steps(separate, steps, warmup, stream) / steps
    status = L.lora_get_status(wss[0]) | L.lora_get_status(lwss[0])
    return {"workload": "q, k, v, o projections (K=4096; N=4096, 1024, 1024, 4096) on the prefill config's "
                        "ids and adapters, one step = all four",
            "M": base.M, "tokens_per_s": round(base.M / (ms_one * 1e-3), 1),
            "ms_per_step": round(ms_one, 5), "method": "lora_linear_layers: segment build + one tiled launch "
                                                       "over the four layers",
            "ms_per_step_four_launches_one_table": round(ms_shared, 5),
            "ms_per_step_table_per_call": round(ms_sep, 5),
            "tflops": round(flops / (ms_one * 1e-3) / 1e12, 1),
            "tensor_frac": round(flops / (ms_one * 1e-3) / 1e12 / load_peaks()[0]["bf16_tflops"], 4),
            "device_status": status}


def run_moe_step(L, device, steps, warmup, stream, peaks):
    """A mixture-of-experts layer's expert GEMM: routing + grouped GEMM +
    weighted finalize through lora_moe, and the grouped GEMM alone."""
    cfg = dict(M=2048, K=2048, N=1536, E=64, topk=8)
    mw = workloads.make_moe(cfg["M"], cfg["K"], cfg["N"], cfg["E"], cfg["topk"], seed=4321, skew=1.0)
    d = device
    sets = []
    for j in range(2):   # two weight sets: 800 MB > 4x L2
        W = mw.W.to(d) if j == 0 else (mw.W.to(d) * 1.0)
        sets.append(dict(x=mw.x.to(d), W=W, ex=mw.expert.to(d), wt=mw.weight.to(d),
                         out=torch.empty(mw.M * mw.topk, mw.N, dtype=torch.bfloat16, device=d),
                         y=torch.empty(mw.M, mw.N, dtype=torch.bfloat16, device=d),
                         ws=L.MoeWorkspace(mw.M, mw.topk, mw.E, d)))
    lib = L.load_library()

    def whole(i):
        s = sets[i % 2]
        L.lora_moe(s["x"], s["W"], s["ex"], s["wt"], s["ws"], out=s["out"], y=s["y"])

    def gemm(i):
        s = sets[i % 2]
        L._check(lib.lora_moe_gemm(L._ptr(s["x"]), mw.M, mw.K, L._ptr(s["W"]), mw.N, mw.E, mw.topk,
                                   L._ptr(s["out"]), s["ws"].ptr, s["ws"].nbytes, L._stream(None)), "lora_moe_gemm")

    whole(0)
    whole(1)
    torch.cuda.synchronize()
    ms_whole = time_steps(whole, steps, warmup, stream) / steps
    ms_gemm = time_steps(gemm, steps, warmup, stream) / steps
    flops = 2 * mw.M * mw.topk * mw.K * mw.N
    tflops = flops / (ms_gemm * 1e-3) / 1e12
    return {"workload": "mixture of experts: M=2048 tokens, K=2048, N=1536, 64 experts, top-8, skewed routing; "
                        "routing + grouped GEMM + weighted finalize",
            "M": mw.M, "tokens_per_s": round(mw.M / (ms_whole * 1e-3), 1), "ms_per_step": round(ms_whole, 5),
            "gemm_us": round(ms_gemm * 1e3, 2), "gemm_tflops": round(tflops, 1),
            "tensor_frac": round(tflops / peaks["bf16_tflops"], 4),
            # the grouped GEMM (two token tiles of an expert per work item)
            "roofline": {"bound": "tensor", "achieved": round(tflops, 1), "peak": peaks["bf16_tflops"],
                         "unit": "TFLOP/s", "frac": round(tflops / peaks["bf16_tflops"], 4),
                         "traffic": profiled_traffic("moe_pair_kernel", "moe"), "kernel": "moe_pair_kernel",
                         "kernel_us": round(ms_gemm * 1e3, 3),
                         "kernel_time_method": "lora_moe_gemm alone, back to back in CUDA graphs over two weight "
                                               "sets, CUDA events on the launching stream",
                         "algorithmic_flops": flops}}


def run_e2e(wl, sets, L, device, steps, warmup, stream):
    """Same metric through the public API with host buffers.  Every step
    copies x and lora_id_map host->device from pinned memory into its input
    set, runs the layer (lora_linear) and brings y back into pinned memory.
    The input sets rotate as in the device-side timing, so the weights come
    from HBM.  Two ways of moving the bytes are timed, both replayed from
    CUDA graphs, and the faster one is the line's value (the other is
    reported beside it): the copy engines, on two side streams, so a step's
    copies overlap the layers of its neighbours (an input set's buffers are
    written again only after its previous layer has read them and its
    previous y has been copied out); or the SMs over the host link
    (run_e2e_host_link).  The copy-engine loop run eagerly on one stream,
    one step after the other, is reported too."""
    ns = len(sets)
    hx = wl.x.pin_memory()
    hids = wl.ids.pin_memory()
    hy = [torch.empty(wl.M, wl.N, dtype=torch.bfloat16).pin_memory() for _ in range(ns)]
    h2d = hx.numel() * hx.element_size() + hids.numel() * hids.element_size()
    d2h = hy[0].numel() * hy[0].element_size()

    def layer(st):
        L.lora_linear(st.x, st.W, st.bias, st.ids, st.pool, wl.scale, st.ws, y=st.y, static_weights=True)

    # eager, one stream: copy in, layer, copy out, step after step
    def eager_step(i):
        st = sets[i % ns]
        st.x.copy_(hx, non_blocking=True)
        st.ids.copy_(hids, non_blocking=True)
        layer(st)
        hy[i % ns].copy_(st.y, non_blocking=True)

    n_eager = min(steps, 2000)
    with torch.cuda.stream(stream):
        for i in range(warmup):
            eager_step(i)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(n_eager):
            eager_step(i)
        e1.record(stream)
    torch.cuda.synchronize()
    ms_eager = e0.elapsed_time(e1) / n_eager

    # CUDA graphs, copies on side streams
    cs_in, cs_out = torch.cuda.Stream(device), torch.cuda.Stream(device)

    def capture(n, first):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(g, stream=stream):
                cur = torch.cuda.current_stream()
                cs_in.wait_stream(cur)
                cs_out.wait_stream(cur)
                read_done, out_done = {}, {}
                for i in range(first, first + n):
                    b = i % ns
                    st = sets[b]
                    with torch.cuda.stream(cs_in):
                        if b in read_done:
                            cs_in.wait_event(read_done[b])
                        st.x.copy_(hx, non_blocking=True)
                        st.ids.copy_(hids, non_blocking=True)
                        ev_in = torch.cuda.Event()
                        ev_in.record(cs_in)
                    cur.wait_event(ev_in)
                    if b in out_done:
                        cur.wait_event(out_done[b])
                    layer(st)
                    ev_l = torch.cuda.Event()
                    ev_l.record(cur)
                    read_done[b] = ev_l
                    with torch.cuda.stream(cs_out):
                        cs_out.wait_event(ev_l)
                        hy[b].copy_(st.y, non_blocking=True)
                        ev_o = torch.cuda.Event()
                        ev_o.record(cs_out)
                        out_done[b] = ev_o
                cur.wait_stream(cs_in)
                cur.wait_stream(cs_out)
        return g

    chunk = min(steps, 200)
    full, rem = divmod(steps, chunk)
    g_full = capture(chunk, 0) if full else None
    g_rem = capture(rem, 0) if rem else None
    for g in (g_full, g_rem):
        if g is not None:
            g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(full):
            g_full.replay()
        if g_rem is not None:
            g_rem.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    # every set's last read-back holds that set's y
    for b in range(min(ns, steps)):
        if not torch.equal(hy[b], sets[b].y.cpu()):
            raise RuntimeError("end-to-end read-back differs from the device output")
    copy_engine = {"value": wl.M / (ms * 1e-3), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                   "d2h_bytes_per_step": d2h, "ms_per_step": ms, "steps": steps,
                   "method": "CUDA graphs of whole steps: pinned H2D of x and ids, lora_linear, D2H of y by the "
                             "copy engines, on two side streams overlapping neighbouring steps; input sets rotated "
                             "as in the device timing"}
    eager = {"value": wl.M / (ms_eager * 1e-3), "ms_per_step": ms_eager, "steps": n_eager}
    try:
        link = run_e2e_host_link(wl, sets, L, steps, stream, hx, hids)
    except L.LoraError as e:   # pinned memory not mapped for the device: the copy engines only
        return {**copy_engine, "host_link": {"unavailable": str(e)}, "eager_one_stream": eager}
    best = link if link["ms_per_step"] < copy_engine["ms_per_step"] else copy_engine
    other = copy_engine if best is link else link
    return {**best, "other_method": {k: other[k] for k in ("value", "ms_per_step", "method")},
            "eager_one_stream": eager}


def run_e2e_host_link(wl, sets, L, steps, stream, hx, hids):
    """The end-to-end step with the SMs moving the bytes across the host
    link: lora_copy_async copies x and lora_id_map from pinned host memory
    into the step's input set, and the layer writes y straight into pinned
    host memory; both are programmatic dependent launches on one stream, so
    a step is two kernels in a row and each may start while the one ahead of
    it finishes.  Replayed from CUDA graphs, input sets rotated."""
    ns = len(sets)
    hy = [torch.full((wl.M, wl.N), float("nan"), dtype=torch.bfloat16).pin_memory() for _ in range(ns)]
    h2d = hx.numel() * hx.element_size() + hids.numel() * hids.element_size()
    d2h = hy[0].numel() * hy[0].element_size()

    def step(i):
        st = sets[i % ns]
        L.copy_async([(st.x, hx), (st.ids, hids)], stream=stream)
        L.lora_linear(st.x, st.W, st.bias, st.ids, st.pool, wl.scale, st.ws, y=hy[i % ns], stream=stream,
                      static_weights=True)

    with torch.cuda.stream(stream):
        for i in range(2 * ns):
            step(i)
    torch.cuda.synchronize()

    def capture(n):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(g, stream=stream):
                for i in range(n):
                    step(i)
        return g

    chunk = min(steps, 200)
    full, rem = divmod(steps, chunk)
    g_full = capture(chunk) if full else None
    g_rem = capture(rem) if rem else None
    for g in (g_full, g_rem):
        if g is not None:
            g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(full):
            g_full.replay()
        if g_rem is not None:
            g_rem.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    for b in range(min(ns, steps)):
        if not torch.equal(hy[b], sets[b].y.cpu()):
            raise RuntimeError("end-to-end host-link output differs from the device output")
    return {"value": wl.M / (ms * 1e-3), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": ms, "steps": steps,
            "method": "CUDA graphs of whole steps on one stream: lora_copy_async (x and ids from pinned host "
                      "memory, copied by the SMs over the host link), then lora_linear writing y straight into "
                      "pinned host memory; input sets rotated as in the device timing"}


def aggregate(ms_local: float, tokens_per_rank: int, world: int, all_reduce_max):
    """Whole-job numbers of `world` independent replicas: the step time is the
    slowest rank's, the throughput counts every rank's tokens."""
    ms = all_reduce_max(ms_local)
    return ms, world * tokens_per_rank / (ms * 1e-3)


def cpu_baseline(name, budget_s=8.0):
    """The CPU oracle as it stands, on whole rows of the same workload."""
    from oracle import oracle
    wl = workloads.make_config(name)
    prep = oracle.Prepared(wl)
    rows_done, t_used, reps = 0, 0.0, 0
    rng = np.random.default_rng(0)
    per_call = min(wl.M, max(1, oracle.num_threads()))
    while t_used < budget_s and reps < 1000:
        rows = rng.integers(0, wl.M, per_call) if per_call < wl.M else np.arange(wl.M)
        t0 = time.perf_counter()
        oracle.lora_linear_rows_prepared(prep, rows)
        t_used += time.perf_counter() - t0
        rows_done += len(rows)
        reps += 1
    return {"value": rows_done / t_used, "unit": "tokens/s", "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"{rows_done} whole output rows of the {name} workload ({reps} calls of {per_call} rows), "
                      f"{t_used:.1f} s of CPU time, fp64 plain loops, OpenMP over rows"}


def roofline(r, wl, kname, config, peaks, peak_kind):
    """Roofline of the dominant kernel.  The decode-sized schedule builds the
    segment table inside its one launch, so a decode step is exactly one
    launch of that kernel: its duration is the step's own back-to-back time
    over the timed region.  The larger schedules follow a separate builder
    launch: their kernel is timed alone with the tables prebuilt.  Beside it,
    the same kernel launched alone after an idle gap (launch start-up
    included, nothing overlapped)."""
    one_launch = kname == "lora_cluster_kernel"
    if one_launch:
        kern_ms, iso_ms = r["ms_per_step"], r["iso_step_ms"]
        method = ("one launch per step (the segment build runs inside the decode kernel): the step's mean "
                  "time over the timed region, back to back in CUDA graphs, CUDA events on the launching stream")
    else:
        kern_ms, iso_ms = r["kernel_ms"], r["iso_kernel_ms"]
        method = ("the fused kernel alone (segment tables prebuilt), mean over back-to-back launches in CUDA "
                  "graphs, CUDA events on the launching stream")
    hbm_bound = wl.M <= 128
    if hbm_bound:
        work, peak, unit, scale, nominal = r["bytes"], peaks["hbm_gbs"], "GB/s", 1e9, NOMINAL_HBM_GBS
        roof = {"bound": "hbm"}
    else:
        work, peak, unit, scale, nominal = r["flops"], peaks["bf16_tflops"], "TFLOP/s", 1e12, NOMINAL_BF16_TFLOPS
        roof = {"bound": "tensor"}
    achieved = work / (kern_ms * 1e-3) / scale
    iso = work / (iso_ms * 1e-3) / scale
    roof.update({"achieved": round(achieved, 1), "peak": peak, "unit": unit, "frac": round(achieved / peak, 4),
                 "traffic": profiled_traffic(kname, config), "kernel": kname,
                 "kernel_us": round(kern_ms * 1e3, 3), "kernel_time_method": method,
                 "isolated_us": round(iso_ms * 1e3, 3), "isolated_achieved": round(iso, 1),
                 "isolated_frac": round(iso / peak, 4),
                 "nominal_peak": nominal, "frac_of_nominal": round(achieved / nominal, 4),
                 "isolated_method": "median of 200 single calls, each after a device synchronize (idle GPU), "
                                    "CUDA events on the launching stream around the one call; the launch's own "
                                    "start-up is included and nothing overlaps it",
                 "algorithmic_bytes": r["bytes"], "algorithmic_flops": r["flops"],
                 "peak_source": f"{peak_kind} ({'MEASURED_PEAKS.json' if peak_kind == 'measured' else 'recipe fallback'})"})
    if one_launch:
        roof["kernel_prebuilt_tables_us"] = round(r["kernel_ms"] * 1e3, 3)
    return roof


def ours(args):
    from segmented_gemm_gb300 import lora as L
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    L.load_library()
    stream = torch.cuda.Stream(device)
    barrier = (lambda: dist.barrier()) if dist else None
    peaks, peak_kind = load_peaks()

    sampler = ClockSampler(local)
    r = run_config(args.config, L, device, args.steps, args.warmup, stream, sampler=sampler,
                   dist_barrier=barrier, compare_plain=True)
    wl = r["wl"]
    def all_reduce_max(v):
        if not dist:
            return v
        t = torch.tensor([v], device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        return float(t.item())

    ms, value = aggregate(r["ms_per_step"], wl.M, world, all_reduce_max)

    # roofline of the dominant kernel (the fused layer)
    kname = dominant_kernel(wl)
    roof = roofline(r, wl, kname, args.config, peaks, peak_kind)

    out = {
        "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 6), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded, bf16-rounded N(0,s) draws)",
        "config": {"workload": CONFIG_TEXT[args.config], "M": wl.M, "K": wl.K, "N": wl.N,
                   "num_adapters": wl.num_adapters, "adapters_present": r["n_present"],
                   "parallelism": f"replicas x{world} (independent batches)",
                   "l2": f"rotating {r['n_sets']} input sets of {r['set_bytes'] / 1e6:.1f} MB "
                         f"({r['n_sets'] * r['set_bytes'] / 1e6:.0f} MB > L2)" if r["n_sets"] > 1 else
                         f"inputs {r['set_bytes'] / 1e6:.0f} MB > 4x L2",
                   "timing": "CUDA graphs of whole steps (segment build + fused layer), CUDA events",
                   "static_weights": "weights loaded once; each call may stream them before the previous "
                                     "call ends (LORA_FLAG_STATIC_WEIGHTS)"},
        "roofline": roof,
        "tflops": round(r["flops"] / (ms * 1e-3) / 1e12, 2),
        "e2e": {k: r["e2e"][k] for k in ("value", "unit", "h2d_bytes_per_step", "d2h_bytes_per_step", "method",
                                          "other_method", "host_link", "eager_one_stream") if k in r["e2e"]},
        # our kernels per timed step: the decode kernel builds its own segment
        # table; the other schedules follow a builder launch
        "gpu_launches": (1 if kname == "lora_cluster_kernel" else 2) * args.steps,
        "clocks": r["clocks"],
        "device_status": r["status"],
        "without_static_weights": r["plain"],
        "torch_base_only": {"us": round(r["base_ms"] * 1e3, 3),
                            "method": "cuBLAS through torch.addmm: x W^T + bias alone (no LoRA term) on the same "
                                      "rotating inputs, back to back in CUDA graphs, CUDA events"},
    }
    if world == 1 and rank == 0 and not args.no_cpu:
        out["cpu_baseline"] = cpu_baseline(args.config)
    if not args.no_sweep and rank == 0:
        sweep = {}
        lines = set(args.sweep.split(","))
        for name in ("prefill", "qkv", "mlp_down", "qkv_sliced", "decode_e4m3", "decode_all_base"):
            if name == args.config or name not in lines:
                continue
            samp = ClockSampler(local)
            nsteps = 30 if name == "mlp_down" else 2000 if name.startswith("decode") else 100
            s = run_config(name, L, device, nsteps, 5 if nsteps < 1000 else 100, stream, e2e=False, sampler=samp)
            kt = s["kernel_ms"] * 1e-3
            sk = dominant_kernel(s["wl"])
            sweep[name] = {
                **({"workload": SWEEP_EXTRA[name]} if name in SWEEP_EXTRA else {}),
                "M": s["wl"].M, "tokens_per_s": round(s["wl"].M / (s["ms_per_step"] * 1e-3), 1),
                "ms_per_step": round(s["ms_per_step"], 5), "kernel_us": round(s["kernel_ms"] * 1e3, 2),
                "kernel_tflops": round(s["flops"] / kt / 1e12, 1),
                "tensor_frac": round(s["flops"] / kt / 1e12 / peaks["bf16_tflops"], 4),
                "hbm_gbs": round(s["bytes"] / kt / 1e9, 1),
                "roofline": roofline(s, s["wl"], sk, name, peaks, peak_kind),
                "torch_base_only_us": round(s["base_ms"] * 1e3, 2),
                "clocks": s["clocks"], "device_status": s["status"]}
            del s
            torch.cuda.empty_cache()
        if "attention_block_prefill" in lines:
            sweep["attention_block_prefill"] = run_layer_step(L, device, 100, 5, stream)
            torch.cuda.empty_cache()
        if "moe_experts" in lines:
            sweep["moe_experts"] = run_moe_step(L, device, 100, 5, stream, peaks)
            torch.cuda.empty_cache()
        out["sweep"] = sweep
    if rank == 0:
        print(json.dumps(out), flush=True)
    if dist:
        dist.destroy_process_group()


# ---------------------------------------------------------------------------
# reference arm: the CPU oracle
# ---------------------------------------------------------------------------

def reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from oracle import oracle
    wl = workloads.make_config(args.config)
    prep = oracle.Prepared(wl)
    rng = np.random.default_rng(0)
    # size each step's sample so the whole run takes about a minute: whole
    # rows (the oracle's row routine) when a step can afford a batch of rows,
    # else single output elements
    budget = 60.0
    per_step = budget / max(1, args.steps + args.warmup)
    threads = oracle.num_threads()
    row_batch = min(wl.M, threads)
    t0 = time.perf_counter()
    oracle.lora_linear_rows_prepared(prep, rng.integers(0, wl.M, row_batch))
    t_rows = time.perf_counter() - t0
    if t_rows <= per_step:
        nb = max(1, int(per_step / t_rows))
        n_rows = min(wl.M, row_batch * nb)

        def step():
            oracle.lora_linear_rows_prepared(prep, rng.integers(0, wl.M, n_rows))
        per_step_tokens = float(n_rows)
        sample = f"each step: {n_rows} random whole output rows of the {args.config} workload"
    else:
        probe_n = 256
        t0 = time.perf_counter()
        oracle.lora_linear_elems(prep, rng.integers(0, wl.M, probe_n), rng.integers(0, wl.N, probe_n))
        per_elem = (time.perf_counter() - t0) / probe_n
        n = int(max(1, min(wl.M * wl.N, per_step / per_elem)))

        def step():
            oracle.lora_linear_elems(prep, rng.integers(0, wl.M, n), rng.integers(0, wl.N, n))
        per_step_tokens = n / wl.N
        sample = (f"each step: {n} random output elements of the {args.config} workload "
                  f"(N elements count as one token)")
    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = time.perf_counter() - t0
    value = args.steps * per_step_tokens / dt
    ms = dt * 1e3 / args.steps
    cores = oracle.num_threads()
    out = {"impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "tokens/s", "n_gpus": 0,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
           "config": {"workload": CONFIG_TEXT[args.config], "M": wl.M, "K": wl.K, "N": wl.N,
                      "num_adapters": wl.num_adapters},
           "cpu_baseline": {"value": round(value, 3), "unit": "tokens/s", "cores": cores, "kind": "oracle",
                            "sample": sample},
           "e2e": {"value": round(value, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", choices=list(CONFIG_TEXT), default="decode")
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--sweep", default=",".join(SWEEP_LINES),
                    help="comma-separated sweep lines to run (default: all of %s)" % ", ".join(SWEEP_LINES))
    ap.add_argument("--max-sets", type=int, default=None,
                    help="cap the rotating input sets (for small ncu captures; the L2 note in config says so)")
    args = ap.parse_args()
    global MAX_SETS
    MAX_SETS = args.max_sets
    args.warmup = max(3, args.warmup)
    if args.impl == "reference":
        reference(args)
    else:
        ours(args)


if __name__ == "__main__":
    main()
