#!/usr/bin/env python
"""Decode-step benchmark of the compressed-KV attention path on one GB300.

Workload (default): the LLaVA-OneVision-7B-shaped decode step -- 28 layers,
B = 1, 28 query / 4 KV heads, D = 128, a history of 14 text + 6273 visual
positions (K INT4, V INT2, group 64, KV head 0 protected in bf16).  One step
= for every layer: kvq_decode_step, which stores the step's own K/V row (a
text position, kept bf16) in the cache and attends over the history plus that
row in one launch (--fused no: the two-call form,
kvq_quantize_append of the row then kvq_decode_attention).  The history is
quantised once before timing (prefill).

value  = algorithmic bytes per step / device time per step (GB/s), where the
         bytes are the compressed cache rows actually attended, q, out and
         the appended row (read + write); ms_per_step is the same time.
e2e    = the same step through the public API with pinned HOST buffers: the
         H2D copy of every layer's q and step K/V and the D2H copy of every
         layer's output are inside the timed region.
L2 is flushed (a write of 2x the L2 size) before every timed step, outside
the timed interval.

--impl reference times the CPU oracle (test infrastructure) on the host
cores, each step a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import synth  # noqa: E402

# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) per launch of the
# roofline kernel from one ncu capture, keyed by the hash of the CUDA sources
# it was taken with (kernel_source_hash) and then by (workload, layers,
# fused).  A source change makes the key miss, so a stale count is reported
# as null rather than carried over.
NCU_TRAFFIC = {
    # kernel source hash -> {(workload, layers, fused): DRAM bytes read + written per launch}
    "6b7fc1ccd8e0d8e4": {("llava_ov_7b", 28, True): 5453440},  # mean of two steady-state launches
}

# Extra workloads timed in every default run (the "sweep" object of the JSON
# line): (workload, history T or None, layer ids or None = all layers).
SWEEP = [
    ("longctx", 4096, None),
    ("longctx", 16384, None),
    ("longctx", 32768, None),
    ("llava15_7b", None, None),
    ("llava_next_13b", None, [0, 4]),
]


def kernel_source_hash() -> str:
    """First 16 hex digits of the SHA-256 of the library's sources (the
    kernels, their headers and the public header), in a fixed order."""
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "bit_mixed_precision_kvq_gb300", "csrc")
    files = sorted(f for f in os.listdir(csrc) if f.endswith((".cu", ".cuh", ".h", ".cpp")))
    for f in files + ["../../include/kvq.h"]:
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]

METRIC = ("decode-attention µs/step and achieved HBM GB/s (compressed bytes) vs 8 TB/s peak")
UNIT = "GB/s"


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="llava_ov_7b")
    ap.add_argument("--T", type=int, default=None, help="history length for the longctx workload")
    ap.add_argument("--layers", type=int, default=None, help="limit layers (parity/debug only)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-sweep", action="store_true",
                    help="skip the other workloads' per-launch lines (long context 4K/16K/32K, "
                         "LLaVA-1.5, LLaVA-Next decode and append)")
    ap.add_argument("--fused", choices=["yes", "no"], default="yes",
                    help="kvq_decode_step (one launch per layer) or append + decode (three)")
    ap.add_argument("--prefill-in-step", choices=["auto", "yes", "no"], default="auto",
                    help="include kvq_quantize_append of the whole bf16 history in every step "
                         "(auto: yes for llava_next_13b, whose step includes the prefill)")
    ap.add_argument("--n-q", type=int, default=1,
                    help="query tokens per sequence and step: > 1 appends n_q rows and runs "
                         "kvq_decode_attention_mq (multi-query decode) per layer")
    ap.add_argument("--preload", choices=["yes", "no"], default="yes",
                    help="kvq_set_cache_preload: each layer's kernel copies its first cache tiles "
                         "while the previous layer's kernel runs (no other kernel writes the caches)")
    ap.add_argument("--probe", action="store_true",
                    help="instead of the decode step: the K-vs-V sensitivity study "
                         "(kvq_sensitivity_probe) on the workload's synthetic cache")
    return ap.parse_args()


# ---------------------------------------------------------------------------
# distributed plumbing (replicas: one independent copy of the workload per rank)
# ---------------------------------------------------------------------------

def dist_setup(use_cuda: bool):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        if use_cuda:
            torch.cuda.set_device(local)
        dist.init_process_group("nccl" if use_cuda else "gloo", rank=rank, world_size=world)
    return rank, world, local


def barrier(world: int, use_cuda: bool):
    if use_cuda:
        torch.cuda.synchronize()
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    if use_cuda:
        torch.cuda.synchronize()


def max_over_ranks(x: float, world: int, use_cuda: bool) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if use_cuda else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x: float, world: int, use_cuda: bool) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if use_cuda else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ---------------------------------------------------------------------------
# clocks (sampled with nvidia-smi during the timed region)
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


# ---------------------------------------------------------------------------
# algorithmic bytes
# ---------------------------------------------------------------------------

def decode_bytes(L, T: int, n_q: int = 1) -> int:
    """Compressed cache bytes a decode over positions [0, T) must read (once,
    whatever the number n_q of query tokens), plus q and out.  A packed
    visual row costs its codes plus its fp16 scale/zero."""
    d = L.d
    vsa, vea = min(d.vis_start, T), min(d.vis_end, T)
    n_vis = vea - vsa
    n_txt = T - n_vis
    bf16_row = 2 * d.D
    packed = sum(int(L.row_bytes[s]) for s in range(4))  # K codes, K s/z, V codes, V s/z
    konly = bf16_row + int(L.row_bytes[2]) + int(L.row_bytes[3])  # bf16 K, packed V
    per_b = (d.H_kv * n_txt * 2 * bf16_row + L.n_prot * n_vis * 2 * bf16_row
             + L.n_packed * n_vis * packed + L.n_konly * n_vis * konly)
    qo = 2 * d.B * n_q * d.H_q * d.D * 2
    return d.B * per_b + qo


def append_bytes(L, n_tok: int) -> int:
    """Read of the step's bf16 K/V rows plus the write of their cache rows
    (text positions: bf16)."""
    d = L.d
    return 2 * (d.B * d.H_kv * n_tok * 2 * 2 * d.D)


def prefill_bytes(L, T: int) -> int:
    """Quantise-append of positions [0, T): read the bf16 K and V rows, write
    their cache rows (packed codes + scale/zero for visual rows of packed
    heads, bf16 otherwise)."""
    d = L.d
    n_vis = min(d.vis_end, T) - min(d.vis_start, T)
    n_txt = T - n_vis
    read = 2 * d.B * d.H_kv * T * 2 * d.D
    packed = sum(int(L.row_bytes[s]) for s in range(4))
    write = d.B * (d.H_kv * n_txt * 4 * d.D + L.n_prot * n_vis * 4 * d.D + L.n_packed * n_vis * packed)
    return read + write


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

class Model:
    """Per-layer caches (history quantised once), per-step inputs, outputs."""

    def __init__(self, w: synth.Workload, dev, n_layers: int, prefill_in_step: bool = False,
                 fused: bool = True, n_q: int = 1, layer_ids=None):
        import bit_mixed_precision_kvq_gb300 as kvq
        self.kvq = kvq
        self.n_q = n_q
        self.fused = fused and n_q == 1  # multi-query: append the rows, then decode
        self.w = w
        self.T_hist = w.T
        self.T = w.T + n_q
        self.prefill_in_step = prefill_in_step
        self.layers = []
        self.ws = {}  # one workspace per unit count (its counter area is sized by it)
        self.layer_ids = list(range(n_layers)) if layer_ids is None else list(layer_ids)
        n_layers = len(self.layer_ids)
        for l in self.layer_ids:
            ls = w.layers[l]
            L = kvq.cache_layout(w.B, w.H_q, w.H_kv, w.D, self.T, w.vis_start, w.vis_end,
                                 ls.k_bits, ls.v_bits, w.group_size, ls.protected)
            cache = torch.empty(int(L.total_bytes), dtype=torch.uint8, device=dev)
            k = synth.make_kv(w, l, "k", dev)
            v = synth.make_kv(w, l, "v", dev)
            kvq.quantize_append(L, cache, k, v, 0)
            layer = dict(L=L, cache=cache)
            if prefill_in_step:  # the bf16 history stays resident as the step's input
                layer["k"], layer["v"] = k, v
            else:
                del k, v
            self.layers.append(layer)
            n = int(L.units)
            nb = kvq.decode_mq_workspace_bytes(L, n_q)
            if n not in self.ws or self.ws[n].numel() < nb:
                self.ws[n] = torch.zeros(nb, dtype=torch.uint8, device=dev)
            layer["ws"] = self.ws[n]
        nL = n_layers
        # per-step device inputs/outputs, packed per layer so that the e2e leg
        # moves them with one copy each way
        ids = self.layer_ids
        if n_q == 1:
            self.q = torch.stack([synth.make_q(w, l, 0, dev) for l in ids])
            self.out = torch.empty((nL, w.B, w.H_q, w.D), dtype=torch.bfloat16, device=dev)
        else:  # [layer][B][n_q][H_q][D]
            self.q = torch.stack([torch.stack([synth.make_q(w, l, s, dev) for s in range(n_q)], 1)
                                  for l in ids])
            self.out = torch.empty((nL, w.B, n_q, w.H_q, w.D), dtype=torch.bfloat16, device=dev)
        # the step's own K/V rows, [layer][B][H_kv][n_q][D]
        self.ks = torch.stack([torch.cat([synth.make_step_kv(w, l, "k", s, dev) for s in range(n_q)], 2)
                               for l in ids])
        self.vs = torch.stack([torch.cat([synth.make_step_kv(w, l, "v", s, dev) for s in range(n_q)], 2)
                               for l in ids])
        self.scale = 1.0 / math.sqrt(w.D)
        torch.cuda.synchronize()

    def step(self):
        kvq = self.kvq
        for l, ly in enumerate(self.layers):
            L = ly["L"]
            if self.prefill_in_step:
                kvq.quantize_append(L, ly["cache"], ly["k"], ly["v"], 0)
            self.decode_layer(l)

    def decode_layer(self, l: int):
        """The step's row into the cache + attention over [0, T)."""
        ly = self.layers[l]
        kvq, L = self.kvq, ly["L"]
        if self.fused:
            kvq.decode_step(L, ly["cache"], self.q[l], self.ks[l], self.vs[l], self.T_hist,
                            self.out[l], self.scale, None, ly["ws"])
        elif self.n_q > 1:
            kvq.quantize_append(L, ly["cache"], self.ks[l], self.vs[l], self.T_hist)
            kvq.decode_attention_mq(L, ly["cache"], self.q[l], self.T, self.out[l], self.scale, None,
                                    ly["ws"])
        else:
            kvq.quantize_append(L, ly["cache"], self.ks[l], self.vs[l], self.T_hist)
            kvq.decode_attention(L, ly["cache"], self.q[l], self.T, self.out[l], self.scale, None,
                                 ly["ws"])

    def launches_per_layer(self) -> int:
        return (1 if self.fused else 3) + (1 if self.prefill_in_step else 0)

    def prefill_layer(self, l: int):
        ly = self.layers[l]
        self.kvq.quantize_append(ly["L"], ly["cache"], ly["k"], ly["v"], 0)

    def step_bytes(self) -> int:
        b = sum(decode_bytes(ly["L"], self.T, self.n_q) + append_bytes(ly["L"], self.n_q)
                for ly in self.layers)
        if self.prefill_in_step:
            b += sum(prefill_bytes(ly["L"], self.T_hist) for ly in self.layers)
        return b


def time_decode_layers(model: "Model", flush, reps: int = 20) -> dict:
    """Per-launch device time of the model's layer decodes: a CUDA graph of
    every layer's decode back to back (as inside a step), L2 flushed before
    each replay, CUDA events on the launching stream; per launch = replay
    time / layers.  Returns median / p10 / p90 in microseconds."""
    n = len(model.layers)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for l in range(n):
            model.decode_layer(l)
    torch.cuda.synchronize()
    for _ in range(3):
        flush()
        g.replay()
    ev = []
    for _ in range(reps):
        flush()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        g.replay()
        b.record()
        ev.append((a, b))
    torch.cuda.synchronize()
    us = np.array([a.elapsed_time(b) * 1e3 / n for a, b in ev])
    return {"median": float(np.median(us)), "p10": float(np.percentile(us, 10)),
            "p90": float(np.percentile(us, 90))}


def time_prefill_layers(model: "Model", flush, reps: int = 3) -> float:
    """Mean device time (us) of one layer's quantise-append of its bf16
    history, L2 flushed before each launch."""
    ev = []
    for _ in range(reps):
        for l in range(len(model.layers)):
            flush()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            model.prefill_layer(l)
            b.record()
            ev.append((a, b))
    torch.cuda.synchronize()
    return float(np.mean([a.elapsed_time(b) * 1e3 for a, b in ev]))


def run_sweep(dev, flush, peak: float) -> list:
    """The other workloads of the pages, one entry each: the per-launch
    decode time (fused step per layer) of the listed layers with its
    algorithmic bytes and roofline fraction, and for LLaVA-Next the
    quantise-append of the bf16 history."""
    rows = []
    for name, T, ids in SWEEP:
        w = synth.workload(name, T)
        prefill = name == "llava_next_13b"
        model = Model(w, dev, w.n_layers, prefill_in_step=prefill, layer_ids=ids)
        model.step()  # eager warm-up
        torch.cuda.synchronize()
        t = time_decode_layers(model, flush)
        layer_bytes = float(np.mean([decode_bytes(ly["L"], model.T) + append_bytes(ly["L"], 1)
                                     for ly in model.layers]))
        gbs = layer_bytes / (t["median"] * 1e-6) / 1e9
        row = {"workload": w.name, "layers": model.layer_ids, "T": model.T,
               "kernel": "kvq_decode_step (one launch per layer)",
               "per_launch_us": round(t["median"], 3), "p10_us": round(t["p10"], 3),
               "p90_us": round(t["p90"], 3), "per_launch_bytes": int(layer_bytes),
               "achieved": round(gbs, 1), "peak": peak, "unit": "GB/s", "frac": round(gbs / peak, 4)}
        rows.append(row)
        if prefill:
            ap_us = time_prefill_layers(model, flush)
            ap_bytes = float(np.mean([prefill_bytes(ly["L"], model.T_hist) for ly in model.layers]))
            ap_gbs = ap_bytes / (ap_us * 1e-6) / 1e9
            rows.append({"workload": w.name, "layers": model.layer_ids, "T": model.T_hist,
                         "kernel": "append_kernel (kvq_quantize_append of the bf16 history)",
                         "per_launch_us": round(ap_us, 2), "per_launch_bytes": int(ap_bytes),
                         "achieved": round(ap_gbs, 1), "peak": peak, "unit": "GB/s",
                         "frac": round(ap_gbs / peak, 4)})
        del model
        torch.cuda.empty_cache()
    return rows


def run_ours(args, rank, world, local):
    import __graft_entry__
    __graft_entry__.build()
    dev = torch.device("cuda", local)
    w = synth.workload(args.workload, args.T)
    n_layers = args.layers or w.n_layers
    prefill = (args.prefill_in_step == "yes" or
               (args.prefill_in_step == "auto" and args.workload == "llava_next_13b"))
    import bit_mixed_precision_kvq_gb300 as kvq
    kvq.set_cache_preload(args.preload == "yes")
    model = Model(w, dev, n_layers, prefill_in_step=prefill, fused=(args.fused == "yes"), n_q=args.n_q)
    props = torch.cuda.get_device_properties(dev)
    l2 = int(getattr(props, "L2_cache_size", 128 << 20))
    flush_buf = torch.empty(max(2 * l2, 256 << 20), dtype=torch.uint8, device=dev)

    def flush():
        flush_buf.fill_(1)

    # eager warm-up (first calls cache the SM count), then capture one step
    model.step()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        model.step()
    torch.cuda.synchronize()
    launches_per_step = model.launches_per_layer() * n_layers

    for _ in range(max(3, args.warmup)):
        flush()
        graph.replay()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    clocks = ClockSampler(local)
    barrier(world, True)
    clocks.start()
    t_wall = time.perf_counter()
    for i in range(args.steps):
        flush()
        ev[i][0].record()
        graph.replay()
        ev[i][1].record()
    barrier(world, True)
    t_wall = time.perf_counter() - t_wall
    clk = clocks.stop()
    step_ms = np.array([a.elapsed_time(b) for a, b in ev])
    dev_ms = float(step_ms.sum())
    dev_ms = max_over_ranks(dev_ms, world, True)
    step_bytes = model.step_bytes()
    total_bytes = sum_over_ranks(float(step_bytes) * args.steps, world, True)
    ms_per_step = dev_ms / args.steps
    value = total_bytes / (dev_ms * 1e-3) / 1e9

    # roofline: the decode of one layer (the fused step kernel, or append +
    # split + combine), timed with events on the launching stream around a
    # CUDA graph of every layer's decode (back-to-back, as in the step), L2
    # flushed before each replay; per launch = replay time / layers
    rl = time_decode_layers(model, flush)
    launch_ms = rl["median"] * 1e-3
    layer_bytes = float(np.mean([decode_bytes(ly["L"], model.T, model.n_q) + append_bytes(ly["L"], model.n_q)
                                 for ly in model.layers]))
    peaks = {}
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            peaks = json.load(f)
    except OSError:
        pass
    peak = float(peaks.get("hbm_gbs", 6800.0))
    achieved = layer_bytes / (launch_ms * 1e-3) / 1e9

    append_line = None
    if prefill:
        ap_us = time_prefill_layers(model, flush)
        ap_bytes = float(np.mean([prefill_bytes(ly["L"], model.T_hist) for ly in model.layers]))
        ap_gbs = ap_bytes / (ap_us * 1e-6) / 1e9
        append_line = {"kernel": "append_kernel (kvq_quantize_append of the bf16 history)",
                       "per_launch_us": round(ap_us, 2), "per_launch_bytes": int(ap_bytes),
                       "achieved": round(ap_gbs, 1), "peak": peak, "unit": "GB/s",
                       "frac": round(ap_gbs / peak, 4)}

    # e2e: pinned host buffers in, outputs back, all inside the timed region
    h_q = torch.empty(model.q.shape, dtype=model.q.dtype, pin_memory=True)
    h_ks = torch.empty(model.ks.shape, dtype=model.ks.dtype, pin_memory=True)
    h_vs = torch.empty(model.vs.shape, dtype=model.vs.dtype, pin_memory=True)
    h_out = torch.empty(model.out.shape, dtype=model.out.dtype, pin_memory=True)
    h_q.copy_(model.q)
    h_ks.copy_(model.ks)
    h_vs.copy_(model.vs)
    e2e_ev = []
    for i in range(args.steps):
        flush()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        model.q.copy_(h_q, non_blocking=True)
        model.ks.copy_(h_ks, non_blocking=True)
        model.vs.copy_(h_vs, non_blocking=True)
        graph.replay()
        h_out.copy_(model.out, non_blocking=True)
        b.record()
        e2e_ev.append((a, b))
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(sum(a.elapsed_time(b) for a, b in e2e_ev), world, True)
    h2d = (h_q.numel() + h_ks.numel() + h_vs.numel()) * 2
    d2h = h_out.numel() * 2
    e2e_value = total_bytes / (e2e_ms * 1e-3) / 1e9

    m_T, m_nq, m_fused = model.T, model.n_q, model.fused
    sweep = None
    if world == 1 and not args.no_sweep and args.workload == "llava_ov_7b" and args.layers is None \
            and args.n_q == 1 and args.fused == "yes":
        del graph, model
        torch.cuda.empty_cache()
        sweep = run_sweep(dev, flush, peak)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, n_layers=min(4, n_layers))

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
        "us_per_step": round(ms_per_step * 1e3, 2),
        "step_us_median_p10_p90": [round(float(np.median(step_ms)) * 1e3, 2),
                                   round(float(np.percentile(step_ms, 10)) * 1e3, 2),
                                   round(float(np.percentile(step_ms, 90)) * 1e3, 2)],
        "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "u8/u4/u2 codes + bf16; fp32 accumulate",
        "data": "synthetic (seeded; shapes of the pages' LLaVA-OneVision-7B video workload)",
        "config": {"workload": f"{w.name}: {n_layers} layers, B={w.B}, H_q={w.H_q}, "
                               f"H_kv={w.H_kv}, D={w.D}, T={m_T} (history {w.T} + current), "
                               f"K{w.layers[0].k_bits}/V{w.layers[0].v_bits} G{w.group_size}, "
                               f"protected {w.layers[0].protected}",
                   "bytes_per_step": step_bytes, "l2": "flushed before every timed step",
                   "graph": "one CUDA graph per step", "parallelism": f"replicas x{world}",
                   "query_tokens": m_nq, "cache_preload": args.preload == "yes"},
        "roofline": {"bound": "hbm",
                     "traffic": (NCU_TRAFFIC.get(kernel_source_hash(), {}).get((w.name, n_layers, m_fused))
                                 if m_nq == 1 else None),
                     "kernel_source_hash": kernel_source_hash(),
                     "kernel": ("split_mma_kernel<..., step> (kvq_decode_step, one launch)" if m_fused
                                else ("kvq_quantize_append + kvq_decode_attention_mq (3 launches)"
                                      if m_nq > 1 else
                                      "kvq_quantize_append + kvq_decode_attention (3 launches)")),
                     "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4),
                     "per_launch_bytes": int(layer_bytes), "per_launch_us": round(launch_ms * 1e3, 3),
                     "per_launch_us_p10_p90": [round(rl["p10"], 3), round(rl["p90"], 3)],
                     "peak_source": "MEASURED_PEAKS.json hbm_gbs (measured)" if peaks else
                                    "fallback 6800 GB/s"},
        "e2e": {"value": round(e2e_value, 2), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms / args.steps, 5)},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk,
        "wall_s_timed_region": round(t_wall, 3),
    }
    if append_line is not None:
        line["append"] = append_line
        line["config"]["step"] = "per layer: quantise-append of the bf16 history + current token, decode"
    if sweep is not None:
        line["sweep"] = sweep
    if cpu is not None:
        line["cpu_baseline"] = cpu
    if rank == 0:
        print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# CPU oracle (test infrastructure) as the baseline / reference arm
# ---------------------------------------------------------------------------

class OracleSample:
    """A bounded sample of the workload for the CPU oracle: the first
    `n_layers` layers of one decode step (history + current token)."""

    def __init__(self, w: synth.Workload, n_layers: int):
        self.w = w
        self.items = []
        self.bytes = 0
        for l in range(n_layers):
            ls = w.layers[l]
            k = torch.cat([synth.make_kv(w, l, "k"), synth.make_step_kv(w, l, "k", 0)], 2)
            v = torch.cat([synth.make_kv(w, l, "v"), synth.make_step_kv(w, l, "v", 0)], 2)
            q = synth.make_q(w, l, 0)
            self.items.append((synth.bf16_bits(q), synth.bf16_bits(k), synth.bf16_bits(v), ls))
            self.bytes += self._bytes(ls, w.T + 1) + 2 * (w.B * w.H_kv * 2 * 2 * w.D)

    def _bytes(self, ls, T):
        w = self.w
        D, G = w.D, w.group_size
        n_vis = min(w.vis_end, T) - min(w.vis_start, T)
        row = lambda b: D * b // 8 + (4 * D // G if b < 16 else 0)  # noqa: E731
        n_prot = len(ls.protected)
        per_b = (w.H_kv * (T - n_vis) * 4 * D + n_prot * n_vis * 4 * D
                 + (w.H_kv - n_prot) * n_vis * (row(ls.k_bits) + row(ls.v_bits)))
        return w.B * per_b + 4 * w.B * w.H_q * D

    def run(self, threads: int):
        import oracle
        w = self.w
        for q, k, v, ls in self.items:
            mask = [1 if h in ls.protected else 0 for h in range(w.H_kv)]
            oracle.decode_reference(q, k, v, w.vis_start, w.vis_end, mask, ls.k_bits, ls.v_bits,
                                    w.group_size, 1.0 / math.sqrt(w.D), threads=threads)


def cpu_baseline(w: synth.Workload, n_layers: int) -> dict:
    import oracle
    oracle.build_oracle()
    cores = oracle.online_cores()
    s = OracleSample(w, n_layers)
    s.run(cores)  # warm
    reps = 0
    t0 = time.perf_counter()
    while True:
        s.run(cores)
        reps += 1
        el = time.perf_counter() - t0
        if el > 10.0 or reps >= 20:
            break
    per = el / reps
    return {"value": round(s.bytes / per / 1e9, 4), "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{n_layers} of {w.n_layers} layers of one {w.name} decode step "
                      f"(history {w.T} + current), {reps} reps",
            "us_per_step_extrapolated": round(per * 1e6 * w.n_layers / n_layers, 1)}


def run_reference(args, rank, world, local):
    if rank != 0:
        return  # the oracle arm runs on rank 0 only; other ranks exit without work
    import oracle
    oracle.build_oracle()
    w = synth.workload(args.workload, args.T)
    cores = oracle.online_cores()
    s = OracleSample(w, n_layers=min(2, args.layers or w.n_layers))
    for _ in range(args.warmup):
        s.run(cores)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        s.run(cores)
    el = time.perf_counter() - t0
    value = s.bytes * args.steps / el / 1e9
    ms = el / args.steps * 1e3
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded)",
        "config": {"workload": f"{w.name}: 2 of {w.n_layers} layers per step (bounded sample), "
                               f"B={w.B}, H_q={w.H_q}, H_kv={w.H_kv}, T={w.T + 1}"},
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": "2 layers of one decode step per step"},
        "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# --probe: K-vs-V sensitivity study
# ---------------------------------------------------------------------------

PROBE_BITS = (8, 4, 2)
PROBE_NOUT = 1024
FP64_NOMINAL_TFLOPS = 1.25  # GB300 FP64, nominal


def run_probe(args):
    """The pages' K-vs-V comparison ("VLM_KV_Quantization", sections 3-4),
    model-free: for every layer of the workload and every bit-width, the same
    synthetic history is appended into a cache with only visual K quantised
    (V bits 16) and one with only visual V quantised (K bits 16), same group
    size, no protected head (the study removes every policy), and
    kvq_sensitivity_probe measures the divergences on each.  The readout is a
    fixed seeded N(0, 1) matrix of PROBE_NOUT rows.  Prints one JSON line with
    the means over (layer, query head) and the probe's device time."""
    import __graft_entry__
    __graft_entry__.build()
    import bit_mixed_precision_kvq_gb300 as kvq
    dev = torch.device("cuda", 0)
    w = synth.workload(args.workload, args.T)
    n_layers = args.layers or w.n_layers
    T = w.T
    g = torch.Generator().manual_seed(20261203)
    R = torch.randn((PROBE_NOUT, w.D), generator=g, dtype=torch.float32).to(dev)
    scale = 1.0 / math.sqrt(w.D)
    sums = {(b, side): np.zeros(3) for b in PROBE_BITS for side in "kv"}
    n_rows = 0
    times = []
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for l in range(n_layers):
        k = synth.make_kv(w, l, "k", dev)
        v = synth.make_kv(w, l, "v", dev)
        q = synth.make_q(w, l, 0, dev)
        for bits in PROBE_BITS:
            for side in "kv":
                kb, vb = (bits, 16) if side == "k" else (16, bits)
                L = kvq.cache_layout(w.B, w.H_q, w.H_kv, w.D, T, w.vis_start, w.vis_end, kb, vb,
                                     w.group_size, [])
                cache = torch.empty(int(L.total_bytes), dtype=torch.uint8, device=dev)
                kvq.quantize_append(L, cache, k, v, 0)
                res = torch.empty((w.B, w.H_q, 3), dtype=torch.float64, device=dev)
                ws = torch.empty(kvq.probe_workspace_bytes(L, T), dtype=torch.uint8, device=dev)
                torch.cuda.synchronize()
                ev0.record()
                kvq.sensitivity_probe(L, cache, q, k, v, T, R, res, scale, ws)
                ev1.record()
                torch.cuda.synchronize()
                times.append(ev0.elapsed_time(ev1) * 1e3)
                sums[(bits, side)] += res.double().sum(dim=(0, 1)).cpu().numpy()
        n_rows += w.B * w.H_q
        del k, v
    table = {}
    for bits in PROBE_BITS:
        mk, mv = sums[(bits, "k")] / n_rows, sums[(bits, "v")] / n_rows
        table[str(bits)] = {"k_kl_attn": mk[0], "k_kl_out": mk[1], "v_kl_out": mv[1],
                            "k_over_v_kl_out": mk[1] / mv[1] if mv[1] > 0 else None,
                            "k_err": mk[2], "v_err": mv[2]}
    us = float(np.median(times))
    flops = 8.0 * w.D * w.B * w.H_q * T  # two score dots and two output sums per position, fp64
    achieved = flops / (us * 1e-6) / 1e12
    line = {
        "metric": "K-vs-V sensitivity (model-free KL of attention weights and of a readout "
                  "distribution, K or V quantised alone)",
        "workload": w.name, "layers": n_layers, "group_size": w.group_size, "T": T,
        "readout_rows": PROBE_NOUT, "bits": table,
        "probe_us_per_layer": us,
        "roofline": {"bound": "alu", "achieved": achieved, "peak": FP64_NOMINAL_TFLOPS,
                     "unit": "TFLOP/s (fp64)", "frac": achieved / FP64_NOMINAL_TFLOPS,
                     "peak_source": "nominal GB300 FP64"},
        "data": "synthetic",
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    if args.probe:
        if not torch.cuda.is_available():
            raise SystemExit("bench.py --probe needs a CUDA GPU")
        run_probe(args)
        return
    if args.impl == "reference":
        rank, world, local = dist_setup(use_cuda=False)
        run_reference(args, rank, world, local)
        return
    if not torch.cuda.is_available():
        raise SystemExit("bench.py (ours) needs a CUDA GPU")
    rank, world, local = dist_setup(use_cuda=True)
    run_ours(args, rank, world, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
