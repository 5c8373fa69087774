"""Benchmark of the MSA hot path on one GB300 (or N independent replicas under torchrun).

One step = one pass of the whole path:
  * prefill at 128K context (index block scores -> per-KV-head top-k -> sparse attention),
    which gives the headline value in tokens/s, and
  * one decode step over a batch of 8 sequences with 1M-token caches (index scan -> top-k
    -> split-KV sparse attention -> log-sum-exp merge), reported as us/step.
Inputs are seeded synthetic tensors resident in HBM; L2 is flushed (a 256 MiB write)
before each timed kernel sequence, outside the timed events.  Times are CUDA events on
the launching stream.  ``--impl reference`` times the fp64 CPU oracle instead, on a
bounded sample of the same workload.
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

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from block_sparse_gqa_02_gb300 import _lib, api  # noqa: E402
from block_sparse_gqa_02_gb300.configs import CONFIGS  # noqa: E402
from block_sparse_gqa_02_gb300.inputs import make_inputs  # noqa: E402

METRIC = "MSA prefill tokens/s and decode µs/step at 128K/1M ctx; % of TC/HBM roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# --------------------------------------------------------------------- work model

def prefill_flops(cfg):
    """Algorithmic FLOPs of one prefill: (index, sparse attention), causal pairs only."""
    T, NI, dI, Hq, d = cfg.seq, cfg.n_heads_kv, cfg.index_dim, cfg.n_heads_q, cfg.head_dim
    index = T * (T + 1) / 2 * NI * 2 * dI
    t = np.arange(T, dtype=np.int64)
    last = np.minimum(T - 1, (t // cfg.q_tile) * cfg.q_tile + cfg.q_tile - 1)
    cb = last // cfg.block_size
    keys = (np.minimum(cfg.top_k, cb + 1) - 1) * cfg.block_size + (t - cfg.block_size * cb + 1)
    sparse = float(keys.sum()) * Hq * 4 * d
    dense = T * (T + 1) / 2 * Hq * 4 * d
    return index, sparse, dense


def decode_bytes(cfg):
    """Compulsory HBM bytes of one decode step: (index scan, selected K/V + rest)."""
    B, L, NI, dI, d, Hq = cfg.batch, cfg.seq, cfg.n_heads_kv, cfg.index_dim, cfg.head_dim, \
        cfg.n_heads_q
    nB = -(-L // cfg.block_size)
    scan = B * L * dI * 2 + B * NI * dI * 2 + B * NI * nB * 4
    sel_keys = min(cfg.top_k * cfg.block_size, L)
    kv = B * NI * sel_keys * d * 2 * 2
    rest = B * NI * nB * 4 + B * Hq * d * 2 * 2 + B * Hq * 4
    dense = B * NI * L * d * 2 * 2 + B * L * dI * 2
    return scan, kv + rest, dense


# DRAM traffic per launch from ncu captures (profiles/), valid only for the kernel source
# that was profiled: a changed kernel reports null until it is captured again.
MEASURED_TRAFFIC = {
    "sparse_prefill_tc.cu": {
        "sha256_16": "588f5883e19a3dce",
        "workload": "p128k",
        "bytes_per_launch": 4.53e9,
        "how": "dram__bytes_read.sum + dram__bytes_write.sum of one launch at 65536 tokens "
               "with the 128K config's heads (1218.7 + 1045.3 MB), scaled by the (token, query "
               "head) rows to 128K (x2)",
    },
    "index_scan_tc.cu": {
        "sha256_16": "966bdbcd089ab6e4",
        "workload": "d1m",
        "bytes_per_launch": 2.18e9,
        "how": "dram__bytes_read.sum + dram__bytes_write.sum of one launch with 131072-token "
               "caches (268.5 + 3.9 MB), scaled by the cache length to 1M (x8)",
    },
}


def measured_traffic(kernel_file: str, workload: str):
    import hashlib
    rec = MEASURED_TRAFFIC.get(kernel_file)
    if rec is None or rec["workload"] != workload:
        return None
    path = os.path.join(ROOT, "block_sparse_gqa_02_gb300", "csrc", kernel_file)
    with open(path, "rb") as f:
        if hashlib.sha256(f.read()).hexdigest()[:16] != rec["sha256_16"]:
            return None
    return rec["bytes_per_launch"]


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    return FALLBACK_PEAKS, "fallback"


# ------------------------------------------------------------------- multi-rank

def max_over_ranks(x: float, world: int, device) -> float:
    """The largest value any rank holds (each rank times its own replica; the job's time is
    the slowest rank's).  A timing reduction only: no data of the path crosses ranks."""
    if world <= 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def whole_job_throughput(units_per_step: float, steps: int, world: int, max_ms: float) -> float:
    """Units all ranks processed divided by the slowest rank's time (weak scaling)."""
    return world * units_per_step * steps / (max_ms / 1e3)


# ------------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples (every 50 ms) of the SM clock and throttle reasons while running."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, FileNotFoundError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        loaded = [s for s, p in zip(sm, power) if p >= 0.5 * max(power)] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm),
                "power_w_max": max(power)}


# -------------------------------------------------------------------- our arm

class Step:
    """Inputs, outputs and events of one workload, resident on the device."""

    def __init__(self, cfg, device):
        self.cfg = cfg
        self.x = make_inputs(cfg, device=device)
        self.shape = _lib.shape_from_config(cfg)
        dt = self.x["q"].dtype
        if cfg.mode == "decode":
            self.bufs = api.alloc_decode_outputs(self.shape, device, dt)
            self.kernels = 4
        else:
            self.bufs = api.alloc_prefill_outputs(self.shape, device, dt)
            self.kernels = 3
        self.ev = []

    def run(self, stream, record=False):
        x, s, b = self.x, self.shape, self.bufs
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(4)] if record else None
        if record:
            evs[0].record(stream)
        _lib.msa_index_scores(s, x["idx_q"], x["idx_k"], b["scores"], stream)
        if record:
            evs[1].record(stream)
        _lib.msa_block_topk(s, b["scores"], b["sel"], stream)
        if record:
            evs[2].record(stream)
        if self.cfg.mode == "decode":
            _lib.msa_sparse_decode(s, x["q"], x["k"], x["v"], b["sel"], b["out"], b["lse"],
                                   b["ws"], None, stream)
        else:
            _lib.msa_sparse_prefill(s, x["q"], x["k"], x["v"], b["sel"], b["out"], b["lse"],
                                    None, 0, stream)
        if record:
            evs[3].record(stream)
            self.ev.append(evs)

    def times_ms(self):
        """Per step: (total, index, topk, attention) in ms."""
        out = []
        for e in self.ev:
            out.append((e[0].elapsed_time(e[3]), e[0].elapsed_time(e[1]),
                        e[1].elapsed_time(e[2]), e[2].elapsed_time(e[3])))
        return np.array(out)


def decode_graph_us(step, stream, flush, n):
    """Mean us per decode step when the step's library calls are replayed from a CUDA graph
    captured once (one launch for the whole step)."""
    g = torch.cuda.CUDAGraph()
    torch.cuda.synchronize()
    with torch.cuda.graph(g, stream=stream):
        step.run(stream, False)
    torch.cuda.synchronize()
    ts = []
    for i in range(n + 3):
        with torch.cuda.stream(stream):
            flush.fill_(1.0)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        with torch.cuda.stream(stream):
            g.replay()                                  # on the stream the events time
        e1.record(stream)
        if i >= 3:
            ts.append((e0, e1))
    torch.cuda.synchronize()
    _lib.msa_get_device_status(stream)
    return float(np.mean([a.elapsed_time(b) for a, b in ts])) * 1e3


def gpu_local_cpus(device):
    """CPUs the GPU's PCI device reports as local (sysfs), within this process's allowed
    set; empty when unknown."""
    try:
        prop = torch.cuda.get_device_properties(device)
        path = (f"/sys/bus/pci/devices/{prop.pci_domain_id:04x}:{prop.pci_bus_id:02x}:"
                f"{prop.pci_device_id:02x}.0/local_cpulist")
        cpus = set()
        with open(path) as f:
            for part in f.read().strip().split(","):
                lo, _, hi = part.partition("-")
                cpus.update(range(int(lo), int(hi or lo) + 1))
        return cpus & os.sched_getaffinity(0)
    except (OSError, ValueError, AttributeError):
        return set()


def e2e_prefill(cfg, step, stream, n_steps):
    """The same metric through the public API with host buffers.  Every step copies its own
    inputs (q, k, v, idx_q, idx_k) from pinned host memory to the device, runs the three
    library calls, and copies out and lse back to pinned host memory.  Steps are pipelined
    the way a serving loop runs them: copy-in streams, a compute stream and copy-out
    streams, with two sets of device buffers, so step i+1's inputs and step i-1's outputs
    move while step i computes.  The serial figure (copy in, compute, copy out, then the
    next step) is reported alongside."""
    names = ["q", "k", "v", "idx_q", "idx_k"]
    dev0 = step.x["q"].device
    # pinned host buffers on the memory next to this GPU: allocate them from the CPUs its
    # PCI device reports as local (a far NUMA node halves the copy bandwidth)
    local = gpu_local_cpus(dev0)
    saved = os.sched_getaffinity(0)
    if local:
        os.sched_setaffinity(0, local)
    try:
        host = {n: step.x[n].cpu().pin_memory() for n in names}
        out_h = [torch.empty(step.bufs["out"].shape, dtype=step.bufs["out"].dtype).pin_memory()
                 for _ in range(2)]
        lse_h = [torch.empty(step.bufs["lse"].shape, dtype=torch.float32).pin_memory()
                 for _ in range(2)]
    finally:
        os.sched_setaffinity(0, saved)
    host_note = (f"pinned buffers allocated from the {len(local)} GPU-local CPUs"
                 if local else "GPU-local CPU list unavailable; default placement")
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = out_h[0].numel() * out_h[0].element_size() + lse_h[0].numel() * 4
    dev = [{n: torch.empty_like(step.x[n]) for n in names} for _ in range(2)]
    bufs = [step.bufs, api.alloc_prefill_outputs(step.shape, dev0, step.x["q"].dtype)]
    # each direction's copies are split over four streams, so that several copy engines move
    # the step's 4.8 GB at once
    lanes = 4
    s_in = [torch.cuda.Stream(dev0) for _ in range(lanes)]
    s_out = [torch.cuda.Stream(dev0) for _ in range(lanes)]
    s_comp = stream

    def chunks(t):
        flat = t.view(-1)
        n = flat.numel()
        return [flat[c * n // lanes:(c + 1) * n // lanes] for c in range(lanes)]
    host_chunks = {nm: chunks(host[nm]) for nm in names}
    dev_chunks = [{nm: chunks(dev[j][nm]) for nm in names} for j in range(2)]
    out_dev_chunks = [chunks(bufs[j]["out"]) for j in range(2)]
    out_host_chunks = [chunks(out_h[j]) for j in range(2)]

    def run(n, pipelined):
        ev_in = [[torch.cuda.Event() for _ in range(lanes)] for _ in range(n)]
        ev_comp = [torch.cuda.Event() for _ in range(n)]
        ev_out = [[torch.cuda.Event() for _ in range(lanes)] for _ in range(n)]
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        t0.record(s_in[0])
        for c in range(1, lanes):
            s_in[c].wait_stream(s_in[0])
        for i in range(n):
            j = i % 2 if pipelined else 0
            for c in range(lanes):
                with torch.cuda.stream(s_in[c]):
                    if i >= 2 and pipelined:
                        s_in[c].wait_event(ev_comp[i - 2])        # set j's inputs are consumed
                    if not pipelined and i >= 1:
                        for e in ev_out[i - 1]:
                            s_in[c].wait_event(e)
                    for nm in names:
                        dev_chunks[j][nm][c].copy_(host_chunks[nm][c], non_blocking=True)
                    ev_in[i][c].record(s_in[c])
            for e in ev_in[i]:
                s_comp.wait_event(e)
            if i >= 2 and pipelined:
                for e in ev_out[i - 2]:
                    s_comp.wait_event(e)                       # set j's outputs are read back
            api.run_prefill(step.shape, dev[j]["q"], dev[j]["k"], dev[j]["v"], dev[j]["idx_q"],
                            dev[j]["idx_k"], bufs[j], s_comp)
            ev_comp[i].record(s_comp)
            for c in range(lanes):
                with torch.cuda.stream(s_out[c]):
                    s_out[c].wait_event(ev_comp[i])
                    out_host_chunks[j][c].copy_(out_dev_chunks[j][c], non_blocking=True)
                    if c == 0:
                        lse_h[j].copy_(bufs[j]["lse"], non_blocking=True)
                    ev_out[i][c].record(s_out[c])
        for e in ev_out[n - 1]:
            s_in[0].wait_event(e)
        t1.record(s_in[0])
        torch.cuda.synchronize()
        return t0.elapsed_time(t1) / n

    def copies_only(n, h2d_on, d2h_on):
        """The step's copies alone (same buffers and streams, no compute): ms per step."""
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        t0.record(s_in[0])
        for c in range(1, lanes):
            s_in[c].wait_stream(s_in[0])
            s_out[c].wait_stream(s_in[0])
        s_out[0].wait_stream(s_in[0])
        for i in range(n):
            for c in range(lanes):
                if h2d_on:
                    with torch.cuda.stream(s_in[c]):
                        for nm in names:
                            dev_chunks[i % 2][nm][c].copy_(host_chunks[nm][c], non_blocking=True)
                if d2h_on:
                    with torch.cuda.stream(s_out[c]):
                        out_host_chunks[i % 2][c].copy_(out_dev_chunks[i % 2][c], non_blocking=True)
                        if c == 0:
                            lse_h[i % 2].copy_(bufs[i % 2]["lse"], non_blocking=True)
        for c in range(lanes):
            s_in[0].wait_stream(s_in[c])
            s_in[0].wait_stream(s_out[c])
        t1.record(s_in[0])
        torch.cuda.synchronize()
        return t0.elapsed_time(t1) / n

    def host_link():
        # this machine's host link on the same buffers: the pipelined step cannot beat the time
        # its copies take with nothing else running (the link is shared with the rest of
        # the machine, so it is taken right before and right after the timed steps)
        ms_h2d = copies_only(2, True, False)
        ms_d2h = copies_only(2, False, True)
        ms_both = copies_only(2, True, True)
        return {"h2d_gbs": h2d / ms_h2d / 1e6, "d2h_gbs": d2h / ms_d2h / 1e6,
                "copies_only_ms_per_step": ms_both,
                "copy_bound_tokens_per_s": cfg.seq * cfg.batch / (ms_both / 1e3)}

    run(2, True)                                       # warm the copy engines
    link_before = host_link()
    ms = run(n_steps, True)
    link_after = host_link()
    ms_serial = run(max(2, n_steps // 2), False)
    return {"value": cfg.seq * cfg.batch / (ms / 1e3), "unit": "tokens/s",
            "ms_per_step": ms, "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "steps": n_steps,
            "pipelined": "copy-in (4 streams) / compute / copy-out (4 streams), two buffer sets",
            "serial_value": cfg.seq * cfg.batch / (ms_serial / 1e3),
            "serial_ms_per_step": ms_serial, "host_memory": host_note,
            "host_link": {"before": link_before, "after": link_after,
                          "note": "the step's own copies timed alone on this box right "
                                  "before and right after the pipelined steps (both "
                                  "directions at once for copies_only_ms_per_step); e2e "
                                  "over copy_bound_tokens_per_s is how close the pipelined "
                                  "step comes to this box's host link"}}, host


def decode_paged(args, device, stream, flush, hbm_peak):
    """The serving form of the decode step: the caches live in shared pools of 128-key
    physical blocks in shuffled order, reached through a block table, with per-sequence
    lengths.  Timed like the contiguous step (CUDA events around the three calls, L2
    flushed before each step) for 8 sequences of 1M tokens (the same bytes as the contiguous
    step) and for 8 sequences of mixed lengths."""
    from block_sparse_gqa_02_gb300.inputs import make_paged_decode_inputs
    cfg = CONFIGS["d1m"]
    res = {"workload": "d1m in shuffled 128-key block pools (paged), batch 8"}
    for name, lens in (("uniform_1m", [cfg.seq] * cfg.batch),
                       ("ragged", [cfg.seq, cfg.seq // 2, cfg.seq // 4, 3 * cfg.seq // 4,
                                   cfg.seq // 8, cfg.seq, 3 * cfg.seq // 8, 5 * cfg.seq // 8])):
        x = make_paged_decode_inputs(cfg, lens, device=device)
        shape = _lib.shape_from_config(cfg, batch=len(lens))
        nb = shape.n_blocks
        scores = torch.empty((len(lens), cfg.n_heads_kv, 1, nb), device=device)
        sel = torch.empty((len(lens), cfg.n_heads_kv, 1, cfg.top_k), dtype=torch.int32,
                          device=device)
        out = torch.empty_like(x["q"])
        lse = torch.empty((len(lens), cfg.n_heads_q, 1), device=device)
        ws = torch.empty(_lib.msa_workspace_bytes(shape, 1) // 4 + 4, device=device)

        def step():
            _lib.msa_index_scores_paged(shape, x["seq_lens"], x["block_table"], x["n_phys"],
                                        x["idx_q"], x["idx_k_pool"], scores, stream)
            _lib.msa_block_topk_ragged(shape, x["seq_lens"], scores, sel, stream)
            _lib.msa_sparse_decode_paged(shape, x["seq_lens"], x["block_table"], x["n_phys"],
                                         x["q"], x["k_pool"], x["v_pool"], sel, out, lse, ws,
                                         stream=stream)
        for _ in range(args.warmup):
            step()
        ts = []
        for _ in range(args.steps):
            with torch.cuda.stream(stream):
                flush.fill_(1.0)
            e0, e1 = torch.cuda.Event(True), torch.cuda.Event(True)
            e0.record(stream)
            step()
            e1.record(stream)
            ts.append((e0, e1))
        stream.synchronize()
        _lib.msa_get_device_status(stream)
        us = float(np.median([a.elapsed_time(b) for a, b in ts])) * 1e3
        tokens = int(sum(lens))
        # index keys streamed, plus the selected K/V blocks (k per KV head, at most the cache)
        sel_keys = sum(min(cfg.top_k * cfg.block_size, L) for L in lens) * cfg.n_heads_kv
        b_step = tokens * cfg.index_dim * 2 + sel_keys * 2 * cfg.head_dim * 2
        res[name] = {"us_per_step": us, "cache_lengths": lens, "cached_tokens": tokens,
                     "step_hbm_gbs": b_step / (us / 1e6) / 1e9,
                     "frac_of_hbm_peak": b_step / (us / 1e6) / 1e9 / hbm_peak}
        del x
        torch.cuda.empty_cache()
    return res


def prefill_1m(args, device, stream, flush, tc_peak):
    """The same prefill pass at 1M context (a secondary measurement, same method)."""
    cfg = CONFIGS["p1m"]
    step = Step(cfg, device)
    for _ in range(args.warmup):
        with torch.cuda.stream(stream):
            flush.fill_(1.0)
        step.run(stream, False)
    torch.cuda.synchronize()
    for _ in range(args.steps_1m):
        with torch.cuda.stream(stream):
            flush.fill_(1.0)
        step.run(stream, True)
    torch.cuda.synchronize()
    _lib.msa_get_device_status(stream)
    t = step.times_ms()
    f_index, f_sparse, f_dense = prefill_flops(cfg)
    ms = float(t[:, 0].mean())
    k_idx, k_topk, k_attn = (float(t[:, i].mean()) for i in (1, 2, 3))
    out = {"workload": f"{cfg.name}: {cfg.description}", "steps": args.steps_1m,
           "tokens_per_s": cfg.seq * cfg.batch / (ms / 1e3), "ms_per_step": ms,
           "kernels_ms": {"index_scores": k_idx, "block_topk": k_topk, "sparse_prefill": k_attn},
           "index_tflops": f_index / (k_idx / 1e3) / 1e12,
           "sparse_tflops": f_sparse / (k_attn / 1e3) / 1e12,
           "index_frac": f_index / (k_idx / 1e3) / 1e12 / tc_peak,
           "sparse_frac": f_sparse / (k_attn / 1e3) / 1e12 / tc_peak,
           "msa_tflops_per_s": (f_index + f_sparse) / (ms / 1e3) / 1e12,
           "dense_flops_avoided": f_dense - f_sparse}
    del step
    torch.cuda.empty_cache()
    return out


def backward_32k(args, device, stream, flush, tc_peak):
    """Training path: gradients of the sparse prefill attention at 32K context, against the
    same tensor peak as the forward (algorithmic work: the five products of the gradient;
    the kernels recompute S and dP once more for the key-block pass)."""
    cfg = CONFIGS["p32k"]
    step = Step(cfg, device)
    step.run(stream, False)
    x, b = step.x, step.bufs
    gen = torch.Generator(device=device).manual_seed(5)
    dout = torch.randn(x["q"].shape, generator=gen, device=device).to(x["q"].dtype)
    dq = torch.empty(x["q"].shape, device=device)
    dk = torch.empty(x["k"].shape, device=device)
    dv = torch.empty(x["v"].shape, device=device)

    ws_bytes = _lib.msa_workspace_bytes(step.shape, 2)
    ws = torch.empty(ws_bytes // 4 + 1, device=device) if ws_bytes else None

    def run():
        _lib.msa_sparse_prefill_backward(step.shape, x["q"], x["k"], x["v"], b["sel"], b["out"],
                                         b["lse"], dout, dq, dk, dv, ws, stream=stream)
    for _ in range(2):
        run()
    ts = []
    for _ in range(3):
        with torch.cuda.stream(stream):
            flush.fill_(1.0)
        e0, e1 = torch.cuda.Event(True), torch.cuda.Event(True)
        e0.record(stream)
        run()
        e1.record(stream)
        stream.synchronize()
        ts.append(e0.elapsed_time(e1))
    _lib.msa_get_device_status(stream)
    ms = float(np.median(ts))
    _, f_sparse, _ = prefill_flops(cfg)
    f_bwd = f_sparse * 2.5          # Q.K^T, dout.V^T, dQ, dK, dV: 10 d per (row, key)

    # the index branch's KL loss and its gradients on the same selection
    loss = torch.empty(1, device=device)
    diq = torch.empty(x["idx_q"].shape, device=device)
    dik = torch.empty(x["idx_k"].shape, device=device)

    kl_ws_bytes = _lib.msa_workspace_bytes(step.shape, 3)
    kl_ws = torch.empty(kl_ws_bytes // 4 + 1, device=device) if kl_ws_bytes else None

    def run_kl():
        _lib.msa_index_kl_loss(step.shape, x["q"], x["k"], b["lse"], x["idx_q"], x["idx_k"],
                               b["sel"], loss, diq, dik, kl_ws, stream=stream)
    run_kl()
    kl_ts = []
    for _ in range(3):
        with torch.cuda.stream(stream):
            flush.fill_(1.0)
        e0, e1 = torch.cuda.Event(True), torch.cuda.Event(True)
        e0.record(stream)
        run_kl()
        e1.record(stream)
        stream.synchronize()
        kl_ts.append(e0.elapsed_time(e1))
    _lib.msa_get_device_status(stream)
    kl_ms = float(np.median(kl_ts))
    # per (token, KV head, visible selected key): the G heads' logits for the target
    # (2 d G) and the index logit, d idx_q and d idx_k (3 x 2 dI)
    G, d, dI = cfg.n_heads_q // cfg.n_heads_kv, cfg.head_dim, cfg.index_dim
    f_kl = f_sparse / (4 * d * G) * (2 * d * G + 6 * dI)
    del step
    torch.cuda.empty_cache()
    return {"workload": f"{cfg.name}: {cfg.description}", "ms": ms,
            "algorithmic_flops": f_bwd, "tflops": f_bwd / (ms / 1e3) / 1e12,
            "frac_of_tensor_peak": f_bwd / (ms / 1e3) / 1e12 / tc_peak,
            "kernel": "tcgen05: dQ pass over query tiles, dK/dV pass over key blocks",
            "index_kl": {"ms": kl_ms, "algorithmic_flops": f_kl,
                         "tflops": f_kl / (kl_ms / 1e3) / 1e12,
                         "frac_of_tensor_peak": f_kl / (kl_ms / 1e3) / 1e12 / tc_peak,
                         "kernel": "tcgen05: normaliser pass (two query tiles per CTA), "
                                   "key-block pass (loss, d idx_q, d idx_k) for G >= 8"}}


def cpu_baseline_prefill(cfg, host, budget_s=15.0, seed=0):
    """The oracle as it stands on the host cores, on uniformly sampled query tiles of the
    same prefill (all heads); tokens/s = q_tile * tiles / time, an unbiased estimate of
    the whole pass because tiles are drawn uniformly."""
    import oracle
    rng = np.random.default_rng(seed)
    n_tiles = -(-cfg.seq // cfg.q_tile)
    done, t0 = [], time.perf_counter()
    while (time.perf_counter() - t0 < budget_s and len(done) < 64) or len(done) < 2:
        m = int(rng.integers(0, n_tiles))
        oracle.msa_prefill(host["q"], host["k"], host["v"], host["idx_q"], host["idx_k"],
                           cfg.block_size, cfg.q_tile, cfg.top_k, tiles=[m])
        done.append(m)
    el = time.perf_counter() - t0
    return {"value": cfg.q_tile * len(done) / el, "unit": "tokens/s", "cores": os.cpu_count(),
            "kind": "oracle",
            "sample": f"{len(done)} uniformly drawn 64-query tiles of the {cfg.name} prefill, "
                      f"all heads, fp64 numpy; extrapolated to tokens/s over {el:.1f} s"}


def run_ours(args, rank, world, device):
    torch.cuda.set_device(device)
    _lib.load()
    pcfg = CONFIGS[args.prefill]
    if args.prefill_seq or args.prefill_heads:
        seq = args.prefill_seq or pcfg.seq
        hq = args.prefill_heads or pcfg.n_heads_q
        pcfg = pcfg.with_(seq=seq, n_heads_q=hq, name=f"{pcfg.name}-T{seq}-H{hq}",
                          description=f"{pcfg.description} (T={seq}, {hq} query heads)")
    dcfg = CONFIGS[args.decode]
    if args.decode_len:
        dcfg = dcfg.with_(seq=args.decode_len, name=f"{dcfg.name}-L{args.decode_len}",
                          description=f"{dcfg.description} (cache length {args.decode_len})")
    stream = torch.cuda.Stream(device)
    pre = Step(pcfg, device)
    dec = Step(dcfg, device) if not args.no_decode else None
    flush = torch.empty(64 << 20, dtype=torch.float32, device=device)   # 256 MiB > L2
    torch.cuda.synchronize()

    def one(step, record):
        with torch.cuda.stream(stream):
            flush.fill_(1.0)
        step.run(stream, record)

    for _ in range(args.warmup):
        one(pre, False)
        if dec:
            one(dec, False)
    _lib.msa_get_device_status(stream)

    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    wall0 = time.perf_counter()
    for _ in range(args.steps):
        one(pre, True)
        if dec:
            one(dec, True)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    wall = time.perf_counter() - wall0
    clk = clocks.stop()
    _lib.msa_get_device_status(stream)

    # the same decode step captured once in a CUDA graph and replayed, one launch per step,
    # as a serving loop runs it (outside the timed region above; its buffers are the same)
    dec_graph_us = decode_graph_us(dec, stream, flush, args.steps) if dec else None

    pt = pre.times_ms()
    dt = dec.times_ms() if dec else None
    pre_ms = max_over_ranks(float(pt[:, 0].sum()), world, device)
    if rank != 0:
        return None

    peaks, peak_src = load_peaks()
    # each tensor kernel is timed on its own, in windows of milliseconds: its peak is the
    # burst figure; the sustained one (a seconds-long loop under the power cap) is given
    # beside it for reference
    tc_peak = peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
    tc_sustained = peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"])
    hbm_peak = peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
    f_index, f_sparse, f_dense = prefill_flops(pcfg)
    k_idx, k_topk, k_attn = (float(pt[:, i].mean()) for i in (1, 2, 3))
    tokens = pcfg.seq * pcfg.batch
    value = whole_job_throughput(tokens, args.steps, world, pre_ms)
    attn_tf = f_sparse / (k_attn / 1e3) / 1e12
    idx_tf = f_index / (k_idx / 1e3) / 1e12
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": pre_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        # the headline workload (the one `value` measures, and the reference arm's); the
        # decode leg names its own inside "decode"
        "config": {"workload": f"{pcfg.name}: {pcfg.description}",
                   "global_batch": pcfg.batch * world, "seq_len": pcfg.seq,
                   "parallelism": "replicas" if world > 1 else "single-gpu",
                   "l2": "flushed by a 256 MiB write before every timed kernel sequence",
                   "timing": "CUDA events on the launching stream around the library calls"},
        "roofline": {"bound": "tensor", "kernel": "sparse prefill attention",
                     "achieved": attn_tf, "peak": tc_peak, "unit": "TFLOP/s",
                     "frac": attn_tf / tc_peak,
                     "traffic": measured_traffic("sparse_prefill_tc.cu", pcfg.name),
                     "traffic_note": MEASURED_TRAFFIC["sparse_prefill_tc.cu"]["how"],
                     "peak_source": f"{peak_src} bf16 burst (dense cuBLAS GEMM)",
                     "frac_of_sustained": attn_tf / tc_sustained,
                     "algorithmic_flops_per_launch": f_sparse},
        "kernels_ms": {"index_scores": k_idx, "block_topk": k_topk, "sparse_prefill": k_attn},
        "index_roofline": {"bound": "tensor", "achieved": idx_tf, "peak": tc_peak,
                           "unit": "TFLOP/s", "frac": idx_tf / tc_peak,
                           "frac_of_sustained": idx_tf / tc_sustained,
                           "algorithmic_flops_per_launch": f_index},
        "dense_flops_avoided": f_dense - f_sparse,
        "msa_prefill_tflops_per_s": (f_index + f_sparse) / (pre_ms / args.steps / 1e3) / 1e12,
        "clocks": clk,
        "gpu_launches": args.steps * (pre.kernels + (dec.kernels if dec else 0)),
        "gpu_launches_note": "library kernels in the timed region of the headline steps "
                             "(prefill 3 + decode 4 per step); the 1M prefill is timed apart",
        "wall_s_timed_region": wall,
    }
    if dec:
        b_scan, b_rest, b_dense = decode_bytes(dcfg)
        d_idx, d_topk, d_attn = (float(dt[:, i].mean()) for i in (1, 2, 3))
        d_total = float(dt[:, 0].mean())
        scan_gbs = b_scan / (d_idx / 1e3) / 1e9
        line["decode"] = {
            "us_per_step": d_total * 1e3, "unit": "us/step", "higher_is_better": False,
            "us_per_step_graph": dec_graph_us,
            "graph_note": "the step's library calls captured in one CUDA graph and replayed "
                          "(same kernels and buffers; L2 flushed before each replay); "
                          "us_per_step and kernels_us time direct launches",
            "workload": f"{dcfg.name}: {dcfg.description}",
            "kernels_us": {"index_scan": d_idx * 1e3, "block_topk": d_topk * 1e3,
                           "sparse_decode+combine": d_attn * 1e3},
            "roofline": {"bound": "hbm", "kernel": "decode index scan", "achieved": scan_gbs,
                         "peak": hbm_peak, "unit": "GB/s", "frac": scan_gbs / hbm_peak,
                         "traffic": measured_traffic("index_scan_tc.cu", dcfg.name),
                         "traffic_note": MEASURED_TRAFFIC["index_scan_tc.cu"]["how"],
                         "algorithmic_bytes_per_launch": b_scan},
            "step_hbm_gbs": (b_scan + b_rest) / (d_total / 1e3) / 1e9,
            "dense_bytes_avoided": b_dense - (b_scan + b_rest),
        }
    # the headline workload through the public API with host buffers, right after its
    # device-timed steps (run after the training leg, the same loop measured 4.4 instead of
    # 6.1 M tokens/s on one box, with the copy bandwidths unchanged)
    if not args.no_e2e:
        e2e, host = e2e_prefill(pcfg, pre, stream, max(8, min(args.steps, 16)))
        line["e2e"] = e2e
    else:
        host = {n: pre.x[n].cpu() for n in ["q", "k", "v", "idx_q", "idx_k"]}
    if not args.no_1m and pcfg.name != "p1m":
        line["prefill_1m"] = prefill_1m(args, device, stream, flush, tc_peak)
    if not args.no_decode and not args.no_paged and args.decode_len == 0:
        line["decode_paged"] = decode_paged(args, device, stream, flush, hbm_peak)
    if not args.no_backward:
        line["backward_32k"] = backward_32k(args, device, stream, flush, tc_peak)
    if not args.no_cpu_baseline and world == 1:
        line["cpu_baseline"] = cpu_baseline_prefill(pcfg, host, args.cpu_budget)
    return line


# --------------------------------------------------------------- reference arm

def run_reference(args):
    """The fp64 oracle as it stands, timed on the host cores on the same workload: each
    step is one uniformly drawn 64-query tile of the prefill (all heads)."""
    import oracle
    cfg = CONFIGS[args.prefill]
    x = make_inputs(cfg, device="cpu")
    rng = np.random.default_rng(1)
    n_tiles = -(-cfg.seq // cfg.q_tile)
    times = []
    for i in range(args.warmup + args.steps):
        m = int(rng.integers(0, n_tiles))
        t0 = time.perf_counter()
        oracle.msa_prefill(x["q"], x["k"], x["v"], x["idx_q"], x["idx_k"], cfg.block_size,
                           cfg.q_tile, cfg.top_k, tiles=[m])
        if i >= args.warmup:
            times.append(time.perf_counter() - t0)
    sec = float(np.mean(times))
    value = cfg.q_tile / sec
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": sec * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{cfg.name}: {cfg.description}", "global_batch": cfg.batch,
                   "seq_len": cfg.seq, "parallelism": "host cores"},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": os.cpu_count(),
                         "kind": "oracle",
                         "sample": f"one uniformly drawn 64-query tile of the {cfg.name} "
                                   "prefill per step, all heads, fp64 numpy"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


# ------------------------------------------------------------------ ablations

def run_ablation(args):
    """What MSA's two changes to DSA buy, measured on synthetic inputs:
    * per-KV-head vs shared (aggregated) selection: recall of each head's planted blocks on
      the 32K planted workload (MSA keeps heads diverse; sharing loses their own plants);
    * block-level vs token-level top-k: time and score-tensor size of the selection step
      at 16K tokens for the same number of attended keys (k blocks of 128 vs 128k tokens).
    """
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    _lib.load()
    cfg = CONFIGS["p32k"]
    x = make_inputs(cfg, device=dev)
    shape = _lib.shape_from_config(cfg)
    dims = (1, 4, shape.n_rows)
    sc = torch.empty(dims + (shape.n_blocks,), device=dev)
    own = torch.empty(dims + (cfg.top_k,), dtype=torch.int32, device=dev)
    shared = torch.empty_like(own)
    _lib.msa_index_scores(shape, x["idx_q"], x["idx_k"], sc)
    _lib.msa_block_topk(shape, sc, own)
    _lib.msa_block_topk_shared(shape, sc, shared)
    torch.cuda.synchronize()
    own_np, sh_np = own.cpu().numpy(), shared.cpu().numpy()

    def recall(sel):
        hit = tot = 0
        for g in range(4):
            for m in range(shape.n_rows):
                cur = (m * 64 + 63) // 128
                for pl in x["plants"][0, g]:
                    if pl < cur:
                        tot += 1
                        hit += int(pl in sel[0, g, m])
        return hit / max(tot, 1)
    distinct = float(np.mean([len({tuple(own_np[0, g, m]) for g in range(4)}) > 1
                              for m in range(shape.n_rows)]))

    def time_topk(T, bs, qt, k, reps=10):
        sh = _lib.make_shape(1, T, T, 16, 4, 128, 128, bs, k, qt, "bf16")
        scores = torch.randn((1, 4, sh.n_rows, sh.n_blocks), device=dev)
        sel = torch.empty((1, 4, sh.n_rows, k), dtype=torch.int32, device=dev)
        for _ in range(3):
            _lib.msa_block_topk(sh, scores, sel)
        ts = []
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(True), torch.cuda.Event(True)
            e0.record()
            _lib.msa_block_topk(sh, scores, sel)
            e1.record()
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1))
        out = {"rows": 4 * sh.n_rows, "candidates_per_row_max": sh.n_blocks, "k": k,
               "ms": float(np.median(ts)), "score_tensor_bytes": scores.numel() * 4}
        del scores, sel
        torch.cuda.empty_cache()
        return out
    T = 16384
    blk = time_topk(T, 128, 64, 16)
    tok = time_topk(T, 1, 1, 16 * 128)
    return {"ablation": "per-KV-head block selection vs shared selection and token-level top-k",
            "data": "synthetic",
            "head_diversity": {"workload": f"{cfg.name}: {cfg.description}",
                               "per_head_plant_recall": recall(own_np),
                               "shared_plant_recall": recall(sh_np),
                               "rows_where_heads_differ": distinct},
            "topk_cost": {"seq": T, "block_level": blk, "token_level": tok,
                          "time_ratio": tok["ms"] / blk["ms"],
                          "score_bytes_ratio": tok["score_tensor_bytes"] /
                          blk["score_tensor_bytes"]}}


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["msa", "reference"], default="msa")
    ap.add_argument("--prefill", default="p128k", choices=["p32k", "p128k", "p1m"])
    ap.add_argument("--prefill-seq", type=int, default=0,
                    help="override the prefill sequence length (smaller cases for profiling)")
    ap.add_argument("--prefill-heads", type=int, default=0,
                    help="override the prefill query-head count (smaller cases for profiling)")
    ap.add_argument("--decode", default="d1m", choices=["d1m"])
    ap.add_argument("--decode-len", type=int, default=0,
                    help="override the decode cache length (smaller cases for profiling)")
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-1m", action="store_true",
                    help="skip the secondary 1M-context prefill measurement")
    ap.add_argument("--steps-1m", type=int, default=3)
    ap.add_argument("--no-paged", action="store_true",
                    help="skip the paged (block-table) decode measurement")
    ap.add_argument("--no-backward", action="store_true",
                    help="skip the training-path (backward) measurement")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--ablation", action="store_true",
                    help="print the selection ablations (shared / token-level) instead")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.ablation:
        if rank == 0:
            print(json.dumps(run_ablation(args)), flush=True)
        return 0
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return 0
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local))
    line = run_ours(args, rank, world, torch.device("cuda", local))
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
