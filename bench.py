#!/usr/bin/env python3
"""Benchmark of the exact-attention hot path on GB300.

One step = one pass over every part of the hot path, each on its own seeded
synthetic workload (inputs resident in HBM, all larger than L2):

  * long-context causal prefill  fa_fwd          B=2, H=Hkv=32, N=8192, d=128,
                                                 1% key rows x8 outliers
  * packed varlen causal prefill fa_fwd_varlen   32 seqs, len U[64,4096], GQA 16/4, d=128
  * paged GQA flash-decoding     fa_decode_paged batch 64, 32q/8kv heads, d=128,
                                                 ctx U[512,32768], 16-token blocks

Reported (one JSON line from rank 0):
  value    prefill TFLOP/s over both prefill launches (algorithmic FLOPs,
           4*N^2*d*H*B halved for causal, summed per sequence for varlen)
  decode   HBM GB/s of the decode step (algorithmic bytes: K/V of every cached
           token, q, out, lse, ctx lengths and block-table entries)
  roofline / roofline_decode   the two kernels against the measured peaks
  e2e      the same metrics with every step's inputs copied in from pinned
           host memory and its results copied back inside the timed region;
           the copies run on two copy streams against double-buffered device
           tensors, so they overlap the neighbouring steps' kernels
  cpu_baseline  the fp64 oracle (NumPy) timed on the host cores on a bounded
           sample of the long-context workload
  next     the further rows (chunked prefill over a paged cache, split-KV
           prefill, FP8 prefill, the backward pass), each on its own workload
  other_configs  the dense d = 64 configuration (B4 H16 N2048), causal and not, and
           paged decode steps at small batches (latency and GB/s)

The split-KV, d = 64 and small-batch decode workloads fit in L2 (or nearly), so
they are timed call by call with L2 flushed (a 256 MiB write) before each call.

``--impl reference`` times the oracle instead (the slow reference arm).
Multi-GPU: one process per GPU (torchrun); every rank runs the full step on
its own GPU (weak scaling, no collective on the data path); the timed region
is bracketed by barriers and the max over ranks is taken.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from exact_attention_33_gb300 import workloads as W  # noqa: E402

METRIC = "prefill TFLOP/s & % bf16 tensor peak; paged-decode HBM GB/s & % of 8 TB/s"
WORKLOAD_TEXT = ("exact-attention hot path: long-context causal prefill B2 H32 N8192 d128 "
                 "(1% x8 key outliers) + packed varlen causal prefill 32 seqs U[64,4096] "
                 "H16/Hkv4 d128 + paged GQA decode batch64 H32/Hkv8 d128 ctx U[512,32768] "
                 "block16")
NOMINAL_HBM_GBS = 8000.0
PROFILES = os.path.join(ROOT, "profiles")
KERNEL_SOURCES = {
    "prefill": ["exact_attention_33_gb300/csrc/prefill.cu", "exact_attention_33_gb300/csrc/ptx.cuh",
                "exact_attention_33_gb300/csrc/fa_internal.h",
                "exact_attention_33_gb300/csrc/checks.cuh"],
    "decode": ["exact_attention_33_gb300/csrc/decode.cu", "exact_attention_33_gb300/csrc/ptx.cuh",
               "exact_attention_33_gb300/csrc/fa_internal.h",
               "exact_attention_33_gb300/csrc/checks.cuh"],
}


# ----------------------------------------------------------------- ranks

def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


def init_dist(world, backend):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend)
    return dist


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int, device=None) -> float:
    """Max of a scalar over all ranks (identity for one rank)."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def weak_scaling_value(units_per_rank: float, world: int, max_seconds: float) -> float:
    """Whole-job throughput: units processed by all ranks over the slowest rank's time."""
    return units_per_rank * world / max_seconds


# ----------------------------------------------------------------- peaks, clocks, profiles

def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "sm_mhz_under_load": (p.get("clocks_under_load") or {}).get("sm_mhz_median"),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "source": "fallback"}


def source_sha(kind: str) -> str:
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES[kind]:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_value(kind: str, pattern: str):
    """A number from the committed ncu summary of the kernel (the first group
    of ``pattern``), if the summary was taken on the current kernel source
    (else None)."""
    name = {"prefill": "prefill_long_causal_d128.txt", "decode": "decode_paged_gqa_d128.txt"}[kind]
    path = os.path.join(PROFILES, name)
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m_sha = re.search(r"source_sha:\s*([0-9a-f]+)", text)
    m_val = re.search(pattern, text)
    if not m_sha or not m_val or m_sha.group(1) != source_sha(kind):
        return None
    return float(m_val.group(1))


def profiled_traffic(kind: str):
    """DRAM bytes per launch (ncu) of the kernel, or None."""
    return profiled_value(kind, r"traffic_bytes_per_launch:\s*([0-9.eE+]+)")


def profiled_tensor_active(kind: str):
    """Fraction of elapsed cycles the tensor pipe was active (ncu), or None."""
    v = profiled_value(kind, r"sm__pipe_tensor_cycles_active \(of elapsed\)\s+([0-9.]+)\s*%")
    return None if v is None else v / 100.0


class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi while running."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self.thread = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            if self.thread is not None:
                self.thread.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for n, val in zip(names, parts[4:8]):
                if val.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------- workloads on the device

def to_dev(bits, torch, device):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


def build_step(torch, device, which=("long", "varlen", "decode"), decode_batch=None):
    """Create the selected workloads on the device; returns a dict of legs."""
    import exact_attention_33_gb300 as fa
    legs = {}
    if "long" in which:
        cfg_l = W.WORKLOADS["long_causal_d128"]
        long_in = W.dense_inputs(cfg_l["B"], cfg_l["N"], cfg_l["H"], cfg_l["Hkv"], cfg_l["d"],
                                 seed=0, outlier_frac=cfg_l["outlier_frac"],
                                 outlier_scale=cfg_l["outlier_scale"])
        _add_long(legs, long_in, cfg_l)
    if "varlen" in which:
        cfg_v = W.WORKLOADS["varlen_gqa_d128"]
        lengths = W.varlen_lengths(cfg_v["num_seqs"], cfg_v["len_lo"], cfg_v["len_hi"])
        var_in = W.varlen_inputs(lengths, cfg_v["H"], cfg_v["Hkv"], cfg_v["d"], seed=0)
        _add_varlen(legs, var_in, lengths, cfg_v)
    if "decode" in which:
        cfg_d = W.WORKLOADS["paged_decode_gqa_d128"]
        ctx = W.decode_ctx_lens(cfg_d["batch"], cfg_d["ctx_lo"], cfg_d["ctx_hi"])
        if decode_batch is not None:
            ctx = ctx[:decode_batch]
        dec_in = W.decode_inputs(ctx, cfg_d["H"], cfg_d["Hkv"], cfg_d["d"], cfg_d["block_size"],
                                 seed=0)
        _add_decode(legs, dec_in, cfg_d)
    for leg in legs.values():
        leg["dev"] = {k: to_dev(v, torch, device) for k, v in leg["host"].items()}
    if "long" in legs:
        lq = legs["long"]["dev"]["q"]
        B, N, H, Hkv, d = legs["long"]["shape"]
        legs["long"]["out"] = torch.empty_like(lq)
        legs["long"]["lse"] = torch.empty((B, H, N), dtype=torch.float32, device=device)
    if "varlen" in legs:
        legs["varlen"]["cu_dev"] = torch.from_numpy(legs["varlen"]["cu"]).to(device)
        vq = legs["varlen"]["dev"]["q"]
        legs["varlen"]["out"] = torch.empty_like(vq)
        legs["varlen"]["lse"] = torch.empty((vq.shape[1], vq.shape[0]), dtype=torch.float32,
                                            device=device)
    if "decode" in legs:
        leg = legs["decode"]
        leg["table_dev"] = torch.from_numpy(leg["table"]).to(device)
        leg["ctx_dev"] = torch.from_numpy(leg["ctx"]).to(device)
        dq = leg["dev"]["q"]
        leg["out"] = torch.empty_like(dq)
        leg["lse"] = torch.empty(dq.shape[:2], dtype=torch.float32, device=device)
        ws = fa.fa_decode_workspace_size(dq.shape[0], dq.shape[1], leg["Hkv"], dq.shape[2],
                                         leg["max_ctx"], 16)
        leg["ws"] = fa.new_workspace(ws, device)
    return legs


def _add_long(legs, long_in, cfg_l):
    legs["long"] = dict(
        host={"q": long_in.q, "k": long_in.k, "v": long_in.v},
        flops=W.prefill_flops(cfg_l["B"], cfg_l["N"], cfg_l["H"], cfg_l["d"], True),
        shape=(cfg_l["B"], cfg_l["N"], cfg_l["H"], cfg_l["Hkv"], cfg_l["d"]))


def _add_varlen(legs, var_in, lengths, cfg_v):
    legs["varlen"] = dict(
        host={"q": var_in.q, "k": var_in.k, "v": var_in.v},
        cu=var_in.cu_seqlens, max_seqlen=var_in.max_seqlen,
        flops=W.varlen_flops(lengths, cfg_v["H"], cfg_v["d"], True),
        total_tokens=var_in.total_tokens)


def _add_decode(legs, dec_in, cfg_d):
    legs["decode"] = dict(
        host={"q": dec_in.q, "k_pool": dec_in.k_pool, "v_pool": dec_in.v_pool},
        table=dec_in.block_table, ctx=dec_in.ctx_lens, max_ctx=dec_in.max_ctx_len,
        bytes=W.decode_bytes(dec_in.ctx_lens, cfg_d["H"], cfg_d["Hkv"], cfg_d["d"],
                             dec_in.block_table.shape[1], cfg_d["block_size"]),
        Hkv=cfg_d["Hkv"])


def run_leg(fa, name, leg, dev, out=None, lse=None):
    out = leg["out"] if out is None else out
    lse = leg["lse"] if lse is None else lse
    if name == "long":
        fa.fa_fwd(dev["q"], dev["k"], dev["v"], causal=True, out=out, lse=lse)
    elif name == "varlen":
        fa.fa_fwd_varlen(dev["q"], dev["k"], dev["v"], leg["cu_dev"], leg["max_seqlen"],
                         causal=True, out=out, lse=lse)
    else:
        fa.fa_decode_paged(dev["q"], dev["k_pool"], dev["v_pool"], leg["table_dev"],
                           leg["ctx_dev"], leg["max_ctx"], out=out, lse=lse,
                           workspace=leg["ws"])


def e2e_pipelined(torch, fa, names, legs, pinned, host_out, steps):
    """End-to-end time (ms) of `steps` steps over the legs `names`: every step
    copies its inputs in from pinned host memory and reads its results back,
    on two copy streams, with the device tensors double-buffered so that step
    k+1's inputs arrive and step k-1's results leave while step k's kernels
    run on the compute stream."""
    comp = torch.cuda.current_stream()
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    devs = {n: [legs[n]["dev"], {k: torch.empty_like(v) for k, v in legs[n]["dev"].items()}]
            for n in names}
    outs = {n: [(legs[n]["out"], legs[n]["lse"]),
                (torch.empty_like(legs[n]["out"]), torch.empty_like(legs[n]["lse"]))]
            for n in names}
    in_done = {n: [None, None] for n in names}
    comp_done = {n: [None, None] for n in names}
    out_done = {n: [None, None] for n in names}
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    t0.record(s_in)
    for it in range(steps):
        b = it % 2
        for n in names:
            with torch.cuda.stream(s_in):
                if comp_done[n][b] is not None:       # step it-2 has read this input buffer
                    s_in.wait_event(comp_done[n][b])
                for k, t in pinned[n].items():
                    devs[n][b][k].copy_(t, non_blocking=True)
                in_done[n][b] = torch.cuda.Event()
                in_done[n][b].record(s_in)
            comp.wait_event(in_done[n][b])
            if out_done[n][b] is not None:            # step it-2's results have left
                comp.wait_event(out_done[n][b])
            run_leg(fa, n, legs[n], devs[n][b], out=outs[n][b][0], lse=outs[n][b][1])
            comp_done[n][b] = torch.cuda.Event()
            comp_done[n][b].record(comp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(comp_done[n][b])
                host_out[n][0].copy_(outs[n][b][0], non_blocking=True)
                host_out[n][1].copy_(outs[n][b][1], non_blocking=True)
                out_done[n][b] = torch.cuda.Event()
                out_done[n][b].record(s_out)
    t1.record(s_out)
    torch.cuda.synchronize()
    return t0.elapsed_time(t1)


def measure_paged_prefill(torch, device, fa, steps, warmup, peak):
    """Chunked prefill over a paged cache (8 sequences, cached prefixes
    U[1024, 16384] plus 1024 new tokens, GQA 32/8, d = 128, causal), timed
    with CUDA events on its own after the main step."""
    cfg = W.WORKLOADS["paged_prefill_gqa_d128"]
    ctx, ql = W.paged_prefill_lengths(cfg["batch"], cfg["prefix_lo"], cfg["prefix_hi"],
                                      cfg["chunk"])
    inp = W.paged_prefill_inputs(ctx, ql, cfg["H"], cfg["Hkv"], cfg["d"], seed=0)
    pl = inp.pool
    q = to_dev(inp.q, torch, device)
    kp = to_dev(pl.k_pool, torch, device)
    vp = to_dev(pl.v_pool, torch, device)
    table = torch.from_numpy(pl.block_table).to(device)
    ctx_d = torch.from_numpy(pl.ctx_lens).to(device)
    cu = torch.from_numpy(inp.cu_seqlens_q).to(device)
    out = torch.empty_like(q)
    lse = torch.empty((q.shape[1], q.shape[0]), dtype=torch.float32, device=device)
    flops = W.paged_prefill_flops(pl.ctx_lens, inp.q_lens, cfg["H"], cfg["d"], True)

    def run():
        fa.fa_fwd_paged(q, kp, vp, table, ctx_d, cu, inp.max_seqlen_q, pl.max_ctx_len,
                        causal=True, out=out, lse=lse)

    for _ in range(warmup):
        run()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        run()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    tf = flops / (ms / 1e3) / 1e12
    return {"workload": "chunked prefill over a paged KV cache: 8 sequences, cached prefix "
                        "U[1024,16384] + 1024-token chunk, H32/Hkv8, d128, causal, block16",
            "ms": ms, "tflops": tf, "frac_of_peak": tf / peak, "flops": flops,
            "launches_per_call": 1}


def measure_fp8_prefill(torch, device, fa, steps, warmup, peak_bf16):
    """FP8 (e4m3) dense causal prefill at the long-context shape (B=2, H=32,
    N=8192, d=128), timed with CUDA events on its own after the main step.
    Its peak is the measured bf16 figure times the nominal fp8 / bf16 tensor
    ratio (4.5 / 2.25 PFLOP/s)."""
    cfg = W.WORKLOADS["long_causal_fp8_d128"]
    inp = W.fp8_inputs(cfg["B"], cfg["N"], cfg["H"], cfg["Hkv"], cfg["d"], seed=0)
    q, k, v = (torch.from_numpy(getattr(inp, n)).to(device) for n in ("q", "k", "v"))
    out = torch.empty(q.shape, dtype=torch.bfloat16, device=device)
    lse = torch.empty((cfg["B"], cfg["H"], cfg["N"]), dtype=torch.float32, device=device)
    flops = W.prefill_flops(cfg["B"], cfg["N"], cfg["H"], cfg["d"], True)

    def run():
        fa.fa_fwd_fp8(q, k, v, inp.q_descale, inp.k_descale, inp.v_descale, causal=True,
                      out=out, lse=lse)

    for _ in range(warmup):
        run()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        run()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    tf = flops / (ms / 1e3) / 1e12
    peak = 2.0 * peak_bf16
    return {"workload": "FP8 e4m3 dense causal prefill, B2 H32 N8192 d128, per-tensor descales "
                        "(N(0,1) quantised)",
            "ms": ms, "tflops": tf, "frac_of_peak": tf / peak, "peak_tflops": peak,
            "peak_source": "measured bf16 burst x 2 (nominal fp8/bf16 ratio)", "flops": flops,
            "launches_per_call": 1}


def measure_fp8_varlen(torch, device, fa, steps, warmup, peak_bf16):
    """FP8 (e4m3) packed varlen causal prefill on the varlen workload (32
    sequences of U[64, 4096] tokens, GQA 16 / 4, d = 128), quantised per
    tensor, timed with CUDA events on its own after the main step."""
    cfg = W.WORKLOADS["varlen_gqa_d128"]
    lengths = W.varlen_lengths(cfg["num_seqs"], cfg["len_lo"], cfg["len_hi"])
    T = int(np.sum(lengths))
    inp = W.fp8_inputs(1, T, cfg["H"], cfg["Hkv"], cfg["d"], seed=0)
    q, k, v = (torch.from_numpy(getattr(inp, n)[0]).to(device) for n in ("q", "k", "v"))
    cu = torch.from_numpy(np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)).to(device)
    out = torch.empty(q.shape, dtype=torch.bfloat16, device=device)
    lse = torch.empty((cfg["H"], T), dtype=torch.float32, device=device)
    flops = W.varlen_flops(lengths, cfg["H"], cfg["d"], True)

    def run():
        fa.fa_fwd_varlen_fp8(q, k, v, cu, int(np.max(lengths)), inp.q_descale, inp.k_descale,
                             inp.v_descale, causal=True, out=out, lse=lse)

    for _ in range(warmup):
        run()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        run()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    tf = flops / (ms / 1e3) / 1e12
    peak = 2.0 * peak_bf16
    return {"workload": "FP8 e4m3 packed varlen causal prefill, 32 seqs U[64,4096], H16/Hkv4, "
                        "d128, per-tensor descales (N(0,1) quantised)",
            "ms": ms, "tflops": tf, "frac_of_peak": tf / peak, "peak_tflops": peak,
            "peak_source": "measured bf16 burst x 2 (nominal fp8/bf16 ratio)", "flops": flops,
            "launches_per_call": 1}


def measure_backward(torch, device, fa, steps, warmup, peak):
    """Backward pass (fa_bwd: dQ, dK, dV) of the long-context causal prefill
    (B=2, H=32, N=8192, d=128, the forward's own workload), timed with CUDA
    events on its own.  Work: the five products of the gradient, 2.5 times
    the forward count (5 * N^2 * d per (batch, head) causal); the kernels
    recompute S and dP once more, which is not counted."""
    cfg = W.WORKLOADS["long_causal_d128"]
    B, N, H, d = cfg["B"], cfg["N"], cfg["H"], cfg["d"]
    inp = W.dense_inputs(B, N, H, cfg["Hkv"], d, seed=0, outlier_frac=cfg["outlier_frac"],
                         outlier_scale=cfg["outlier_scale"])
    q, k, v = (to_dev(getattr(inp, n), torch, device) for n in ("q", "k", "v"))
    do = to_dev(W.normal_bf16_bits((B, N, H, d), 0, 3), torch, device)
    out, lse = fa.fa_fwd(q, k, v, causal=True)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(fa.fa_bwd_workspace_size(B, H, N), dtype=torch.uint8, device=device)
    flops = 2.5 * W.prefill_flops(B, N, H, d, True)

    def run():
        fa.fa_bwd(q, k, v, out, lse, do, causal=True, dq=dq, dk=dk, dv=dv, workspace=ws)

    for _ in range(warmup):
        run()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        run()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    tf = flops / (ms / 1e3) / 1e12
    return {"workload": "backward of the long-context causal prefill: B2 H32 N8192 d128 "
                        "(dQ, dK, dV from O, lse, dO)",
            "ms": ms, "tflops": tf, "frac_of_peak": tf / peak, "flops": flops,
            "launches_per_call": 3}


def measure_backward_varlen(torch, device, fa, steps, warmup, peak):
    """Backward pass of a packed varlen batch (fa_bwd_varlen) on the varlen
    workload (32 sequences of U[64, 4096] tokens, GQA 16 / 4, d = 128,
    causal), timed with CUDA events on its own.  Work: 2.5 times the
    forward's causal products of each sequence, as for the dense backward."""
    cfg = W.WORKLOADS["varlen_gqa_d128"]
    lengths = W.varlen_lengths(cfg["num_seqs"], cfg["len_lo"], cfg["len_hi"])
    H, Hkv, d = cfg["H"], cfg["Hkv"], cfg["d"]
    inp = W.varlen_inputs(lengths, H, Hkv, d, seed=0)
    T = inp.total_tokens
    q, k, v = (to_dev(getattr(inp, n), torch, device) for n in ("q", "k", "v"))
    do = to_dev(W.normal_bf16_bits((T, H, d), 0, 3), torch, device)
    cu = torch.from_numpy(inp.cu_seqlens.astype(np.int32)).to(device)
    max_len = int(np.max(lengths))
    out, lse = fa.fa_fwd_varlen(q, k, v, cu, max_len, causal=True)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(fa.fa_bwd_workspace_size(len(lengths), H, max_len), dtype=torch.uint8,
                     device=device)
    flops = 2.5 * W.varlen_flops(lengths, H, d, True)

    def run():
        fa.fa_bwd_varlen(q, k, v, out, lse, do, cu, max_len, causal=True, dq=dq, dk=dk, dv=dv,
                         workspace=ws)

    for _ in range(warmup):
        run()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        run()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    tf = flops / (ms / 1e3) / 1e12
    return {"workload": "backward of the packed varlen causal prefill: 32 seqs U[64,4096], "
                        "H16/Hkv4, d128 (dQ, dK, dV from O, lse, dO)",
            "ms": ms, "tflops": tf, "frac_of_peak": tf / peak, "flops": flops,
            "launches_per_call": 3}


L2_FLUSH_BYTES = 256 << 20   # twice the GB300's L2
SLEEP_CYCLES = 200_000        # ~0.1 ms of device time before each timed call


def time_flushed(torch, fn, steps, warmup, flush):
    """Mean device time of fn() over `steps` calls, each timed alone with CUDA
    events on the current stream after `flush` (a buffer larger than L2) has
    been rewritten, so no call finds its inputs or partial states in L2.  The
    time is the device's alone: fn() is enqueued before its start event runs."""
    for _ in range(warmup):
        fn()
    stream = torch.cuda.current_stream()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    for e0, e1 in ev:
        flush.zero_()
        # a short device-side wait lets the host enqueue fn() before the start
        # event is reached, so host launch overhead never enters the timing
        torch.cuda._sleep(SLEEP_CYCLES)
        e0.record(stream)
        fn()
        e1.record(stream)
    torch.cuda.synchronize()
    return sum(e0.elapsed_time(e1) for e0, e1 in ev) / steps


def measure_splitkv(torch, device, fa, steps, warmup, peak):
    """Split-KV dense prefill (fa_fwd_splitkv, automatic split count) on a
    long sequence with few heads (B=1, H=4, N=8192, d=128, causal: 128
    query-tile pairs, fewer than the SMs), timed beside fa_fwd on the same
    inputs."""
    cfg = W.WORKLOADS["splitkv_small_bh_d128"]
    B, N, H, d = cfg["B"], cfg["N"], cfg["H"], cfg["d"]
    inp = W.dense_inputs(B, N, H, cfg["Hkv"], d, seed=0)
    q, k, v = (to_dev(getattr(inp, n), torch, device) for n in ("q", "k", "v"))
    out = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=device)
    ws = fa.new_workspace(fa.fa_fwd_splitkv_workspace_size(B, H, N, d, 0), device)
    flops = W.prefill_flops(B, N, H, d, True)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
    ms = time_flushed(torch, lambda: fa.fa_fwd_splitkv(q, k, v, causal=True, out=out, lse=lse,
                                                       workspace=ws), steps, warmup, flush)
    ms_plain = time_flushed(torch, lambda: fa.fa_fwd(q, k, v, causal=True, out=out, lse=lse),
                            steps, warmup, flush)
    tf = flops / (ms / 1e3) / 1e12
    return {"workload": "split-KV causal prefill, few heads: B1 H4 N8192 d128 "
                        "(L2 flushed before each launch)",
            "ms": ms, "tflops": tf, "frac_of_peak": tf / peak, "flops": flops,
            "unsplit_ms": ms_plain, "unsplit_tflops": flops / (ms_plain / 1e3) / 1e12,
            "launches_per_call": 2}


def measure_dense_d64(torch, device, fa, steps, warmup, modes=(False, True), fp8=True):
    """The dense configuration of the workload list (B=4, H=Hkv=16, N=2048,
    d=64, bf16 N(0,1)), non-causal and causal (``modes``: the causal flags
    to run), and (``fp8``) the same shape on e4m3 inputs quantised per
    tensor.  Its inputs fit in L2, so L2 is flushed (a 256 MiB write)
    before every timed launch and only the launch is timed."""
    cfg = W.WORKLOADS["dense_d64"]
    B, N, H, Hkv, d = cfg["B"], cfg["N"], cfg["H"], cfg["Hkv"], cfg["d"]
    inp = W.dense_inputs(B, N, H, Hkv, d, seed=0)
    q, k, v = (to_dev(getattr(inp, n), torch, device) for n in ("q", "k", "v"))
    out = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=device)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
    res = {"workload": "dense prefill B4 H16 N2048 d64 (L2 flushed before each launch)"}
    for causal in modes:
        ms = time_flushed(torch, lambda: fa.fa_fwd(q, k, v, causal=causal, out=out, lse=lse),
                          steps, warmup, flush)
        flops = W.prefill_flops(B, N, H, d, causal)
        res["causal" if causal else "non_causal"] = {"ms": ms, "tflops": flops / (ms / 1e3) / 1e12,
                                                     "flops": flops}
    if fp8:
        f8 = W.fp8_inputs(B, N, H, Hkv, d, seed=0)
        fq, fk, fv = (torch.from_numpy(getattr(f8, n)).to(device) for n in ("q", "k", "v"))
        for causal in modes:
            ms = time_flushed(
                torch, lambda: fa.fa_fwd_fp8(fq, fk, fv, f8.q_descale, f8.k_descale, f8.v_descale,
                                             causal=causal, out=out, lse=lse),
                steps, warmup, flush)
            flops = W.prefill_flops(B, N, H, d, causal)
            res["fp8_causal" if causal else "fp8_non_causal"] = {
                "ms": ms, "tflops": flops / (ms / 1e3) / 1e12, "flops": flops}
    if fa.fa_device_status(clear=True) != 0:
        raise RuntimeError("device status word set during the dense d64 leg")
    return res


def measure_decode_small_batches(torch, device, fa, steps, warmup):
    """Paged decode at serving batch sizes (32 query / 8 KV heads, d = 128,
    16-token blocks, equal contexts): the latency of one step, L2 flushed
    (a 256 MiB write) before each timed call, and its HBM rate."""
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
    res = {"workload": "paged GQA decode steps at small batches (L2 flushed before each call)"}
    for batch, ctx_len in ((1, 4096), (1, 32768), (8, 8192), (16, 32768)):
        ctx = [ctx_len] * batch
        inp = W.decode_inputs(ctx, 32, 8, 128, seed=1)
        q = to_dev(inp.q, torch, device)
        kp, vp = to_dev(inp.k_pool, torch, device), to_dev(inp.v_pool, torch, device)
        table = torch.from_numpy(inp.block_table).to(device)
        cl = torch.from_numpy(inp.ctx_lens).to(device)
        out = torch.empty_like(q)
        lse = torch.empty((batch, 32), dtype=torch.float32, device=device)
        ws = fa.new_workspace(fa.fa_decode_workspace_size(batch, 32, 8, 128, ctx_len), device)
        nbytes = W.decode_bytes(inp.ctx_lens, 32, 8, 128, inp.block_table.shape[1], 16)
        ms = time_flushed(torch, lambda: fa.fa_decode_paged(q, kp, vp, table, cl, ctx_len,
                                                            out=out, lse=lse, workspace=ws),
                          steps, warmup, flush)
        res[f"batch{batch}_ctx{ctx_len}"] = {"us": ms * 1e3, "gbs": nbytes / (ms / 1e3) / 1e9,
                                             "bytes": nbytes}
    if fa.fa_device_status(clear=True) != 0:
        raise RuntimeError("device status word set during the small-batch decode leg")
    return res


NEXT_LEGS = ("paged_prefill", "splitkv", "fp8_prefill", "fp8_varlen", "backward",
             "backward_varlen")
# legs that --profile-leg can run alone (one launch kind each, for ncu captures)
PROFILE_LEGS = NEXT_LEGS + ("dense_d64", "dense_d64_causal", "decode_small")


def run_next_leg(name, torch, device, fa, steps, warmup, peak):
    fn = {"paged_prefill": measure_paged_prefill, "splitkv": measure_splitkv,
          "fp8_prefill": measure_fp8_prefill, "fp8_varlen": measure_fp8_varlen,
          "backward": measure_backward, "backward_varlen": measure_backward_varlen,
          "dense_d64": lambda t, dv, f, s, w, pk: measure_dense_d64(t, dv, f, s, w, (False,), False),
          "dense_d64_causal": lambda t, dv, f, s, w, pk: measure_dense_d64(t, dv, f, s, w, (True,),
                                                                           False),
          "decode_small": lambda t, dv, f, s, w, pk: measure_decode_small_batches(t, dv, f, s, w),
          }[name]
    res = fn(torch, device, fa, steps, warmup, peak)
    if fa.fa_device_status(clear=True) != 0:
        raise RuntimeError(f"device status word set during the {name} leg")
    return res


LEG_ORDER = ("long", "varlen", "decode")
LAUNCHES_PER_STEP = {"long": 1, "varlen": 1, "decode": 2}


# ----------------------------------------------------------------- oracle timing

def oracle_sample_tflops(max_seconds=20.0, rows_per_pair=None, pairs=4, seed=5):
    """Time the fp64 oracle on a seeded sample of the long-context workload.

    Each sampled (batch, head) pair runs the oracle on all 8192 query rows
    (or ``rows_per_pair`` seeded rows); the work counted is the causal
    algorithmic FLOPs of the rows evaluated.  Returns (TFLOP/s, sample text).
    """
    import oracle
    cfg = W.WORKLOADS["long_causal_d128"]
    N, d, H = cfg["N"], cfg["d"], cfg["H"]
    rng = np.random.default_rng(seed)
    done_flops, spent, used = 0.0, 0.0, []
    # one (batch, head) slice at a time keeps host memory small
    for idx in rng.choice(cfg["B"] * H, pairs, replace=False):
        b, h = int(idx) // H, int(idx) % H
        inp = _long_slice(b, h)
        rows = None
        if rows_per_pair is not None:
            rows = np.sort(np.random.default_rng(seed + 1).choice(N, rows_per_pair, replace=False))
        t0 = time.perf_counter()
        oracle.attention_one(inp[0], inp[1], inp[2], causal=True, rows=rows)
        dt = time.perf_counter() - t0
        r = np.arange(N) if rows is None else rows
        done_flops += 4.0 * d * float(np.sum(r + 1))
        spent += dt
        used.append((b, h))
        if spent > max_seconds:
            break
    desc = (f"oracle on {len(used)} (batch, head) pairs {used} of the long-context causal "
            f"workload, {'all' if rows_per_pair is None else rows_per_pair} query rows each")
    return done_flops / spent / 1e12, desc, spent


_LONG_CACHE = {}


def _long_slice(b, h):
    """fp64 (q, k, v) of one (batch, head) of the long-context workload."""
    if "inp" not in _LONG_CACHE:
        cfg = W.WORKLOADS["long_causal_d128"]
        _LONG_CACHE["inp"] = W.dense_inputs(cfg["B"], cfg["N"], cfg["H"], cfg["Hkv"], cfg["d"],
                                            seed=0, outlier_frac=cfg["outlier_frac"],
                                            outlier_scale=cfg["outlier_scale"])
    inp = _LONG_CACHE["inp"]
    g = h // (inp.H // inp.Hkv)
    f = W.bf16_bits_to_f64
    return (f(inp.q[b][:, h:h + 1]), f(inp.k[b][:, g:g + 1]), f(inp.v[b][:, g:g + 1]))


def blas_threads():
    for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        if os.environ.get(var):
            try:
                return int(os.environ[var])
            except ValueError:
                pass
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads") for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    return os.cpu_count() or 1


# ----------------------------------------------------------------- arms

def bench_reference(args, rank, world):
    """The oracle as it stands, on the host cores, each step a bounded sample."""
    if rank != 0:
        return 0
    # each step: one (batch, head) pair, 1024 seeded query rows (about 1-3 s)
    steps, warmup = args.steps, args.warmup
    per_step, total_flops, total_t, desc = [], 0.0, 0.0, ""
    for it in range(warmup + steps):
        tf, desc, spent = oracle_sample_tflops(max_seconds=0.0, rows_per_pair=1024, pairs=1,
                                               seed=100 + it)
        if it >= warmup:
            per_step.append(spent)
            total_t += spent
            total_flops += tf * 1e12 * spent
    value = total_flops / total_t / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": steps, "warmup": warmup, "ms_per_step": 1e3 * total_t / steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": WORKLOAD_TEXT,
                   "sample": "per step: the oracle on one seeded (batch, head) pair of the "
                             "long-context causal prefill, 1024 seeded query rows",
                   "parallelism": "host cores, rank 0 only"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": blas_threads(),
                         "kind": "oracle", "sample": desc},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def bench_ours(args, rank, world, local):
    import torch
    import exact_attention_33_gb300 as fa

    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    init_dist(world, "nccl")
    fa.load_library()
    fa.fa_device_status(clear=True)
    order = [n for n in LEG_ORDER if n in args.legs]
    legs = build_step(torch, device, order, args.decode_batch)
    stream = torch.cuda.current_stream()

    def step(ev=None):
        for i, name in enumerate(order):
            if ev is not None:
                ev[i][0].record(stream)
            run_leg(fa, name, legs[name], legs[name]["dev"])
            if ev is not None:
                ev[i][1].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    events = [[[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in order]
              for _ in range(args.steps)]
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clocks:
        time.sleep(0.3)
        barrier(world)
        torch.cuda.synchronize()
        t_start.record(stream)
        for it in range(args.steps):
            step(events[it])
        t_end.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        time.sleep(0.2)
    total_ms = t_start.elapsed_time(t_end)
    leg_ms = {name: [events[it][i][0].elapsed_time(events[it][i][1]) for it in range(args.steps)]
              for i, name in enumerate(order)}
    status = fa.fa_device_status(clear=True)
    if status != 0:
        raise RuntimeError(f"device status word set during the bench: {status:#x}")

    # ---- end to end: pinned host inputs in, results out, inside the timed region
    pinned = {name: {k: torch.from_numpy(np.ascontiguousarray(v).view(np.int16))
                     .view(torch.bfloat16).pin_memory()
                     for k, v in legs[name]["host"].items()} for name in order}
    host_out = {name: (torch.empty(legs[name]["out"].shape, dtype=torch.bfloat16).pin_memory(),
                       torch.empty(legs[name]["lse"].shape, dtype=torch.float32).pin_memory())
                for name in order}
    h2d = sum(t.numel() * t.element_size() for n in order for t in pinned[n].values())
    d2h = sum(o.numel() * o.element_size() + l.numel() * l.element_size()
              for o, l in host_out.values())
    e2e_steps = max(2, min(args.steps, 10))
    pre = [n for n in ("long", "varlen") if n in order]
    barrier(world)
    e2e_pre_ms = e2e_pipelined(torch, fa, pre, legs, pinned, host_out, e2e_steps) if pre else None
    e2e_dec_ms = (e2e_pipelined(torch, fa, ["decode"], legs, pinned, host_out, e2e_steps)
                  if "decode" in order else None)
    barrier(world)

    nxt = {}
    other = {}
    if args.next_legs and "long" in order:
        peaks0 = measured_peaks()
        for name in NEXT_LEGS:
            nxt[name] = run_next_leg(name, torch, device, fa,
                                     min(args.steps, 20 if name.startswith("backward") else 50),
                                     args.warmup, peaks0["bf16_tflops"])
        other["dense_d64"] = measure_dense_d64(torch, device, fa, min(args.steps, 50),
                                               args.warmup)
        other["decode_small_batches"] = measure_decode_small_batches(
            torch, device, fa, min(args.steps, 50), args.warmup)

    # ---- numbers (max over ranks of each time)
    K = args.steps
    t = {n: max_over_ranks(sum(leg_ms[n]) / 1e3, world, device) for n in order}
    te_pre = max_over_ranks(e2e_pre_ms / 1e3, world, device) if pre else None
    te_dec = max_over_ranks(e2e_dec_ms / 1e3, world, device) if "decode" in order else None
    t_total = max_over_ranks(total_ms / 1e3, world, device)
    f_pre = sum(legs[n]["flops"] for n in pre)
    prefill_tflops = (weak_scaling_value(f_pre * K, world, sum(t[n] for n in pre)) / 1e12
                      if pre else None)
    e2e_tflops = (weak_scaling_value(f_pre * e2e_steps, world, te_pre) / 1e12
                  if pre else None)
    dbytes = legs["decode"]["bytes"] if "decode" in order else None
    decode_gbs = weak_scaling_value(dbytes * K, world, t["decode"]) / 1e9 if dbytes else None
    e2e_gbs = weak_scaling_value(dbytes * e2e_steps, world, te_dec) / 1e9 if dbytes else None

    if rank != 0:
        return 0
    peaks = measured_peaks()
    clk = clocks.summary()
    timed_s = total_ms / 1e3
    tensor_peak = peaks["bf16_tflops_sustained"] if timed_s > 2.0 else peaks["bf16_tflops"]
    leg_info, roof, roof_dec = {}, None, None
    if "long" in order:
        f = legs["long"]["flops"]
        leg_info["long_causal_prefill"] = {"ms": 1e3 * t["long"] / K,
                                           "tflops": f * K / t["long"] / 1e12}
        ach = f / (statistics.mean(leg_ms["long"]) / 1e3) / 1e12
        roof = {"bound": "tensor", "kernel": "prefill_kernel<128,causal> (long-context launch)",
                "achieved": ach, "peak": tensor_peak, "unit": "TFLOP/s",
                "frac": ach / tensor_peak, "traffic": profiled_traffic("prefill"),
                "peak_source": peaks["source"] + (" sustained" if timed_s > 2.0 else " burst"),
                # clock-independent view: the peak above is cuBLAS at the power-capped
                # clock of its own measurement; the kernel ran at the sampled clock
                "tensor_pipe_active_ncu": profiled_tensor_active("prefill"),
                "peak_measured_at_sm_mhz": peaks.get("sm_mhz_under_load"),
                "sm_mhz": clk.get("sm_mhz")}
    if "varlen" in order:
        f = legs["varlen"]["flops"]
        leg_info["varlen_causal_prefill"] = {"ms": 1e3 * t["varlen"] / K,
                                             "tflops": f * K / t["varlen"] / 1e12}
    if "decode" in order:
        leg_info["paged_decode"] = {"ms": 1e3 * t["decode"] / K,
                                    "gbs": dbytes * K / t["decode"] / 1e9}
        ach = dbytes / (statistics.mean(leg_ms["decode"]) / 1e3) / 1e9
        roof_dec = {"bound": "hbm", "kernel": "decode_split_kernel + decode_combine_kernel",
                    "achieved": ach, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                    "frac": ach / peaks["hbm_gbs"], "traffic": profiled_traffic("decode"),
                    "peak_source": peaks["source"]}
    if args.cpu_seconds > 0:
        cpu_tf, cpu_desc, _ = oracle_sample_tflops(max_seconds=args.cpu_seconds)
        cpu = {"value": cpu_tf, "unit": "TFLOP/s", "cores": blas_threads(), "kind": "oracle",
               "sample": cpu_desc}
    else:
        cpu = None
    line = {
        "metric": METRIC,
        "value": prefill_tflops,
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": 1e3 * t_total / K,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {
            "workload": WORKLOAD_TEXT,
            "legs": order,
            "decode_batch": args.decode_batch or 64,
            "prefill_flops_per_step": f_pre,
            "decode_bytes_per_step": dbytes,
            "l2": "step inputs are larger than L2 (no flush needed); the split-KV, d=64 "
                  "and small-batch decode legs flush it before each timed call",
            "parallelism": f"replicas x{world}",
        },
        "decode": None if dbytes is None else {
            "value": decode_gbs, "unit": "GB/s",
            "frac_of_8tbs": decode_gbs / world / NOMINAL_HBM_GBS,
            "frac_of_measured": decode_gbs / world / peaks["hbm_gbs"],
            "ms_per_step": 1e3 * t["decode"] / K},
        "legs": leg_info,
        "roofline": roof,
        "roofline_decode": roof_dec,
        "e2e": {"value": e2e_tflops, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "decode_gbs": e2e_gbs, "steps": e2e_steps,
                "pipelined": "inputs of step k+1 copied in and results of step k-1 read back "
                             "on two copy streams while step k runs (double-buffered device "
                             "tensors)"},
        "next": nxt or None,
        "other_configs": other or None,
        "gpu_launches": sum(LAUNCHES_PER_STEP[n] for n in order) * K,
        "clocks": clk,
        "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=15.0,
                    help="budget of the oracle CPU-baseline sample (0: skip)")
    ap.add_argument("--legs", default="long,varlen,decode",
                    help="comma-separated subset of the step (for profiling runs)")
    ap.add_argument("--no-next", dest="next_legs", action="store_false",
                    help="skip the separately timed legs (paged prefill, split-KV, FP8, backward)")
    ap.add_argument("--decode-batch", type=int, default=None,
                    help="use only the first B decode sequences (for profiling runs)")
    ap.add_argument("--profile-leg", choices=PROFILE_LEGS, default=None,
                    help="run only this separately timed leg, --steps times (for ncu runs)")
    args = ap.parse_args(argv)
    args.legs = [x for x in args.legs.split(",") if x]
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    rank, world, local = dist_env()
    if args.profile_leg:
        import torch
        import exact_attention_33_gb300 as fa
        fa.load_library()
        res = run_next_leg(args.profile_leg, torch, torch.device("cuda", 0), fa, args.steps,
                           args.warmup, measured_peaks()["bf16_tflops"])
        print(json.dumps({"profile_leg": args.profile_leg, **res}))
        return 0
    if args.impl == "reference":
        return bench_reference(args, rank, world)
    return bench_ours(args, rank, world, local)


if __name__ == "__main__":
    sys.exit(main())
