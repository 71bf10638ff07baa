#!/usr/bin/env python3
"""Benchmark of the hybrid-attention decode hot path on GB300 (one JSON line on rank 0).

Workload (default, `decode_single_layer`): 32 requests, H=32, D=128, bf16 KV, fp32 linear
state, seq_lens ~ U{128..4096} with blocks shuffled across a pool; one step = one decode
token for every request through one Full layer (KV append at position seq_len - 1 fused
into the split-K paged decode, plus the split combine) and one Linear layer (in-place state
step). Metric: req-tokens/s per layer
= B * layers / step time. Inputs live in HBM before timing; the per-step working set
(~1.2 GB of KV and 128 MiB of state) is far larger than L2, so no flush is needed.

`value` is device time (CUDA events on the launching stream). `e2e` is the same step
through the public dispatcher (hyb_layer_dispatch) with the step's q/k/v and metadata
copied from pinned host memory and the outputs copied back, inside the timed region.
`--impl reference` times the CPU oracle instead (bounded sample per step, host cores).
With torchrun (N > 1) every rank runs its own replica (the path shards by request with
no exchange) and rank 0 reports the aggregate.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "hybrid attn decode req-tokens/s per layer; HBM GB/s and % of GB300 roofline"
UNIT = "req-tokens/s per layer"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2500)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--workload", default="decode_single_layer",
                    choices=["decode_single_layer", "hybrid_32layer", "prefill_chunked", "long_context_decode",
                             "sliding_window", "state_precision", "block32", "bucketing", "prefill_lengths"],
                    help="decode_single_layer is the headline; the others are timed alone (e.g. for profiling)")
    ap.add_argument("--no-rows", action="store_true", help="skip the per-row measurements of the other workloads")
    return ap.parse_args()


# ------------------------------------------------------------------ distributed
class Dist:
    def __init__(self, n):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if self.world > 1:
            import torch.distributed as dist
            dist.init_process_group("gloo")       # timing barrier / max only; no data exchange
            self.pg = dist

    def barrier(self):
        if self.pg:
            self.pg.barrier()

    def max(self, x: float) -> float:
        if not self.pg:
            return x
        import torch
        t = torch.tensor([x], dtype=torch.float64)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def sum(self, x: float) -> float:
        if not self.pg:
            return x
        import torch
        t = torch.tensor([x], dtype=torch.float64)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.SUM)
        return float(t.item())


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi samples during the timed region (SM clock, throttle reasons)."""
    Q = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.lines = []
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits", "-lms", "100",
                 "-i", str(self.idx)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            threading.Thread(target=self._read, daemon=True).start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self, which):
        setattr(self, which, time.time())

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        rows = [l for (t, l) in self.lines if self.t0 and self.t1 and self.t0 - 0.15 <= t <= self.t1 + 0.15]
        if not rows:
            rows = [l for (_, l) in self.lines]
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            f = [x.strip() for x in r.split(",")]
            if len(f) < 10:
                continue
            try:
                sm.append(float(f[2]))
                mx = float(f[3])
            except ValueError:
                continue
            for name, val in zip(names, f[6:10]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------ peaks
def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        return float(j["hbm_gbs"]), float(j["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, "fallback"


def traffic_record(kernel: str, src: str):
    """ncu dram bytes per launch recorded under profiles/, valid only while the kernel
    source is unchanged since the capture (sha256 of the .cu file)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        rec = json.load(f).get(kernel)
    if not rec:
        return None
    with open(os.path.join(ROOT, "paged_kv_linear_gb300", "csrc", src), "rb") as f:
        if hashlib.sha256(f.read()).hexdigest() != rec.get("source_sha256"):
            return None
    return rec


# ------------------------------------------------------------------ workload
def build_workload(seed, device):
    import torch
    db = W.decode_single_layer(seed)
    B, H, D, NB, MB = db.B, db.H, db.D, db.pool.num_blocks, db.pool.max_blocks
    g = W.rng(seed + 1)
    wl = dict(db=db, B=B, H=H, D=D, NB=NB, MB=MB)
    wl["kc"] = W.device_rows_(torch.empty((NB, H, 16, D), dtype=torch.bfloat16, device=device), seed * 10 + 1, D)
    wl["vc"] = W.device_rows_(torch.empty((NB, H, 16, D), dtype=torch.bfloat16, device=device), seed * 10 + 2, D)
    wl["state"] = W.device_state_(torch.empty((B, H, D, D), device=device), seed * 10 + 3, db.seq_lens, D)
    wl["host"] = {n: W.rows(g, (B, H, D), D, W.BF16) for n in ("qf", "kf", "vf", "ql", "kl", "vl")}
    wl["slots_h"] = g.permutation(B).astype(np.int32)
    return wl


# ------------------------------------------------------------------ other rows
def _time(fn, stream, iters, warmup=3):
    """Average device time (ms) of fn() over `iters` calls, CUDA events on `stream`."""
    import torch
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            fn()
        stream.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(iters):
            fn()
        e1.record(stream)
        stream.synchronize()
    return e0.elapsed_time(e1) / iters


def _traffic(kernel, src):
    rec = traffic_record(kernel, src)
    return int(rec["bytes_per_launch"]) if rec else None


def _roof(bound, achieved, peak, unit, kernel, alg, traffic=None, **extra):
    r = {"kernel": kernel, "bound": bound, "achieved": round(achieved, 1), "peak": peak, "unit": unit,
         "frac": round(achieved / peak, 4), "traffic": traffic, "algorithmic": alg}
    r.update(extra)
    return r


def row_long_context(hyb, device, stream, iters, seed=0):
    """8 requests x 131072 tokens: split-K paged decode over 8192 random blocks each, and the
    Linear step on 8 x 32 x 128 x 128 fp32 states."""
    import torch
    hbm, _, _ = measured_peaks()
    db = W.decode_long_context(seed)
    B, H, D, NB = db.B, db.H, db.D, db.pool.num_blocks
    d = hyb.dims(H, D, NB, db.pool.max_blocks, W.BF16)
    kc = W.device_rows_(torch.empty((NB, H, 16, D), dtype=torch.bfloat16, device=device), 51, D)
    vc = W.device_rows_(torch.empty_like(kc), 52, D)
    st = W.device_state_(torch.empty((B, H, D, D), device=device), 53, db.seq_lens, D)
    g = W.rng(seed + 5)
    q = torch.from_numpy(W.rows(g, (B, H, D), D, W.BF16).view(np.int16)).to(device).view(torch.bfloat16)
    out = torch.empty_like(q)
    bt = torch.from_numpy(db.pool.block_tables).to(device)
    lens = torch.from_numpy(db.seq_lens).to(device)
    slots = torch.arange(B, dtype=torch.int32, device=device)
    n = int(db.seq_lens.max())
    ws_n = hyb.hyb_paged_attn_decode_workspace_size(B, n, d)
    ws = torch.empty(ws_n, dtype=torch.uint8, device=device)
    sh = stream.cuda_stream
    t_dec = _time(lambda: hyb.check(hyb.hyb_paged_attn_decode(out, q, kc, vc, bt, lens, B, n, d, ws, ws_n, sh)), stream, iters)
    t_lin = _time(lambda: hyb.check(hyb.hyb_linear_attn_step(out, q, q, q, st, B, slots, B, H, D, W.BF16, sh)), stream, iters)
    dec_bytes = int(db.seq_lens.sum()) * H * D * 4 + 2 * B * H * D * 2
    lin_bytes = B * H * D * D * 8
    res = {"workload": "long_context_decode: 8 requests x 131072 tokens, H=32, D=128, 8192 random blocks each",
           "value": round(B * 2 / ((t_dec + t_lin) * 1e-3), 1), "unit": UNIT,
           "ms": {"paged_decode": round(t_dec, 4), "linear_step": round(t_lin, 4)},
           "roofline": _roof("hbm", dec_bytes / (t_dec * 1e-3) / 1e9, hbm, "GB/s", "paged_decode (split-K + combine)", dec_bytes),
           "linear_step": _roof("hbm", lin_bytes / (t_lin * 1e-3) / 1e9, hbm, "GB/s", "linear_step", lin_bytes)}
    del kc, vc, st
    torch.cuda.empty_cache()
    return res


def row_hybrid_32layer(hyb, device, stream, iters, seed=0):
    """32 layers [F,F,F,Lin] x 8, batch 64 (80% ~128, 20% ~2048 tokens): one decode token per
    request through all layers via hyb_layer_dispatch."""
    import torch
    hbm, _, _ = measured_peaks()
    db = W.decode_hybrid_32layer(seed)
    lt = db.extra["layer_types"]
    B, H, D, NB, MB = db.B, db.H, db.D, db.pool.num_blocks, db.pool.max_blocks
    d = hyb.dims(H, D, NB, MB, W.BF16)
    g = W.rng(seed + 9)
    mk = lambda: torch.from_numpy(W.rows(g, (B, H, D), D, W.BF16).view(np.int16)).to(device).view(torch.bfloat16)
    keep, ios = [], []
    for l, t in enumerate(lt):
        q, k, v, o = mk(), mk(), mk(), torch.empty((B, H, D), dtype=torch.bfloat16, device=device)
        if t == 0:
            kc = W.device_rows_(torch.empty((NB, H, 16, D), dtype=torch.bfloat16, device=device), 100 + l, D)
            vc = W.device_rows_(torch.empty_like(kc), 200 + l, D)
            keep += [q, k, v, o, kc, vc]
            ios.append(hyb.layer_io(o, q, k, v, kc, vc))
        else:
            sp = W.device_state_(torch.empty((B, H, D, D), device=device), 300 + l, db.seq_lens, D)
            keep += [q, k, v, o, sp]
            ios.append(hyb.layer_io(o, q, k, v, state_pool=sp, num_state_slots=B))
    bt = torch.from_numpy(db.pool.block_tables).to(device)
    lens = torch.from_numpy(db.seq_lens).to(device)
    slots = torch.from_numpy(g.permutation(B).astype(np.int32)).to(device)
    msl = int(db.seq_lens.max())
    ws_n = hyb.hyb_paged_attn_decode_workspace_size(B, msl, d)
    ws = torch.empty(ws_n, dtype=torch.uint8, device=device)
    # no slot mapping: each Full layer appends its new rows at seq_len - 1 via the block table
    meta = hyb.batch_meta(B, B, seq_lens=lens, block_tables=bt, state_slots=slots, max_seq_len=msl)
    sh = stream.cuda_stream

    def step():
        hyb.check(hyb.hyb_layer_dispatch(lt, 32, 0, ios, meta, d, 64, ws, ws_n, sh))
    hyb.hyb_launch_count(reset=True)
    step()
    launches = hyb.hyb_launch_count(reset=True)
    t = _time(step, stream, iters)
    # the same step captured once into a CUDA graph and replayed (no per-launch host work)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        step()                                   # every first-call set-up done before capture
        stream.synchronize()
        with torch.cuda.graph(graph, stream=stream):
            step()
    t_graph = _time(graph.replay, stream, iters)
    n_full, n_lin = int((lt == 0).sum()), int((lt == 1).sum())
    alg = n_full * (int(db.seq_lens.sum()) * H * D * 4 + 2 * B * H * D * 2) + n_lin * B * H * D * D * 8
    res = {"workload": "hybrid_32layer: [full,full,full,linear] x 8, batch 64, 80% ~lognormal(128) / 20% ~lognormal(2048)",
           "value": round(B * 32 / (t * 1e-3), 1), "unit": UNIT, "ms_per_step": round(t, 4),
           "launches_per_step": int(launches),
           "roofline": _roof("hbm", alg / (t * 1e-3) / 1e9, hbm, "GB/s", "whole 32-layer step (dispatch)", alg),
           "cuda_graph": {"value": round(B * 32 / (t_graph * 1e-3), 1), "ms_per_step": round(t_graph, 4),
                          "roofline": _roof("hbm", alg / (t_graph * 1e-3) / 1e9, hbm, "GB/s",
                                            "whole 32-layer step (graph replay)", alg)}}
    del graph
    del keep, ios
    torch.cuda.empty_cache()
    return res


def row_prefill(hyb, device, stream, iters, seed=0):
    """8 requests x 8192-token prompts, H=32, D=128: Full layer = slot mapping + KV append +
    tensor-core causal prefill over the paged cache; Linear layer = tensor-core chunked
    prefill (chunk 64) from a zero state."""
    import torch
    hbm, tf, _ = measured_peaks()
    pb = W.prefill_chunked(seed)
    B, H, D, NB = len(pb.q_lens), pb.H, pb.D, pb.pool.num_blocks
    cu_h = W.cu_from_lens(pb.q_lens)
    T = int(cu_h[-1])
    d = hyb.dims(H, D, NB, pb.pool.max_blocks, W.BF16)
    mk = lambda s: W.device_rows_(torch.empty((T, H, D), dtype=torch.bfloat16, device=device), s, D)
    q, k, v, ql, kl, vl = (mk(60 + i) for i in range(6))
    out, lo = torch.empty_like(q), torch.empty_like(q)
    kc = torch.zeros((NB, H, 16, D), dtype=torch.bfloat16, device=device)
    vc = torch.zeros_like(kc)
    st = torch.zeros((B, H, D, D), device=device)
    bt = torch.from_numpy(pb.pool.block_tables).to(device)
    cu = torch.from_numpy(cu_h).to(device)
    slots = torch.arange(B, dtype=torch.int32, device=device)
    reset = torch.ones(B, dtype=torch.uint8, device=device)
    slot = torch.empty(T, dtype=torch.int64, device=device)
    sh = stream.cuda_stream
    L = int(pb.q_lens.max())
    t_slot = _time(lambda: hyb.check(hyb.hyb_slot_mapping(slot, bt, cu, None, B, T, d, sh)), stream, iters)
    t_app = _time(lambda: hyb.check(hyb.hyb_paged_kv_append(k, v, slot, T, kc, vc, d, sh)), stream, iters)
    t_pf = _time(lambda: hyb.check(hyb.hyb_paged_attn_prefill_causal(out, q, kc, vc, bt, cu, None, B, T, L, d, sh)), stream, iters)
    t_lin = _time(lambda: hyb.check(hyb.hyb_linear_attn_chunked_prefill(lo, ql, kl, vl, cu, None, st, B, slots, reset,
                                                                        B, T, L, H, D, pb.chunk, W.BF16, sh)), stream, iters)
    st_, fl = hyb.hyb_device_status(clear=True)
    if st_ != 0:
        raise RuntimeError(f"device-side check flags {fl:#x}")
    n = pb.q_lens.astype(np.float64)
    pf_flops = 4.0 * H * D * float((n * (n + 1) / 2).sum())              # QK^T + PV over the causal triangle
    lin_flops = T * H * (4.0 * pb.chunk * D + 4.0 * D * D)                # per token-head: 4CD + 4D^2
    lin_bytes = 4 * T * H * D * 2 + B * H * D * D * 4                     # q,k,v read, o written, state written
    app_bytes = 2 * 2 * T * H * D * 2
    ai = lin_flops / lin_bytes
    lin_gbs = lin_bytes / (t_lin * 1e-3) / 1e9
    lin_tf = lin_flops / (t_lin * 1e-3) / 1e12
    res = {"workload": "prefill_chunked: 8 requests x 8192-token prompts, H=32, D=128, chunk 64",
           "value": round(T * 2 / ((t_slot + t_app + t_pf + t_lin) * 1e-3), 1), "unit": "prompt tokens/s per layer",
           "ms": {"slot_mapping": round(t_slot, 4), "kv_append": round(t_app, 4), "prefill_causal": round(t_pf, 4),
                  "linear_chunked_prefill": round(t_lin, 4)},
           "roofline": _roof("tensor", pf_flops / (t_pf * 1e-3) / 1e12, tf, "TFLOP/s", "prefill_tc_kernel (causal, paged)",
                             pf_flops, traffic=_traffic("prefill_tc", "prefill_tc.cu"),
                             peak_source="measured bf16_tflops (burst)"),
           "linear_chunked_prefill": _roof("hbm", lin_gbs, hbm, "GB/s", "linear_prefill_tc_kernel", lin_bytes,
                                           traffic=_traffic("linear_prefill_tc", "linear_tc.cu"),
                                           tflops=round(lin_tf, 1), tensor_frac=round(lin_tf / tf, 4),
                                           arithmetic_intensity=round(ai, 1),
                                           frac_of_min_peak_ai_bw=round(lin_tf / min(tf, ai * hbm / 1e3), 4)),
           "kv_append": _roof("hbm", app_bytes / (t_app * 1e-3) / 1e9, hbm, "GB/s", "kv_append_kernel", app_bytes,
                              traffic=_traffic("kv_append", "append.cu"))}
    del q, k, v, ql, kl, vl, out, lo, kc, vc, st
    torch.cuda.empty_cache()
    return res


def row_sliding_window(hyb, device, stream, iters, seed=0):
    """Sliding-window Full layers: decode of 8 requests x 131072 cached tokens with window
    8192 (only the window's blocks are read), and tensor-core causal prefill of 8 x 8192
    prompts with window 4096."""
    import torch
    hbm, tf, _ = measured_peaks()
    Wd, Wp = 8192, 4096
    db = W.decode_long_context(seed)
    B, H, D, NB = db.B, db.H, db.D, db.pool.num_blocks
    d = hyb.dims(H, D, NB, db.pool.max_blocks, W.BF16, window=Wd)
    kc = W.device_rows_(torch.empty((NB, H, 16, D), dtype=torch.bfloat16, device=device), 71, D)
    vc = W.device_rows_(torch.empty_like(kc), 72, D)
    g = W.rng(seed + 7)
    q = torch.from_numpy(W.rows(g, (B, H, D), D, W.BF16).view(np.int16)).to(device).view(torch.bfloat16)
    out = torch.empty_like(q)
    bt = torch.from_numpy(db.pool.block_tables).to(device)
    lens = torch.from_numpy(db.seq_lens).to(device)
    n = int(db.seq_lens.max())
    ws_n = hyb.hyb_paged_attn_decode_workspace_size(B, n, d)
    ws = torch.empty(max(ws_n, 16), dtype=torch.uint8, device=device)
    sh = stream.cuda_stream
    t_dec = _time(lambda: hyb.check(hyb.hyb_paged_attn_decode(out, q, kc, vc, bt, lens, B, n, d, ws, ws_n, sh)), stream, iters)
    dec_bytes = int(np.minimum(db.seq_lens, Wd).sum()) * H * D * 4 + 2 * B * H * D * 2
    del kc, vc
    torch.cuda.empty_cache()

    pb = W.prefill_chunked(seed)
    B, H, D, NB = len(pb.q_lens), pb.H, pb.D, pb.pool.num_blocks
    cu_h = W.cu_from_lens(pb.q_lens)
    T = int(cu_h[-1])
    dp = hyb.dims(H, D, NB, pb.pool.max_blocks, W.BF16, window=Wp)
    qp = W.device_rows_(torch.empty((T, H, D), dtype=torch.bfloat16, device=device), 73, D)
    kcp = W.device_rows_(torch.empty((NB, H, 16, D), dtype=torch.bfloat16, device=device), 74, D)
    vcp = W.device_rows_(torch.empty_like(kcp), 75, D)
    outp = torch.empty_like(qp)
    btp = torch.from_numpy(pb.pool.block_tables).to(device)
    cu = torch.from_numpy(cu_h).to(device)
    L = int(pb.q_lens.max())
    t_pf = _time(lambda: hyb.check(hyb.hyb_paged_attn_prefill_causal(outp, qp, kcp, vcp, btp, cu, None, B, T, L, dp, sh)),
                 stream, iters)
    st_, fl = hyb.hyb_device_status(clear=True)
    if st_ != 0:
        raise RuntimeError(f"device-side check flags {fl:#x}")
    keys = sum(float(np.minimum(np.arange(1, m + 1), Wp).sum()) for m in pb.q_lens)
    pf_flops = 4.0 * H * D * keys                                          # QK^T + PV inside the band
    res = {"workload": "sliding_window: decode 8 x 131072 cached tokens with window 8192; "
                       "prefill 8 x 8192 prompts with window 4096; H=32, D=128",
           "value": round(B * 1 / (t_dec * 1e-3), 1), "unit": "req-tokens/s per layer (windowed decode)",
           "ms": {"paged_decode_window": round(t_dec, 4), "prefill_causal_window": round(t_pf, 4)},
           "roofline": _roof("hbm", dec_bytes / (t_dec * 1e-3) / 1e9, hbm, "GB/s",
                             "paged_decode, window 8192 (split-K + combine)", dec_bytes),
           "prefill_window": _roof("tensor", pf_flops / (t_pf * 1e-3) / 1e12, tf, "TFLOP/s",
                                   "prefill_tc_kernel, window 4096", pf_flops,
                                   peak_source="measured bf16_tflops (burst)")}
    del qp, kcp, vcp, outp
    torch.cuda.empty_cache()
    return res


def row_state_precision(hyb, device, stream, iters, seed=0):
    """Linear decode step with the fp32 state the pages prescribe vs bf16 and fp16 state
    pools: time per step on 32 requests x 32 heads x 128 x 128, and the output drift of the
    16-bit states against the fp32 state over 16384 decode steps (4 requests x 4 heads,
    fp32 q/k/v, zero initial state)."""
    import torch
    hbm, _, _ = measured_peaks()
    B, H, D = 32, 32, 128
    g = W.rng(seed + 11)
    mk = lambda: torch.from_numpy(W.rows(g, (B, H, D), D, W.BF16).view(np.int16)).to(device).view(torch.bfloat16)
    q, k, v = mk(), mk(), mk()
    out = torch.empty_like(q)
    slots = torch.arange(B, dtype=torch.int32, device=device)
    st32 = W.device_state_(torch.empty((B, H, D, D), device=device), 81, np.full(B, 2048), D)
    st16 = {sd: st32.to(torch.bfloat16 if sd == W.BF16 else torch.float16) for sd in (W.BF16, hyb.HYB_F16)}
    sh = stream.cuda_stream
    t = {"fp32": _time(lambda: hyb.check(hyb.hyb_linear_attn_step(out, q, k, v, st32, B, slots, B, H, D, W.BF16, sh)),
                       stream, iters)}
    for sd, name in ((W.BF16, "bf16"), (hyb.HYB_F16, "fp16")):
        t[name] = _time(lambda: hyb.check(hyb.hyb_linear_attn_step_lowp(out, q, k, v, st16[sd], sd, B, slots, B, H, D,
                                                                        W.BF16, sh)), stream, iters)
    byt = {"fp32": B * H * D * D * 8, "bf16": B * H * D * D * 4, "fp16": B * H * D * D * 4}
    del st32, st16
    # drift: the same fp32 q/k/v stream through the three state types
    Bd, Hd, T = 4, 4, 16384
    qs = W.device_rows_(torch.empty((T, Bd, Hd, D), device=device), 82, D)
    ks = W.device_rows_(torch.empty_like(qs), 83, D)
    vs = W.device_rows_(torch.empty_like(qs), 84, D)
    outs = {n: torch.empty_like(qs) for n in ("fp32", "bf16", "fp16")}
    pools = {"fp32": torch.zeros((Bd, Hd, D, D), device=device),
             "bf16": torch.zeros((Bd, Hd, D, D), dtype=torch.bfloat16, device=device),
             "fp16": torch.zeros((Bd, Hd, D, D), dtype=torch.float16, device=device)}
    sl = torch.arange(Bd, dtype=torch.int32, device=device)
    with torch.cuda.stream(stream):
        for i in range(T):
            hyb.check(hyb.hyb_linear_attn_step(outs["fp32"][i], qs[i], ks[i], vs[i], pools["fp32"], Bd, sl, Bd, Hd, D,
                                               W.F32, sh))
            hyb.check(hyb.hyb_linear_attn_step_lowp(outs["bf16"][i], qs[i], ks[i], vs[i], pools["bf16"], W.BF16, Bd, sl,
                                                    Bd, Hd, D, W.F32, sh))
            hyb.check(hyb.hyb_linear_attn_step_lowp(outs["fp16"][i], qs[i], ks[i], vs[i], pools["fp16"], hyb.HYB_F16, Bd,
                                                    sl, Bd, Hd, D, W.F32, sh))
    stream.synchronize()
    st_, fl = hyb.hyb_device_status(clear=True)
    if st_ != 0:
        raise RuntimeError(f"device-side check flags {fl:#x}")
    drift = {}
    for n in ("bf16", "fp16"):
        drift[n] = {}
        for tt in (256, 1024, 4096, 16384):
            ref = outs["fp32"][tt - 64:tt]
            drift[n][str(tt)] = float((outs[n][tt - 64:tt] - ref).abs().max() / ref.abs().max())
    del qs, ks, vs, outs, pools
    torch.cuda.empty_cache()
    return {"workload": "state_precision: linear step, 32 requests x 32 heads x 128 x 128; drift over 16384 steps",
            "value": round(B / (t["fp32"] * 1e-3), 1), "unit": "req-tokens/s per layer (fp32 state linear step)",
            "ms": {n: round(x, 4) for n, x in t.items()},
            "roofline": {n: _roof("hbm", byt[n] / (t[n] * 1e-3) / 1e9, hbm, "GB/s", f"linear step, {n} state", byt[n])
                         for n in t},
            "drift_vs_fp32_state": {"metric": "max |o - o_fp32| / max |o_fp32| over the 64 steps before t",
                                    "steps": T, **drift}}


def row_block32(hyb, device, stream, iters, seed=0):
    """32-token blocks (the vLLM/SGLang page's size): paged decode of the 32-request batch
    (lengths 128..4096) and tensor-core causal prefill of 8 x 8192 prompts, each pool laid
    out in 32-token blocks."""
    import torch
    hbm, tf, _ = measured_peaks()
    bs = 32
    g = W.rng(seed + 13)
    lens = W.lens_uniform(g, 32, 128, 4096)
    pool = W.block_pool(g, lens, block_size=bs)
    B, H, D, NB = 32, 32, 128, pool.num_blocks
    d = hyb.dims(H, D, NB, pool.max_blocks, W.BF16, block_size=bs)
    kc = W.device_rows_(torch.empty((NB, H, bs, D), dtype=torch.bfloat16, device=device), 91, D)
    vc = W.device_rows_(torch.empty_like(kc), 92, D)
    q = torch.from_numpy(W.rows(g, (B, H, D), D, W.BF16).view(np.int16)).to(device).view(torch.bfloat16)
    out = torch.empty_like(q)
    bt = torch.from_numpy(pool.block_tables).to(device)
    ln = torch.from_numpy(lens).to(device)
    n = int(lens.max())
    ws_n = hyb.hyb_paged_attn_decode_workspace_size(B, n, d)
    ws = torch.empty(max(ws_n, 16), dtype=torch.uint8, device=device)
    sh = stream.cuda_stream
    t_dec = _time(lambda: hyb.check(hyb.hyb_paged_attn_decode(out, q, kc, vc, bt, ln, B, n, d, ws, ws_n, sh)),
                  stream, iters)
    dec_bytes = int(lens.sum()) * H * D * 4 + 2 * B * H * D * 2
    del kc, vc
    pb = W.prefill_chunked(seed)
    Bp = len(pb.q_lens)
    cu_h = W.cu_from_lens(pb.q_lens)
    T = int(cu_h[-1])
    ppool = W.block_pool(W.rng(seed + 14), pb.q_lens, block_size=bs)
    dp = hyb.dims(H, D, ppool.num_blocks, ppool.max_blocks, W.BF16, block_size=bs)
    qp = W.device_rows_(torch.empty((T, H, D), dtype=torch.bfloat16, device=device), 93, D)
    kcp = W.device_rows_(torch.empty((ppool.num_blocks, H, bs, D), dtype=torch.bfloat16, device=device), 94, D)
    vcp = W.device_rows_(torch.empty_like(kcp), 95, D)
    outp = torch.empty_like(qp)
    btp = torch.from_numpy(ppool.block_tables).to(device)
    cu = torch.from_numpy(cu_h).to(device)
    L = int(pb.q_lens.max())
    t_pf = _time(lambda: hyb.check(hyb.hyb_paged_attn_prefill_causal(outp, qp, kcp, vcp, btp, cu, None, Bp, T, L, dp, sh)),
                 stream, iters)
    st_, fl = hyb.hyb_device_status(clear=True)
    if st_ != 0:
        raise RuntimeError(f"device-side check flags {fl:#x}")
    nq = pb.q_lens.astype(np.float64)
    pf_flops = 4.0 * H * D * float((nq * (nq + 1) / 2).sum())
    del qp, kcp, vcp, outp
    torch.cuda.empty_cache()
    return {"workload": "block32: decode 32 requests x U{128..4096} and prefill 8 x 8192, H=32, D=128, 32-token blocks",
            "value": round(B / (t_dec * 1e-3), 1), "unit": "req-tokens/s per layer (decode, 32-token blocks)",
            "ms": {"paged_decode": round(t_dec, 4), "prefill_causal": round(t_pf, 4)},
            "roofline": _roof("hbm", dec_bytes / (t_dec * 1e-3) / 1e9, hbm, "GB/s",
                              "paged_decode, 32-token blocks (split-K + combine)", dec_bytes),
            "prefill": _roof("tensor", pf_flops / (t_pf * 1e-3) / 1e12, tf, "TFLOP/s",
                             "prefill_tc_kernel, 32-token blocks", pf_flops,
                             peak_source="measured bf16_tflops (burst)")}


def row_bucketing(hyb, device, stream, iters, seed=0):
    """Length-bucketed batching: the 32-layer decode step of the 64-request 80%/20% mix run as
    one call in arrival order, as one call sorted by length, and as two calls (requests with
    <= 512 cached tokens, then the rest). The kernels take ragged batches without padding, so
    bucketing only changes the order and the number of launches."""
    import torch
    hbm, _, _ = measured_peaks()
    db = W.decode_hybrid_32layer(seed)
    lt = db.extra["layer_types"]
    B, H, D, NB, MB = db.B, db.H, db.D, db.pool.num_blocks, db.pool.max_blocks
    d = hyb.dims(H, D, NB, MB, W.BF16)
    g = W.rng(seed + 19)
    keep, per_layer = [], []
    for l, t in enumerate(lt):
        q = W.device_rows_(torch.empty((B, H, D), dtype=torch.bfloat16, device=device), 400 + l, D)
        o = torch.empty_like(q)
        if t == 0:
            kc = W.device_rows_(torch.empty((NB, H, 16, D), dtype=torch.bfloat16, device=device), 500 + l, D)
            vc = W.device_rows_(torch.empty_like(kc), 600 + l, D)
            keep += [q, o, kc, vc]
            per_layer.append((q, o, kc, vc, None))
        else:
            sp = W.device_state_(torch.empty((B, H, D, D), device=device), 700 + l, db.seq_lens, D)
            keep += [q, o, sp]
            per_layer.append((q, o, None, None, sp))
    sh = stream.cuda_stream

    def plan(order):
        """One dispatch call over the requests in `order` (rows r of q/k/v/out = order[r])."""
        n = len(order)
        lens = db.seq_lens[order]
        bt = torch.from_numpy(np.ascontiguousarray(db.pool.block_tables[order])).to(device)
        ln = torch.from_numpy(lens).to(device)
        slots = torch.from_numpy(np.asarray(order, np.int32)).to(device)
        msl = int(lens.max())
        ws_n = hyb.hyb_paged_attn_decode_workspace_size(n, msl, d)
        ws = torch.empty(max(ws_n, 16), dtype=torch.uint8, device=device)
        rows = torch.from_numpy(np.asarray(order, np.int64)).to(device)
        ios = []
        bufs = [bt, ln, slots, ws]
        for (q, o, kc, vc, sp) in per_layer:
            qb, ob = q[rows].contiguous(), o[rows].contiguous()
            bufs += [qb, ob]
            ios.append(hyb.layer_io(ob, qb, qb, qb, kc, vc) if kc is not None
                       else hyb.layer_io(ob, qb, qb, qb, state_pool=sp, num_state_slots=B))
        meta = hyb.batch_meta(n, n, seq_lens=ln, block_tables=bt, state_slots=slots, max_seq_len=msl)

        def run():                         # new rows at seq_len - 1 via the block table
            hyb.check(hyb.hyb_layer_dispatch(lt, len(lt), 0, ios, meta, d, 64, ws, ws_n, sh))
        return run, bufs

    arrival = np.arange(B)
    by_len = np.argsort(-db.seq_lens, kind="stable")
    short = np.nonzero(db.seq_lens <= 512)[0]
    long_ = np.nonzero(db.seq_lens > 512)[0]
    res_ms = {}
    for name, groups in (("one_call_arrival_order", [arrival]), ("one_call_sorted_by_length", [by_len]),
                         ("two_buckets_short_then_long", [short, long_])):
        runs = [plan(gr) for gr in groups if len(gr)]
        res_ms[name] = round(_time(lambda: [r() for r, _ in runs], stream, iters), 4)
        del runs
    alg = int((lt == 0).sum()) * (int(db.seq_lens.sum()) * H * D * 4 + 2 * B * H * D * 2) + \
        int((lt == 1).sum()) * B * H * D * D * 8
    t0 = res_ms["one_call_arrival_order"]
    del keep, per_layer
    torch.cuda.empty_cache()
    return {"workload": "bucketing: 32-layer decode step, batch 64, 80% ~128 / 20% ~2048 cached tokens",
            "value": round(B * 32 / (t0 * 1e-3), 1), "unit": UNIT, "ms_per_step": res_ms,
            "buckets": {"short_le_512": int(len(short)), "long": int(len(long_))},
            "roofline": _roof("hbm", alg / (t0 * 1e-3) / 1e9, hbm, "GB/s", "whole 32-layer step, one call", alg)}


def row_prefill_lengths(hyb, device, stream, iters, seed=0):
    """Tensor-core causal prefill at one CTA count (8 192 pairs of query tiles) and five
    prompt lengths, 32 x 2048 ... 2 x 32768 tokens, H=32, D=128: how the per-CTA fill and
    drain weigh against the per-key-step cost."""
    import torch
    _, tf, _ = measured_peaks()
    res = {"workload": "prefill_lengths: causal prefill, 8192 CTAs, B x L = 32x2048 .. 2x32768, H=32, D=128",
           "unit": "TFLOP/s", "cases": {}}
    for B, L in ((32, 2048), (16, 4096), (8, 8192), (4, 16384), (2, 32768)):
        pb = W.prefill_chunked(seed, B=B, L=L)
        H, D, NB = pb.H, pb.D, pb.pool.num_blocks
        cu_h = W.cu_from_lens(pb.q_lens)
        T = int(cu_h[-1])
        d = hyb.dims(H, D, NB, pb.pool.max_blocks, W.BF16)
        q = W.device_rows_(torch.empty((T, H, D), dtype=torch.bfloat16, device=device), 61, D)
        kc = W.device_rows_(torch.empty((NB, H, 16, D), dtype=torch.bfloat16, device=device), 5, D)
        vc = W.device_rows_(torch.empty_like(kc), 6, D)
        bt = torch.from_numpy(pb.pool.block_tables).to(device)
        cu = torch.from_numpy(cu_h).to(device)
        out = torch.empty_like(q)
        sh = stream.cuda_stream
        t = _time(lambda: hyb.check(hyb.hyb_paged_attn_prefill_causal(out, q, kc, vc, bt, cu, None, B, T, L, d, sh)),
                  stream, min(iters, 10))
        n = pb.q_lens.astype(np.float64)
        fl = 4.0 * H * D * float((n * (n + 1) / 2).sum())
        res["cases"][f"{B}x{L}"] = {"ms": round(t, 4), "TFLOP/s": round(fl / (t * 1e-3) / 1e12, 1),
                                    "frac": round(fl / (t * 1e-3) / 1e12 / tf, 4)}
        del q, kc, vc, out
        torch.cuda.empty_cache()
    st_, fl = hyb.hyb_device_status(clear=True)
    if st_ != 0:
        raise RuntimeError(f"device-side check flags {fl:#x}")
    return res


ROWS = {"long_context_decode": row_long_context, "hybrid_32layer": row_hybrid_32layer,
        "prefill_chunked": row_prefill, "sliding_window": row_sliding_window,
        "state_precision": row_state_precision, "block32": row_block32, "bucketing": row_bucketing}
EXTRA_ROWS = {"prefill_lengths": row_prefill_lengths}   # --workload only, not in the default rows


def bench_ours(args, dist):
    import torch
    from paged_kv_linear_gb300 import _build
    if dist.rank == 0 or dist.world == 1:
        _build.build()
    dist.barrier()
    _build.build()
    import paged_kv_linear_gb300 as hyb

    torch.cuda.set_device(dist.local)
    device = torch.device("cuda", dist.local)
    if args.workload != "decode_single_layer":          # one other workload, timed alone
        stream = torch.cuda.Stream(device=device)
        r = {**ROWS, **EXTRA_ROWS}[args.workload](hyb, device, stream, max(args.steps, 1), args.seed + dist.rank)
        r.update({"metric": METRIC, "n_gpus": dist.world, "steps": args.steps, "warmup": 3,
                  "higher_is_better": True, "dtype": "bf16", "data": "synthetic"})
        return r
    wl = build_workload(args.seed + dist.rank, device)
    B, H, D, NB, MB, db = wl["B"], wl["H"], wl["D"], wl["NB"], wl["MB"], wl["db"]
    d = hyb.dims(H, D, NB, MB, W.BF16)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16) if a.dtype == np.uint16 else a).to(device)
    bf = lambda a: dev(a).view(torch.bfloat16) if a.dtype == np.uint16 else dev(a)
    x = {n: bf(a) for n, a in wl["host"].items()}
    bt = dev(db.pool.block_tables)
    lens = dev(db.seq_lens)
    slots = dev(wl["slots_h"])
    msl = int(db.seq_lens.max())
    ws_n = hyb.hyb_paged_attn_decode_workspace_size(B, msl, d)
    ws = torch.empty(max(ws_n, 16), dtype=torch.uint8, device=device)
    out_f = torch.empty((B, H, D), dtype=torch.bfloat16, device=device)
    out_l = torch.empty_like(out_f)
    stream = torch.cuda.Stream(device=device)
    sh = stream.cuda_stream
    L = 2
    n_ops = 2
    names = ["paged_decode", "linear_step"]

    def step(ev=None):
        if ev: ev[0].record(stream)
        # Full layer: KV append (at position seq_len - 1 through the block table) and paged
        # decode in one launch, plus the split combine
        hyb.check(hyb.hyb_paged_attn_decode_append(out_f, x["qf"], x["kf"], x["vf"], None, wl["kc"], wl["vc"],
                                                   bt, lens, B, msl, d, ws, ws_n, sh))
        if ev: ev[1].record(stream)
        hyb.check(hyb.hyb_linear_attn_step(out_l, x["ql"], x["kl"], x["vl"], wl["state"], B, slots, B, H, D, W.BF16, sh))
        if ev: ev[2].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    # An event recorded between two kernels keeps the second from launching while the first
    # drains (programmatic dependent launch), so per-op events would slow the step they
    # measure (0.222 against 0.205 ms here). One event pair brackets all K steps for the
    # step time; every INSTR-th step also carries per-op events for the breakdown and the
    # decode kernel's roofline.
    INSTR = 8
    instr = [s for s in range(args.steps) if s % INSTR == 0]
    evs = {s: [torch.cuda.Event(enable_timing=True) for _ in range(n_ops + 1)] for s in instr}
    loop_ev = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
    clocks = ClockSampler(dist.local)
    clocks.start()
    time.sleep(0.3)
    dist.barrier()
    torch.cuda.synchronize()
    hyb.hyb_launch_count(reset=True)
    clocks.mark("t0")
    with torch.cuda.stream(stream):
        loop_ev[0].record(stream)
        for s in range(args.steps):
            step(evs.get(s))
        loop_ev[1].record(stream)
    torch.cuda.synchronize()
    clocks.mark("t1")
    launches = hyb.hyb_launch_count(reset=True)
    dist.barrier()
    clocks.stop()
    per_op = np.zeros(n_ops)
    step_ms = []                                  # instrumented steps (per-op events)
    for e in evs.values():
        step_ms.append(e[0].elapsed_time(e[n_ops]))
        for i in range(n_ops):
            per_op[i] += e[i].elapsed_time(e[i + 1])
    per_op /= len(evs)
    ms_step = dist.max(loop_ev[0].elapsed_time(loop_ev[1]) / args.steps)
    units = dist.sum(B * L)                       # request-tokens per layer-step over all ranks
    value = units / (ms_step * 1e-3)
    st, flags = hyb.hyb_device_status(clear=True)
    if st != 0:
        raise RuntimeError(f"device-side check flags {flags:#x}")

    # ---- roofline of the dominant kernel (paged decode: split-K kernel + combine)
    hbm_peak, tf_peak, peak_kind = measured_peaks()
    tokens = int(db.seq_lens.sum())
    # K+V read, q read, out write, and the new K/V rows read and written into the cache
    alg_bytes = tokens * H * D * 2 * 2 + 2 * B * H * D * 2 + 4 * B * H * D * 2
    achieved = alg_bytes / (per_op[0] * 1e-3) / 1e9
    trec = traffic_record("paged_decode", "decode.cu")
    roofline = {"kernel": "paged_decode with the KV append fused (split-K + combine)", "bound": "hbm",
                "achieved": round(achieved, 1),
                "peak": hbm_peak, "unit": "GB/s", "frac": round(achieved / hbm_peak, 4),
                "traffic": (int(trec["bytes_per_launch"]) if trec else None),
                "algorithmic_bytes": alg_bytes, "peak_source": f"{peak_kind} hbm_gbs"}
    lin_bytes = B * H * D * D * 4 * 2
    ops = {n: {"ms": round(float(t), 5)} for n, t in zip(names, per_op)}
    ops["paged_decode"]["GB/s"] = round(achieved, 1)
    ops["linear_step"]["GB/s"] = round(lin_bytes / (per_op[1] * 1e-3) / 1e9, 1)
    ops["linear_step"]["frac"] = round(ops["linear_step"]["GB/s"] / hbm_peak, 4)
    ops["linear_step"]["traffic"] = _traffic("linear_step", "linear.cu")

    # ---- end to end through the public dispatcher, host buffers, copies timed. All of a
    # step's inputs sit in one pinned host buffer and go over in one copy; both layers'
    # outputs come back in one copy.
    host_arrays = dict(wl["host"])
    host_arrays.update({"lens": db.seq_lens, "bt": db.pool.block_tables, "slots": wl["slots_h"]})
    offs, total = {}, 0
    for n, a in host_arrays.items():
        offs[n] = total
        total += (a.nbytes + 255) // 256 * 256
    h_all = torch.empty(total, dtype=torch.uint8).pin_memory()
    h_all_np = h_all.numpy()
    for n, a in host_arrays.items():
        h_all_np[offs[n]:offs[n] + a.nbytes] = np.ascontiguousarray(a).view(np.uint8).reshape(-1)
    h2d = sum(a.nbytes for a in host_arrays.values())
    # Two sets of device buffers: step s copies its inputs into set s % 2 on a copy stream
    # while the compute stream still runs step s - 1, and reads its outputs back while step
    # s + 1 computes (the pipelining a serving loop does).
    sets = []
    for _ in range(2):
        d_all = torch.empty(total, dtype=torch.uint8, device=device)

        def dview(n, d_all=d_all):
            a = host_arrays[n]
            t = d_all[offs[n]:offs[n] + a.nbytes]
            t = t.view(torch.bfloat16) if a.dtype == np.uint16 else t.view(getattr(torch, a.dtype.name))
            return t.view(a.shape)

        d_in = {n: dview(n) for n in wl["host"]}
        d_meta = {n: dview(n) for n in ("lens", "bt", "slots")}
        out_all = torch.empty(2 * B * H * D, dtype=torch.bfloat16, device=device)
        e_out_f, e_out_l = out_all[:B * H * D].view(B, H, D), out_all[B * H * D:].view(B, H, D)
        meta = hyb.batch_meta(B, B, seq_lens=d_meta["lens"], block_tables=d_meta["bt"],
                              state_slots=d_meta["slots"], max_seq_len=msl)   # new rows at seq_len - 1 via the table
        ios = [hyb.layer_io(e_out_f, d_in["qf"], d_in["kf"], d_in["vf"], wl["kc"], wl["vc"]),
               hyb.layer_io(e_out_l, d_in["ql"], d_in["kl"], d_in["vl"], state_pool=wl["state"],
                            num_state_slots=B)]
        sets.append(dict(d_all=d_all, d_meta=d_meta, out_all=out_all, meta=meta, ios=ios,
                         h_out=torch.empty(2 * B * H * D, dtype=torch.int16).pin_memory(),
                         loaded=torch.cuda.Event(), computed=torch.cuda.Event(), read=torch.cuda.Event()))
    d2h = sets[0]["h_out"].numel() * sets[0]["h_out"].element_size()
    h2d_stream = torch.cuda.Stream(device=device)   # one stream per direction: a read-back
    d2h_stream = torch.cuda.Stream(device=device)   # must not hold up the next step's inputs

    def e2e_step(i):
        st = sets[i % 2]
        if i >= 2:
            h2d_stream.wait_event(st["read"])        # step i - 2's outputs are back (so it is done)
        with torch.cuda.stream(h2d_stream):
            st["d_all"].copy_(h_all, non_blocking=True)
            st["loaded"].record(h2d_stream)
        stream.wait_event(st["loaded"])
        hyb.check(hyb.hyb_layer_dispatch([0, 1], 2, 0, st["ios"], st["meta"], d, 64, ws, ws_n, sh))
        st["computed"].record(stream)
        d2h_stream.wait_event(st["computed"])
        with torch.cuda.stream(d2h_stream):
            st["h_out"].copy_(st["out_all"].view(torch.int16), non_blocking=True)
            st["read"].record(d2h_stream)

    e2e_steps = max(10, min(args.steps, 500))
    with torch.cuda.stream(stream):
        for i in range(3):
            e2e_step(i)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        dist.barrier()
        e0.record(stream)
        h2d_stream.wait_event(e0)                # no copy of the timed steps starts before e0
        for i in range(e2e_steps):
            e2e_step(i)
        for st in sets:                          # the last steps' outputs are on the host
            stream.wait_event(st["read"])
        e1.record(stream)
        torch.cuda.synchronize()
    e2e_ms = dist.max(e0.elapsed_time(e1) / e2e_steps)
    e2e_val = units / (e2e_ms * 1e-3)

    # ---- CPU oracle beside it (rank 0, N = 1 only)
    cpu = None
    if dist.world == 1:
        cpu = cpu_baseline_decode(wl, budget_s=10.0)

    # ---- the other rows of the hot path, each against its own roofline (N = 1 only)
    rows = None
    if dist.world == 1 and not args.no_rows:
        del wl
        torch.cuda.empty_cache()
        rows = {name: fn(hyb, device, stream, 20, args.seed) for name, fn in ROWS.items()}

    return {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": dist.world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 5),
        "ms_per_step_p50": round(float(np.percentile(step_ms, 50)), 5),
        "ms_per_step_p99": round(float(np.percentile(step_ms, 99)), 5),
        "timing": (f"ms_per_step: one CUDA event pair around all {args.steps} steps; p50/p99 and ops: "
                   f"the {len(evs)} steps (every {INSTR}th) that also carry per-op events"),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1)/sqrt(D) q/k/v, shuffled block pool, N(0,seq/D^2) states)",
        "config": {"workload": "decode_single_layer: 32 requests, H=32, D=128, block 16, seq_lens U{128..4096}, "
                               "1 Full paged-decode + 1 Linear step", "B": B, "H": H, "D": D,
                   "layers": ["full", "linear"], "kv_tokens": tokens, "pool_blocks": NB,
                   "l2": "no flush: per-step working set %.2f GB > 129 MB L2" % ((alg_bytes + lin_bytes) / 1e9),
                   "parallelism": f"replicas x{dist.world}"},
        "roofline": roofline, "ops": ops,
        "e2e": {"value": round(e2e_val, 1), "unit": UNIT, "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h),
                "path": "hyb_layer_dispatch; inputs in one pinned buffer, one copy each way, "
                        "on copy streams double-buffered against the compute stream"},
        "gpu_launches": int(launches),
        "clocks": clocks.summary(),
        "cpu_baseline": cpu,
        "rows": rows,
    }


def cpu_baseline_decode(wl, budget_s=15.0, requests=None):
    """Times the CPU oracle (as it stands) on a bounded sample of the same workload: whole
    requests through the Full-layer decode and the Linear step, all heads."""
    import oracle
    db = wl["db"]
    H, D = wl["H"], wl["D"]
    cores = oracle.set_threads(0)
    kc = wl["kc"].cpu().view(__import__("torch").int16).numpy().view(np.uint16)
    vc = wl["vc"].cpu().view(__import__("torch").int16).numpy().view(np.uint16)
    st = wl["state"].cpu().numpy()
    hq = wl["host"]
    done, t_used = 0, 0.0
    order = list(range(wl["B"])) if requests is None else list(requests)
    passes = 0
    while t_used < budget_s:             # repeat the whole batch until ~budget_s of CPU work
        for b in order:
            t0 = time.perf_counter()
            oracle.full_decode(hq["qf"][b:b + 1], kc, vc, db.pool.block_tables[b:b + 1],
                               db.seq_lens[b:b + 1], D ** -0.5)
            oracle.linear_step(hq["ql"][b:b + 1], hq["kl"][b:b + 1], hq["vl"][b:b + 1], st,
                               wl["slots_h"][b:b + 1])
            t_used += time.perf_counter() - t0
            done += 1
            if t_used > budget_s:
                break
        passes += 1
    res = {"value": round(done * 2 / t_used, 2), "unit": UNIT, "cores": cores, "kind": "oracle",
           "sample": f"{done} request-steps ({passes} pass(es) over the {wl['B']} requests, all {H} heads; "
                     f"Full decode + Linear step), fp64 C oracle with OpenMP over (request, head), "
                     f"{t_used:.1f} s"}
    # the same oracle on one core, over a short sample (first requests of the batch)
    oracle.set_threads(1)
    done1, t1 = 0, 0.0
    for b in order:
        if t1 > budget_s / 5:
            break
        t0 = time.perf_counter()
        oracle.full_decode(hq["qf"][b:b + 1], kc, vc, db.pool.block_tables[b:b + 1], db.seq_lens[b:b + 1], D ** -0.5)
        oracle.linear_step(hq["ql"][b:b + 1], hq["kl"][b:b + 1], hq["vl"][b:b + 1], st, wl["slots_h"][b:b + 1])
        t1 += time.perf_counter() - t0
        done1 += 1
    oracle.set_threads(cores)
    res["single_thread"] = {"value": round(done1 * 2 / t1, 2), "unit": UNIT, "cores": 1,
                            "sample": f"the first {done1} requests of the batch, {t1:.1f} s"}
    return res


def bench_reference(args, dist):
    """The CPU oracle as the reference arm: each step is one request (rotating through the
    batch) through both layers, on the host cores."""
    if dist.rank != 0:
        return None
    import oracle
    oracle.build()
    db = W.decode_single_layer(args.seed)
    g = W.rng(args.seed + 1)
    B, H, D = db.B, db.H, db.D
    cores = oracle.set_threads(0)
    # pool contents for the sampled requests only (host-drawn, same shapes)
    kc = np.empty((db.pool.num_blocks, H, 16, D), np.uint16)
    vc = np.empty_like(kc)
    gk = W.rng(args.seed + 7)
    kc[:] = W.rows(gk, kc.shape, D, W.BF16)
    vc[:] = W.rows(gk, vc.shape, D, W.BF16)
    st = W.synthetic_state(g, B, H, D, db.seq_lens)
    q, k, v = (W.rows(g, (B, H, D), D, W.BF16) for _ in range(3))
    slots = np.arange(B, dtype=np.int32)

    def one(b):
        oracle.full_decode(q[b:b + 1], kc, vc, db.pool.block_tables[b:b + 1], db.seq_lens[b:b + 1], D ** -0.5)
        oracle.linear_step(q[b:b + 1], k[b:b + 1], v[b:b + 1], st, slots[b:b + 1])

    for i in range(args.warmup):
        one(i % B)
    t0 = time.perf_counter()
    for i in range(args.steps):
        one(i % B)
    dt = time.perf_counter() - t0
    ms = dt * 1e3 / args.steps
    val = 2 / (ms * 1e-3)
    return {"impl": "reference", "metric": METRIC, "value": round(val, 2), "unit": UNIT, "n_gpus": dist.world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "decode_single_layer: 32 requests, H=32, D=128, block 16, seq_lens U{128..4096}, "
                                   "1 Full paged-decode + 1 Linear step", "sample_per_step": "1 request, all heads"},
            "cpu_baseline": {"value": round(val, 2), "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": "1 request per step (rotating over the 32), all 32 heads, Full decode + Linear step"},
            "e2e": {"value": round(val, 2), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    args = parse()
    dist = Dist(args.gpus)
    if args.impl == "reference":
        res = bench_reference(args, dist)
    else:
        res = bench_ours(args, dist)
    if dist.rank == 0 and res is not None:
        print(json.dumps(res), flush=True)
    if dist.pg:
        dist.pg.destroy_process_group()


if __name__ == "__main__":
    main()
