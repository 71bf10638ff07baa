#!/usr/bin/env python3
"""Benchmark of the hybrid-attention decode hot path on GB300 (one JSON line on rank 0).

Headline workload (`hybrid_32layer`): a 32-layer hybrid model, layer types
[full, full, full, linear] x 8, batch 64 with 80 % of the requests around 128 cached tokens
and 20 % around 2048 (lognormal), H=32, D=128, bf16 KV in 16-token blocks shuffled across a
pool, fp32 linear states. One step = one decode token for every request through all 32
layers in one hyb_layer_dispatch call: each Full layer is one launch of the paged decode
with the KV append fused in (new row at seq_len - 1 through the block table) plus its split
combine, each Linear layer one in-place state step. Metric: req-tokens/s per layer
= B * 32 / step time. Inputs live in HBM before timing; a step streams ~15.8 GB of KV and
state, far more than the 129 MB L2, so no flush is needed.

`value` is device time (CUDA events on the launching stream). `e2e` is the same step through
the same public call with all 32 layers' q/k/v and the batch metadata copied from pinned host
memory and all outputs copied back, inside the timed region. `rows` time the other
workloads (single-layer decode batch, 131K-context decode, chunked prefill, and the
variants), each against its own roofline and, for the four workloads of the method, beside
the CPU oracle. `--impl reference` times the CPU oracle on the headline workload instead
(bounded sample per step, host cores). With torchrun (N > 1) every rank runs its own
replica (the path shards by request with no exchange) and rank 0 reports the aggregate.
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
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--workload", default="hybrid_32layer",
                    choices=["hybrid_32layer", *ROWS, *EXTRA_ROWS],
                    help="hybrid_32layer is the headline; the others are timed alone (e.g. for profiling)")
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


# ------------------------------------------------------------------ timing helpers
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


def _u16(t):
    """A device bf16 tensor as host bf16 bit patterns (numpy uint16)."""
    import torch
    return t.cpu().view(torch.int16).numpy().view(np.uint16)


def _dev_bf16(a, device):
    """Host bf16 bit patterns (numpy uint16) as a device bf16 tensor."""
    import torch
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(device).view(torch.bfloat16)


def _check_device(hyb):
    st_, fl = hyb.hyb_device_status(clear=True)
    if st_ != 0:
        raise RuntimeError(f"device-side check flags {fl:#x}")


# ------------------------------------------------------------------ 32-layer hybrid batch
def build_hybrid(seed, device):
    """The 32-layer hybrid decode batch: every layer's q/k/v drawn on the host (bf16 bit
    patterns, [L][3][B][H][D]); each Full layer's K and V pools and each Linear layer's state
    pool filled on the device (seeded)."""
    import torch
    db = W.decode_hybrid_32layer(seed)
    lt = [int(x) for x in db.extra["layer_types"]]
    L = len(lt)
    B, H, D, NB, MB = db.B, db.H, db.D, db.pool.num_blocks, db.pool.max_blocks
    g = W.rng(seed + 9)
    qkv = W.rows(g, (L, 3, B, H, D), D, W.BF16)
    slots = g.permutation(B).astype(np.int32)
    kv, st = {}, {}
    for l, t in enumerate(lt):
        if t == 0:
            kv[l] = tuple(W.device_rows_(torch.empty((NB, H, 16, D), dtype=torch.bfloat16, device=device),
                                         base + l, D) for base in (100, 200))
        else:
            st[l] = W.device_state_(torch.empty((B, H, D, D), device=device), 300 + l, db.seq_lens, D)
    return dict(db=db, lt=lt, L=L, B=B, H=H, D=D, NB=NB, MB=MB, qkv=qkv, slots=slots, kv=kv, st=st)


def hybrid_bytes(wl):
    """Algorithmic bytes of one Full-layer decode launch (K and V of every cached token read
    once, q read, out written, the new K/V rows read and written into the cache) and of one
    whole 32-layer step (every Linear layer reads and writes its fp32 states and moves its
    q/k/v/out rows)."""
    B, H, D = wl["B"], wl["H"], wl["D"]
    tokens = int(wl["db"].seq_lens.sum())
    full = tokens * H * D * 2 * 2 + 2 * B * H * D * 2 + 4 * B * H * D * 2
    lin = B * H * D * D * 4 * 2 + 4 * B * H * D * 2
    n_full = sum(1 for t in wl["lt"] if t == 0)
    return full, lin, n_full * full + (wl["L"] - n_full) * lin


def cpu_baseline_hybrid(wl, budget_s=8.0, max_passes=20):
    """Times the CPU oracle (as it stands) on the whole 32-layer step: all 64 requests through
    every layer in order (Full: slot of position seq_len - 1, KV append, paged decode; Linear:
    state step). Every layer's pools are copied to the host once first (not timed); whole
    passes are repeated until ~budget_s of CPU work."""
    import oracle
    db, lt, B, L, D = wl["db"], wl["lt"], wl["B"], wl["L"], wl["D"]
    cores = oracle.set_threads(0)
    qkv = wl["qkv"]
    cu = np.arange(B + 1, dtype=np.int32)
    pos = (db.seq_lens - 1).astype(np.int32)
    host = {l: (tuple(_u16(x) for x in wl["kv"][l]) if t == 0 else wl["st"][l].cpu().numpy()) for l, t in enumerate(lt)}
    passes, t_used = 0, 0.0
    while passes < 1 or (t_used < budget_s and passes < max_passes):
        for l, t in enumerate(lt):
            t0 = time.perf_counter()
            if t == 0:
                kc, vc = host[l]
                slot = oracle.slot_mapping(db.pool.block_tables, cu, pos)
                oracle.kv_append(qkv[l, 1], qkv[l, 2], slot, kc, vc)
                oracle.full_decode(qkv[l, 0], kc, vc, db.pool.block_tables, db.seq_lens, D ** -0.5)
            else:
                oracle.linear_step(qkv[l, 0], qkv[l, 1], qkv[l, 2], host[l], wl["slots"])
            t_used += time.perf_counter() - t0
        passes += 1
    del host
    return {"value": round(passes * B * L / t_used, 2), "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"the whole step, {passes} pass(es): all {B} requests x {L} layers (24 Full: slot, KV "
                      f"append, paged decode; 8 Linear: state step), all heads; fp64 C oracle with OpenMP over "
                      f"(request, head); {t_used:.1f} s of CPU work (host copies of the pools made once, not timed)"}


# ------------------------------------------------------------------ single-layer decode batch
def build_single_layer(seed, device):
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


def cpu_baseline_decode(wl, budget_s=6.0):
    """Times the CPU oracle (as it stands) on the single-layer decode batch: whole passes over
    the 32 requests (slot of position seq_len - 1, KV append, paged decode; Linear step), all
    heads, repeated until ~budget_s of CPU work."""
    import oracle
    db, B, D = wl["db"], wl["B"], wl["D"]
    cores = oracle.set_threads(0)
    kc, vc = _u16(wl["kc"]), _u16(wl["vc"])
    st = wl["state"].cpu().numpy()
    hq = wl["host"]
    cu = np.arange(B + 1, dtype=np.int32)
    pos = (db.seq_lens - 1).astype(np.int32)
    passes, t_used = 0, 0.0
    while passes < 1 or t_used < budget_s:
        t0 = time.perf_counter()
        slot = oracle.slot_mapping(db.pool.block_tables, cu, pos)
        oracle.kv_append(hq["kf"], hq["vf"], slot, kc, vc)
        oracle.full_decode(hq["qf"], kc, vc, db.pool.block_tables, db.seq_lens, D ** -0.5)
        oracle.linear_step(hq["ql"], hq["kl"], hq["vl"], st, wl["slots_h"])
        t_used += time.perf_counter() - t0
        passes += 1
    return {"value": round(passes * B * 2 / t_used, 2), "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"the whole step, {passes} pass(es): all {B} requests x (Full: slot, KV append, paged "
                      f"decode; Linear step), all heads; fp64 C oracle with OpenMP over (request, head); "
                      f"{t_used:.1f} s"}


def row_single_layer(hyb, device, stream, iters, seed=0, cpu=True):
    """32 requests, seq_lens ~ U{128..4096}: one Full layer (paged decode with the KV append
    fused, plus the split combine) and one Linear layer (in-place state step). The per-op
    split comes from a second pass with an event between the two ops."""
    import torch
    hbm, _, _ = measured_peaks()
    wl = build_single_layer(seed, device)
    B, H, D, NB, MB, db = wl["B"], wl["H"], wl["D"], wl["NB"], wl["MB"], wl["db"]
    d = hyb.dims(H, D, NB, MB, W.BF16)
    x = {n: _dev_bf16(a, device) for n, a in wl["host"].items()}
    bt = torch.from_numpy(db.pool.block_tables).to(device)
    lens = torch.from_numpy(db.seq_lens).to(device)
    slots = torch.from_numpy(wl["slots_h"]).to(device)
    msl = int(db.seq_lens.max())
    ws_n = hyb.hyb_paged_attn_decode_workspace_size(B, msl, d)
    ws = torch.empty(max(ws_n, 16), dtype=torch.uint8, device=device)
    out_f, out_l = (torch.empty((B, H, D), dtype=torch.bfloat16, device=device) for _ in range(2))
    sh = stream.cuda_stream
    dec = lambda: hyb.check(hyb.hyb_paged_attn_decode_append(out_f, x["qf"], x["kf"], x["vf"], None, wl["kc"],
                                                             wl["vc"], bt, lens, B, msl, d, ws, ws_n, sh))
    lin = lambda: hyb.check(hyb.hyb_linear_attn_step(out_l, x["ql"], x["kl"], x["vl"], wl["state"], B, slots,
                                                     B, H, D, W.BF16, sh))
    t_step = _time(lambda: (dec(), lin()), stream, iters)
    # per-op split: an event between the ops (it holds back the programmatic early launch of
    # the next kernel, so this pass runs a little slower than the step above)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(iters)]
    with torch.cuda.stream(stream):
        for e in evs:
            e[0].record(stream)
            dec()
            e[1].record(stream)
            lin()
            e[2].record(stream)
    stream.synchronize()
    _check_device(hyb)
    t_dec = float(np.mean([e[0].elapsed_time(e[1]) for e in evs]))
    t_lin = float(np.mean([e[1].elapsed_time(e[2]) for e in evs]))
    tokens = int(db.seq_lens.sum())
    dec_bytes = tokens * H * D * 2 * 2 + 2 * B * H * D * 2 + 4 * B * H * D * 2
    lin_bytes = B * H * D * D * 4 * 2
    res = {"workload": "decode_single_layer: 32 requests, H=32, D=128, block 16, seq_lens U{128..4096}, "
                       "1 Full paged-decode (KV append fused) + 1 Linear step",
           "value": round(B * 2 / (t_step * 1e-3), 1), "unit": UNIT, "ms_per_step": round(t_step, 5),
           "kv_tokens": tokens,
           "ms": {"paged_decode": round(t_dec, 5), "linear_step": round(t_lin, 5)},
           "roofline": _roof("hbm", dec_bytes / (t_dec * 1e-3) / 1e9, hbm, "GB/s",
                             "paged_decode with the KV append fused (split-K + combine)", dec_bytes,
                             traffic=_traffic("paged_decode", "decode.cu")),
           "linear_step": _roof("hbm", lin_bytes / (t_lin * 1e-3) / 1e9, hbm, "GB/s",
                                "linear_step (in the step: the decode before it evicts L2)", lin_bytes,
                                traffic=_traffic("linear_step", "linear.cu")),
           "l2": "no flush: per-step working set %.2f GB > 129 MB L2" % ((dec_bytes + lin_bytes) / 1e9)}
    if cpu:
        res["cpu_baseline"] = cpu_baseline_decode(wl)
    del wl, x
    torch.cuda.empty_cache()
    return res


def cpu_baseline_long(db, kc, vc, q_h, st, H, D, budget_s=6.0, max_passes=10):
    """Times the CPU oracle (as it stands) on the whole 131K-context step: each of the 8
    requests through the paged decode over its 8192 blocks and the Linear step. Each
    request's blocks are gathered on the device and copied to the host once first (not
    timed), in logical order; whole passes repeat until ~budget_s of CPU work."""
    import torch
    import oracle
    cores = oracle.set_threads(0)
    B = db.B
    st_h = st.cpu().numpy()
    kv = []
    for b in range(B):
        nb = int(db.pool.blocks_per_req[b])
        idx = torch.from_numpy(db.pool.block_tables[b, :nb].astype(np.int64)).to(kc.device)
        kv.append((_u16(kc.index_select(0, idx)), _u16(vc.index_select(0, idx)), np.arange(nb, dtype=np.int32)[None, :]))
    passes, t_used = 0, 0.0
    while passes < 1 or (t_used < budget_s and passes < max_passes):
        for b in range(B):
            kb, vb, tbl = kv[b]
            t0 = time.perf_counter()
            oracle.full_decode(q_h[b:b + 1], kb, vb, tbl, db.seq_lens[b:b + 1], D ** -0.5)
            oracle.linear_step(q_h[b:b + 1], q_h[b:b + 1], q_h[b:b + 1], st_h, np.array([b], np.int32))
            t_used += time.perf_counter() - t0
        passes += 1
    del kv
    return {"value": round(passes * B * 2 / t_used, 3), "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"the whole step, {passes} pass(es): all {B} requests x (paged decode over 131072 tokens, "
                      f"Linear step), all {H} heads; fp64 C oracle with OpenMP over (request, head); {t_used:.1f} s "
                      f"(each request's blocks gathered to the host once first, not timed)"}


def row_long_context(hyb, device, stream, iters, seed=0, cpu=True):
    """8 requests x 131072 tokens: split-K paged decode over 8192 random blocks each, and the
    Linear step on 8 x 32 x 128 x 128 fp32 states. The Linear step's states (16.8 MB per
    batch) would stay in L2 across back-to-back calls, so it rotates over 16 state pools
    (268 MB, twice the L2)."""
    import torch
    hbm, _, _ = measured_peaks()
    db = W.decode_long_context(seed)
    B, H, D, NB = db.B, db.H, db.D, db.pool.num_blocks
    d = hyb.dims(H, D, NB, db.pool.max_blocks, W.BF16)
    kc = W.device_rows_(torch.empty((NB, H, 16, D), dtype=torch.bfloat16, device=device), 51, D)
    vc = W.device_rows_(torch.empty_like(kc), 52, D)
    NR = 16
    sts = [W.device_state_(torch.empty((B, H, D, D), device=device), 53 + i, db.seq_lens, D) for i in range(NR)]
    g = W.rng(seed + 5)
    q_h = W.rows(g, (B, H, D), D, W.BF16)
    q = _dev_bf16(q_h, device)
    out = torch.empty_like(q)
    bt = torch.from_numpy(db.pool.block_tables).to(device)
    lens = torch.from_numpy(db.seq_lens).to(device)
    slots = torch.arange(B, dtype=torch.int32, device=device)
    n = int(db.seq_lens.max())
    ws_n = hyb.hyb_paged_attn_decode_workspace_size(B, n, d)
    ws = torch.empty(ws_n, dtype=torch.uint8, device=device)
    sh = stream.cuda_stream
    t_dec = _time(lambda: hyb.check(hyb.hyb_paged_attn_decode(out, q, kc, vc, bt, lens, B, n, d, ws, ws_n, sh)),
                  stream, iters)
    it = [0]

    def lin():
        it[0] += 1
        hyb.check(hyb.hyb_linear_attn_step(out, q, q, q, sts[it[0] % NR], B, slots, B, H, D, W.BF16, sh))
    t_lin = _time(lin, stream, max(iters, 4 * NR))
    _check_device(hyb)
    dec_bytes = int(db.seq_lens.sum()) * H * D * 4 + 2 * B * H * D * 2
    lin_bytes = B * H * D * D * 8
    res = {"workload": "long_context_decode: 8 requests x 131072 tokens, H=32, D=128, 8192 random blocks each",
           "value": round(B * 2 / ((t_dec + t_lin) * 1e-3), 1), "unit": UNIT,
           "ms": {"paged_decode": round(t_dec, 4), "linear_step": round(t_lin, 4)},
           "roofline": _roof("hbm", dec_bytes / (t_dec * 1e-3) / 1e9, hbm, "GB/s", "paged_decode (split-K + combine)",
                             dec_bytes),
           "linear_step": _roof("hbm", lin_bytes / (t_lin * 1e-3) / 1e9, hbm, "GB/s",
                                f"linear_step, rotating over {NR} state pools ({NR * lin_bytes // 2 / 1e6:.0f} MB)",
                                lin_bytes)}
    if cpu:
        res["cpu_baseline"] = cpu_baseline_long(db, kc, vc, q_h, sts[0], H, D)
    del kc, vc, sts
    torch.cuda.empty_cache()
    return res


def cpu_baseline_prefill(pb, k0, v0, q0, ql0, kl0, vl0, H, D, every=4):
    """Times the CPU oracle (as it stands) on a labelled subset of the chunked-prefill workload
    and extrapolates by work: request 0's slot mapping and KV append (all 8192 rows) and its
    causal prefill on every `every`-th query row (a uniform sample of the causal triangle);
    request 0's Linear prefill as the token recurrence over all 8192 tokens (all heads). The
    full workload is 8 such requests and all query rows."""
    import oracle
    cores = oracle.set_threads(0)
    n = int(pb.q_lens[0])
    nb = (n + 15) // 16
    g = W.rng(77)
    tbl = g.permutation(nb).astype(np.int32)[None, :]
    kc = np.zeros((nb, H, 16, D), np.uint16)
    vc = np.zeros_like(kc)
    cu = np.array([0, n], np.int32)
    rows = np.arange(every - 1, n, every, dtype=np.int32)
    t0 = time.perf_counter()
    slot = oracle.slot_mapping(tbl, cu)
    oracle.kv_append(k0, v0, slot, kc, vc)
    t_app = time.perf_counter() - t0
    t0 = time.perf_counter()
    oracle.full_prefill(q0, kc, vc, tbl, cu, None, D ** -0.5, rows=rows)
    t_rows = time.perf_counter() - t0
    t0 = time.perf_counter()
    oracle.linear_recurrence(ql0, kl0, vl0, cu)
    t_lin = time.perf_counter() - t0
    Bn = len(pb.q_lens)
    keys_all = float(sum(m * (m + 1) / 2 for m in pb.q_lens.astype(np.float64)))
    keys_rows = float((rows + 1).astype(np.float64).sum())
    est = Bn * t_app + t_rows * keys_all / keys_rows + Bn * t_lin
    T = int(pb.q_lens.sum())
    return {"value": round(T * 2 / est, 2), "unit": "prompt tokens/s per layer", "cores": cores, "kind": "oracle",
            "extrapolated": True,
            "sample": f"request 0 of {Bn}: slot mapping + KV append of its {n} rows ({t_app:.2f} s), causal prefill "
                      f"of every {every}th query row ({len(rows)} rows, {t_rows:.1f} s), token recurrence over its "
                      f"{n} tokens ({t_lin:.1f} s), all {H} heads; extrapolated by work to {Bn} requests and every "
                      f"row ({est:.0f} s estimated); fp64 C oracle with OpenMP over (request, head)"}


def row_prefill(hyb, device, stream, iters, seed=0, cpu=True):
    """8 requests x 8192-token prompts, H=32, D=128: Full layer = slot mapping + KV append +
    tensor-core causal prefill over the paged cache; Linear layer = tensor-core chunked
    prefill (interface chunk 64; the kernel computes 128-token chunks, which the chunk form
    allows since it equals the recurrence for any cut) from a zero state."""
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
    t_pf = _time(lambda: hyb.check(hyb.hyb_paged_attn_prefill_causal(out, q, kc, vc, bt, cu, None, B, T, L, d, sh)),
                 stream, iters)
    lws = torch.empty(hyb.hyb_linear_attn_chunked_prefill_workspace_size(), dtype=torch.uint8, device=device)
    t_lin = _time(lambda: hyb.check(hyb.hyb_linear_attn_chunked_prefill(lo, ql, kl, vl, cu, None, st, B, slots, reset,
                                                                        B, T, L, H, D, pb.chunk, W.BF16, lws,
                                                                        lws.numel(), sh)),
                  stream, iters)
    _check_device(hyb)
    n = pb.q_lens.astype(np.float64)
    pf_flops = 4.0 * H * D * float((n * (n + 1) / 2).sum())              # QK^T + PV over the causal triangle
    lin_flops = T * H * (4.0 * pb.chunk * D + 4.0 * D * D)                # per token-head: 4CD + 4D^2 at C = 64
    lin_bytes = 4 * T * H * D * 2 + B * H * D * D * 4                     # q,k,v read, o written, state written
    app_bytes = 2 * 2 * T * H * D * 2
    ai = lin_flops / lin_bytes
    lin_gbs = lin_bytes / (t_lin * 1e-3) / 1e9
    lin_tf = lin_flops / (t_lin * 1e-3) / 1e12
    res = {"workload": "prefill_chunked: 8 requests x 8192-token prompts, H=32, D=128, interface chunk 64 "
                       "(computed as 128-token chunks)",
           "value": round(T * 2 / ((t_slot + t_app + t_pf + t_lin) * 1e-3), 1), "unit": "prompt tokens/s per layer",
           "ms": {"slot_mapping": round(t_slot, 4), "kv_append": round(t_app, 4), "prefill_causal": round(t_pf, 4),
                  "linear_chunked_prefill": round(t_lin, 4)},
           "roofline": _roof("tensor", pf_flops / (t_pf * 1e-3) / 1e12, tf, "TFLOP/s", "prefill_tc_kernel (causal, paged)",
                             pf_flops, traffic=_traffic("prefill_tc", "prefill_tc.cu"),
                             peak_source="measured bf16_tflops (burst)"),
           "linear_chunked_prefill": _roof("hbm", lin_gbs, hbm, "GB/s", "linear_prefill_tc_kernel (128-token chunks)",
                                           lin_bytes, traffic=_traffic("linear_prefill_tc", "linear_tc.cu"),
                                           tflops=round(lin_tf, 1), tensor_frac=round(lin_tf / tf, 4),
                                           arithmetic_intensity=round(ai, 1),
                                           frac_of_min_peak_ai_bw=round(lin_tf / min(tf, ai * hbm / 1e3), 4)),
           "kv_append": _roof("hbm", app_bytes / (t_app * 1e-3) / 1e9, hbm, "GB/s", "kv_append_kernel", app_bytes,
                              traffic=_traffic("kv_append", "append.cu"))}
    if cpu:
        n0 = int(pb.q_lens[0])
        res["cpu_baseline"] = cpu_baseline_prefill(pb, _u16(k[:n0]), _u16(v[:n0]), _u16(q[:n0]), _u16(ql[:n0]),
                                                   _u16(kl[:n0]), _u16(vl[:n0]), H, D)
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


def row_prefill_prefix(hyb, device, stream, iters, seed=0):
    """Chunked prefill over a cached prefix: the last 2048-token chunk of 8 x 8192-token
    prompts, H=32, D=128. Full layer = slot mapping + KV append of the chunk + tensor-core
    causal prefill over the 6144 cached tokens and the chunk; Linear layer = tensor-core
    chunked prefill (interface chunk 64) continuing each chain from its carried state."""
    import torch
    hbm, tf, _ = measured_peaks()
    B, H, D, P, C = 8, 32, 128, 6144, 2048
    g = W.rng(seed + 21)
    pool = W.block_pool(g, np.full(B, P + C, np.int32))
    NB = pool.num_blocks
    d = hyb.dims(H, D, NB, pool.max_blocks, W.BF16)
    q_lens = np.full(B, C, np.int32)
    ctx_h = np.full(B, P, np.int32)
    cu_h = W.cu_from_lens(q_lens)
    T = int(cu_h[-1])
    mk = lambda s_: W.device_rows_(torch.empty((T, H, D), dtype=torch.bfloat16, device=device), s_, D)
    q, k, v, ql, kl, vl = (mk(70 + i) for i in range(6))
    out, lo = torch.empty_like(q), torch.empty_like(q)
    # the pool holds the cached prefix (random rows); the append writes the chunk behind it
    kc = W.device_rows_(torch.empty((NB, H, 16, D), dtype=torch.bfloat16, device=device), 76, D)
    vc = W.device_rows_(torch.empty_like(kc), 77, D)
    st = W.device_state_(torch.empty((B, H, D, D), device=device), 78, ctx_h, D)
    bt = torch.from_numpy(pool.block_tables).to(device)
    cu = torch.from_numpy(cu_h).to(device)
    ctx = torch.from_numpy(ctx_h).to(device)
    slots = torch.arange(B, dtype=torch.int32, device=device)
    reset = torch.zeros(B, dtype=torch.uint8, device=device)
    slot = torch.empty(T, dtype=torch.int64, device=device)
    lws = torch.empty(hyb.hyb_linear_attn_chunked_prefill_workspace_size(), dtype=torch.uint8, device=device)
    sh = stream.cuda_stream
    t_slot = _time(lambda: hyb.check(hyb.hyb_slot_mapping(slot, bt, cu, ctx, B, T, d, sh)), stream, iters)
    t_app = _time(lambda: hyb.check(hyb.hyb_paged_kv_append(k, v, slot, T, kc, vc, d, sh)), stream, iters)
    t_pf = _time(lambda: hyb.check(hyb.hyb_paged_attn_prefill_causal(out, q, kc, vc, bt, cu, ctx, B, T, C, d, sh)),
                 stream, iters)
    t_lin = _time(lambda: hyb.check(hyb.hyb_linear_attn_chunked_prefill(lo, ql, kl, vl, cu, ctx, st, B, slots, reset,
                                                                        B, T, C, H, D, 64, W.BF16, lws,
                                                                        lws.numel(), sh)),
                  stream, iters)
    _check_device(hyb)
    i = np.arange(1, C + 1, dtype=np.float64)
    pf_flops = 4.0 * H * D * B * float((P + i).sum())                    # each new row sees P + i keys
    lin_flops = T * H * (4.0 * 64 * D + 4.0 * D * D)
    lin_bytes = 4 * T * H * D * 2 + 2 * B * H * D * D * 4                # q,k,v read, o written; state read + written
    lin_gbs = lin_bytes / (t_lin * 1e-3) / 1e9
    res = {"workload": "prefill_prefix: 8 requests, 2048-token chunk over a 6144-token cached prefix, H=32, D=128, "
                       "interface chunk 64 (computed as 128-token chunks), Linear state carried",
           "value": round(T * 2 / ((t_slot + t_app + t_pf + t_lin) * 1e-3), 1), "unit": "prompt tokens/s per layer",
           "ms": {"slot_mapping": round(t_slot, 4), "kv_append": round(t_app, 4), "prefill_causal": round(t_pf, 4),
                  "linear_chunked_prefill": round(t_lin, 4)},
           "roofline": _roof("tensor", pf_flops / (t_pf * 1e-3) / 1e12, tf, "TFLOP/s",
                             "prefill_tc_kernel (causal over a cached prefix, paged)", pf_flops,
                             peak_source="measured bf16_tflops (burst)"),
           "linear_chunked_prefill": _roof("hbm", lin_gbs, hbm, "GB/s",
                                           "linear_prefill_tc_kernel (128-token chunks, state carried)", lin_bytes)}
    del q, k, v, ql, kl, vl, out, lo, kc, vc, st
    torch.cuda.empty_cache()
    return res


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
    # one pool per state type is 67 MB (fp32) or 34 MB (16-bit): back-to-back calls would be
    # served from the 129 MB L2, so each type rotates over pools totalling 268 MB
    st32 = [W.device_state_(torch.empty((B, H, D, D), device=device), 81 + i, np.full(B, 2048), D) for i in range(4)]
    st16 = {sd: [st32[i % 4].to(torch.bfloat16 if sd == W.BF16 else torch.float16) for i in range(8)]
            for sd in (W.BF16, hyb.HYB_F16)}
    sh = stream.cuda_stream
    it = [0]

    def step32():
        it[0] += 1
        hyb.check(hyb.hyb_linear_attn_step(out, q, k, v, st32[it[0] % 4], B, slots, B, H, D, W.BF16, sh))

    def step16(sd):
        it[0] += 1
        hyb.check(hyb.hyb_linear_attn_step_lowp(out, q, k, v, st16[sd][it[0] % 8], sd, B, slots, B, H, D, W.BF16, sh))
    n_it = max(iters, 32)
    t = {"fp32": _time(step32, stream, n_it)}
    for sd, name in ((W.BF16, "bf16"), (hyb.HYB_F16, "fp16")):
        t[name] = _time(lambda: step16(sd), stream, n_it)
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
            "roofline": {n: _roof("hbm", byt[n] / (t[n] * 1e-3) / 1e9, hbm, "GB/s",
                                  f"linear step, {n} state, rotating over pools totalling 268 MB", byt[n])
                         for n in t},
            "drift_vs_fp32_state": {"metric": "max |o - o_fp32| / max |o_fp32| over the 64 steps before t",
                                    "steps": T, **drift}}


ROWS = {"decode_single_layer": row_single_layer, "long_context_decode": row_long_context,
        "prefill_chunked": row_prefill, "prefill_prefix": row_prefill_prefix, "sliding_window": row_sliding_window,
        "state_precision": row_state_precision, "block32": row_block32, "bucketing": row_bucketing}
EXTRA_ROWS = {"prefill_lengths": row_prefill_lengths}   # --workload only, not in the default rows
CPU_ROWS = ("decode_single_layer", "long_context_decode", "prefill_chunked")   # rows timed beside the oracle


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
    if args.workload != "hybrid_32layer":               # one other workload, timed alone
        stream = torch.cuda.Stream(device=device)
        fn = {**ROWS, **EXTRA_ROWS}[args.workload]
        kw = {"cpu": False} if args.workload in CPU_ROWS else {}
        r = fn(hyb, device, stream, max(args.steps, 1), args.seed + dist.rank, **kw)
        r.update({"metric": METRIC, "n_gpus": dist.world, "steps": args.steps, "warmup": 3,
                  "higher_is_better": True, "dtype": "bf16", "data": "synthetic"})
        return r
    wl = build_hybrid(args.seed + dist.rank, device)
    db, lt, L, B, H, D, NB, MB = (wl[n] for n in ("db", "lt", "L", "B", "H", "D", "NB", "MB"))
    d = hyb.dims(H, D, NB, MB, W.BF16)
    qkv = _dev_bf16(wl["qkv"], device)                  # [L][3][B][H][D]
    out = torch.empty((L, B, H, D), dtype=torch.bfloat16, device=device)
    bt = torch.from_numpy(db.pool.block_tables).to(device)
    lens = torch.from_numpy(db.seq_lens).to(device)
    slots = torch.from_numpy(wl["slots"]).to(device)
    msl = int(db.seq_lens.max())
    ws_n = hyb.hyb_paged_attn_decode_workspace_size(B, msl, d)
    ws = torch.empty(max(ws_n, 16), dtype=torch.uint8, device=device)
    stream = torch.cuda.Stream(device=device)
    sh = stream.cuda_stream

    def layer_ios(qkv_t, out_t):
        return [hyb.layer_io(out_t[l], qkv_t[l, 0], qkv_t[l, 1], qkv_t[l, 2], *wl["kv"][l]) if t == 0 else
                hyb.layer_io(out_t[l], qkv_t[l, 0], qkv_t[l, 1], qkv_t[l, 2], state_pool=wl["st"][l],
                             num_state_slots=B)
                for l, t in enumerate(lt)]
    ios = layer_ios(qkv, out)
    # no slot mapping: each Full layer appends its new rows at seq_len - 1 through the block table
    meta = hyb.batch_meta(B, B, seq_lens=lens, block_tables=bt, state_slots=slots, max_seq_len=msl)

    def step():
        hyb.check(hyb.hyb_layer_dispatch(lt, L, 0, ios, meta, d, 64, ws, ws_n, sh))

    # runs of consecutive layers of one type: [full x3], [linear], ... (8 periods)
    runs = []
    for l, t in enumerate(lt):
        if runs and runs[-1][0] == t:
            runs[-1][2] += 1
        else:
            runs.append([t, l, 1])

    def step_by_runs(ev):
        """The launches of step(), one dispatch call per run of same-type layers, with an event
        between runs: inside a run the kernels keep their early (programmatic) launch."""
        ev[0].record(stream)
        for k, (t, l0, n) in enumerate(runs):
            hyb.check(hyb.hyb_layer_dispatch(lt[l0:l0 + n], n, 0, ios[l0:l0 + n], meta, d, 64, ws, ws_n, sh))
            ev[k + 1].record(stream)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
    torch.cuda.synchronize()
    # An event between two kernels holds back the early (programmatic dependent) launch of the
    # second, so events slow the step they time. One event pair brackets all K steps for the
    # step time; every INSTR-th step runs as one dispatch call per run of same-type layers
    # with an event between runs, for the per-layer split and the decode kernel's roofline.
    INSTR = 10
    evs = {s: [torch.cuda.Event(enable_timing=True) for _ in range(len(runs) + 1)]
           for s in range(0, args.steps, INSTR)}
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
            if s in evs:
                step_by_runs(evs[s])
            else:
                step()
        loop_ev[1].record(stream)
    torch.cuda.synchronize()
    clocks.mark("t1")
    launches = hyb.hyb_launch_count(reset=True)
    dist.barrier()
    clocks.stop()
    ms_step = dist.max(loop_ev[0].elapsed_time(loop_ev[1]) / args.steps)
    units = dist.sum(B * L)                              # request-tokens per layer-step over all ranks
    value = units / (ms_step * 1e-3)
    run_ms = np.array([[e[k].elapsed_time(e[k + 1]) for k in range(len(runs))] for e in evs.values()])
    _check_device(hyb)
    n_full = sum(n for t, _, n in runs if t == 0)
    full_runs = np.array([t == 0 for t, _, _ in runs])
    full_ms = float(run_ms[:, full_runs].sum(1).mean()) / n_full          # per Full layer
    lin_ms = float(run_ms[:, ~full_runs].sum(1).mean()) / (L - n_full)    # per Linear layer
    step_inst_ms = float(run_ms.sum(1).mean())

    # ---- roofline of the dominant kernel: a Full layer's paged decode (KV append fused,
    # split-K kernel + combine), averaged over the 24 Full layers of the instrumented steps
    hbm_peak, _, peak_kind = measured_peaks()
    full_bytes, lin_bytes, step_bytes = hybrid_bytes(wl)
    achieved = full_bytes / (full_ms * 1e-3) / 1e9
    trec = traffic_record("paged_decode_hybrid", "decode.cu")
    roofline = {"kernel": "paged_decode with the KV append fused (split-K + combine), one Full layer of the step",
                "bound": "hbm", "achieved": round(achieved, 1), "peak": hbm_peak, "unit": "GB/s",
                "frac": round(achieved / hbm_peak, 4),
                "traffic": (int(trec["bytes_per_launch"]) if trec else None),
                "algorithmic_bytes": full_bytes, "launches_averaged": n_full * len(evs),
                "timing": (f"CUDA events around each run of 3 Full layers in the {len(evs)} instrumented steps "
                           f"(every {INSTR}th of the timed loop); time of the runs / layers"),
                "peak_source": f"{peak_kind} hbm_gbs"}
    ops = {"full_layer": {"ms": round(full_ms, 5), "GB/s": round(achieved, 1), "layers": n_full,
                          "share_of_step": round(n_full * full_ms / step_inst_ms, 4)},
           "linear_layer": {"ms": round(lin_ms, 5), "GB/s": round(lin_bytes / (lin_ms * 1e-3) / 1e9, 1),
                            "frac": round(lin_bytes / (lin_ms * 1e-3) / 1e9 / hbm_peak, 4), "layers": L - n_full,
                            "traffic": _traffic("linear_step_hybrid", "linear.cu"),
                            "share_of_step": round((L - n_full) * lin_ms / step_inst_ms, 4)},
           "instrumented_step_ms": round(step_inst_ms, 5),
           "note": (f"from the {len(evs)} instrumented steps (every {INSTR}th), one dispatch call per run of "
                    "same-type layers with events between runs; the early launch is lost only at run edges")}
    step_roof = _roof("hbm", step_bytes / (ms_step * 1e-3) / 1e9, hbm_peak, "GB/s", "whole 32-layer step (dispatch)",
                      step_bytes)

    # ---- step-time distribution: a separate pass, one event pair per step
    NP = 200
    pev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(NP)]
    with torch.cuda.stream(stream):
        for a, b in pev:
            a.record(stream)
            step()
            b.record(stream)
    torch.cuda.synchronize()
    per_step = np.array([a.elapsed_time(b) for a, b in pev])

    # ---- the same step captured once into a CUDA graph and replayed
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        step()
        stream.synchronize()
        with torch.cuda.graph(graph, stream=stream):
            step()
    t_graph = _time(graph.replay, stream, 100)
    del graph

    # ---- end to end through the public dispatcher, host buffers, copies timed. All of a
    # step's inputs (32 layers' q/k/v and the batch metadata) sit in one pinned host buffer and
    # go over in one copy; all 32 layers' outputs come back in one copy.
    host_arrays = {"qkv": wl["qkv"], "lens": db.seq_lens, "bt": db.pool.block_tables, "slots": wl["slots"]}
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

        out_all = torch.empty((L, B, H, D), dtype=torch.bfloat16, device=device)
        e_meta = hyb.batch_meta(B, B, seq_lens=dview("lens"), block_tables=dview("bt"), state_slots=dview("slots"),
                                max_seq_len=msl)
        sets.append(dict(d_all=d_all, out_all=out_all, meta=e_meta, ios=layer_ios(dview("qkv"), out_all),
                         h_out=torch.empty(out_all.numel(), dtype=torch.int16).pin_memory(),
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
        hyb.check(hyb.hyb_layer_dispatch(lt, L, 0, st["ios"], st["meta"], d, 64, ws, ws_n, sh))
        st["computed"].record(stream)
        d2h_stream.wait_event(st["computed"])
        with torch.cuda.stream(d2h_stream):
            st["h_out"].copy_(st["out_all"].view(-1).view(torch.int16), non_blocking=True)
            st["read"].record(d2h_stream)

    e2e_steps = max(10, min(args.steps, 200))
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
    _check_device(hyb)
    # The Full layers' outputs are the same every step (same inputs; the append rewrites the
    # same slots): the last end-to-end step's host copy must equal the device-timed step's.
    last = sets[(e2e_steps - 1) % 2]["h_out"].view(L, B, H, D)
    dev_out = out.view(torch.int16).cpu()
    full_idx = [l for l, t in enumerate(lt) if t == 0]
    e2e_match = bool(torch.equal(last[full_idx], dev_out[full_idx]))
    del sets

    # ---- CPU oracle beside it (rank 0, N = 1 only)
    cpu = cpu_baseline_hybrid(wl) if dist.world == 1 else None

    # ---- the other workloads, each against its own roofline (N = 1 only)
    rows = None
    if dist.world == 1 and not args.no_rows:
        tokens = int(db.seq_lens.sum())
        del wl, qkv, out, ios
        torch.cuda.empty_cache()
        rows = {name: fn(hyb, device, stream, 20, args.seed) for name, fn in ROWS.items()}
    else:
        tokens = int(db.seq_lens.sum())

    res = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": dist.world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 5),
        "ms_per_step_p50": round(float(np.percentile(per_step, 50)), 5),
        "ms_per_step_p99": round(float(np.percentile(per_step, 99)), 5),
        "timing": (f"ms_per_step: one CUDA event pair around all {args.steps} steps; p50/p99: a separate pass "
                   f"of {NP} steps with one event pair each"),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1)/sqrt(D) q/k/v, shuffled block pool, N(0,seq/D^2) states)",
        "config": {"workload": "hybrid_32layer: 32 layers [full,full,full,linear] x 8, batch 64 (80% ~lognormal(128), "
                               "20% ~lognormal(2048) cached tokens), H=32, D=128, block 16, one decode token per "
                               "request through all layers",
                   "B": B, "H": H, "D": D, "layers": "[full,full,full,linear] x 8", "kv_tokens": tokens,
                   "pool_blocks": NB,
                   "l2": "no flush: per-step working set %.2f GB > 129 MB L2" % (step_bytes / 1e9),
                   "parallelism": f"replicas x{dist.world}"},
        "roofline": roofline, "step_roofline": step_roof, "ops": ops,
        "cuda_graph": {"value": round(units / (t_graph * 1e-3), 1), "ms_per_step": round(t_graph, 5),
                       "note": "the same step captured once and replayed (no per-launch host work)"},
        "e2e": {"value": round(e2e_val, 1), "unit": UNIT, "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h),
                "path": "hyb_layer_dispatch over all 32 layers; inputs in one pinned buffer, one copy each way, "
                        "on copy streams double-buffered against the compute stream",
                "full_layer_outputs_equal_device_step": e2e_match},
        "gpu_launches": int(launches),
        "clocks": clocks.summary(),
        "cpu_baseline": cpu,
        "rows": rows,
    }
    return res


def bench_reference(args, dist):
    """The CPU oracle as the reference arm, on the headline workload: each step is the batch's
    requests through one period [full, full, full, linear] of the 32-layer pattern (rotating
    over the requests when the run is long), on the host cores."""
    if dist.rank != 0:
        return None
    import oracle
    oracle.build()
    db = W.decode_hybrid_32layer(args.seed)
    g = W.rng(args.seed + 9)
    B, H, D = db.B, db.H, db.D
    cores = oracle.set_threads(0)
    period = [0, 0, 0, 1]
    P = len(period)
    # One K and one V pool image (0.36 GB each, larger than the host caches) shared by the
    # period's Full layers; each layer has its own q/k/v rows.
    import torch
    kc, vc = (W.device_rows_(torch.empty((db.pool.num_blocks, H, 16, D), dtype=torch.bfloat16), 100 + i, D)
              .view(torch.int16).numpy().view(np.uint16) for i in range(2))     # host tensors, seeded
    qkv = W.rows(g, (P, 3, B, H, D), D, W.BF16)
    st = W.synthetic_state(g, B, H, D, db.seq_lens)
    slots = g.permutation(B).astype(np.int32)
    # requests per step: the whole batch unless the run is long (keeps it to a few minutes)
    R = max(1, min(B, (B * 100) // max(args.steps + args.warmup, 1)))

    def one(i):
        r = np.arange(i * R, i * R + R) % B
        bt, ln = db.pool.block_tables[r], db.seq_lens[r]
        cu = np.arange(R + 1, dtype=np.int32)
        for l, t in enumerate(period):
            q, k, v = qkv[l, 0][r], qkv[l, 1][r], qkv[l, 2][r]
            if t == 0:
                slot = oracle.slot_mapping(bt, cu, (ln - 1).astype(np.int32))
                oracle.kv_append(k, v, slot, kc, vc)
                oracle.full_decode(q, kc, vc, bt, ln, D ** -0.5)
            else:
                oracle.linear_step(q, k, v, st, slots[r])

    for i in range(args.warmup):
        one(i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        one(i)
    dt = time.perf_counter() - t0
    ms = dt * 1e3 / args.steps
    val = R * P / (ms * 1e-3)
    sample = (f"{R} of the {B} requests per step (rotating) through one period [full, full, full, linear] of the "
              f"32-layer pattern (Full: slot, KV append, paged decode; Linear: state step), all {H} heads; the "
              f"period's Full layers share one 0.36 GB K and V pool image")
    return {"impl": "reference", "metric": METRIC, "value": round(val, 2), "unit": UNIT, "n_gpus": dist.world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "hybrid_32layer: 32 layers [full,full,full,linear] x 8, batch 64 (80% "
                                   "~lognormal(128), 20% ~lognormal(2048) cached tokens), H=32, D=128, block 16, "
                                   "one decode token per request through all layers",
                       "sample_per_step": sample},
            "cpu_baseline": {"value": round(val, 2), "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
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

