#!/usr/bin/env python3
"""Benchmark of the hybrid compressed/sparse attention hot path on one B300.

A step is one decode step of one CSA attention layer over a batch of 4
sequences at 1,048,576 cached tokens (V4-Pro shape: 128 query heads, head dim
128, m = 4 -> 262,144 compressed entries, int8 indexer dim 64, top-k 1024,
128-token window):
  1. hsa_compress   -- fold the block completed by the new token into its entry
  2. hsa_index_topk -- int8 scores of all 262,144 entries, exact top-1024
  3. hsa_attn_decode -- split-KV attention over the 1024 entries + 128 raw tokens,
                        log-sum-exp merge of the splits.
Inputs are seeded synthetic tensors; the timed steps rotate over R replicas of
the per-step inputs whose indexer keys alone exceed 4x the L2 cache, so every
step reads them from HBM.  One CUDA graph holds a block of steps; the timed
region is exactly K steps.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl {hsa,reference}]
Prints one JSON line on rank 0.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import platform
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from compressed_attention_compress_b300.inputs import WORKLOADS, block_weights  # noqa: E402

WL = WORKLOADS["pro_csa_decode"]

# DRAM bytes (read + write) of one index_fused_kernel launch on this workload, from the
# ncu capture summarised in profiles/index_fused_kernel_pro_csa_1M_B4.md; reported only
# while the kernel's sources are the ones that capture ran.
INDEX_TRAFFIC = {
    "bytes": 67258368 + 110336,
    "sources": {
        "compressed_attention_compress_b300/csrc/index_fused.cu":
            "fd9e0083f6ed2eebb211bcb3ff11a3142598ba316ffa91176b925dcc9d2cf824",
        "compressed_attention_compress_b300/csrc/common.cuh":
            "1c50e4616466d69022320548d2a47c9c9d2aef65c6b5dca650519a168e3275b2",
        "compressed_attention_compress_b300/csrc/block_scan.cuh":
            "ac0c74255584e15eaea3aa69860c5b08cd4267e432e4e9db82d6c3de8245161a",
    },
}


def index_traffic():
    import hashlib
    for rel, want in INDEX_TRAFFIC["sources"].items():
        with open(os.path.join(ROOT, rel), "rb") as f:
            if hashlib.sha256(f.read()).hexdigest() != want:
                return None
    return INDEX_TRAFFIC["bytes"]
METRIC = "decode queries/s at 1M ctx (V4-Pro-shaped CSA layer, B=4)"
UNIT = "queries/s"


# ----------------------------------------------------------------- helpers

def algorithmic_bytes(wl, cnt_total: int):
    """Bytes the method must move in one decode step (raw cache outside the window not counted)."""
    B, E, DI, d = wl.B, wl.N // wl.m, wl.DI, wl.d
    idx_bytes = B * E * DI + B * DI + 2 * B * wl.topk * 4 + 2 * B * 4      # keys, queries, idx/cnt write+read
    gather = cnt_total * 2 * d * 2                                          # selected K and V entries
    window = B * min(wl.window, wl.N) * 2 * d * 2
    qo = 2 * B * wl.H * d * 2
    compress = B * wl.m * 2 * d * 2 + B * 2 * d * 2
    return {"index_topk": idx_bytes, "step": idx_bytes + gather + window + qo + compress}


class ClockSampler:
    """Samples the SM clock and throttle reasons during the timed region: NVML
    (what nvidia-smi reads) polled from a thread, else an `nvidia-smi -lms` child."""

    _NAMES = {0x8: "hw_slowdown", 0x40: "hw_thermal_slowdown", 0x20: "sw_thermal_slowdown", 0x4: "sw_power_cap",
              0x80: "hw_power_brake_slowdown"}

    def __init__(self, dev_index: int, period_s: float = 0.005):
        self.samples, self.reasons, self.max_mhz = [], set(), None
        self.period, self._stop = period_s, threading.Event()
        self.mode, self.err = None, None
        try:
            import pynvml
            pynvml.nvmlInit()
            self.nvml = pynvml
            self.h = pynvml.nvmlDeviceGetHandleByIndex(dev_index)
            self.max_mhz = pynvml.nvmlDeviceGetMaxClockInfo(self.h, pynvml.NVML_CLOCK_SM)
            self.mode = "nvml"
        except Exception as e:  # noqa: BLE001
            self.err = f"nvml: {e}"
            self.mode = "smi"
        self.dev_index = dev_index

    def _run(self):
        while not self._stop.is_set():
            try:
                self.samples.append(self.nvml.nvmlDeviceGetClockInfo(self.h, self.nvml.NVML_CLOCK_SM))
                r = self.nvml.nvmlDeviceGetCurrentClocksEventReasons(self.h)
                for bit, name in self._NAMES.items():
                    if r & bit:
                        self.reasons.add(name)
            except Exception as e:  # noqa: BLE001
                self.err = f"nvml poll: {e}"
            time.sleep(self.period)

    def __enter__(self):
        if self.mode == "nvml":
            self.t = threading.Thread(target=self._run, daemon=True)
            self.t.start()
        else:
            q = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                 "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
            try:
                self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.dev_index), f"--query-gpu={q}",
                                              "--format=csv,noheader,nounits", "-lms", "50"],
                                             stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            except Exception as e:  # noqa: BLE001
                self.proc = None
                self.err = (self.err or "") + f"; smi: {e}"
        return self

    def __exit__(self, *a):
        if self.mode == "nvml":
            self._stop.set()
            self.t.join()
        elif getattr(self, "proc", None) is not None:
            self.proc.terminate()
            out, _ = self.proc.communicate(timeout=10)
            names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
            for line in out.splitlines():
                f = [x.strip() for x in line.split(",")]
                if len(f) < 6:
                    continue
                try:
                    self.samples.append(float(f[0]))
                    self.max_mhz = float(f[1])
                except ValueError:
                    continue
                for n, v in zip(names, f[2:6]):
                    if v.lower() == "active":
                        self.reasons.add(n)

    def summary(self):
        d = {"sm_mhz": statistics.median(self.samples) if self.samples else None, "sm_max_mhz": self.max_mhz,
             "reasons": sorted(self.reasons), "samples": len(self.samples), "source": self.mode}
        if self.err:
            d["note"] = self.err
        return d


def load_peaks(kind: str = "hbm_gbs"):
    """(peak, source): the measured copy bandwidth (GB/s) or bf16 GEMM rate (TFLOP/s)
    of this GPU model, else the earlier single-B300 measurement."""
    fallback = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        if kind in j:
            return float(j[kind]), "measured"
    return fallback[kind], "fallback"


# ------------------------------------------------------------ distributed

def dist_setup(args):
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, ws: int) -> float:
    if ws <= 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------- hsa arm

class DecodeBench:
    """Device buffers and the three C-ABI calls of one decode step."""

    def __init__(self, wl, replicas: int, seed_base: int, dev):
        from compressed_attention_compress_b300 import _lib as L
        self.L, self.wl, self.dev, self.R = L, wl, dev, replicas
        B, N, H, d, m, DI = wl.B, wl.N, wl.H, wl.d, wl.m, wl.DI
        E = N // m
        g = torch.Generator(device=dev)
        g.manual_seed(seed_base)

        def randn_bf16(shape):
            out = torch.empty(shape, dtype=torch.bfloat16, device=dev)
            flat = out.view(-1, shape[-1])
            step = 1 << 22
            for r0 in range(0, flat.shape[0], step):
                r1 = min(flat.shape[0], r0 + step)
                flat[r0:r1] = torch.randn((r1 - r0, shape[-1]), generator=g, device=dev).to(torch.bfloat16)
            return out

        def randint8(shape):
            return torch.randint(-127, 128, shape, generator=g, device=dev, dtype=torch.int16).to(torch.int8)

        self.k_raw = randn_bf16((B, N, d))
        self.v_raw = randn_bf16((B, N, d))
        self.w = block_weights(m, seed_base + 6).to(dev)
        self.kc = torch.empty((B, E, d), dtype=torch.bfloat16, device=dev)
        self.vc = torch.empty_like(self.kc)
        zeros = torch.zeros(B, dtype=torch.int64, device=dev)
        full = torch.full((B,), N, dtype=torch.int64, device=dev)
        L.hsa_compress(self.k_raw, self.v_raw, zeros, full, E, self.w, m, self.kc, self.vc)  # build the cache
        self.ctx = full
        self.pos0 = full - 1
        self.tb = full - m                # the block completed by the new token
        self.te = full
        self.q = [randn_bf16((B, H, d)) for _ in range(replicas)]
        self.qi = [randint8((B, 1, DI)) for _ in range(replicas)]
        self.ki = [randint8((B, E, DI)) for _ in range(replicas)]
        self.idx = [torch.empty((B, 1, wl.topk), dtype=torch.int32, device=dev) for _ in range(replicas)]
        self.cnt = [torch.empty((B, 1), dtype=torch.int32, device=dev) for _ in range(replicas)]
        self.out = [torch.empty((B, H, d), dtype=torch.bfloat16, device=dev) for _ in range(replicas)]
        self.lse = [torch.empty((B, H), dtype=torch.float32, device=dev) for _ in range(replicas)]
        self.ws_i = L.workspace(L.hsa_index_topk_workspace_size(B, 1, DI, E, wl.topk), device=dev)
        self.ws_a = L.workspace(L.hsa_attn_decode_workspace_size(torch.bfloat16, B, H, d, E, m, wl.topk, wl.window),
                                device=dev)
        torch.cuda.synchronize(dev)

    def compress(self, r):
        self.L.hsa_compress(self.k_raw, self.v_raw, self.tb, self.te, 1, self.w, self.wl.m, self.kc, self.vc)

    def index(self, r):
        self.L.hsa_index_topk(self.qi[r], self.ki[r], self.pos0, self.wl.m, self.wl.topk, self.idx[r], self.cnt[r],
                              self.ws_i)

    def attn(self, r):
        wl = self.wl
        self.L.hsa_attn_decode(self.q[r], self.kc, self.vc, wl.m, self.idx[r].view(wl.B, wl.topk),
                               self.cnt[r].view(wl.B), self.k_raw, self.v_raw, wl.window, self.ctx, wl.scale,
                               self.out[r], self.lse[r], self.ws_a)

    def step(self, r):
        self.compress(r)
        self.index(r)
        self.attn(r)


KERNELS_PER_STEP = 3  # compress, fused indexer/top-k, cluster attention (split merge inside)


def capture_block(bench, steps, start, events=None):
    """One CUDA graph of `steps` consecutive steps (replica (start+i) % R).  The new
    block's compression runs on a second stream, beside the indexer (which does not
    read the compressed cache); attention waits for both.  With `events`
    ([step][4] external CUDA events) the three calls run one after another on one
    stream, with the time recorded before and after each."""
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    side = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.graph(g, stream=s):
        for i in range(steps):
            r = (start + i) % bench.R
            if events is not None:
                events[i][0].record()
                bench.compress(r)
                events[i][1].record()
                bench.index(r)
                events[i][2].record()
                bench.attn(r)
                events[i][3].record()
                continue
            fork, join = torch.cuda.Event(), torch.cuda.Event()
            fork.record(s)
            side.wait_event(fork)
            with torch.cuda.stream(side):
                bench.compress(r)
            join.record(side)
            bench.index(r)
            s.wait_event(join)
            bench.attn(r)
    torch.cuda.current_stream().wait_stream(s)
    return g


def time_graph(fn, R: int, steps: int = 64, reps: int = 20) -> float:
    """ms per call of fn(replica) in a CUDA graph of `steps` calls over R replicas."""
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.graph(g, stream=s):
        for i in range(steps):
            fn(i % R)
    torch.cuda.current_stream().wait_stream(s)
    g.replay()
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record()
    for _ in range(reps):
        g.replay()
    t1.record()
    torch.cuda.synchronize()
    return t0.elapsed_time(t1) / (reps * steps)


def time_state_append(bench, steps: int = 64, reps: int = 20) -> float:
    """ms per call of the state-cache form of the step's compression (hsa_compress_append:
    one new token per sequence, completing its block), in a CUDA graph of `steps` calls."""
    wl, L = bench.wl, bench.L
    B, N, d = wl.B, wl.N, wl.d
    st_k = torch.zeros((B, d), dtype=torch.float32, device=bench.dev)
    st_v = torch.zeros_like(st_k)
    kn, vn = bench.k_raw[:, N - 1:N], bench.v_raw[:, N - 1:N]
    pos = bench.ctx - 1
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.graph(g, stream=s):
        for _ in range(steps):
            L.hsa_compress_append(kn, vn, pos, bench.w, wl.m, st_k, st_v, bench.kc, bench.vc)
    torch.cuda.current_stream().wait_stream(s)
    g.replay()
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record()
    for _ in range(reps):
        g.replay()
    t1.record()
    torch.cuda.synchronize()
    return t0.elapsed_time(t1) / (reps * steps)


def time_v4_details(bench, steps: int = 64, reps: int = 20) -> dict:
    """ms per call of the V4-detail kernels a decode step adds around the same attention
    kernels: RMSNorm + partial RoPE of the step's queries and of each sequence's new
    entry, and the sink + inverse rotation of the output (CUDA graphs of `steps` calls)."""
    wl, L, dev = bench.wl, bench.L, bench.dev
    B, H, d, m = wl.B, wl.H, wl.d, wl.m
    q = bench.q[0].clone()
    zeros = torch.zeros(B, dtype=torch.int64, device=dev)
    ones = torch.ones(B, dtype=torch.int64, device=dev)
    pos = bench.ctx - 1
    E_new = torch.div(bench.ctx, m, rounding_mode="floor")
    gamma = torch.ones(d, device=dev)
    sink = torch.zeros(H, device=dev)
    out = bench.out[0].clone()
    lse = torch.zeros((B, H), dtype=torch.float32, device=dev)
    kc = bench.kc.clone()
    calls = {
        "v4_prep_query": lambda: L.hsa_rmsnorm_rope(q.view(B, 1, H, d), zeros, ones, 1, pos, 1, 0, gamma),
        "v4_prep_entry": lambda: L.hsa_rmsnorm_rope(kc, E_new - 1, E_new, 1, None, m, m - 1, gamma),
        "v4_finalize": lambda: L.hsa_attn_finalize(out, lse, pos, sink),
    }
    res = {}
    for name, fn in calls.items():
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.graph(g, stream=s):
            for _ in range(steps):
                fn()
        torch.cuda.current_stream().wait_stream(s)
        g.replay()
        torch.cuda.synchronize()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record()
        for _ in range(reps):
            g.replay()
        t1.record()
        torch.cuda.synchronize()
        res[name] = t0.elapsed_time(t1) / (reps * steps)
    return res


def run_hsa(args, ws, rank, local):
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    R, BLOCK = args.replicas, args.block
    bench = DecodeBench(WL, R, 1000 * WL.wid + 100 * rank, dev)
    # eager warm-up (also sets kernel attributes before any capture)
    for i in range(max(args.warmup, 3)):
        bench.step(i % R)
    torch.cuda.synchronize()

    K = args.steps
    nblk, tail = divmod(K, BLOCK)
    g_main = capture_block(bench, BLOCK, 0)
    g_tail = capture_block(bench, tail, (nblk * BLOCK) % R) if tail else None
    # graph warm-up
    for _ in range(max(1, args.warmup // BLOCK)):
        g_main.replay()
    torch.cuda.synchronize()

    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(local)
    barrier(ws)
    torch.cuda.synchronize()
    with sampler:
        t0.record()
        for _ in range(nblk):
            g_main.replay()
        if g_tail is not None:
            g_tail.replay()
        t1.record()
        torch.cuda.synchronize()
    barrier(ws)
    ms_total = t0.elapsed_time(t1)
    ms_total = max_over_ranks(ms_total, ws)
    ms_step = ms_total / K

    # Per-op device time: the same steps replayed with an event record node
    # between the calls (the nodes themselves add a little time per step, so the
    # step time above comes from the uninstrumented graph).
    ev = [[torch.cuda.Event(enable_timing=True, external=True) for _ in range(4)] for _ in range(BLOCK)]
    g_ev = capture_block(bench, BLOCK, 0, ev)
    per_op = {"compress": [], "index_topk": [], "attn_decode": []}
    reps = max(1, min(8, nblk))
    for _ in range(reps):
        g_ev.replay()
        torch.cuda.synchronize()
        for i in range(BLOCK):
            per_op["compress"].append(ev[i][0].elapsed_time(ev[i][1]))
            per_op["index_topk"].append(ev[i][1].elapsed_time(ev[i][2]))
            per_op["attn_decode"].append(ev[i][2].elapsed_time(ev[i][3]))
    op_ms = {k: statistics.fmean(v) for k, v in per_op.items()}
    op_ms["compress_append"] = time_state_append(bench)
    op_ms.update(time_v4_details(bench))
    op_ms["attn_decode_shared_kv"] = time_graph(lambda r: bench.L.hsa_attn_decode(
        bench.q[r], bench.kc, bench.kc, WL.m, bench.idx[r].view(WL.B, WL.topk), bench.cnt[r].view(WL.B),
        bench.k_raw, bench.k_raw, WL.window, bench.ctx, WL.scale, bench.out[r], bench.lse[r], bench.ws_a), bench.R)

    cnt_total = int(sum(int(c.sum()) for c in bench.cnt[:1]))
    bytes_ = algorithmic_bytes(WL, cnt_total)
    peak, peak_kind = load_peaks()
    queries = WL.B * ws
    value = queries / (ms_step * 1e-3)

    # end to end through the public API: pinned host inputs in, result out, every step
    e2e = None if args.profile else run_e2e(bench, args, dev)

    out = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": K, "warmup": args.warmup,
        "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16 (int8 indexer, int32 scores, fp32 accumulate)", "data": "synthetic (seeded N(0,1) bf16, uniform int8)",
        "config": {"workload": WL.name, "global_batch": WL.B * ws, "seq_len": WL.N, "parallelism": f"replicas x{ws}",
                   "l2": f"rotating {R} input replicas: {R * WL.B * (WL.N // WL.m) * WL.DI / 2**20:.0f} MiB of indexer keys > 4x L2",
                   "graph_block": BLOCK},
        "hbm_gbs_step": bytes_["step"] / (ms_step * 1e-3) / 1e9,
        "gpu_launches": KERNELS_PER_STEP * K,
        "e2e": e2e,
    }
    if op_ms["index_topk"]:
        ach = bytes_["index_topk"] / (op_ms["index_topk"] * 1e-3) / 1e9
        out["roofline"] = {"kernel": "index_fused_kernel (hsa_index_topk; one launch per step)", "bound": "hbm",
                           "achieved": ach, "peak": peak, "unit": "GB/s", "frac": ach / peak,
                           "traffic": args.traffic if args.traffic is not None else index_traffic(),
                           "peak_source": peak_kind,
                           "algorithmic_bytes_per_launch": bytes_["index_topk"]}
        step_ach = bytes_["step"] / (ms_step * 1e-3) / 1e9
        out["step_roofline"] = {"bound": "hbm", "achieved": step_ach, "peak": peak, "unit": "GB/s",
                                "frac": step_ach / peak, "algorithmic_bytes_per_step": bytes_["step"]}
        out["op_ms"] = op_ms
    out["clocks"] = sampler.summary()
    return out, bench


def run_e2e(bench, args, dev):
    """Same metric through the Python/C-ABI calls with host buffers: each step copies
    its inputs (q, indexer query) from pinned host memory, runs the three calls, reads
    the output back to pinned host memory, and waits for it.  The step's copies and
    calls are captured once per input replica into a CUDA graph (compression on a
    second stream beside the indexer, as a serving loop would run them); every step
    replays one graph and synchronises; the attention's query is copied on the second
    stream.  `eager_*` is the same step issued call by call on one stream."""
    wl = bench.wl
    R = bench.R
    hq = [bench.q[r].cpu().pin_memory() for r in range(R)]
    hqi = [bench.qi[r].cpu().pin_memory() for r in range(R)]
    hout = torch.empty((wl.B, wl.H, wl.d), dtype=torch.bfloat16).pin_memory()
    dq = torch.empty_like(bench.q[0])
    dqi = torch.empty_like(bench.qi[0])
    steps = max(20, min(args.steps, 2000))

    def calls(r, side=None):
        if side is None:
            dq.copy_(hq[r], non_blocking=True)
            dqi.copy_(hqi[r], non_blocking=True)
            bench.compress(r)
        else:
            # the attention's query travels beside the indexer's, with the compression
            fork, join = torch.cuda.Event(), torch.cuda.Event()
            fork.record()
            side.wait_event(fork)
            with torch.cuda.stream(side):
                dq.copy_(hq[r], non_blocking=True)
                bench.compress(r)
            join.record(side)
            dqi.copy_(hqi[r], non_blocking=True)
        bench.L.hsa_index_topk(dqi, bench.ki[r], bench.pos0, wl.m, wl.topk, bench.idx[r], bench.cnt[r], bench.ws_i)
        if side is not None:
            torch.cuda.current_stream().wait_event(join)
        bench.L.hsa_attn_decode(dq, bench.kc, bench.vc, wl.m, bench.idx[r].view(wl.B, wl.topk), bench.cnt[r].view(wl.B),
                                bench.k_raw, bench.v_raw, wl.window, bench.ctx, wl.scale, bench.out[r], bench.lse[r],
                                bench.ws_a)
        hout.copy_(bench.out[r], non_blocking=True)

    def timed(one):
        for i in range(5):
            one(i)
        t = time.perf_counter()
        for i in range(steps):
            one(i)
        return (time.perf_counter() - t) / steps

    def eager(i):
        calls(i % R)
        torch.cuda.current_stream().synchronize()

    dt_eager = timed(eager)

    graphs = []
    side = torch.cuda.Stream()
    cap = torch.cuda.Stream()
    cap.wait_stream(torch.cuda.current_stream())
    for r in range(R):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cap):
            calls(r, side)
        graphs.append(g)
    torch.cuda.current_stream().wait_stream(cap)
    torch.cuda.synchronize()

    def replay(i):
        graphs[i % R].replay()
        torch.cuda.current_stream().synchronize()

    dt = timed(replay)
    h2d = hq[0].numel() * 2 + hqi[0].numel()
    d2h = hout.numel() * 2
    return {"value": wl.B / dt, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "ms_per_step": dt * 1e3, "steps": steps,
            "launch": "one CUDA graph per step (replayed, then synchronised)",
            "eager_value": wl.B / dt_eager, "eager_ms_per_step": dt_eager * 1e3}


# --------------------------------------------------- chunked prefill rows

def prefill_flops(wl) -> float:
    """4*H*d FLOP per (query row, attended item): QK^T and PV, multiply-add = 2 FLOP."""
    p = np.arange(wl.N - wl.T, wl.N, dtype=np.int64)
    E = (p + 1) // wl.m
    sel = np.minimum(E, wl.topk) if wl.kind == "csa" else E
    items = sel + np.minimum(wl.window, p + 1)
    return 4.0 * wl.B * wl.H * wl.d * float(items.sum())


def run_prefill(dev, reps: int):
    """Chunked prefill of 8192 new tokens on a 1,048,576-token cache, one HCA and one CSA
    layer.  Each call is timed alone with CUDA events on the launching stream, L2
    flushed (a 256 MiB write) before every run; median of `reps` runs after 2 warm-ups."""
    from compressed_attention_compress_b300 import _lib as L
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    peak_tc = load_peaks(kind="bf16_tflops")
    peak_bw, _ = load_peaks()

    def timed(fn):
        ts = []
        for i in range(reps + 2):
            flush.fill_(i & 255)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            torch.cuda.synchronize(dev)
            if i >= 2:
                ts.append(e0.elapsed_time(e1))
        return statistics.median(ts)

    res = {}
    for name in ("prefill_hca", "prefill_csa"):
        wl = WORKLOADS[name]
        B, N, H, d, m, T = wl.B, wl.N, wl.H, wl.d, wl.m, wl.T
        E = N // m
        g = torch.Generator(device=dev)
        g.manual_seed(1000 * wl.wid)
        kr = torch.randn((B, N, d), generator=g, device=dev).to(torch.bfloat16)
        vr = torch.randn((B, N, d), generator=g, device=dev).to(torch.bfloat16)
        q = torch.randn((B, T, H, d), generator=g, device=dev).to(torch.bfloat16)
        w = block_weights(m, 1000 * wl.wid + 6).to(dev)
        kc = torch.empty((B, E, d), dtype=torch.bfloat16, device=dev)
        vc = torch.empty_like(kc)
        zeros = torch.zeros(B, dtype=torch.int64, device=dev)
        full = torch.full((B,), N, dtype=torch.int64, device=dev)
        pos0 = full - T
        L.hsa_compress(kr, vr, zeros, pos0, (N - T) // m, w, m, kc, vc)  # the cache before the chunk
        out = torch.empty((B, T, H, d), dtype=torch.bfloat16, device=dev)
        r = {"workload": wl.name}
        r["compress_chunk_ms"] = timed(lambda: L.hsa_compress(kr, vr, pos0, full, T // m, w, m, kc, vc))
        # the learned attention-like compressor (window 2m for CSA, m for HCA) on the same chunk
        Lw = 2 * m if wl.kind == "csa" else m
        u_l = torch.randn((d,), generator=g, device=dev) / d ** 0.5
        b_l = torch.randn((Lw,), generator=g, device=dev)
        r["compress_learned_chunk_ms"] = timed(lambda: L.hsa_compress_learned(kr, vr, pos0, full, T // m, u_l, b_l, m,
                                                                              kc, vc))
        idx = cnt = None
        if wl.kind == "csa":
            qi = torch.randint(-127, 128, (B, T, wl.DI), generator=g, device=dev, dtype=torch.int16).to(torch.int8)
            ki = torch.randint(-127, 128, (B, E, wl.DI), generator=g, device=dev, dtype=torch.int16).to(torch.int8)
            idx = torch.empty((B, T, wl.topk), dtype=torch.int32, device=dev)
            cnt = torch.empty((B, T), dtype=torch.int32, device=dev)
            ws_i = L.workspace(L.hsa_index_topk_workspace_size(B, T, wl.DI, E, wl.topk), device=dev)
            r["index_ms"] = timed(lambda: L.hsa_index_topk(qi, ki, pos0, m, wl.topk, idx, cnt, ws_i))
            p = np.arange(N - T, N, dtype=np.int64)
            macs = float(B * ((p + 1) // m).sum() * wl.DI)
            r["index_tflops"] = 2 * macs / (r["index_ms"] * 1e-3) / 1e12
            r["index_frac_of_bf16_peak"] = r["index_tflops"] / peak_tc[0]
        ws_a = L.workspace(L.hsa_attn_prefill_workspace_size(torch.bfloat16, B, T, H, d, E, m,
                                                             wl.topk if wl.kind == "csa" else 0, wl.window),
                           device=dev)
        r["attn_ms"] = timed(lambda: L.hsa_attn_prefill(q, kc, vc, m, idx, cnt, kr, vr, wl.window, pos0, wl.scale,
                                                        out, ws=ws_a))
        flop = prefill_flops(wl)
        r["attn_tflops"] = flop / (r["attn_ms"] * 1e-3) / 1e12
        r["attn_frac_of_bf16_peak"] = r["attn_tflops"] / peak_tc[0]
        # V4's shared key/value entry: one buffer passed as both K and V (each item loaded once)
        r["attn_shared_kv_ms"] = timed(lambda: L.hsa_attn_prefill(q, kc, kc, m, idx, cnt, kr, kr, wl.window, pos0,
                                                                  wl.scale, out, ws=ws_a))
        if wl.kind == "csa":
            gather = float(B * T) * (wl.topk + wl.window) * 2 * d * 2
            r["attn_gather_gbs"] = gather / (r["attn_ms"] * 1e-3) / 1e9
            layer = r["compress_chunk_ms"] + r["index_ms"] + r["attn_ms"]
            r["layer_ms"] = layer
            r["layer_tflops"] = (flop + 2 * macs) / (layer * 1e-3) / 1e12
        else:
            r["layer_ms"] = r["compress_chunk_ms"] + r["attn_ms"]
        r["peak_bf16_tflops"] = peak_tc[0]
        r["peak_source"] = peak_tc[1]
        res[name] = {k: (round(v, 4) if isinstance(v, float) else v) for k, v in r.items()}
        del kr, vr, q, kc, vc, out
        torch.cuda.empty_cache()
    return res


# ------------------------------------------------------ oracle (CPU) arm

def oracle_sample_setup(seconds_hint=True):
    """One sequence of the workload on the host, its compressed cache built by the oracle."""
    import oracle
    from compressed_attention_compress_b300.inputs import bf16_bits, make_inputs
    oracle.build()
    x = make_inputs(WL, B=1)
    m = WL.m
    E = WL.N // m
    kr, vr = bf16_bits(x.k_raw), bf16_bits(x.v_raw)
    kc = oracle.compress(kr, x.w.numpy(), m, [0], [WL.N], E, out_dtype=np.float32)
    vc = oracle.compress(vr, x.w.numpy(), m, [0], [WL.N], E, out_dtype=np.float32)
    return oracle, x, kr, vr, kc, vc


def oracle_query(oracle, x, kr, vr, kc, vc, rep: int):
    """One decode query through the oracle: compress the new block, index + top-k, attention."""
    from compressed_attention_compress_b300.inputs import bf16_bits
    m, N = WL.m, WL.N
    p = N - 1
    newblk = oracle.compress(kr[:, N - m:], x.w.numpy(), m, [0], [m], 1, out_dtype=np.float32)
    kc[:, -1] = newblk[:, 0]
    oi, oc = oracle.index_topk_rows(x.q_idx.numpy().reshape(1, WL.DI), [0], [p], x.k_idx.numpy(), m, WL.topk)
    o, l = oracle.attn_rows(bf16_bits(x.q).reshape(1, WL.H, WL.d), [0], [p], kc, vc, m, oi, kr, vr, WL.window,
                            WL.scale)
    return o


def cpu_baseline(budget_s: float):
    """Time the oracle as it stands on a bounded sample (whole decode queries of sequence 0)."""
    t_setup = time.perf_counter()
    oracle, x, kr, vr, kc, vc = oracle_sample_setup()
    setup = time.perf_counter() - t_setup
    n = 0
    t = time.perf_counter()
    while True:
        oracle_query(oracle, x, kr, vr, kc, vc, n)
        n += 1
        if time.perf_counter() - t >= budget_s:
            break
    dt = time.perf_counter() - t
    return {"value": n / dt, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"{n} full decode queries of sequence 0 (index over 262144 entries, top-1024, attention over "
                      f"1152 items x 128 heads, new-block compress); {dt:.1f} s timed, cache build {setup:.1f} s untimed",
            "cpu": platform.processor() or platform.machine()}


def run_reference(args, ws, rank):
    if rank != 0:
        return None
    oracle, x, kr, vr, kc, vc = oracle_sample_setup()
    for i in range(args.warmup if args.warmup < 3 else 3):
        oracle_query(oracle, x, kr, vr, kc, vc, i)
    K = args.steps
    # each step is one decode query (one of the B sequences' worth of work); bound the run to minutes
    per = None
    t = time.perf_counter()
    done = 0
    for i in range(K):
        oracle_query(oracle, x, kr, vr, kc, vc, i)
        done += 1
        el = time.perf_counter() - t
        per = el / done
        if el > args.ref_budget:
            break
    dt = time.perf_counter() - t
    value = done / dt
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": done,
            "warmup": args.warmup, "ms_per_step": dt / done * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64 (oracle)", "data": "synthetic",
            "config": {"workload": WL.name, "global_batch": 1, "seq_len": WL.N, "parallelism": "host cores"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
                             "sample": f"{done} of the {K} requested steps, one decode query each (sequence 0); "
                                       f"run bounded to {args.ref_budget:.0f} s"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=64)
    ap.add_argument("--impl", choices=["hsa", "reference"], default="hsa")
    ap.add_argument("--replicas", type=int, default=8)
    ap.add_argument("--block", type=int, default=64, help="steps per captured CUDA graph")
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--ref-budget", type=float, default=120.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--traffic", type=float, default=None, help="ncu dram bytes per index_topk launch, if known")
    ap.add_argument("--no-prefill", action="store_true", help="skip the chunked-prefill rows")
    ap.add_argument("--prefill-reps", type=int, default=10)
    ap.add_argument("--prefill-only", action="store_true",
                    help="only the chunked-prefill rows (for profiling their kernels)")
    ap.add_argument("--profile", action="store_true",
                    help="small run for ncu captures: 2 replicas, no end-to-end or CPU legs")
    args = ap.parse_args()
    if args.profile:
        args.replicas, args.block, args.no_cpu_baseline = 2, max(1, min(args.block, args.steps)), True
        args.no_prefill = True
    # the oracle's host threads are started before any GPU work
    ws, rank, local = dist_setup(args)
    if args.impl == "reference":
        res = run_reference(args, ws, rank)
        if res is not None:
            print(json.dumps(res), flush=True)
        return
    if args.prefill_only:
        torch.cuda.set_device(local)
        res = run_prefill(torch.device("cuda", local), args.prefill_reps)
        if rank == 0:
            print(json.dumps({"prefill": res}), flush=True)
        return
    res, bench = run_hsa(args, ws, rank, local)
    del bench
    torch.cuda.empty_cache()
    if not args.no_prefill:
        res["prefill"] = run_prefill(torch.device("cuda", local), args.prefill_reps)
    if rank == 0:
        if not args.no_cpu_baseline and ws == 1:
            res["cpu_baseline"] = cpu_baseline(args.cpu_budget)
        print(json.dumps(res), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
