#!/usr/bin/env python3
"""Benchmark of the hybrid compressed/sparse attention hot path on B300.

The headline step is one decode step of one CSA attention layer over a batch of
4 sequences at 1,048,576 cached tokens (V4-Pro shape: 128 query heads, head dim
128, m = 4 -> 262,144 compressed entries, int8 indexer dim 64, top-k 1024,
128-token window):
  1. hsa_compress    -- fold the block completed by the new token into its entry
  2. hsa_index_topk  -- int8 scores of all 262,144 entries, exact top-1024
  3. hsa_attn_decode -- attention over the 1024 entries + 128 raw tokens, split
                        over 128-item tiles and merged by log-sum-exp.
The same timing runs two more decode rows: the V4-Flash-shaped CSA step (B = 8
at 131,072 tokens, 64 heads, top-k 512) and the HCA step (B = 16, lengths
uniform in [262144, 1048576], m = 128, dense over all entries + window).

Inputs are seeded synthetic tensors.  Every per-step buffer (query, indexer
keys, raw and compressed caches, outputs) exists in R replicas that the steps
rotate over, and the replicas' bytes exceed 4x the L2 cache, so a step reads its
inputs from HBM.  CUDA graphs hold the steps; the timed region is exactly K
steps (barrier + synchronize on both sides, max over ranks), followed by at
least 20 further replays of the same K steps whose median is reported beside it.
The chunked-prefill rows (8192 new tokens on a 1M-token cache, one HCA and one
CSA layer) time each call alone after an L2 flush.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl {hsa,reference}]
Prints one JSON line on rank 0.  With --gpus N > 1 and no launcher environment,
the script starts N ranks itself (one process per GPU, NCCL), each running the
same replicas on its own GPU (weak scaling, no data-path collective).
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import math
import os
import platform
import socket
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from compressed_attention_compress_b300.inputs import WORKLOADS, block_weights, context_lengths, T_LEN  # noqa: E402

HEADLINE = "pro_csa_decode"
EXTRA_DECODE = ("flash_csa_decode", "hca_decode")
METRIC = "decode queries/s at 1M ctx (V4-Pro-shaped CSA layer, B=4)"
UNIT = "queries/s"

# DRAM bytes (read + write) of one launch of a kernel on a workload, from an ncu
# capture of that kernel; reported only while the kernel's sources are the ones
# that capture ran (sha256 of each file).
TRAFFIC = {
    ("index_fused_kernel", "pro_csa_decode"): {
        "bytes": 67240960 + 509952,
        "sources": {
            "compressed_attention_compress_b300/csrc/index_fused.cu":
                "07a532c05edea268a0dd2b2fd8e9e3d7969f8ad7693ca4309344da283dddfc61",
            "compressed_attention_compress_b300/csrc/common.cuh":
                "79620607484ca1168ae52da7bbf685b100d0e8e9f3444486c3871e963c3a346d",
            "compressed_attention_compress_b300/csrc/block_scan.cuh":
                "fcbf6072ec91c580a5c6abf47cd7a369531be3b55ac0e10c9af50cbdb7c7dd8d",
        },
    },
}


def measured_traffic(kernel: str, workload: str):
    t = TRAFFIC.get((kernel, workload))
    if t is None:
        return None
    for rel, want in t["sources"].items():
        with open(os.path.join(ROOT, rel), "rb") as f:
            if hashlib.sha256(f.read()).hexdigest() != want:
                return None
    return t["bytes"]


# ----------------------------------------------------------------- helpers

def algorithmic_bytes(wl, ctx, cnt_total: int):
    """Bytes the method must move in one decode step (raw cache outside the window
    not counted): indexer keys and query, the top-k written and read back, the
    selected (CSA) or all visible (HCA) compressed K and V rows, the window's raw K
    and V rows, q and out, and the new block's compression."""
    B, d, m = wl.B, wl.d, wl.m
    E = [int(c) // m for c in ctx]
    win = sum(min(wl.window, int(c)) for c in ctx)
    if wl.kind == "csa":
        index = sum(E) * wl.DI + B * wl.DI + 2 * B * wl.topk * 4 + 2 * B * 4
        entries = cnt_total * 2 * d * 2
    else:
        index = 0
        entries = sum(E) * 2 * d * 2
    window = win * 2 * d * 2
    qo = 2 * B * wl.H * d * 2
    compress = B * m * 2 * d * 2 + B * 2 * d * 2
    attn = entries + window + qo + (2 * B * wl.topk * 4 if wl.kind == "csa" else 0)
    return {"index_topk": index, "attn_decode": attn, "compress": compress,
            "step": index + entries + window + qo + compress}


def pci_bus_id(dev_index: int):
    """PCI bus id of CUDA device `dev_index` in NVML's form, so that NVML and
    nvidia-smi read the same GPU whatever CUDA_VISIBLE_DEVICES maps; None if unknown."""
    try:
        p = torch.cuda.get_device_properties(dev_index)
        return f"{p.pci_domain_id:08X}:{p.pci_bus_id:02X}:{p.pci_device_id:02X}.0"
    except Exception:  # noqa: BLE001
        return None


class _CtypesNvml:
    """Read-only NVML through libnvidia-ml (clock and clock-event reasons), for
    when the pynvml module is not importable."""

    def __init__(self, bus_id):
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit_v2 failed")
        self.h = ctypes.c_void_p()
        if self.lib.nvmlDeviceGetHandleByPciBusId_v2(bus_id.encode(), ctypes.byref(self.h)) != 0:
            raise RuntimeError(f"nvmlDeviceGetHandleByPciBusId_v2({bus_id}) failed")
        fn = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None)
        self._reasons_fn = fn if fn is not None else self.lib.nvmlDeviceGetCurrentClocksThrottleReasons

    def sm_clock(self):
        c = ctypes.c_uint()
        self.lib.nvmlDeviceGetClockInfo(self.h, ctypes.c_int(1), ctypes.byref(c))  # NVML_CLOCK_SM
        return c.value

    def max_sm_clock(self):
        c = ctypes.c_uint()
        self.lib.nvmlDeviceGetMaxClockInfo(self.h, ctypes.c_int(1), ctypes.byref(c))
        return c.value

    def reasons(self):
        r = ctypes.c_ulonglong()
        self._reasons_fn(self.h, ctypes.byref(r))
        return r.value


class ClockSampler:
    """Samples the SM clock and clock-event (throttle) reasons while the timed work
    runs: NVML (pynvml, else libnvidia-ml through ctypes) polled from a thread,
    else an `nvidia-smi -lms` child.  Only reads; changes no setting."""

    _NAMES = {0x8: "hw_slowdown", 0x40: "hw_thermal_slowdown", 0x20: "sw_thermal_slowdown", 0x4: "sw_power_cap",
              0x80: "hw_power_brake_slowdown"}

    def __init__(self, dev_index: int, period_s: float = 0.01):
        self.samples, self.reasons, self.max_mhz = [], set(), None
        self.period, self._stop = period_s, threading.Event()
        self.mode, self.err = None, None
        self.bus_id = pci_bus_id(dev_index)
        self.dev_index = dev_index
        try:
            import pynvml
            pynvml.nvmlInit()
            h = pynvml.nvmlDeviceGetHandleByPciBusId(self.bus_id)
            self._clock = lambda: pynvml.nvmlDeviceGetClockInfo(h, pynvml.NVML_CLOCK_SM)
            self._reasons = lambda: pynvml.nvmlDeviceGetCurrentClocksEventReasons(h)
            self.max_mhz = pynvml.nvmlDeviceGetMaxClockInfo(h, pynvml.NVML_CLOCK_SM)
            self.mode = "nvml"
        except Exception as e:  # noqa: BLE001
            self.err = f"pynvml: {e}"
            try:
                n = _CtypesNvml(self.bus_id)
                self._clock, self._reasons = n.sm_clock, n.reasons
                self.max_mhz = n.max_sm_clock()
                self.mode = "nvml-ctypes"
            except Exception as e2:  # noqa: BLE001
                self.err += f"; libnvidia-ml: {e2}"
                self.mode = "smi"

    def _run(self):
        while not self._stop.is_set():
            try:
                self.samples.append(self._clock())
                r = self._reasons()
                for bit, name in self._NAMES.items():
                    if r & bit:
                        self.reasons.add(name)
            except Exception as e:  # noqa: BLE001
                self.err = f"poll: {e}"
            time.sleep(self.period)

    def __enter__(self):
        if self.mode != "smi":
            self.t = threading.Thread(target=self._run, daemon=True)
            self.t.start()
        else:
            q = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                 "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
            try:
                self.proc = subprocess.Popen(["nvidia-smi", "-i", self.bus_id or str(self.dev_index), f"--query-gpu={q}",
                                              "--format=csv,noheader,nounits", "-lms", "50"],
                                             stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
                time.sleep(0.5)  # the child's first sample
            except Exception as e:  # noqa: BLE001
                self.proc = None
                self.err = (self.err or "") + f"; smi: {e}"
        return self

    def __exit__(self, *a):
        if self.mode != "smi":
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
             "reasons": sorted(self.reasons), "samples": len(self.samples), "source": self.mode,
             "window": "warm-up, the timed K steps and the repeated replays"}
        if self.err and not self.samples:
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

def dist_setup():
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
    dev = "cuda" if torch.cuda.is_available() and dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_entry(local_rank: int, argv, n: int, port: int):
    os.environ.update({"RANK": str(local_rank), "LOCAL_RANK": str(local_rank), "WORLD_SIZE": str(n),
                       "LOCAL_WORLD_SIZE": str(n), "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    main(argv)


def spawn_ranks(argv, n: int):
    """Start n ranks of this script (one process per GPU) when no launcher did."""
    import torch.multiprocessing as mp
    mp.start_processes(_rank_entry, args=(argv, n, _free_port()), nprocs=n, start_method="spawn", join=True)


# ------------------------------------------------------------- decode rows

class DecodeBench:
    """Device buffers of R input replicas and the C-ABI calls of one decode step."""

    def __init__(self, wl, replicas: int, seed_base: int, dev, fused: bool = False):
        from compressed_attention_compress_b300 import _lib as L
        self.L, self.wl, self.dev, self.R = L, wl, dev, replicas
        B, N, H, d, m = wl.B, wl.N, wl.H, wl.d, wl.m
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

        if wl.len_hi:
            ctx = context_lengths(B, wl.len_lo, wl.len_hi, 1000 * wl.wid + T_LEN)
        else:
            ctx = torch.full((B,), N, dtype=torch.int64)
        self.ctx_host = ctx
        self.ctx = ctx.to(dev)
        self.pos0 = self.ctx - 1
        # the block the newest complete block boundary closes, one per sequence
        last = torch.div(self.ctx, m, rounding_mode="floor") * m
        self.tb, self.te = (last - m).clamp(min=0), last
        self.w = block_weights(m, seed_base + 6).to(dev)
        zeros = torch.zeros(B, dtype=torch.int64, device=dev)
        self.k_raw, self.v_raw, self.kc, self.vc, self.q = [], [], [], [], []
        self.qi, self.ki, self.idx, self.cnt, self.out, self.lse = [], [], [], [], [], []
        for r in range(replicas):
            kr, vr = randn_bf16((B, N, d)), randn_bf16((B, N, d))
            kc = torch.empty((B, E, d), dtype=torch.bfloat16, device=dev)
            vc = torch.empty_like(kc)
            L.hsa_compress(kr, vr, zeros, self.ctx, E, self.w, m, kc, vc)  # the cache before the step
            self.k_raw.append(kr)
            self.v_raw.append(vr)
            self.kc.append(kc)
            self.vc.append(vc)
            self.q.append(randn_bf16((B, H, d)))
            self.out.append(torch.empty((B, H, d), dtype=torch.bfloat16, device=dev))
            self.lse.append(torch.empty((B, H), dtype=torch.float32, device=dev))
            if wl.kind == "csa":
                self.qi.append(randint8((B, 1, wl.DI)))
                self.ki.append(randint8((B, E, wl.DI)))
                self.idx.append(torch.empty((B, 1, wl.topk), dtype=torch.int32, device=dev))
                self.cnt.append(torch.empty((B, 1), dtype=torch.int32, device=dev))
        self.ws_i = None
        if wl.kind == "csa":
            self.ws_i = L.workspace(L.hsa_index_topk_workspace_size(B, 1, wl.DI, E, wl.topk), device=dev)
        self.ws_a = L.workspace(L.hsa_attn_decode_workspace_size(torch.bfloat16, B, H, d, E, m,
                                                                 wl.topk if wl.kind == "csa" else 0, wl.window),
                                device=dev)
        # CSA: the one-launch decode step (hsa_decode_csa) when the shape fits it, else
        # the two calls hsa_index_topk + hsa_attn_decode
        self.fused = False
        if wl.kind == "csa" and fused:
            try:
                self.ws_f = L.workspace(L.hsa_decode_csa_workspace_size(B, H, d, wl.DI, E), device=dev)
                self.fused = True
            except L.HSAError:
                self.fused = False
        torch.cuda.synchronize(dev)
        if self.fused:
            self.calls = ("compress", "decode_step")
        elif wl.kind == "csa":
            self.calls = ("compress", "index_topk", "attn_decode")
        else:
            self.calls = ("compress", "attn_decode")

    def replica_bytes(self) -> int:
        per = sum(t.numel() * t.element_size() for t in (self.k_raw[0], self.v_raw[0], self.kc[0], self.vc[0]))
        if self.wl.kind == "csa":
            per += self.ki[0].numel()
        return per

    def compress(self, r):
        self.L.hsa_compress(self.k_raw[r], self.v_raw[r], self.tb, self.te, 1, self.w, self.wl.m, self.kc[r],
                            self.vc[r])

    def index(self, r, qi=None):
        self.L.hsa_index_topk(self.qi[r] if qi is None else qi, self.ki[r], self.pos0, self.wl.m, self.wl.topk,
                              self.idx[r], self.cnt[r], self.ws_i)

    def attn(self, r, q=None, kv_shared=False):
        wl = self.wl
        csa = wl.kind == "csa"
        vc = self.kc[r] if kv_shared else self.vc[r]
        vr = self.k_raw[r] if kv_shared else self.v_raw[r]
        self.L.hsa_attn_decode(self.q[r] if q is None else q, self.kc[r], vc, wl.m,
                               self.idx[r].view(wl.B, wl.topk) if csa else None,
                               self.cnt[r].view(wl.B) if csa else None, self.k_raw[r], vr, wl.window, self.ctx,
                               wl.scale, self.out[r], self.lse[r], self.ws_a)

    def decode_step(self, r, qi=None, q=None):
        wl = self.wl
        self.L.hsa_decode_csa(self.qi[r] if qi is None else qi, self.ki[r], wl.m, wl.topk,
                              self.idx[r].view(wl.B, wl.topk), self.cnt[r].view(wl.B), self.q[r] if q is None else q,
                              self.kc[r], self.vc[r], self.k_raw[r], self.v_raw[r], wl.window, self.ctx, wl.scale,
                              self.out[r], self.lse[r], self.ws_f)

    def step(self, r):
        self.compress(r)
        if self.fused:
            self.decode_step(r)
            return
        if self.wl.kind == "csa":
            self.index(r)
        self.attn(r)

    def cnt_total(self) -> int:
        if self.wl.kind != "csa":
            return 0
        return int(self.cnt[0].sum())


def capture_steps(bench, steps, start, events=None):
    """One CUDA graph of `steps` consecutive steps (replica (start + i) % R).  With
    the one-launch decode step the new block's compression runs first (the step
    reads the compressed cache); with two calls it runs on a second stream beside
    the indexer (which does not read it) and the attention waits for both.  With `events`
    ([step][calls + 1] CUDA events) the calls run one after another on one stream
    with an event recorded before and after each."""
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    side = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.graph(g, stream=s):
        for i in range(steps):
            r = (start + i) % bench.R
            if events is not None:
                ev = events[i]
                ev[0].record()
                bench.compress(r)
                ev[1].record()
                if bench.fused:
                    bench.decode_step(r)
                    ev[-1].record()
                    continue
                if bench.wl.kind == "csa":
                    bench.index(r)
                    ev[2].record()
                bench.attn(r)
                ev[-1].record()
                continue
            if bench.fused:
                bench.compress(r)
                bench.decode_step(r)
                continue
            if bench.wl.kind == "csa":
                fork, join = torch.cuda.Event(), torch.cuda.Event()
                fork.record(s)
                side.wait_event(fork)
                with torch.cuda.stream(side):
                    bench.compress(r)
                join.record(side)
                bench.index(r)
                s.wait_event(join)
            else:
                bench.compress(r)
            bench.attn(r)
    torch.cuda.current_stream().wait_stream(s)
    return g


def time_decode(bench, K: int, W: int, block: int, ws: int, min_repeat_s: float = 1.0):
    """Exactly K steps timed once (barrier + synchronize on both sides, max over
    ranks), then the same K steps replayed at least 20 times (and for at least
    `min_repeat_s`), each replay timed alone; returns both and the replay median."""
    for i in range(max(W, 3)):  # eager warm-up (also sets kernel attributes before any capture)
        bench.step(i % bench.R)
    torch.cuda.synchronize()
    graphs = []
    done = 0
    while done < K:
        n = min(block, K - done)
        graphs.append(capture_steps(bench, n, done % bench.R))
        done += n

    def replay_all():
        for g in graphs:
            g.replay()

    for _ in range(max(1, math.ceil(max(W, 3) / K))):  # graph warm-up: at least W steps
        replay_all()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    barrier(ws)
    torch.cuda.synchronize()
    t0.record()
    replay_all()
    t1.record()
    torch.cuda.synchronize()
    barrier(ws)
    ms_total = max_over_ranks(t0.elapsed_time(t1), ws)
    reps = []
    wall0 = time.perf_counter()
    while len(reps) < 20 or time.perf_counter() - wall0 < min_repeat_s:
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        replay_all()
        e1.record()
        e1.synchronize()
        reps.append(e0.elapsed_time(e1) / K)
        if len(reps) >= 100000:
            break
    med = max_over_ranks(statistics.median(reps), ws)
    return {"ms_per_step": ms_total / K, "ms_per_step_median": med, "replays": len(reps),
            "ms_per_step_min": min(reps), "ms_per_step_max": max(reps)}


def per_call_ms(bench, steps: int = 64, reps: int = 4) -> dict:
    """Device time of each call of the step: the steps replayed with an event
    record between the calls (those nodes add ~1-2 us per call, so the step time
    comes from the uninstrumented graphs)."""
    n = len(bench.calls) + 1
    ev = [[torch.cuda.Event(enable_timing=True, external=True) for _ in range(n)] for _ in range(steps)]
    g = capture_steps(bench, steps, 0, ev)
    acc = {c: [] for c in bench.calls}
    for _ in range(reps):
        g.replay()
        torch.cuda.synchronize()
        for i in range(steps):
            for c, name in enumerate(bench.calls):
                acc[name].append(ev[i][c].elapsed_time(ev[i][c + 1]))
    return {k: statistics.fmean(v) for k, v in acc.items()}


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
    pos = bench.ctx - 1
    return time_graph(lambda r: L.hsa_compress_append(bench.k_raw[r][:, N - 1:N], bench.v_raw[r][:, N - 1:N], pos,
                                                      bench.w, wl.m, st_k, st_v, bench.kc[r], bench.vc[r]),
                      bench.R, steps, reps)


def time_v4_details(bench, steps: int = 64, reps: int = 20):
    """ms per call of a V4-detail decode step's calls (CUDA graphs of `steps` calls): the
    attention with the query prep, sink and inverse rotation inside it
    (hsa_attn_decode_v4), and the new block's compression with the entry's RMSNorm +
    partial RoPE as it is written (hsa_compress_v4).  Also, for comparison, the same
    details as separate passes around the plain calls (query prep, entry prep, finalize)."""
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
    kc = bench.kc[0].clone()

    def attn_v4(r):
        L.hsa_attn_decode_v4(q, bench.kc[r], bench.kc[r], m, bench.idx[r].view(B, wl.topk), bench.cnt[r].view(B),
                             bench.k_raw[r], bench.k_raw[r], wl.window, bench.ctx, wl.scale, bench.out[r],
                             bench.lse[r], bench.ws_a, gamma, 1e-6, 64, 10000.0, sink)

    fused = {
        "attn_decode_v4": time_graph(attn_v4, bench.R, steps, reps),
        "compress_v4": time_graph(lambda r: L.hsa_compress_v4(bench.k_raw[r], bench.tb, bench.te, 1, bench.w, m, kc,
                                                              gamma), bench.R, steps, reps),
    }
    unfused = {
        "v4_prep_query": time_graph(lambda r: L.hsa_rmsnorm_rope(q.view(B, 1, H, d), zeros, ones, 1, pos, 1, 0, gamma),
                                    1, steps, reps),
        "v4_prep_entry": time_graph(lambda r: L.hsa_rmsnorm_rope(kc, E_new - 1, E_new, 1, None, m, m - 1, gamma), 1,
                                    steps, reps),
        "v4_finalize": time_graph(lambda r: L.hsa_attn_finalize(out, lse, pos, sink), 1, steps, reps),
    }
    return fused, unfused


def decode_row(wl, bench, t, op_ms, ws):
    """JSON row of one decode workload: rate, bandwidth and roofline fractions."""
    peak, peak_kind = load_peaks()
    ms = t["ms_per_step"]
    by = algorithmic_bytes(wl, bench.ctx_host.tolist(), bench.cnt_total())
    row = {"workload": wl.name, "queries_per_s": wl.B * ws / (ms * 1e-3), "ms_per_step": ms,
           "ms_per_step_median": t["ms_per_step_median"], "replays": t["replays"],
           "algorithmic_bytes_per_step": by["step"], "hbm_gbs_step": by["step"] / (ms * 1e-3) / 1e9,
           "step_frac_of_hbm": by["step"] / (ms * 1e-3) / 1e9 / peak,
           "step_frac_of_hbm_median": by["step"] / (t["ms_per_step_median"] * 1e-3) / 1e9 / peak,
           "peak_gbs": peak, "peak_source": peak_kind, "op_ms": op_ms,
           "l2": f"{bench.R} rotating replicas of every per-step buffer, {bench.R * bench.replica_bytes() / 2**30:.1f} GiB"}
    by["decode_step"] = by["index_topk"] + by["attn_decode"]
    for call in ("index_topk", "attn_decode", "decode_step"):
        if call in op_ms and by[call]:
            ach = by[call] / (op_ms[call] * 1e-3) / 1e9
            row[f"{call}_gbs"] = ach
            row[f"{call}_frac_of_hbm"] = ach / peak
    row["path"] = "hsa_decode_csa (one launch)" if bench.fused else (
        "hsa_index_topk + hsa_attn_decode" if wl.kind == "csa" else "hsa_attn_decode")
    return row


def run_decode(args, ws, rank, local, name, replicas, fused=False):
    dev = torch.device("cuda", local)
    wl = WORKLOADS[name]
    bench = DecodeBench(wl, replicas, 1000 * wl.wid + 100 * rank, dev, fused=fused)
    t = time_decode(bench, args.steps, args.warmup, args.block, ws)
    op_ms = per_call_ms(bench, steps=min(64, max(8, args.block)))
    row = decode_row(wl, bench, t, op_ms, ws)
    return row, bench


def run_hsa(args, ws, rank, local):
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    wl = WORKLOADS[HEADLINE]
    sampler = ClockSampler(local)
    with sampler:
        head, bench = run_decode(args, ws, rank, local, HEADLINE, args.replicas)
    op_ms = head["op_ms"]
    op_ms["compress_append"] = time_state_append(bench)
    v4_fused, v4_unfused = time_v4_details(bench)
    op_ms.update(v4_fused)
    op_ms["attn_decode_shared_kv"] = time_graph(lambda r: bench.attn(r, kv_shared=True), bench.R)
    by = algorithmic_bytes(wl, bench.ctx_host.tolist(), bench.cnt_total())
    peak, peak_kind = load_peaks()
    ms_step = head["ms_per_step"]
    queries = wl.B * ws
    e2e = None if args.profile else run_e2e(bench, args)
    if bench.fused:
        kname, call = "decode_step_kernel", "decode_step"
        kbytes = by["index_topk"] + by["attn_decode"]
        kdesc = "decode_step_kernel (hsa_decode_csa: indexer, top-k and attention; one launch per step)"
    else:
        kname, call, kbytes = "index_fused_kernel", "index_topk", by["index_topk"]
        kdesc = "index_fused_kernel (hsa_index_topk; one launch per step)"
    ach = kbytes / (op_ms[call] * 1e-3) / 1e9
    out = {
        "metric": METRIC, "value": queries / (ms_step * 1e-3), "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16 (int8 indexer, int32 scores, fp32 accumulate)",
        "data": "synthetic (seeded N(0,1) bf16, uniform int8)",
        "config": {"workload": wl.name, "global_batch": wl.B * ws, "seq_len": wl.N,
                   "parallelism": f"replicas x{ws}" if ws > 1 else "one GPU",
                   "l2": head["l2"] + " (> 4x L2: inputs larger than L2, no flush)",
                   "graph_block": args.block},
        "value_median_of_replays": queries / (head["ms_per_step_median"] * 1e-3),
        "ms_per_step_median_of_replays": head["ms_per_step_median"], "replays": head["replays"],
        "hbm_gbs_step": head["hbm_gbs_step"],
        "gpu_launches": len(bench.calls) * args.steps,
        "e2e": e2e,
        "roofline": {"kernel": kdesc, "bound": "hbm",
                     "achieved": ach, "peak": peak, "unit": "GB/s", "frac": ach / peak,
                     "traffic": args.traffic if args.traffic is not None else measured_traffic(kname, HEADLINE),
                     "peak_source": peak_kind, "algorithmic_bytes_per_launch": kbytes,
                     "duration": "mean per-call device time of the step's calls replayed with events between them"},
        "step_roofline": {"bound": "hbm", "achieved": head["hbm_gbs_step"], "peak": peak, "unit": "GB/s",
                          "frac": head["step_frac_of_hbm"], "frac_median_of_replays": head["step_frac_of_hbm_median"],
                          "algorithmic_bytes_per_step": by["step"]},
        "op_ms": op_ms,
        "v4_unfused_ms": v4_unfused,
        "clocks": sampler.summary(),
    }
    del bench
    torch.cuda.empty_cache()
    rows = {}
    # the decode rows through the two calls, and the CSA ones also through the
    # one-launch step (hsa_decode_csa) where its plan fits the shape
    todo = [(name, False) for name in args.decode_rows]
    if not args.profile:
        todo += [(name, True) for name in [HEADLINE] + list(args.decode_rows) if WORKLOADS[name].kind == "csa"]
    for name, fused in todo:
        key = name + ("_one_launch" if fused else "")
        s2 = ClockSampler(local)
        with s2:
            row, b2 = run_decode(args, ws, rank, local, name, args.replicas, fused=fused)
        if fused and not b2.fused:
            rows[key] = {"workload": WORKLOADS[name].name,
                         "unsupported": "hsa_decode_csa: the shape does not fit one resident launch "
                                        "(TMEM-using kernels are resident one CTA per SM)"}
        else:
            row["clocks"] = s2.summary()
            rows[key] = row
        del b2
        torch.cuda.empty_cache()
    out["decode_rows"] = rows
    return out


def run_e2e(bench, args):
    """Same metric through the Python/C-ABI calls with host buffers: each step copies
    its inputs (q, indexer query) from pinned host memory, runs the three calls and
    copies the output back to pinned host memory, every step inside the timed region.

    `value` pipelines the steps over two input slots and three streams: step i's
    inputs are copied in on a copy stream as soon as slot i % 2 is free (step i - 2
    has run), its calls run as one CUDA graph on the compute stream once they have
    landed, its output is copied out on a third stream behind them, and the host
    waits for step i - 2's output before it issues step i (two steps in flight, as a
    serving loop over independent requests would run).  `sync_value` is one graph per
    step (copies, calls, copy back) replayed and waited for before the next step;
    `eager_value` the same step issued call by call and waited for."""
    wl = bench.wl
    R = bench.R
    S = 2  # input slots = steps in flight
    hq = [bench.q[r].cpu().pin_memory() for r in range(R)]
    hqi = [bench.qi[r].cpu().pin_memory() for r in range(R)]
    hout = [torch.empty((wl.B, wl.H, wl.d), dtype=torch.bfloat16).pin_memory() for _ in range(S)]
    dq = [torch.empty_like(bench.q[0]) for _ in range(S)]
    dqi = [torch.empty_like(bench.qi[0]) for _ in range(S)]
    steps = max(20, min(args.steps, 2000))

    def copies_in(r, s):
        dq[s].copy_(hq[r], non_blocking=True)
        dqi[s].copy_(hqi[r], non_blocking=True)

    def compute(r, s, side=None):
        # inputs already in slot s; the compression runs beside the indexer when a
        # second stream is given (the one-launch step reads the compressed cache)
        if bench.fused:
            bench.compress(r)
            bench.decode_step(r, qi=dqi[s], q=dq[s])
            return
        if side is None:
            bench.compress(r)
        else:
            fork, join = torch.cuda.Event(), torch.cuda.Event()
            fork.record()
            side.wait_event(fork)
            with torch.cuda.stream(side):
                bench.compress(r)
            join.record(side)
        bench.index(r, qi=dqi[s])
        if side is not None:
            torch.cuda.current_stream().wait_event(join)
        bench.attn(r, q=dq[s])

    def timed(one):
        for i in range(5):
            one(i)
        torch.cuda.synchronize()
        t = time.perf_counter()
        for i in range(steps):
            one(i)
        torch.cuda.synchronize()
        return (time.perf_counter() - t) / steps

    def eager(i):
        r, s = i % R, 0
        copies_in(r, s)
        compute(r, s)
        hout[s].copy_(bench.out[r], non_blocking=True)
        torch.cuda.current_stream().synchronize()

    dt_eager = timed(eager)

    side = torch.cuda.Stream()
    cap = torch.cuda.Stream()
    cap.wait_stream(torch.cuda.current_stream())
    # one graph per replica of the whole step (copies in, calls, copy out), and one of
    # the calls alone per (replica, slot)
    whole, calls_only = [], {}
    for r in range(R):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cap):
            copies_in(r, 0)
            compute(r, 0, side)
            hout[0].copy_(bench.out[r], non_blocking=True)
        whole.append(g)
        for s in range(S):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=cap):
                compute(r, s, side)
            calls_only[(r, s)] = g
    torch.cuda.current_stream().wait_stream(cap)
    torch.cuda.synchronize()

    def replay(i):
        whole[i % R].replay()
        torch.cuda.current_stream().synchronize()

    dt_sync = timed(replay)

    # Pipelined: graph P[r] runs step r's calls (inputs in slot r % 2) and, beside
    # them on two more streams, copies step r - 1's output out and step r + 1's
    # inputs in (R is even, so replica and slot agree step after step).  Graphs run
    # back to back on one stream; the host waits for graph i - 1 (so for step i - 2's
    # output) after it launches graph i.  The first step's inputs and the last
    # step's output are copied outside the graphs, inside the timed region.
    assert R % S == 0
    s_a, s_b = torch.cuda.Stream(), torch.cuda.Stream()
    piped_g = []
    cap.wait_stream(torch.cuda.current_stream())
    for r in range(R):
        g = torch.cuda.CUDAGraph()
        rp, rn = (r - 1) % R, (r + 1) % R
        with torch.cuda.graph(g, stream=cap):
            fork, j1, j2 = torch.cuda.Event(), torch.cuda.Event(), torch.cuda.Event()
            fork.record()
            s_a.wait_event(fork)
            s_b.wait_event(fork)
            with torch.cuda.stream(s_a):
                hout[rp % S].copy_(bench.out[rp], non_blocking=True)
            j1.record(s_a)
            with torch.cuda.stream(s_b):
                copies_in(rn, rn % S)
            j2.record(s_b)
            compute(r, r % S, side)
            torch.cuda.current_stream().wait_event(j1)
            torch.cuda.current_stream().wait_event(j2)
        piped_g.append(g)
    torch.cuda.current_stream().wait_stream(cap)
    torch.cuda.synchronize()
    done = [torch.cuda.Event() for _ in range(2)]

    def run_piped(n, start):
        copies_in(start % R, start % S)
        for i in range(start, start + n):
            piped_g[i % R].replay()
            done[i % 2].record()
            if i > start:
                done[(i - 1) % 2].synchronize()  # graph i - 1 is done: step i - 2's output is on the host
        last = (start + n - 1) % R
        hout[last % S].copy_(bench.out[last], non_blocking=True)
        torch.cuda.current_stream().synchronize()

    run_piped(8, 0)
    torch.cuda.synchronize()
    t = time.perf_counter()
    run_piped(steps, 0)
    dt = (time.perf_counter() - t) / steps

    h2d = hq[0].numel() * 2 + hqi[0].numel()
    d2h = hout[0].numel() * 2
    return {"value": wl.B / dt, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "ms_per_step": dt * 1e3, "steps": steps,
            "launch": "pipelined: one CUDA graph per step runs its calls and, beside them, copies the previous "
                      "step's output out and the next step's inputs in (2 input slots); graphs back to back on one "
                      "stream, the host waits for graph i-1 after launching graph i",
            "sync_value": wl.B / dt_sync, "sync_ms_per_step": dt_sync * 1e3,
            "sync_launch": "one CUDA graph per step (copies in, calls, copy out), replayed and waited for",
            "eager_value": wl.B / dt_eager, "eager_ms_per_step": dt_eager * 1e3}


# --------------------------------------------------- chunked prefill rows

def prefill_items(wl, rows=None):
    """Attended items per query row (selected or visible entries + window)."""
    p = np.arange(wl.N - wl.T, wl.N, dtype=np.int64)
    if rows is not None:
        p = p[rows]
    E = (p + 1) // wl.m
    sel = np.minimum(E, wl.topk) if wl.kind == "csa" else E
    return sel + np.minimum(wl.window, p + 1)


def prefill_flops(wl, rows=None) -> float:
    """4*H*d FLOP per (query row, attended item): QK^T and PV, multiply-add = 2 FLOP."""
    return 4.0 * wl.B * wl.H * wl.d * float(prefill_items(wl, rows).sum())


def run_prefill(dev, reps: int):
    """Chunked prefill of 8192 new tokens on a 1,048,576-token cache, one HCA and one CSA
    layer.  Each call is timed alone with CUDA events on the launching stream, L2
    flushed (a 256 MiB write) before every run; median of `reps` runs after 2 warm-ups."""
    from compressed_attention_compress_b300 import _lib as L
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    peak_tc = load_peaks(kind="bf16_tflops")

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
        macs = 0.0
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

def oracle_sample_setup():
    """One sequence of the headline workload on the host, its compressed cache built by the oracle."""
    import oracle
    from compressed_attention_compress_b300.inputs import bf16_bits, make_inputs
    oracle.build()
    wl = WORKLOADS[HEADLINE]
    x = make_inputs(wl, B=1)
    m = wl.m
    E = wl.N // m
    kr, vr = bf16_bits(x.k_raw), bf16_bits(x.v_raw)
    kc = oracle.compress(kr, x.w.numpy(), m, [0], [wl.N], E, out_dtype=np.float32)
    vc = oracle.compress(vr, x.w.numpy(), m, [0], [wl.N], E, out_dtype=np.float32)
    return oracle, x, kr, vr, kc, vc


def oracle_query(oracle, x, kr, vr, kc, vc):
    """One decode query through the oracle: compress the new block, index + top-k, attention."""
    from compressed_attention_compress_b300.inputs import bf16_bits
    wl = WORKLOADS[HEADLINE]
    m, N = wl.m, wl.N
    p = N - 1
    newblk = oracle.compress(kr[:, N - m:], x.w.numpy(), m, [0], [m], 1, out_dtype=np.float32)
    kc[:, -1] = newblk[:, 0]
    oi, oc = oracle.index_topk_rows(x.q_idx.numpy().reshape(1, wl.DI), [0], [p], x.k_idx.numpy(), m, wl.topk)
    o, l = oracle.attn_rows(bf16_bits(x.q).reshape(1, wl.H, wl.d), [0], [p], kc, vc, m, oi, kr, vr, wl.window,
                            wl.scale)
    return o


def cpu_baseline(budget_s: float):
    """Time the oracle as it stands on a bounded sample (whole decode queries of sequence 0)."""
    t_setup = time.perf_counter()
    oracle, x, kr, vr, kc, vc = oracle_sample_setup()
    setup = time.perf_counter() - t_setup
    n = 0
    t = time.perf_counter()
    while True:
        oracle_query(oracle, x, kr, vr, kc, vc)
        n += 1
        if time.perf_counter() - t >= budget_s:
            break
    dt = time.perf_counter() - t
    return {"value": n / dt, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"{n} full decode queries of sequence 0 (index over 262144 entries, top-1024, attention over "
                      f"1152 items x 128 heads, new-block compress); {dt:.1f} s timed, cache build {setup:.1f} s untimed",
            "cpu": platform.processor() or platform.machine()}


def cpu_baseline_prefill(budget_s: float):
    """The oracle on a row sample of each chunked-prefill layer: for the CSA layer,
    indexer + top-k + attention of single query rows; for the HCA layer, attention of
    single query rows.  Rows are taken every 512th from the chunk's start, one at a
    time, until `budget_s` per layer; the rate is reported in query rows/s and in the
    attention's TFLOP/s (4*H*d FLOP per attended item)."""
    import oracle
    from compressed_attention_compress_b300.inputs import bf16_bits, make_inputs
    oracle.build()
    res = {}
    for name in ("prefill_hca", "prefill_csa"):
        wl = WORKLOADS[name]
        x = make_inputs(wl)
        m, T, N = wl.m, wl.T, wl.N
        E = N // m
        kr, vr = bf16_bits(x.k_raw), bf16_bits(x.v_raw)
        kc = oracle.compress(kr, x.w.numpy(), m, [0], [N], E, out_dtype=np.float32)
        vc = oracle.compress(vr, x.w.numpy(), m, [0], [N], E, out_dtype=np.float32)
        qb = bf16_bits(x.q.reshape(T, wl.H, wl.d))
        done = []
        t = time.perf_counter()
        for row in range(0, T, 512):
            p = N - T + row
            oi = None
            if wl.kind == "csa":
                oi, _ = oracle.index_topk_rows(x.q_idx.numpy().reshape(T, wl.DI)[row:row + 1], [0], [p],
                                               x.k_idx.numpy(), m, wl.topk)
            oracle.attn_rows(qb[row:row + 1], [0], [p], kc, vc, m, oi, kr, vr, wl.window, wl.scale)
            done.append(row)
            if time.perf_counter() - t >= budget_s:
                break
        dt = time.perf_counter() - t
        flop = prefill_flops(wl, np.array(done))
        res[name] = {"value": len(done) / dt, "unit": "query rows/s", "tflops": flop / dt / 1e12,
                     "cores": oracle.num_threads(), "kind": "oracle",
                     "sample": f"{len(done)} query rows (every 512th of the 8192-token chunk), {dt:.1f} s"}
        del x, kr, vr, kc, vc
    return res


def run_reference(args, ws, rank):
    if rank != 0:
        return None
    oracle, x, kr, vr, kc, vc = oracle_sample_setup()
    for _ in range(min(args.warmup, 3)):
        oracle_query(oracle, x, kr, vr, kc, vc)
    K = args.steps
    wl = WORKLOADS[HEADLINE]
    t = time.perf_counter()
    done = 0
    for _ in range(K):
        oracle_query(oracle, x, kr, vr, kc, vc)
        done += 1
        if time.perf_counter() - t > args.ref_budget:
            break
    dt = time.perf_counter() - t
    value = done / dt
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": done,
            "warmup": args.warmup, "ms_per_step": dt / done * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64 (oracle)", "data": "synthetic",
            "config": {"workload": wl.name, "global_batch": 1, "seq_len": wl.N, "parallelism": "host cores"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
                             "sample": f"{done} of the {K} requested steps, one decode query each (sequence 0); "
                                       f"run bounded to {args.ref_budget:.0f} s"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def run_dry(args, ws, rank):
    """Launcher self-check without a GPU: every rank joins the process group, times a
    trivial host loop, and rank 0 reports the max over ranks (tests the multi-rank
    plumbing of this script on CPU ranks)."""
    barrier(ws)
    t = time.perf_counter()
    acc = 0
    for i in range(args.steps):
        acc += i
    dt = max_over_ranks(time.perf_counter() - t, ws)
    barrier(ws)
    if rank == 0:
        return {"impl": "dry-run", "n_gpus": ws, "steps": args.steps, "seconds_max_over_ranks": dt,
                "world_size": ws}
    return None


def parse(argv):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
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
    ap.add_argument("--decode-rows", default=",".join(EXTRA_DECODE),
                    help="comma-separated extra decode workloads timed beside the headline")
    ap.add_argument("--profile", action="store_true",
                    help="small run for ncu captures: 2 replicas, no end-to-end, CPU or extra legs")
    ap.add_argument("--dry-run", action="store_true", help="launcher self-check on CPU ranks (no GPU work)")
    ap.add_argument("--only", default=None, choices=sorted(k for k in WORKLOADS if "decode" in k),
                    help="time only this decode workload (its row alone, for profiling its kernels)")
    args = ap.parse_args(argv)
    args.decode_rows = [r for r in args.decode_rows.split(",") if r]
    if args.profile:
        args.replicas, args.block, args.no_cpu_baseline = 2, max(1, min(args.block, args.steps)), True
        args.no_prefill, args.decode_rows = True, []
    return args


def main(argv=None):
    argv = sys.argv[1:] if argv is None else argv
    args = parse(argv)
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        spawn_ranks(argv, args.gpus)
        return
    ws, rank, local = dist_setup()
    try:
        if args.dry_run:
            res = run_dry(args, ws, rank)
        elif args.impl == "reference":
            res = run_reference(args, ws, rank)
        elif args.only:
            torch.cuda.set_device(local)
            row, _ = run_decode(args, ws, rank, local, args.only, args.replicas, fused=False)
            res = {"only": args.only, "row": row}
        elif args.prefill_only:
            torch.cuda.set_device(local)
            res = {"prefill": run_prefill(torch.device("cuda", local), args.prefill_reps)}
        else:
            res = run_hsa(args, ws, rank, local)
            torch.cuda.empty_cache()
            if not args.no_prefill:
                res["prefill"] = run_prefill(torch.device("cuda", local), args.prefill_reps)
            if rank == 0 and not args.no_cpu_baseline and ws == 1:
                res["cpu_baseline"] = cpu_baseline(args.cpu_budget)
                res["prefill"] = res.get("prefill") or {}
                res["prefill"]["cpu_baseline"] = cpu_baseline_prefill(args.cpu_budget / 2)
        if rank == 0 and res is not None:
            print(json.dumps(res), flush=True)
    finally:
        if ws > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
