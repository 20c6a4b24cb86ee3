"""Seeded synthetic inputs for the five hybrid-attention workloads.

This module only draws random numbers and states shapes; it holds none of the
method's arithmetic.  Both the CUDA path (through the tests and the benchmark)
and the CPU oracle receive exactly these tensors.

Recipe (every tensor is drawn on the CPU with its own ``torch.Generator``
seeded ``1000 * workload_id + tensor_id``):

* q, raw K, raw V ~ N(0, 1) in fp32, then rounded to bf16 (kept fp32 for the
  fp32 workload);
* indexer vectors: integers uniform in [-127, 127], stored as int8;
* block weights: w_raw ~ U(0, 1], w = w_raw / sum(w_raw) in fp64, stored fp32;
* HCA decode context lengths: uniform integers in [262144, 1048576].

The shapes follow the pages' model configurations (V4-Flash: top-k 512, V4-Pro:
top-k 1024, 128-token window, CSA m = 4, HCA m = 128), as fixed for this
library; no public dataset is involved.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch

T_Q, T_K, T_V, T_QI, T_KI, T_W, T_LEN = 1, 2, 3, 4, 5, 6, 7


@dataclasses.dataclass(frozen=True)
class Workload:
    """One synthetic workload: shapes, dtype and the layer kind."""
    wid: int            # workload id (seed base)
    name: str
    kind: str           # "csa" or "hca"
    phase: str          # "decode" or "prefill"
    B: int
    N: int              # cached tokens per sequence (decode: includes the new token)
    H: int
    d: int
    m: int
    window: int
    topk: int = 0       # CSA only
    DI: int = 0         # CSA only
    T: int = 1          # query tokens per sequence (prefill); decode has 1
    dtype: str = "bf16"  # "bf16" or "f32"
    len_lo: int = 0     # HCA decode: per-sequence length range (inclusive)
    len_hi: int = 0

    @property
    def E_cap(self) -> int:
        return self.N // self.m

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)


def _tiny_csa_prefill() -> Workload:
    return Workload(1, "tiny CSA prefill, fp32, N=4096 H=8 d=64 m=4 k=64 W=128",
                    "csa", "prefill", B=1, N=4096, H=8, d=64, m=4, window=128, topk=64, DI=32,
                    T=4096, dtype="f32")


def _flash_csa_decode() -> Workload:
    return Workload(2, "V4-Flash-shaped CSA decode, B=8 ctx=131072 H=64 d=128 m=4 k=512 W=128",
                    "csa", "decode", B=8, N=131072, H=64, d=128, m=4, window=128, topk=512, DI=64)


def _pro_csa_decode() -> Workload:
    return Workload(3, "V4-Pro-shaped CSA decode at 1M ctx, B=4 ctx=1048576 H=128 d=128 m=4 k=1024 W=128",
                    "csa", "decode", B=4, N=1048576, H=128, d=128, m=4, window=128, topk=1024, DI=64)


def _hca_decode() -> Workload:
    return Workload(4, "HCA decode, B=16 ctx~U[262144,1048576] H=64 d=128 m=128 W=128",
                    "hca", "decode", B=16, N=1048576, H=64, d=128, m=128, window=128,
                    len_lo=262144, len_hi=1048576)


def _prefill_csa() -> Workload:
    return Workload(5, "chunked prefill CSA layer: 8192 tokens on a 1048576-token cache, H=64 d=128 m=4 k=1024 W=128",
                    "csa", "prefill", B=1, N=1048576 + 8192, H=64, d=128, m=4, window=128, topk=1024,
                    DI=64, T=8192)


def _prefill_hca() -> Workload:
    return Workload(15, "chunked prefill HCA layer: 8192 tokens on a 1048576-token cache, H=64 d=128 m=128 W=128",
                    "hca", "prefill", B=1, N=1048576 + 8192, H=64, d=128, m=128, window=128, T=8192)


WORKLOADS = {
    "tiny_csa_prefill": _tiny_csa_prefill(),
    "flash_csa_decode": _flash_csa_decode(),
    "pro_csa_decode": _pro_csa_decode(),
    "hca_decode": _hca_decode(),
    "prefill_csa": _prefill_csa(),
    "prefill_hca": _prefill_hca(),
}


def gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return g


def normal_bf16(shape, seed: int, dtype: str = "bf16", chunk_rows: int = 1 << 22) -> torch.Tensor:
    """N(0,1) drawn in fp32 then rounded (RNE) to bf16, or kept fp32.

    Drawn in slabs along the first axes to bound host memory for 1M-token caches.
    """
    g = gen(seed)
    out_dtype = torch.bfloat16 if dtype == "bf16" else torch.float32
    numel = math.prod(shape)
    last = shape[-1]
    rows = numel // last
    out = torch.empty((rows, last), dtype=out_dtype)
    for r0 in range(0, rows, chunk_rows):
        r1 = min(rows, r0 + chunk_rows)
        out[r0:r1] = torch.randn((r1 - r0, last), generator=g, dtype=torch.float32).to(out_dtype)
    return out.view(*shape)


def uniform_int8(shape, seed: int, lo: int = -127, hi: int = 127) -> torch.Tensor:
    g = gen(seed)
    return torch.randint(lo, hi + 1, shape, generator=g, dtype=torch.int16).to(torch.int8)


def block_weights(m: int, seed: int) -> torch.Tensor:
    """w_raw ~ U(0,1], normalised in fp64, stored fp32 (|sum(w) - 1| < 1e-6)."""
    g = gen(seed)
    w_raw = 1.0 - torch.rand((m,), generator=g, dtype=torch.float64)
    w = (w_raw / w_raw.sum()).to(torch.float32)
    assert abs(float(w.double().sum()) - 1.0) < 1e-6
    return w


def context_lengths(B: int, lo: int, hi: int, seed: int) -> torch.Tensor:
    g = gen(seed)
    return torch.randint(lo, hi + 1, (B,), generator=g, dtype=torch.int64)


@dataclasses.dataclass
class Inputs:
    """Host tensors for one workload (CPU, pinned-able)."""
    wl: Workload
    q: torch.Tensor               # decode [B, H, d]; prefill [B, T, H, d]
    k_raw: torch.Tensor           # [B, N, d]
    v_raw: torch.Tensor           # [B, N, d]
    w: torch.Tensor               # [m] fp32
    ctx_len: torch.Tensor         # [B] int64 (decode: query position = ctx_len - 1)
    q_pos0: torch.Tensor          # [B] int64 (prefill: first query position)
    q_idx: Optional[torch.Tensor] = None  # decode [B, DI]; prefill [B, T, DI] int8
    k_idx: Optional[torch.Tensor] = None  # [B, E_cap, DI] int8


def make_inputs(wl: Workload, N: Optional[int] = None, B: Optional[int] = None,
                T: Optional[int] = None, seed_offset: int = 0) -> Inputs:
    """Draw one workload's inputs; N, B, T override the sizes (for reduced cases)."""
    N = wl.N if N is None else N
    B = wl.B if B is None else B
    T = wl.T if T is None else T
    base = 1000 * wl.wid + seed_offset
    if wl.phase == "decode":
        q = normal_bf16((B, wl.H, wl.d), base + T_Q, wl.dtype)
        if wl.len_hi:
            lo, hi = min(wl.len_lo, N), min(wl.len_hi, N)
            ctx = context_lengths(B, lo, hi, base + T_LEN)
        else:
            ctx = torch.full((B,), N, dtype=torch.int64)
        q_pos0 = ctx - 1
    else:
        q = normal_bf16((B, T, wl.H, wl.d), base + T_Q, wl.dtype)
        ctx = torch.full((B,), N, dtype=torch.int64)
        q_pos0 = torch.full((B,), N - T, dtype=torch.int64)
    k_raw = normal_bf16((B, N, wl.d), base + T_K, wl.dtype)
    v_raw = normal_bf16((B, N, wl.d), base + T_V, wl.dtype)
    w = block_weights(wl.m, base + T_W)
    q_idx = k_idx = None
    if wl.kind == "csa":
        E_cap = N // wl.m
        qshape = (B, wl.DI) if wl.phase == "decode" else (B, T, wl.DI)
        q_idx = uniform_int8(qshape, base + T_QI)
        k_idx = uniform_int8((B, E_cap, wl.DI), base + T_KI)
    return Inputs(wl, q, k_raw, v_raw, w, ctx, q_pos0, q_idx, k_idx)


def bf16_bits(t: torch.Tensor):
    """A bf16 (or fp32) CPU tensor as a numpy array the oracle reads exactly."""
    t = t.contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view("uint16")
    return t.numpy()
