"""Shared helpers of the parity tests: run the CUDA path and the oracle on the
same seeded inputs.  The CUDA path is reached only through the C-ABI binding;
the oracle only through ``oracle``.  Neither sees the other's results."""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle
from compressed_attention_compress_b300.inputs import bf16_bits

# spec tolerance for bf16 outputs against the fp64 oracle
BF16_MAX_ABS, BF16_MEAN_ABS = 2e-2, 2e-3
# fp32 storage: the fp32 kernels accumulate in fp32 over at most a few thousand terms
F32_MAX_ABS, F32_MEAN_ABS = 1e-4, 1e-5
LSE_ABS = 2e-2


def host_np(t: torch.Tensor):
    """CPU tensor -> numpy array the oracle reads exactly (bf16 as raw bits)."""
    return bf16_bits(t.cpu())


def assert_close_out(gpu, ref, dtype, what="out"):
    g = gpu.float().cpu().numpy().astype(np.float64)
    err = np.abs(g - ref)
    mx, mean = float(err.max(initial=0.0)), float(err.mean()) if err.size else 0.0
    if dtype == torch.bfloat16:
        assert mx <= BF16_MAX_ABS and mean <= BF16_MEAN_ABS, f"{what}: max {mx:.3g} mean {mean:.3g}"
    else:
        assert mx <= F32_MAX_ABS and mean <= F32_MEAN_ABS, f"{what}: max {mx:.3g} mean {mean:.3g}"
    return mx, mean


def assert_close_lse(gpu, ref):
    g = gpu.cpu().numpy().astype(np.float64)
    both_inf = np.isneginf(g) & np.isneginf(ref)
    assert (np.isneginf(g) == np.isneginf(ref)).all(), "lse -inf pattern differs"
    err = np.abs(np.where(both_inf, 0.0, np.where(both_inf, 0.0, g) - np.where(both_inf, 0.0, ref)))
    assert float(err.max(initial=0.0)) <= LSE_ABS, f"lse max err {float(err.max()):.3g}"


def gpu_compress(k_raw, v_raw, w, m, tok_begin, tok_end, E_cap, lib):
    """Compress on the GPU; k_raw/v_raw device [B, N, d]."""
    B, N, d = k_raw.shape
    kc = torch.zeros((B, E_cap, d), dtype=k_raw.dtype, device=k_raw.device)
    vc = torch.zeros_like(kc)
    tb = torch.as_tensor(tok_begin, dtype=torch.int64).to(k_raw.device)
    te = torch.as_tensor(tok_end, dtype=torch.int64).to(k_raw.device)
    max_blocks = int(max(int(e) // m - int(b) // m for b, e in zip(tok_begin, tok_end))) if B else 0
    lib.hsa_compress(k_raw, v_raw, tb, te, max(max_blocks, 0), w.to(k_raw.device), m, kc, vc)
    return kc, vc


def gpu_index(q_idx, k_idx, q_pos0, m, topk, lib):
    """q_idx device [B, T, DI]; returns (idx [B,T,topk], cnt [B,T]) on device."""
    B, T, DI = q_idx.shape
    E_cap = k_idx.shape[1]
    idx = torch.empty((B, T, topk), dtype=torch.int32, device=q_idx.device)
    cnt = torch.empty((B, T), dtype=torch.int32, device=q_idx.device)
    ws = lib.workspace(lib.hsa_index_topk_workspace_size(B, T, DI, E_cap, topk), device=q_idx.device)
    for _ in range(2):  # twice on one workspace: each call must leave it ready for the next
        lib.hsa_index_topk(q_idx, k_idx, q_pos0.to(q_idx.device), m, topk, idx, cnt, ws)
    return idx, cnt


def oracle_index_rows(q_idx_np, k_idx_np, rows_b, rows_p, m, topk):
    return oracle.index_topk_rows(q_idx_np, rows_b, rows_p, k_idx_np, m, topk)


def scale_of(d):
    return 1.0 / math.sqrt(d)
