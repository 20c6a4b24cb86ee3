"""Parity of the whole hot path (compress -> index/top-k -> attention) on the
five workloads at their full sizes, in the launch configuration bench.py uses.

Decode workloads are checked on every sequence.  On the 8192-token chunked
prefill every query row's top-k indices and count are checked; outputs and
log-sum-exps on every 16th row plus the first and last 64 rows (644 rows), which
the oracle computes one by one.  Top-k indices and counts must match
bit-exactly, outputs within the bf16 tolerance (max 2e-2, mean 2e-3) of the
fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
from compressed_attention_compress_b300.inputs import WORKLOADS, bf16_bits, make_inputs
from hsa_testlib import assert_close_lse, assert_close_out

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from compressed_attention_compress_b300 import _lib
    return _lib


def _gpu_cache(lib, x, dev):
    wl = x.wl
    B, N, d = x.k_raw.shape
    E = N // wl.m
    kr, vr = x.k_raw.to(dev), x.v_raw.to(dev)
    kc = torch.empty((B, E, d), dtype=kr.dtype, device=dev)
    vc = torch.empty_like(kc)
    lib.hsa_compress(kr, vr, torch.zeros(B, dtype=torch.int64, device=dev), x.ctx_len.to(dev), E, x.w.to(dev), wl.m,
                     kc, vc)
    return kr, vr, kc, vc


def _oracle_cache(x, E, ctx):
    B = x.k_raw.shape[0]
    kc = oracle.compress(bf16_bits(x.k_raw), x.w.numpy(), x.wl.m, [0] * B, ctx, E, out_dtype=np.float32)
    vc = oracle.compress(bf16_bits(x.v_raw), x.w.numpy(), x.wl.m, [0] * B, ctx, E, out_dtype=np.float32)
    return kc, vc


@pytest.mark.parametrize("name", ["flash_csa_decode", "pro_csa_decode", "hca_decode"])
def test_decode_workload(lib, name):
    wl = WORKLOADS[name]
    x = make_inputs(wl)
    dev = torch.device("cuda", 0)
    B, N, H, d, m = wl.B, wl.N, wl.H, wl.d, wl.m
    E = N // m
    kr, vr, kc, vc = _gpu_cache(lib, x, dev)
    ctx = x.ctx_len.to(dev)
    idx = cnt = None
    if wl.kind == "csa":
        idx = torch.empty((B, 1, wl.topk), dtype=torch.int32, device=dev)
        cnt = torch.empty((B, 1), dtype=torch.int32, device=dev)
        ws = lib.workspace(lib.hsa_index_topk_workspace_size(B, 1, wl.DI, E, wl.topk), device=dev)
        lib.hsa_index_topk(x.q_idx.view(B, 1, wl.DI).to(dev), x.k_idx.to(dev), x.q_pos0.to(dev), m, wl.topk, idx,
                           cnt, ws)
    out = torch.empty((B, H, d), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((B, H), dtype=torch.float32, device=dev)
    wsa = lib.workspace(lib.hsa_attn_decode_workspace_size(torch.bfloat16, B, H, d, E, m, wl.topk, wl.window),
                        device=dev)
    lib.hsa_attn_decode(x.q.to(dev), kc, vc, m, None if idx is None else idx.view(B, wl.topk),
                        None if cnt is None else cnt.view(B), kr, vr, wl.window, ctx, wl.scale, out, lse, wsa)
    lib.hsa_check()

    rows_p = (x.ctx_len - 1).numpy()
    oidx = None
    if wl.kind == "csa":
        oidx, ocnt = oracle.index_topk_rows(x.q_idx.numpy(), np.arange(B), rows_p, x.k_idx.numpy(), m, wl.topk)
        assert np.array_equal(cnt.view(B).cpu().numpy(), ocnt)
        assert np.array_equal(idx.view(B, wl.topk).cpu().numpy(), oidx)
    okc, ovc = _oracle_cache(x, E, x.ctx_len.numpy())
    ro, rl = oracle.attn_rows(bf16_bits(x.q), np.arange(B), rows_p, okc, ovc, m, oidx, bf16_bits(x.k_raw),
                              bf16_bits(x.v_raw), wl.window, wl.scale)
    assert_close_out(out, ro, torch.bfloat16)
    assert_close_lse(lse, rl)


@pytest.mark.parametrize("name", ["flash_csa_decode", "pro_csa_decode"])
def test_decode_step_workload(lib, name):
    # the one-launch decode step on the full-size decode workloads
    wl = WORKLOADS[name]
    x = make_inputs(wl)
    dev = torch.device("cuda", 0)
    B, N, H, d, m = wl.B, wl.N, wl.H, wl.d, wl.m
    E = N // m
    kr, vr, kc, vc = _gpu_cache(lib, x, dev)
    idx = torch.empty((B, wl.topk), dtype=torch.int32, device=dev)
    cnt = torch.empty((B,), dtype=torch.int32, device=dev)
    out = torch.empty((B, H, d), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((B, H), dtype=torch.float32, device=dev)
    ws = lib.workspace(lib.hsa_decode_csa_workspace_size(B, H, d, wl.DI, E), device=dev)
    lib.hsa_decode_csa(x.q_idx.to(dev), x.k_idx.to(dev), m, wl.topk, idx, cnt, x.q.to(dev), kc, vc, kr, vr,
                       wl.window, x.ctx_len.to(dev), wl.scale, out, lse, ws)
    lib.hsa_check()
    rows_p = (x.ctx_len - 1).numpy()
    oidx, ocnt = oracle.index_topk_rows(x.q_idx.numpy(), np.arange(B), rows_p, x.k_idx.numpy(), m, wl.topk)
    assert np.array_equal(cnt.cpu().numpy(), ocnt)
    assert np.array_equal(idx.cpu().numpy(), oidx)
    okc, ovc = _oracle_cache(x, E, x.ctx_len.numpy())
    ro, rl = oracle.attn_rows(bf16_bits(x.q), np.arange(B), rows_p, okc, ovc, m, oidx, bf16_bits(x.k_raw),
                              bf16_bits(x.v_raw), wl.window, wl.scale)
    assert_close_out(out, ro, torch.bfloat16)
    assert_close_lse(lse, rl)


def _sample_rows(T):
    """Rows whose outputs are compared on long chunks: every 16th, the first 64 and the last 64."""
    rows = set(range(min(64, T))) | set(range(max(0, T - 64), T)) | set(range(0, T, 16))
    return np.array(sorted(rows), dtype=np.int64)


@pytest.mark.parametrize("name", ["tiny_csa_prefill", "prefill_csa", "prefill_hca"])
def test_prefill_workload(lib, name):
    wl = WORKLOADS[name]
    x = make_inputs(wl)
    dev = torch.device("cuda", 0)
    B, N, H, d, m, T = wl.B, wl.N, wl.H, wl.d, wl.m, wl.T
    E = N // m
    dt = torch.bfloat16 if wl.dtype == "bf16" else torch.float32
    kr, vr, kc, vc = _gpu_cache(lib, x, dev)
    pos0 = x.q_pos0.to(dev)
    idx = cnt = None
    if wl.kind == "csa":
        idx = torch.empty((B, T, wl.topk), dtype=torch.int32, device=dev)
        cnt = torch.empty((B, T), dtype=torch.int32, device=dev)
        ws = lib.workspace(lib.hsa_index_topk_workspace_size(B, T, wl.DI, E, wl.topk), device=dev)
        lib.hsa_index_topk(x.q_idx.to(dev), x.k_idx.to(dev), pos0, m, wl.topk, idx, cnt, ws)
        del ws
    out = torch.empty((B, T, H, d), dtype=dt, device=dev)
    lse = torch.empty((B, T, H), dtype=torch.float32, device=dev)
    wsa = lib.workspace(lib.hsa_attn_prefill_workspace_size(dt, B, T, H, d, E, m, wl.topk, wl.window), device=dev)
    lib.hsa_attn_prefill(x.q.to(dev), kc, vc, m, idx, cnt, kr, vr, wl.window, pos0, wl.scale, out, lse, wsa)
    lib.hsa_check()

    assert B == 1
    rows = _sample_rows(T) if T > 4096 else np.arange(T, dtype=np.int64)
    rows_b = np.zeros(len(rows), np.int64)
    rows_p = int(x.q_pos0[0]) + rows
    oidx = None
    if wl.kind == "csa":
        # every query row's selection, bit-exact
        all_rows = np.arange(T, dtype=np.int64)
        aidx, acnt = oracle.index_topk_rows(x.q_idx.numpy().reshape(B * T, wl.DI), np.zeros(T, np.int64),
                                            int(x.q_pos0[0]) + all_rows, x.k_idx.numpy(), m, wl.topk)
        gcnt = cnt.view(B * T).cpu().numpy()
        gidx = idx.view(B * T, wl.topk).cpu().numpy()
        bad = np.flatnonzero((gcnt != acnt) | (gidx != aidx).any(axis=1))
        assert bad.size == 0, f"{bad.size} of {T} rows differ from the oracle's top-k, first {bad[:8].tolist()}"
        oidx = aidx[rows]
    okc, ovc = _oracle_cache(x, E, x.ctx_len.numpy())
    qr = bf16_bits(x.q.reshape(B * T, H, d))[rows]
    ro, rl = oracle.attn_rows(qr, rows_b, rows_p, okc, ovc, m, oidx, bf16_bits(x.k_raw), bf16_bits(x.v_raw),
                              wl.window, wl.scale)
    assert_close_out(out.view(B * T, H, d)[torch.from_numpy(rows).to(dev)], ro, dt)
    assert_close_lse(lse.view(B * T, H)[torch.from_numpy(rows).to(dev)], rl)
