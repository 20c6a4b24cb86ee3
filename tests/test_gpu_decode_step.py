"""hsa_decode_csa (the CSA decode step in one launch) against the oracle and
against the two-call path (hsa_index_topk + hsa_attn_decode): the selection must
match bit-exactly, outputs and log-sum-exps within the bf16 tolerance."""
import numpy as np
import pytest
import torch

import oracle
from hsa_testlib import assert_close_lse, assert_close_out, host_np, scale_of

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from compressed_attention_compress_b300 import _lib
    return _lib


def _randn(shape, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(shape, generator=g).to(torch.bfloat16)


def _randint8(shape, seed, lo=-127, hi=127):
    g = torch.Generator().manual_seed(seed)
    return torch.randint(lo, hi + 1, shape, generator=g, dtype=torch.int16).to(torch.int8)


def _case(lib, B, H, DI, topk, ctx, m=4, W=128, seed=0, lo=-127, hi=127, shared_kv=False, k_idx=None):
    d = 128
    N = max(ctx) + 5
    E_cap = N // m
    kc, vc = _randn((B, E_cap, d), seed + 1), _randn((B, E_cap, d), seed + 2)
    kr, vr = _randn((B, N, d), seed + 3), _randn((B, N, d), seed + 4)
    if shared_kv:
        vc, vr = kc, kr
    q = _randn((B, H, d), seed + 5)
    qi = _randint8((B, DI), seed + 6, lo, hi)
    ki = _randint8((B, E_cap, DI), seed + 7, lo, hi) if k_idx is None else k_idx
    dev = "cuda"
    g = {n: t.to(dev) for n, t in dict(kc=kc, vc=vc, kr=kr, vr=vr, q=q, qi=qi, ki=ki).items()}
    if shared_kv:
        g["vc"], g["vr"] = g["kc"], g["kr"]
    ctx_d = torch.tensor(ctx, dtype=torch.int64, device=dev)
    idx = torch.empty((B, topk), dtype=torch.int32, device=dev)
    cnt = torch.empty((B,), dtype=torch.int32, device=dev)
    out = torch.empty((B, H, d), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((B, H), dtype=torch.float32, device=dev)
    ws = lib.workspace(lib.hsa_decode_csa_workspace_size(B, H, d, DI, E_cap), device=dev)
    for _ in range(2):  # twice: the workspace must be left ready for the next call
        lib.hsa_decode_csa(g["qi"], g["ki"], m, topk, idx, cnt, g["q"], g["kc"], g["vc"], g["kr"], g["vr"], W, ctx_d,
                           scale_of(d), out, lse, ws)
    lib.hsa_check()
    rows_p = np.asarray(ctx) - 1
    oidx, ocnt = oracle.index_topk_rows(qi.numpy(), np.arange(B), rows_p, ki.numpy(), m, topk)
    assert np.array_equal(cnt.cpu().numpy(), ocnt)
    assert np.array_equal(idx.cpu().numpy(), oidx)
    ro, rl = oracle.attn_rows(host_np(q), np.arange(B), rows_p, host_np(kc), host_np(vc), m, oidx, host_np(kr),
                              host_np(vr), W, scale_of(d))
    assert_close_out(out, ro, torch.bfloat16)
    assert_close_lse(lse, rl)
    # the two-call path selects the same entries
    idx2 = torch.empty((B, 1, topk), dtype=torch.int32, device=dev)
    cnt2 = torch.empty((B, 1), dtype=torch.int32, device=dev)
    wsi = lib.workspace(lib.hsa_index_topk_workspace_size(B, 1, DI, E_cap, topk), device=dev)
    lib.hsa_index_topk(g["qi"].view(B, 1, DI), g["ki"], ctx_d - 1, m, topk, idx2, cnt2, wsi)
    assert torch.equal(idx2.view(B, topk), idx) and torch.equal(cnt2.view(B), cnt)


@pytest.mark.parametrize("H", [64, 128])
def test_decode_step_basic(lib, H):
    # long, medium and short sequences (E < topk), window partly before position 0
    _case(lib, B=3, H=H, DI=64, topk=256, ctx=[4 * 3000 + 2, 4 * 700, 130], seed=10)


def test_decode_step_no_entries_and_no_window(lib):
    _case(lib, B=2, H=128, DI=64, topk=64, ctx=[3, 4 * 900 + 1], seed=20)
    _case(lib, B=2, H=64, DI=64, topk=64, ctx=[4 * 900 + 1, 4 * 300], W=0, seed=21)


@pytest.mark.parametrize("DI", [32, 128])
def test_decode_step_indexer_dims(lib, DI):
    _case(lib, B=2, H=128, DI=DI, topk=512, ctx=[4 * 5000, 4 * 2500 + 3], seed=30 + DI)


def test_decode_step_heavy_ties(lib):
    # scores in a few values: the threshold bin holds thousands of keys
    _case(lib, B=2, H=64, DI=64, topk=512, ctx=[4 * 6000, 4 * 3000], lo=-1, hi=1, seed=40)


def test_decode_step_all_equal_keys(lib):
    # every score equal: the first topk entries by index
    B, DI, ctx = 2, 64, [4 * 4000, 4 * 1000]
    ki = torch.zeros((B, (max(ctx) + 5) // 4, DI), dtype=torch.int8)
    _case(lib, B=B, H=128, DI=DI, topk=300, ctx=ctx, seed=50, k_idx=ki)


def test_decode_step_shared_kv(lib):
    _case(lib, B=2, H=128, DI=64, topk=128, ctx=[4 * 2000, 4 * 1000 + 1], seed=60, shared_kv=True)
