"""V4 attention details on the GPU (Q/KV RMSNorm, partial RoPE, shared K=V entry with
the output's inverse rotation, attention sink): hsa_rmsnorm_rope on the query, the
entries and the window tokens, the unchanged attention kernels with one buffer as
both K and V, then hsa_attn_finalize -- against the oracle's direct definition."""
import numpy as np
import pytest
import torch

import oracle
from tests.hsa_testlib import assert_close_lse, assert_close_out, host_np

pytestmark = pytest.mark.gpu
RD, THETA, EPS = 64, 10000.0, 1e-6


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from compressed_attention_compress_b300 import _lib
    oracle.build()
    return _lib


def _prep(lib, x, n_begin, n_end, max_rows, pos_base, stride, offset, gamma):
    dev = x.device
    lib.hsa_rmsnorm_rope(x, torch.as_tensor(n_begin, dtype=torch.int64, device=dev),
                         torch.as_tensor(n_end, dtype=torch.int64, device=dev), max_rows,
                         None if pos_base is None else torch.as_tensor(pos_base, dtype=torch.int64, device=dev),
                         stride, offset, gamma, EPS, RD, THETA)


def _inputs(seed, B, E_cap, N, H, d):
    g = torch.Generator().manual_seed(seed)
    ent = (torch.randn((B, E_cap, d), generator=g) * 3).to(torch.bfloat16)
    raw = (torch.randn((B, N, d), generator=g) * 2).to(torch.bfloat16)
    gq = torch.rand((d,), generator=g) + 0.5
    gk = torch.rand((d,), generator=g) + 0.5
    sink = torch.randn((H,), generator=g) * 2
    return ent, raw, gq, gk, sink, g


@pytest.mark.parametrize("use_sink,fused,H", [(True, False, 64), (False, False, 64), (True, True, 64),
                                               (False, True, 64), (True, True, 128)])
def test_v4_decode_csa(lib, use_sink, fused, H):
    """fused: the raw query into hsa_attn_decode_v4 (query prep, sink and inverse rotation
    inside the attention kernel); else hsa_rmsnorm_rope, hsa_attn_decode, hsa_attn_finalize"""
    dev = torch.device("cuda")
    B, d, m, W, topk = 2, 128, 4, 128, 256
    E_cap = 2048
    N = E_cap * m
    ent, raw, gq, gk, sink, g = _inputs(31, B, E_cap, N, H, d)
    q = torch.randn((B, H, d), generator=g).to(torch.bfloat16)
    ctx = np.array([N, 5000])
    E = ctx // m
    idx = np.full((B, topk), -1, np.int32)
    for b in range(B):
        idx[b] = np.sort(np.random.default_rng(b).choice(E[b], topk, replace=False))
    scale = 1.0 / d ** 0.5
    qd, entd, rawd = q.to(dev), ent.to(dev), raw.to(dev)
    gqd, gkd = gq.to(dev), gk.to(dev)
    if not fused:
        _prep(lib, qd.view(B, 1, H, d), [0] * B, [1] * B, 1, ctx - 1, 1, 0, gqd)
    _prep(lib, entd, [0] * B, E.tolist(), E_cap, None, m, m - 1, gkd)
    _prep(lib, rawd, np.maximum(ctx - W, 0).tolist(), ctx.tolist(), W, None, 1, 0, gkd)
    out = torch.empty((B, H, d), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((B, H), dtype=torch.float32, device=dev)
    ws = lib.workspace(lib.hsa_attn_decode_workspace_size(torch.bfloat16, B, H, d, E_cap, m, topk, W))
    ctxd = torch.as_tensor(ctx, dtype=torch.int64, device=dev)
    if fused:
        lib.hsa_attn_decode_v4(qd, entd, entd, m, torch.from_numpy(idx).to(dev), None, rawd, rawd, W, ctxd, scale, out,
                               lse, ws, gqd, EPS, RD, THETA, sink.to(dev) if use_sink else None)
        assert torch.equal(qd.cpu(), q)  # the raw query is left as it was
    else:
        lib.hsa_attn_decode(qd, entd, entd, m, torch.from_numpy(idx).to(dev), None, rawd, rawd, W, ctxd, scale, out,
                            lse, ws)
        lib.hsa_attn_finalize(out, lse, ctxd - 1, sink.to(dev) if use_sink else None, RD, THETA)
    lib.hsa_check()
    ro, rl = oracle.attn_v4_rows(host_np(q), np.arange(B), ctx - 1, host_np(ent), m, idx, host_np(raw), W, scale,
                                 gq.double().numpy(), gk.double().numpy(), EPS, RD, THETA,
                                 sink.double().numpy() if use_sink else None)
    assert_close_out(out, ro, torch.bfloat16)
    assert_close_lse(lse, rl)


def test_v4_prefill_hca(lib):
    """dense (HCA) prefill through the tensor-core kernel, with sink and rotation"""
    dev = torch.device("cuda")
    B, T, H, d, m, W = 1, 64, 64, 128, 128, 128
    E_cap = 96
    N = E_cap * m
    ent, raw, gq, gk, sink, g = _inputs(32, B, E_cap, N, H, d)
    q = torch.randn((B, T, H, d), generator=g).to(torch.bfloat16)
    pos0 = np.array([N - T])
    scale = 1.0 / d ** 0.5
    qd, entd, rawd = q.to(dev), ent.to(dev), raw.to(dev)
    gqd, gkd = gq.to(dev), gk.to(dev)
    E_last = (pos0[0] + T) // m
    _prep(lib, qd, [0], [T], T, pos0, 1, 0, gqd)
    _prep(lib, entd, [0], [E_last], E_cap, None, m, m - 1, gkd)
    _prep(lib, rawd, [max(0, pos0[0] - W + 1)], [pos0[0] + T], W + T, None, 1, 0, gkd)
    out = torch.empty((B, T, H, d), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((B, T, H), dtype=torch.float32, device=dev)
    p0 = torch.as_tensor(pos0, dtype=torch.int64, device=dev)
    lib.hsa_attn_prefill(qd, entd, entd, m, None, None, rawd, rawd, W, p0, scale, out, lse)
    lib.hsa_attn_finalize(out, lse, p0, sink.to(dev), RD, THETA)
    lib.hsa_check()
    rows_p = pos0[0] + np.arange(T)
    ro, rl = oracle.attn_v4_rows(host_np(q.view(T, H, d)), np.zeros(T, np.int64), rows_p, host_np(ent), m, None,
                                 host_np(raw), W, scale, gq.double().numpy(), gk.double().numpy(), EPS, RD, THETA,
                                 sink.double().numpy())
    assert_close_out(out.view(T, H, d), ro, torch.bfloat16)
    assert_close_lse(lse.view(T, H), rl)


def test_rmsnorm_rope_matches_definition(lib):
    """the prepared vectors themselves: fp32 storage, rotation at large positions"""
    dev = torch.device("cuda")
    B, n, H, d = 2, 5, 3, 128
    g = torch.Generator().manual_seed(33)
    x = torch.randn((B, n, H, d), generator=g, dtype=torch.float32)
    gam = torch.rand((d,), generator=g) + 0.5
    base = np.array([1_000_003, 17])
    xd = x.to(dev)
    _prep(lib, xd, [1, 0], [4, 5], 5, base, 7, 2, gam.to(dev))
    got = xd.cpu().double().numpy()
    want = x.double().numpy().copy()
    for b in range(B):
        for r in range(1 if b == 0 else 0, 4 if b == 0 else 5):
            pos = base[b] + r * 7 + 2
            for h in range(H):
                v = x[b, r, h].double().numpy()
                v = v / np.sqrt((v * v).mean() + EPS) * gam.double().numpy()
                k = np.arange(RD // 2)
                ang = pos * THETA ** (-2.0 * k / RD)
                z = (v[d - RD::2] + 1j * v[d - RD + 1::2]) * np.exp(1j * ang)
                v[d - RD::2], v[d - RD + 1::2] = z.real, z.imag
                want[b, r, h] = v
    np.testing.assert_allclose(got, want, atol=2e-5, rtol=1e-5)


def test_v4_decode_from_raw_tokens(lib):
    """the V4 decode path with each preparation inside a kernel that writes or reads the
    vectors: entries compressed and prepared as they are written (hsa_compress_v4), the raw
    query into hsa_attn_decode_v4 (query prep, sink, inverse rotation inside), window tokens
    prepared when they are written -- against the oracle on the raw tokens"""
    dev = torch.device("cuda")
    B, H, d, m, W, topk = 2, 128, 128, 4, 128, 256
    E_cap = 2048
    N = E_cap * m
    _, raw, gq, gk, sink, g = _inputs(33, B, E_cap, N, H, d)
    w = torch.rand((m,), generator=g, dtype=torch.float64) + 0.1
    w = (w / w.sum()).float()
    q = torch.randn((B, H, d), generator=g).to(torch.bfloat16)
    ctx = np.array([N, 5001])
    E = ctx // m
    idx = np.full((B, topk), -1, np.int32)
    for b in range(B):
        idx[b] = np.sort(np.random.default_rng(40 + b).choice(E[b], topk, replace=False))
    scale = 1.0 / d ** 0.5
    rawd = raw.to(dev)
    gqd, gkd, wd = gq.to(dev), gk.to(dev), w.to(dev)
    tb = torch.zeros(B, dtype=torch.int64, device=dev)
    te = torch.as_tensor(ctx, dtype=torch.int64, device=dev)
    kc = torch.zeros((B, E_cap, d), dtype=torch.bfloat16, device=dev)
    lib.hsa_compress_v4(rawd, tb, te, E_cap, wd, m, kc, gkd, EPS, RD, THETA)
    # the same entries by hsa_compress, then hsa_rmsnorm_rope: equal up to the rounding
    # of the intermediate entry
    kc2 = torch.zeros_like(kc)
    lib.hsa_compress(rawd, rawd, tb, te, E_cap, wd, m, kc2, kc2.clone())
    _prep(lib, kc2, [0] * B, E.tolist(), E_cap, None, m, m - 1, gkd)
    torch.testing.assert_close(kc.float(), kc2.float(), rtol=2 ** -6, atol=2e-2)
    rawp = rawd.clone()
    _prep(lib, rawp, np.maximum(ctx - W, 0).tolist(), ctx.tolist(), W, None, 1, 0, gkd)
    qd = q.to(dev)
    out = torch.empty((B, H, d), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((B, H), dtype=torch.float32, device=dev)
    ws = lib.workspace(lib.hsa_attn_decode_workspace_size(torch.bfloat16, B, H, d, E_cap, m, topk, W))
    ctxd = torch.as_tensor(ctx, dtype=torch.int64, device=dev)
    lib.hsa_attn_decode_v4(qd, kc, kc, m, torch.from_numpy(idx).to(dev), None, rawp, rawp, W, ctxd, scale, out, lse,
                           ws, gqd, EPS, RD, THETA, sink.to(dev))
    lib.hsa_check()
    ent = oracle.compress(host_np(raw), w.numpy(), m, [0] * B, ctx.tolist(), E_cap)
    ro, rl = oracle.attn_v4_rows(host_np(q), np.arange(B), ctx - 1, ent, m, idx, host_np(raw), W, scale,
                                 gq.double().numpy(), gk.double().numpy(), EPS, RD, THETA, sink.double().numpy())
    assert_close_out(out, ro, torch.bfloat16)
    assert_close_lse(lse, rl)
