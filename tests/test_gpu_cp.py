"""GPU parity of the context-parallel exchange kernels (hsa_index_scores,
hsa_topk_merge, hsa_lse_merge) against their definitions, and the CSA and HCA CP
decode steps on the GPU (ranks emulated as threads of one process, per-rank steps
through the C ABI) against the single-GPU path and the oracle."""
import numpy as np
import pytest
import torch

import oracle
from compressed_attention_compress_b300 import cp
from tests.cp_testlib import ThreadGroup
from tests.hsa_testlib import assert_close_lse, assert_close_out, host_np

pytestmark = pytest.mark.gpu
INT32_MIN = -(1 << 31)


@pytest.fixture(scope="module")
def L():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from compressed_attention_compress_b300 import _lib
    oracle.build()
    return _lib


def test_index_scores_exact(L):
    g = torch.Generator().manual_seed(21)
    B, T, E, DI, k = 3, 5, 700, 64, 96
    q = torch.randint(-128, 128, (B, T, DI), generator=g, dtype=torch.int16).to(torch.int8)
    kk = torch.randint(-128, 128, (B, E, DI), generator=g, dtype=torch.int16).to(torch.int8)
    idx = torch.randint(-3, E, (B, T, k), generator=g, dtype=torch.int32)
    cnt = torch.randint(0, k + 1, (B, T), generator=g, dtype=torch.int32)
    sc = torch.empty((B, T, k), dtype=torch.int32, device="cuda")
    L.hsa_index_scores(q.cuda(), kk.cuda(), idx.cuda(), cnt.cuda(), sc)
    qn, kn = q.numpy().astype(np.int64), kk.numpy().astype(np.int64)
    ref = np.full((B, T, k), INT32_MIN, dtype=np.int64)
    for b in range(B):
        for t in range(T):
            for s in range(int(cnt[b, t])):
                j = int(idx[b, t, s])
                if j >= 0:
                    ref[b, t, s] = qn[b, t] @ kn[b, j]
    assert np.array_equal(sc.cpu().numpy().astype(np.int64), ref)


def _merge_ref(scores, idx, topk):
    rows = idx.shape[0]
    out = np.full((rows, topk), -1, dtype=np.int64)
    cnt = np.zeros(rows, dtype=np.int64)
    for r in range(rows):
        pairs = sorted((-int(s), int(j)) for s, j in zip(scores[r], idx[r]) if j >= 0)[:topk]
        sel = sorted(j for _, j in pairs)
        cnt[r] = len(sel)
        out[r, :len(sel)] = sel
    return out, cnt


@pytest.mark.parametrize("rows,n,topk,vals", [(4, 2048, 512, 1 << 20), (3, 4096, 1024, 5), (2, 100, 512, 1 << 30),
                                              (5, 33, 7, 3)])
def test_topk_merge_exact(L, rows, n, topk, vals):
    g = np.random.default_rng(rows * 1000 + n)
    scores = g.integers(-vals, vals, (rows, n)).astype(np.int32)
    if vals >= 1 << 30:
        scores[0, :8] = [INT32_MIN + 1, 2**31 - 1, 0, -1, 1, INT32_MIN + 1, 2**31 - 1, 5]  # extreme keys
    idx = np.full((rows, n), -1, dtype=np.int32)
    for r in range(rows):
        keep = np.sort(g.choice(10 * n, size=int(g.integers(0, n + 1)), replace=False))
        slots = np.sort(g.choice(n, size=len(keep), replace=False))
        idx[r, slots] = keep  # ascending over the non-empty slots, gaps anywhere
    out = torch.empty((rows, topk), dtype=torch.int32, device="cuda")
    cnt = torch.empty((rows,), dtype=torch.int32, device="cuda")
    L.hsa_topk_merge(torch.from_numpy(scores).cuda(), torch.from_numpy(idx).cuda(), topk, out, cnt)
    ro, rc = _merge_ref(scores, idx, topk)
    assert np.array_equal(cnt.cpu().numpy(), rc)
    assert np.array_equal(out.cpu().numpy().astype(np.int64), ro)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_lse_merge(L, dtype):
    g = torch.Generator().manual_seed(7)
    S, rows, H, d = 5, 6, 16, 128
    o = torch.randn((S, rows, H, d), generator=g).to(dtype)
    lse = torch.randn((S, rows, H), generator=g) * 4
    lse[1, 2] = -float("inf")           # an empty part
    lse[:, 3, 5] = -float("inf")        # every part empty for one (row, head)
    out = torch.empty((rows, H, d), dtype=dtype, device="cuda")
    lo = torch.empty((rows, H), dtype=torch.float32, device="cuda")
    L.hsa_lse_merge(o.cuda(), lse.cuda(), out, lo)
    on = o.float().numpy().astype(np.float64)
    ref_o = np.empty((rows, H, d))
    ref_l = np.empty((rows, H))
    for r in range(rows):
        ref_o[r], ref_l[r] = oracle.lse_merge(on[:, r], lse[:, r].numpy().astype(np.float64))
    assert_close_out(out, ref_o, dtype)
    assert_close_lse(lo, ref_l)


@pytest.mark.parametrize("world", [1, 2, 4])
def test_cp_decode_step_device(L, world):
    """Flash-like shape on a 32k-token context: the sharded step selects exactly the
    single-GPU top-k and its output matches the oracle of the unsharded step."""
    B, H, d, m, DI, topk, W = 2, 64, 128, 4, 64, 512, 128
    E_cap = 8192
    N = E_cap * m
    dev = torch.device("cuda")
    g = torch.Generator().manual_seed(40 + world)
    kc = torch.randn((B, E_cap, d), generator=g).to(torch.bfloat16)
    vc = torch.randn((B, E_cap, d), generator=g).to(torch.bfloat16)
    k_raw = torch.randn((B, N, d), generator=g).to(torch.bfloat16)
    v_raw = torch.randn((B, N, d), generator=g).to(torch.bfloat16)
    q = torch.randn((B, H, d), generator=g).to(torch.bfloat16)
    k_idx = torch.randint(-127, 128, (B, E_cap, DI), generator=g, dtype=torch.int16).to(torch.int8)
    q_idx = torch.randint(-127, 128, (B, 1, DI), generator=g, dtype=torch.int16).to(torch.int8)
    ctx = torch.tensor([N, 3 * N // 5 + 3], dtype=torch.int64)
    scale = 1.0 / d ** 0.5

    # single-GPU path on the whole sequence
    idx1 = torch.empty((B, 1, topk), dtype=torch.int32, device=dev)
    cnt1 = torch.empty((B, 1), dtype=torch.int32, device=dev)
    ws = L.workspace(L.hsa_index_topk_workspace_size(B, 1, DI, E_cap, topk))
    L.hsa_index_topk(q_idx.to(dev), k_idx.to(dev), (ctx - 1).to(dev), m, topk, idx1, cnt1, ws)

    def rank_fn(r, ag):
        e0, e1 = cp.shard_bounds(E_cap, world, r)
        sh = cp.Shard(rank=r, world=world, e0=e0, kc=kc[:, e0:e1].contiguous().to(dev),
                      vc=vc[:, e0:e1].contiguous().to(dev), k_idx=k_idx[:, e0:e1].contiguous().to(dev),
                      k_raw=k_raw.to(dev), v_raw=v_raw.to(dev), window_rank=world - 1)
        ops = cp.DeviceOps(B, H, d, DI, e1 - e0, m, topk, W)
        out, lse, sel = cp.cp_decode_step(sh, q.to(dev), q_idx.to(dev), ctx.to(dev), m=m, topk=topk, window=W,
                                          scale=scale, allgather=ag, ops=ops)
        torch.cuda.synchronize()
        return out, lse, sel

    res = ThreadGroup(world).run(rank_fn)
    ref_idx = idx1.view(B, topk).cpu().numpy()
    ro, rl = oracle.attn_rows(host_np(q), np.arange(B), ctx.numpy() - 1, host_np(kc), host_np(vc), m, ref_idx,
                              host_np(k_raw), host_np(v_raw), W, scale)
    for out, lse, sel in res:
        assert np.array_equal(sel.cpu().numpy(), ref_idx)
        assert_close_out(out, ro, torch.bfloat16)
        assert_close_lse(lse, rl)
    L.hsa_check()


@pytest.mark.parametrize("world,E_cap", [(1, 2048), (2, 2048), (4, 2048), (5, 2048), (4, 3)])
def test_cp_decode_step_dense_device(L, world, E_cap):
    """HCA shape (m = 128, 128-token window) on a 256k-token context: each rank's
    attention over all its visible entries, merged, matches the oracle of the
    unsharded dense step (at world 1 a rank's 2,048 entries plus the window exceed
    one tensor-core call, so its list goes in two pieces merged on the rank; with 3
    entries over 4 ranks one rank holds none and attends to the window alone)."""
    B, H, d, m, W = 2, 64, 128, 128, 128
    N = E_cap * m
    dev = torch.device("cuda")
    g = torch.Generator().manual_seed(60 + world)
    kc = torch.randn((B, E_cap, d), generator=g).to(torch.bfloat16)
    vc = torch.randn((B, E_cap, d), generator=g).to(torch.bfloat16)
    k_raw = torch.randn((B, N, d), generator=g).to(torch.bfloat16)
    v_raw = torch.randn((B, N, d), generator=g).to(torch.bfloat16)
    q = torch.randn((B, H, d), generator=g).to(torch.bfloat16)
    ctx = torch.tensor([N, N // 3 + 77], dtype=torch.int64)   # the second stops inside rank 0's or 1's range
    scale = 1.0 / d ** 0.5

    def rank_fn(r, ag):
        e0, e1 = cp.shard_bounds(E_cap, world, r)
        sh = cp.Shard(rank=r, world=world, e0=e0, kc=kc[:, e0:e1].contiguous().to(dev),
                      vc=vc[:, e0:e1].contiguous().to(dev), k_idx=torch.empty(0, dtype=torch.int8, device=dev),
                      k_raw=k_raw.to(dev), v_raw=v_raw.to(dev), window_rank=world - 1)
        ops = cp.DeviceOps(B, H, d, 0, e1 - e0, m, e1 - e0, W)
        out, lse = cp.cp_decode_step_dense(sh, q.to(dev), ctx.to(dev), m=m, window=W, scale=scale,
                                           allgather=ag, ops=ops)
        torch.cuda.synchronize()
        return out, lse

    res = ThreadGroup(world).run(rank_fn)
    ro, rl = oracle.attn_rows(host_np(q), np.arange(B), ctx.numpy() - 1, host_np(kc), host_np(vc), m, None,
                              host_np(k_raw), host_np(v_raw), W, scale)
    for out, lse in res:
        assert_close_out(out, ro, torch.bfloat16)
        assert_close_lse(lse, rl)
    L.hsa_check()


@pytest.mark.parametrize("world", [2, 3])
@pytest.mark.parametrize("csa", [True, False], ids=["csa", "hca"])
def test_cp_prefill_rows_device(L, world, csa):
    """Prefill rows sharded over ranks, cache replicated: each rank's selection is the
    single call's for its rows, bit for bit, and the gathered outputs match it."""
    B, T, H, d, W, DI, topk = 1, 48, 64, 128, 128, 64, 512
    m, E_cap = (4, 8192) if csa else (128, 256)
    N = E_cap * m
    dev = torch.device("cuda")
    g = torch.Generator().manual_seed(70 + world + 10 * csa)
    kc = torch.randn((B, E_cap, d), generator=g).to(torch.bfloat16).to(dev)
    vc = torch.randn((B, E_cap, d), generator=g).to(torch.bfloat16).to(dev)
    k_raw = torch.randn((B, N, d), generator=g).to(torch.bfloat16).to(dev)
    v_raw = torch.randn((B, N, d), generator=g).to(torch.bfloat16).to(dev)
    q = torch.randn((B, T, H, d), generator=g).to(torch.bfloat16).to(dev)
    k_idx = torch.randint(-127, 128, (B, E_cap, DI), generator=g, dtype=torch.int16).to(torch.int8).to(dev)
    q_idx = torch.randint(-127, 128, (B, T, DI), generator=g, dtype=torch.int16).to(torch.int8).to(dev)
    pos0 = torch.tensor([N - T], dtype=torch.int64, device=dev)
    scale = 1.0 / d ** 0.5
    ops = cp.DeviceOps(B, H, d, DI if csa else 0, E_cap, m, topk, W)
    args = (q, q_idx if csa else None, k_idx if csa else None, kc, vc, k_raw, v_raw, pos0)
    kw = dict(m=m, topk=topk, window=W, scale=scale, ops=ops)
    _, ref_o, ref_l, ref_idx = cp.cp_prefill_rows(0, 1, *args, **kw)

    def rank_fn(r, ag):
        res = cp.cp_prefill_rows(r, world, *args, **kw, allgather=ag)
        t0, t1 = cp.row_bounds(T, world, r)
        torch.cuda.synchronize()
        return res, t0, t1

    for (_, out, lse, idx), t0, t1 in ThreadGroup(world).run(rank_fn):
        if csa:
            assert torch.equal(idx, ref_idx[:, t0:t1])
        assert_close_out(out.reshape(B * T, H, d), ref_o.reshape(B * T, H, d).float().cpu().numpy(), torch.bfloat16)
        assert_close_lse(lse.reshape(B * T, H), ref_l.reshape(B * T, H).cpu().numpy())
    L.hsa_check()
