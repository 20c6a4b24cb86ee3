"""Context-parallel exchange of one long sequence (entry sharding across ranks):
the protocols of cp.cp_decode_step (CSA) and cp.cp_decode_step_dense (HCA) run by
2 gloo ranks in separate processes and by 1-4 ranks emulated as threads, with the
per-rank steps computed by the oracle, against the single-process oracle of the
same decode step."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

import oracle
from compressed_attention_compress_b300 import cp
from tests.cp_testlib import (OracleOps, PrefillOracleOps, ThreadGroup, cp_case, full_reference,
                              full_reference_dense, prefill_case)

M, H, D, DI, TOPK, W = 4, 4, 16, 32, 8, 8
M_HCA = 16          # HCA-layer block size of the dense cases (the window W < M_HCA)
SCALE = 1.0 / np.sqrt(D)


def _shard(x, world, rank, E_cap, window_rank):
    e0, e1 = cp.shard_bounds(E_cap, world, rank)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a))
    return cp.Shard(rank=rank, world=world, e0=e0, kc=t(x["kc"][:, e0:e1]), vc=t(x["vc"][:, e0:e1]),
                    k_idx=t(x["k_idx"][:, e0:e1]), k_raw=t(x["k_raw"]), v_raw=t(x["v_raw"]), window_rank=window_rank)


def _run_rank(rank, world, x, E_cap, ctx, allgather, window_rank):
    sh = _shard(x, world, rank, E_cap, window_rank)
    ops = OracleOps(sh.e0, E_cap)
    return cp.cp_decode_step(sh, torch.from_numpy(x["q"]), torch.from_numpy(x["q_idx"]),
                             torch.tensor(ctx, dtype=torch.int64), m=M, topk=TOPK, window=W, scale=SCALE,
                             allgather=allgather, ops=ops)


def _run_rank_dense(rank, world, x, E_cap, ctx, allgather, window_rank):
    sh = _shard(x, world, rank, E_cap, window_rank)
    ops = OracleOps(sh.e0, E_cap)
    return cp.cp_decode_step_dense(sh, torch.from_numpy(x["q"]), torch.tensor(ctx, dtype=torch.int64), m=M_HCA,
                                   window=W, scale=SCALE, allgather=allgather, ops=ops)


def _check_dense(res, x, ctx):
    ref_o, ref_l = full_reference_dense(x, ctx, M_HCA, W, SCALE)
    for out, lse in res:
        np.testing.assert_allclose(out.numpy(), ref_o, atol=1e-10, rtol=0)
        np.testing.assert_allclose(lse.numpy(), ref_l, atol=1e-10, rtol=0)


def _check(res, x, ctx):
    ref_idx, ref_o, ref_l = full_reference(x, ctx, M, TOPK, W, SCALE)
    for out, lse, sel in res:
        assert np.array_equal(sel.numpy(), ref_idx), (sel, ref_idx)
        np.testing.assert_allclose(out.numpy(), ref_o, atol=1e-10, rtol=0)
        np.testing.assert_allclose(lse.numpy(), ref_l, atol=1e-10, rtol=0)


CASES = [
    # (seed, B, E_cap, ctx_len per sequence, ties)
    (11, 2, 64, [256, 256], False),       # every entry visible
    (12, 2, 64, [81, 256], False),        # sequence 0: rank 1's entries are not visible yet
    (13, 3, 64, [256, 130, 7], True),     # heavy ties (3 distinct indexer values); a sequence with one entry
]


DENSE_CASES = [
    # (seed, B, E_cap, ctx_len per sequence)
    (21, 2, 24, [384, 384]),              # every entry visible
    (22, 3, 24, [200, 384, 15]),          # rank 1's entries not visible for sequence 0; no entry at all for 2
    (23, 1, 5, [75]),                     # 5 entries: ragged shards, an empty one on 4 ranks; a partial block
]


PREFILL_CASES = [
    # (seed, B, T, E_cap, q_pos0 per sequence, csa)
    (31, 2, 13, 40, [147, 20], True),     # CSA: index and attention per row; sequence 1 starts with few entries
    (32, 1, 5, 40, [100], False),         # HCA; 5 rows over up to 4 ranks
    (33, 1, 2, 40, [60], True),           # fewer rows than ranks: some ranks have none
]


def _prefill_run(rank, world, x, pos0, csa, allgather):
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a))
    return cp.cp_prefill_rows(rank, world, t(x["q"]), t(x["q_idx"]) if csa else None, t(x["k_idx"]) if csa else None,
                              t(x["kc"]), t(x["vc"]), t(x["k_raw"]), t(x["v_raw"]),
                              torch.tensor(pos0, dtype=torch.int64), m=M, topk=TOPK, window=W, scale=SCALE,
                              ops=PrefillOracleOps(), allgather=allgather)


def _prefill_check(res, x, pos0, csa):
    ops = PrefillOracleOps()
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a))
    pos = torch.tensor(pos0, dtype=torch.int64)
    idx = cnt = None
    if csa:
        idx, cnt = ops.index_topk_rows(t(x["q_idx"]), t(x["k_idx"]), pos, M, TOPK)
    ro, rl = ops.attn_prefill(t(x["q"]), t(x["kc"]), t(x["vc"]), M, idx, cnt, t(x["k_raw"]), t(x["v_raw"]), W, pos,
                              SCALE)
    for t0, out, lse, _ in res:
        assert t0 == 0
        np.testing.assert_array_equal(out.numpy(), ro.numpy())
        np.testing.assert_array_equal(lse.numpy(), rl.numpy())


def _gloo_worker(rank, world, port, case, dense=False, prefill=False):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        oracle.build()
        if prefill:
            seed, B, T, E_cap, pos0, csa = case
            x = prefill_case(seed, B, T, E_cap, M, H, D, DI)
            _prefill_check([_prefill_run(rank, world, x, pos0, csa, cp.torch_allgather())], x, pos0, csa)
            return
        if dense:
            seed, B, E_cap, ctx = case
            x = cp_case(seed, B, E_cap, M_HCA, H, D, DI)
            res = _run_rank_dense(rank, world, x, E_cap, ctx, cp.torch_allgather(), window_rank=world - 1)
            _check_dense([res], x, ctx)
            return
        seed, B, E_cap, ctx, ties = case
        x = cp_case(seed, B, E_cap, M, H, D, DI, ties)
        res = _run_rank(rank, world, x, E_cap, ctx, cp.torch_allgather(), window_rank=world - 1)
        _check([res], x, ctx)
    finally:
        dist.destroy_process_group()


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


@pytest.mark.parametrize("case", CASES, ids=["full", "short", "ties"])
def test_cp_gloo_two_ranks(case):
    oracle.build()
    mp.spawn(_gloo_worker, args=(2, _free_port(), case), nprocs=2, join=True)


@pytest.mark.parametrize("world", [1, 3, 4])
@pytest.mark.parametrize("case", CASES, ids=["full", "short", "ties"])
def test_cp_thread_ranks(case, world):
    oracle.build()
    seed, B, E_cap, ctx, ties = case
    x = cp_case(seed, B, E_cap, M, H, D, DI, ties)
    tg = ThreadGroup(world)
    res = tg.run(lambda r, ag: _run_rank(r, world, x, E_cap, ctx, ag, window_rank=0))
    _check(res, x, ctx)


@pytest.mark.parametrize("case", DENSE_CASES, ids=["full", "short", "ragged"])
def test_cp_dense_gloo_two_ranks(case):
    oracle.build()
    mp.spawn(_gloo_worker, args=(2, _free_port(), case, True), nprocs=2, join=True)


@pytest.mark.parametrize("world", [1, 3, 4])
@pytest.mark.parametrize("case", DENSE_CASES, ids=["full", "short", "ragged"])
def test_cp_dense_thread_ranks(case, world):
    oracle.build()
    seed, B, E_cap, ctx = case
    x = cp_case(seed, B, E_cap, M_HCA, H, D, DI)
    tg = ThreadGroup(world)
    res = tg.run(lambda r, ag: _run_rank_dense(r, world, x, E_cap, ctx, ag, window_rank=world // 2))
    _check_dense(res, x, ctx)


@pytest.mark.parametrize("case", PREFILL_CASES, ids=["csa", "hca", "few_rows"])
def test_cp_prefill_rows_gloo_two_ranks(case):
    oracle.build()
    mp.spawn(_gloo_worker, args=(2, _free_port(), case, False, True), nprocs=2, join=True)


@pytest.mark.parametrize("world", [1, 3, 4])
@pytest.mark.parametrize("case", PREFILL_CASES, ids=["csa", "hca", "few_rows"])
def test_cp_prefill_rows_thread_ranks(case, world):
    """Rows sharded, cache replicated: the gathered outputs equal the unsharded oracle
    bit for bit (each row's selection and attention use only that row's data)."""
    oracle.build()
    seed, B, T, E_cap, pos0, csa = case
    x = prefill_case(seed, B, T, E_cap, M, H, D, DI)
    tg = ThreadGroup(world)
    _prefill_check(tg.run(lambda r, ag: _prefill_run(r, world, x, pos0, csa, ag)), x, pos0, csa)


def test_cp_union_of_local_topk_is_global_topk():
    """The property the exchange rests on, by brute force: for random shardings the
    top-k of the union of the shards' top-k lists equals the global top-k."""
    g = np.random.default_rng(5)
    for _ in range(200):
        n, k = int(g.integers(1, 60)), int(g.integers(1, 12))
        s = g.integers(-5, 6, n)                       # many ties
        cuts = np.sort(g.integers(0, n + 1, int(g.integers(0, 4))))
        bounds = [0, *cuts.tolist(), n]
        order = lambda ids: sorted(ids, key=lambda j: (-s[j], j))
        union = []
        for a, b in zip(bounds[:-1], bounds[1:]):
            union += order(range(a, b))[:k]
        assert sorted(order(union)[:k]) == sorted(order(range(n))[:k])


def test_split_list_and_row_bounds():
    """Host helpers: the pieces of a per-rank list cover it once, in order, each call at
    most TC_SLOTS slots with the window on the first piece only; row ranges cover a
    chunk once, nearly equal, in rank order."""
    for n in [1, 2, 100, 1919, 1920, 1921, 2048, 4096, 5000]:
        for w in [0, 1, 128, 2047]:
            ps = cp.split_list(n, w)
            assert ps[0][0] == 0 and ps[-1][1] == n
            assert all(a[1] == b[0] for a, b in zip(ps, ps[1:]))
            assert ps[0][2] == w and all(p[2] == 0 for p in ps[1:])
            assert all(c1 > c0 and c1 - c0 + ww <= cp.TC_SLOTS for c0, c1, ww in ps)
    for T in [1, 5, 13, 48, 8192]:
        for world in [1, 2, 3, 4, 7]:
            rb = [cp.row_bounds(T, world, r) for r in range(world)]
            assert rb[0][0] == 0 and rb[-1][1] == T
            assert all(a[1] == b[0] for a, b in zip(rb, rb[1:]))
            assert max(t1 - t0 for t0, t1 in rb) <= -(-T // world)
