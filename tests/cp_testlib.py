"""Helpers of the context-parallel tests: the per-rank steps computed by the oracle
(CPU), an in-process emulation of several ranks (threads and a shared
all-gather), and seeded sharded inputs.  The exchange itself is the library's
``cp.cp_decode_step``."""
from __future__ import annotations

import threading

import numpy as np
import torch

import oracle

INT32_MIN = -(1 << 31)


class OracleOps:
    """Per-rank steps of the CP decode computed by the oracle, for one rank's shard.
    `kc_full`-sized buffers are built with only this rank's entries filled, so a
    rank that touched another rank's entries would read zeros and fail the test."""

    def __init__(self, e0: int, E_cap: int):
        self.e0, self.E_cap = e0, E_cap

    def index_topk(self, q_idx, k_idx, E_loc, m, topk):
        B = q_idx.shape[0]
        idx = np.full((B, 1, topk), -1, dtype=np.int32)
        cnt = np.zeros((B, 1), dtype=np.int32)
        for b in range(B):
            e = int(E_loc[b])
            if e == 0:
                continue
            i, c = oracle.index_topk_rows(q_idx[b, :1].numpy(), [0], [e * m - 1], k_idx[b:b + 1].numpy(), m, topk)
            idx[b, 0], cnt[b, 0] = i[0], c[0]
        return torch.from_numpy(idx), torch.from_numpy(cnt)

    def index_scores(self, q_idx, k_idx, idx, cnt):
        B, T, topk = idx.shape
        out = np.full((B, T, topk), INT32_MIN, dtype=np.int64)
        q = q_idx.numpy().astype(np.int64)
        k = k_idx.numpy().astype(np.int64)
        for b in range(B):
            for t in range(T):
                for s in range(int(cnt[b, t])):
                    j = int(idx[b, t, s])
                    if j >= 0:
                        out[b, t, s] = int(q[b, t] @ k[b, j])
        return torch.from_numpy(out.astype(np.int32))

    def topk_merge(self, scores, idx, topk):
        rows = idx.shape[0]
        out = np.full((rows, topk), -1, dtype=np.int32)
        cnt = np.zeros((rows,), dtype=np.int32)
        for r in range(rows):
            pairs = [(-int(s), int(j)) for s, j in zip(scores[r].tolist(), idx[r].tolist()) if j >= 0]
            best = sorted(sorted(pairs)[:topk], key=lambda x: x[1])
            cnt[r] = len(best)
            out[r, :len(best)] = [j for _, j in best]
        return torch.from_numpy(out), torch.from_numpy(cnt)

    def attn_partial(self, q, kc, vc, m, loc_idx, k_raw, v_raw, window, ctx_len, scale):
        B, H, d = q.shape
        n = kc.shape[1]
        kf = np.zeros((B, self.E_cap, d))
        vf = np.zeros((B, self.E_cap, d))
        kf[:, self.e0:self.e0 + n] = kc.numpy()
        vf[:, self.e0:self.e0 + n] = vc.numpy()
        gidx = np.where(loc_idx.numpy() >= 0, loc_idx.numpy() + self.e0, -1).astype(np.int32)
        o, l = oracle.attn_rows(q.numpy(), np.arange(B), ctx_len.numpy() - 1, kf, vf, m, gidx,
                                k_raw.numpy(), v_raw.numpy(), window, scale)
        return torch.from_numpy(o), torch.from_numpy(l)

    def lse_merge(self, parts_o, parts_lse):
        S, B, H, d = parts_o.shape
        out = np.empty((B, H, d))
        lse = np.empty((B, H))
        for b in range(B):
            out[b], lse[b] = oracle.lse_merge(parts_o[:, b].numpy(), parts_lse[:, b].numpy())
        return torch.from_numpy(out), torch.from_numpy(lse)


class ThreadGroup:
    """`world` ranks as threads of one process: all_gather through shared slots."""

    def __init__(self, world: int):
        self.world = world
        self.slots = [None] * world
        self.bar = threading.Barrier(world, timeout=120)

    def allgather_for(self, rank: int):
        def ag(t):
            self.slots[rank] = t
            self.bar.wait()
            out = torch.stack(list(self.slots))
            self.bar.wait()
            return out
        return ag

    def run(self, fn):
        """fn(rank, allgather) in `world` threads; returns the per-rank results."""
        res, errs = [None] * self.world, []

        def body(r):
            try:
                res[r] = fn(r, self.allgather_for(r))
            except BaseException as e:  # noqa: BLE001 - reported below
                errs.append(e)
                self.bar.abort()

        th = [threading.Thread(target=body, args=(r,)) for r in range(self.world)]
        for t in th:
            t.start()
        for t in th:
            t.join()
        if errs:
            raise errs[0]
        return res


def cp_case(seed: int, B: int, E_cap: int, m: int, H: int, d: int, DI: int, ties: bool = False):
    """Seeded full-sequence inputs (fp64 values, int8 indexer vectors)."""
    g = np.random.default_rng(seed)
    N = E_cap * m
    kc = g.standard_normal((B, E_cap, d))
    vc = g.standard_normal((B, E_cap, d))
    k_raw = g.standard_normal((B, N, d))
    v_raw = g.standard_normal((B, N, d))
    q = g.standard_normal((B, H, d))
    hi = 3 if ties else 128
    k_idx = g.integers(-hi + 1, hi, (B, E_cap, DI)).astype(np.int8)
    q_idx = g.integers(-127, 128, (B, 1, DI)).astype(np.int8)
    return dict(kc=kc, vc=vc, k_raw=k_raw, v_raw=v_raw, q=q, k_idx=k_idx, q_idx=q_idx)


def full_reference(x, ctx_len, m, topk, window, scale):
    """Single-process oracle of the same step: global top-k, then attention."""
    B = x["q"].shape[0]
    p = np.asarray(ctx_len) - 1
    idx, cnt = oracle.index_topk_rows(x["q_idx"][:, 0], np.arange(B), p, x["k_idx"], m, topk)
    o, l = oracle.attn_rows(x["q"], np.arange(B), p, x["kc"], x["vc"], m, idx, x["k_raw"], x["v_raw"], window, scale)
    return idx, o, l


def full_reference_dense(x, ctx_len, m, window, scale):
    """Single-process oracle of the HCA step: attention over every visible entry."""
    B = x["q"].shape[0]
    p = np.asarray(ctx_len) - 1
    o, l = oracle.attn_rows(x["q"], np.arange(B), p, x["kc"], x["vc"], m, None, x["k_raw"], x["v_raw"], window,
                            scale)
    return o, l


class PrefillOracleOps:
    """Per-rank prefill steps (replicated cache) computed by the oracle."""

    def index_topk_rows(self, q_idx, k_idx, q_pos0, m, topk):
        B, T, DI = q_idx.shape
        rows_b = np.repeat(np.arange(B), T)
        rows_p = (q_pos0.numpy()[:, None] + np.arange(T)[None, :]).reshape(-1)
        idx, cnt = oracle.index_topk_rows(q_idx.numpy().reshape(B * T, DI), rows_b, rows_p, k_idx.numpy(), m, topk)
        return torch.from_numpy(idx.reshape(B, T, topk)), torch.from_numpy(cnt.reshape(B, T))

    def attn_prefill(self, q, kc, vc, m, idx, cnt, k_raw, v_raw, window, q_pos0, scale):
        B, T, H, d = q.shape
        rows_b = np.repeat(np.arange(B), T)
        rows_p = (q_pos0.numpy()[:, None] + np.arange(T)[None, :]).reshape(-1)
        ia = None if idx is None else idx.numpy().reshape(B * T, -1)
        o, l = oracle.attn_rows(q.numpy().reshape(B * T, H, d), rows_b, rows_p, kc.numpy(), vc.numpy(), m, ia,
                                k_raw.numpy(), v_raw.numpy(), window, scale)
        return torch.from_numpy(o.reshape(B, T, H, d)), torch.from_numpy(l.reshape(B, T, H))


def prefill_case(seed: int, B: int, T: int, E_cap: int, m: int, H: int, d: int, DI: int):
    """Seeded chunk inputs: q [B, T, H, d] fp64, q_idx [B, T, DI] int8, and a replicated cache."""
    g = np.random.default_rng(seed)
    N = E_cap * m
    return dict(q=g.standard_normal((B, T, H, d)), q_idx=g.integers(-127, 128, (B, T, DI)).astype(np.int8),
                kc=g.standard_normal((B, E_cap, d)), vc=g.standard_normal((B, E_cap, d)),
                k_raw=g.standard_normal((B, N, d)), v_raw=g.standard_normal((B, N, d)),
                k_idx=g.integers(-127, 128, (B, E_cap, DI)).astype(np.int8))
