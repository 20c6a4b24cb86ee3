"""Context parallelism for this attention path: decode over one long sequence whose
compressed entries are sharded across ranks (CSA and HCA layers), and chunked
prefill with the query rows sharded.

Rank r of `world` holds a contiguous range [e0, e0 + n_local) of every sequence's
compressed entries (Kc, Vc and the indexer keys kI); the rank `window_rank` also
holds the newest raw tokens.  One decode step (QbitAI article "DeepSeek V4报告太详尽了！",
section 混合注意力机制: CSA steps 2-3 and the sliding-window paragraph) becomes:

  1. every rank scores its own visible entries and keeps its local top-k
     (`index_topk`), with their exact scores (`index_scores`);
  2. all-gather of the (score, global index) pairs; every rank merges them into
     the global top-k (`topk_merge`) -- the top-k of the union of the local
     top-k lists is the top-k of the whole sequence, because an entry outside
     its rank's list has k entries of that rank ranked above it;
  3. every rank attends to the selected entries it holds, the window rank adds
     the raw window (`attn_partial`, giving out and lse);
  4. all-gather of the partial (out, lse) and the log-sum-exp merge (`lse_merge`).

The exchange is written once, against two small interfaces: `allgather(t)`
returns the rank-ordered stack of every rank's `t` (torch.distributed, or an
emulation of several ranks in one process), and `ops` computes the per-rank
steps.  `DeviceOps` runs them through the library's CUDA kernels (C ABI).
Dense (HCA) layers (QbitAI article, the HCA paragraph: dense attention over every
compressed entry) shard the same way with steps 1-2 left out: every rank attends to
all of its visible entries, the window rank adds the window, and the partials are
merged (`cp_decode_step_dense`).
A prefill chunk can instead shard its query rows with the cache replicated
(`cp_prefill_rows`): every row's selection and attention use only that row's data,
so ranks need no exchange besides gathering the outputs.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Callable

import torch


@dataclass
class Shard:
    """What one rank holds.  kc, vc: [B, n_local, d]; k_idx: [B, n_local, DI] int8;
    k_raw, v_raw: the raw cache indexed by global token position [B, N_cap, d]
    (read only on `window_rank`, only at the last `window` positions)."""
    rank: int
    world: int
    e0: int
    kc: torch.Tensor
    vc: torch.Tensor
    k_idx: torch.Tensor
    k_raw: torch.Tensor
    v_raw: torch.Tensor
    window_rank: int

    @property
    def n_local(self) -> int:
        return self.kc.shape[1]


def shard_bounds(E_cap: int, world: int, rank: int) -> tuple[int, int]:
    """Contiguous, nearly equal entry ranges: rank r holds [e0, e1)."""
    per = (E_cap + world - 1) // world
    e0 = min(E_cap, rank * per)
    return e0, min(E_cap, e0 + per)


def torch_allgather(group=None) -> Callable[[torch.Tensor], torch.Tensor]:
    """all-gather over a torch.distributed process group, stacked in rank order."""
    import torch.distributed as dist

    def ag(t: torch.Tensor) -> torch.Tensor:
        t = t.contiguous()
        parts = [torch.empty_like(t) for _ in range(dist.get_world_size(group))]
        dist.all_gather(parts, t, group=group)
        return torch.stack(parts)

    return ag


def cp_decode_step(sh: Shard, q: torch.Tensor, q_idx: torch.Tensor, ctx_len: torch.Tensor, *, m: int, topk: int,
                   window: int, scale: float, allgather: Callable[[torch.Tensor], torch.Tensor], ops):
    """One CSA decode step of B sequences (query at p = ctx_len - 1).
    q [B, H, d]; q_idx [B, 1, DI] int8; ctx_len int64 [B].
    Returns (out [B, H, d], lse [B, H] fp32, selected global indices [B, topk])."""
    B = q.shape[0]
    E = torch.div(ctx_len, m, rounding_mode="floor")
    E_loc = (E - sh.e0).clamp(min=0, max=sh.n_local)
    # 1. local top-k and its scores
    idx_l, cnt_l = ops.index_topk(q_idx, sh.k_idx, E_loc, m, topk)
    sc_l = ops.index_scores(q_idx, sh.k_idx, idx_l, cnt_l)
    gidx = torch.where(idx_l >= 0, idx_l + sh.e0, torch.full_like(idx_l, -1))
    # 2. gather every rank's pairs (rank-major: global indices ascending) and merge
    all_sc = allgather(sc_l.reshape(B, topk))
    all_ix = allgather(gidx.reshape(B, topk))
    pairs_sc = all_sc.permute(1, 0, 2).reshape(B, -1).contiguous()
    pairs_ix = all_ix.permute(1, 0, 2).reshape(B, -1).contiguous()
    sel, _ = ops.topk_merge(pairs_sc, pairs_ix, topk)
    # 3. attention over the selected entries this rank holds (+ the window on one rank)
    mine = (sel >= sh.e0) & (sel < sh.e0 + sh.n_local)
    loc = torch.where(mine, sel - sh.e0, torch.full_like(sel, -1))
    w = window if sh.rank == sh.window_rank else 0
    o_r, lse_r = ops.attn_partial(q, sh.kc, sh.vc, m, loc, sh.k_raw, sh.v_raw, w, ctx_len, scale)
    # 4. gather the partials and merge them
    out, lse = ops.lse_merge(allgather(o_r), allgather(lse_r))
    return out, lse, sel


def cp_decode_step_dense(sh: Shard, q: torch.Tensor, ctx_len: torch.Tensor, *, m: int, window: int, scale: float,
                         allgather: Callable[[torch.Tensor], torch.Tensor], ops):
    """One HCA decode step of B sequences (query at p = ctx_len - 1): every rank attends
    to all of its visible entries (listed explicitly, so the same per-rank attention
    serves), the window rank adds the raw window, and one all-gather of the partial
    (out, lse) feeds the log-sum-exp merge.  `sh.k_idx` is not read.
    Returns (out [B, H, d], lse [B, H] fp32)."""
    B = q.shape[0]
    E = torch.div(ctx_len, m, rounding_mode="floor")
    E_loc = (E - sh.e0).clamp(min=0, max=sh.n_local).to(q.device)
    ar = torch.arange(sh.n_local, dtype=torch.int32, device=q.device)
    loc = torch.where(ar[None, :] < E_loc[:, None], ar[None, :].expand(B, -1),
                      torch.full((B, sh.n_local), -1, dtype=torch.int32, device=q.device))
    w = window if sh.rank == sh.window_rank else 0
    o_r, lse_r = ops.attn_partial(q, sh.kc, sh.vc, m, loc.contiguous(), sh.k_raw, sh.v_raw, w, ctx_len, scale)
    return ops.lse_merge(allgather(o_r), allgather(lse_r))


def row_bounds(T: int, world: int, rank: int) -> tuple[int, int]:
    """Contiguous, nearly equal query-row ranges of a T-token chunk: rank r takes [t0, t1)."""
    per = (T + world - 1) // world
    t0 = min(T, rank * per)
    return t0, min(T, t0 + per)


def cp_prefill_rows(rank: int, world: int, q: torch.Tensor, q_idx, k_idx, kc, vc, k_raw, v_raw,
                    q_pos0: torch.Tensor, *, m: int, topk: int, window: int, scale: float, ops,
                    allgather: Callable[[torch.Tensor], torch.Tensor] | None = None):
    """Chunked prefill with the chunk's query rows sharded over ranks and the cache
    replicated (no exchange): rank r selects (CSA: q_idx and k_idx given; HCA: None)
    and attends for the tokens [t0, t1) of its row range, whose positions start at
    q_pos0 + t0.  q [B, T, H, d], q_idx [B, T, DI].  Returns (t0, out [B, t1 - t0, H, d],
    lse, this rank's idx or None); with `allgather`, (0, out, lse) of the whole chunk
    (every rank's range padded to the longest for the gather) and this rank's idx."""
    B, T = q.shape[:2]
    t0, t1 = row_bounds(T, world, rank)
    pos = (q_pos0 + t0).contiguous()
    idx = cnt = None
    if t1 > t0:
        if q_idx is not None:
            idx, cnt = ops.index_topk_rows(q_idx[:, t0:t1].contiguous(), k_idx, pos, m, topk)
        out, lse = ops.attn_prefill(q[:, t0:t1].contiguous(), kc, vc, m, idx, cnt, k_raw, v_raw, window, pos,
                                    scale)
    else:  # more ranks than rows: nothing here
        out = torch.empty((B, 0) + tuple(q.shape[2:]), dtype=q.dtype, device=q.device)
        lse = torch.empty((B, 0, q.shape[2]), dtype=torch.float32, device=q.device)
    if allgather is None:
        return t0, out, lse, idx
    per = (T + world - 1) // world
    pad_o = torch.zeros((B, per) + tuple(out.shape[2:]), dtype=out.dtype, device=out.device)
    pad_l = torch.zeros((B, per) + tuple(lse.shape[2:]), dtype=lse.dtype, device=lse.device)
    pad_o[:, :t1 - t0] = out
    pad_l[:, :t1 - t0] = lse
    go, gl = allgather(pad_o), allgather(pad_l)  # [world, B, per, ...]
    lens = [row_bounds(T, world, r)[1] - row_bounds(T, world, r)[0] for r in range(world)]
    full_o = torch.cat([go[r, :, :lens[r]] for r in range(world)], 1)
    full_l = torch.cat([gl[r, :, :lens[r]] for r in range(world)], 1)
    return 0, full_o, full_l, idx


TC_SLOTS = 2048  # selected entries + window one call of the tensor-core decode kernel takes


def split_list(n: int, window: int, slots: int = TC_SLOTS):
    """Pieces [(c0, c1, window)] of an n-entry list for calls of at most `slots` slots:
    the window goes with the first piece."""
    first = max(1, slots - window)
    out = [(0, min(n, first), window)]
    c0 = out[0][1]
    while c0 < n:
        out.append((c0, min(n, c0 + slots), 0))
        c0 = out[-1][1]
    return out


class DeviceOps:
    """The per-rank steps on this process's GPU through the library's C ABI
    (workspaces are allocated once here and reused; the library allocates nothing)."""

    def __init__(self, B: int, H: int, d: int, DI: int, n_local: int, m: int, topk: int, window: int,
                 dtype=torch.bfloat16, device="cuda"):
        """DI = 0: no indexer (the dense step); its attention lists every local entry,
        so pass topk = n_local.  A list longer than one tensor-core call takes is cut
        into pieces (`split_list`) whose partials are merged here."""
        from . import _lib as L
        self.L = L
        self.topk = topk
        self.window = window
        self.ws_i = (L.workspace(L.hsa_index_topk_workspace_size(B, 1, DI, n_local, topk), device=device)
                     if DI else None)
        sizes = [L.hsa_attn_decode_workspace_size(dtype, B, H, d, n_local, m, c1 - c0, w)
                 for c0, c1, w in split_list(max(topk, 1), window)]
        self.ws_a = L.workspace(max(sizes), device=device)

    def index_topk(self, q_idx, k_idx, E_loc, m, topk):
        B = q_idx.shape[0]
        # local positions whose visible-entry count is E_loc: floor((p + 1) / m) = E_loc
        pos0 = (E_loc * m - 1).to(torch.int64).contiguous()
        idx = torch.empty((B, 1, topk), dtype=torch.int32, device=q_idx.device)
        cnt = torch.empty((B, 1), dtype=torch.int32, device=q_idx.device)
        self.L.hsa_index_topk(q_idx, k_idx, pos0, m, topk, idx, cnt, self.ws_i)
        return idx, cnt

    def index_scores(self, q_idx, k_idx, idx, cnt):
        sc = torch.empty_like(idx)
        self.L.hsa_index_scores(q_idx, k_idx, idx, cnt, sc)
        return sc

    def topk_merge(self, scores, idx, topk):
        rows = idx.shape[0]
        out = torch.empty((rows, topk), dtype=torch.int32, device=idx.device)
        cnt = torch.empty((rows,), dtype=torch.int32, device=idx.device)
        self.L.hsa_topk_merge(scores, idx, topk, out, cnt)
        return out, cnt

    def attn_partial(self, q, kc, vc, m, loc_idx, k_raw, v_raw, window, ctx_len, scale):
        B, H, d = q.shape
        if loc_idx.shape[1] == 0:  # a rank holding no entry: one empty slot, the window alone
            loc_idx = torch.full((B, 1), -1, dtype=torch.int32, device=q.device)
        parts = split_list(loc_idx.shape[1], window)
        outs, lses = [], []
        for c0, c1, w in parts:
            out = torch.empty_like(q)
            lse = torch.empty((B, H), dtype=torch.float32, device=q.device)
            self.L.hsa_attn_decode(q, kc, vc, m, loc_idx[:, c0:c1].contiguous(), None, k_raw, v_raw, w, ctx_len,
                                   scale, out, lse, self.ws_a)
            outs.append(out)
            lses.append(lse)
        if len(parts) == 1:
            return outs[0], lses[0]
        return self.lse_merge(torch.stack(outs), torch.stack(lses))

    def index_topk_rows(self, q_idx, k_idx, q_pos0, m, topk):
        """Top-k of several query rows per sequence (prefill rows): idx [B, T, topk], cnt [B, T]."""
        B, T, DI = q_idx.shape
        idx = torch.empty((B, T, topk), dtype=torch.int32, device=q_idx.device)
        cnt = torch.empty((B, T), dtype=torch.int32, device=q_idx.device)
        ws = self.L.workspace(self.L.hsa_index_topk_workspace_size(B, T, DI, k_idx.shape[1], topk),
                              device=q_idx.device)
        self.L.hsa_index_topk(q_idx, k_idx, q_pos0, m, topk, idx, cnt, ws)
        return idx, cnt

    def attn_prefill(self, q, kc, vc, m, idx, cnt, k_raw, v_raw, window, q_pos0, scale):
        B, T, H, d = q.shape
        out = torch.empty_like(q)
        lse = torch.empty((B, T, H), dtype=torch.float32, device=q.device)
        topk = idx.shape[-1] if idx is not None else 0
        ws = self.L.workspace(self.L.hsa_attn_prefill_workspace_size(q.dtype, B, T, H, d, kc.shape[1], m, topk,
                                                                     window), device=q.device)
        self.L.hsa_attn_prefill(q, kc, vc, m, idx, cnt, k_raw, v_raw, window, q_pos0, scale, out, lse, ws)
        return out, lse

    def lse_merge(self, parts_o, parts_lse):
        out = torch.empty(parts_o.shape[1:], dtype=parts_o.dtype, device=parts_o.device)
        lse = torch.empty(parts_lse.shape[1:], dtype=torch.float32, device=parts_o.device)
        self.L.hsa_lse_merge(parts_o.contiguous(), parts_lse.contiguous(), out, lse)
        return out, lse
