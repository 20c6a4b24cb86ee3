"""Pins for the CPU oracle: each check ties it to something other than itself.

The pages print no worked numerical example for this path, so the oracle is
pinned by (a) the counts the pages do print (tests/golden), (b) special cases
that reduce to a textbook routine (torch's scaled_dot_product_attention in
fp64, numpy integer matmul, scipy softmax / logsumexp, itertools enumeration),
(c) closed forms and invariants.  Each pin is chosen so that a plausible slip
in the oracle (a dropped term, an off-by-one block or window bound, a wrong
sign, a transposed operand, a wrong tie rule) fails at least one of them.
"""
import itertools
import math
import os

import numpy as np
import pytest
import scipy.special
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
RNG = np.random.default_rng(12345)


def _golden_rows(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("|")[0].strip()
            if line and not line.startswith("#"):
                rows.append([int(v) for v in line.split()])
    return rows


# ----------------------------------------------------------------- counts ---

@pytest.mark.parametrize("tokens,m,expected", _golden_rows("entry_counts.txt"))
def test_entry_counts_golden(tokens, m, expected):
    # A sequence of `tokens` tokens: the query at the last position p = tokens - 1.
    assert oracle.num_entries(tokens - 1, m) == expected


def test_entry_count_strict_causality():
    # Block j is visible at p iff (j+1)*m - 1 <= p: a block ending exactly at p counts,
    # a block still incomplete at p does not.
    for m in (1, 4, 128):
        for p in range(0, 3 * m + 2):
            visible = [j for j in range(0, p + 2) if (j + 1) * m - 1 <= p]
            assert oracle.num_entries(p, m) == len(visible)


@pytest.mark.parametrize("tokens,m,topk,expected", _golden_rows("topk_counts.txt"))
def test_topk_count_golden(tokens, m, topk, expected):
    E = tokens // m
    kI = RNG.integers(-127, 128, size=(1, E, 8), dtype=np.int64).astype(np.int8)
    q = RNG.integers(-127, 128, size=(1, 8), dtype=np.int64).astype(np.int8)
    idx, cnt = oracle.index_topk_rows(q, [0], [tokens - 1], kI, m, topk)
    assert cnt[0] == expected
    assert (idx[0] >= 0).sum() == expected


@pytest.mark.parametrize("p,W,expected", _golden_rows("window.txt"))
def test_window_size_golden(p, W, expected):
    # q = 0 makes every logit 0, so lse = ln |S|; with no entries |S| is the window size.
    N = p + 1
    z = np.zeros((1, N, 1), dtype=np.float32)
    kc = np.zeros((1, 1, 1), dtype=np.float32)
    q = np.zeros((1, 1, 1), dtype=np.float32)
    idx = np.full((1, 1), -1, dtype=np.int32)
    _, lse = oracle.attn_rows(q, [0], [p], kc, kc, N, idx, z, z, W, 1.0)
    assert round(math.exp(lse[0, 0])) == expected


# ------------------------------------------------------------- compressor ---

def _x(B, N, d):
    return RNG.standard_normal((B, N, d)).astype(np.float32)


@pytest.mark.parametrize("m", [4, 128])
def test_compress_one_hot_copies_token(m):
    B, N, d = 2, 3 * m + 1, 5
    x = _x(B, N, d)
    for r0 in (0, m - 1, m // 2):
        w = np.zeros(m, dtype=np.float32)
        w[r0] = 1.0
        E = N // m
        out = oracle.compress(x, w, m, [0, 0], [N, N], E)
        np.testing.assert_array_equal(out, x[:, r0:E * m:m, :].astype(np.float64))


def test_compress_uniform_weights_is_block_mean():
    m, B, N, d = 4, 2, 41, 3
    x = _x(B, N, d)
    w = np.full(m, 0.25, dtype=np.float32)
    E = N // m
    out = oracle.compress(x, w, m, [0, 0], [N, N], E)
    ref = x[:, :E * m].astype(np.float64).reshape(B, E, m, d).mean(axis=2)
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-14)


def test_compress_m1_identity():
    x = _x(1, 17, 4)
    out = oracle.compress(x, np.ones(1, np.float32), 1, [0], [17], 17)
    np.testing.assert_array_equal(out, x.astype(np.float64))


def test_compress_linear_and_weighted():
    m, B, N, d = 4, 1, 24, 6
    x, y = _x(B, N, d), _x(B, N, d)
    w = RNG.random(m).astype(np.float32)
    E = N // m
    cx = oracle.compress(x, w, m, [0], [N], E)
    cy = oracle.compress(y, w, m, [0], [N], E)
    cxy = oracle.compress(2 * x.astype(np.float64) - 3 * y.astype(np.float64), w, m, [0], [N], E)
    np.testing.assert_allclose(cxy, 2 * cx - 3 * cy, atol=1e-12)
    # explicit weighted sum of the block via an einsum
    ref = np.einsum("r,bjrc->bjc", w.astype(np.float64), x.astype(np.float64).reshape(B, E, m, d))
    np.testing.assert_allclose(cx, ref, atol=1e-13)


def test_compress_token_range():
    m, N, d = 4, 40, 2
    x = _x(1, N, d)
    w = RNG.random(m).astype(np.float32)
    full = oracle.compress(x, w, m, [0], [N], N // m)
    part = oracle.compress(x, w, m, [13], [35], N // m)   # blocks 3 .. 7
    np.testing.assert_array_equal(part[:, 3:8], full[:, 3:8])
    assert not part[:, :3].any() and not part[:, 8:].any()


def test_compress_bf16_reads_exactly():
    x = torch.randn(1, 8, 4).to(torch.bfloat16)
    bits = x.view(torch.int16).numpy().view(np.uint16)
    out = oracle.compress(bits, np.ones(1, np.float32), 1, [0], [8], 8)
    np.testing.assert_array_equal(out, x.double().numpy())


# ------------------------------------------------------------------ top-k ---

def _brute_topk_set(s, k):
    """The unique set S (|S| = min(k, E)) with every member beating every non-member
    under (score desc, index asc), found by exhaustive enumeration."""
    E = len(s)
    n = min(k, E)
    found = []
    for S in itertools.combinations(range(E), n):
        rest = [j for j in range(E) if j not in S]
        if all(s[i] > s[j] or (s[i] == s[j] and i < j) for i in S for j in rest):
            found.append(list(S))
    assert len(found) == 1
    return found[0]


def _topk_property(idx_row, cnt, s, E, k):
    n = min(k, E)
    assert cnt == n
    sel = idx_row[:n]
    assert (idx_row[n:] == -1).all()
    assert (np.diff(sel) > 0).all() and (sel >= 0).all() and (sel < E).all()
    chosen = set(sel.tolist())
    rest = [j for j in range(E) if j not in chosen]
    if rest and n:
        worst = min(sel, key=lambda i: (s[i], -i))
        best_rest = max(rest, key=lambda j: (s[j], -j))
        assert (s[worst], -worst) > (s[best_rest], -best_rest)


@pytest.mark.parametrize("values", [(-127, 127), (-1, 1), (0, 0), (-128, 127)])
def test_topk_exhaustive_tiny(values):
    lo, hi = values
    for trial in range(20):
        E_cap, DI, m = 9, 3, 2
        kI = RNG.integers(lo, hi + 1, size=(1, E_cap, DI)).astype(np.int8)
        q = RNG.integers(lo, hi + 1, size=(3, DI)).astype(np.int8)
        ps = [1, 9, 2 * E_cap - 1]
        for k in (1, 3, 4, 12):
            idx, cnt = oracle.index_topk_rows(q, [0, 0, 0], ps, kI, m, k)
            for r, p in enumerate(ps):
                E = (p + 1) // m
                s = (kI[0, :E].astype(np.int64) @ q[r].astype(np.int64)).tolist()
                want = _brute_topk_set(s, k)
                got = idx[r][idx[r] >= 0].tolist()
                assert got == want
                assert cnt[r] == len(want)


@pytest.mark.parametrize("lo,hi", [(-127, 127), (-1, 1)])
def test_topk_property_medium(lo, hi):
    B, E_cap, DI, m, k = 2, 700, 16, 4, 37
    kI = RNG.integers(lo, hi + 1, size=(B, E_cap, DI)).astype(np.int8)
    rows_b = [0, 1, 1, 0, 1]
    rows_p = [4 * E_cap - 1, 4 * E_cap - 2, 150, 3, 2]
    q = RNG.integers(lo, hi + 1, size=(len(rows_b), DI)).astype(np.int8)
    idx, cnt = oracle.index_topk_rows(q, rows_b, rows_p, kI, m, k)
    for r, (b, p) in enumerate(zip(rows_b, rows_p)):
        E = (p + 1) // m
        s = (kI[b, :E].astype(np.int64) @ q[r].astype(np.int64))
        _topk_property(idx[r], cnt[r], s, E, k)


def test_topk_all_equal_scores_take_lowest_indices():
    kI = np.zeros((1, 50, 8), dtype=np.int8)
    q = RNG.integers(-127, 128, size=(1, 8)).astype(np.int8)
    idx, cnt = oracle.index_topk_rows(q, [0], [199], kI, 4, 10)
    assert idx[0].tolist() == list(range(10)) and cnt[0] == 10


def test_topk_k_at_least_E_takes_all():
    kI = RNG.integers(-127, 128, size=(1, 30, 8)).astype(np.int8)
    q = RNG.integers(-127, 128, size=(1, 8)).astype(np.int8)
    idx, cnt = oracle.index_topk_rows(q, [0], [4 * 7 + 2], kI, 4, 16)  # E = 7
    assert idx[0].tolist() == list(range(7)) + [-1] * 9 and cnt[0] == 7


def test_topk_no_visible_entry():
    kI = RNG.integers(-127, 128, size=(1, 30, 8)).astype(np.int8)
    q = RNG.integers(-127, 128, size=(1, 8)).astype(np.int8)
    idx, cnt = oracle.index_topk_rows(q, [0], [2], kI, 4, 5)  # E(2) = 0 for m = 4
    assert cnt[0] == 0 and (idx[0] == -1).all()


def test_topk_planted_winners_selected():
    E, DI, k = 500, 64, 16
    q = RNG.integers(-127, 128, size=(1, DI)).astype(np.int8)
    kI = RNG.integers(-3, 4, size=(1, E, DI)).astype(np.int8)
    planted = sorted(RNG.choice(E, size=k, replace=False).tolist())
    kI[0, planted] = np.clip(q[0].astype(np.int16), -127, 127).astype(np.int8)
    idx, cnt = oracle.index_topk_rows(q, [0], [4 * E - 1], kI, 4, k)
    assert idx[0].tolist() == planted


def test_topk_score_sign_and_operand():
    # a single entry that is the exact negative of q must lose to every zero entry
    DI = 16
    q = RNG.integers(1, 128, size=(1, DI)).astype(np.int8)
    kI = np.zeros((1, 5, DI), dtype=np.int8)
    kI[0, 0] = -q[0]
    kI[0, 4] = 1
    idx, _ = oracle.index_topk_rows(q, [0], [19], kI, 4, 2)
    assert idx[0].tolist() == [1, 4]


# -------------------------------------------------------------- attention ---

def _sdpa(q, k, v, mask):
    """torch fp64 textbook attention.  q [T, H, d], k, v [S, d], mask [T, S] bool or float."""
    qt = torch.from_numpy(np.asarray(q, np.float64)).permute(1, 0, 2)  # [H, T, d]
    kt = torch.from_numpy(np.asarray(k, np.float64)).unsqueeze(0).expand(qt.shape[0], -1, -1)
    vt = torch.from_numpy(np.asarray(v, np.float64)).unsqueeze(0).expand(qt.shape[0], -1, -1)
    mt = torch.from_numpy(mask)
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mt)
    return o.permute(1, 0, 2).numpy()


def _prefill_rows(T):
    return np.zeros(T, np.int64), np.arange(T, dtype=np.int64)


def test_attn_m1_dense_no_window_is_causal_attention():
    T, H, d = 23, 3, 8
    q = RNG.standard_normal((T, H, d)).astype(np.float32)
    k = RNG.standard_normal((1, T, d)).astype(np.float32)
    v = RNG.standard_normal((1, T, d)).astype(np.float32)
    rb, rp = _prefill_rows(T)
    out, _ = oracle.attn_rows(q, rb, rp, k, v, 1, None, k, v, 0, 1 / math.sqrt(d))
    causal = np.tril(np.ones((T, T), dtype=bool))
    np.testing.assert_allclose(out, _sdpa(q, k[0], v[0], causal), atol=1e-12)


def test_attn_m1_dense_window_adds_ln2_bias():
    T, H, d, W = 30, 2, 8, 5
    q = RNG.standard_normal((T, H, d)).astype(np.float32)
    k = RNG.standard_normal((1, T, d)).astype(np.float32)
    v = RNG.standard_normal((1, T, d)).astype(np.float32)
    rb, rp = _prefill_rows(T)
    out, _ = oracle.attn_rows(q, rb, rp, k, v, 1, None, k, v, W, 1 / math.sqrt(d))
    i = np.arange(T)[:, None]
    j = np.arange(T)[None, :]
    bias = np.where(j <= i, 0.0, -np.inf) + np.where((j <= i) & (j > i - W), math.log(2.0), 0.0)
    np.testing.assert_allclose(out, _sdpa(q, k[0], v[0], bias), atol=1e-12)


def test_attn_no_entries_is_sliding_window_attention():
    T, H, d, W, m = 40, 2, 8, 7, 4
    q = RNG.standard_normal((T, H, d)).astype(np.float32)
    k = RNG.standard_normal((1, T, d)).astype(np.float32)
    v = RNG.standard_normal((1, T, d)).astype(np.float32)
    kc = RNG.standard_normal((1, T // m, d)).astype(np.float32)
    rb, rp = _prefill_rows(T)
    idx = np.full((T, 3), -1, dtype=np.int32)
    out, _ = oracle.attn_rows(q, rb, rp, kc, kc, m, idx, k, v, W, 1 / math.sqrt(d))
    i = np.arange(T)[:, None]
    j = np.arange(T)[None, :]
    band = (j <= i) & (j > i - W)
    np.testing.assert_allclose(out, _sdpa(q, k[0], v[0], band), atol=1e-12)


def test_attn_selected_entries_plus_window_one_softmax():
    # Attention over [kc ; k_raw] with a per-query mask built from idx and the window bound.
    N, H, d, W, m, k = 64, 4, 8, 6, 4, 5
    E = N // m
    ps = np.array([3, 10, 33, 63], dtype=np.int64)
    q = RNG.standard_normal((len(ps), H, d)).astype(np.float32)
    kr = RNG.standard_normal((1, N, d)).astype(np.float32)
    vr = RNG.standard_normal((1, N, d)).astype(np.float32)
    kc = RNG.standard_normal((1, E, d)).astype(np.float32)
    vc = RNG.standard_normal((1, E, d)).astype(np.float32)
    idx = np.full((len(ps), k), -1, dtype=np.int32)
    for r, p in enumerate(ps):
        Ep = (p + 1) // m
        sel = sorted(RNG.choice(Ep, size=min(k, Ep), replace=False).tolist()) if Ep else []
        idx[r, :len(sel)] = sel
    out, _ = oracle.attn_rows(q, np.zeros(len(ps), np.int64), ps, kc, vc, m, idx, kr, vr, W, 0.3)
    keys = np.concatenate([kc[0], kr[0]])
    vals = np.concatenate([vc[0], vr[0]])
    for r, p in enumerate(ps):
        mask = np.zeros((1, E + N), dtype=bool)
        for j in idx[r]:
            if j >= 0:
                mask[0, j] = True
        for t in range(max(0, p - W + 1), p + 1):
            mask[0, E + t] = True
        ref = _sdpa(q[r:r + 1].astype(np.float64) * (0.3 * math.sqrt(d)), keys, vals, mask)
        np.testing.assert_allclose(out[r], ref[0], atol=1e-12)


def test_attn_zero_query_gives_mean_of_values():
    N, H, d, W, m = 50, 2, 4, 9, 4
    kr = RNG.standard_normal((1, N, d)).astype(np.float32)
    vr = RNG.standard_normal((1, N, d)).astype(np.float32)
    kc = RNG.standard_normal((1, N // m, d)).astype(np.float32)
    vc = RNG.standard_normal((1, N // m, d)).astype(np.float32)
    p = 45
    idx = np.array([[2, 5, 7, -1]], dtype=np.int32)
    out, lse = oracle.attn_rows(np.zeros((1, H, d), np.float32), [0], [p], kc, vc, m, idx, kr, vr, W, 1.0)
    members = np.concatenate([vc[0, [2, 5, 7]], vr[0, p - W + 1:p + 1]])
    np.testing.assert_allclose(out[0], np.broadcast_to(members.astype(np.float64).mean(0), (H, d)), atol=1e-14)
    np.testing.assert_allclose(lse[0], math.log(len(members)), atol=1e-14)


def test_attn_one_hot_values_expose_probabilities():
    # V rows are unit vectors, so the output is the probability vector itself:
    # it must sum to 1 and equal scipy's softmax of the logits; lse = logsumexp.
    n_ent, W, H = 6, 5, 3
    d = n_ent + W
    N = 40
    m = 4
    p = 37
    kc = RNG.standard_normal((1, N // m, d)).astype(np.float32)
    kr = RNG.standard_normal((1, N, d)).astype(np.float32)
    vc = np.zeros((1, N // m, d), np.float32)
    vr = np.zeros((1, N, d), np.float32)
    sel = [0, 1, 3, 4, 6, 8]
    for i, j in enumerate(sel):
        vc[0, j, i] = 1.0
    win = list(range(p - W + 1, p + 1))
    for i, t in enumerate(win):
        vr[0, t, n_ent + i] = 1.0
    q = RNG.standard_normal((1, H, d)).astype(np.float32)
    scale = 0.37
    out, lse = oracle.attn_rows(q, [0], [p], kc, vc, m, np.array([sel], np.int32), kr, vr, W, scale)
    keys = np.concatenate([kc[0, sel], kr[0, win]]).astype(np.float64)
    logits = scale * (q[0].astype(np.float64) @ keys.T)
    np.testing.assert_allclose(out[0].sum(-1), 1.0, atol=1e-14)
    np.testing.assert_allclose(out[0], scipy.special.softmax(logits, axis=-1), atol=1e-14)
    np.testing.assert_allclose(lse[0], scipy.special.logsumexp(logits, axis=-1), atol=1e-13)


def test_attn_empty_set():
    z = np.zeros((1, 8, 2), np.float32)
    out, lse = oracle.attn_rows(np.ones((1, 1, 2), np.float32), [0], [2], z, z, 4,
                                np.full((1, 2), -1, np.int32), z, z, 0, 1.0)
    assert (out == 0).all() and lse[0, 0] == -np.inf


def test_attn_dense_equals_all_selected():
    N, H, d, W, m = 77, 2, 6, 4, 4
    p = 70
    E = (p + 1) // m
    kr = RNG.standard_normal((1, N, d)).astype(np.float32)
    vr = RNG.standard_normal((1, N, d)).astype(np.float32)
    kc = RNG.standard_normal((1, N // m, d)).astype(np.float32)
    vc = RNG.standard_normal((1, N // m, d)).astype(np.float32)
    q = RNG.standard_normal((1, H, d)).astype(np.float32)
    a, la = oracle.attn_rows(q, [0], [p], kc, vc, m, None, kr, vr, W, 0.5)
    b, lb = oracle.attn_rows(q, [0], [p], kc, vc, m, np.arange(E, dtype=np.int32)[None], kr, vr, W, 0.5)
    np.testing.assert_allclose(a, b, atol=1e-14)
    np.testing.assert_allclose(la, lb, atol=1e-14)


def test_lse_merge_of_partition_equals_whole():
    N, H, d, W, m = 90, 3, 5, 6, 4
    p = 89
    kr = RNG.standard_normal((1, N, d)).astype(np.float32)
    vr = RNG.standard_normal((1, N, d)).astype(np.float32)
    kc = RNG.standard_normal((1, N // m, d)).astype(np.float32)
    vc = RNG.standard_normal((1, N // m, d)).astype(np.float32)
    q = RNG.standard_normal((1, H, d)).astype(np.float32)
    sel = np.array([1, 4, 5, 9, 12, 20], np.int32)
    whole, lw = oracle.attn_rows(q, [0], [p], kc, vc, m, sel[None], kr, vr, W, 0.4)
    pa, la = oracle.attn_rows(q, [0], [p], kc, vc, m, sel[None, :2], kr, vr, 0, 0.4)
    pb, lb = oracle.attn_rows(q, [0], [p], kc, vc, m, sel[None, 2:], kr, vr, 0, 0.4)
    pc, lc = oracle.attn_rows(q, [0], [p], kc, vc, m, np.full((1, 1), -1, np.int32), kr, vr, W, 0.4)
    pe, le = oracle.attn_rows(q, [0], [p], kc, vc, m, np.full((1, 1), -1, np.int32), kr, vr, 0, 0.4)
    merged, lm = oracle.lse_merge(np.stack([pa[0], pb[0], pe[0], pc[0]]), np.stack([la[0], lb[0], le[0], lc[0]]))
    np.testing.assert_allclose(merged, whole[0], atol=1e-13)
    np.testing.assert_allclose(lm, lw[0], atol=1e-13)


def test_pipeline_tiny_against_textbook():
    # compress (uniform weights = block mean) -> top-k -> attention, against an
    # independent numpy/torch construction of the same set and softmax.
    B, N, d, H, m, W, k, DI = 1, 48, 4, 2, 4, 5, 3, 6
    x_k = RNG.standard_normal((B, N, d)).astype(np.float32)
    x_v = RNG.standard_normal((B, N, d)).astype(np.float32)
    w = np.full(m, 0.25, np.float32)
    E = N // m
    kc = oracle.compress(x_k, w, m, [0], [N], E)
    vc = oracle.compress(x_v, w, m, [0], [N], E)
    kI = RNG.integers(-127, 128, size=(B, E, DI)).astype(np.int8)
    ps = np.arange(N, dtype=np.int64)
    qI = RNG.integers(-127, 128, size=(N, DI)).astype(np.int8)
    idx, cnt = oracle.index_topk_rows(qI, np.zeros(N, np.int64), ps, kI, m, k)
    q = RNG.standard_normal((N, H, d)).astype(np.float32)
    out, _ = oracle.attn_rows(q, np.zeros(N, np.int64), ps, kc, vc, m, idx, x_k, x_v, W, 1 / math.sqrt(d))
    kc_ref = x_k[0].astype(np.float64).reshape(E, m, d).mean(1)
    vc_ref = x_v[0].astype(np.float64).reshape(E, m, d).mean(1)
    keys = np.concatenate([kc_ref, x_k[0]])
    vals = np.concatenate([vc_ref, x_v[0]])
    for p in range(N):
        Ep = (p + 1) // m
        s = kI[0, :Ep].astype(np.int64) @ qI[p].astype(np.int64)
        order = sorted(range(Ep), key=lambda j: (-s[j], j))[:k]
        mask = np.zeros((1, E + N), bool)
        mask[0, order] = True
        mask[0, E + max(0, p - W + 1):E + p + 1] = True
        ref = _sdpa(q[p:p + 1], keys, vals, mask)
        np.testing.assert_allclose(out[p], ref[0], atol=1e-12)
        assert sorted(order) == idx[p][:cnt[p]].tolist()


# ------------------------------------------------ V4 attention details ---
# (QbitAI article, hybrid attention: the Q/KV normalisation, partial RoPE, shared
# K=V entry with the output's inverse rotation, and attention sink paragraphs)

def _rms(x, gamma=None, eps=1e-6):
    x = np.asarray(x, dtype=np.float64)
    y = x / np.sqrt((x * x).mean(-1, keepdims=True) + eps)
    return y if gamma is None else y * gamma


def _rot(x, pos, rd, theta=10000.0):
    """rotate channel pairs (d-rd+2k, d-rd+2k+1) by pos * theta^(-2k/rd) (numpy, complex form)"""
    x = np.array(x, dtype=np.float64)
    d = x.shape[-1]
    k = np.arange(rd // 2)
    ang = np.asarray(pos, dtype=np.float64)[..., None] * theta ** (-2.0 * k / rd)
    z = (x[..., d - rd::2] + 1j * x[..., d - rd + 1::2]) * np.exp(1j * ang)
    x[..., d - rd::2], x[..., d - rd + 1::2] = z.real, z.imag
    return x


def _v4_case(seed, B=1, E_cap=16, m=4, H=3, d=16, N=None):
    g = np.random.default_rng(seed)
    N = N or E_cap * m
    return (g.standard_normal((B, 1, H, d)), g.standard_normal((B, E_cap, d)) * 3,
            g.standard_normal((B, N, d)) * 2, g.uniform(0.5, 1.5, d), g.uniform(0.5, 1.5, d))


def test_v4_without_rope_is_plain_attention_on_normalised_inputs():
    q, ent, raw, gq, gk = _v4_case(1)
    m, W, p = 4, 5, 50
    o, l = oracle.attn_v4_rows(q[0], [0], [p], ent, m, None, raw, W, 0.3, gq, gk, 1e-6, 0, 10000.0, None)
    ro, rl = oracle.attn_rows(_rms(q[0], gq), [0], [p], _rms(ent, gk), _rms(ent, gk), m, None, _rms(raw, gk),
                              _rms(raw, gk), W, 0.3)
    np.testing.assert_allclose(o, ro, atol=1e-12)
    np.testing.assert_allclose(l, rl, atol=1e-12)


@pytest.mark.parametrize("rd", [2, 8, 16])
def test_v4_one_item_is_relative_rotation(rd):
    """one attended entry: softmax weight 1, out = R(t - p) N(e) in closed form"""
    q, ent, raw, gq, gk = _v4_case(2)
    m, p, j = 4, 61, 9
    idx = np.full((1, 4), -1, np.int32)
    idx[0, 2] = j
    o, l = oracle.attn_v4_rows(q[0], [0], [p], ent, m, idx, raw, 0, 0.7, gq, gk, 1e-6, rd, 10000.0, None)
    t = (j + 1) * m - 1
    want = _rot(_rms(ent[0, j], gk), t - p, rd)
    for h in range(q.shape[2]):
        np.testing.assert_allclose(o[0, h], want, atol=1e-12)
        qv = _rot(_rms(q[0, 0, h], gq), p, rd)
        kv = _rot(_rms(ent[0, j], gk), t, rd)
        assert abs(l[0, h] - 0.7 * qv @ kv) < 1e-12


def test_v4_shift_of_every_position_leaves_output_unchanged():
    """window-only attention at positions p and p + shift over the same token vectors"""
    g = np.random.default_rng(3)
    d, H, W, shift = 16, 2, 6, 37
    q = g.standard_normal((1, H, d))
    toks = g.standard_normal((W, d))
    N = 200
    ent = np.zeros((1, N, d))
    outs = []
    for p in (80, 80 + shift):
        raw = np.zeros((1, N, d))
        raw[0, p - W + 1:p + 1] = toks
        outs.append(oracle.attn_v4_rows(q, [0], [p], ent, 1, np.full((1, 1), -1, np.int32), raw, W, 0.25,
                                        None, None, 1e-6, 16, 10000.0, None)[0])
    np.testing.assert_allclose(outs[0], outs[1], atol=1e-10)


def test_v4_sink_weight_closed_form_and_limit():
    q, ent, raw, gq, gk = _v4_case(4)
    m, p, j = 4, 40, 3
    idx = np.array([[j]], np.int32)
    base, bl = oracle.attn_v4_rows(q[0], [0], [p], ent, m, idx, raw, 0, 0.5, gq, gk, 1e-6, 8, 10000.0, None)
    z = np.array([0.3, -1.0, 2.0])
    o, l = oracle.attn_v4_rows(q[0], [0], [p], ent, m, idx, raw, 0, 0.5, gq, gk, 1e-6, 8, 10000.0, z)
    w = np.exp(bl[0]) / (np.exp(bl[0]) + np.exp(z))           # one item: weight e^l / (e^l + e^z)
    np.testing.assert_allclose(o[0], base[0] * w[:, None], atol=1e-12)
    np.testing.assert_allclose(l[0], np.logaddexp(bl[0], z), atol=1e-12)
    o2, l2 = oracle.attn_v4_rows(q[0], [0], [p], ent, m, idx, raw, 0, 0.5, gq, gk, 1e-6, 8, 10000.0,
                                 np.full(3, -np.inf))
    np.testing.assert_allclose(o2, base, atol=0)
    # sink only (empty set): out 0, lse = z
    o3, l3 = oracle.attn_v4_rows(q[0], [0], [p], ent, m, np.full((1, 1), -1, np.int32), raw, 0, 0.5, gq, gk,
                                 1e-6, 8, 10000.0, z)
    assert not o3.any() and np.allclose(l3[0], z)


# ------------------------------------------------- learned compressor ---
# (QbitAI article, hybrid attention: CSA step 1 -- attention-like merge with learned
# weights -- and the HCA paragraph -- no overlap; window/score reading in hsa_oracle.c)

def _kv(seed, B=2, N=40, d=8):
    g = np.random.default_rng(seed)
    return g.standard_normal((B, N, d)), g.standard_normal((B, N, d)), g.standard_normal(d)


def test_learned_zero_scores_is_block_mean():
    k, v, _ = _kv(1)
    m = 4
    kc, vc = oracle.compress_learned(k, v, np.zeros(8), np.zeros(m), m, m, [0, 4], [40, 37], 10)
    rk = oracle.compress(k, np.full(m, 1.0 / m), m, [0, 4], [40, 37], 10)
    rv = oracle.compress(v, np.full(m, 1.0 / m), m, [0, 4], [40, 37], 10)
    np.testing.assert_allclose(kc, rk, atol=1e-14)
    np.testing.assert_allclose(vc, rv, atol=1e-14)


@pytest.mark.parametrize("r", [0, 3, 5, 7])
def test_learned_one_open_bias_copies_that_token(r):
    k, v, u = _kv(2)
    m, L = 4, 8
    bias = np.full(L, -np.inf)
    bias[r] = 0.0
    kc, vc = oracle.compress_learned(k, v, u, bias, m, L, [8, 8], [40, 40], 10)
    for j in range(2, 10):
        t = (j + 1) * m - L + r
        np.testing.assert_array_equal(kc[:, j], k[:, t])
        np.testing.assert_array_equal(vc[:, j], v[:, t])


def test_learned_bias_shift_and_masked_overlap():
    k, v, u = _kv(3)
    m = 4
    bias = np.random.default_rng(4).standard_normal(2 * m)
    a = oracle.compress_learned(k, v, u, bias, m, 2 * m, [0, 0], [40, 40], 10)
    b = oracle.compress_learned(k, v, u, bias + 3.7, m, 2 * m, [0, 0], [40, 40], 10)
    np.testing.assert_allclose(a[0], b[0], atol=1e-12)
    np.testing.assert_allclose(a[1], b[1], atol=1e-12)
    # the earlier block masked out: the same as no overlap
    masked = np.concatenate([np.full(m, -np.inf), bias[m:]])
    c = oracle.compress_learned(k, v, u, masked, m, 2 * m, [0, 0], [40, 40], 10)
    d = oracle.compress_learned(k, v, u, bias[m:], m, m, [0, 0], [40, 40], 10)
    np.testing.assert_allclose(c[0], d[0], atol=1e-14)
    np.testing.assert_allclose(c[1], d[1], atol=1e-14)


def test_learned_weights_follow_scores():
    """two-token window, closed form: a_1 = sigmoid(s_1 - s_0)"""
    k, v, u = _kv(5, B=1, N=12, d=6)
    m, L = 1, 2
    bias = np.array([0.2, -0.5])
    kc, vc = oracle.compress_learned(k, v, u, bias, m, L, [1], [12], 12)
    for j in range(1, 12):
        s0, s1 = u @ k[0, j - 1] + bias[0], u @ k[0, j] + bias[1]
        a1 = 1.0 / (1.0 + np.exp(s0 - s1))
        np.testing.assert_allclose(kc[0, j], (1 - a1) * k[0, j - 1] + a1 * k[0, j], atol=1e-12)
        np.testing.assert_allclose(vc[0, j], (1 - a1) * v[0, j - 1] + a1 * v[0, j], atol=1e-12)
    # entry 0 has only token 0 in range
    kc0, _ = oracle.compress_learned(k, v, u, bias, m, L, [0], [1], 12)
    np.testing.assert_allclose(kc0[0, 0], k[0, 0], atol=1e-15)
