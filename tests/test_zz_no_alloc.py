"""hsa_index_topk_noalloc: the indexer for callers that cannot allocate device
memory (their memory belongs to another allocator's pool, or their host code may
not call cudaMalloc), so they cannot hand the library a workspace.  It must give
exactly what hsa_index_topk gives with a workspace, call after call, although
every call reuses the same built-in scratch.  Collected last on purpose."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from compressed_attention_compress_b300 import _lib
    return _lib


def _inputs(B, E, DI, seed, lo=-127, hi=127):
    g = torch.Generator().manual_seed(seed)
    q = torch.randint(lo, hi + 1, (B, 1, DI), generator=g, dtype=torch.int16).to(torch.int8)
    k = torch.randint(lo, hi + 1, (B, E, DI), generator=g, dtype=torch.int16).to(torch.int8)
    return q.cuda(), k.cuda()


def _with_workspace(lib, q, k, pos0, m, topk):
    B, T, DI = q.shape
    idx = torch.empty((B, T, topk), dtype=torch.int32, device="cuda")
    cnt = torch.empty((B, T), dtype=torch.int32, device="cuda")
    ws = lib.workspace(lib.hsa_index_topk_workspace_size(B, T, DI, k.shape[1], topk))
    lib.hsa_index_topk(q, k, pos0, m, topk, idx, cnt, ws)
    return idx, cnt


def _no_alloc(lib, q, k, pos0, m, topk):
    B, T, _ = q.shape
    idx = torch.full((B, T, topk), 7, dtype=torch.int32, device="cuda")
    cnt = torch.full((B, T), 7, dtype=torch.int32, device="cuda")
    lib.hsa_index_topk_noalloc(q, k, pos0, m, topk, idx, cnt)
    return idx, cnt


@pytest.mark.parametrize("shape", [(4, 262144, 64, 1024), (8, 32768, 64, 512)])
def test_no_alloc_matches_workspace_entry_point_on_two_calls(lib, shape):
    B, E, DI, topk = shape
    m = 4
    # two calls in a row with different inputs (the second one starts from whatever
    # the first left in the shared scratch); one row is short (fewer than k entries)
    for call, (seed, lo, hi) in enumerate([(11, -127, 127), (12, -1, 1)]):
        q, k = _inputs(B, E, DI, seed, lo, hi)
        pos0 = torch.full((B,), m * E - 1, dtype=torch.int64, device="cuda")
        pos0[1] = m * (topk // 2) + 1
        ref_idx, ref_cnt = _with_workspace(lib, q, k, pos0, m, topk)
        got_idx, got_cnt = _no_alloc(lib, q, k, pos0, m, topk)
        torch.cuda.synchronize()
        assert torch.equal(got_cnt, ref_cnt), f"call {call}: counts differ"
        assert torch.equal(got_idx, ref_idx), f"call {call}: indices differ"
    lib.hsa_check()


def test_no_alloc_rejects_sizes_beyond_its_scratch(lib):
    B, E, DI, topk, m = 64, 262144, 64, 1024, 4
    need = lib.hsa_index_topk_workspace_size(B, 1, DI, E, topk)
    assert need > lib.NOALLOC_SCRATCH_BYTES
    q = torch.zeros((B, 1, DI), dtype=torch.int8, device="cuda")
    k = torch.zeros((B, E, DI), dtype=torch.int8, device="cuda")
    pos0 = torch.full((B,), m * E - 1, dtype=torch.int64, device="cuda")
    idx = torch.empty((B, 1, topk), dtype=torch.int32, device="cuda")
    cnt = torch.empty((B, 1), dtype=torch.int32, device="cuda")
    with pytest.raises(lib.HSAError) as ei:
        lib.hsa_index_topk_noalloc(q, k, pos0, m, topk, idx, cnt)
    assert ei.value.status == lib.HSA_ERR_WORKSPACE
    assert str(lib.NOALLOC_SCRATCH_BYTES) in str(ei.value)
    # nothing was enqueued; a call within the limit still works
    q2, k2 = _inputs(2, 4096, DI, 13)
    pos2 = torch.full((2,), m * 4096 - 1, dtype=torch.int64, device="cuda")
    ref = _with_workspace(lib, q2, k2, pos2, m, 100)
    got = _no_alloc(lib, q2, k2, pos2, m, 100)
    assert torch.equal(got[0], ref[0]) and torch.equal(got[1], ref[1])
    lib.hsa_check()
