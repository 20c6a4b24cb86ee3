"""hsa_compress_append (partial-block state cache): tokens appended in chunks of
any size give entries bit-identical to hsa_compress over the same tokens, within
tolerance of the oracle's fp64 compression, and states equal to the partial sums
of the incomplete blocks."""
import numpy as np
import pytest
import torch

import oracle
from tests.hsa_testlib import assert_close_out, host_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from compressed_attention_compress_b300 import _lib
    oracle.build()
    return _lib


@pytest.mark.parametrize("dtype,d,m", [(torch.bfloat16, 128, 4), (torch.bfloat16, 128, 128), (torch.float32, 64, 3)])
def test_append_matches_batch_compress(lib, dtype, d, m):
    dev = torch.device("cuda")
    B, N = 3, 1100
    E_cap = N // m + 1
    g = torch.Generator().manual_seed(90 + m)
    k = torch.randn((B, N, d), generator=g).to(dtype)
    v = torch.randn((B, N, d), generator=g).to(dtype)
    w = torch.rand((m,), generator=g, dtype=torch.float64) + 1e-3
    w = (w / w.sum()).to(torch.float32)
    starts = [0, m * 3, m * 7]  # each sequence starts at a block boundary
    chunks = [1, 1, 3, 7, 1, 64, 2, 129, 1, 5, 300, 1, 1, 17]
    kd, vd, wd = k.to(dev), v.to(dev), w.to(dev)
    kc = torch.zeros((B, E_cap, d), dtype=dtype, device=dev)
    vc = torch.zeros_like(kc)
    st_k = torch.full((B, d), float("nan"), dtype=torch.float32, device=dev)  # no initial value needed
    st_v = torch.full((B, d), float("nan"), dtype=torch.float32, device=dev)
    pos = list(starts)
    for T in chunks:
        T = min(T, N - max(pos))
        if T <= 0:
            break
        kn = torch.stack([kd[b, pos[b]:pos[b] + T] for b in range(B)])
        vn = torch.stack([vd[b, pos[b]:pos[b] + T] for b in range(B)])
        lib.hsa_compress_append(kn, vn, torch.tensor(pos, dtype=torch.int64, device=dev), wd, m, st_k, st_v, kc, vc)
        pos = [p + T for p in pos]
    # the same blocks through the batch kernel
    kc2 = torch.zeros_like(kc)
    vc2 = torch.zeros_like(vc)
    lib.hsa_compress(kd, vd, torch.tensor(starts, device=dev), torch.tensor(pos, device=dev),
                     max((pos[b] // m) - (starts[b] // m) for b in range(B)), wd, m, kc2, vc2)
    lib.hsa_check()
    assert torch.equal(kc.view(torch.int16 if dtype == torch.bfloat16 else torch.int32),
                       kc2.view(torch.int16 if dtype == torch.bfloat16 else torch.int32))
    assert torch.equal(vc.view(torch.int16 if dtype == torch.bfloat16 else torch.int32),
                       vc2.view(torch.int16 if dtype == torch.bfloat16 else torch.int32))
    # against the oracle, block by block, and the states against the partial sums
    for b in range(B):
        j0, j1 = starts[b] // m, pos[b] // m
        ref = oracle.compress(host_np(k[b:b + 1]), w.numpy(), m, [starts[b]], [pos[b]], E_cap)
        assert_close_out(kc[b:b + 1, j0:j1], ref[:, j0:j1], dtype, "kc")
        r = pos[b] % m
        if r:
            part = (w[:r].double()[:, None] * k[b, pos[b] - r:pos[b]].double()).sum(0).numpy()
            np.testing.assert_allclose(st_k[b].cpu().numpy(), part, atol=1e-5, rtol=1e-5)


def test_append_negative_position_flags(lib):
    dev = torch.device("cuda")
    d, m = 128, 4
    k = torch.zeros((1, 1, d), dtype=torch.bfloat16, device=dev)
    st = torch.zeros((1, d), dtype=torch.float32, device=dev)
    kc = torch.zeros((1, 8, d), dtype=torch.bfloat16, device=dev)
    lib.hsa_compress_append(k, k.clone(), torch.tensor([-1], device=dev), torch.full((m,), 0.25, device=dev), m,
                            st, st.clone(), kc, kc.clone())
    with pytest.raises(lib.HSAError) as ei:
        lib.hsa_check()
    assert ei.value.status == lib.HSA_ERR_DEVICE_FLAG
