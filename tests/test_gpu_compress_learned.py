"""hsa_compress_learned (attention-like pooling with learned weights, overlapping CSA
windows) against the oracle's definition."""
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


@pytest.mark.parametrize("dtype,d,m,L,N", [(torch.bfloat16, 128, 4, 8, 4096), (torch.bfloat16, 128, 128, 128, 8192),
                                           (torch.float32, 64, 3, 6, 999)])
def test_learned_compress_parity(lib, dtype, d, m, L, N):
    dev = torch.device("cuda")
    B = 2
    E_cap = N // m + 2
    g = torch.Generator().manual_seed(50 + m)
    k = torch.randn((B, N, d), generator=g).to(dtype)
    v = torch.randn((B, N, d), generator=g).to(dtype)
    u = torch.randn((d,), generator=g) / d ** 0.5
    bias = torch.randn((L,), generator=g)
    tb, te = [0, 5 * m + 1], [N, N - 2 * m]
    kc = torch.zeros((B, E_cap, d), dtype=dtype, device=dev)
    vc = torch.zeros_like(kc)
    max_blocks = max(te[b] // m - tb[b] // m for b in range(B))
    lib.hsa_compress_learned(k.to(dev), v.to(dev), torch.tensor(tb, device=dev), torch.tensor(te, device=dev),
                             max_blocks, u.to(dev), bias.to(dev), m, kc, vc)
    lib.hsa_check()
    rk, rv = oracle.compress_learned(host_np(k), host_np(v), u.double().numpy(), bias.double().numpy(), m, L, tb, te,
                                     E_cap)
    assert_close_out(kc, rk, dtype, "kc")
    assert_close_out(vc, rv, dtype, "vc")
