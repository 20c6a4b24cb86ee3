"""The boundary's pointer classifier on a GPU: device memory of the current
device is accepted, host memory (pinned or pageable) is refused before anything
is enqueued.  Only the classifier itself is called with host addresses; no
launching entry point ever receives one."""
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


def test_device_memory_is_accepted(lib):
    t = torch.zeros(1024, dtype=torch.uint8, device="cuda")
    lib.hsa_check_pointer(t.data_ptr())
    lib.hsa_check_pointer(t[256:].data_ptr())  # inside an allocation


def test_pinned_host_memory_is_refused(lib):
    t = torch.zeros(1024, dtype=torch.uint8).pin_memory()
    with pytest.raises(lib.HSAError) as e:
        lib.hsa_check_pointer(t.data_ptr())
    assert e.value.status == lib.HSA_ERR_INVALID_ARG and "pinned" in str(e.value)


def test_pageable_host_memory_is_refused(lib):
    a = np.zeros(1024, dtype=np.uint8)
    with pytest.raises(lib.HSAError) as e:
        lib.hsa_check_pointer(a.ctypes.data)
    assert e.value.status == lib.HSA_ERR_INVALID_ARG and "pageable" in str(e.value)


def test_null_is_refused(lib):
    with pytest.raises(lib.HSAError) as e:
        lib.hsa_check_pointer(0)
    assert e.value.status == lib.HSA_ERR_INVALID_ARG


def _v4_decode_args(lib, H=64, d=128, dtype=torch.bfloat16, topk=128):
    B, m, W, E_cap = 1, 4, 128, 512
    dev = "cuda"
    q = torch.zeros((B, H, d), dtype=dtype, device=dev)
    kc = torch.zeros((B, E_cap, d), dtype=dtype, device=dev)
    raw = torch.zeros((B, E_cap * m, d), dtype=dtype, device=dev)
    idx = torch.zeros((B, topk), dtype=torch.int32, device=dev)
    ctx = torch.full((B,), E_cap * m, dtype=torch.int64, device=dev)
    out = torch.empty((B, H, d), dtype=dtype, device=dev)
    lse = torch.empty((B, H), dtype=torch.float32, device=dev)
    n = lib.hsa_attn_decode_workspace_size(dtype, B, H, d, E_cap, m, topk, W)
    ws = lib.workspace(n, device=dev)
    return dict(q=q, kc=kc, vc=kc, m=m, idx=idx, cnt=None, k_raw=raw, v_raw=raw, window=W, ctx_len=ctx,
                scale=d ** -0.5, out=out, lse=lse, ws=ws)


def test_attn_decode_v4_refuses_other_paths(lib):
    # the fused V4 attention runs on the tensor-core CSA decode path only
    for kw in (dict(H=32), dict(dtype=torch.float32)):
        args = _v4_decode_args(lib, **kw)
        with pytest.raises(lib.HSAError) as e:
            lib.hsa_attn_decode_v4(**args)
        assert e.value.status == lib.HSA_ERR_UNSUPPORTED
    args = _v4_decode_args(lib)
    args["idx"] = None
    with pytest.raises(lib.HSAError) as e:
        lib.hsa_attn_decode_v4(**args)
    assert e.value.status == lib.HSA_ERR_UNSUPPORTED
    lib.hsa_check()  # nothing was enqueued


@pytest.mark.parametrize("bad", [dict(rope_dims=3), dict(rope_dims=130), dict(theta=0.0), dict(eps=-1.0)])
def test_attn_decode_v4_bad_parameters(lib, bad):
    args = _v4_decode_args(lib)
    with pytest.raises(lib.HSAError) as e:
        lib.hsa_attn_decode_v4(**args, **bad)
    assert e.value.status == lib.HSA_ERR_INVALID_ARG
    lib.hsa_check()


def test_compress_v4_bad_parameters(lib):
    B, N, d, m = 1, 64, 128, 4
    k = torch.zeros((B, N, d), dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros((B, N // m, d), dtype=torch.bfloat16, device="cuda")
    tb = torch.zeros(B, dtype=torch.int64, device="cuda")
    te = torch.full((B,), N, dtype=torch.int64, device="cuda")
    w = torch.full((m,), 1.0 / m, device="cuda")
    for bad, status in ((dict(rope_dims=5), lib.HSA_ERR_INVALID_ARG), (dict(theta=-1.0), lib.HSA_ERR_INVALID_ARG)):
        with pytest.raises(lib.HSAError) as e:
            lib.hsa_compress_v4(k, tb, te, N // m, w, m, kc, **bad)
        assert e.value.status == status
    k96 = torch.zeros((B, N, 96), dtype=torch.bfloat16, device="cuda")
    kc96 = torch.zeros((B, N // m, 96), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(lib.HSAError) as e:
        lib.hsa_compress_v4(k96, tb, te, N // m, w, m, kc96, rope_dims=32)
    assert e.value.status == lib.HSA_ERR_UNSUPPORTED  # d must be a multiple of 64
    lib.hsa_check()
