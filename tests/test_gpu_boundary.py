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
