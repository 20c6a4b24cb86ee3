"""CPU checks of the C-ABI library: it builds, loads without a GPU, exports every
symbol include/hsa.h declares, and rejects bad host arguments before touching
the device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "hsa.h")).read()
    return sorted(set(re.findall(r"HSA_API\s+[\w\s\*]+?\b(hsa_\w+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    from compressed_attention_compress_b300 import build
    build.build()
    from compressed_attention_compress_b300 import _lib
    return _lib


def test_header_declares_the_boundary():
    names = _declared()
    for n in ("hsa_compress", "hsa_index_topk", "hsa_attn_decode", "hsa_attn_prefill", "hsa_last_error",
              "hsa_check", "hsa_index_topk_workspace_size", "hsa_attn_decode_workspace_size"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    raw = ctypes.CDLL(lib.LIB_PATH)
    for n in _declared():
        assert hasattr(raw, n), n
    assert sorted(lib.EXPORTS) == _declared()


def test_version_and_empty_error(lib):
    assert lib.lib.hsa_version() >= 100
    assert isinstance(lib.lib.hsa_last_error(), bytes)


def test_host_validation_without_device(lib):
    L = lib.lib
    # negative batch: rejected before any CUDA call
    st = L.hsa_compress(None, None, lib.HSA_BF16, -1, 128, 0, 0, 0, None, None, 0, None, 4, None, None, 0, 0, 0,
                        None)
    assert st == lib.HSA_ERR_INVALID_ARG and b"bad size" in L.hsa_last_error()
    # unsupported dtype
    st = L.hsa_compress(None, None, 7, 1, 128, 0, 0, 0, None, None, 1, None, 4, None, None, 0, 0, 0, None)
    assert st == lib.HSA_ERR_UNSUPPORTED
    # unsupported indexer dim / topk
    st = L.hsa_index_topk(None, 0, 0, None, 0, 0, 10, 1, 1, 48, None, 4, 8, None, None, None, 0, None)
    assert st == lib.HSA_ERR_UNSUPPORTED
    st = L.hsa_index_topk(None, 0, 0, None, 0, 0, 10, 1, 1, 64, None, 4, 0, None, None, None, 0, None)
    assert st == lib.HSA_ERR_UNSUPPORTED
    # null pointers with work to do
    st = L.hsa_index_topk(None, 0, 0, None, 0, 0, 10, 1, 1, 64, None, 4, 8, None, None, None, 0, None)
    assert st == lib.HSA_ERR_INVALID_ARG
    # empty work is a no-op success
    st = L.hsa_index_topk(None, 0, 0, None, 0, 0, 10, 0, 1, 64, None, 4, 8, None, None, None, 0, None)
    assert st == lib.HSA_OK
    # bf16 attention with an unsupported head dim is refused on the host
    st = L.hsa_attn_prefill(ctypes.c_void_p(16), lib.HSA_BF16, 1, 1, 16, 96, ctypes.c_void_p(16), ctypes.c_void_p(16),
                            96, 96, 4, 4, None, None, 0, ctypes.c_void_p(16), ctypes.c_void_p(16), 96, 96, 16, 8,
                            ctypes.c_void_p(16), 0.1, ctypes.c_void_p(16), None, None, 0, None)
    assert st == lib.HSA_ERR_UNSUPPORTED


def test_python_binding_refuses_to_run_without_the_library(tmp_path, monkeypatch):
    import importlib
    import compressed_attention_compress_b300._lib as L
    monkeypatch.setattr(L, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(ImportError):
        L._load()
    importlib.reload(L)


def test_pointer_classifier_refuses_without_a_device(lib):
    # no GPU here: nothing can be classified as device memory
    import numpy as np
    a = np.zeros(16, dtype=np.uint8)
    assert lib.lib.hsa_check_pointer(a.ctypes.data) == lib.HSA_ERR_INVALID_ARG
    assert lib.lib.hsa_check_pointer(None) == lib.HSA_ERR_INVALID_ARG
