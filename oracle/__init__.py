"""CPU oracle for hybrid compressed/sparse attention -- TEST INFRASTRUCTURE ONLY.

Only the test-suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` import this package.  The product library never imports, links or
calls it, and it shares no code with the CUDA path: the arithmetic lives in
``hsa_oracle.c`` (plain C, fp64), this module only marshals numpy arrays.

Each function below names the passage it follows; the C file carries the full
statement of the method and the readings taken where the pages are silent.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "hsa_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")

F32, BF16, F64 = 0, 1, 2
_ERRORS = {
    -1: "block, entry or token outside its buffer",
    -2: "indexer score does not fit in int32",
    -3: "selected index is not a visible entry",
    -4: "bad argument",
    -5: "out of host memory",
}


def build(force: bool = False) -> str:
    """Compile hsa_oracle.c into liboracle.so (gcc, fp64, no fast-math, OpenMP)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
               "-fno-fast-math", "-Wall", "-o", _LIB_PATH, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
    return _LIB_PATH


_lib = None


def _get():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        I64, I32, D = ctypes.c_int64, ctypes.c_int, ctypes.c_double
        lib.orc_num_entries.restype = I64
        lib.orc_num_entries.argtypes = [I64, I32]
        lib.orc_num_threads.restype = I32
        lib.orc_compress.restype = I32
        lib.orc_compress.argtypes = [P, I32, I32, I64, I32, P, P, P, I32, P, I32, I64]
        lib.orc_index_topk_rows.restype = I32
        lib.orc_index_topk_rows.argtypes = [I64, P, P, P, P, I32, I64, I32, I32, I32, P, P]
        lib.orc_attn_rows.restype = I32
        lib.orc_attn_rows.argtypes = [I64, P, I32, P, P, I32, I32, P, P, I32, I64, I32, P, I32,
                                      P, P, I32, I64, I32, D, P, P]
        lib.orc_lse_merge.restype = I32
        lib.orc_lse_merge.argtypes = [I32, P, P, I32, I32, P, P]
        lib.orc_compress_learned.restype = I32
        lib.orc_compress_learned.argtypes = [P, P, I32, I32, I64, I32, P, P, I32, I32, P, P, P, P, I32, I64]
        lib.orc_attn_v4_rows.restype = I32
        lib.orc_attn_v4_rows.argtypes = [I64, P, I32, P, P, I32, I32, P, I32, I64, I32, P, I32, P, I32, I64, I32,
                                         D, P, P, D, I32, D, P, P, P]
        _lib = lib
    return _lib


def _check(rc: int):
    if rc != 0:
        raise ValueError(f"oracle error {rc}: {_ERRORS.get(rc, 'unknown')}")


def _float_arr(x):
    """Return (contiguous array, dtype code). bf16 data travels as uint16 bit patterns."""
    x = np.ascontiguousarray(x)
    if x.dtype == np.float32:
        return x, F32
    if x.dtype == np.float64:
        return x, F64
    if x.dtype == np.uint16:
        return x, BF16
    raise TypeError(f"unsupported oracle dtype {x.dtype}")


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def num_threads() -> int:
    return _get().orc_num_threads()


def num_entries(p: int, m: int) -> int:
    """E(p) = floor((p+1)/m): complete blocks ending at or before p (strict causality)."""
    return _get().orc_num_entries(int(p), int(m))


def compress(x, w, m, tok_begin, tok_end, E_cap, out_dtype=np.float64):
    """KV compression (QbitAI article, hybrid attention: CSA step 1 / HCA).

    x: [B, N_cap, d] float32/float64 or bf16 bits as uint16; w: [m] float32.
    Returns [B, E_cap, d] with entries j in [tok_begin/m, tok_end/m) filled,
    zeros elsewhere.
    """
    xa, xdt = _float_arr(x)
    B, N_cap, d = xa.shape
    w = np.ascontiguousarray(w, dtype=np.float32)
    assert w.shape == (m,)
    tb = np.ascontiguousarray(tok_begin, dtype=np.int64).reshape(B)
    te = np.ascontiguousarray(tok_end, dtype=np.int64).reshape(B)
    out = np.zeros((B, E_cap, d), dtype=out_dtype)
    odt = F64 if out.dtype == np.float64 else F32
    _check(_get().orc_compress(_ptr(xa), xdt, B, N_cap, d, _ptr(tb), _ptr(te), _ptr(w), m,
                               _ptr(out), odt, E_cap))
    return out


def index_topk_rows(q, row_b, row_p, kI, m, topk):
    """Lightning indexer + exact top-k (QbitAI article, hybrid attention: CSA step 2).

    q: [n_rows, DI] int8; kI: [B, E_cap, DI] int8.  Returns (idx [n_rows, topk]
    int32 ascending and -1 padded, cnt [n_rows] int32).
    """
    q = np.ascontiguousarray(q, dtype=np.int8)
    kI = np.ascontiguousarray(kI, dtype=np.int8)
    n_rows, DI = q.shape
    B, E_cap, DI2 = kI.shape
    assert DI == DI2
    rb = np.ascontiguousarray(row_b, dtype=np.int64).reshape(n_rows)
    rp = np.ascontiguousarray(row_p, dtype=np.int64).reshape(n_rows)
    idx = np.empty((n_rows, max(topk, 0)), dtype=np.int32)
    cnt = np.empty((n_rows,), dtype=np.int32)
    _check(_get().orc_index_topk_rows(n_rows, _ptr(q), _ptr(rb), _ptr(rp), _ptr(kI), B, E_cap, DI,
                                      m, topk, _ptr(idx), _ptr(cnt)))
    return idx, cnt


def attn_rows(q, row_b, row_p, kc, vc, m, idx, k_raw, v_raw, window, scale):
    """Attention over selected (or all) compressed entries plus the raw window, one softmax.

    QbitAI article, hybrid attention: CSA step 3 (MQA over the top-k), HCA (dense),
    and the sliding-window paragraph.  q: [n_rows, H, d]; kc, vc: [B, E_cap, d];
    idx: [n_rows, topk] int32 or None (dense); k_raw, v_raw: [B, N_cap, d].
    Returns (out [n_rows, H, d] float64, lse [n_rows, H] float64).
    """
    qa, qdt = _float_arr(q)
    n_rows, H, d = qa.shape
    kca, cdt = _float_arr(kc)
    vca, cdt2 = _float_arr(vc)
    assert cdt == cdt2 and kca.shape == vca.shape
    B, E_cap, d2 = kca.shape
    kra, rdt = _float_arr(k_raw)
    vra, rdt2 = _float_arr(v_raw)
    assert rdt == rdt2 and kra.shape == vra.shape
    _, N_cap, d3 = kra.shape
    assert d == d2 == d3
    rb = np.ascontiguousarray(row_b, dtype=np.int64).reshape(n_rows)
    rp = np.ascontiguousarray(row_p, dtype=np.int64).reshape(n_rows)
    if idx is None:
        ia, topk, iptr = None, 0, None
    else:
        ia = np.ascontiguousarray(idx, dtype=np.int32)
        assert ia.shape[0] == n_rows
        topk = ia.shape[1]
        iptr = _ptr(ia)
    out = np.empty((n_rows, H, d), dtype=np.float64)
    lse = np.empty((n_rows, H), dtype=np.float64)
    _check(_get().orc_attn_rows(n_rows, _ptr(qa), qdt, _ptr(rb), _ptr(rp), H, d, _ptr(kca), _ptr(vca),
                                cdt, E_cap, m, iptr, topk, _ptr(kra), _ptr(vra), rdt, N_cap,
                                window, float(scale), _ptr(out), _ptr(lse)))
    return out, lse


def lse_merge(o_parts, lse_parts):
    """Log-sum-exp merge of attention over disjoint parts of one set (split-KV decode).

    o_parts: [S, H, d] float64; lse_parts: [S, H] float64 -> (out [H, d], lse [H]).
    """
    o = np.ascontiguousarray(o_parts, dtype=np.float64)
    ls = np.ascontiguousarray(lse_parts, dtype=np.float64)
    S, H, d = o.shape
    out = np.empty((H, d), dtype=np.float64)
    lse = np.empty((H,), dtype=np.float64)
    _check(_get().orc_lse_merge(S, _ptr(o), _ptr(ls), H, d, _ptr(out), _ptr(lse)))
    return out, lse


def attn_v4_rows(q, row_b, row_p, ent, m, idx, raw, window, scale, gamma_q=None, gamma_kv=None, eps=1e-6,
                 rope_dims=64, theta=10000.0, sink=None):
    """V4 attention details (QbitAI article, hybrid attention: the Q/KV normalisation,
    partial RoPE, shared K=V entry with the output's inverse rotation, and attention
    sink paragraphs) over the same set as attn_rows.  q: [n_rows, H, d]; ent: [B, E_cap, d]
    (key and value); raw: [B, N_cap, d]; gamma_*: [d] or None; sink: [H] or None.
    Returns (out [n_rows, H, d] float64, lse [n_rows, H] float64)."""
    qa, qdt = _float_arr(q)
    n_rows, H, d = qa.shape
    ea, edt = _float_arr(ent)
    B, E_cap, d2 = ea.shape
    ra, rdt = _float_arr(raw)
    _, N_cap, d3 = ra.shape
    assert d == d2 == d3
    rb = np.ascontiguousarray(row_b, dtype=np.int64).reshape(n_rows)
    rp = np.ascontiguousarray(row_p, dtype=np.int64).reshape(n_rows)
    if idx is None:
        iptr, topk = None, 0
    else:
        ia = np.ascontiguousarray(idx, dtype=np.int32)
        iptr, topk = _ptr(ia), ia.shape[1]
    gq = None if gamma_q is None else np.ascontiguousarray(gamma_q, dtype=np.float64)
    gk = None if gamma_kv is None else np.ascontiguousarray(gamma_kv, dtype=np.float64)
    sk = None if sink is None else np.ascontiguousarray(sink, dtype=np.float64)
    out = np.empty((n_rows, H, d), dtype=np.float64)
    lse = np.empty((n_rows, H), dtype=np.float64)
    _check(_get().orc_attn_v4_rows(n_rows, _ptr(qa), qdt, _ptr(rb), _ptr(rp), H, d, _ptr(ea), edt, E_cap, m, iptr,
                                   topk, _ptr(ra), rdt, N_cap, window, float(scale),
                                   None if gq is None else _ptr(gq), None if gk is None else _ptr(gk), float(eps),
                                   int(rope_dims), float(theta), None if sk is None else _ptr(sk), _ptr(out),
                                   _ptr(lse)))
    return out, lse


def compress_learned(k, v, u, bias, m, L, tok_begin, tok_end, E_cap, out_dtype=np.float64):
    """Learned, attention-like compression (QbitAI article, hybrid attention: CSA step 1
    and the HCA paragraph; the window/score reading is stated in hsa_oracle.c).
    k, v: [B, N_cap, d]; u: [d]; bias: [L].  Returns (kc, vc) [B, E_cap, d]."""
    ka, kdt = _float_arr(k)
    va, vdt = _float_arr(v)
    assert kdt == vdt and ka.shape == va.shape
    B, N_cap, d = ka.shape
    ua = np.ascontiguousarray(u, dtype=np.float64)
    ba = np.ascontiguousarray(bias, dtype=np.float64)
    assert ua.shape == (d,) and ba.shape == (L,)
    tb = np.ascontiguousarray(tok_begin, dtype=np.int64)
    te = np.ascontiguousarray(tok_end, dtype=np.int64)
    kc = np.zeros((B, E_cap, d), dtype=out_dtype)
    vc = np.zeros((B, E_cap, d), dtype=out_dtype)
    code = 2 if out_dtype == np.float64 else 0
    _check(_get().orc_compress_learned(_ptr(ka), _ptr(va), kdt, B, N_cap, d, _ptr(ua), _ptr(ba), m, L, _ptr(tb),
                                       _ptr(te), _ptr(kc), _ptr(vc), code, E_cap))
    return kc, vc

