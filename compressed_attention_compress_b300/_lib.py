"""Thin ctypes binding of libhsa.so (include/hsa.h).

Argument marshalling only: every step runs in the library's CUDA kernels.
Functions keep the C names; tensors are torch CUDA tensors (device memory and
streams come from torch), sizes and strides are taken from them.  There is no
CPU path: if the shared library is missing or fails to load, importing this
module raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libhsa.so")

HSA_OK, HSA_ERR_INVALID_ARG, HSA_ERR_UNSUPPORTED, HSA_ERR_WORKSPACE, HSA_ERR_CUDA, HSA_ERR_DEVICE_FLAG = range(6)
HSA_F32, HSA_BF16 = 0, 1
_STATUS = {0: "HSA_OK", 1: "HSA_ERR_INVALID_ARG", 2: "HSA_ERR_UNSUPPORTED", 3: "HSA_ERR_WORKSPACE",
           4: "HSA_ERR_CUDA", 5: "HSA_ERR_DEVICE_FLAG"}

# every symbol include/hsa.h declares
EXPORTS = ["hsa_last_error", "hsa_version", "hsa_check", "hsa_check_pointer", "hsa_compress", "hsa_compress_v4", "hsa_compress_append", "hsa_compress_learned", "hsa_index_topk_workspace_size",
           "hsa_index_topk", "hsa_index_topk_noalloc", "hsa_attn_decode_workspace_size", "hsa_attn_decode", "hsa_attn_decode_v4", "hsa_decode_csa_workspace_size", "hsa_decode_csa",
           "hsa_attn_prefill_workspace_size", "hsa_attn_prefill", "hsa_index_scores", "hsa_topk_merge",
           "hsa_lse_merge", "hsa_rmsnorm_rope", "hsa_attn_finalize"]
NOALLOC_SCRATCH_BYTES = 16 << 20


class HSAError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{_STATUS.get(status, status)}: {msg}")
        self.status = status


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with `python -m compressed_attention_compress_b300.build`")
    lib = ctypes.CDLL(LIB_PATH)
    P, I, I64, SZ, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float
    lib.hsa_last_error.restype = ctypes.c_char_p
    lib.hsa_last_error.argtypes = []
    lib.hsa_version.restype = I
    lib.hsa_check.restype = I
    lib.hsa_check.argtypes = [P]
    lib.hsa_check_pointer.restype = I
    lib.hsa_check_pointer.argtypes = [P]
    lib.hsa_compress.restype = I
    lib.hsa_compress.argtypes = [P, P, I, I, I, I64, I64, I64, P, P, I64, P, I, P, P, I64, I64, I64, P]
    lib.hsa_compress_v4.restype = I
    lib.hsa_compress_v4.argtypes = [P, I, I, I, I64, I64, I64, P, P, I64, P, I, P, I64, I64, I64, P, F, I, F, P]
    lib.hsa_compress_learned.restype = I
    lib.hsa_compress_learned.argtypes = [P, P, I, I, I, I64, I64, I64, P, P, I64, P, P, I, I, P, P, I64, I64, I64, P]
    lib.hsa_compress_append.restype = I
    lib.hsa_compress_append.argtypes = [P, P, I, I, I, I, I64, I64, P, P, I, P, P, I64, P, P, I64, I64, I64, P]
    lib.hsa_index_topk_workspace_size.restype = I
    lib.hsa_index_topk_workspace_size.argtypes = [I, I, I, I64, I, ctypes.POINTER(SZ)]
    lib.hsa_index_topk.restype = I
    lib.hsa_index_topk.argtypes = [P, I64, I64, P, I64, I64, I64, I, I, I, P, I, I, P, P, P, SZ, P]
    lib.hsa_index_topk_noalloc.restype = I
    lib.hsa_index_topk_noalloc.argtypes = [P, I64, I64, P, I64, I64, I64, I, I, I, P, I, I, P, P, P]
    lib.hsa_attn_decode_workspace_size.restype = I
    lib.hsa_attn_decode_workspace_size.argtypes = [I, I, I, I, I64, I, I, I, ctypes.POINTER(SZ)]
    lib.hsa_attn_decode.restype = I
    lib.hsa_attn_decode.argtypes = [P, I, I, I, I, P, P, I64, I64, I64, I, P, P, I, P, P, I64, I64, I64, I, P, F,
                                    P, P, P, SZ, P]
    lib.hsa_attn_decode_v4.restype = I
    # as hsa_attn_decode, with gamma_q, eps, rope_dims, theta and sink before out
    lib.hsa_attn_decode_v4.argtypes = lib.hsa_attn_decode.argtypes[:22] + [P, F, I, F, P] + lib.hsa_attn_decode.argtypes[22:]
    lib.hsa_decode_csa_workspace_size.restype = I
    lib.hsa_decode_csa_workspace_size.argtypes = [I, I, I, I, I64, ctypes.POINTER(SZ)]
    lib.hsa_decode_csa.restype = I
    lib.hsa_decode_csa.argtypes = [P, I64, P, I64, I64, I64, I, I, I, P, P, P, I, I, I, I, P, P, I64, I64, P, P, I64,
                                   I64, I64, I, P, F, P, P, P, SZ, P]
    lib.hsa_attn_prefill_workspace_size.restype = I
    lib.hsa_attn_prefill_workspace_size.argtypes = [I, I, I, I, I, I64, I, I, I, ctypes.POINTER(SZ)]
    lib.hsa_attn_prefill.restype = I
    lib.hsa_attn_prefill.argtypes = [P, I, I, I, I, I, P, P, I64, I64, I64, I, P, P, I, P, P, I64, I64, I64, I, P,
                                     F, P, P, P, SZ, P]
    lib.hsa_index_scores.restype = I
    lib.hsa_index_scores.argtypes = [P, I64, I64, P, I64, I64, I64, I, I, I, P, P, I, P, P]
    lib.hsa_topk_merge.restype = I
    lib.hsa_topk_merge.argtypes = [P, P, I, I, I, P, P, P]
    lib.hsa_lse_merge.restype = I
    lib.hsa_lse_merge.argtypes = [P, P, I, I, I, I, I, P, P, P]
    lib.hsa_rmsnorm_rope.restype = I
    lib.hsa_rmsnorm_rope.argtypes = [P, I, I, I, I, I64, I64, I64, P, P, I64, P, I64, I64, P, F, I, F, P]
    lib.hsa_attn_finalize.restype = I
    lib.hsa_attn_finalize.argtypes = [P, P, I, I, I, I, I, P, P, I, F, P]
    return lib


lib = _load()


def _chk(status: int):
    if status != HSA_OK:
        raise HSAError(status, lib.hsa_last_error().decode())


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _dt(t):
    if t.dtype == torch.bfloat16:
        return HSA_BF16
    if t.dtype == torch.float32:
        return HSA_F32
    raise HSAError(HSA_ERR_UNSUPPORTED, f"dtype {t.dtype}")


def hsa_check(stream=None):
    _chk(lib.hsa_check(_stream(stream)))


def hsa_check_pointer(ptr: int):
    """Raise HSAError unless the address `ptr` is device memory of the current device (or managed)."""
    _chk(lib.hsa_check_pointer(ctypes.c_void_p(ptr)))


def hsa_compress_v4(k, tok_begin, tok_end, max_blocks, w, m, kc, gamma=None, eps=1e-6, rope_dims=64, theta=10000.0,
                    stream=None):
    """k [B, N_cap, d] -> kc [B, E_cap, d]: compressed V4 entries (one entry is key and value),
    normalised with gamma and rotated to their block's last token as they are written."""
    B, N_cap, d = k.shape
    _chk(lib.hsa_compress_v4(_p(k), _dt(k), B, d, k.stride(0), k.stride(1), N_cap, _p(tok_begin), _p(tok_end),
                             int(max_blocks), _p(w), int(m), _p(kc), kc.stride(0), kc.stride(1), kc.shape[1],
                             _p(gamma), float(eps), int(rope_dims), float(theta), _stream(stream)))


def hsa_compress(k, v, tok_begin, tok_end, max_blocks, w, m, kc, vc, stream=None):
    """k, v [B, N_cap, d]; kc, vc [B, E_cap, d] (channel stride 1); tok_* int64 [B] on device."""
    B, N_cap, d = k.shape
    assert v.shape == k.shape and v.stride() == k.stride() and kc.stride() == vc.stride()
    _chk(lib.hsa_compress(_p(k), _p(v), _dt(k), B, d, k.stride(0), k.stride(1), N_cap, _p(tok_begin), _p(tok_end),
                          int(max_blocks), _p(w), int(m), _p(kc), _p(vc), kc.stride(0), kc.stride(1), kc.shape[1],
                          _stream(stream)))


def hsa_compress_learned(k, v, tok_begin, tok_end, max_blocks, u, bias, m, kc, vc, stream=None):
    """Learned attention-like compression: window L = bias.numel() tokens ending at each block's last token."""
    B, N_cap, d = k.shape
    assert v.shape == k.shape and v.stride() == k.stride() and kc.stride() == vc.stride()
    _chk(lib.hsa_compress_learned(_p(k), _p(v), _dt(k), B, d, k.stride(0), k.stride(1), N_cap, _p(tok_begin),
                                  _p(tok_end), int(max_blocks), _p(u), _p(bias), int(m), int(bias.numel()), _p(kc),
                                  _p(vc), kc.stride(0), kc.stride(1), kc.shape[1], _stream(stream)))


def hsa_compress_append(k_new, v_new, pos0, w, m, state_k, state_v, kc, vc, stream=None):
    """k_new, v_new [B, T, d]; pos0 int64 [B] (position of the first new token); state_k/v fp32 [B, d];
    kc, vc [B, E_cap, d] receive the entries of blocks completed by the new tokens."""
    B, T, d = k_new.shape
    assert v_new.shape == k_new.shape and v_new.stride() == k_new.stride() and kc.stride() == vc.stride()
    assert state_k.stride() == state_v.stride() and state_k.dtype == torch.float32
    _chk(lib.hsa_compress_append(_p(k_new), _p(v_new), _dt(k_new), B, T, d, k_new.stride(0), k_new.stride(1),
                                 _p(pos0), _p(w), int(m), _p(state_k), _p(state_v), state_k.stride(0), _p(kc),
                                 _p(vc), kc.stride(0), kc.stride(1), kc.shape[1], _stream(stream)))


def hsa_index_topk_workspace_size(B, T, DI, E_cap, topk):
    n = ctypes.c_size_t(0)
    _chk(lib.hsa_index_topk_workspace_size(B, T, DI, E_cap, topk, ctypes.byref(n)))
    return n.value


def hsa_index_topk(q_idx, k_idx, q_pos0, m, topk, idx_out, cnt_out, ws, stream=None):
    """q_idx int8 [B, T, DI]; k_idx int8 [B, E_cap, DI]; idx_out int32 [B, T, topk]; cnt_out int32 [B, T]."""
    B, T, DI = q_idx.shape
    E_cap = k_idx.shape[1]
    _chk(lib.hsa_index_topk(_p(q_idx), q_idx.stride(0), q_idx.stride(1), _p(k_idx), k_idx.stride(0), k_idx.stride(1),
                            E_cap, B, T, DI, _p(q_pos0), int(m), int(topk), _p(idx_out), _p(cnt_out), _p(ws),
                            ws.numel() * ws.element_size() if ws is not None else 0, _stream(stream)))


def hsa_index_topk_noalloc(q_idx, k_idx, q_pos0, m, topk, idx_out, cnt_out, stream=None):
    """hsa_index_topk without a workspace, for callers that cannot allocate device
    memory: the library's built-in 16 MiB scratch is used instead.  Same result."""
    B, T, DI = q_idx.shape
    E_cap = k_idx.shape[1]
    _chk(lib.hsa_index_topk_noalloc(_p(q_idx), q_idx.stride(0), q_idx.stride(1), _p(k_idx), k_idx.stride(0),
                                    k_idx.stride(1), E_cap, B, T, DI, _p(q_pos0), int(m), int(topk), _p(idx_out),
                                    _p(cnt_out), _stream(stream)))


def hsa_attn_decode_workspace_size(dtype, B, H, d, E_cap, m, topk, window):
    n = ctypes.c_size_t(0)
    dt = HSA_BF16 if dtype == torch.bfloat16 else HSA_F32
    _chk(lib.hsa_attn_decode_workspace_size(dt, B, H, d, E_cap, m, topk, window, ctypes.byref(n)))
    return n.value


def hsa_attn_decode(q, kc, vc, m, idx, cnt, k_raw, v_raw, window, ctx_len, scale, out, lse=None, ws=None,
                    stream=None):
    """q [B, H, d]; kc/vc [B, E_cap, d]; idx int32 [B, topk] or None (HCA); out [B, H, d]; lse fp32 [B, H]."""
    B, H, d = q.shape
    topk = idx.shape[-1] if idx is not None else 0
    _chk(lib.hsa_attn_decode(_p(q), _dt(q), B, H, d, _p(kc), _p(vc), kc.stride(0), kc.stride(1), kc.shape[1],
                             int(m), _p(idx), _p(cnt), topk, _p(k_raw), _p(v_raw), k_raw.stride(0), k_raw.stride(1),
                             k_raw.shape[1], int(window), _p(ctx_len), float(scale), _p(out), _p(lse), _p(ws),
                             ws.numel() * ws.element_size() if ws is not None else 0, _stream(stream)))


def hsa_attn_decode_v4(q, kc, vc, m, idx, cnt, k_raw, v_raw, window, ctx_len, scale, out, lse=None, ws=None,
                       gamma_q=None, eps=1e-6, rope_dims=64, theta=10000.0, sink=None, stream=None):
    """hsa_attn_decode with the V4 query preparation (RMSNorm, partial RoPE) and the sink and
    inverse rotation of the output inside the attention kernel; q is the raw query."""
    B, H, d = q.shape
    topk = idx.shape[-1] if idx is not None else 0
    _chk(lib.hsa_attn_decode_v4(_p(q), _dt(q), B, H, d, _p(kc), _p(vc), kc.stride(0), kc.stride(1), kc.shape[1],
                                int(m), _p(idx), _p(cnt), topk, _p(k_raw), _p(v_raw), k_raw.stride(0),
                                k_raw.stride(1), k_raw.shape[1], int(window), _p(ctx_len), float(scale), _p(gamma_q),
                                float(eps), int(rope_dims), float(theta), _p(sink), _p(out), _p(lse), _p(ws),
                                ws.numel() * ws.element_size() if ws is not None else 0, _stream(stream)))


def hsa_decode_csa_workspace_size(B, H, d, DI, E_cap):
    n = ctypes.c_size_t(0)
    _chk(lib.hsa_decode_csa_workspace_size(B, H, d, DI, E_cap, ctypes.byref(n)))
    return n.value


def hsa_decode_csa(q_idx, k_idx, m, topk, idx_out, cnt_out, q, kc, vc, k_raw, v_raw, window, ctx_len, scale, out,
                   lse=None, ws=None, stream=None):
    """One CSA decode step: q_idx int8 [B, DI] (or [B, 1, DI]); k_idx int8 [B, E_cap, DI]; idx_out int32
    [B, topk]; cnt_out int32 [B]; q [B, H, d]; kc/vc [B, E_cap, d]; out [B, H, d]; lse fp32 [B, H]."""
    B, H, d = q.shape
    qi = q_idx.reshape(B, -1)
    DI = qi.shape[1]
    E_cap = k_idx.shape[1]
    _chk(lib.hsa_decode_csa(_p(qi), qi.stride(0), _p(k_idx), k_idx.stride(0), k_idx.stride(1), E_cap, DI, int(m),
                            int(topk), _p(idx_out), _p(cnt_out), _p(q), _dt(q), B, H, d, _p(kc), _p(vc), kc.stride(0),
                            kc.stride(1), _p(k_raw), _p(v_raw), k_raw.stride(0), k_raw.stride(1), k_raw.shape[1],
                            int(window), _p(ctx_len), float(scale), _p(out), _p(lse), _p(ws),
                            ws.numel() * ws.element_size() if ws is not None else 0, _stream(stream)))


def hsa_attn_prefill_workspace_size(dtype, B, T, H, d, E_cap, m, topk, window):
    n = ctypes.c_size_t(0)
    dt = HSA_BF16 if dtype == torch.bfloat16 else HSA_F32
    _chk(lib.hsa_attn_prefill_workspace_size(dt, B, T, H, d, E_cap, m, topk, window, ctypes.byref(n)))
    return n.value


def hsa_attn_prefill(q, kc, vc, m, idx, cnt, k_raw, v_raw, window, q_pos0, scale, out, lse=None, ws=None,
                     stream=None):
    """q [B, T, H, d]; idx int32 [B, T, topk] or None (HCA); out [B, T, H, d]; lse fp32 [B, T, H]."""
    B, T, H, d = q.shape
    topk = idx.shape[-1] if idx is not None else 0
    _chk(lib.hsa_attn_prefill(_p(q), _dt(q), B, T, H, d, _p(kc), _p(vc), kc.stride(0), kc.stride(1), kc.shape[1],
                              int(m), _p(idx), _p(cnt), topk, _p(k_raw), _p(v_raw), k_raw.stride(0),
                              k_raw.stride(1), k_raw.shape[1], int(window), _p(q_pos0), float(scale), _p(out),
                              _p(lse), _p(ws), ws.numel() * ws.element_size() if ws is not None else 0,
                              _stream(stream)))


def hsa_index_scores(q_idx, k_idx, idx, cnt, scores, stream=None):
    """q_idx int8 [B, T, DI]; k_idx int8 [B, E_cap, DI]; idx int32 [B, T, topk]; cnt int32 [B, T] or None;
    scores int32 [B, T, topk] (INT32_MIN for empty slots)."""
    B, T, DI = q_idx.shape
    _chk(lib.hsa_index_scores(_p(q_idx), q_idx.stride(0), q_idx.stride(1), _p(k_idx), k_idx.stride(0),
                              k_idx.stride(1), k_idx.shape[1], B, T, DI, _p(idx), _p(cnt), idx.shape[-1], _p(scores),
                              _stream(stream)))


def hsa_topk_merge(scores, idx, topk, idx_out, cnt_out, stream=None):
    """scores, idx int32 [rows, n] (idx < 0 empty; non-empty indices ascending per row);
    idx_out int32 [rows, topk]; cnt_out int32 [rows]."""
    rows, n = idx.shape
    _chk(lib.hsa_topk_merge(_p(scores), _p(idx), rows, n, int(topk), _p(idx_out), _p(cnt_out), _stream(stream)))


def hsa_lse_merge(parts_o, parts_lse, out, lse_out=None, stream=None):
    """parts_o [S, rows, H, d]; parts_lse fp32 [S, rows, H]; out [rows, H, d]; lse_out fp32 [rows, H]."""
    S, rows, H, d = parts_o.shape
    _chk(lib.hsa_lse_merge(_p(parts_o), _p(parts_lse), _dt(parts_o), S, rows, H, d, _p(out), _p(lse_out),
                           _stream(stream)))


def hsa_rmsnorm_rope(x, n_begin, n_end, max_rows, pos_base=None, pos_stride=1, pos_offset=0, gamma=None,
                     eps=1e-6, rope_dims=64, theta=10000.0, stream=None):
    """In place x <- R(pos) RMSNorm(x) on rows [n_begin[b], n_end[b]) of x [B, n_cap, d] or [B, n_cap, H, d];
    pos = pos_base[b] + n * pos_stride + pos_offset."""
    if x.dim() == 3:
        B, n_cap, d = x.shape
        H = 1
    else:
        B, n_cap, H, d = x.shape
        assert x.stride(2) == d
    _chk(lib.hsa_rmsnorm_rope(_p(x), _dt(x), B, H, d, x.stride(0), x.stride(1), n_cap, _p(n_begin), _p(n_end),
                              int(max_rows), _p(pos_base), int(pos_stride), int(pos_offset), _p(gamma), float(eps),
                              int(rope_dims), float(theta), _stream(stream)))


def hsa_attn_finalize(out, lse, q_pos0, sink=None, rope_dims=64, theta=10000.0, stream=None):
    """Sink and inverse rotation on (out [B, T, H, d] or [B, H, d], lse) in place; p = q_pos0[b] + t."""
    if out.dim() == 3:
        B, H, d = out.shape
        T = 1
    else:
        B, T, H, d = out.shape
    _chk(lib.hsa_attn_finalize(_p(out), _p(lse), _dt(out), B, T, H, d, _p(q_pos0), _p(sink), int(rope_dims),
                               float(theta), _stream(stream)))


def workspace(nbytes: int, device="cuda"):
    """A zero-filled, 256-byte aligned workspace (torch allocations are 512-byte aligned)."""
    return torch.zeros(max(int(nbytes), 1), dtype=torch.uint8, device=device)
