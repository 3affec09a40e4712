"""ctypes binding of libusp.so: the C entry points of include/usp.h, same names.

Argument marshalling only: tensors become device pointers, the stream becomes
torch's current CUDA stream unless one is given, and a non-zero status raises
``UspError``.  Every step of the path runs in the library's CUDA kernels; there
is no CPU fallback, and a missing library or a CPU tensor is an error.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libusp.so")
_lib = None

# status codes (include/usp.h)
USP_OK = 0
USP_ERR_INVALID_ARG = 1
USP_ERR_INDIVISIBLE = 2
USP_ERR_UNSUPPORTED = 3
USP_ERR_ALIGNMENT = 4
USP_ERR_BAD_SEQLENS = 5
USP_ERR_BAD_POSITIONS = 6
USP_ERR_TIMEOUT = 7
USP_ERR_CUDA = 8
USP_ERR_WORKSPACE = 9

EXPORTED = [
    "usp_status_string", "usp_version",
    "usp_relayout_fwd", "usp_relayout_bwd", "usp_relayout_fwd_qkv",
    "usp_cu_seqlens_workspace_bytes", "usp_cu_seqlens_from_position_ids",
    "usp_cu_seqlens_from_position_ids_noalloc",
    "usp_attn_fwd", "usp_attn_bwd_workspace_bytes", "usp_attn_bwd",
    "usp_attn_bwd_preprocess", "usp_attn_bwd_dkdv", "usp_attn_bwd_dq",
    "usp_hybrid_relayout_fwd", "usp_hybrid_relayout_bwd", "usp_hybrid_relayout_fwd_qkv",
    "usp_ring_fwd_merge", "usp_ring_grad_accumulate", "usp_attn_bwd_fast_workspace_bytes",
    "usp_a2a_pack_seq_to_head", "usp_a2a_unpack_seq_to_head", "usp_a2a_pack_head_to_seq",
    "usp_a2a_unpack_head_to_seq",
]

USP_RING_FIRST = 1
USP_RING_LAST = 2


class UspError(RuntimeError):
    def __init__(self, code: int, where: str = ""):
        self.code = int(code)
        super().__init__(f"{where}: {status_string(code)}" if where else status_string(code))


class AttnParams(ctypes.Structure):
    """usp_attn_params (include/usp.h)."""
    _fields_ = [
        ("B", ctypes.c_int), ("S", ctypes.c_int), ("Hq", ctypes.c_int), ("Hkv", ctypes.c_int),
        ("D", ctypes.c_int), ("P", ctypes.c_int), ("causal", ctypes.c_int),
        ("window_left", ctypes.c_int), ("softmax_scale", ctypes.c_float),
        ("cu_seqlens", ctypes.c_void_p), ("n_docs", ctypes.c_void_p), ("sinks", ctypes.c_void_p),
        ("io_layout", ctypes.c_int), ("ring", ctypes.c_int), ("ring_step", ctypes.c_int),
        ("head_first", ctypes.c_int), ("head_count", ctypes.c_int),
    ]


USP_IO_HEAD = 0
USP_IO_SEQ = 1
USP_IO_SEQ_KV_HEAD = 2


def lib_path() -> str:
    return _LIB_PATH


def load() -> ctypes.CDLL:
    """Load libusp.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        raise RuntimeError(f"{_LIB_PATH} is missing: build it with ulysses_sequence_long_gb300._build.build()")
    L = ctypes.CDLL(_LIB_PATH)
    vp, i32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    L.usp_status_string.restype = ctypes.c_char_p
    L.usp_status_string.argtypes = [i32]
    L.usp_version.restype = i32
    L.usp_relayout_fwd.argtypes = [vp, vp, i32, i32, i32, i32, i32, i32, vp]
    L.usp_relayout_bwd.argtypes = [vp, vp, i32, i32, i32, i32, i32, i32, vp]
    L.usp_relayout_fwd_qkv.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, vp]
    L.usp_cu_seqlens_workspace_bytes.restype = sz
    L.usp_cu_seqlens_workspace_bytes.argtypes = [i32, i32]
    L.usp_cu_seqlens_from_position_ids.argtypes = [vp, i32, i32, i32, vp, vp, vp, vp, sz, vp, vp]
    L.usp_cu_seqlens_from_position_ids_noalloc.argtypes = [vp, i32, i32, i32, vp, vp, vp, vp, vp]
    L.usp_attn_fwd.argtypes = [ctypes.POINTER(AttnParams), vp, vp, vp, vp, vp, vp, vp]
    L.usp_attn_bwd_workspace_bytes.restype = sz
    L.usp_attn_bwd_workspace_bytes.argtypes = [ctypes.POINTER(AttnParams)]
    L.usp_attn_bwd_fast_workspace_bytes.restype = sz
    L.usp_attn_bwd_fast_workspace_bytes.argtypes = [ctypes.POINTER(AttnParams)]
    L.usp_attn_bwd.argtypes = [ctypes.POINTER(AttnParams), vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp, vp]
    L.usp_attn_bwd_preprocess.argtypes = [ctypes.POINTER(AttnParams), vp, vp, vp, vp, vp, sz, vp, vp]
    L.usp_attn_bwd_dkdv.argtypes = [ctypes.POINTER(AttnParams), vp, vp, vp, vp, vp, vp, vp, vp, sz, vp, vp]
    L.usp_attn_bwd_dq.argtypes = [ctypes.POINTER(AttnParams), vp, vp, vp, vp, vp, vp, vp, sz, vp, vp]
    L.usp_hybrid_relayout_fwd.argtypes = [vp, vp, i32, i32, i32, i32, i32, i32, i32, vp]
    L.usp_hybrid_relayout_bwd.argtypes = [vp, vp, i32, i32, i32, i32, i32, i32, i32, vp]
    L.usp_hybrid_relayout_fwd_qkv.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, i32, i32, vp]
    L.usp_ring_fwd_merge.argtypes = [ctypes.POINTER(AttnParams), vp, vp, vp, vp, vp, vp, i32, vp]
    L.usp_ring_grad_accumulate.argtypes = [vp, vp, vp, sz, i32, vp]
    for name in ("usp_a2a_pack_seq_to_head", "usp_a2a_unpack_seq_to_head", "usp_a2a_pack_head_to_seq",
                 "usp_a2a_unpack_head_to_seq"):
        getattr(L, name).argtypes = [vp, vp, i32, i32, i32, i32, i32, i32, vp]
    for name in ("usp_relayout_fwd", "usp_relayout_bwd", "usp_relayout_fwd_qkv",
                 "usp_cu_seqlens_from_position_ids", "usp_cu_seqlens_from_position_ids_noalloc",
                 "usp_attn_fwd", "usp_attn_bwd",
                 "usp_attn_bwd_preprocess", "usp_attn_bwd_dkdv", "usp_attn_bwd_dq",
                 "usp_hybrid_relayout_fwd", "usp_hybrid_relayout_bwd", "usp_hybrid_relayout_fwd_qkv",
                 "usp_ring_fwd_merge", "usp_ring_grad_accumulate", "usp_a2a_pack_seq_to_head",
                 "usp_a2a_unpack_seq_to_head", "usp_a2a_pack_head_to_seq", "usp_a2a_unpack_head_to_seq"):
        getattr(L, name).restype = i32
    _lib = L
    return L


def status_string(code: int) -> str:
    return load().usp_status_string(int(code)).decode()


def _check(rc: int, where: str) -> None:
    if rc != USP_OK:
        raise UspError(rc, where)


def _dev(t: Optional[torch.Tensor], name: str, dtype=None):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor (the library has no CPU path)")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def usp_relayout_fwd(x_seq, x_head, B, S, H, D, P, stream=None):
    _check(load().usp_relayout_fwd(_dev(x_seq, "x_seq"), _dev(x_head, "x_head"), B, S, H, D, P,
                                   x_seq.element_size(), _stream(stream)), "usp_relayout_fwd")


def usp_relayout_bwd(x_head, x_seq, B, S, H, D, P, stream=None):
    _check(load().usp_relayout_bwd(_dev(x_head, "x_head"), _dev(x_seq, "x_seq"), B, S, H, D, P,
                                   x_head.element_size(), _stream(stream)), "usp_relayout_bwd")


def usp_relayout_fwd_qkv(q_seq, k_seq, v_seq, q_head, k_head, v_head, B, S, Hq, Hkv, D, P, stream=None):
    _check(load().usp_relayout_fwd_qkv(_dev(q_seq, "q_seq"), _dev(k_seq, "k_seq"), _dev(v_seq, "v_seq"),
                                       _dev(q_head, "q_head"), _dev(k_head, "k_head"), _dev(v_head, "v_head"),
                                       B, S, Hq, Hkv, D, P, q_seq.element_size(), _stream(stream)),
           "usp_relayout_fwd_qkv")


def usp_cu_seqlens_workspace_bytes(B, S) -> int:
    return int(load().usp_cu_seqlens_workspace_bytes(B, S))


def usp_cu_seqlens_from_position_ids(pos, B, S, P, cu_seqlens, n_docs, max_len, ws, dev_status=None,
                                     stream=None):
    _check(load().usp_cu_seqlens_from_position_ids(
        _dev(pos, "pos", torch.int32), B, S, P, _dev(cu_seqlens, "cu_seqlens", torch.int32),
        _dev(n_docs, "n_docs", torch.int32), _dev(max_len, "max_len", torch.int32), _dev(ws, "ws"),
        ws.numel() * ws.element_size(), _dev(dev_status, "dev_status", torch.int32), _stream(stream)),
        "usp_cu_seqlens_from_position_ids")


def usp_cu_seqlens_from_position_ids_noalloc(pos, B, S, P, cu_seqlens, n_docs, max_len, dev_status=None,
                                             stream=None):
    """The scan without a workspace: its scratch is a fixed array inside the library (B*S <= 2^24)."""
    _check(load().usp_cu_seqlens_from_position_ids_noalloc(
        _dev(pos, "pos", torch.int32), B, S, P, _dev(cu_seqlens, "cu_seqlens", torch.int32),
        _dev(n_docs, "n_docs", torch.int32), _dev(max_len, "max_len", torch.int32),
        _dev(dev_status, "dev_status", torch.int32), _stream(stream)),
        "usp_cu_seqlens_from_position_ids_noalloc")


def attn_params(B, S, Hq, Hkv, D, P, cu_seqlens, n_docs, causal=True, window_left=-1, softmax_scale=0.0,
                sinks=None, io_layout=USP_IO_HEAD, ring=1, ring_step=0, head_first=0, head_count=0) -> AttnParams:
    return AttnParams(B, S, Hq, Hkv, D, P, 1 if causal else 0, window_left, softmax_scale,
                      _dev(cu_seqlens, "cu_seqlens", torch.int32), _dev(n_docs, "n_docs", torch.int32),
                      _dev(sinks, "sinks", torch.float32), int(io_layout), int(ring), int(ring_step),
                      int(head_first), int(head_count))


def usp_attn_fwd(params: AttnParams, q, k, v, o, lse, dev_status=None, stream=None):
    _check(load().usp_attn_fwd(ctypes.byref(params), _dev(q, "q", torch.bfloat16), _dev(k, "k", torch.bfloat16),
                               _dev(v, "v", torch.bfloat16), _dev(o, "o", torch.bfloat16),
                               _dev(lse, "lse", torch.float32), _dev(dev_status, "dev_status", torch.int32),
                               _stream(stream)), "usp_attn_fwd")


def usp_attn_bwd_workspace_bytes(params: AttnParams) -> int:
    return int(load().usp_attn_bwd_workspace_bytes(ctypes.byref(params)))


def usp_attn_bwd_fast_workspace_bytes(params: AttnParams) -> int:
    return int(load().usp_attn_bwd_fast_workspace_bytes(ctypes.byref(params)))


def usp_attn_bwd(params: AttnParams, q, k, v, o, lse, dO, dq, dk, dv, dsinks, ws, dev_status=None, stream=None):
    _check(load().usp_attn_bwd(
        ctypes.byref(params), _dev(q, "q", torch.bfloat16), _dev(k, "k", torch.bfloat16),
        _dev(v, "v", torch.bfloat16), _dev(o, "o", torch.bfloat16), _dev(lse, "lse", torch.float32),
        _dev(dO, "dO", torch.bfloat16), _dev(dq, "dq", torch.bfloat16), _dev(dk, "dk", torch.bfloat16),
        _dev(dv, "dv", torch.bfloat16), _dev(dsinks, "dsinks", torch.float32), _dev(ws, "ws"),
        ws.numel() * ws.element_size(), _dev(dev_status, "dev_status", torch.int32), _stream(stream)),
        "usp_attn_bwd")


def usp_attn_bwd_preprocess(params: AttnParams, o, lse, dO, dsinks, ws, dev_status=None, stream=None):
    _check(load().usp_attn_bwd_preprocess(
        ctypes.byref(params), _dev(o, "o", torch.bfloat16), _dev(lse, "lse", torch.float32),
        _dev(dO, "dO", torch.bfloat16), _dev(dsinks, "dsinks", torch.float32), _dev(ws, "ws"),
        ws.numel() * ws.element_size(), _dev(dev_status, "dev_status", torch.int32), _stream(stream)),
        "usp_attn_bwd_preprocess")


def usp_attn_bwd_dkdv(params: AttnParams, q, k, v, lse, dO, dk, dv, ws, dev_status=None, stream=None):
    _check(load().usp_attn_bwd_dkdv(
        ctypes.byref(params), _dev(q, "q", torch.bfloat16), _dev(k, "k", torch.bfloat16),
        _dev(v, "v", torch.bfloat16), _dev(lse, "lse", torch.float32), _dev(dO, "dO", torch.bfloat16),
        _dev(dk, "dk", torch.bfloat16), _dev(dv, "dv", torch.bfloat16), _dev(ws, "ws"),
        ws.numel() * ws.element_size(), _dev(dev_status, "dev_status", torch.int32), _stream(stream)),
        "usp_attn_bwd_dkdv")


def usp_attn_bwd_dq(params: AttnParams, q, k, v, lse, dO, dq, ws, dev_status=None, stream=None):
    _check(load().usp_attn_bwd_dq(
        ctypes.byref(params), _dev(q, "q", torch.bfloat16), _dev(k, "k", torch.bfloat16),
        _dev(v, "v", torch.bfloat16), _dev(lse, "lse", torch.float32), _dev(dO, "dO", torch.bfloat16),
        _dev(dq, "dq", torch.bfloat16), _dev(ws, "ws"), ws.numel() * ws.element_size(),
        _dev(dev_status, "dev_status", torch.int32), _stream(stream)),
        "usp_attn_bwd_dq")


def usp_hybrid_relayout_fwd(x_seq, x_head, B, S, H, D, ring, ulysses, stream=None):
    _check(load().usp_hybrid_relayout_fwd(_dev(x_seq, "x_seq"), _dev(x_head, "x_head"), B, S, H, D, ring, ulysses,
                                          x_seq.element_size(), _stream(stream)), "usp_hybrid_relayout_fwd")


def usp_hybrid_relayout_bwd(x_head, x_seq, B, S, H, D, ring, ulysses, stream=None):
    _check(load().usp_hybrid_relayout_bwd(_dev(x_head, "x_head"), _dev(x_seq, "x_seq"), B, S, H, D, ring, ulysses,
                                          x_head.element_size(), _stream(stream)), "usp_hybrid_relayout_bwd")


def usp_hybrid_relayout_fwd_qkv(q_seq, k_seq, v_seq, q_head, k_head, v_head, B, S, Hq, Hkv, D, ring, ulysses,
                                stream=None):
    _check(load().usp_hybrid_relayout_fwd_qkv(
        _dev(q_seq, "q_seq"), _dev(k_seq, "k_seq"), _dev(v_seq, "v_seq"), _dev(q_head, "q_head"),
        _dev(k_head, "k_head"), _dev(v_head, "v_head"), B, S, Hq, Hkv, D, ring, ulysses, q_seq.element_size(),
        _stream(stream)), "usp_hybrid_relayout_fwd_qkv")


def usp_ring_fwd_merge(params: AttnParams, o_step, lse_step, o_acc, lse_acc, o, lse, flags, stream=None):
    _check(load().usp_ring_fwd_merge(
        ctypes.byref(params), _dev(o_step, "o_step", torch.bfloat16), _dev(lse_step, "lse_step", torch.float32),
        _dev(o_acc, "o_acc", torch.float32), _dev(lse_acc, "lse_acc", torch.float32), _dev(o, "o", torch.bfloat16),
        _dev(lse, "lse", torch.float32), int(flags), _stream(stream)), "usp_ring_fwd_merge")


def usp_ring_grad_accumulate(g_step, g_acc, g_out, flags, stream=None):
    _check(load().usp_ring_grad_accumulate(
        _dev(g_step, "g_step", torch.bfloat16), _dev(g_acc, "g_acc", torch.float32),
        _dev(g_out, "g_out", torch.bfloat16), g_step.numel(), int(flags), _stream(stream)),
        "usp_ring_grad_accumulate")


def _a2a(name, src, dst, B, S_local, H, D, P, stream):
    _check(getattr(load(), name)(_dev(src, "src"), _dev(dst, "dst"), B, S_local, H, D, P, src.element_size(),
                                 _stream(stream)), name)


def usp_a2a_pack_seq_to_head(x_local, send, B, S_local, H, D, P, stream=None):
    _a2a("usp_a2a_pack_seq_to_head", x_local, send, B, S_local, H, D, P, stream)


def usp_a2a_unpack_seq_to_head(recv, x_head, B, S_local, H, D, P, stream=None):
    _a2a("usp_a2a_unpack_seq_to_head", recv, x_head, B, S_local, H, D, P, stream)


def usp_a2a_pack_head_to_seq(x_head, send, B, S_local, H, D, P, stream=None):
    _a2a("usp_a2a_pack_head_to_seq", x_head, send, B, S_local, H, D, P, stream)


def usp_a2a_unpack_head_to_seq(recv, x_local, B, S_local, H, D, P, stream=None):
    _a2a("usp_a2a_unpack_head_to_seq", recv, x_local, B, S_local, H, D, P, stream)
