"""ctypes binding to the C ABI in include/attn.h: argument marshalling only.

Every step of the attention path runs in the CUDA library; this module only
turns PyTorch tensors into pointers and sizes, passes the current CUDA stream
and raises on a non-zero status.  There is no fallback: if the library is not
built, every call raises ``ExtensionMissing``.
"""

from __future__ import annotations

import ctypes
import math
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "lib", "libexact_attention.so")

ATTN_OK = 0
ATTN_ERR_INVALID_ARG = 1
ATTN_ERR_UNSUPPORTED = 2
ATTN_ERR_CUDA = 3
ATTN_ERR_DEVICE_TIMEOUT = 4
ATTN_BF16 = 0
ATTN_FP16 = 1

EXPORTS = ("attn_fwd", "attn_fwd_varlen", "attn_fwd_qkvpacked", "attn_bwd", "attn_bwd_varlen",
           "attn_bwd_qkvpacked", "attn_bwd_workspace_bytes", "attn_decode", "attn_decode_fused",
           "attn_decode_paged",
           "attn_decode_noalloc",
           "attn_decode_workspace_bytes",
           "attn_decode_chunk", "attn_check_device_status", "attn_debug_set",
           "attn_status_string", "attn_version")
NOALLOC_MAX_BYTES = 16 << 20  # ATTN_DECODE_NOALLOC_MAX_BYTES in attn.h


class ExtensionMissing(RuntimeError):
    pass


class AttnError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{msg} (status {status})")
        self.status = status


_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load the shared library and declare the C signatures (no CUDA call is made)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ExtensionMissing(
            f"{path} is not built; run `python -m exact_attention_43_gb300.build` "
            "(or __graft_entry__.build())")
    lib = ctypes.CDLL(path)
    vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    lib.attn_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, i, f, i, vp]
    lib.attn_fwd.restype = i
    lib.attn_fwd_varlen.argtypes = [vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, i, i, i, i, f,
                                    i, vp]
    lib.attn_fwd_varlen.restype = i
    lib.attn_fwd_qkvpacked.argtypes = [vp, vp, vp, i, i, i, i, i, i, i, f, i, vp]
    lib.attn_fwd_qkvpacked.restype = i
    lib.attn_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, f, i, vp]
    lib.attn_bwd.restype = i
    lib.attn_bwd_varlen.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, i,
                                    i, i, i, f, i, vp]
    lib.attn_bwd_varlen.restype = i
    lib.attn_bwd_qkvpacked.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, i, f, i, vp]
    lib.attn_bwd_qkvpacked.restype = i
    lib.attn_bwd_workspace_bytes.argtypes = [i, i, i, i]
    lib.attn_bwd_workspace_bytes.restype = sz
    lib.attn_decode.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, i, vp]
    lib.attn_decode.restype = i
    lib.attn_decode_fused.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, i, vp]
    lib.attn_decode_fused.restype = i
    lib.attn_decode_paged.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, i, i, vp]
    lib.attn_decode_paged.restype = i
    lib.attn_decode_noalloc.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, i, vp]
    lib.attn_decode_noalloc.restype = i
    lib.attn_decode_workspace_bytes.argtypes = [i, i, i, i, i]
    lib.attn_decode_workspace_bytes.restype = sz
    lib.attn_decode_chunk.argtypes = [i, i]
    lib.attn_decode_chunk.restype = i
    lib.attn_check_device_status.argtypes = [vp]
    lib.attn_check_device_status.restype = i
    lib.attn_debug_set.argtypes = [i, ctypes.c_uint]
    lib.attn_debug_set.restype = i
    lib.attn_status_string.argtypes = [i]
    lib.attn_status_string.restype = ctypes.c_char_p
    lib.attn_version.argtypes = []
    lib.attn_version.restype = i
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return load().attn_status_string(status).decode()


def _check(status: int, what: str):
    if status != ATTN_OK:
        raise AttnError(status, f"{what}: {status_string(status)}")


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return ATTN_BF16
    if t.dtype == torch.float16:
        return ATTN_FP16
    raise TypeError(f"unsupported dtype {t.dtype}: bf16 or fp16")


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _ptr(t):
    return None if t is None else t.data_ptr()


def _cuda16(t, name):
    """The device of `t`, which must be a 16-bit (bf16 / fp16) CUDA tensor."""
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    _dtype_code(t)
    return t.device


def _expect(t, name, shape, dtype, device):
    """Raise unless `t` is a contiguous tensor of this shape and dtype on `device`:
    the library trusts the sizes it is given, so nothing may be smaller than they say."""
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.device != device:
        raise ValueError(f"{name} must be on {device}, got {t.device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def attn_fwd(q, k, v, *, causal: bool, scale: float | None = None, out=None, lse=None,
             return_lse: bool = True, stream=None):
    """Prefill attention: q [B,Hq,Sq,D], k/v [B,Hkv,Skv,D] (contiguous CUDA tensors).

    Returns (O, LSE) with O like q and LSE [B,Hq,Sq] float32 (None when
    return_lse is False and no lse buffer was given).
    """
    lib = load()
    dev = _cuda16(q, "q")
    B, Hq, Sq, D = q.shape
    Hkv, Skv = k.shape[1], k.shape[2]
    _expect(q, "q", (B, Hq, Sq, D), q.dtype, dev)
    _expect(k, "k", (B, Hkv, Skv, D), q.dtype, dev)
    _expect(v, "v", (B, Hkv, Skv, D), q.dtype, dev)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty_like(q)
    _expect(out, "out", q.shape, q.dtype, dev)
    if lse is None and return_lse:
        lse = torch.empty((B, Hq, Sq), dtype=torch.float32, device=q.device)
    if lse is not None:
        _expect(lse, "lse", (B, Hq, Sq), torch.float32, dev)
    st = lib.attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, Hq, Hkv, Sq, Skv, D,
                      1 if causal else 0, float(scale), _dtype_code(q), _stream(stream))
    _check(st, "attn_fwd")
    return out, lse


def attn_fwd_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q: int, max_seqlen_k: int, *,
                    causal: bool = True, window=(-1, -1), scale=None, out=None, lse=None,
                    return_lse: bool = True, stream=None):
    """Packed variable-length prefill: q [total_q,Hq,D], k/v [total_k,Hkv,D], cu_seqlens_* [B+1]
    int32 (all CUDA); window = (left, right), -1 for no bound.  Returns (O, LSE [Hq,total_q])."""
    lib = load()
    dev = _cuda16(q, "q")
    total_q, Hq, D = q.shape
    total_k, Hkv = k.shape[0], k.shape[1]
    _expect(q, "q", (total_q, Hq, D), q.dtype, dev)
    _expect(k, "k", (total_k, Hkv, D), q.dtype, dev)
    _expect(v, "v", (total_k, Hkv, D), q.dtype, dev)
    if cu_seqlens_q.dim() != 1 or cu_seqlens_q.numel() < 1:
        raise ValueError("cu_seqlens_q must hold B + 1 offsets")
    B = cu_seqlens_q.numel() - 1
    _expect(cu_seqlens_q, "cu_seqlens_q", (B + 1,), torch.int32, dev)
    _expect(cu_seqlens_k, "cu_seqlens_k", (B + 1,), torch.int32, dev)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty_like(q)
    _expect(out, "out", q.shape, q.dtype, dev)
    if lse is None and return_lse:
        lse = torch.empty((Hq, total_q), dtype=torch.float32, device=q.device)
    if lse is not None:
        _expect(lse, "lse", (Hq, total_q), torch.float32, dev)
    wl, wr = window
    st = lib.attn_fwd_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(cu_seqlens_q),
                             _ptr(cu_seqlens_k), B, Hq, Hkv, total_q, total_k, int(max_seqlen_q),
                             int(max_seqlen_k), D, 1 if causal else 0, int(wl), int(wr),
                             float(scale), _dtype_code(q), _stream(stream))
    _check(st, "attn_fwd_varlen")
    return out, lse


def attn_fwd_qkvpacked(qkv, *, causal: bool = True, window=(-1, -1), scale=None, out=None,
                       lse=None, return_lse: bool = True, stream=None):
    """Prefill reading Q, K, V in place from qkv [B,S,3,H,D] (CUDA).  Returns (O [B,S,H,D],
    LSE [H,B,S])."""
    lib = load()
    dev = _cuda16(qkv, "qkv")
    if qkv.dim() != 5 or qkv.shape[2] != 3:
        raise ValueError("qkv must be [B, S, 3, H, D]")
    B, S, _, H, D = qkv.shape
    _expect(qkv, "qkv", (B, S, 3, H, D), qkv.dtype, dev)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty((B, S, H, D), dtype=qkv.dtype, device=qkv.device)
    _expect(out, "out", (B, S, H, D), qkv.dtype, dev)
    if lse is None and return_lse:
        lse = torch.empty((H, B, S), dtype=torch.float32, device=qkv.device)
    if lse is not None:
        _expect(lse, "lse", (H, B, S), torch.float32, dev)
    wl, wr = window
    st = lib.attn_fwd_qkvpacked(_ptr(qkv), _ptr(out), _ptr(lse), B, S, H, D, 1 if causal else 0,
                                int(wl), int(wr), float(scale), _dtype_code(qkv), _stream(stream))
    _check(st, "attn_fwd_qkvpacked")
    return out, lse


def attn_bwd(q, k, v, o, lse, dout, *, causal: bool = True, scale=None, dq=None, dk=None, dv=None,
             stream=None):
    """Gradients of attn_fwd: q, o, dout [B,Hq,Sq,D], k, v [B,Hkv,Skv,D], lse [B,Hq,Sq] float32
    (the forward's outputs o and lse).  Returns (dQ, dK, dV)."""
    lib = load()
    dev = _cuda16(q, "q")
    B, Hq, Sq, D = q.shape
    Hkv, Skv = k.shape[1], k.shape[2]
    for t, name in ((q, "q"), (o, "o"), (dout, "dout")):
        _expect(t, name, (B, Hq, Sq, D), q.dtype, dev)
    for t, name in ((k, "k"), (v, "v")):
        _expect(t, name, (B, Hkv, Skv, D), q.dtype, dev)
    _expect(lse, "lse", (B, Hq, Sq), torch.float32, dev)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    _expect(dq, "dq", q.shape, q.dtype, dev)
    _expect(dk, "dk", k.shape, q.dtype, dev)
    _expect(dv, "dv", v.shape, q.dtype, dev)
    st = lib.attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout), _ptr(dq), _ptr(dk),
                      _ptr(dv), B, Hq, Hkv, Sq, Skv, D, 1 if causal else 0, float(scale),
                      _dtype_code(q), _stream(stream))
    _check(st, "attn_bwd")
    return dq, dk, dv


def attn_bwd_varlen(q, k, v, o, lse, dout, cu_seqlens_q, cu_seqlens_k, max_seqlen_q: int,
                    max_seqlen_k: int, *, causal: bool = True, window=(-1, -1), scale=None, dq=None,
                    dk=None, dv=None, stream=None):
    """Gradients of attn_fwd_varlen: q, o, dout [total_q,Hq,D], k, v [total_k,Hkv,D], lse
    [Hq,total_q] float32 (the forward's outputs), cu_seqlens_* [B+1] int32.  Returns
    (dQ, dK, dV); rows of tokens outside every sequence are not written."""
    lib = load()
    dev = _cuda16(q, "q")
    total_q, Hq, D = q.shape
    total_k, Hkv = k.shape[0], k.shape[1]
    for t, name in ((q, "q"), (o, "o"), (dout, "dout")):
        _expect(t, name, (total_q, Hq, D), q.dtype, dev)
    for t, name in ((k, "k"), (v, "v")):
        _expect(t, name, (total_k, Hkv, D), q.dtype, dev)
    _expect(lse, "lse", (Hq, total_q), torch.float32, dev)
    if cu_seqlens_q.dim() != 1 or cu_seqlens_q.numel() < 1:
        raise ValueError("cu_seqlens_q must hold B + 1 offsets")
    B = cu_seqlens_q.numel() - 1
    _expect(cu_seqlens_q, "cu_seqlens_q", (B + 1,), torch.int32, dev)
    _expect(cu_seqlens_k, "cu_seqlens_k", (B + 1,), torch.int32, dev)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    _expect(dq, "dq", q.shape, q.dtype, dev)
    _expect(dk, "dk", k.shape, q.dtype, dev)
    _expect(dv, "dv", v.shape, q.dtype, dev)
    wl, wr = window
    st = lib.attn_bwd_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout), _ptr(dq),
                             _ptr(dk), _ptr(dv), _ptr(cu_seqlens_q), _ptr(cu_seqlens_k), B, Hq, Hkv,
                             total_q, total_k, int(max_seqlen_q), int(max_seqlen_k), D,
                             1 if causal else 0, int(wl), int(wr), float(scale), _dtype_code(q),
                             _stream(stream))
    _check(st, "attn_bwd_varlen")
    return dq, dk, dv


def attn_bwd_qkvpacked(qkv, o, lse, dout, *, causal: bool = True, window=(-1, -1), scale=None,
                       dqkv=None, stream=None):
    """Gradient of attn_fwd_qkvpacked: qkv [B,S,3,H,D], o and dout [B,S,H,D], lse [H,B,S]
    float32.  Returns dqkv [B,S,3,H,D] (dQ, dK, dV at the places of Q, K, V)."""
    lib = load()
    dev = _cuda16(qkv, "qkv")
    if qkv.dim() != 5 or qkv.shape[2] != 3:
        raise ValueError("qkv must be [B, S, 3, H, D]")
    B, S, _, H, D = qkv.shape
    _expect(qkv, "qkv", (B, S, 3, H, D), qkv.dtype, dev)
    _expect(o, "o", (B, S, H, D), qkv.dtype, dev)
    _expect(dout, "dout", (B, S, H, D), qkv.dtype, dev)
    _expect(lse, "lse", (H, B, S), torch.float32, dev)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    dqkv = torch.empty_like(qkv) if dqkv is None else dqkv
    _expect(dqkv, "dqkv", qkv.shape, qkv.dtype, dev)
    wl, wr = window
    st = lib.attn_bwd_qkvpacked(_ptr(qkv), _ptr(o), _ptr(lse), _ptr(dout), _ptr(dqkv), B, S, H, D,
                                1 if causal else 0, int(wl), int(wr), float(scale),
                                _dtype_code(qkv), _stream(stream))
    _check(st, "attn_bwd_qkvpacked")
    return dqkv


def _decode_shapes(q, k_cache, v_cache, seq_lens, out):
    """Check the contiguous-cache decode arguments; returns (B, Hq, Hkv, max_S, D)."""
    dev = _cuda16(q, "q")
    B, Hq, D = q.shape
    Hkv, max_S = k_cache.shape[1], k_cache.shape[2]
    _expect(q, "q", (B, Hq, D), q.dtype, dev)
    _expect(k_cache, "k_cache", (B, Hkv, max_S, D), q.dtype, dev)
    _expect(v_cache, "v_cache", (B, Hkv, max_S, D), q.dtype, dev)
    _expect(seq_lens, "seq_lens", (B,), torch.int32, dev)
    if out is not None:
        _expect(out, "out", (B, Hq, D), q.dtype, dev)
    return B, Hq, Hkv, max_S, D


def attn_decode(q, k_cache, v_cache, seq_lens, *, num_splits: int = 0, out=None, stream=None):
    """Flash-decoding: q [B,Hq,D], caches [B,Hkv,max_S,D], seq_lens [B] int32 (all CUDA)."""
    lib = load()
    B, Hq, Hkv, max_S, D = _decode_shapes(q, k_cache, v_cache, seq_lens, out)
    if out is None:
        out = torch.empty_like(q)
    st = lib.attn_decode(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(seq_lens), _ptr(out), B, Hq,
                         Hkv, max_S, D, num_splits, _dtype_code(q), _stream(stream))
    _check(st, "attn_decode")
    return out


def attn_decode_fused(q, k_cache, v_cache, seq_lens, *, num_splits: int = 0, out=None,
                      stream=None):
    """``attn_decode`` in one kernel launch: the last split CTA of each (sequence,
    head group) merges the group's chunk partials.  Calls that may overlap on the
    GPU share the library's merge counters: order them on one stream."""
    lib = load()
    B, Hq, Hkv, max_S, D = _decode_shapes(q, k_cache, v_cache, seq_lens, out)
    if out is None:
        out = torch.empty_like(q)
    st = lib.attn_decode_fused(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(seq_lens), _ptr(out),
                               B, Hq, Hkv, max_S, D, num_splits, _dtype_code(q), _stream(stream))
    _check(st, "attn_decode_fused")
    return out


def attn_decode_paged(q, k_pages, v_pages, block_table, seq_lens, *, num_splits: int = 0, out=None,
                      stream=None):
    """Flash-decoding over a paged cache: q [B,Hq,D], pages [num_pages,Hkv,page_size,D],
    block_table [B,max_pages] int32, seq_lens [B] int32 (all CUDA)."""
    lib = load()
    dev = _cuda16(q, "q")
    B, Hq, D = q.shape
    num_pages, Hkv, page_size = k_pages.shape[0], k_pages.shape[1], k_pages.shape[2]
    if block_table.dim() != 2:
        raise ValueError("block_table must be [B, max_pages]")
    max_pages = block_table.shape[1]
    _expect(q, "q", (B, Hq, D), q.dtype, dev)
    _expect(k_pages, "k_pages", (num_pages, Hkv, page_size, D), q.dtype, dev)
    _expect(v_pages, "v_pages", (num_pages, Hkv, page_size, D), q.dtype, dev)
    _expect(block_table, "block_table", (B, max_pages), torch.int32, dev)
    _expect(seq_lens, "seq_lens", (B,), torch.int32, dev)
    if out is None:
        out = torch.empty_like(q)
    _expect(out, "out", (B, Hq, D), q.dtype, dev)
    st = lib.attn_decode_paged(_ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(block_table),
                               _ptr(seq_lens), _ptr(out), B, Hq, Hkv, num_pages, page_size,
                               max_pages, D, num_splits, _dtype_code(q), _stream(stream))
    _check(st, "attn_decode_paged")
    return out


def attn_decode_noalloc(q, k_cache, v_cache, seq_lens, *, num_splits: int = 0, out=None,
                        stream=None):
    """attn_decode for callers that may not allocate GPU memory during the call.

    Same inputs and result as ``attn_decode``; the chunk partials go to a fixed
    16 MiB scratch array the library reserves per device instead of a
    per-call allocation.  ``out`` must be given (the wrapper allocates nothing
    either when it is).  Problems whose partials exceed the scratch raise
    AttnError (ATTN_ERR_UNSUPPORTED).  Calls that may overlap on the GPU share
    the scratch and race: order them on one stream.
    """
    lib = load()
    if out is None:
        raise ValueError("attn_decode_noalloc needs a preallocated `out`")
    B, Hq, Hkv, max_S, D = _decode_shapes(q, k_cache, v_cache, seq_lens, out)
    st = lib.attn_decode_noalloc(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(seq_lens), _ptr(out),
                                 B, Hq, Hkv, max_S, D, num_splits, _dtype_code(q), _stream(stream))
    _check(st, "attn_decode_noalloc")
    return out


def decode_chunk(max_S: int, num_splits: int) -> int:
    return load().attn_decode_chunk(max_S, num_splits)


def decode_workspace_bytes(B, Hq, max_S, D, num_splits) -> int:
    return load().attn_decode_workspace_bytes(B, Hq, max_S, D, num_splits)


def check_device_status(stream=None) -> int:
    """Synchronise the stream and return (and clear) the library's device status."""
    return load().attn_check_device_status(_stream(stream))


def debug_set(fault: int, wait_limit_us: int = 0) -> int:
    return load().attn_debug_set(fault, wait_limit_us)


def version() -> int:
    return load().attn_version()
