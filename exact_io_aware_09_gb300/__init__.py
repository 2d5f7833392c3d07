"""Python binding of libattn_gb300.so (exact attention for GB300 / sm_103a).

The functions below only marshal arguments (torch tensors -> device pointers, sizes, the
current CUDA stream) and call the C ABI declared in ``include/attn.h``; every step of the
computation runs in the library's CUDA kernels.  There is no CPU or PyTorch fallback: if the
library is missing the import fails, and an unsupported request raises ``AttnError``.
"""
from __future__ import annotations

import ctypes
import math
import os

__all__ = [
    "AttnError", "attn_fwd", "attn_fwd_window", "attn_fwd_block_sparse", "attn_fwd_fp8",
    "attn_fwd_fp8_workspace_bytes", "attn_fwd_fp8_workspace_offsets",
    "attn_bwd", "attn_bwd_workspace_bytes",
    "attn_decode_splitkv", "attn_decode_workspace_bytes", "attn_decode_paged",
    "attn_decode_splitkv_static", "attn_decode_static_scratch_bytes",
    "attn_poll_status", "attn_status_string", "attn_fwd_kv_tiles", "attn_fwd_kv_span",
    "attn_fwd_set_d64_kernel", "D64_AUTO", "D64_PAIR", "D64_SINGLE",
    "attn_bwd_kv_order", "attn_selftest_timeout",
    "attn_version", "library_path", "lib",
]

_PKG = os.path.dirname(os.path.abspath(__file__))
library_path = os.path.join(_PKG, "libattn_gb300.so")

if not os.path.exists(library_path):
    raise ImportError(
        f"{library_path} is missing: build it first (python exact_io_aware_09_gb300/build.py "
        "or __graft_entry__.build()); there is no fallback implementation")

lib = ctypes.CDLL(library_path)

_P = ctypes.c_void_p
_I = ctypes.c_int
_F = ctypes.c_float
_SZ = ctypes.c_size_t
lib.attn_fwd.argtypes = [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _P, _I]
lib.attn_fwd.restype = _I
lib.attn_bwd_workspace_bytes.argtypes = [_I, _I, _I]
lib.attn_bwd_workspace_bytes.restype = _SZ
lib.attn_bwd.argtypes = [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _I, _P,
                         _SZ, _P]
lib.attn_bwd.restype = _I
lib.attn_fwd_fp8_workspace_bytes.argtypes = [_I] * 6
lib.attn_fwd_fp8_workspace_bytes.restype = _SZ
lib.attn_fwd_fp8_workspace_offsets.argtypes = [_I] * 6 + [_P]
lib.attn_fwd_fp8_workspace_offsets.restype = _I
lib.attn_fwd_fp8.argtypes = [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _P, _P, _SZ, _P, _I]
lib.attn_fwd_fp8.restype = _I
lib.attn_fwd_window.argtypes = [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _P, _I]
lib.attn_fwd_window.restype = _I
lib.attn_fwd_block_sparse.argtypes = [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _P, _F, _P,
                                      _I]
lib.attn_fwd_block_sparse.restype = _I
lib.attn_decode_workspace_bytes.argtypes = [_I, _I, _I, _I, _I]
lib.attn_decode_workspace_bytes.restype = _SZ
lib.attn_decode_splitkv.argtypes = [_P, _P, _P, _P, _I, _I, _P, _P, _I, _I, _I, _I, _I, _F, _I,
                                    _P, _SZ, _P]
lib.attn_decode_splitkv.restype = _I
lib.attn_decode_splitkv_static.argtypes = [_P, _P, _P, _P, _I, _I, _P, _P, _I, _I, _I, _I, _I,
                                           _F, _I, _P]
lib.attn_decode_splitkv_static.restype = _I
lib.attn_decode_paged.argtypes = [_P, _P, _P, _P, _P, _I, _I, _I, _I, _P, _P, _I, _I, _I, _I, _I, _F,
                                  _I, _P, _SZ, _P]
lib.attn_decode_paged.restype = _I
lib.attn_decode_static_scratch_bytes.argtypes = []
lib.attn_decode_static_scratch_bytes.restype = _SZ
lib.attn_poll_status.argtypes = [_P]
lib.attn_poll_status.restype = _I
lib.attn_status_string.argtypes = [_I]
lib.attn_status_string.restype = ctypes.c_char_p
lib.attn_fwd_kv_tiles.argtypes = [_I, _I, _I, _I, _I, _I, ctypes.POINTER(_I), ctypes.POINTER(_I)]
lib.attn_fwd_kv_tiles.restype = _I
lib.attn_fwd_set_d64_kernel.argtypes = [_I]
lib.attn_fwd_set_d64_kernel.restype = _I
lib.attn_bwd_kv_order.argtypes = [_I] * 7 + [ctypes.POINTER(ctypes.c_uint16), _I, ctypes.POINTER(_I)]
lib.attn_bwd_kv_order.restype = _I
lib.attn_fwd_kv_span.argtypes = [_I, _I, _I, _I, _I, _I, _I] + [ctypes.POINTER(_I)] * 4
lib.attn_fwd_kv_span.restype = _I
lib.attn_selftest_timeout.argtypes = [_I, _P]
lib.attn_selftest_timeout.restype = _I
lib.attn_version.argtypes = []
lib.attn_version.restype = ctypes.c_char_p

ATTN_F16, ATTN_BF16 = 0, 1


class AttnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {attn_status_string(status)} (status {status})")


def attn_status_string(status: int) -> str:
    return lib.attn_status_string(int(status)).decode()


def attn_version() -> str:
    return lib.attn_version().decode()


def _torch():
    import torch

    return torch


def _stream_handle(stream, device=None):
    """The raw handle of ``stream`` (a torch stream or an integer handle); None = torch's
    current stream of ``device`` (of the current device when that is None too).  A torch
    stream must belong to ``device``."""
    torch = _torch()
    if stream is None:
        stream = torch.cuda.current_stream(device)
    elif device is not None and getattr(stream, "device", device) != device:
        raise AttnError(-1, f"stream on {stream.device}, tensors on {device}")
    return ctypes.c_void_p(int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream))


def _on_device(where, first, *others):
    """Checks that every given tensor sits on ``first``'s CUDA device and returns a context
    that makes that device current, so that the library's launches, its per-device state and
    torch's default stream all refer to the device that holds the data."""
    torch = _torch()
    if not first.is_cuda:
        raise AttnError(-1, f"{where}: tensors must be CUDA tensors")
    for t in others:
        if t is not None and t.device != first.device:
            raise AttnError(-1, f"{where}: tensors on {first.device} and {t.device}")
    return torch.cuda.device(first.device)


def _dtype_code(t) -> int:
    torch = _torch()
    if t.dtype == torch.float16:
        return ATTN_F16
    if t.dtype == torch.bfloat16:
        return ATTN_BF16
    raise AttnError(-2, f"dtype {t.dtype}")


def _check(status: int, where: str):
    if status != 0:
        raise AttnError(status, where)


def _dev_ptr(t, name):
    if t is None:
        return None
    if not t.is_cuda or not t.is_contiguous():
        raise AttnError(-1, f"{name} must be a contiguous CUDA tensor")
    return ctypes.c_void_p(t.data_ptr())


def attn_fwd(q, k, v, o=None, lse=None, causal: bool = False, scale: float | None = None,
             stream=None):
    """Exact attention forward.  q [B,Hq,N_q,d], k/v [B,Hkv,N_kv,d] fp16/bf16 CUDA tensors.

    Returns (o [B,Hq,N_q,d] same dtype, lse [B,Hq,N_q] fp32).  Enqueued on ``stream``
    (default: torch's current stream); no synchronisation.
    """
    torch = _torch()
    B, Hq, N_q, d = q.shape
    _, Hkv, N_kv, _ = k.shape
    if k.shape != v.shape or k.shape[0] != B or k.shape[3] != d or k.dtype != q.dtype or v.dtype != q.dtype:
        raise AttnError(-1, "attn_fwd: q/k/v shapes or dtypes disagree")
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq, N_q), device=q.device, dtype=torch.float32)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    with _on_device("attn_fwd", q, k, v, o, lse):
        st = lib.attn_fwd(_dev_ptr(q, "q"), _dev_ptr(k, "k"), _dev_ptr(v, "v"), _dev_ptr(o, "o"),
                          _dev_ptr(lse, "lse"), B, Hq, Hkv, N_q, N_kv, d, int(bool(causal)),
                          float(scale), _stream_handle(stream, q.device), _dtype_code(q))
    _check(st, "attn_fwd")
    return o, lse


def _fwd_prep(q, k, v, o, lse, scale):
    torch = _torch()
    B, Hq, N_q, d = q.shape
    _, Hkv, N_kv, _ = k.shape
    if k.shape != v.shape or k.shape[0] != B or k.shape[3] != d or k.dtype != q.dtype or v.dtype != q.dtype:
        raise AttnError(-1, "attn_fwd: q/k/v shapes or dtypes disagree")
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq, N_q), device=q.device, dtype=torch.float32)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    return B, Hq, Hkv, N_q, N_kv, d, o, lse, float(scale)


def attn_bwd_workspace_bytes(B: int, Hq: int, N_q: int) -> int:
    return int(lib.attn_bwd_workspace_bytes(B, Hq, N_q))


def attn_bwd(q, k, v, o, dout, lse, causal: bool = False, scale: float | None = None,
             dq=None, dk=None, dv=None, workspace=None, stream=None):
    """Gradients (dq, dk, dv) of attn_fwd for the incoming gradient ``dout`` (shape of o).

    q/o/dout [B,Hq,N_q,d], k/v [B,Hkv,N_kv,d] 16-bit CUDA tensors, lse [B,Hq,N_q] fp32 as
    attn_fwd returns it.  Deterministic.
    """
    torch = _torch()
    B, Hq, N_q, d = q.shape
    _, Hkv, N_kv, _ = k.shape
    for t, nm in ((o, "o"), (dout, "dout")):
        if t.shape != q.shape or t.dtype != q.dtype:
            raise AttnError(-1, f"attn_bwd: {nm} must match q")
    if k.shape != v.shape or k.dtype != q.dtype or v.dtype != q.dtype or lse.dtype != torch.float32:
        raise AttnError(-1, "attn_bwd: k/v/lse shapes or dtypes disagree")
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if workspace is None:
        workspace = torch.empty(max(int(lib.attn_bwd_workspace_bytes(B, Hq, N_q)), 1),
                                device=q.device, dtype=torch.uint8)
    with _on_device("attn_bwd", q, k, v, o, dout, lse, dq, dk, dv, workspace):
        st = lib.attn_bwd(_dev_ptr(q, "q"), _dev_ptr(k, "k"), _dev_ptr(v, "v"), _dev_ptr(o, "o"),
                          _dev_ptr(dout, "dout"), _dev_ptr(lse, "lse"), _dev_ptr(dq, "dq"),
                          _dev_ptr(dk, "dk"), _dev_ptr(dv, "dv"), B, Hq, Hkv, N_q, N_kv, d,
                          int(bool(causal)), float(scale), _dtype_code(q),
                          _dev_ptr(workspace, "workspace"), workspace.numel(),
                          _stream_handle(stream, q.device))
    _check(st, "attn_bwd")
    return dq, dk, dv


def attn_fwd_fp8_workspace_bytes(B, Hq, Hkv, N_q, N_kv, d) -> int:
    return int(lib.attn_fwd_fp8_workspace_bytes(B, Hq, Hkv, N_q, N_kv, d))


def attn_fwd_fp8_workspace_offsets(B, Hq, Hkv, N_q, N_kv, d):
    """Byte offsets of (Q codes, K codes, V^T codes, Q scales, K scales, V scales, scratch)."""
    off = (ctypes.c_size_t * 7)()
    _check(lib.attn_fwd_fp8_workspace_offsets(B, Hq, Hkv, N_q, N_kv, d, off),
           "attn_fwd_fp8_workspace_offsets")
    return list(off)


def attn_fwd_fp8(q, k, v, signs=None, o=None, lse=None, causal: bool = False,
                 scale: float | None = None, workspace=None, stream=None):
    """FP8 prefill with incoherent processing.  signs: int8 CUDA tensor [d] of +-1 (None: no
    rotation).  Shapes and return value as attn_fwd (d = 128)."""
    torch = _torch()
    B, Hq, Hkv, N_q, N_kv, d, o, lse, scale = _fwd_prep(q, k, v, o, lse, scale)
    if signs is not None and (signs.dtype != torch.int8 or tuple(signs.shape) != (d,)):
        raise AttnError(-1, "attn_fwd_fp8: signs must be int8 [d]")
    if workspace is None:
        workspace = torch.empty(max(1, attn_fwd_fp8_workspace_bytes(B, Hq, Hkv, N_q, N_kv, d)),
                                device=q.device, dtype=torch.uint8)
    with _on_device("attn_fwd_fp8", q, k, v, o, lse, signs, workspace):
        st = lib.attn_fwd_fp8(_dev_ptr(q, "q"), _dev_ptr(k, "k"), _dev_ptr(v, "v"),
                              _dev_ptr(o, "o"), _dev_ptr(lse, "lse"), B, Hq, Hkv, N_q, N_kv, d,
                              int(bool(causal)), scale,
                              _dev_ptr(signs, "signs") if signs is not None else None,
                              _dev_ptr(workspace, "workspace"), workspace.numel(),
                              _stream_handle(stream, q.device), _dtype_code(q))
    _check(st, "attn_fwd_fp8")
    return o, lse


def attn_fwd_window(q, k, v, window: int, o=None, lse=None, scale: float | None = None,
                    stream=None):
    """Sliding-window prefill: key j visible to row i iff 0 <= i + N_kv - N_q - j <= window.

    Shapes and return value as attn_fwd.
    """
    B, Hq, Hkv, N_q, N_kv, d, o, lse, scale = _fwd_prep(q, k, v, o, lse, scale)
    with _on_device("attn_fwd_window", q, k, v, o, lse):
        st = lib.attn_fwd_window(_dev_ptr(q, "q"), _dev_ptr(k, "k"), _dev_ptr(v, "v"),
                                 _dev_ptr(o, "o"), _dev_ptr(lse, "lse"), B, Hq, Hkv, N_q, N_kv, d,
                                 int(window), scale, _stream_handle(stream, q.device),
                                 _dtype_code(q))
    _check(st, "attn_fwd_window")
    return o, lse


def attn_fwd_block_sparse(q, k, v, block_mask, causal: bool = False, o=None, lse=None,
                          scale: float | None = None, stream=None):
    """Block-sparse prefill.  block_mask: uint8 CUDA tensor [ceil(N_q/128), ceil(N_kv/128)],
    nonzero = compute that (query tile, key tile) block.  Shapes and return value as attn_fwd.
    """
    torch = _torch()
    B, Hq, Hkv, N_q, N_kv, d, o, lse, scale = _fwd_prep(q, k, v, o, lse, scale)
    shape = ((N_q + 127) // 128, (N_kv + 127) // 128)
    if (block_mask.dtype != torch.uint8 or tuple(block_mask.shape) != shape
            or not block_mask.is_contiguous()):
        raise AttnError(-1, f"attn_fwd_block_sparse: block_mask must be contiguous uint8 {shape}")
    with _on_device("attn_fwd_block_sparse", q, k, v, o, lse, block_mask):
        st = lib.attn_fwd_block_sparse(_dev_ptr(q, "q"), _dev_ptr(k, "k"), _dev_ptr(v, "v"),
                                       _dev_ptr(o, "o"), _dev_ptr(lse, "lse"), B, Hq, Hkv, N_q,
                                       N_kv, d, int(bool(causal)),
                                       _dev_ptr(block_mask, "block_mask"), scale,
                                       _stream_handle(stream, q.device), _dtype_code(q))
    _check(st, "attn_fwd_block_sparse")
    return o, lse


def attn_fwd_kv_span(q_tile: int, block_m: int, block_n: int, N_q: int, N_kv: int,
                     causal: bool, window: int = -1):
    """(j_begin, j_end, lo_masked, hi_masked) of the prefill schedule for one query tile."""
    out = [_I(0) for _ in range(4)]
    _check(lib.attn_fwd_kv_span(q_tile, block_m, block_n, N_q, N_kv, int(bool(causal)),
                                int(window), *[ctypes.byref(x) for x in out]), "attn_fwd_kv_span")
    return tuple(x.value for x in out)


def attn_decode_paged(q, k_pages, v_pages, block_table, seqlens_k, max_seqlen_k: int, o=None,
                      lse=None, split_size: int = 512, scale: float | None = None, workspace=None,
                      stream=None):
    """One split-KV decode step over a paged cache.

    q [B,Hq,d]; k_pages/v_pages [num_pages, page_size, Hkv, d]; block_table int32 CUDA
    [B, max_pages_per_seq]; seqlens_k int32 CUDA [B].  Returns (o [B,Hq,d], lse [B,Hq] fp32).
    """
    torch = _torch()
    B, Hq, d = q.shape
    num_pages, page_size, Hkv, _ = k_pages.shape
    if v_pages.shape != k_pages.shape or k_pages.dtype != q.dtype or v_pages.dtype != q.dtype:
        raise AttnError(-1, "attn_decode_paged: page pools disagree with q")
    if block_table.dtype != torch.int32 or block_table.dim() != 2 or block_table.shape[0] != B:
        raise AttnError(-1, "attn_decode_paged: block_table must be int32 [B, max_pages]")
    if seqlens_k.dtype != torch.int32 or tuple(seqlens_k.shape) != (B,):
        raise AttnError(-1, "attn_decode_paged: seqlens_k must be int32 [B]")
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq), device=q.device, dtype=torch.float32)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    need = attn_decode_workspace_bytes(B, Hq, max_seqlen_k, split_size, d)
    if workspace is None:
        workspace = torch.empty(max(need, 1), device=q.device, dtype=torch.uint8)
    with _on_device("attn_decode_paged", q, k_pages, v_pages, block_table, seqlens_k, o, lse,
                    workspace):
        st = lib.attn_decode_paged(_dev_ptr(q, "q"), _dev_ptr(k_pages, "k_pages"),
                                   _dev_ptr(v_pages, "v_pages"),
                                   _dev_ptr(block_table, "block_table"),
                                   _dev_ptr(seqlens_k, "seqlens_k"), num_pages, page_size,
                                   block_table.shape[1], int(max_seqlen_k), _dev_ptr(o, "o"),
                                   _dev_ptr(lse, "lse"), B, Hq, Hkv, d, int(split_size),
                                   float(scale), _dtype_code(q), _dev_ptr(workspace, "workspace"),
                                   workspace.numel(), _stream_handle(stream, q.device))
    _check(st, "attn_decode_paged")
    return o, lse


def attn_decode_workspace_bytes(B: int, Hq: int, max_seqlen_k: int, split_size: int, d: int) -> int:
    return int(lib.attn_decode_workspace_bytes(B, Hq, max_seqlen_k, split_size, d))


def attn_decode_splitkv(q, k_cache, v_cache, cu_seqlens_k, max_seqlen_k: int, o=None, lse=None,
                        split_size: int = 512, scale: float | None = None, workspace=None,
                        stream=None):
    """One split-KV decode step.

    q [B,Hq,d]; k_cache/v_cache [capacity,Hkv,d]; cu_seqlens_k int32 CUDA [B+1].
    ``workspace``: a uint8 CUDA tensor of at least attn_decode_workspace_bytes(...) bytes
    (allocated here when omitted).  Returns (o [B,Hq,d], lse [B,Hq] fp32).
    """
    torch = _torch()
    B, Hq, d = q.shape
    cap, Hkv, _ = k_cache.shape
    if cu_seqlens_k.dtype != torch.int32 or cu_seqlens_k.numel() != B + 1:
        raise AttnError(-1, "attn_decode_splitkv: cu_seqlens_k must be int32 [B+1]")
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq), device=q.device, dtype=torch.float32)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    need = attn_decode_workspace_bytes(B, Hq, max_seqlen_k, split_size, d)
    if workspace is None:
        workspace = torch.empty(max(need, 16), device=q.device, dtype=torch.uint8)
    with _on_device("attn_decode_splitkv", q, k_cache, v_cache, cu_seqlens_k, o, lse,
                    workspace):
        st = lib.attn_decode_splitkv(_dev_ptr(q, "q"), _dev_ptr(k_cache, "k_cache"),
                                     _dev_ptr(v_cache, "v_cache"),
                                     _dev_ptr(cu_seqlens_k, "cu_seqlens_k"), cap,
                                     int(max_seqlen_k), _dev_ptr(o, "o"), _dev_ptr(lse, "lse"), B,
                                     Hq, Hkv, d, int(split_size), float(scale), _dtype_code(q),
                                     _dev_ptr(workspace, "workspace"), workspace.numel(),
                                     _stream_handle(stream, q.device))
    _check(st, "attn_decode_splitkv")
    return o, lse


def attn_decode_static_scratch_bytes() -> int:
    return int(lib.attn_decode_static_scratch_bytes())


def attn_decode_splitkv_static(q, k_cache, v_cache, cu_seqlens_k, max_seqlen_k: int, o=None,
                               lse=None, split_size: int = 512, scale: float | None = None,
                               stream=None):
    """attn_decode_splitkv without a workspace, for callers that cannot allocate device memory
    during a decode step.

    The partial states go to a fixed 32 MiB scratch array owned by the library (one per GPU,
    kept until exit); requests needing more raise AttnError(ATTN_ERR_WORKSPACE).  All calls
    share that array, so calls must not overlap on the GPU.  The first call on each GPU looks
    the array up; make it before any stream capture.  ``o`` and ``lse`` are allocated here only
    when omitted -- pass them to keep the call allocation-free.
    """
    torch = _torch()
    B, Hq, d = q.shape
    cap, Hkv, _ = k_cache.shape
    if cu_seqlens_k.dtype != torch.int32 or cu_seqlens_k.numel() != B + 1:
        raise AttnError(-1, "attn_decode_splitkv_static: cu_seqlens_k must be int32 [B+1]")
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq), device=q.device, dtype=torch.float32)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    with _on_device("attn_decode_splitkv_static", q, k_cache, v_cache, cu_seqlens_k, o, lse):
        st = lib.attn_decode_splitkv_static(_dev_ptr(q, "q"), _dev_ptr(k_cache, "k_cache"),
                                            _dev_ptr(v_cache, "v_cache"),
                                            _dev_ptr(cu_seqlens_k, "cu_seqlens_k"), cap,
                                            int(max_seqlen_k), _dev_ptr(o, "o"),
                                            _dev_ptr(lse, "lse"), B, Hq, Hkv, d, int(split_size),
                                            float(scale), _dtype_code(q),
                                            _stream_handle(stream, q.device))
    _check(st, "attn_decode_splitkv_static")
    return o, lse


def attn_poll_status(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device status word."""
    return int(lib.attn_poll_status(_stream_handle(stream)))


def attn_fwd_kv_tiles(q_tile: int, block_m: int, block_n: int, N_q: int, N_kv: int, causal: bool):
    """(n_tiles, first_masked) of the prefill schedule for one query tile (host only)."""
    n = _I(0)
    fm = _I(0)
    _check(lib.attn_fwd_kv_tiles(q_tile, block_m, block_n, N_q, N_kv, int(bool(causal)),
                                 ctypes.byref(n), ctypes.byref(fm)), "attn_fwd_kv_tiles")
    return n.value, fm.value


D64_AUTO, D64_PAIR, D64_SINGLE = 0, 1, 2


def attn_fwd_set_d64_kernel(mode: int) -> int:
    """Choose the d = 64 prefill kernel for later calls (D64_AUTO, D64_PAIR: two query tiles per
    work item, D64_SINGLE: one); returns the previous mode."""
    r = int(lib.attn_fwd_set_d64_kernel(int(mode)))
    if r < 0:
        raise AttnError(r, "attn_fwd_set_d64_kernel")
    return r


def attn_bwd_kv_order(B: int, Hq: int, Hkv: int, N_q: int, N_kv: int, causal: bool, n_sm: int,
                      cap: int = 2048):
    """Launch order of attn_bwd's dK/dV blocks on n_sm SMs (host only): the job of every block,
    or an empty list when the default order (job = block index) stands."""
    buf = (ctypes.c_uint16 * max(cap, 1))()
    n = _I(0)
    _check(lib.attn_bwd_kv_order(B, Hq, Hkv, N_q, N_kv, int(bool(causal)), n_sm, buf, cap,
                                 ctypes.byref(n)), "attn_bwd_kv_order")
    return list(buf[:n.value])


def attn_selftest_timeout(limit_us: int, stream=None) -> None:
    _check(lib.attn_selftest_timeout(int(limit_us), _stream_handle(stream)), "attn_selftest_timeout")
