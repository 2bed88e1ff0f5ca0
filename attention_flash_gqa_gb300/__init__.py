"""Fused flash-style GQA attention for NVIDIA GB300 (sm_103a).

Thin Python binding over the C ABI in ``include/attn.h`` (``libattn_gb300.so``):
argument marshalling only. Every step of the computation runs in the library's
CUDA kernels; there is no CPU or PyTorch fallback, and importing a function whose
library is missing raises immediately.

PyTorch is used for device memory and streams: tensors are passed by data pointer,
outputs and workspaces are allocated with ``torch.empty`` when not supplied, and
work is queued on the current CUDA stream unless ``stream`` is given.

Entry points (same names as the C ABI):

* ``attn_fwd(q, k, v, ...)``          q [B,S,Hq,D], k/v [B,S,Hkv,D] -> (o, lse[B,Hq,S])
* ``attn_fwd_varlen(q, k, v, cu_seqlens, max_seqlen, ...)``  packed [T,H,D] -> (o, lse[Hq,T])
* ``attn_fwd_paged(q, k_cache, v_cache, block_table, seq_lens, cu_q, max_q_len, ...)``
  chunked prefill over a paged cache: packed new tokens [T,Hq,D] -> (o, lse[Hq,T])
* ``attn_bwd(q, k, v, o, lse, dO, ...)``  -> (dQ, dK, dV); dense or packed (cu_seqlens)
* ``attn_merge_lse(o_parts, lse_parts, ...)`` attention results over disjoint key sets -> (o, lse)
* ``attn_decode_paged(q, k_cache, v_cache, block_table, seq_lens, ...)`` -> (o, lse[B,Hq])
* ``attn_workspace_size``, ``attn_get_device_status``, ``attn_status_string``
* ``attn_selftest_wait_timeout`` (exercises the bounded-wait failure reporting)
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

__all__ = [
    "AttnError", "attn_fwd", "attn_fwd_varlen", "attn_fwd_paged", "attn_bwd", "attn_decode_paged", "attn_workspace_size",
    "attn_get_device_status", "attn_status_string", "library_path", "load_library",
    "attn_launch_count", "attn_profile_start", "attn_profile_stop", "attn_decode_paged_noalloc",
    "attn_selftest_wait_timeout", "attn_merge_lse",
    "ATTN_OP_FWD", "ATTN_OP_FWD_VARLEN", "ATTN_OP_BWD", "ATTN_OP_BWD_VARLEN", "ATTN_OP_DECODE_PAGED",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libattn_gb300.so")
_lock = threading.Lock()
_lib = None

ATTN_OP_FWD, ATTN_OP_FWD_VARLEN, ATTN_OP_BWD, ATTN_OP_BWD_VARLEN, ATTN_OP_DECODE_PAGED = 0, 1, 2, 3, 4
STATUS = {0: "ATTN_OK", 1: "ATTN_ERR_INVALID_ARG", 2: "ATTN_ERR_UNSUPPORTED", 3: "ATTN_ERR_MISALIGNED",
          4: "ATTN_ERR_WORKSPACE", 5: "ATTN_ERR_LAUNCH", 6: "ATTN_ERR_DEVICE_TIMEOUT", 7: "ATTN_ERR_DEVICE_BOUNDS",
          8: "ATTN_ERR_NO_DEVICE"}


class AttnError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {STATUS.get(status, status)}")
        self.status = status


def library_path() -> str:
    return _LIB_PATH


def load_library():
    """Load libattn_gb300.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(f"{_LIB_PATH} is missing: build it first (python -m attention_flash_gqa_gb300._build "
                               "or __graft_entry__.build()); there is no fallback implementation")
        lib = ctypes.CDLL(_LIB_PATH)
        P, I, F, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        lib.attn_fwd.argtypes = [P, P, P, P, P, I, I, I, I, I, F, I, I, P, Z, P]
        lib.attn_fwd_varlen.argtypes = [P, P, P, P, P, P, I, I, I, I, I, I, F, I, I, P, Z, P]
        lib.attn_fwd_paged.argtypes = [P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, I, I, F, I, I, P]
        lib.attn_merge_lse.argtypes = [P, P, P, P, I, I, I, I, I, P]
        lib.attn_merge_lse.restype = I
        lib.attn_bwd.argtypes = [P, P, P, P, P, P, P, P, P, I, I, I, I, I, F, I, I, P, I, I, P, Z, P]
        lib.attn_decode_paged.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, I, I, F, I, P, Z, P]
        lib.attn_workspace_size.argtypes = [I, I, I, I, I, I, I, I]
        lib.attn_workspace_size.restype = Z
        lib.attn_get_device_status.argtypes = [P]
        lib.attn_selftest_wait_timeout.argtypes = [I, P]
        lib.attn_status_string.argtypes = [I]
        lib.attn_status_string.restype = ctypes.c_char_p
        lib.attn_version.restype = I
        lib.attn_decode_paged_noalloc.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, I, I, F, I, P]
        lib.attn_decode_paged_noalloc.restype = I
        lib.attn_decode_paged_noalloc_max_bytes.restype = Z
        lib.attn_launch_count.restype = ctypes.c_ulonglong
        lib.attn_profile_start.restype = I
        lib.attn_profile_stop.argtypes = [ctypes.c_char_p, Z]
        lib.attn_profile_stop.restype = I
        for f in (lib.attn_fwd, lib.attn_fwd_varlen, lib.attn_fwd_paged, lib.attn_bwd, lib.attn_decode_paged, lib.attn_get_device_status):
            f.restype = I
        _lib = lib
        return lib


def attn_status_string(status: int) -> str:
    return load_library().attn_status_string(int(status)).decode()


def attn_workspace_size(op: int, B: int = 0, Hq: int = 0, Hkv: int = 0, S: int = 0, D: int = 0, num_seqs: int = 0,
                        max_pages_per_seq: int = 0) -> int:
    return int(load_library().attn_workspace_size(op, B, Hq, Hkv, S, D, num_seqs, max_pages_per_seq))


def attn_launch_count() -> int:
    """Kernel launches issued by the library in this process (monotonic)."""
    return int(load_library().attn_launch_count())


def attn_profile_start() -> None:
    """Bracket every library kernel launch with CUDA events from now on (clears old records)."""
    _check(load_library().attn_profile_start(), "attn_profile_start")


def attn_profile_stop() -> dict:
    """Stop profiling; returns {kernel name: (launches, total device ms)}."""
    buf = ctypes.create_string_buffer(1 << 14)
    n = load_library().attn_profile_stop(buf, len(buf))
    if n < 0:
        raise AttnError(-n, "attn_profile_stop")
    out = {}
    for line in buf.value.decode().splitlines():
        name, cnt, ms = line.split()
        out[name] = (int(cnt), float(ms))
    return out


def _stream_ptr(stream, device):
    import torch

    s = stream if stream is not None else torch.cuda.current_stream(device)
    return ctypes.c_void_p(s.cuda_stream)


def attn_get_device_status(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device fault flags as a status code."""
    import torch

    return int(load_library().attn_get_device_status(_stream_ptr(stream, torch.cuda.current_device())))


def attn_selftest_wait_timeout(limit_ms: int = 100, stream=None) -> None:
    """Enqueue the bounded-wait self-test (a wait that nothing completes gives up after
    limit_ms and records ATTN_ERR_DEVICE_TIMEOUT); read it with attn_get_device_status()."""
    import torch

    _check(int(load_library().attn_selftest_wait_timeout(int(limit_ms), _stream_ptr(stream, torch.cuda.current_device()))),
           "attn_selftest_wait_timeout")


def _check(status: int, what: str):
    if status != 0:
        raise AttnError(status, what)


def _bf16(t, name):
    import torch

    if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous bfloat16 CUDA tensor")
    return ctypes.c_void_p(t.data_ptr())


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


_ws_cache: dict = {}


def _workspace(nbytes: int, device, zero: bool, key: str):
    """Reusable workspace per (device, purpose); grown when too small (allocation is torch's)."""
    import torch

    k = (str(device), key)
    buf = _ws_cache.get(k)
    if buf is None or buf.numel() < nbytes:
        buf = (torch.zeros if zero else torch.empty)(max(nbytes, 256), dtype=torch.uint8, device=device)
        _ws_cache[k] = buf
    return buf


def attn_fwd(q, k, v, o=None, lse=None, *, causal: bool = True, window: int = 0, scale: float | None = None,
             stream=None):
    """Forward of causal (optionally sliding-window) GQA attention, dense [B, S, H, D] layout."""
    import torch

    B, S, Hq, D = q.shape
    Hkv = k.shape[2]
    scale = float(scale if scale is not None else 1.0 / math.sqrt(D))
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq, S), dtype=torch.float32, device=q.device)
    with torch.cuda.device(q.device):  # the library works on the current device
        rc = load_library().attn_fwd(_bf16(q, "q"), _bf16(k, "k"), _bf16(v, "v"), _bf16(o, "o"), _ptr(lse), B, Hq, Hkv,
                                     S, D, scale, int(causal), int(window), None, 0, _stream_ptr(stream, q.device))
    _check(rc, "attn_fwd")
    return o, lse


def attn_fwd_varlen(q, k, v, cu_seqlens, max_seqlen: int, o=None, lse=None, *, causal: bool = True, window: int = 0,
                    scale: float | None = None, stream=None):
    """Forward over packed sequences: q [T, Hq, D], k/v [T, Hkv, D], cu_seqlens int32 [n+1] on the device."""
    import torch

    T, Hq, D = q.shape
    Hkv = k.shape[1]
    scale = float(scale if scale is not None else 1.0 / math.sqrt(D))
    if cu_seqlens.dtype != torch.int32 or not cu_seqlens.is_cuda:
        raise ValueError("cu_seqlens must be an int32 CUDA tensor")
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((Hq, T), dtype=torch.float32, device=q.device)
    with torch.cuda.device(q.device):  # the library works on the current device
        rc = load_library().attn_fwd_varlen(_bf16(q, "q"), _bf16(k, "k"), _bf16(v, "v"), _bf16(o, "o"), _ptr(lse),
                                            _ptr(cu_seqlens), cu_seqlens.numel() - 1, T, int(max_seqlen), Hq, Hkv, D,
                                            scale, int(causal), int(window), None, 0, _stream_ptr(stream, q.device))
    _check(rc, "attn_fwd_varlen")
    return o, lse


def attn_fwd_paged(q, k_cache, v_cache, block_table, seq_lens, cu_q, max_q_len: int, o=None, lse=None, *,
                   causal: bool = True, window: int = 0, scale: float | None = None, stream=None):
    """Chunked prefill: q [T,Hq,D] new tokens packed by cu_q, caches [pages,16,Hkv,D], block_table int32
    [R,max_pages], seq_lens int32 [R] (cached tokens including the new ones), cu_q int32 [R+1]."""
    import torch

    T, Hq, D = q.shape
    num_pages, page_size, Hkv, _ = k_cache.shape
    scale = float(scale if scale is not None else 1.0 / math.sqrt(D))
    for t, n in ((block_table, "block_table"), (seq_lens, "seq_lens"), (cu_q, "cu_q")):
        if t.dtype != torch.int32 or not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{n} must be a contiguous int32 CUDA tensor")
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((Hq, T), dtype=torch.float32, device=q.device)
    with torch.cuda.device(q.device):  # the library works on the current device
        rc = load_library().attn_fwd_paged(
            _bf16(q, "q"), _bf16(k_cache, "k_cache"), _bf16(v_cache, "v_cache"), _ptr(block_table), _ptr(seq_lens),
            _ptr(cu_q), _bf16(o, "o"), _ptr(lse), cu_q.numel() - 1, T, int(max_q_len), Hq, Hkv, D, page_size,
            block_table.shape[1], num_pages, scale, int(causal), int(window), _stream_ptr(stream, q.device))
    _check(rc, "attn_fwd_paged")
    return o, lse


def attn_merge_lse(o_parts, lse_parts, o=None, lse=None, *, stream=None):
    """Combine results over disjoint key sets: o_parts [P,B,S,H,D] (or [P,T,H,D]) bf16, lse_parts
    [P,B,H,S] (or [P,H,T]) fp32 -> (o, lse) in the forward's layouts. o / lse may be o_parts[0] /
    lse_parts[0] (in-place running merge)."""
    import torch

    packed = o_parts.dim() == 4
    if packed:
        P, S, H, D = o_parts.shape
        B = 1
    else:
        P, B, S, H, D = o_parts.shape
    if lse_parts.dtype != torch.float32 or not lse_parts.is_cuda or not lse_parts.is_contiguous():
        raise ValueError("lse_parts must be a contiguous float32 CUDA tensor")
    if tuple(lse_parts.shape) != ((P, H, S) if packed else (P, B, H, S)):
        raise ValueError("lse_parts shape does not match o_parts")
    if o is None:
        o = torch.empty(o_parts.shape[1:], dtype=torch.bfloat16, device=o_parts.device)
    if lse is None:
        lse = torch.empty(lse_parts.shape[1:], dtype=torch.float32, device=o_parts.device)
    with torch.cuda.device(o_parts.device):  # the library works on the current device
        rc = load_library().attn_merge_lse(_bf16(o_parts, "o_parts"), _ptr(lse_parts), _bf16(o, "o"), _ptr(lse), P, B,
                                           S, H, D, _stream_ptr(stream, o_parts.device))
    _check(rc, "attn_merge_lse")
    return o, lse


def attn_bwd(q, k, v, o, lse, dO, dq=None, dk=None, dv=None, *, causal: bool = True, window: int = 0,
             scale: float | None = None, cu_seqlens=None, max_seqlen: int = 0, workspace=None, stream=None):
    """Gradients (dQ, dK, dV). Dense [B,S,H,D] when cu_seqlens is None, else packed [T,H,D]."""
    import torch

    if cu_seqlens is None:
        B, S, Hq, D = q.shape
        Hkv = k.shape[2]
        nseq = 0
    else:
        B, (S, Hq, D) = 1, q.shape
        Hkv = k.shape[1]
        nseq = cu_seqlens.numel() - 1
    scale = float(scale if scale is not None else 1.0 / math.sqrt(D))
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    need = attn_workspace_size(ATTN_OP_BWD if cu_seqlens is None else ATTN_OP_BWD_VARLEN, B, Hq, Hkv, S, D, nseq)
    if workspace is None:
        workspace = _workspace(need, q.device, False, "bwd")
    with torch.cuda.device(q.device):  # the library works on the current device
        rc = load_library().attn_bwd(_bf16(q, "q"), _bf16(k, "k"), _bf16(v, "v"), _bf16(o, "o"), _ptr(lse),
                                     _bf16(dO, "dO"), _bf16(dq, "dQ"), _bf16(dk, "dK"), _bf16(dv, "dV"), B, Hq, Hkv, S, D,
                                     scale, int(causal), int(window), _ptr(cu_seqlens), nseq, int(max_seqlen),
                                     _ptr(workspace), workspace.numel() * workspace.element_size(),
                                     _stream_ptr(stream, q.device))
    _check(rc, "attn_bwd")
    return dq, dk, dv


def attn_decode_paged(q, k_cache, v_cache, block_table, seq_lens, o=None, lse=None, *, scale: float | None = None,
                      window: int = 0, workspace=None, stream=None):
    """Single-token decode: q [B,Hq,D], caches [pages,16,Hkv,D], block_table int32 [B,max_pages], seq_lens int32 [B];
    window > 0: the query sees only the last `window` keys."""
    import torch

    B, Hq, D = q.shape
    num_pages, page_size, Hkv, _ = k_cache.shape
    scale = float(scale if scale is not None else 1.0 / math.sqrt(D))
    for t, n in ((block_table, "block_table"), (seq_lens, "seq_lens")):
        if t.dtype != torch.int32 or not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{n} must be a contiguous int32 CUDA tensor")
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    need = attn_workspace_size(ATTN_OP_DECODE_PAGED, B, Hq, Hkv, 0, D)
    if workspace is None:
        workspace = _workspace(need, q.device, False, "decode")
    with torch.cuda.device(q.device):  # the library works on the current device
        rc = load_library().attn_decode_paged(_bf16(q, "q"), _bf16(k_cache, "k_cache"), _bf16(v_cache, "v_cache"),
                                              _ptr(block_table), _ptr(seq_lens), _bf16(o, "o"), _ptr(lse), B, Hq, Hkv, D,
                                              page_size, block_table.shape[1], num_pages, scale, int(window),
                                              _ptr(workspace),
                                              workspace.numel() * workspace.element_size(), _stream_ptr(stream, q.device))
    _check(rc, "attn_decode_paged")
    return o, lse


def attn_decode_paged_noalloc(q, k_cache, v_cache, block_table, seq_lens, o, lse, *, scale: float | None = None,
                              window: int = 0, stream=None):
    """attn_decode_paged without a workspace: the library's built-in scratch buffer is used.

    For callers that cannot allocate device memory on their decode path, so the outputs
    ``o`` [B,Hq,D] and ``lse`` [B,Hq] must be supplied by the caller. Calls that overlap
    on the GPU share the buffer and race; see include/attn.h for the size limit.
    """
    import torch

    B, Hq, D = q.shape
    num_pages, page_size, Hkv, _ = k_cache.shape
    scale = float(scale if scale is not None else 1.0 / math.sqrt(D))
    for t, n in ((block_table, "block_table"), (seq_lens, "seq_lens")):
        if t.dtype != torch.int32 or not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{n} must be a contiguous int32 CUDA tensor")
    with torch.cuda.device(q.device):  # the library works on the current device
        rc = load_library().attn_decode_paged_noalloc(
            _bf16(q, "q"), _bf16(k_cache, "k_cache"), _bf16(v_cache, "v_cache"), _ptr(block_table), _ptr(seq_lens),
            _bf16(o, "o"), _ptr(lse), B, Hq, Hkv, D, page_size, block_table.shape[1], num_pages, scale, int(window),
            _stream_ptr(stream, q.device))
    _check(rc, "attn_decode_paged_noalloc")
    return o, lse
