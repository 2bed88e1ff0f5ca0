"""fp64 CPU oracle for fused GQA attention (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The attention library never does, and the
oracle never imports the library: the two share nothing but the seeded input
generator in ``synth``.

All arithmetic lives in ``oracle.c`` (plain C, fp64, one query row at a time);
this module only compiles it and marshals numpy arrays through ctypes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()

_p = ctypes.c_void_p
_i = ctypes.c_int
_d = ctypes.c_double
_l = ctypes.c_long


def build(force: bool = False, mutant: int = 0, out: str | None = None) -> str:
    """Compile the oracle with gcc. ``mutant`` > 0 plants a known mistake (for the pin tests)."""
    out = out or LIB_PATH
    if force or mutant or not os.path.exists(out) or os.path.getmtime(out) < os.path.getmtime(_SRC):
        tmp = out + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", f"-DORACLE_MUTANT={int(mutant)}",
                               "-o", tmp, _SRC, "-lm", "-lpthread"])
        os.replace(tmp, out)
    return out


def _ptr(a):
    return None if a is None else a.ctypes.data


def _u16(a):
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError("bf16 inputs are passed as uint16 bit patterns")
    return a


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


class Oracle:
    """Handle on one compiled oracle library."""

    def __init__(self, path: str | None = None):
        path = path or build()
        self.path = path
        lib = ctypes.CDLL(path)
        lib.oracle_attn_fwd.argtypes = [_p, _p, _p, _i, _i, _i, _i, _i, _d, _i, _i, _p, _p, _i]
        lib.oracle_attn_bwd.argtypes = [_p, _p, _p, _p, _i, _i, _i, _i, _i, _d, _i, _i, _p, _p, _p, _p, _p, _p, _i]
        lib.oracle_attn_fwd_varlen.argtypes = [_p, _p, _p, _p, _i, _i, _i, _i, _d, _i, _i, _p, _p, _i]
        lib.oracle_attn_bwd_varlen.argtypes = [_p, _p, _p, _p, _p, _i, _i, _i, _i, _d, _i, _i, _p, _p, _p, _p, _i]
        lib.oracle_attn_fwd_rows.argtypes = [_p, _p, _p, _p, _i, _i, _i, _i, _i, _d, _i, _i, _p, _l, _p, _p, _i]
        lib.oracle_attn_dq_rows.argtypes = [_p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _d, _i, _i, _p, _l, _p, _i]
        lib.oracle_attn_dkv_rows.argtypes = [_p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _d, _i, _i, _p, _l, _p, _p, _i]
        lib.oracle_attn_decode_paged.argtypes = [_p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _i, _d, _i, _p, _p, _i]
        lib.oracle_attn_prefill_paged.argtypes = [_p, _p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _i, _d, _i, _p, _p,
                                                  _i]
        lib.oracle_merge_lse.argtypes = [_p, _p, _i, _i, _i, _i, _i, _p, _p]
        lib.oracle_mutant_id.restype = _i
        self.lib = lib
        self.mutant = lib.oracle_mutant_id()

    @staticmethod
    def _check(rc, what):
        if rc != 0:
            raise ValueError(f"oracle {what} rejected its arguments (rc={rc})")

    # ---- dense [B, S, H, D] -------------------------------------------------------
    def fwd(self, q, k, v, scale, causal=1, window=0, nthreads=None):
        q, k, v = _u16(q), _u16(k), _u16(v)
        B, S, Hq, D = q.shape
        Hkv = k.shape[2]
        o = np.empty((B, S, Hq, D), np.float64)
        lse = np.empty((B, Hq, S), np.float64)
        self._check(self.lib.oracle_attn_fwd(_ptr(q), _ptr(k), _ptr(v), B, Hq, Hkv, S, D, scale, causal, window,
                                             _ptr(o), _ptr(lse), nthreads or default_threads()), "fwd")
        return o, lse

    def bwd(self, q, k, v, do, scale, causal=1, window=0, nthreads=None):
        """Returns dq, dk, dv, o, delta, max |Delta - dO.o| over rows."""
        q, k, v, do = _u16(q), _u16(k), _u16(v), _u16(do)
        B, S, Hq, D = q.shape
        Hkv = k.shape[2]
        dq = np.empty((B, S, Hq, D), np.float64)
        dk = np.empty((B, S, Hkv, D), np.float64)
        dv = np.empty((B, S, Hkv, D), np.float64)
        o = np.empty((B, S, Hq, D), np.float64)
        delta = np.empty((B, Hq, S), np.float64)
        gap = ctypes.c_double(0.0)
        self._check(self.lib.oracle_attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(do), B, Hq, Hkv, S, D, scale, causal,
                                             window, _ptr(dq), _ptr(dk), _ptr(dv), _ptr(o), _ptr(delta),
                                             ctypes.addressof(gap), nthreads or default_threads()), "bwd")
        return dq, dk, dv, o, delta, gap.value

    # ---- packed varlen [T, H, D] --------------------------------------------------
    def fwd_varlen(self, q, k, v, cu_seqlens, scale, causal=1, window=0, nthreads=None):
        q, k, v = _u16(q), _u16(k), _u16(v)
        cu = np.ascontiguousarray(cu_seqlens, dtype=np.int32)
        T, Hq, D = q.shape
        Hkv = k.shape[1]
        o = np.empty((T, Hq, D), np.float64)
        lse = np.empty((Hq, T), np.float64)
        self._check(self.lib.oracle_attn_fwd_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(cu), len(cu) - 1, Hq, Hkv, D,
                                                    scale, causal, window, _ptr(o), _ptr(lse),
                                                    nthreads or default_threads()), "fwd_varlen")
        return o, lse

    def bwd_varlen(self, q, k, v, do, cu_seqlens, scale, causal=1, window=0, nthreads=None):
        q, k, v, do = _u16(q), _u16(k), _u16(v), _u16(do)
        cu = np.ascontiguousarray(cu_seqlens, dtype=np.int32)
        T, Hq, D = q.shape
        Hkv = k.shape[1]
        dq = np.empty((T, Hq, D), np.float64)
        dk = np.empty((T, Hkv, D), np.float64)
        dv = np.empty((T, Hkv, D), np.float64)
        gap = ctypes.c_double(0.0)
        self._check(self.lib.oracle_attn_bwd_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(do), _ptr(cu), len(cu) - 1, Hq,
                                                    Hkv, D, scale, causal, window, _ptr(dq), _ptr(dk), _ptr(dv),
                                                    ctypes.addressof(gap), nthreads or default_threads()),
                    "bwd_varlen")
        return dq, dk, dv, gap.value

    # ---- sampled rows (dense when cu_seqlens is None, else packed) ---------------------
    def _rows_args(self, q, cu_seqlens):
        if cu_seqlens is None:
            B, S = q.shape[0], q.shape[1]
            return None, B, S, q.shape[2], q.shape[3]
        cu = np.ascontiguousarray(cu_seqlens, dtype=np.int32)
        return cu, len(cu) - 1, 0, q.shape[1], q.shape[2]

    def fwd_rows(self, q, k, v, rows, scale, causal=1, window=0, cu_seqlens=None, nthreads=None):
        """rows: int64 [n, 3] of (sequence, query head, query index)."""
        q, k, v = _u16(q), _u16(k), _u16(v)
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        cu, nb, S, Hq, D = self._rows_args(q, cu_seqlens)
        Hkv = k.shape[-2]
        o = np.empty((len(rows), D), np.float64)
        lse = np.empty(len(rows), np.float64)
        self._check(self.lib.oracle_attn_fwd_rows(_ptr(q), _ptr(k), _ptr(v), _ptr(cu), nb, S, Hq, Hkv, D, scale,
                                                  causal, window, _ptr(rows), len(rows), _ptr(o), _ptr(lse),
                                                  nthreads or default_threads()), "fwd_rows")
        return o, lse

    def dq_rows(self, q, k, v, do, rows, scale, causal=1, window=0, cu_seqlens=None, nthreads=None):
        q, k, v, do = _u16(q), _u16(k), _u16(v), _u16(do)
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        cu, nb, S, Hq, D = self._rows_args(q, cu_seqlens)
        Hkv = k.shape[-2]
        dq = np.empty((len(rows), D), np.float64)
        self._check(self.lib.oracle_attn_dq_rows(_ptr(q), _ptr(k), _ptr(v), _ptr(do), _ptr(cu), nb, S, Hq, Hkv, D,
                                                 scale, causal, window, _ptr(rows), len(rows), _ptr(dq),
                                                 nthreads or default_threads()), "dq_rows")
        return dq

    def dkv_rows(self, q, k, v, do, rows, scale, causal=1, window=0, cu_seqlens=None, nthreads=None):
        """rows: int64 [n, 3] of (sequence, kv head, key index)."""
        q, k, v, do = _u16(q), _u16(k), _u16(v), _u16(do)
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        cu, nb, S, Hq, D = self._rows_args(q, cu_seqlens)
        Hkv = k.shape[-2]
        dk = np.empty((len(rows), D), np.float64)
        dv = np.empty((len(rows), D), np.float64)
        self._check(self.lib.oracle_attn_dkv_rows(_ptr(q), _ptr(k), _ptr(v), _ptr(do), _ptr(cu), nb, S, Hq, Hkv, D,
                                                  scale, causal, window, _ptr(rows), len(rows), _ptr(dk), _ptr(dv),
                                                  nthreads or default_threads()), "dkv_rows")
        return dk, dv

    # ---- paged decode ---------------------------------------------------------------------
    def decode_paged(self, q, k_cache, v_cache, block_table, seq_lens, scale, window=0, nthreads=None):
        q, kc, vc = _u16(q), _u16(k_cache), _u16(v_cache)
        bt = np.ascontiguousarray(block_table, dtype=np.int32)
        sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
        B, Hq, D = q.shape
        num_pages, ps, Hkv, _ = kc.shape
        o = np.empty((B, Hq, D), np.float64)
        lse = np.empty((B, Hq), np.float64)
        self._check(self.lib.oracle_attn_decode_paged(_ptr(q), _ptr(kc), _ptr(vc), _ptr(bt), _ptr(sl), B, Hq, Hkv, D,
                                                      ps, bt.shape[1], num_pages, scale, window, _ptr(o), _ptr(lse),
                                                      nthreads or default_threads()), "decode_paged")
        return o, lse


    def prefill_paged(self, q, k_cache, v_cache, block_table, seq_lens, cu_q, scale, window=0, nthreads=None):
        """New queries q [T, Hq, D] (request b: rows cu_q[b]..cu_q[b+1]-1, the last n_b of its
        seq_lens[b] cached tokens) over the paged cache -> o [T, Hq, D], lse [Hq, T]."""
        q, kc, vc = _u16(q), _u16(k_cache), _u16(v_cache)
        bt = np.ascontiguousarray(block_table, dtype=np.int32)
        sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
        cu = np.ascontiguousarray(cu_q, dtype=np.int32)
        T, Hq, D = q.shape
        num_pages, ps, Hkv, _ = kc.shape
        o = np.zeros((T, Hq, D), np.float64)
        lse = np.full((Hq, T), -np.inf, np.float64)
        self._check(self.lib.oracle_attn_prefill_paged(_ptr(q), _ptr(kc), _ptr(vc), _ptr(bt), _ptr(sl), _ptr(cu),
                                                       len(sl), Hq, Hkv, D, ps, bt.shape[1], num_pages, scale, window,
                                                       _ptr(o), _ptr(lse), nthreads or default_threads()),
                    "prefill_paged")
        return o, lse


    def merge_lse(self, o_parts, lse_parts):
        """Combine attention results over disjoint key sets. o_parts [P, B, S, H, D] (or
        [P, T, H, D]) as bf16 bit patterns (uint16/int16) or floats; lse_parts [P, B, H, S]
        (or [P, H, T]). Returns o [B, S, H, D] (or [T, H, D]) and lse [B, H, S] (or [H, T])."""
        o_parts = np.asarray(o_parts)
        if o_parts.dtype in (np.uint16, np.int16):
            o_parts = (o_parts.astype(np.uint16).astype(np.uint32) << 16).view(np.float32)
        packed = o_parts.ndim == 4
        if packed:
            o_parts = o_parts[:, None]
            lse_parts = np.asarray(lse_parts)[:, None]
        o_parts = np.ascontiguousarray(o_parts, dtype=np.float64)
        lse_parts = np.ascontiguousarray(lse_parts, dtype=np.float64)
        P, B, S, H, D = o_parts.shape
        if lse_parts.shape != (P, B, H, S):
            raise ValueError("lse_parts shape does not match o_parts")
        o = np.empty((B, S, H, D), np.float64)
        lse = np.empty((B, H, S), np.float64)
        self._check(self.lib.oracle_merge_lse(_ptr(o_parts), _ptr(lse_parts), P, B, S, H, D, _ptr(o), _ptr(lse)),
                    "merge_lse")
        return (o[0], lse[0]) if packed else (o, lse)


_default = None


def get() -> Oracle:
    """The oracle as built from source (no planted mistake)."""
    global _default
    with _lock:
        if _default is None:
            _default = Oracle()
    return _default
