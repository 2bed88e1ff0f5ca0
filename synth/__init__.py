"""Seeded synthetic inputs for the attention workloads.

This package draws numbers and lays them out in the shapes of the workloads; it
computes nothing about attention. Both the fp64 oracle and the CUDA path are fed
from here, so they see the same bf16 bits.

Recipe (all draws counter based, see ``synth.c``):

* dense / sliding-window / tiny: q, k, v, dO ~ N(0, 1) rounded to bf16 (RNE),
  streams 1, 2, 3, 4 of the seed. The sliding-window workload additionally
  scales 1 % of the entries of q and of k (independent Bernoulli draws) by 30
  before rounding.
* varlen: sequence lengths uniform integers in [512, 4096] (stream 10), packed
  back to back; ``cu_seqlens`` is their int32 prefix sum starting at 0.
* paged decode: context lengths uniform integers in [256, 1024] (stream 11);
  a Fisher-Yates permutation of the 4096 pool pages (stream 12) is dealt in
  order to the requests, ``ceil(L / 16)`` pages each; unused block-table entries
  are -1. The whole pool and q are N(0, 1) bf16 (streams 13, 14, 1).
* sliding-window decode, head_dim 256: contexts uniform integers in [1024, 4096] (stream 11),
  the pool sized to the requests' pages plus 64 and dealt as for paged decode.
* chunked prefill over a paged cache: as paged decode, with each request's last
  q_len tokens new (q packed by ``cu_q``, stream 1).
* merge of results over disjoint key sets: part outputs N(0, 1) bf16 (stream 15);
  part lse = 8 + 2 * (a bf16 N(0, 1) draw, stream 16), exact in fp32; optionally a
  percentage of (part, row) entries empty (lse = -inf) by uniform draws (stream 17).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB = os.path.join(_HERE, "libsynth.so")
_lock = threading.Lock()
_lib = None

STREAM_Q, STREAM_K, STREAM_V, STREAM_DO = 1, 2, 3, 4
STREAM_SEQLENS, STREAM_CTX, STREAM_PERM, STREAM_KCACHE, STREAM_VCACHE = 10, 11, 12, 13, 14
STREAM_OPARTS, STREAM_LSEPARTS, STREAM_EMPTY = 15, 16, 17


def build(force: bool = False) -> str:
    """Compile ``libsynth.so`` next to its source (gcc, no extra flags that differ by host)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm", "-lpthread"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            lib.synth_normal_bf16.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64, ctypes.c_double,
                                              ctypes.c_double, ctypes.c_void_p, ctypes.c_int]
            lib.synth_uniform_int.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64, ctypes.c_int64,
                                              ctypes.c_int64, ctypes.c_void_p]
            lib.synth_permutation.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_int64, ctypes.c_void_p]
            lib.synth_mix64.argtypes = [ctypes.c_uint64]
            lib.synth_mix64.restype = ctypes.c_uint64
            lib.synth_unit.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64]
            lib.synth_unit.restype = ctypes.c_double
            _lib = lib
    return _lib


def _threads() -> int:
    return max(1, min(64, os.cpu_count() or 1))


def normal_bf16(seed: int, stream: int, shape, outlier_frac: float = 0.0, outlier_scale: float = 1.0) -> np.ndarray:
    """bf16 bit patterns (uint16) of N(0,1) draws, optionally with sparse scaled outliers."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16)
    _load().synth_normal_bf16(seed, stream, n, float(outlier_frac), float(outlier_scale),
                              out.ctypes.data, _threads())
    return out.reshape(shape)


def uniform_int(seed: int, stream: int, n: int, lo: int, hi: int) -> np.ndarray:
    out = np.empty(n, dtype=np.int64)
    if _load().synth_uniform_int(seed, stream, n, lo, hi, out.ctypes.data) != 0:
        raise ValueError("hi < lo")
    return out


def permutation(seed: int, stream: int, n: int) -> np.ndarray:
    out = np.empty(n, dtype=np.int64)
    _load().synth_permutation(seed, stream, n, out.ctypes.data)
    return out


def mix64(z: int) -> int:
    return int(_load().synth_mix64(z))


def unit(seed: int, stream: int, i: int) -> float:
    return float(_load().synth_unit(seed, stream, i))


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32."""
    return (bits.astype(np.uint32) << 16).view(np.float32)


def f32_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 bit patterns (round to nearest even; inputs finite)."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    b = b + 0x7FFF + ((b >> 16) & 1)
    return (b >> 16).astype(np.uint16)


# --------------------------------------------------------------------------------------
# Workloads
# --------------------------------------------------------------------------------------

@dataclass
class Dense:
    """Dense (or sliding-window) causal prefill problem in [B, S, H, D] layout."""
    name: str
    B: int
    Hq: int
    Hkv: int
    S: int
    D: int
    window: int
    scale: float
    q: np.ndarray = field(repr=False)
    k: np.ndarray = field(repr=False)
    v: np.ndarray = field(repr=False)
    do: np.ndarray = field(repr=False)
    causal: int = 1


@dataclass
class Varlen:
    """Packed variable-length causal prefill problem in [T, H, D] layout."""
    name: str
    seqlens: np.ndarray
    cu_seqlens: np.ndarray
    Hq: int
    Hkv: int
    D: int
    window: int
    scale: float
    q: np.ndarray = field(repr=False)
    k: np.ndarray = field(repr=False)
    v: np.ndarray = field(repr=False)
    do: np.ndarray = field(repr=False)
    causal: int = 1

    @property
    def total_tokens(self) -> int:
        return int(self.cu_seqlens[-1])

    @property
    def max_seqlen(self) -> int:
        return int(self.seqlens.max()) if len(self.seqlens) else 0


@dataclass
class Paged:
    """Single-token decode over a paged KV cache."""
    name: str
    B: int
    Hq: int
    Hkv: int
    D: int
    page_size: int
    num_pages: int
    max_pages: int
    scale: float
    seq_lens: np.ndarray
    block_table: np.ndarray = field(repr=False)
    q: np.ndarray = field(repr=False)
    k_cache: np.ndarray = field(repr=False)
    v_cache: np.ndarray = field(repr=False)
    window: int = 0  # > 0: the query sees only the last `window` keys


def dense(B, Hq, Hkv, S, D, window=0, seed=0, outlier_frac=0.0, outlier_scale=1.0, scale=None,
          name="dense", with_do=True) -> Dense:
    q = normal_bf16(seed, STREAM_Q, (B, S, Hq, D), outlier_frac, outlier_scale)
    k = normal_bf16(seed, STREAM_K, (B, S, Hkv, D), outlier_frac, outlier_scale)
    v = normal_bf16(seed, STREAM_V, (B, S, Hkv, D))
    do = normal_bf16(seed, STREAM_DO, (B, S, Hq, D)) if with_do else None
    return Dense(name, B, Hq, Hkv, S, D, window, float(scale if scale is not None else D ** -0.5), q, k, v, do)


def varlen_from_lengths(seqlens, Hq, Hkv, D, window=0, seed=0, scale=None, name="varlen", with_do=True) -> Varlen:
    seqlens = np.asarray(seqlens, dtype=np.int64)
    cu = np.zeros(len(seqlens) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(seqlens)
    T = int(cu[-1])
    q = normal_bf16(seed, STREAM_Q, (T, Hq, D))
    k = normal_bf16(seed, STREAM_K, (T, Hkv, D))
    v = normal_bf16(seed, STREAM_V, (T, Hkv, D))
    do = normal_bf16(seed, STREAM_DO, (T, Hq, D)) if with_do else None
    return Varlen(name, seqlens.astype(np.int32), cu, Hq, Hkv, D, window,
                  float(scale if scale is not None else D ** -0.5), q, k, v, do)


def varlen(num_seqs, lo, hi, Hq, Hkv, D, window=0, seed=0, name="varlen", with_do=True) -> Varlen:
    lens = uniform_int(seed, STREAM_SEQLENS, num_seqs, lo, hi)
    return varlen_from_lengths(lens, Hq, Hkv, D, window, seed, name=name, with_do=with_do)


def paged_from_lengths(seq_lens, Hq, Hkv, D, page_size=16, num_pages=4096, seed=0, scale=None,
                       max_pages=None, name="paged", window=0) -> Paged:
    seq_lens = np.asarray(seq_lens, dtype=np.int64)
    B = len(seq_lens)
    need = (seq_lens + page_size - 1) // page_size
    if max_pages is None:
        max_pages = int(max(1, need.max() if B else 1))
    if need.sum() > num_pages or (B and need.max() > max_pages):
        raise ValueError("page pool too small for the requested lengths")
    perm = permutation(seed, STREAM_PERM, num_pages)
    bt = np.full((B, max_pages), -1, dtype=np.int32)
    pos = 0
    for b in range(B):
        n = int(need[b])
        bt[b, :n] = perm[pos:pos + n]
        pos += n
    q = normal_bf16(seed, STREAM_Q, (B, Hq, D))
    kc = normal_bf16(seed, STREAM_KCACHE, (num_pages, page_size, Hkv, D))
    vc = normal_bf16(seed, STREAM_VCACHE, (num_pages, page_size, Hkv, D))
    return Paged(name, B, Hq, Hkv, D, page_size, num_pages, max_pages,
                 float(scale if scale is not None else D ** -0.5), seq_lens.astype(np.int32), bt, q, kc, vc,
                 int(window))


@dataclass
class PagedPrefill:
    """Chunked prefill over a paged KV cache: request b has seq_lens[b] cached tokens, the last
    q_lens[b] of which are new queries (packed rows cu_q[b] .. cu_q[b+1]-1 of q)."""
    name: str
    Hq: int
    Hkv: int
    D: int
    page_size: int
    num_pages: int
    max_pages: int
    window: int
    scale: float
    seq_lens: np.ndarray
    q_lens: np.ndarray
    cu_q: np.ndarray
    block_table: np.ndarray = field(repr=False)
    q: np.ndarray = field(repr=False)
    k_cache: np.ndarray = field(repr=False)
    v_cache: np.ndarray = field(repr=False)

    @property
    def B(self) -> int:
        return len(self.seq_lens)

    @property
    def total_q(self) -> int:
        return int(self.cu_q[-1])

    @property
    def max_q(self) -> int:
        return int(self.q_lens.max()) if len(self.q_lens) else 0


def prefill_paged_from_lengths(seq_lens, q_lens, Hq, Hkv, D, page_size=16, num_pages=None, window=0, seed=0,
                               scale=None, max_pages=None, name="prefill_paged") -> PagedPrefill:
    seq_lens = np.asarray(seq_lens, dtype=np.int64)
    q_lens = np.asarray(q_lens, dtype=np.int64)
    if np.any(q_lens > seq_lens) or np.any(q_lens < 0):
        raise ValueError("each request needs 0 <= q_len <= seq_len")
    need = (seq_lens + page_size - 1) // page_size
    if num_pages is None:
        num_pages = int(max(1, need.sum()) + 8)
    base = paged_from_lengths(seq_lens, Hq, Hkv, D, page_size, num_pages, seed, scale, max_pages, name)
    cu_q = np.zeros(len(q_lens) + 1, dtype=np.int32)
    cu_q[1:] = np.cumsum(q_lens)
    q = normal_bf16(seed, STREAM_Q, (int(cu_q[-1]), Hq, D))
    return PagedPrefill(name, Hq, Hkv, D, page_size, num_pages, base.max_pages, int(window), base.scale,
                        seq_lens.astype(np.int32), q_lens.astype(np.int32), cu_q, base.block_table, q, base.k_cache,
                        base.v_cache)


def paged(B, lo, hi, Hq, Hkv, D, page_size=16, num_pages=4096, seed=0, max_pages=None, name="paged") -> Paged:
    lens = uniform_int(seed, STREAM_CTX, B, lo, hi)
    if max_pages is None:
        max_pages = (hi + page_size - 1) // page_size
    return paged_from_lengths(lens, Hq, Hkv, D, page_size, num_pages, seed, max_pages=max_pages, name=name)


@dataclass
class MergeParts:
    """Results over P disjoint key sets in the forward's layouts: o_parts [P, B, S, H, D] bf16
    bits, lse_parts [P, B, H, S] fp32 (-inf = no key in that part for that row)."""
    name: str
    P: int
    B: int
    S: int
    H: int
    D: int
    o_parts: np.ndarray = field(repr=False)
    lse_parts: np.ndarray = field(repr=False)


def merge_parts(P, B, S, H, D, seed=0, empty_pct=0, name="merge_parts") -> MergeParts:
    o = normal_bf16(seed, STREAM_OPARTS, (P, B, S, H, D))
    lb = normal_bf16(seed, STREAM_LSEPARTS, (P, B, H, S))
    lse = (lb.astype(np.uint32) << 16).view(np.float32) * np.float32(2.0) + np.float32(8.0)
    if empty_pct:
        draw = uniform_int(seed, STREAM_EMPTY, P * B * H * S, 0, 99).reshape(P, B, H, S)
        lse[draw < empty_pct] = -np.inf
    return MergeParts(name, P, B, S, H, D, o, lse.astype(np.float32))


# The five workloads, named by what they are.
def tiny_d512_causal(seed=0) -> Dense:
    return dense(1, 2, 1, 128, 512, 0, seed, name="tiny_d512_causal")


def dense_d512_causal(seed=0, with_do=True) -> Dense:
    return dense(2, 32, 4, 4096, 512, 0, seed, name="dense_d512_causal", with_do=with_do)


def swa_d256_w1024(seed=0, with_do=True) -> Dense:
    return dense(2, 32, 16, 8192, 256, 1024, seed, outlier_frac=0.01, outlier_scale=30.0,
                 name="swa_d256_w1024", with_do=with_do)


def dense_d128_causal(seed=0, with_do=True) -> Dense:
    """Qwen3-class heads (head_dim 128, 32 query heads over 8 KV heads) at the dense workload's
    batch and length."""
    return dense(2, 32, 8, 4096, 128, 0, seed, name="dense_d128_causal", with_do=with_do)


def dense_d64_causal(seed=0, with_do=True) -> Dense:
    return dense(2, 32, 8, 4096, 64, 0, seed, name="dense_d64_causal", with_do=with_do)


def varlen_d512_causal(seed=0, with_do=True) -> Varlen:
    return varlen(8, 512, 4096, 32, 4, 512, 0, seed, name="varlen_d512_causal", with_do=with_do)


def prefill_paged_d512(seed=0) -> PagedPrefill:
    """Chunked prefill of 512 new tokens per request over a paged cache: 8 requests with
    contexts uniform in [1024, 4096] (the varlen workload's length law), head_dim 512, GQA 8:1."""
    ctx = uniform_int(seed, STREAM_CTX, 8, 1024, 4096)
    return prefill_paged_from_lengths(ctx, np.full(8, 512), 32, 4, 512, page_size=16, seed=seed,
                                      name="prefill_paged_d512")


def merge_cp8_d512(seed=0) -> MergeParts:
    """The combining step of an 8-way context-parallel ring over a 16k-token sequence, seen from
    one rank: its 2048 query tokens' results from 8 key chunks, 32 heads of dim 512."""
    return merge_parts(8, 1, 2048, 32, 512, seed, name="merge_cp8_d512")


def decode_paged_swa_d256(seed=0) -> Paged:
    """Sliding-window decode at head_dim 256 (the window workload's heads and window: Hq 32,
    Hkv 16, W 1024) for 64 requests with contexts uniform in [1024, 4096], so the window binds."""
    lens = uniform_int(seed, STREAM_CTX, 64, 1024, 4096)
    need = int(((lens + 15) // 16).sum())
    return paged_from_lengths(lens, 32, 16, 256, 16, need + 64, seed, max_pages=256, name="decode_paged_swa_d256",
                              window=1024)


def decode_paged_d128(seed=0) -> Paged:
    return paged(64, 256, 1024, 32, 8, 128, 16, 4096, seed, max_pages=64, name="decode_paged_d128")
