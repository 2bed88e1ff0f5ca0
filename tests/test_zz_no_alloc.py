"""The allocation-free decode entry point (attn_decode_paged_noalloc) against the
regular one (attn_decode_paged with a caller workspace).

Callers that cannot allocate device memory on their decode path (a plug-in whose host
application owns the device-memory budget, a latency-critical loop that must not pay
cudaMalloc's implicit synchronisation) use the variant whose scratch is a buffer built
into the library. It must give the same results as the workspace path, including on a
second call that finds the previous call's leftovers in the shared buffer.

This file is collected last so a stop-at-first-failure run has already run every other
test; it also passes on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import attention_flash_gqa_gb300 as attn
import synth
from gpu_util import check, check_lse, to_dev, to_np


@pytest.fixture(scope="module")
def lib():
    from attention_flash_gqa_gb300 import _build

    _build.build()
    return attn.load_library()


def _device_case(pp):
    q, kc, vc = to_dev(pp.q), to_dev(pp.k_cache), to_dev(pp.v_cache)
    bt = torch.from_numpy(pp.block_table).cuda()
    sl = torch.from_numpy(pp.seq_lens).cuda()
    return q, kc, vc, bt, sl


_CASES = [
    # (problem, window): the benchmarked head_dim 128 decode, a ragged batch with empty and one-page
    # requests, and a windowed head_dim 256 batch (KV heads in blocks, contexts past the window)
    (lambda: synth.decode_paged_d128(seed=3), 0),
    (lambda: synth.paged_from_lengths([5, 1024, 0, 17, 300, 640], 32, 8, 128, page_size=16, num_pages=512,
                                      seed=4, max_pages=64), 0),
    (lambda: synth.paged_from_lengths([300, 17, 1024, 2000, 1500], 32, 16, 256, page_size=16, num_pages=512,
                                      seed=5, max_pages=128), 1024),
]


@pytest.mark.gpu
def test_noalloc_matches_workspace_path_on_two_calls(lib):
    """Both entry points run the same kernels on the same inputs, so their results must be the
    same bits; each case makes two calls in a row on the shared buffer (the second finds the
    first call's leftovers, and the cases change the batch and head size between calls)."""
    torch.cuda.set_device(0)
    for make, window in _CASES:
        pp = make()
        q, kc, vc, bt, sl = _device_case(pp)
        ref_o, ref_lse = attn.attn_decode_paged(q, kc, vc, bt, sl, scale=pp.scale, window=window)
        for _ in range(2):
            o = torch.full_like(q, 5.0)
            lse = torch.full((pp.B, pp.Hq), 5.0, dtype=torch.float32, device="cuda")
            attn.attn_decode_paged_noalloc(q, kc, vc, bt, sl, o, lse, scale=pp.scale, window=window)
            torch.cuda.synchronize()
            assert attn.attn_get_device_status() == 0
            assert torch.equal(o.view(torch.int16), ref_o.view(torch.int16))
            assert torch.equal(lse, ref_lse)
            # and so within the tolerance of every parity test
            check("o", to_np(o), to_np(ref_o))
            check_lse("lse", to_np(lse), to_np(ref_lse))


def test_noalloc_rejects_problems_beyond_the_buffer(lib):
    """Needs no GPU: the size check comes before anything touches the device."""
    cap = lib.attn_decode_paged_noalloc_max_bytes()
    assert cap == 16 << 20
    fake = ctypes.c_void_p(1 << 20)
    args = [fake] * 7

    def call(B, Hq):
        return lib.attn_decode_paged_noalloc(*args, B, Hq, 8, 128, 16, 64, 4096, 0.088, 0, None)

    assert attn.attn_workspace_size(attn.ATTN_OP_DECODE_PAGED, 481, 32, 8, 0, 128) > cap
    assert call(481, 32) == 4  # ATTN_ERR_WORKSPACE
    assert call(4096, 64) == 4
    assert call(-1, 32) == 1  # ATTN_ERR_INVALID_ARG


def test_noalloc_rejects_unsupported_head_sizes_without_sizing_them(lib):
    """Needs no GPU: a head size no decode kernel takes is rejected as unsupported (and the
    workspace size of such a problem is 0) instead of reaching the size arithmetic."""
    fake = ctypes.c_void_p(1 << 20)
    args = [fake] * 7
    for D in (2048, 64, 100):
        assert attn.attn_workspace_size(attn.ATTN_OP_DECODE_PAGED, 8, 32, 8, 0, D) == 0
        assert lib.attn_decode_paged_noalloc(*args, 8, 32, 8, D, 16, 64, 4096, 0.088, 0, None) == 2
    assert attn.attn_workspace_size(attn.ATTN_OP_DECODE_PAGED, 8, 32, 6, 0, 128) == 0  # 32 % 6 != 0
    assert lib.attn_decode_paged_noalloc(*args, 8, 32, 6, 128, 16, 64, 4096, 0.088, 0, None) == 1
