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


@pytest.mark.gpu
def test_noalloc_matches_workspace_path_on_two_calls(lib):
    torch.cuda.set_device(0)
    cases = [synth.decode_paged_d128(seed=3),
             synth.paged_from_lengths([5, 1024, 0, 17, 300, 640], 32, 8, 128, page_size=16, num_pages=512,
                                      seed=4, max_pages=64)]
    for pp in cases:  # two calls in a row on the shared buffer, different batches
        q, kc, vc, bt, sl = _device_case(pp)
        ref_o, ref_lse = attn.attn_decode_paged(q, kc, vc, bt, sl, scale=pp.scale)
        o = torch.empty_like(q)
        lse = torch.empty((pp.B, pp.Hq), dtype=torch.float32, device="cuda")
        attn.attn_decode_paged_noalloc(q, kc, vc, bt, sl, o, lse, scale=pp.scale)
        torch.cuda.synchronize()
        assert attn.attn_get_device_status() == 0
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
