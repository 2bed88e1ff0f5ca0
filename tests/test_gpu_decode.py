"""Paged decode beyond the head_dim 128 workload: sliding windows, head_dim 256, KV heads split
into blocks, against the fp64 oracle; and the sliding-window head_dim 256 workload at full size."""
import numpy as np
import pytest
import torch

import attention_flash_gqa_gb300 as attn
import synth
from gpu_util import check, check_lse, to_dev, to_np

pytestmark = pytest.mark.gpu

LENS = [1, 15, 16, 17, 33, 256, 1024, 0, 700, 5, 2049]


@pytest.fixture(scope="module", autouse=True)
def _built():
    from attention_flash_gqa_gb300 import _build

    _build.build()
    attn.load_library()
    torch.cuda.set_device(0)


def run(pp, window=None):
    q, kc, vc = to_dev(pp.q), to_dev(pp.k_cache), to_dev(pp.v_cache)
    bt = torch.from_numpy(pp.block_table).cuda()
    sl = torch.from_numpy(pp.seq_lens).cuda()
    o, lse = attn.attn_decode_paged(q, kc, vc, bt, sl, scale=pp.scale, window=pp.window if window is None else window)
    torch.cuda.synchronize()
    assert attn.attn_get_device_status() == 0
    return to_np(o), to_np(lse)


def compare(orc, pp, window):
    o, lse = run(pp, window)
    ro, rl = orc.decode_paged(pp.q, pp.k_cache, pp.v_cache, pp.block_table, pp.seq_lens, pp.scale, window)
    check("o", o, ro)
    check_lse("lse", lse, rl)
    empty = [i for i, L in enumerate(pp.seq_lens) if L == 0]
    for i in empty:
        assert np.all(o[i] == 0) and np.all(np.isneginf(lse[i]))


@pytest.mark.parametrize("window", [1, 15, 16, 17, 100, 1024, 5000])
def test_decode_window_d128(orc, window):
    pp = synth.paged_from_lengths(LENS, 32, 8, 128, page_size=16, num_pages=512, seed=window, max_pages=160)
    compare(orc, pp, window)


@pytest.mark.parametrize("Hq,Hkv", [(32, 16), (16, 4), (4, 4), (8, 2), (2, 2), (24, 6)])
@pytest.mark.parametrize("window", [0, 1, 40, 1024])
def test_decode_d256(orc, Hq, Hkv, window):
    pp = synth.paged_from_lengths(LENS, Hq, Hkv, 256, page_size=16, num_pages=512, seed=Hq * 7 + Hkv + window,
                                  max_pages=160)
    compare(orc, pp, window)


@pytest.mark.parametrize("Hq,Hkv", [(64, 8), (128, 16), (16, 16)])
def test_decode_d128_head_blocks(orc, Hq, Hkv):
    """More KV heads than one unit holds: the heads are served in blocks by the grid's y."""
    pp = synth.paged_from_lengths(LENS, Hq, Hkv, 128, page_size=16, num_pages=512, seed=Hq + Hkv, max_pages=160)
    compare(orc, pp, 0)
    compare(orc, pp, 300)


@pytest.mark.parametrize("Hq,Hkv,D", [(8, 4, 256), (32, 8, 128), (8, 4, 128), (4, 4, 128), (16, 2, 128)])
@pytest.mark.parametrize("W", [37, 0])
def test_decode_window_unused_tokens_are_never_read(orc, Hq, Hkv, D, W):
    """Tokens before the window and slots past the end hold NaN: neither reaches the result. At
    head_dim 128 with groups up to 4 the page's products are matrix instructions over whole
    pages, so the NaN rows sit inside the operands and must be masked, not skipped."""
    pp = synth.paged_from_lengths([40, 100, 17, 16, 1], Hq, Hkv, D, page_size=16, num_pages=24, seed=5 + D + Hq,
                                  max_pages=7)
    kc, vc = pp.k_cache.copy(), pp.v_cache.copy()
    for b, L in enumerate(pp.seq_lens):
        before = list(range(0, max(0, L - W))) if W > 0 else []
        for t in before + list(range(L, ((L + 15) // 16) * 16)):
            page = pp.block_table[b, t // 16]
            kc[page, t % 16] = 0x7FC0
            vc[page, t % 16] = 0x7FC0
    bad = synth.Paged(**{**pp.__dict__, "k_cache": kc, "v_cache": vc})
    o, lse = run(bad, W)
    ro, rl = orc.decode_paged(pp.q, pp.k_cache, pp.v_cache, pp.block_table, pp.seq_lens, pp.scale, W)
    check("o", o, ro)
    check_lse("lse", lse, rl)


def test_decode_noalloc_window_d256(orc):
    pp = synth.paged_from_lengths([300, 17, 1024], 32, 16, 256, page_size=16, num_pages=128, seed=8, max_pages=64)
    q, kc, vc = to_dev(pp.q), to_dev(pp.k_cache), to_dev(pp.v_cache)
    bt = torch.from_numpy(pp.block_table).cuda()
    sl = torch.from_numpy(pp.seq_lens).cuda()
    o = torch.empty_like(q)
    lse = torch.empty((pp.B, pp.Hq), dtype=torch.float32, device="cuda")
    attn.attn_decode_paged_noalloc(q, kc, vc, bt, sl, o, lse, scale=pp.scale, window=100)
    torch.cuda.synchronize()
    assert attn.attn_get_device_status() == 0
    ro, rl = orc.decode_paged(pp.q, pp.k_cache, pp.v_cache, pp.block_table, pp.seq_lens, pp.scale, 100)
    check("o", to_np(o), ro)
    check_lse("lse", to_np(lse), rl)


def test_decode_swa_d256_full_workload(orc):
    """The benchmarked sliding-window workload (64 requests, contexts U[1024, 4096], Hq 32, Hkv 16,
    D 256, W 1024) in the benchmark's launch, every output against the oracle."""
    pp = synth.decode_paged_swa_d256(seed=0)
    o, lse = run(pp)
    ro, rl = orc.decode_paged(pp.q, pp.k_cache, pp.v_cache, pp.block_table, pp.seq_lens, pp.scale, pp.window)
    check("o", o, ro)
    check_lse("lse", lse, rl)


def test_decode_all_requests_empty():
    """No request has a cached token: the decode grid does nothing and the merge writes o = 0,
    lse = -inf for every (request, head)."""
    pp = synth.paged_from_lengths([0, 0, 0], 32, 8, 128, page_size=16, num_pages=16, seed=1, max_pages=4)
    o, lse = run(pp)
    assert np.all(o == 0) and np.all(np.isneginf(lse))


@pytest.mark.parametrize("lens", [[152 * 16 * 3 + 5], [152 * 16 * 2, 3]])
def test_decode_one_request_over_every_cta(orc, lens):
    """A request longer than the grid has CTAs: every CTA holds a piece of it, so the merge
    folds more than a hundred partial slots in several rounds."""
    pp = synth.paged_from_lengths(lens, 32, 8, 128, page_size=16, num_pages=1024, seed=len(lens), max_pages=512)
    compare(orc, pp, 0)


@pytest.mark.parametrize("direction", ["rising", "falling"])
def test_decode_scores_drifting_along_the_context(orc, direction):
    """Keys scaled by a factor that grows (or shrinks) along the context, so a page's scores keep
    exceeding the running maximum by far more than the lazy-update threshold (or never do)."""
    pp = synth.paged_from_lengths([1500, 700, 40], 32, 8, 128, page_size=16, num_pages=256, seed=9, max_pages=128)
    kc = pp.k_cache.view(np.uint16).copy()
    kf = (kc.astype(np.uint32) << 16).view(np.float32)
    for b, L in enumerate(pp.seq_lens):
        for p in range((int(L) + 15) // 16):
            pos = p * 16 + np.arange(16)
            f = 1.0 + pos / 60.0 if direction == "rising" else 1.0 + (int(L) - pos) / 60.0
            page = pp.block_table[b, p]
            kf[page] *= f[:, None, None].astype(np.float32)
    k_new = (kf.view(np.uint32) + 0x8000 >> 16).astype(np.uint16)  # round to bf16
    pp = synth.Paged(**{**pp.__dict__, "k_cache": k_new.view(pp.k_cache.dtype)})
    compare(orc, pp, 0)


def test_decode_max_batch_tiny_contexts(orc):
    """The largest batch the call accepts (4096 requests), contexts of 0 to 33 tokens: every CTA's
    range spans many requests, most of them in one page, some empty."""
    lens = [int(x) for x in np.random.default_rng(4096).choice([0, 1, 2, 5, 15, 16, 17, 33], 4096)]
    pp = synth.paged_from_lengths(lens, 8, 2, 128, page_size=16, num_pages=8192, seed=40, max_pages=3)
    compare(orc, pp, 0)


@pytest.mark.parametrize("window", [1, 17, 300])
def test_decode_window_head_blocks_group8(orc, window):
    """A GQA group of 8 at head_dim 128 (KV heads in blocks of 4) with a sliding window."""
    pp = synth.paged_from_lengths(LENS, 64, 8, 128, page_size=16, num_pages=512, seed=window, max_pages=160)
    compare(orc, pp, window)


def test_decode_back_to_back_with_q_rewritten_between(orc):
    """Three decode calls on one stream sharing one workspace, with an ordinary kernel (a torch
    copy) rewriting q before each call. Each decode grid may launch while the previous call's
    merge still runs, so it must wait for that merge before it reads q or writes the partials the
    merge still reads. Every output matches the oracle for the q it was given."""
    pps = [synth.paged_from_lengths([900, 1, 0, 513, 40, 2048, 77, 16], 32, 8, 128, num_pages=640, seed=s,
                                    max_pages=130) for s in (11, 12, 13)]
    base = pps[0]
    kc, vc = to_dev(base.k_cache), to_dev(base.v_cache)
    bt, sl = torch.from_numpy(base.block_table).cuda(), torch.from_numpy(base.seq_lens).cuda()
    qs = [to_dev(p.q) for p in pps]
    q = torch.empty_like(qs[0])
    ws = torch.empty(attn.attn_workspace_size(attn.ATTN_OP_DECODE_PAGED, base.B, base.Hq, base.Hkv, 0, base.D),
                     dtype=torch.uint8, device="cuda")
    outs = []
    for i in range(3):
        q.copy_(qs[i])  # an ordinary kernel on the same stream, just before the call
        o, lse = attn.attn_decode_paged(q, kc, vc, bt, sl, scale=base.scale, workspace=ws)
        outs.append((o, lse))
    torch.cuda.synchronize()
    assert attn.attn_get_device_status() == 0
    for p, (o, lse) in zip(pps, outs):
        ro, rl = orc.decode_paged(p.q, base.k_cache, base.v_cache, base.block_table, base.seq_lens, base.scale)
        check("o", to_np(o), ro)
        check_lse("lse", to_np(lse), rl)


@pytest.mark.parametrize("fill", [0x00, 0xFF])
def test_decode_long_contexts_over_repeated_calls(orc, fill):
    """Sixteen requests with long and ragged contexts (several pages per CTA), three calls in a row
    on one workspace that starts as zeros or as 0xFF bytes: every call writes all of the partials
    it reads, so whatever the workspace held before does not matter. Every call matches the
    oracle."""
    lens = [3000, 17, 2500, 1, 0, 4100, 800, 1601, 2048, 333, 3999, 64, 1200, 16, 2777, 900]
    pp = synth.paged_from_lengths(lens, 32, 8, 128, num_pages=1600, seed=21, max_pages=260)
    assert sum((L + 15) // 16 for L in lens) >= 4 * torch.cuda.get_device_properties(0).multi_processor_count
    q, kc, vc = to_dev(pp.q), to_dev(pp.k_cache), to_dev(pp.v_cache)
    bt, sl = torch.from_numpy(pp.block_table).cuda(), torch.from_numpy(pp.seq_lens).cuda()
    ws = torch.full((attn.attn_workspace_size(attn.ATTN_OP_DECODE_PAGED, pp.B, pp.Hq, pp.Hkv, 0, pp.D),), fill,
                    dtype=torch.uint8, device="cuda")
    ro, rl = orc.decode_paged(pp.q, pp.k_cache, pp.v_cache, pp.block_table, pp.seq_lens, pp.scale, 0)
    for _ in range(3):
        o, lse = attn.attn_decode_paged(q, kc, vc, bt, sl, scale=pp.scale, workspace=ws)
        torch.cuda.synchronize()
        assert attn.attn_get_device_status() == 0
        check("o", to_np(o), ro)
        check_lse("lse", to_np(lse), rl)
