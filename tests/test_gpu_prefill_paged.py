"""Chunked prefill over a paged KV cache: the CUDA path (attn_fwd_paged) against the fp64
oracle, element by element, plus the full-size workload on sampled requests and heads, the
first-prefill identity with the varlen forward, and the edge cases (empty requests, one new
token, partial last pages holding NaN, bad page ids, inconsistent requests)."""
import numpy as np
import pytest
import torch

import attention_flash_gqa_gb300 as attn
import synth
from gpu_util import check, check_lse, to_dev, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from attention_flash_gqa_gb300 import _build

    _build.build()
    attn.load_library()
    torch.cuda.set_device(0)


def _i32(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()


def run_prefill(pp, block_table=None, seq_lens=None, k_cache=None, v_cache=None, max_q=None):
    q = to_dev(pp.q)
    kc = to_dev(pp.k_cache if k_cache is None else k_cache)
    vc = to_dev(pp.v_cache if v_cache is None else v_cache)
    bt = _i32(pp.block_table if block_table is None else block_table)
    sl = _i32(pp.seq_lens if seq_lens is None else seq_lens)
    o = torch.zeros_like(q)
    lse = torch.full((pp.Hq, pp.total_q), 7.0, dtype=torch.float32, device="cuda")
    o, lse = attn.attn_fwd_paged(q, kc, vc, bt, sl, _i32(pp.cu_q), pp.max_q if max_q is None else max_q, o, lse,
                                 window=pp.window, scale=pp.scale)
    torch.cuda.synchronize()
    return to_np(o), to_np(lse)


def compare(orc, pp):
    o, lse = run_prefill(pp)
    assert attn.attn_get_device_status() == 0
    ro, rl = orc.prefill_paged(pp.q, pp.k_cache, pp.v_cache, pp.block_table, pp.seq_lens, pp.cu_q, pp.scale,
                               pp.window)
    check("o", o, ro)
    check_lse("lse", lse, rl)
    return o, lse


# contexts and new-token counts: a single token (decode), a whole first prefill, new tokens
# starting mid-page and mid-tile, an empty request, several query tiles with a ragged tail
LENS = [(1, 1), (16, 16), (17, 5), (300, 300), (1000, 128), (129, 0), (700, 257), (2049, 131)]


@pytest.mark.parametrize("D,Hq,Hkv,window", [(512, 8, 2, 0), (512, 4, 4, 0), (256, 8, 1, 0), (256, 4, 2, 100),
                                             (512, 4, 1, 1000), (256, 2, 1, 129)])
def test_prefill_paged(orc, D, Hq, Hkv, window):
    seq, nq = zip(*LENS)
    pp = synth.prefill_paged_from_lengths(seq, nq, Hq, Hkv, D, window=window, seed=D + Hq + window)
    compare(orc, pp)


def test_prefill_paged_unused_page_slots_are_never_read(orc):
    """Cache slots past each request's end in its last page, and every page no request owns,
    hold NaN: the result equals the oracle's on the clean cache."""
    seq, nq = zip(*LENS)
    pp = synth.prefill_paged_from_lengths(seq, nq, 8, 2, 512, seed=11)
    nan = np.uint16(0x7FC0)
    kc, vc = pp.k_cache.copy(), pp.v_cache.copy()
    owned = np.zeros(pp.num_pages, bool)
    for b, L in enumerate(pp.seq_lens):
        npg = (int(L) + 15) // 16
        owned[pp.block_table[b, :npg]] = True
        if L % 16:
            last = pp.block_table[b, npg - 1]
            kc[last, L % 16:] = nan
            vc[last, L % 16:] = nan
    kc[~owned] = nan
    vc[~owned] = nan
    o, lse = run_prefill(pp, k_cache=kc, v_cache=vc)
    assert attn.attn_get_device_status() == 0
    ro, rl = orc.prefill_paged(pp.q, pp.k_cache, pp.v_cache, pp.block_table, pp.seq_lens, pp.cu_q, pp.scale)
    check("o", o, ro)
    check_lse("lse", lse, rl)


def test_prefill_paged_first_prefill_equals_varlen():
    """With n_b = L_b for every request the paged forward is the varlen forward over the same
    tokens: same tiles, same products, so the same bits."""
    lens = [300, 1, 129, 1024, 77]
    pp = synth.prefill_paged_from_lengths(lens, lens, 8, 2, 512, seed=5)
    o, lse = run_prefill(pp)
    assert attn.attn_get_device_status() == 0
    # gather the caches into packed [T, Hkv, D] keys / values
    ks, vs = [], []
    for b, L in enumerate(lens):
        pages = pp.block_table[b, :(L + 15) // 16]
        ks.append(pp.k_cache[pages].reshape(-1, pp.Hkv, pp.D)[:L])
        vs.append(pp.v_cache[pages].reshape(-1, pp.Hkv, pp.D)[:L])
    k, v = to_dev(np.concatenate(ks)), to_dev(np.concatenate(vs))
    ov, lv = attn.attn_fwd_varlen(to_dev(pp.q), k, v, _i32(pp.cu_q), max(lens), scale=pp.scale)
    torch.cuda.synchronize()
    assert np.array_equal(o, to_np(ov))
    assert np.array_equal(lse, to_np(lv))


def test_prefill_paged_full_workload_sampled(orc):
    """The benchmarked workload (8 requests, contexts U[1024, 4096], 512 new tokens each,
    Hq = 32, Hkv = 4, D = 512) in the benchmark's launch; the oracle checks two requests on
    the query heads of two KV heads."""
    pp = synth.prefill_paged_d512(seed=0)
    o, lse = run_prefill(pp)
    assert attn.attn_get_device_status() == 0
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    G = pp.Hq // pp.Hkv
    for b in (0, 5):
        for g in (0, 3):
            heads = slice(g * G, (g + 1) * G)
            rows = slice(int(pp.cu_q[b]), int(pp.cu_q[b + 1]))
            sub = synth.PagedPrefill(
                pp.name, G, 1, pp.D, pp.page_size, pp.num_pages, pp.max_pages, pp.window, pp.scale,
                pp.seq_lens[b:b + 1], pp.q_lens[b:b + 1], np.array([0, pp.q_lens[b]], np.int32),
                pp.block_table[b:b + 1], np.ascontiguousarray(pp.q[rows, heads]),
                np.ascontiguousarray(pp.k_cache[:, :, g:g + 1]), np.ascontiguousarray(pp.v_cache[:, :, g:g + 1]))
            ro, rl = orc.prefill_paged(sub.q, sub.k_cache, sub.v_cache, sub.block_table, sub.seq_lens, sub.cu_q,
                                       sub.scale)
            check(f"o[req {b}, kv head {g}]", o[rows, heads], ro)
            check_lse(f"lse[req {b}, kv head {g}]", lse[heads, rows], rl)


def test_prefill_paged_no_new_tokens():
    pp = synth.prefill_paged_from_lengths([40, 0, 16], [0, 0, 0], 4, 2, 256, seed=3)
    assert pp.total_q == 0
    q = torch.empty((0, 4, 256), dtype=torch.bfloat16, device="cuda")
    o, lse = attn.attn_fwd_paged(q, to_dev(pp.k_cache), to_dev(pp.v_cache), _i32(pp.block_table),
                                 _i32(pp.seq_lens), _i32(pp.cu_q), 0)
    torch.cuda.synchronize()
    assert o.shape == (0, 4, 256) and lse.shape == (4, 0)
    assert attn.attn_get_device_status() == 0


def test_prefill_paged_bad_page_id_is_reported_not_read(orc):
    """A page id outside the pool is never dereferenced (page 0 is read instead) and the
    fault is reported; requests with valid tables are unaffected."""
    pp = synth.prefill_paged_from_lengths([200, 200], [64, 64], 4, 2, 256, seed=9)
    bt = pp.block_table.copy()
    bt[1, 3] = 1 << 30
    o, lse = run_prefill(pp, block_table=bt)
    assert attn.attn_get_device_status() == 7  # ATTN_ERR_DEVICE_BOUNDS
    ro, rl = orc.prefill_paged(pp.q, pp.k_cache, pp.v_cache, pp.block_table, pp.seq_lens, pp.cu_q, pp.scale)
    check("o[req 0]", o[:64], ro[:64])
    check_lse("lse[req 0]", lse[:, :64], rl[:, :64])
    assert np.isfinite(o[64:]).all()
    assert attn.attn_get_device_status() == 0  # cleared by the previous read


def test_prefill_paged_inconsistent_request_is_reported(orc):
    """A request with more new tokens than cached ones is skipped (its rows stay as they were)
    and reported; the other requests are computed."""
    pp = synth.prefill_paged_from_lengths([200, 100, 50], [64, 64, 20], 4, 2, 256, seed=4)
    sl = pp.seq_lens.copy()
    sl[1] = 10
    o, lse = run_prefill(pp, seq_lens=sl)
    assert attn.attn_get_device_status() == 7
    ro, rl = orc.prefill_paged(pp.q, pp.k_cache, pp.v_cache, pp.block_table, pp.seq_lens, pp.cu_q, pp.scale)
    keep = np.r_[0:64, 128:148]
    check("o[valid]", o[keep], ro[keep])
    check_lse("lse[valid]", lse[:, keep], rl[:, keep])
    assert np.all(o[64:128] == 0) and np.all(lse[:, 64:128] == 7.0)


def test_prefill_paged_rejects_bad_arguments():
    pp = synth.prefill_paged_from_lengths([40], [8], 4, 2, 256, seed=1)
    q, kc, vc = to_dev(pp.q), to_dev(pp.k_cache), to_dev(pp.v_cache)
    bt, sl, cu = _i32(pp.block_table), _i32(pp.seq_lens), _i32(pp.cu_q)
    with pytest.raises(attn.AttnError) as e:  # page_size 8 is not supported
        attn.attn_fwd_paged(q, kc.view(-1, 8, 2, 256), vc.view(-1, 8, 2, 256), bt, sl, cu, 8)
    assert e.value.status == 2
    with pytest.raises(attn.AttnError) as e:  # D = 96 is not a supported head size
        attn.attn_fwd_paged(q[..., :96].contiguous(), kc[..., :96].contiguous(), vc[..., :96].contiguous(), bt,
                            sl, cu, 8)
    assert e.value.status == 2
