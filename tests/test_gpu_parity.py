"""CUDA path vs the fp64 oracle, element by element, at sizes the oracle finishes in
seconds that still span several 128-row tiles and a ragged tail, plus edge cases."""
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


def run_dense(p, with_bwd=True):
    q, k, v = to_dev(p.q), to_dev(p.k), to_dev(p.v)
    o, lse = attn.attn_fwd(q, k, v, window=p.window, scale=p.scale)
    out = {"o": o, "lse": lse}
    if with_bwd:
        do = to_dev(p.do)
        dq, dk, dv = attn.attn_bwd(q, k, v, o, lse, do, window=p.window, scale=p.scale)
        out.update(dq=dq, dk=dk, dv=dv)
    torch.cuda.synchronize()
    assert attn.attn_get_device_status() == 0
    return {k: to_np(v) for k, v in out.items()}


def compare_dense(orc, p, with_bwd=True):
    got = run_dense(p, with_bwd)
    ro, rl = orc.fwd(p.q, p.k, p.v, p.scale, 1, p.window)
    check("o", got["o"], ro)
    check_lse("lse", got["lse"], rl)
    if with_bwd:
        rdq, rdk, rdv, *_ = orc.bwd(p.q, p.k, p.v, p.do, p.scale, 1, p.window)
        check("dq", got["dq"], rdq)
        check("dk", got["dk"], rdk)
        check("dv", got["dv"], rdv)


def test_tiny_d512_causal(orc):
    """B=1, Hq=2, Hkv=1, S=128, D=512, scale 1/sqrt(512): the smallest workload, whole."""
    compare_dense(orc, synth.tiny_d512_causal(seed=0))


@pytest.mark.parametrize("B,Hq,Hkv,S,D", [(2, 4, 2, 300, 512), (1, 2, 1, 129, 512), (1, 8, 1, 257, 512),
                                          (2, 4, 4, 300, 256), (1, 6, 2, 385, 256), (1, 2, 1, 1, 512)])
def test_dense_causal(orc, B, Hq, Hkv, S, D):
    compare_dense(orc, synth.dense(B, Hq, Hkv, S, D, 0, seed=S + D))


@pytest.mark.parametrize("window", [1, 2, 127, 128, 129, 299, 300, 600])
def test_sliding_window_edges(orc, window):
    """Window widths around the 128-key tile and the sequence length (W >= S = causal)."""
    compare_dense(orc, synth.dense(1, 2, 1, 300, 256, window, seed=window))


def test_sliding_window_outliers_finite(orc):
    """1 % of q and k entries scaled by 30 (as in the sliding-window workload): the
    backward must stay finite and match."""
    p = synth.dense(1, 4, 2, 640, 256, 256, seed=3, outlier_frac=0.01, outlier_scale=30.0)
    compare_dense(orc, p)


def test_d512_window(orc):
    compare_dense(orc, synth.dense(1, 4, 1, 400, 512, 200, seed=9))


@pytest.mark.parametrize("D,scale,window", [(512, 0.3, 0), (256, 0.02, 0), (256, 0.15, 90), (128, 0.5, 0), (64, 0.05, 40)])
def test_scale_other_than_inverse_sqrt_d(orc, D, scale, window):
    """A softmax scale that is not 1/sqrt(D), larger and smaller: the scale must enter S, the
    saved lse, dS and dK (every place it appears), not a constant derived from D."""
    compare_dense(orc, synth.dense(1, 4, 2, 260, D, window, seed=D + window, scale=scale))


@pytest.mark.parametrize("D", [512, 256])
def test_wide_gqa_group(orc, D):
    """16 query heads over one KV head: the backward sums dK / dV over the whole group."""
    compare_dense(orc, synth.dense(1, 16, 1, 200, D, 0, seed=16 + D))


@pytest.mark.parametrize("Hq,Hkv,window", [(2, 2, 0), (3, 1, 0), (6, 3, 130), (4, 2, 0), (8, 2, 300)])
def test_d512_forward_paths(orc, Hq, Hkv, window):
    """Head_dim 512: even GQA groups run the forward in CTA pairs (two query heads of a group on
    two SMs sharing one MMA), odd groups (1, 3) in single CTAs; both against the oracle, with a
    ragged last tile and, for some, a window."""
    compare_dense(orc, synth.dense(1, Hq, Hkv, 333, 512, window, seed=Hq * 7 + Hkv + window))


def test_forward_is_deterministic():
    p = synth.dense(1, 4, 2, 300, 512, 0, seed=4, with_do=False)
    q, k, v = to_dev(p.q), to_dev(p.k), to_dev(p.v)
    o1, l1 = attn.attn_fwd(q, k, v, scale=p.scale)
    o2, l2 = attn.attn_fwd(q, k, v, scale=p.scale)
    torch.cuda.synchronize()
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16)) and torch.equal(l1, l2)


@pytest.mark.parametrize("D,window", [(512, 0), (512, 150), (256, 0), (256, 100)])
def test_varlen(orc, D, window):
    lens = [1, 127, 128, 129, 300, 0, 513]
    vp = synth.varlen_from_lengths(lens, 4, 1, D, window, seed=D + window)
    q, k, v, do = (to_dev(x) for x in (vp.q, vp.k, vp.v, vp.do))
    cu = torch.from_numpy(vp.cu_seqlens).cuda()
    o, lse = attn.attn_fwd_varlen(q, k, v, cu, vp.max_seqlen, window=window, scale=vp.scale)
    dq, dk, dv = attn.attn_bwd(q, k, v, o, lse, do, window=window, scale=vp.scale, cu_seqlens=cu,
                               max_seqlen=vp.max_seqlen)
    torch.cuda.synchronize()
    assert attn.attn_get_device_status() == 0
    ro, rl = orc.fwd_varlen(vp.q, vp.k, vp.v, vp.cu_seqlens, vp.scale, 1, window)
    rdq, rdk, rdv, _ = orc.bwd_varlen(vp.q, vp.k, vp.v, vp.do, vp.cu_seqlens, vp.scale, 1, window)
    check("o", to_np(o), ro)
    check_lse("lse", to_np(lse), rl)
    check("dq", to_np(dq), rdq)
    check("dk", to_np(dk), rdk)
    check("dv", to_np(dv), rdv)


@pytest.mark.parametrize("D,window", [(512, 0), (256, 64)])
def test_varlen_many_short_sequences(orc, D, window):
    """Forty sequences, many shorter than a tile, some empty or of one or two tokens: every query
    tile stays inside its own sequence and every key range ends at its own sequence's end."""
    lens = [int(x) for x in np.random.default_rng(D + window).choice([0, 1, 2, 3, 17, 64, 127, 128, 129, 200], 40)]
    vp = synth.varlen_from_lengths(lens, 4, 2, D, window, seed=D + 1)
    q, k, v, do = (to_dev(x) for x in (vp.q, vp.k, vp.v, vp.do))
    cu = torch.from_numpy(vp.cu_seqlens).cuda()
    o, lse = attn.attn_fwd_varlen(q, k, v, cu, vp.max_seqlen, window=window, scale=vp.scale)
    dq, dk, dv = attn.attn_bwd(q, k, v, o, lse, do, window=window, scale=vp.scale, cu_seqlens=cu,
                               max_seqlen=vp.max_seqlen)
    torch.cuda.synchronize()
    assert attn.attn_get_device_status() == 0
    ro, rl = orc.fwd_varlen(vp.q, vp.k, vp.v, vp.cu_seqlens, vp.scale, 1, window)
    rdq, rdk, rdv, _ = orc.bwd_varlen(vp.q, vp.k, vp.v, vp.do, vp.cu_seqlens, vp.scale, 1, window)
    check("o", to_np(o), ro)
    check_lse("lse", to_np(lse), rl)
    check("dq", to_np(dq), rdq)
    check("dk", to_np(dk), rdk)
    check("dv", to_np(dv), rdv)


def test_varlen_equals_dense_per_sequence():
    """The packed result of each sequence is bitwise the dense result of that sequence alone."""
    lens = [200, 77]
    vp = synth.varlen_from_lengths(lens, 4, 2, 512, 0, seed=31, with_do=False)
    q, k, v = (to_dev(x) for x in (vp.q, vp.k, vp.v))
    cu = torch.from_numpy(vp.cu_seqlens).cuda()
    o, lse = attn.attn_fwd_varlen(q, k, v, cu, vp.max_seqlen, scale=vp.scale)
    for s, L in enumerate(lens):
        a = int(vp.cu_seqlens[s])
        od, ld = attn.attn_fwd(q[a:a + L][None].contiguous(), k[a:a + L][None].contiguous(),
                               v[a:a + L][None].contiguous(), scale=vp.scale)
        torch.cuda.synchronize()
        assert torch.equal(o[a:a + L].view(torch.int16), od[0].view(torch.int16))
        assert torch.equal(lse[:, a:a + L], ld[0])


# (planted cu_seqlens, max_seqlen, indices of the sequences whose slices stay valid); the true
# lengths are [200, 100, 300] (cu [0, 200, 300, 600], T = 600)
_BAD_CU = {
    "decreasing": ([0, 200, 100, 600], 300, [0]),         # seq 1 ends before it starts; seq 2 then exceeds 300
    "past_the_end": ([0, 200, 300, 700], 300, [0, 1]),    # seq 2 ends beyond the 600 packed rows
    "negative_start": ([-5, 200, 300, 600], 300, [1, 2]), # seq 0 starts before row 0
    "longer_than_max": ([0, 200, 300, 600], 250, [0, 1]), # seq 2 (300 tokens) is longer than max_seqlen
}


@pytest.mark.parametrize("D", [512, 256, 128])
@pytest.mark.parametrize("case", sorted(_BAD_CU))
def test_varlen_bad_cu_seqlens_is_reported_not_touched(orc, D, case):
    """A malformed prefix sum from the caller (the varlen path stands in for a 2-D padding mask)
    must not turn into out-of-range accesses: each sequence's slice is checked on the device, a
    bad one is reported as ATTN_ERR_DEVICE_BOUNDS and none of its rows is read or written, and
    the sequences whose slices are valid are still computed (forward and backward)."""
    lens = [200, 100, 300]
    bad_cu, max_seqlen, good = _BAD_CU[case]
    vp = synth.varlen_from_lengths(lens, 4, 2, D, 0, seed=D + len(case))
    T = int(vp.cu_seqlens[-1])
    q, k, v, do = (to_dev(x) for x in (vp.q, vp.k, vp.v, vp.do))
    cu_ok = torch.from_numpy(vp.cu_seqlens).cuda()
    cu_bad = torch.tensor(bad_cu, dtype=torch.int32, device="cuda")
    # reference rows: the valid slices of the planted prefix sum are slices of the true one
    ro, rl = orc.fwd_varlen(vp.q, vp.k, vp.v, vp.cu_seqlens, vp.scale, 1, 0)
    rdq, rdk, rdv, _ = orc.bwd_varlen(vp.q, vp.k, vp.v, vp.do, vp.cu_seqlens, vp.scale, 1, 0)
    good_rows = np.concatenate([np.arange(vp.cu_seqlens[s], vp.cu_seqlens[s + 1]) for s in good])
    untouched = np.setdiff1d(np.arange(T), good_rows)

    o = torch.zeros_like(q)
    lse = torch.full((4, T), 7.0, dtype=torch.float32, device="cuda")
    attn.attn_fwd_varlen(q, k, v, cu_bad, max_seqlen, o, lse, scale=vp.scale)
    assert attn.attn_get_device_status() == 7  # ATTN_ERR_DEVICE_BOUNDS
    on, ln = to_np(o), to_np(lse)
    check("o[valid]", on[good_rows], ro[good_rows])
    check_lse("lse[valid]", ln[:, good_rows], rl[:, good_rows])
    assert np.all(on[untouched] == 0) and np.all(ln[:, untouched] == 7.0)

    # backward with the forward of the true prefix sum as input, then the planted one
    o_ok, lse_ok = attn.attn_fwd_varlen(q, k, v, cu_ok, vp.max_seqlen, scale=vp.scale)
    dq = torch.full_like(q, 3.0)
    dk = torch.full_like(k, 3.0)
    dv = torch.full_like(v, 3.0)
    attn.attn_bwd(q, k, v, o_ok, lse_ok, do, dq, dk, dv, scale=vp.scale, cu_seqlens=cu_bad, max_seqlen=max_seqlen)
    assert attn.attn_get_device_status() == 7
    dqn, dkn, dvn = to_np(dq), to_np(dk), to_np(dv)
    check("dq[valid]", dqn[good_rows], rdq[good_rows])
    check("dk[valid]", dkn[good_rows], rdk[good_rows])
    check("dv[valid]", dvn[good_rows], rdv[good_rows])
    assert np.all(dqn[untouched] == 0)  # the accumulator of a skipped slice stays zero
    assert np.all(dkn[untouched] == 3.0) and np.all(dvn[untouched] == 3.0)
    assert attn.attn_get_device_status() == 0  # cleared by the previous read


def run_decode(pp, workspace=None):
    q, kc, vc = to_dev(pp.q), to_dev(pp.k_cache), to_dev(pp.v_cache)
    bt = torch.from_numpy(pp.block_table).cuda()
    sl = torch.from_numpy(pp.seq_lens).cuda()
    o, lse = attn.attn_decode_paged(q, kc, vc, bt, sl, scale=pp.scale, workspace=workspace)
    torch.cuda.synchronize()
    return to_np(o), to_np(lse)


@pytest.mark.parametrize("Hq,Hkv", [(32, 8), (8, 8), (16, 8), (64, 8), (8, 2)])
def test_decode_paged(orc, Hq, Hkv):
    lens = [1, 15, 16, 17, 33, 256, 1024, 0, 700, 5]
    pp = synth.paged_from_lengths(lens, Hq, Hkv, 128, page_size=16, num_pages=256, seed=Hq + Hkv, max_pages=64)
    o, lse = run_decode(pp)
    assert attn.attn_get_device_status() == 0
    ro, rl = orc.decode_paged(pp.q, pp.k_cache, pp.v_cache, pp.block_table, pp.seq_lens, pp.scale)
    check("o", o, ro)
    check_lse("lse", lse, rl)
    assert np.all(o[7] == 0) and np.all(np.isneginf(lse[7]))  # empty request


def test_decode_repeated_calls_reuse_workspace(orc):
    """The workspace's contents on entry do not matter: it starts as arbitrary bytes, and a
    second call on it gives the same bits as the first."""
    pp = synth.paged_from_lengths([900, 1000, 3, 512], 32, 8, 128, page_size=16, num_pages=512, seed=2, max_pages=64)
    g = torch.Generator(device="cuda").manual_seed(3)
    ws = torch.randint(0, 256, (attn.attn_workspace_size(attn.ATTN_OP_DECODE_PAGED, 4, 32, 8, 0, 128),),
                       dtype=torch.uint8, device="cuda", generator=g)
    o1, l1 = run_decode(pp, ws)
    o2, l2 = run_decode(pp, ws)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
    ro, rl = orc.decode_paged(pp.q, pp.k_cache, pp.v_cache, pp.block_table, pp.seq_lens, pp.scale)
    check("o", o2, ro)
    check_lse("lse", l2, rl)


def test_decode_bad_page_id_is_reported_not_read(orc):
    """A page id outside the pool is never dereferenced: its tokens are skipped and the
    fault is reported by attn_get_device_status; other requests are unaffected."""
    pp = synth.paged_from_lengths([40, 40], 32, 8, 128, page_size=16, num_pages=16, seed=8, max_pages=4)
    bt = pp.block_table.copy()
    bt[1, 1] = 10_000_000
    bad = synth.Paged(**{**pp.__dict__, "block_table": bt})
    o, lse = run_decode(bad)
    assert attn.attn_get_device_status() == 7  # ATTN_ERR_DEVICE_BOUNDS
    ro, rl = orc.decode_paged(pp.q, pp.k_cache, pp.v_cache, pp.block_table, pp.seq_lens, pp.scale)
    check("o[0]", o[0], ro[0])
    assert np.isfinite(o[1]).all() and np.isfinite(lse[1]).all()
    assert attn.attn_get_device_status() == 0  # cleared by the previous read


def test_bounded_wait_gives_up_and_reports(orc):
    """Failure detection without a fault: a pipeline wait that nothing completes gives up after
    its limit, the kernel records ATTN_ERR_DEVICE_TIMEOUT and returns; the status is read on the
    host, cleared, and the context stays usable (a forward afterwards still matches the oracle)."""
    assert attn.attn_get_device_status() == 0
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record()
    attn.attn_selftest_wait_timeout(50)
    t1.record()
    assert attn.attn_get_device_status() == 6  # ATTN_ERR_DEVICE_TIMEOUT
    assert t0.elapsed_time(t1) >= 45.0  # it really waited out its limit
    assert attn.attn_get_device_status() == 0  # cleared by the previous read
    with pytest.raises(attn.AttnError):
        attn.attn_selftest_wait_timeout(0)  # limit out of range: rejected before anything runs
    compare_dense(orc, synth.dense(1, 2, 1, 200, 256, 0, seed=31), with_bwd=True)
