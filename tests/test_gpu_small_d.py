"""head_dim 128 and 64 (Qwen3-class heads): the forward in its dense, windowed, varlen and paged
forms against the fp64 oracle."""
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


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("B,Hq,Hkv,S,W", [(2, 4, 2, 300, 0), (1, 8, 1, 385, 0), (1, 6, 2, 129, 0), (2, 4, 4, 700, 129),
                                          (1, 2, 1, 1, 0), (1, 4, 1, 513, 1), (1, 4, 2, 640, 300)])
def test_forward_small_d(orc, D, B, Hq, Hkv, S, W):
    p = synth.dense(B, Hq, Hkv, S, D, W, seed=S + D + W, with_do=False)
    q, k, v = to_dev(p.q), to_dev(p.k), to_dev(p.v)
    o, lse = attn.attn_fwd(q, k, v, window=W, scale=p.scale)
    torch.cuda.synchronize()
    assert attn.attn_get_device_status() == 0
    ro, rl = orc.fwd(p.q, p.k, p.v, p.scale, 1, W)
    check("o", to_np(o), ro)
    check_lse("lse", to_np(lse), rl)


@pytest.mark.parametrize("D", [64, 128])
def test_forward_small_d_varlen(orc, D):
    vp = synth.varlen_from_lengths([1, 127, 128, 129, 300, 0, 513], 8, 2, D, seed=D, with_do=False)
    q, k, v = to_dev(vp.q), to_dev(vp.k), to_dev(vp.v)
    cu = torch.from_numpy(vp.cu_seqlens).cuda()
    o, lse = attn.attn_fwd_varlen(q, k, v, cu, vp.max_seqlen, scale=vp.scale)
    torch.cuda.synchronize()
    assert attn.attn_get_device_status() == 0
    ro, rl = orc.fwd_varlen(vp.q, vp.k, vp.v, vp.cu_seqlens, vp.scale)
    check("o", to_np(o), ro)
    check_lse("lse", to_np(lse), rl)


@pytest.mark.parametrize("D,window", [(64, 0), (128, 0), (128, 100), (64, 37)])
def test_prefill_paged_small_d(orc, D, window):
    seq = [1, 16, 17, 300, 1000, 129, 700, 2049]
    nq = [1, 16, 5, 300, 128, 0, 257, 131]
    pp = synth.prefill_paged_from_lengths(seq, nq, 8, 2, D, window=window, seed=D + window)
    q, kc, vc = to_dev(pp.q), to_dev(pp.k_cache), to_dev(pp.v_cache)
    bt, sl, cu = (torch.from_numpy(x).cuda() for x in (pp.block_table, pp.seq_lens, pp.cu_q))
    o, lse = attn.attn_fwd_paged(q, kc, vc, bt, sl, cu, pp.max_q, window=window, scale=pp.scale)
    torch.cuda.synchronize()
    assert attn.attn_get_device_status() == 0
    ro, rl = orc.prefill_paged(pp.q, pp.k_cache, pp.v_cache, pp.block_table, pp.seq_lens, pp.cu_q, pp.scale, window)
    check("o", to_np(o), ro)
    check_lse("lse", to_np(lse), rl)


def _bwd_dense(orc, p):
    q, k, v, do = to_dev(p.q), to_dev(p.k), to_dev(p.v), to_dev(p.do)
    o, lse = attn.attn_fwd(q, k, v, window=p.window, scale=p.scale)
    dq, dk, dv = attn.attn_bwd(q, k, v, o, lse, do, window=p.window, scale=p.scale)
    torch.cuda.synchronize()
    assert attn.attn_get_device_status() == 0
    rdq, rdk, rdv, *_ = orc.bwd(p.q, p.k, p.v, p.do, p.scale, 1, p.window)
    check("dq", to_np(dq), rdq)
    check("dk", to_np(dk), rdk)
    check("dv", to_np(dv), rdv)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("B,Hq,Hkv,S,W", [(2, 4, 2, 300, 0), (1, 8, 1, 385, 0), (1, 6, 2, 129, 0), (2, 4, 4, 700, 129),
                                          (1, 2, 1, 1, 0), (1, 4, 1, 513, 1), (1, 4, 2, 640, 300)])
def test_backward_small_d(orc, D, B, Hq, Hkv, S, W):
    _bwd_dense(orc, synth.dense(B, Hq, Hkv, S, D, W, seed=S + D + W + 1))


@pytest.mark.parametrize("D", [64, 128])
def test_backward_small_d_outliers(orc, D):
    """Scaled outliers in q and k (1 % of entries x 30, as in the window workload): finite, in tolerance."""
    _bwd_dense(orc, synth.dense(1, 4, 2, 520, D, 256, seed=D, outlier_frac=0.01, outlier_scale=30.0))


@pytest.mark.parametrize("D", [64, 128])
def test_backward_small_d_varlen(orc, D):
    vp = synth.varlen_from_lengths([1, 127, 128, 129, 300, 0, 513], 8, 2, D, seed=D + 5)
    q, k, v, do = to_dev(vp.q), to_dev(vp.k), to_dev(vp.v), to_dev(vp.do)
    cu = torch.from_numpy(vp.cu_seqlens).cuda()
    o, lse = attn.attn_fwd_varlen(q, k, v, cu, vp.max_seqlen, scale=vp.scale)
    dq, dk, dv = attn.attn_bwd(q, k, v, o, lse, do, scale=vp.scale, cu_seqlens=cu, max_seqlen=vp.max_seqlen)
    torch.cuda.synchronize()
    assert attn.attn_get_device_status() == 0
    rdq, rdk, rdv, *_ = orc.bwd_varlen(vp.q, vp.k, vp.v, vp.do, vp.cu_seqlens, vp.scale)
    check("dq", to_np(dq), rdq)
    check("dk", to_np(dk), rdk)
    check("dv", to_np(dv), rdv)


@pytest.mark.parametrize("D", [64, 128, 256, 512])
@pytest.mark.parametrize("W", [0, 300])
def test_forward_running_max_keeps_moving(orc, D, W):
    """Keys scaled up along the sequence, so the scores of every later key tile exceed the
    running maximum by far more than the lazy-rescale threshold: O is rescaled in tensor memory
    on almost every step (with two score buffers at D >= 256 and three at D <= 128)."""
    p = synth.dense(1, 4, 2, 700, D, W, seed=D + W, with_do=False)
    kb = p.k.view(np.uint16).copy()
    kf = (kb.astype(np.uint32) << 16).view(np.float32)
    kf *= (1.0 + np.arange(p.S, dtype=np.float32) / 40.0)[None, :, None, None]
    k_new = ((kf.view(np.uint32) + 0x8000) >> 16).astype(np.uint16)
    q, k, v = to_dev(p.q), to_dev(k_new.view(p.k.dtype)), to_dev(p.v)
    o, lse = attn.attn_fwd(q, k, v, window=W, scale=p.scale)
    torch.cuda.synchronize()
    assert attn.attn_get_device_status() == 0
    ro, rl = orc.fwd(p.q, k_new.view(p.k.dtype), p.v, p.scale, 1, W)
    check("o", to_np(o), ro)
    check_lse("lse", to_np(lse), rl)
