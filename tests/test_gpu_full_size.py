"""The benchmarked workloads at full size, in the launch configuration the benchmark times, and
the largest shape the suite runs (2^32 elements of q).

The oracle computes sampled output rows one by one (forward rows, dQ rows, and dK/dV
rows of keys whose query set is affordable); every output tensor must be finite.
"""
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


def all_finite(*ts):
    return all(bool(torch.isfinite(t.float()).all()) for t in ts)


def sample_q_rows(rng, nb, Hq, lens, n):
    rows = []
    for _ in range(n):
        b = int(rng.integers(nb))
        rows.append((b, int(rng.integers(Hq)), int(rng.integers(lens[b]))))
    for b in range(nb):  # the first and last rows of every sequence
        rows.append((b, int(rng.integers(Hq)), 0))
        rows.append((b, int(rng.integers(Hq)), int(lens[b]) - 1))
    return np.array(rows, np.int64)


def gather_rows(t, rows, packed=False):
    """t: numpy [B, S, H, D] (or [T, H, D] packed with cu offsets applied by caller)."""
    return np.stack([t[b, i, h] for b, h, i in rows])


def dense_case(orc, p, key_rows):
    q, k, v, do = (to_dev(x) for x in (p.q, p.k, p.v, p.do))
    o, lse = attn.attn_fwd(q, k, v, window=p.window, scale=p.scale)
    dq, dk, dv = attn.attn_bwd(q, k, v, o, lse, do, window=p.window, scale=p.scale)
    torch.cuda.synchronize()
    assert attn.attn_get_device_status() == 0
    assert all_finite(o, lse, dq, dk, dv)
    rng = np.random.default_rng(0)
    rows = sample_q_rows(rng, p.B, p.Hq, [p.S] * p.B, 24)
    ro, rl = orc.fwd_rows(p.q, p.k, p.v, rows, p.scale, 1, p.window)
    rdq = orc.dq_rows(p.q, p.k, p.v, p.do, rows, p.scale, 1, p.window)
    on, ln, dqn = to_np(o), to_np(lse), to_np(dq)
    check("o rows", np.stack([on[b, i, h] for b, h, i in rows]), ro)
    check_lse("lse rows", np.array([ln[b, h, i] for b, h, i in rows]), rl)
    check("dq rows", np.stack([dqn[b, i, h] for b, h, i in rows]), rdq)
    krows = np.array(key_rows, np.int64)
    rdk, rdv = orc.dkv_rows(p.q, p.k, p.v, p.do, krows, p.scale, 1, p.window)
    dkn, dvn = to_np(dk), to_np(dv)
    check("dk rows", np.stack([dkn[b, j, g] for b, g, j in krows]), rdk)
    check("dv rows", np.stack([dvn[b, j, g] for b, g, j in krows]), rdv)


def test_dense_d512_causal_full(orc):
    """B=2, Hq=32, Hkv=4, S=4096, D=512: dK/dV on keys near the end (few queries see them) and on
    the first keys and one mid-sequence key of two (batch, KV head) pairs. Key 0 is seen by all
    4096 queries of all 8 heads of its group: the longest accumulation in tensor memory (256
    steps of its key tile) checked at full size."""
    p = synth.dense_d512_causal(seed=0)
    S = p.S
    keys = [(0, 0, S - 1), (1, 3, S - 2), (0, 2, S - 129), (1, 1, S - 200), (0, 3, S - 128), (1, 0, S - 64),
            (0, 0, 0), (0, 0, 1), (0, 0, 127), (1, 2, 0), (1, 2, S // 2), (1, 2, S // 2 - 1)]
    dense_case(orc, p, keys)


def test_swa_d256_w1024_full(orc):
    """B=2, Hq=32, Hkv=16, S=8192, D=256, W=1024, 1 % x30 outliers; every gradient finite."""
    p = synth.swa_d256_w1024(seed=0)
    rng = np.random.default_rng(1)
    keys = [(int(rng.integers(2)), int(rng.integers(16)), int(rng.integers(8192))) for _ in range(6)]
    keys += [(0, 0, 0), (1, 15, 8191), (0, 5, 1023), (1, 7, 1024)]
    dense_case(orc, p, keys)


def test_varlen_d512_causal_full(orc):
    vp = synth.varlen_d512_causal(seed=0)
    q, k, v, do = (to_dev(x) for x in (vp.q, vp.k, vp.v, vp.do))
    cu = torch.from_numpy(vp.cu_seqlens).cuda()
    o, lse = attn.attn_fwd_varlen(q, k, v, cu, vp.max_seqlen, scale=vp.scale)
    dq, dk, dv = attn.attn_bwd(q, k, v, o, lse, do, scale=vp.scale, cu_seqlens=cu, max_seqlen=vp.max_seqlen)
    torch.cuda.synchronize()
    assert attn.attn_get_device_status() == 0
    assert all_finite(o, lse, dq, dk, dv)
    rng = np.random.default_rng(2)
    ns = len(vp.seqlens)
    rows = sample_q_rows(rng, ns, vp.Hq, vp.seqlens, 24)
    ro, rl = orc.fwd_rows(vp.q, vp.k, vp.v, rows, vp.scale, cu_seqlens=vp.cu_seqlens)
    rdq = orc.dq_rows(vp.q, vp.k, vp.v, vp.do, rows, vp.scale, cu_seqlens=vp.cu_seqlens)
    on, ln, dqn = to_np(o), to_np(lse), to_np(dq)
    cu_np = vp.cu_seqlens
    check("o rows", np.stack([on[cu_np[s] + i, h] for s, h, i in rows]), ro)
    check_lse("lse rows", np.array([ln[h, cu_np[s] + i] for s, h, i in rows]), rl)
    check("dq rows", np.stack([dqn[cu_np[s] + i, h] for s, h, i in rows]), rdq)
    # late keys of every sequence, and the first key of every sequence (seen by all its queries)
    krows = np.array([(s, int(rng.integers(vp.Hkv)), int(vp.seqlens[s]) - 1 - int(rng.integers(100)))
                      for s in range(ns)] + [(s, int(rng.integers(vp.Hkv)), 0) for s in range(ns)], np.int64)
    rdk, rdv = orc.dkv_rows(vp.q, vp.k, vp.v, vp.do, krows, vp.scale, cu_seqlens=vp.cu_seqlens)
    dkn, dvn = to_np(dk), to_np(dv)
    check("dk rows", np.stack([dkn[cu_np[s] + j, g] for s, g, j in krows]), rdk)
    check("dv rows", np.stack([dvn[cu_np[s] + j, g] for s, g, j in krows]), rdv)


def test_decode_paged_d128_full(orc):
    """batch 64, Hq=32, Hkv=8, D=128, lengths U[256,1024], page 16, 4096-page permuted pool: all outputs."""
    pp = synth.decode_paged_d128(seed=0)
    q, kc, vc = to_dev(pp.q), to_dev(pp.k_cache), to_dev(pp.v_cache)
    bt = torch.from_numpy(pp.block_table).cuda()
    sl = torch.from_numpy(pp.seq_lens).cuda()
    o, lse = attn.attn_decode_paged(q, kc, vc, bt, sl, scale=pp.scale)
    torch.cuda.synchronize()
    assert attn.attn_get_device_status() == 0
    ro, rl = orc.decode_paged(pp.q, pp.k_cache, pp.v_cache, pp.block_table, pp.seq_lens, pp.scale)
    check("o", to_np(o), ro)
    check_lse("lse", to_np(lse), rl)


def test_forward_beyond_2_31_elements(orc):
    """The largest shape this suite runs: q holds 2^32 elements (B 1, S 131072, Hq 32, D 512), so
    any 32-bit element index in the output or lse addressing would wrap. Sampled rows, among
    them the last, are checked against the oracle; every output is finite."""
    p = synth.dense(1, 32, 1, 131072, 512, 0, seed=3, with_do=False)
    q, k, v = to_dev(p.q), to_dev(p.k), to_dev(p.v)
    o, lse = attn.attn_fwd(q, k, v, scale=p.scale)
    torch.cuda.synchronize()
    assert attn.attn_get_device_status() == 0
    assert all_finite(o, lse)
    rows = np.array([[0, 0, 0], [0, 31, 131071], [0, 17, 131071], [0, 5, 65536], [0, 30, 100000], [0, 12, 4097]],
                    dtype=np.int64)
    ro, rl = orc.fwd_rows(p.q, p.k, p.v, rows, p.scale)
    got_o = np.stack([to_np(o[0, s, hh]) for _, hh, s in rows])
    got_l = np.array([float(lse[0, hh, s]) for _, hh, s in rows])
    check("o[sampled rows]", got_o, ro)
    check_lse("lse[sampled rows]", got_l, rl)
