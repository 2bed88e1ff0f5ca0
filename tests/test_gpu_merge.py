"""Merge of attention results over disjoint key sets (attn_merge_lse) against the fp64 oracle,
plus the end-to-end identity that ties it to the forward: a sliding-window forward and a
shifted causal forward over the remaining keys merge into the full causal forward."""
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


def run_merge(mp):
    op = to_dev(mp.o_parts)
    lp = torch.from_numpy(mp.lse_parts).cuda()
    o, lse = attn.attn_merge_lse(op, lp)
    torch.cuda.synchronize()
    return to_np(o), lse.cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("P", [1, 2, 3, 5, 8])
@pytest.mark.parametrize("D", [64, 128, 256, 512])
def test_merge_lse(orc, P, D):
    mp = synth.merge_parts(P, 2, 37, 3, D, seed=P * 1000 + D, empty_pct=15)
    o, lse = run_merge(mp)
    ro, rl = orc.merge_lse(mp.o_parts, mp.lse_parts)
    check("o", o, ro)
    check_lse("lse", lse, rl)


def test_merge_lse_empty_parts_are_never_read(orc):
    """Parts whose lse is -inf hold NaN in o: nothing of it reaches the result. Rows empty in
    every part give o = 0 and lse = -inf."""
    mp = synth.merge_parts(4, 1, 50, 2, 128, seed=3, empty_pct=40)
    lse = mp.lse_parts.copy()
    lse[:, 0, :, :5] = -np.inf  # s = 0..4 empty everywhere
    o_parts = mp.o_parts.copy()
    empty = np.isneginf(lse)  # [P, B, H, S]
    o_parts[np.transpose(empty, (0, 1, 3, 2))] = 0x7FC0  # NaN in every empty (part, row)
    bad = synth.MergeParts(mp.name, mp.P, mp.B, mp.S, mp.H, mp.D, o_parts, lse)
    o, got = run_merge(bad)
    ro, rl = orc.merge_lse(mp.o_parts, lse)
    check("o", o, ro)
    check_lse("lse", got, rl)
    assert np.all(o[0, :5] == 0) and np.all(np.isneginf(got[0, :, :5]))


def test_merge_lse_in_place_running_merge(orc):
    """Folding parts one at a time into part 0's buffers (o == o_parts[0], lse == lse_parts[0])
    agrees with merging all at once."""
    mp = synth.merge_parts(5, 1, 64, 4, 256, seed=9, empty_pct=10)
    op = to_dev(mp.o_parts)
    lp = torch.from_numpy(mp.lse_parts).cuda()
    pair_o = torch.empty((2,) + tuple(op.shape[1:]), dtype=torch.bfloat16, device="cuda")
    pair_l = torch.empty((2,) + tuple(lp.shape[1:]), dtype=torch.float32, device="cuda")
    pair_o[0].copy_(op[0])
    pair_l[0].copy_(lp[0])
    for p in range(1, mp.P):
        pair_o[1].copy_(op[p])
        pair_l[1].copy_(lp[p])
        attn.attn_merge_lse(pair_o, pair_l, pair_o[0], pair_l[0])
    torch.cuda.synchronize()
    ro, rl = orc.merge_lse(mp.o_parts, mp.lse_parts)
    check("o (running merge)", to_np(pair_o[0]), ro)
    check_lse("lse (running merge)", pair_l[0].cpu().numpy().astype(np.float64), rl)


@pytest.mark.parametrize("D,S,W", [(256, 700, 300), (512, 385, 129)])
def test_window_and_shifted_causal_merge_to_causal(orc, D, S, W):
    """Keys of query i split into its window (i-W, i] and the rest [0, i-W]: the first part is the
    sliding-window forward, the second the causal forward of q[W:] over k[:S-W]. Their merge is
    the full causal forward."""
    p = synth.dense(2, 4, 2, S, D, 0, seed=S + W)
    q, k, v = to_dev(p.q), to_dev(p.k), to_dev(p.v)
    B, Hq = p.B, p.Hq
    o_parts = torch.zeros((2, B, S, Hq, D), dtype=torch.bfloat16, device="cuda")
    l_parts = torch.full((2, B, Hq, S), float("-inf"), dtype=torch.float32, device="cuda")
    attn.attn_fwd(q, k, v, o_parts[0], l_parts[0], window=W, scale=p.scale)
    o2, l2 = attn.attn_fwd(q[:, W:].contiguous(), k[:, :S - W].contiguous(), v[:, :S - W].contiguous(),
                           scale=p.scale)
    o_parts[1, :, W:] = o2
    l_parts[1, :, :, W:] = l2
    o, lse = attn.attn_merge_lse(o_parts, l_parts)
    of, lf = attn.attn_fwd(q, k, v, scale=p.scale)
    torch.cuda.synchronize()
    assert attn.attn_get_device_status() == 0
    ro, rl = orc.fwd(p.q, p.k, p.v, p.scale, 1, 0)
    check("merged o vs oracle causal", to_np(o), ro)
    check_lse("merged lse vs oracle causal", lse.cpu().numpy().astype(np.float64), rl)
    check("merged o vs causal forward", to_np(o), to_np(of))
    check_lse("merged lse vs causal forward", lse.cpu().numpy().astype(np.float64),
              lf.cpu().numpy().astype(np.float64))


def test_merge_lse_full_workload_sampled(orc):
    """The benchmarked merge (8 parts, 2048 tokens, 32 heads, D 512) in the benchmark's launch;
    the oracle checks 96 sampled token rows across all heads."""
    mp = synth.merge_cp8_d512(seed=0)
    o, lse = run_merge(mp)
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    rows = np.unique(np.concatenate([[0, 1, mp.S - 1], np.random.default_rng(4).integers(0, mp.S, 93)]))
    ro, rl = orc.merge_lse(mp.o_parts[:, :, rows], mp.lse_parts[:, :, :, rows])
    check("o[sampled rows]", o[:, rows], ro)
    check_lse("lse[sampled rows]", lse[:, :, rows], rl)
