"""Pins that tie the fp64 oracle to things other than itself.

Each ``pin_*`` takes an ``oracle.Oracle`` and raises AssertionError when the
oracle disagrees with:

* a library routine computing the same definition (torch's fp64 CPU
  scaled_dot_product_attention with its own GQA broadcast, torch.logsumexp, and
  torch autograd for the gradient),
* central finite differences of L = sum(dO * O) through the oracle's own forward
  (pins the backward to the forward, whatever formula either uses),
* closed forms (scale 0, window 1, identical keys, all-ones values),
* invariants (wide window = causal, varlen = per-sequence dense, paged =
  contiguous, decode = last prefill row, paged prefill = gathered keys with a
  bottom-right mask and one new token = decode, GQA = repeat-KV MHA, key shifts),
* the hand-worked examples under ``tests/golden``.

The same pins run against deliberately broken builds of the oracle
(``test_oracle_mutants.py``) to show each plausible mistake is caught.
"""
from __future__ import annotations

import json
import os

import numpy as np
import torch

import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _f(bits):
    return synth.bf16_to_f32(bits).astype(np.float64)


def _bf16_exact(x):
    """bf16 bits of values that must be exactly representable."""
    x = np.asarray(x, dtype=np.float64)
    bits = synth.f32_to_bf16(x.astype(np.float32))
    assert np.array_equal(_f(bits), x), "test value not representable in bf16"
    return bits


def _mask(S, causal, window, Sk=None):
    Sk = S if Sk is None else Sk
    i = np.arange(S)[:, None]
    j = np.arange(Sk)[None, :]
    m = np.ones((S, Sk), bool)
    if causal:
        m &= j <= i
    if window > 0:
        m &= (i - j) < window
    return m


def _torch_ref(q, k, v, do, scale, causal, window):
    """torch fp64 reference: SDPA with enable_gqa and a boolean mask, autograd for grads."""
    qt = torch.tensor(_f(q)).permute(0, 2, 1, 3).contiguous().requires_grad_(True)  # B,H,S,D
    kt = torch.tensor(_f(k)).permute(0, 2, 1, 3).contiguous().requires_grad_(True)
    vt = torch.tensor(_f(v)).permute(0, 2, 1, 3).contiguous().requires_grad_(True)
    S = q.shape[1]
    mask = torch.tensor(_mask(S, causal, window))
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask, scale=scale, enable_gqa=True)
    G = q.shape[2] // k.shape[2]
    scores = (qt @ kt.repeat_interleave(G, dim=1).transpose(-1, -2)) * scale
    lse = torch.logsumexp(scores.masked_fill(~mask, float("-inf")), dim=-1)
    grads = None
    if do is not None:
        dot = torch.tensor(_f(do)).permute(0, 2, 1, 3)
        grads = torch.autograd.grad(o, (qt, kt, vt), dot)
        grads = [g.permute(0, 2, 1, 3).detach().numpy() for g in grads]
    return o.detach().permute(0, 2, 1, 3).numpy(), lse.detach().numpy(), grads


def _close(a, b, tol, what):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    assert a.shape == b.shape, f"{what}: shape {a.shape} vs {b.shape}"
    fin = np.isfinite(b)
    assert np.array_equal(np.isfinite(a), fin), f"{what}: finiteness differs"
    assert np.array_equal(a[~fin], b[~fin]), f"{what}: non-finite values differ"
    err = np.max(np.abs(a[fin] - b[fin])) if fin.any() else 0.0
    scale = max(1.0, np.max(np.abs(b[fin])) if fin.any() else 1.0)
    assert err <= tol * scale, f"{what}: max abs err {err:.3e} > {tol:.1e} * {scale:.3g}"


# ------------------------------------------------------------------------------------
def pin_torch_forward(orc):
    for (B, S, Hq, Hkv, D, window, seed) in [(2, 37, 4, 2, 16, 0, 1), (1, 45, 6, 3, 8, 7, 2), (1, 20, 2, 2, 32, 1, 3)]:
        p = synth.dense(B, Hq, Hkv, S, D, window, seed=seed, with_do=False)
        o, lse = orc.fwd(p.q, p.k, p.v, p.scale, 1, window)
        to, tlse, _ = _torch_ref(p.q, p.k, p.v, None, p.scale, 1, window)
        _close(o, to, 1e-12, "o vs torch sdpa")
        _close(lse, tlse, 1e-12, "lse vs torch logsumexp")


def pin_torch_backward(orc):
    for (B, S, Hq, Hkv, D, window, seed) in [(2, 33, 4, 2, 16, 0, 4), (1, 41, 6, 2, 8, 9, 5)]:
        p = synth.dense(B, Hq, Hkv, S, D, window, seed=seed)
        dq, dk, dv, o, delta, gap = orc.bwd(p.q, p.k, p.v, p.do, p.scale, 1, window)
        to, _, (tdq, tdk, tdv) = _torch_ref(p.q, p.k, p.v, p.do, p.scale, 1, window)
        _close(o, to, 1e-12, "bwd o vs torch")
        _close(dq, tdq, 1e-11, "dq vs torch autograd")
        _close(dk, tdk, 1e-11, "dk vs torch autograd")
        _close(dv, tdv, 1e-11, "dv vs torch autograd")
        # Delta = sum_j p dp must equal dO . o
        assert gap < 1e-10, f"Delta two ways differ by {gap}"
        _close(delta, np.einsum("bshd,bshd->bhs", _f(p.do), to), 1e-11, "Delta vs dO.o")


def pin_finite_differences(orc):
    """dL/dx for L = sum(dO * O), by Richardson-extrapolated central differences."""
    rng = np.random.default_rng(11)
    B, S, Hq, Hkv, D, window = 1, 12, 4, 2, 8, 5
    p = synth.dense(B, Hq, Hkv, S, D, window, seed=21)
    dq, dk, dv, *_ = orc.bwd(p.q, p.k, p.v, p.do, p.scale, 1, window)
    dof = _f(p.do)

    def loss(q, k, v):
        o, _ = orc.fwd(q, k, v, p.scale, 1, window, nthreads=1)
        return float(np.sum(dof * o))

    checked = 0
    for name, arr, grad in (("q", p.q, dq), ("k", p.k, dk), ("v", p.v, dv)):
        flat = arr.reshape(-1)
        picks = rng.permutation(flat.size)
        n_ok = 0
        for idx in picks:
            x = float(_f(flat[idx:idx + 1])[0])
            h = 2.0 ** -4
            cands = [x + h, x - h, x + h / 2, x - h / 2]
            bits = synth.f32_to_bf16(np.array(cands, np.float32))
            if not np.array_equal(_f(bits), np.array(cands)):
                continue

            def at(val_bits):
                a = arr.copy().reshape(-1)
                a[idx] = val_bits
                a = a.reshape(arr.shape)
                if name == "q":
                    return loss(a, p.k, p.v)
                if name == "k":
                    return loss(p.q, a, p.v)
                return loss(p.q, p.k, a)

            d1 = (at(bits[0]) - at(bits[1])) / (2 * h)
            d2 = (at(bits[2]) - at(bits[3])) / h
            fd = (4 * d2 - d1) / 3
            an = float(grad.reshape(-1)[idx])
            assert abs(fd - an) <= 2e-4 * max(1.0, abs(an)), f"d{name}[{idx}]: finite diff {fd} vs analytic {an}"
            n_ok += 1
            checked += 1
            if n_ok >= 6:
                break
        assert n_ok >= 3, f"too few representable perturbations for {name}"
    assert checked >= 9


def pin_closed_forms(orc):
    B, S, Hq, Hkv, D = 1, 19, 4, 2, 8
    p = synth.dense(B, Hq, Hkv, S, D, 0, seed=7, with_do=False)
    G = Hq // Hkv
    vf = _f(p.v)
    for window in (0, 4):
        # scale 0: uniform weights over the allowed keys
        o, lse = orc.fwd(p.q, p.k, p.v, 0.0, 1, window)
        m = _mask(S, 1, window)
        cnt = m.sum(1)
        for h in range(Hq):
            g = h // G
            expect = (m.astype(np.float64) @ vf[0, :, g, :]) / cnt[:, None]
            _close(o[0, :, h, :], expect, 1e-13, "scale=0 mean of allowed values")
            _close(lse[0, h], np.log(cnt), 1e-13, "scale=0 lse = ln(count)")
    # window 1: each row sees only itself
    o, lse = orc.fwd(p.q, p.k, p.v, p.scale, 1, 1)
    qf, kf = _f(p.q), _f(p.k)
    for h in range(Hq):
        g = h // G
        _close(o[0, :, h, :], vf[0, :, g, :], 1e-13, "window=1 copies v_i")
        _close(lse[0, h], p.scale * np.sum(qf[0, :, h, :] * kf[0, :, g, :], axis=1), 1e-12, "window=1 lse = s_ii")
    # all-ones values: every output is exactly one (rows of P sum to one)
    ones = np.full_like(p.v, synth.f32_to_bf16(np.array([1.0], np.float32))[0])
    o, _ = orc.fwd(p.q, p.k, ones, p.scale, 1, 0)
    _close(o, np.ones_like(o), 1e-13, "rows of P sum to one")
    # identical keys: uniform weights, lse = s + ln(count)
    k_same = np.broadcast_to(p.k[:, :1], p.k.shape).copy()
    o, lse = orc.fwd(p.q, k_same, p.v, p.scale, 1, 0)
    cnt = np.arange(1, S + 1)
    for h in range(Hq):
        g = h // G
        expect = np.cumsum(vf[0, :, g, :], axis=0) / cnt[:, None]
        _close(o[0, :, h, :], expect, 1e-12, "identical keys: running mean")
        s = p.scale * _f(p.q)[0, :, h, :] @ _f(k_same)[0, 0, g, :]
        _close(lse[0, h], s + np.log(cnt), 1e-12, "identical keys lse")


def pin_invariants(orc):
    # window >= S reproduces causal
    p = synth.dense(1, 4, 2, 23, 16, 0, seed=8)
    o0, l0 = orc.fwd(p.q, p.k, p.v, p.scale, 1, 0)
    for w in (23, 24, 100):
        o1, l1 = orc.fwd(p.q, p.k, p.v, p.scale, 1, w)
        _close(o1, o0, 0, f"window {w} >= S equals causal")
        _close(l1, l0, 0, f"window {w} >= S lse equals causal")
    g0 = orc.bwd(p.q, p.k, p.v, p.do, p.scale, 1, 0)
    g1 = orc.bwd(p.q, p.k, p.v, p.do, p.scale, 1, 64)
    for a, b, n in zip(g0[:3], g1[:3], ("dq", "dk", "dv")):
        _close(b, a, 0, f"wide window {n} equals causal")

    # GQA equals MHA on repeated K/V; GQA dK/dV equal group sums of MHA dK/dV
    G = p.Hq // p.Hkv
    kr = np.repeat(p.k, G, axis=2)
    vr = np.repeat(p.v, G, axis=2)
    om, lm = orc.fwd(p.q, kr, vr, p.scale, 1, 0)
    _close(o0, om, 1e-13, "GQA = repeat-KV MHA (o)")
    _close(l0, lm, 1e-13, "GQA = repeat-KV MHA (lse)")
    gm = orc.bwd(p.q, kr, vr, p.do, p.scale, 1, 0)
    _close(g0[0], gm[0], 1e-12, "GQA dq = MHA dq")
    _close(g0[1], gm[1].reshape(1, 23, p.Hkv, G, 16).sum(3), 1e-12, "GQA dk = group-summed MHA dk")
    _close(g0[2], gm[2].reshape(1, 23, p.Hkv, G, 16).sum(3), 1e-12, "GQA dv = group-summed MHA dv")

    # key shift: k_j + u changes every score of row i by scale*q_i.u, so o is unchanged
    rng = np.random.default_rng(3)
    S, Hq, Hkv, D = 9, 2, 1, 4
    q = _bf16_exact(rng.integers(-8, 9, (1, S, Hq, D)) / 8.0)
    k = _bf16_exact(rng.integers(-8, 9, (1, S, Hkv, D)) / 8.0)
    v = _bf16_exact(rng.integers(-8, 9, (1, S, Hkv, D)) / 8.0)
    u = rng.integers(-8, 9, D) / 8.0
    ks = _bf16_exact(_f(k) + u)
    o_a, l_a = orc.fwd(q, k, v, 0.5, 1, 3)
    o_b, l_b = orc.fwd(q, ks, v, 0.5, 1, 3)
    _close(o_b, o_a, 1e-13, "key shift leaves o unchanged")
    _close(l_b, l_a + 0.5 * np.einsum("bshd,d->bhs", _f(q), u), 1e-12, "key shift moves lse by scale q.u")


def pin_varlen(orc):
    lens = [5, 1, 17, 0, 9]
    for window in (0, 4):
        vp = synth.varlen_from_lengths(lens, 4, 2, 16, window, seed=12)
        o, lse = orc.fwd_varlen(vp.q, vp.k, vp.v, vp.cu_seqlens, vp.scale, 1, window)
        dq, dk, dv, gap = orc.bwd_varlen(vp.q, vp.k, vp.v, vp.do, vp.cu_seqlens, vp.scale, 1, window)
        assert gap < 1e-10
        for s, L in enumerate(lens):
            a, b = vp.cu_seqlens[s], vp.cu_seqlens[s + 1]
            if L == 0:
                continue
            sl = lambda x: x[a:b][None]
            od, ld = orc.fwd(sl(vp.q), sl(vp.k), sl(vp.v), vp.scale, 1, window)
            _close(o[a:b], od[0], 0, "varlen o = dense per sequence")
            _close(lse[:, a:b], ld[0], 0, "varlen lse = dense per sequence")
            gd = orc.bwd(sl(vp.q), sl(vp.k), sl(vp.v), sl(vp.do), vp.scale, 1, window)
            _close(dq[a:b], gd[0][0], 0, "varlen dq = dense")
            _close(dk[a:b], gd[1][0], 0, "varlen dk = dense")
            _close(dv[a:b], gd[2][0], 0, "varlen dv = dense")
    # packing two sequences as one with a cross-document mask would differ: the
    # second sequence must not see the first
    vp = synth.varlen_from_lengths([6, 6], 2, 1, 8, 0, seed=13)
    o, _ = orc.fwd_varlen(vp.q, vp.k, vp.v, vp.cu_seqlens, vp.scale)
    o_joint, _ = orc.fwd(vp.q[None], vp.k[None], vp.v[None], vp.scale)
    assert np.max(np.abs(o[6:] - o_joint[0, 6:])) > 1e-3, "varlen must not leak across sequences"


def pin_paged(orc):
    pp = synth.paged_from_lengths([1, 16, 17, 40, 33], 8, 2, 32, page_size=16, num_pages=64, seed=14, max_pages=4)
    o, lse = orc.decode_paged(pp.q, pp.k_cache, pp.v_cache, pp.block_table, pp.seq_lens, pp.scale)
    for b in range(pp.B):
        L = int(pp.seq_lens[b])
        tok = np.arange(L)
        pages = pp.block_table[b, tok // 16]
        kk = pp.k_cache[pages, tok % 16][None]  # [1, L, Hkv, D] contiguous copy
        vv = pp.v_cache[pages, tok % 16][None]
        # decode == last row of the prefill over the same contiguous keys
        qq = np.repeat(pp.q[b][None, None], L, axis=1)  # query rows; only row L-1 matters
        od, ld = orc.fwd(qq, kk, vv, pp.scale, 1, 0)
        _close(o[b], od[0, L - 1], 1e-13, "decode = last prefill row (o)")
        _close(lse[b], ld[0, :, L - 1], 1e-13, "decode = last prefill row (lse)")
    # relabelling the pool (permuting pages and the table with them) changes nothing
    perm = np.random.default_rng(5).permutation(pp.num_pages)
    inv = np.argsort(perm)
    kc2 = pp.k_cache[inv]
    vc2 = pp.v_cache[inv]
    bt2 = np.where(pp.block_table >= 0, perm[np.maximum(pp.block_table, 0)], -1).astype(np.int32)
    o2, l2 = orc.decode_paged(pp.q, kc2, vc2, bt2, pp.seq_lens, pp.scale)
    _close(o2, o, 0, "page relabelling (o)")
    _close(l2, lse, 0, "page relabelling (lse)")
    # a sliding window: the query at position L-1 sees keys max(0, L-W) .. L-1 (torch fp64 attention
    # over exactly those keys); windows of 1, inside a page, a whole page, across pages, beyond L
    for D in (32, 256):
        pw = synth.paged_from_lengths([1, 16, 17, 40, 33, 100], 4, 2, D, page_size=16, num_pages=64, seed=16 + D,
                                      max_pages=7)
        for W in (1, 7, 16, 17, 50):
            ow, lw = orc.decode_paged(pw.q, pw.k_cache, pw.v_cache, pw.block_table, pw.seq_lens, pw.scale, W)
            for b in range(pw.B):
                L = int(pw.seq_lens[b])
                tok = np.arange(max(0, L - W), L)
                pages = pw.block_table[b, tok // 16]
                kt = torch.tensor(_f(pw.k_cache[pages, tok % 16])).permute(1, 0, 2)[None]  # 1, Hkv, n, D
                vt = torch.tensor(_f(pw.v_cache[pages, tok % 16])).permute(1, 0, 2)[None]
                qt = torch.tensor(_f(pw.q[b]))[None, :, None, :]  # 1, Hq, 1, D
                to = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=pw.scale, enable_gqa=True)
                G = pw.Hq // pw.Hkv
                tl = torch.logsumexp((qt @ kt.repeat_interleave(G, dim=1).transpose(-1, -2)) * pw.scale, dim=-1)
                _close(ow[b], to[0, :, 0].numpy(), 1e-12, f"windowed decode o vs torch (W={W}, D={D})")
                _close(lw[b], tl[0, :, 0].numpy(), 1e-12, f"windowed decode lse vs torch (W={W}, D={D})")
    # an empty request gives o = 0 and lse = -inf, never NaN
    pe = synth.paged_from_lengths([0, 3], 4, 1, 16, page_size=16, num_pages=4, seed=15, max_pages=1)
    o3, l3 = orc.decode_paged(pe.q, pe.k_cache, pe.v_cache, pe.block_table, pe.seq_lens, pe.scale)
    assert np.all(o3[0] == 0) and np.all(np.isneginf(l3[0])) and np.all(np.isfinite(o3[1]))


def pin_prefill_paged(orc):
    """Chunked prefill over a paged cache vs torch fp64 SDPA on the gathered contiguous keys
    with a bottom-right aligned mask (new query i of a request sits at position L - n + i),
    with and without a window; single new token = decode; page relabelling changes nothing."""
    for window in (0, 7):
        pp = synth.prefill_paged_from_lengths([1, 16, 17, 40, 33, 9], [1, 5, 17, 12, 0, 9], 6, 2, 16, page_size=16,
                                              window=window, seed=21)
        o, lse = orc.prefill_paged(pp.q, pp.k_cache, pp.v_cache, pp.block_table, pp.seq_lens, pp.cu_q, pp.scale,
                                   window)
        for b in range(pp.B):
            L, n, r0 = int(pp.seq_lens[b]), int(pp.q_lens[b]), int(pp.cu_q[b])
            if n == 0:
                continue
            tok = np.arange(L)
            pages = pp.block_table[b, tok // 16]
            kt = torch.tensor(_f(pp.k_cache[pages, tok % 16])).permute(1, 0, 2)[None]  # 1, Hkv, L, D
            vt = torch.tensor(_f(pp.v_cache[pages, tok % 16])).permute(1, 0, 2)[None]
            qt = torch.tensor(_f(pp.q[r0:r0 + n])).permute(1, 0, 2)[None]  # 1, Hq, n, D
            pos = np.arange(L - n, L)[:, None]
            j = np.arange(L)[None, :]
            m = j <= pos
            if window > 0:
                m &= (pos - j) < window
            mask = torch.tensor(m)
            to = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask, scale=pp.scale,
                                                                  enable_gqa=True)
            G = pp.Hq // pp.Hkv
            sc = (qt @ kt.repeat_interleave(G, dim=1).transpose(-1, -2)) * pp.scale
            tl = torch.logsumexp(sc.masked_fill(~mask, float("-inf")), dim=-1)
            _close(o[r0:r0 + n], to[0].permute(1, 0, 2).numpy(), 1e-12, f"prefill_paged o vs torch (W={window})")
            _close(lse[:, r0:r0 + n], tl[0].numpy(), 1e-12, f"prefill_paged lse vs torch (W={window})")
    # one new token per request is the decode
    pd = synth.paged_from_lengths([5, 16, 33], 8, 2, 32, page_size=16, num_pages=8, seed=22, max_pages=3)
    od, ld = orc.decode_paged(pd.q, pd.k_cache, pd.v_cache, pd.block_table, pd.seq_lens, pd.scale)
    cu = np.arange(pd.B + 1, dtype=np.int32)
    op, lp = orc.prefill_paged(pd.q, pd.k_cache, pd.v_cache, pd.block_table, pd.seq_lens, cu, pd.scale)
    _close(op, od, 0, "prefill_paged with one token = decode (o)")
    _close(lp.T, ld, 0, "prefill_paged with one token = decode (lse)")
    # relabelling the pool changes nothing
    pp = synth.prefill_paged_from_lengths([40, 23], [40, 7], 4, 1, 16, page_size=16, seed=23)
    o, lse = orc.prefill_paged(pp.q, pp.k_cache, pp.v_cache, pp.block_table, pp.seq_lens, pp.cu_q, pp.scale)
    perm = np.random.default_rng(6).permutation(pp.num_pages)
    inv = np.argsort(perm)
    bt2 = np.where(pp.block_table >= 0, perm[np.maximum(pp.block_table, 0)], -1).astype(np.int32)
    o2, l2 = orc.prefill_paged(pp.q, pp.k_cache[inv], pp.v_cache[inv], bt2, pp.seq_lens, pp.cu_q, pp.scale)
    _close(o2, o, 0, "prefill_paged page relabelling (o)")
    _close(l2, lse, 0, "prefill_paged page relabelling (lse)")


def _sdpa_part(q, k, v, scale, mask):
    """torch fp64 attention of q [1,H,S,D] over the keys k, v [1,H,n,D] that `mask` [S,n] allows:
    (o [S,H,D], lse [H,S]); rows with no allowed key give o = 0, lse = -inf."""
    sc = (q @ k.transpose(-1, -2)) * scale
    sc = sc.masked_fill(~mask, float("-inf"))
    lse = torch.logsumexp(sc, dim=-1)  # 1, H, S
    p = torch.exp(sc - torch.where(torch.isfinite(lse), lse, torch.zeros_like(lse))[..., None])
    o = p @ v
    return o[0].permute(1, 0, 2).numpy(), lse[0].numpy()


def pin_merge_lse(orc):
    """Merging attention results over disjoint key chunks reproduces torch fp64 attention over
    all keys (non-causal and causal, so some chunks have rows with no allowed key); closed forms:
    one part is the identity, two equal parts keep o and add ln 2 to lse, lse of order 1e4 does
    not overflow, all-empty rows give o = 0 / lse = -inf; the order of the parts does not matter."""
    rng = np.random.default_rng(31)
    S, H, D = 23, 3, 16
    q = torch.tensor(_f(synth.normal_bf16(31, 1, (S, H, D)))).permute(1, 0, 2)[None]
    k = torch.tensor(_f(synth.normal_bf16(31, 2, (S, H, D)))).permute(1, 0, 2)[None]
    v = torch.tensor(_f(synth.normal_bf16(31, 3, (S, H, D)))).permute(1, 0, 2)[None]
    cuts = [0, 5, 6, 6, 17, 23]  # chunks of 5, 1, 0, 11, 6 keys
    for causal in (False, True):
        i = np.arange(S)[:, None]
        full = (np.arange(S)[None, :] <= i) if causal else np.ones((S, S), bool)
        ref_o, ref_l = _sdpa_part(q, k, v, 0.37, torch.tensor(full))
        parts_o, parts_l = [], []
        for a, b in zip(cuts[:-1], cuts[1:]):
            po, pl = _sdpa_part(q, k[:, :, a:b], v[:, :, a:b], 0.37, torch.tensor(full[:, a:b]))
            parts_o.append(po)
            parts_l.append(pl)
        po, pl = np.stack(parts_o), np.stack(parts_l)
        o, lse = orc.merge_lse(po, pl)
        _close(o, ref_o, 1e-12, f"merge of key chunks = attention over all keys (o, causal={causal})")
        _close(lse, ref_l, 1e-12, f"merge of key chunks = attention over all keys (lse, causal={causal})")
        perm = rng.permutation(len(parts_o))
        o2, l2 = orc.merge_lse(po[perm], pl[perm])
        _close(o2, o, 1e-13, "merge is independent of the order of the parts (o)")
        _close(l2, lse, 1e-13, "merge is independent of the order of the parts (lse)")
    x = rng.standard_normal((1, 4, 2, 8))
    lx = rng.standard_normal((1, 2, 4)) * 3
    o, lse = orc.merge_lse(x, lx)
    _close(o, x[0], 0, "one part is the identity (o)")
    _close(lse, lx[0], 0, "one part is the identity (lse)")
    o, lse = orc.merge_lse(np.stack([x[0], x[0]]), np.stack([lx[0], lx[0]]))
    _close(o, x[0], 1e-15, "two equal parts keep o")
    _close(lse, lx[0] + np.log(2.0), 1e-14, "two equal parts add ln 2 to lse")
    big = np.stack([np.full((2, 4), 1.0e4), np.full((2, 4), 1.0e4 - 1.0)])
    y = rng.standard_normal((2, 4, 2, 8))
    o, lse = orc.merge_lse(y, big)
    w1 = 1.0 / (1.0 + np.exp(-1.0))
    _close(lse, np.full((2, 4), 1.0e4 + np.log1p(np.exp(-1.0))), 1e-11, "lse of order 1e4 merges without overflow")
    _close(o, w1 * y[0] + (1 - w1) * y[1], 1e-11, "lse of order 1e4 (one ulp of lse is 2e-12): weights 1/(1+e^-1) and e^-1/(1+e^-1)")
    empty = np.full((3, 2, 4), -np.inf)
    o, lse = orc.merge_lse(rng.standard_normal((3, 4, 2, 8)), empty)
    assert np.all(o == 0) and np.all(np.isneginf(lse)), "rows with no key in any part: o = 0, lse = -inf"


def pin_golden(orc):
    for name in ("two_token_causal.json", "three_token_window2.json"):
        g = json.load(open(os.path.join(GOLDEN, name)))
        q = _bf16_exact(np.array(g["q"], float)[None, :, None, :])
        k = _bf16_exact(np.array(g["k"], float)[None, :, None, :])
        v = _bf16_exact(np.array(g["v"], float)[None, :, None, :])
        o, lse = orc.fwd(q, k, v, g["scale"], g["causal"], g["window"])
        _close(o[0, :, 0, :], np.array(g["o"], float), 1e-14, f"{name} o")
        _close(lse[0, 0], np.array(g["lse"], float), 1e-14, f"{name} lse")
        if "dO" in g:
            do = _bf16_exact(np.array(g["dO"], float)[None, :, None, :])
            dq, dk, dv, *_ = orc.bwd(q, k, v, do, g["scale"], g["causal"], g["window"])
            _close(dq[0, :, 0, :], np.array(g["dq"], float), 1e-14, f"{name} dq")
            _close(dk[0, :, 0, :], np.array(g["dk"], float), 1e-14, f"{name} dk")
            _close(dv[0, :, 0, :], np.array(g["dv"], float), 1e-14, f"{name} dv")


def pin_sampled_rows(orc):
    """The row-sampling entry points agree with the whole-problem ones."""
    p = synth.dense(2, 4, 2, 29, 16, 0, seed=16)
    for window in (0, 6):
        o, lse = orc.fwd(p.q, p.k, p.v, p.scale, 1, window)
        dq, dk, dv, *_ = orc.bwd(p.q, p.k, p.v, p.do, p.scale, 1, window)
        rows = np.array([[0, 0, 0], [1, 3, 28], [0, 2, 13], [1, 1, 5]], np.int64)
        ro, rl = orc.fwd_rows(p.q, p.k, p.v, rows, p.scale, 1, window)
        rdq = orc.dq_rows(p.q, p.k, p.v, p.do, rows, p.scale, 1, window)
        for r, (b, h, i) in enumerate(rows):
            _close(ro[r], o[b, i, h], 1e-13, "fwd_rows")
            _close(rl[r], lse[b, h, i], 1e-13, "fwd_rows lse")
            _close(rdq[r], dq[b, i, h], 1e-12, "dq_rows")
        krows = np.array([[0, 0, 0], [1, 1, 28], [0, 1, 10], [1, 0, 3]], np.int64)
        rdk, rdv = orc.dkv_rows(p.q, p.k, p.v, p.do, krows, p.scale, 1, window)
        for r, (b, g, j) in enumerate(krows):
            _close(rdk[r], dk[b, j, g], 1e-12, "dkv_rows dk")
            _close(rdv[r], dv[b, j, g], 1e-12, "dkv_rows dv")
    # packed sequences: rows are (sequence, head, index within the sequence)
    vp = synth.varlen_from_lengths([7, 19, 3], 4, 2, 16, 0, seed=17)
    o, lse = orc.fwd_varlen(vp.q, vp.k, vp.v, vp.cu_seqlens, vp.scale)
    dq, dk, dv, _ = orc.bwd_varlen(vp.q, vp.k, vp.v, vp.do, vp.cu_seqlens, vp.scale)
    rows = np.array([[0, 1, 6], [1, 3, 0], [1, 2, 18], [2, 0, 2]], np.int64)
    ro, rl = orc.fwd_rows(vp.q, vp.k, vp.v, rows, vp.scale, cu_seqlens=vp.cu_seqlens)
    rdq = orc.dq_rows(vp.q, vp.k, vp.v, vp.do, rows, vp.scale, cu_seqlens=vp.cu_seqlens)
    krows = np.array([[0, 0, 6], [1, 1, 0], [1, 0, 18], [2, 1, 1]], np.int64)
    rdk, rdv = orc.dkv_rows(vp.q, vp.k, vp.v, vp.do, krows, vp.scale, cu_seqlens=vp.cu_seqlens)
    for r, (s, h, i) in enumerate(rows):
        t = vp.cu_seqlens[s] + i
        _close(ro[r], o[t, h], 1e-13, "varlen fwd_rows")
        _close(rl[r], lse[h, t], 1e-13, "varlen fwd_rows lse")
        _close(rdq[r], dq[t, h], 1e-12, "varlen dq_rows")
    for r, (s, g, j) in enumerate(krows):
        t = vp.cu_seqlens[s] + j
        _close(rdk[r], dk[t, g], 1e-12, "varlen dkv_rows dk")
        _close(rdv[r], dv[t, g], 1e-12, "varlen dkv_rows dv")


ALL_PINS = [pin_golden, pin_torch_forward, pin_torch_backward, pin_finite_differences, pin_closed_forms,
            pin_invariants, pin_varlen, pin_paged, pin_prefill_paged, pin_merge_lse, pin_sampled_rows]
