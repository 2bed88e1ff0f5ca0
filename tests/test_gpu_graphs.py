"""The C ABI under CUDA-graph capture: calls captured once and replayed, as a serving loop or a
training step does. The decode call launches two kernels with programmatic stream
serialisation, which a capture must keep as programmatic edges; the forward and backward use
tensor maps encoded on the host at capture time and cluster launches. Every replay must give the
oracle's result."""
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


def capture(fns):
    """Warm every call up on a side stream, then capture them in order into one graph."""
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for f in fns:
            f()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for f in fns:
            f()
    return g


def test_decode_graph_two_pools(orc):
    """Two decode calls over two different KV pools (and two output buffers) in one graph,
    replayed three times; both results match the oracle after every replay."""
    pa = synth.paged_from_lengths([900, 1, 0, 513, 40, 2048], 32, 8, 128, num_pages=512, seed=5, max_pages=128)
    pb = synth.paged_from_lengths([900, 1, 0, 513, 40, 2048], 32, 8, 128, num_pages=512, seed=6, max_pages=128)
    bta, btb = torch.from_numpy(pa.block_table).cuda(), torch.from_numpy(pb.block_table).cuda()
    sl = torch.from_numpy(pa.seq_lens).cuda()
    qa, ka, va = to_dev(pa.q), to_dev(pa.k_cache), to_dev(pa.v_cache)
    qb, kb, vb = to_dev(pb.q), to_dev(pb.k_cache), to_dev(pb.v_cache)
    oa, ob = torch.empty_like(qa), torch.empty_like(qb)
    la = torch.empty((pa.B, pa.Hq), dtype=torch.float32, device="cuda")
    lb = torch.empty_like(la)
    ws = torch.empty(attn.attn_workspace_size(attn.ATTN_OP_DECODE_PAGED, pa.B, pa.Hq, pa.Hkv, 0, pa.D),
                     dtype=torch.uint8, device="cuda")
    g = capture([lambda: attn.attn_decode_paged(qa, ka, va, bta, sl, oa, la, scale=pa.scale, workspace=ws),
                 lambda: attn.attn_decode_paged(qb, kb, vb, btb, sl, ob, lb, scale=pb.scale, workspace=ws)])
    ra = orc.decode_paged(pa.q, pa.k_cache, pa.v_cache, pa.block_table, pa.seq_lens, pa.scale)
    rb = orc.decode_paged(pb.q, pb.k_cache, pb.v_cache, pb.block_table, pb.seq_lens, pb.scale)
    for _ in range(3):
        oa.zero_(), ob.zero_(), la.zero_(), lb.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert attn.attn_get_device_status() == 0
        check("o pool a", to_np(oa), ra[0])
        check_lse("lse pool a", to_np(la), ra[1])
        check("o pool b", to_np(ob), rb[0])
        check_lse("lse pool b", to_np(lb), rb[1])


@pytest.mark.parametrize("D,window", [(512, 0), (256, 100), (128, 0)])
def test_forward_backward_graph(orc, D, window):
    """One forward + backward captured and replayed twice on new inputs copied into the
    captured buffers: the second replay sees the second input set."""
    p1 = synth.dense(1, 4, 2, 300, D, window, seed=D)
    p2 = synth.dense(1, 4, 2, 300, D, window, seed=D + 1)
    q, k, v, do = (to_dev(x) for x in (p1.q, p1.k, p1.v, p1.do))
    o = torch.empty_like(q)
    lse = torch.empty((1, 4, 300), dtype=torch.float32, device="cuda")
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(attn.attn_workspace_size(attn.ATTN_OP_BWD, 1, 4, 2, 300, D), dtype=torch.uint8, device="cuda")
    g = capture([lambda: attn.attn_fwd(q, k, v, o, lse, window=window, scale=p1.scale),
                 lambda: attn.attn_bwd(q, k, v, o, lse, do, dq, dk, dv, window=window, scale=p1.scale, workspace=ws)])
    for p in (p1, p2):
        for dst, src in ((q, p.q), (k, p.k), (v, p.v), (do, p.do)):
            dst.copy_(to_dev(src))
        g.replay()
        torch.cuda.synchronize()
        assert attn.attn_get_device_status() == 0
        ro, rl = orc.fwd(p.q, p.k, p.v, p.scale, 1, window)
        rdq, rdk, rdv, *_ = orc.bwd(p.q, p.k, p.v, p.do, p.scale, 1, window)
        check("o", to_np(o), ro)
        check_lse("lse", to_np(lse), rl)
        check("dq", to_np(dq), rdq)
        check("dk", to_np(dk), rdk)
        check("dv", to_np(dv), rdv)
