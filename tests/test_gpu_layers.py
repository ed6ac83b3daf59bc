"""GPU parity of the multi-layer reverse replay (response_replay_gb300/layers.py): three
layers' prompts captured under one page table, each layer's forward and backward
checked against the fp64 oracle on that layer's own pools, the backward run last layer
first with dK / dV allocated per layer; a second backward over the same keys adds."""
import numpy as np
import pytest
import torch

import oracle
from parity_util import TOL_GRAD, TOL_LSE, TOL_O, rel_err, u16
from response_replay_gb300 import binding as B
from response_replay_gb300 import layers as L
from response_replay_gb300 import synthetic as syn
from response_replay_gb300 import torch_api as api

pytestmark = pytest.mark.gpu


def test_three_layers_reverse_replay(cuda):
    P, R, hq, hkv, ps, splits, nl = 2000, 300, 8, 2, 64, 5, 3
    scale = 128 ** -0.5
    pr0 = syn.make_prompt(P, hkv, 128, ps, 900, cuda, extra_pages=2, sharp=True)
    lc = L.LayeredKVCache(nl, pr0.num_pages, pr0.page_table, ps, hkv, P, device=cuda,
                          fill=float("nan"))
    saved, d_os = [], []
    for l in range(nl):
        pr = syn.make_prompt(P, hkv, 128, ps, 900 + 7 * l, cuda, sharp=True)
        lc.capture(l, pr.k[:P].contiguous(), pr.v[:P].contiguous())
        br = syn.make_branch(R, hq, hkv, 128, 950 + l, cuda, sharp=True)
        o, lse = api.replay_fwd(lc[l], br.q, br.k, br.v, scale, splits)
        saved.append((br.q, br.k, br.v, o, lse))
        d_os.append(br.d_o)
    got = {}

    def consume(l, dq, dk, dv):
        got[l] = (dq.cpu().numpy(), dk.cpu().numpy(), dv.cpu().numpy())

    order = []

    def upstream(l):
        order.append(l)
        return d_os[l]

    L.reverse_replay_bwd(lc, saved, upstream, consume, scale, splits)
    torch.cuda.synchronize()
    assert B.ls_last_device_error(0) == B.LS_OK
    assert order == [2, 1, 0]
    pt = pr0.page_table.cpu().numpy()
    for l in range(nl):
        q, k, v, o, lse = saved[l]
        pb = oracle.AttnProblem(u16(lc.k_pools[l]), u16(lc.v_pools[l]), pt, P, u16(q), u16(k),
                                u16(v), scale, splits)
        o_ref, lse_ref = oracle.attn_fwd(pb)
        assert rel_err(o.float().cpu().numpy(), o_ref) <= TOL_O, l
        assert float(np.abs(lse.cpu().numpy() - lse_ref).max()) <= TOL_LSE, l
        refs = oracle.attn_bwd(pb, u16(d_os[l]))
        for name, x, ref in zip(("dq", "dk", "dv"), got[l], refs):
            assert rel_err(x, ref) <= TOL_GRAD, (l, name)

    # a second backward over layer 1's keys adds to its dK / dV (the oracle is linear
    # in dO, so the sum of the two oracle gradients is the reference)
    q, k, v, o, lse = saved[1]
    g = L.KVGradPages(R, hkv, cuda)
    g.backward(lc[1], q, k, v, o, lse, d_os[1], scale, splits)
    d_o2 = syn.make_branch(R, hq, hkv, 128, 977, cuda, sharp=True).d_o
    g.backward(lc[1], q, k, v, o, lse, d_o2, scale, splits)
    torch.cuda.synchronize()
    pb = oracle.AttnProblem(u16(lc.k_pools[1]), u16(lc.v_pools[1]), pt, P, u16(q), u16(k),
                            u16(v), scale, splits)
    _, dk1, dv1 = oracle.attn_bwd(pb, u16(d_os[1]))
    _, dk2, dv2 = oracle.attn_bwd(pb, u16(d_o2))
    assert g.touches == 2
    assert rel_err(g.dk.cpu().numpy(), dk1 + dk2) <= TOL_GRAD
    assert rel_err(g.dv.cpu().numpy(), dv1 + dv2) <= TOL_GRAD


def test_streamed_layers_match_resident_layers(cuda):
    """Three layers' prompt pages captured into pinned host memory and streamed through
    the two-slot GPU page cache one layer ahead: forward (layers in order) and backward
    (last layer first) bit-identical to the same layers held in GPU memory, one layer
    against the oracle."""
    P, R, hq, hkv, ps, splits, nl = 3000, 200, 8, 2, 64, 5, 3
    scale = 128 ** -0.5
    pr0 = syn.make_prompt(P, hkv, 128, ps, 700, cuda, extra_pages=2, sharp=True)
    res = L.LayeredKVCache(nl, pr0.num_pages, pr0.page_table, ps, hkv, P, device=cuda)
    st = L.StreamedLayers(nl, pr0.num_pages, pr0.page_table, ps, hkv, P, device=cuda)
    brs = []
    for l in range(nl):
        pr = syn.make_prompt(P, hkv, 128, ps, 700 + 3 * l, cuda, sharp=True)
        res.capture(l, pr.k[:P].contiguous(), pr.v[:P].contiguous())
        st.capture(l, pr.k[:P].contiguous(), pr.v[:P].contiguous())
        brs.append(syn.make_branch(R, hq, hkv, 128, 720 + l, cuda, sharp=True))
    outs_r, outs_s = [], []
    st.prefetch(0)
    for l in range(nl):
        c = st.cache(l)
        if l + 1 < nl:
            st.prefetch(l + 1)
        br = brs[l]
        outs_s.append(api.replay_fwd(c, br.q, br.k, br.v, scale, splits))
        st.release(l)
        outs_r.append(api.replay_fwd(res[l], br.q, br.k, br.v, scale, splits))
    st.prefetch(nl - 1)
    for l in reversed(range(nl)):
        c = st.cache(l)
        if l > 0:
            st.prefetch(l - 1)
        br = brs[l]
        o, lse = outs_s[l]
        g_s = api.replay_bwd(c, br.q, br.k, br.v, o, lse, br.d_o, scale, splits)
        st.release(l)
        g_r = api.replay_bwd(res[l], br.q, br.k, br.v, o, lse, br.d_o, scale, splits)
        torch.cuda.synchronize()
        for a, b in zip(g_s, g_r):
            assert torch.equal(a, b), l
    torch.cuda.synchronize()
    assert B.ls_last_device_error(0) == B.LS_OK
    for (o_s, l_s), (o_r, l_r) in zip(outs_s, outs_r):
        assert torch.equal(o_s, o_r) and torch.equal(l_s, l_r)
    assert not st.host[1].k_pool.is_cuda and st.host[1].k_pool.is_pinned()
    pt = pr0.page_table.cpu().numpy()
    pb = oracle.AttnProblem(u16(st.host[1].k_pool), u16(st.host[1].v_pool), pt, P,
                            u16(brs[1].q), u16(brs[1].k), u16(brs[1].v), scale, splits)
    o_ref, lse_ref = oracle.attn_fwd(pb)
    assert rel_err(outs_s[1][0].float().cpu().numpy(), o_ref) <= TOL_O
    assert float(np.abs(outs_s[1][1].cpu().numpy() - lse_ref).max()) <= TOL_LSE
