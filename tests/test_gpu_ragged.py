"""Ragged members replayed in one forward and one backward launch
(ls_replay_attn_fwd_ragged / ls_replay_attn_bwd_ragged): every member is checked
against the fp64 oracle run on that member's slices alone, and against the
one-response calls.  Members' lengths are empty, one token, short (the grouped-query
packed layout), long and not multiples of the tile."""
import numpy as np
import pytest
import torch

import oracle
from parity_util import TOL_GRAD, TOL_LSE, TOL_O, rel_err, u16
from response_replay_gb300 import binding as B
from response_replay_gb300 import synthetic as syn
from response_replay_gb300 import torch_api as api

pytestmark = pytest.mark.gpu


def make(P, lens, hq, hkv, ps, seed, device):
    pr = syn.make_prompt(max(P, 1), hkv, 128, ps, seed, device, extra_pages=2, sharp=True)
    if P == 0:
        pr.page_table = pr.page_table[:0]
    cache = api.PagedKVCache(pr.num_pages, pr.page_table, ps, hkv, P, device=device,
                             fill=float("nan"))
    if P > 0:
        cache.capture(pr.k[:P].contiguous(), pr.v[:P].contiguous())
    br = syn.make_branch(int(sum(lens)), hq, hkv, 128, seed + 1, device, sharp=True)
    return cache, br


def member_problem(cache, P, br, s, e, scale, splits):
    torch.cuda.synchronize()
    pt = cache.page_table.cpu().numpy() if P > 0 else np.zeros(1, np.int32)
    return oracle.AttnProblem(u16(cache.k_pool), u16(cache.v_pool), pt, P, u16(br.q[s:e]),
                              u16(br.k[s:e]), u16(br.v[s:e]), scale, splits)


@pytest.mark.parametrize("P,lens,hq,hkv,ps,splits", [
    (3000, [300, 17, 1000, 1, 64, 0, 255], 12, 2, 64, 5),
    (0, [130, 5, 260], 6, 3, 64, 2),
    (2000, [16, 3, 40, 21], 12, 2, 32, 3),          # 80 tokens: grouped-query packing
    (777, [129, 128, 127, 300], 8, 1, 16, 1000),
])
def test_ragged_members_match_oracle(cuda, P, lens, hq, hkv, ps, splits):
    scale = 128 ** -0.5
    cache, br = make(P, lens, hq, hkv, ps, 500 + P + len(lens), cuda)
    o, lse = api.replay_fwd_ragged(cache, br.q, br.k, br.v, lens, scale, splits)
    dq, dk, dv = api.replay_bwd_ragged(cache, br.q, br.k, br.v, o, lse, br.d_o, lens, scale,
                                       splits)
    torch.cuda.synchronize()
    assert B.ls_last_device_error(0) == B.LS_OK
    off = np.concatenate([[0], np.cumsum(lens)]).astype(int)
    for m, R in enumerate(lens):
        s, e = off[m], off[m + 1]
        if R == 0:
            continue
        pb = member_problem(cache, P, br, s, e, scale, splits)
        o_ref, lse_ref = oracle.attn_fwd(pb)
        assert rel_err(o[s:e].float().cpu().numpy(), o_ref) <= TOL_O, m
        assert float(np.abs(lse[s:e].cpu().numpy() - lse_ref).max()) <= TOL_LSE, m
        dq_ref, dk_ref, dv_ref = oracle.attn_bwd(pb, u16(br.d_o[s:e]))
        for name, x, ref in (("dq", dq, dq_ref), ("dk", dk, dk_ref), ("dv", dv, dv_ref)):
            err = rel_err(x[s:e].cpu().numpy(), ref)
            assert err <= TOL_GRAD, (m, name, err)
        # the one-response calls on the member's slices
        o1, l1 = api.replay_fwd(cache, br.q[s:e], br.k[s:e], br.v[s:e], scale, splits)
        assert (o1.float() - o[s:e].float()).abs().max().item() <= 2 ** -7
        assert (l1 - lse[s:e]).abs().max().item() <= 1e-5


def test_ragged_cycle_of_the_reuse_workload(cuda):
    """One cycle of the 4,194,304-position workload's ragged lengths (8 members, 959 to
    7,773 tokens, 33,371 in all) over a 4,096-position prompt: sampled rows of every
    member and its last keys against the oracle; accumulate adds."""
    w = syn.WORKLOADS["p4m_reuse"]
    lens = list(w.R[:8])
    P, scale, splits = 4096, 128 ** -0.5, 4
    cache, br = make(P, lens, w.hq, w.hkv, 256, 77, cuda)
    o, lse = api.replay_fwd_ragged(cache, br.q, br.k, br.v, lens, scale, splits)
    dq, dk, dv = api.replay_bwd_ragged(cache, br.q, br.k, br.v, o, lse, br.d_o, lens, scale,
                                       splits)
    torch.cuda.synchronize()
    off = np.concatenate([[0], np.cumsum(lens)]).astype(int)
    rng = np.random.default_rng(3)
    for m, R in enumerate(lens):
        s, e = off[m], off[m + 1]
        pb = member_problem(cache, P, br, s, e, scale, splits)
        ts = np.array([0, R - 1] + list(rng.integers(0, R, 3)), np.int32)
        hs = rng.integers(0, w.hq, len(ts)).astype(np.int32)
        o_ref, lse_ref = oracle.attn_fwd_rows(pb, ts, hs)
        assert rel_err(o[s:e].float().cpu().numpy()[ts, hs], o_ref) <= TOL_O, m
        assert float(np.abs(lse[s:e].cpu().numpy()[ts, hs] - lse_ref).max()) <= TOL_LSE, m
        d_o = u16(br.d_o[s:e])
        dq_ref = oracle.attn_bwd_dq_rows(pb, d_o, ts, hs)
        assert rel_err(dq[s:e].cpu().numpy()[ts, hs], dq_ref) <= TOL_GRAD, m
        js = np.repeat(np.array([R - 1], np.int32), w.hkv)
        kv = np.arange(w.hkv, dtype=np.int32)
        dk_ref, dv_ref = oracle.attn_bwd_dkdv_keys(pb, d_o, js, kv)
        assert rel_err(dk[s:e].cpu().numpy()[js, kv], dk_ref) <= TOL_GRAD, m
        assert rel_err(dv[s:e].cpu().numpy()[js, kv], dv_ref) <= TOL_GRAD, m
    g2 = api.replay_bwd_ragged(cache, br.q, br.k, br.v, o, lse, br.d_o, lens, scale, splits,
                               dq=dq.clone(), dk=dk.clone(), dv=dv.clone(), accumulate=True)
    for a, b in zip((dq, dk, dv), g2):
        torch.testing.assert_close(b, 2 * a, rtol=1e-6, atol=1e-7)
    assert B.ls_last_device_error(0) == B.LS_OK


def test_ragged_argument_checks(cuda):
    cache, br = make(256, [8, 8], 4, 2, 64, 9, cuda)
    for bad in ([], [-1, 17], [1] * 65):  # no member, a negative length, too many members
        with pytest.raises(B.LongstrawError):
            B.ls_replay_attn_fwd_ragged_workspace(cache.struct, bad, 4, 2)
        with pytest.raises(B.LongstrawError):
            B.ls_replay_attn_bwd_ragged_workspace(cache.struct, bad, 4, 2)
    with pytest.raises(ValueError):
        api.replay_fwd_ragged(cache, br.q, br.k, br.v, [8, 9], 0.1, 2)
