"""GPU parity of the batched forward (ls_replay_attn_fwd_members): several responses of
equal length over one captured prompt in one launch.  Every member is checked against
the fp64 oracle run on that member alone, and against the one-member call."""
import numpy as np
import pytest
import torch

import oracle
from parity_util import TOL_LSE, TOL_O, rel_err, u16
from response_replay_gb300 import synthetic as syn
from response_replay_gb300 import torch_api as api
from response_replay_gb300 import binding as B

pytestmark = pytest.mark.gpu


def make_members(P, R, hq, hkv, ps, M, seed, device, sharp=True):
    pr = syn.make_prompt(max(P, 1), hkv, syn.HEAD_DIM, ps, seed, device, extra_pages=2,
                         sharp=sharp)
    if P == 0:
        pr.page_table = pr.page_table[:0]
    cache = api.PagedKVCache(pr.num_pages, pr.page_table, ps, hkv, P, device=device,
                             fill=float("nan"))
    if P > 0:
        cache.capture(pr.k[:P].contiguous(), pr.v[:P].contiguous())
    brs = [syn.make_branch(R, hq, hkv, syn.HEAD_DIM, seed + 1 + m, device, sharp=sharp)
           for m in range(M)]
    q = torch.stack([b.q for b in brs]).contiguous()
    k = torch.stack([b.k for b in brs]).contiguous()
    v = torch.stack([b.v for b in brs]).contiguous()
    return cache, q, k, v


def oracle_member(cache, P, q, k, v, m, scale, splits):
    torch.cuda.synchronize()
    pt = cache.page_table.cpu().numpy() if P > 0 else np.zeros(1, np.int32)
    pb = oracle.AttnProblem(u16(cache.k_pool), u16(cache.v_pool), pt, P, u16(q[m]), u16(k[m]),
                            u16(v[m]), scale, splits)
    return oracle.attn_fwd(pb)


# Short responses (grouped-query packing) put the members' tokens into shared tiles: a
# tile holds floor(128 / g) tokens of consecutive members, so member boundaries fall
# inside tiles (R = 16, g = 6), several members share one tile (R = 1), a unit spans 32
# one-token members (g = 8), units straddle members (R = 77), P = 0.  Long responses
# (R >= 256) and g = 1 keep units per member (two 128-token tiles, ragged last unit).
# One member is the one-response kernel.  More splits than tiles included.
@pytest.mark.parametrize("P,R,hq,hkv,ps,splits,M", [
    (3000, 16, 24, 4, 64, 5, 8),
    (1000, 1, 6, 1, 16, 3, 5),
    (1500, 1, 16, 2, 64, 3, 100),
    (5000, 77, 12, 2, 128, 7, 3),
    (2000, 300, 6, 2, 64, 4, 3),
    (0, 50, 4, 1, 64, 2, 4),
    (4096, 130, 5, 5, 64, 1000, 2),
    (777, 255, 24, 3, 32, 4, 1),
])
def test_members_match_oracle_per_member(cuda, P, R, hq, hkv, ps, splits, M):
    scale = syn.HEAD_DIM ** -0.5
    cache, q, k, v = make_members(P, R, hq, hkv, ps, M, P * 3 + R + M, cuda)
    o, lse = api.replay_fwd_members(cache, q, k, v, scale, splits)
    assert B.ls_last_device_error(0) == B.LS_OK
    for m in range(M):
        o_ref, lse_ref = oracle_member(cache, P, q, k, v, m, scale, splits)
        o_g, l_g = o[m].float().cpu().numpy(), lse[m].cpu().numpy()
        assert np.isfinite(o_g).all() and np.isfinite(l_g).all()
        assert rel_err(o_g, o_ref) <= TOL_O, m
        assert float(np.abs(l_g - lse_ref).max()) <= TOL_LSE, m
        # the one-member call on member m's slices: same arithmetic, other split points
        o1, l1 = api.replay_fwd(cache, q[m], k[m], v[m], scale, splits)
        assert (o1.float() - o[m].float()).abs().max().item() <= 2 ** -7
        assert (l1 - lse[m]).abs().max().item() <= 1e-5


@pytest.mark.parametrize("R", [5, 45, 300])
def test_members_isolated(cuda, R):
    """Member 1's response keys and values are huge (finite): they would dominate every
    row that could see them, yet members 0 and 2 match the oracle run on their own
    inputs.  R = 5 and 45 pack the members into shared tiles, R = 300 gives each member
    its own units."""
    P, hq, hkv, ps, splits, M = 2048, 8, 2, 64, 3, 3
    scale = syn.HEAD_DIM ** -0.5
    cache, q, k, v = make_members(P, R, hq, hkv, ps, M, 77, cuda)
    k[1].fill_(30.0)
    v[1].fill_(1.0e4)
    o, lse = api.replay_fwd_members(cache, q, k, v, scale, splits)
    for m in (0, 2):
        o_ref, lse_ref = oracle_member(cache, P, q, k, v, m, scale, splits)
        assert rel_err(o[m].float().cpu().numpy(), o_ref) <= TOL_O
        assert float(np.abs(lse[m].cpu().numpy() - lse_ref).max()) <= TOL_LSE


def test_members_zero_is_noop_and_bad_args(cuda):
    cache, q, k, v = make_members(256, 8, 4, 2, 64, 2, 5, cuda)
    scale = syn.HEAD_DIM ** -0.5
    o = torch.full_like(q, 3.0)
    lse = torch.full(q.shape[:3], 3.0, dtype=torch.float32, device=cuda)
    B.ls_replay_attn_fwd_members(cache.struct, q.data_ptr(), k.data_ptr(), v.data_ptr(), 8, 0,
                                 4, scale, 2, o.data_ptr(), lse.data_ptr(), 0, 0)
    torch.cuda.synchronize()
    assert (o.float() == 3.0).all() and (lse == 3.0).all()
    with pytest.raises(B.LongstrawError):
        B.ls_replay_attn_fwd_members(cache.struct, q.data_ptr(), k.data_ptr(), v.data_ptr(), 8,
                                     -1, 4, scale, 2, o.data_ptr(), lse.data_ptr(), 0, 0)


def test_members_full_prompt_short_responses_sampled(cuda):
    """The 2,097,152-position prompt with 8 members of 16 tokens (the pre-step scoring
    shape): sampled rows of every member against the oracle."""
    w = syn.WORKLOADS["p2m"]
    seed = syn.seed_of("p2m")
    pr = syn.make_prompt(w.P, w.hkv, 128, w.page_size, seed, cuda)
    cache = api.PagedKVCache(pr.num_pages, pr.page_table, w.page_size, w.hkv, w.P, device=cuda)
    cache.capture(pr.k, pr.v)
    del pr
    M, R = 8, 16
    brs = [syn.make_branch(R, w.hq, w.hkv, 128, seed + 1 + m, cuda) for m in range(M)]
    q = torch.stack([b.q for b in brs]).contiguous()
    k = torch.stack([b.k for b in brs]).contiguous()
    v = torch.stack([b.v for b in brs]).contiguous()
    scale = 128 ** -0.5
    o, lse = api.replay_fwd_members(cache, q, k, v, scale, w.num_splits)
    torch.cuda.synchronize()
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
    rng = np.random.default_rng(seed)
    pt = cache.page_table.cpu().numpy()
    kp, vp = u16(cache.k_pool), u16(cache.v_pool)
    for m in (0, 3, 7):
        pb = oracle.AttnProblem(kp, vp, pt, w.P, u16(q[m]), u16(k[m]), u16(v[m]), scale,
                                w.num_splits)
        ts = np.array([0, R - 1, int(rng.integers(0, R))], dtype=np.int32)
        hs = rng.integers(0, w.hq, 3).astype(np.int32)
        o_ref, lse_ref = oracle.attn_fwd_rows(pb, ts, hs)
        o_g = o[m].float().cpu().numpy()[ts, hs]
        assert float(np.abs(o_g - o_ref).max() / np.abs(o_ref).max()) <= TOL_O
        assert float(np.abs(lse[m].cpu().numpy()[ts, hs] - lse_ref).max()) <= TOL_LSE
