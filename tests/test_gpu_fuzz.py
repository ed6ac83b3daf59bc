"""Seeded random shapes for replay attention, forward and backward, against the fp64
oracle: prompt lengths from 0 up, response lengths from 1 token to a few tiles, every
grouped-query ratio up to 8, page sizes 16-256, split counts from 1 to more than the
prompt has tiles, scores of unit spread or near-uniform, ragged member lists with
empty members, and latent (MLA-style) replays, forward and backward, with 1-128 heads
and 32-4096-row pages.
The shapes are drawn once from a fixed seed, so every run checks the same cases; each is
small enough for the oracle to finish in about a second."""
import numpy as np
import pytest
import torch

import oracle
from parity_util import TOL_GRAD, TOL_LSE, TOL_O, Case, rel_err, u16
from response_replay_gb300 import binding as B
from response_replay_gb300 import torch_api as api

pytestmark = pytest.mark.gpu

MAX_WORK = 6_000_000  # R * (P + R) * Hq per case: about a second of oracle time


def _draw_single(n, seed):
    rng = np.random.default_rng(seed)
    cases = []
    while len(cases) < n:
        hkv = int(rng.choice([1, 2, 3, 4]))
        g = int(rng.choice([1, 2, 3, 4, 5, 6, 8]))
        P = 0 if rng.random() < 0.12 else int(rng.integers(1, 4500))
        R = int(np.exp(rng.uniform(0, np.log(420))))
        ps = int(rng.choice([16, 32, 64, 128, 256]))
        splits = int(rng.choice([1, 2, 3, 7, 16, 64, 1000]))
        sharp = bool(rng.random() < 0.7)
        scale = float(rng.choice([128 ** -0.5, 0.05, 0.15]))
        if R * (P + R) * g * hkv > MAX_WORK:
            continue
        cases.append((P, R, g * hkv, hkv, ps, splits, sharp, scale))
    return cases


def _draw_ragged(n, seed):
    rng = np.random.default_rng(seed)
    cases = []
    while len(cases) < n:
        hkv = int(rng.choice([1, 2, 4]))
        g = int(rng.choice([1, 3, 6]))
        P = 0 if rng.random() < 0.15 else int(rng.integers(1, 3000))
        lens = [int(x) for x in rng.integers(0, 260, size=int(rng.integers(1, 6)))]
        if sum(lens) == 0:
            continue
        ps = int(rng.choice([16, 64, 256]))
        splits = int(rng.choice([1, 4, 1000]))
        if sum(r * (P + r) for r in lens) * g * hkv > MAX_WORK:
            continue
        cases.append((P, lens, g * hkv, hkv, ps, splits))
    return cases


SINGLE = _draw_single(28, 20261203)
RAGGED = _draw_ragged(8, 20261204)


@pytest.mark.parametrize("P,R,hq,hkv,ps,splits,sharp,scale", SINGLE)
def test_random_shape_fwd_bwd(cuda, P, R, hq, hkv, ps, splits, sharp, scale):
    case = Case(P, R, hq, hkv, ps, splits, seed=3 * P + 7 * R + hq, device=cuda, sharp=sharp,
                scale=scale)
    o, lse = case.fwd()
    pb = case.problem()
    o_ref, lse_ref = oracle.attn_fwd(pb)
    assert rel_err(o.float().cpu().numpy(), o_ref) <= TOL_O
    assert float(np.abs(lse.cpu().numpy() - lse_ref).max()) <= TOL_LSE
    dq, dk, dv = case.bwd(o, lse)
    dq_ref, dk_ref, dv_ref = oracle.attn_bwd(pb, case.d_o_host())
    for name, x, ref in (("dq", dq, dq_ref), ("dk", dk, dk_ref), ("dv", dv, dv_ref)):
        err = rel_err(x.cpu().numpy(), ref)
        assert err <= TOL_GRAD, (name, err)
    assert B.ls_last_device_error(0) == B.LS_OK


@pytest.mark.parametrize("P,lens,hq,hkv,ps,splits", RAGGED)
def test_random_ragged_members(cuda, P, lens, hq, hkv, ps, splits):
    from test_gpu_ragged import make, member_problem
    scale = 128 ** -0.5
    cache, br = make(P, lens, hq, hkv, ps, 900 + P + sum(lens), cuda)
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


def _draw_latent(n, seed):
    rng = np.random.default_rng(seed)
    cases = []
    while len(cases) < n:
        H = int(rng.choice([1, 3, 16, 20, 64, 128]))
        P = 0 if rng.random() < 0.15 else int(rng.integers(1, 6000))
        R = int(np.exp(rng.uniform(0, np.log(200))))
        ps = int(rng.choice([32, 64, 256, 4096]))
        splits = int(rng.choice([1, 2, 5, 64, 1000]))
        sharp = bool(rng.random() < 0.7)
        if R * (P + R) * H > 3_000_000:
            continue
        cases.append((P, R, H, ps, splits, sharp))
    return cases


LATENT = _draw_latent(10, 20261205)


@pytest.mark.parametrize("P,R,H,ps,splits,sharp", LATENT)
def test_random_latent_replay(cuda, P, R, H, ps, splits, sharp):
    from test_gpu_mla import SCALE, make, problem
    cache, br = make(P, R, H, ps, 40 + P + R + H, cuda, sharp=sharp, extra_pages=1)
    o, lse = api.mla_replay_fwd(cache, br.q, br.lat, SCALE, splits)
    torch.cuda.synchronize()
    assert B.ls_last_device_error(0) == B.LS_OK
    pb = problem(cache, br, P)
    o_ref, lse_ref = oracle.mla_fwd(pb)
    assert rel_err(o.float().cpu().numpy(), o_ref) <= TOL_O
    assert float(np.abs(lse.cpu().numpy() - lse_ref).max()) <= TOL_LSE
    dq, dlat = api.mla_replay_bwd(cache, br.q, br.lat, o, lse, br.d_o, SCALE, splits)
    torch.cuda.synchronize()
    assert B.ls_last_device_error(0) == B.LS_OK
    dq_ref, dlat_ref = oracle.mla_bwd(pb, u16(br.d_o))
    assert rel_err(dq.cpu().numpy(), dq_ref) <= TOL_GRAD
    assert rel_err(dlat.cpu().numpy(), dlat_ref) <= TOL_GRAD
