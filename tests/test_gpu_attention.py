"""GPU parity of replay attention (forward and backward) and page capture against the
fp64 oracle, element by element, through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
from parity_util import TOL_GRAD, TOL_LSE, TOL_O, Case, rel_err, u16
from response_replay_gb300 import synthetic as syn
from response_replay_gb300 import torch_api as api
from response_replay_gb300 import binding as B

pytestmark = pytest.mark.gpu


def check_fwd(case, o, lse, pb=None):
    pb = pb or case.problem()
    o_ref, lse_ref = oracle.attn_fwd(pb)
    o_gpu = o.float().cpu().numpy()
    lse_gpu = lse.cpu().numpy()
    assert np.isfinite(o_gpu).all() and np.isfinite(lse_gpu).all()
    e_o, e_l = rel_err(o_gpu, o_ref), float(np.abs(lse_gpu - lse_ref).max())
    assert e_o <= TOL_O, f"O rel err {e_o}"
    assert e_l <= TOL_LSE, f"LSE abs err {e_l}"
    return pb


def check_bwd(case, dq, dk, dv, pb):
    dq_ref, dk_ref, dv_ref = oracle.attn_bwd(pb, case.d_o_host())
    for name, x, ref in (("dq", dq, dq_ref), ("dk", dk, dk_ref), ("dv", dv, dv_ref)):
        xg = x.cpu().numpy()
        assert np.isfinite(xg).all(), name
        e = rel_err(xg, ref)
        assert e <= TOL_GRAD, f"{name} rel err {e}"


# The small workload: P = 4096 in 64-token pages, Hq 8 / Hkv 2, 4 splits, G = 2 x 256.
@pytest.mark.parametrize("member", [0, 1])
@pytest.mark.parametrize("sharp", [False, True])
def test_small_workload_fwd_bwd(cuda, member, sharp):
    w = syn.WORKLOADS["p4k"]
    case = Case(w.P, w.R[member], w.hq, w.hkv, w.page_size, w.num_splits,
                syn.seed_of("p4k") + 10 * member, cuda, sharp=sharp)
    o, lse = case.fwd()
    pb = check_fwd(case, o, lse)
    dq, dk, dv = case.bwd(o, lse)
    check_bwd(case, dq, dk, dv, pb)
    assert B.ls_last_device_error(0) == B.LS_OK


# Ragged shapes: prompt not a multiple of the tile or page, response not a multiple of
# the query block, several split counts (more splits than tiles included), P = 0, R = 1.
@pytest.mark.parametrize("P,R,hq,hkv,ps,splits", [
    (1000, 200, 6, 2, 16, 3),
    (1000, 200, 6, 2, 16, 1000),
    (3000, 77, 4, 4, 256, 2),
    (0, 130, 6, 3, 64, 4),
    (777, 1, 8, 1, 32, 5),
    (129, 65, 2, 1, 128, 1),
    (5000, 300, 12, 2, 64, 7),
])
def test_ragged_fwd_bwd(cuda, P, R, hq, hkv, ps, splits):
    case = Case(P, R, hq, hkv, ps, splits, seed=P * 7 + R, device=cuda, sharp=True)
    o, lse = case.fwd()
    pb = check_fwd(case, o, lse)
    dq, dk, dv = case.bwd(o, lse)
    check_bwd(case, dq, dk, dv, pb)


# Short responses (R < 256): the forward packs the g query heads of a KV head into a
# unit's rows (floor(128 / g) whole tokens per tile, g not dividing 128 leaves spare
# rows); g = 1 and R = 1 included, P = 0, more splits than tiles.
@pytest.mark.parametrize("P,R,hq,hkv,ps,splits", [
    (3000, 77, 12, 2, 64, 5),
    (1000, 1, 6, 1, 16, 3),
    (5000, 200, 8, 2, 128, 7),
    (777, 255, 24, 3, 32, 4),
    (0, 50, 4, 1, 64, 2),
    (2048, 10, 3, 1, 16, 1000),
    (4096, 130, 5, 5, 64, 4),
    # a tile holds a divisor of g heads: g = 6 packs 2 heads x 64 tokens at R = 48 / 64
    # (forward) and 64 / 128 (both passes); 127 tokens take one head per tile backward
    (3000, 64, 12, 2, 64, 5),
    (2000, 48, 24, 4, 128, 3),
    (1500, 128, 6, 1, 64, 4),
    (1000, 127, 12, 2, 32, 7),
    (2500, 96, 8, 2, 64, 3),
])
def test_short_response_packed_fwd_bwd(cuda, P, R, hq, hkv, ps, splits):
    case = Case(P, R, hq, hkv, ps, splits, seed=P * 5 + R + hq, device=cuda, sharp=True)
    o, lse = case.fwd()
    pb = check_fwd(case, o, lse)
    dq, dk, dv = case.bwd(o, lse)
    check_bwd(case, dq, dk, dv, pb)
    assert B.ls_last_device_error(0) == B.LS_OK


def test_split_count_does_not_change_result(cuda):
    case = Case(4096, 256, 8, 2, 64, 1, seed=5, device=cuda, sharp=True)
    outs = [case.fwd(num_splits=s) for s in (1, 3, 32, 1000)]
    o0, l0 = outs[0]
    for o, l in outs[1:]:
        assert (o.float() - o0.float()).abs().max().item() <= 2 ** -7
        assert (l - l0).abs().max().item() <= 1e-5


def test_bwd_accumulate_adds(cuda):
    case = Case(512, 96, 4, 2, 64, 2, seed=9, device=cuda, sharp=True)
    o, lse = case.fwd()
    dq1, dk1, dv1 = case.bwd(o, lse)
    dq2, dk2, dv2 = case.bwd(o, lse, dq=dq1.clone(), dk=dk1.clone(), dv=dv1.clone(),
                             accumulate=True)
    torch.testing.assert_close(dq2, 2 * dq1, rtol=1e-6, atol=1e-7)
    torch.testing.assert_close(dk2, 2 * dk1, rtol=1e-6, atol=1e-7)
    torch.testing.assert_close(dv2, 2 * dv1, rtol=1e-6, atol=1e-7)


def test_deterministic(cuda):
    case = Case(4096, 256, 8, 2, 64, 4, seed=11, device=cuda, sharp=True)
    o1, l1 = case.fwd()
    o2, l2 = case.fwd()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    g1 = case.bwd(o1, l1)
    g2 = case.bwd(o1, l1)
    for a, b in zip(g1, g2):
        assert torch.equal(a, b)


def test_capture_bit_exact_against_oracle(cuda):
    P, hkv, ps = 1000, 3, 16
    pr = syn.make_prompt(P, hkv, 128, ps, 21, cuda, extra_pages=5)
    cache = api.PagedKVCache(pr.num_pages, pr.page_table, ps, hkv, P, device=cuda, fill=float("nan"))
    k_before = u16(cache.k_pool).copy()
    v_before = u16(cache.v_pool).copy()
    # chunked capture: [0, 333) then [333, 1000)
    cache.capture(pr.k[:333].contiguous(), pr.v[:333].contiguous(), 0)
    cache.capture(pr.k[333:].contiguous(), pr.v[333:].contiguous(), 333)
    torch.cuda.synchronize()
    oracle.capture_kv(k_before, v_before, pr.page_table.cpu().numpy(), ps, u16(pr.k), u16(pr.v), 0)
    assert np.array_equal(u16(cache.k_pool), k_before)
    assert np.array_equal(u16(cache.v_pool), v_before)
    cache.validate()
    assert B.ls_last_device_error(0) == B.LS_OK


def test_bad_page_id_is_reported_not_faulted(cuda):
    P, hkv, ps = 256, 1, 64
    pr = syn.make_prompt(P, hkv, 128, ps, 23, cuda)
    bad = pr.page_table.clone()
    bad[2] = pr.num_pages + 5           # outside the pool
    cache = api.PagedKVCache(pr.num_pages, bad, ps, hkv, P, device=cuda, fill=0.0)
    cache.capture(pr.k, pr.v)
    assert B.ls_last_device_error(0) == B.LS_ERR_DEVICE_CHECK
    br = syn.make_branch(8, 2, hkv, 128, 24, cuda)
    api.replay_fwd(cache, br.q, br.k, br.v, 0.1, 2)
    assert B.ls_last_device_error(0) == B.LS_ERR_DEVICE_CHECK
    cache.validate()
    assert B.ls_last_device_error(0) == B.LS_ERR_DEVICE_CHECK
    dup = pr.page_table.clone()
    dup[1] = dup[0]                     # a physical page used twice
    api.PagedKVCache(pr.num_pages, dup, ps, hkv, P, device=cuda).validate()
    assert B.ls_last_device_error(0) == B.LS_ERR_DEVICE_CHECK
    assert B.ls_last_device_error(0) == B.LS_OK   # cleared by the read
