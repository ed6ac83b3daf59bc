"""Prompt pages held in pinned host memory (Grace memory behind NVLink-C2C on a GB300
node), read and written by the kernels in place: capture bit-exact against the oracle,
forward and backward against the oracle and bit-identical to the same pages in GPU
memory (the kernels are deterministic and read the same values)."""
import numpy as np
import pytest
import torch

import oracle
from parity_util import TOL_GRAD, TOL_LSE, TOL_O, Case, rel_err, u16
from response_replay_gb300 import binding as B
from response_replay_gb300 import synthetic as syn
from response_replay_gb300 import torch_api as api

pytestmark = pytest.mark.gpu


def host_copy(cache: api.PagedKVCache) -> api.PagedKVCache:
    kh = torch.empty(cache.k_pool.shape, dtype=torch.bfloat16, pin_memory=True)
    vh = torch.empty(cache.v_pool.shape, dtype=torch.bfloat16, pin_memory=True)
    kh.copy_(cache.k_pool)
    vh.copy_(cache.v_pool)
    return api.PagedKVCache(cache.k_pool.shape[0], cache.page_table, cache.page_size,
                            cache.num_kv_heads, cache.num_tokens, k_pool=kh, v_pool=vh)


def test_capture_into_host_pages_bit_exact(cuda):
    P, hkv, ps = 1000, 3, 16
    pr = syn.make_prompt(P, hkv, 128, ps, 31, cuda, extra_pages=5)
    cache = api.PagedKVCache(pr.num_pages, pr.page_table, ps, hkv, P, host_pools=True,
                             fill=float("nan"))
    assert not cache.k_pool.is_cuda and cache.k_pool.is_pinned()
    k_before = u16(cache.k_pool).copy()
    v_before = u16(cache.v_pool).copy()
    cache.capture(pr.k[:400].contiguous(), pr.v[:400].contiguous(), 0)
    cache.capture(pr.k[400:].contiguous(), pr.v[400:].contiguous(), 400)
    torch.cuda.synchronize()
    oracle.capture_kv(k_before, v_before, pr.page_table.cpu().numpy(), ps, u16(pr.k), u16(pr.v), 0)
    assert np.array_equal(u16(cache.k_pool), k_before)
    assert np.array_equal(u16(cache.v_pool), v_before)
    assert B.ls_last_device_error(0) == B.LS_OK


@pytest.mark.parametrize("P,R,hq,hkv,ps,splits", [
    (4096, 256, 8, 2, 64, 4),       # the small workload's shape
    (3000, 77, 12, 2, 64, 5),       # grouped-query packing, ragged tail
    (5000, 300, 12, 2, 64, 7),
])
def test_host_pages_match_oracle_and_gpu_pages(cuda, P, R, hq, hkv, ps, splits):
    case = Case(P, R, hq, hkv, ps, splits, seed=P + R, device=cuda, sharp=True)
    hc = host_copy(case.cache)
    br = case.br
    o_d, l_d = case.fwd()
    o_h, l_h = api.replay_fwd(hc, br.q, br.k, br.v, case.scale, splits)
    g_d = case.bwd(o_d, l_d)
    g_h = api.replay_bwd(hc, br.q, br.k, br.v, o_h, l_h, br.d_o, case.scale, splits)
    torch.cuda.synchronize()
    assert B.ls_last_device_error(0) == B.LS_OK
    assert torch.equal(o_h, o_d) and torch.equal(l_h, l_d)
    for a, b in zip(g_h, g_d):
        assert torch.equal(a, b)
    pb = case.problem()
    o_ref, lse_ref = oracle.attn_fwd(pb)
    assert rel_err(o_h.float().cpu().numpy(), o_ref) <= TOL_O
    assert float(np.abs(l_h.cpu().numpy() - lse_ref).max()) <= TOL_LSE
    for x, ref in zip(g_h, oracle.attn_bwd(pb, case.d_o_host())):
        assert rel_err(x.cpu().numpy(), ref) <= TOL_GRAD


def test_host_pages_ragged_members(cuda):
    P, lens, hq, hkv, ps, splits = 2000, [16, 300, 1, 77], 12, 2, 32, 3
    pr = syn.make_prompt(P, hkv, 128, ps, 41, cuda, extra_pages=2, sharp=True)
    cache = api.PagedKVCache(pr.num_pages, pr.page_table, ps, hkv, P, device=cuda)
    cache.capture(pr.k[:P].contiguous(), pr.v[:P].contiguous())
    hc = host_copy(cache)
    br = syn.make_branch(int(sum(lens)), hq, hkv, 128, 42, cuda, sharp=True)
    scale = 128 ** -0.5
    o_d, l_d = api.replay_fwd_ragged(cache, br.q, br.k, br.v, lens, scale, splits)
    o_h, l_h = api.replay_fwd_ragged(hc, br.q, br.k, br.v, lens, scale, splits)
    g_d = api.replay_bwd_ragged(cache, br.q, br.k, br.v, o_d, l_d, br.d_o, lens, scale, splits)
    g_h = api.replay_bwd_ragged(hc, br.q, br.k, br.v, o_h, l_h, br.d_o, lens, scale, splits)
    torch.cuda.synchronize()
    assert B.ls_last_device_error(0) == B.LS_OK
    assert torch.equal(o_h, o_d) and torch.equal(l_h, l_d)
    for a, b in zip(g_h, g_d):
        assert torch.equal(a, b)
