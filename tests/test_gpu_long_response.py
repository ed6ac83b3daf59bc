"""dK/dV of the response's own keys over long responses, first keys included.

The gradient of response key j sums over every later row t >= j and every query head
of its group, so key 0 of a long response has the longest reduction of the backward.
Two checks cover it:
  * the fp64 oracle on every key of a 2,048-token response over a 2,048-position prompt
    with sharp inputs (scores of unit spread);
  * the all-zero-key closed forms (tests/closed_forms.py, pinned against the oracle) at
    R = 4,096 and 8,192 with and without a prompt, and R = 4,096 over the full
    2,097,152-position prompt, where the oracle would need hours:
    keys 0, 1, R/2 and R - 1 of every KV head, plus O and LSE of every row.
"""
import numpy as np
import pytest
import torch

import oracle
from closed_forms import key_gradients, uniform_attention
from parity_util import TOL_GRAD, TOL_LSE, TOL_O, Case, rel_err, u16
from response_replay_gb300 import synthetic as syn
from response_replay_gb300 import torch_api as api
from response_replay_gb300 import binding as B

pytestmark = pytest.mark.gpu


def test_whole_response_every_key_sharp(cuda):
    case = Case(2048, 2048, 6, 1, 64, 5, seed=31, device=cuda, sharp=True)
    o, lse = case.fwd()
    dq, dk, dv = case.bwd(o, lse)
    pb = case.problem()
    o_ref, lse_ref = oracle.attn_fwd(pb)
    assert rel_err(o.float().cpu().numpy(), o_ref) <= TOL_O
    assert float(np.abs(lse.cpu().numpy() - lse_ref).max()) <= TOL_LSE
    dq_ref, dk_ref, dv_ref = oracle.attn_bwd(pb, case.d_o_host())
    for name, x, ref in (("dq", dq, dq_ref), ("dk", dk, dk_ref), ("dv", dv, dv_ref)):
        e = rel_err(x.cpu().numpy(), ref)
        assert e <= TOL_GRAD, (name, e)
    # the first keys carry the longest sums: checked on their own scale too
    for x, ref in ((dk, dk_ref), (dv, dv_ref)):
        assert rel_err(x[:4].cpu().numpy(), ref[:4]) <= TOL_GRAD


@pytest.mark.parametrize("P,R", [(0, 4096), (4096, 4096), (0, 8192), (4096, 8192),
                                 (2097152, 4096)])
def test_long_response_first_keys_closed_form(cuda, P, R):
    hq, hkv, ps, splits, d = 24, 4, 256, 4, 128
    scale = d ** -0.5
    seed = 40 + R + P
    pr = syn.make_prompt(max(P, 1), hkv, d, ps, seed, cuda, extra_pages=1)
    if P == 0:
        pr.page_table = pr.page_table[:0]
    cache = api.PagedKVCache(pr.num_pages, pr.page_table, ps, hkv, P, device=cuda, fill=0.0)
    if P > 0:
        cache.capture(torch.zeros_like(pr.k), pr.v)
    br = syn.make_branch(R, hq, hkv, d, seed + 1, cuda, sharp=True)
    k0 = torch.zeros_like(br.k)
    o, lse = api.replay_fwd(cache, br.q, k0, br.v, scale, splits)
    dq, dk, dv = api.replay_bwd(cache, br.q, k0, br.v, o, lse, br.d_o, scale, splits)
    torch.cuda.synchronize()
    assert B.ls_last_device_error(0) == B.LS_OK
    vp = pr.v[:P].sum(0, dtype=torch.float64).cpu().numpy() if P > 0 else np.zeros((hkv, d))
    vr = br.v.double().cpu().numpy()
    lse_ref, o_ref = uniform_attention(P, vp, vr)
    g = hq // hkv
    assert float(np.abs(lse.cpu().numpy() - lse_ref[:, None]).max()) <= TOL_LSE
    assert rel_err(o.float().cpu().numpy(), np.repeat(o_ref, g, axis=1)) <= TOL_O
    assert torch.count_nonzero(dq).item() == 0          # every key is zero
    js = np.repeat(np.array([0, 1, R // 2, R - 1]), hkv)
    kvhs = np.tile(np.arange(hkv), 4)
    dk_ref, dv_ref = key_gradients(P, scale, br.q.double().cpu().numpy(), vr,
                                   br.d_o.double().cpu().numpy(), o_ref, js, kvhs)
    dk_g = dk.cpu().numpy()[js, kvhs]
    dv_g = dv.cpu().numpy()[js, kvhs]
    for i in range(len(js)):   # each key on its own scale
        assert rel_err(dk_g[i], dk_ref[i]) <= TOL_GRAD, ("dk", js[i], kvhs[i])
        assert rel_err(dv_g[i], dv_ref[i]) <= TOL_GRAD, ("dv", js[i], kvhs[i])
