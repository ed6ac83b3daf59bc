"""The all-zero-key closed forms (tests/closed_forms.py) agree with the fp64 oracle on
small inputs, so the long-response GPU tests that use them rest on the same
definitions as every other parity test."""
import numpy as np
import pytest

import oracle
from closed_forms import key_gradients, uniform_attention


@pytest.mark.parametrize("P,R,hq,hkv,ps", [(0, 37, 6, 2, 16), (100, 50, 4, 1, 32),
                                           (64, 9, 3, 3, 64)])
def test_zero_key_closed_forms_match_oracle(P, R, hq, hkv, ps):
    rng = np.random.default_rng(P + R)
    d = 128
    pages = max(1, (P + ps - 1) // ps)
    k_pool = np.zeros((pages + 1, hkv, ps, d))
    v_pool = rng.standard_normal((pages + 1, hkv, ps, d))
    pt = rng.permutation(pages + 1)[:pages].astype(np.int32)
    q = rng.standard_normal((R, hq, d))
    kr = np.zeros((R, hkv, d))
    vr = rng.standard_normal((R, hkv, d))
    d_o = rng.standard_normal((R, hq, d))
    scale = d ** -0.5
    pb = oracle.AttnProblem(k_pool, v_pool, pt, P, q, kr, vr, scale, 3)
    o_ref, lse_ref = oracle.attn_fwd(pb)
    _, dk_ref, dv_ref = oracle.attn_bwd(pb, d_o)
    # the prompt's values in position order
    vp = np.zeros((hkv, d))
    for p in range(P):
        vp += v_pool[pt[p // ps], :, p % ps, :]
    lse, o = uniform_attention(P, vp, vr)
    g = hq // hkv
    assert np.abs(lse[:, None] - lse_ref).max() < 1e-12
    assert np.abs(np.repeat(o, g, axis=1) - o_ref).max() < 1e-12
    js = np.repeat(np.arange(R), hkv)
    kvhs = np.tile(np.arange(hkv), R)
    dk, dv = key_gradients(P, scale, q, vr, d_o, o, js, kvhs)
    assert np.abs(dk - dk_ref[js, kvhs]).max() < 1e-10
    assert np.abs(dv - dv_ref[js, kvhs]).max() < 1e-10
