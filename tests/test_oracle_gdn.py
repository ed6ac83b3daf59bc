"""Pins of the Gated-DeltaNet replay oracle (oracle/gdn_oracle.c) against things other
than itself: a hand-worked example, closed forms (no update: pure decay; unit keys with
beta = 1: exact overwrite), replay from a captured state equal to running the whole
sequence, the chunked form of the rule (tests/gdn_chunked.py, a second derivation) for
the forward and every gradient, and central finite differences of <dO, o>."""
import json
import os

import numpy as np
import pytest

import gdn_chunked
import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "gdn_hand_example.json")


def rand_problem(R, H, dk, dv, seed, scale=0.5):
    rng = np.random.default_rng(seed)
    k = rng.standard_normal((R, H, dk))
    k /= np.linalg.norm(k, axis=2, keepdims=True)          # unit keys, as GDN normalises them
    q = rng.standard_normal((R, H, dk))
    v = rng.standard_normal((R, H, dv))
    g = np.log(rng.uniform(0.6, 1.0, (R, H)))
    beta = rng.uniform(0.05, 0.95, (R, H))
    s0 = rng.standard_normal((H, dv, dk))
    return oracle.GdnProblem(s0, q, k, v, g, beta, scale)


def test_hand_example():
    ex = json.load(open(GOLDEN))
    toks = ex["tokens"]
    pb = oracle.GdnProblem(np.array([ex["state0"]]), np.array([[t["q"]] for t in toks]),
                           np.array([[t["k"]] for t in toks]), np.array([[t["v"]] for t in toks]),
                           np.log(np.array([[t["alpha"]] for t in toks])),
                           np.array([[t["beta"]] for t in toks]), ex["scale"])
    o, s = oracle.gdn_fwd(pb)
    assert np.allclose(o[:, 0], ex["o"], atol=1e-12)
    assert np.allclose(s[0], ex["state_out"], atol=1e-12)


def test_no_update_is_pure_decay():
    pb = rand_problem(9, 2, 5, 3, 1)
    pb.beta[:] = 0.0
    o, s = oracle.gdn_fwd(pb)
    G = np.cumsum(pb.g, axis=0)                             # [R][H]
    want = np.einsum("th,hab,thb->tha", np.exp(G), pb.state0, pb.scale * pb.q)
    assert np.abs(o - want).max() < 1e-12
    assert np.abs(s - np.exp(G[-1])[:, None, None] * pb.state0).max() < 1e-12


def test_unit_keys_beta_one_overwrite():
    """alpha = 1, beta = 1 and keys from an orthonormal basis: the rule writes v_t at k_t,
    so S_t k_t = v_t and a query equal to k_t reads v_t back (times scale)."""
    R, dk, dv = 6, 4, 3
    rng = np.random.default_rng(2)
    basis = np.linalg.qr(rng.standard_normal((dk, dk)))[0]
    idx = [0, 2, 1, 2, 3, 0]                                # keys revisited
    k = basis[idx][:, None, :]
    v = rng.standard_normal((R, 1, dv))
    pb = oracle.GdnProblem(rng.standard_normal((1, dv, dk)), k.copy(), k, v, np.zeros((R, 1)),
                           np.ones((R, 1)), 2.0)
    o, _ = oracle.gdn_fwd(pb)
    assert np.abs(o[:, 0] - 2.0 * v[:, 0]).max() < 1e-12


def test_replay_from_captured_state_equals_whole_sequence():
    whole = rand_problem(23, 3, 6, 5, 3)
    Pn = 15
    head = oracle.GdnProblem(whole.state0, whole.q[:Pn], whole.k[:Pn], whole.v[:Pn],
                             whole.g[:Pn], whole.beta[:Pn], whole.scale)
    _, captured = oracle.gdn_fwd(head)
    tail = oracle.GdnProblem(captured, whole.q[Pn:], whole.k[Pn:], whole.v[Pn:], whole.g[Pn:],
                             whole.beta[Pn:], whole.scale)
    o_whole, s_whole = oracle.gdn_fwd(whole)
    o_tail, s_tail = oracle.gdn_fwd(tail)
    assert np.array_equal(o_whole[Pn:], o_tail)
    assert np.array_equal(s_whole, s_tail)


@pytest.mark.parametrize("R,C", [(11, 4), (16, 4), (7, 8), (130, 64)])
def test_chunked_form_matches(R, C):
    pb = rand_problem(R, 2, 6, 5, 4 + R)
    o, s = oracle.gdn_fwd(pb)
    oc, sc = gdn_chunked.fwd(pb.state0, pb.q, pb.k, pb.v, pb.g, pb.beta, pb.scale, C)
    assert np.abs(o - oc).max() < 1e-10 and np.abs(s - sc).max() < 1e-10
    d_o = np.random.default_rng(R).standard_normal(o.shape)
    ref = oracle.gdn_bwd(pb, d_o)
    got = gdn_chunked.bwd(pb.state0, pb.q, pb.k, pb.v, pb.g, pb.beta, pb.scale, d_o, C)
    for name, a, b in zip(("dq", "dk", "dv", "dg", "dbeta", "dstate0"), ref, got):
        assert np.abs(a - b).max() < 1e-9 * max(1.0, np.abs(a).max()), name


def test_gradients_by_finite_differences():
    pb = rand_problem(7, 2, 4, 3, 5)
    d_o = np.random.default_rng(6).standard_normal((7, 2, 3))
    dq, dk, dv, dg, db, ds0 = oracle.gdn_bwd(pb, d_o)

    def f():
        return float(np.sum(oracle.gdn_fwd(pb)[0] * d_o))

    eps = 1e-6
    for arr, grad in ((pb.q, dq), (pb.k, dk), (pb.v, dv), (pb.g, dg), (pb.beta, db),
                      (pb.state0, ds0)):
        flat, gflat = arr.reshape(-1), grad.reshape(-1)
        for i in range(0, flat.size, max(1, flat.size // 9)):
            x = flat[i]
            flat[i] = x + eps
            fp = f()
            flat[i] = x - eps
            fm = f()
            flat[i] = x
            assert abs((fp - fm) / (2 * eps) - gflat[i]) < 1e-6 * max(1.0, abs(gflat[i]))
