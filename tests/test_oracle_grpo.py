"""Pins of the fp64 GRPO oracle against closed forms, a hand-worked example, a
library log-softmax and finite differences."""
import json
import os

import numpy as np
import pytest
from scipy.special import log_softmax

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rand_case(lens, V, seed, G=None, rewards=None):
    rng = np.random.default_rng(seed)
    T = int(sum(lens))
    logits = rng.standard_normal((T, V)) * 2.0
    targets = rng.integers(0, V, T).astype(np.int32)
    if rewards is None:
        rewards = rng.standard_normal(len(lens) if G is None else G)
    return logits, targets, np.asarray(rewards, np.float64), rng


def lib_logp(logits, targets):
    return log_softmax(logits, axis=1)[np.arange(len(targets)), targets]


def test_hand_worked_example():
    with open(os.path.join(GOLDEN, "grpo_hand_example.json")) as f:
        ex = json.load(f)
    rng = np.random.default_rng(0)
    logits = rng.standard_normal((3, 4))
    targets = np.array([1, 3, 0], np.int32)
    logp_old = lib_logp(logits, targets) - np.log(ex["rho"])
    r = oracle.grpo(logits, targets, logp_old, ex["rewards"], ex["resp_lens"], 0, 2, ex["eps"],
                    1e-6, 1)
    np.testing.assert_allclose(r.adv, ex["adv_ddof1"], rtol=0, atol=1e-14)
    np.testing.assert_allclose(r.ratio, ex["rho"], rtol=0, atol=1e-14)
    assert abs(r.loss - ex["expect_loss_ddof1"]) < 1e-14
    np.testing.assert_allclose(r.coef, ex["expect_coef_ddof1"], rtol=0, atol=1e-14)
    np.testing.assert_array_equal(r.zeroed, ex["expect_zeroed_ddof1"])
    r0 = oracle.grpo(logits, targets, logp_old, ex["rewards"], ex["resp_lens"], 0, 2, ex["eps"],
                     1e-6, 0)
    np.testing.assert_allclose(r0.adv, ex["adv_ddof0"], rtol=0, atol=1e-14)


def test_equal_rewards_give_exact_zero():
    """All members rewarded alike: every advantage is 0, so the loss and every gradient
    coefficient are exactly 0 (no rounding residue from the mean)."""
    logits, targets, _, rng = rand_case([5, 3, 4], 16, 1)
    for rw in (0.3, 1.0, -7.1):
        r = oracle.grpo(logits, targets, lib_logp(logits, targets) + rng.normal(0, .3, 12),
                        [rw] * 3, [5, 3, 4], 0, 3, 0.2)
        assert r.loss == 0.0
        assert (r.adv == 0).all() and (r.coef == 0).all() and (r.zeroed == 0).all()


def test_on_policy_ratio_one():
    """logp_old = logp: rho = 1 in the band, loss = -(1/G) sum_i A_i = 0 (the advantages
    sum to zero) and dL/dlogp_t = -A_i / (G R_i)."""
    lens = [4, 2, 6, 3]
    logits, targets, rewards, _ = rand_case(lens, 32, 2)
    r = oracle.grpo(logits, targets, lib_logp(logits, targets), rewards, lens, 0, 4, 0.2)
    np.testing.assert_allclose(r.ratio, 1.0, atol=1e-14)
    assert abs(r.loss) < 1e-14
    member = np.repeat(np.arange(4), lens)
    np.testing.assert_allclose(r.coef, -r.adv[member] / (4 * np.array(lens)[member]), atol=1e-15)


def test_clip_branch_on_favourable_side_zeroes_gradient():
    lens = [3, 3]
    logits, targets, _, _ = rand_case(lens, 8, 3)
    lp = lib_logp(logits, targets)
    rewards = [0.0, 1.0]                              # A0 < 0, A1 > 0
    shift = np.array([+0.5, +0.5, +0.5, -0.5, -0.5, -0.5])
    # member 0 (A<0): rho = e^-0.5 < 0.8 -> clipped; member 1 (A>0): rho = e^0.5 > 1.2 -> clipped
    r = oracle.grpo(logits, targets, lp + shift, rewards, lens, 0, 2, 0.2)
    assert (r.zeroed == 1).all() and (r.coef == 0).all()
    # the unfavourable side keeps the gradient: flip the shifts
    r2 = oracle.grpo(logits, targets, lp - shift, rewards, lens, 0, 2, 0.2)
    assert (r2.zeroed == 0).all() and (r2.coef != 0).all()


def test_constant_logits_lse():
    V = 50
    logits = np.full((3, V), 1.25)
    r = oracle.grpo(logits, np.array([0, 7, 49], np.int32), np.zeros(3), [0.0, 1.0], [1, 2], 0, 2,
                    0.2)
    np.testing.assert_allclose(r.lse, np.log(V) + 1.25, atol=1e-14)
    np.testing.assert_allclose(r.logp, -np.log(V), atol=1e-14)


def test_unclipped_limit_matches_library_log_softmax():
    """eps -> infinity leaves the plain surrogate -(1/G) sum_i (1/R_i) sum_t rho A_i
    (the unclipped form the 2M-token runs used)."""
    lens = [7, 1, 5]
    logits, targets, rewards, rng = rand_case(lens, 40, 4)
    old = lib_logp(logits, targets) + rng.normal(0, 0.4, sum(lens))
    r = oracle.grpo(logits, targets, old, rewards, lens, 0, 3, 1e30)
    rho = np.exp(lib_logp(logits, targets) - old)
    A = (rewards - rewards.mean()) / (rewards.std(ddof=1) + 1e-6)
    member = np.repeat(np.arange(3), lens)
    expect = -np.sum(rho * A[member] / np.array(lens)[member]) / 3
    assert abs(r.loss - expect) < 1e-13 * max(1, abs(expect))


def test_dlogits_match_finite_differences():
    """d(loss)/d(logits) against central differences of the oracle's own loss, on a case
    with tokens on both sides of the band (none within 1e-3 of a boundary)."""
    lens = [3, 2, 4]
    V = 6
    logits, targets, rewards, rng = rand_case(lens, V, 5)
    old = lib_logp(logits, targets) + rng.choice([-0.6, -0.05, 0.05, 0.6], size=9)
    r = oracle.grpo(logits, targets, old, rewards, lens, 0, 3, 0.2)
    assert (np.abs(np.abs(r.ratio - 1) - 0.2) > 1e-3).all()
    assert r.zeroed.any() and (r.coef != 0).any()
    g = oracle.grpo_dlogits_rows(logits, range(9), targets, r.lse, r.coef)
    h = 1e-6
    fd = np.zeros_like(logits)
    for t in range(9):
        for v in range(V):
            lp, lm = logits.copy(), logits.copy()
            lp[t, v] += h
            lm[t, v] -= h
            fp = oracle.grpo(lp, targets, old, rewards, lens, 0, 3, 0.2).loss
            fm = oracle.grpo(lm, targets, old, rewards, lens, 0, 3, 0.2).loss
            fd[t, v] = (fp - fm) / (2 * h)
    np.testing.assert_allclose(g, fd, atol=1e-8)


def test_member_range_partial_losses_add_up():
    """Serial replay calls the loss once per member with the whole group's rewards; the
    per-member losses must add up to the whole-group loss."""
    lens = [4, 3, 5]
    logits, targets, rewards, rng = rand_case(lens, 12, 6)
    old = lib_logp(logits, targets) + rng.normal(0, 0.3, 12)
    full = oracle.grpo(logits, targets, old, rewards, lens, 0, 3, 0.2)
    off = np.cumsum([0] + lens)
    parts = [oracle.grpo(logits[off[i]:off[i + 1]], targets[off[i]:off[i + 1]],
                         old[off[i]:off[i + 1]], rewards, lens, i, i + 1, 0.2) for i in range(3)]
    assert abs(sum(p.loss for p in parts) - full.loss) < 1e-15
    np.testing.assert_array_equal(np.concatenate([p.coef for p in parts]), full.coef)


def test_invalid_arguments():
    logits = np.zeros((3, 4))
    t = np.zeros(3, np.int32)
    with pytest.raises(ValueError):   # lengths do not cover T
        oracle.grpo(logits, t, np.zeros(3), [0, 1], [1, 1], 0, 2, 0.2)
    with pytest.raises(ValueError):   # G = 1 with sample std
        oracle.grpo(logits, t, np.zeros(3), [1.0], [3], 0, 1, 0.2, std_ddof=1)
    with pytest.raises(ValueError):   # target outside the vocabulary
        oracle.grpo(logits, np.array([0, 4, 0], np.int32), np.zeros(3), [0, 1], [1, 2], 0, 2, 0.2)


def test_logp_matches_library_log_softmax_and_lse_closed_form():
    logits, targets, _, _ = rand_case([5, 4], 37, 7)
    lse, logp, kl = oracle.grpo_logp(logits, targets)
    assert kl is None
    np.testing.assert_allclose(logp, lib_logp(logits, targets), atol=1e-13)
    np.testing.assert_allclose(lse, np.log(np.exp(logits).sum(axis=1)), atol=1e-12)
    # constant rows: lse = log V + c, logp = -log V
    c = np.full((3, 50), -2.5)
    lse_c, logp_c, _ = oracle.grpo_logp(c, np.array([0, 9, 49], np.int32))
    np.testing.assert_allclose(lse_c, np.log(50) - 2.5, atol=1e-14)
    np.testing.assert_allclose(logp_c, -np.log(50), atol=1e-14)
    # the loss oracle computes the same logp
    r = oracle.grpo(logits, targets, np.zeros(9), [0.0, 1.0], [5, 4], 0, 2, 0.2)
    np.testing.assert_array_equal(r.logp, logp)


def test_kl_estimate_closed_cases():
    """kl = exp(d) - d - 1 with d = ref - logp: zero when the policies agree, 1 - ln 2 at
    d = ln 2, e^-1 at d = -1, non-negative, and d^2/2 to third order for small d."""
    logits, targets, _, rng = rand_case([6, 6], 20, 8)
    lp = lib_logp(logits, targets)
    _, logp, kl = oracle.grpo_logp(logits, targets, lp)
    assert (kl == 0).all()
    d = np.array([np.log(2.0), -1.0, 0.0, 0.7, -2.3, 1e-3, -1e-3, 3.0, 0.1, -0.1, 2.0, -0.5])
    _, _, kl = oracle.grpo_logp(logits, targets, logp + d)
    np.testing.assert_allclose(kl[0], 1 - np.log(2.0), atol=1e-14)
    np.testing.assert_allclose(kl[1], np.exp(-1.0), atol=1e-14)
    assert (kl >= 0).all()
    small = np.abs(d) < 0.2
    np.testing.assert_allclose(kl[small], d[small] ** 2 / 2, atol=np.abs(d[small]).max() ** 3)


def test_logp_rejects_bad_arguments():
    with pytest.raises(ValueError):
        oracle.grpo_logp(np.zeros((2, 4)), np.array([0, 4], np.int32))
