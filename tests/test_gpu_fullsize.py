"""Parity at the benchmark's full sizes, in the launch configuration bench.py times:
the oracle recomputes sampled outputs one by one (attention rows (t, h), response keys
near the end of the branch for dK/dV, GRPO token rows), and properties that hold at any
size are checked on the whole output."""
import numpy as np
import pytest
import torch

import oracle
from parity_util import TOL_DLOGITS, TOL_GRAD, TOL_LOGP, TOL_LSE, TOL_O, loss_tolerance, u16
from response_replay_gb300 import synthetic as syn
from response_replay_gb300 import torch_api as api

pytestmark = pytest.mark.gpu


def sample_rows(R, hq, n, seed):
    rng = np.random.default_rng(seed)
    ts = np.concatenate([[0, R - 1], rng.integers(0, R, n - 2)]).astype(np.int32)
    hs = rng.integers(0, hq, n).astype(np.int32)
    return ts, hs


def rel(x, ref):
    return float(np.abs(x - ref).max() / max(np.abs(ref).max(), 1e-30))


@pytest.mark.parametrize("name,nrows,keys,member,R_short", [
    ("p128k", 48, 6, 0, None), ("p1m", 24, 3, 0, None), ("p2m", 16, 2, 0, None),
    ("p4m_reuse", 8, 2, 5, None), ("p2m", 16, 2, 0, 48), ("p2m", 16, 2, 0, 16)])
def test_attention_full_size_sampled(cuda, name, nrows, keys, member, R_short):
    """p4m_reuse: P = 4,194,304 with one of its seeded ragged response lengths;
    R_short: the 2,097,152-position prompt replayed by a short response (packed heads)."""
    w = syn.WORKLOADS[name]
    seed = syn.seed_of(name)
    pr = syn.make_prompt(w.P, w.hkv, 128, w.page_size, seed, cuda)
    cache = api.PagedKVCache(pr.num_pages, pr.page_table, w.page_size, w.hkv, w.P, device=cuda)
    cache.capture(pr.k, pr.v)
    del pr
    R = w.R[member] if R_short is None else R_short
    br = syn.make_branch(R, w.hq, w.hkv, 128, seed + 1, cuda)
    scale = 128 ** -0.5
    o, lse = api.replay_fwd(cache, br.q, br.k, br.v, scale, w.num_splits)
    dq, dk, dv = api.replay_bwd(cache, br.q, br.k, br.v, o, lse, br.d_o, scale, w.num_splits)
    torch.cuda.synchronize()
    # whole-output properties
    for t in (o.float(), lse, dq, dk, dv):
        assert torch.isfinite(t).all()
    # sampled outputs against the oracle
    pb = oracle.AttnProblem(u16(cache.k_pool), u16(cache.v_pool), cache.page_table.cpu().numpy(),
                            w.P, u16(br.q), u16(br.k), u16(br.v), scale, w.num_splits)
    ts, hs = sample_rows(R, w.hq, nrows, seed)
    o_ref, lse_ref = oracle.attn_fwd_rows(pb, ts, hs)
    o_g = o.float().cpu().numpy()[ts, hs]
    assert rel(o_g, o_ref) <= TOL_O
    assert np.abs(lse.cpu().numpy()[ts, hs] - lse_ref).max() <= TOL_LSE
    d_o = u16(br.d_o)
    dq_ref = oracle.attn_bwd_dq_rows(pb, d_o, ts, hs)
    assert rel(dq.cpu().numpy()[ts, hs], dq_ref) <= TOL_GRAD
    js = np.repeat(np.arange(R - keys, R, dtype=np.int32), w.hkv)
    kvhs = np.tile(np.arange(w.hkv, dtype=np.int32), keys)
    dk_ref, dv_ref = oracle.attn_bwd_dkdv_keys(pb, d_o, js, kvhs)
    assert rel(dk.cpu().numpy()[js, kvhs], dk_ref) <= TOL_GRAD
    assert rel(dv.cpu().numpy()[js, kvhs], dv_ref) <= TOL_GRAD


@pytest.mark.parametrize("name", ["p128k", "p2m"])
def test_grpo_full_size_member(cuda, name):
    """One member's call (R_i tokens x V = 151936 bf16) with the whole group's rewards."""
    w = syn.WORKLOADS[name]
    inp = syn.make_grpo(w.R, w.vocab, w.logits_dtype, w.rewards, syn.seed_of(name), cuda,
                        shift_frac=w.shift_frac)
    lens = np.array(w.R, np.int32)
    i = 1
    t0, t1 = int(lens[:i].sum()), int(lens[:i + 1].sum())
    logits = inp.logits[t0:t1].contiguous()
    zl = u16(logits)
    tg = inp.targets[t0:t1].cpu().numpy()
    rewards = inp.rewards.cpu().numpy()
    logp = oracle.grpo(zl, tg, np.zeros(t1 - t0), rewards, lens, i, i + 1, 0.2).logp
    logp_old = (logp + inp.noise[t0:t1].cpu().numpy()).astype(np.float32)
    lo = torch.from_numpy(logp_old).to(cuda)
    loss, dlog, logp_gpu, stats = api.grpo_loss_fwd_bwd(logits, inp.targets[t0:t1].contiguous(),
                                                        lo, inp.rewards, inp.resp_lens, i, i + 1,
                                                        0.2)
    ref = oracle.grpo(zl, tg, logp_old.astype(np.float64), rewards, lens, i, i + 1, 0.2)
    assert abs(loss.item() - ref.loss) <= loss_tolerance(ref.loss, ref.adv)
    assert np.abs(logp_gpu.cpu().numpy() - ref.logp).max() <= TOL_LOGP
    rng = np.random.default_rng(7)
    rows = [r for r in rng.choice(t1 - t0, 24, replace=False)
            if abs(abs(ref.ratio[r] - 1) - 0.2) >= 1e-5]
    g_ref = oracle.grpo_dlogits_rows(zl, rows, tg, ref.lse, ref.coef)
    g = dlog[rows].float().cpu().numpy()
    for k in range(len(rows)):
        s = np.abs(g_ref[k]).max()
        assert (np.abs(g[k] - g_ref[k]).max() / s if s > 0 else np.abs(g[k]).max()) <= TOL_DLOGITS["bf16"]
    # every row of dlogits sums to ~0 (softmax gradient) - a property at any size
    sums = dlog.float().sum(1).cpu().numpy()
    assert np.abs(sums).max() <= 1e-2 * max(np.abs(ref.coef).max(), 1e-30) + 1e-6
