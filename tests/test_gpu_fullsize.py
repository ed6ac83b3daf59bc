"""Parity at the benchmark's full sizes, in the launch configuration bench.py times:
the oracle recomputes sampled outputs one by one (attention rows (t, h), the last keys
of the response for dK/dV on every KV head, GRPO token rows), and properties that hold
at any size are checked on the whole output.

Each prompt size runs twice: with the workloads' near-uniform inputs (Q, K ~
N(0,1)/sqrt(128), scores of spread ~0.008) and with sharp inputs (Q, K ~ N(0,1), scores
of unit spread), which gives the running max, the compensated row sums over millions
of keys and the log-sum-exp merge of hundreds of splits real dynamic range.  The first
keys of long responses are covered in tests/test_gpu_long_response.py."""
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


_CACHES = {}


def full_cache(name, sharp, device):
    """The workload's captured prompt (one at a time is kept: the 4,194,304-position
    pools hold 8.6 GB)."""
    key = (name, sharp)
    if key not in _CACHES:
        _CACHES.clear()
        torch.cuda.empty_cache()
        w = syn.WORKLOADS[name]
        seed = syn.seed_of(name)
        pr = syn.make_prompt(w.P, w.hkv, 128, w.page_size, seed, device, sharp=sharp)
        cache = api.PagedKVCache(pr.num_pages, pr.page_table, w.page_size, w.hkv, w.P,
                                 device=device)
        cache.capture(pr.k, pr.v)
        del pr
        torch.cuda.synchronize()
        _CACHES[key] = (cache, u16(cache.k_pool), u16(cache.v_pool),
                        cache.page_table.cpu().numpy())
    return _CACHES[key]


# (workload, sampled rows, end keys per KV head, replay index, short R, sharp).  For the
# 4,194,304-position prompt, replays from three of its eight cycles (the longest R of
# all 64, 8,164 tokens, is replay 28); R_short replays the 2,097,152-position prompt with
# a short response (grouped-query packing).
CASES = [
    ("p128k", 48, 6, 0, None, False), ("p128k", 48, 6, 3, None, True),
    ("p1m", 24, 3, 0, None, False), ("p1m", 24, 3, 5, None, True),
    ("p2m", 16, 2, 0, None, False), ("p2m", 16, 2, 7, None, True),
    ("p4m_reuse", 8, 2, 5, None, False), ("p4m_reuse", 8, 2, 28, None, True),
    ("p4m_reuse", 8, 2, 59, None, True),
    ("p2m", 16, 2, 0, 48, False), ("p2m", 16, 2, 0, 16, True),
]


@pytest.mark.parametrize("name,nrows,keys,member,R_short,sharp", CASES)
def test_attention_full_size_sampled(cuda, name, nrows, keys, member, R_short, sharp):
    w = syn.WORKLOADS[name]
    seed = syn.seed_of(name)
    cache, kp, vp, pt = full_cache(name, sharp, cuda)
    R = w.R[member] if R_short is None else R_short
    br = syn.make_branch(R, w.hq, w.hkv, 128, seed + 1 + member, cuda, sharp=sharp)
    scale = 128 ** -0.5
    o, lse = api.replay_fwd(cache, br.q, br.k, br.v, scale, w.num_splits)
    dq, dk, dv = api.replay_bwd(cache, br.q, br.k, br.v, o, lse, br.d_o, scale, w.num_splits)
    torch.cuda.synchronize()
    # whole-output properties
    for t in (o.float(), lse, dq, dk, dv):
        assert torch.isfinite(t).all()
    # sampled outputs against the oracle
    pb = oracle.AttnProblem(kp, vp, pt, w.P, u16(br.q), u16(br.k), u16(br.v), scale,
                            w.num_splits)
    ts, hs = sample_rows(R, w.hq, nrows, seed + member)
    o_ref, lse_ref = oracle.attn_fwd_rows(pb, ts, hs)
    o_g = o.float().cpu().numpy()[ts, hs]
    assert rel(o_g, o_ref) <= TOL_O
    assert np.abs(lse.cpu().numpy()[ts, hs] - lse_ref).max() <= TOL_LSE
    if sharp:  # the rows are not near-uniform: the LSE sits well above log(P + t + 1)
        assert np.abs(lse_ref - np.log(w.P + ts + 1.0)).max() > 0.1
    d_o = u16(br.d_o)
    dq_ref = oracle.attn_bwd_dq_rows(pb, d_o, ts, hs)
    assert rel(dq.cpu().numpy()[ts, hs], dq_ref) <= TOL_GRAD
    js = np.repeat(np.arange(R - keys, R, dtype=np.int32), w.hkv)
    kvhs = np.tile(np.arange(w.hkv, dtype=np.int32), keys)
    dk_ref, dv_ref = oracle.attn_bwd_dkdv_keys(pb, d_o, js, kvhs)
    assert rel(dk.cpu().numpy()[js, kvhs], dk_ref) <= TOL_GRAD
    assert rel(dv.cpu().numpy()[js, kvhs], dv_ref) <= TOL_GRAD


@pytest.mark.parametrize("name", ["p128k", "p1m", "p2m"])
def test_grpo_full_size_member(cuda, name):
    """One member's call (R_i tokens x V = 151936 bf16) with the whole group's rewards.
    p1m shifts about 20% of the old log-probabilities by +-0.5, so the clip zeroes the
    gradient of many tokens: their count must match the oracle's."""
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
    near = np.abs(np.abs(ref.ratio - 1) - 0.2) < 1e-5       # clip-boundary ties
    rng = np.random.default_rng(7)
    rows = [r for r in rng.choice(t1 - t0, 24, replace=False) if not near[r]]
    if w.shift_frac > 0:  # rows whose gradient the clip zeroed are among the checked ones
        rows += [int(r) for r in np.flatnonzero((ref.zeroed != 0) & ~near)[:8]]
    g_ref = oracle.grpo_dlogits_rows(zl, rows, tg, ref.lse, ref.coef)
    g = dlog[rows].float().cpu().numpy()
    for k in range(len(rows)):
        s = np.abs(g_ref[k]).max()
        assert (np.abs(g[k] - g_ref[k]).max() / s if s > 0 else np.abs(g[k]).max()) <= TOL_DLOGITS["bf16"]
    # every row of dlogits sums to ~0 (softmax gradient) - a property at any size
    sums = dlog.float().sum(1).cpu().numpy()
    assert np.abs(sums).max() <= 1e-2 * max(np.abs(ref.coef).max(), 1e-30) + 1e-6
    # tokens whose gradient the clip zeroed: the same count up to boundary ties
    st = stats.cpu().numpy()
    assert abs(float(st[0]) - float(ref.zeroed.sum())) <= near.sum()
    if w.shift_frac > 0:
        assert ref.zeroed.sum() > 0.02 * (t1 - t0)
