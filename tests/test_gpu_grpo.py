"""GPU parity of the fused GRPO loss / logits gradient against the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
from parity_util import TOL_DLOGITS, TOL_LOGP, loss_tolerance, rel_err, u16
from response_replay_gb300 import synthetic as syn
from response_replay_gb300 import torch_api as api
from response_replay_gb300 import binding as B

pytestmark = pytest.mark.gpu


def host_logits(logits: torch.Tensor) -> np.ndarray:
    return u16(logits) if logits.dtype == torch.bfloat16 else logits.cpu().numpy()


def run_case(inp, eps, mb, me, std_ddof=1, rows_to_check=None, logp_old=None):
    """One call over members [mb, me); returns gpu outputs and the oracle result."""
    lens = inp.resp_lens.cpu().numpy()
    off = np.concatenate([[0], np.cumsum(lens)])
    t0, t1 = int(off[mb]), int(off[me])
    logits = inp.logits[t0:t1].contiguous()
    zl = host_logits(logits)
    targets = inp.targets[t0:t1].contiguous()
    if logp_old is None:
        # logp_old = logp + noise, logp from the oracle (fp64), rounded to fp32
        logp = oracle.grpo(zl, targets.cpu().numpy(), np.zeros(t1 - t0), inp.rewards.cpu().numpy(),
                           lens, mb, me, eps).logp
        logp_old = (logp + inp.noise[t0:t1].cpu().numpy()).astype(np.float32)
    lo = torch.from_numpy(np.asarray(logp_old, np.float32)).to(logits.device)
    loss, dlog, logp_gpu, stats = api.grpo_loss_fwd_bwd(logits, targets, lo, inp.rewards,
                                                        inp.resp_lens, mb, me, eps,
                                                        std_ddof=std_ddof)
    ref = oracle.grpo(zl, targets.cpu().numpy(), lo.cpu().numpy().astype(np.float64),
                      inp.rewards.cpu().numpy(), lens, mb, me, eps, 1e-6, std_ddof)
    return loss, dlog, logp_gpu, stats, ref, zl, targets.cpu().numpy()


def check(inp, eps, mb, me, dtype, std_ddof=1, rows=None, **kw):
    loss, dlog, logp_gpu, stats, ref, zl, tg = run_case(inp, eps, mb, me, std_ddof, **kw)
    assert abs(loss.item() - ref.loss) <= loss_tolerance(ref.loss, ref.adv), (loss.item(), ref.loss)
    assert np.abs(logp_gpu.cpu().numpy() - ref.logp).max() <= TOL_LOGP
    T = zl.shape[0]
    rows = range(T) if rows is None else rows
    near = np.abs(np.abs(ref.ratio - 1.0) - eps) < 1e-5      # clip-boundary ties excluded
    rows = [r for r in rows if not near[r]]
    g_ref = oracle.grpo_dlogits_rows(zl, rows, tg, ref.lse, ref.coef)
    g = dlog[rows].float().cpu().numpy()
    for i, r in enumerate(rows):
        scale = np.abs(g_ref[i]).max()
        if scale == 0:
            assert (g[i] == 0).all()
        else:
            assert np.abs(g[i] - g_ref[i]).max() / scale <= TOL_DLOGITS[dtype], r
    st = stats.cpu().numpy()
    assert st[0] == ref.zeroed.sum()
    return ref


# The small workload: V = 4096 fp32 logits N(0,2), G = 2 x 256, Bernoulli(0.5) rewards.
def test_small_workload(cuda):
    w = syn.WORKLOADS["p4k"]
    for seed_off in range(3):
        inp = syn.make_grpo(w.R, w.vocab, w.logits_dtype, w.rewards, syn.seed_of("p4k") + seed_off,
                            cuda)
        check(inp, 0.2, 0, w.G, "fp32")


@pytest.mark.parametrize("V,dtype", [(151936, "bf16"), (1001, "bf16"), (1001, "fp32"),
                                     (7, "fp32"), (33, "bf16")])
def test_vocab_sizes_and_alignment(cuda, V, dtype):
    lens = [5, 9, 3]
    inp = syn.make_grpo(lens, V, dtype, "normal", 100 + V, cuda, shift_frac=0.3)
    check(inp, 0.2, 0, 3, dtype)


def test_serial_member_calls_accumulate(cuda):
    """Serial replay: one call per member, each seeing the whole group's rewards, adding
    into one loss scalar; per-member gradients and the accumulated loss match."""
    lens = [40, 24, 64, 8]
    inp = syn.make_grpo(lens, 4096, "bf16", "uniform01", 31, cuda, shift_frac=0.2)
    off = np.concatenate([[0], np.cumsum(lens)])
    loss_acc = torch.zeros(1, dtype=torch.float32, device=cuda)
    total, adv = 0.0, None
    for i in range(4):
        ref = check(inp, 0.2, i, i + 1, "bf16")        # per-member parity (fresh loss)
        t0, t1 = int(off[i]), int(off[i + 1])
        logp_old = torch.from_numpy(
            (ref.logp + inp.noise[t0:t1].cpu().numpy()).astype(np.float32)).to(cuda)
        api.grpo_loss_fwd_bwd(inp.logits[t0:t1].contiguous(), inp.targets[t0:t1].contiguous(),
                              logp_old, inp.rewards, inp.resp_lens, i, i + 1, 0.2, loss=loss_acc,
                              accumulate=i > 0)
        total += ref.loss
        adv = ref.adv
    assert abs(loss_acc.item() - total) <= loss_tolerance(total, adv) + 1e-7


def test_equal_rewards_exact_zero(cuda):
    lens = [16, 16, 16]
    inp = syn.make_grpo(lens, 512, "bf16", "normal", 41, cuda)
    inp.rewards.fill_(0.3)
    loss, dlog, _, stats, ref, _, _ = run_case(inp, 0.2, 0, 3)
    assert loss.item() == 0.0 and ref.loss == 0.0
    assert (dlog == 0).all()


def test_std_ddof0(cuda):
    inp = syn.make_grpo([6, 6], 256, "fp32", "bernoulli0.5", 43, cuda)
    inp.rewards.copy_(torch.tensor([0.0, 1.0]))
    ref = check(inp, 0.2, 0, 2, "fp32", std_ddof=0)
    np.testing.assert_allclose(ref.adv, [-0.999998000004, 0.999998000004], atol=1e-12)


def test_length_mismatch_reported(cuda):
    inp = syn.make_grpo([4, 4], 64, "fp32", "normal", 47, cuda)
    bad = torch.tensor([4, 5], dtype=torch.int32, device=cuda)
    lo = torch.zeros(8, dtype=torch.float32, device=cuda)
    loss = torch.full((1,), 7.0, device=cuda)
    api.grpo_loss_fwd_bwd(inp.logits, inp.targets, lo, inp.rewards, bad, 0, 2, 0.2, loss=loss)
    assert B.ls_last_device_error(0) == B.LS_ERR_DEVICE_CHECK
    assert loss.item() == 7.0   # nothing written
