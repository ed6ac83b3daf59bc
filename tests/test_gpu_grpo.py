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


# Rows that are whole 16-byte units take the streamed kernel (bulk copies through a
# shared-memory ring of 30 KB chunks, the last six chunks of a row held for pass 2):
# 151,936 bf16 = 10 chunks (4 re-loaded), fp32 = 20 chunks, 92,160 bf16 = exactly the six
# held chunks, 107,512 bf16 = seven chunks with a ragged last one, 16 / 8 = one short
# chunk.  Other V (1001, 7, 33) take the one-CTA-per-row kernel.
@pytest.mark.parametrize("V,dtype", [(151936, "bf16"), (151936, "fp32"), (1001, "bf16"),
                                     (1001, "fp32"), (7, "fp32"), (33, "bf16"), (16, "bf16"),
                                     (8, "fp32"), (4104, "bf16"), (92160, "bf16"),
                                     (107512, "bf16")])
def test_vocab_sizes_and_alignment(cuda, V, dtype):
    lens = [5, 9, 3]
    inp = syn.make_grpo(lens, V, dtype, "normal", 100 + V, cuda, shift_frac=0.3)
    check(inp, 0.2, 0, 3, dtype)


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_unaligned_logits_buffer_rejected(cuda, dtype):
    """Device pointers must be 16-byte aligned: a logits view at an odd element offset is
    refused before any launch."""
    lens = [3, 4]
    V = 64
    inp = syn.make_grpo(lens, V, dtype, "normal", 211, cuda)
    buf = torch.empty(sum(lens) * V + 1, dtype=inp.logits.dtype, device=cuda)
    buf[1:].copy_(inp.logits.flatten())
    logits = buf[1:].view(sum(lens), V)
    assert logits.data_ptr() % 16 != 0
    lo = torch.zeros(sum(lens), dtype=torch.float32, device=cuda)
    with pytest.raises(B.LongstrawError):
        api.grpo_loss_fwd_bwd(logits, inp.targets, lo, inp.rewards, inp.resp_lens, 0, 2, 0.2)


def test_many_rows_per_cta(cuda):
    """T much larger than the number of CTAs: every ring stage is refilled many times and
    the held chunks of one row give way to the next row's."""
    lens = [700, 1100, 300, 948]
    inp = syn.make_grpo(lens, 40960, "bf16", "normal", 223, cuda, shift_frac=0.3)
    check(inp, 0.2, 0, 4, "bf16")


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


def test_member_slices_at_any_token_offset(cuda):
    """Ragged members: each call passes its member's slices of token-major buffers
    (logits rows stay 16-byte aligned; targets, logp_old and logp_out start at odd token
    offsets such as 37) without copies, and matches the oracle."""
    lens = [37, 90, 5, 128]
    inp = syn.make_grpo(lens, 4096, "bf16", "normal", 53, cuda, shift_frac=0.2)
    off = np.concatenate([[0], np.cumsum(lens)])
    zl = u16(inp.logits)
    tg = inp.targets.cpu().numpy()
    logp = oracle.grpo(zl, tg, np.zeros(off[-1]), inp.rewards.cpu().numpy(), lens, 0, 4, 0.2).logp
    lo = torch.from_numpy((logp + inp.noise.cpu().numpy()).astype(np.float32)).to(cuda)
    lp_out = torch.full((int(off[-1]),), float("nan"), device=cuda)
    for i in range(4):
        t0, t1 = int(off[i]), int(off[i + 1])
        loss, dlog, _, _ = api.grpo_loss_fwd_bwd(inp.logits[t0:t1], inp.targets[t0:t1], lo[t0:t1],
                                                 inp.rewards, inp.resp_lens, i, i + 1, 0.2,
                                                 logp_out=lp_out[t0:t1])
        ref = oracle.grpo(zl[t0:t1], tg[t0:t1], lo[t0:t1].cpu().numpy().astype(np.float64),
                          inp.rewards.cpu().numpy(), lens, i, i + 1, 0.2)
        assert abs(loss.item() - ref.loss) <= loss_tolerance(ref.loss, ref.adv)
        near = np.abs(np.abs(ref.ratio - 1.0) - 0.2) < 1e-5
        rows = [r for r in range(t1 - t0) if not near[r]]
        g_ref = oracle.grpo_dlogits_rows(zl[t0:t1], rows, tg[t0:t1], ref.lse, ref.coef)
        assert rel_err(dlog[rows].float().cpu().numpy(), g_ref) <= TOL_DLOGITS["bf16"]
    assert np.abs(lp_out.cpu().numpy() - logp).max() <= TOL_LOGP


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


# ---- pre-step scoring (log-softmax gather, KL estimate against a reference policy)

def check_logp(logits, targets, ref=None):
    zl = host_logits(logits)
    tg = targets.cpu().numpy()
    ref_t = None if ref is None else torch.from_numpy(ref.astype(np.float32)).to(logits.device)
    logp, lse, kl = api.grpo_logp(logits, targets, ref_t, with_lse=True)
    lse_ref, logp_ref, kl_ref = oracle.grpo_logp(zl, tg, None if ref is None else
                                                 ref.astype(np.float32).astype(np.float64))
    assert np.abs(logp.cpu().numpy() - logp_ref).max(initial=0.0) <= TOL_LOGP
    assert np.abs(lse.cpu().numpy() - lse_ref).max(initial=0.0) <= TOL_LOGP
    if ref is not None:
        # kl'(d) = e^d - 1, so an error e in logp moves kl by about |e^d - 1| e
        d = ref.astype(np.float32).astype(np.float64) - logp_ref
        tol = TOL_LOGP * np.abs(np.expm1(d)) + 1e-6
        assert (np.abs(kl.cpu().numpy() - kl_ref) <= tol).all()
        assert (kl.cpu().numpy() >= -1e-7).all()
    assert B.ls_last_device_error(0) == B.LS_OK


@pytest.mark.parametrize("T,V,dtype", [(9, 37, torch.float32), (128, 4096, torch.float32),
                                       (64, 1001, torch.bfloat16), (48, 151936, torch.bfloat16),
                                       (0, 64, torch.float32), (700, 12296, torch.bfloat16),
                                       (700, 12288, torch.float32)])
def test_grpo_logp_parity(cuda, T, V, dtype):
    g = torch.Generator(device="cpu").manual_seed(T * 131 + V)
    logits = (torch.randn(T, V, generator=g) * 2.0).to(dtype).to(cuda)
    targets = torch.randint(0, V, (T,), generator=g, dtype=torch.int32).to(cuda)
    check_logp(logits, targets)
    if T > 0:
        rng = np.random.default_rng(T + V)
        lp = oracle.grpo_logp(host_logits(logits), targets.cpu().numpy())[1]
        ref = lp + rng.choice([0.0, 1e-3, -0.4, 0.9, -2.0], size=T)
        check_logp(logits, targets, ref)


def test_grpo_logp_full_member(cuda):
    """The 2,097,152-position workload's first member: 4,096 tokens x 151,936 bf16 logits."""
    w = syn.WORKLOADS["p2m"]
    inp = syn.make_grpo(list(w.R[:1]), w.vocab, w.logits_dtype, w.rewards, syn.seed_of("p2m"),
                        cuda, shift_frac=w.shift_frac)
    lp = oracle.grpo_logp(host_logits(inp.logits), inp.targets.cpu().numpy())[1]
    check_logp(inp.logits, inp.targets, lp + inp.noise.cpu().numpy())


def test_grpo_logp_bad_target_reported(cuda):
    logits = torch.randn(4, 16, device=cuda)
    targets = torch.tensor([0, 16, 3, -1], dtype=torch.int32, device=cuda)
    logp, _, _ = api.grpo_logp(logits, targets)
    assert B.ls_last_device_error(0) == B.LS_ERR_DEVICE_CHECK
    lp = logp.cpu().numpy()
    assert np.isnan(lp[1]) and np.isnan(lp[3]) and np.isfinite(lp[[0, 2]]).all()


@pytest.mark.parametrize("V,dtype", [(151936, "bf16"), (1001, "fp32")])
def test_deterministic(cuda, V, dtype):
    """Whichever CTA finishes last and reduces the loss, the sum runs in one fixed order:
    repeated calls agree bit for bit (streamed kernel at V = 151,936 bf16, one-CTA-per-row
    kernel at V = 1001)."""
    lens = [300, 211, 97]
    inp = syn.make_grpo(lens, V, dtype, "normal", 333, cuda, shift_frac=0.3)
    lo = (torch.randn(sum(lens), device=cuda) * 0.05 - 12.0).contiguous()
    outs = []
    for _ in range(3):
        loss, dlog, logp, stats = api.grpo_loss_fwd_bwd(inp.logits, inp.targets, lo, inp.rewards,
                                                        inp.resp_lens, 0, 3, 0.2)
        outs.append((loss.clone(), dlog.clone(), logp.clone(), stats.clone()))
    for other in outs[1:]:
        for a, b in zip(outs[0], other):
            assert torch.equal(a, b)
