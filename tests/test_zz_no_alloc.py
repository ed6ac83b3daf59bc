"""The allocation-free GRPO entry point (ls_grpo_loss_fwd_bwd_noalloc).

It exists for callers that cannot allocate device memory when they compute the loss
(a host framework that plans all device memory in advance and allows no allocation
mid-step). It must give the same results as ls_grpo_loss_fwd_bwd, call after call,
even though every call reuses the same library-owned scratch array. This file is
collected last, so a run that stops at the first failure has run every other test.
"""
import numpy as np
import pytest
import torch

import oracle
from parity_util import TOL_DLOGITS, TOL_LOGP, loss_tolerance, u16
from response_replay_gb300 import binding as B
from response_replay_gb300 import synthetic as syn
from response_replay_gb300 import torch_api as api

pytestmark = pytest.mark.gpu


def _noalloc(inp, logp_old, mb, me, eps, loss, dlog, logp, stats, accumulate=False):
    T, V = inp.logits.shape
    dt = B.LS_BF16 if inp.logits.dtype == torch.bfloat16 else B.LS_FP32
    B.ls_grpo_loss_fwd_bwd_noalloc(
        inp.logits.data_ptr(), dt, T, V, inp.targets.data_ptr(), logp_old.data_ptr(),
        inp.rewards.data_ptr(), inp.resp_lens.data_ptr(), inp.rewards.numel(), mb, me, eps,
        1e-6, 1, int(accumulate), loss.data_ptr(), dlog.data_ptr(), logp.data_ptr(),
        stats.data_ptr(), torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("dtype,V", [("bf16", 151936), ("fp32", 1001)])
def test_noalloc_matches_workspace_entry_point_twice(cuda, dtype, V):
    lens = [37, 64, 21]
    for call in range(2):  # two calls in a row share (and reuse) the scratch array
        inp = syn.make_grpo(lens, V, dtype, "normal", 900 + 7 * call + V, cuda, shift_frac=0.3)
        # logp_old = logp + noise, logp from the library's own (workspace) entry point
        lp0 = torch.zeros(sum(lens), dtype=torch.float32, device=cuda)
        _, _, logp, _ = api.grpo_loss_fwd_bwd(inp.logits, inp.targets, lp0, inp.rewards,
                                              inp.resp_lens, 0, 3, 0.2)
        logp_old = (logp + inp.noise).contiguous()
        ref_loss, ref_dlog, ref_logp, ref_stats = api.grpo_loss_fwd_bwd(
            inp.logits, inp.targets, logp_old, inp.rewards, inp.resp_lens, 0, 3, 0.2)
        loss = torch.full((1,), 123.0, device=cuda)
        dlog = torch.full_like(inp.logits, float("nan"))
        logp_n = torch.full_like(logp, float("nan"))
        stats = torch.full((4,), float("nan"), device=cuda)
        _noalloc(inp, logp_old, 0, 3, 0.2, loss, dlog, logp_n, stats)
        torch.cuda.synchronize()
        assert B.ls_last_device_error(0) == B.LS_OK
        r = ref_loss.item()
        assert abs(loss.item() - r) <= loss_tolerance(r, np.ones(1)) + 1e-7
        assert (logp_n - ref_logp).abs().max().item() <= TOL_LOGP
        g, gr = dlog.float(), ref_dlog.float()
        scale = gr.abs().amax(dim=1).clamp_min(1e-30)
        assert ((g - gr).abs().amax(dim=1) / scale).max().item() <= TOL_DLOGITS[dtype]
        assert torch.equal(stats[0], ref_stats[0])
        assert (stats[1:] - ref_stats[1:]).abs().max().item() <= 1e-4 * max(1.0, ref_stats[1].abs().item())
        # and against the fp64 oracle directly
        zl = u16(inp.logits) if dtype == "bf16" else inp.logits.cpu().numpy()
        o = oracle.grpo(zl, inp.targets.cpu().numpy(), logp_old.cpu().numpy().astype(np.float64),
                        inp.rewards.cpu().numpy(), np.array(lens), 0, 3, 0.2)
        assert abs(loss.item() - o.loss) <= loss_tolerance(o.loss, o.adv)
        assert np.abs(logp_n.cpu().numpy() - o.logp).max() <= TOL_LOGP
        near = np.abs(np.abs(o.ratio - 1.0) - 0.2) < 1e-5
        rows = [r for r in range(0, sum(lens), 7) if not near[r]]
        g_ref = oracle.grpo_dlogits_rows(zl, rows, inp.targets.cpu().numpy(), o.lse, o.coef)
        g_rows = dlog[rows].float().cpu().numpy()
        for k in range(len(rows)):
            s = np.abs(g_ref[k]).max()
            err = np.abs(g_rows[k] - g_ref[k]).max() / s if s > 0 else np.abs(g_rows[k]).max()
            assert err <= TOL_DLOGITS[dtype], rows[k]


def test_noalloc_serial_member_accumulation(cuda):
    """Serial replay: one call per member into one loss scalar, as with the workspace form."""
    lens = [40, 24, 64]
    inp = syn.make_grpo(lens, 4096, "bf16", "uniform01", 77, cuda)
    logp_old = (inp.noise * 0).contiguous()
    off = np.concatenate([[0], np.cumsum(lens)])
    ref = torch.zeros(1, device=cuda)
    got = torch.zeros(1, device=cuda)
    stats = torch.empty(4, device=cuda)
    for i in range(3):
        s, e = int(off[i]), int(off[i + 1])
        sub = syn.GrpoInputs(inp.logits[s:e].contiguous(), inp.targets[s:e].contiguous(),
                             inp.rewards, inp.resp_lens, inp.noise[s:e])
        api.grpo_loss_fwd_bwd(sub.logits, sub.targets, logp_old[s:e].contiguous(), inp.rewards,
                              inp.resp_lens, i, i + 1, 0.2, loss=ref, accumulate=i > 0)
        _noalloc(sub, logp_old[s:e].contiguous(), i, i + 1, 0.2, got,
                 torch.empty_like(sub.logits), torch.empty(e - s, device=cuda), stats,
                 accumulate=i > 0)
    torch.cuda.synchronize()
    assert abs(got.item() - ref.item()) <= loss_tolerance(ref.item(), np.ones(1)) + 1e-7


def test_noalloc_largest_group(cuda):
    """G = 1,024 members (the largest member tables the scratch holds), two tokens of a
    few members in the call, against the workspace entry point."""
    G = 1024
    lens = torch.full((G,), 2, dtype=torch.int32, device=cuda)
    mb, me = 1000, 1003
    inp = syn.make_grpo([2] * (me - mb), 64, "fp32", "normal", 5, cuda)
    rewards = torch.randn(G, generator=syn.gen(cuda, 6), device=cuda)
    lo = inp.noise.contiguous()
    ref_loss, ref_dlog, ref_logp, _ = api.grpo_loss_fwd_bwd(inp.logits, inp.targets, lo, rewards,
                                                            lens, mb, me, 0.2)
    big = syn.GrpoInputs(inp.logits, inp.targets, rewards, lens, inp.noise)
    loss = torch.zeros(1, device=cuda)
    dlog = torch.empty_like(inp.logits)
    logp = torch.empty(inp.logits.shape[0], device=cuda)
    stats = torch.empty(4, device=cuda)
    _noalloc(big, lo, mb, me, 0.2, loss, dlog, logp, stats)
    torch.cuda.synchronize()
    assert B.ls_last_device_error(0) == B.LS_OK
    assert abs(loss.item() - ref_loss.item()) <= loss_tolerance(ref_loss.item(), np.ones(1)) + 1e-9
    assert torch.equal(logp, ref_logp)
    assert (dlog - ref_dlog).abs().max().item() <= 1e-6 * ref_dlog.abs().max().item()


def test_noalloc_rejects_sizes_beyond_its_scratch(cuda):
    logits = torch.empty((1, 8), dtype=torch.float32, device=cuda)  # never read
    t = torch.zeros(2048, dtype=torch.int32, device=cuda)
    f = torch.zeros(2048, device=cuda)
    for T, G in ((262145, 2), (2, 1025)):
        with pytest.raises(B.LongstrawError) as ei:
            B.ls_grpo_loss_fwd_bwd_noalloc(logits.data_ptr(), B.LS_FP32, T, 8, t.data_ptr(),
                                           f.data_ptr(), f.data_ptr(), t.data_ptr(), G, 0, 2,
                                           0.2, 1e-6, 1, 0, f.data_ptr(), logits.data_ptr(), None,
                                           None, 0)
        assert ei.value.status == B.LS_ERR_WORKSPACE


def test_noalloc_call_captured_in_a_cuda_graph(cuda):
    """After one eager call (which looks up the scratch array on this device), the call
    can be captured in a CUDA graph; replaying the graph gives bit-identical outputs to an
    eager call on the same inputs."""
    lens = [40, 25, 63]
    inp = syn.make_grpo(lens, 2048, "bf16", "normal", 4242, cuda, shift_frac=0.3)
    logp_old = inp.noise.contiguous()
    T = sum(lens)
    outs = [(torch.zeros(1, device=cuda), torch.empty_like(inp.logits),
             torch.empty(T, device=cuda), torch.empty(4, device=cuda)) for _ in range(2)]
    _noalloc(inp, logp_old, 0, 3, 0.2, *outs[0])          # eager (first call on the device)
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            _noalloc(inp, logp_old, 0, 3, 0.2, *outs[1])
    torch.cuda.current_stream().wait_stream(s)
    for t in outs[1]:
        t.fill_(float("nan"))                              # every output is written anew
    graph.replay()
    torch.cuda.synchronize()
    assert B.ls_last_device_error(0) == B.LS_OK
    for a, b in zip(outs[0], outs[1]):
        assert torch.equal(a, b)
