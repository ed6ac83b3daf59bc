"""The library's calls inside a CUDA graph: they are stream-ordered, allocate nothing
once the workspaces exist and never synchronize, so a replay step captured once and
replayed gives bit-identical results to eager calls, also after its inputs change in
place."""
import numpy as np
import pytest
import torch

from parity_util import Case
from response_replay_gb300 import binding as B
from response_replay_gb300 import synthetic as syn
from response_replay_gb300 import torch_api as api

pytestmark = pytest.mark.gpu


def test_replay_step_in_a_cuda_graph(cuda):
    P, R, hq, hkv, ps, splits = 2048, 200, 8, 2, 64, 3
    case = Case(P, R, hq, hkv, ps, splits, seed=71, device=cuda, sharp=True)
    br, cache, scale = case.br, case.cache, case.scale
    pk = case.prompt.k[:P].contiguous()
    pv = case.prompt.v[:P].contiguous()
    lens = [R, 150]
    g = syn.make_grpo(lens, 4096, "bf16", "normal", 72, cuda, shift_frac=0.3)
    logits = g.logits[:R].contiguous()
    targets = g.targets[:R].contiguous()
    logp_old = (torch.randn(R, device=cuda) * 0.05 - 8.0).contiguous()
    M, Rs = 3, 5
    sq = torch.stack([syn.make_branch(Rs, hq, hkv, 128, 80 + m, cuda).q for m in range(M)])
    sk = torch.stack([syn.make_branch(Rs, hq, hkv, 128, 90 + m, cuda).k for m in range(M)])
    sv = torch.stack([syn.make_branch(Rs, hq, hkv, 128, 95 + m, cuda).v for m in range(M)])
    sq, sk, sv = sq.contiguous(), sk.contiguous(), sv.contiguous()

    o = torch.empty_like(br.q)
    lse = torch.empty((R, hq), dtype=torch.float32, device=cuda)
    dq = torch.empty((R, hq, 128), dtype=torch.float32, device=cuda)
    dk = torch.empty((R, hkv, 128), dtype=torch.float32, device=cuda)
    dv = torch.empty_like(dk)
    loss = torch.zeros(1, dtype=torch.float32, device=cuda)
    dlog = torch.empty_like(logits)
    lp = torch.empty(R, dtype=torch.float32, device=cuda)
    stats = torch.empty(4, dtype=torch.float32, device=cuda)
    mo = torch.empty_like(sq)
    mlse = torch.empty(sq.shape[:3], dtype=torch.float32, device=cuda)
    s_lp = torch.empty(R, dtype=torch.float32, device=cuda)
    s_kl = torch.empty(R, dtype=torch.float32, device=cuda)

    def step():
        cache.capture(pk, pv)
        api.replay_fwd(cache, br.q, br.k, br.v, scale, splits, o=o, lse=lse)
        api.grpo_loss_fwd_bwd(logits, targets, logp_old, g.rewards, g.resp_lens, 0, 1, 0.2,
                              loss=loss, dlogits=dlog, logp_out=lp, stats=stats)
        api.replay_bwd(cache, br.q, br.k, br.v, o, lse, br.d_o, scale, splits, dq=dq, dk=dk,
                       dv=dv)
        api.replay_fwd_members(cache, sq, sk, sv, scale, splits, o=mo, lse=mlse)
        B.ls_grpo_logp(logits.data_ptr(), B.LS_BF16, R, 4096, targets.data_ptr(),
                       logp_old.data_ptr(), s_lp.data_ptr(), 0, s_kl.data_ptr(),
                       torch.cuda.current_stream().cuda_stream)

    outs = (o, lse, dq, dk, dv, loss, dlog, lp, stats, mo, mlse, s_lp, s_kl)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # eager warm-up: every workspace exists before capture
        step()
        step()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    eager = [t.clone() for t in outs]

    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for t in outs:
        t.fill_(float("nan")) if t.is_floating_point() else t.zero_()
    graph.replay()
    torch.cuda.synchronize()
    assert B.ls_last_device_error(0) == B.LS_OK
    for a, b in zip(outs, eager):
        assert torch.equal(a, b)

    # new inputs, same buffers: the replay follows them
    br.q.mul_(0.5)
    logits.mul_(1.5)
    sq.mul_(-1.0)
    graph.replay()
    torch.cuda.synchronize()
    replayed = [t.clone() for t in outs]
    step()
    torch.cuda.synchronize()
    for a, b in zip(replayed, outs):
        assert torch.equal(a, b)
    assert not torch.equal(replayed[0], eager[0])


def test_latent_replay_in_a_cuda_graph(cuda):
    """The latent capture, forward and backward captured once: replays bit-identical to
    eager calls, and they follow the inputs when these change in place."""
    P, R, H, ps, splits, scale = 3000, 70, 16, 64, 5, 192 ** -0.5
    pr = syn.make_latent_prompt(P, ps, 401, cuda, extra_pages=1)
    lat = pr.lat[:P].contiguous()
    cache = api.LatentCache(pr.num_pages, pr.page_table, ps, P, device=cuda)
    br = syn.make_latent_branch(R, H, 402, cuda, sharp=True)
    o = torch.empty((R, H, 512), dtype=torch.bfloat16, device=cuda)
    lse = torch.empty((R, H), dtype=torch.float32, device=cuda)
    dq = torch.empty((R, H, 576), dtype=torch.float32, device=cuda)
    dl = torch.empty((R, 576), dtype=torch.float32, device=cuda)

    def step():
        cache.capture(lat)
        api.mla_replay_fwd(cache, br.q, br.lat, scale, splits, o=o, lse=lse)
        api.mla_replay_bwd(cache, br.q, br.lat, o, lse, br.d_o, scale, splits, dq=dq, dlat=dl)

    outs = (o, lse, dq, dl)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # eager warm-up: every workspace exists before capture
        step()
        step()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    eager = [t.clone() for t in outs]

    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for t in outs:
        t.fill_(float("nan"))
    graph.replay()
    torch.cuda.synchronize()
    assert B.ls_last_device_error(0) == B.LS_OK
    for a, b in zip(outs, eager):
        assert torch.equal(a, b)

    br.q.mul_(0.5)
    br.d_o.mul_(-1.0)
    graph.replay()
    torch.cuda.synchronize()
    replayed = [t.clone() for t in outs]
    step()
    torch.cuda.synchronize()
    for a, b in zip(replayed, outs):
        assert torch.equal(a, b)
    assert not torch.equal(replayed[2], eager[2])
