"""GPU parity of Gated-DeltaNet replay from a captured state (ls_gdn_replay_fwd / _bwd)
against the fp64 token-by-token oracle, element by element: chunk-aligned and ragged
lengths, one and several heads, the capture (running a prompt from a zero state) and
replay from the captured state, accumulation, and the 4,096-token, 32-head layer."""
import numpy as np
import pytest
import torch

import oracle
from parity_util import rel_err, u16
from response_replay_gb300 import binding as B
from response_replay_gb300 import synthetic as syn
from response_replay_gb300 import torch_api as api

pytestmark = pytest.mark.gpu

TOL_O = 1e-2      # o is bf16
TOL_F32 = 1e-3    # fp32 outputs (state, gradients), relative to the tensor's max


def problem(inp, scale):
    return oracle.GdnProblem(inp.state0.double().cpu().numpy(), u16(inp.q), u16(inp.k), u16(inp.v),
                             inp.g.double().cpu().numpy(), inp.beta.double().cpu().numpy(), scale)


def check(inp, scale, grads=True):
    o, s_out = api.gdn_replay_fwd(inp.state0, inp.q, inp.k, inp.v, inp.g, inp.beta, scale,
                                  with_state=True)
    torch.cuda.synchronize()
    pb = problem(inp, scale)
    o_ref, s_ref = oracle.gdn_fwd(pb)
    assert rel_err(o.float().cpu().numpy(), o_ref) <= TOL_O
    assert rel_err(s_out.cpu().numpy(), s_ref) <= TOL_F32
    if grads:
        got = api.gdn_replay_bwd(inp.state0, inp.q, inp.k, inp.v, inp.g, inp.beta, inp.d_o, scale)
        torch.cuda.synchronize()
        ref = oracle.gdn_bwd(pb, u16(inp.d_o))
        for name, x, r in zip(("dq", "dk", "dv", "dg", "dbeta"), got, ref):
            e = rel_err(x.cpu().numpy(), r)
            assert e <= TOL_F32, (name, e)
    assert B.ls_last_device_error(0) == B.LS_OK


@pytest.mark.parametrize("R,H", [(1, 1), (37, 2), (64, 1), (130, 3), (300, 2), (512, 4)])
def test_gdn_matches_oracle(cuda, R, H):
    inp = syn.make_gdn(R, H, 100 + R + H, cuda)
    check(inp, 128 ** -0.5)


def test_gdn_strong_decay_and_writes(cuda):
    """Fast decay (exp(g) in [0.3, 0.7]) and large states: the within-chunk decay ratios
    span many orders of magnitude."""
    inp = syn.make_gdn(200, 2, 7, cuda, decay=(0.3, 0.7), state_std=3.0)
    check(inp, 0.2)


def test_gdn_capture_then_replay(cuda):
    """Running the prompt from a zero state and keeping state_out (the capture), then
    replaying the response from it, gives the response outputs of running the whole
    sequence, and matches the oracle's replay."""
    Pn, R, H = 192, 100, 2
    whole = syn.make_gdn(Pn + R, H, 11, cuda)
    zero = torch.zeros_like(whole.state0)
    _, captured = api.gdn_replay_fwd(zero, whole.q[:Pn].contiguous(), whole.k[:Pn].contiguous(),
                                     whole.v[:Pn].contiguous(), whole.g[:Pn].contiguous(),
                                     whole.beta[:Pn].contiguous(), 0.1, with_state=True)
    o_tail, _ = api.gdn_replay_fwd(captured, whole.q[Pn:].contiguous(), whole.k[Pn:].contiguous(),
                                   whole.v[Pn:].contiguous(), whole.g[Pn:].contiguous(),
                                   whole.beta[Pn:].contiguous(), 0.1)
    o_whole, _ = api.gdn_replay_fwd(zero, whole.q, whole.k, whole.v, whole.g, whole.beta, 0.1)
    torch.cuda.synchronize()
    assert (o_tail.float() - o_whole[Pn:].float()).abs().max().item() <= 2e-2 * o_whole.float().abs().max().item()
    pb = oracle.GdnProblem(np.zeros((H, 128, 128)), u16(whole.q), u16(whole.k), u16(whole.v),
                           whole.g.double().cpu().numpy(), whole.beta.double().cpu().numpy(), 0.1)
    o_ref, _ = oracle.gdn_fwd(pb)
    assert rel_err(o_tail.float().cpu().numpy(), o_ref[Pn:]) <= TOL_O


def test_gdn_accumulate_and_zero_length(cuda):
    inp = syn.make_gdn(70, 2, 13, cuda)
    g1 = api.gdn_replay_bwd(inp.state0, inp.q, inp.k, inp.v, inp.g, inp.beta, inp.d_o, 0.1)
    g2 = api.gdn_replay_bwd(inp.state0, inp.q, inp.k, inp.v, inp.g, inp.beta, inp.d_o, 0.1,
                            grads=tuple(x.clone() for x in g1), accumulate=True)
    for a, b in zip(g1, g2):
        torch.testing.assert_close(b, 2 * a, rtol=1e-6, atol=1e-6)
    empty = syn.make_gdn(0, 2, 14, cuda)
    _, s = api.gdn_replay_fwd(inp.state0, empty.q, empty.k, empty.v, empty.g, empty.beta, 0.1,
                              with_state=True)
    torch.cuda.synchronize()
    assert torch.equal(s, inp.state0)


def test_gdn_full_layer(cuda):
    """One layer's replay at the benchmark's size: 4,096 response tokens, 32 heads."""
    inp = syn.make_gdn(4096, 32, 17, cuda)
    check(inp, 128 ** -0.5)
