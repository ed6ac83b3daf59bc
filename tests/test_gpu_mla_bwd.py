"""GPU parity of the latent (MLA-style) replay backward against the fp64 oracle, through
the C ABI: dq and the response rows' gradient element by element at small sizes (several
row tiles, both dq parts, split pieces, ragged prompt tails, P = 0, one token per unit at
128 heads, response lengths over several 128-row key tiles, odd head counts), split-count
invariance and determinism, latent pages in pinned host memory (bit-identical to the
same pages in GPU memory), and sampled rows and keys over a 2,097,152-position prompt."""
import numpy as np
import pytest
import torch

import oracle
from parity_util import TOL_GRAD, rel_err, u16
from response_replay_gb300 import binding as B
from response_replay_gb300 import torch_api as api
from test_gpu_mla import SCALE, make, problem

pytestmark = pytest.mark.gpu


def run(cache, br, splits):
    o, lse = api.mla_replay_fwd(cache, br.q, br.lat, SCALE, splits)
    dq, dlat = api.mla_replay_bwd(cache, br.q, br.lat, o, lse, br.d_o, SCALE, splits)
    torch.cuda.synchronize()
    assert B.ls_last_device_error(0) == B.LS_OK
    return dq, dlat


@pytest.mark.parametrize("P,R,H,ps,splits,sharp", [
    (1000, 7, 16, 64, 3, True),
    (0, 40, 8, 32, 2, True),
    (777, 1, 128, 32, 5, True),
    (3000, 33, 64, 256, 1000, False),
    (129, 130, 4, 32, 1, True),
    (2048, 16, 64, 128, 7, True),
    (500, 300, 3, 64, 4, True),
    (0, 260, 1, 32, 1, True),
])
def test_mla_bwd_matches_oracle(cuda, P, R, H, ps, splits, sharp):
    cache, br = make(P, R, H, ps, 170 + P + R, cuda, sharp=sharp)
    dq, dlat = run(cache, br, splits)
    dq_ref, dlat_ref = oracle.mla_bwd(problem(cache, br, P), u16(br.d_o))
    dq_g, dl_g = dq.cpu().numpy(), dlat.cpu().numpy()
    assert np.isfinite(dq_g).all() and np.isfinite(dl_g).all()
    assert rel_err(dq_g, dq_ref) <= TOL_GRAD, rel_err(dq_g, dq_ref)
    assert rel_err(dl_g, dlat_ref) <= TOL_GRAD, rel_err(dl_g, dlat_ref)
    # the rotary part of the response rows takes the key term only, and it is not zero
    assert np.abs(dl_g[:, 512:]).max() > 0


def test_mla_bwd_split_count_and_determinism(cuda):
    """One forward, backwards at several split counts: partial dq sums differ only in
    fp32 order; the response rows' walk does not depend on the splits at all."""
    cache, br = make(4096, 20, 32, 64, 5, cuda)
    o, lse = api.mla_replay_fwd(cache, br.q, br.lat, SCALE, 4)

    def bwd(s):
        r = api.mla_replay_bwd(cache, br.q, br.lat, o, lse, br.d_o, SCALE, s)
        torch.cuda.synchronize()
        assert B.ls_last_device_error(0) == B.LS_OK
        return r
    outs = [bwd(s) for s in (1, 4, 64, 1000)]
    dq0, dl0 = outs[0]
    for dq, dl in outs[1:]:
        assert (dq - dq0).abs().max().item() <= 1e-5 * dq0.abs().max().item()
        assert torch.equal(dl, dl0)
    dq1, dl1 = bwd(64)
    assert torch.equal(dq1, outs[2][0]) and torch.equal(dl1, outs[2][1])


def test_mla_bwd_host_pool_matches_device_pool(cuda):
    P, R, H, ps = 3000, 24, 32, 128
    dev_cache, br = make(P, R, H, ps, 19, cuda)
    host_cache, _ = make(P, R, H, ps, 19, cuda, host_pool=True)
    assert not host_cache.pool.is_cuda and host_cache.pool.is_pinned()
    dq_d, dl_d = run(dev_cache, br, 8)
    dq_h, dl_h = run(host_cache, br, 8)
    assert torch.equal(dq_d, dq_h) and torch.equal(dl_d, dl_h)
    dq_ref, dl_ref = oracle.mla_bwd(problem(host_cache, br, P), u16(br.d_o))
    assert rel_err(dq_h.cpu().numpy(), dq_ref) <= TOL_GRAD
    assert rel_err(dl_h.cpu().numpy(), dl_ref) <= TOL_GRAD


def test_mla_bwd_bad_page_is_reported(cuda):
    cache, br = make(500, 4, 8, 32, 3, cuda)
    o, lse = api.mla_replay_fwd(cache, br.q, br.lat, SCALE, 2)
    torch.cuda.synchronize()
    assert B.ls_last_device_error(0) == B.LS_OK
    cache.page_table[2] = cache.pool.shape[0] + 5
    api.mla_replay_bwd(cache, br.q, br.lat, o, lse, br.d_o, SCALE, 2)
    assert B.ls_last_device_error(0) == B.LS_ERR_DEVICE_CHECK
    assert B.ls_last_device_error(0) == B.LS_OK


def test_mla_bwd_argument_checks(cuda):
    cache, br = make(300, 4, 8, 32, 3, cuda)
    o, lse = api.mla_replay_fwd(cache, br.q, br.lat, SCALE, 1)
    with pytest.raises(B.LongstrawError):      # non-positive scale
        api.mla_replay_bwd(cache, br.q, br.lat, o, lse, br.d_o, -1.0, 1)
    with pytest.raises(B.LongstrawError):      # no workspace
        B.ls_mla_replay_bwd(cache.struct, br.q.data_ptr(), br.lat.data_ptr(), o.data_ptr(),
                            lse.data_ptr(), br.d_o.data_ptr(), 4, 8, SCALE, 1,
                            o.data_ptr(), o.data_ptr(), 0, 0, 0)
    dq, dl = api.mla_replay_bwd(cache, br.q[:0], br.lat[:0], o[:0], lse[:0], br.d_o[:0],
                                SCALE, 1)   # R = 0: no-op
    assert dq.shape == (0, 8, 576) and dl.shape == (0, 576)


def test_mla_bwd_full_prompt_sampled(cuda):
    """2,097,152 latent positions in 256-row pages, 64 heads, a 64-token response with
    scores of unit spread: dq of sampled rows, the gradient of the last response rows."""
    P, R, H, ps = 2097152, 64, 64, 256
    cache, br = make(P, R, H, ps, 2027, cuda, extra_pages=1)
    dq, dlat = run(cache, br, 256)
    assert torch.isfinite(dq).all() and torch.isfinite(dlat).all()
    pb = problem(cache, br, P)
    g = u16(br.d_o)
    rng = np.random.default_rng(11)
    ts = np.concatenate([[0, R - 1], rng.integers(0, R, 4)]).astype(np.int32)
    hs = rng.integers(0, H, len(ts)).astype(np.int32)
    dq_ref = oracle.mla_bwd_dq_rows(pb, g, ts, hs)
    assert rel_err(dq.cpu().numpy()[ts, hs], dq_ref) <= TOL_GRAD
    js = np.array([R - 1, R - 2], np.int32)
    dl_ref = oracle.mla_bwd_dlat_keys(pb, g, js)
    assert rel_err(dlat.cpu().numpy()[js], dl_ref) <= TOL_GRAD
