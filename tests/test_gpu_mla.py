"""GPU parity of the latent (MLA-style) replay forward against the fp64 oracle, through
the C ABI: element by element at small sizes (several row tiles and split pieces,
ragged prompt tails, P = 0, one token per tile at 128 heads), latent pages in pinned
host memory (bit-identical to the same pages in GPU memory), layers streamed from host
memory through the two-slot GPU page cache, the capture, a bad page id, and sampled rows
over a 2,097,152-position prompt."""
import numpy as np
import pytest
import torch

import oracle
from parity_util import TOL_LSE, TOL_O, rel_err, u16
from response_replay_gb300 import binding as B
from response_replay_gb300 import synthetic as syn
from response_replay_gb300 import torch_api as api

pytestmark = pytest.mark.gpu

SCALE = 192 ** -0.5


def make(P, R, H, ps, seed, device, sharp=True, host_pool=False, extra_pages=2):
    pr = syn.make_latent_prompt(max(P, 1), ps, seed, device, extra_pages=extra_pages)
    pt = pr.page_table if P > 0 else pr.page_table[:0]
    cache = api.LatentCache(pr.num_pages, pt, ps, P, device=device, fill=float("nan"),
                            host_pool=host_pool)
    if P > 0:
        cache.capture(pr.lat[:P].contiguous())
    br = syn.make_latent_branch(R, H, seed + 1, device, sharp=sharp)
    return cache, br


def problem(cache, br, P):
    torch.cuda.synchronize()
    pt = cache.page_table.cpu().numpy() if P > 0 else np.zeros(1, np.int32)
    return oracle.MlaProblem(u16(cache.pool), pt, P, u16(br.q), u16(br.lat), SCALE)


@pytest.mark.parametrize("P,R,H,ps,splits,sharp", [
    (1000, 7, 16, 64, 3, True),
    (0, 40, 8, 32, 2, True),
    (777, 1, 128, 32, 5, True),
    (3000, 33, 64, 256, 1000, False),
    (129, 130, 4, 32, 1, True),
    (2048, 16, 64, 128, 7, True),
    (5000, 3, 20, 64, 16, True),
])
def test_mla_fwd_matches_oracle(cuda, P, R, H, ps, splits, sharp):
    cache, br = make(P, R, H, ps, 70 + P + R, cuda, sharp=sharp)
    o, lse = api.mla_replay_fwd(cache, br.q, br.lat, SCALE, splits)
    torch.cuda.synchronize()
    assert B.ls_last_device_error(0) == B.LS_OK
    o_ref, lse_ref = oracle.mla_fwd(problem(cache, br, P))
    o_g = o.float().cpu().numpy()
    assert np.isfinite(o_g).all()
    assert rel_err(o_g, o_ref) <= TOL_O
    assert float(np.abs(lse.cpu().numpy() - lse_ref).max()) <= TOL_LSE


def test_mla_split_count_and_determinism(cuda):
    cache, br = make(4096, 20, 32, 64, 5, cuda)
    outs = [api.mla_replay_fwd(cache, br.q, br.lat, SCALE, s) for s in (1, 4, 64, 1000)]
    o0, l0 = outs[0]
    for o, l in outs[1:]:
        assert (o.float() - o0.float()).abs().max().item() <= 2 ** -6
        assert (l - l0).abs().max().item() <= 1e-5
    o1, l1 = api.mla_replay_fwd(cache, br.q, br.lat, SCALE, 64)
    assert torch.equal(o1, outs[2][0]) and torch.equal(l1, outs[2][1])


def test_mla_host_pool_matches_device_pool(cuda):
    P, R, H, ps = 3000, 24, 32, 128
    dev_cache, br = make(P, R, H, ps, 9, cuda)
    host_cache, _ = make(P, R, H, ps, 9, cuda, host_pool=True)
    assert not host_cache.pool.is_cuda and host_cache.pool.is_pinned()
    o_d, l_d = api.mla_replay_fwd(dev_cache, br.q, br.lat, SCALE, 8)
    o_h, l_h = api.mla_replay_fwd(host_cache, br.q, br.lat, SCALE, 8)
    torch.cuda.synchronize()
    assert B.ls_last_device_error(0) == B.LS_OK
    assert torch.equal(o_d, o_h) and torch.equal(l_d, l_h)
    o_ref, lse_ref = oracle.mla_fwd(problem(host_cache, br, P))
    assert rel_err(o_h.float().cpu().numpy(), o_ref) <= TOL_O
    assert float(np.abs(l_h.cpu().numpy() - lse_ref).max()) <= TOL_LSE


def test_latent_capture_bit_exact(cuda):
    P, ps = 1000, 64
    pr = syn.make_latent_prompt(P, ps, 13, cuda, extra_pages=3)
    cache = api.LatentCache(pr.num_pages, pr.page_table, ps, P, device=cuda, fill=1.5)
    cache.capture(pr.lat[:400].contiguous(), 0)
    cache.capture(pr.lat[400:].contiguous(), 400)
    torch.cuda.synchronize()
    pool = u16(cache.pool)
    pt = pr.page_table.cpu().numpy()
    lat = u16(pr.lat)
    want = np.full(pool.shape, u16(torch.tensor([1.5], dtype=torch.bfloat16))[0], np.uint16)
    for p in range(P):
        want[pt[p // ps], p % ps] = lat[p]
    np.testing.assert_array_equal(pool, want)


def test_mla_bad_page_is_reported(cuda):
    cache, br = make(500, 4, 8, 32, 3, cuda)
    cache.page_table[2] = cache.pool.shape[0] + 5
    api.mla_replay_fwd(cache, br.q, br.lat, SCALE, 2)
    assert B.ls_last_device_error(0) == B.LS_ERR_DEVICE_CHECK
    assert B.ls_last_device_error(0) == B.LS_OK


def test_mla_argument_checks(cuda):
    cache, br = make(300, 4, 8, 32, 3, cuda)
    st = cache.struct
    bad = B.ls_latent_cache(st.pool, st.page_table, st.num_pages, st.num_logical_pages, 16,
                            st.num_tokens)
    with pytest.raises(B.LongstrawError):      # page size below 32
        B.ls_mla_replay_fwd_workspace(bad, 4, 8, 1)
    with pytest.raises(B.LongstrawError):      # non-positive scale
        api.mla_replay_fwd(cache, br.q, br.lat, 0.0, 1)
    o, lse = api.mla_replay_fwd(cache, br.q[:0], br.lat[:0], SCALE, 1)   # R = 0: no-op
    assert o.shape == (0, 8, 512)


def test_mla_full_prompt_sampled_rows(cuda):
    """2,097,152 latent positions in 256-row pages, 64 heads, a 64-token response."""
    P, R, H, ps = 2097152, 64, 64, 256
    cache, br = make(P, R, H, ps, 2026, cuda, extra_pages=1)
    o, lse = api.mla_replay_fwd(cache, br.q, br.lat, SCALE, 256)
    torch.cuda.synchronize()
    assert B.ls_last_device_error(0) == B.LS_OK
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
    rng = np.random.default_rng(7)
    ts = np.concatenate([[0, R - 1], rng.integers(0, R, 6)]).astype(np.int32)
    hs = rng.integers(0, H, len(ts)).astype(np.int32)
    o_ref, lse_ref = oracle.mla_fwd_rows(problem(cache, br, P), ts, hs)
    assert rel_err(o.float().cpu().numpy()[ts, hs], o_ref) <= TOL_O
    assert float(np.abs(lse.cpu().numpy()[ts, hs] - lse_ref).max()) <= TOL_LSE
    # the rows are sharp: the LSE sits well above log(P + t + 1)
    assert np.abs(lse_ref - np.log(P + ts + 1.0)).max() > 0.1


def test_streamed_latent_layers_match_resident(cuda):
    """Three layers' latent pages captured into pinned host memory and streamed through the
    two-slot GPU page cache one layer ahead (forward in layer order, backward in reverse):
    every layer's forward and backward bit-identical to the same pages held in GPU
    memory, one layer's forward against the oracle."""
    from response_replay_gb300 import layers as L
    P, R, H, ps, splits, nl = 3000, 40, 16, 64, 5, 3
    pr0 = syn.make_latent_prompt(P, ps, 900, cuda, extra_pages=2)
    st = L.StreamedLatentLayers(nl, pr0.num_pages, pr0.page_table, ps, P, device=cuda)
    res, brs = [], []
    for l in range(nl):
        lat = syn.make_latent_prompt(P, ps, 900 + 3 * l, cuda).lat[:P].contiguous()
        c = api.LatentCache(pr0.num_pages, pr0.page_table, ps, P, device=cuda)
        c.capture(lat)
        res.append(c)
        st.capture(l, lat)
        brs.append(syn.make_latent_branch(R, H, 920 + l, cuda, sharp=True))
    st.prefetch(0)
    outs = []
    for l in range(nl):
        c = st.cache(l)
        if l + 1 < nl:
            st.prefetch(l + 1)
        outs.append(api.mla_replay_fwd(c, brs[l].q, brs[l].lat, SCALE, splits))
        st.release(l)
    # the backward in reverse layer order through the same two slots
    st.prefetch(nl - 1)
    grads = [None] * nl
    for l in reversed(range(nl)):
        c = st.cache(l)
        if l > 0:
            st.prefetch(l - 1)
        grads[l] = api.mla_replay_bwd(c, brs[l].q, brs[l].lat, outs[l][0], outs[l][1],
                                      brs[l].d_o, SCALE, splits)
        st.release(l)
    torch.cuda.synchronize()
    assert B.ls_last_device_error(0) == B.LS_OK
    for l in range(nl):
        o_r, l_r = api.mla_replay_fwd(res[l], brs[l].q, brs[l].lat, SCALE, splits)
        assert torch.equal(outs[l][0], o_r) and torch.equal(outs[l][1], l_r), l
        dq_r, dl_r = api.mla_replay_bwd(res[l], brs[l].q, brs[l].lat, o_r, l_r, brs[l].d_o,
                                        SCALE, splits)
        assert torch.equal(grads[l][0], dq_r) and torch.equal(grads[l][1], dl_r), l
    assert not st.host[1].pool.is_cuda and st.host[1].pool.is_pinned()
    o_ref, lse_ref = oracle.mla_fwd(problem(st.host[1], brs[1], P))
    assert rel_err(outs[1][0].float().cpu().numpy(), o_ref) <= TOL_O
    assert float(np.abs(outs[1][1].cpu().numpy() - lse_ref).max()) <= TOL_LSE
