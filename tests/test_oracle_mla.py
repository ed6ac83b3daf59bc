"""Pins of the fp64 latent-attention (MLA-style) oracle against things other than itself:
a brute-force softmax over the gathered rows, the q = 0 closed form, the attention
oracle (itself pinned) in the equivalent one-KV-head problem, and page-table
invariance.  A wrong page lookup, a dropped rotary term, the rotary part leaking into
the output, a wrong causal bound or a wrong scale fails at least one."""
import numpy as np
import pytest

import oracle


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round-to-nearest-even bf16 bit patterns of x."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)


def bf16_value(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def latent_problem(P, R, H, d_c, d_r, ps, seed, extra_pages=2, scale=0.1, zero_q=False):
    """Random latent pages (shuffled, stale rows NaN) and a branch; also the prompt rows
    in logical order as fp64 for brute force."""
    rng = np.random.default_rng(seed)
    D = d_c + d_r
    logical = (P + ps - 1) // ps
    num_pages = logical + extra_pages
    pt = rng.permutation(num_pages)[:logical].astype(np.int32)
    pool = np.full((num_pages, ps, D), 0x7FC0, np.uint16)   # bf16 NaN in unused slots
    rows = bf16_bits(rng.standard_normal((P, D)))
    for p in range(P):
        pool[pt[p // ps], p % ps] = rows[p]
    q = bf16_bits(np.zeros((R, H, D)) if zero_q else rng.standard_normal((R, H, D)))
    resp = bf16_bits(rng.standard_normal((R, D)))
    pb = oracle.MlaProblem(pool, pt if P > 0 else np.zeros(1, np.int32), P, q, resp, scale,
                           d_c=d_c)
    return pb, bf16_value(rows)


def brute_force(pb, rows):
    """Textbook softmax over the full key matrix [prompt rows; response rows]."""
    R, H, D = pb.q.shape
    keys = np.concatenate([rows, bf16_value(pb.lat_resp)], 0)      # [P + R, D]
    q = bf16_value(pb.q)
    o = np.zeros((R, H, pb.d_c))
    lse = np.zeros((R, H))
    for t in range(R):
        vis = keys[:pb.P + t + 1]
        s = pb.scale * q[t] @ vis.T                                 # [H, P + t + 1]
        m = s.max(1, keepdims=True)
        w = np.exp(s - m)
        lse[t] = m[:, 0] + np.log(w.sum(1))
        o[t] = (w / w.sum(1, keepdims=True)) @ vis[:, :pb.d_c]
    return o, lse


@pytest.mark.parametrize("P,R,H,d_c,d_r,ps", [
    (37, 5, 3, 16, 8, 8), (0, 6, 2, 12, 4, 4), (64, 1, 4, 8, 0, 16), (100, 9, 2, 20, 6, 32),
])
def test_matches_brute_force(P, R, H, d_c, d_r, ps):
    pb, rows = latent_problem(P, R, H, d_c, d_r, ps, seed=P + 10 * R + H)
    o, lse = oracle.mla_fwd(pb)
    o_bf, lse_bf = brute_force(pb, rows)
    np.testing.assert_allclose(o, o_bf, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lse_bf, rtol=0, atol=1e-12)


def test_zero_query_is_mean_of_visible_latents():
    P, R, H, d_c, d_r = 50, 7, 3, 10, 6
    pb, rows = latent_problem(P, R, H, d_c, d_r, 16, seed=3, zero_q=True)
    o, lse = oracle.mla_fwd(pb)
    lat = np.concatenate([rows, bf16_value(pb.lat_resp)], 0)[:, :d_c]
    for t in range(R):
        np.testing.assert_allclose(o[t], np.broadcast_to(lat[:P + t + 1].mean(0), (H, d_c)),
                                   rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse[t], np.log(P + t + 1.0), rtol=0, atol=1e-12)


def test_equals_one_kv_head_attention():
    """Latent attention is attention with one KV head whose key is the whole row and whose
    value is the row with its rotary part zeroed (output columns past d_c are then 0)."""
    P, R, H, d_c, d_r, ps = 70, 6, 4, 12, 4, 16
    pb, rows = latent_problem(P, R, H, d_c, d_r, ps, seed=11)
    o, lse = oracle.mla_fwd(pb)
    kp = bf16_value(pb.lat_pool)[:, None]                        # [pages][1][ps][D]
    vp = kp.copy()
    vp[..., d_c:] = 0.0
    kr = bf16_value(pb.lat_resp)[:, None]
    vr = kr.copy()
    vr[..., d_c:] = 0.0
    ap = oracle.AttnProblem(np.nan_to_num(kp), np.nan_to_num(vp), pb.page_table, P,
                            bf16_value(pb.q), kr, vr, pb.scale, 3)
    o_a, lse_a = oracle.attn_fwd(ap)
    np.testing.assert_allclose(o, o_a[..., :d_c], rtol=0, atol=1e-12)
    assert np.abs(o_a[..., d_c:]).max() == 0.0
    np.testing.assert_allclose(lse, lse_a, rtol=0, atol=1e-12)


def test_page_table_invariance():
    """The same prompt rows on one identity-mapped page give the same result."""
    P, R, H, d_c, d_r, ps = 45, 4, 2, 8, 8, 8
    pb, rows = latent_problem(P, R, H, d_c, d_r, ps, seed=21)
    one = np.zeros((1, P, d_c + d_r), np.uint16)
    one[0] = bf16_bits(rows)
    pb1 = oracle.MlaProblem(one, np.zeros(1, np.int32), P, pb.q, pb.lat_resp, pb.scale, d_c=d_c)
    o, lse = oracle.mla_fwd(pb)
    o1, lse1 = oracle.mla_fwd(pb1)
    np.testing.assert_array_equal(o, o1)
    np.testing.assert_array_equal(lse, lse1)


def test_rows_sampler_and_bad_page():
    P, R, H, d_c, d_r, ps = 33, 5, 3, 8, 4, 8
    pb, rows = latent_problem(P, R, H, d_c, d_r, ps, seed=5)
    o, lse = oracle.mla_fwd(pb)
    ts, hs = np.array([0, 4, 2, 4]), np.array([2, 0, 1, 2])
    o_r, lse_r = oracle.mla_fwd_rows(pb, ts, hs)
    np.testing.assert_array_equal(o_r, o[ts, hs])
    np.testing.assert_array_equal(lse_r, lse[ts, hs])
    bad = pb.page_table.copy()
    bad[1] = pb.lat_pool.shape[0]
    with pytest.raises(ValueError):
        oracle.mla_fwd(oracle.MlaProblem(pb.lat_pool, bad, P, pb.q, pb.lat_resp, pb.scale,
                                         d_c=d_c))


# ----------------------------------------------------------------------------- backward
# Pins of lso_mla_bwd: central finite differences of L = <dO, O> through the forward
# oracle (pinned above), with steps that are exact in bf16 so the perturbed inputs are
# what the forward reads; and the one-key closed form.  A dropped D term, a missing
# scale, the value term of d lat missing or leaking into the rotary part, a wrong causal
# bound on d lat, or a gradient given to the prompt rows fails at least one of them.

def _loss(pb, g):
    o, _ = oracle.mla_fwd(pb)
    return float((o * bf16_value(g)).sum())


def _fd(pb, g, arr, idx):
    """Richardson-extrapolated central difference of L in arr[idx], taken at the value 1.0
    (set beforehand), with steps 1/64 and 1/128 (1 +- h exact in bf16)."""
    def central(h):
        arr[idx] = bf16_bits(np.array([1.0 + h]))[0]
        lp = _loss(pb, g)
        arr[idx] = bf16_bits(np.array([1.0 - h]))[0]
        lm = _loss(pb, g)
        arr[idx] = bf16_bits(np.array([1.0]))[0]
        return (lp - lm) / (2 * h)
    d1, d2 = central(1 / 64), central(1 / 128)
    return (4 * d2 - d1) / 3


@pytest.mark.parametrize("P,R,H,d_c,d_r,ps", [(23, 4, 2, 8, 4, 8), (0, 5, 3, 6, 2, 4)])
def test_bwd_matches_finite_differences(P, R, H, d_c, d_r, ps):
    pb, _ = latent_problem(P, R, H, d_c, d_r, ps, seed=77 + P + R, scale=0.3)
    rng = np.random.default_rng(5 + P)
    g = bf16_bits(rng.standard_normal((R, H, d_c)))
    D = d_c + d_r
    probes_q = [(R - 1, H - 1, D - 1), (0, 0, 0), (R // 2, 1 % H, d_c), (R - 1, 0, d_c - 1)]
    probes_l = [(0, 0), (0, D - 1), (R - 1, 1), (R // 2, d_c), (R - 2, d_c - 1)]
    for (t, h, d) in probes_q:
        pb.q[t, h, d] = bf16_bits(np.array([1.0]))[0]
    for (j, d) in probes_l:
        pb.lat_resp[j, d] = bf16_bits(np.array([1.0]))[0]
    dq, dlat = oracle.mla_bwd(pb, g)
    scale_q = np.abs(dq).max()
    scale_l = np.abs(dlat).max()
    for (t, h, d) in probes_q:
        fd = _fd(pb, g, pb.q, (t, h, d))
        assert abs(fd - dq[t, h, d]) <= 1e-6 * scale_q + 1e-5 * abs(fd), ((t, h, d), fd, dq[t, h, d])
    for (j, d) in probes_l:
        fd = _fd(pb, g, pb.lat_resp, (j, d))
        assert abs(fd - dlat[j, d]) <= 1e-6 * scale_l + 1e-5 * abs(fd), ((j, d), fd, dlat[j, d])


def test_bwd_one_key_closed_form():
    """A one-token response over an empty prompt attends only to its own row: P = 1, so
    dS = 0, dq = 0, and the row's gradient is the heads' dO summed (value role only)."""
    H, d_c, d_r = 4, 10, 6
    pb, _ = latent_problem(0, 1, H, d_c, d_r, 8, seed=11)
    g = bf16_bits(np.random.default_rng(2).standard_normal((1, H, d_c)))
    dq, dlat = oracle.mla_bwd(pb, g)
    np.testing.assert_allclose(dq, 0.0, rtol=0, atol=1e-12)
    want = np.concatenate([bf16_value(g)[0].sum(0), np.zeros(d_r)])
    np.testing.assert_allclose(dlat[0], want, rtol=0, atol=1e-12)


def test_bwd_rows_and_keys_match_full():
    P, R, H, d_c, d_r, ps = 41, 7, 3, 12, 4, 16
    pb, _ = latent_problem(P, R, H, d_c, d_r, ps, seed=19)
    g = bf16_bits(np.random.default_rng(3).standard_normal((R, H, d_c)))
    dq, dlat = oracle.mla_bwd(pb, g)
    ts = np.array([0, R - 1, 3, 3], np.int32)
    hs = np.array([0, H - 1, 1, 2], np.int32)
    np.testing.assert_allclose(oracle.mla_bwd_dq_rows(pb, g, ts, hs), dq[ts, hs], rtol=0,
                               atol=1e-13)
    js = np.array([R - 1, 0, 4], np.int32)
    np.testing.assert_allclose(oracle.mla_bwd_dlat_keys(pb, g, js), dlat[js], rtol=0,
                               atol=1e-12)


def test_bwd_equals_one_kv_head_attention():
    """The same one-KV-head problem as above, backward: dq equals the attention oracle's
    dQ (itself pinned), and the response rows' gradient equals its dK + dV (the latent is
    both the key and the value; dO padded with zeros past d_c leaves dV's rotary part 0)."""
    P, R, H, d_c, d_r, ps = 70, 6, 4, 12, 4, 16
    pb, rows = latent_problem(P, R, H, d_c, d_r, ps, seed=13)
    g = bf16_bits(np.random.default_rng(4).standard_normal((R, H, d_c)))
    dq, dlat = oracle.mla_bwd(pb, g)
    kp = bf16_value(pb.lat_pool)[:, None]
    vp = kp.copy()
    vp[..., d_c:] = 0.0
    kr = bf16_value(pb.lat_resp)[:, None]
    vr = kr.copy()
    vr[..., d_c:] = 0.0
    ap = oracle.AttnProblem(np.nan_to_num(kp), np.nan_to_num(vp), pb.page_table, P,
                            bf16_value(pb.q), kr, vr, pb.scale, 3)
    g_pad = np.zeros((R, H, d_c + d_r), np.uint16)
    g_pad[..., :d_c] = g
    dq_a, dk_a, dv_a = oracle.attn_bwd(ap, g_pad)
    np.testing.assert_allclose(dq, dq_a, rtol=0, atol=1e-12)
    assert np.abs(dv_a[..., d_c:]).max() == 0.0
    np.testing.assert_allclose(dlat, (dk_a + dv_a)[:, 0], rtol=0, atol=1e-12)
