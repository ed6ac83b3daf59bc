"""Pins of the fp64 attention oracle against things other than itself.

Each test checks the oracle against a fact fixed by the pages or by mathematics:
a brute-force monolithic softmax, the split/merge invariant, closed forms, the
library causal-attention routine in the special case with no prompt, finite
differences for the gradients, and a hand-worked example. A dropped term, a wrong
index into the page table, a transposed operand or a wrong sign fails at least one.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def paged_problem(P, R, hq, hkv, d, ps, seed, extra_pages=3, splits=1, dtype=np.float64,
                  scale=None, nan_fill=True):
    """Random paged cache + branch in fp64 (or another float dtype). Returns the
    problem and the logical-order prompt keys/values for brute force."""
    rng = np.random.default_rng(seed)
    logical = (P + ps - 1) // ps
    num_pages = logical + extra_pages
    pt = rng.permutation(num_pages)[:logical].astype(np.int32)
    kp = np.full((num_pages, hkv, ps, d), np.nan if nan_fill else 0.0)
    vp = np.full((num_pages, hkv, ps, d), np.nan if nan_fill else 0.0)
    K = rng.standard_normal((P, hkv, d))
    V = rng.standard_normal((P, hkv, d))
    for p in range(P):
        kp[pt[p // ps], :, p % ps] = K[p]
        vp[pt[p // ps], :, p % ps] = V[p]
    q = rng.standard_normal((R, hq, d))
    kr = rng.standard_normal((R, hkv, d))
    vr = rng.standard_normal((R, hkv, d))
    pb = oracle.AttnProblem(kp.astype(dtype), vp.astype(dtype), pt, P, q.astype(dtype),
                            kr.astype(dtype), vr.astype(dtype),
                            scale if scale is not None else d ** -0.5, splits)
    return pb, K, V


def brute_force_fwd(pb, K, V):
    """Monolithic softmax over all visible keys of each row (textbook definition)."""
    R, hq, hkv, d = pb.dims
    g = hq // hkv
    P = pb.P
    o = np.zeros((R, hq, d))
    lse = np.zeros((R, hq))
    for h in range(hq):
        kvh = h // g
        keys = np.concatenate([K[:, kvh], pb.k_resp[:, kvh]], 0)
        vals = np.concatenate([V[:, kvh], pb.v_resp[:, kvh]], 0)
        s = pb.scale * pb.q[:, h] @ keys.T                     # [R, P + R]
        mask = np.zeros_like(s, dtype=bool)
        for t in range(R):
            mask[t, P + t + 1:] = True                          # causal within response
        s = np.where(mask, -np.inf, s)
        m = s.max(1, keepdims=True)
        w = np.exp(s - m)
        lse[:, h] = (m[:, 0] + np.log(w.sum(1)))
        o[:, h] = (w / w.sum(1, keepdims=True)) @ vals
    return o, lse


@pytest.mark.parametrize("P,ps", [(200, 16), (256, 64), (64, 64), (37, 8)])
@pytest.mark.parametrize("splits", [1, 2, 3, 1000])
def test_fwd_matches_brute_force_for_any_split(P, ps, splits):
    pb, K, V = paged_problem(P, R=9, hq=4, hkv=2, d=8, ps=ps, seed=P + ps)
    pages = (P + ps - 1) // ps
    pb.num_splits = min(splits, pages)
    o, lse = oracle.attn_fwd(pb)
    ob, lseb = brute_force_fwd(pb, K, V)
    assert np.isfinite(o).all()
    np.testing.assert_allclose(o, ob, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lseb, rtol=0, atol=1e-12)


def test_split_invariance_more_splits_than_pages():
    """Splits beyond the page count are empty (lse = -inf) and must not change anything."""
    pb, K, V = paged_problem(100, R=5, hq=2, hkv=1, d=4, ps=32, seed=1)
    pb.num_splits = 1
    o1, l1 = oracle.attn_fwd(pb)
    pb.num_splits = 17
    o2, l2 = oracle.attn_fwd(pb)
    np.testing.assert_allclose(o2, o1, atol=1e-13)
    np.testing.assert_allclose(l2, l1, atol=1e-13)


def test_zero_query_closed_form():
    """q = 0 makes every visible score 0: O_t = mean of the P + t + 1 visible values,
    LSE_t = log(P + t + 1)."""
    pb, K, V = paged_problem(96, R=7, hq=4, hkv=2, d=8, ps=32, seed=3, splits=3)
    pb.q = np.zeros_like(pb.q)
    o, lse = oracle.attn_fwd(pb)
    R, hq, hkv, d = pb.dims
    for t in range(R):
        for h in range(hq):
            kvh = h // 2
            vis = np.concatenate([V[:, kvh], pb.v_resp[: t + 1, kvh]], 0)
            np.testing.assert_allclose(o[t, h], vis.mean(0), atol=1e-13)
            assert abs(lse[t, h] - np.log(pb.P + t + 1)) < 1e-13


def _sdpa_ref(q, k, v, scale, causal):
    """torch fp64 scaled_dot_product_attention with GQA heads expanded."""
    R, hq, d = q.shape
    hkv = k.shape[1]
    g = hq // hkv
    qt = torch.from_numpy(q).permute(1, 0, 2)
    kt = torch.from_numpy(k).permute(1, 0, 2).repeat_interleave(g, 0)
    vt = torch.from_numpy(v).permute(1, 0, 2).repeat_interleave(g, 0)
    return qt, kt, vt


def test_no_prompt_equals_causal_sdpa():
    """P = 0: the method reduces to ordinary causal self-attention of the response."""
    rng = np.random.default_rng(5)
    R, hq, hkv, d = 13, 6, 2, 16
    q, kr, vr = (rng.standard_normal(s) for s in ((R, hq, d), (R, hkv, d), (R, hkv, d)))
    pb = oracle.AttnProblem(np.zeros((1, hkv, 16, d)), np.zeros((1, hkv, 16, d)),
                            np.zeros(1, np.int32), 0, q, kr, vr, 0.3, 1)
    o, lse = oracle.attn_fwd(pb)
    qt, kt, vt = _sdpa_ref(q, kr, vr, 0.3, True)
    ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, is_causal=True, scale=0.3)
    np.testing.assert_allclose(o, ref.permute(1, 0, 2).numpy(), atol=1e-12)


def test_single_query_is_decode_attention():
    """R = 1: one query attending to all P prompt keys and its own key (decode)."""
    pb, K, V = paged_problem(300, R=1, hq=4, hkv=1, d=8, ps=64, seed=7, splits=2)
    o, lse = oracle.attn_fwd(pb)
    keys = np.concatenate([K, pb.k_resp], 0)      # [P + 1, 1, d]
    vals = np.concatenate([V, pb.v_resp], 0)
    qt, kt, vt = _sdpa_ref(pb.q, keys, vals, pb.scale, False)
    ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=pb.scale)
    np.testing.assert_allclose(o, ref.permute(1, 0, 2).numpy(), atol=1e-12)


def test_one_page_identity_table_equals_shuffled_pages():
    """A single page holding the whole prompt (identity table) and a shuffled multi-page
    placement of the same logical prompt give identical results: the page table only
    moves data, it never changes which key a position reads."""
    P, hkv, d = 128, 2, 8
    pb, K, V = paged_problem(P, R=4, hq=4, hkv=hkv, d=d, ps=16, seed=11)
    one = oracle.AttnProblem(K.transpose(1, 0, 2)[None].copy(), V.transpose(1, 0, 2)[None].copy(),
                             np.zeros(1, np.int32), P, pb.q, pb.k_resp, pb.v_resp, pb.scale, 1)
    o1, l1 = oracle.attn_fwd(one)
    o2, l2 = oracle.attn_fwd(pb)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_hand_worked_example():
    """Tiny example worked by hand (tests/golden/attn_hand_example.json)."""
    with open(os.path.join(GOLDEN, "attn_hand_example.json")) as f:
        ex = json.load(f)
    kp = np.array(ex["k_pool"], np.float64)
    vp = np.array(ex["v_pool"], np.float64)
    pb = oracle.AttnProblem(kp, vp, np.array(ex["page_table"], np.int32), ex["P"],
                            np.array(ex["q"], np.float64), np.array(ex["k_resp"], np.float64),
                            np.array(ex["v_resp"], np.float64), ex["scale"], ex["num_splits"])
    o, lse = oracle.attn_fwd(pb)
    np.testing.assert_allclose(o, np.array(ex["expect_o"]), atol=1e-15)
    np.testing.assert_allclose(lse, np.array(ex["expect_lse"]), atol=1e-15)


def test_sampled_rows_match_full():
    pb, K, V = paged_problem(160, R=11, hq=6, hkv=2, d=8, ps=32, seed=13, splits=2)
    o, lse = oracle.attn_fwd(pb)
    ts = [0, 3, 10, 10, 5]
    hs = [0, 5, 2, 3, 1]
    o_r, lse_r = oracle.attn_fwd_rows(pb, ts, hs)
    np.testing.assert_array_equal(o_r, o[ts, hs])
    np.testing.assert_array_equal(lse_r, lse[ts, hs])


# ---------------------------------------------------------------- backward


def _loss_fn(pb, d_o):
    o, _ = oracle.attn_fwd(pb)
    return float((o * d_o).sum())


def _fd_grad(pb, d_o, attr, idx_list, h=1e-6):
    out = []
    for idx in idx_list:
        arr = getattr(pb, attr)
        old = arr[idx]
        arr[idx] = old + h
        fp = _loss_fn(pb, d_o)
        arr[idx] = old - h
        fm = _loss_fn(pb, d_o)
        arr[idx] = old
        out.append((fp - fm) / (2 * h))
    return np.array(out)


def test_bwd_matches_finite_differences():
    """Central differences of f = <dO, O> w.r.t. Q, K_resp and V_resp (fp64, h = 1e-6)."""
    pb, K, V = paged_problem(48, R=6, hq=4, hkv=2, d=4, ps=16, seed=17, splits=2)
    rng = np.random.default_rng(18)
    d_o = rng.standard_normal(pb.q.shape)
    dq, dk, dv = oracle.attn_bwd(pb, d_o)
    all_q = [tuple(i) for i in np.ndindex(*pb.q.shape)]
    all_k = [tuple(i) for i in np.ndindex(*pb.k_resp.shape)]
    fq = _fd_grad(pb, d_o, "q", all_q)
    fk = _fd_grad(pb, d_o, "k_resp", all_k)
    fv = _fd_grad(pb, d_o, "v_resp", all_k)
    np.testing.assert_allclose(dq.reshape(-1), fq, atol=2e-8, rtol=1e-6)
    np.testing.assert_allclose(dk.reshape(-1), fk, atol=2e-8, rtol=1e-6)
    np.testing.assert_allclose(dv.reshape(-1), fv, atol=2e-8, rtol=1e-6)


def test_no_prompt_bwd_equals_autograd_sdpa():
    rng = np.random.default_rng(19)
    R, hq, hkv, d = 9, 4, 2, 8
    q, kr, vr = (rng.standard_normal(s) for s in ((R, hq, d), (R, hkv, d), (R, hkv, d)))
    d_o = rng.standard_normal((R, hq, d))
    pb = oracle.AttnProblem(np.zeros((1, hkv, 8, d)), np.zeros((1, hkv, 8, d)),
                            np.zeros(1, np.int32), 0, q, kr, vr, 0.5, 1)
    dq, dk, dv = oracle.attn_bwd(pb, d_o)
    qt = torch.from_numpy(q).requires_grad_()
    kt = torch.from_numpy(kr).requires_grad_()
    vt = torch.from_numpy(vr).requires_grad_()
    g = hq // hkv
    o = torch.nn.functional.scaled_dot_product_attention(
        qt.permute(1, 0, 2), kt.permute(1, 0, 2).repeat_interleave(g, 0),
        vt.permute(1, 0, 2).repeat_interleave(g, 0), is_causal=True, scale=0.5)
    (o.permute(1, 0, 2) * torch.from_numpy(d_o)).sum().backward()
    np.testing.assert_allclose(dq, qt.grad.numpy(), atol=1e-12)
    np.testing.assert_allclose(dk, kt.grad.numpy(), atol=1e-12)
    np.testing.assert_allclose(dv, vt.grad.numpy(), atol=1e-12)


def test_bwd_sampled_match_full():
    pb, K, V = paged_problem(96, R=10, hq=6, hkv=2, d=8, ps=32, seed=23, splits=2)
    rng = np.random.default_rng(24)
    d_o = rng.standard_normal(pb.q.shape)
    dq, dk, dv = oracle.attn_bwd(pb, d_o)
    ts, hs = [0, 9, 4], [5, 0, 3]
    np.testing.assert_allclose(oracle.attn_bwd_dq_rows(pb, d_o, ts, hs), dq[ts, hs], atol=1e-14)
    js, kvhs = [9, 0, 5, 7], [1, 0, 1, 0]
    dk_s, dv_s = oracle.attn_bwd_dkdv_keys(pb, d_o, js, kvhs)
    np.testing.assert_allclose(dk_s, dk[js, kvhs], atol=1e-14)
    np.testing.assert_allclose(dv_s, dv[js, kvhs], atol=1e-14)


def test_bf16_inputs_widen_exactly():
    """bf16 bit patterns give exactly the result of the same values passed as fp64."""
    pb, K, V = paged_problem(64, R=4, hq=2, hkv=1, d=8, ps=16, seed=29, nan_fill=False)
    to_bits = lambda a: torch.from_numpy(a).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    from_bits = lambda b: torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).double().numpy()
    bits = {n: to_bits(getattr(pb, n)) for n in ("k_pool", "v_pool", "q", "k_resp", "v_resp")}
    pb_b = oracle.AttnProblem(bits["k_pool"], bits["v_pool"], pb.page_table, pb.P, bits["q"],
                              bits["k_resp"], bits["v_resp"], pb.scale, 1)
    pb_d = oracle.AttnProblem(*(from_bits(bits[n]) for n in ("k_pool", "v_pool")), pb.page_table,
                              pb.P, *(from_bits(bits[n]) for n in ("q", "k_resp", "v_resp")),
                              pb.scale, 1)
    o1, l1 = oracle.attn_fwd(pb_b)
    o2, l2 = oracle.attn_fwd(pb_d)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_bad_page_id_rejected():
    pb, K, V = paged_problem(64, R=2, hq=2, hkv=1, d=4, ps=16, seed=31)
    pb.page_table = pb.page_table.copy()
    pb.page_table[1] = pb.k_pool.shape[0]
    with pytest.raises(ValueError):
        oracle.attn_fwd(pb)


# ---------------------------------------------------------------- capture


def test_capture_scatter_bit_exact_and_sentinels_intact():
    rng = np.random.default_rng(37)
    ps, hkv, d = 16, 2, 8
    P = 100                                    # ragged last page
    logical = (P + ps - 1) // ps
    num_pages = logical + 2
    pt = rng.permutation(num_pages)[:logical].astype(np.int32)
    sentinel = np.uint16(0x7FC1)               # a bf16 NaN pattern
    kp = np.full((num_pages, hkv, ps, d), sentinel, np.uint16)
    vp = np.full((num_pages, hkv, ps, d), sentinel, np.uint16)
    k = rng.integers(0, 0x7F00, size=(P, hkv, d), dtype=np.uint16)
    v = rng.integers(0, 0x7F00, size=(P, hkv, d), dtype=np.uint16)
    # two calls: a chunked capture must equal one whole capture
    oracle.capture_kv(kp, vp, pt, ps, k[:37].copy(), v[:37].copy(), 0)
    oracle.capture_kv(kp, vp, pt, ps, k[37:].copy(), v[37:].copy(), 37)
    ek = np.full_like(kp, sentinel)
    ev = np.full_like(vp, sentinel)
    pos = np.arange(P)
    ek[pt[pos // ps], :, pos % ps] = k           # numpy fancy-index scatter
    ev[pt[pos // ps], :, pos % ps] = v
    assert np.array_equal(kp, ek) and np.array_equal(vp, ev)
    # round trip: gathering back through the table returns the input
    assert np.array_equal(kp[pt[pos // ps], :, pos % ps], k)
    untouched = np.setdiff1d(np.arange(num_pages), pt)
    assert (kp[untouched] == sentinel).all()
    assert (kp[pt[-1], :, P % ps:] == sentinel).all()


def test_capture_rejects_out_of_table():
    kp = np.zeros((2, 1, 4, 2), np.uint16)
    with pytest.raises(ValueError):
        oracle.capture_kv(kp, kp.copy(), np.array([0, 1], np.int32), 4,
                          np.zeros((3, 1, 2), np.uint16), np.zeros((3, 1, 2), np.uint16), 7)
