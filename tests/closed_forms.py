"""Closed forms of replay attention for inputs whose every key is zero.

With k_j = 0 for every prompt and response key, every score s_{t,j} = scale <q_t, k_j>
is 0, so each response row t attends uniformly to the P prompt positions and the
response keys j <= t: P_{t,j} = 1 / (P + t + 1).  The definitions of the replay forward
and backward (LongStraw explainer, "Serial replay makes G a schedule"; paper digest,
Method, last paragraph, for the stopgrad prompt state) then reduce to sums that cost
O(R d) per output instead of O(R (P + R) d):

  lse_t   = log(P + t + 1)
  o_t     = (sum_prompt v + sum_{j <= t} v_j) / (P + t + 1)          (same for every head
                                                                      of a KV group)
  D_t,h   = <dO_t,h, o_t>
  dS      = (<dO_t,h, v_j> - D_t,h) / (P + t + 1)                     for j <= t
  dk_j    = scale sum_{h in group} sum_{t >= j} dS q_t,h
  dv_j    = sum_{h in group} sum_{t >= j} dO_t,h / (P + t + 1)
  dq_t    = 0

This lets a test check the gradients of the response's first keys, whose sums run over
every later row of a long response, at lengths where the fp64 oracle would need hours.
Test infrastructure: pinned against the oracle on small inputs (tests/test_closed_forms.py).
"""
from __future__ import annotations

import numpy as np


def uniform_attention(P: int, v_prompt_sum: np.ndarray, v_resp: np.ndarray):
    """lse [R] and o [R][hkv][d] for all-zero keys.  v_prompt_sum: [hkv][d] (the sum of
    the prompt's values per KV head), v_resp: [R][hkv][d]."""
    R = v_resp.shape[0]
    n = P + np.arange(R, dtype=np.float64) + 1.0
    o = (v_prompt_sum[None] + np.cumsum(v_resp, axis=0)) / n[:, None, None]
    return np.log(n), o


def key_gradients(P: int, scale: float, q: np.ndarray, v_resp: np.ndarray, d_o: np.ndarray,
                  o: np.ndarray, js, kvhs):
    """dk, dv [n][d] of response keys (js[i], kvhs[i]) for all-zero keys.
    q, d_o: [R][hq][d]; v_resp, o: [R][hkv][d] (o from uniform_attention)."""
    R, hq, d = q.shape
    hkv = v_resp.shape[1]
    g = hq // hkv
    inv_n = 1.0 / (P + np.arange(R, dtype=np.float64) + 1.0)
    dk = np.zeros((len(js), d))
    dv = np.zeros((len(js), d))
    for i, (j, c) in enumerate(zip(js, kvhs)):
        for h in range(c * g, (c + 1) * g):
            do_h = d_o[j:, h, :]                       # rows t >= j
            dd = np.einsum("td,td->t", do_h, o[j:, c, :])
            ds = (do_h @ v_resp[j, c, :] - dd) * inv_n[j:]
            dk[i] += scale * (ds @ q[j:, h, :])
            dv[i] += inv_n[j:] @ do_h
    return dk, dv
