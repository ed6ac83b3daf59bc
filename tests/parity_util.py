"""Shared helpers of the GPU parity tests: build a paged cache + branch on the GPU from
the seeded generators, run the CUDA path through the C ABI, hand the same inputs to
the oracle, and compare with the tolerances the tests use."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from response_replay_gb300 import synthetic as syn
from response_replay_gb300 import torch_api as api

# Tolerances (floating point): outputs at unit scale are compared as
# max|x - ref| / max|ref| (the error relative to the tensor's own scale).
TOL_O = 1e-2        # O (bf16 output)
TOL_LSE = 1e-3      # LSE, absolute
TOL_GRAD = 1e-2     # dQ, dK, dV
TOL_LOGP = 1e-4     # absolute
TOL_LOSS = 1e-4     # relative, see loss_tolerance
TOL_DLOGITS = {"bf16": 1e-2, "fp32": 1e-4}  # per row, relative to the row's max |ref|


def rel_err(x, ref) -> float:
    x = np.asarray(x, np.float64)
    ref = np.asarray(ref, np.float64)
    scale = np.abs(ref).max()
    return float(np.abs(x - ref).max() / (scale if scale > 0 else 1.0))


def u16(t: torch.Tensor) -> np.ndarray:
    return syn.bf16_bits(t)


class Case:
    """A paged prompt cache (captured through the C ABI) plus one response branch."""

    def __init__(self, P, R, hq, hkv, page_size, num_splits, seed, device, sharp=False,
                 extra_pages=2, scale=None):
        self.P, self.R, self.hq, self.hkv = P, R, hq, hkv
        self.page_size, self.num_splits = page_size, num_splits
        self.scale = scale if scale is not None else syn.HEAD_DIM ** -0.5
        pr = syn.make_prompt(max(P, 1), hkv, syn.HEAD_DIM, page_size, seed, device,
                             extra_pages=extra_pages, sharp=sharp)
        if P == 0:
            pr.page_table = pr.page_table[:0]
        self.prompt = pr
        self.cache = api.PagedKVCache(pr.num_pages, pr.page_table, page_size, hkv, P,
                                      device=device, fill=float("nan"))
        if P > 0:
            self.cache.capture(pr.k[:P].contiguous(), pr.v[:P].contiguous())
        self.br = syn.make_branch(R, hq, hkv, syn.HEAD_DIM, seed + 1, device, sharp=sharp)

    def fwd(self, num_splits=None):
        return api.replay_fwd(self.cache, self.br.q, self.br.k, self.br.v, self.scale,
                              num_splits or self.num_splits)

    def bwd(self, o, lse, num_splits=None, **kw):
        return api.replay_bwd(self.cache, self.br.q, self.br.k, self.br.v, o, lse, self.br.d_o,
                              self.scale, num_splits or self.num_splits, **kw)

    def problem(self) -> oracle.AttnProblem:
        """The same inputs, on the host, for the oracle (pools read back as captured)."""
        torch.cuda.synchronize()
        pt = self.prompt.page_table.cpu().numpy()
        return oracle.AttnProblem(u16(self.cache.k_pool), u16(self.cache.v_pool),
                                  pt if self.P > 0 else np.zeros(1, np.int32), self.P,
                                  u16(self.br.q), u16(self.br.k), u16(self.br.v), self.scale,
                                  self.num_splits)

    def d_o_host(self) -> np.ndarray:
        return u16(self.br.d_o)


def loss_tolerance(loss_ref: float, adv: np.ndarray) -> float:
    """|dL| allowed: 1e-4 of max(|L|, 1e-3 mean|A|): the loss nearly cancels because the
    advantages sum to zero, so a purely relative bound would be vacuous near 0."""
    return TOL_LOSS * max(abs(loss_ref), 1e-3 * float(np.mean(np.abs(adv))))
