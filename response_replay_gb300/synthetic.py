"""Seeded synthetic inputs for the replay-attention and GRPO-loss path.

This module only draws random numbers and lays them out; it holds none of the
method's arithmetic, so both the CUDA path and the fp64 oracle can be fed from it.
Where an input is defined in terms of the method (logp_old = logp + noise), this
module returns only the random part (the noise, the shift mask) and the caller adds
it to a logp computed by whichever side it trusts.

The five workloads follow the shapes of the LongStraw runs (explainer, "Serial
replay makes G a schedule": 2,097,152 positions, G in {2, 8}; "The numbers, and the
ceiling": one captured prefix reused over 8 consecutive G=8 cycles at 4,456,448
positions). Those runs used synthetic rewards and responses (explainer, "The fine
print"), so synthetic data here stands in for nothing else.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

HEAD_DIM = 128


@dataclass(frozen=True)
class Workload:
    """Sizes of one replay workload (single attention layer)."""
    name: str
    P: int                 # captured prompt tokens
    hq: int                # query heads
    hkv: int               # key/value heads
    page_size: int
    num_splits: int
    G: int                 # group members
    R: tuple               # response length of each member
    vocab: int
    logits_dtype: str      # "fp32" | "bf16"
    rewards: str           # reward distribution tag
    shift_frac: float = 0.0  # fraction of tokens whose logp_old is shifted by +-0.5
    cycles: int = 1        # replay cycles over one capture
    d: int = HEAD_DIM
    extra: dict = field(default_factory=dict)

    @property
    def T(self) -> int:
        return int(sum(self.R))

    @property
    def pages(self) -> int:
        return (self.P + self.page_size - 1) // self.page_size


def _ragged(seed: int, n: int, lo: int, hi: int) -> tuple:
    rng = np.random.default_rng(seed)
    return tuple(int(x) for x in rng.integers(lo, hi + 1, size=n))


# The five configurations (one attention layer each).
WORKLOADS = {
    "p4k": Workload("p4k", P=4096, hq=8, hkv=2, page_size=64, num_splits=4, G=2, R=(256, 256),
                    vocab=4096, logits_dtype="fp32", rewards="bernoulli0.5"),
    "p128k": Workload("p128k", P=131072, hq=24, hkv=4, page_size=128, num_splits=32, G=8,
                      R=(1024,) * 8, vocab=151936, logits_dtype="bf16", rewards="bernoulli0.5"),
    "p1m": Workload("p1m", P=1048576, hq=24, hkv=4, page_size=256, num_splits=128, G=8,
                    R=(2048,) * 8, vocab=151936, logits_dtype="bf16", rewards="uniform01",
                    shift_frac=0.2),
    "p2m": Workload("p2m", P=2097152, hq=24, hkv=4, page_size=256, num_splits=256, G=8,
                    R=(4096,) * 8, vocab=151936, logits_dtype="bf16", rewards="normal"),
    "p4m_reuse": Workload("p4m_reuse", P=4194304, hq=24, hkv=4, page_size=256, num_splits=256,
                          G=8, R=_ragged(20260716 + 4, 64, 512, 8192), vocab=151936,
                          logits_dtype="bf16", rewards="bernoulli0.3", cycles=8),
}
WORKLOAD_ORDER = ["p4k", "p128k", "p1m", "p2m", "p4m_reuse"]


def seed_of(name: str) -> int:
    return 20260716 + WORKLOAD_ORDER.index(name) if name in WORKLOAD_ORDER else 20260716


def gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """Host uint16 bit patterns of a bf16 tensor (no rounding: already bf16)."""
    assert t.dtype == torch.bfloat16
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


@dataclass
class PromptCache:
    """Prompt K/V to capture and the page placement. Tensors live on `device`."""
    k: torch.Tensor            # [P][hkv][d] bf16
    v: torch.Tensor            # [P][hkv][d] bf16
    page_table: torch.Tensor   # [logical pages] int32, distinct physical page ids
    num_pages: int             # physical pages in the pool (>= logical pages)
    page_size: int


def make_prompt(P: int, hkv: int, d: int, page_size: int, seed: int, device="cpu",
                extra_pages: int = 0, sharp: bool = False) -> PromptCache:
    """K, V ~ N(0,1) scaled by 1/sqrt(d) (unscaled K when sharp); page table a
    seeded random choice of distinct physical pages out of pages + extra_pages."""
    g = gen(device, seed)
    ks = 1.0 if sharp else d ** -0.5
    k = (torch.randn(P, hkv, d, generator=g, device=device) * ks).to(torch.bfloat16)
    v = (torch.randn(P, hkv, d, generator=g, device=device) * d ** -0.5).to(torch.bfloat16)
    logical = (P + page_size - 1) // page_size
    num_pages = logical + extra_pages
    rng = np.random.default_rng(seed)
    pt = rng.permutation(num_pages)[:logical].astype(np.int32)
    return PromptCache(k, v, torch.from_numpy(pt).to(device), num_pages, page_size)


@dataclass
class Branch:
    """One response branch: queries, its own keys/values and the output cotangent."""
    q: torch.Tensor        # [R][hq][d] bf16
    k: torch.Tensor        # [R][hkv][d] bf16
    v: torch.Tensor        # [R][hkv][d] bf16
    d_o: torch.Tensor      # [R][hq][d] bf16


def make_branch(R: int, hq: int, hkv: int, d: int, seed: int, device="cpu",
                sharp: bool = False) -> Branch:
    """Q, K, V ~ N(0,1) scaled by 1/sqrt(d) (Q and K unscaled when sharp); dO ~ N(0,1)."""
    g = gen(device, seed)
    qs = 1.0 if sharp else d ** -0.5
    q = (torch.randn(R, hq, d, generator=g, device=device) * qs).to(torch.bfloat16)
    k = (torch.randn(R, hkv, d, generator=g, device=device) * qs).to(torch.bfloat16)
    v = (torch.randn(R, hkv, d, generator=g, device=device) * d ** -0.5).to(torch.bfloat16)
    d_o = torch.randn(R, hq, d, generator=g, device=device).to(torch.bfloat16)
    return Branch(q, k, v, d_o)


@dataclass
class GrpoInputs:
    logits: torch.Tensor       # [T][V] fp32 or bf16
    targets: torch.Tensor      # [T] int32
    rewards: torch.Tensor      # [G] fp32
    resp_lens: torch.Tensor    # [G] int32
    noise: torch.Tensor        # [T] fp32: logp_old = logp + noise


def draw_rewards(kind: str, G: int, rng: np.random.Generator) -> np.ndarray:
    if kind == "bernoulli0.5":
        return (rng.random(G) < 0.5).astype(np.float32)
    if kind == "bernoulli0.3":
        return (rng.random(G) < 0.3).astype(np.float32)
    if kind == "uniform01":
        return rng.random(G).astype(np.float32)
    if kind == "normal":
        return rng.standard_normal(G).astype(np.float32)
    raise ValueError(kind)


def make_grpo(resp_lens, vocab: int, logits_dtype: str, rewards: str, seed: int,
              device="cpu", shift_frac: float = 0.0, logit_std: float = 2.0,
              noise_std: float = 0.05) -> GrpoInputs:
    """Logits ~ N(0, logit_std); targets uniform in [0, V); noise ~ N(0, noise_std),
    plus +-0.5 (equiprobable sign) on an independent Bernoulli(shift_frac) subset."""
    lens = np.asarray(resp_lens, dtype=np.int32)
    T = int(lens.sum())
    g = gen(device, seed)
    dt = torch.float32 if logits_dtype == "fp32" else torch.bfloat16
    logits = (torch.randn(T, vocab, generator=g, device=device) * logit_std).to(dt)
    rng = np.random.default_rng(seed)
    targets = rng.integers(0, vocab, size=T).astype(np.int32)
    r = draw_rewards(rewards, len(lens), rng)
    noise = rng.standard_normal(T) * noise_std
    if shift_frac > 0:
        mask = rng.random(T) < shift_frac
        sign = np.where(rng.random(T) < 0.5, -1.0, 1.0)
        noise = noise + mask * sign * 0.5
    return GrpoInputs(logits, torch.from_numpy(targets).to(device),
                      torch.from_numpy(r).to(device), torch.from_numpy(lens).to(device),
                      torch.from_numpy(noise.astype(np.float32)).to(device))


@dataclass
class GdnInputs:
    """Inputs of a Gated-DeltaNet replay (one layer): the captured state and the response
    tokens' projections."""
    state0: torch.Tensor   # [H][128][128] fp32 (d_v x d_k)
    q: torch.Tensor        # [R][H][128] bf16, unit rows
    k: torch.Tensor        # [R][H][128] bf16, unit rows
    v: torch.Tensor        # [R][H][128] bf16
    g: torch.Tensor        # [R][H] fp32, log decay
    beta: torch.Tensor     # [R][H] fp32 in (0, 1)
    d_o: torch.Tensor      # [R][H][128] bf16


def make_gdn(R: int, H: int, seed: int, device="cpu", d: int = HEAD_DIM,
             decay=(0.9, 1.0), state_std: float = 0.1) -> GdnInputs:
    """q, k: N(0,1) rows normalised to unit length (the layer normalises them); v, dO:
    N(0,1); decay exp(g) ~ U(decay); beta = sigmoid(N(0,1)); state0 ~ N(0, state_std)."""
    gg = gen(device, seed)
    q = torch.randn(R, H, d, generator=gg, device=device)
    k = torch.randn(R, H, d, generator=gg, device=device)
    q = (q / q.norm(dim=2, keepdim=True).clamp_min(1e-6)).to(torch.bfloat16)
    k = (k / k.norm(dim=2, keepdim=True).clamp_min(1e-6)).to(torch.bfloat16)
    v = torch.randn(R, H, d, generator=gg, device=device).to(torch.bfloat16)
    d_o = torch.randn(R, H, d, generator=gg, device=device).to(torch.bfloat16)
    u = torch.rand(R, H, generator=gg, device=device)
    g = torch.log(decay[0] + (decay[1] - decay[0]) * u).float().contiguous()
    beta = torch.sigmoid(torch.randn(R, H, generator=gg, device=device)).float().contiguous()
    state0 = (torch.randn(H, d, d, generator=gg, device=device) * state_std).float()
    return GdnInputs(state0, q, k, v, g, beta, d_o)


LATENT_ROW = 576   # latent (512) + rotary key (64) values per position
LATENT_DIM = 512   # latent values (the output width)


@dataclass
class LatentPrompt:
    """Prompt rows of a latent-attention layer to capture, and the page placement."""
    lat: torch.Tensor          # [P][576] bf16, logical order
    page_table: torch.Tensor   # [ceil(P / page_size)] int32
    num_pages: int
    page_size: int


@dataclass
class LatentBranch:
    """One response branch of a latent-attention layer."""
    q: torch.Tensor            # [R][H][576] bf16 absorbed queries
    lat: torch.Tensor          # [R][576] bf16 the response's own rows
    d_o: torch.Tensor          # [R][H][512] bf16 output gradient


def make_latent_prompt(P: int, page_size: int, seed: int, device="cpu",
                       extra_pages: int = 0) -> LatentPrompt:
    """Rows ~ N(0,1); page table a seeded random choice of distinct physical pages."""
    g = gen(device, seed)
    lat = torch.randn(P, LATENT_ROW, generator=g, device=device).to(torch.bfloat16)
    logical = (P + page_size - 1) // page_size
    num_pages = logical + extra_pages
    rng = np.random.default_rng(seed)
    pt = rng.permutation(num_pages)[:logical].astype(np.int32)
    return LatentPrompt(lat, torch.from_numpy(pt).to(device), num_pages, page_size)


def make_latent_branch(R: int, H: int, seed: int, device="cpu", sharp: bool = False) -> LatentBranch:
    """Rows ~ N(0,1); queries N(0,1) (sharp: scores of spread ~1.7 at scale 1/sqrt(192))
    or N(0,1)/sqrt(576) (near-uniform); output gradient N(0,1), drawn last."""
    g = gen(device, seed)
    qs = 1.0 if sharp else LATENT_ROW ** -0.5
    q = (torch.randn(R, H, LATENT_ROW, generator=g, device=device) * qs).to(torch.bfloat16)
    lat = torch.randn(R, LATENT_ROW, generator=g, device=device).to(torch.bfloat16)
    d_o = torch.randn(R, H, LATENT_DIM, generator=g, device=device).to(torch.bfloat16)
    return LatentBranch(q, lat, d_o)
