"""PyTorch-facing helpers over the C ABI.

PyTorch supplies device memory and streams; every step of the computation runs in the
CUDA kernels behind include/longstraw.h.  These helpers allocate outputs and workspace
with torch, check shapes and dtypes, and pass raw pointers to the binding.
"""
from __future__ import annotations

import torch

from . import binding as B

HEAD_DIM = 128


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _check(t: torch.Tensor, name: str, dtype, shape=None):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name}: expected {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: expected shape {tuple(shape)}, got {tuple(t.shape)}")


_workspaces: dict = {}


def workspace(nbytes: int, device: torch.device, key: str = "default") -> torch.Tensor:
    """A reusable uint8 workspace of at least nbytes on `device` (grown on demand).
    Calls that share a key must not overlap on the GPU."""
    k = (device.index if device.index is not None else torch.cuda.current_device(), key)
    ws = _workspaces.get(k)
    if ws is None or ws.numel() < max(nbytes, 1):
        ws = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)
        _workspaces[k] = ws
    return ws


def _check_pool(t: torch.Tensor, name: str, shape):
    """A page pool: GPU memory, or pinned host memory the GPU reads directly."""
    if not t.is_cuda and not (t.device.type == "cpu" and t.is_pinned()):
        raise ValueError(f"{name} must be a CUDA tensor or a pinned host tensor")
    if t.dtype != torch.bfloat16:
        raise ValueError(f"{name}: expected torch.bfloat16, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: expected shape {tuple(shape)}, got {tuple(t.shape)}")


class PagedKVCache:
    """K/V page pools plus page table of one attention layer (ls_kv_cache).

    host_pools=True places the pools in pinned host memory (on a Grace-Blackwell node,
    Grace memory read over NVLink-C2C); the kernels read and write them there."""

    def __init__(self, num_pages: int, page_table: torch.Tensor, page_size: int, num_kv_heads: int,
                 num_tokens: int, device=None, fill: float | None = None,
                 k_pool: torch.Tensor | None = None, v_pool: torch.Tensor | None = None,
                 host_pools: bool = False):
        device = torch.device(device) if device is not None else page_table.device
        shape = (num_pages, num_kv_heads, page_size, HEAD_DIM)
        if k_pool is None:
            if host_pools:
                k_pool = torch.empty(shape, dtype=torch.bfloat16, pin_memory=True)
                v_pool = torch.empty(shape, dtype=torch.bfloat16, pin_memory=True)
            else:
                k_pool = torch.empty(shape, dtype=torch.bfloat16, device=device)
                v_pool = torch.empty(shape, dtype=torch.bfloat16, device=device)
            if fill is not None:
                k_pool.fill_(fill)
                v_pool.fill_(fill)
        _check_pool(k_pool, "k_pool", shape)
        _check_pool(v_pool, "v_pool", shape)
        _check(page_table, "page_table", torch.int32)
        self.k_pool, self.v_pool, self.page_table = k_pool, v_pool, page_table
        self.page_size, self.num_kv_heads, self.num_tokens = page_size, num_kv_heads, num_tokens
        self.struct = B.ls_kv_cache(k_pool.data_ptr(), v_pool.data_ptr(), page_table.data_ptr(),
                                    num_pages, page_table.numel(), page_size, num_kv_heads,
                                    HEAD_DIM, num_tokens)

    @property
    def device(self):
        return self.page_table.device

    def capture(self, k: torch.Tensor, v: torch.Tensor, start_pos: int = 0, stream=None) -> None:
        n = k.shape[0]
        _check(k, "k", torch.bfloat16, (n, self.num_kv_heads, HEAD_DIM))
        _check(v, "v", torch.bfloat16, (n, self.num_kv_heads, HEAD_DIM))
        B.ls_capture_kv(self.struct, k.data_ptr(), v.data_ptr(), start_pos, n, _stream(stream))

    def validate(self, stream=None) -> None:
        nbytes = B.ls_validate_page_table_workspace(self.struct)
        ws = torch.empty(nbytes, dtype=torch.uint8, device=self.device)
        B.ls_validate_page_table(self.struct, ws.data_ptr(), nbytes, _stream(stream))


def replay_fwd(cache: PagedKVCache, q: torch.Tensor, k_resp: torch.Tensor, v_resp: torch.Tensor,
               softmax_scale: float, num_splits: int, o: torch.Tensor | None = None,
               lse: torch.Tensor | None = None, stream=None):
    R, hq, _ = q.shape
    _check(q, "q", torch.bfloat16, (R, hq, HEAD_DIM))
    _check(k_resp, "k_resp", torch.bfloat16, (R, cache.num_kv_heads, HEAD_DIM))
    _check(v_resp, "v_resp", torch.bfloat16, (R, cache.num_kv_heads, HEAD_DIM))
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((R, hq), dtype=torch.float32, device=q.device)
    _check(o, "o", torch.bfloat16, q.shape)
    _check(lse, "lse", torch.float32, (R, hq))
    nbytes = B.ls_replay_attn_fwd_workspace(cache.struct, R, hq, num_splits)
    ws = workspace(nbytes, q.device, "fwd")
    B.ls_replay_attn_fwd(cache.struct, q.data_ptr(), k_resp.data_ptr(), v_resp.data_ptr(), R, hq,
                         softmax_scale, num_splits, o.data_ptr(), lse.data_ptr(), ws.data_ptr(),
                         ws.numel(), _stream(stream))
    return o, lse


def replay_fwd_members(cache: PagedKVCache, q: torch.Tensor, k_resp: torch.Tensor,
                       v_resp: torch.Tensor, softmax_scale: float, num_splits: int,
                       o: torch.Tensor | None = None, lse: torch.Tensor | None = None,
                       stream=None):
    """Forward of several equal-length responses over the prompt in one launch:
    q [members][R][Hq][128], k_resp / v_resp [members][R][Hkv][128]."""
    M, R, hq, _ = q.shape
    hkv = cache.num_kv_heads
    _check(q, "q", torch.bfloat16, (M, R, hq, HEAD_DIM))
    _check(k_resp, "k_resp", torch.bfloat16, (M, R, hkv, HEAD_DIM))
    _check(v_resp, "v_resp", torch.bfloat16, (M, R, hkv, HEAD_DIM))
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((M, R, hq), dtype=torch.float32, device=q.device)
    _check(o, "o", torch.bfloat16, q.shape)
    _check(lse, "lse", torch.float32, (M, R, hq))
    nbytes = B.ls_replay_attn_fwd_members_workspace(cache.struct, R, M, hq, num_splits)
    ws = workspace(nbytes, q.device, "fwd")
    B.ls_replay_attn_fwd_members(cache.struct, q.data_ptr(), k_resp.data_ptr(),
                                 v_resp.data_ptr(), R, M, hq, softmax_scale, num_splits,
                                 o.data_ptr(), lse.data_ptr(), ws.data_ptr(), ws.numel(),
                                 _stream(stream))
    return o, lse


def replay_bwd(cache: PagedKVCache, q, k_resp, v_resp, o, lse, d_o, softmax_scale: float,
               num_splits: int, dq=None, dk=None, dv=None, accumulate: bool = False, stream=None):
    R, hq, _ = q.shape
    hkv = cache.num_kv_heads
    for t, n in ((q, "q"), (o, "o"), (d_o, "d_o")):
        _check(t, n, torch.bfloat16, (R, hq, HEAD_DIM))
    _check(k_resp, "k_resp", torch.bfloat16, (R, hkv, HEAD_DIM))
    _check(v_resp, "v_resp", torch.bfloat16, (R, hkv, HEAD_DIM))
    _check(lse, "lse", torch.float32, (R, hq))
    if dq is None:
        dq = torch.empty((R, hq, HEAD_DIM), dtype=torch.float32, device=q.device)
    if dk is None:
        dk = torch.empty((R, hkv, HEAD_DIM), dtype=torch.float32, device=q.device)
    if dv is None:
        dv = torch.empty((R, hkv, HEAD_DIM), dtype=torch.float32, device=q.device)
    _check(dq, "dq", torch.float32, (R, hq, HEAD_DIM))
    _check(dk, "dk", torch.float32, (R, hkv, HEAD_DIM))
    _check(dv, "dv", torch.float32, (R, hkv, HEAD_DIM))
    nbytes = B.ls_replay_attn_bwd_workspace(cache.struct, R, hq, num_splits)
    ws = workspace(nbytes, q.device, "bwd")
    B.ls_replay_attn_bwd(cache.struct, q.data_ptr(), k_resp.data_ptr(), v_resp.data_ptr(),
                         o.data_ptr(), lse.data_ptr(), d_o.data_ptr(), R, hq, softmax_scale,
                         num_splits, int(accumulate), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                         ws.data_ptr(), ws.numel(), _stream(stream))
    return dq, dk, dv


def grpo_loss_fwd_bwd(logits: torch.Tensor, targets: torch.Tensor, logp_old: torch.Tensor,
                      rewards: torch.Tensor, resp_lens: torch.Tensor, member_begin: int,
                      member_end: int, eps: float, adv_eps: float = 1e-6, std_ddof: int = 1,
                      loss: torch.Tensor | None = None, accumulate: bool = False,
                      dlogits: torch.Tensor | None = None, logp_out: torch.Tensor | None = None,
                      stats: torch.Tensor | None = None, stream=None):
    """Returns (loss[1], dlogits, logp[T], stats[4]); loss accumulates when asked."""
    T, V = logits.shape
    if logits.dtype == torch.bfloat16:
        dt = B.LS_BF16
    elif logits.dtype == torch.float32:
        dt = B.LS_FP32
    else:
        raise ValueError("logits must be bf16 or fp32")
    _check(logits, "logits", logits.dtype)
    _check(targets, "targets", torch.int32, (T,))
    _check(logp_old, "logp_old", torch.float32, (T,))
    G = rewards.numel()
    _check(rewards, "rewards", torch.float32, (G,))
    _check(resp_lens, "resp_lens", torch.int32, (G,))
    dev = logits.device
    if loss is None:
        loss = torch.zeros(1, dtype=torch.float32, device=dev)
    if dlogits is None:
        dlogits = torch.empty_like(logits)
    if logp_out is None:
        logp_out = torch.empty(T, dtype=torch.float32, device=dev)
    if stats is None:
        stats = torch.empty(4, dtype=torch.float32, device=dev)
    _check(dlogits, "dlogits", logits.dtype, (T, V))
    nbytes = B.ls_grpo_workspace(T, G)
    ws = workspace(nbytes, dev, "grpo")
    B.ls_grpo_loss_fwd_bwd(logits.data_ptr(), dt, T, V, targets.data_ptr(), logp_old.data_ptr(),
                           rewards.data_ptr(), resp_lens.data_ptr(), G, member_begin, member_end,
                           eps, adv_eps, std_ddof, int(accumulate), loss.data_ptr(),
                           dlogits.data_ptr(), logp_out.data_ptr(), stats.data_ptr(),
                           ws.data_ptr(), ws.numel(), _stream(stream))
    return loss, dlogits, logp_out, stats


def grpo_logp(logits: torch.Tensor, targets: torch.Tensor, ref_logp: torch.Tensor | None = None,
              with_lse: bool = False, stream=None):
    """Pre-step scoring: returns (logp[T], lse[T] or None, kl[T] or None)."""
    T, V = logits.shape
    if logits.dtype == torch.bfloat16:
        dt = B.LS_BF16
    elif logits.dtype == torch.float32:
        dt = B.LS_FP32
    else:
        raise ValueError("logits must be bf16 or fp32")
    _check(logits, "logits", logits.dtype)
    _check(targets, "targets", torch.int32, (T,))
    dev = logits.device
    logp = torch.empty(T, dtype=torch.float32, device=dev)
    lse = torch.empty(T, dtype=torch.float32, device=dev) if with_lse else None
    kl = None
    if ref_logp is not None:
        _check(ref_logp, "ref_logp", torch.float32, (T,))
        kl = torch.empty(T, dtype=torch.float32, device=dev)
    B.ls_grpo_logp(logits.data_ptr(), dt, T, V, targets.data_ptr(),
                   ref_logp.data_ptr() if ref_logp is not None else None, logp.data_ptr(),
                   lse.data_ptr() if lse is not None else None,
                   kl.data_ptr() if kl is not None else None, _stream(stream))
    return logp, lse, kl


def replay_fwd_ragged(cache: PagedKVCache, q: torch.Tensor, k_resp: torch.Tensor,
                      v_resp: torch.Tensor, lens, softmax_scale: float, num_splits: int,
                      o: torch.Tensor | None = None, lse: torch.Tensor | None = None, stream=None):
    """Forward of ragged members laid out back to back: q [T][Hq][128], k_resp / v_resp
    [T][Hkv][128], lens the members' lengths (summing to T)."""
    T, hq, _ = q.shape
    lens = [int(x) for x in lens]
    if sum(lens) != T:
        raise ValueError("member lengths must add up to the token count")
    _check(q, "q", torch.bfloat16, (T, hq, HEAD_DIM))
    _check(k_resp, "k_resp", torch.bfloat16, (T, cache.num_kv_heads, HEAD_DIM))
    _check(v_resp, "v_resp", torch.bfloat16, (T, cache.num_kv_heads, HEAD_DIM))
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((T, hq), dtype=torch.float32, device=q.device)
    nbytes = B.ls_replay_attn_fwd_ragged_workspace(cache.struct, lens, hq, num_splits)
    ws = workspace(nbytes, q.device, "fwd")
    B.ls_replay_attn_fwd_ragged(cache.struct, q.data_ptr(), k_resp.data_ptr(), v_resp.data_ptr(),
                                lens, hq, softmax_scale, num_splits, o.data_ptr(), lse.data_ptr(),
                                ws.data_ptr(), ws.numel(), _stream(stream))
    return o, lse


def replay_bwd_ragged(cache: PagedKVCache, q, k_resp, v_resp, o, lse, d_o, lens,
                      softmax_scale: float, num_splits: int, dq=None, dk=None, dv=None,
                      accumulate: bool = False, stream=None):
    """Backward of ragged members laid out back to back (see replay_fwd_ragged)."""
    T, hq, _ = q.shape
    hkv = cache.num_kv_heads
    lens = [int(x) for x in lens]
    if sum(lens) != T:
        raise ValueError("member lengths must add up to the token count")
    for t, n in ((q, "q"), (o, "o"), (d_o, "d_o")):
        _check(t, n, torch.bfloat16, (T, hq, HEAD_DIM))
    _check(lse, "lse", torch.float32, (T, hq))
    dev = q.device
    if dq is None:
        dq = torch.empty((T, hq, HEAD_DIM), dtype=torch.float32, device=dev)
    if dk is None:
        dk = torch.empty((T, hkv, HEAD_DIM), dtype=torch.float32, device=dev)
    if dv is None:
        dv = torch.empty((T, hkv, HEAD_DIM), dtype=torch.float32, device=dev)
    nbytes = B.ls_replay_attn_bwd_ragged_workspace(cache.struct, lens, hq, num_splits)
    ws = workspace(nbytes, dev, "bwd")
    B.ls_replay_attn_bwd_ragged(cache.struct, q.data_ptr(), k_resp.data_ptr(), v_resp.data_ptr(),
                                o.data_ptr(), lse.data_ptr(), d_o.data_ptr(), lens, hq,
                                softmax_scale, num_splits, int(accumulate), dq.data_ptr(),
                                dk.data_ptr(), dv.data_ptr(), ws.data_ptr(), ws.numel(),
                                _stream(stream))
    return dq, dk, dv


def gdn_replay_fwd(state0: torch.Tensor, q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                   g: torch.Tensor, beta: torch.Tensor, scale: float, o: torch.Tensor | None = None,
                   state_out: torch.Tensor | None = None, with_state: bool = False, stream=None):
    """Gated-DeltaNet replay of R tokens from a captured state: state0 fp32 [H][128][128],
    q/k/v bf16 [R][H][128], g/beta fp32 [R][H].  Returns (o, state_out or None)."""
    R, H, _ = q.shape
    _check(state0, "state0", torch.float32, (H, HEAD_DIM, HEAD_DIM))
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _check(t, n, torch.bfloat16, (R, H, HEAD_DIM))
    _check(g, "g", torch.float32, (R, H))
    _check(beta, "beta", torch.float32, (R, H))
    if o is None:
        o = torch.empty_like(q)
    if state_out is None and with_state:
        state_out = torch.empty_like(state0)
    nbytes = B.ls_gdn_replay_fwd_workspace(R, H)
    ws = workspace(nbytes, q.device, "gdn")
    B.ls_gdn_replay_fwd(state0.data_ptr(), q.data_ptr(), k.data_ptr(), v.data_ptr(), g.data_ptr(),
                        beta.data_ptr(), R, H, scale, o.data_ptr(),
                        state_out.data_ptr() if state_out is not None else None, ws.data_ptr(),
                        ws.numel(), _stream(stream))
    return o, state_out


def gdn_replay_bwd(state0, q, k, v, g, beta, d_o, scale: float, grads=None,
                   accumulate: bool = False, stream=None):
    """Gradients (dq, dk, dv, dg, dbeta) of the replay with the captured state stopgrad."""
    R, H, _ = q.shape
    _check(d_o, "d_o", torch.bfloat16, (R, H, HEAD_DIM))
    if grads is None:
        dev = q.device
        grads = (torch.empty((R, H, HEAD_DIM), dtype=torch.float32, device=dev),
                 torch.empty((R, H, HEAD_DIM), dtype=torch.float32, device=dev),
                 torch.empty((R, H, HEAD_DIM), dtype=torch.float32, device=dev),
                 torch.empty((R, H), dtype=torch.float32, device=dev),
                 torch.empty((R, H), dtype=torch.float32, device=dev))
    dq, dk, dv, dg, db = grads
    nbytes = B.ls_gdn_replay_bwd_workspace(R, H)
    ws = workspace(nbytes, q.device, "gdn")
    B.ls_gdn_replay_bwd(state0.data_ptr(), q.data_ptr(), k.data_ptr(), v.data_ptr(), g.data_ptr(),
                        beta.data_ptr(), d_o.data_ptr(), R, H, scale, int(accumulate),
                        dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), dg.data_ptr(), db.data_ptr(),
                        ws.data_ptr(), ws.numel(), _stream(stream))
    return dq, dk, dv, dg, db


def last_device_error(stream=None) -> int:
    return B.ls_last_device_error(_stream(stream))


# ---------------------------------------------------------------- latent (MLA) replay

LATENT_DIM = 512           # c_j: the values attention averages
LATENT_ROW = 576           # c_j followed by the 64-value rotary key


class LatentCache:
    """Latent (MLA-style) pages of one layer plus page table (ls_latent_cache): rows of
    LATENT_ROW bf16 values shared by all heads.  host_pool=True places the pool in pinned
    host memory (Grace memory on a Grace-Blackwell node), read there by the kernels."""

    def __init__(self, num_pages: int, page_table: torch.Tensor, page_size: int, num_tokens: int,
                 device=None, fill: float | None = None, pool: torch.Tensor | None = None,
                 host_pool: bool = False):
        device = torch.device(device) if device is not None else page_table.device
        shape = (num_pages, page_size, LATENT_ROW)
        if pool is None:
            pool = (torch.empty(shape, dtype=torch.bfloat16, pin_memory=True) if host_pool
                    else torch.empty(shape, dtype=torch.bfloat16, device=device))
            if fill is not None:
                pool.fill_(fill)
        _check_pool(pool, "pool", shape)
        _check(page_table, "page_table", torch.int32)
        self.pool, self.page_table = pool, page_table
        self.page_size, self.num_tokens = page_size, num_tokens
        self.struct = B.ls_latent_cache(pool.data_ptr(), page_table.data_ptr(), num_pages,
                                        page_table.numel(), page_size, num_tokens)

    @property
    def device(self):
        return self.page_table.device

    def capture(self, lat: torch.Tensor, start_pos: int = 0, stream=None) -> None:
        n = lat.shape[0]
        _check(lat, "lat", torch.bfloat16, (n, LATENT_ROW))
        B.ls_capture_latent(self.struct, lat.data_ptr(), start_pos, n, _stream(stream))


def mla_replay_fwd(cache: LatentCache, q: torch.Tensor, lat_resp: torch.Tensor,
                   softmax_scale: float, num_splits: int, o: torch.Tensor | None = None,
                   lse: torch.Tensor | None = None, stream=None):
    """q [R][H][576] absorbed queries, lat_resp [R][576] the response's own rows ->
    o [R][H][512] (bf16), lse [R][H] (fp32)."""
    R, H, _ = q.shape
    _check(q, "q", torch.bfloat16, (R, H, LATENT_ROW))
    _check(lat_resp, "lat_resp", torch.bfloat16, (R, LATENT_ROW))
    if o is None:
        o = torch.empty((R, H, LATENT_DIM), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((R, H), dtype=torch.float32, device=q.device)
    _check(o, "o", torch.bfloat16, (R, H, LATENT_DIM))
    _check(lse, "lse", torch.float32, (R, H))
    nbytes = B.ls_mla_replay_fwd_workspace(cache.struct, R, H, num_splits)
    ws = workspace(nbytes, q.device, "mla_fwd")
    B.ls_mla_replay_fwd(cache.struct, q.data_ptr(), lat_resp.data_ptr(), R, H, softmax_scale,
                        num_splits, o.data_ptr(), lse.data_ptr(), ws.data_ptr(), ws.numel(),
                        _stream(stream))
    return o, lse


def mla_replay_bwd(cache: LatentCache, q: torch.Tensor, lat_resp: torch.Tensor, o: torch.Tensor,
                   lse: torch.Tensor, d_o: torch.Tensor, softmax_scale: float, num_splits: int,
                   dq: torch.Tensor | None = None, dlat: torch.Tensor | None = None, stream=None):
    """Backward of mla_replay_fwd with the prompt rows stopgrad: o, lse from the forward,
    d_o [R][H][512] bf16 -> dq [R][H][576] and dlat [R][576] (fp32, the gradient of the
    response's own rows)."""
    R, H, _ = q.shape
    _check(q, "q", torch.bfloat16, (R, H, LATENT_ROW))
    _check(lat_resp, "lat_resp", torch.bfloat16, (R, LATENT_ROW))
    _check(o, "o", torch.bfloat16, (R, H, LATENT_DIM))
    _check(lse, "lse", torch.float32, (R, H))
    _check(d_o, "d_o", torch.bfloat16, (R, H, LATENT_DIM))
    if dq is None:
        dq = torch.empty((R, H, LATENT_ROW), dtype=torch.float32, device=q.device)
    if dlat is None:
        dlat = torch.empty((R, LATENT_ROW), dtype=torch.float32, device=q.device)
    _check(dq, "dq", torch.float32, (R, H, LATENT_ROW))
    _check(dlat, "dlat", torch.float32, (R, LATENT_ROW))
    nbytes = B.ls_mla_replay_bwd_workspace(cache.struct, R, H, num_splits)
    ws = workspace(nbytes, q.device, "mla_bwd")
    B.ls_mla_replay_bwd(cache.struct, q.data_ptr(), lat_resp.data_ptr(), o.data_ptr(),
                        lse.data_ptr(), d_o.data_ptr(), R, H, softmax_scale, num_splits,
                        dq.data_ptr(), dlat.data_ptr(), ws.data_ptr(), ws.numel(),
                        _stream(stream))
    return dq, dlat
