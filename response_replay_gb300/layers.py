"""Several attention layers over one captured prompt, and their backward in reverse
layer order.

A model replays a response through its layers forward, then runs the backward from the
last layer to the first (explainer "LongStraw: fitting million-token RL onto a fixed GPU
budget", section "Two incompatible architectures, same transaction", Qwen bullet: the
response's blocks are replayed in reverse, and K/V gradient pages exist only once a
response backward touches them).  The layers are joined by the model's weights, which
this library does not hold: the caller supplies each layer's upstream gradient dO and
takes its dQ / dK / dV.  This module holds the part that needs no weights:

- ``LayeredKVCache``: the captured prompt K/V of L layers.  The prompt's token -> page
  map is the same in every layer, so one page table serves all of them; the pools are
  one [L][pages][Hkv][page][128] allocation for K and one for V, and layer l is an
  ordinary ``PagedKVCache`` over slice l.
- ``KVGradPages``: one response's dK / dV in one layer, allocated by the first backward
  that touches them and written by it (no zero fill); a later backward over the same
  keys adds to them (the C ABI's ``accumulate`` flag).
- ``reverse_replay_bwd``: the backward of one response through all layers, last layer
  first.  A layer's dK / dV are allocated at that layer's backward and dropped once the
  caller's consumer returns, so one layer's K/V gradients are alive at a time.
- ``StreamedLayers``: the L layers' prompt pages in pinned host memory (Grace memory on a
  GB300 node), streamed into a two-slot page cache in GPU memory one layer ahead of the
  replay that reads them (explainer, same section, GLM bullet: the prompt's pages held in
  CPU memory); ``StreamedLatentLayers`` does the same for latent (MLA-style) pages.

Every step of the computation is a call of the replay backward in the CUDA library.
"""
from __future__ import annotations

from typing import Callable, Sequence

import torch

from . import torch_api as api


class LayeredKVCache:
    """Captured prompt K/V of ``num_layers`` attention layers under one page table."""

    def __init__(self, num_layers: int, num_pages: int, page_table: torch.Tensor,
                 page_size: int, num_kv_heads: int, num_tokens: int, device=None,
                 fill: float | None = None):
        if num_layers < 1:
            raise ValueError("num_layers must be at least 1")
        device = torch.device(device) if device is not None else page_table.device
        shape = (num_layers, num_pages, num_kv_heads, page_size, api.HEAD_DIM)
        self.k_pools = torch.empty(shape, dtype=torch.bfloat16, device=device)
        self.v_pools = torch.empty(shape, dtype=torch.bfloat16, device=device)
        if fill is not None:
            self.k_pools.fill_(fill)
            self.v_pools.fill_(fill)
        self.page_table = page_table
        self.layers = [api.PagedKVCache(num_pages, page_table, page_size, num_kv_heads,
                                        num_tokens, device=device, k_pool=self.k_pools[l],
                                        v_pool=self.v_pools[l])
                       for l in range(num_layers)]

    def __len__(self) -> int:
        return len(self.layers)

    def __getitem__(self, layer: int) -> api.PagedKVCache:
        return self.layers[layer]

    def capture(self, layer: int, k: torch.Tensor, v: torch.Tensor, start_pos: int = 0,
                stream=None) -> None:
        self.layers[layer].capture(k, v, start_pos, stream)


class KVGradPages:
    """dK / dV [R][Hkv][128] fp32 of one response in one layer, allocated on first touch."""

    def __init__(self, R: int, num_kv_heads: int, device):
        self.shape = (R, num_kv_heads, api.HEAD_DIM)
        self.device = torch.device(device)
        self.dk = self.dv = None
        self.touches = 0

    @property
    def allocated(self) -> bool:
        return self.dk is not None

    def backward(self, cache: api.PagedKVCache, q, k_resp, v_resp, o, lse, d_o,
                 softmax_scale: float, num_splits: int, dq=None, stream=None):
        """One replay backward over this response's keys; returns dQ.  The first call
        allocates dK / dV and writes them, later calls add to them.  A dQ passed in is
        written on the first call and added to on later ones, like dK / dV."""
        first = self.dk is None
        if first:
            self.dk = torch.empty(self.shape, dtype=torch.float32, device=self.device)
            self.dv = torch.empty(self.shape, dtype=torch.float32, device=self.device)
            if dq is None:
                dq = torch.empty(q.shape, dtype=torch.float32, device=self.device)
        elif dq is None:
            dq = torch.zeros(q.shape, dtype=torch.float32, device=self.device)
        dq, _, _ = api.replay_bwd(cache, q, k_resp, v_resp, o, lse, d_o, softmax_scale,
                                  num_splits, dq=dq, dk=self.dk, dv=self.dv,
                                  accumulate=not first, stream=stream)
        self.touches += 1
        return dq

    def release(self):
        """Hands dK / dV to the caller and drops this object's references."""
        dk, dv = self.dk, self.dv
        self.dk = self.dv = None
        return dk, dv


def reverse_replay_bwd(layers: LayeredKVCache, saved: Sequence[tuple],
                       upstream: Callable[[int], torch.Tensor],
                       consume: Callable[[int, torch.Tensor, torch.Tensor, torch.Tensor], None],
                       softmax_scale: float, num_splits: int, stream=None) -> None:
    """Backward of one response through every layer, last layer first.

    saved[l] = (q, k_resp, v_resp, o, lse) of layer l from the forward replay;
    upstream(l) returns layer l's dO (called after layer l + 1 was consumed, so it may
    depend on what the consumer did with it); consume(l, dq, dk, dv) receives layer l's
    gradients, which this function does not keep."""
    if len(saved) != len(layers):
        raise ValueError("one saved entry per layer is required")
    for l in reversed(range(len(layers))):
        q, k_resp, v_resp, o, lse = saved[l]
        grads = KVGradPages(k_resp.shape[0], k_resp.shape[1], q.device)
        dq = grads.backward(layers[l], q, k_resp, v_resp, o, lse, upstream(l), softmax_scale,
                            num_splits, stream=stream)
        dk, dv = grads.release()
        consume(l, dq, dk, dv)


class _TwoSlotLayers:
    """Every layer's captured pages in pinned host memory (on a Grace-Blackwell node,
    Grace memory: room for every layer of a long prompt, which HBM would not hold),
    streamed into a two-slot page cache in GPU memory one layer ahead of the replay that
    reads them.

    The kernels could read the host pages directly, but every unit of a long replay
    re-reads the prompt and those reads are not kept in L2, so a long replay from host
    pages is bound by the host link many times over.  Copied once into GPU memory, a
    layer's pages serve every unit at HBM speed, and the copy of the next layer runs on
    its own stream while the current layer is replayed.

    Use: ``prefetch(l)`` starts layer l's copy into slot l % 2 (the copy waits for the
    work already queued on the current stream and for the release of the slot's previous
    layer; a slot whose layer was never released is not overwritten: ValueError);
    ``cache(l)`` returns the layer's cache in GPU memory and makes the current stream wait
    for its copy; ``release(l)`` marks the point on the current stream after which the
    slot may be overwritten.  Capture writes the host pages directly (``capture``).
    Subclasses name the caches and their page pools."""

    def __init__(self, host: list, slots: list, device, bytes_per_layer: int):
        self.device = device
        self.host = host
        self.slots = slots
        self.copy_stream = torch.cuda.Stream(device)
        self.ready = [torch.cuda.Event() for _ in range(2)]
        self.free = [torch.cuda.Event() for _ in range(2)]
        self.held = [False, False]       # a layer was copied into the slot
        self.released = [False, False]   # ... and released since (free[s] marks when)
        self.layer_in = [None, None]     # layer held (or being copied) by each slot
        self.bytes_per_layer = bytes_per_layer

    @staticmethod
    def _pools(cache) -> tuple:
        raise NotImplementedError

    def __len__(self) -> int:
        return len(self.host)

    def _stale(self, layer: int) -> None:
        for s in range(2):              # a slot holding this layer is now stale
            if self.layer_in[s] == layer:
                self.layer_in[s] = None

    def _slot(self, layer: int) -> int:
        for s in range(2):
            if self.layer_in[s] == layer:
                return s
        return layer % 2

    def prefetch(self, layer: int) -> None:
        s = self._slot(layer)
        if self.layer_in[s] == layer:
            return
        if self.held[s] and not self.released[s]:
            raise ValueError(f"slot {s} still holds layer {self.layer_in[s]}: release it "
                             f"before prefetching layer {layer}")
        cs = self.copy_stream
        # the capture that wrote the host pages and the work queued so far come first, and
        # the slot's previous layer's last reader (marked by its release)
        cs.wait_stream(torch.cuda.current_stream(self.device))
        if self.held[s]:
            cs.wait_event(self.free[s])
        with torch.cuda.stream(cs):
            for dst, src in zip(self._pools(self.slots[s]), self._pools(self.host[layer])):
                dst.copy_(src, non_blocking=True)
            self.ready[s].record(cs)
        self.layer_in[s] = layer
        self.held[s] = True
        self.released[s] = False

    def cache(self, layer: int):
        self.prefetch(layer)
        s = self._slot(layer)
        torch.cuda.current_stream(self.device).wait_event(self.ready[s])
        return self.slots[s]

    def release(self, layer: int) -> None:
        s = self._slot(layer)
        if self.layer_in[s] == layer:
            self.free[s].record(torch.cuda.current_stream(self.device))
            self.released[s] = True


class StreamedLayers(_TwoSlotLayers):
    """The captured prompt K/V pages of L attention layers in pinned host memory,
    streamed through a two-slot GPU page cache (see _TwoSlotLayers)."""

    def __init__(self, num_layers: int, num_pages: int, page_table: torch.Tensor,
                 page_size: int, num_kv_heads: int, num_tokens: int, device=None):
        if num_layers < 1:
            raise ValueError("num_layers must be at least 1")
        device = torch.device(device) if device is not None else page_table.device
        shape = (num_pages, num_kv_heads, page_size, api.HEAD_DIM)
        host = [api.PagedKVCache(num_pages, page_table, page_size, num_kv_heads, num_tokens,
                                 host_pools=True) for _ in range(num_layers)]
        slots = [api.PagedKVCache(num_pages, page_table, page_size, num_kv_heads, num_tokens,
                                  device=device) for _ in range(2)]
        super().__init__(host, slots, device, 2 * int(torch.Size(shape).numel()) * 2)

    @staticmethod
    def _pools(cache) -> tuple:
        return cache.k_pool, cache.v_pool

    def capture(self, layer: int, k: torch.Tensor, v: torch.Tensor, start_pos: int = 0,
                stream=None) -> None:
        self.host[layer].capture(k, v, start_pos, stream)
        self._stale(layer)


class StreamedLatentLayers(_TwoSlotLayers):
    """The captured latent (MLA-style) pages of L latent-attention layers in pinned host
    memory (the GLM layers' CPU-resident latent pages of the explainer, GLM bullet),
    streamed through a two-slot GPU page cache (see _TwoSlotLayers)."""

    def __init__(self, num_layers: int, num_pages: int, page_table: torch.Tensor,
                 page_size: int, num_tokens: int, device=None):
        if num_layers < 1:
            raise ValueError("num_layers must be at least 1")
        device = torch.device(device) if device is not None else page_table.device
        host = [api.LatentCache(num_pages, page_table, page_size, num_tokens, host_pool=True)
                for _ in range(num_layers)]
        slots = [api.LatentCache(num_pages, page_table, page_size, num_tokens, device=device)
                 for _ in range(2)]
        super().__init__(host, slots, device, num_pages * page_size * api.LATENT_ROW * 2)

    @staticmethod
    def _pools(cache) -> tuple:
        return (cache.pool,)

    def capture(self, layer: int, lat: torch.Tensor, start_pos: int = 0, stream=None) -> None:
        self.host[layer].capture(lat, start_pos, stream)
        self._stale(layer)
