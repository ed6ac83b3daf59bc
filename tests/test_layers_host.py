"""Host logic of the multi-layer reverse replay (response_replay_gb300/layers.py) on the
CPU: layers run last first, each layer's dK / dV are allocated by its own backward and
handed on, a first touch writes and later touches add.  The replay backward itself is
replaced by a stand-in that records its calls (the CUDA path is checked in
test_gpu_layers.py)."""
import torch

from response_replay_gb300 import layers as L
from response_replay_gb300 import torch_api as api


def fake_bwd(calls):
    def run(cache, q, k, v, o, lse, d_o, scale, splits, dq=None, dk=None, dv=None,
            accumulate=False, stream=None):
        calls.append((cache, accumulate, dk.data_ptr(), float(d_o.sum())))
        val = float(d_o.sum())
        for t in (dq, dk, dv):
            if accumulate:
                t += val
            else:
                t.fill_(val)
        return dq, dk, dv
    return run


def saved_entry(R=5, hq=4, hkv=2):
    q = torch.zeros(R, hq, api.HEAD_DIM)
    kv = torch.zeros(R, hkv, api.HEAD_DIM)
    return (q, kv, kv, q, torch.zeros(R, hq))


def test_layers_run_last_first_and_hold_one_layer(monkeypatch):
    calls, seen = [], []
    monkeypatch.setattr(api, "replay_bwd", fake_bwd(calls))
    layers = ["layer0", "layer1", "layer2"]
    saved = [saved_entry() for _ in layers]

    def upstream(l):
        return torch.full((5, 4, api.HEAD_DIM), float(l + 1))

    def consume(l, dq, dk, dv):
        seen.append(l)
        assert len(calls) == len(seen)            # layer l's backward ran just before
        assert dk.shape == (5, 2, api.HEAD_DIM) and dv.shape == dk.shape
        assert torch.all(dk == float(upstream(l).sum()))

    L.reverse_replay_bwd(layers, saved, upstream, consume, 0.1, 4)
    assert seen == [2, 1, 0]
    assert [c[0] for c in calls] == ["layer2", "layer1", "layer0"]
    assert all(not c[1] for c in calls)          # each layer's first touch writes


def test_grad_pages_allocate_on_first_touch_and_add_after(monkeypatch):
    calls = []
    monkeypatch.setattr(api, "replay_bwd", fake_bwd(calls))
    g = L.KVGradPages(5, 2, "cpu")
    assert not g.allocated
    q, k, v, o, lse = saved_entry()
    dq1 = g.backward("c", q, k, v, o, lse, torch.ones(5, 4, api.HEAD_DIM), 0.1, 2)
    assert g.allocated and g.touches == 1 and calls[0][1] is False
    ptr = g.dk.data_ptr()
    dq2 = g.backward("c", q, k, v, o, lse, 2 * torch.ones(5, 4, api.HEAD_DIM), 0.1, 2)
    assert calls[1][1] is True and g.dk.data_ptr() == ptr   # same buffers, added to
    n = 5 * 4 * api.HEAD_DIM
    assert torch.all(g.dk == n + 2 * n)
    assert torch.all(dq1 == n) and torch.all(dq2 == 2 * n)  # fresh dQ per call
    dk, dv = g.release()
    assert not g.allocated and torch.all(dv == 3 * n)


def test_saved_must_match_layers(monkeypatch):
    monkeypatch.setattr(api, "replay_bwd", fake_bwd([]))
    try:
        L.reverse_replay_bwd(["a", "b"], [saved_entry()], lambda l: None,
                             lambda *a: None, 0.1, 1)
    except ValueError:
        return
    raise AssertionError("mismatched saved list accepted")
