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


class _Log:
    """Records stream / event operations of the two-slot layer cache."""

    def __init__(self):
        self.ops = []


def _fake_cuda(monkeypatch, log):
    class Event:
        n = 0

        def __init__(self):
            Event.n += 1
            self.name = f"e{Event.n}"

        def record(self, stream=None):
            log.ops.append(("record", self.name, getattr(stream, "name", "cur")))

    class Stream:
        def __init__(self, device=None, name="copy"):
            self.name = name

        def wait_stream(self, other):
            log.ops.append(("wait_stream", self.name, other.name))

        def wait_event(self, ev):
            log.ops.append(("wait_event", self.name, ev.name))

    class Ctx:
        def __init__(self, s):
            self.s = s

        def __enter__(self):
            return self.s

        def __exit__(self, *a):
            return False

    current = Stream(name="cur")
    monkeypatch.setattr(torch.cuda, "Stream", Stream)
    monkeypatch.setattr(torch.cuda, "Event", Event)
    monkeypatch.setattr(torch.cuda, "current_stream", lambda device=None: current)
    monkeypatch.setattr(torch.cuda, "stream", lambda s: Ctx(s))


class _Pool:
    def __init__(self, log, name):
        self.log, self.name = log, name

    def copy_(self, src, non_blocking=False):
        self.log.ops.append(("copy", self.name, src.name))


class _Cache:
    def __init__(self, log, name):
        self.pool = _Pool(log, name)
        self.captured = 0

    def capture(self, lat, start_pos=0, stream=None):
        self.captured += 1


def test_two_slot_layers_order_their_copies(monkeypatch):
    """Layer l goes to slot l % 2; a slot's copy waits for the current stream (the capture
    and the slot's last reader) and, once the slot has held a layer, for that layer's
    release; a resident layer is not copied again; a new capture makes its slot stale."""
    log = _Log()
    _fake_cuda(monkeypatch, log)
    host = [_Cache(log, f"host{l}") for l in range(3)]
    slots = [_Cache(log, f"slot{s}") for s in range(2)]

    class Layers(L._TwoSlotLayers):
        @staticmethod
        def _pools(cache):
            return (cache.pool,)

    st = Layers(host, slots, "cpu", 123)
    assert len(st) == 3 and st.bytes_per_layer == 123
    st.prefetch(0)
    assert ("copy", "slot0", "host0") in log.ops
    assert ("wait_stream", "copy", "cur") in log.ops
    assert not any(op[0] == "wait_event" and op[1] == "copy" for op in log.ops)
    n = len(log.ops)
    assert st.cache(0) is slots[0]                      # no second copy, a wait for it
    assert [op for op in log.ops[n:] if op[0] == "copy"] == []
    assert log.ops[-1][0] == "wait_event" and log.ops[-1][1] == "cur"
    st.prefetch(1)
    assert log.ops[-2] == ("copy", "slot1", "host1")
    st.release(0)
    release_ev = log.ops[-1][1]
    assert log.ops[-1][0] == "record" and log.ops[-1][2] == "cur"
    n = len(log.ops)
    st.prefetch(2)                                      # reuses slot 0 after its release
    new = log.ops[n:]
    assert ("wait_event", "copy", release_ev) in new
    assert ("copy", "slot0", "host2") in new
    assert new.index(("wait_event", "copy", release_ev)) < new.index(("copy", "slot0", "host2"))
    assert st.layer_in == [2, 1]
    n = len(log.ops)
    st.prefetch(1)                                      # resident: nothing to do
    assert log.ops[n:] == []
    # layer 1 was never released: its slot is not overwritten
    st._stale(1)                                        # as a new capture into layer 1 does
    assert st.layer_in == [2, None]
    try:
        st.prefetch(1)
        raise AssertionError("prefetch over an unreleased slot")
    except ValueError:
        pass
    st.layer_in[1] = 1
    st.release(1)
    st._stale(1)
    st.prefetch(1)                                      # stale after a capture: copied again
    assert log.ops[-2] == ("copy", "slot1", "host1")
