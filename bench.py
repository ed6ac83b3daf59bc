"""Benchmark of the replay hot path on the 2,097,152-position workload.

One step = capture of the prompt K/V into pages (P = 2,097,152, Hkv = 4, 256-token
pages) + serial replay of G = 8 members (R = 4096, Hq = 24): per member the replay
attention forward, the GRPO loss / logits gradient (V = 151,936 bf16) and the replay
attention backward with dQ/dK/dV accumulated across members.  Inputs are synthetic,
seeded, resident in HBM before the timed region (except for the e2e figure, which
copies them in from pinned host memory every step).

Prints one JSON line.  value = algorithmic replay-attention fwd+bwd FLOPs of the step
/ step time (TFLOP/s); components add prompt-KV GB/s and GRPO tokens/s.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "replay attn fwd+bwd TFLOP/s & prompt-KV GB/s at P=2.1M; GRPO loss tokens/s"
WORKLOAD = "p2m"          # the configuration the metric is quoted on (P = 2,097,152)
D = 128
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ------------------------------------------------------------------ work accounting

def attn_flops(P: int, R: int, hq: int) -> tuple[float, float]:
    """Algorithmic FLOPs of one member's forward and backward (exact counts: the
    prompt part is dense R x P, the response part is the causal triangle)."""
    tri = R * (R + 1) / 2
    fwd = 4.0 * hq * D * (R * P + tri)
    bwd = hq * D * (6.0 * R * P + 10.0 * tri)
    return fwd, bwd


def prompt_kv_bytes(P: int, hkv: int) -> float:
    return float(P) * hkv * D * 2 * 2          # K and V, bf16


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def kernel_source_hash(kernel_file: str) -> str:
    """First 16 hex digits of the sha256 of a kernel's .cu file followed by every shared
    header of the library (so a change to a header the kernel uses also counts)."""
    csrc = os.path.join(ROOT, "response_replay_gb300", "csrc")
    h = hashlib.sha256()
    for name in [kernel_file] + sorted(f for f in os.listdir(csrc) if f.endswith((".h", ".cuh"))):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def traffic_from_profile(kernel_file: str, kernel: str):
    """DRAM bytes per launch of `kernel` from the committed ncu summary, or None when
    the summary is missing or was taken on a different version of the kernel source."""
    prof = os.path.join(ROOT, "profiles", f"{kernel}_{WORKLOAD}.md")
    try:
        with open(prof) as f:
            txt = f.read()
        h = kernel_source_hash(kernel_file)
    except OSError:
        return None
    m = re.search(r"source_sha256_16:\s*([0-9a-f]{16})", txt)
    t = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", txt)
    if not m or not t or m.group(1) != h:
        return None
    return float(t.group(1))


# ------------------------------------------------------------------ ranks

def max_over_ranks(x: float, world: int, device=None) -> float:
    """The largest value of x over all ranks (every rank receives it): the whole job
    takes as long as its slowest rank."""
    if world <= 1:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank_step: float, world: int, ms_per_step: float) -> float:
    """Units per second of the whole job: every rank processes the same number of
    independent units per step (weak scaling), and the step lasts the slowest rank's
    time."""
    return units_per_rank_step * world / (ms_per_step * 1e-3)


def cpu_model() -> str:
    """The host CPU's model name (what the oracle baseline ran on), or "unknown"."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def rank_seed(base: int, rank: int) -> int:
    """Each rank replays its own independent problem, drawn from its own seed."""
    return base + 1000 * rank


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines: list[str] = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.t.join(timeout=2)

    def summary(self) -> dict:
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        sm.sort()
        return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------ our arm

def run_ours(args, rank: int, world: int, local_rank: int):
    import numpy as np
    import torch

    from response_replay_gb300 import synthetic as syn
    from response_replay_gb300 import torch_api as api
    from response_replay_gb300 import binding as B

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    w = syn.WORKLOADS[args.workload]
    C = w.cycles                   # replay cycles over one capture (8 on p4m_reuse)
    G = w.G if args.members is None else args.members   # members replayed per cycle
    seed = rank_seed(syn.seed_of(args.workload), rank)
    scale = D ** -0.5
    stream = torch.cuda.current_stream()

    # ---- resident inputs
    pr = syn.make_prompt(w.P, w.hkv, D, w.page_size, seed, dev)
    cache = api.PagedKVCache(pr.num_pages, pr.page_table, w.page_size, w.hkv, w.P, device=dev)
    group_lens = [list(w.R[c * w.G:(c + 1) * w.G]) for c in range(C)]  # whole groups
    replays = [(c, i) for c in range(C) for i in range(G)]
    Rs = {(c, i): group_lens[c][i] for c, i in replays}
    Rmax = max(Rs.values())
    branches = {(c, i): syn.make_branch(Rs[c, i], w.hq, w.hkv, D, seed + 1 + c * w.G + i, dev)
                for c, i in replays}
    gins, offs, logp_olds = [], [], []
    for c in range(C):
        lens = group_lens[c][:G]
        gin = syn.make_grpo(lens, w.vocab, w.logits_dtype, w.rewards, seed + 7919 * c, dev,
                            shift_frac=w.shift_frac)
        if G < w.G:
            # fewer members replayed (profiling): the loss still sees the whole group
            gin.rewards = torch.from_numpy(syn.draw_rewards(
                w.rewards, w.G, np.random.default_rng(seed + 7919 * c))).to(dev)
            gin.resp_lens = torch.tensor(group_lens[c], dtype=torch.int32, device=dev)
        off = [0]
        for n in lens:
            off.append(off[-1] + n)
        # logp_old = logp + noise: logp from one untimed call of the library itself
        logp = torch.empty(off[-1], dtype=torch.float32, device=dev)
        zero = torch.zeros(off[-1], dtype=torch.float32, device=dev)
        for i in range(G):
            api.grpo_loss_fwd_bwd(gin.logits[off[i]:off[i + 1]], gin.targets[off[i]:off[i + 1]],
                                  zero[off[i]:off[i + 1]], gin.rewards, gin.resp_lens, i, i + 1,
                                  0.2, logp_out=logp[off[i]:off[i + 1]],
                                  dlogits=torch.empty_like(gin.logits[off[i]:off[i + 1]]))
        logp_olds.append((logp + gin.noise).contiguous())
        gins.append(gin)
        offs.append(off)
        del zero
    T_step = sum(o_[-1] for o_ in offs)
    o = torch.empty((Rmax, w.hq, D), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((Rmax, w.hq), dtype=torch.float32, device=dev)
    dq = torch.zeros((Rmax, w.hq, D), dtype=torch.float32, device=dev)
    dk = torch.zeros((Rmax, w.hkv, D), dtype=torch.float32, device=dev)
    dv = torch.zeros((Rmax, w.hkv, D), dtype=torch.float32, device=dev)
    dlog = torch.empty((Rmax, w.vocab), dtype=gins[0].logits.dtype, device=dev)
    loss = torch.zeros(1, dtype=torch.float32, device=dev)
    stats = torch.empty(4, dtype=torch.float32, device=dev)
    lp_out = torch.empty(max(o_[-1] for o_ in offs), dtype=torch.float32, device=dev)

    def ev():
        e = torch.cuda.Event(enable_timing=True)
        e.record(stream)
        return e

    def member(c, i, m=None, before_loss=None, inp=None):
        """One replay (member i of cycle c): forward, GRPO loss (accumulating), backward
        with gradient accumulation.  inp: another set of device input buffers (the e2e
        double buffer); default the resident one."""
        R = Rs[c, i]
        if inp is None:
            br = branches[c, i]
            q, kr, vr, d_o = br.q, br.k, br.v, br.d_o
            gin = gins[c]
            logits, targets, lpo = gin.logits, gin.targets, logp_olds[c]
            rewards, lens = gin.rewards, gin.resp_lens
        else:
            q, kr, vr, d_o = inp.br[i]
            logits, targets, lpo, rewards, lens = (inp.logits, inp.targets, inp.logp_old,
                                                   inp.rewards, inp.lens)
        first = c == 0 and i == 0
        api.replay_fwd(cache, q, kr, vr, scale, w.num_splits, o=o[:R], lse=lse[:R],
                       stream=stream)
        if m is not None:
            m.append(ev())
        if before_loss is not None:
            before_loss()
        s, e = offs[c][i], offs[c][i + 1]
        api.grpo_loss_fwd_bwd(logits[s:e], targets[s:e], lpo[s:e], rewards, lens, i, i + 1, 0.2,
                              loss=loss, accumulate=not first, dlogits=dlog[: e - s],
                              logp_out=lp_out[s:e], stats=stats, stream=stream)
        if m is not None:
            m.append(ev())
        api.replay_bwd(cache, q, kr, vr, o[:R], lse[:R], d_o, scale, w.num_splits, dq=dq[:R],
                       dk=dk[:R], dv=dv[:R], accumulate=not first, stream=stream)
        if m is not None:
            m.append(ev())

    # --batched: each cycle's members replay in one ragged forward and one ragged backward
    # launch (their tokens back to back) and one loss call over the cycle's members
    if args.batched:
        cyc = {}
        for c in range(C):
            bs = [branches[c, i] for i in range(G)]
            cyc[c] = tuple(torch.cat([getattr(b, f) for b in bs]).contiguous()
                           for f in ("q", "k", "v", "d_o"))
        Tc = max(o_[-1] for o_ in offs)
        o_c = torch.empty((Tc, w.hq, D), dtype=torch.bfloat16, device=dev)
        lse_c = torch.empty((Tc, w.hq), dtype=torch.float32, device=dev)
        dq_c = torch.zeros((Tc, w.hq, D), dtype=torch.float32, device=dev)
        dk_c = torch.zeros((Tc, w.hkv, D), dtype=torch.float32, device=dev)
        dv_c = torch.zeros((Tc, w.hkv, D), dtype=torch.float32, device=dev)
        dlog_c = torch.empty((Tc, w.vocab), dtype=gins[0].logits.dtype, device=dev)

    def cycle(c, m=None):
        """Cycle c's members in one ragged launch per pass (see --batched)."""
        T = offs[c][-1]
        lens = group_lens[c][:G]
        q, kr, vr, d_o = cyc[c]
        gin = gins[c]
        first = c == 0
        api.replay_fwd_ragged(cache, q, kr, vr, lens, scale, w.num_splits, o=o_c[:T],
                              lse=lse_c[:T], stream=stream)
        if m is not None:
            m.append(ev())
        api.grpo_loss_fwd_bwd(gin.logits, gin.targets, logp_olds[c], gin.rewards, gin.resp_lens,
                              0, G, 0.2, loss=loss, accumulate=not first, dlogits=dlog_c[:T],
                              logp_out=lp_out[:T], stats=stats, stream=stream)
        if m is not None:
            m.append(ev())
        api.replay_bwd_ragged(cache, q, kr, vr, o_c[:T], lse_c[:T], d_o, lens, scale,
                              w.num_splits, dq=dq_c[:T], dk=dk_c[:T], dv=dv_c[:T],
                              accumulate=not first, stream=stream)
        if m is not None:
            m.append(ev())

    groups = list(range(C)) if args.batched else replays

    def step(marks=None):
        m = [ev()] if marks is not None else None
        cache.capture(pr.k, pr.v, 0, stream)
        if m is not None:
            m.append(ev())
        for gr in groups:
            if args.batched:
                cycle(gr, m)
            else:
                member(*gr, m)
        return m

    # kernel launches of one step, as counted by the library itself
    n0 = B.ls_kernel_launches()
    step()
    torch.cuda.synchronize()
    launches = B.ls_kernel_launches() - n0

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()

    # ---- timed region (device-resident inputs)
    marks_all = []
    with ClockSampler(local_rank) as clk:
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        t0 = ev()
        for _ in range(args.steps):
            marks_all.append(step(marks=True))
        t1 = ev()
        torch.cuda.synchronize()
    total_ms = max_over_ranks(t0.elapsed_time(t1), world, dev)
    assert B.ls_last_device_error(0) == B.LS_OK
    assert torch.isfinite(loss).all() and torch.isfinite(dq_c if args.batched else dq).all()

    cap_ms = fwd_ms = grpo_ms = bwd_ms = 0.0
    n_rep = len(replays)
    for m in marks_all:
        cap_ms += m[0].elapsed_time(m[1])
        for r in range(len(groups)):
            a = 1 + 3 * r
            fwd_ms += m[a].elapsed_time(m[a + 1])
            grpo_ms += m[a + 1].elapsed_time(m[a + 2])
            bwd_ms += m[a + 2].elapsed_time(m[a + 3])
    K = args.steps
    flops = [attn_flops(w.P, Rs[r], w.hq) for r in replays]
    f_fwd = sum(f for f, _ in flops)     # per step, all replays
    f_bwd = sum(b for _, b in flops)
    step_flops = f_fwd + f_bwd
    ms_per_step = total_ms / K
    value = whole_job_rate(step_flops, world, ms_per_step) / 1e12
    kv_bytes = prompt_kv_bytes(w.P, w.hkv)
    comps = {
        "attn_fwd_tflops": K * f_fwd / (fwd_ms * 1e-3) / 1e12,
        "attn_bwd_tflops": K * f_bwd / (bwd_ms * 1e-3) / 1e12,
        "prompt_kv_gbs": 2 * n_rep * K * kv_bytes / ((fwd_ms + bwd_ms) * 1e-3) / 1e9,
        "grpo_tokens_per_s": T_step * K / (grpo_ms * 1e-3),
        "capture_gbs": 2 * kv_bytes * K / (cap_ms * 1e-3) / 1e9,
        "ms_capture": cap_ms / K, "ms_fwd_per_member": fwd_ms / (K * n_rep),
        "ms_grpo_per_member": grpo_ms / (K * n_rep), "ms_bwd_per_member": bwd_ms / (K * n_rep),
    }
    pk, pk_src = peaks()
    peak = pk.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"])
    # dominant call: the backward or the forward, whichever takes longer over the step;
    # achieved = its algorithmic FLOPs over all replays / its summed CUDA-event time
    if bwd_ms >= fwd_ms:
        dom, dom_flops, dom_ms, kfile, kname = "replay_attn_bwd", f_bwd, bwd_ms / K, \
            "replay_bwd_dq_tc.cu", "bwd_dq_tc_kernel"
    else:
        dom, dom_flops, dom_ms, kfile, kname = "replay_attn_fwd", f_fwd, fwd_ms / K, \
            "replay_fwd_tc.cu", "replay_fwd_tc_kernel"
    achieved = dom_flops / (dom_ms * 1e-3) / 1e12
    roofline = {"bound": "tensor", "kernel": kname, "timed": f"{dom} calls (CUDA events)",
                "achieved": achieved, "peak": peak, "peak_source": f"{pk_src} bf16 sustained",
                "unit": "TFLOP/s", "frac": achieved / peak,
                "traffic": traffic_from_profile(kfile, kname) if args.workload == WORKLOAD
                else None}

    # ---- e2e: the same step through the public API with inputs copied in from pinned
    # host memory every step and the loss read back
    e2e = None
    if not args.no_e2e and C > 1:
        e2e = {"value": None, "unit": "TFLOP/s", "skipped": "multi-cycle workload: its "
               f"{C} cycles' logits alone are {sum(g_.logits.numel() for g_ in gins) * 2 / 1e9:.0f} "
               "GB of pinned host memory per input set"}
    if not args.no_e2e and C == 1 and not args.batched:
        gin, logp_old, off = gins[0], logp_olds[0], offs[0]
        branch_list = [branches[0, i] for i in range(G)]
        host = {}

        def pin(t):
            h = torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
            h.copy_(t)
            return h

        host["k"], host["v"] = pin(pr.k), pin(pr.v)
        host["br"] = [(pin(b.q), pin(b.k), pin(b.v), pin(b.d_o)) for b in branch_list]
        host["logits"] = pin(gin.logits)
        host["targets"], host["logp_old"] = pin(gin.targets), pin(logp_old)
        host["rewards"], host["lens"] = pin(gin.rewards), pin(gin.resp_lens)
        loss_h = torch.empty(1, dtype=torch.float32, pin_memory=True)
        h2d = sum(t.numel() * t.element_size() for t in
                  [host["k"], host["v"], host["logits"], host["targets"], host["logp_old"],
                   host["rewards"], host["lens"]] + [x for b in host["br"] for x in b])
        d2h = 4

        # Inputs go through two sets of device buffers: step s + 1's inputs are copied
        # into one set while step s computes on the other (a set is refilled only after
        # the step that read it has finished).  Every step's inputs are copied inside the
        # timed region; only the first step's copies have no earlier step to hide behind.
        # Within a set the copies run on two copy streams (prompt K on one and V on the
        # other in page-aligned chunks, then each member's tensors), each piece marked by
        # an event; the compute stream waits for exactly the pieces its next call reads.
        copy_streams = [torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)]
        n_chunks = 8
        P = pr.k.shape[0]
        unit = w.page_size
        bounds = [(P // unit) * c // n_chunks * unit for c in range(n_chunks)] + [P]

        class InputSet:
            def __init__(self, k, v, br, logits, targets, lpo, rewards, lens):
                self.k, self.v, self.br = k, v, br
                self.logits, self.targets, self.logp_old = logits, targets, lpo
                self.rewards, self.lens = rewards, lens

        sets = [InputSet(pr.k, pr.v, [(b.q, b.k, b.v, b.d_o) for b in branch_list], gin.logits,
                         gin.targets, logp_old, gin.rewards, gin.resp_lens)]
        el = torch.empty_like
        sets.append(InputSet(el(pr.k), el(pr.v), [tuple(el(x) for x in t) for t in sets[0].br],
                             el(gin.logits), el(gin.targets), el(logp_old), el(gin.rewards),
                             el(gin.resp_lens)))

        def mark(st):
            e = torch.cuda.Event()
            e.record(st)
            return e

        def issue_copies(dst, after):
            """Enqueue one step's host->device copies into set dst once `after` has
            happened; returns the events of its pieces."""
            for cs in copy_streams:
                cs.wait_event(after)
            cs0, cs1 = copy_streams
            with torch.cuda.stream(cs0):
                dst.rewards.copy_(host["rewards"], non_blocking=True)
                dst.lens.copy_(host["lens"], non_blocking=True)
            kv_ev = []
            for c in range(n_chunks):
                s, e = bounds[c], bounds[c + 1]
                with torch.cuda.stream(cs0):
                    dst.k[s:e].copy_(host["k"][s:e], non_blocking=True)
                with torch.cuda.stream(cs1):
                    dst.v[s:e].copy_(host["v"][s:e], non_blocking=True)
                kv_ev.append((mark(cs0), mark(cs1)))
            br_ev, lg_ev = [], []
            for i, (b, hb) in enumerate(zip(dst.br, host["br"])):
                with torch.cuda.stream(copy_streams[i % 2]):
                    for d_, s_ in zip(b, hb):
                        d_.copy_(s_, non_blocking=True)
                br_ev.append(mark(copy_streams[i % 2]))
                # the member's logits rows, half on each copy stream
                s, e = off[i], off[i + 1]
                mid = (s + e) // 2
                evs = []
                for cs, (a0, a1) in zip(copy_streams, ((s, mid), (mid, e))):
                    with torch.cuda.stream(cs):
                        dst.logits[a0:a1].copy_(host["logits"][a0:a1], non_blocking=True)
                        dst.targets[a0:a1].copy_(host["targets"][a0:a1], non_blocking=True)
                        dst.logp_old[a0:a1].copy_(host["logp_old"][a0:a1], non_blocking=True)
                    evs.append(mark(cs))
                lg_ev.append(evs)
            return kv_ev, br_ev, lg_ev

        def compute(src, evs):
            """One step on input set src once its pieces have landed; returns the event
            after which src may be refilled."""
            kv_ev, br_ev, lg_ev = evs
            for c in range(n_chunks):
                stream.wait_event(kv_ev[c][0])
                stream.wait_event(kv_ev[c][1])
                s, e = bounds[c], bounds[c + 1]
                cache.capture(src.k[s:e], src.v[s:e], s, stream)
            for i in range(G):
                # the forward reads only the member's q / k / v / dO (and the captured
                # prompt); the loss also waits for its logits rows, whose events follow
                # the rewards and lengths copied first on copy stream 0
                stream.wait_event(br_ev[i])
                member(0, i, before_loss=lambda i=i: [stream.wait_event(e) for e in lg_ev[i]],
                       inp=src)
            loss_h.copy_(loss, non_blocking=True)
            return mark(stream)

        def e2e_steps(n):
            free = [mark(stream), mark(stream)]  # when each set may be refilled
            evs = issue_copies(sets[0], free[0])
            for st in range(n):
                nxt = issue_copies(sets[(st + 1) % 2], free[(st + 1) % 2]) if st + 1 < n else None
                free[st % 2] = compute(sets[st % 2], evs)
                evs = nxt

        e2e_steps(1)
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        a = ev()
        e2e_steps(args.steps)
        b = ev()
        torch.cuda.synchronize()
        e_ms = max_over_ranks(a.elapsed_time(b), world, dev)
        e2e = {"value": whole_job_rate(step_flops, world, e_ms / K) / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": d2h,
               "ms_per_step": e_ms / K}

    # ---- pre-step scoring (outside the step): log-softmax gather of one member's tokens
    # with the KL estimate against reference log-probabilities; HBM-bound, V*b read per
    # token
    gin, off = gins[0], offs[0]
    s0, s1 = off[0], off[1]
    ref_lp = logp_olds[0][s0:s1]
    api.grpo_logp(gin.logits[s0:s1], gin.targets[s0:s1], ref_lp, stream=stream)
    torch.cuda.synchronize()
    # hold the stream for a few ms so that all K calls are queued before the first
    # starts: the events then time the kernels, not the host's call overhead
    torch.cuda._sleep(20_000_000)
    ea, eb = ev(), None
    for _ in range(K):
        api.grpo_logp(gin.logits[s0:s1], gin.targets[s0:s1], ref_lp, stream=stream)
    eb = ev()
    torch.cuda.synchronize()
    sc_ms = ea.elapsed_time(eb) / K
    tok_bytes = w.vocab * gin.logits.element_size()
    comps["grpo_logp_tokens_per_s"] = (s1 - s0) / (sc_ms * 1e-3)
    comps["grpo_logp_hbm_frac"] = (s1 - s0) * tok_bytes / (sc_ms * 1e-3) / 1e9 / pk.get(
        "hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])

    # ---- pre-step scoring, attention half: the forward of G short responses over the
    # captured prompt, one batched launch (the members' tokens packed into shared tiles)
    # against G one-member launches.  Short responses are HBM-bound one by one; batched,
    # each prompt K/V tile serves every member's rows of its KV head at once.
    for Rsc in (2, 16):
        sbr = [syn.make_branch(Rsc, w.hq, w.hkv, D, seed + 101 + i, dev) for i in range(w.G)]
        sq = torch.stack([b.q for b in sbr]).contiguous()
        sk = torch.stack([b.k for b in sbr]).contiguous()
        sv = torch.stack([b.v for b in sbr]).contiguous()
        so = torch.empty_like(sq)
        slse = torch.empty(sq.shape[:3], dtype=torch.float32, device=dev)

        def scoring_batched():
            api.replay_fwd_members(cache, sq, sk, sv, scale, w.num_splits, o=so, lse=slse,
                                   stream=stream)

        def scoring_serial():
            for i in range(w.G):
                api.replay_fwd(cache, sq[i], sk[i], sv[i], scale, w.num_splits, o=so[i],
                               lse=slse[i], stream=stream)

        for name, fn in (("batched", scoring_batched), ("serial", scoring_serial)):
            fn()
            torch.cuda.synchronize()
            torch.cuda._sleep(20_000_000)  # queue the K calls before the first starts
            ea = ev()
            for _ in range(K):
                fn()
            eb = ev()
            torch.cuda.synchronize()
            comps[f"prestep_fwd_{w.G}x{Rsc}_{name}_ms"] = ea.elapsed_time(eb) / K
        comps[f"prestep_fwd_{w.G}x{Rsc}_batched_kv_hbm_frac"] = kv_bytes / (
            comps[f"prestep_fwd_{w.G}x{Rsc}_batched_ms"] * 1e-3) / 1e9 / pk.get(
            "hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])

    # ---- CPU baseline: the oracle on a bounded sample of the same workload
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline_attention(cache, branches[0, 0], w, scale, budget_s=args.cpu_budget)

    rl = sorted(Rs.values())
    if C == 1 and rl[0] == rl[-1]:
        replay_desc = f"G={G} serial replays R={rl[0]}"
    else:
        how = ("each cycle's members in one ragged forward, one loss and one ragged backward "
               "call" if args.batched else "serial replays")
        replay_desc = (f"one capture, {C} cycles x G={G} ({n_rep} replays), {how}, ragged R "
                       f"in [{rl[0]}, {rl[-1]}] (mean {sum(rl) / len(rl):.0f})")
    out = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded; shapes of the pages' "
                + ("4,456,448-position prefix-reuse runs)" if C > 1 else "2,097,152-position runs)"),
        "config": {"workload": f"{args.workload}: P={w.P:,} prompt positions, Hq={w.hq}, "
                               f"Hkv={w.hkv}, d=128, {w.page_size}-token pages shuffled, "
                               f"{w.num_splits} KV splits; " + replay_desc + "; GRPO "
                               f"V={w.vocab:,} {w.logits_dtype} logits",
                   "members": n_rep,
                   "l2": f"inputs larger than L2 (prompt KV {prompt_kv_bytes(w.P, w.hkv)/1e9:.2f} "
                         f"GB per pass)"},
        "components": comps, "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
        "gpu_launches": launches * K,
        "clocks": clk.summary(),
    }
    if rank == 0:
        print(json.dumps(out), flush=True)


def cpu_baseline_attention(cache, br, w, scale, budget_s: float):
    """Time the fp64 oracle on sampled rows of the same workload (forward + dQ of each
    sampled row over the full prompt) and express it in the metric's unit."""
    import numpy as np

    import oracle
    from response_replay_gb300 import synthetic as syn

    pb = oracle.AttnProblem(syn.bf16_bits(cache.k_pool), syn.bf16_bits(cache.v_pool),
                            cache.page_table.cpu().numpy(), w.P, syn.bf16_bits(br.q),
                            syn.bf16_bits(br.k), syn.bf16_bits(br.v), scale, w.num_splits)
    d_o = syn.bf16_bits(br.d_o)
    rng = np.random.default_rng(0)
    R = br.q.shape[0]
    threads = oracle.num_threads()

    def run(n):
        ts = rng.integers(0, R, n).astype(np.int32)
        hs = rng.integers(0, w.hq, n).astype(np.int32)
        t0 = time.perf_counter()
        oracle.attn_fwd_rows(pb, ts, hs)
        oracle.attn_bwd_dq_rows(pb, d_o, ts, hs)
        dt = time.perf_counter() - t0
        fl = sum(4.0 * D * (w.P + t + 1) + 6.0 * D * (w.P + t + 1) for t in ts)
        return fl, dt

    n = max(threads, 1)
    fl, dt = run(n)
    if dt < budget_s / 4:
        n2 = int(n * min(64, max(1.0, (budget_s * 0.75) / max(dt, 1e-3))))
        n2 = max(n, (n2 // max(threads, 1)) * max(threads, 1))
        fl, dt = run(n2)
        n = n2
    return {"value": fl / dt / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
            "cpu": cpu_model(),
            "sample": f"{n} random (t, h) rows of one member: fp64 forward + dQ over all "
                      f"{w.P} prompt keys and the causal response keys; {dt:.1f} s"}


# ------------------------------------------------------------------ short-response sweep

def run_short_sweep(args, local_rank: int):
    """Supplementary, labelled sweep (not the headline line): one replay of short
    responses R over the 2,097,152-position prompt, where the forward streams the prompt
    K/V once per KV head and HBM bandwidth, not the tensor cores, is the bound.  One JSON
    line per R: forward and backward times, prompt-KV GB/s of each pass against the
    measured copy bandwidth, the FLOP rate, and the batched forward of all G members'
    responses of R tokens (pre-step scoring) in one launch."""
    import torch

    from response_replay_gb300 import synthetic as syn
    from response_replay_gb300 import torch_api as api

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    w = syn.WORKLOADS[WORKLOAD]
    seed = syn.seed_of(WORKLOAD)
    scale = D ** -0.5
    pr = syn.make_prompt(w.P, w.hkv, D, w.page_size, seed, dev)
    cache = api.PagedKVCache(pr.num_pages, pr.page_table, w.page_size, w.hkv, w.P, device=dev)
    cache.capture(pr.k, pr.v)
    del pr
    pk, _ = peaks()
    hbm = pk.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
    kv_bytes = prompt_kv_bytes(w.P, w.hkv)
    stream = torch.cuda.current_stream()
    for R in [int(x) for x in args.sweep_short.split(",")]:
        br = syn.make_branch(R, w.hq, w.hkv, D, seed + 1, dev)
        o = torch.empty((R, w.hq, D), dtype=torch.bfloat16, device=dev)
        lse = torch.empty((R, w.hq), dtype=torch.float32, device=dev)
        dq = torch.empty((R, w.hq, D), dtype=torch.float32, device=dev)
        dk = torch.empty((R, w.hkv, D), dtype=torch.float32, device=dev)
        dv = torch.empty((R, w.hkv, D), dtype=torch.float32, device=dev)

        def fwd():
            api.replay_fwd(cache, br.q, br.k, br.v, scale, w.num_splits, o=o, lse=lse, stream=stream)

        def bwd():
            api.replay_bwd(cache, br.q, br.k, br.v, o, lse, br.d_o, scale, w.num_splits, dq=dq,
                           dk=dk, dv=dv, stream=stream)

        def timed(fn):
            for _ in range(args.warmup):
                fn()
            torch.cuda.synchronize()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for _ in range(args.steps):
                fn()
            b.record(stream)
            torch.cuda.synchronize()
            return a.elapsed_time(b) / args.steps

        # pre-step scoring: the forward of all G members' responses of R tokens in one launch
        G = w.G
        mq = torch.stack([syn.make_branch(R, w.hq, w.hkv, D, seed + 11 + i, dev).q
                          for i in range(G)]).contiguous()
        mk = br.k.unsqueeze(0).repeat(G, 1, 1, 1).contiguous()
        mv = br.v.unsqueeze(0).repeat(G, 1, 1, 1).contiguous()
        mo = torch.empty_like(mq)
        mlse = torch.empty(mq.shape[:3], dtype=torch.float32, device=dev)

        def fwd_members():
            api.replay_fwd_members(cache, mq, mk, mv, scale, w.num_splits, o=mo, lse=mlse,
                                   stream=stream)

        f_ms, b_ms = timed(fwd), timed(bwd)
        m_ms = timed(fwd_members)
        f_fl, b_fl = attn_flops(w.P, R, w.hq)
        print(json.dumps({
            "sweep": "short responses over the 2,097,152-position prompt (supplementary)",
            "R": R, "config": {"workload": f"P={w.P:,}, Hq={w.hq}, Hkv={w.hkv}, d=128, "
                                           f"{w.page_size}-token pages, {w.num_splits} splits"},
            "fwd_ms": f_ms, "bwd_ms": b_ms,
            "fwd_kv_gbs": kv_bytes / (f_ms * 1e-3) / 1e9,
            "bwd_kv_gbs": kv_bytes / (b_ms * 1e-3) / 1e9,
            "fwd_frac_of_hbm": kv_bytes / (f_ms * 1e-3) / 1e9 / hbm,
            "bwd_frac_of_hbm": kv_bytes / (b_ms * 1e-3) / 1e9 / hbm,
            "fwd_tflops": f_fl / (f_ms * 1e-3) / 1e12, "bwd_tflops": b_fl / (b_ms * 1e-3) / 1e12,
            "members": G, "members_fwd_ms": m_ms,
            "members_fwd_frac_of_hbm": kv_bytes / (m_ms * 1e-3) / 1e9 / hbm,
            "members_fwd_speedup_over_calls": G * f_ms / m_ms,
            "hbm_peak_gbs": hbm, "steps": args.steps, "warmup": args.warmup,
        }), flush=True)


# ------------------------------------------------------------------ host-resident pages

def run_host_sweep(args, local_rank: int):
    """Supplementary, labelled lines (not the headline): the 2,097,152-position prompt's
    pages held in pinned host memory (Grace memory, read over NVLink-C2C by the kernels
    themselves) against the same pages in HBM.  One JSON line per R with forward and
    backward times in both placements, the prompt-KV GB/s of each pass, and the measured
    host-to-device copy bandwidth (a 4 GiB copy from pinned memory) for comparison."""
    import torch

    from response_replay_gb300 import synthetic as syn
    from response_replay_gb300 import torch_api as api

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    w = syn.WORKLOADS[WORKLOAD]
    seed = syn.seed_of(WORKLOAD)
    scale = D ** -0.5
    pr = syn.make_prompt(w.P, w.hkv, D, w.page_size, seed, dev)
    dcache = api.PagedKVCache(pr.num_pages, pr.page_table, w.page_size, w.hkv, w.P, device=dev)
    dcache.capture(pr.k, pr.v)
    hcache = api.PagedKVCache(pr.num_pages, pr.page_table, w.page_size, w.hkv, w.P,
                              host_pools=True)
    hcache.capture(pr.k, pr.v)  # written over the link by the capture kernel
    del pr
    stream = torch.cuda.current_stream()

    def timed(fn, steps):
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(steps):
            fn()
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / steps

    # copy-engine bandwidth from pinned host memory, for scale
    src = torch.empty(1 << 31, dtype=torch.int16, pin_memory=True)
    dst = torch.empty(1 << 31, dtype=torch.int16, device=dev)
    copy_ms = timed(lambda: dst.copy_(src, non_blocking=True), max(args.steps, 3))
    h2d_gbs = src.numel() * 2 / (copy_ms * 1e-3) / 1e9
    del src, dst
    kv_bytes = prompt_kv_bytes(w.P, w.hkv)
    for R in [int(x) for x in args.sweep_host.split(",")]:
        br = syn.make_branch(R, w.hq, w.hkv, D, seed + 1, dev)
        o = torch.empty((R, w.hq, D), dtype=torch.bfloat16, device=dev)
        lse = torch.empty((R, w.hq), dtype=torch.float32, device=dev)
        dq = torch.empty((R, w.hq, D), dtype=torch.float32, device=dev)
        dk = torch.empty((R, w.hkv, D), dtype=torch.float32, device=dev)
        dv = torch.empty((R, w.hkv, D), dtype=torch.float32, device=dev)
        res = {}
        for name, cache in (("hbm", dcache), ("host", hcache)):
            def fwd():
                api.replay_fwd(cache, br.q, br.k, br.v, scale, w.num_splits, o=o, lse=lse,
                               stream=stream)

            def bwd():
                api.replay_bwd(cache, br.q, br.k, br.v, o, lse, br.d_o, scale, w.num_splits,
                               dq=dq, dk=dk, dv=dv, stream=stream)

            steps = args.steps if R < 1024 else max(1, args.steps // 5)
            res[name] = (timed(fwd, steps), timed(bwd, steps))
        f_fl, b_fl = attn_flops(w.P, R, w.hq)
        (fh, bh), (fd, bd) = res["host"], res["hbm"]
        print(json.dumps({
            "sweep": "prompt pages in host (Grace) memory vs HBM, 2,097,152 positions "
                     "(supplementary)",
            "R": R, "config": {"workload": f"P={w.P:,}, Hq={w.hq}, Hkv={w.hkv}, d=128, "
                                           f"{w.page_size}-token pages, {w.num_splits} splits"},
            "host_fwd_ms": fh, "host_bwd_ms": bh, "hbm_fwd_ms": fd, "hbm_bwd_ms": bd,
            "host_fwd_kv_gbs": kv_bytes / (fh * 1e-3) / 1e9,
            "host_bwd_kv_gbs": kv_bytes / (bh * 1e-3) / 1e9,
            "host_fwd_tflops": f_fl / (fh * 1e-3) / 1e12,
            "host_bwd_tflops": b_fl / (bh * 1e-3) / 1e12,
            "h2d_copy_gbs": h2d_gbs, "steps": args.steps, "warmup": args.warmup,
        }), flush=True)


# ------------------------------------------------------------------ latent (MLA) replay

MLA_ROW, MLA_DC = 576, 512


def mla_flops(P: int, R: int, H: int) -> tuple[float, float]:
    """(algorithmic, executed) FLOPs of one latent replay forward: per (query row, visible
    key) 2 x 576 for the score and 2 x 512 for the output; the kernel computes every
    score twice (once per half of the output columns)."""
    pairs = R * H * (P + (R + 1) / 2)
    return pairs * 2 * (MLA_ROW + MLA_DC), pairs * 2 * (2 * MLA_ROW + MLA_DC)


def mla_bwd_flops(P: int, R: int, H: int) -> tuple[float, float]:
    """(algorithmic, executed) FLOPs of one latent replay backward.  Algorithmic: per
    (query row, visible key) 2 x (576 score + 512 dP + 576 dq); per (query row, response
    key j <= t) 2 x (512 + 576) for the response row's gradient.  Executed on the tensor
    pipe: the dq kernel's 128-lane products hold 64 query rows, so per (row, key) they cost
    2 x 2 x (576 + 320 + 256) (S|dP, and the dq products on all 128 lanes); the
    response-row kernel walks 128-key tiles over 16-row blocks from each tile's first
    token, 2 x (2 x 2 x 576 + 576 + 512) per walked (row, key)."""
    pairs = R * H * (P + (R + 1) / 2)
    resp_pairs = R * H * (R + 1) / 2
    alg = pairs * 2 * (2 * MLA_ROW + MLA_DC) + resp_pairs * 2 * (MLA_ROW + MLA_DC)
    rb_hi = -(-R * H // 16)
    walked = sum(128 * 16 * (rb_hi - 8 * kt * H) for kt in range(-(-R // 128)))
    exe = pairs * 2 * 2 * (MLA_ROW + 320 + 256) + walked * 2 * (4 * MLA_ROW + MLA_ROW + MLA_DC)
    return alg, exe


def run_mla_sweep(args, local_rank: int):
    """Supplementary, labelled lines (not the headline): the latent (MLA-style) replay
    forward over a prompt of P (default 2,097,152) 576-value latent rows (256-row pages,
    256 splits), H query heads, with the pool in HBM and (for short responses) in pinned host
    memory read over the host link; one JSON line per R."""
    import torch

    from response_replay_gb300 import synthetic as syn
    from response_replay_gb300 import torch_api as api

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    P, ps, splits, H = args.mla_p, 256, 256, args.mla_heads
    scale = 192 ** -0.5
    pr = syn.make_latent_prompt(max(P, 1), ps, 4242, dev)  # P = 0: causal response only
    pt = pr.page_table if P > 0 else pr.page_table[:0]
    dcache = api.LatentCache(pr.num_pages, pt, ps, P, device=dev)
    if P > 0:
        dcache.capture(pr.lat)
    hcache = None
    if args.mla_host_max_r > 0 and P > 0:
        hcache = api.LatentCache(pr.num_pages, pt, ps, P, host_pool=True)
        hcache.capture(pr.lat)  # written over the link by the capture kernel
    del pr
    stream = torch.cuda.current_stream()

    def timed(fn, steps):
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(steps):
            fn()
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / steps

    h2d_gbs = None
    Rs = [int(x) for x in args.sweep_mla.split(",")]
    if any(R <= args.mla_host_max_r for R in Rs):  # copy-engine rate from pinned memory
        src = torch.empty(1 << 31, dtype=torch.int16, pin_memory=True)
        dst = torch.empty(1 << 31, dtype=torch.int16, device=dev)
        copy_ms = timed(lambda: dst.copy_(src, non_blocking=True), max(args.steps, 3))
        h2d_gbs = src.numel() * 2 / (copy_ms * 1e-3) / 1e9
        del src, dst
    pk, pk_src = peaks()
    peak = pk.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
    lat_bytes = P * MLA_ROW * 2
    for R in Rs:
        br = syn.make_latent_branch(R, H, 4243, dev, sharp=True)
        o = torch.empty((R, H, MLA_DC), dtype=torch.bfloat16, device=dev)
        lse = torch.empty((R, H), dtype=torch.float32, device=dev)
        line = {"sweep": f"latent (MLA-style) replay forward, {P:,} positions (supplementary)",
                "R": R, "config": {"workload": f"P={P:,} latent rows of {MLA_ROW} bf16 "
                                               f"({MLA_DC} latent + 64 rotary), H={H}, "
                                               f"{ps}-row pages, {splits} splits"}}
        for name, cache in (("hbm", dcache), ("host", hcache)):
            if name == "host" and (cache is None or R > args.mla_host_max_r):
                continue
            ms = timed(lambda: api.mla_replay_fwd(cache, br.q, br.lat, scale, splits, o=o,
                                                  lse=lse, stream=stream), args.steps)
            alg, exe = mla_flops(P, R, H)
            line.update({f"{name}_fwd_ms": ms,
                         f"{name}_tflops": alg / (ms * 1e-3) / 1e12,
                         f"{name}_executed_tflops": exe / (ms * 1e-3) / 1e12,
                         f"{name}_latent_gbs": lat_bytes / (ms * 1e-3) / 1e9})
        if args.mla_bwd:
            d_o = br.d_o
            dq = torch.empty((R, H, MLA_ROW), dtype=torch.float32, device=dev)
            dl = torch.empty((R, MLA_ROW), dtype=torch.float32, device=dev)
            api.mla_replay_fwd(dcache, br.q, br.lat, scale, splits, o=o, lse=lse, stream=stream)
            alg, exe = mla_bwd_flops(P, R, H)
            for name, cache in (("hbm", dcache), ("host", hcache)):
                if name == "host" and (cache is None or R > args.mla_host_max_r):
                    continue
                ms = timed(lambda: api.mla_replay_bwd(cache, br.q, br.lat, o, lse, d_o, scale,
                                                      splits, dq=dq, dlat=dl, stream=stream),
                           args.steps)
                line.update({f"{name}_bwd_ms": ms,
                             f"{name}_bwd_tflops": alg / (ms * 1e-3) / 1e12,
                             f"{name}_bwd_executed_tflops": exe / (ms * 1e-3) / 1e12,
                             f"{name}_bwd_latent_gbs": lat_bytes / (ms * 1e-3) / 1e9})
            line["bwd_executed_frac_of_bf16_burst"] = line["hbm_bwd_executed_tflops"] / peak
        line.update({"executed_frac_of_bf16_burst": line["hbm_executed_tflops"] / peak,
                     "peak": f"{pk_src} bf16 burst {peak}", "h2d_copy_gbs": h2d_gbs,
                     "steps": args.steps, "warmup": args.warmup})
        print(json.dumps(line), flush=True)


def run_mla_layers_sweep(args, local_rank: int):
    """Supplementary, labelled line (not the headline): one response of R tokens replayed
    (forward, and with --mla-bwd the backward in reverse layer order) through L
    latent-attention layers over a 2,097,152-row latent prompt, with
    every layer's pages (a) in GPU memory and (b) in pinned host memory, streamed into a
    two-slot GPU page cache one layer ahead (each layer's copy overlapping the previous
    layer's replay)."""
    import torch

    from response_replay_gb300 import layers as Lm
    from response_replay_gb300 import synthetic as syn
    from response_replay_gb300 import torch_api as api

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    P, ps, splits, H, nl, R = args.mla_p, 256, 256, args.mla_heads, args.sweep_mla_layers, \
        args.mla_layers_r
    scale = 192 ** -0.5
    pr0 = syn.make_latent_prompt(P, ps, 5100, dev)
    st = Lm.StreamedLatentLayers(nl, pr0.num_pages, pr0.page_table, ps, P, device=dev)
    res, brs = [], []
    for l in range(nl):
        lat = syn.make_latent_prompt(P, ps, 5100 + l, dev).lat
        c = api.LatentCache(pr0.num_pages, pr0.page_table, ps, P, device=dev)
        c.capture(lat)
        st.capture(l, lat)
        res.append(c)
        del lat
        brs.append(syn.make_latent_branch(R, H, 5200 + l, dev, sharp=True))
    stream = torch.cuda.current_stream()
    os_ = [torch.empty((R, H, MLA_DC), dtype=torch.bfloat16, device=dev) for _ in range(nl)]
    lses = [torch.empty((R, H), dtype=torch.float32, device=dev) for _ in range(nl)]
    dq = torch.empty((R, H, MLA_ROW), dtype=torch.float32, device=dev)
    dl = torch.empty((R, MLA_ROW), dtype=torch.float32, device=dev)

    def bwd(c, l):
        api.mla_replay_bwd(c, brs[l].q, brs[l].lat, os_[l], lses[l], brs[l].d_o, scale, splits,
                           dq=dq, dlat=dl, stream=stream)

    def resident():
        for l in range(nl):
            api.mla_replay_fwd(res[l], brs[l].q, brs[l].lat, scale, splits, o=os_[l],
                               lse=lses[l], stream=stream)
        if args.mla_bwd:
            for l in reversed(range(nl)):
                bwd(res[l], l)

    def streamed():
        st.prefetch(0)
        for l in range(nl):
            c = st.cache(l)
            if l + 1 < nl:
                st.prefetch(l + 1)
            api.mla_replay_fwd(c, brs[l].q, brs[l].lat, scale, splits, o=os_[l], lse=lses[l],
                               stream=stream)
            st.release(l)
        if args.mla_bwd:  # backward in reverse layer order through the same two slots
            st.prefetch(nl - 1)
            for l in reversed(range(nl)):
                c = st.cache(l)
                if l > 0:
                    st.prefetch(l - 1)
                bwd(c, l)
                st.release(l)

    def timed(fn):
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(args.steps):
            fn()
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / args.steps

    ms_res, ms_str = timed(resident), timed(streamed)
    # the copy alone, from pinned host memory into a slot
    cp = timed(lambda: st.slots[0].pool.copy_(st.host[0].pool, non_blocking=True))
    alg, _ = mla_flops(P, R, H)
    if args.mla_bwd:
        alg += mla_bwd_flops(P, R, H)[0]
    print(json.dumps({
        "sweep": f"latent replay through {nl} layers ({'forward, then backward in reverse' if args.mla_bwd else 'forward'}), "
                 "pages streamed from host memory vs held in HBM (supplementary)",
        "config": {"workload": f"P={P:,} latent rows of {MLA_ROW} bf16, H={H}, R={R}, "
                               f"{ps}-row pages, {splits} splits, {nl} layers"},
        "hbm_ms": ms_res, "streamed_ms": ms_str, "slowdown": ms_str / ms_res,
        "hbm_tflops": nl * alg / (ms_res * 1e-3) / 1e12,
        "streamed_tflops": nl * alg / (ms_str * 1e-3) / 1e12,
        "layer_copy_ms": cp, "layer_bytes": st.bytes_per_layer,
        "layer_copy_gbs": st.bytes_per_layer / (cp * 1e-3) / 1e9,
        "steps": args.steps, "warmup": args.warmup,
    }), flush=True)


# ------------------------------------------------------------------ streamed layers

def run_layers_sweep(args, local_rank: int):
    """Supplementary, labelled line (not the headline): one response of R = 4,096 tokens
    replayed through L layers over the 2,097,152-position prompt, forward in layer order
    and backward last layer first, with the layers' prompt pages (a) all in GPU memory and
    (b) in pinned host memory, streamed into a two-slot GPU page cache one layer ahead of
    use (each layer's copy overlapping the previous layer's replay)."""
    import torch

    from response_replay_gb300 import layers as L
    from response_replay_gb300 import synthetic as syn
    from response_replay_gb300 import torch_api as api

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    w = syn.WORKLOADS[WORKLOAD]
    seed = syn.seed_of(WORKLOAD)
    scale = D ** -0.5
    nl = int(args.sweep_layers)
    R = w.R[0]
    pr = syn.make_prompt(w.P, w.hkv, D, w.page_size, seed, dev)
    res = L.LayeredKVCache(nl, pr.num_pages, pr.page_table, w.page_size, w.hkv, w.P, device=dev)
    st = L.StreamedLayers(nl, pr.num_pages, pr.page_table, w.page_size, w.hkv, w.P, device=dev)
    for l in range(nl):  # the same prompt K/V in every layer (the values do not matter here)
        res.capture(l, pr.k, pr.v)
        st.capture(l, pr.k, pr.v)
    del pr
    br = syn.make_branch(R, w.hq, w.hkv, D, seed + 1, dev)
    o = [torch.empty((R, w.hq, D), dtype=torch.bfloat16, device=dev) for _ in range(nl)]
    lse = [torch.empty((R, w.hq), dtype=torch.float32, device=dev) for _ in range(nl)]
    dq = torch.empty((R, w.hq, D), dtype=torch.float32, device=dev)
    dk = torch.empty((R, w.hkv, D), dtype=torch.float32, device=dev)
    dv = torch.empty((R, w.hkv, D), dtype=torch.float32, device=dev)

    def step(get, pre, rel):
        for l in range(nl):
            c = get(l)
            if l + 1 < nl:
                pre(l + 1)
            api.replay_fwd(c, br.q, br.k, br.v, scale, w.num_splits, o=o[l], lse=lse[l])
            rel(l)
        pre(nl - 1)
        for l in reversed(range(nl)):
            c = get(l)
            if l > 0:
                pre(l - 1)
            api.replay_bwd(c, br.q, br.k, br.v, o[l], lse[l], br.d_o, scale, w.num_splits,
                           dq=dq, dk=dk, dv=dv)
            rel(l)

    none = lambda l: None  # noqa: E731
    runs = {"hbm": lambda: step(lambda l: res[l], none, none),
            "streamed": lambda: step(st.cache, st.prefetch, st.release)}
    out = {}
    for name, fn in runs.items():
        for _ in range(max(args.warmup, 1)):
            fn()
        torch.cuda.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(args.steps):
            fn()
        b.record()
        torch.cuda.synchronize()
        out[name] = a.elapsed_time(b) / args.steps
    f_fl, b_fl = attn_flops(w.P, R, w.hq)
    print(json.dumps({
        "sweep": "layers' prompt pages streamed from host (Grace) memory vs held in HBM "
                 "(supplementary)",
        "layers": nl, "R": R,
        "config": {"workload": f"P={w.P:,}, Hq={w.hq}, Hkv={w.hkv}, d=128, {w.page_size}-token "
                               f"pages, {w.num_splits} splits; forward over the layers, then "
                               f"backward last layer first"},
        "hbm_ms": out["hbm"], "streamed_ms": out["streamed"],
        "streamed_over_hbm": out["streamed"] / out["hbm"],
        "streamed_tflops": nl * (f_fl + b_fl) / (out["streamed"] * 1e-3) / 1e12,
        "hbm_tflops": nl * (f_fl + b_fl) / (out["hbm"] * 1e-3) / 1e12,
        "copy_bytes_per_layer": st.bytes_per_layer,
        "host_pinned_bytes": nl * st.bytes_per_layer,
        "steps": args.steps, "warmup": args.warmup,
    }), flush=True)


# ------------------------------------------------------------------ self-attention sweep

def run_self_sweep(args, local_rank: int):
    """Supplementary, labelled lines (not the headline): replay with no prompt (P = 0),
    i.e. plain causal attention of a long response, where the response-key part of the
    backward (dK/dV over the causal triangle) is about half the backward's work.  One
    JSON line per R with forward and backward time and algorithmic TFLOP/s."""
    import torch

    from response_replay_gb300 import synthetic as syn
    from response_replay_gb300 import torch_api as api

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    hq, hkv, ps = 24, 4, 256
    pr = syn.make_prompt(1, hkv, D, ps, 11, dev)
    cache = api.PagedKVCache(pr.num_pages, pr.page_table[:0], ps, hkv, 0, device=dev)
    pk, _ = peaks()
    stream = torch.cuda.current_stream()
    scale = D ** -0.5
    for R in [int(x) for x in args.sweep_self.split(",")]:
        br = syn.make_branch(R, hq, hkv, D, 12, dev, sharp=True)
        o = torch.empty((R, hq, D), dtype=torch.bfloat16, device=dev)
        lse = torch.empty((R, hq), dtype=torch.float32, device=dev)
        dq = torch.empty((R, hq, D), dtype=torch.float32, device=dev)
        dk = torch.empty((R, hkv, D), dtype=torch.float32, device=dev)
        dv = torch.empty((R, hkv, D), dtype=torch.float32, device=dev)

        def fwd():
            api.replay_fwd(cache, br.q, br.k, br.v, scale, 1, o=o, lse=lse, stream=stream)

        def bwd():
            api.replay_bwd(cache, br.q, br.k, br.v, o, lse, br.d_o, scale, 1, dq=dq, dk=dk,
                           dv=dv, stream=stream)

        def timed(fn):
            for _ in range(args.warmup):
                fn()
            torch.cuda.synchronize()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for _ in range(args.steps):
                fn()
            b.record(stream)
            torch.cuda.synchronize()
            return a.elapsed_time(b) / args.steps

        f_ms, b_ms = timed(fwd), timed(bwd)
        f_fl, b_fl = attn_flops(0, R, hq)
        print(json.dumps({
            "sweep": "causal self-attention of one response, no prompt (supplementary)",
            "R": R, "config": {"workload": f"P=0, R={R}, Hq={hq}, Hkv={hkv}, d=128"},
            "fwd_ms": f_ms, "bwd_ms": b_ms,
            "fwd_tflops": f_fl / (f_ms * 1e-3) / 1e12, "bwd_tflops": b_fl / (b_ms * 1e-3) / 1e12,
            "bf16_tflops_burst": pk.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]),
            "steps": args.steps, "warmup": args.warmup,
        }), flush=True)


# ------------------------------------------------------------------ Gated-DeltaNet replay

GDN_HEADS = 32


def gdn_flops(R: int, H: int) -> tuple[float, float]:
    """fp32 FLOPs the chunked Gated-DeltaNet replay executes per layer (64-token chunks,
    128 x 128 state): per chunk and head the forward does K K^T, the triangular inverse,
    W and U0, the state hand-off, Q K^T, Q S^T and P U; the backward recomputes the
    forward's chunk algebra and runs the adjoint products and its own hand-off."""
    C, d = 64, 128
    nc = -(-R // C) * H
    fwd = 2.0 * (C * C * d + C ** 3 / 6 + 2 * C * C * d + 2 * C * d * d + C * C * d + C * d * d
                 + C * C * d)
    bwd_extra = 2.0 * (2 * C * C * d + 2 * C * d * d + C * C * d + 2 * C * d * d + C * C * d
                       + 2 * C * C * d + C * C * d + C * d * d + (C * d * d + C * C * d)
                       + (2 * C * d * d + 3 * C * C * d))
    rec = fwd - 2.0 * (C * C * d + C * d * d + C * C * d)   # the forward minus its output
    return nc * fwd, nc * (rec + bwd_extra)


def alu_peak_tflops(sm_mhz: float = 2070.0, sms: int = 152) -> float:
    """fp32 FMA peak of the CUDA cores: 128 FMA lanes per SM per clock, 2 FLOPs each."""
    return sms * 128 * 2 * sm_mhz * 1e6 / 1e12


def run_gdn_sweep(args, local_rank: int):
    """Supplementary, labelled lines: one Gated-DeltaNet layer replayed from a captured
    state (32 heads, 128 x 128 state), forward and backward times per response length,
    against the CUDA cores' fp32 peak (the chunk algebra runs in fp32 on them)."""
    import torch

    from response_replay_gb300 import synthetic as syn
    from response_replay_gb300 import torch_api as api

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()
    for R in [int(x) for x in args.sweep_gdn.split(",")]:
        inp = syn.make_gdn(R, GDN_HEADS, 21, dev)
        scale = D ** -0.5
        o = torch.empty_like(inp.q)
        grads = api.gdn_replay_bwd(inp.state0, inp.q, inp.k, inp.v, inp.g, inp.beta, inp.d_o,
                                   scale)

        def fwd():
            api.gdn_replay_fwd(inp.state0, inp.q, inp.k, inp.v, inp.g, inp.beta, scale, o=o,
                               stream=stream)

        def bwd():
            api.gdn_replay_bwd(inp.state0, inp.q, inp.k, inp.v, inp.g, inp.beta, inp.d_o, scale,
                               grads=grads, stream=stream)

        def timed(fn):
            for _ in range(args.warmup):
                fn()
            torch.cuda.synchronize()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for _ in range(args.steps):
                fn()
            b.record(stream)
            torch.cuda.synchronize()
            return a.elapsed_time(b) / args.steps

        f_ms, b_ms = timed(fwd), timed(bwd)
        f_fl, b_fl = gdn_flops(R, GDN_HEADS)
        peak = alu_peak_tflops()
        print(json.dumps({
            "sweep": "Gated-DeltaNet replay from a captured state, one layer (supplementary)",
            "R": R, "config": {"workload": f"R={R} response tokens, H={GDN_HEADS} heads, "
                                           "128 x 128 fp32 state, 64-token chunks"},
            "fwd_ms": f_ms, "bwd_ms": b_ms,
            "fwd_tflops": f_fl / (f_ms * 1e-3) / 1e12, "bwd_tflops": b_fl / (b_ms * 1e-3) / 1e12,
            "roofline": {"bound": "alu", "peak": peak, "unit": "TFLOP/s",
                         "peak_source": "152 SMs x 128 fp32 FMA lanes x 2 x 2.07 GHz",
                         "fwd_frac": f_fl / (f_ms * 1e-3) / 1e12 / peak,
                         "bwd_frac": b_fl / (b_ms * 1e-3) / 1e12 / peak},
            "steps": args.steps, "warmup": args.warmup,
        }), flush=True)


# ------------------------------------------------------------------ reference arm

def run_reference(args, rank: int, world: int):
    """The oracle as the reference arm: each step is a bounded sample of the same
    workload on the host cores (rank 0 only)."""
    if rank != 0:
        return
    import numpy as np

    import oracle
    from response_replay_gb300 import synthetic as syn

    w = syn.WORKLOADS[WORKLOAD]
    R = w.R[0]
    seed = syn.seed_of(WORKLOAD)
    rng = np.random.default_rng(seed)
    # host-side inputs of the same shapes (bf16 bit patterns of N(0,1)/sqrt(d) values)
    import torch
    pr = syn.make_prompt(w.P, w.hkv, D, w.page_size, seed, "cpu")
    pool_k = np.zeros((pr.num_pages, w.hkv, w.page_size, D), np.uint16)
    pool_v = np.zeros_like(pool_k)
    oracle.capture_kv(pool_k, pool_v, pr.page_table.numpy(), w.page_size, syn.bf16_bits(pr.k),
                      syn.bf16_bits(pr.v), 0)
    br = syn.make_branch(R, w.hq, w.hkv, D, seed + 1, "cpu")
    pb = oracle.AttnProblem(pool_k, pool_v, pr.page_table.numpy(), w.P, syn.bf16_bits(br.q),
                            syn.bf16_bits(br.k), syn.bf16_bits(br.v), D ** -0.5, w.num_splits)
    d_o = syn.bf16_bits(br.d_o)
    threads = oracle.num_threads()
    n = max(threads, 1) * args.ref_rows_per_core

    def sample_step():
        ts = rng.integers(0, R, n).astype(np.int32)
        hs = rng.integers(0, w.hq, n).astype(np.int32)
        oracle.attn_fwd_rows(pb, ts, hs)
        oracle.attn_bwd_dq_rows(pb, d_o, ts, hs)
        return sum(10.0 * D * (w.P + t + 1) for t in ts)

    for _ in range(args.warmup):
        sample_step()
    t0 = time.perf_counter()
    fl = 0.0
    for _ in range(args.steps):
        fl += sample_step()
    dt = time.perf_counter() - t0
    v = fl / dt / 1e12
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": v, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": "P=2,097,152, Hq=24, Hkv=4, d=128, R=4096 "
                                                    "(sampled rows)"},
        "cpu_baseline": {"value": v, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "cpu": cpu_model(),
                         "sample": f"{n} random (t, h) rows per step: fp64 forward + dQ over "
                                   f"the full prompt"},
        "e2e": {"value": v, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--members", type=int, default=None, help="replay fewer members (debug)")
    ap.add_argument("--batched", action="store_true",
                    help="replay each cycle's members in one ragged launch per pass")
    ap.add_argument("--workload", default=WORKLOAD,
                    help="p2m (default, the metric's configuration); smaller ones for profiling")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--ref-rows-per-core", type=int, default=2)
    ap.add_argument("--sweep-self", default=None,
                    help="comma-separated response lengths: supplementary no-prompt (causal "
                         "self-attention) lines instead of the headline step")
    ap.add_argument("--sweep-gdn", default=None,
                    help="comma-separated response lengths: supplementary Gated-DeltaNet "
                         "replay lines instead of the headline step")
    ap.add_argument("--sweep-layers", default=None,
                    help="number of layers: supplementary line with the layers' prompt pages "
                         "streamed from pinned host memory against held in HBM")
    ap.add_argument("--sweep-host", default=None,
                    help="comma-separated response lengths: supplementary lines with the "
                         "prompt pages in pinned host memory against HBM")
    ap.add_argument("--sweep-mla", default=None,
                    help="comma-separated response lengths: supplementary latent (MLA-style) "
                         "replay lines instead of the headline step")
    ap.add_argument("--mla-bwd", action="store_true",
                    help="with --sweep-mla / --sweep-mla-layers: also time the latent replay "
                         "backward")
    ap.add_argument("--sweep-mla-layers", type=int, default=0,
                    help="number of latent-attention layers: supplementary line with their "
                         "pages streamed from pinned host memory against held in HBM")
    ap.add_argument("--mla-layers-r", type=int, default=256)
    ap.add_argument("--mla-heads", type=int, default=64)
    ap.add_argument("--mla-p", type=int, default=2097152)
    ap.add_argument("--mla-host-max-r", type=int, default=16)
    ap.add_argument("--sweep-short", default=None,
                    help="comma-separated response lengths: supplementary short-R sweep "
                         "(one JSON line each) instead of the headline step")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        print("note: fewer than 3 warm-up steps", file=sys.stderr)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if args.sweep_short:
        if rank == 0:
            run_short_sweep(args, local_rank)
        return
    if args.sweep_self:
        if rank == 0:
            run_self_sweep(args, local_rank)
        return
    if args.sweep_host:
        if rank == 0:
            run_host_sweep(args, local_rank)
        return
    if args.sweep_layers:
        if rank == 0:
            run_layers_sweep(args, local_rank)
        return
    if args.sweep_mla:
        if rank == 0:
            run_mla_sweep(args, local_rank)
        return
    if args.sweep_mla_layers:
        if rank == 0:
            run_mla_layers_sweep(args, local_rank)
        return
    if args.sweep_gdn:
        if rank == 0:
            run_gdn_sweep(args, local_rank)
        return
    if world > 1:
        import torch
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl")
    try:
        run_ours(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
