"""CPU tests of the host side: the work schedule, the C ABI's exports and its argument
checks (no compute call needs a GPU: every rejected call returns before any launch)."""
import ctypes as C
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "response_replay_gb300", "csrc")


def test_schedule_invariants(tmp_path):
    exe = tmp_path / "sched_check"
    subprocess.run(["g++", "-std=c++17", "-O1", "-I", CSRC,
                    os.path.join(os.path.dirname(__file__), "sched_check.cpp"), "-o", str(exe)],
                   check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "schedules ok" in r.stdout


@pytest.fixture(scope="module")
def lib():
    from response_replay_gb300 import binding
    if not os.path.exists(binding.LIB_PATH):
        from response_replay_gb300 import build
        build.build()
    return binding.lib()


def test_library_exports_every_declared_symbol(lib):
    with open(os.path.join(ROOT, "include", "longstraw.h")) as f:
        hdr = f.read()
    declared = set(re.findall(r"\b(ls_[a-z_0-9]+)\s*\(", hdr))
    assert {"ls_capture_kv", "ls_replay_attn_fwd", "ls_replay_attn_bwd",
            "ls_grpo_loss_fwd_bwd"} <= declared
    for name in sorted(declared):
        assert hasattr(lib, name), f"{name} declared in include/longstraw.h but not exported"
    out = subprocess.run(["nm", "-D", "--defined-only",
                          os.path.join(ROOT, "response_replay_gb300", "_build",
                                       "liblongstraw.so")], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (ls_[a-z_0-9]+)\b", out))
    assert declared <= exported


def _cache(**kw):
    from response_replay_gb300.binding import ls_kv_cache
    d = dict(k_pool=256, v_pool=512, page_table=1024, num_pages=8, num_logical_pages=8,
             page_size=64, num_kv_heads=2, head_dim=128, num_tokens=512)
    d.update(kw)
    return ls_kv_cache(**d)


def test_argument_checks_reject_before_launch(lib):
    from response_replay_gb300 import binding as B
    sz = C.c_size_t(0)
    ok = _cache()
    cases = [
        (_cache(head_dim=64), B.LS_ERR_UNSUPPORTED),
        (_cache(page_size=48), B.LS_ERR_UNSUPPORTED),
        (_cache(page_size=8), B.LS_ERR_UNSUPPORTED),
        (_cache(num_tokens=513), B.LS_ERR_INVALID_ARG),
        (_cache(k_pool=260), B.LS_ERR_INVALID_ARG),
        (_cache(num_kv_heads=0), B.LS_ERR_INVALID_ARG),
    ]
    for c, want in cases:
        assert lib.ls_replay_attn_fwd_workspace(C.byref(c), 128, 8, 4, C.byref(sz)) == want
    # Hq not a multiple of the kv heads; zero splits
    assert lib.ls_replay_attn_fwd_workspace(C.byref(ok), 128, 7, 4, C.byref(sz)) == B.LS_ERR_INVALID_ARG
    assert lib.ls_replay_attn_fwd_workspace(C.byref(ok), 128, 8, 0, C.byref(sz)) == B.LS_ERR_INVALID_ARG
    # capture past the table
    assert lib.ls_capture_kv(C.byref(ok), 256, 256, 500, 13, None) == B.LS_ERR_INVALID_ARG
    # misaligned q
    assert lib.ls_replay_attn_fwd(C.byref(ok), 258, 256, 256, 16, 8, 0.1, 4, 256, 256, 256, 1 << 20,
                                  None) == B.LS_ERR_INVALID_ARG
    # GRPO: sample std with one member; member range outside the group; bad dtype
    assert lib.ls_grpo_loss_fwd_bwd(256, 0, 4, 16, 256, 256, 256, 256, 1, 0, 1, 0.2, 1e-6, 1, 0, 256,
                                    256, None, None, 256, 1 << 20, None) == B.LS_ERR_INVALID_ARG
    assert lib.ls_grpo_loss_fwd_bwd(256, 0, 4, 16, 256, 256, 256, 256, 2, 0, 3, 0.2, 1e-6, 1, 0, 256,
                                    256, None, None, 256, 1 << 20, None) == B.LS_ERR_INVALID_ARG
    assert lib.ls_grpo_loss_fwd_bwd(256, 7, 4, 16, 256, 256, 256, 256, 2, 0, 2, 0.2, 1e-6, 1, 0, 256,
                                    256, None, None, 256, 1 << 20, None) == B.LS_ERR_INVALID_ARG
    # GRPO workspace too small
    need = C.c_size_t(0)
    assert lib.ls_grpo_workspace(4, 2, C.byref(need)) == 0 and need.value > 0
    assert lib.ls_grpo_loss_fwd_bwd(256, 0, 4, 16, 256, 256, 256, 256, 2, 0, 2, 0.2, 1e-6, 1, 0, 256,
                                    256, None, None, 256, need.value - 1, None) == B.LS_ERR_WORKSPACE
    # batched forward: negative member count, members x R beyond 2^30, bad scale,
    # misaligned output; zero members or R = 0 is a no-op (no pointer is touched)
    assert lib.ls_replay_attn_fwd_members_workspace(C.byref(ok), 16, -1, 8, 4, C.byref(sz)) == \
        B.LS_ERR_INVALID_ARG
    assert lib.ls_replay_attn_fwd_members_workspace(C.byref(ok), 1 << 20, 2048, 8, 4,
                                                    C.byref(sz)) == B.LS_ERR_UNSUPPORTED
    assert lib.ls_replay_attn_fwd_members(C.byref(ok), 256, 256, 256, 16, -2, 8, 0.1, 4, 256, 256,
                                          256, 1 << 20, None) == B.LS_ERR_INVALID_ARG
    assert lib.ls_replay_attn_fwd_members(C.byref(ok), 256, 256, 256, 16, 3, 8, 0.0, 4, 256, 256,
                                          256, 1 << 20, None) == B.LS_ERR_INVALID_ARG
    assert lib.ls_replay_attn_fwd_members(C.byref(ok), 256, 256, 256, 16, 3, 8, 0.1, 4, 264, 256,
                                          256, 1 << 20, None) == B.LS_ERR_INVALID_ARG
    assert lib.ls_replay_attn_fwd_members(C.byref(ok), None, None, None, 16, 0, 8, 0.1, 4, None,
                                          None, None, 0, None) == B.LS_OK
    assert lib.ls_replay_attn_fwd_members(C.byref(ok), None, None, None, 0, 3, 8, 0.1, 4, None,
                                          None, None, 0, None) == B.LS_OK
    # pre-step scoring: bad dtype, KL output without reference log-probs, misaligned logits
    assert lib.ls_grpo_logp(256, 7, 4, 16, 256, None, 256, None, None, None) == \
        B.LS_ERR_INVALID_ARG
    assert lib.ls_grpo_logp(256, 0, 4, 16, 256, None, 256, None, 256, None) == \
        B.LS_ERR_INVALID_ARG
    assert lib.ls_grpo_logp(258, 0, 4, 16, 256, None, 256, None, None, None) == \
        B.LS_ERR_INVALID_ARG
    # per-token arrays need 4-byte alignment (member slices at any token offset), not less
    assert lib.ls_grpo_logp(256, 0, 4, 16, 258, None, 256, None, None, None) == \
        B.LS_ERR_INVALID_ARG
    assert lib.ls_grpo_loss_fwd_bwd(256, 0, 4, 16, 256, 262, 256, 256, 2, 0, 2, 0.2, 1e-6, 1, 0,
                                    256, 256, None, None, 256, 1 << 20, None) == \
        B.LS_ERR_INVALID_ARG
    assert B.status_string(B.LS_ERR_TIMEOUT)


def test_noalloc_scratch_holds_its_largest_call(lib):
    """The allocation-free GRPO entry point runs on a fixed 4.125 MiB array: the
    workspace of its largest accepted call (262,144 tokens, 1,024 members) must fit."""
    need = C.c_size_t(0)
    assert lib.ls_grpo_workspace(262144, 1024, C.byref(need)) == 0
    assert need.value <= (4 << 20) + (128 << 10)
