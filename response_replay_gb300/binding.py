"""ctypes binding of include/longstraw.h.

Argument marshalling only: every function below forwards to the C entry point of the
same name in liblongstraw.so, which validates the arguments and launches the CUDA
kernels.  Pointers are passed as integers (device addresses, e.g. tensor.data_ptr()),
streams as integers (torch.cuda.Stream.cuda_stream; 0 = legacy default stream).

There is no fallback: if the CUDA library has not been built, the first call raises.
"""
from __future__ import annotations

import ctypes as C
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "liblongstraw.so")

LS_OK, LS_ERR_INVALID_ARG, LS_ERR_UNSUPPORTED, LS_ERR_WORKSPACE, LS_ERR_CUDA, \
    LS_ERR_TIMEOUT, LS_ERR_DEVICE_CHECK = range(7)
LS_BF16, LS_FP32 = 0, 1

EXPORTED = (
    "ls_capture_kv", "ls_replay_attn_fwd_workspace", "ls_replay_attn_fwd",
    "ls_replay_attn_bwd_workspace", "ls_replay_attn_bwd", "ls_grpo_workspace",
    "ls_grpo_loss_fwd_bwd", "ls_validate_page_table", "ls_validate_page_table_workspace",
    "ls_last_device_error", "ls_status_string", "ls_kernel_launches",
    "ls_grpo_loss_fwd_bwd_noalloc", "ls_selftest_wait_timeout", "ls_grpo_logp",
    "ls_replay_attn_fwd_members_workspace", "ls_replay_attn_fwd_members",
    "ls_gdn_replay_fwd_workspace", "ls_gdn_replay_fwd", "ls_gdn_replay_bwd_workspace",
    "ls_gdn_replay_bwd", "ls_replay_attn_fwd_ragged_workspace", "ls_replay_attn_fwd_ragged",
    "ls_replay_attn_bwd_ragged_workspace", "ls_replay_attn_bwd_ragged",
    "ls_capture_latent", "ls_mla_replay_fwd_workspace", "ls_mla_replay_fwd",
    "ls_mla_replay_bwd_workspace", "ls_mla_replay_bwd",
)


class ls_kv_cache(C.Structure):
    _fields_ = [
        ("k_pool", C.c_void_p), ("v_pool", C.c_void_p), ("page_table", C.c_void_p),
        ("num_pages", C.c_int32), ("num_logical_pages", C.c_int32), ("page_size", C.c_int32),
        ("num_kv_heads", C.c_int32), ("head_dim", C.c_int32), ("num_tokens", C.c_int64),
    ]


class ls_latent_cache(C.Structure):
    _fields_ = [
        ("pool", C.c_void_p), ("page_table", C.c_void_p), ("num_pages", C.c_int32),
        ("num_logical_pages", C.c_int32), ("page_size", C.c_int32), ("num_tokens", C.c_int64),
    ]


class LongstrawError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn}: {status_string(status)} (status {status})")


_lib = None


def lib() -> C.CDLL:
    """The loaded CUDA library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build the CUDA library first "
                "(python -c 'import __graft_entry__ as g; g.build()')")
        l = C.CDLL(LIB_PATH)
        P, i32, i64, sz, f32 = C.c_void_p, C.c_int, C.c_int64, C.c_size_t, C.c_float
        cache = C.POINTER(ls_kv_cache)
        lcache = C.POINTER(ls_latent_cache)
        szp = C.POINTER(C.c_size_t)
        sig = {
            "ls_capture_latent": [lcache, P, i64, i64, P],
            "ls_mla_replay_fwd_workspace": [lcache, i32, i32, i32, szp],
            "ls_mla_replay_fwd": [lcache, P, P, i32, i32, f32, i32, P, P, P, sz, P],
            "ls_mla_replay_bwd_workspace": [lcache, i32, i32, i32, szp],
            "ls_mla_replay_bwd": [lcache, P, P, P, P, P, i32, i32, f32, i32, P, P, P, sz, P],
            "ls_capture_kv": [cache, P, P, i64, i64, P],
            "ls_replay_attn_fwd_workspace": [cache, i32, i32, i32, szp],
            "ls_replay_attn_fwd": [cache, P, P, P, i32, i32, f32, i32, P, P, P, sz, P],
            "ls_replay_attn_fwd_members_workspace": [cache, i32, i32, i32, i32, szp],
            "ls_replay_attn_fwd_members": [cache, P, P, P, i32, i32, i32, f32, i32, P, P, P, sz,
                                           P],
            "ls_replay_attn_bwd_workspace": [cache, i32, i32, i32, szp],
            "ls_replay_attn_bwd": [cache, P, P, P, P, P, P, i32, i32, f32, i32, i32, P, P, P, P,
                                   sz, P],
            "ls_grpo_workspace": [i64, i32, szp],
            "ls_grpo_loss_fwd_bwd": [P, i32, i64, i32, P, P, P, P, i32, i32, i32, f32, f32, i32,
                                     i32, P, P, P, P, P, sz, P],
            "ls_grpo_loss_fwd_bwd_noalloc": [P, i32, i64, i32, P, P, P, P, i32, i32, i32, f32,
                                             f32, i32, i32, P, P, P, P, P],
            "ls_validate_page_table": [cache, P, sz, P],
            "ls_validate_page_table_workspace": [cache, szp],
            "ls_last_device_error": [P],
            "ls_selftest_wait_timeout": [P],
            "ls_grpo_logp": [P, i32, i64, i32, P, P, P, P, P, P],
            "ls_status_string": [i32],
            "ls_replay_attn_fwd_ragged_workspace": [cache, P, i32, i32, i32, szp],
            "ls_replay_attn_fwd_ragged": [cache, P, P, P, P, i32, i32, f32, i32, P, P, P, sz, P],
            "ls_replay_attn_bwd_ragged_workspace": [cache, P, i32, i32, i32, szp],
            "ls_replay_attn_bwd_ragged": [cache, P, P, P, P, P, P, P, i32, i32, f32, i32, i32, P,
                                          P, P, P, sz, P],
            "ls_gdn_replay_fwd_workspace": [i32, i32, szp],
            "ls_gdn_replay_bwd_workspace": [i32, i32, szp],
            "ls_gdn_replay_fwd": [P, P, P, P, P, P, i32, i32, f32, P, P, P, sz, P],
            "ls_gdn_replay_bwd": [P, P, P, P, P, P, P, i32, i32, f32, i32, P, P, P, P, P, P, sz,
                                  P],
        }
        for name, args in sig.items():
            f = getattr(l, name)
            f.argtypes = args
            f.restype = C.c_int
        l.ls_status_string.restype = C.c_char_p
        l.ls_kernel_launches.argtypes = []
        l.ls_kernel_launches.restype = C.c_uint64
        _lib = l
    return _lib


def status_string(status: int) -> str:
    return lib().ls_status_string(status).decode()


def _ok(fn: str, status: int) -> None:
    if status != LS_OK:
        raise LongstrawError(fn, status)


def _size(fn: str, *args) -> int:
    out = C.c_size_t(0)
    _ok(fn, getattr(lib(), fn)(*args, C.byref(out)))
    return out.value


def ls_capture_kv(cache: ls_kv_cache, k: int, v: int, start_pos: int, n: int,
                  stream: int = 0) -> None:
    _ok("ls_capture_kv", lib().ls_capture_kv(C.byref(cache), k, v, start_pos, n, stream))


def ls_replay_attn_fwd_workspace(cache: ls_kv_cache, R: int, Hq: int, num_splits: int) -> int:
    return _size("ls_replay_attn_fwd_workspace", C.byref(cache), R, Hq, num_splits)


def ls_replay_attn_fwd(cache: ls_kv_cache, q: int, k_resp: int, v_resp: int, R: int, Hq: int,
                       softmax_scale: float, num_splits: int, o: int, lse: int, workspace: int,
                       workspace_bytes: int, stream: int = 0) -> None:
    _ok("ls_replay_attn_fwd",
        lib().ls_replay_attn_fwd(C.byref(cache), q, k_resp, v_resp, R, Hq, softmax_scale,
                                 num_splits, o, lse, workspace, workspace_bytes, stream))


def ls_replay_attn_fwd_members_workspace(cache: ls_kv_cache, R: int, members: int, Hq: int,
                                         num_splits: int) -> int:
    return _size("ls_replay_attn_fwd_members_workspace", C.byref(cache), R, members, Hq,
                 num_splits)


def ls_replay_attn_fwd_members(cache: ls_kv_cache, q: int, k_resp: int, v_resp: int, R: int,
                               members: int, Hq: int, softmax_scale: float, num_splits: int,
                               o: int, lse: int, workspace: int, workspace_bytes: int,
                               stream: int = 0) -> None:
    _ok("ls_replay_attn_fwd_members",
        lib().ls_replay_attn_fwd_members(C.byref(cache), q, k_resp, v_resp, R, members, Hq,
                                         softmax_scale, num_splits, o, lse, workspace,
                                         workspace_bytes, stream))


def ls_replay_attn_bwd_workspace(cache: ls_kv_cache, R: int, Hq: int, num_splits: int) -> int:
    return _size("ls_replay_attn_bwd_workspace", C.byref(cache), R, Hq, num_splits)


def ls_replay_attn_bwd(cache: ls_kv_cache, q: int, k_resp: int, v_resp: int, o: int, lse: int,
                       d_o: int, R: int, Hq: int, softmax_scale: float, num_splits: int,
                       accumulate: int, dq: int, dk_resp: int, dv_resp: int, workspace: int,
                       workspace_bytes: int, stream: int = 0) -> None:
    _ok("ls_replay_attn_bwd",
        lib().ls_replay_attn_bwd(C.byref(cache), q, k_resp, v_resp, o, lse, d_o, R, Hq,
                                 softmax_scale, num_splits, accumulate, dq, dk_resp, dv_resp,
                                 workspace, workspace_bytes, stream))


def ls_grpo_workspace(T: int, G: int) -> int:
    return _size("ls_grpo_workspace", T, G)


def ls_grpo_loss_fwd_bwd(logits: int, dtype: int, T: int, V: int, targets: int, logp_old: int,
                         rewards: int, resp_lens: int, G: int, member_begin: int, member_end: int,
                         eps: float, adv_eps: float, std_ddof: int, accumulate_loss: int,
                         loss: int, dlogits: int, logp_out: int | None, stats: int | None,
                         workspace: int, workspace_bytes: int, stream: int = 0) -> None:
    _ok("ls_grpo_loss_fwd_bwd",
        lib().ls_grpo_loss_fwd_bwd(logits, dtype, T, V, targets, logp_old, rewards, resp_lens, G,
                                   member_begin, member_end, eps, adv_eps, std_ddof,
                                   accumulate_loss, loss, dlogits, logp_out, stats, workspace,
                                   workspace_bytes, stream))


def ls_grpo_loss_fwd_bwd_noalloc(logits: int, dtype: int, T: int, V: int, targets: int,
                                 logp_old: int, rewards: int, resp_lens: int, G: int,
                                 member_begin: int, member_end: int, eps: float, adv_eps: float,
                                 std_ddof: int, accumulate_loss: int, loss: int, dlogits: int,
                                 logp_out: int | None, stats: int | None,
                                 stream: int = 0) -> None:
    """The GRPO loss without a caller workspace (library-owned fixed scratch; limits
    T <= 262,144 and G <= 1,024; calls must not overlap on the GPU)."""
    _ok("ls_grpo_loss_fwd_bwd_noalloc",
        lib().ls_grpo_loss_fwd_bwd_noalloc(logits, dtype, T, V, targets, logp_old, rewards,
                                           resp_lens, G, member_begin, member_end, eps, adv_eps,
                                           std_ddof, accumulate_loss, loss, dlogits, logp_out,
                                           stats, stream))


def ls_validate_page_table_workspace(cache: ls_kv_cache) -> int:
    return _size("ls_validate_page_table_workspace", C.byref(cache))


def ls_validate_page_table(cache: ls_kv_cache, workspace: int, workspace_bytes: int,
                           stream: int = 0) -> None:
    _ok("ls_validate_page_table",
        lib().ls_validate_page_table(C.byref(cache), workspace, workspace_bytes, stream))


def ls_kernel_launches() -> int:
    """Kernel launches issued by the library so far in this process."""
    return lib().ls_kernel_launches()


def ls_grpo_logp(logits: int, dtype: int, T: int, V: int, targets: int, ref_logp: int | None,
                 logp_out: int, lse_out: int | None, kl_out: int | None, stream: int = 0) -> None:
    _ok("ls_grpo_logp", lib().ls_grpo_logp(logits, dtype, T, V, targets, ref_logp, logp_out,
                                           lse_out, kl_out, stream))


def ls_selftest_wait_timeout(stream: int = 0) -> None:
    """Enqueue a bounded wait that must run out (see include/longstraw.h)."""
    _ok("ls_selftest_wait_timeout", lib().ls_selftest_wait_timeout(stream))


def ls_last_device_error(stream: int = 0) -> int:
    """Synchronise `stream`; return the recorded device-side status (LS_OK if none)."""
    return lib().ls_last_device_error(stream)


def ls_gdn_replay_fwd_workspace(R: int, H: int) -> int:
    return _size("ls_gdn_replay_fwd_workspace", R, H)


def ls_gdn_replay_bwd_workspace(R: int, H: int) -> int:
    return _size("ls_gdn_replay_bwd_workspace", R, H)


def ls_gdn_replay_fwd(state0: int, q: int, k: int, v: int, g: int, beta: int, R: int, H: int,
                      scale: float, o: int, state_out: int | None, workspace: int,
                      workspace_bytes: int, stream: int = 0) -> None:
    _ok("ls_gdn_replay_fwd",
        lib().ls_gdn_replay_fwd(state0, q, k, v, g, beta, R, H, scale, o, state_out, workspace,
                                workspace_bytes, stream))


def ls_gdn_replay_bwd(state0: int, q: int, k: int, v: int, g: int, beta: int, d_o: int, R: int,
                      H: int, scale: float, accumulate: int, dq: int, dk: int, dv: int, dg: int,
                      dbeta: int, workspace: int, workspace_bytes: int, stream: int = 0) -> None:
    _ok("ls_gdn_replay_bwd",
        lib().ls_gdn_replay_bwd(state0, q, k, v, g, beta, d_o, R, H, scale, accumulate, dq, dk,
                                dv, dg, dbeta, workspace, workspace_bytes, stream))


def ls_capture_latent(cache: ls_latent_cache, lat: int, start_pos: int, n: int,
                      stream: int = 0) -> None:
    _ok("ls_capture_latent", lib().ls_capture_latent(C.byref(cache), lat, start_pos, n, stream))


def ls_mla_replay_fwd_workspace(cache: ls_latent_cache, R: int, H: int, num_splits: int) -> int:
    return _size("ls_mla_replay_fwd_workspace", C.byref(cache), R, H, num_splits)


def ls_mla_replay_fwd(cache: ls_latent_cache, q: int, lat_resp: int, R: int, H: int,
                      softmax_scale: float, num_splits: int, o: int, lse: int, workspace: int,
                      workspace_bytes: int, stream: int = 0) -> None:
    _ok("ls_mla_replay_fwd",
        lib().ls_mla_replay_fwd(C.byref(cache), q, lat_resp, R, H, softmax_scale, num_splits, o,
                                lse, workspace, workspace_bytes, stream))


def ls_mla_replay_bwd_workspace(cache: ls_latent_cache, R: int, H: int, num_splits: int) -> int:
    return _size("ls_mla_replay_bwd_workspace", C.byref(cache), R, H, num_splits)


def ls_mla_replay_bwd(cache: ls_latent_cache, q: int, lat_resp: int, o: int, lse: int, d_o: int,
                      R: int, H: int, softmax_scale: float, num_splits: int, dq: int, dlat: int,
                      workspace: int, workspace_bytes: int, stream: int = 0) -> None:
    _ok("ls_mla_replay_bwd",
        lib().ls_mla_replay_bwd(C.byref(cache), q, lat_resp, o, lse, d_o, R, H, softmax_scale,
                                num_splits, dq, dlat, workspace, workspace_bytes, stream))


def _lens(lens) -> tuple:
    arr = (C.c_int32 * len(lens))(*[int(x) for x in lens])
    return arr, len(lens)


def ls_replay_attn_fwd_ragged_workspace(cache: ls_kv_cache, lens, Hq: int, num_splits: int) -> int:
    arr, n = _lens(lens)
    return _size("ls_replay_attn_fwd_ragged_workspace", C.byref(cache), arr, n, Hq, num_splits)


def ls_replay_attn_fwd_ragged(cache: ls_kv_cache, q: int, k_resp: int, v_resp: int, lens, Hq: int,
                              softmax_scale: float, num_splits: int, o: int, lse: int,
                              workspace: int, workspace_bytes: int, stream: int = 0) -> None:
    """lens: the members' response lengths (host)."""
    arr, n = _lens(lens)
    _ok("ls_replay_attn_fwd_ragged",
        lib().ls_replay_attn_fwd_ragged(C.byref(cache), q, k_resp, v_resp, arr, n, Hq,
                                        softmax_scale, num_splits, o, lse, workspace,
                                        workspace_bytes, stream))


def ls_replay_attn_bwd_ragged_workspace(cache: ls_kv_cache, lens, Hq: int, num_splits: int) -> int:
    arr, n = _lens(lens)
    return _size("ls_replay_attn_bwd_ragged_workspace", C.byref(cache), arr, n, Hq, num_splits)


def ls_replay_attn_bwd_ragged(cache: ls_kv_cache, q: int, k_resp: int, v_resp: int, o: int, lse: int,
                              d_o: int, lens, Hq: int, softmax_scale: float, num_splits: int,
                              accumulate: int, dq: int, dk_resp: int, dv_resp: int, workspace: int,
                              workspace_bytes: int, stream: int = 0) -> None:
    arr, n = _lens(lens)
    _ok("ls_replay_attn_bwd_ragged",
        lib().ls_replay_attn_bwd_ragged(C.byref(cache), q, k_resp, v_resp, o, lse, d_o, arr, n,
                                        Hq, softmax_scale, num_splits, accumulate, dq, dk_resp,
                                        dv_resp, workspace, workspace_bytes, stream))
