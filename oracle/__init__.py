"""fp64 CPU oracle for the response-replay hot path (ctypes wrapper).

TEST INFRASTRUCTURE ONLY. The tests, ``__graft_entry__.smoke()`` and the
benchmark's ``cpu_baseline`` leg may import this package; the product package
``response_replay_gb300`` never does, and this package never imports it.

All arithmetic happens in ``longstraw_oracle.c`` (plain C, fp64). This module only
marshals numpy arrays. bf16 inputs are passed as their uint16 bit patterns and
widened exactly to double inside the C code.

Functions and the definitions they follow (LongStraw pages):
  capture_kv       -- literal page scatter (digest, Method step 1).
  attn_fwd[_rows]  -- exact attention over captured pages + causal response keys,
                      prompt split into ranges merged by log-sum-exp (explainer,
                      "Two incompatible architectures", Qwen bullet).
  attn_bwd[...]    -- conditional-response gradient, prompt state stopgrad
                      (digest, Method, last paragraph).
  grpo             -- clipped surrogate with group-relative advantages (digest,
                      Method, L_policy equation).
  grpo_logp        -- pre-step scoring: log-softmax gather of the target and the
                      per-token KL estimate exp(d) - d - 1, d = ref - logp, against a
                      reference policy (the pages fix no KL form; their 2M-token runs
                      used beta = 0).
  gdn_fwd/gdn_bwd  -- Gated-DeltaNet replay from a captured recurrent state (digest,
                      Method step 1 and "Qwen implementation"): the gated delta rule of
                      Yang, Kautz & Hatamizadeh (ICLR 2025) as a token-by-token loop,
                      and its reverse-mode gradient (gdn_oracle.c).
"""
from __future__ import annotations

import ctypes as C
import os
from dataclasses import dataclass

import numpy as np

from . import build as _build

BF16, F32, F64 = 0, 1, 2

_lib = None


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        l = C.CDLL(path)
        P = C.c_void_p
        i32, i64, dbl = C.c_int32, C.c_int64, C.c_double
        l.lso_capture_kv.argtypes = [P, P, P, i64, i64, i32, i32, i32, P, P, i64, i64]
        l.lso_attn_fwd.argtypes = [P, P, P]
        l.lso_attn_fwd_rows.argtypes = [P, i32, P, P, P, P]
        l.lso_attn_bwd.argtypes = [P, P, i32, P, P, P]
        l.lso_attn_bwd_dq_rows.argtypes = [P, P, i32, i32, P, P, P]
        l.lso_attn_bwd_dkdv_keys.argtypes = [P, P, i32, i32, P, P, P, P]
        l.lso_grpo.argtypes = [P, i32, i64, i32, P, P, P, P, i32, i32, i32, dbl, dbl, i32,
                               P, P, P, P, P, P, P]
        l.lso_grpo_dlogits_row.argtypes = [P, i32, i32, i32, dbl, dbl, P]
        l.lso_grpo_logp.argtypes = [P, i32, i64, i32, P, P, P, P, P]
        l.lso_gdn_fwd.argtypes = [P, P, P]
        l.lso_gdn_bwd.argtypes = [P, P, i32, P, P, P, P, P, P]
        l.lso_mla_fwd.argtypes = [P, P, P]
        l.lso_mla_fwd_rows.argtypes = [P, i32, P, P, P, P]
        l.lso_mla_bwd.argtypes = [P, P, P, P]
        l.lso_mla_bwd_dq_rows.argtypes = [P, P, i32, P, P, P]
        l.lso_mla_bwd_dlat_keys.argtypes = [P, P, i32, P, P]
        l.lso_num_threads.argtypes = []
        for f in ("lso_capture_kv", "lso_attn_fwd", "lso_attn_fwd_rows", "lso_attn_bwd",
                  "lso_attn_bwd_dq_rows", "lso_attn_bwd_dkdv_keys", "lso_grpo",
                  "lso_grpo_dlogits_row", "lso_grpo_logp", "lso_gdn_fwd", "lso_gdn_bwd",
                  "lso_mla_fwd", "lso_mla_fwd_rows", "lso_mla_bwd", "lso_mla_bwd_dq_rows",
                  "lso_mla_bwd_dlat_keys", "lso_num_threads"):
            getattr(l, f).restype = C.c_int
        _lib = l
    return _lib


def num_threads() -> int:
    return lib().lso_num_threads()


class _Attn(C.Structure):
    _fields_ = [
        ("k_pool", C.c_void_p), ("v_pool", C.c_void_p), ("pool_dtype", C.c_int32),
        ("page_size", C.c_int32), ("page_table", C.c_void_p), ("num_pages", C.c_int64),
        ("num_logical_pages", C.c_int64), ("P", C.c_int64), ("hkv", C.c_int32),
        ("d", C.c_int32), ("q", C.c_void_p), ("k_resp", C.c_void_p), ("v_resp", C.c_void_p),
        ("in_dtype", C.c_int32), ("R", C.c_int32), ("hq", C.c_int32),
        ("num_splits", C.c_int32), ("scale", C.c_double),
    ]


def _dtype_code(a: np.ndarray) -> int:
    if a.dtype == np.uint16:
        return BF16
    if a.dtype == np.float32:
        return F32
    if a.dtype == np.float64:
        return F64
    raise TypeError(f"unsupported element type {a.dtype} (bf16 is passed as uint16 bits)")


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(C.c_void_p)


def _check(rc: int, what: str):
    if rc == 1:
        raise ValueError(f"oracle {what}: invalid argument")
    if rc == 2:
        raise MemoryError(f"oracle {what}: out of memory")
    if rc != 0:
        raise RuntimeError(f"oracle {what}: error {rc}")


def capture_kv(k_pool: np.ndarray, v_pool: np.ndarray, page_table: np.ndarray,
               page_size: int, k: np.ndarray, v: np.ndarray, start_pos: int) -> None:
    """In-place scatter of k, v ([n][hkv][d] uint16) into the pools
    ([num_pages][hkv][page_size][d] uint16)."""
    for a in (k_pool, v_pool, k, v):
        assert a.dtype == np.uint16 and a.flags.c_contiguous
    pt = np.ascontiguousarray(page_table, dtype=np.int32)
    num_pages, hkv, ps, d = k_pool.shape
    assert ps == page_size
    n = k.shape[0]
    _check(lib().lso_capture_kv(_ptr(k_pool), _ptr(v_pool), _ptr(pt), num_pages, pt.shape[0],
                                page_size, hkv, d, _ptr(k), _ptr(v), start_pos, n),
           "capture_kv")


@dataclass
class AttnProblem:
    """One response branch over a paged prompt cache (host arrays).

    k_pool, v_pool: [num_pages][hkv][page_size][d]; page_table: [num_logical_pages]
    int32; q: [R][hq][d]; k_resp, v_resp: [R][hkv][d]. bf16 arrays as uint16 bits,
    or float32 / float64.
    """
    k_pool: np.ndarray
    v_pool: np.ndarray
    page_table: np.ndarray
    P: int
    q: np.ndarray
    k_resp: np.ndarray
    v_resp: np.ndarray
    scale: float
    num_splits: int = 1

    def _struct(self) -> tuple[_Attn, list]:
        keep = []

        def c(a):
            a = np.ascontiguousarray(a)
            keep.append(a)
            return a

        kp, vp, q, kr, vr = (c(x) for x in (self.k_pool, self.v_pool, self.q, self.k_resp,
                                            self.v_resp))
        pt = c(np.asarray(self.page_table, dtype=np.int32))
        assert _dtype_code(kp) == _dtype_code(vp)
        assert _dtype_code(q) == _dtype_code(kr) == _dtype_code(vr)
        num_pages, hkv, ps, d = kp.shape
        R, hq, d2 = q.shape
        assert d2 == d and kr.shape == (R, hkv, d) and vr.shape == (R, hkv, d)
        s = _Attn(k_pool=kp.ctypes.data, v_pool=vp.ctypes.data, pool_dtype=_dtype_code(kp),
                  page_size=ps, page_table=pt.ctypes.data, num_pages=num_pages,
                  num_logical_pages=pt.shape[0], P=self.P, hkv=hkv, d=d,
                  q=q.ctypes.data, k_resp=kr.ctypes.data, v_resp=vr.ctypes.data,
                  in_dtype=_dtype_code(q), R=R, hq=hq, num_splits=self.num_splits,
                  scale=float(self.scale))
        return s, keep

    @property
    def dims(self):
        R, hq, d = self.q.shape
        return R, hq, self.k_resp.shape[1], d


def attn_fwd(pb: AttnProblem) -> tuple[np.ndarray, np.ndarray]:
    """O [R][hq][d] and LSE [R][hq] (natural log), fp64."""
    R, hq, hkv, d = pb.dims
    s, keep = pb._struct()
    o = np.zeros((R, hq, d), np.float64)
    lse = np.zeros((R, hq), np.float64)
    _check(lib().lso_attn_fwd(C.byref(s), _ptr(o), _ptr(lse)), "attn_fwd")
    return o, lse


def attn_fwd_rows(pb: AttnProblem, ts, hs) -> tuple[np.ndarray, np.ndarray]:
    """O [n][d], LSE [n] for the rows (ts[i], hs[i])."""
    R, hq, hkv, d = pb.dims
    ts = np.ascontiguousarray(ts, dtype=np.int32)
    hs = np.ascontiguousarray(hs, dtype=np.int32)
    s, keep = pb._struct()
    o = np.zeros((len(ts), d), np.float64)
    lse = np.zeros((len(ts),), np.float64)
    _check(lib().lso_attn_fwd_rows(C.byref(s), len(ts), _ptr(ts), _ptr(hs), _ptr(o), _ptr(lse)),
           "attn_fwd_rows")
    return o, lse


def attn_bwd(pb: AttnProblem, d_o: np.ndarray):
    """dQ [R][hq][d], dK, dV [R][hkv][d] (response keys only), fp64."""
    R, hq, hkv, d = pb.dims
    d_o = np.ascontiguousarray(d_o)
    s, keep = pb._struct()
    dq = np.zeros((R, hq, d), np.float64)
    dk = np.zeros((R, hkv, d), np.float64)
    dv = np.zeros((R, hkv, d), np.float64)
    _check(lib().lso_attn_bwd(C.byref(s), _ptr(d_o), _dtype_code(d_o), _ptr(dq), _ptr(dk),
                              _ptr(dv)), "attn_bwd")
    return dq, dk, dv


def attn_bwd_dq_rows(pb: AttnProblem, d_o: np.ndarray, ts, hs) -> np.ndarray:
    R, hq, hkv, d = pb.dims
    d_o = np.ascontiguousarray(d_o)
    ts = np.ascontiguousarray(ts, dtype=np.int32)
    hs = np.ascontiguousarray(hs, dtype=np.int32)
    s, keep = pb._struct()
    dq = np.zeros((len(ts), d), np.float64)
    _check(lib().lso_attn_bwd_dq_rows(C.byref(s), _ptr(d_o), _dtype_code(d_o), len(ts),
                                      _ptr(ts), _ptr(hs), _ptr(dq)), "attn_bwd_dq_rows")
    return dq


def attn_bwd_dkdv_keys(pb: AttnProblem, d_o: np.ndarray, js, kvhs):
    R, hq, hkv, d = pb.dims
    d_o = np.ascontiguousarray(d_o)
    js = np.ascontiguousarray(js, dtype=np.int32)
    kvhs = np.ascontiguousarray(kvhs, dtype=np.int32)
    s, keep = pb._struct()
    dk = np.zeros((len(js), d), np.float64)
    dv = np.zeros((len(js), d), np.float64)
    _check(lib().lso_attn_bwd_dkdv_keys(C.byref(s), _ptr(d_o), _dtype_code(d_o), len(js),
                                        _ptr(js), _ptr(kvhs), _ptr(dk), _ptr(dv)),
           "attn_bwd_dkdv_keys")
    return dk, dv


@dataclass
class GrpoResult:
    loss: float
    adv: np.ndarray
    lse: np.ndarray
    logp: np.ndarray
    ratio: np.ndarray
    coef: np.ndarray
    zeroed: np.ndarray


def grpo(logits: np.ndarray, targets, logp_old, rewards, resp_lens, member_begin: int,
         member_end: int, eps: float, adv_eps: float = 1e-6, std_ddof: int = 1) -> GrpoResult:
    """Loss and per-token quantities for the members [member_begin, member_end) whose
    tokens are the rows of logits [T][V] (uint16 bf16 bits, float32 or float64)."""
    logits = np.ascontiguousarray(logits)
    T, V = logits.shape
    targets = np.ascontiguousarray(targets, dtype=np.int32)
    logp_old = np.ascontiguousarray(logp_old, dtype=np.float64)
    rewards = np.ascontiguousarray(rewards, dtype=np.float64)
    resp_lens = np.ascontiguousarray(resp_lens, dtype=np.int32)
    G = rewards.shape[0]
    loss = np.zeros(1, np.float64)
    adv = np.zeros(G, np.float64)
    lse, logp, ratio, coef = (np.zeros(T, np.float64) for _ in range(4))
    zeroed = np.zeros(T, np.int32)
    _check(lib().lso_grpo(_ptr(logits), _dtype_code(logits), T, V, _ptr(targets), _ptr(logp_old),
                          _ptr(rewards), _ptr(resp_lens), G, member_begin, member_end,
                          float(eps), float(adv_eps), std_ddof, _ptr(loss), _ptr(adv), _ptr(lse),
                          _ptr(logp), _ptr(ratio), _ptr(coef), _ptr(zeroed)), "grpo")
    return GrpoResult(float(loss[0]), adv, lse, logp, ratio, coef, zeroed)


def grpo_logp(logits: np.ndarray, targets, ref_logp=None):
    """Pre-step scoring: (lse, logp, kl) per token row of logits [T][V]; kl is None
    without reference log-probabilities."""
    logits = np.ascontiguousarray(logits)
    T, V = logits.shape
    targets = np.ascontiguousarray(targets, dtype=np.int32)
    lse = np.zeros(T, np.float64)
    logp = np.zeros(T, np.float64)
    kl = None
    ref_p = None
    if ref_logp is not None:
        ref_logp = np.ascontiguousarray(ref_logp, dtype=np.float64)
        kl = np.zeros(T, np.float64)
        ref_p = _ptr(ref_logp)
    _check(lib().lso_grpo_logp(_ptr(logits), _dtype_code(logits), T, V, _ptr(targets), ref_p,
                               _ptr(lse), _ptr(logp), _ptr(kl) if kl is not None else None),
           "grpo_logp")
    return lse, logp, kl


def grpo_dlogits_rows(logits: np.ndarray, rows, targets, lse, coef) -> np.ndarray:
    """dL/dlogits for the listed token rows: [len(rows)][V] fp64."""
    logits = np.ascontiguousarray(logits)
    T, V = logits.shape
    out = np.zeros((len(rows), V), np.float64)
    code = _dtype_code(logits)
    for i, r in enumerate(rows):
        row = logits[r]
        _check(lib().lso_grpo_dlogits_row(row.ctypes.data_as(C.c_void_p), code, V,
                                          int(targets[r]), float(lse[r]), float(coef[r]),
                                          out[i].ctypes.data_as(C.c_void_p)), "grpo_dlogits_row")
    return out


class _Gdn(C.Structure):
    _fields_ = [
        ("state0", C.c_void_p), ("q", C.c_void_p), ("k", C.c_void_p), ("v", C.c_void_p),
        ("in_dtype", C.c_int32), ("g", C.c_void_p), ("beta", C.c_void_p), ("R", C.c_int32),
        ("H", C.c_int32), ("dk", C.c_int32), ("dv", C.c_int32), ("scale", C.c_double),
    ]


@dataclass
class GdnProblem:
    """Gated-DeltaNet replay of R response tokens from a captured state (host arrays).

    state0: [H][dv][dk] float64; q, k: [R][H][dk], v: [R][H][dv] (bf16 as uint16 bits,
    float32 or float64, all the same type); g (log of the decay), beta: [R][H]."""
    state0: np.ndarray
    q: np.ndarray
    k: np.ndarray
    v: np.ndarray
    g: np.ndarray
    beta: np.ndarray
    scale: float

    def _struct(self):
        keep = []

        def c(a, dt=None):
            a = np.ascontiguousarray(a, dtype=dt) if dt is not None else np.ascontiguousarray(a)
            keep.append(a)
            return a

        s0 = c(self.state0, np.float64)
        q, k, v = c(self.q), c(self.k), c(self.v)
        assert _dtype_code(q) == _dtype_code(k) == _dtype_code(v)
        g, b = c(self.g, np.float64), c(self.beta, np.float64)
        R, H, dk = q.shape
        dv = v.shape[2]
        assert k.shape == (R, H, dk) and v.shape[:2] == (R, H) and s0.shape == (H, dv, dk)
        assert g.shape == (R, H) and b.shape == (R, H)
        st = _Gdn(state0=s0.ctypes.data, q=q.ctypes.data, k=k.ctypes.data, v=v.ctypes.data,
                  in_dtype=_dtype_code(q), g=g.ctypes.data, beta=b.ctypes.data, R=R, H=H, dk=dk,
                  dv=dv, scale=float(self.scale))
        return st, keep

    @property
    def dims(self):
        R, H, dk = self.q.shape
        return R, H, dk, self.v.shape[2]


def gdn_fwd(pb: GdnProblem):
    """o [R][H][dv] and the state after the last token [H][dv][dk], fp64."""
    R, H, dk, dv = pb.dims
    st, keep = pb._struct()
    o = np.zeros((R, H, dv), np.float64)
    s_out = np.zeros((H, dv, dk), np.float64)
    _check(lib().lso_gdn_fwd(C.byref(st), _ptr(o), _ptr(s_out)), "gdn_fwd")
    return o, s_out


def gdn_bwd(pb: GdnProblem, d_o: np.ndarray):
    """dq, dk [R][H][dk], dv [R][H][dv], dg, dbeta [R][H] and the gradient that would
    reach the captured state [H][dv][dk] (dropped by the replay: stopgrad), fp64."""
    R, H, dk, dv = pb.dims
    d_o = np.ascontiguousarray(d_o)
    st, keep = pb._struct()
    dq = np.zeros((R, H, dk))
    dkk = np.zeros((R, H, dk))
    dvv = np.zeros((R, H, dv))
    dg = np.zeros((R, H))
    db = np.zeros((R, H))
    ds0 = np.zeros((H, dv, dk))
    _check(lib().lso_gdn_bwd(C.byref(st), _ptr(d_o), _dtype_code(d_o), _ptr(dq), _ptr(dkk),
                             _ptr(dvv), _ptr(dg), _ptr(db), _ptr(ds0)), "gdn_bwd")
    return dq, dkk, dvv, dg, db, ds0


class _Mla(C.Structure):
    _fields_ = [
        ("lat_pool", C.c_void_p), ("page_size", C.c_int32), ("page_table", C.c_void_p),
        ("num_pages", C.c_int64), ("num_logical_pages", C.c_int64), ("P", C.c_int64),
        ("q", C.c_void_p), ("lat_resp", C.c_void_p), ("R", C.c_int32), ("H", C.c_int32),
        ("d_c", C.c_int32), ("d_r", C.c_int32), ("scale", C.c_double),
    ]


@dataclass
class MlaProblem:
    """One response branch over latent (MLA-style) pages (host arrays, bf16 as uint16).

    lat_pool: [num_pages][page_size][d_c + d_r]; page_table: [num_logical_pages] int32;
    q: [R][H][d_c + d_r]; lat_resp: [R][d_c + d_r]."""
    lat_pool: np.ndarray
    page_table: np.ndarray
    P: int
    q: np.ndarray
    lat_resp: np.ndarray
    scale: float
    d_c: int = 512

    def _struct(self):
        keep = []

        def c(a, dt):
            a = np.ascontiguousarray(a, dtype=dt)
            keep.append(a)
            return a

        lp, q, lr = c(self.lat_pool, np.uint16), c(self.q, np.uint16), c(self.lat_resp, np.uint16)
        pt = c(self.page_table, np.int32)
        num_pages, ps, D = lp.shape
        R, H, D2 = q.shape
        assert D2 == D and lr.shape == (R, D) and 0 < self.d_c <= D
        st = _Mla(lat_pool=lp.ctypes.data, page_size=ps, page_table=pt.ctypes.data,
                  num_pages=num_pages, num_logical_pages=pt.shape[0], P=self.P,
                  q=q.ctypes.data, lat_resp=lr.ctypes.data, R=R, H=H, d_c=self.d_c,
                  d_r=D - self.d_c, scale=float(self.scale))
        return st, keep


def mla_fwd(pb: MlaProblem):
    """O [R][H][d_c] and LSE [R][H] (natural log), fp64."""
    R, H, _ = pb.q.shape
    st, keep = pb._struct()
    o = np.zeros((R, H, pb.d_c), np.float64)
    lse = np.zeros((R, H), np.float64)
    _check(lib().lso_mla_fwd(C.byref(st), _ptr(o), _ptr(lse)), "mla_fwd")
    return o, lse


def mla_fwd_rows(pb: MlaProblem, ts, hs):
    """O [n][d_c], LSE [n] for the rows (ts[i], hs[i])."""
    ts = np.ascontiguousarray(ts, dtype=np.int32)
    hs = np.ascontiguousarray(hs, dtype=np.int32)
    st, keep = pb._struct()
    o = np.zeros((len(ts), pb.d_c), np.float64)
    lse = np.zeros((len(ts),), np.float64)
    _check(lib().lso_mla_fwd_rows(C.byref(st), len(ts), _ptr(ts), _ptr(hs), _ptr(o),
                                  _ptr(lse)), "mla_fwd_rows")
    return o, lse


def mla_bwd(pb: MlaProblem, d_o):
    """dq [R][H][D] and d lat [R][D] (the response's own rows; prompt rows stopgrad), fp64.
    d_o: bf16 bits (uint16) [R][H][d_c]."""
    R, H, D = pb.q.shape
    d_o = np.ascontiguousarray(d_o, dtype=np.uint16)
    assert d_o.shape == (R, H, pb.d_c)
    st, keep = pb._struct()
    dq = np.zeros((R, H, D), np.float64)
    dlat = np.zeros((R, D), np.float64)
    _check(lib().lso_mla_bwd(C.byref(st), _ptr(d_o), _ptr(dq), _ptr(dlat)), "mla_bwd")
    return dq, dlat


def mla_bwd_dq_rows(pb: MlaProblem, d_o, ts, hs):
    """dq [n][D] for the rows (ts[i], hs[i])."""
    ts = np.ascontiguousarray(ts, dtype=np.int32)
    hs = np.ascontiguousarray(hs, dtype=np.int32)
    d_o = np.ascontiguousarray(d_o, dtype=np.uint16)
    st, keep = pb._struct()
    dq = np.zeros((len(ts), pb.q.shape[2]), np.float64)
    _check(lib().lso_mla_bwd_dq_rows(C.byref(st), _ptr(d_o), len(ts), _ptr(ts), _ptr(hs),
                                     _ptr(dq)), "mla_bwd_dq_rows")
    return dq


def mla_bwd_dlat_keys(pb: MlaProblem, d_o, js):
    """d lat [n][D] for the response rows js[i]."""
    js = np.ascontiguousarray(js, dtype=np.int32)
    d_o = np.ascontiguousarray(d_o, dtype=np.uint16)
    st, keep = pb._struct()
    dl = np.zeros((len(js), pb.q.shape[2]), np.float64)
    _check(lib().lso_mla_bwd_dlat_keys(C.byref(st), _ptr(d_o), len(js), _ptr(js), _ptr(dl)),
           "mla_bwd_dlat_keys")
    return dl
