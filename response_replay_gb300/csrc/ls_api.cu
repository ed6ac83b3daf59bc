// ls_api.cu -- the extern "C" entry points of include/longstraw.h: argument checks,
// workspace layout, the per-device error word and the kernel launches.
#include <math.h>
#include <stdlib.h>
#include <atomic>
#include <mutex>

#include "../../include/longstraw.h"
#include "ls_dkdv.h"
#include "ls_internal.h"

// One error word per device (module globals are instantiated per device).  Kernels
// OR LS_DEVERR_* bits into it; ls_last_device_error reads and clears it.
__device__ uint32_t g_ls_device_error;

namespace {
std::atomic<uint64_t> g_launches{0};
}  // namespace

void ls_note_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

namespace {

constexpr int kMaxDevices = 64;
constexpr int kHeadDim = 128;

struct DevInfo {
  int sms = 0;
  int pairs = 0;  // CTA pairs resident at once for the pair dQ kernel (0: none)
  uint32_t* err = nullptr;
};
DevInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

// SM count and error-word address of the current device (looked up once per device,
// with that device current).
ls_status dev_info(DevInfo* out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return LS_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_dev_mu);
  DevInfo& d = g_dev[dev];
  if (d.sms == 0) {
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return LS_ERR_CUDA;
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_ls_device_error) != cudaSuccess) return LS_ERR_CUDA;
    d.err = static_cast<uint32_t*>(p);
    int pairs = 0;
    if (ls_bwd_pair_workers(&pairs) != cudaSuccess) {
      pairs = 0;
      (void)cudaGetLastError();  // not fatal: the one-CTA dQ kernel runs instead
    }
    d.pairs = pairs;
    d.sms = sms;
  }
  *out = d;
  return LS_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }
// Per-token arrays of the loss and scoring calls are read and written one element at a
// time, so a member's slice of a token-major buffer (any token offset) is accepted.
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3) == 0; }

int ilog2_exact(int x) {
  if (x <= 0 || (x & (x - 1))) return -1;
  int l = 0;
  while ((1 << l) < x) ++l;
  return l;
}

// Checks shared by every call that reads the cache.
ls_status check_cache(const ls_kv_cache* c) {
  if (!c) return LS_ERR_INVALID_ARG;
  if (c->head_dim != kHeadDim) return LS_ERR_UNSUPPORTED;
  const int l = ilog2_exact(c->page_size);
  if (l < 4 || l > 12) return LS_ERR_UNSUPPORTED;
  if (c->num_kv_heads <= 0 || c->num_pages <= 0 || c->num_logical_pages < 0 || c->num_tokens < 0)
    return LS_ERR_INVALID_ARG;
  if ((int64_t)c->num_pages * c->num_kv_heads * c->page_size >= (1ll << 31)) return LS_ERR_UNSUPPORTED;
  if (c->num_tokens > (int64_t)c->num_logical_pages * c->page_size) return LS_ERR_INVALID_ARG;
  if (!c->k_pool || !c->v_pool || !aligned16(c->k_pool) || !aligned16(c->v_pool))
    return LS_ERR_INVALID_ARG;
  if (c->num_logical_pages > 0 && !c->page_table) return LS_ERR_INVALID_ARG;
  return LS_OK;
}

ls_status from_cuda(cudaError_t e) { return e == cudaSuccess ? LS_OK : LS_ERR_CUDA; }

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// ---- replay attention: argument block, schedule and workspace layout

ls_status check_replay(const ls_kv_cache* c, int R, int Hq, int num_splits) {
  ls_status s = check_cache(c);
  if (s != LS_OK) return s;
  if (R < 0 || Hq <= 0 || num_splits < 1) return LS_ERR_INVALID_ARG;
  if (Hq % c->num_kv_heads != 0) return LS_ERR_INVALID_ARG;
  return LS_OK;
}

// resp_tokens: the response tokens a unit's causal item can reach (R, or members x R
// for packed members).  Token-block-major units when the prompt is short next to them.
// seg: the response's segments (NULL: one response of resp_tokens).
LsSched make_sched_units(const ls_kv_cache* c, int units, int num_splits, int tile, int ctas,
                         int64_t resp_tokens, const LsSegs* seg = nullptr) {
  const int ntiles = (int)((c->num_tokens + tile - 1) / tile);
  LsSched s = ls_make_sched(units, ntiles, num_splits, ctas);
  const int64_t resp_tiles = (resp_tokens + tile - 1) / tile;
  s.tb_major = (int64_t)ntiles < 8 * resp_tiles ? 1 : 0;
  if (seg) {
    s.seg = *seg;
  } else {
    s.seg.n = 1;
    s.seg.off[0] = 0;
    s.seg.off[1] = (int32_t)resp_tokens;
  }
  return s;
}

// Backward dQ geometry: CTA pairs (two-tile units over pairs of SMs) when the device
// fits them, else one CTA per unit of one tile.  LS_BWD_PAIR=0 / 1 in the environment
// selects the one-CTA / pair kernel.
struct BwdGeom {
  int pair, pack, units, unit_rows, workers;
};
BwdGeom bwd_geom(int R, int Hq, int Hkv, const DevInfo& d) {
  static const int env = [] {
    const char* e = getenv("LS_BWD_PAIR");
    return e ? atoi(e) : -1;
  }();
  BwdGeom g;
  g.pair = (env == 1 && d.pairs > 0) ? 1 : 0;
  if (g.pair) {
    g.pack = ls_bwd_pair_pack(R, Hq, Hkv);
    g.units = ls_bwd_pair_units(R, Hq, Hkv);
    g.unit_rows = ls_bwd_pair_unit_rows();
    g.workers = d.pairs;
  } else {
    g.pack = ls_bwd_pack(R, Hq, Hkv);
    g.units = ls_bwd_units(R, Hq, Hkv);
    g.unit_rows = ls_bwd_unit_rows();
    g.workers = d.sms * ls_bwd_ctas_per_sm();
  }
  return g;
}

// Forward geometry of `members` responses of R tokens.  Short responses (grouped-query
// packing) pack the members' tokens into shared tiles as one sequence of members x R
// tokens; otherwise every member has its own units.
struct FwdGeom {
  int pack, tiles, units, upm, rt;
  bool ok;
};
FwdGeom fwd_geom(int R, int members, int Hq, int Hkv) {
  FwdGeom f;
  f.pack = ls_fwd_pack(R, Hq, Hkv);
  f.ok = (int64_t)members * R <= (1 << 30);
  if (!f.ok) return f;
  // the packed-members walk holds at most two key tiles per member (short responses);
  // longer members take per-member units of one head
  if (members > 1 && R >= 2 * ls_fwd_tile()) f.pack = 1;
  if (members > 1 && f.pack > 1) {
    const int tpt = ls_fwd_tile() / f.pack;
    f.rt = members * R;
    f.tiles = f.rt <= tpt ? 1 : 2;
    const int tpu = f.tiles * tpt;
    f.units = (int)((int64_t)(Hq / f.pack) * ((f.rt + tpu - 1) / tpu));
    f.upm = INT32_MAX;
  } else {
    f.rt = R;
    f.tiles = f.pack == 1 ? 2 : ls_fwd_tiles(R, Hq, Hkv);
    const int upm = f.pack == 1 ? ls_num_units(R, Hq, Hkv, ls_fwd_unit_rows())
                                : ls_fwd_units(R, Hq, Hkv);
    f.ok = (int64_t)members * upm <= (1 << 30);
    f.units = members * upm;
    f.upm = members > 1 ? upm : INT32_MAX;
  }
  return f;
}

struct FwdWs {
  size_t part_o, part_lse, total;
};
FwdWs fwd_ws(const LsSched& sc, int unit_rows) {
  FwdWs w;
  size_t p = 0;
  // one partial (o, lse) per tail piece when the tail units are cut into pieces
  const size_t slots = sc.has_partials() ? (size_t)sc.num_pieces() : 0;
  w.part_o = p;
  p = align256(p + slots * unit_rows * kHeadDim * 4);
  w.part_lse = p;
  p = align256(p + slots * unit_rows * 4);
  w.total = p;
  return w;
}

struct BwdWs {
  size_t delta, dt, lse2t, part_dq, part_dkdv, total;
};
BwdWs bwd_ws(const LsSched& sc, int unit_rows, int R, int Hq, int Hkv, int sms,
             const LsSegs* segs = nullptr) {
  BwdWs w;
  size_t p = 0;
  const size_t rp = (size_t)(R + 127) / 128 * 128;
  w.delta = p;
  p = align256(p + (size_t)R * Hq * 4);
  w.dt = p;
  p = align256(p + rp * Hq * 4);
  w.lse2t = p;
  p = align256(p + rp * Hq * 4);
  w.part_dq = p;
  p = align256(p + (sc.has_partials() ? (size_t)sc.num_pieces() * unit_rows * kHeadDim * 4 : 0));
  w.part_dkdv = p;
  p = align256(p + ls_dkdv_part_bytes(R, Hq, Hkv, sms, segs));
  w.total = p;
  return w;
}

LsAttnArgs attn_args(const ls_kv_cache* c, const void* q, const void* kr, const void* vr, int R,
                     int Hq, float scale, uint32_t* err) {
  LsAttnArgs a;
  a.k_pool = c->k_pool;
  a.v_pool = c->v_pool;
  a.page_table = c->page_table;
  a.num_pages = c->num_pages;
  a.ps_log2 = ilog2_exact(c->page_size);
  a.P = c->num_tokens;
  a.hkv = c->num_kv_heads;
  a.hq = Hq;
  a.g = Hq / c->num_kv_heads;
  a.pack = 1;
  a.tiles = 2;
  a.R = R;
  a.members = 1;
  a.upm = INT32_MAX;
  a.rt = R;
  a.q = q;
  a.k_resp = kr;
  a.v_resp = vr;
  a.scale = scale;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.err = err;
  return a;
}

// Segments of ragged members laid out back to back (host lens); the total in *T and the
// longest member in *rmax.
ls_status make_segs(const int32_t* lens, int members, LsSegs* seg, int* T, int* rmax) {
  if (!lens || members < 1 || members > kLsMaxSegs) return LS_ERR_INVALID_ARG;
  int64_t t = 0;
  int m = 0;
  seg->n = members;
  seg->off[0] = 0;
  for (int i = 0; i < members; ++i) {
    if (lens[i] < 0) return LS_ERR_INVALID_ARG;
    t += lens[i];
    if (t > (1 << 30)) return LS_ERR_UNSUPPORTED;
    seg->off[i + 1] = (int32_t)t;
    if (lens[i] > m) m = lens[i];
  }
  *T = (int)t;
  *rmax = m;
  return LS_OK;
}

}  // namespace

extern "C" {

uint64_t ls_kernel_launches(void) { return g_launches.load(std::memory_order_relaxed); }

const char* ls_status_string(ls_status s) {
  switch (s) {
    case LS_OK: return "ok";
    case LS_ERR_INVALID_ARG: return "invalid argument";
    case LS_ERR_UNSUPPORTED: return "unsupported configuration";
    case LS_ERR_WORKSPACE: return "workspace missing or too small";
    case LS_ERR_CUDA: return "CUDA error";
    case LS_ERR_TIMEOUT: return "device pipeline wait timed out";
    case LS_ERR_DEVICE_CHECK: return "device-side argument check failed";
  }
  return "unknown status";
}

ls_status ls_capture_kv(const ls_kv_cache* cache, const void* k, const void* v, int64_t start_pos,
                        int64_t n, ls_stream_t stream) {
  ls_status s = check_cache(cache);
  if (s != LS_OK) return s;
  if (start_pos < 0 || n < 0) return LS_ERR_INVALID_ARG;
  if (start_pos + n > (int64_t)cache->num_logical_pages * cache->page_size) return LS_ERR_INVALID_ARG;
  if (n == 0) return LS_OK;
  if (!k || !v || !aligned16(k) || !aligned16(v)) return LS_ERR_INVALID_ARG;
  DevInfo d;
  if ((s = dev_info(&d)) != LS_OK) return s;
  return from_cuda(ls_launch_capture(k, v, cache->k_pool, cache->v_pool, cache->page_table,
                                     cache->num_pages, ilog2_exact(cache->page_size),
                                     cache->num_kv_heads, start_pos, n, d.sms, d.err,
                                     (cudaStream_t)stream));
}

ls_status ls_replay_attn_fwd_members_workspace(const ls_kv_cache* cache, int R, int members,
                                               int Hq, int num_splits, size_t* bytes) {
  ls_status s = check_replay(cache, R, Hq, num_splits);
  if (s != LS_OK) return s;
  if (!bytes || members < 0) return LS_ERR_INVALID_ARG;
  const FwdGeom f = fwd_geom(R, members > 0 ? members : 1, Hq, cache->num_kv_heads);
  if (!f.ok) return LS_ERR_UNSUPPORTED;
  DevInfo d;
  if ((s = dev_info(&d)) != LS_OK) return s;
  LsSched sc = make_sched_units(cache, f.units, num_splits, ls_fwd_tile(),
                                d.sms * ls_fwd_ctas_per_sm(), f.rt);
  if (members > 1) sc.tb_major = 0;  // the members' layouts walk their units group major
  *bytes = fwd_ws(sc, ls_fwd_unit_rows()).total;
  return LS_OK;
}

ls_status ls_replay_attn_fwd_members(const ls_kv_cache* cache, const void* q, const void* k_resp,
                                     const void* v_resp, int R, int members, int Hq,
                                     float softmax_scale, int num_splits, void* o, float* lse,
                                     void* workspace, size_t workspace_bytes,
                                     ls_stream_t stream) {
  ls_status s = check_replay(cache, R, Hq, num_splits);
  if (s != LS_OK) return s;
  if (!isfinite(softmax_scale) || !(softmax_scale > 0.f) || members < 0) return LS_ERR_INVALID_ARG;
  if (R == 0 || members == 0) return LS_OK;
  const FwdGeom f = fwd_geom(R, members, Hq, cache->num_kv_heads);
  if (!f.ok) return LS_ERR_UNSUPPORTED;
  const void* ptrs[] = {q, k_resp, v_resp, o, lse};
  for (const void* p : ptrs)
    if (!p || !aligned16(p)) return LS_ERR_INVALID_ARG;
  DevInfo d;
  if ((s = dev_info(&d)) != LS_OK) return s;
  LsSched sc = make_sched_units(cache, f.units, num_splits, ls_fwd_tile(),
                                d.sms * ls_fwd_ctas_per_sm(), f.rt);
  if (members > 1) sc.tb_major = 0;  // the members' layouts walk their units group major
  const FwdWs w = fwd_ws(sc, ls_fwd_unit_rows());
  if (w.total > 0 && (!workspace || workspace_bytes < w.total || !aligned16(workspace)))
    return LS_ERR_WORKSPACE;
  LsAttnArgs a = attn_args(cache, q, k_resp, v_resp, R, Hq, softmax_scale, d.err);
  a.pack = f.pack;
  a.tiles = f.tiles;
  a.members = members;
  a.upm = f.upm;
  a.rt = f.rt;
  LsFwdOut out;
  out.o = o;
  out.lse = lse;
  out.part_o = reinterpret_cast<float*>(static_cast<char*>(workspace) + w.part_o);
  out.part_lse = reinterpret_cast<float*>(static_cast<char*>(workspace) + w.part_lse);
  return from_cuda(ls_launch_replay_fwd(a, sc, out, (cudaStream_t)stream));
}

ls_status ls_replay_attn_fwd_workspace(const ls_kv_cache* cache, int R, int Hq, int num_splits,
                                       size_t* bytes) {
  return ls_replay_attn_fwd_members_workspace(cache, R, 1, Hq, num_splits, bytes);
}

ls_status ls_replay_attn_fwd(const ls_kv_cache* cache, const void* q, const void* k_resp,
                             const void* v_resp, int R, int Hq, float softmax_scale, int num_splits,
                             void* o, float* lse, void* workspace, size_t workspace_bytes,
                             ls_stream_t stream) {
  return ls_replay_attn_fwd_members(cache, q, k_resp, v_resp, R, 1, Hq, softmax_scale, num_splits,
                                    o, lse, workspace, workspace_bytes, stream);
}

}  // extern "C"

namespace {

// Backward of one response of R tokens cut into the segments `seg` (one segment: a
// single response; several: ragged members back to back, each seeing the prompt and its
// own keys).  resp_max: the longest segment.
ls_status bwd_workspace_impl(const ls_kv_cache* cache, int R, const LsSegs& seg, int resp_max,
                             int Hq, int num_splits, size_t* bytes) {
  ls_status s = check_replay(cache, R, Hq, num_splits);
  if (s != LS_OK) return s;
  if (!bytes) return LS_ERR_INVALID_ARG;
  if (seg.n > 1 && (R + 127) / 128 > kLsMaxDkTiles) return LS_ERR_UNSUPPORTED;
  DevInfo d;
  if ((s = dev_info(&d)) != LS_OK) return s;
  const BwdGeom g = bwd_geom(R, Hq, cache->num_kv_heads, d);
  const LsSched sc = make_sched_units(cache, g.units, num_splits, ls_bwd_tile(), g.workers,
                                      resp_max, &seg);
  *bytes = bwd_ws(sc, g.unit_rows, R, Hq, cache->num_kv_heads, d.sms, &seg).total;
  return LS_OK;
}

ls_status bwd_impl(const ls_kv_cache* cache, const void* q, const void* k_resp, const void* v_resp,
                   const void* o, const float* lse, const void* d_o, int R, const LsSegs& seg,
                   int resp_max, int Hq, float softmax_scale, int num_splits, int accumulate,
                   float* dq, float* dk_resp, float* dv_resp, void* workspace,
                   size_t workspace_bytes, ls_stream_t stream) {
  ls_status s = check_replay(cache, R, Hq, num_splits);
  if (s != LS_OK) return s;
  if (!isfinite(softmax_scale) || !(softmax_scale > 0.f)) return LS_ERR_INVALID_ARG;
  if (R == 0) return LS_OK;
  if (seg.n > 1 && (R + 127) / 128 > kLsMaxDkTiles) return LS_ERR_UNSUPPORTED;
  const void* ptrs[] = {q, k_resp, v_resp, o, lse, d_o, dq, dk_resp, dv_resp};
  for (const void* p : ptrs)
    if (!p || !aligned16(p)) return LS_ERR_INVALID_ARG;
  DevInfo d;
  if ((s = dev_info(&d)) != LS_OK) return s;
  const BwdGeom g = bwd_geom(R, Hq, cache->num_kv_heads, d);
  const LsSched sc = make_sched_units(cache, g.units, num_splits, ls_bwd_tile(), g.workers,
                                      resp_max, &seg);
  const BwdWs w = bwd_ws(sc, g.unit_rows, R, Hq, cache->num_kv_heads, d.sms, &seg);
  if (!workspace || workspace_bytes < w.total || !aligned16(workspace)) return LS_ERR_WORKSPACE;
  LsAttnArgs a = attn_args(cache, q, k_resp, v_resp, R, Hq, softmax_scale, d.err);
  a.pack = g.pack;
  LsBwdIn b;
  b.o = o;
  b.lse = lse;
  b.d_o = d_o;
  b.delta = reinterpret_cast<float*>(static_cast<char*>(workspace) + w.delta);
  b.dt = reinterpret_cast<float*>(static_cast<char*>(workspace) + w.dt);
  b.lse2t = reinterpret_cast<float*>(static_cast<char*>(workspace) + w.lse2t);
  b.part_dq = reinterpret_cast<float*>(static_cast<char*>(workspace) + w.part_dq);
  b.part_dkdv = reinterpret_cast<float*>(static_cast<char*>(workspace) + w.part_dkdv);
  b.dq = dq;
  b.dk = dk_resp;
  b.dv = dv_resp;
  b.accumulate = accumulate != 0;
  b.pair = g.pair;
  return from_cuda(ls_launch_replay_bwd(a, sc, b, d.sms, (cudaStream_t)stream));
}

LsSegs single_seg(int R) {
  LsSegs s;
  s.n = 1;
  s.off[0] = 0;
  s.off[1] = R;
  return s;
}

}  // namespace

extern "C" {

ls_status ls_replay_attn_bwd_workspace(const ls_kv_cache* cache, int R, int Hq, int num_splits,
                                       size_t* bytes) {
  return bwd_workspace_impl(cache, R, single_seg(R), R, Hq, num_splits, bytes);
}

ls_status ls_replay_attn_bwd(const ls_kv_cache* cache, const void* q, const void* k_resp,
                             const void* v_resp, const void* o, const float* lse, const void* d_o,
                             int R, int Hq, float softmax_scale, int num_splits, int accumulate,
                             float* dq, float* dk_resp, float* dv_resp, void* workspace,
                             size_t workspace_bytes, ls_stream_t stream) {
  return bwd_impl(cache, q, k_resp, v_resp, o, lse, d_o, R, single_seg(R), R, Hq, softmax_scale,
                  num_splits, accumulate, dq, dk_resp, dv_resp, workspace, workspace_bytes, stream);
}

ls_status ls_replay_attn_bwd_ragged_workspace(const ls_kv_cache* cache, const int32_t* lens,
                                              int members, int Hq, int num_splits, size_t* bytes) {
  LsSegs seg;
  int T = 0, rmax = 0;
  ls_status s = make_segs(lens, members, &seg, &T, &rmax);
  if (s != LS_OK) return s;
  return bwd_workspace_impl(cache, T, seg, rmax, Hq, num_splits, bytes);
}

ls_status ls_replay_attn_bwd_ragged(const ls_kv_cache* cache, const void* q, const void* k_resp,
                                    const void* v_resp, const void* o, const float* lse,
                                    const void* d_o, const int32_t* lens, int members, int Hq,
                                    float softmax_scale, int num_splits, int accumulate, float* dq,
                                    float* dk_resp, float* dv_resp, void* workspace,
                                    size_t workspace_bytes, ls_stream_t stream) {
  LsSegs seg;
  int T = 0, rmax = 0;
  ls_status s = make_segs(lens, members, &seg, &T, &rmax);
  if (s != LS_OK) return s;
  return bwd_impl(cache, q, k_resp, v_resp, o, lse, d_o, T, seg, rmax, Hq, softmax_scale,
                  num_splits, accumulate, dq, dk_resp, dv_resp, workspace, workspace_bytes, stream);
}

ls_status ls_replay_attn_fwd_ragged_workspace(const ls_kv_cache* cache, const int32_t* lens,
                                              int members, int Hq, int num_splits, size_t* bytes) {
  LsSegs seg;
  int T = 0, rmax = 0;
  ls_status s = make_segs(lens, members, &seg, &T, &rmax);
  if (s != LS_OK) return s;
  s = check_replay(cache, T, Hq, num_splits);
  if (s != LS_OK) return s;
  if (!bytes) return LS_ERR_INVALID_ARG;
  const FwdGeom f = fwd_geom(T, 1, Hq, cache->num_kv_heads);
  if (!f.ok) return LS_ERR_UNSUPPORTED;
  DevInfo d;
  if ((s = dev_info(&d)) != LS_OK) return s;
  const LsSched sc = make_sched_units(cache, f.units, num_splits, ls_fwd_tile(),
                                      d.sms * ls_fwd_ctas_per_sm(), rmax, &seg);
  *bytes = fwd_ws(sc, ls_fwd_unit_rows()).total;
  return LS_OK;
}

ls_status ls_replay_attn_fwd_ragged(const ls_kv_cache* cache, const void* q, const void* k_resp,
                                    const void* v_resp, const int32_t* lens, int members, int Hq,
                                    float softmax_scale, int num_splits, void* o, float* lse,
                                    void* workspace, size_t workspace_bytes, ls_stream_t stream) {
  LsSegs seg;
  int T = 0, rmax = 0;
  ls_status s = make_segs(lens, members, &seg, &T, &rmax);
  if (s != LS_OK) return s;
  s = check_replay(cache, T, Hq, num_splits);
  if (s != LS_OK) return s;
  if (!isfinite(softmax_scale) || !(softmax_scale > 0.f)) return LS_ERR_INVALID_ARG;
  if (T == 0) return LS_OK;
  const FwdGeom f = fwd_geom(T, 1, Hq, cache->num_kv_heads);
  if (!f.ok) return LS_ERR_UNSUPPORTED;
  const void* ptrs[] = {q, k_resp, v_resp, o, lse};
  for (const void* p : ptrs)
    if (!p || !aligned16(p)) return LS_ERR_INVALID_ARG;
  DevInfo d;
  if ((s = dev_info(&d)) != LS_OK) return s;
  const LsSched sc = make_sched_units(cache, f.units, num_splits, ls_fwd_tile(),
                                      d.sms * ls_fwd_ctas_per_sm(), rmax, &seg);
  const FwdWs w = fwd_ws(sc, ls_fwd_unit_rows());
  if (w.total > 0 && (!workspace || workspace_bytes < w.total || !aligned16(workspace)))
    return LS_ERR_WORKSPACE;
  LsAttnArgs a = attn_args(cache, q, k_resp, v_resp, T, Hq, softmax_scale, d.err);
  a.pack = f.pack;
  a.tiles = f.tiles;
  a.members = 1;
  a.upm = f.upm;
  a.rt = f.rt;
  LsFwdOut out;
  out.o = o;
  out.lse = lse;
  out.part_o = reinterpret_cast<float*>(static_cast<char*>(workspace) + w.part_o);
  out.part_lse = reinterpret_cast<float*>(static_cast<char*>(workspace) + w.part_lse);
  return from_cuda(ls_launch_replay_fwd(a, sc, out, (cudaStream_t)stream));
}

ls_status ls_grpo_workspace(int64_t T, int G, size_t* bytes) {
  if (T < 0 || G <= 0 || !bytes) return LS_ERR_INVALID_ARG;
  *bytes = ls_grpo_ws_bytes(T, G);
  return LS_OK;
}

ls_status ls_grpo_loss_fwd_bwd(const void* logits, ls_dtype dtype, int64_t T, int V,
                               const int32_t* targets, const float* logp_old, const float* rewards,
                               const int32_t* resp_lens, int G, int member_begin, int member_end,
                               float eps, float adv_eps, int std_ddof, int accumulate_loss,
                               float* loss, void* dlogits, float* logp_out, float* stats,
                               void* workspace, size_t workspace_bytes, ls_stream_t stream) {
  if (dtype != LS_BF16 && dtype != LS_FP32) return LS_ERR_INVALID_ARG;
  if (T < 0 || V <= 0 || V > (1 << 30) || G <= 0 || std_ddof < 0 || G - std_ddof < 1)
    return LS_ERR_INVALID_ARG;
  if (member_begin < 0 || member_end > G || member_begin > member_end) return LS_ERR_INVALID_ARG;
  if (!(eps >= 0.f) || !isfinite(adv_eps) || adv_eps < 0.f) return LS_ERR_INVALID_ARG;
  if (!rewards || !resp_lens || !loss || !aligned16(rewards) || !aligned16(resp_lens) ||
      !aligned16(loss))
    return LS_ERR_INVALID_ARG;
  if (T > 0) {
    const void* rows[] = {logits, dlogits};
    for (const void* p : rows)
      if (!p || !aligned16(p)) return LS_ERR_INVALID_ARG;
    const void* tok[] = {targets, logp_old};
    for (const void* p : tok)
      if (!p || !aligned4(p)) return LS_ERR_INVALID_ARG;
    if (logp_out && !aligned4(logp_out)) return LS_ERR_INVALID_ARG;
  }
  if (stats && !aligned16(stats)) return LS_ERR_INVALID_ARG;
  const size_t need = ls_grpo_ws_bytes(T, G);
  if (!workspace || workspace_bytes < need || !aligned16(workspace)) return LS_ERR_WORKSPACE;
  DevInfo d;
  ls_status s = dev_info(&d);
  if (s != LS_OK) return s;
  LsGrpoArgs a;
  a.logits = logits;
  a.is_bf16 = dtype == LS_BF16;
  a.T = T;
  a.V = V;
  a.targets = targets;
  a.logp_old = logp_old;
  a.rewards = rewards;
  a.resp_lens = resp_lens;
  a.G = G;
  a.member_begin = member_begin;
  a.member_end = member_end;
  a.eps = eps;
  a.adv_eps = adv_eps;
  a.std_ddof = std_ddof;
  a.accumulate_loss = accumulate_loss != 0;
  a.loss = loss;
  a.dlogits = dlogits;
  a.logp_out = logp_out;
  a.stats = stats;
  a.workspace = workspace;
  a.err = d.err;
  return from_cuda(ls_launch_grpo(a, d.sms, (cudaStream_t)stream));
}

ls_status ls_validate_page_table_workspace(const ls_kv_cache* cache, size_t* bytes) {
  ls_status s = check_cache(cache);
  if (s != LS_OK) return s;
  if (!bytes) return LS_ERR_INVALID_ARG;
  *bytes = align256(((size_t)cache->num_pages + 31) / 32 * 4);
  return LS_OK;
}

ls_status ls_validate_page_table(const ls_kv_cache* cache, void* workspace, size_t workspace_bytes,
                                 ls_stream_t stream) {
  size_t need = 0;
  ls_status s = ls_validate_page_table_workspace(cache, &need);
  if (s != LS_OK) return s;
  if (!workspace || workspace_bytes < need || !aligned16(workspace)) return LS_ERR_WORKSPACE;
  DevInfo d;
  if ((s = dev_info(&d)) != LS_OK) return s;
  const int32_t logical =
      (int32_t)((cache->num_tokens + cache->page_size - 1) / cache->page_size);
  if (logical == 0) return LS_OK;
  return from_cuda(ls_launch_validate_pages(cache->page_table, logical, cache->num_pages,
                                            static_cast<uint32_t*>(workspace), d.err,
                                            (cudaStream_t)stream));
}

ls_status ls_grpo_logp(const void* logits, ls_dtype dtype, int64_t T, int V,
                       const int32_t* targets, const float* ref_logp, float* logp_out,
                       float* lse_out, float* kl_out, ls_stream_t stream) {
  if (dtype != LS_BF16 && dtype != LS_FP32) return LS_ERR_INVALID_ARG;
  if (T < 0 || V <= 0 || V > (1 << 30)) return LS_ERR_INVALID_ARG;
  if (kl_out && !ref_logp) return LS_ERR_INVALID_ARG;
  if (T > 0) {
    if (!logits || !aligned16(logits)) return LS_ERR_INVALID_ARG;
    const void* ptrs[] = {targets, logp_out};
    for (const void* p : ptrs)
      if (!p || !aligned4(p)) return LS_ERR_INVALID_ARG;
    const void* opt[] = {ref_logp, lse_out, kl_out};
    for (const void* p : opt)
      if (p && !aligned4(p)) return LS_ERR_INVALID_ARG;
  }
  DevInfo d;
  ls_status s = dev_info(&d);
  if (s != LS_OK) return s;
  return from_cuda(ls_launch_grpo_logp(logits, dtype == LS_BF16, T, V, targets, ref_logp,
                                       logp_out, lse_out, kl_out, d.err, d.sms,
                                       (cudaStream_t)stream));
}

ls_status ls_gdn_replay_fwd_workspace(int R, int H, size_t* bytes) {
  if (R < 0 || H <= 0 || !bytes) return LS_ERR_INVALID_ARG;
  if ((int64_t)R * H >= (1ll << 31) || (R + 63) / 64 * (int64_t)H > 65535) return LS_ERR_UNSUPPORTED;
  *bytes = ls_gdn_ws_bytes(R, H, false);
  return LS_OK;
}

ls_status ls_gdn_replay_bwd_workspace(int R, int H, size_t* bytes) {
  if (R < 0 || H <= 0 || !bytes) return LS_ERR_INVALID_ARG;
  if ((int64_t)R * H >= (1ll << 31) || (R + 63) / 64 * (int64_t)H > 65535) return LS_ERR_UNSUPPORTED;
  *bytes = ls_gdn_ws_bytes(R, H, true);
  return LS_OK;
}

ls_status ls_gdn_replay_fwd(const float* state0, const void* q, const void* k, const void* v,
                            const float* g, const float* beta, int R, int H, float scale, void* o,
                            float* state_out, void* workspace, size_t workspace_bytes,
                            ls_stream_t stream) {
  size_t need = 0;
  ls_status s = ls_gdn_replay_fwd_workspace(R, H, &need);
  if (s != LS_OK) return s;
  if (!isfinite(scale)) return LS_ERR_INVALID_ARG;
  if (!state0 || !aligned16(state0) || (state_out && !aligned16(state_out))) return LS_ERR_INVALID_ARG;
  if (R == 0) {  // no tokens: the state passes through unchanged
    if (state_out && state_out != state0)
      return from_cuda(cudaMemcpyAsync(state_out, state0, (size_t)H * 128 * 128 * 4,
                                       cudaMemcpyDeviceToDevice, (cudaStream_t)stream));
    return LS_OK;
  }
  const void* ptrs[] = {q, k, v, g, beta, o};
  for (const void* p : ptrs)
    if (!p || !aligned16(p)) return LS_ERR_INVALID_ARG;
  if (!workspace || workspace_bytes < need || !aligned16(workspace)) return LS_ERR_WORKSPACE;
  DevInfo d;
  if ((s = dev_info(&d)) != LS_OK) return s;
  LsGdnArgs a{state0, q, k, v, g, beta, R, H, scale, d.err};
  return from_cuda(ls_launch_gdn_fwd(a, o, state_out, workspace, (cudaStream_t)stream));
}

ls_status ls_gdn_replay_bwd(const float* state0, const void* q, const void* k, const void* v,
                            const float* g, const float* beta, const void* d_o, int R, int H,
                            float scale, int accumulate, float* dq, float* dk, float* dv, float* dg,
                            float* dbeta, void* workspace, size_t workspace_bytes,
                            ls_stream_t stream) {
  size_t need = 0;
  ls_status s = ls_gdn_replay_bwd_workspace(R, H, &need);
  if (s != LS_OK) return s;
  if (!isfinite(scale)) return LS_ERR_INVALID_ARG;
  if (R == 0) return LS_OK;
  const void* ptrs[] = {state0, q, k, v, g, beta, d_o, dq, dk, dv, dg, dbeta};
  for (const void* p : ptrs)
    if (!p || !aligned16(p)) return LS_ERR_INVALID_ARG;
  if (!workspace || workspace_bytes < need || !aligned16(workspace)) return LS_ERR_WORKSPACE;
  DevInfo d;
  if ((s = dev_info(&d)) != LS_OK) return s;
  LsGdnArgs a{state0, q, k, v, g, beta, R, H, scale, d.err};
  return from_cuda(ls_launch_gdn_bwd(a, d_o, accumulate != 0, dq, dk, dv, dg, dbeta, workspace,
                                     (cudaStream_t)stream));
}

// ---- latent (MLA-style) replay

}  // extern "C"

namespace {

ls_status check_latent(const ls_latent_cache* c) {
  if (!c) return LS_ERR_INVALID_ARG;
  const int l = ilog2_exact(c->page_size);
  if (l < 5 || l > 12) return LS_ERR_UNSUPPORTED;
  if (c->num_pages <= 0 || c->num_logical_pages < 0 || c->num_tokens < 0) return LS_ERR_INVALID_ARG;
  if ((int64_t)c->num_pages * c->page_size >= (1ll << 31)) return LS_ERR_UNSUPPORTED;
  if (c->num_tokens > (int64_t)c->num_logical_pages * c->page_size) return LS_ERR_INVALID_ARG;
  if (!c->pool || !aligned16(c->pool)) return LS_ERR_INVALID_ARG;
  if (c->num_logical_pages > 0 && !c->page_table) return LS_ERR_INVALID_ARG;
  return LS_OK;
}

// Units: (row tile of 128 token-major (t, h) rows) x (half of the output columns).
ls_status mla_sched(const ls_latent_cache* c, int R, int H, int num_splits, LsSched* sc,
                    size_t* part_o, size_t* part_lse, size_t* total) {
  if (R < 0 || H <= 0 || num_splits < 1) return LS_ERR_INVALID_ARG;
  const int64_t rows = (int64_t)R * H;
  const int64_t units = 2 * ((rows + ls_mla_unit_rows() - 1) / ls_mla_unit_rows());
  if (rows >= (1ll << 31) || units >= (1ll << 30)) return LS_ERR_UNSUPPORTED;
  DevInfo d;
  const ls_status s = dev_info(&d);
  if (s != LS_OK) return s;
  const int tile = ls_mla_tile();
  // a 1-token response of 64 heads is two units: let them spread over every SM
  *sc = ls_make_sched((int)units, (int)((c->num_tokens + tile - 1) / tile), num_splits, d.sms,
                      256);
  const size_t pieces = sc->has_partials() ? (size_t)sc->num_pieces() : 0;
  *part_o = 0;
  *part_lse = align256(pieces * ls_mla_unit_rows() * ls_mla_half() * sizeof(float));
  *total = *part_lse + align256(pieces * ls_mla_unit_rows() * sizeof(float));
  return LS_OK;
}

// Backward units: row tiles of 64 (t, h) rows (all 576 dq columns each).  Workspace:
// D per row, partial dq of tail-unit pieces, partial d lat of units cut between CTAs.
ls_status mla_bwd_sched(const ls_latent_cache* c, int R, int H, int num_splits, LsSched* sc,
                        size_t* off_pdq, size_t* off_pdl, size_t* total, int* sms) {
  if (R < 0 || H <= 0 || num_splits < 1) return LS_ERR_INVALID_ARG;
  const int64_t rows = (int64_t)R * H;
  const int64_t units = (rows + ls_mla_bwd_unit_rows() - 1) / ls_mla_bwd_unit_rows();
  if (rows >= (1ll << 31) || units >= (1ll << 30)) return LS_ERR_UNSUPPORTED;
  DevInfo d;
  const ls_status s = dev_info(&d);
  if (s != LS_OK) return s;
  const int tile = ls_mla_bwd_tile();
  // one 64-row unit holds a 1-token response of 64 heads: let it spread over every SM
  *sc = ls_make_sched((int)units, (int)((c->num_tokens + tile - 1) / tile), num_splits, d.sms,
                      256);
  const size_t pieces = sc->has_partials() ? (size_t)sc->num_pieces() : 0;
  const size_t pc = (size_t)ls_mla_bwd_part_cols();
  *off_pdq = align256((size_t)rows * sizeof(float));
  *off_pdl = *off_pdq + align256(pieces * ls_mla_bwd_unit_rows() * 576 * sizeof(float));
  *total = *off_pdl +
           align256((size_t)2 * ls_mla_bwd_dlat_ctas(R, H, d.sms) * 128 * pc * sizeof(float));
  *sms = d.sms;
  return LS_OK;
}

}  // namespace

extern "C" {

ls_status ls_capture_latent(const ls_latent_cache* cache, const void* lat, int64_t start_pos,
                            int64_t n, ls_stream_t stream) {
  ls_status s = check_latent(cache);
  if (s != LS_OK) return s;
  if (start_pos < 0 || n < 0) return LS_ERR_INVALID_ARG;
  if (start_pos + n > (int64_t)cache->num_logical_pages * cache->page_size) return LS_ERR_INVALID_ARG;
  if (n == 0) return LS_OK;
  if (!lat || !aligned16(lat)) return LS_ERR_INVALID_ARG;
  DevInfo d;
  if ((s = dev_info(&d)) != LS_OK) return s;
  return from_cuda(ls_launch_capture_latent(lat, cache->pool, cache->page_table, cache->num_pages,
                                            ilog2_exact(cache->page_size), start_pos, n, d.sms,
                                            d.err, (cudaStream_t)stream));
}

ls_status ls_mla_replay_fwd_workspace(const ls_latent_cache* cache, int R, int H, int num_splits,
                                      size_t* bytes) {
  ls_status s = check_latent(cache);
  if (s != LS_OK) return s;
  if (!bytes) return LS_ERR_INVALID_ARG;
  LsSched sc;
  size_t po, pl;
  return mla_sched(cache, R, H, num_splits, &sc, &po, &pl, bytes);
}

ls_status ls_mla_replay_fwd(const ls_latent_cache* cache, const void* q, const void* lat_resp,
                            int R, int H, float softmax_scale, int num_splits, void* o,
                            float* lse, void* workspace, size_t workspace_bytes,
                            ls_stream_t stream) {
  ls_status s = check_latent(cache);
  if (s != LS_OK) return s;
  if (!isfinite(softmax_scale) || !(softmax_scale > 0.f)) return LS_ERR_INVALID_ARG;
  LsSched sc;
  size_t po, pl, total;
  if ((s = mla_sched(cache, R, H, num_splits, &sc, &po, &pl, &total)) != LS_OK) return s;
  if (R == 0) return LS_OK;
  const void* ptrs[] = {q, lat_resp, o, lse};
  for (const void* p : ptrs)
    if (!p || !aligned16(p)) return LS_ERR_INVALID_ARG;
  if (total > 0 && (!workspace || workspace_bytes < total || !aligned16(workspace)))
    return LS_ERR_WORKSPACE;
  DevInfo d;
  if ((s = dev_info(&d)) != LS_OK) return s;
  LsMlaArgs a;
  a.pool = cache->pool;
  a.page_table = cache->page_table;
  a.num_pages = cache->num_pages;
  a.ps_log2 = ilog2_exact(cache->page_size);
  a.P = cache->num_tokens;
  a.q = q;
  a.lat_resp = lat_resp;
  a.R = R;
  a.H = H;
  a.scale_log2 = softmax_scale * 1.4426950408889634f;
  a.o = o;
  a.lse = lse;
  a.part_o = reinterpret_cast<float*>(static_cast<char*>(workspace) + po);
  a.part_lse = reinterpret_cast<float*>(static_cast<char*>(workspace) + pl);
  a.err = d.err;
  return from_cuda(ls_launch_mla_fwd(a, sc, (cudaStream_t)stream));
}

ls_status ls_mla_replay_bwd_workspace(const ls_latent_cache* cache, int R, int H, int num_splits,
                                      size_t* bytes) {
  ls_status s = check_latent(cache);
  if (s != LS_OK) return s;
  if (!bytes) return LS_ERR_INVALID_ARG;
  LsSched sc;
  size_t a, b;
  int sms;
  return mla_bwd_sched(cache, R, H, num_splits, &sc, &a, &b, bytes, &sms);
}

ls_status ls_mla_replay_bwd(const ls_latent_cache* cache, const void* q, const void* lat_resp,
                            const void* o, const float* lse, const void* d_o, int R, int H,
                            float softmax_scale, int num_splits, float* dq, float* dlat,
                            void* workspace, size_t workspace_bytes, ls_stream_t stream) {
  ls_status s = check_latent(cache);
  if (s != LS_OK) return s;
  if (!isfinite(softmax_scale) || !(softmax_scale > 0.f)) return LS_ERR_INVALID_ARG;
  LsSched sc;
  size_t off_pdq, off_pdl, total;
  int sms;
  if ((s = mla_bwd_sched(cache, R, H, num_splits, &sc, &off_pdq, &off_pdl, &total, &sms)) != LS_OK)
    return s;
  if (R == 0) return LS_OK;
  const void* ptrs[] = {q, lat_resp, o, lse, d_o, dq, dlat};
  for (const void* p : ptrs)
    if (!p || !aligned16(p)) return LS_ERR_INVALID_ARG;
  if (!workspace || workspace_bytes < total || !aligned16(workspace)) return LS_ERR_WORKSPACE;
  DevInfo d;
  if ((s = dev_info(&d)) != LS_OK) return s;
  LsMlaBwdArgs a;
  a.pool = cache->pool;
  a.page_table = cache->page_table;
  a.num_pages = cache->num_pages;
  a.ps_log2 = ilog2_exact(cache->page_size);
  a.P = cache->num_tokens;
  a.q = q;
  a.lat_resp = lat_resp;
  a.o = o;
  a.lse = lse;
  a.d_o = d_o;
  a.R = R;
  a.H = H;
  a.scale = softmax_scale;
  a.scale_log2 = softmax_scale * 1.4426950408889634f;
  char* ws = static_cast<char*>(workspace);
  a.delta = reinterpret_cast<float*>(ws);
  a.dq = dq;
  a.dlat = dlat;
  a.part_dq = reinterpret_cast<float*>(ws + off_pdq);
  a.part_dlat = reinterpret_cast<float*>(ws + off_pdl);
  a.err = d.err;
  return from_cuda(ls_launch_mla_bwd(a, sc, sms, (cudaStream_t)stream));
}

ls_status ls_selftest_wait_timeout(ls_stream_t stream) {
  DevInfo d;
  ls_status s = dev_info(&d);
  if (s != LS_OK) return s;
  return from_cuda(ls_launch_wait_timeout(d.err, (cudaStream_t)stream));
}

ls_status ls_last_device_error(ls_stream_t stream) {
  DevInfo d;
  ls_status s = dev_info(&d);
  if (s != LS_OK) return s;
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return LS_ERR_CUDA;
  uint32_t v = 0;
  if (cudaMemcpy(&v, d.err, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess) return LS_ERR_CUDA;
  if (v == 0) return LS_OK;
  const uint32_t zero = 0;
  if (cudaMemcpy(d.err, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess)
    return LS_ERR_CUDA;
  return (v & LS_DEVERR_TIMEOUT) ? LS_ERR_TIMEOUT : LS_ERR_DEVICE_CHECK;
}

}  // extern "C"
