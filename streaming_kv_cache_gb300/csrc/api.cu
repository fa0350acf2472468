// C-ABI entry points of libskv: argument validation and kernel launches.
// Nothing here allocates device memory or synchronises the stream.
#include <stdint.h>
#include <string.h>

#include <atomic>

#include "common.cuh"
#include "kernels.h"
#include "skv.h"

namespace {

thread_local int g_last_cuda = 0;

int cuda_fail(cudaError_t e) {
  g_last_cuda = (int)e;
  return SKV_ERR_CUDA;
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

// 1 = sm_103 device, -1 = other device, 0 = not asked yet; cached per
// device ordinal (host threads may fill an entry at the same time: they
// store the same value, and the atomic makes that well defined).
std::atomic<int> g_dev_ok[64];

int check_device() {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (dev < 0 || dev >= 64) return SKV_ERR_UNSUPPORTED;
  int ok = g_dev_ok[dev].load(std::memory_order_relaxed);
  if (ok == 0) {
    int major = 0, minor = 0;
    if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess)
      return cuda_fail(e);
    if ((e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess)
      return cuda_fail(e);
    ok = (major == 10 && minor == 3) ? 1 : -1;
    g_dev_ok[dev].store(ok, std::memory_order_relaxed);
  }
  return ok == 1 ? SKV_OK : SKV_ERR_UNSUPPORTED;
}

int check_cache(const skv_cache* c) {
  if (!c) return SKV_ERR_INVALID;
  if (c->n_cache < 0 || c->n_view < 1 || c->n_frame < 1 || c->frame_len < 1 ||
      c->prefix_len < 0 || c->tail_cap < 0 || c->n_kv_head < 1)
    return SKV_ERR_INVALID;
  if (c->head_dim != 64 && c->head_dim != 128) return SKV_ERR_INVALID;
  const long long need = (long long)c->prefix_len +
                         (long long)c->n_view * c->n_frame * c->frame_len + c->tail_cap;
  if (need > 0x3FFFFFFFLL) return SKV_ERR_INVALID;
  if (c->row_cap < need || (c->row_cap & 7) != 0) return SKV_ERR_INVALID;
  if (c->rope_len < need) return SKV_ERR_INVALID;
  if (c->rope_mode != 0 && c->rope_mode != 1) return SKV_ERR_INVALID;
  if (c->n_cache == 0) return SKV_OK;  // nothing to touch: calls return early
  if (!c->k || !c->vt || !c->head || !c->rope || !c->status) return SKV_ERR_INVALID;
  if (!aligned16(c->k) || !aligned16(c->vt) || !aligned16(c->rope)) return SKV_ERR_INVALID;
  if (((uintptr_t)c->head & 3u) || ((uintptr_t)c->status & 3u)) return SKV_ERR_INVALID;
  return SKV_OK;
}

// The frame insert's arrival counters: only kv_stream_insert reads cache->sync.
int check_sync(const skv_cache* c) {
  if (c->n_cache == 0) return SKV_OK;
  if (!c->sync || ((uintptr_t)c->sync & 3u)) return SKV_ERR_INVALID;
  return SKV_OK;
}

// Shapes the tensor-core prefill kernel covers: its per-CTA tables hold the
// ring heads of at most kMaxViews views and at most kPrefillMaxKeyTiles
// 128-row key tiles per (cache, kv head), and output rows (token, head) are
// indexed in 32 bits.  Checked here so that a call outside them enqueues
// nothing (the tail prefill writes rows before it attends).
constexpr int kMaxViews = 64;
constexpr long long kPrefillMaxKeyTiles = 1024;
constexpr long long kPrefillKeyTile = 128;

int check_prefill_shape(const skv_cache* c, long long n_query, int n_q_head) {
  if (c->n_view > kMaxViews) return SKV_ERR_UNSUPPORTED;
  if ((c->row_cap + kPrefillKeyTile - 1) / kPrefillKeyTile > kPrefillMaxKeyTiles) return SKV_ERR_UNSUPPORTED;
  if ((long long)c->n_cache * n_query * n_q_head > 0x7FFFFFFFLL) return SKV_ERR_UNSUPPORTED;
  return SKV_OK;
}

}  // namespace

namespace skv {

// The argument checks kv_stream_insert makes, except those of cache->sync,
// without enqueueing anything; lets a caller validate before it enqueues
// work of its own.
int check_insert_args(const skv_cache* cache, const void* k_new, const void* v_new) {
  int rc = check_cache(cache);
  if (rc) return rc;
  if (cache->n_cache == 0) return SKV_OK;
  if (!k_new || !v_new || !aligned16(k_new) || !aligned16(v_new)) return SKV_ERR_INVALID;
  return check_device();
}

int record_cuda_error(cudaError_t e) { return cuda_fail(e); }

}  // namespace skv

extern "C" {

int skv_version(void) { return SKV_VERSION; }

const char* skv_status_string(int code) {
  switch (code) {
    case SKV_OK: return "ok";
    case SKV_ERR_INVALID: return "invalid argument (null/misaligned pointer or bad shape)";
    case SKV_ERR_UNSUPPORTED: return "unsupported (no sm_103 device current, or shape outside the kernels)";
    case SKV_ERR_CUDA: return "CUDA call failed (see skv_last_cuda_error)";
    case SKV_ERR_TOO_LARGE: return "n_cache * n_view exceeds the static scratch of kv_stream_insert_noalloc";
    case SKV_DEV_TIMEOUT: return "device: a bounded wait gave up";
    case SKV_DEV_BAD_HEAD: return "device: ring head outside [0, F)";
    case SKV_DEV_TAIL_OVERFLOW: return "device: tail_len + blk exceeds tail_cap";
    case SKV_DEV_BAD_TAIL: return "device: negative tail_len";
    default: return code > 0 ? "device: several status bits set" : "unknown status";
  }
}

int skv_last_cuda_error(void) { return g_last_cuda; }

int32_t skv_row_cap(int32_t P, int32_t V, int32_t F, int32_t T, int32_t tail_cap) {
  if (P < 0 || V < 1 || F < 1 || T < 1 || tail_cap < 0) return -1;
  const long long need = (long long)P + (long long)V * F * T + tail_cap;
  const long long cap = (need + 127) / 128 * 128;
  return cap > 0x3FFFFFFFLL ? -1 : (int32_t)cap;
}

int skv_build_rope_table(float* tab, int32_t n_pos, int32_t head_dim, double theta, void* stream) {
  if (!tab || n_pos < 1 || head_dim < 2 || (head_dim & 1) || !(theta > 0.0) || !aligned16(tab))
    return SKV_ERR_INVALID;
  int rc = check_device();
  if (rc) return rc;
  cudaError_t e = skv::launch_rope_table(tab, n_pos, head_dim, theta, (cudaStream_t)stream);
  return e == cudaSuccess ? SKV_OK : cuda_fail(e);
}

int skv_build_mrope_table(float* tab, int32_t n_pos, int32_t head_dim, double theta, int32_t P,
                          int32_t V, int32_t F, int32_t T, int32_t grid_w, uint64_t h_mask,
                          uint64_t w_mask, void* stream) {
  if (!tab || n_pos < 1 || head_dim < 2 || (head_dim & 1) || head_dim / 2 > 64 || !(theta > 0.0) ||
      !aligned16(tab))
    return SKV_ERR_INVALID;
  if (P < 0 || V < 1 || F < 1 || T < 1 || grid_w < 1 || T % grid_w || (h_mask & w_mask))
    return SKV_ERR_INVALID;
  if ((long long)P + (long long)V * F * T > 0x3FFFFFFFLL) return SKV_ERR_INVALID;
  int rc = check_device();
  if (rc) return rc;
  skv::MRopeGeom m{P, V, F, T, grid_w, h_mask, w_mask};
  cudaError_t e = skv::launch_mrope_table(tab, n_pos, head_dim, theta, m, (cudaStream_t)stream);
  return e == cudaSuccess ? SKV_OK : cuda_fail(e);
}

int kv_write_rows(const skv_cache* cache, int32_t row0, int32_t n_rows, const void* k_src,
                  const void* v_src, void* stream) {
  int rc = check_cache(cache);
  if (rc) return rc;
  if (row0 < 0 || n_rows < 0 || (long long)row0 + n_rows > cache->row_cap) return SKV_ERR_INVALID;
  if (n_rows == 0 || cache->n_cache == 0) return SKV_OK;
  if (!k_src || !v_src || !aligned16(k_src) || !aligned16(v_src)) return SKV_ERR_INVALID;
  if ((rc = check_device())) return rc;
  const skv::Geom g = skv::geom_of(*cache);
  cudaError_t e = skv::launch_write_rows(g, cache->k, cache->vt, k_src, v_src, 1, n_rows, 0, row0,
                                         cache->head, cache->sync, nullptr, cache->status,
                                         (cudaStream_t)stream);
  return e == cudaSuccess ? SKV_OK : cuda_fail(e);
}

int kv_stream_insert(const skv_cache* cache, const void* k_new, const void* v_new, void* stream) {
  int rc = check_cache(cache);
  if (rc) return rc;
  if ((rc = check_sync(cache))) return rc;
  if (cache->n_cache == 0) return SKV_OK;
  if (!k_new || !v_new || !aligned16(k_new) || !aligned16(v_new)) return SKV_ERR_INVALID;
  if ((rc = check_device())) return rc;
  const skv::Geom g = skv::geom_of(*cache);
  cudaError_t e = skv::launch_write_rows(g, cache->k, cache->vt, k_new, v_new, g.V, g.T, 1, 0,
                                         cache->head, cache->sync, nullptr, cache->status,
                                         (cudaStream_t)stream);
  return e == cudaSuccess ? SKV_OK : cuda_fail(e);
}

int stream_attn_prefill(const skv_cache* cache, int32_t n_q_head, const void* q_new, void* out,
                        float* lse, float sm_scale, void* stream) {
  int rc = check_cache(cache);
  if (rc) return rc;
  if (n_q_head < 1 || n_q_head % cache->n_kv_head) return SKV_ERR_INVALID;
  if (128 % (n_q_head / cache->n_kv_head)) return SKV_ERR_UNSUPPORTED;
  if ((rc = check_prefill_shape(cache, (long long)cache->n_view * cache->frame_len, n_q_head))) return rc;
  if (!(sm_scale > 0.f) || sm_scale != sm_scale) return SKV_ERR_INVALID;
  if (cache->n_cache == 0) return SKV_OK;
  if (!q_new || !out || !aligned16(q_new) || !aligned16(out)) return SKV_ERR_INVALID;
  if (lse && ((uintptr_t)lse & 3u)) return SKV_ERR_INVALID;
  if ((rc = check_device())) return rc;
  const skv::Geom g = skv::geom_of(*cache);
  skv::PrefillQuery qs{};
  qs.nf = 1;                        // the newest frame of every view
  qs.NQ = g.V * g.T;
  cudaError_t e = skv::launch_prefill_tc(g, n_q_head, qs, q_new, out, lse, cache->k, cache->vt, cache->rope,
                                         cache->head, sm_scale, cache->status, cache->wait_ns,
                                         (cudaStream_t)stream);
  return e == cudaSuccess ? SKV_OK : cuda_fail(e);
}

int stream_attn_prefill_insert(const skv_cache* cache, int32_t n_q_head, const void* k_new,
                               const void* v_new, const void* q_new, void* out, float* lse,
                               float sm_scale, void* stream) {
  int rc = check_cache(cache);
  if (rc) return rc;
  if ((rc = check_sync(cache))) return rc;
  if (n_q_head < 1 || n_q_head % cache->n_kv_head) return SKV_ERR_INVALID;
  if (128 % (n_q_head / cache->n_kv_head)) return SKV_ERR_UNSUPPORTED;
  if ((rc = check_prefill_shape(cache, (long long)cache->n_view * cache->frame_len, n_q_head))) return rc;
  if (!(sm_scale > 0.f) || sm_scale != sm_scale) return SKV_ERR_INVALID;
  if (cache->n_cache == 0) return SKV_OK;
  if (!k_new || !v_new || !q_new || !out) return SKV_ERR_INVALID;
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(q_new) || !aligned16(out)) return SKV_ERR_INVALID;
  if (lse && ((uintptr_t)lse & 3u)) return SKV_ERR_INVALID;
  if ((rc = check_device())) return rc;
  const skv::Geom g = skv::geom_of(*cache);
  cudaStream_t st = (cudaStream_t)stream;
  skv::PrefillQuery qs{};
  qs.nf = 1;
  qs.NQ = g.V * g.T;
  cudaError_t e;
  if (skv::prefill_insert_fusable(g)) {
    e = skv::launch_prefill_tc(g, n_q_head, qs, q_new, out, lse, cache->k, cache->vt, cache->rope, cache->head,
                               sm_scale, cache->status, cache->wait_ns, st, k_new, v_new, cache->sync);
  } else {
    // the two steps one after the other on the stream
    e = skv::launch_write_rows(g, cache->k, cache->vt, k_new, v_new, g.V, g.T, 1, 0, cache->head, cache->sync,
                               nullptr, cache->status, st);
    if (e == cudaSuccess)
      e = skv::launch_prefill_tc(g, n_q_head, qs, q_new, out, lse, cache->k, cache->vt, cache->rope, cache->head,
                                 sm_scale, cache->status, cache->wait_ns, st);
  }
  return e == cudaSuccess ? SKV_OK : cuda_fail(e);
}

int stream_attn_prefill_tail(const skv_cache* cache, int32_t n_q_head, int32_t n_tok,
                             const int32_t* tail_len, const void* q_tail, const void* k_tail,
                             const void* v_tail, void* out, float* lse, float sm_scale,
                             void* stream) {
  int rc = check_cache(cache);
  if (rc) return rc;
  if (n_q_head < 1 || n_q_head % cache->n_kv_head) return SKV_ERR_INVALID;
  if (n_tok < 1 || n_tok > cache->tail_cap) return SKV_ERR_INVALID;
  if (128 % (n_q_head / cache->n_kv_head)) return SKV_ERR_UNSUPPORTED;
  if ((rc = check_prefill_shape(cache, n_tok, n_q_head))) return rc;
  if (!(sm_scale > 0.f) || sm_scale != sm_scale) return SKV_ERR_INVALID;
  if (cache->n_cache == 0) return SKV_OK;
  if (!tail_len || !q_tail || !k_tail || !v_tail || !out) return SKV_ERR_INVALID;
  if (!aligned16(q_tail) || !aligned16(k_tail) || !aligned16(v_tail) || !aligned16(out))
    return SKV_ERR_INVALID;
  if (((uintptr_t)tail_len & 3u) || (lse && ((uintptr_t)lse & 3u))) return SKV_ERR_INVALID;
  if ((rc = check_device())) return rc;
  const skv::Geom g = skv::geom_of(*cache);
  cudaStream_t st = (cudaStream_t)stream;
  // the tokens' K/V into the tail, then their attention (same stream order)
  cudaError_t e = skv::launch_write_rows(g, cache->k, cache->vt, k_tail, v_tail, 1, n_tok, 2, 0,
                                         cache->head, cache->sync, tail_len, cache->status, st);
  if (e != cudaSuccess) return cuda_fail(e);
  skv::PrefillQuery qs{};
  qs.n_tail = n_tok;
  qs.tail_len = tail_len;
  qs.NQ = n_tok;
  e = skv::launch_prefill_tc(g, n_q_head, qs, q_tail, out, lse, cache->k, cache->vt, cache->rope, cache->head,
                             sm_scale, cache->status, cache->wait_ns, st);
  return e == cudaSuccess ? SKV_OK : cuda_fail(e);
}

int stream_attn_window(const skv_cache* cache, int32_t n_q_head, const void* q_win, void* out,
                       float* lse, float sm_scale, void* stream) {
  int rc = check_cache(cache);
  if (rc) return rc;
  if (n_q_head < 1 || n_q_head % cache->n_kv_head) return SKV_ERR_INVALID;
  if (128 % (n_q_head / cache->n_kv_head)) return SKV_ERR_UNSUPPORTED;
  if ((rc = check_prefill_shape(cache, (long long)cache->prefix_len +
                                           (long long)cache->n_view * cache->n_frame * cache->frame_len,
                                n_q_head)))
    return rc;
  if (!(sm_scale > 0.f) || sm_scale != sm_scale) return SKV_ERR_INVALID;
  if (cache->n_cache == 0) return SKV_OK;
  if (!q_win || !out || !aligned16(q_win) || !aligned16(out)) return SKV_ERR_INVALID;
  if (lse && ((uintptr_t)lse & 3u)) return SKV_ERR_INVALID;
  if ((rc = check_device())) return rc;
  const skv::Geom g = skv::geom_of(*cache);
  skv::PrefillQuery qs{};
  qs.nf = g.F;                      // every frame of every view, and the prefix
  qs.prefix = true;
  qs.NQ = g.n_visual();
  qs.q_view0 = g.P;
  cudaError_t e = skv::launch_prefill_tc(g, n_q_head, qs, q_win, out, lse, cache->k, cache->vt, cache->rope,
                                         cache->head, sm_scale, cache->status, cache->wait_ns,
                                         (cudaStream_t)stream);
  return e == cudaSuccess ? SKV_OK : cuda_fail(e);
}

size_t skv_verify_workspace_bytes(const skv_cache* cache, int32_t n_q_head, int32_t blk) {
  if (check_cache(cache) || n_q_head < 1 || n_q_head % cache->n_kv_head || blk < 1) return 0;
  return skv::verify_ws_bytes(skv::geom_of(*cache), n_q_head, blk);
}

int stream_attn_verify(const skv_cache* cache, int32_t n_q_head, int32_t blk,
                       const int32_t* tail_len, const void* q_blk, const void* k_blk,
                       const void* v_blk, void* out, const int32_t* target_ids,
                       const int32_t* draft_ids, int32_t* accept_len, int32_t* next_token,
                       void* ws, size_t ws_bytes, float sm_scale, void* stream) {
  int rc = check_cache(cache);
  if (rc) return rc;
  if (n_q_head < 1 || n_q_head % cache->n_kv_head) return SKV_ERR_INVALID;
  if (blk < 1 || blk > cache->tail_cap) return SKV_ERR_INVALID;
  {
    // block rows are taken 64 (more than 64: 128) at a time per kv head, whole tokens each
    const int G = n_q_head / cache->n_kv_head;
    if (G > 64 || ((long long)blk * G > 128 && 128 % G)) return SKV_ERR_UNSUPPORTED;
  }
  if (!(sm_scale > 0.f) || sm_scale != sm_scale) return SKV_ERR_INVALID;
  if (cache->n_cache == 0) return SKV_OK;
  if (!tail_len || !q_blk || !k_blk || !v_blk || !out) return SKV_ERR_INVALID;
  if (!aligned16(q_blk) || !aligned16(k_blk) || !aligned16(v_blk) || !aligned16(out))
    return SKV_ERR_INVALID;
  const bool ids = target_ids && draft_ids;
  if (ids && (!accept_len || !next_token)) return SKV_ERR_INVALID;
  const size_t ws_need = skv_verify_workspace_bytes(cache, n_q_head, blk);
  if (ws_bytes < ws_need || (ws_need && (!ws || !aligned16(ws)))) return SKV_ERR_INVALID;
  if (cache->n_view > kMaxViews) return SKV_ERR_UNSUPPORTED;   // the verify kernel keeps the ring heads on chip
  if ((rc = check_device())) return rc;
  const skv::Geom g = skv::geom_of(*cache);
  cudaStream_t st = (cudaStream_t)stream;
  // the block's K/V into the tail, and the accept length from the ids
  cudaError_t e = skv::launch_write_rows(g, cache->k, cache->vt, k_blk, v_blk, 1, blk, 2, 0,
                                         cache->head, cache->sync, tail_len, cache->status, st,
                                         ids ? target_ids : nullptr, ids ? draft_ids : nullptr,
                                         ids ? accept_len : nullptr, ids ? next_token : nullptr);
  if (e != cudaSuccess) return cuda_fail(e);
  e = skv::launch_verify_tc(g, n_q_head, blk, tail_len, q_blk, out, cache->k, cache->vt, cache->rope,
                            cache->head, ws, ws_bytes, sm_scale, cache->status, cache->wait_ns, st);
  if (e != cudaSuccess) return cuda_fail(e);
  return SKV_OK;
}

}  // extern "C"
