// Host side of the C ABI (include/qevict.h): validation, budget arithmetic, arena layout,
// schedule checks and kernel launches.  The library never allocates device memory.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <new>
#include <vector>

#include "cache_dev.cuh"
#include "common.cuh"
#include "diag_dev.cuh"
#include "qevict.h"

namespace qv {
cudaError_t launch_init(const CacheDev &C, cudaStream_t s);
cudaError_t launch_wait_selftest(const CacheDev &C, cudaStream_t s);
cudaError_t launch_route(const CacheDev &C, int unit0, int n_units, const __nv_bfloat16 *kp,
                         const __nv_bfloat16 *vp, int layer, int mig_blocks, cudaStream_t s);
cudaError_t launch_prefill_setup(const CacheDev &C, const __nv_bfloat16 *kp, const __nv_bfloat16 *vp, int layer,
                                 const float *s0, cudaStream_t s);
cudaError_t launch_prefill_scores(const CacheDev &C, const __nv_bfloat16 *q, const __nv_bfloat16 *k, float *s0,
                                  cudaStream_t s);
cudaError_t launch_decode(const CacheDev &C, const DecodeIO &io, cudaStream_t s);
cudaError_t launch_flush(const CacheDev &C, cudaStream_t s);
int route_max_windows();
cudaError_t launch_diag_collect(const CacheDev &R, const DiagDev &Dg, cudaStream_t s);
cudaError_t launch_diag_event(const CacheDev &P, const CacheDev &R, const DiagDev &Dg, int e, cudaStream_t s);
}  // namespace qv

struct qevict_cache {
  qevict_config cfg;
  qevict_budget_info bud;
  qevict_layout lay;
  qv::CacheDev dev;
  int64_t off_s0buf;            // fp32 [B][prompt windows] scratch for computed prefill scores
  std::vector<int> t_host;      // tokens cached per layer (host mirror)
  std::vector<int> prefilled;
  int routes_done;
  int last_decode_layer;        // layer of the last decode enqueued, -1 after any other call
  int rope_set;                 // rope = 1: the RoPE table has been copied in
};

namespace {

constexpr int D = 128;

int64_t align256(int64_t x) { return (x + 255) & ~int64_t(255); }

int device_sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 152;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
    cudaGetLastError();
    return 152;
  }
  return n;
}

qevict_status check_config(const qevict_config *c) {
  if (!c) return QEVICT_EINVAL;
  if (c->batch < 1 || c->n_layers < 1 || c->h_kv < 1 || c->h_q < c->h_kv || c->h_q % c->h_kv) return QEVICT_EINVAL;
  const int G = c->h_q / c->h_kv;
  if (G != 1 && G != 2 && G != 4 && G != 8) return QEVICT_EINVAL;
  if (c->d_head != D) return QEVICT_EINVAL;
  if (!((c->window == 32 && c->bits == 2) || (c->window == 64 && c->bits == 4))) return QEVICT_EINVAL;
  if (c->ranker < 0 || c->ranker > 3 || c->no_promotion < 0 || c->no_promotion > 1) return QEVICT_EINVAL;
  if (!(c->decay >= 0.f && c->decay <= 1.f) || !(c->pnorm == 0.f || c->pnorm >= 1.f)) return QEVICT_EINVAL;
  if (c->rope < 0 || c->rope > 1 || c->reserved0 != 0) return QEVICT_EINVAL;
  if (c->n_sink < 1 || c->n_sink > 16 || c->n_recent < c->window || c->omega < 1 ||
      c->omega > 256)
    return QEVICT_EINVAL;
  if (c->q_den < 1 || c->q_num < 0 || c->q_num > c->q_den) return QEVICT_EINVAL;
  if (c->b_total < 0 || (c->b_total == 0 && (c->budget_den < 1 || c->budget_num < 0))) return QEVICT_EINVAL;
  if (c->prompt_len <= c->n_sink || c->max_len < c->prompt_len) return QEVICT_EINVAL;
  return QEVICT_OK;
}

qevict_status compute_budget(const qevict_config *c, qevict_budget_info *b) {
  qevict_status st = check_config(c);
  if (st != QEVICT_OK) return st;
  const int64_t c_tok = 4LL * c->h_kv * c->d_head;            // bf16 K + V of one token
  const int64_t tok_bytes = c_tok + 4;                          // + int32 position
  b->full_bytes = c_tok * c->prompt_len;                        // Eq. (7) per layer and sequence
  if (c->b_total) {
    b->b_total = c->b_total;
  } else {   // the product may pass 2^63 for extreme fractions: clamp in 128 bits
    const __int128 bt = (__int128)b->full_bytes * c->budget_num / c->budget_den;
    b->b_total = bt > (__int128)INT64_MAX ? INT64_MAX : (int64_t)bt;
  }
  b->b_sink = c->n_sink * tok_bytes;
  b->b_local = (int64_t)(c->n_recent + c->window) * tok_bytes;
  b->b_hist = b->b_total - b->b_sink - b->b_local;
  b->payload = 2LL * c->h_kv * c->window * c->d_head * c->bits / 8 + 4LL * c->h_kv * c->d_head +
               4LL * c->h_kv * c->window;
  b->m_q = b->payload + 4LL * c->window + 16;
  b->m_f = (int64_t)c->window * c_tok + 4LL * c->window + 8 + b->payload;
  b->n_windows = (c->max_len - c->n_sink + c->window - 1) / c->window;
  b->ring_windows = (c->n_recent + c->window + c->omega + c->window - 1) / c->window;
  if (b->b_hist < 0) {
    b->k_f = b->k_q = 0;
    return QEVICT_EBUDGET;
  }
  // Eq. (3) with q = q_num / q_den in exact integers (128-bit products)
  const __int128 nf = (__int128)(c->q_den - c->q_num) * b->b_hist, df = (__int128)c->q_den * b->m_f;
  const __int128 nq = (__int128)c->q_num * b->b_hist, dq = (__int128)c->q_den * b->m_q;
  const __int128 ikf = nf / df, ikq = nq / dq;
  b->k_f = ikf > 0x3fffffff ? 0x3fffffff : (int32_t)ikf;
  b->k_q = ikq > 0x3fffffff ? 0x3fffffff : (int32_t)ikq;
  if (b->n_windows > qv::route_max_windows()) return QEVICT_EINVAL;
  return QEVICT_OK;
}

struct Plan {
  qevict_layout lay;
  qv::CacheDev dev;
  int64_t off_s0buf;
};

void make_plan(const qevict_config *c, const qevict_budget_info *b, Plan *p) {
  std::memset(p, 0, sizeof(*p));
  const int N = b->n_windows, R = b->ring_windows, W = c->window;
  const int kf_cap = std::min(b->k_f, N), kq_cap = std::min(b->k_q, N);
  const int lp_cap = (int)std::min<int64_t>((int64_t)b->k_f + b->k_q, N);
  const int64_t qb = b->payload / c->h_kv;
  const int U = c->batch * c->n_layers;
  int64_t off = 0;
  auto region = [&](int64_t per_unit, int64_t &o, int64_t &st) {
    st = align256(std::max<int64_t>(per_unit, 16));
    o = off;
    off += st * U;
  };
  qevict_layout &L = p->lay;
  region(2LL * c->h_kv * c->n_sink * D * 2, L.off_sink, L.stride_sink);
  region(2LL * c->h_kv * R * W * D * 2, L.off_ring, L.stride_ring);
  region((int64_t)kf_cap * c->h_kv * 2 * W * D * 2, L.off_fpool, L.stride_fpool);
  region((int64_t)lp_cap * c->h_kv * qb, L.off_ledger, L.stride_ledger);
  region(4LL * c->h_kv * N, L.off_score, L.stride_score);
  region(N, L.off_state, L.stride_state);
  region(4LL * N, L.off_fslot, L.stride_fslot);
  region(4LL * N, L.off_lslot, L.stride_lslot);
  region(8LL * kf_cap, L.off_ftab, L.stride_ftab);
  region(8LL * kq_cap, L.off_qtab, L.stride_qtab);
  region(4LL * qv::META_INTS, L.off_meta, L.stride_meta);
  region(4LL * N, L.off_agg, L.stride_agg);
  qv::CacheDev &C = p->dev;
  region(16LL * N, C.off_qtask, C.st_qtask);
  region(16LL * N, C.off_mtask, C.st_mtask);
  // decode split-K partitions: at most one CTA per SM for the whole batch (a decode CTA fills an SM, so a
  // grid above the SM count would run a second, nearly empty wave)
  const int sms = device_sm_count();
  const int max_items = 1 + (R + 1) + kf_cap + kq_cap;
  int n_split = sms / (c->batch * c->h_kv);
  n_split = std::max(1, std::min(n_split, std::max(1, max_items / 4)));
  auto global = [&](int64_t bytes) {
    const int64_t o = off;
    off += align256(std::max<int64_t>(bytes, 16));
    return o;
  };
  C.off_counters = global(8LL * qv::N_COUNTERS * U);
  C.off_status = global(256);
  C.off_splitctr = global(4LL * c->n_layers * c->batch * c->h_kv);
  C.off_thead = global(4LL * c->n_layers * c->batch * c->h_kv);
  C.st_part_layer = align256(4LL * c->batch * c->h_kv * n_split * qv::PART_FLOATS);
  C.off_part = global(C.st_part_layer * c->n_layers);
  // per-step window log-masses: one record of G floats (the KV head's query heads) per item
  C.st_mu_layer = align256(4LL * c->batch * c->h_kv * c->omega * max_items * (c->h_q / c->h_kv));
  C.off_mu = global(C.st_mu_layer * c->n_layers);
  C.st_mstat_layer = align256(4LL * c->batch * c->h_kv * c->omega * 16);
  C.off_mstat = global(C.st_mstat_layer * c->n_layers);
  C.off_flushctr = global(4LL * c->n_layers * c->batch);
  C.off_rowstat = global(4LL * c->batch * c->h_q * c->prompt_len);
  C.off_colsum = global(4LL * c->batch * c->h_q * c->prompt_len);
  const int npw = (c->prompt_len - c->n_sink + W - 1) / W;
  p->off_s0buf = global(4LL * c->batch * npw);
  // rope = 1: max_len rows of the caller's table; the decode kernel reads rows 0..31 in any case
  C.off_rope = L.off_rope = global(c->rope ? 512LL * std::max(c->max_len, 32) : 16);
  L.qblock = qb;
  L.arena_bytes = off;
  L.n_split = n_split;
  C.off_sink = L.off_sink;     C.st_sink = L.stride_sink;
  C.off_ring = L.off_ring;     C.st_ring = L.stride_ring;
  C.off_fpool = L.off_fpool;   C.st_fpool = L.stride_fpool;
  C.off_ledger = L.off_ledger; C.st_ledger = L.stride_ledger;
  C.off_score = L.off_score;   C.st_score = L.stride_score;
  C.off_state = L.off_state;   C.st_state = L.stride_state;
  C.off_fslot = L.off_fslot;   C.st_fslot = L.stride_fslot;
  C.off_lslot = L.off_lslot;   C.st_lslot = L.stride_lslot;
  C.off_ftab = L.off_ftab;     C.st_ftab = L.stride_ftab;
  C.off_qtab = L.off_qtab;     C.st_qtab = L.stride_qtab;
  C.off_meta = L.off_meta;     C.st_meta = L.stride_meta;
  C.off_agg = L.off_agg;       C.st_agg = L.stride_agg;
  C.B = c->batch;
  C.L = c->n_layers;
  C.h_q = c->h_q;
  C.h_kv = c->h_kv;
  C.G = c->h_q / c->h_kv;
  C.n_sink = c->n_sink;
  C.n_recent = c->n_recent;
  C.W = W;
  C.bits = c->bits;
  C.omega = c->omega;
  C.k_f = b->k_f;
  C.k_q = b->k_q;
  C.n_windows = N;
  C.ring_windows = R;
  C.n_split = n_split;
  C.max_items = max_items;
  C.prompt_len = c->prompt_len;
  C.max_len = c->max_len;
  C.ranker = c->ranker;
  C.no_promotion = c->no_promotion;
  C.decay = c->decay == 0.f ? 0.99f : c->decay;
  C.pnorm = c->pnorm == 0.f ? 3.0f : c->pnorm;
  C.rope = c->rope;
  C.slot_cap = -1;
}

qevict_status cuda_status(cudaError_t e) { return e == cudaSuccess ? QEVICT_OK : QEVICT_ECUDA; }

}  // namespace

extern "C" {

qevict_status qevict_budget(const qevict_config *cfg, qevict_budget_info *out) {
  if (!out) return QEVICT_EINVAL;
  return compute_budget(cfg, out);
}

qevict_status qevict_cache_bytes(const qevict_config *cfg, size_t *bytes) {
  if (!bytes) return QEVICT_EINVAL;
  qevict_budget_info b;
  qevict_status st = compute_budget(cfg, &b);
  if (st != QEVICT_OK) return st;
  Plan p;
  make_plan(cfg, &b, &p);
  *bytes = (size_t)p.lay.arena_bytes;
  return QEVICT_OK;
}

qevict_status qevict_init_cache(const qevict_config *cfg, void *d_arena, size_t bytes, qevict_stream_t stream,
                                qevict_cache **out) {
  if (!out || !d_arena || ((uintptr_t)d_arena & 255)) return QEVICT_EINVAL;
  qevict_budget_info b;
  qevict_status st = compute_budget(cfg, &b);
  if (st != QEVICT_OK) return st;
  Plan p;
  make_plan(cfg, &b, &p);
  if ((int64_t)bytes < p.lay.arena_bytes) return QEVICT_ENOMEM;
  qevict_cache *c = new (std::nothrow) qevict_cache();
  if (!c) return QEVICT_ENOMEM;
  c->cfg = *cfg;
  c->bud = b;
  c->lay = p.lay;
  c->dev = p.dev;
  c->dev.arena = static_cast<uint8_t *>(d_arena);
  c->dev.status_word = reinterpret_cast<int *>(c->dev.arena + c->dev.off_status);
  c->off_s0buf = p.off_s0buf;
  c->t_host.assign(cfg->n_layers, 0);
  c->prefilled.assign(cfg->n_layers, 0);
  c->routes_done = 0;
  c->last_decode_layer = -1;
  c->rope_set = 0;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemsetAsync(d_arena, 0, (size_t)p.lay.arena_bytes, s);
  if (e == cudaSuccess) e = qv::launch_init(c->dev, s);
  if (e != cudaSuccess) {
    delete c;
    return QEVICT_ECUDA;
  }
  *out = c;
  return QEVICT_OK;
}

qevict_status qevict_get_layout(const qevict_cache *cache, qevict_layout *out) {
  if (!cache || !out) return QEVICT_EINVAL;
  *out = cache->lay;
  return QEVICT_OK;
}

qevict_status qevict_set_rope_table(qevict_cache *cache, const float *d_table, int64_t rows, qevict_stream_t stream) {
  if (!cache || !d_table || !cache->cfg.rope || rows < cache->cfg.max_len) return QEVICT_EINVAL;
  for (int l = 0; l < cache->cfg.n_layers; ++l)
    if (cache->prefilled[l]) return QEVICT_ESCHEDULE;
  if (cudaMemcpyAsync(cache->dev.arena + cache->dev.off_rope, d_table, 512 * (size_t)cache->cfg.max_len,
                      cudaMemcpyDeviceToDevice, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return QEVICT_ECUDA;
  cache->rope_set = 1;
  return QEVICT_OK;
}

qevict_status qevict_prefill_scores(const qevict_cache *cache, const void *q_prompt, const void *k_prompt,
                                    float *s0_out, qevict_stream_t stream) {
  if (!cache || !q_prompt || !k_prompt || !s0_out || (((uintptr_t)q_prompt | (uintptr_t)k_prompt) & 15))
    return QEVICT_EINVAL;
  return cuda_status(qv::launch_prefill_scores(cache->dev, static_cast<const __nv_bfloat16 *>(q_prompt),
                                               static_cast<const __nv_bfloat16 *>(k_prompt), s0_out,
                                               reinterpret_cast<cudaStream_t>(stream)));
}

qevict_status qevict_prefill_route(qevict_cache *cache, int32_t layer, const void *k_prompt, const void *v_prompt,
                                   const float *s0, const void *q_prompt, qevict_stream_t stream) {
  if (!cache || layer < 0 || layer >= cache->cfg.n_layers || !k_prompt || !v_prompt) return QEVICT_EINVAL;
  if ((((uintptr_t)k_prompt | (uintptr_t)v_prompt) & 1) || ((uintptr_t)s0 & 3)) return QEVICT_EINVAL;
  if (!s0 && (!q_prompt || (((uintptr_t)q_prompt | (uintptr_t)k_prompt) & 15))) return QEVICT_EINVAL;
  if (cache->prefilled[layer] || (cache->cfg.rope && !cache->rope_set)) return QEVICT_ESCHEDULE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const auto *kp = static_cast<const __nv_bfloat16 *>(k_prompt);
  const auto *vp = static_cast<const __nv_bfloat16 *>(v_prompt);
  if (!s0) {
    float *buf = reinterpret_cast<float *>(cache->dev.arena + cache->off_s0buf);
    cudaError_t e = qv::launch_prefill_scores(cache->dev, static_cast<const __nv_bfloat16 *>(q_prompt), kp, buf, s);
    if (e != cudaSuccess) return QEVICT_ECUDA;
    s0 = buf;
  }
  cudaError_t e = qv::launch_prefill_setup(cache->dev, kp, vp, layer, s0, s);
  // the prompt's windows all migrate at once: about four migration CTAs per SM over the batch
  const int mig_blocks = std::max(8, 4 * device_sm_count() / cache->cfg.batch);
  if (e == cudaSuccess)
    e = qv::launch_route(cache->dev, layer * cache->cfg.batch, cache->cfg.batch, kp, vp, layer, mig_blocks, s);
  if (e != cudaSuccess) return QEVICT_ECUDA;
  cache->prefilled[layer] = 1;
  cache->t_host[layer] = cache->cfg.prompt_len;
  cache->last_decode_layer = -1;
  return QEVICT_OK;
}

qevict_status qevict_decode_step(qevict_cache *cache, int32_t layer, const void *q, const void *k_new,
                                 const void *v_new, void *out, qevict_stream_t stream) {
  if (!cache || layer < 0 || layer >= cache->cfg.n_layers || !q || !k_new || !v_new || !out) return QEVICT_EINVAL;
  // q and k_new are read as bf16 pairs, v_new and out element by element
  if ((((uintptr_t)q | (uintptr_t)k_new) & 3) || (((uintptr_t)v_new | (uintptr_t)out) & 1)) return QEVICT_EINVAL;
  if (!cache->prefilled[layer]) return QEVICT_ESCHEDULE;
  const int T = cache->t_host[layer];
  if (T >= cache->cfg.max_len) return QEVICT_ESCHEDULE;
  // a routing event is due every omega decode steps; the recent ring holds no more than that
  if (T - cache->cfg.prompt_len >= (cache->routes_done + 1) * cache->cfg.omega) return QEVICT_ESCHEDULE;
  qv::DecodeIO io;
  io.q = static_cast<const __nv_bfloat16 *>(q);
  io.k_new = static_cast<const __nv_bfloat16 *>(k_new);
  io.v_new = static_cast<const __nv_bfloat16 *>(v_new);
  io.out = static_cast<__nv_bfloat16 *>(out);
  io.layer = layer;
  io.scale_log2 = 1.4426950408889634f / std::sqrt((float)D);
  io.inv_hq = 1.0f / (float)cache->cfg.h_q;
  io.wait_first = (cache->last_decode_layer == layer) ? 1 : 0;
  cudaError_t e = qv::launch_decode(cache->dev, io, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return QEVICT_ECUDA;
  cache->last_decode_layer = layer;
  cache->t_host[layer] = T + 1;
  return QEVICT_OK;
}

static qevict_status route_due(const qevict_cache *cache) {
  const int due = cache->cfg.prompt_len + (cache->routes_done + 1) * cache->cfg.omega;
  for (int l = 0; l < cache->cfg.n_layers; ++l)
    if (!cache->prefilled[l] || cache->t_host[l] != due) return QEVICT_ESCHEDULE;
  return QEVICT_OK;
}

qevict_status qevict_route(qevict_cache *cache, qevict_stream_t stream) {
  if (!cache) return QEVICT_EINVAL;
  if (route_due(cache) != QEVICT_OK) return QEVICT_ESCHEDULE;
  cudaError_t e = qv::launch_flush(cache->dev, reinterpret_cast<cudaStream_t>(stream));
  if (e == cudaSuccess)
    e = qv::launch_route(cache->dev, 0, cache->cfg.batch * cache->cfg.n_layers, nullptr, nullptr, 0, 8,
                         reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return QEVICT_ECUDA;
  cache->routes_done += 1;
  cache->last_decode_layer = -1;
  return QEVICT_OK;
}

qevict_status qevict_flush_scores(qevict_cache *cache, qevict_stream_t stream) {
  if (!cache) return QEVICT_EINVAL;
  for (int l = 0; l < cache->cfg.n_layers; ++l)
    if (!cache->prefilled[l]) return QEVICT_ESCHEDULE;
  if (qv::launch_flush(cache->dev, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return QEVICT_ECUDA;
  cache->last_decode_layer = -1;
  return QEVICT_OK;
}

static qevict_status read_status(qevict_cache *cache, cudaStream_t s) {
  int st = 0;
  if (cudaMemcpyAsync(&st, cache->dev.status_word, sizeof(int), cudaMemcpyDeviceToHost, s) !=
          cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return QEVICT_ECUDA;
  return st ? QEVICT_EDEVICE : QEVICT_OK;
}

qevict_status qevict_read_counters(qevict_cache *cache, int64_t *host7, qevict_stream_t stream) {
  if (!cache || !host7) return QEVICT_EINVAL;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int U = cache->cfg.batch * cache->cfg.n_layers;
  std::vector<long long> buf((size_t)U * qv::N_COUNTERS);
  if (cudaMemcpyAsync(buf.data(), cache->dev.arena + cache->dev.off_counters, buf.size() * sizeof(long long),
                      cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return QEVICT_ECUDA;
  qevict_status st = read_status(cache, s);
  for (int k = 0; k < 7; ++k) {
    long long t = 0;
    for (int u = 0; u < U; ++u) t += buf[(size_t)u * qv::N_COUNTERS + k];
    host7[k] = t;
  }
  return st;
}

qevict_status qevict_read_status(const qevict_cache *cache, int32_t *host_word, qevict_stream_t stream) {
  if (!cache || !host_word) return QEVICT_EINVAL;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(host_word, cache->dev.status_word, sizeof(int32_t), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return QEVICT_ECUDA;
  return QEVICT_OK;
}

qevict_status qevict_check(qevict_cache *cache, qevict_stream_t stream) {
  if (!cache) return QEVICT_EINVAL;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int L = cache->cfg.n_layers;
  std::vector<int> m((size_t)L * qv::META_INTS);
  for (int l = 0; l < L; ++l)
    if (cudaMemcpyAsync(&m[(size_t)l * qv::META_INTS],
                        cache->dev.arena + cache->dev.off_meta + cache->dev.st_meta * (int64_t)(l * cache->cfg.batch),
                        4 * qv::META_INTS, cudaMemcpyDeviceToHost, s) != cudaSuccess)
      return QEVICT_ECUDA;
  qevict_status st = read_status(cache, s);
  if (st == QEVICT_ECUDA) return st;
  for (int l = 0; l < L; ++l)
    if (cache->prefilled[l]) {
      cache->t_host[l] = m[(size_t)l * qv::META_INTS + qv::M_T];
      cache->routes_done = m[(size_t)l * qv::META_INTS + qv::M_NEVENT];
    }
  return st;
}

qevict_status qevict_debug_cap_free_slots(qevict_cache *cache, int32_t cap) {
  if (!cache || cap < -1) return QEVICT_EINVAL;
  cache->dev.slot_cap = cap;
  return QEVICT_OK;
}

qevict_status qevict_selftest_wait(qevict_cache *cache, qevict_stream_t stream) {
  if (!cache) return QEVICT_EINVAL;
  return qv::launch_wait_selftest(cache->dev, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? QEVICT_OK
                                                                                                       : QEVICT_ECUDA;
}

qevict_status qevict_get_tuple(const qevict_cache *cache, int32_t layer, int32_t seq, qevict_tuple *out) {
  if (!cache || !out || layer < 0 || layer >= cache->cfg.n_layers || seq < 0 || seq >= cache->cfg.batch)
    return QEVICT_EINVAL;
  const qv::CacheDev &C = cache->dev;
  const int u = layer * cache->cfg.batch + seq;
  out->sink = C.at<uint8_t>(C.off_sink, C.st_sink, u);
  out->ring = C.at<uint8_t>(C.off_ring, C.st_ring, u);
  out->fpool = C.at<uint8_t>(C.off_fpool, C.st_fpool, u);
  out->ledger = C.at<uint8_t>(C.off_ledger, C.st_ledger, u);
  out->score = C.at<float>(C.off_score, C.st_score, u);
  out->state = C.at<uint8_t>(C.off_state, C.st_state, u);
  out->f_slot = C.at<int32_t>(C.off_fslot, C.st_fslot, u);
  out->l_slot = C.at<int32_t>(C.off_lslot, C.st_lslot, u);
  out->f_table = C.at<int32_t>(C.off_ftab, C.st_ftab, u);
  out->q_table = C.at<int32_t>(C.off_qtab, C.st_qtab, u);
  out->meta = C.at<int32_t>(C.off_meta, C.st_meta, u);
  return QEVICT_OK;
}

namespace {
struct ExportHeader {
  char magic[8];
  int64_t arena_bytes;
  qevict_config cfg;
};
constexpr char kExportMagic[8] = {'Q', 'E', 'V', 'I', 'C', 'T', 'S', '1'};
}  // namespace

qevict_status qevict_export_bytes(const qevict_cache *cache, size_t *bytes) {
  if (!cache || !bytes) return QEVICT_EINVAL;
  *bytes = sizeof(ExportHeader) + (size_t)cache->lay.arena_bytes;
  return QEVICT_OK;
}

qevict_status qevict_export_state(const qevict_cache *cache, void *host_buf, size_t bytes, qevict_stream_t stream) {
  if (!cache || !host_buf) return QEVICT_EINVAL;
  if (bytes < sizeof(ExportHeader) + (size_t)cache->lay.arena_bytes) return QEVICT_ENOMEM;
  ExportHeader h;
  std::memset(&h, 0, sizeof(h));
  std::memcpy(h.magic, kExportMagic, sizeof(h.magic));
  h.arena_bytes = cache->lay.arena_bytes;
  h.cfg = cache->cfg;
  std::memcpy(host_buf, &h, sizeof(h));
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(static_cast<uint8_t *>(host_buf) + sizeof(h), cache->dev.arena, (size_t)h.arena_bytes,
                      cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return QEVICT_ECUDA;
  return QEVICT_OK;
}

qevict_status qevict_import_state(qevict_cache *cache, const void *host_buf, size_t bytes, qevict_stream_t stream) {
  if (!cache || !host_buf || bytes < sizeof(ExportHeader)) return QEVICT_EINVAL;
  ExportHeader h;
  std::memcpy(&h, host_buf, sizeof(h));
  if (std::memcmp(h.magic, kExportMagic, sizeof(h.magic)) != 0 || h.arena_bytes != cache->lay.arena_bytes ||
      std::memcmp(&h.cfg, &cache->cfg, sizeof(qevict_config)) != 0 ||
      bytes < sizeof(ExportHeader) + (size_t)h.arena_bytes)
    return QEVICT_EINVAL;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(cache->dev.arena, static_cast<const uint8_t *>(host_buf) + sizeof(h), (size_t)h.arena_bytes,
                      cudaMemcpyHostToDevice, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return QEVICT_ECUDA;
  // host bookkeeping follows the imported meta records: a layer is prefilled once T > 0
  const int L = cache->cfg.n_layers;
  const uint8_t *arena = static_cast<const uint8_t *>(host_buf) + sizeof(h);
  for (int l = 0; l < L; ++l) {
    int32_t m[qv::META_INTS];
    std::memcpy(m, arena + cache->dev.off_meta + cache->dev.st_meta * (int64_t)(l * cache->cfg.batch), sizeof(m));
    cache->prefilled[l] = m[qv::M_T] > 0 ? 1 : 0;
    cache->t_host[l] = m[qv::M_T];
    if (m[qv::M_T] > 0) cache->routes_done = m[qv::M_NEVENT];
    // a prefilled rope = 1 cache had its table set, and the table travels inside the arena
    if (m[qv::M_T] > 0 && cache->cfg.rope) cache->rope_set = 1;
  }
  cache->last_decode_layer = -1;
  return QEVICT_OK;
}

// ----------------------------------------------------------------------------- routing diagnostics

struct qevict_diag {
  qevict_cache *policy, *fullkv;
  qv::DiagDev dev;
  int events;
};

namespace {

qevict_status diag_check(const qevict_cache *P, const qevict_cache *R, const qevict_diag_config *dc, int *horizon,
                         int *lir_m) {
  if (!P || !R || P == R || !dc) return QEVICT_EINVAL;
  const qevict_config &a = P->cfg, &b = R->cfg;
  if (a.batch != b.batch || a.n_layers != b.n_layers || a.h_q != b.h_q || a.h_kv != b.h_kv || a.d_head != b.d_head ||
      a.n_sink != b.n_sink || a.n_recent != b.n_recent || a.window != b.window || a.bits != b.bits ||
      a.omega != b.omega || a.prompt_len != b.prompt_len || a.max_len != b.max_len || a.rope != b.rope)
    return QEVICT_EINVAL;
  if (a.ranker != 0 || R->bud.k_f < R->bud.n_windows) return QEVICT_EINVAL;
  const int H = dc->horizon ? dc->horizon : 32, m = dc->lir_m ? dc->lir_m : 3;
  if (H < a.omega || H % a.omega || H / a.omega > qv::DG_MAX_OPEN || a.omega > qv::DG_MAX_OMEGA || m < 1 ||
      dc->horizon < 0 || dc->lir_m < 0)
    return QEVICT_EINVAL;
  *horizon = H;
  *lir_m = m;
  return QEVICT_OK;
}

qv::DiagDev diag_plan(const qevict_cache *P, int horizon, int lir_m, int64_t *bytes) {
  qv::DiagDev d = {};
  d.U = P->cfg.batch * P->cfg.n_layers;
  d.N = P->bud.n_windows;
  d.Hq = P->cfg.h_q;
  d.n_open = horizon / P->cfg.omega;
  d.horizon = horizon;
  d.lir_m = lir_m;
  int64_t off = 0;
  auto take = [&](int64_t n) {
    const int64_t o = off;
    off += align256(std::max<int64_t>(n, 16));
    return o;
  };
  const int64_t UN = (int64_t)d.U * d.N;
  d.off_evict = take(4 * UN);   // the three -1 regions first: one memset covers them
  d.off_since = take(4 * UN);
  d.off_evT = take(4LL * d.U * qv::DG_MAX_OPEN);
  d.off_evId = take(4LL * d.U * qv::DG_MAX_OPEN);
  d.off_runpol = take(4 * UN);
  d.off_runorc = take(4 * UN);
  d.off_xpol = take(4 * UN);
  d.off_xorc = take(4 * UN);
  d.off_ret = take(UN);
  d.off_fnum = take(8LL * d.U * d.Hq * qv::DG_MAX_OPEN);
  d.off_fden = take(8LL * d.U * d.Hq * qv::DG_MAX_OPEN);
  d.off_acc = take(8LL * d.U * qv::DA_N);
  *bytes = off;
  return d;
}

}  // namespace

qevict_status qevict_diag_bytes(const qevict_cache *policy, const qevict_diag_config *dc, size_t *bytes) {
  if (!policy || !dc || !bytes || dc->horizon < 0 || dc->lir_m < 0) return QEVICT_EINVAL;
  const int H = dc->horizon ? dc->horizon : 32, om = policy->cfg.omega;
  if (H < om || H % om || H / om > qv::DG_MAX_OPEN) return QEVICT_EINVAL;
  int64_t b = 0;
  diag_plan(policy, H, 3, &b);
  *bytes = (size_t)b;
  return QEVICT_OK;
}

qevict_status qevict_diag_init(qevict_cache *policy, qevict_cache *fullkv, const qevict_diag_config *dc, void *d_buf,
                               size_t bytes, qevict_stream_t stream, qevict_diag **out) {
  if (!out || !d_buf || ((uintptr_t)d_buf & 255)) return QEVICT_EINVAL;
  int H = 0, m = 0;
  qevict_status st = diag_check(policy, fullkv, dc, &H, &m);
  if (st != QEVICT_OK) return st;
  for (const qevict_cache *c : {policy, fullkv}) {
    if (c->routes_done != 0) return QEVICT_ESCHEDULE;
    for (int l = 0; l < c->cfg.n_layers; ++l)
      if (!c->prefilled[l] || c->t_host[l] != c->cfg.prompt_len) return QEVICT_ESCHEDULE;
  }
  int64_t need = 0;
  qv::DiagDev d = diag_plan(policy, H, m, &need);
  if ((int64_t)bytes < need) return QEVICT_ENOMEM;
  d.base = static_cast<uint8_t *>(d_buf);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemsetAsync(d_buf, 0, (size_t)need, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(d.base + d.off_evict, 0xFF, (size_t)(d.off_evId - d.off_evict), s);
  if (e == cudaSuccess) e = qv::launch_diag_event(policy->dev, fullkv->dev, d, 0, s);
  if (e != cudaSuccess) return QEVICT_ECUDA;
  qevict_diag *dg = new (std::nothrow) qevict_diag();
  if (!dg) return QEVICT_ENOMEM;
  dg->policy = policy;
  dg->fullkv = fullkv;
  dg->dev = d;
  dg->events = 1;
  *out = dg;
  return QEVICT_OK;
}

qevict_status qevict_diag_route(qevict_diag *diag, qevict_stream_t stream) {
  if (!diag) return QEVICT_EINVAL;
  if (route_due(diag->policy) != QEVICT_OK || route_due(diag->fullkv) != QEVICT_OK) return QEVICT_ESCHEDULE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (qv::launch_diag_collect(diag->fullkv->dev, diag->dev, s) != cudaSuccess) return QEVICT_ECUDA;
  qevict_status st = qevict_route(diag->policy, stream);
  if (st == QEVICT_OK) st = qevict_route(diag->fullkv, stream);
  if (st != QEVICT_OK) return st;
  if (qv::launch_diag_event(diag->policy->dev, diag->fullkv->dev, diag->dev, diag->events, s) != cudaSuccess)
    return QEVICT_ECUDA;
  diag->events += 1;
  return QEVICT_OK;
}

qevict_status qevict_diag_read(qevict_diag *diag, qevict_diag_report *out, qevict_stream_t stream) {
  if (!diag || !out) return QEVICT_EINVAL;
  const qv::DiagDev &d = diag->dev;
  std::vector<double> acc((size_t)d.U * qv::DA_N);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(acc.data(), d.base + d.off_acc, acc.size() * sizeof(double), cudaMemcpyDeviceToHost, s) !=
      cudaSuccess)
    return QEVICT_ECUDA;
  qevict_status st = read_status(diag->policy, s);
  if (st == QEVICT_OK) st = read_status(diag->fullkv, s);
  if (st == QEVICT_ECUDA) return st;
  std::memset(out, 0, sizeof(*out));
  double fs = 0, fc = 0, cs = 0, cc = 0, qs = 0, rs = 0, qc = 0;
  for (int u = 0; u < d.U; ++u) {
    const double *a = acc.data() + (size_t)u * qv::DA_N;
    fs += a[qv::DA_FMM_SUM];
    fc += a[qv::DA_FMM_CNT];
    cs += a[qv::DA_CHURN_SUM];
    cc += a[qv::DA_CHURN_CNT];
    qs += a[qv::DA_QSA_SUM];
    rs += a[qv::DA_RQ_SUM];
    qc += a[qv::DA_QSA_CNT];
    for (int z = 0; z < 4; ++z) out->tier_mass[z] += a[qv::DA_MU + z] / d.U;
    out->lir_eligible += (int64_t)a[qv::DA_LIR + 0];
    out->lir_rescued += (int64_t)a[qv::DA_LIR + 1];
    out->lir_fullkv_eligible += (int64_t)a[qv::DA_LIR + 2];
    out->lir_fullkv_rescued += (int64_t)a[qv::DA_LIR + 3];
    for (int k = 0; k < qv::DG_MAX_LAG * 4; ++k) (&out->lag[0][0][0])[k] += (int64_t)a[qv::DA_LAG + k];
    if (u == 0) out->events = (int64_t)a[qv::DA_EVENTS];
  }
  out->fmm = fc > 0 ? fs / fc : 0.0;
  out->fmm_terms = (int64_t)fc;
  out->churn = cc > 0 ? cs / cc : 0.0;
  out->churn_terms = (int64_t)cc;
  out->qsa = qc > 0 ? qs / qc : 0.0;
  out->r_q = qc > 0 ? rs / qc : 0.0;
  out->qsa_terms = (int64_t)qc;
  return st;
}

qevict_status qevict_diag_destroy(qevict_diag *diag) {
  delete diag;
  return QEVICT_OK;
}

qevict_status qevict_destroy(qevict_cache *cache) {
  delete cache;
  return QEVICT_OK;
}

const char *qevict_status_string(qevict_status s) {
  switch (s) {
    case QEVICT_OK: return "ok";
    case QEVICT_EINVAL: return "invalid argument";
    case QEVICT_EBUDGET: return "budget below the protected sink and recent bytes";
    case QEVICT_ENOMEM: return "arena too small";
    case QEVICT_ESCHEDULE: return "call out of schedule (prefill / Omega routing cadence / cache full)";
    case QEVICT_ECUDA: return "CUDA launch or copy failed";
    case QEVICT_EDEVICE: return "a kernel recorded a fault in the device status word";
  }
  return "unknown status";
}

}  // extern "C"
