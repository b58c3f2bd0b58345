// Device view of a cache: the caller's arena plus the byte offsets of every region.
// Built once on the host (api.cu) and passed by value to every kernel.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

namespace qv {

struct CacheDev {
  uint8_t *arena;
  // per-unit regions: unit u = layer * B + seq
  int64_t off_sink, st_sink;
  int64_t off_ring, st_ring;
  int64_t off_fpool, st_fpool;
  int64_t off_ledger, st_ledger;
  int64_t off_score, st_score;
  int64_t off_state, st_state;
  int64_t off_fslot, st_fslot;
  int64_t off_lslot, st_lslot;
  int64_t off_ftab, st_ftab;
  int64_t off_qtab, st_qtab;
  int64_t off_meta, st_meta;
  int64_t off_agg, st_agg;         // float [N]: ranker value (rankers 1-3)
  int64_t off_qtask, st_qtask;     // int4 quantise tasks [n_windows]
  int64_t off_mtask, st_mtask;     // int4 promote/copy tasks [n_windows]
  // global regions
  int64_t off_counters;            // int64 [U][N_COUNTERS]
  int64_t off_status;              // int32, inside the arena (status_word points at it for a cache)
  int64_t off_splitctr;            // uint32 [L][B][h_kv]
  int64_t off_thead;               // int32 [L][B][h_kv] tokens cached, one copy per KV head: the decode
                                   // CTAs of a head read theirs, its last CTA advances it
  int64_t off_part, st_part_layer; // float [L][B][h_kv][n_split][PART_FLOATS]
  // per-window log2-sum-exp of the decode steps since the last score flush, by step slot
  // (tokens cached at the step minus those at the flush) and stable item index
  int64_t off_mu, st_mu_layer;     // float [L][B][h_kv][omega][max_items][G]
  int64_t off_mstat, st_mstat_layer;   // float [L][B][h_kv][omega][16]: merged max M[8], 1/L[8] per step
  int64_t off_flushctr;            // uint32 [L][B] score-flush arrivals
  int64_t off_rowstat;             // float [B][h_q][P] prefill row log2-sum-exp
  int64_t off_colsum;              // float [B][h_q][P] prefill column sums
  int64_t off_rope;                // float [max_len][64][2] (cos, sin) of every position (rope = 1)
  // sizes
  int B, L, h_q, h_kv, G, n_sink, n_recent, W, bits, omega;
  int k_f, k_q, n_windows, ring_windows, n_split, max_items, prompt_len, max_len;
  int ranker, no_promotion;
  float decay, pnorm;
  int rope;                        // 1: Quantized keys are kept before RoPE
  int slot_cap;                    // >= 0: routing sees at most this many free F / ledger slots (a
                                   // host-set test cap that makes the slot-exhaustion guard reachable)
  int *status_word;                // device status word every bounded wait and guard reports to

  // Stable index of a window's mass record between two routing events: 1 + i for the i-th recent
  // window from the first unrouted one, then the Full table entries, then the Quantized ones.
  __host__ __device__ int loc_items() const { return ring_windows + 1; }
  __host__ __device__ int kf_cap() const { return k_f < n_windows ? k_f : n_windows; }

  template <typename T>
  __host__ __device__ T *at(int64_t off, int64_t st, int u) const {
    return reinterpret_cast<T *>(arena + off + st * (int64_t)u);
  }
  __host__ __device__ const float *rope_tab() const { return reinterpret_cast<const float *>(arena + off_rope); }
  __host__ __device__ int *status() const { return status_word; }
};

constexpr int PART_FLOATS = 16 + 8 * 128;   // m[8], l[8], O[8][128] per split

struct DecodeIO {
  const __nv_bfloat16 *q;       // [B][h_q][D]
  const __nv_bfloat16 *k_new;   // [B][h_kv][D]
  const __nv_bfloat16 *v_new;   // [B][h_kv][D]
  __nv_bfloat16 *out;           // [B][h_q][D]
  int layer;
  float scale_log2;             // log2(e) / sqrt(D)
  float inv_hq;                 // 1 / h_q
  int wait_first;               // 1: the previous kernel in the stream may be this layer's decode
};

}  // namespace qv
