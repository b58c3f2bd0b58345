// Routing event and migration kernels.
//
// QEvict (arXiv 2608.05326) §4.3 Eq. (4)-(6) and App. A Algorithm 1:
//   candidates = F ∪ Q ∪ windows aged out of the recent region; rank by the cumulative score
//   (descending; ties to the older window); first K_f -> Full, next K_q -> Quantized, rest ->
//   Evicted.  Quantise a window only on its first demotion (write-once ledger), reactivate a
//   dormant ledger on re-demotion, rebuild a promoted window in bf16 from its ledger (the ledger
//   turns dormant), release evicted windows, rebuild the tables in window order.
//
// route_kernel: one CTA per (sequence, layer) unit; sort, tier assignment, deterministic slot
//   allocation (after the releases, newcomers in ascending window id take the lowest free slots),
//   task lists, tables, counters.
// quant_kernel: one CTA per (task, KV head): asymmetric min/max INT2 quantisation (keys per
//   channel over the window's tokens, values per token over the channels), fp16 scale/offset.
// move_kernel: one CTA per (task, KV head): promotion (ledger -> bf16 F slot) or a copy of an
//   aged window into its F slot.  Runs after quant_kernel so sources are read before any freed F
//   slot is rewritten.
// With pre-RoPE keys (rope = 1, QEvict §4.3 "Cache Execution") quant_kernel first takes a window's
// keys back to the pre-RoPE domain at its positions, and move_kernel rotates rebuilt keys forward.
#include "cache_dev.cuh"
#include "common.cuh"
#include "smem_optin.h"

namespace qv {

constexpr int RT_THREADS = 1024;
constexpr int RT_MAXN = 8192;          // windows per unit the router handles
constexpr int MIG_THREADS = 128;

enum : int { SRC_FSLOT = 0, SRC_RING = 1, SRC_PROMPT = 2 };
enum : int { MOVE_PROMOTE = 0, MOVE_COPY = 1 };
enum : int { OLD_AGED = 4 };

struct PromptIO {                     // prefill sources of one layer (NULL during decode routing)
  const __nv_bfloat16 *k;             // [B][P][h_kv][D]
  const __nv_bfloat16 *v;
  int layer;
};

// Exclusive scan of a[0..n) in place over the CTA; returns the total.  n <= RT_MAXN.
__device__ int block_exscan(int *a, int n, int *wsum) {
  const int tid = threadIdx.x, nt = blockDim.x;
  const int per = (n + nt - 1) / nt;
  const int lo = min(n, tid * per), hi = min(n, lo + per);
  int s = 0;
  for (int i = lo; i < hi; ++i) s += a[i];
  const int lane = tid & 31, warp = tid >> 5;
  int x = s;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, off);
    if (lane >= off) x += y;
  }
  if (lane == 31) wsum[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = lane < (nt >> 5) ? wsum[lane] : 0;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, off);
      if (lane >= off) w += y;
    }
    wsum[lane] = w;   // inclusive warp totals
  }
  __syncthreads();
  int run = x - s + (warp ? wsum[warp - 1] : 0);
  const int total = wsum[(nt >> 5) - 1];
  for (int i = lo; i < hi; ++i) {
    const int v = a[i];
    a[i] = run;
    run += v;
  }
  __syncthreads();
  return total;
}

__device__ int block_sum(int v, int *wsum) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int off = 16; off; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  __syncthreads();
  if (lane == 0) wsum[warp] = v;
  __syncthreads();
  int t = 0;
  for (int w = 0; w < (int)(blockDim.x >> 5); ++w) t += wsum[w];
  __syncthreads();
  return t;
}

__global__ void __launch_bounds__(RT_THREADS, 1) route_kernel(const CacheDev C, const PromptIO pio, int unit0,
                                                              int prefill) {
  extern __shared__ __align__(16) uint8_t smem[];
  unsigned long long *keys = reinterpret_cast<unsigned long long *>(smem);          // [RT_MAXN]
  int *scanA = reinterpret_cast<int *>(smem + 8 * RT_MAXN);                          // [RT_MAXN]
  int *scanB = scanA + RT_MAXN;                                                      // [RT_MAXN]
  unsigned char *newt = reinterpret_cast<unsigned char *>(scanB + RT_MAXN);          // [RT_MAXN]
  __shared__ int wsum[32];

  const int tid = threadIdx.x, nt = blockDim.x;
  const int unit = unit0 + blockIdx.x;
  int *meta = C.at<int>(C.off_meta, C.st_meta, unit);
  unsigned char *state = C.at<unsigned char>(C.off_state, C.st_state, unit);
  int *fslot = C.at<int>(C.off_fslot, C.st_fslot, unit);
  int *lslot = C.at<int>(C.off_lslot, C.st_lslot, unit);
  float *score = C.at<float>(C.off_score, C.st_score, unit);
  int2 *ftab = C.at<int2>(C.off_ftab, C.st_ftab, unit);
  int2 *qtab = C.at<int2>(C.off_qtab, C.st_qtab, unit);
  int4 *qtask = C.at<int4>(C.off_qtask, C.st_qtask, unit);
  int4 *mtask = C.at<int4>(C.off_mtask, C.st_mtask, unit);
  const int N = C.n_windows, W = C.W;
  const int T = meta[M_T], nr_old = meta[M_NROUTE];
  const int n_new = n_hist_dev(T, C.n_recent, C.n_sink, W);
  const int n_acc = T > C.n_sink ? min(N, (T - 1 - C.n_sink) / W + 1) : 0;
  const int kf_cap = min(C.k_f, N), lp_cap = min(C.k_f + C.k_q, N);
  if (n_new > N || n_new > RT_MAXN || n_new < nr_old) {
    if (tid == 0) atomicOr(C.status(), QV_ERR_STATE);
    return;
  }

  // 1. the window's attention is the sum of the per-KV-head partials.  Cumulative ranking keeps the
  //    running score in head 0; the other rankers (QEvict App. J) fold the event's attention u
  //    (Eq. (20)) into agg, S = decay * S + u (Eq. (22)) or S = S + u^p (Eq. (23)), and restart u.
  const int ranker = C.ranker;
  float *agg = C.at<float>(C.off_agg, C.st_agg, unit);
  for (int w = tid; w < n_acc; w += nt) {
    float s = score[w];
    for (int g = 1; g < C.h_kv; ++g) {
      s += score[(size_t)g * N + w];
      score[(size_t)g * N + w] = 0.f;
    }
    if (ranker == 0) {
      score[w] = s;
    } else {
      score[w] = 0.f;
      if (ranker == 1) agg[w] = fmaf(C.decay, agg[w], s);
      else if (ranker == 2) agg[w] += powf(s, C.pnorm);
    }
  }
  if (ranker == 3) {
    // key norm (Eq. (24)): mean over the window's tokens of the key's L2 norm across all KV heads,
    // taken once, when the window leaves the recent region; one warp per window, a lane per token
    const int warp = tid >> 5, lane = tid & 31, b = unit % C.B;
    const __nv_bfloat16 *ring = C.at<const __nv_bfloat16>(C.off_ring, C.st_ring, unit);
    for (int w = nr_old + warp; w < n_new; w += nt / 32) {
      float sum = 0.f;
      for (int t = lane; t < W; t += 32) {
        const int pos = C.n_sink + w * W + t;
        float ss = 0.f;
        for (int g = 0; g < C.h_kv; ++g) {
          if (prefill) {
            const __nv_bfloat16 *kr = pio.k + (((size_t)b * C.prompt_len + pos) * C.h_kv + g) * D;
            for (int d = 0; d < D; ++d) {
              const float x = __bfloat162float(kr[d]);
              ss = fmaf(x, x, ss);
            }
          } else {
            const __nv_bfloat16 *kb = ring + ((size_t)(g * 2) * C.ring_windows + w % C.ring_windows) * W * D;
            for (int d = 0; d < D; ++d) {
              const float x = __bfloat162float(kb[fnk_index(t, d)]);
              ss = fmaf(x, x, ss);
            }
          }
        }
        sum += sqrtf(ss);
      }
#pragma unroll
      for (int off = 16; off; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
      if (lane == 0) agg[w] = sum / (float)W;
    }
  }
  __syncthreads();
  // 2. candidates (Eq. (4)): windows still in F or Q plus the newly aged ones
  for (int w = tid; w < n_new; w += nt) {
    const int tier = state[w] & 3;
    scanA[w] = (w >= nr_old || tier == TIER_FULL || tier == TIER_QUANT) ? 1 : 0;
    newt[w] = 0xFF;
  }
  __syncthreads();
  for (int w = tid; w < n_new; w += nt) scanB[w] = scanA[w];
  __syncthreads();
  const int count = block_exscan(scanB, n_new, wsum);
  int p2 = 2;
  while (p2 < count) p2 <<= 1;
  for (int i = tid; i < p2; i += nt) keys[i] = ~0ull;
  __syncthreads();
  for (int w = tid; w < n_new; w += nt)
    if (scanA[w]) {
      // the rank value is >= +0, so its bit pattern orders like the value; ~bits sorts descending
      // (key norms: ascending), ties by window id ascending
      const unsigned sb = __float_as_uint(ranker == 0 ? score[w] : agg[w]);
      keys[scanB[w]] = ((unsigned long long)(ranker == 3 ? sb : ~sb) << 32) | (unsigned)w;
    }
  __syncthreads();
  // 3. bitonic sort, ascending keys = (score desc, window id asc)
  for (int k = 2; k <= p2; k <<= 1)
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = tid; i < p2; i += nt) {
        const int ixj = i ^ j;
        if (ixj > i) {
          const unsigned long long a = keys[i], c = keys[ixj];
          if (((i & k) == 0) ? (a > c) : (a < c)) {
            keys[i] = c;
            keys[ixj] = a;
          }
        }
      }
      __syncthreads();
    }
  // 4. Eq. (5): TopK_{K_f} -> Full, next K_q -> Quantized, rest -> Evicted
  if (!C.no_promotion) {
    for (int r = tid; r < count; r += nt) {
      const int w = (int)(keys[r] & 0xffffffffu);
      newt[w] = r < C.k_f ? TIER_FULL : ((long long)r < (long long)C.k_f + C.k_q ? TIER_QUANT : TIER_EVICT);
    }
  } else {
    // QEvict App. K: a quantized window cannot return to the full tier, so Full takes the best-ranked
    // candidates that are not quantized and Quantized the best of the rest
    auto eligible = [&](int w) { return !(w < nr_old && (state[w] & 3) == TIER_QUANT); };
    for (int r = tid; r < count; r += nt) scanA[r] = eligible((int)(keys[r] & 0xffffffffu)) ? 1 : 0;
    __syncthreads();
    block_exscan(scanA, count, wsum);
    for (int r = tid; r < count; r += nt) {
      const int w = (int)(keys[r] & 0xffffffffu);
      const bool f = eligible(w) && scanA[r] < C.k_f;
      scanB[r] = f ? 0 : 1;
      newt[w] = f ? TIER_FULL : 0xFE;
    }
    __syncthreads();
    block_exscan(scanB, count, wsum);
    for (int r = tid; r < count; r += nt) {
      const int w = (int)(keys[r] & 0xffffffffu);
      if (newt[w] != TIER_FULL) newt[w] = scanB[r] < C.k_q ? TIER_QUANT : TIER_EVICT;
    }
  }
  __syncthreads();

  // 5. releases first: the slots of surviving windows mark the pools (scanA = F pool, scanB = ledger)
  int *poolF = scanA, *poolL = scanB;
  for (int s = tid; s < RT_MAXN; s += nt) poolF[s] = poolL[s] = 0;
  __syncthreads();
  for (int w = tid; w < n_new; w += nt) {
    const int nv = newt[w];
    if (nv == 0xFF) continue;
    const int old = w < nr_old ? (state[w] & 3) : OLD_AGED;
    const int led = w < nr_old ? ((state[w] >> 2) & 3) : LED_NONE;
    if (old == TIER_FULL && nv == TIER_FULL) {
      const int fs = fslot[w];
      if (fs >= 0 && fs < kf_cap) poolF[fs] = 1;
      else atomicOr(C.status(), QV_ERR_STATE);
    }
    const bool keepL = (old == TIER_QUANT && nv != TIER_EVICT) ||
                       (old == TIER_FULL && nv != TIER_EVICT && led == LED_DORMANT);
    if (keepL) {
      const int ls = lslot[w];
      if (ls >= 0 && ls < lp_cap) poolL[ls] = 1;
      else atomicOr(C.status(), QV_ERR_STATE);
    }
  }
  __syncthreads();
  for (int s = tid; s < RT_MAXN; s += nt) {   // free flags
    poolF[s] = (s < kf_cap && !poolF[s]) ? 1 : 0;
    poolL[s] = (s < lp_cap && !poolL[s]) ? 1 : 0;
  }
  __syncthreads();
  const int totF = block_exscan(poolF, kf_cap, wsum);
  const int totL = block_exscan(poolL, lp_cap, wsum);
  // k-th free slot, ascending: slotF[k] / slotL[k] (the sort keys are dead now)
  int *slotF = reinterpret_cast<int *>(keys), *slotL = slotF + RT_MAXN;
  for (int s = tid; s < kf_cap; s += nt)
    if ((s + 1 < kf_cap ? poolF[s + 1] : totF) != poolF[s]) slotF[poolF[s]] = s;
  for (int s = tid; s < lp_cap; s += nt)
    if ((s + 1 < lp_cap ? poolL[s + 1] : totL) != poolL[s]) slotL[poolL[s]] = s;
  __syncthreads();

  // 6. newcomers in ascending window id take the lowest free slots (needF: bit 4, needL: bit 5 of newt)
  int *rankF = scanA, *rankL = scanB;
  for (int w = tid; w < n_new; w += nt) {
    const int nv = newt[w];
    int nf = 0, nl = 0;
    if (nv != 0xFF) {
      const int old = w < nr_old ? (state[w] & 3) : OLD_AGED;
      const int led = w < nr_old ? ((state[w] >> 2) & 3) : LED_NONE;
      nf = (nv == TIER_FULL && old != TIER_FULL) ? 1 : 0;
      nl = (nv == TIER_QUANT && (old == OLD_AGED || (old == TIER_FULL && led != LED_DORMANT))) ? 1 : 0;
      newt[w] = (unsigned char)(nv | (nf << 4) | (nl << 5));
    }
    rankF[w] = nf;
    rankL[w] = nl;
  }
  __syncthreads();
  const int nNeedF = block_exscan(rankF, n_new, wsum);
  const int nNeedL = block_exscan(rankL, n_new, wsum);
  // Unreachable with in-range slot ids: a busy F slot belongs to a window that keeps one of the K_f
  // Full places and a newcomer takes another, so nNeedF <= totF; the ledger holds K_f + K_q places the
  // same way.  A test cap set on the host (slot_cap >= 0) hides free slots so that the guard can be
  // exercised.  Should it fire, this event changes no tier, table or slot and migrates nothing.
  const int capF = C.slot_cap >= 0 ? min(totF, C.slot_cap) : totF;
  const int capL = C.slot_cap >= 0 ? min(totL, C.slot_cap) : totL;
  if (nNeedF > capF || nNeedL > capL) {
    if (tid == 0) {
      atomicOr(C.status(), QV_ERR_SLOT);
      meta[M_NQUANT] = 0;
      meta[M_NMOVE] = 0;
    }
    return;
  }

  int c_promo = 0, c_demo = 0, c_firstq = 0, c_react = 0, c_evict = 0, c_agedf = 0, c_agedq = 0;
  for (int w = tid; w < n_new; w += nt) {
    const int nv = newt[w];
    if (nv == 0xFF) continue;
    const int tnew = nv & 3;
    const bool needF = (nv >> 4) & 1, needL = (nv >> 5) & 1;
    const int old = w < nr_old ? (state[w] & 3) : OLD_AGED;
    const int led = w < nr_old ? ((state[w] >> 2) & 3) : LED_NONE;
    const int ofs = w < nr_old ? fslot[w] : -1;
    const int ols = w < nr_old ? lslot[w] : -1;
    const int src_kind = prefill ? SRC_PROMPT : SRC_RING;
    if (tnew == TIER_EVICT) {
      state[w] = TIER_EVICT;
      fslot[w] = -1;
      lslot[w] = -1;
      ++c_evict;
    } else if (tnew == TIER_QUANT) {
      int ls = ols;
      if (needL) {
        ls = slotL[rankL[w]];
        qtask[rankL[w]] = make_int4(w, old == TIER_FULL ? SRC_FSLOT : src_kind, old == TIER_FULL ? ofs : w, ls);
        ++c_firstq;
      }
      if (old == TIER_FULL) {
        ++c_demo;
        if (led == LED_DORMANT) ++c_react;
      }
      if (old == OLD_AGED) ++c_agedq;
      state[w] = (unsigned char)(TIER_QUANT | (LED_ACTIVE << 2));
      fslot[w] = -1;
      lslot[w] = ls;
    } else {   // Full
      int fs = ofs;
      int ledn = led;
      if (needF) {
        fs = slotF[rankF[w]];
        if (old == TIER_QUANT) {
          mtask[rankF[w]] = make_int4(w, MOVE_PROMOTE, ols, fs);
          ledn = LED_DORMANT;
          ++c_promo;
        } else {
          mtask[rankF[w]] = make_int4(w, MOVE_COPY | (src_kind << 4), w, fs);
          ledn = LED_NONE;
          ++c_agedf;
        }
      }
      state[w] = (unsigned char)(TIER_FULL | (ledn << 2));
      fslot[w] = fs;
      lslot[w] = (ledn == LED_NONE) ? -1 : ols;
    }
  }
  __syncthreads();
  // 7. tables in ascending window id (QEvict Algorithm 1: reconstruct in chronological order)
  for (int w = tid; w < n_new; w += nt) {
    const int t = state[w] & 3;
    rankF[w] = (t == TIER_FULL) ? 1 : 0;
    rankL[w] = (t == TIER_QUANT) ? 1 : 0;
  }
  __syncthreads();
  const int nF = block_exscan(rankF, n_new, wsum);
  const int nQ = block_exscan(rankL, n_new, wsum);
  for (int w = tid; w < n_new; w += nt) {
    const int t = state[w] & 3;
    if (t == TIER_FULL && qv_inbounds(rankF[w] < kf_cap, C.status())) ftab[rankF[w]] = make_int2(w, fslot[w]);
    if (t == TIER_QUANT && qv_inbounds(rankL[w] < min(C.k_q, N), C.status()))
      qtab[rankL[w]] = make_int2(w, lslot[w]);
  }
  const int tp = block_sum(c_promo, wsum), td = block_sum(c_demo, wsum), tf = block_sum(c_firstq, wsum);
  const int tr = block_sum(c_react, wsum), te = block_sum(c_evict, wsum), ta = block_sum(c_agedf, wsum);
  const int tq = block_sum(c_agedq, wsum);
  if (tid == 0) {
    long long *ctr = reinterpret_cast<long long *>(C.arena + C.off_counters) + (size_t)unit * N_COUNTERS;
    ctr[0] += tp;
    ctr[1] += td;
    ctr[2] += tf;
    ctr[3] += tr;
    ctr[4] += te;
    ctr[5] += ta;
    ctr[6] += tq;
    meta[M_NROUTE] = n_new;
    meta[M_FCOUNT] = nF;
    meta[M_QCOUNT] = nQ;
    meta[M_NQUANT] = nNeedL;
    meta[M_NMOVE] = nNeedF;
    if (!prefill) meta[M_NEVENT] += 1;
  }
}

// ----------------------------------------------------------------------------- quantise once

template <int W>
__device__ void load_window(const CacheDev &C, const PromptIO &pio, int unit, int b, int g, int kind, int src,
                            float (*xk)[D + 1], float (*xv)[D + 1]) {
  using Gm = Geo<W, 2>;
  const int tid = threadIdx.x;
  if (kind == SRC_PROMPT) {
    const int P = C.prompt_len;
    for (int idx = tid; idx < W * D; idx += blockDim.x) {
      const int tok = idx / D, dim = idx % D;
      const int pos = C.n_sink + src * W + tok;
      const size_t o = (((size_t)b * P + pos) * C.h_kv + g) * D + dim;
      xk[tok][dim] = __bfloat162float(pio.k[o]);
      xv[tok][dim] = __bfloat162float(pio.v[o]);
    }
    return;
  }
  const __nv_bfloat16 *kb, *vb;
  if (kind == SRC_FSLOT) {
    kb = C.at<const __nv_bfloat16>(C.off_fpool, C.st_fpool, unit) + ((size_t)src * C.h_kv + g) * 2 * Gm::BLK;
    vb = kb + Gm::BLK;
  } else {
    const __nv_bfloat16 *ring = C.at<const __nv_bfloat16>(C.off_ring, C.st_ring, unit);
    const int rs = src % C.ring_windows;
    kb = ring + ((size_t)(g * 2 + 0) * C.ring_windows + rs) * Gm::BLK;
    vb = ring + ((size_t)(g * 2 + 1) * C.ring_windows + rs) * Gm::BLK;
  }
  for (int idx = tid; idx < W * D; idx += blockDim.x) {
    const int tok = idx / D, dim = idx % D;
    xk[tok][dim] = __bfloat162float(kb[fnk_index(tok, dim)]);
    xv[tok][dim] = __bfloat162float(vb[fnv_index(tok, dim)]);
  }
}

// code = clamp(rint((x - m) / s), 0, 2^BITS - 1) in float32 with IEEE subtraction and division,
// 0 when s == 0
template <int BITS>
__device__ __forceinline__ unsigned quant_code(float x, float s, float m) {
  if (s == 0.f) return 0u;
  const float t = rintf(__fdiv_rn(__fsub_rn(x, m), s));
  return (unsigned)fminf(fmaxf(t, 0.f), (float)((1 << BITS) - 1));
}

template <int W, int BITS>
constexpr int quant_smem_bytes() {   // xk, xv [W][D+1] fp32 + the packed K and V codes
  return 2 * W * (D + 1) * 4 + 2 * Geo<W, BITS>::CODE_BYTES;
}

template <int W, int BITS>
__global__ void __launch_bounds__(MIG_THREADS) quant_kernel(const CacheDev C, const PromptIO pio, int unit0) {
  using Gm = Geo<W, BITS>;
  constexpr float LEVELS = (float)((1 << BITS) - 1);
  extern __shared__ __align__(16) uint8_t qsm[];
  auto xk = reinterpret_cast<float(*)[D + 1]>(qsm);
  auto xv = reinterpret_cast<float(*)[D + 1]>(qsm + W * (D + 1) * 4);
  uint32_t *cw = reinterpret_cast<uint32_t *>(qsm + 2 * W * (D + 1) * 4);
  const int unit = unit0 + blockIdx.y;
  const int b = unit % C.B;
  const int *meta = C.at<const int>(C.off_meta, C.st_meta, unit);
  const int ntask = meta[M_NQUANT];
  const int4 *qtask = C.at<const int4>(C.off_qtask, C.st_qtask, unit);
  uint8_t *ledger = C.at<uint8_t>(C.off_ledger, C.st_ledger, unit);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int kf_cap = min(C.k_f, C.n_windows), lp_cap = min(C.k_f + C.k_q, C.n_windows);
  if (!qv_inbounds(ntask >= 0 && ntask <= C.n_windows, C.status())) return;
  for (int job = blockIdx.x; job < ntask * C.h_kv; job += gridDim.x) {
    const int4 tk = qtask[job / C.h_kv];
    const int g = job % C.h_kv;
    // task: window, source kind, source (F slot / window id / prompt window), ledger slot
    const bool src_ok = tk.y == SRC_FSLOT ? (tk.z >= 0 && tk.z < kf_cap)
                      : tk.y == SRC_RING  ? (tk.z >= 0 && tk.z < C.n_windows)
                      : tk.y == SRC_PROMPT && tk.z >= 0 && C.n_sink + (tk.z + 1) * W <= C.prompt_len;
    if (!qv_inbounds(src_ok && tk.x >= 0 && tk.x < C.n_windows && tk.w >= 0 && tk.w < lp_cap, C.status()))
      continue;   // the same for every thread of the CTA
    __syncthreads();
    load_window<W>(C, pio, unit, b, g, tk.y, tk.z, xk, xv);
    for (int i = threadIdx.x; i < 2 * Gm::CODE_BYTES / 4; i += blockDim.x) cw[i] = 0u;
    __syncthreads();
    if (C.rope) {
      // keys back to the pre-RoPE domain at the window's positions (QEvict §4.3), pairs (i, i + 64):
      // x_i c + x_{i+64} s and x_{i+64} c - x_i s, each product and sum rounded on its own
      const float *cs = C.rope_tab() + (size_t)(C.n_sink + tk.x * W) * D;
      for (int idx = tid; idx < W * (D / 2); idx += blockDim.x) {
        const int tok = idx / (D / 2), i = idx % (D / 2);
        const float c = cs[tok * D + 2 * i], sn = cs[tok * D + 2 * i + 1];
        const float a = xk[tok][i], bb = xk[tok][i + D / 2];
        xk[tok][i] = __fadd_rn(__fmul_rn(a, c), __fmul_rn(bb, sn));
        xk[tok][i + D / 2] = __fsub_rn(__fmul_rn(bb, c), __fmul_rn(a, sn));
      }
      __syncthreads();
    }
    uint8_t *blk = ledger + ((size_t)tk.w * C.h_kv + g) * Gm::QB;
    // scatter a code into its fragment-native position (shared-memory words, copied out below)
    auto put = [&](bool is_v, int tok, int dim, unsigned c) {
      int byte, shift;
      code_pos<BITS>(is_v, tok, dim, byte, shift);
      const int gb = byte + (is_v ? Gm::CODE_BYTES : 0);
      atomicOr(&cw[gb >> 2], c << (8 * (gb & 3) + shift));
    };
    // keys: one group per channel across the window's tokens
    {
      const int dim = tid;   // MIG_THREADS == D
      float mn = xk[0][dim], mx = xk[0][dim];
      for (int t = 1; t < W; ++t) {
        mn = fminf(mn, xk[t][dim]);
        mx = fmaxf(mx, xk[t][dim]);
      }
      const __half s16 = __float2half_rn(__fdiv_rn(__fsub_rn(mx, mn), LEVELS));
      const __half m16 = __float2half_rn(mn);
      const float s = __half2float(s16), m = __half2float(m16);
      reinterpret_cast<__half *>(blk + Gm::OFF_KS)[dim] = s16;
      reinterpret_cast<__half *>(blk + Gm::OFF_KM)[dim] = m16;
      for (int t = 0; t < W; ++t) put(false, t, dim, quant_code<BITS>(xk[t][dim], s, m));
    }
    // values: one group per token across the channels
    for (int t = warp; t < W; t += MIG_THREADS / 32) {
      float mn = INFINITY, mx = -INFINITY;
      for (int d = lane; d < D; d += 32) {
        mn = fminf(mn, xv[t][d]);
        mx = fmaxf(mx, xv[t][d]);
      }
#pragma unroll
      for (int off = 16; off; off >>= 1) {
        mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, off));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      }
      const __half s16 = __float2half_rn(__fdiv_rn(__fsub_rn(mx, mn), LEVELS));
      const __half m16 = __float2half_rn(mn);
      const float s = __half2float(s16), m = __half2float(m16);
      if (lane == 0) {
        reinterpret_cast<__half *>(blk + Gm::OFF_VS)[t] = s16;
        reinterpret_cast<__half *>(blk + Gm::OFF_VM)[t] = m16;
      }
      for (int d = lane; d < D; d += 32) put(true, t, d, quant_code<BITS>(xv[t][d], s, m));
    }
    __syncthreads();
    for (int i = tid; i < 2 * Gm::CODE_BYTES / 4; i += blockDim.x) reinterpret_cast<uint32_t *>(blk)[i] = cw[i];
  }
}

// ----------------------------------------------------------------------------- promote / copy

template <int W, int BITS>
__global__ void __launch_bounds__(MIG_THREADS) move_kernel(const CacheDev C, const PromptIO pio, int unit0) {
  using Gm = Geo<W, BITS>;
  __shared__ __align__(16) uint8_t led[Gm::QB];
  const int unit = unit0 + blockIdx.y;
  const int b = unit % C.B;
  const int *meta = C.at<const int>(C.off_meta, C.st_meta, unit);
  const int ntask = meta[M_NMOVE];
  const int4 *mtask = C.at<const int4>(C.off_mtask, C.st_mtask, unit);
  const uint8_t *ledger = C.at<const uint8_t>(C.off_ledger, C.st_ledger, unit);
  const __nv_bfloat16 *ring = C.at<const __nv_bfloat16>(C.off_ring, C.st_ring, unit);
  __nv_bfloat16 *fpool = C.at<__nv_bfloat16>(C.off_fpool, C.st_fpool, unit);
  const int tid = threadIdx.x;
  const int kf_cap = min(C.k_f, C.n_windows), lp_cap = min(C.k_f + C.k_q, C.n_windows);
  if (!qv_inbounds(ntask >= 0 && ntask <= C.n_windows, C.status())) return;
  for (int job = blockIdx.x; job < ntask * C.h_kv; job += gridDim.x) {
    const int4 tk = mtask[job / C.h_kv];
    const int g = job % C.h_kv;
    // task: window, kind | source kind << 4, source (ledger slot / window id / prompt window), F slot
    const int k0 = tk.y & 15, s0k = tk.y >> 4;
    const bool src_ok = k0 == MOVE_PROMOTE ? (tk.z >= 0 && tk.z < lp_cap)
                      : s0k == SRC_RING    ? (tk.z >= 0 && tk.z < C.n_windows)
                      : s0k == SRC_PROMPT && tk.z >= 0 && C.n_sink + (tk.z + 1) * W <= C.prompt_len;
    if (!qv_inbounds(src_ok && tk.x >= 0 && tk.x < C.n_windows && tk.w >= 0 && tk.w < kf_cap, C.status()))
      continue;   // the same for every thread of the CTA
    __nv_bfloat16 *dk = fpool + ((size_t)tk.w * C.h_kv + g) * 2 * Gm::BLK;
    __nv_bfloat16 *dv = dk + Gm::BLK;
    const int kind = tk.y & 15, src_kind = tk.y >> 4;
    __syncthreads();
    if (kind == MOVE_PROMOTE) {
      // x_hat = bf16(fp32(code * s + m)), the ledger's approximation rebuilt in bf16
      const uint8_t *src = ledger + ((size_t)tk.z * C.h_kv + g) * Gm::QB;
      for (int i = tid; i < Gm::QB / 16; i += blockDim.x)
        reinterpret_cast<uint4 *>(led)[i] = reinterpret_cast<const uint4 *>(src)[i];
      __syncthreads();
      const __half *ks = reinterpret_cast<const __half *>(led + Gm::OFF_KS);
      const __half *km = reinterpret_cast<const __half *>(led + Gm::OFF_KM);
      const __half *vsp = reinterpret_cast<const __half *>(led + Gm::OFF_VS);
      const __half *vmp = reinterpret_cast<const __half *>(led + Gm::OFF_VM);
      auto dq = [&](bool is_v, int tok, int dim) -> float {
        int byte, shift;
        code_pos<BITS>(is_v, tok, dim, byte, shift);
        const float c = (float)((led[byte + (is_v ? Gm::OFF_VCODE : 0)] >> shift) & ((1u << BITS) - 1u));
        const float s = __half2float(is_v ? vsp[tok] : ks[dim]);
        const float m = __half2float(is_v ? vmp[tok] : km[dim]);
        return __bfloat162float(__float2bfloat16_rn(__fmaf_rn(c, s, m)));
      };
      if (!C.rope) {
        for (int idx = tid; idx < 2 * W * D; idx += blockDim.x) {
          const bool is_v = idx >= W * D;
          const int e = is_v ? idx - W * D : idx, tok = e / D, dim = e % D;
          const __nv_bfloat16 x = __float2bfloat16_rn(dq(is_v, tok, dim));
          if (is_v) dv[fnv_index(tok, dim)] = x;
          else dk[fnk_index(tok, dim)] = x;
        }
      } else {
        for (int idx = tid; idx < W * D; idx += blockDim.x) {
          const int tok = idx / D, dim = idx % D;
          dv[fnv_index(tok, dim)] = __float2bfloat16_rn(dq(true, tok, dim));
        }
        // pre-RoPE keys rotated back to the window's positions (QEvict §4.3), then bf16:
        // x_i c - x_{i+64} s and x_{i+64} c + x_i s, each product and sum rounded on its own
        const float *cs = C.rope_tab() + (size_t)(C.n_sink + tk.x * W) * D;
        for (int idx = tid; idx < W * (D / 2); idx += blockDim.x) {
          const int tok = idx / (D / 2), i = idx % (D / 2);
          const float c = cs[tok * D + 2 * i], sn = cs[tok * D + 2 * i + 1];
          const float a = dq(false, tok, i), bb = dq(false, tok, i + D / 2);
          dk[fnk_index(tok, i)] = __float2bfloat16_rn(__fsub_rn(__fmul_rn(a, c), __fmul_rn(bb, sn)));
          dk[fnk_index(tok, i + D / 2)] = __float2bfloat16_rn(__fadd_rn(__fmul_rn(bb, c), __fmul_rn(a, sn)));
        }
      }
    } else if (src_kind == SRC_RING) {
      const int rs = tk.z % C.ring_windows;
      const uint4 *sk = reinterpret_cast<const uint4 *>(ring + ((size_t)(g * 2 + 0) * C.ring_windows + rs) * Gm::BLK);
      const uint4 *sv = reinterpret_cast<const uint4 *>(ring + ((size_t)(g * 2 + 1) * C.ring_windows + rs) * Gm::BLK);
      for (int i = tid; i < Gm::BLK * 2 / 16; i += blockDim.x) {
        reinterpret_cast<uint4 *>(dk)[i] = sk[i];
        reinterpret_cast<uint4 *>(dv)[i] = sv[i];
      }
    } else {   // prompt rows -> fragment-native block
      const int P = C.prompt_len;
      for (int idx = tid; idx < W * D; idx += blockDim.x) {
        const int tok = idx / D, dim = idx % D;
        const size_t o = (((size_t)b * P + C.n_sink + (size_t)tk.z * W + tok) * C.h_kv + g) * D + dim;
        dk[fnk_index(tok, dim)] = pio.k[o];
        dv[fnv_index(tok, dim)] = pio.v[o];
      }
    }
  }
}

// ----------------------------------------------------------------------------- prefill setup / init

// Stores the sink rows and the recent windows of one layer's prompt, the initial scores and T = P.
template <int W>
__global__ void prefill_setup_kernel(const CacheDev C, const PromptIO pio, const float *s0) {
  using Gm = Geo<W, 2>;
  const int b = blockIdx.x, g = blockIdx.y;
  const int unit = pio.layer * C.B + b;
  const int P = C.prompt_len;
  const int nh = n_hist_dev(P, C.n_recent, C.n_sink, W);
  const int npw = (P - C.n_sink + W - 1) / W;   // windows starting inside the prompt
  __nv_bfloat16 *sink = C.at<__nv_bfloat16>(C.off_sink, C.st_sink, unit) + (size_t)g * 2 * C.n_sink * D;
  __nv_bfloat16 *ring = C.at<__nv_bfloat16>(C.off_ring, C.st_ring, unit);
  for (int idx = threadIdx.x; idx < C.n_sink * D; idx += blockDim.x) {
    const int t = idx / D, d = idx % D;
    const size_t o = (((size_t)b * P + t) * C.h_kv + g) * D + d;
    sink[idx] = pio.k[o];
    sink[C.n_sink * D + idx] = pio.v[o];
  }
  const int lo = C.n_sink + nh * W;
  for (int idx = threadIdx.x; idx < (P - lo) * D; idx += blockDim.x) {
    const int pos = lo + idx / D, d = idx % D;
    const int j = (pos - C.n_sink) / W, tok = (pos - C.n_sink) % W, rs = j % C.ring_windows;
    const size_t o = (((size_t)b * P + pos) * C.h_kv + g) * D + d;
    ring[((size_t)(g * 2 + 0) * C.ring_windows + rs) * Gm::BLK + fnk_index(tok, d)] = pio.k[o];
    ring[((size_t)(g * 2 + 1) * C.ring_windows + rs) * Gm::BLK + fnv_index(tok, d)] = pio.v[o];
  }
  if (threadIdx.x == 0) reinterpret_cast<int *>(C.arena + C.off_thead)[(size_t)unit * C.h_kv + g] = P;
  if (g == 0) {
    float *score = C.at<float>(C.off_score, C.st_score, unit);
    for (int w = threadIdx.x; w < npw; w += blockDim.x) score[w] = s0[(size_t)b * npw + w];
    if (threadIdx.x == 0) {
      int *meta = C.at<int>(C.off_meta, C.st_meta, unit);
      meta[M_T] = P;
      meta[M_FLUSHT] = P;
      meta[M_NROUTE] = 0;
      meta[M_FCOUNT] = 0;
      meta[M_QCOUNT] = 0;
    }
  }
}

__global__ void init_slots_kernel(const CacheDev C) {
  const int unit = blockIdx.x;
  int *fs = C.at<int>(C.off_fslot, C.st_fslot, unit);
  int *ls = C.at<int>(C.off_lslot, C.st_lslot, unit);
  for (int w = threadIdx.x; w < C.n_windows; w += blockDim.x) {
    fs[w] = -1;
    ls[w] = -1;
  }
}

// Failure-reporting self-test: one thread waits, through the library's bounded wait, on an mbarrier
// phase that nothing completes.  The wait gives up after its limit, records QV_ERR_TIMEOUT in the
// status word and the kernel returns: the context stays usable.
__global__ void wait_selftest_kernel(const CacheDev C) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
    mbar_wait(&bar, 0, C.status());
  }
}

// ----------------------------------------------------------------------------- launchers

int route_smem_bytes() { return 8 * RT_MAXN + 4 * RT_MAXN * 2 + RT_MAXN; }
int route_max_windows() { return RT_MAXN; }

cudaError_t launch_init(const CacheDev &C, cudaStream_t s) {
  init_slots_kernel<<<C.B * C.L, 256, 0, s>>>(C);
  return cudaGetLastError();
}

cudaError_t launch_wait_selftest(const CacheDev &C, cudaStream_t s) {
  wait_selftest_kernel<<<1, 32, 0, s>>>(C);
  return cudaGetLastError();
}

template <int W, int BITS>
static cudaError_t launch_migrate(const CacheDev &C, const PromptIO &pio, int unit0, int n_units, int mig_blocks,
                                  cudaStream_t s) {
  constexpr int qsm = quant_smem_bytes<W, BITS>();
  static SmemOptIn optin;   // per device: the dynamic shared memory opt-in
  if (qsm > 48 * 1024) {
    const cudaError_t e = optin.ensure(quant_kernel<W, BITS>, qsm);
    if (e != cudaSuccess) return e;
  }
  dim3 grid(mig_blocks, n_units);
  quant_kernel<W, BITS><<<grid, MIG_THREADS, qsm, s>>>(C, pio, unit0);
  move_kernel<W, BITS><<<grid, MIG_THREADS, 0, s>>>(C, pio, unit0);
  return cudaGetLastError();
}

cudaError_t launch_route(const CacheDev &C, int unit0, int n_units, const __nv_bfloat16 *kp,
                         const __nv_bfloat16 *vp, int layer, int mig_blocks, cudaStream_t s) {
  static SmemOptIn optin;
  const cudaError_t e = optin.ensure(route_kernel, route_smem_bytes());
  if (e != cudaSuccess) return e;
  const int prefill = kp != nullptr;
  PromptIO pio{kp, vp, layer};
  route_kernel<<<n_units, RT_THREADS, route_smem_bytes(), s>>>(C, pio, unit0, prefill);
  if (C.W == 32 && C.bits == 2) return launch_migrate<32, 2>(C, pio, unit0, n_units, mig_blocks, s);
  if (C.W == 64 && C.bits == 4) return launch_migrate<64, 4>(C, pio, unit0, n_units, mig_blocks, s);
  return cudaErrorInvalidValue;
}

cudaError_t launch_prefill_setup(const CacheDev &C, const __nv_bfloat16 *kp, const __nv_bfloat16 *vp, int layer,
                                 const float *s0, cudaStream_t s) {
  PromptIO pio{kp, vp, layer};
  if (C.W == 32)
    prefill_setup_kernel<32><<<dim3(C.B, C.h_kv), 256, 0, s>>>(C, pio, s0);
  else if (C.W == 64)
    prefill_setup_kernel<64><<<dim3(C.B, C.h_kv), 256, 0, s>>>(C, pio, s0);
  else
    return cudaErrorInvalidValue;
  return cudaGetLastError();
}

}  // namespace qv
