// Routing diagnostics of QEvict (arXiv 2608.05326) App. I and App. K, measured against a FullKV run.
//
// Two caches decode the same inputs: the evaluated policy P and a FullKV cache R whose budget keeps
// every window Full, so R's per-step window masses are the FullKV attention A_tau(w) of App. I.1.
// At every routing event:
//   diag_collect_kernel  (before R's score flush) reads R's recorded masses of the steps since the
//     previous event and adds, for every routing event still inside its horizon H, the mass on the
//     windows P had evicted by then and on every state that existed then (App. I.2 Eq. (13));
//   diag_event_kernel    (after both caches routed) closes the events whose horizon is complete,
//     opens this one, and records the selection churn (Eq. (14)), the tier attention-mass shares
//     (Eq. (15)), QSA and R_Q over P's Quantized windows (Eq. (16)-(17)), Global LIR episodes of P's
//     Full tier and of the FullKV top-K_f selection (Eq. (18)), and lagged transition counts of P's
//     Full tier (Eq. (19)).
// States are windows; an episode starts when a window leaves the selected set; FMM counts only
// events whose whole horizon was decoded.
#include "cache_dev.cuh"
#include "common.cuh"
#include "smem_optin.h"
#include "diag_dev.cuh"

namespace qv {

constexpr int DG_COLLECT_THREADS = 256;
constexpr int DG_EVENT_THREADS = 1024;

__device__ __forceinline__ float warp_sum_f(float v) {
#pragma unroll
  for (int off = 16; off; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  return v;
}

// One CTA per (KV head g, sequence, layer) of R.  Only two kinds of window enter the sums: those the
// policy has evicted by an open event (FMM numerator) and those that did not exist yet at an open event
// (left out of its denominator, which is then the step count minus their attention: every step's
// attention sums to one over the sinks and the windows).
__global__ void __launch_bounds__(DG_COLLECT_THREADS) diag_collect_kernel(const CacheDev R, const DiagDev Dg) {
  const int g = blockIdx.x, b = blockIdx.y, layer = blockIdx.z;
  const int unit = layer * R.B + b, bg = b * R.h_kv + g;
  const int G = R.G, NO = Dg.n_open;
  __shared__ int s_meta[8];
  __shared__ float st[DG_MAX_OMEGA * 16];                  // merged max and 1/L of each pending step
  __shared__ int s_evT[DG_MAX_OPEN], s_evId[DG_MAX_OPEN];
  __shared__ unsigned s_inh[DG_MAX_OMEGA];                 // per step: the open events it counts for
  __shared__ float acc_ev[8][DG_MAX_OPEN], acc_nx[8][DG_MAX_OPEN];
  const int *meta = R.at<const int>(R.off_meta, R.st_meta, unit);
  if (threadIdx.x < 8) s_meta[threadIdx.x] = meta[threadIdx.x];
  if (threadIdx.x < DG_MAX_OPEN) {
    s_evT[threadIdx.x] = threadIdx.x < NO ? Dg.ev_T(unit)[threadIdx.x] : -1;
    s_evId[threadIdx.x] = threadIdx.x < NO ? Dg.ev_id(unit)[threadIdx.x] : -1;
  }
  if (threadIdx.x < 8 * DG_MAX_OPEN) {
    (&acc_ev[0][0])[threadIdx.x] = 0.f;
    (&acc_nx[0][0])[threadIdx.x] = 0.f;
  }
  __syncthreads();
  const int T = s_meta[M_T], F = s_meta[M_FLUSHT], j0 = s_meta[M_NROUTE];
  const int nF = s_meta[M_FCOUNT], nQ = s_meta[M_QCOUNT];
  const int nk = T - F;
  if (nk < 0 || nk > R.omega || nk > DG_MAX_OMEGA) {
    if (threadIdx.x == 0) atomicOr(R.status(), QV_ERR_STATE);
    return;
  }
  const float *ms = reinterpret_cast<const float *>(R.arena + R.off_mstat + R.st_mstat_layer * layer) +
                    (size_t)bg * R.omega * 16;
  for (int i = threadIdx.x; i < nk * 16; i += blockDim.x) st[i] = ms[i];
  for (int k = threadIdx.x; k < nk; k += blockDim.x) {
    const int Tk = F + k + 1;   // tokens cached after step k; its query sits at position Tk - 1
    unsigned m = 0;
    for (int j = 0; j < NO; ++j)
      if (s_evT[j] >= 0 && Tk > s_evT[j] && Tk - s_evT[j] <= Dg.horizon) m |= 1u << j;
    s_inh[k] = m;
  }
  __syncthreads();
  const float *mu = reinterpret_cast<const float *>(R.arena + R.off_mu + R.st_mu_layer * layer) +
                    (size_t)bg * R.omega * R.max_items * R.G;
  const int2 *ftab = R.at<const int2>(R.off_ftab, R.st_ftab, unit);
  const int2 *qtab = R.at<const int2>(R.off_qtab, R.st_qtab, unit);
  const int *evict = Dg.evict(unit);
  const int LOC = R.loc_items(), KFC = R.kf_cap();
  float ev[8][DG_MAX_OPEN], nx[8][DG_MAX_OPEN];
#pragma unroll
  for (int h = 0; h < 8; ++h)
#pragma unroll
    for (int j = 0; j < DG_MAX_OPEN; ++j) ev[h][j] = nx[h][j] = 0.f;
  for (int idx = 1 + threadIdx.x; idx < R.max_items; idx += blockDim.x) {
    int w, k0 = 0;
    if (idx <= LOC) {   // recent window j0 + idx - 1, present from the step that caches its first position
      w = j0 + idx - 1;
      if (w >= R.n_windows) continue;
      k0 = max(0, R.n_sink + w * R.W - F);
    } else if (idx <= LOC + KFC) {
      const int f = idx - 1 - LOC;
      if (f >= nF) continue;
      w = ftab[f].x;
    } else {
      const int q = idx - 1 - LOC - KFC;
      if (q >= nQ) continue;
      w = qtab[q].x;
    }
    const int ew = evict[w];
    unsigned evb = 0, nxb = 0;
    for (int j = 0; j < NO; ++j) {
      if (s_evT[j] < 0) continue;
      if (ew >= 0 && ew <= s_evId[j]) evb |= 1u << j;                 // evicted by event j
      if (R.n_sink + w * R.W >= s_evT[j]) nxb |= 1u << j;             // did not exist at event j
    }
    if (!(evb | nxb)) continue;
    for (int k = k0; k < nk; ++k) {
      const unsigned me = evb & s_inh[k], mn = nxb & s_inh[k];
      if (!(me | mn)) continue;
      const float *m = mu + ((size_t)k * R.max_items + idx) * R.G;
      const float *Mk = st + k * 16;
#pragma unroll
      for (int h = 0; h < 8; ++h) {
        if (h >= G) continue;
        const float a = exp2f(m[h] - Mk[h]) * Mk[8 + h];
#pragma unroll
        for (int j = 0; j < DG_MAX_OPEN; ++j) {
          if (me >> j & 1u) ev[h][j] += a;
          if (mn >> j & 1u) nx[h][j] += a;
        }
      }
    }
  }
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int h = 0; h < 8; ++h) {
    if (h >= G) continue;
#pragma unroll
    for (int j = 0; j < DG_MAX_OPEN; ++j) {
      if (j >= NO) continue;
      const float x = warp_sum_f(ev[h][j]), y = warp_sum_f(nx[h][j]);
      if (lane == 0) {
        atomicAdd(&acc_ev[h][j], x);
        atomicAdd(&acc_nx[h][j], y);
      }
    }
  }
  __syncthreads();
  if (threadIdx.x < G * NO) {
    const int h = threadIdx.x % G, j = threadIdx.x / G;
    int steps = 0;
    for (int k = 0; k < nk; ++k) steps += (s_inh[k] >> j) & 1u;
    if (steps) {
      const size_t o = ((size_t)unit * R.h_q + (size_t)g * G + h) * DG_MAX_OPEN + j;
      Dg.fnum()[o] += (double)acc_ev[h][j];
      Dg.fden()[o] += (double)steps - (double)acc_nx[h][j];
    }
  }
}

__device__ int block_sum_i(int v, int *ws) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int off = 16; off; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  __syncthreads();
  if (lane == 0) ws[warp] = v;
  __syncthreads();
  if (warp == 0) {
    int t = lane < (int)(blockDim.x >> 5) ? ws[lane] : 0;
#pragma unroll
    for (int off = 16; off; off >>= 1) t += __shfl_xor_sync(0xffffffffu, t, off);
    if (lane == 0) ws[32] = t;
  }
  __syncthreads();
  return ws[32];
}

__device__ __forceinline__ double warp_sum_d(double v) {
#pragma unroll
  for (int off = 16; off; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  return v;
}

// One CTA per (sequence, layer) unit; runs after both caches routed at event e.  Double-precision sums
// stay in one warp: this GPU's FP64 rate is low.
__global__ void __launch_bounds__(DG_EVENT_THREADS, 1) diag_event_kernel(const CacheDev P, const CacheDev R,
                                                                         const DiagDev Dg, int e) {
  extern __shared__ __align__(16) uint8_t dsm[];
  const int N = P.n_windows;
  float *s_full = reinterpret_cast<float *>(dsm);        // [N] FullKV window scores
  float *s_pol = s_full + N;                             // [N] policy window scores
  uint8_t *s_tier = reinterpret_cast<uint8_t *>(s_pol + N);   // [N] policy tier (Local for unrouted)
  __shared__ int ws[33];
  __shared__ unsigned hist[256];
  __shared__ unsigned long long s_prefix;
  __shared__ int s_want;
  __shared__ int s_lag[DG_MAX_LAG * 4], s_lir[4];
  const int unit = blockIdx.x, tid = threadIdx.x, nt = blockDim.x, lane = tid & 31, warp = tid >> 5;
  const int *pm = P.at<const int>(P.off_meta, P.st_meta, unit);
  const int *rm = R.at<const int>(R.off_meta, R.st_meta, unit);
  const int T = pm[M_T], n_route = pm[M_NROUTE];
  if (rm[M_T] != T || rm[M_NROUTE] != n_route) {
    if (tid == 0) atomicOr(P.status(), QV_ERR_STATE);
    return;
  }
  const int NO = Dg.n_open, Hq = P.h_q;
  double *acc = Dg.acc(unit);
  int *evT = Dg.ev_T(unit), *evId = Dg.ev_id(unit);
  double *fnum = Dg.fnum() + (size_t)unit * Hq * DG_MAX_OPEN, *fden = Dg.fden() + (size_t)unit * Hq * DG_MAX_OPEN;

  // 1. events whose horizon is complete: FMM of every head (Eq. (13)), one warp; then open this event
  if (warp == 0) {
    double fs = 0.0, fc = 0.0;
    for (int j = 0; j < NO; ++j) {
      if (evT[j] < 0 || T - evT[j] < Dg.horizon) continue;
      for (int h = lane; h < Hq; h += 32) {
        const double den = fden[h * DG_MAX_OPEN + j];
        if (den > 0.0) {
          fs += fnum[h * DG_MAX_OPEN + j] / den;
          fc += 1.0;
        }
      }
    }
    fs = warp_sum_d(fs);
    fc = warp_sum_d(fc);
    __syncwarp();
    if (lane == 0) {
      acc[DA_FMM_SUM] += fs;
      acc[DA_FMM_CNT] += fc;
      int slot = -1;
      for (int j = 0; j < NO; ++j) {
        if (evT[j] >= 0 && T - evT[j] >= Dg.horizon) evT[j] = -1;
        if (evT[j] < 0 && slot < 0) slot = j;
      }
      if (slot < 0) {
        atomicOr(P.status(), QV_ERR_STATE);
      } else {
        evT[slot] = T;
        evId[slot] = e;
        for (int h = 0; h < Hq; ++h) fnum[h * DG_MAX_OPEN + slot] = fden[h * DG_MAX_OPEN + slot] = 0.0;
      }
    }
  }
  if (tid < DG_MAX_LAG * 4) s_lag[tid] = 0;
  if (tid < 4) s_lir[tid] = 0;

  // 2. per window: evictions, the retained set, both runs' scores (sums of the KV-head partials, head order)
  const uint8_t *state = P.at<const uint8_t>(P.off_state, P.st_state, unit);
  const float *sp = P.at<const float>(P.off_score, P.st_score, unit);
  const float *sr = R.at<const float>(R.off_score, R.st_score, unit);
  int *evict = Dg.evict(unit);
  uint8_t *ret = Dg.ret(unit);
  int inter = 0, uni = 0;
  for (int w = tid; w < N; w += nt) {
    const bool routed = w < n_route;
    const int tier = routed ? (state[w] & 3) : TIER_LOCAL;
    if (routed && tier == TIER_EVICT && evict[w] < 0) evict[w] = e;
    const int now = routed && (tier == TIER_FULL || tier == TIER_QUANT);
    const int prev = ret[w];
    inter += prev & now;
    uni += prev | now;
    ret[w] = (uint8_t)now;
    float a = sr[w], c = sp[w];
    for (int g = 1; g < P.h_kv; ++g) {
      a += sr[(size_t)g * N + w];
      c += sp[(size_t)g * N + w];
    }
    s_full[w] = a;
    s_pol[w] = c;
    s_tier[w] = (uint8_t)tier;
  }
  inter = block_sum_i(inter, ws);   // its barriers also publish the shared arrays
  uni = block_sum_i(uni, ws);

  // 3. one warp: QSA / R_Q over the Quantized windows (Eq. (16)-(17)), tier shares over the windows that
  //    exist (Eq. (15)), churn (Eq. (14))
  if (warp == 0) {
    double dot = 0, nq = 0, nf = 0, sq = 0, sf = 0, mz[4] = {0, 0, 0, 0};
    for (int w = lane; w < N; w += 32) {
      const double a = s_full[w], c = s_pol[w];
      const int tier = s_tier[w];
      if (tier == TIER_QUANT) {
        dot += c * a;
        nq += c * c;
        nf += a * a;
        sq += c;
        sf += a;
      }
      if (P.n_sink + w * P.W < T) mz[tier] += a;
    }
    dot = warp_sum_d(dot);
    nq = warp_sum_d(nq);
    nf = warp_sum_d(nf);
    sq = warp_sum_d(sq);
    sf = warp_sum_d(sf);
#pragma unroll
    for (int z = 0; z < 4; ++z) mz[z] = warp_sum_d(mz[z]);
    if (lane == 0) {
      if (e >= 1 && uni > 0) {
        acc[DA_CHURN_SUM] += 1.0 - (double)inter / (double)uni;
        acc[DA_CHURN_CNT] += 1.0;
      }
      if (e >= 1 && nq > 0 && nf > 0) {   // a non-empty Quantized tier
        acc[DA_QSA_SUM] += dot / sqrt(nq * nf);
        acc[DA_RQ_SUM] += sq / sf;
        acc[DA_QSA_CNT] += 1.0;
      }
      const double tot = mz[0] + mz[1] + mz[2] + mz[3];
      // shares in the order Full, Quantized, Evicted, Local
      acc[DA_MU + 0] = tot > 0 ? mz[TIER_FULL] / tot : 0.0;
      acc[DA_MU + 1] = tot > 0 ? mz[TIER_QUANT] / tot : 0.0;
      acc[DA_MU + 2] = tot > 0 ? mz[TIER_EVICT] / tot : 0.0;
      acc[DA_MU + 3] = tot > 0 ? mz[TIER_LOCAL] / tot : 0.0;
      acc[DA_EVENTS] = e + 1;
    }
  }

  // 4. the FullKV top-K_f selection: radix select of the K_f-th smallest key (score descending, window
  //    id ascending) among the routed windows, 8 bits per pass
  auto key_of = [&](int w) -> unsigned long long {
    return ((unsigned long long)(~__float_as_uint(s_full[w])) << 32) | (unsigned)w;
  };
  const bool all_in = n_route <= P.k_f;
  if (tid == 0) {
    s_prefix = 0ull;
    s_want = P.k_f;   // 1-based rank of the last selected key
  }
  unsigned long long mask = 0ull;
  for (int shift = 56; shift >= 0 && !all_in; shift -= 8) {
    for (int i = tid; i < 256; i += nt) hist[i] = 0u;
    __syncthreads();
    const unsigned long long prefix = s_prefix;
    for (int w = tid; w < n_route; w += nt) {
      const unsigned long long k = key_of(w);
      if ((k & mask) == prefix) atomicAdd(&hist[(k >> shift) & 255u], 1u);
    }
    __syncthreads();
    if (warp == 0) {
      // lane l holds bins 8l .. 8l+7; find the bin where the running count reaches the wanted rank
      unsigned c[8], sum = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        c[i] = hist[8 * lane + i];
        sum += c[i];
      }
      unsigned incl = sum;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const unsigned y = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += y;
      }
      const unsigned want = (unsigned)s_want;
      unsigned before = incl - sum;
      if (before < want && want <= incl) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          if (before < want && want <= before + c[i]) {
            s_prefix = prefix | ((unsigned long long)(8 * lane + i) << shift);
            s_want = (int)(want - before);
          }
          before += c[i];
        }
      }
    }
    mask |= 255ull << shift;
    __syncthreads();
  }
  const unsigned long long kth = s_prefix;

  // 5. selections X of the policy's Full tier and of the FullKV top-K_f: history, LIR episodes, lags
  uint32_t *xp = Dg.xpol(unit), *xo = Dg.xorc(unit);
  int *rp = Dg.runpol(unit), *ro = Dg.runorc(unit), *since = Dg.since(unit);
  const int m = Dg.lir_m;
  for (int w = tid; w < n_route; w += nt) {
    const uint32_t Xp = s_tier[w] == TIER_FULL ? 1u : 0u, Xo = (all_in || key_of(w) <= kth) ? 1u : 0u;
    if (since[w] < 0) {
      since[w] = e;
      xp[w] = xo[w] = 0u;
      rp[w] = ro[w] = -1;
    }
    const uint32_t hp = (xp[w] << 1) | Xp, ho = (xo[w] << 1) | Xo;
    xp[w] = hp;
    xo[w] = ho;
    // an episode is a run of inactive events after the window was selected: eligible at m, rescued on return
    auto lir = [&](int &run, uint32_t X, int *cnt) {
      if (X) {
        if (run >= m) atomicAdd(&cnt[1], 1);
        run = 0;
      } else if (run >= 0) {
        ++run;
        if (run == m) atomicAdd(&cnt[0], 1);
      }
    };
    int r0 = rp[w], r1 = ro[w];
    lir(r0, Xp, s_lir);
    lir(r1, Xo, s_lir + 2);
    rp[w] = r0;
    ro[w] = r1;
    const int span = min(DG_MAX_LAG, e - since[w]);
    for (int d = 1; d <= span; ++d) atomicAdd(&s_lag[(d - 1) * 4 + (int)(((hp >> d) & 1u) * 2u + Xp)], 1);
  }
  __syncthreads();
  if (tid < 4) acc[DA_LIR + tid] += (double)s_lir[tid];
  if (tid < DG_MAX_LAG * 4) acc[DA_LAG + tid] += (double)s_lag[tid];
}

cudaError_t launch_diag_collect(const CacheDev &R, const DiagDev &Dg, cudaStream_t s) {
  diag_collect_kernel<<<dim3(R.h_kv, R.B, R.L), DG_COLLECT_THREADS, 0, s>>>(R, Dg);
  return cudaGetLastError();
}

cudaError_t launch_diag_event(const CacheDev &P, const CacheDev &R, const DiagDev &Dg, int e, cudaStream_t s) {
  const size_t smem = (size_t)P.n_windows * 9;
  static SmemOptIn optin;
  const cudaError_t err = optin.ensure(diag_event_kernel, 8192 * 9);
  if (err != cudaSuccess) return err;
  diag_event_kernel<<<P.B * P.L, DG_EVENT_THREADS, smem, s>>>(P, R, Dg, e);
  return cudaGetLastError();
}

}  // namespace qv
