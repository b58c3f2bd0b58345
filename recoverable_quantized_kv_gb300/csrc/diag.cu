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
#include "diag_dev.cuh"

namespace qv {

constexpr int DG_COLLECT_THREADS = 256;
constexpr int DG_EVENT_THREADS = 1024;

__device__ __forceinline__ float warp_sum_f(float v) {
#pragma unroll
  for (int off = 16; off; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  return v;
}

// One CTA per (KV head g, sequence, layer) of R.
__global__ void __launch_bounds__(DG_COLLECT_THREADS) diag_collect_kernel(const CacheDev R, const DiagDev Dg) {
  const int g = blockIdx.x, b = blockIdx.y, layer = blockIdx.z;
  const int unit = layer * R.B + b, bg = b * R.h_kv + g;
  const int G = R.G, NO = Dg.n_open;
  __shared__ int s_meta[8];
  __shared__ float st[DG_MAX_OMEGA * 16];                  // merged max and 1/L of each pending step
  __shared__ int s_evT[DG_MAX_OPEN], s_evId[DG_MAX_OPEN];
  __shared__ float acc_tot[8], acc_ex[8][DG_MAX_OPEN], acc_ev[8][DG_MAX_OPEN];
  const int *meta = R.at<const int>(R.off_meta, R.st_meta, unit);
  if (threadIdx.x < 8) s_meta[threadIdx.x] = meta[threadIdx.x];
  if (threadIdx.x < NO) {
    s_evT[threadIdx.x] = Dg.ev_T(unit)[threadIdx.x];
    s_evId[threadIdx.x] = Dg.ev_id(unit)[threadIdx.x];
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
  const float *mu = reinterpret_cast<const float *>(R.arena + R.off_mu + R.st_mu_layer * layer) +
                    (size_t)bg * R.omega * R.max_items * 8;
  const int2 *ftab = R.at<const int2>(R.off_ftab, R.st_ftab, unit);
  const int2 *qtab = R.at<const int2>(R.off_qtab, R.st_qtab, unit);
  const int *evict = Dg.evict(unit);
  const int LOC = R.loc_items(), KFC = R.kf_cap();
  const int lane = threadIdx.x & 31;
  for (int k = 0; k < nk; ++k) {
    const int Tk = F + k + 1;   // tokens cached after step k; its query sits at position Tk - 1
    if (threadIdx.x < 8 * (1 + 2 * DG_MAX_OPEN)) {
      const int h = threadIdx.x & 7, j = threadIdx.x >> 3;
      if (j == 0) acc_tot[h] = 0.f;
      else if (j <= DG_MAX_OPEN) acc_ex[h][j - 1] = 0.f;
      else acc_ev[h][j - 1 - DG_MAX_OPEN] = 0.f;
    }
    __syncthreads();
    // per thread: its items' masses for every head, split by open event
    float tot[8], ex[8][DG_MAX_OPEN], ev[8][DG_MAX_OPEN];
#pragma unroll
    for (int h = 0; h < 8; ++h) {
      tot[h] = 0.f;
#pragma unroll
      for (int j = 0; j < DG_MAX_OPEN; ++j) ex[h][j] = ev[h][j] = 0.f;
    }
    for (int idx = 1 + threadIdx.x; idx < R.max_items; idx += blockDim.x) {
      int w;
      if (idx <= LOC) {   // recent window j0 + idx - 1, present once its first position is cached
        w = j0 + idx - 1;
        if (w >= R.n_windows || R.n_sink + w * R.W > F + k) continue;
      } else if (idx <= LOC + KFC) {
        const int f = idx - 1 - LOC;
        if (f >= nF) continue;
        w = ftab[f].x;
      } else {
        const int q = idx - 1 - LOC - KFC;
        if (q >= nQ) continue;
        w = qtab[q].x;
      }
      const float *m = mu + ((size_t)k * R.max_items + idx) * 8;
      const float *Mk = st + k * 16;
      const int ew = evict[w];
#pragma unroll
      for (int h = 0; h < 8; ++h) {
        if (h >= G) continue;
        const float a = exp2f(m[h] - Mk[h]) * Mk[8 + h];
        tot[h] += a;
#pragma unroll
        for (int j = 0; j < DG_MAX_OPEN; ++j) {
          if (j >= NO || s_evT[j] < 0) continue;
          if (R.n_sink + w * R.W < s_evT[j]) ex[h][j] += a;                  // existed at event j
          if (ew >= 0 && ew <= s_evId[j]) ev[h][j] += a;                     // evicted by then
        }
      }
    }
#pragma unroll
    for (int h = 0; h < 8; ++h) {
      if (h >= G) continue;
      const float t = warp_sum_f(tot[h]);
      if (lane == 0) atomicAdd(&acc_tot[h], t);
#pragma unroll
      for (int j = 0; j < DG_MAX_OPEN; ++j) {
        if (j >= NO) continue;
        const float x = warp_sum_f(ex[h][j]), y = warp_sum_f(ev[h][j]);
        if (lane == 0) {
          atomicAdd(&acc_ex[h][j], x);
          atomicAdd(&acc_ev[h][j], y);
        }
      }
    }
    __syncthreads();
    // the sinks hold the rest of the step's attention; the step counts for an event inside its horizon
    if (threadIdx.x < G * NO) {
      const int h = threadIdx.x % G, j = threadIdx.x / G;
      if (s_evT[j] >= 0 && Tk > s_evT[j] && Tk - s_evT[j] <= Dg.horizon) {
        const size_t o = ((size_t)unit * R.h_q + (size_t)g * G + h) * DG_MAX_OPEN + j;
        Dg.fnum()[o] += (double)acc_ev[h][j];
        Dg.fden()[o] += (double)(1.f - acc_tot[h]) + (double)acc_ex[h][j];
      }
    }
    __syncthreads();
  }
}

__device__ double block_sum_d(double v, double *wsum) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int off = 16; off; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  __syncthreads();
  if (lane == 0) wsum[warp] = v;
  __syncthreads();
  double t = 0.0;
  for (int w = 0; w < (int)(blockDim.x >> 5); ++w) t += wsum[w];
  __syncthreads();
  return t;
}

// One CTA per (sequence, layer) unit; runs after both caches routed at event e.
__global__ void __launch_bounds__(DG_EVENT_THREADS, 1) diag_event_kernel(const CacheDev P, const CacheDev R,
                                                                         const DiagDev Dg, int e) {
  extern __shared__ float s_full[];   // [n_windows] FullKV scores (the oracle selection ranks them)
  __shared__ double wsum[32];
  __shared__ int s_lag[DG_MAX_LAG * 4], s_lir[4];
  const int unit = blockIdx.x, tid = threadIdx.x, nt = blockDim.x;
  const int *pm = P.at<const int>(P.off_meta, P.st_meta, unit);
  const int *rm = R.at<const int>(R.off_meta, R.st_meta, unit);
  const int T = pm[M_T], n_route = pm[M_NROUTE];
  if (rm[M_T] != T || rm[M_NROUTE] != n_route) {
    if (tid == 0) atomicOr(P.status(), QV_ERR_STATE);
    return;
  }
  const int N = P.n_windows, NO = Dg.n_open, Hq = P.h_q;
  double *acc = Dg.acc(unit);
  int *evT = Dg.ev_T(unit), *evId = Dg.ev_id(unit);
  double *fnum = Dg.fnum() + (size_t)unit * Hq * DG_MAX_OPEN, *fden = Dg.fden() + (size_t)unit * Hq * DG_MAX_OPEN;

  // 1. events whose horizon is complete: FMM of every head (Eq. (13)); then open this event
  if (tid == 0) {
    for (int j = 0; j < NO; ++j) {
      if (evT[j] < 0 || T - evT[j] < Dg.horizon) continue;
      for (int h = 0; h < Hq; ++h) {
        const double den = fden[h * DG_MAX_OPEN + j];
        if (den > 0.0) {
          acc[DA_FMM_SUM] += fnum[h * DG_MAX_OPEN + j] / den;
          acc[DA_FMM_CNT] += 1.0;
        }
      }
      evT[j] = -1;
    }
    int slot = -1;
    for (int j = 0; j < NO && slot < 0; ++j)
      if (evT[j] < 0) slot = j;
    if (slot < 0) {
      atomicOr(P.status(), QV_ERR_STATE);
    } else {
      evT[slot] = T;
      evId[slot] = e;
      for (int h = 0; h < Hq; ++h) fnum[h * DG_MAX_OPEN + slot] = fden[h * DG_MAX_OPEN + slot] = 0.0;
    }
  }
  if (tid < DG_MAX_LAG * 4) s_lag[tid] = 0;
  if (tid < 4) s_lir[tid] = 0;

  // 2. per window: evictions, retained sets, scores, tier masses
  const uint8_t *state = P.at<const uint8_t>(P.off_state, P.st_state, unit);
  const float *sp = P.at<const float>(P.off_score, P.st_score, unit);
  const float *sr = R.at<const float>(R.off_score, R.st_score, unit);
  int *evict = Dg.evict(unit);
  uint8_t *ret = Dg.ret(unit);
  double inter = 0, uni = 0, dot = 0, nq = 0, nf = 0, sq = 0, sf = 0, mz[4] = {0, 0, 0, 0};
  for (int w = tid; w < N; w += nt) {
    const bool routed = w < n_route;
    const int tier = routed ? (state[w] & 3) : TIER_LOCAL;
    if (routed && tier == TIER_EVICT && evict[w] < 0) evict[w] = e;
    const int now = routed && (tier == TIER_FULL || tier == TIER_QUANT);
    const int prev = ret[w];
    inter += (double)(prev & now);
    uni += (double)(prev | now);
    ret[w] = (uint8_t)now;
    float a = sr[w], c = sp[w];   // window scores: the sum of the KV-head partials in head order
    for (int g = 1; g < P.h_kv; ++g) {
      a += sr[(size_t)g * N + w];
      c += sp[(size_t)g * N + w];
    }
    s_full[w] = a;
    if (tier == TIER_QUANT) {
      dot += (double)c * a;
      nq += (double)c * c;
      nf += (double)a * a;
      sq += c;
      sf += a;
    }
    if (P.n_sink + w * P.W < T) mz[tier] += a;
  }
  inter = block_sum_d(inter, wsum);
  uni = block_sum_d(uni, wsum);
  dot = block_sum_d(dot, wsum);
  nq = block_sum_d(nq, wsum);
  nf = block_sum_d(nf, wsum);
  sq = block_sum_d(sq, wsum);
  sf = block_sum_d(sf, wsum);
#pragma unroll
  for (int z = 0; z < 4; ++z) mz[z] = block_sum_d(mz[z], wsum);   // also orders s_full before step 3
  if (tid == 0) {
    if (e >= 1 && uni > 0) {
      acc[DA_CHURN_SUM] += 1.0 - inter / uni;
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

  // 3. selections X of the policy's Full tier and of the FullKV top-K_f: history, LIR episodes, lags
  uint32_t *xp = Dg.xpol(unit), *xo = Dg.xorc(unit);
  int *rp = Dg.runpol(unit), *ro = Dg.runorc(unit), *since = Dg.since(unit);
  const int m = Dg.lir_m;
  for (int w = tid; w < n_route; w += nt) {
    const int tier = state[w] & 3;
    const float a = s_full[w];
    int rank = 0;
    for (int v = 0; v < n_route; ++v) {
      const float b = s_full[v];
      rank += (b > a || (b == a && v < w)) ? 1 : 0;
    }
    const uint32_t Xp = tier == TIER_FULL ? 1u : 0u, Xo = rank < P.k_f ? 1u : 0u;
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
  const size_t smem = (size_t)P.n_windows * sizeof(float);
  static bool attr_set[64] = {};
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_set[dev]) {
    err = cudaFuncSetAttribute(diag_event_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 8192 * 4);
    if (err != cudaSuccess) return err;
    attr_set[dev] = true;
  }
  diag_event_kernel<<<P.B * P.L, DG_EVENT_THREADS, smem, s>>>(P, R, Dg, e);
  return cudaGetLastError();
}

}  // namespace qv
