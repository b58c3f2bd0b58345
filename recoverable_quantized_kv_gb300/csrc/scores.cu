// Prefill window scores from prompt attention.
//
// QEvict (arXiv 2608.05326) §4.2, last paragraph: during prefill, prompt attention initialises the
// window scores.  Every prompt query tau attends causally over keys i <= tau; the initial score of
// window j is (1/H_q) * sum_h sum_tau sum_{i in w_j, i <= tau} a_tau^h(i).
//
// Two passes over the prompt, no score matrix is stored:
//   pass 1 (one thread per query row): row log2-sum-exp of the scaled logits, online;
//   pass 2 (one thread per key column): column sum of 2^(logit - rowLSE) over the queries at or
//            after the key;
//   pass 3: per-window sums over the heads in a fixed order (deterministic).
// Key / query tiles are staged in shared memory and read as broadcasts.
#include "cache_dev.cuh"
#include "common.cuh"

namespace qv {

constexpr int SC_ROWS = 128;   // threads per CTA = rows (pass 1) or columns (pass 2)
constexpr int SC_TILE = 32;    // keys (pass 1) or queries (pass 2) per shared-memory tile

__global__ void __launch_bounds__(SC_ROWS) rowstat_kernel(const CacheDev C, const __nv_bfloat16 *q,
                                                          const __nv_bfloat16 *k, float scale_log2) {
  __shared__ __align__(16) float kt[SC_TILE][D];
  const int P = C.prompt_len;
  const int h = blockIdx.y, b = blockIdx.z, g = h / C.G;
  const int r0 = blockIdx.x * SC_ROWS, tau = r0 + threadIdx.x;
  float qr[D];
  if (tau < P) {
    const __nv_bfloat16 *qp = q + (((size_t)b * P + tau) * C.h_q + h) * D;
#pragma unroll
    for (int d = 0; d < D; ++d) qr[d] = __bfloat162float(qp[d]);
  } else {
#pragma unroll
    for (int d = 0; d < D; ++d) qr[d] = 0.f;
  }
  float m = -INFINITY, l = 0.f;
  const int last = min(P - 1, r0 + SC_ROWS - 1);
  for (int k0 = 0; k0 <= last; k0 += SC_TILE) {
    __syncthreads();
    for (int idx = threadIdx.x; idx < SC_TILE * D; idx += SC_ROWS) {
      const int kk = k0 + idx / D;
      kt[idx / D][idx % D] = kk < P ? __bfloat162float(k[(((size_t)b * P + kk) * C.h_kv + g) * D + idx % D]) : 0.f;
    }
    __syncthreads();
    const int n = min(SC_TILE, tau - k0 + 1);
    for (int kk = 0; kk < n; ++kk) {
      float acc = 0.f;
#pragma unroll
      for (int d = 0; d < D; d += 4) {
        const float4 kv = *reinterpret_cast<const float4 *>(&kt[kk][d]);
        acc = fmaf(qr[d], kv.x, acc);
        acc = fmaf(qr[d + 1], kv.y, acc);
        acc = fmaf(qr[d + 2], kv.z, acc);
        acc = fmaf(qr[d + 3], kv.w, acc);
      }
      const float s = acc * scale_log2;
      if (s > m) {
        l = l * exp2f(m - s) + 1.f;
        m = s;
      } else {
        l += exp2f(s - m);
      }
    }
  }
  if (tau < P) reinterpret_cast<float *>(C.arena + C.off_rowstat)[((size_t)b * C.h_q + h) * P + tau] = m + __log2f(l);
}

__global__ void __launch_bounds__(SC_ROWS) colsum_kernel(const CacheDev C, const __nv_bfloat16 *q,
                                                         const __nv_bfloat16 *k, float scale_log2) {
  __shared__ __align__(16) float qt[SC_TILE][D];
  __shared__ float rs[SC_TILE];
  const int P = C.prompt_len;
  const int h = blockIdx.y, b = blockIdx.z, g = h / C.G;
  const int c0 = blockIdx.x * SC_ROWS, i = c0 + threadIdx.x;
  const float *rowstat = reinterpret_cast<const float *>(C.arena + C.off_rowstat) + ((size_t)b * C.h_q + h) * P;
  float kr[D];
  if (i < P) {
    const __nv_bfloat16 *kp = k + (((size_t)b * P + i) * C.h_kv + g) * D;
#pragma unroll
    for (int d = 0; d < D; ++d) kr[d] = __bfloat162float(kp[d]);
  } else {
#pragma unroll
    for (int d = 0; d < D; ++d) kr[d] = 0.f;
  }
  float col = 0.f;
  for (int t0 = (c0 / SC_TILE) * SC_TILE; t0 < P; t0 += SC_TILE) {
    __syncthreads();
    for (int idx = threadIdx.x; idx < SC_TILE * D; idx += SC_ROWS) {
      const int tt = t0 + idx / D;
      qt[idx / D][idx % D] = tt < P ? __bfloat162float(q[(((size_t)b * P + tt) * C.h_q + h) * D + idx % D]) : 0.f;
    }
    if (threadIdx.x < SC_TILE) rs[threadIdx.x] = t0 + threadIdx.x < P ? rowstat[t0 + threadIdx.x] : 0.f;
    __syncthreads();
    if (i >= P) continue;
    const int from = max(0, i - t0), to = min(SC_TILE, P - t0);
    for (int tt = from; tt < to; ++tt) {
      float acc = 0.f;
#pragma unroll
      for (int d = 0; d < D; d += 4) {
        const float4 qv = *reinterpret_cast<const float4 *>(&qt[tt][d]);
        acc = fmaf(kr[d], qv.x, acc);
        acc = fmaf(kr[d + 1], qv.y, acc);
        acc = fmaf(kr[d + 2], qv.z, acc);
        acc = fmaf(kr[d + 3], qv.w, acc);
      }
      col += exp2f(acc * scale_log2 - rs[tt]);
    }
  }
  if (i < P) reinterpret_cast<float *>(C.arena + C.off_colsum)[((size_t)b * C.h_q + h) * P + i] = col;
}

__global__ void window_sum_kernel(const CacheDev C, float *s0) {
  const int P = C.prompt_len, W = C.W;
  const int b = blockIdx.y;
  const int npw = (P - C.n_sink + W - 1) / W;
  const int j = blockIdx.x * blockDim.x + threadIdx.x;
  if (j >= npw) return;
  const float *col = reinterpret_cast<const float *>(C.arena + C.off_colsum) + (size_t)b * C.h_q * P;
  const int lo = C.n_sink + j * W, hi = min(P, lo + W);
  float s = 0.f;
  for (int h = 0; h < C.h_q; ++h)
    for (int i = lo; i < hi; ++i) s += col[(size_t)h * P + i];
  s0[(size_t)b * npw + j] = s / (float)C.h_q;
}

cudaError_t launch_prefill_scores(const CacheDev &C, const __nv_bfloat16 *q, const __nv_bfloat16 *k, float *s0,
                                  cudaStream_t stream) {
  const float scale_log2 = 1.4426950408889634f / sqrtf((float)D);
  const int P = C.prompt_len;
  dim3 grid((P + SC_ROWS - 1) / SC_ROWS, C.h_q, C.B);
  rowstat_kernel<<<grid, SC_ROWS, 0, stream>>>(C, q, k, scale_log2);
  colsum_kernel<<<grid, SC_ROWS, 0, stream>>>(C, q, k, scale_log2);
  const int npw = (P - C.n_sink + C.W - 1) / C.W;
  window_sum_kernel<<<dim3((npw + 127) / 128, C.B), 128, 0, stream>>>(C, s0);
  return cudaGetLastError();
}


// ----------------------------------------------------------------------------- deferred score updates
//
// QEvict §4.2 Eq. (1): after every decode step the score of window w grows by the attention mass
// the step put on it, S(w) += (1/H_q) sum_h sum_{i in w} a^h(i).  The decode kernel records, per
// step, every window's log2-sum-exp per query head (mu) and the merged max M and 1/L per head; this
// kernel turns them into masses 2^(mu - M) / L and adds them to the per-KV-head score partials one
// step at a time in decode order, the same floating-point sequence as adding after every step.
// Scores are read only by the router, which flushes first.  One CTA per (KV head, sequence, layer).
__global__ void __launch_bounds__(256) flush_kernel(const CacheDev C, float inv_hq) {
  extern __shared__ float st[];   // [omega][16]
  const int g = blockIdx.x, b = blockIdx.y, layer = blockIdx.z;
  const int unit = layer * C.B + b, bg = b * C.h_kv + g;
  int *meta = C.at<int>(C.off_meta, C.st_meta, unit);
  __shared__ int s_meta[8];
  if (threadIdx.x < 8) s_meta[threadIdx.x] = meta[threadIdx.x];
  __syncthreads();
  const int T = s_meta[M_T], F = s_meta[M_FLUSHT], j0 = s_meta[M_NROUTE];
  const int nF = s_meta[M_FCOUNT], nQ = s_meta[M_QCOUNT];
  const int nk = T - F;
  if (nk < 0 || nk > C.omega) {
    if (threadIdx.x == 0) atomicOr(C.status(), QV_ERR_STATE);
  } else if (nk > 0) {
    const float *ms = reinterpret_cast<const float *>(C.arena + C.off_mstat + C.st_mstat_layer * layer) +
                      (size_t)bg * C.omega * 16;
    for (int i = threadIdx.x; i < nk * 16; i += blockDim.x) st[i] = ms[i];
    __syncthreads();
    const float *mu = reinterpret_cast<const float *>(C.arena + C.off_mu + C.st_mu_layer * layer) +
                      (size_t)bg * C.omega * C.max_items * 8;
    float *score = C.at<float>(C.off_score, C.st_score, unit) + (size_t)g * C.n_windows;
    const int2 *ftab = C.at<const int2>(C.off_ftab, C.st_ftab, unit);
    const int2 *qtab = C.at<const int2>(C.off_qtab, C.st_qtab, unit);
    const int LOC = C.loc_items(), KFC = C.kf_cap();
    const int G = C.G;
    for (int idx = 1 + threadIdx.x; idx < C.max_items; idx += blockDim.x) {
      int w, k0 = 0;
      if (idx <= LOC) {   // recent window j0 + idx - 1: in the step of T_k tokens once T_k >= n_sink + w W
        w = j0 + idx - 1;
        if (w >= C.n_windows) continue;
        k0 = max(0, C.n_sink + w * C.W - F);
        if (k0 >= nk) continue;
      } else if (idx <= LOC + KFC) {
        const int f = idx - 1 - LOC;
        if (f >= nF) continue;
        w = ftab[f].x;
      } else {
        const int q = idx - 1 - LOC - KFC;
        if (q >= nQ) continue;
        w = qtab[q].x;
      }
      float s = score[w];
      for (int k = k0; k < nk; ++k) {
        const float *m = mu + ((size_t)k * C.max_items + idx) * 8;
        const float *Mk = st + k * 16;
        float a = 0.f;
        for (int h = 0; h < G; ++h) a = fmaf(exp2f(m[h] - Mk[h]), Mk[8 + h], a);
        s = s + a * inv_hq;
      }
      score[w] = s;
    }
  }
  // the last of the unit's CTAs to finish records the flush (every CTA has read M_FLUSHT by then)
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned *ctr = reinterpret_cast<unsigned *>(C.arena + C.off_flushctr) + unit;
    unsigned prev;
    asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], 1;" : "=r"(prev) : "l"(ctr) : "memory");
    if (prev == (unsigned)(C.h_kv - 1)) {
      *ctr = 0u;
      if (nk >= 0 && nk <= C.omega) meta[M_FLUSHT] = T;
    }
  }
}

cudaError_t launch_flush(const CacheDev &C, cudaStream_t s) {
  flush_kernel<<<dim3(C.h_kv, C.B, C.L), 256, (size_t)C.omega * 16 * sizeof(float), s>>>(C, 1.0f / (float)C.h_q);
  return cudaGetLastError();
}

}  // namespace qv
