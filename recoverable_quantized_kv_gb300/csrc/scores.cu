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

}  // namespace qv
