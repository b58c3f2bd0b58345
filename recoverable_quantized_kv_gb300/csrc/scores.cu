// Prefill window scores from prompt attention.
//
// QEvict (arXiv 2608.05326) §4.2, last paragraph: during prefill, prompt attention initialises the
// window scores.  Every prompt query tau attends causally over keys i <= tau; the initial score of
// window j is (1/H_q) * sum_h sum_tau sum_{i in w_j, i <= tau} a_tau^h(i).
//
// Two passes over the prompt, no score matrix is stored:
//   pass 1: row log2-sum-exp of the scaled logits of every query, online;
//   pass 2: column sum of 2^(logit - rowLSE) of every key over the queries at or after it;
//   pass 3: per-window sums over the heads in a fixed order (deterministic).
#include "cache_dev.cuh"
#include "common.cuh"

namespace qv {

// Both passes are flash-attention-shaped contractions on the tensor cores (mma.m16n8k16, bf16 in,
// fp32 accumulate).  A CTA of 4 warps owns 64 rows (queries in pass 1, keys in pass 2), each warp
// 16 of them with its A fragments in registers; the other operand streams through shared memory in
// 64-row tiles (double-buffered with cp.async, rows padded to 136 elements so ldmatrix is free of
// bank conflicts), and every row's reduction stays inside its 4 owning lanes.
constexpr int SC_WARPS = 4;
constexpr int SC_TILE = 64;            // rows per CTA and rows per streamed tile
constexpr int SC_LD = D + 8;           // padded shared-memory row, elements

__device__ __forceinline__ void cp_async16(void *smem_dst, const void *gsrc, bool valid) {
  const int n = valid ? 16 : 0;        // zero-fill rows past the prompt
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(smem_dst)), "l"(gsrc), "r"(n) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

__device__ __forceinline__ void ldsm_x4(const void *p, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(smem_u32(p)));
}

// Stage rows [r0, r0 + 64) of a [B][P][heads][D] bf16 tensor (head hh of sequence b) into a
// padded shared tile; rows at or past P are zero-filled.
__device__ __forceinline__ void stage_tile(__nv_bfloat16 *dst, const __nv_bfloat16 *src, int b, int P, int heads,
                                           int hh, int r0) {
  for (int idx = threadIdx.x; idx < SC_TILE * (D / 8); idx += SC_WARPS * 32) {
    const int r = idx / (D / 8), c = (idx % (D / 8)) * 8;
    const int row = r0 + r;
    const bool valid = row < P;
    const __nv_bfloat16 *g = src + (((size_t)b * P + (valid ? row : 0)) * heads + hh) * D + c;
    cp_async16(dst + r * SC_LD + c, g, valid);
  }
  cp_async_commit();
}

// A fragments of 16 rows [r0, r0 + 16) x 128 dims straight from global (zero rows past P).
__device__ __forceinline__ void load_a_frags(uint32_t (&a)[8][4], const __nv_bfloat16 *src, int b, int P, int heads,
                                             int hh, int r0) {
  const int lane = threadIdx.x & 31, gl = lane >> 2, tl = lane & 3;
  const int ra = r0 + gl, rb = r0 + gl + 8;
  const uint32_t *pa = reinterpret_cast<const uint32_t *>(src + (((size_t)b * P + min(ra, P - 1)) * heads + hh) * D);
  const uint32_t *pb = reinterpret_cast<const uint32_t *>(src + (((size_t)b * P + min(rb, P - 1)) * heads + hh) * D);
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    a[j][0] = ra < P ? __ldg(pa + 8 * j + tl) : 0u;
    a[j][1] = rb < P ? __ldg(pb + 8 * j + tl) : 0u;
    a[j][2] = ra < P ? __ldg(pa + 8 * j + tl + 4) : 0u;
    a[j][3] = rb < P ? __ldg(pb + 8 * j + tl + 4) : 0u;
  }
}

// S[16 x 64] = A (16 rows x 128) . B^T, B = the 64 staged rows; s[n][*] covers tile columns 8n..8n+7.
__device__ __forceinline__ void tile_mma(float (&s)[8][4], const uint32_t (&a)[8][4], const __nv_bfloat16 *tile) {
  const int lane = threadIdx.x & 31;
  // ldmatrix x4 row addresses: matrices (n, dims 16j..+7), (n, 16j+8..), (n+1, 16j..), (n+1, 16j+8..)
  const int mrow = (lane & 7) + ((lane >> 4) << 3), mcol = ((lane >> 3) & 1) * 8;
#pragma unroll
  for (int n = 0; n < 8; ++n) s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.f;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
#pragma unroll
    for (int n = 0; n < 8; n += 2) {
      uint32_t b0, b1, b2, b3;
      ldsm_x4(tile + (8 * n + mrow) * SC_LD + 16 * j + mcol, b0, b1, b2, b3);
      mma_bf16(s[n], a[j][0], a[j][1], a[j][2], a[j][3], b0, b1);
      mma_bf16(s[n + 1], a[j][0], a[j][1], a[j][2], a[j][3], b2, b3);
    }
  }
}

// Pass 1: rowstat[b][h][tau] = log2 sum_{i <= tau} 2^(q_tau . k_i * scale_log2).
__global__ void __launch_bounds__(SC_WARPS * 32) rowstat_kernel(const CacheDev C, const __nv_bfloat16 *q,
                                                                const __nv_bfloat16 *k, float scale_log2) {
  __shared__ __align__(128) __nv_bfloat16 kt[2][SC_TILE * SC_LD];
  const int P = C.prompt_len;
  const int h = blockIdx.y, b = blockIdx.z, g = h / C.G;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gl = lane >> 2, tl = lane & 3;
  const int q0 = blockIdx.x * SC_TILE, r0 = q0 + 16 * warp;
  uint32_t qa[8][4];
  load_a_frags(qa, q, b, P, C.h_q, h, r0);
  float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};   // rows gl, gl+8; l is this lane's partial sum
  const int ntiles = q0 / SC_TILE + 1;   // key tiles up to the diagonal
  stage_tile(kt[0], k, b, P, C.h_kv, g, 0);
  for (int t = 0; t < ntiles; ++t) {
    if (t + 1 < ntiles) {
      stage_tile(kt[(t + 1) & 1], k, b, P, C.h_kv, g, (t + 1) * SC_TILE);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    float s[8][4];
    tile_mma(s, qa, kt[t & 1]);
    const int k0 = t * SC_TILE;
    float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int n = 0; n < 8; ++n)
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int row = r0 + gl + ((c >> 1) << 3), key = k0 + 8 * n + 2 * tl + (c & 1);
        const float v = (key <= row && key < P) ? s[n][c] * scale_log2 : -INFINITY;
        s[n][c] = v;
        mx[c >> 1] = fmaxf(mx[c >> 1], v);
      }
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
      mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
      const float mn = fmaxf(m[r], mx[r]);
      if (mn != -INFINITY) {
        l[r] *= exp2f(m[r] - mn);
        m[r] = mn;
      }
    }
#pragma unroll
    for (int n = 0; n < 8; ++n)
#pragma unroll
      for (int c = 0; c < 4; ++c)
        if (s[n][c] != -INFINITY) l[c >> 1] += exp2f(s[n][c] - m[c >> 1]);
    __syncthreads();   // the tile is consumed before the next stage overwrites it
  }
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    l[r] += __shfl_xor_sync(0xffffffffu, l[r], 1);
    l[r] += __shfl_xor_sync(0xffffffffu, l[r], 2);
    const int row = r0 + gl + 8 * r;
    if (tl == 0 && row < P)
      reinterpret_cast<float *>(C.arena + C.off_rowstat)[((size_t)b * C.h_q + h) * P + row] = m[r] + __log2f(l[r]);
  }
}

// Pass 2: colsum[b][h][i] = sum_{tau >= i} 2^(q_tau . k_i * scale_log2 - rowstat[tau]).  Keys are
// the rows here (S^T = K Q^T), so a key's sum over queries stays in its 4 lanes.
__global__ void __launch_bounds__(SC_WARPS * 32) colsum_kernel(const CacheDev C, const __nv_bfloat16 *q,
                                                               const __nv_bfloat16 *k, float scale_log2) {
  __shared__ __align__(128) __nv_bfloat16 qt[2][SC_TILE * SC_LD];
  __shared__ float rs[2][SC_TILE];
  const int P = C.prompt_len;
  const int h = blockIdx.y, b = blockIdx.z, g = h / C.G;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gl = lane >> 2, tl = lane & 3;
  const int i0 = blockIdx.x * SC_TILE, r0 = i0 + 16 * warp;
  const float *rowstat = reinterpret_cast<const float *>(C.arena + C.off_rowstat) + ((size_t)b * C.h_q + h) * P;
  uint32_t ka[8][4];
  load_a_frags(ka, k, b, P, C.h_kv, g, r0);
  float col[2] = {0.f, 0.f};   // keys gl, gl+8: this lane's partial sums
  const int t0 = i0 / SC_TILE, ntiles = (P + SC_TILE - 1) / SC_TILE;
  auto stage = [&](int t, int buf) {
    if (threadIdx.x < SC_TILE) {
      const int row = t * SC_TILE + threadIdx.x;
      rs[buf][threadIdx.x] = row < P ? rowstat[row] : 0.f;
    }
    stage_tile(qt[buf], q, b, P, C.h_q, h, t * SC_TILE);
  };
  stage(t0, 0);
  for (int t = t0; t < ntiles; ++t) {
    const int buf = (t - t0) & 1;
    if (t + 1 < ntiles) {
      stage(t + 1, buf ^ 1);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    float s[8][4];
    tile_mma(s, ka, qt[buf]);
    const int qq0 = t * SC_TILE;
#pragma unroll
    for (int n = 0; n < 8; ++n)
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int key = r0 + gl + ((c >> 1) << 3), qc = 8 * n + 2 * tl + (c & 1), query = qq0 + qc;
        if (query >= key && query < P) col[c >> 1] += exp2f(s[n][c] * scale_log2 - rs[buf][qc]);
      }
    __syncthreads();
  }
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    col[r] += __shfl_xor_sync(0xffffffffu, col[r], 1);
    col[r] += __shfl_xor_sync(0xffffffffu, col[r], 2);
    const int key = r0 + gl + 8 * r;
    if (tl == 0 && key < P) reinterpret_cast<float *>(C.arena + C.off_colsum)[((size_t)b * C.h_q + h) * P + key] = col[r];
  }
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
  dim3 grid((P + SC_TILE - 1) / SC_TILE, C.h_q, C.B);
  rowstat_kernel<<<grid, SC_WARPS * 32, 0, stream>>>(C, q, k, scale_log2);
  colsum_kernel<<<grid, SC_WARPS * 32, 0, stream>>>(C, q, k, scale_log2);
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
