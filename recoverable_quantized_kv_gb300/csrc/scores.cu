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
#include <cuda.h>
#include <cudaTypedefs.h>

#include "cache_dev.cuh"
#include "common.cuh"
#include "smem_optin.h"

namespace qv {

// Both passes run on the 5th-generation tensor cores.  A CTA (one per SM) owns two row tiles of 128 rows
// (queries in pass 1, keys in pass 2) of one (sequence, head); both multiply every streamed 128-row tile
// of the other operand, so each tile is read once for 256 rows.  A producer thread loads tiles with TMA
// (tensor maps over the [B][P][heads][128] prompt tensors, 128-byte swizzle, rows past the prompt
// zero-filled) into a four-stage ring; one thread issues tcgen05.mma (M = N = 128, K = 16 per
// instruction, bf16 in, fp32 out) into two TMEM accumulators per row tile (all 512 columns); sixteen
// epilogue warps read TMEM with tcgen05.ld: eight per row tile, warp w taking the 32 lanes (rows)
// 32 (w % 4) .. and the 64 columns 64 ((w / 4) % 2) .., so every thread reduces half a row without
// shuffles and the two halves meet once at the end.  Every wait is bounded; the TMEM columns are
// released on every path.
constexpr int TC_ROWS = 128;                         // rows per row tile and per streamed tile
constexpr int TC_RT = 2;                             // row tiles per CTA
constexpr int TC_STAGES = 4;
constexpr int TC_EPI = 8 * TC_RT;                    // epilogue warps
constexpr int TC_THREADS = (TC_EPI + 2) * 32;        // + 1 TMA producer warp + 1 MMA issuer warp
constexpr int TC_PRODUCER = TC_EPI, TC_ISSUER = TC_EPI + 1;
constexpr int TC_TILE_BYTES = TC_ROWS * D * 2;       // 32 KB: two 128-byte-swizzled blocks of 64 dims
constexpr int TC_KBLOCK = TC_TILE_BYTES / 2;
constexpr int TC_TMEM_COLS = TC_RT * 2 * TC_ROWS;    // two fp32 accumulators of 128 columns per row tile
constexpr int TC_OFF_B = TC_RT * TC_TILE_BYTES;
constexpr int TC_OFF_RS = TC_OFF_B + TC_STAGES * TC_TILE_BYTES;   // [RT][2][128] negated row statistics
constexpr int TC_OFF_HALF = TC_OFF_RS + TC_RT * 2 * TC_ROWS * 4;  // [RT][2][128] second-half partials
constexpr int TC_OFF_BAR = TC_OFF_HALF + TC_RT * 2 * TC_ROWS * 4;
constexpr int TC_NBAR = 2 * TC_STAGES + 4 * TC_RT + 2;            // full, empty, tfull, tempty, afull, fin
constexpr int TC_SMEM = 1024 + TC_OFF_BAR + TC_NBAR * 8 + 16;
static_assert(TC_TMEM_COLS <= 512 && TC_SMEM <= 232448, "one CTA per SM");

// tcgen05 shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups 1024 B apart
__device__ __forceinline__ uint64_t umma_desc(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
// instruction descriptor, kind::f16: fp32 accumulator, bf16 A and B, both K-major, M = N = 128
constexpr uint32_t TC_IDESC = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(TC_ROWS >> 3) << 17) |
                              ((uint32_t)(TC_ROWS >> 4) << 24);

__device__ __forceinline__ void tma_load_4d(void *dst, const CUtensorMap *map, int x, int y, int z, int w,
                                            uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5}], "
      "[%6];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_commit(uint64_t *bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}
__device__ __forceinline__ void tc_mma(uint32_t tmem, uint64_t da, uint64_t db, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(tmem),
      "l"(da), "l"(db), "r"(TC_IDESC), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ float ex2(float x) {   // 2^x on the special-function unit, subnormal results as 0
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// The three-input maximum.
__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// 64 consecutive fp32 columns of this thread's TMEM lane: two 32-column loads, one wait
__device__ __forceinline__ void tmem_ld64(uint32_t addr, float (&v)[64]) {
  uint32_t r[64];
#pragma unroll
  for (int h = 0; h < 2; ++h)
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
        "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[32 * h + 0]), "=r"(r[32 * h + 1]), "=r"(r[32 * h + 2]), "=r"(r[32 * h + 3]), "=r"(r[32 * h + 4]),
          "=r"(r[32 * h + 5]), "=r"(r[32 * h + 6]), "=r"(r[32 * h + 7]), "=r"(r[32 * h + 8]), "=r"(r[32 * h + 9]),
          "=r"(r[32 * h + 10]), "=r"(r[32 * h + 11]), "=r"(r[32 * h + 12]), "=r"(r[32 * h + 13]),
          "=r"(r[32 * h + 14]), "=r"(r[32 * h + 15]), "=r"(r[32 * h + 16]), "=r"(r[32 * h + 17]),
          "=r"(r[32 * h + 18]), "=r"(r[32 * h + 19]), "=r"(r[32 * h + 20]), "=r"(r[32 * h + 21]),
          "=r"(r[32 * h + 22]), "=r"(r[32 * h + 23]), "=r"(r[32 * h + 24]), "=r"(r[32 * h + 25]),
          "=r"(r[32 * h + 26]), "=r"(r[32 * h + 27]), "=r"(r[32 * h + 28]), "=r"(r[32 * h + 29]),
          "=r"(r[32 * h + 30]), "=r"(r[32 * h + 31])
        : "r"(addr + 32 * h));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int j = 0; j < 64; ++j) v[j] = __uint_as_float(r[j]);
}

// COL = false, pass 1: rowstat[b][h][tau] = log2 sum_{i <= tau} 2^(q_tau . k_i * scale_log2).
// COL = true,  pass 2: colsum[b][h][i] = sum_{tau >= i} 2^(q_tau . k_i * scale_log2 - rowstat[tau]).
template <bool COL>
__global__ void __launch_bounds__(TC_THREADS, 1) tc_score_kernel(const __grid_constant__ CUtensorMap tq,
                                                                 const __grid_constant__ CUtensorMap tk,
                                                                 const CacheDev C, int *status, float scale_log2) {
  extern __shared__ uint8_t tc_smem_raw[];
  uint8_t *sm = tc_smem_raw + ((1024 - (smem_u32(tc_smem_raw) & 1023)) & 1023);   // swizzle atoms: 1024-aligned
  uint64_t *bars = reinterpret_cast<uint64_t *>(sm + TC_OFF_BAR);
  uint64_t *full = bars, *empty = bars + TC_STAGES;
  uint64_t *tfull = bars + 2 * TC_STAGES, *tempty = tfull + 2 * TC_RT;   // [RT][2] each
  uint64_t *afull = tempty + 2 * TC_RT, *fin = afull + 1;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + TC_NBAR);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int P = C.prompt_len, nrt = (P + TC_ROWS - 1) / TC_ROWS, npair = (nrt + TC_RT - 1) / TC_RT;
  const int h = blockIdx.y, b = blockIdx.z, g = h / C.G;
  const int pr = COL ? (int)blockIdx.x : npair - 1 - (int)blockIdx.x;   // pass 1: the longest rows first
  // tile range [lo[r], hi[r]] of row tile rt = TC_RT pr + r (empty past the prompt)
  int lo[TC_RT], hi[TC_RT];
#pragma unroll
  for (int r = 0; r < TC_RT; ++r) {
    const int rt = TC_RT * pr + r;
    lo[r] = COL ? rt : 0;
    hi[r] = rt < nrt ? (COL ? nrt - 1 : rt) : -1;
  }
  const int t_lo = COL ? TC_RT * pr : 0, t_hi = COL ? nrt - 1 : min(TC_RT * pr + TC_RT - 1, nrt - 1);

  if (threadIdx.x == 0) {
    for (int i = 0; i < TC_NBAR; ++i) {
      const bool te = &bars[i] >= tempty && &bars[i] < tempty + 2 * TC_RT;
      mbar_init(&bars[i], te ? 8 * 32 : 1);
    }
    fence_mbar_init();
  }
  if (warp == TC_ISSUER) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(TC_TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // A: pass 1 the queries of head h, pass 2 the keys of KV head g; the streamed tiles the other operand
  const CUtensorMap *mapA = COL ? &tk : &tq, *mapB = COL ? &tq : &tk;
  const int headA = COL ? g : h, headB = COL ? h : g;

  if (warp == TC_PRODUCER) {
    if (lane == 0) {   // ---- TMA producer
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(mapA)) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(mapB)) : "memory");
      mbar_arrive_expect_tx(afull, TC_RT * TC_TILE_BYTES);
      for (int r = 0; r < TC_RT; ++r) {
        uint8_t *dst = sm + r * TC_TILE_BYTES;
        tma_load_4d(dst, mapA, 0, headA, (TC_RT * pr + r) * TC_ROWS, b, afull);
        tma_load_4d(dst + TC_KBLOCK, mapA, 64, headA, (TC_RT * pr + r) * TC_ROWS, b, afull);
      }
      int issued = 0;
      for (int i = 0; i <= t_hi - t_lo; ++i) {
        const int s = i % TC_STAGES;
        if (!mbar_wait(&empty[s], ((i / TC_STAGES) & 1) ^ 1, status)) break;
        uint8_t *dst = sm + TC_OFF_B + TC_TILE_BYTES * s;
        mbar_arrive_expect_tx(&full[s], TC_TILE_BYTES);
        tma_load_4d(dst, mapB, 0, headB, (t_lo + i) * TC_ROWS, b, &full[s]);
        tma_load_4d(dst + TC_KBLOCK, mapB, 64, headB, (t_lo + i) * TC_ROWS, b, &full[s]);
        issued = i + 1;
      }
      // copies still in flight land before the CTA leaves (normally all were consumed already)
      for (int i = max(0, issued - TC_STAGES); i < issued; ++i)
        mbar_wait(&full[i % TC_STAGES], (i / TC_STAGES) & 1, status);
      mbar_wait(afull, 0, status);
    }
  } else if (warp == TC_ISSUER) {
    if (lane == 0) {   // ---- MMA issuer
      bool ok = mbar_wait(afull, 0, status);
      int cnt[TC_RT];
#pragma unroll
      for (int r = 0; r < TC_RT; ++r) cnt[r] = 0;
      for (int i = 0; ok && i <= t_hi - t_lo; ++i) {
        const int s = i % TC_STAGES, t = t_lo + i;
        if (!mbar_wait(&full[s], (i / TC_STAGES) & 1, status)) break;
        const uint32_t b0 = smem_u32(sm + TC_OFF_B + TC_TILE_BYTES * s);
#pragma unroll
        for (int r = 0; r < TC_RT; ++r) {
          if (t < lo[r] || t > hi[r]) continue;
          const int buf = cnt[r] & 1;
          if (!mbar_wait(&tempty[2 * r + buf], ((cnt[r] >> 1) & 1) ^ 1, status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_u32(sm + r * TC_TILE_BYTES);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * TC_KBLOCK + (kk & 3) * 32;   // 16 dims = 32 B inside a 128-B row
            tc_mma(tmem + (2 * r + buf) * TC_ROWS, umma_desc(a0 + off), umma_desc(b0 + off), kk > 0 ? 1u : 0u);
          }
          tc_commit(&tfull[2 * r + buf]);
          ++cnt[r];
        }
        tc_commit(&empty[s]);
      }
      tc_commit(fin);   // every MMA issued above has completed once this arrives
      mbar_wait(fin, 0, status);
    }
  } else {
    // ---- epilogue: group r = warp / 8; thread = TMEM lane = row of row tile rt, columns half * 64 .. + 63
    const int r = warp >> 3, wq = warp & 3, half = (warp >> 2) & 1, cbeg = 64 * half;
    const int rt = TC_RT * pr + r, r0 = rt * TC_ROWS, row = 32 * wq + lane;
    const int nt = hi[r] - lo[r] + 1;   // tiles of this row tile (0 past the prompt)
    const uint32_t lane_addr = tmem + ((uint32_t)(32 * wq) << 16) + 2 * r * TC_ROWS + cbeg;
    float *hp = reinterpret_cast<float *>(sm + TC_OFF_HALF) + r * 2 * TC_ROWS;
    float *rsb = reinterpret_cast<float *>(sm + TC_OFF_RS) + r * 2 * TC_ROWS;
    const int barid = 1 + r;
    bool ok = true;
    if (!COL) {
      const int qrow = r0 + row;
      float m = -INFINITY, l = 0.f;
      for (int i = 0; i < nt; ++i) {
        const int buf = i & 1, t = lo[r] + i;
        if (ok) ok = mbar_wait(&tfull[2 * r + buf], (i >> 1) & 1, status);
        tc_fence_after();
        const bool diag = t == rt;   // key tile t meets the query tile on the diagonal
        float v[64];
        tmem_ld64(lane_addr + buf * TC_ROWS, v);
        if (diag) {
#pragma unroll
          for (int j = 0; j < 64; ++j)
            if (cbeg + j > row) v[j] = -INFINITY;   // causal: keys after the query
        }
        float mx0 = v[0], mx1 = v[1];   // two chains of three-input maxima
#pragma unroll
        for (int j = 2; j < 62; j += 4) {
          mx0 = max3(mx0, v[j], v[j + 1]);
          mx1 = max3(mx1, v[j + 2], v[j + 3]);
        }
        mx0 = max3(mx0, v[62], v[63]);
        const float mn = fmaxf(m, fmaxf(mx0, mx1) * scale_log2);
        if (mn != -INFINITY) {   // the tile holds a key at or before the query
          float a0 = l * ex2(m - mn), a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
          for (int j = 0; j < 64; j += 4) {   // 2^(s scale - mn) two at a time, four accumulators
            float x0, x1, x2, x3;
            fma2(x0, x1, v[j], v[j + 1], scale_log2, scale_log2, -mn, -mn);
            fma2(x2, x3, v[j + 2], v[j + 3], scale_log2, scale_log2, -mn, -mn);
            add2(a0, a1, ex2(x0), ex2(x1));
            add2(a2, a3, ex2(x2), ex2(x3));
          }
          l = (a0 + a1) + (a2 + a3);
          m = mn;
        }
        tc_fence_before();
        mbar_arrive(&tempty[2 * r + buf]);
      }
      // the two column halves of a row meet: (m, l) pairs merge by log-sum-exp
      if (half) {
        hp[row] = m;
        hp[TC_ROWS + row] = l;
      }
      asm volatile("bar.sync %0, %1;" ::"r"(barid), "r"(8 * 32) : "memory");
      if (!half && nt > 0) {
        const float m2 = hp[row], l2 = hp[TC_ROWS + row], mm = fmaxf(m, m2);
        const float ls = (m == -INFINITY ? 0.f : l * exp2f(m - mm)) + (m2 == -INFINITY ? 0.f : l2 * exp2f(m2 - mm));
        if (qrow < P) reinterpret_cast<float *>(C.arena + C.off_rowstat)[((size_t)b * C.h_q + h) * P + qrow] = mm + __log2f(ls);
      }
    } else {
      const int key = r0 + row;
      const float *rowstat = reinterpret_cast<const float *>(C.arena + C.off_rowstat) + ((size_t)b * C.h_q + h) * P;
      float col = 0.f;
      int tau = lo[r] * TC_ROWS + row;
      float nxt = (!half && nt > 0 && tau < P) ? rowstat[tau] : 0.f;   // the statistic of query tau, a tile ahead
      for (int i = 0; i < nt; ++i) {
        const int t = lo[r] + i, buf = i & 1;
        if (!half) rsb[buf * TC_ROWS + row] = -nxt;   // negated: the FMA adds it
        tau += TC_ROWS;
        if (!half && i + 1 < nt) nxt = tau < P ? rowstat[tau] : 0.f;
        asm volatile("bar.sync %0, %1;" ::"r"(barid), "r"(8 * 32) : "memory");   // the tile's row statistics
        if (ok) ok = mbar_wait(&tfull[2 * r + buf], (i >> 1) & 1, status);
        tc_fence_after();
        const bool diag = t == rt, tail = (t + 1) * TC_ROWS > P;
        const float *rs = rsb + buf * TC_ROWS + cbeg;
        float v[64];
        tmem_ld64(lane_addr + buf * TC_ROWS, v);
        if (!diag && !tail) {
          float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
          for (int j = 0; j < 64; j += 4) {
            const float4 q4 = *reinterpret_cast<const float4 *>(rs + j);
            float x0, x1, x2, x3;
            fma2(x0, x1, v[j], v[j + 1], scale_log2, scale_log2, q4.x, q4.y);
            fma2(x2, x3, v[j + 2], v[j + 3], scale_log2, scale_log2, q4.z, q4.w);
            add2(a0, a1, ex2(x0), ex2(x1));
            add2(a2, a3, ex2(x2), ex2(x3));
          }
          col += (a0 + a1) + (a2 + a3);
        } else {
#pragma unroll
          for (int j = 0; j < 64; ++j) {
            const int c = cbeg + j;
            const bool valid = (!diag || c >= row) && t * TC_ROWS + c < P;   // causal, inside the prompt
            col += valid ? ex2(fmaf(v[j], scale_log2, rs[j])) : 0.f;
          }
        }
        tc_fence_before();
        mbar_arrive(&tempty[2 * r + buf]);
      }
      if (half) hp[row] = col;
      asm volatile("bar.sync %0, %1;" ::"r"(barid), "r"(8 * 32) : "memory");
      if (!half && nt > 0 && key < P)
        reinterpret_cast<float *>(C.arena + C.off_colsum)[((size_t)b * C.h_q + h) * P + key] = col + hp[row];
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == TC_ISSUER) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TC_TMEM_COLS) : "memory");
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

namespace {
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// [B][P][heads][128] bf16 as a 4-D tensor map; a box is 64 dims x 1 head x 128 rows, 128-byte swizzled
bool prompt_map(CUtensorMap *map, const __nv_bfloat16 *base, int B, int P, int heads) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return false;
  const cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)heads, (cuuint64_t)P, (cuuint64_t)B};
  const cuuint64_t strides[3] = {(cuuint64_t)D * 2, (cuuint64_t)heads * D * 2, (cuuint64_t)P * heads * D * 2};
  const cuuint32_t box[4] = {64, 1, (cuuint32_t)TC_ROWS, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<__nv_bfloat16 *>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
}  // namespace

cudaError_t launch_prefill_scores(const CacheDev &C, const __nv_bfloat16 *q, const __nv_bfloat16 *k, float *s0,
                                  cudaStream_t stream) {
  const float scale_log2 = 1.4426950408889634f / sqrtf((float)D);
  const int P = C.prompt_len;
  if (((uintptr_t)q | (uintptr_t)k) & 15) return cudaErrorInvalidValue;   // tensor maps: 16-byte aligned bases
  CUtensorMap tq, tk;
  if (!prompt_map(&tq, q, C.B, P, C.h_q) || !prompt_map(&tk, k, C.B, P, C.h_kv)) return cudaErrorInvalidValue;
  static SmemOptIn optin_rows, optin_cols;
  cudaError_t e = optin_rows.ensure(tc_score_kernel<false>, TC_SMEM);
  if (e == cudaSuccess) e = optin_cols.ensure(tc_score_kernel<true>, TC_SMEM);
  if (e != cudaSuccess) return e;
  int *status = C.status();
  const int nrt = (P + TC_ROWS - 1) / TC_ROWS;
  dim3 grid((nrt + TC_RT - 1) / TC_RT, C.h_q, C.B);
  tc_score_kernel<false><<<grid, TC_THREADS, TC_SMEM, stream>>>(tq, tk, C, status, scale_log2);
  tc_score_kernel<true><<<grid, TC_THREADS, TC_SMEM, stream>>>(tq, tk, C, status, scale_log2);
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
  int nF = s_meta[M_FCOUNT], nQ = s_meta[M_QCOUNT];
  if (!qv_inbounds(nF >= 0 && nF <= C.kf_cap() && nQ >= 0 && nQ <= min(C.k_q, C.n_windows), C.status()))
    nF = nQ = 0;
  const int nk = T - F;
  if (nk < 0 || nk > C.omega) {
    if (threadIdx.x == 0) atomicOr(C.status(), QV_ERR_STATE);
  } else if (nk > 0) {
    const float *ms = reinterpret_cast<const float *>(C.arena + C.off_mstat + C.st_mstat_layer * layer) +
                      (size_t)bg * C.omega * 16;
    for (int i = threadIdx.x; i < nk * 16; i += blockDim.x) st[i] = ms[i];
    __syncthreads();
    const float *mu = reinterpret_cast<const float *>(C.arena + C.off_mu + C.st_mu_layer * layer) +
                      (size_t)bg * C.omega * C.max_items * C.G;
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
      if (!qv_inbounds(w >= 0 && w < C.n_windows, C.status())) continue;
      float s = score[w];
      for (int k = k0; k < nk; ++k) {
        const float *m = mu + ((size_t)k * C.max_items + idx) * C.G;
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
