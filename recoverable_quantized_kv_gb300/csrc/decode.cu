// Decode step of one layer: append + split-K GQA attention over sink / recent / Full (bf16) /
// Quantized (INT2 dequantised in registers) windows + per-window attention mass + score update.
//
// QEvict (arXiv 2608.05326) §4.1: o = softmax(q K_acc^T / sqrt(d)) V_acc over the accessible set;
// §4.2 Eq. (1): the window score accumulates (1/H_q) sum_h sum_{i in w} a^h(i).
//
// Grid (n_split, h_kv, batch); at batch 1 (h_kv, 1, n_split), so that the CTAs dispatched last are
// one split of every KV head.  Each CTA owns a slice of the recent, Full and Quantized windows of
// one (sequence, KV head), proportional to its split's weight.  One producer warp streams the
// slice's windows through a CTA-wide ring of 4 KB shared-memory slots with 1-D bulk copies (TMA),
// each completing on an mbarrier; eleven consumer warps take items (a window, or two Quantized INT2
// windows; the Quantized items first, the bf16 windows last) from a shared queue, wait for their
// chunks, compute, and release the slots.  The G query heads of the KV head ride on the N side of
// mma.m16n8k16 (tokens on M for Q K^T, dims on M for P V), so both products run on tensor cores.
// Softmax is online per warp; per-window masses are kept as log2-sum-exp values, normalised into the
// window scores when the scores are flushed.  The last CTA of the (sequence, KV head) to finish
// (counted with one atomic, no waiting) merges the splits and stores the step's merged max and 1/L
// for that flush.
// With pre-RoPE Quantized keys (QEvict §4.3 "Cache Execution") the kernel variant ROPE rotates the
// dequantised keys to their positions in registers before the key MMAs.
#include "cache_dev.cuh"
#include "common.cuh"
#include "smem_optin.h"

namespace qv {

constexpr int DEC_WARPS = 12;          // 11 consumer warps + 1 producer warp (168 registers a thread)
constexpr int DEC_CONSUMERS = DEC_WARPS - 1;
constexpr int DEC_SLOTS = 36;          // CTA-wide ring of 4 KB slots filled by bulk copies
constexpr int DEC_STAGE_BYTES = 4096;
// per consumer warp: the key look-up tables of the windows in hand (INT2: bf16 bytes of the 4 values
// of 128 channels; INT4: fp32 scale and offset of 128 channels), 8 k-steps x 4 lane classes x 32 B
// each, then (ROPE) the cos/sin rows of the window's first position of each 32-token half.  They live
// in the warp's own output region of the CTA merge, which the warp writes only after its last window.
constexpr int DEC_TBL_BYTES = 1024;
// Scale of the output accumulators of the INT2 kernels: P V of Quantized windows runs on value codes
// held as fp16 subnormals (c * 4^tau * 2^-24) against P * s * 4^(3 - tau), so its products come out
// at 2^-18; bf16 windows scale their P by the same 2^-18, and the CTA merge scales back.
template <int BITS>
struct OScale {
  static constexpr float P = BITS == 2 ? 0x1p-18f : 1.f;
  static constexpr float INV = BITS == 2 ? 0x1p18f : 1.f;
};
// CTA merge: running max / sum / rescale per (warp, head), CTA max, and every warp's outputs
constexpr int DEC_CO_OFF = (3 * DEC_CONSUMERS * 8 + 16) * 4;   // bytes before the outputs
constexpr int DEC_MRG_FLOATS = 3 * DEC_CONSUMERS * 8 + 16 + DEC_CONSUMERS * 128 * 8;
// ROPE: cos/sin of the in-window offsets 0..31, 16 KB shared by the consumer warps
constexpr int DEC_REL_BYTES = 32 * 64 * 2 * 4;

// Chunk stream geometry of one (window, bits) format.  A bf16 window streams its K block then its
// V block in 4 KB chunks; a Quantized window streams its ledger record (codes, then parameters).
// Consumers take windows from a queue, so a consumer can wait on a chunk up to
// DEC_CONSUMERS * MAX_CHUNKS chunks past the first one not yet issued.  Giving every slot PHASES
// "full" barriers used in turn keeps every parity wait unambiguous: the chunk PHASES * DEC_SLOTS
// earlier on the same barrier has always landed by then.
template <int W, int BITS, bool ROPE>
struct DecGeo {
  static constexpr int HALVES = W / 32;                        // 32-token halves of a window
  static constexpr int KCH = W / 16;                           // 4 KB chunks of one K (or V) block
  static constexpr int BF_CHUNKS = 2 * KCH;
  static constexpr int Q_CHUNKS = (Geo<W, BITS>::QB + DEC_STAGE_BYTES - 1) / DEC_STAGE_BYTES;
  static constexpr int MAX_CHUNKS = BF_CHUNKS > Q_CHUNKS ? BF_CHUNKS : Q_CHUNKS;
  static constexpr int PHASES = 1 + (DEC_CONSUMERS * MAX_CHUNKS + DEC_SLOTS - 1) / DEC_SLOTS;
  static constexpr int FULL = PHASES * DEC_SLOTS;
  static constexpr int REL_OFF = DEC_SLOTS * DEC_STAGE_BYTES;
  static constexpr int BAR_OFF = REL_OFF + (ROPE ? DEC_REL_BYTES : 0);
  static constexpr int MRG_OFF = BAR_OFF + (FULL + DEC_SLOTS) * 8;
  static constexpr int SMEM = MRG_OFF + DEC_MRG_FLOATS * 4;
  static_assert((PHASES - 1) * DEC_SLOTS >= DEC_CONSUMERS * MAX_CHUNKS, "too few full barriers per slot");
  static_assert(W == 32 || Geo<W, BITS>::CODE_BYTES == DEC_STAGE_BYTES, "INT4 code blocks fill one chunk each");
  static_assert(2 * DEC_TBL_BYTES + HALVES * 512 <= 128 * 8 * 4, "per-warp tables fit the warp's output region");
  static_assert(SMEM <= 232448, "shared memory per CTA");
  static_assert(MRG_OFF % 16 == 0 && DEC_CO_OFF % 16 == 0, "16-byte aligned per-warp tables");
};

__device__ __forceinline__ uint32_t ldg32(const void *p) { return __ldg(reinterpret_cast<const uint32_t *>(p)); }
__device__ __forceinline__ uint32_t ldg16(const void *p) { return __ldg(reinterpret_cast<const unsigned short *>(p)); }

// 2^x on the special-function unit (relative error about 2^-22); results below 2^-126 flush to zero,
// which drops nothing from a probability sum whose largest term is 1.
__device__ __forceinline__ float ex2_ftz(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// One online-softmax step over NMT 16-token groups of S^T fragments (rows tokens, cols heads).
// s holds raw logits q.k; `scale` (log2(e) / sqrt(d)) takes them to log2 units inside the
// exponent's FMA, and the item's max is taken on raw logits and scaled once (a positive factor keeps
// the order).  Rows flagged invalid are excluded.  On return s holds the probabilities relative to
// the running max m_run (log2 units), tsum the sum of this lane's head over the item (heads 2tl and
// 2tl + 1 on even and odd gl).  The running max only
// moves when some logit of the item exceeds it (one warp vote decides); otherwise every
// probability is already <= 1 and nothing accumulated so far (o, macc, l_run) needs rescaling.
template <int NMT>
__device__ __forceinline__ void online_step(float (&s)[NMT][4], const bool (&valid)[NMT][2], float (&m_run)[2],
                                            float &l_run, float (&o)[8][4], float (&macc)[2],
                                            float &tsum, const float scale) {
  const bool odd = (threadIdx.x >> 2) & 1;
  float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
  for (int mt = 0; mt < NMT; ++mt)
#pragma unroll
    for (int r = 0; r < 2; ++r)
      if (valid[mt][r]) {
        mx[0] = fmaxf(mx[0], s[mt][2 * r]);
        mx[1] = fmaxf(mx[1], s[mt][2 * r + 1]);
      }
  mx[0] *= scale;
  mx[1] *= scale;
  if (!__all_sync(0xffffffffu, mx[0] <= m_run[0] && mx[1] <= m_run[1])) {
    float corr[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const float mnew = fmaxf(m_run[h], warp_max_xor_g(mx[h]));
      corr[h] = exp2f(m_run[h] - (mnew == -INFINITY ? 0.f : mnew));
      m_run[h] = mnew;
      macc[h] *= corr[h];
    }
    l_run *= odd ? corr[1] : corr[0];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      o[i][0] *= corr[0];
      o[i][2] *= corr[0];
      o[i][1] *= corr[1];
      o[i][3] *= corr[1];
    }
  }
  float base[2], ps[2] = {0.f, 0.f};
#pragma unroll
  for (int h = 0; h < 2; ++h) base[h] = m_run[h] == -INFINITY ? 0.f : m_run[h];
#pragma unroll
  for (int mt = 0; mt < NMT; ++mt)
#pragma unroll
    for (int r = 0; r < 2; ++r)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const float p = valid[mt][r] ? ex2_ftz(fmaf(s[mt][2 * r + h], scale, -base[h])) : 0.f;
        s[mt][2 * r + h] = p;
        ps[h] += p;
      }
  float v = odd ? ps[1] : ps[0];
  v += __shfl_xor_sync(0xffffffffu, odd ? ps[0] : ps[1], 4);
  v += __shfl_xor_sync(0xffffffffu, v, 8);
  v += __shfl_xor_sync(0xffffffffu, v, 16);
  tsum = v;
  l_run += v;
}

// online_step for NW windows of 32 tokens at once (S^T fragments s[w][mt]): one max vote and at most
// one rescale for all of them; tsum[w] is window w's sum of this lane's head, l_run gains them all.
// Windows with valid[w] false contribute nothing (probabilities 0).
template <int NW>
__device__ __forceinline__ void online_step_w(float (&s)[NW][2][4], const bool (&valid)[NW], float (&m_run)[2],
                                              float &l_run, float (&o)[8][4], float (&macc)[2], float (&tsum)[NW],
                                              const float scale) {
  const bool odd = (threadIdx.x >> 2) & 1;
  float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
  for (int w = 0; w < NW; ++w)
    if (valid[w]) {
#pragma unroll
      for (int mt = 0; mt < 2; ++mt) {
        mx[0] = fmaxf(mx[0], fmaxf(s[w][mt][0], s[w][mt][2]));
        mx[1] = fmaxf(mx[1], fmaxf(s[w][mt][1], s[w][mt][3]));
      }
    }
  mx[0] *= scale;
  mx[1] *= scale;
  if (!__all_sync(0xffffffffu, mx[0] <= m_run[0] && mx[1] <= m_run[1])) {
    float corr[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const float mnew = fmaxf(m_run[h], warp_max_xor_g(mx[h]));
      corr[h] = exp2f(m_run[h] - (mnew == -INFINITY ? 0.f : mnew));
      m_run[h] = mnew;
      macc[h] *= corr[h];
    }
    l_run *= odd ? corr[1] : corr[0];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      o[i][0] *= corr[0];
      o[i][2] *= corr[0];
      o[i][1] *= corr[1];
      o[i][3] *= corr[1];
    }
  }
  float base[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) base[h] = m_run[h] == -INFINITY ? 0.f : m_run[h];
  float v[NW];
#pragma unroll
  for (int w = 0; w < NW; ++w) {
    float ps[2] = {0.f, 0.f};
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
      for (int r = 0; r < 2; ++r)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const float p = valid[w] ? ex2_ftz(fmaf(s[w][mt][2 * r + h], scale, -base[h])) : 0.f;
          s[w][mt][2 * r + h] = p;
          ps[h] += p;
        }
    v[w] = odd ? ps[1] : ps[0];
    v[w] += __shfl_xor_sync(0xffffffffu, odd ? ps[0] : ps[1], 4);
  }
#pragma unroll
  for (int w = 0; w < NW; ++w) v[w] += __shfl_xor_sync(0xffffffffu, v[w], 8);
#pragma unroll
  for (int w = 0; w < NW; ++w) {
    v[w] += __shfl_xor_sync(0xffffffffu, v[w], 16);
    tsum[w] = v[w];
    l_run += v[w];
  }
}

// B fragments of P^T for k-step kk from the S^T accumulator layout (8x8 transposes), times `scale`
// (a power of two: exact).
template <int NMT>
__device__ __forceinline__ void p_to_b(const float (&p)[NMT][4], uint32_t (&pb)[NMT][2], const float scale) {
#pragma unroll
  for (int kk = 0; kk < NMT; ++kk) {
    pb[kk][0] = movmatrix_trans(pack_bf16(p[kk][0] * scale, p[kk][1] * scale));
    pb[kk][1] = movmatrix_trans(pack_bf16(p[kk][2] * scale, p[kk][3] * scale));
  }
}

__device__ __forceinline__ float h2f_lo(uint32_t v) { return __half2float(__ushort_as_half((unsigned short)(v & 0xFFFF))); }
__device__ __forceinline__ float h2f_hi(uint32_t v) { return __half2float(__ushort_as_half((unsigned short)(v >> 16))); }

__device__ __forceinline__ uint32_t word_of(const uint4 &v, int k) {
  return k == 0 ? v.x : (k == 1 ? v.y : (k == 2 ? v.z : v.w));
}

// Exact bf16(fp32(code * s + m)) for keys via per-channel byte tables: lo/hi bytes of the 4
// dequantised values of channel pair A (2t, 2t+1) and B (2t+8, 2t+9) of k-step j.  sel01 / sel23
// are the byte-permute selectors of the field (its low 16 bits are used).
__device__ __forceinline__ void lut_k_regs(uint32_t sel01, uint32_t sel23, const uint4 &TA, const uint4 &TB,
                                           uint32_t &a0, uint32_t &a1, uint32_t &a2, uint32_t &a3) {
  uint32_t lo = __byte_perm(TA.x, TA.y, sel01), hi = __byte_perm(TA.z, TA.w, sel01);
  a0 = __byte_perm(lo, hi, 0x5140);
  a1 = __byte_perm(lo, hi, 0x7362);
  lo = __byte_perm(TB.x, TB.y, sel23);
  hi = __byte_perm(TB.z, TB.w, sel23);
  a2 = __byte_perm(lo, hi, 0x5140);
  a3 = __byte_perm(lo, hi, 0x7362);
}

// INT4 value codes as exact fp16 integers: the codes at nibble p (0 or 1) of both fp16 halves land
// in the mantissas under exponent 2^10 (value 1024 + 16^p c); one packed fma recovers c.
__device__ __forceinline__ uint32_t dq_v4(uint32_t w, int p) {
  static constexpr uint32_t SCL[2] = {0x3C003C00u, 0x2C002C00u};   // 1, 1/16
  static constexpr uint32_t OFF[2] = {0xE400E400u, 0xD400D400u};   // -1024, -64
  const uint32_t x = (w & (0x000F000Fu << (4 * p))) | 0x64006400u;
  uint32_t r;
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(x), "r"(SCL[p]), "r"(OFF[p]));
  return r;
}

// Byte r of two words holding one 4-bit code per byte, as exact floats: the mantissa of 2^23 + c, less
// 2^23 in one packed subtraction.
__device__ __forceinline__ void nib_f2(uint32_t e, uint32_t o, int r, float &ce, float &co) {
  ce = __uint_as_float(__byte_perm(e, 0x4B000000u, 0x7540u | r));
  co = __uint_as_float(__byte_perm(o, 0x4B000000u, 0x7540u | r));
  sub2(ce, co, ce, co, 8388608.0f, 8388608.0f);
}
// bf16(fp32(c * s + m)) of two channels (c exact floats), packed low / high, each FMA rounded on its own
__device__ __forceinline__ uint32_t dq_k4(float c0, float c1, float s0, float s1, float m0, float m1) {
  float d0, d1;
  fma2(d0, d1, c0, c1, s0, s1, m0, m1);
  return pack_bf16(d0, d1);
}

__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                        uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_half(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&v);
}

// Key look-up table of one INT2 window for this lane's four channels d = 4*lane + k: the bf16 values
// bf16(fp32(c*s + m)) for c = 0..3, split into low and high bytes, stored where lut_k_regs reads them
// (k-step j, lane class t, channel pair A or B, value half).
__device__ __forceinline__ void ktab_int2(const uint8_t *ch, uint8_t *tbl, int lane) {
  using Gm = Geo<32, 2>;
  const uint2 sp = *reinterpret_cast<const uint2 *>(ch + Gm::OFF_KS + 8 * lane);
  const uint2 mp = *reinterpret_cast<const uint2 *>(ch + Gm::OFF_KM + 8 * lane);
  float sc[4] = {h2f_lo(sp.x), h2f_hi(sp.x), h2f_lo(sp.y), h2f_hi(sp.y)};
  float mn[4] = {h2f_lo(mp.x), h2f_hi(mp.x), h2f_lo(mp.y), h2f_hi(mp.y)};
  float v1[4], v2[4], v3[4];   // c*s + m for c = 1, 2, 3, each product and sum rounded on its own
#pragma unroll
  for (int k = 0; k < 4; k += 2) {
    v1[k] = sc[k], v1[k + 1] = sc[k + 1];
    add2(v1[k], v1[k + 1], mn[k], mn[k + 1]);
    fma2(v2[k], v2[k + 1], 2.f, 2.f, sc[k], sc[k + 1], mn[k], mn[k + 1]);
    fma2(v3[k], v3[k + 1], 3.f, 3.f, sc[k], sc[k + 1], mn[k], mn[k + 1]);
  }
  uint32_t lo[4], hi[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const uint32_t p01 = pack_bf16(mn[k], v1[k]), p23 = pack_bf16(v2[k], v3[k]);
    lo[k] = __byte_perm(p01, p23, 0x6420);
    hi[k] = __byte_perm(p01, p23, 0x7531);
  }
  // channel d = 4 lane + k sits at k-step j = lane / 4, lane class t = 2 (lane & 1) + k / 2, channel pair
  // (lane / 2) & 1, value half k & 1: channels k = 0, 1 fill one 16-byte run (low bytes, then high
  // bytes), k = 2, 3 the run 32 bytes on
  uint4 *tw = reinterpret_cast<uint4 *>(tbl) + ((lane >> 2) * 4 + 2 * (lane & 1)) * 2 + ((lane >> 1) & 1);
  tw[0] = make_uint4(lo[0], lo[1], hi[0], hi[1]);
  tw[2] = make_uint4(lo[2], lo[3], hi[2], hi[3]);
}

// S^T = K q^T over the 32 tokens of NW INT2 windows at once (their MMA chains interleave): exact
// bf16 keys from the byte tables, the G query heads on the N side.  kc: each window's two 16-byte
// pieces of this lane's K codes; tbl: the windows' tables, DEC_TBL_BYTES apart.
template <int NW>
__device__ __forceinline__ void keys_int2(const uint4 (&kc)[NW][2], const uint8_t *tbl, const uint32_t (&qb)[8][2],
                                          float (&s)[NW][2][4], int tl) {
#pragma unroll
  for (int jp = 0; jp < 4; ++jp) {
    // selectors of both fields of a code word at once: k-step 2jp in the low half, 2jp+1 high
    uint32_t sa[NW][2], sb[NW][2];
#pragma unroll
    for (int w = 0; w < NW; ++w)
#pragma unroll
      for (int mt = 0; mt < 2; ++mt) {
        const uint32_t wd = word_of(kc[w][mt], jp);
        sa[w][mt] = (wd & 0x33333333u) | 0x40404040u;
        sb[w][mt] = ((wd >> 2) & 0x33333333u) | 0x40404040u;
      }
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      const int j = 2 * jp + hf;
#pragma unroll
      for (int w = 0; w < NW; ++w) {
        const uint4 TA = lds128(tbl + w * DEC_TBL_BYTES + (j * 4 + tl) * 32);
        const uint4 TB = lds128(tbl + w * DEC_TBL_BYTES + (j * 4 + tl) * 32 + 16);
#pragma unroll
        for (int mt = 0; mt < 2; ++mt) {
          uint32_t a0, a1, a2, a3;
          lut_k_regs(hf ? sa[w][mt] >> 16 : sa[w][mt], hf ? sb[w][mt] >> 16 : sb[w][mt], TA, TB, a0, a1, a2, a3);
          mma_bf16(s[w][mt], a0, a1, a2, a3, qb[j][0], qb[j][1]);
        }
      }
    }
  }
}

// P V of one INT2 window (QEvict §4.3: values quantised per token, x = c*s + m), for this lane's
// probabilities p (S^T layout, tokens 16kk + gl and + 8).  o += sum_t p_t s_t c_t at the 2^-18
// scale of OScale<2>, macc += sum_t p_t m_t per lane head (its lanes are summed at the merge).
// The codes enter the tensor core as fp16 subnormals c * 4^tau * 2^-24 (one mask each), and the P
// operand of token pair tau carries p * s * 4^(3 - tau), so every product is c p s 2^-18.  That P
// stays below the fp16 range while every token scale s <= 1023; a window with a larger scale takes
// the products at 2^-24 into a zeroed tile and adds them 64-fold instead.
__device__ __forceinline__ void pv_int2(const float (&p)[2][4], const uint8_t *ch, float (&o)[8][4], float (&macc)[2],
                                        int lane) {
  using Gm = Geo<32, 2>;
  const int gl = lane >> 2;
  const __half *vsp = reinterpret_cast<const __half *>(ch + Gm::OFF_VS);
  const __half *vmp = reinterpret_cast<const __half *>(ch + Gm::OFF_VM);
  float sv[2][2], pm0 = 0.f, pm1 = 0.f;
#pragma unroll
  for (int kk = 0; kk < 2; ++kk) {
    const int t0 = 16 * kk + gl, t1 = t0 + 8;
    sv[kk][0] = __half2float(vsp[t0]);
    sv[kk][1] = __half2float(vsp[t1]);
    const float m0v = __half2float(vmp[t0]), m1v = __half2float(vmp[t1]);
    fma2(pm0, pm1, p[kk][2], p[kk][3], m1v, m1v, pm0, pm1);
    fma2(pm0, pm1, p[kk][0], p[kk][1], m0v, m0v, pm0, pm1);
  }
  macc[0] += pm0;
  macc[1] += pm1;
  const uint4 vw0 = lds128(ch + Gm::OFF_VCODE + lane * 16), vw1 = lds128(ch + Gm::OFF_VCODE + 512 + lane * 16);
  const float smax = fmaxf(fmaxf(sv[0][0], sv[0][1]), fmaxf(sv[1][0], sv[1][1]));
  const bool wide = __any_sync(0xffffffffu, !(smax <= 1023.f));
  // P operand of k-step kk: b0 holds tokens 16kk + 2tl .. (pair tau = 2kk), b1 tokens 16kk + 8 + 2tl ..
  // (tau = 2kk + 1), each scaled by 4^(3 - tau) (2^-6 more on the wide path)
  const float wsc = wide ? 0.015625f : 1.f;
  uint32_t pb[2][2];
#pragma unroll
  for (int kk = 0; kk < 2; ++kk) {
    const float f0 = (kk ? 4.f : 64.f) * wsc, f1 = (kk ? 1.f : 16.f) * wsc;
    const float s0 = sv[kk][0] * f0, s1 = sv[kk][1] * f1;
    float x0, x1, x2, x3;
    mul2(x0, x1, p[kk][0], p[kk][1], s0, s0);
    mul2(x2, x3, p[kk][2], p[kk][3], s1, s1);
    pb[kk][0] = movmatrix_trans(pack_half(x0, x1));
    pb[kk][1] = movmatrix_trans(pack_half(x2, x3));
  }
  if (!wide) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t w = word_of(i < 4 ? vw0 : vw1, i & 3), w8 = w >> 8;
#pragma unroll
      for (int kk = 0; kk < 2; ++kk) {
        const uint32_t m0 = 0x00030003u << (4 * kk), m1 = m0 << 2;
        mma_f16(o[i], w & m0, w8 & m0, w & m1, w8 & m1, pb[kk][0], pb[kk][1]);
      }
    }
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t w = word_of(i < 4 ? vw0 : vw1, i & 3), w8 = w >> 8;
      float t[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int kk = 0; kk < 2; ++kk) {
        const uint32_t m0 = 0x00030003u << (4 * kk), m1 = m0 << 2;
        mma_f16(t, w & m0, w8 & m0, w & m1, w8 & m1, pb[kk][0], pb[kk][1]);
      }
#pragma unroll
      for (int r = 0; r < 4; ++r) o[i][r] = fmaf(64.f, t[r], o[i][r]);
    }
  }
}

// cos/sin of the in-window offset tt for channels 16jj + 2tl + 8hh and + 1, as (cos, cos, sin, sin) of the
// two channels, from the offset table:
// 16 B per (offset, k-step jj, channel half, lane class), the two halves swapped on odd offsets so
// that the lanes of neighbouring token rows read different banks
__device__ __forceinline__ float4 rel_cs(const uint8_t *rel, int tt, int jj, int hh, int tl) {
  return *reinterpret_cast<const float4 *>(rel + ((((tt * 4 + jj) * 2 + (hh ^ (tt & 1))) * 4 + tl) * 16));
}

// RoPE of one token's channel pairs (i, i + 64) and (i + 1, i + 65) (QEvict §4.3: RoPE re-applied
// after dequantisation): a0, a1 are the pre-RoPE values of channels i, i + 1 and b0, b1 of i + 64,
// i + 65.  The angle of position p0 + tt comes by angle addition from the window's row cb and the
// offset's row rt, both (cos, cos, sin, sin) of the two channels (ncb: the window row's sines negated);
// the rotation x_i c - x_{i+64} s, x_{i+64} c + x_i s rounds every product and sum on its own, two
// channels per packed instruction.  ka, kb: the bf16 pairs (i, i + 1) and (i + 64, i + 65).
__device__ __forceinline__ void rope_rot(float a0, float a1, float b0, float b1, const float4 &cb, const float2 &ncb,
                                         const float4 &rt, uint32_t &ka, uint32_t &kb) {
  float c0, c1, s0, s1, u0, u1, w0, w1;
  mul2(u0, u1, ncb.x, ncb.y, rt.z, rt.w);          // -sin(p0) sin(t)
  fma2(c0, c1, cb.x, cb.y, rt.x, rt.y, u0, u1);     // cos(p0 + t)
  mul2(w0, w1, cb.x, cb.y, rt.z, rt.w);            // cos(p0) sin(t)
  fma2(s0, s1, cb.z, cb.w, rt.x, rt.y, w0, w1);     // sin(p0 + t)
  float p0, p1, q0, q1;
  mul2(p0, p1, a0, a1, c0, c1);
  mul2(q0, q1, b0, b1, s0, s1);
  sub2(p0, p1, p0, p1, q0, q1);                    // x_i c - x_{i+64} s
  mul2(u0, u1, b0, b1, c0, c1);
  mul2(w0, w1, a0, a1, s0, s1);
  add2(u0, u1, w0, w1);                            // x_{i+64} c + x_i s
  ka = pack_bf16(p0, p1);
  kb = pack_bf16(u0, u1);
}

// a window's RoPE row (cos, sin, cos, sin of channels 2l, 2l + 1) reordered to (cos, cos, sin, sin)
__device__ __forceinline__ float4 cc_ss(const float4 &v) { return make_float4(v.x, v.z, v.y, v.w); }

template <int W, int BITS, bool ROPE>
// 12 warps, three on each SM sub-partition, whose register file share (16K registers) allows 168 each
__global__ void __launch_bounds__(DEC_WARPS * 32, 1) decode_kernel(const CacheDev C, const DecodeIO io) {
  static_assert((W == 32 && BITS == 2) || (W == 64 && BITS == 4), "formats: W=32 INT2, W=64 INT4");
  using Gm = Geo<W, BITS>;
  using Dg = DecGeo<W, BITS, ROPE>;
  constexpr int NMT = 2;                 // 16-token groups of a 32-token half
  constexpr int HALVES = Dg::HALVES;
  constexpr int KCH = Dg::KCH, BFC = Dg::BF_CHUNKS, QCH = Dg::Q_CHUNKS;
  extern __shared__ __align__(128) uint8_t smem[];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gl = lane >> 2, tl = lane & 3;
  const bool one_seq = C.B == 1;
  const int split = one_seq ? blockIdx.z : blockIdx.x, g = one_seq ? blockIdx.x : blockIdx.y,
            b = one_seq ? 0 : blockIdx.z;
  const int unit = io.layer * C.B + b;
  const int G = C.G;
  // Programmatic dependent launch.  This kernel may start while the previous kernel in the stream
  // (the decode of another layer) finishes; that kernel writes only its own layer's state, and every
  // kernel before it has completed (each decode kernel lets its successor start only after its own
  // wait below).  So this layer's meta record and tables can be read right away; the window copies
  // and the step's inputs (q, k_new, v_new) wait.  When the previous decode was the same layer,
  // wait first.
  if (io.wait_first) asm volatile("griddepcontrol.wait;" ::: "memory");
  int *status = C.status();
  int *meta = C.at<int>(C.off_meta, C.st_meta, unit);
  int *thead = reinterpret_cast<int *>(C.arena + C.off_thead) + (size_t)unit * C.h_kv + g;
  int T = *thead, n_route = meta[M_NROUTE], nF = meta[M_FCOUNT], nQ = meta[M_QCOUNT];
  if (!qv_inbounds(nF >= 0 && nF <= C.kf_cap() && nQ >= 0 && nQ <= min(C.k_q, C.n_windows) && n_route >= 0 &&
                       T > C.n_sink && T < C.max_len && (T - C.n_sink) / C.W - n_route < C.ring_windows,
                   status))
    nF = nQ = 0, n_route = max(0, (T - C.n_sink) / C.W);
  // this step's slot in the per-step mass records: steps since the scores last absorbed them
  int mslot = T - meta[M_FLUSHT];
  if (mslot < 0 || mslot >= C.omega) {
    if (threadIdx.x == 0) atomicOr(C.status(), QV_ERR_STATE);
    mslot = mslot < 0 ? 0 : C.omega - 1;
  }
  const int2 *ftab = C.at<const int2>(C.off_ftab, C.st_ftab, unit);
  const int2 *qtab = C.at<const int2>(C.off_qtab, C.st_qtab, unit);
  const __nv_bfloat16 *sink = C.at<const __nv_bfloat16>(C.off_sink, C.st_sink, unit) + (size_t)g * 2 * C.n_sink * D;
  __nv_bfloat16 *ring = C.at<__nv_bfloat16>(C.off_ring, C.st_ring, unit) + (size_t)g * 2 * C.ring_windows * Gm::BLK;
  const uint8_t *fpool = C.at<const uint8_t>(C.off_fpool, C.st_fpool, unit);
  const uint8_t *ledger = C.at<const uint8_t>(C.off_ledger, C.st_ledger, unit);
  const int bg = b * C.h_kv + g;
  float *mu = reinterpret_cast<float *>(C.arena + C.off_mu + C.st_mu_layer * io.layer) +
              ((size_t)bg * C.omega + mslot) * C.max_items * G;
  float *part = reinterpret_cast<float *>(C.arena + C.off_part + C.st_part_layer * io.layer) +
                (size_t)bg * C.n_split * PART_FLOATS;

  const int jn = (T - C.n_sink) / W;   // window of the new token at position T
  const int j0 = n_route;
  const int nL = jn - n_route + 1;
  // this CTA's slice of every class; item ids: 0 sink, 1..nL recent, then F, then Q.  Slice
  // weights, in sixteenths of a share.  At batch 1 the last split takes 11: its CTAs are
  // dispatched last, onto the SMs that the previous layer's split merges free, so they start about a
  // microsecond after the others and without copies issued before the programmatic-launch wait.
  // (At larger batches the previous kernel merges on B * h_kv SMs and every loop is long: equal
  // shares.)  n is at most the router's window capacity, so the products fit 32 bits.
  const int ns = C.n_split;
  const int last_w = one_seq ? 11 : 16, wtot = 16 * (ns - 1) + last_w;
  auto cut = [&](int s, int n) { return s >= ns ? n : (int)((unsigned)n * (16u * s) / (unsigned)wtot); };
  const int L0 = cut(split, nL), L1 = cut(split + 1, nL);
  const int F0 = cut(split, nF), F1 = cut(split + 1, nF);
  const int Q0 = cut(split, nQ), Q1 = cut(split + 1, nQ);
  const int has_sink = split == 0 ? 1 : 0;
  // Quantized windows per queue item: INT2 windows without RoPE go in pairs, whose MMA chains and
  // softmax a warp runs together; the last item of an odd count holds one window
  constexpr int QPER = (BITS == 2 && !ROPE) ? 2 : 1;
  const int nq = Q1 - Q0, nqi = (nq + QPER - 1) / QPER;   // Quantized windows and items of this CTA
  const int cta_items = has_sink + nqi + (L1 - L0) + (F1 - F0);
  // queue order [sink][Quantized][recent][Full]: the short bf16 items come last and fill the tail
  auto item_of = [&](int k) -> int {   // the item's (first) window
    if (has_sink) {
      if (k == 0) return 0;
      k -= 1;
    }
    if (k < nqi) return 1 + nL + nF + Q0 + QPER * k;
    k -= nqi;
    if (k < L1 - L0) return 1 + L0 + k;
    return 1 + nL + F0 + (k - (L1 - L0));
  };

  uint8_t *slots = smem;
  uint8_t *tbl = smem + Dg::MRG_OFF + DEC_CO_OFF + (warp < DEC_CONSUMERS ? warp : 0) * (D * 8 * 4);
  uint8_t *rel = smem + Dg::REL_OFF;
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + Dg::BAR_OFF);   // [Dg::FULL]
  uint64_t *empty = full + Dg::FULL;                                    // [DEC_SLOTS]
  __shared__ int q_next;    // next queue position to hand to a consumer warp

  // ---- chunk stream.  The CTA's windows in queue order [sink][Quantized][recent][Full]; a bf16
  // window is KCH K chunks then KCH V chunks (4 KB each), a Quantized window QCH chunks of its
  // ledger record, the sink none.  Chunk c lives in slot c % DEC_SLOTS and completes on
  // full[c % Dg::FULL].
  const int nb = (L1 - L0) + (F1 - F0);            // bf16 windows of this CTA
  const int n_total = BFC * nb + QCH * (Q1 - Q0);  // chunks of this CTA
  auto chunk_start = [&](int pos) -> int {
    const int k = pos - has_sink;
    if (k <= 0) return 0;
    return k <= nqi ? QCH * min(QPER * k, nq) : QCH * nq + BFC * (k - nqi);
  };
  // global source of chunk c
  auto chunk_src = [&](int c, const void *&src, uint32_t &bytes) {
    // the window of chunk c: Quantized window c / QCH of the CTA (chunks count windows, not queue
    // items, which pair Quantized windows), then the bf16 windows
    int it, sub;
    if (c < QCH * nq) {
      it = 1 + nL + nF + Q0 + c / QCH;
      sub = c % QCH;
    } else {
      const int bi = (c - QCH * nq) / BFC;   // bf16 window of the CTA: recent, then Full
      it = bi < L1 - L0 ? 1 + L0 + bi : 1 + nL + F0 + (bi - (L1 - L0));
      sub = (c - QCH * nq) % BFC;
    }
    if (it <= nL) {
      const int rs = (j0 + it - 1) % C.ring_windows;
      const __nv_bfloat16 *kb = ring + (size_t)rs * Gm::BLK;
      const __nv_bfloat16 *vb = ring + (size_t)(C.ring_windows + rs) * Gm::BLK;
      src = sub < KCH ? (const void *)(kb + sub * 2048) : (const void *)(vb + (sub - KCH) * 2048);
      bytes = DEC_STAGE_BYTES;
    } else if (it <= nL + nF) {
      int slot = __ldg(&ftab[it - 1 - nL].y);
      if (!qv_inbounds(slot >= 0 && slot < C.kf_cap(), status)) slot = 0;
      src = fpool + ((size_t)slot * C.h_kv + g) * 2 * Gm::BLK * 2 + (size_t)sub * DEC_STAGE_BYTES;
      bytes = DEC_STAGE_BYTES;
    } else {
      int slot = __ldg(&qtab[it - 1 - nL - nF].y);
      if (!qv_inbounds(slot >= 0 && slot < min(C.k_f + C.k_q, C.n_windows), status)) slot = 0;
      src = ledger + ((size_t)slot * C.h_kv + g) * Gm::QB + (size_t)sub * DEC_STAGE_BYTES;
      bytes = min(DEC_STAGE_BYTES, Gm::QB - sub * DEC_STAGE_BYTES);
    }
  };
  // the producer's first batch: one chunk per lane, its source looked up before the barrier
  const bool producer = warp == DEC_CONSUMERS;
  const void *src0 = nullptr;
  uint32_t bytes0 = 0;
  if (producer && lane < n_total) chunk_src(lane, src0, bytes0);
  if (threadIdx.x < Dg::FULL + DEC_SLOTS) {
    mbar_init(&full[threadIdx.x], 1);
    fence_mbar_init();
  }
  if (threadIdx.x == 0) q_next = 0;
  __syncthreads();

  float m_run[2] = {-INFINITY, -INFINITY}, l_run = 0.f, macc[2] = {0.f, 0.f};
  float o[8][4];
#pragma unroll
  for (int i = 0; i < 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;

  bool ok = true;
  auto wait_chunk = [&](int c) -> const uint8_t * {
    if (!mbar_wait(&full[c % Dg::FULL], (uint32_t)((c / Dg::FULL) & 1), status)) ok = false;
    return slots + (c % DEC_SLOTS) * DEC_STAGE_BYTES;
  };
  auto release_chunk = [&](int c) {
    if (lane == 0) mbar_arrive(&empty[c % DEC_SLOTS]);
  };

  if (producer) {
    // ---------------- producer warp: lane l issues chunk base + l of every batch of 32; a chunk
    // reuses its slot once the consumer of the chunk DEC_SLOTS earlier has released it
    // The cache windows of this layer do not depend on the previous kernel, so the first copies go
    // out before the wait, on an SM the previous kernel has already left.  (When the
    // previous kernel may be this layer's own decode, everything waited above.)
    // How many: the previous layer's last CTAs are merging their splits from L2 meanwhile, and a deep
    // burst of copies delays those loads; 16 chunks measured best for INT2, the whole batch for INT4.
    constexpr int PRE = BITS == 2 ? 16 : 32;
    int base0 = 0;
    if (!io.wait_first) {
      if (lane < PRE && lane < n_total) {
        mbar_arrive_expect_tx(&full[lane], bytes0);
        bulk_g2s(slots + lane * DEC_STAGE_BYTES, src0, bytes0, &full[lane]);
      }
      base0 = 32;
      asm volatile("griddepcontrol.wait;" ::: "memory");
      if (lane >= PRE && lane < n_total) {   // the rest of the first batch
        mbar_arrive_expect_tx(&full[lane], bytes0);
        bulk_g2s(slots + lane * DEC_STAGE_BYTES, src0, bytes0, &full[lane]);
      }
    }
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    int done = n_total;           // chunks before this one were all issued
    bool mine = false;            // this lane issued its chunk of the batch that stopped early
    for (int base = base0; base < n_total; base += 32) {
      const int c = base + lane;
      bool good = true;
      mine = false;
      if (c < n_total) {
        const void *src = src0;
        uint32_t bytes = bytes0;
        if (base > 0) chunk_src(c, src, bytes);
        if (c >= DEC_SLOTS) good = mbar_wait(&empty[c % DEC_SLOTS], (uint32_t)(((c / DEC_SLOTS) - 1) & 1), status);
        if (good) {
          uint64_t *bar = &full[c % Dg::FULL];
          mbar_arrive_expect_tx(bar, bytes);
          bulk_g2s(slots + (c % DEC_SLOTS) * DEC_STAGE_BYTES, src, bytes, bar);
          mine = true;
        }
      }
      if (!__all_sync(0xffffffffu, good)) {   // a wait ran out: stop issuing
        done = base;
        break;
      }
      mine = false;
    }
    // no copy may still be landing when the CTA ends.  Every earlier chunk of a slot landed before
    // the slot was reused, so only the last DEC_SLOTS chunks issued in order (and those of a batch
    // that stopped early) can still be in flight; none of them shares a barrier phase with another.
    for (int k = (done > DEC_SLOTS ? done - DEC_SLOTS : 0) + lane; k < done; k += 32)
      mbar_wait(&full[k % Dg::FULL], (uint32_t)((k / Dg::FULL) & 1), status);
    if (mine) {
      const int k = done + lane;
      mbar_wait(&full[k % Dg::FULL], (uint32_t)((k / Dg::FULL) & 1), status);
    }
    __syncwarp();
  } else {
  // ---------------- consumer warps
  // the step's inputs come from the previous kernel in a model: wait for it, then let the next start
  if (!io.wait_first) asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // q as the B operand of S^T = K q^T: b0 = q[head gl][16j+2tl .. +1], b1 = the same at +8
  uint32_t qb[8][2];
  {
    const __nv_bfloat16 *qh = io.q + ((size_t)b * C.h_q + (size_t)g * G + gl) * D;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      qb[j][0] = gl < G ? ldg32(qh + 16 * j + 2 * tl) : 0u;
      qb[j][1] = gl < G ? ldg32(qh + 16 * j + 2 * tl + 8) : 0u;
    }
  }
  if constexpr (ROPE) {
    // the offset table: rows 0..31 of the RoPE table, laid out as rel_cs reads it
    const float *tab = C.rope_tab();
    for (int k = threadIdx.x; k < DEC_REL_BYTES / 16; k += DEC_CONSUMERS * 32) {
      const int t = k >> 5, jj = (k >> 3) & 3, t4 = k & 3, hh = ((k >> 2) & 1) ^ (t & 1);
      *reinterpret_cast<float4 *>(rel + 16 * k) =
          cc_ss(__ldg(reinterpret_cast<const float4 *>(tab + ((size_t)t * 64 + 16 * jj + 2 * t4 + 8 * hh) * 2)));
    }
    asm volatile("bar.sync 1, %0;" ::"r"(DEC_CONSUMERS * 32) : "memory");   // consumer warps only
  }
  while (ok) {
    int pos = 0;
    if (lane == 0) pos = atomicAdd(&q_next, 1);
    pos = __shfl_sync(0xffffffffu, pos, 0);
    if (pos >= cta_items) break;
    const int c0 = chunk_start(pos);
    const int it = item_of(pos);
    float tsum;
    if (it == 0) {
      // ---------------- sink tokens (no mass): fragments straight from the compact sink rows
      float sacc[1][4] = {{0.f, 0.f, 0.f, 0.f}};
      const __nv_bfloat16 *sk = sink, *sv = sink + (size_t)C.n_sink * D;
      const bool r0 = gl < C.n_sink, r1 = gl + 8 < C.n_sink;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const uint32_t a0 = r0 ? ldg32(sk + gl * D + 16 * j + 2 * tl) : 0u;
        const uint32_t a1 = r1 ? ldg32(sk + (gl + 8) * D + 16 * j + 2 * tl) : 0u;
        const uint32_t a2 = r0 ? ldg32(sk + gl * D + 16 * j + 2 * tl + 8) : 0u;
        const uint32_t a3 = r1 ? ldg32(sk + (gl + 8) * D + 16 * j + 2 * tl + 8) : 0u;
        mma_bf16(sacc[0], a0, a1, a2, a3, qb[j][0], qb[j][1]);
      }
      const bool valid[1][2] = {{r0, r1}};
      online_step<1>(sacc, valid, m_run, l_run, o, macc, tsum, io.scale_log2);
      uint32_t pb[1][2];
      p_to_b<1>(sacc, pb, OScale<BITS>::P);
      const int t0 = 2 * tl, t1 = 2 * tl + 8;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int d0 = 16 * i + gl, d1 = d0 + 8;
        auto vv = [&](int t, int d) -> uint32_t { return t < C.n_sink ? ldg16(sv + t * D + d) : 0u; };
        const uint32_t a0 = vv(t0, d0) | (vv(t0 + 1, d0) << 16);
        const uint32_t a1 = vv(t0, d1) | (vv(t0 + 1, d1) << 16);
        const uint32_t a2 = vv(t1, d0) | (vv(t1 + 1, d0) << 16);
        const uint32_t a3 = vv(t1, d1) | (vv(t1 + 1, d1) << 16);
        mma_bf16(o[i], a0, a1, a2, a3, pb[0][0], pb[0][1]);
      }
      continue;
    }

    // log2-sum-exp of the window's logits per head, over its 32-token halves
    float wmu = -INFINITY;   // this lane's head: 2tl + (gl & 1)
    auto add_half_mass = [&]() {
      const float x = tsum > 0.f ? (gl & 1 ? m_run[1] : m_run[0]) + __log2f(tsum) : -INFINITY;
      const float hi = fmaxf(wmu, x), lo = fminf(wmu, x);
      wmu = lo == -INFINITY ? hi : hi + __log2f(1.f + exp2f(lo - hi));
    };

    if (it <= nL + nF) {
      // ---------------- bf16 window (recent or Full), one 32-token half at a time
      const bool is_local = it <= nL;
      const int wid = j0 + it - 1;   // the recent window (meaningful only when is_local)
      const int newtok = (is_local && wid == jn) ? T - (C.n_sink + jn * W) : -1;
#pragma unroll 1
      for (int hv = 0; hv < HALVES; ++hv) {
        bool valid[NMT][2];
        float s[NMT][4];
#pragma unroll
        for (int mt = 0; mt < NMT; ++mt) s[mt][0] = s[mt][1] = s[mt][2] = s[mt][3] = 0.f;
        const bool patch = newtok >= 0 && (newtok >> 5) == hv;
        const uint8_t *kc[NMT];
#pragma unroll
        for (int mt = 0; mt < NMT; ++mt) kc[mt] = wait_chunk(c0 + 2 * hv + mt);
        if (patch && ok) {
          // append: the new token enters the recent ring (global) and this warp's staged copy
          const int rs = jn % C.ring_windows;
          __nv_bfloat16 *kb = ring + (size_t)rs * Gm::BLK;
          const __nv_bfloat16 *kn = io.k_new + ((size_t)b * C.h_kv + g) * D;
          uint8_t *kst = const_cast<uint8_t *>(kc[(newtok >> 4) & 1]);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int d = 4 * lane + 2 * h;
            const uint32_t pair = ldg32(kn + d);
            const int idx = fnk_index(newtok, d);
            *reinterpret_cast<uint32_t *>(kb + idx) = pair;
            *reinterpret_cast<uint32_t *>(kst + (idx - (newtok >> 4) * 2048) * 2) = pair;
          }
          fence_proxy_async();   // this generic write must precede the slot's next bulk copy
          __syncwarp();
        }
#pragma unroll
        for (int mt = 0; mt < NMT; ++mt) {
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const uint4 a = lds128(kc[mt] + (j * 32 + lane) * 16);
            mma_bf16(s[mt], a.x, a.y, a.z, a.w, qb[j][0], qb[j][1]);
          }
        }
        __syncwarp();
#pragma unroll
        for (int mt = 0; mt < NMT; ++mt) release_chunk(c0 + 2 * hv + mt);
#pragma unroll
        for (int mt = 0; mt < NMT; ++mt) {
          const int tok0 = 32 * hv + 16 * mt + gl;
          if (is_local) {
            const int p0 = C.n_sink + wid * W + tok0;
            valid[mt][0] = p0 <= T;
            valid[mt][1] = p0 + 8 <= T;
          } else {
            valid[mt][0] = valid[mt][1] = true;
          }
        }
        online_step<NMT>(s, valid, m_run, l_run, o, macc, tsum, io.scale_log2);
        uint32_t pb[NMT][2];
        p_to_b<NMT>(s, pb, OScale<BITS>::P);
        const uint8_t *vc[NMT];
#pragma unroll
        for (int kk = 0; kk < NMT; ++kk) vc[kk] = wait_chunk(c0 + KCH + 2 * hv + kk);
        if (patch && ok) {
          const int rs = jn % C.ring_windows;
          __nv_bfloat16 *vb = ring + (size_t)(C.ring_windows + rs) * Gm::BLK;
          const __nv_bfloat16 *vn = io.v_new + ((size_t)b * C.h_kv + g) * D;
          uint8_t *vst = const_cast<uint8_t *>(vc[(newtok >> 4) & 1]);
#pragma unroll
          for (int h = 0; h < 4; ++h) {
            const int d = 4 * lane + h;
            const unsigned short x = (unsigned short)ldg16(vn + d);
            const int idx = fnv_index(newtok, d);
            reinterpret_cast<unsigned short *>(vb)[idx] = x;
            reinterpret_cast<unsigned short *>(vst)[idx - (newtok >> 4) * 2048] = x;
          }
          fence_proxy_async();
          __syncwarp();
        }
#pragma unroll
        for (int kk = 0; kk < NMT; ++kk) {
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const uint4 a = lds128(vc[kk] + (i * 32 + lane) * 16);
            mma_bf16(o[i], a.x, a.y, a.z, a.w, pb[kk][0], pb[kk][1]);
          }
        }
        __syncwarp();
#pragma unroll
        for (int kk = 0; kk < NMT; ++kk) release_chunk(c0 + KCH + 2 * hv + kk);
        add_half_mass();
      }
    } else if constexpr (BITS == 2 && !ROPE) {
      // ---------------- Quantized windows, W = 32, two per item: INT2 codes + fp16 scale/offset in one
      // chunk each.  The two windows' key products run as interleaved MMA chains and share one online
      // softmax step over their 64 tokens; their masses stay separate.
      const int qi = it - 1 - nL - nF;          // Q-table index of the first window
      const bool hasB = qi + 1 < Q1;            // the item's second window
      const uint8_t *ch[2];
      ch[0] = wait_chunk(c0);
      ch[1] = hasB ? wait_chunk(c0 + 1) : ch[0];
      ktab_int2(ch[0], tbl, lane);
      ktab_int2(ch[1], tbl + DEC_TBL_BYTES, lane);
      __syncwarp();
      uint4 kc[2][2];
#pragma unroll
      for (int w = 0; w < 2; ++w) {
        kc[w][0] = lds128(ch[w] + lane * 16);
        kc[w][1] = lds128(ch[w] + 512 + lane * 16);
      }
      float s2[2][2][4];
#pragma unroll
      for (int w = 0; w < 2; ++w)
#pragma unroll
        for (int mt = 0; mt < 2; ++mt) s2[w][mt][0] = s2[w][mt][1] = s2[w][mt][2] = s2[w][mt][3] = 0.f;
      keys_int2<2>(kc, tbl, qb, s2, tl);
      const bool vw[2] = {true, hasB};
      float ts[2];
      online_step_w<2>(s2, vw, m_run, l_run, o, macc, ts, io.scale_log2);
      pv_int2(s2[0], ch[0], o, macc, lane);
      if (hasB) pv_int2(s2[1], ch[1], o, macc, lane);
      __syncwarp();
      release_chunk(c0);
      if (hasB) release_chunk(c0 + 1);
      // the windows' log2-sum-exp per head (see below), under their stable indices
      if (gl < 2 && 2 * tl + gl < G) {
        const float mr = gl & 1 ? m_run[1] : m_run[0];
        const int sidx = 1 + qi + C.loc_items() + C.kf_cap();   // as for single windows below
        mu[(size_t)sidx * G + 2 * tl + gl] = ts[0] > 0.f ? mr + __log2f(ts[0]) : -INFINITY;
        if (hasB) mu[(size_t)(sidx + 1) * G + 2 * tl + gl] = ts[1] > 0.f ? mr + __log2f(ts[1]) : -INFINITY;
      }
      continue;
    } else if constexpr (BITS == 2) {
      // ---------------- Quantized window with pre-RoPE keys, W = 32: INT2 codes + fp16 scale/offset
      // in one chunk
      bool valid[NMT][2];
      float s[NMT][4];
#pragma unroll
      for (int mt = 0; mt < NMT; ++mt) s[mt][0] = s[mt][1] = s[mt][2] = s[mt][3] = 0.f;
      // this lane's 16 B of the RoPE row of the window's first position
      const int wq = __ldg(&qtab[it - 1 - nL - nF].x);
      const float4 csr = __ldg(reinterpret_cast<const float4 *>(C.rope_tab() + (size_t)(C.n_sink + wq * W) * D) + lane);
      const uint8_t *ch = wait_chunk(c0);
      ktab_int2(ch, tbl, lane);
      *reinterpret_cast<float4 *>(tbl + 2 * DEC_TBL_BYTES + 16 * lane) = cc_ss(csr);
      __syncwarp();
      const uint4 kcw0 = lds128(ch + lane * 16), kcw1 = lds128(ch + 512 + lane * 16);
      // k-steps jj and jj + 4 hold the RoPE partners (channels c and c + 64) in the same registers
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {
        const uint4 TA0 = lds128(tbl + (jj * 4 + tl) * 32), TB0 = lds128(tbl + (jj * 4 + tl) * 32 + 16);
        const uint4 TA1 = lds128(tbl + ((jj + 4) * 4 + tl) * 32), TB1 = lds128(tbl + ((jj + 4) * 4 + tl) * 32 + 16);
        const uint8_t *csw = tbl + 2 * DEC_TBL_BYTES + (16 * jj + 2 * tl) * 8;
        const float4 cb0 = *reinterpret_cast<const float4 *>(csw), cb1 = *reinterpret_cast<const float4 *>(csw + 64);
        const float2 ncb0 = make_float2(-cb0.z, -cb0.w), ncb1 = make_float2(-cb1.z, -cb1.w);
#pragma unroll
        for (int mt = 0; mt < NMT; ++mt) {
          // k-step j sits in code word j / 2, low half for even j
          const uint4 &kc = mt == 0 ? kcw0 : kcw1;
          const uint32_t wa = word_of(kc, jj >> 1) >> (16 * (jj & 1));
          const uint32_t wb = word_of(kc, 2 + (jj >> 1)) >> (16 * (jj & 1));
          uint32_t ka[4], kb[4];
          lut_k_regs((wa & 0x3333u) | 0x4040u, ((wa >> 2) & 0x3333u) | 0x4040u, TA0, TB0, ka[0], ka[1], ka[2], ka[3]);
          lut_k_regs((wb & 0x3333u) | 0x4040u, ((wb >> 2) & 0x3333u) | 0x4040u, TA1, TB1, kb[0], kb[1], kb[2], kb[3]);
#pragma unroll
          for (int r = 0; r < 4; ++r) {
            const int tt = 16 * mt + gl + 8 * (r & 1);
            rope_rot(bf16_lo(ka[r]), bf16_hi(ka[r]), bf16_lo(kb[r]), bf16_hi(kb[r]), (r >> 1) ? cb1 : cb0, (r >> 1) ? ncb1 : ncb0,
                     rel_cs(rel, tt, jj, r >> 1, tl), ka[r], kb[r]);
          }
          mma_bf16(s[mt], ka[0], ka[1], ka[2], ka[3], qb[jj][0], qb[jj][1]);
          mma_bf16(s[mt], kb[0], kb[1], kb[2], kb[3], qb[jj + 4][0], qb[jj + 4][1]);
        }
      }
#pragma unroll
      for (int mt = 0; mt < NMT; ++mt) {
        valid[mt][0] = valid[mt][1] = true;
      }
      online_step<NMT>(s, valid, m_run, l_run, o, macc, tsum, io.scale_log2);
      pv_int2(s, ch, o, macc, lane);
      __syncwarp();
      release_chunk(c0);
      add_half_mass();
    } else {
      // ---------------- Quantized window, W = 64: INT4 codes; chunks K codes | V codes | parameters
      float4 csr[HALVES];   // ROPE: this lane's 16 B of the RoPE rows of each half's first position
      if constexpr (ROPE) {
        const int wq = __ldg(&qtab[it - 1 - nL - nF].x);
#pragma unroll
        for (int hv = 0; hv < HALVES; ++hv)
          csr[hv] = __ldg(reinterpret_cast<const float4 *>(C.rope_tab() + (size_t)(C.n_sink + wq * W + 32 * hv) * D) + lane);
      }
      const uint8_t *kch = wait_chunk(c0);
      const uint8_t *vch = wait_chunk(c0 + 1);
      const uint8_t *pch = wait_chunk(c0 + 2);
      // per-channel fp32 (scale, offset) for the four channels 2t, 2t+1, 2t+8, 2t+9 of every
      // (k-step j, lane class t): 8 floats, scales then offsets
      {
        const uint2 sp = *reinterpret_cast<const uint2 *>(pch + (Gm::OFF_KS - 2 * Gm::CODE_BYTES) + 8 * lane);
        const uint2 mp = *reinterpret_cast<const uint2 *>(pch + (Gm::OFF_KM - 2 * Gm::CODE_BYTES) + 8 * lane);
        float *tf = reinterpret_cast<float *>(tbl);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint32_t sw = k < 2 ? sp.x : sp.y, mw = k < 2 ? mp.x : mp.y;
          const int d = 4 * lane + k, j = d >> 4, c16 = d & 15;
          const int t = (c16 & 7) >> 1, which = c16 >> 3, half = c16 & 1;
          const int base = (j * 4 + t) * 8 + which * 2 + half;
          tf[base] = (k & 1) ? h2f_hi(sw) : h2f_lo(sw);
          tf[base + 4] = (k & 1) ? h2f_hi(mw) : h2f_lo(mw);
        }
      }
      if constexpr (ROPE) {
#pragma unroll
        for (int hv = 0; hv < HALVES; ++hv)
          *reinterpret_cast<float4 *>(tbl + DEC_TBL_BYTES + hv * 512 + 16 * lane) = cc_ss(csr[hv]);
      }
      __syncwarp();
      const __half *vsp = reinterpret_cast<const __half *>(pch + (Gm::OFF_VS - 2 * Gm::CODE_BYTES));
      const __half *vmp = reinterpret_cast<const __half *>(pch + (Gm::OFF_VM - 2 * Gm::CODE_BYTES));
#pragma unroll 1
      for (int hv = 0; hv < HALVES; ++hv) {
        bool valid[NMT][2];
        float s[NMT][4];
#pragma unroll
        for (int mt = 0; mt < NMT; ++mt) s[mt][0] = s[mt][1] = s[mt][2] = s[mt][3] = 0.f;
        // keys: tile (token group tg, k-step j) is word ((tile/4)*32 + lane)*4 + tile%4 of the K codes
#pragma unroll
        for (int mt = 0; mt < NMT; ++mt) {
          const int tg = 2 * hv + mt;
          const uint4 w03 = lds128(kch + (((2 * tg) * 32 + lane) * 4) * 4);
          const uint4 w47 = lds128(kch + (((2 * tg + 1) * 32 + lane) * 4) * 4);
          if constexpr (ROPE) {
            // pre-RoPE keys bf16(fp32(c * s + m)), rotated to their positions; k-steps jj and jj + 4
            // hold the RoPE partners in the same registers
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
              const uint32_t wa = word_of(w03, jj), wb = word_of(w47, jj);
              const uint32_t Ea = wa & 0x0F0F0F0Fu, Oa = (wa >> 4) & 0x0F0F0F0Fu;
              const uint32_t Eb = wb & 0x0F0F0F0Fu, Ob = (wb >> 4) & 0x0F0F0F0Fu;
              const float4 sa = *reinterpret_cast<const float4 *>(tbl + (jj * 4 + tl) * 32);
              const float4 ma = *reinterpret_cast<const float4 *>(tbl + (jj * 4 + tl) * 32 + 16);
              const float4 sb = *reinterpret_cast<const float4 *>(tbl + ((jj + 4) * 4 + tl) * 32);
              const float4 mb = *reinterpret_cast<const float4 *>(tbl + ((jj + 4) * 4 + tl) * 32 + 16);
              const uint8_t *csw = tbl + DEC_TBL_BYTES + hv * 512 + (16 * jj + 2 * tl) * 8;
              const float4 cb0 = *reinterpret_cast<const float4 *>(csw), cb1 = *reinterpret_cast<const float4 *>(csw + 64);
              const float2 ncb0 = make_float2(-cb0.z, -cb0.w), ncb1 = make_float2(-cb1.z, -cb1.w);
              uint32_t ka[4], kb[4];
#pragma unroll
              for (int r = 0; r < 4; ++r) {
                const bool h8 = r >= 2;   // channels 2t + 8, 2t + 9
                float ca0, ca1, cb0f, cb1f;
                nib_f2(Ea, Oa, r, ca0, ca1);
                nib_f2(Eb, Ob, r, cb0f, cb1f);
                const uint32_t pa = dq_k4(ca0, ca1, h8 ? sa.z : sa.x, h8 ? sa.w : sa.y, h8 ? ma.z : ma.x, h8 ? ma.w : ma.y);
                const uint32_t pbk = dq_k4(cb0f, cb1f, h8 ? sb.z : sb.x, h8 ? sb.w : sb.y, h8 ? mb.z : mb.x, h8 ? mb.w : mb.y);
                const float a0 = bf16_lo(pa), a1 = bf16_hi(pa), b0 = bf16_lo(pbk), b1 = bf16_hi(pbk);
                rope_rot(a0, a1, b0, b1, h8 ? cb1 : cb0, h8 ? ncb1 : ncb0, rel_cs(rel, 16 * mt + gl + 8 * (r & 1), jj, r >> 1, tl),
                         ka[r], kb[r]);
              }
              mma_bf16(s[mt], ka[0], ka[1], ka[2], ka[3], qb[jj][0], qb[jj][1]);
              mma_bf16(s[mt], kb[0], kb[1], kb[2], kb[3], qb[jj + 4][0], qb[jj + 4][1]);
            }
          } else {
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const uint32_t w = word_of(j < 4 ? w03 : w47, j & 3);
            const uint32_t E = w & 0x0F0F0F0Fu, Od = (w >> 4) & 0x0F0F0F0Fu;
            const float4 sc = *reinterpret_cast<const float4 *>(tbl + (j * 4 + tl) * 32);
            const float4 mn = *reinterpret_cast<const float4 *>(tbl + (j * 4 + tl) * 32 + 16);
            float c[4][2];
#pragma unroll
            for (int r = 0; r < 4; ++r) nib_f2(E, Od, r, c[r][0], c[r][1]);
            const uint32_t a0 = dq_k4(c[0][0], c[0][1], sc.x, sc.y, mn.x, mn.y);
            const uint32_t a1 = dq_k4(c[1][0], c[1][1], sc.x, sc.y, mn.x, mn.y);
            const uint32_t a2 = dq_k4(c[2][0], c[2][1], sc.z, sc.w, mn.z, mn.w);
            const uint32_t a3 = dq_k4(c[3][0], c[3][1], sc.z, sc.w, mn.z, mn.w);
            mma_bf16(s[mt], a0, a1, a2, a3, qb[j][0], qb[j][1]);
          }
          }
        }
#pragma unroll
        for (int mt = 0; mt < NMT; ++mt) {
          valid[mt][0] = valid[mt][1] = true;
        }
        online_step<NMT>(s, valid, m_run, l_run, o, macc, tsum, io.scale_log2);
        uint32_t pbh[NMT][2];
        float pm0 = 0.f, pm1 = 0.f;
#pragma unroll
        for (int kk = 0; kk < NMT; ++kk) {
          const int t0 = 32 * hv + 16 * kk + gl, t1 = t0 + 8;
          const float s0v = __half2float(vsp[t0]), s1v = __half2float(vsp[t1]);
          const float m0v = __half2float(vmp[t0]), m1v = __half2float(vmp[t1]);
          fma2(pm0, pm1, s[kk][2], s[kk][3], m1v, m1v, pm0, pm1);
          fma2(pm0, pm1, s[kk][0], s[kk][1], m0v, m0v, pm0, pm1);
          float x0, x1, x2, x3;
          mul2(x0, x1, s[kk][0], s[kk][1], s0v, s0v);
          mul2(x2, x3, s[kk][2], s[kk][3], s1v, s1v);
          pbh[kk][0] = movmatrix_trans(pack_half(x0, x1));
          pbh[kk][1] = movmatrix_trans(pack_half(x2, x3));
        }
        macc[0] += pm0;
        macc[1] += pm1;
        // values: tile (token group tg, dim tile i) is word ((tile/4)*32 + lane)*4 + tile%4 of the V
        // codes; its registers 0, 1 sit at nibbles 0, 1 of each half, registers 2, 3 at nibbles 2, 3
#pragma unroll
        for (int kk = 0; kk < NMT; ++kk) {
          const int tg = 2 * hv + kk;
          const uint4 w03 = lds128(vch + (((2 * tg) * 32 + lane) * 4) * 4);
          const uint4 w47 = lds128(vch + (((2 * tg + 1) * 32 + lane) * 4) * 4);
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const uint32_t w = word_of(i < 4 ? w03 : w47, i & 3);
            const uint32_t w8 = w >> 8;
            mma_f16(o[i], dq_v4(w, 0), dq_v4(w, 1), dq_v4(w8, 0), dq_v4(w8, 1), pbh[kk][0], pbh[kk][1]);
          }
        }
        add_half_mass();
      }
      __syncwarp();
      release_chunk(c0);
      release_chunk(c0 + 1);
      release_chunk(c0 + 2);
    }
    // the window's log2-sum-exp per head: its mass is 2^(mu - M) / L with the merged max M and sum
    // L; recorded under the window's stable index (recent, then Full, then Quantized)
    if (gl < 2 && 2 * tl + gl < G) {
      const int sidx = it <= nL ? it : (it <= nL + nF ? it - nL + C.loc_items() : it - nL - nF + C.loc_items() + C.kf_cap());
      mu[(size_t)sidx * G + 2 * tl + gl] = wmu;
    }
  }
  }   // consumer warps

  // ---------------- merge the consumer warps of this CTA into one split partial; each consumer
  // warp stores its state as soon as its queue runs dry, into a region of its own
  const int lgG = __ffs(G) - 1;
  float *cm = reinterpret_cast<float *>(smem + Dg::MRG_OFF);   // [DEC_CONSUMERS][8] running max
  float *cl = cm + DEC_CONSUMERS * 8;            // [DEC_CONSUMERS][8] running sum
  float *cf = cl + DEC_CONSUMERS * 8;            // [DEC_CONSUMERS][8] rescale factor to the CTA max
  float *sM = cf + DEC_CONSUMERS * 8;            // [16] CTA max per head, then the merged max and 1/L
  float *cO = sM + 16;                           // [DEC_CONSUMERS][D][8] unnormalised outputs
  if (warp < DEC_CONSUMERS) {
    // the Quantized values' offset term was summed per lane; its lanes of each head meet once, here
    macc[0] = warp_sum_xor_g(macc[0]);
    macc[1] = warp_sum_xor_g(macc[1]);
    if (gl < 2) {
      cm[warp * 8 + 2 * tl + gl] = gl ? m_run[1] : m_run[0];
      cl[warp * 8 + 2 * tl + gl] = l_run;
    }
    if (2 * tl < G) {   // heads 2tl, 2tl+1 of dims 16i+gl and 16i+gl+8, as float2
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        float *r = cO + ((size_t)warp * D + 16 * i + gl) * 8 + 2 * tl;
        constexpr float U = OScale<BITS>::INV;   // the accumulators' scale, undone here
        *reinterpret_cast<float2 *>(r) = make_float2(fmaf(o[i][0], U, macc[0]), fmaf(o[i][1], U, macc[1]));
        *reinterpret_cast<float2 *>(r + 64) = make_float2(fmaf(o[i][2], U, macc[0]), fmaf(o[i][3], U, macc[1]));
      }
    }
  }
  __syncthreads();   // also: every bulk copy into the slot ring has landed (producer drain)
  if (threadIdx.x < DEC_CONSUMERS * 8) {
    const int h = threadIdx.x & 7;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < DEC_CONSUMERS; ++w) M = fmaxf(M, cm[w * 8 + h]);
    cf[threadIdx.x] = M == -INFINITY ? 0.f : exp2f(cm[threadIdx.x] - M);
    if (threadIdx.x < 8) sM[h] = M;
  }
  __syncthreads();
  float *mypart = part + (size_t)split * PART_FLOATS;
  for (int idx = threadIdx.x; idx < G * D; idx += blockDim.x) {
    const int h = idx & (G - 1), d = idx >> lgG;
    float acc = 0.f;
#pragma unroll
    for (int w = 0; w < DEC_CONSUMERS; ++w) acc = fmaf(cO[((size_t)w * D + d) * 8 + h], cf[w * 8 + h], acc);
    mypart[16 + h * D + d] = acc;
  }
  if (threadIdx.x < G) {
    float l = 0.f;
#pragma unroll
    for (int w = 0; w < DEC_CONSUMERS; ++w) l = fmaf(cl[w * 8 + threadIdx.x], cf[w * 8 + threadIdx.x], l);
    mypart[threadIdx.x] = sM[threadIdx.x];
    mypart[8 + threadIdx.x] = l;
  }

  // ---------------- the last CTA of this (sequence, KV head) merges the splits
  __shared__ int s_last;
  __syncthreads();   // every partial write of this CTA happens before thread 0's release below
  unsigned *splitctr = reinterpret_cast<unsigned *>(C.arena + C.off_splitctr) + ((size_t)io.layer * C.B + b) * C.h_kv + g;
  if (threadIdx.x == 0) {
    unsigned prev;
    asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], 1;" : "=r"(prev) : "l"(splitctr) : "memory");
    s_last = prev == (unsigned)(C.n_split - 1);
  }
  __syncthreads();
  if (!s_last) return;

  // outputs: one warp covers 32 dims of one head; lane sp holds split sp's (m, l), the merged max M
  // and sum L come from warp reductions, and each lane folds every split's output for its dim.  A
  // thread may own several (head, dim) items: the loads of all of them are issued before any is
  // used, so the partials cross the L2 once (per 32 splits).
  const int nsp = C.n_split;
  constexpr int IPT = (8 * D + DEC_WARPS * 32 - 1) / (DEC_WARPS * 32);   // (head, dim) items per thread
  float M[IPT], L[IPT], O[IPT];
#pragma unroll
  for (int k = 0; k < IPT; ++k) M[k] = -INFINITY, L[k] = 0.f, O[k] = 0.f;
  for (int s0 = 0; s0 < nsp; s0 += 32) {
    const int n = min(32, nsp - s0);
    float ov[IPT][32], lk[IPT], mk[IPT];
#pragma unroll
    for (int k = 0; k < IPT; ++k) {
      const int idx = threadIdx.x + k * DEC_WARPS * 32;   // the same head across a warp (D % 32 == 0)
      const bool valid = idx < G * D;
      const int h = valid ? idx / D : 0;
      const float *po = part + 16 + (valid ? idx : 0) + (size_t)s0 * PART_FLOATS;
#pragma unroll
      for (int x = 0; x < 32; ++x) ov[k][x] = (valid && x < n) ? __ldcg(po + (size_t)x * PART_FLOATS) : 0.f;
      const float *ph = part + h + (size_t)(s0 + lane) * PART_FLOATS;
      lk[k] = (valid && lane < n) ? __ldcg(ph + 8) : 0.f;
      mk[k] = (valid && lane < n) ? __ldcg(ph) : -INFINITY;
    }
#pragma unroll
    for (int k = 0; k < IPT; ++k) {
      if (threadIdx.x + k * DEC_WARPS * 32 >= G * D) continue;   // uniform over the warp
      const float l = lk[k], m = mk[k];
      float Mc = l > 0.f ? m : -INFINITY;
#pragma unroll
      for (int x = 16; x >= 1; x >>= 1) Mc = fmaxf(Mc, __shfl_xor_sync(0xffffffffu, Mc, x));
      const float Mn = fmaxf(M[k], Mc);   // finite: the newest token's window always holds mass
      const float cold = M[k] == -INFINITY ? 0.f : exp2f(M[k] - Mn);
      const float e = l > 0.f ? exp2f(m - Mn) : 0.f;
      float Lc = l * e;
#pragma unroll
      for (int x = 16; x >= 1; x >>= 1) Lc += __shfl_xor_sync(0xffffffffu, Lc, x);
      float Oc0 = 0.f, Oc1 = 0.f;
#pragma unroll
      for (int x = 0; x < 32; x += 2) {
        Oc0 = fmaf(ov[k][x], __shfl_sync(0xffffffffu, e, x), Oc0);
        Oc1 = fmaf(ov[k][x + 1], __shfl_sync(0xffffffffu, e, x + 1), Oc1);
      }
      L[k] = fmaf(L[k], cold, Lc);
      O[k] = fmaf(O[k], cold, Oc0 + Oc1);
      M[k] = Mn;
    }
  }
#pragma unroll
  for (int k = 0; k < IPT; ++k) {
    const int idx = threadIdx.x + k * DEC_WARPS * 32;
    if (idx >= G * D) continue;
    const int h = idx / D, d = idx % D;
    const float inv = 1.f / L[k];
    io.out[((size_t)b * C.h_q + (size_t)g * G + h) * D + d] = __float2bfloat16_rn(O[k] * inv);
    if (d == 0) {   // this step's merged max and 1/L: the window masses are applied when scores are flushed
      float *ms = reinterpret_cast<float *>(C.arena + C.off_mstat + C.st_mstat_layer * io.layer) +
                  ((size_t)bg * C.omega + mslot) * 16;
      ms[h] = M[k];
      ms[8 + h] = inv;
    }
  }
  // every CTA of this KV head has read T and arrived: the head's copy of T advances (head 0's also
  // in the unit's meta record, which the router and the score flush read)
  if (threadIdx.x == 0) {
    *splitctr = 0u;
    *thead = T + 1;
    if (g == 0) meta[M_T] = T + 1;
  }
}

template <int W, int BITS, bool ROPE>
static cudaError_t launch_decode_fmt(const CacheDev &C, const DecodeIO &io, cudaStream_t stream) {
  using Dg = DecGeo<W, BITS, ROPE>;
  auto kern = decode_kernel<W, BITS, ROPE>;
  static SmemOptIn optin;   // per device: the dynamic shared memory opt-in of this kernel
  const cudaError_t e = optin.ensure(kern, Dg::SMEM);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = C.B == 1 ? dim3(C.h_kv, 1, C.n_split) : dim3(C.n_split, C.h_kv, C.B);
  cfg.blockDim = dim3(DEC_WARPS * 32);
  cfg.dynamicSmemBytes = Dg::SMEM;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, C, io);
}

cudaError_t launch_decode(const CacheDev &C, const DecodeIO &io, cudaStream_t stream) {
  if (C.W == 32 && C.bits == 2)
    return C.rope ? launch_decode_fmt<32, 2, true>(C, io, stream) : launch_decode_fmt<32, 2, false>(C, io, stream);
  if (C.W == 64 && C.bits == 4)
    return C.rope ? launch_decode_fmt<64, 4, true>(C, io, stream) : launch_decode_fmt<64, 4, false>(C, io, stream);
  return cudaErrorInvalidValue;
}

}  // namespace qv
