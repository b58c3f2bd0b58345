// Device-side building blocks shared by the QEvict kernels (sm_103a).
//
// Layout maps (fragment-native blocks, code fields), PTX wrappers for the
// mbarrier / 1-D bulk-copy (TMA) pipeline, mma.sync / movmatrix, and the
// bounded waits every kernel uses.  No wait in this library spins without a
// limit: a wait that runs out records QV_ERR_TIMEOUT in the device status word
// and returns false so the kernel can leave cleanly.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace qv {

constexpr int D = 128;            // head dimension (fixed)
constexpr int META_INTS = 16;     // per-unit meta words
// M_FLUSHT: tokens cached when the window scores last absorbed the decode steps' masses
enum : int { M_T = 0, M_NROUTE = 1, M_FCOUNT = 2, M_QCOUNT = 3, M_NQUANT = 4, M_NMOVE = 5, M_NEVENT = 6, M_FLUSHT = 7 };

enum : int { TIER_LOCAL = 0, TIER_FULL = 1, TIER_QUANT = 2, TIER_EVICT = 3 };
enum : int { LED_NONE = 0, LED_ACTIVE = 1, LED_DORMANT = 2 };
enum : int { QV_ERR_TIMEOUT = 1, QV_ERR_SLOT = 2, QV_ERR_STATE = 4, QV_ERR_BOUNDS = 8 };

// Checked builds (compiled with -DQEVICT_CHECK, libqevict_check.so) test every index read from
// device data before the access it guards: an index outside its buffer records QV_ERR_BOUNDS in the
// device status word and the access is skipped.  Other builds compile the test away.
#ifdef QEVICT_CHECK
__device__ __forceinline__ bool qv_inbounds(bool ok, int *status) {
  if (!ok) atomicOr(status, QV_ERR_BOUNDS);
  return ok;
}
#else
__device__ __forceinline__ bool qv_inbounds(bool, int *) { return true; }
#endif
enum : int { N_COUNTERS = 8 };    // 7 used: promo, demo, firstq, react, evict, aged_f, aged_q

// ----------------------------------------------------------------------------- layout maps

// m16n8k16 A-operand register map for a 16x16 tile: element (r, c) sits in
// lane (r%8)*4 + (c%8)/2, register r/8 + 2*(c/8), half c%2.
__host__ __device__ __forceinline__ int frag_lane(int r, int c) { return ((r & 7) << 2) | ((c & 7) >> 1); }
__host__ __device__ __forceinline__ int frag_reg(int r, int c) { return (r >> 3) | ((c >> 3) << 1); }

// K block of one window: A operand of S^T = K q^T (rows = tokens, cols = dims).
__host__ __device__ __forceinline__ int fnk_index(int tok, int dim) {
  const int r = tok & 15, c = dim & 15, grp = (tok >> 4) * 8 + (dim >> 4);
  return ((grp * 32 + frag_lane(r, c)) << 3) | (frag_reg(r, c) << 1) | (c & 1);
}
// V block of one window: A operand of O^T = V^T P^T (rows = dims, cols = tokens).
__host__ __device__ __forceinline__ int fnv_index(int tok, int dim) {
  const int r = dim & 15, c = tok & 15, grp = (tok >> 4) * 8 + (dim >> 4);
  return ((grp * 32 + frag_lane(r, c)) << 3) | (frag_reg(r, c) << 1) | (c & 1);
}

// Position of the INT2 code of element (tok, dim) inside a window's K or V code block (1 KB for
// W = 32): returns the byte offset and the bit shift inside that byte.  Each lane of the decode warp
// owns 32 bytes, stored as two 16-byte pieces at piece*512 + lane*16 (conflict-free 128-bit loads).
//  K: the codes of one m16n8k16 A-register group (16 tokens x 16 channels) form a 16-bit field per
//     lane; element e = reg*2 + half sits at bit 4e (e < 4) or 4(e-4)+2 (e >= 4), so masking with
//     0x3333 yields byte-permute selectors directly.
//  V: one 32-bit word per 16-dim tile i (word i of the lane's 32 bytes): the register of row half
//     rh = (dim%16)/8 and token pair tau = 2*(tok/16) + (tok%16)/8 keeps its two codes (even, odd
//     token) at bits b and b+16 with b = 8*rh + 2*tau.  One mask (after a shift by 8 for rh = 1)
//     leaves them as the mantissas of two fp16 subnormals, c * 4^tau * 2^-24: the power of 4 depends
//     on the token pair only, so the P operand of those tokens can carry its inverse.
__host__ __device__ __forceinline__ void code_pos2(bool is_v, int tok, int dim, int &byte, int &shift) {
  int lb, bit;
  if (!is_v) {
    const int r = tok & 15, c = dim & 15, grp = (tok >> 4) * 8 + (dim >> 4);
    const int lane = frag_lane(r, c);
    const int e = (frag_reg(r, c) << 1) | (c & 1);
    bit = e < 4 ? 4 * e : 4 * (e - 4) + 2;
    lb = grp * 2 + (bit >> 3);
    byte = (lb >> 4) * 512 + lane * 16 + (lb & 15);
  } else {
    const int rr = dim & 15, c = tok & 15, i = dim >> 4;
    const int lane = frag_lane(rr, c);
    const int tau = 2 * (tok >> 4) + (c >> 3);
    bit = 8 * (rr >> 3) + 2 * tau + 16 * (c & 1);
    lb = 4 * i + (bit >> 3);
    byte = (lb >> 4) * 512 + lane * 16 + (lb & 15);
  }
  shift = bit & 7;
}

// Position of the INT4 code of element (tok, dim) inside a window's K or V code block (4 KB for
// W = 64): one 32-bit word per (16x16 tile, lane), tile = (tok/16)*8 + dim/16, stored at word
// ((tile/4)*32 + lane)*4 + tile%4 (a lane's four consecutive tiles are one 128-bit load).
//  K: element e = reg*2 + dim%2 of the lane's A registers sits at bits 4e.
//  V: register reg's two codes (even, odd token) sit at bits 4*reg and 16 + 4*reg, so registers
//     0, 1 (and 2, 3 after a shift by 8) are one mask away from fp16 mantissas.
__host__ __device__ __forceinline__ void code_pos4(bool is_v, int tok, int dim, int &byte, int &shift) {
  const int tile = (tok >> 4) * 8 + (dim >> 4);
  const int r = is_v ? (dim & 15) : (tok & 15), c = is_v ? (tok & 15) : (dim & 15);
  const int lane = frag_lane(r, c);
  const int word = ((tile >> 2) * 32 + lane) * 4 + (tile & 3);
  const int bit = is_v ? 4 * frag_reg(r, c) + 16 * (c & 1) : 4 * ((frag_reg(r, c) << 1) | (c & 1));
  byte = word * 4 + (bit >> 3);
  shift = bit & 7;
}

template <int BITS>
__host__ __device__ __forceinline__ void code_pos(bool is_v, int tok, int dim, int &byte, int &shift) {
  if (BITS == 2)
    code_pos2(is_v, tok, dim, byte, shift);
  else
    code_pos4(is_v, tok, dim, byte, shift);
}

template <int W, int BITS>
struct Geo {
  static constexpr int BLK = W * D;                     // elements of one K or V block
  static constexpr int GROUPS = W / 16;                 // 16-token groups per window
  static constexpr int CODE_BYTES = W * D * BITS / 8;   // K (or V) codes of one window and head
  static constexpr int OFF_VCODE = CODE_BYTES;
  static constexpr int OFF_KS = 2 * CODE_BYTES;         // fp16 K scale [D]
  static constexpr int OFF_KM = OFF_KS + 2 * D;         // fp16 K offset [D]
  static constexpr int OFF_VS = OFF_KM + 2 * D;         // fp16 V scale [W]
  static constexpr int OFF_VM = OFF_VS + 2 * W;         // fp16 V offset [W]
  static constexpr int QB = OFF_VM + 2 * W;             // ledger bytes per (slot, head)
};

// ----------------------------------------------------------------------------- small PTX wrappers

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait on an mbarrier phase: gives up after ~200 ms, records the timeout and returns false.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, int *status) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 0;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 255u) == 255u && globaltimer_ns() - t0 > 200000000ull) {
      atomicOr(status, QV_ERR_TIMEOUT);
      return false;
    }
  }
}

// Packed fp32 pairs: two values per instruction, each product and sum rounded on its own (RN).
__device__ __forceinline__ void fma2(float &dx, float &dy, float ax, float ay, float bx, float by, float cx, float cy) {
  asm("{\n .reg .b64 ra, rb, rc, rd;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n mov.b64 rc, {%6, %7};\n"
      " fma.rn.f32x2 rd, ra, rb, rc;\n mov.b64 {%0, %1}, rd;\n}"
      : "=f"(dx), "=f"(dy)
      : "f"(ax), "f"(ay), "f"(bx), "f"(by), "f"(cx), "f"(cy));
}
__device__ __forceinline__ void add2(float &ax, float &ay, float bx, float by) {
  asm("{\n .reg .b64 ra, rb, rd;\n mov.b64 ra, {%0, %1};\n mov.b64 rb, {%2, %3};\n add.rn.f32x2 rd, ra, rb;\n"
      " mov.b64 {%0, %1}, rd;\n}"
      : "+f"(ax), "+f"(ay)
      : "f"(bx), "f"(by));
}
__device__ __forceinline__ void sub2(float &dx, float &dy, float ax, float ay, float bx, float by) {
  asm("{\n .reg .b64 ra, rb, rd;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n sub.rn.f32x2 rd, ra, rb;\n"
      " mov.b64 {%0, %1}, rd;\n}"
      : "=f"(dx), "=f"(dy)
      : "f"(ax), "f"(ay), "f"(bx), "f"(by));
}
__device__ __forceinline__ void mul2(float &dx, float &dy, float ax, float ay, float bx, float by) {
  asm("{\n .reg .b64 ra, rb, rd;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n mul.rn.f32x2 rd, ra, rb;\n"
      " mov.b64 {%0, %1}, rd;\n}"
      : "=f"(dx), "=f"(dy)
      : "f"(ax), "f"(ay), "f"(bx), "f"(by));
}

// 1-D bulk copy global -> shared (TMA), completion counted on `bar` in bytes.
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ uint4 lds128(const void *p) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(smem_u32(p)));
  return v;
}

// D += A * B, m16n8k16, bf16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Transpose of an 8x8 b16 matrix held one register per lane (row lane/4, cols 2*(lane%4)+{0,1}).
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t a) {
  uint32_t d;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
  return d;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);   // RN-even, lo in the low half
  return *reinterpret_cast<uint32_t *>(&v);
}

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

template <typename T>
__device__ __forceinline__ T warp_max_xor_g(T v) {   // reduce over lanes sharing lane%4
  v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 4));
  v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 8));
  v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 16));
  return v;
}
__device__ __forceinline__ float warp_sum_xor_g(float v) {
  v += __shfl_xor_sync(0xffffffffu, v, 4);
  v += __shfl_xor_sync(0xffffffffu, v, 8);
  v += __shfl_xor_sync(0xffffffffu, v, 16);
  return v;
}

// Windows whose tokens have all left the recent region when T tokens are cached.
__device__ __forceinline__ int n_hist_dev(int T, int n_recent, int n_sink, int W) {
  const int x = T - n_recent - n_sink;
  return x > 0 ? x / W : 0;
}

}  // namespace qv
