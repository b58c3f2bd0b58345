// Device view of the routing-diagnostics state (csrc/diag.cu): per-unit window histories, the open
// Future-Missed-Mass events and the per-unit accumulators, all inside one caller-owned buffer.
#pragma once

#include <stdint.h>

namespace qv {

constexpr int DG_MAX_OPEN = 8;     // events inside their horizon at once: horizon / omega
constexpr int DG_MAX_LAG = 8;      // lagged transitions for Delta = 1 .. 8
constexpr int DG_MAX_OMEGA = 256;

// per-unit accumulators (double): sums and counts of the per-event terms
enum : int {
  DA_FMM_SUM = 0, DA_FMM_CNT = 1, DA_CHURN_SUM = 2, DA_CHURN_CNT = 3, DA_QSA_SUM = 4, DA_RQ_SUM = 5, DA_QSA_CNT = 6,
  DA_EVENTS = 7,
  DA_MU = 8,     // [4] tier shares at the last event: Full, Quantized, Evicted, Local
  DA_LIR = 12,   // [4] policy eligible, rescued; FullKV-selection eligible, rescued
  DA_LAG = 16,   // [DG_MAX_LAG][2][2]
  DA_N = 16 + DG_MAX_LAG * 4
};

struct DiagDev {
  uint8_t *base;
  int U, N, Hq, n_open, horizon, lir_m;
  int64_t off_evict, off_since, off_evT;   // int32, initialised to -1
  int64_t off_evId, off_runpol, off_runorc, off_xpol, off_xorc, off_ret, off_fnum, off_fden, off_acc;

  __host__ __device__ int *evict(int u) const { return reinterpret_cast<int *>(base + off_evict) + (size_t)u * N; }
  __host__ __device__ int *since(int u) const { return reinterpret_cast<int *>(base + off_since) + (size_t)u * N; }
  __host__ __device__ int *ev_T(int u) const { return reinterpret_cast<int *>(base + off_evT) + (size_t)u * DG_MAX_OPEN; }
  __host__ __device__ int *ev_id(int u) const { return reinterpret_cast<int *>(base + off_evId) + (size_t)u * DG_MAX_OPEN; }
  __host__ __device__ int *runpol(int u) const { return reinterpret_cast<int *>(base + off_runpol) + (size_t)u * N; }
  __host__ __device__ int *runorc(int u) const { return reinterpret_cast<int *>(base + off_runorc) + (size_t)u * N; }
  __host__ __device__ uint32_t *xpol(int u) const { return reinterpret_cast<uint32_t *>(base + off_xpol) + (size_t)u * N; }
  __host__ __device__ uint32_t *xorc(int u) const { return reinterpret_cast<uint32_t *>(base + off_xorc) + (size_t)u * N; }
  __host__ __device__ uint8_t *ret(int u) const { return base + off_ret + (size_t)u * N; }
  // [U][Hq][DG_MAX_OPEN]: attention on the evicted windows / on every existing state, summed over steps
  __host__ __device__ double *fnum() const { return reinterpret_cast<double *>(base + off_fnum); }
  __host__ __device__ double *fden() const { return reinterpret_cast<double *>(base + off_fden); }
  __host__ __device__ double *acc(int u) const { return reinterpret_cast<double *>(base + off_acc) + (size_t)u * DA_N; }
};

}  // namespace qv
