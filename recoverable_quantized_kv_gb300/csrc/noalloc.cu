// Prefill window scoring for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc at all: code that runs inside a framework owning every byte
// of device memory through its own pool, plugins handed only their input and output buffers, or
// code paths where an allocation would synchronise the device.  qevict_prefill_scores needs a
// cache (and its arena) only for scratch space; this entry point takes plain sizes and the caller's
// inputs and output, and keeps its scratch in a fixed array that is part of the library image.
//
// The scratch is a file-scope device array of QEVICT_NOALLOC_SCRATCH_FLOATS floats (8 MiB); every
// GPU that loads the library holds it until the process exits.  Host code cannot use the array's
// name as a device address, so the first call on each device looks the address up once, with that
// device current, and later calls reuse it.  Every call shares the array: the two kernels overwrite
// every element they later read, so nothing has to be cleared between calls, but calls that overlap
// on the GPU (for example on two streams) race on the scratch and must be ordered by the caller.
// The scoring kernels' bounded waits report to a status word of this file (not to any cache's);
// qevict_prefill_scores_noalloc_status reads and clears it.
#include <cuda_runtime.h>

#include <mutex>

#include "cache_dev.cuh"
#include "common.cuh"
#include "qevict.h"

namespace qv {
cudaError_t launch_prefill_scores(const CacheDev &C, const __nv_bfloat16 *q, const __nv_bfloat16 *k, float *s0,
                                  cudaStream_t s);
}

namespace {

constexpr long long kScratchFloats = QEVICT_NOALLOC_SCRATCH_FLOATS;
static __device__ __align__(256) float g_noalloc_scratch[kScratchFloats];
static __device__ int g_noalloc_status;   // the scoring kernels' bounded waits record timeouts here

constexpr int kMaxDevices = 64;
std::mutex g_mu;
float *g_scratch_addr[kMaxDevices] = {};   // device address of g_noalloc_scratch, per device
int *g_status_addr[kMaxDevices] = {};      // device address of g_noalloc_status, per device

// The device addresses of the scratch and of the status word on the current device, looked up
// once per device with that device current.
qevict_status device_addresses(float **scratch, int **status) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return QEVICT_ECUDA;
  if (dev < 0 || dev >= kMaxDevices) return QEVICT_EINVAL;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_addr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return QEVICT_ECUDA;
    void *st = nullptr;
    if (cudaGetSymbolAddress(&st, g_noalloc_status) != cudaSuccess || !st) return QEVICT_ECUDA;
    g_scratch_addr[dev] = static_cast<float *>(p);
    g_status_addr[dev] = static_cast<int *>(st);
  }
  *scratch = g_scratch_addr[dev];
  *status = g_status_addr[dev];
  return QEVICT_OK;
}

}  // namespace

extern "C" qevict_status qevict_prefill_scores_noalloc_status(qevict_stream_t stream) {
  float *scratch = nullptr;
  int *status = nullptr;
  const qevict_status st = device_addresses(&scratch, &status);
  if (st != QEVICT_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int word = 0;
  if (cudaMemcpyAsync(&word, status, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaMemsetAsync(status, 0, sizeof(int), s) != cudaSuccess || cudaStreamSynchronize(s) != cudaSuccess)
    return QEVICT_ECUDA;
  return word ? QEVICT_EDEVICE : QEVICT_OK;
}

extern "C" qevict_status qevict_prefill_scores_noalloc(int32_t batch, int32_t prompt_len, int32_t h_q, int32_t h_kv,
                                                       int32_t n_sink, int32_t window, const void *q_prompt,
                                                       const void *k_prompt, float *s0_out, qevict_stream_t stream) {
  if (!q_prompt || !k_prompt || !s0_out || (((uintptr_t)q_prompt | (uintptr_t)k_prompt) & 15) ||
      ((uintptr_t)s0_out & 3) || batch < 1 || h_kv < 1 || h_q < h_kv || h_q % h_kv || window < 1 || n_sink < 0 ||
      prompt_len <= n_sink)
    return QEVICT_EINVAL;
  const int G = h_q / h_kv;
  if (G != 1 && G != 2 && G != 4 && G != 8) return QEVICT_EINVAL;
  const long long per_array = (long long)batch * h_q * prompt_len;   // row statistics, then column sums
  if (2 * per_array > kScratchFloats) return QEVICT_ENOMEM;
  float *scratch = nullptr;
  int *status = nullptr;
  const qevict_status st = device_addresses(&scratch, &status);
  if (st != QEVICT_OK) return st;
  qv::CacheDev C = {};
  C.arena = reinterpret_cast<uint8_t *>(scratch);
  C.off_rowstat = 0;
  C.off_colsum = per_array * (long long)sizeof(float);
  C.status_word = status;   // a word of its own, outside the scratch
  C.B = batch;
  C.h_q = h_q;
  C.h_kv = h_kv;
  C.G = G;
  C.n_sink = n_sink;
  C.W = window;
  C.prompt_len = prompt_len;
  const cudaError_t e = qv::launch_prefill_scores(C, static_cast<const __nv_bfloat16 *>(q_prompt),
                                                  static_cast<const __nv_bfloat16 *>(k_prompt), s0_out,
                                                  reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? QEVICT_OK : QEVICT_ECUDA;
}
