// fm_gemm_consumer_noalloc: the skinny GEMM + fused consumer of fm_gemm_consumer,
// for callers that cannot allocate device memory.
//
// Some callers have no way to get scratch memory on the device: code running
// under an allocator that must not be re-entered, a real-time control loop that
// forbids allocation after start-up, or a host framework that hands this library
// only its own input and output buffers. fm_gemm_consumer needs a scratch buffer
// for its fp32 split-K partial planes; this variant uses a fixed-size array that
// lives in the library's device image instead, so the call allocates nothing
// (no cudaMalloc, no cudaFree, no allocating library routine).
//
// The array is file-scope device memory: every GPU that loads the library holds
// it until the process exits. Its name is only a host-side stand-in, so its
// device address is looked up with cudaGetSymbolAddress on the first call on
// each device (with that device current); that first call should therefore come
// before any stream capture. All calls share the array and it keeps the last
// call's contents; the GEMM overwrites every partial it later reads, so nothing
// in it has to start at zero. Calls that overlap on the GPU (different streams,
// or different threads without ordering) race on the array.

#include <mutex>

#include "internal.h"

namespace {

constexpr size_t kScratchBytes = 8u << 20;   // 8 MiB of fp32 partial planes
constexpr int kMaxDevices = 64;

static __device__ __align__(256) float g_scratch[kScratchBytes / sizeof(float)];
static __device__ int g_err_word;   // bounded-wait error bits of these launches

std::mutex g_mutex;
float* g_scratch_addr[kMaxDevices] = {};
int* g_err_addr[kMaxDevices] = {};

}  // namespace

namespace fm {

// The device address of this file's error word on device `dev`, or nullptr when no
// call has set it up there yet (then no launch of this entry point could have set it).
int* noalloc_error_word(int dev) {
  if (dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_mutex);
  return g_err_addr[dev];
}

}  // namespace fm

extern "C" int fm_gemm_consumer_noalloc(const void* a, int M, int K, const void* w_packed, int N, int fmt, int s,
                                        const float* s_a, const float* s_w, const float* bias, float* x,
                                        const float* gate, const float* scale, const float* shift, float eps,
                                        const float* s_q, void* q, void* stream) {
  size_t need = 0;
  const char* why = "";
  int st = fm::gemm_consumer_scratch_bytes(M, N, K, fmt, s, &need, &why);
  if (st != FM_OK) return fm::record_error(st, why);
  if (need > kScratchBytes)
    return fm::record_error(FM_ERR_WORKSPACE,
                            "fm_gemm_consumer_noalloc: the split-K partials of this shape exceed the 8 MiB built-in "
                            "scratch (s/cluster x M x N x 4 bytes); use fm_gemm_consumer with caller scratch");
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return fm::record_error(FM_ERR_CUDA, "fm_gemm_consumer_noalloc: no usable current device");
  float* scratch = nullptr;
  int* err_word = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_scratch_addr[dev]) {   // once per device, with that device current
      void* sp = nullptr;
      void* ep = nullptr;
      if (cudaGetSymbolAddress(&sp, g_scratch) != cudaSuccess || cudaGetSymbolAddress(&ep, g_err_word) != cudaSuccess)
        return fm::record_error(FM_ERR_CUDA, "fm_gemm_consumer_noalloc: cudaGetSymbolAddress failed");
      g_scratch_addr[dev] = static_cast<float*>(sp);
      g_err_addr[dev] = static_cast<int*>(ep);
    }
    scratch = g_scratch_addr[dev];
    err_word = g_err_addr[dev];
  }
  const fm::GemmConsumerArgs g{a, M, K, N, fmt, s, w_packed, s_a, s_w, bias, x, gate, scale, shift, eps, s_q, q};
  st = fm::gemm_consumer_run(g, scratch, kScratchBytes, err_word, static_cast<cudaStream_t>(stream), &why);
  return st == FM_OK ? FM_OK : fm::record_error(st, why);
}
