// Hand-off diagnostics: what it costs to pass work from one stage of a layer-step to
// the next (the decision pays seven such boundaries per layer-step).
//
//  * fm_test_pdl_chain: a kernel boundary under programmatic dependent launch inside a
//    CUDA graph, as the decision launches its kernels: a graph of `kernels` nearly
//    empty dependent kernels (each signals its dependents at entry, then waits for its
//    predecessor), optionally launched as thread-block clusters and with stores to
//    make visible at completion, timed per kernel.
//  * fm_test_grid_barrier: a grid-wide barrier inside one cooperatively launched
//    kernel (every CTA co-resident by construction): rounds of an arrive counter in
//    global memory, ordered either by release/acquire at gpu scope or by full fences
//    around relaxed atomics. Every wait is bounded; a wait that runs out sets the error
//    word, which also releases every other waiter.
//
// Neither is part of the method; they measure the boundaries the decision's kernel
// sequence is made of.
#include <cuda_runtime.h>

#include <cstdint>

#include "fmad.h"
#include "internal.h"
#include "ptx.cuh"

namespace fm {
namespace {

__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void red_release_gpu_add(unsigned* p, unsigned v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// words[0]: the arrive counter; words[1]: the error word. mode 0: arrive by a release
// reduction, poll by acquire loads; 1: a full fence, a relaxed atomic add, volatile
// polls and a full fence after; 2: as 0, but CTA 0 never arrives (the bounded-wait
// failure path: every CTA gives up after budget_ns). out[2b] = CTA b's time over the
// rounds it completed (ns), out[2b + 1] = that number of rounds.
__global__ void grid_barrier_kernel(unsigned* words, int rounds, int mode, unsigned long long budget_ns,
                                    unsigned long long* out) {
  __shared__ int s_stop;
  unsigned* counter = words;
  int* err = reinterpret_cast<int*>(words + 1);
  if (threadIdx.x == 0) s_stop = 0;
  __syncthreads();
  const uint64_t t0 = global_ns();
  int done = 0;
  for (int r = 1; r <= rounds; ++r) {
    if (threadIdx.x == 0) {
      if (!(mode == 2 && blockIdx.x == 0)) {
        if (mode == 1) {
          __threadfence();
          atomicAdd(counter, 1u);
        } else {
          red_release_gpu_add(counter, 1u);
        }
      }
      const unsigned target = static_cast<unsigned>(r) * gridDim.x;
      const uint64_t ts = global_ns();
      for (;;) {
        const unsigned v = mode == 1 ? *reinterpret_cast<volatile unsigned*>(counter) : ld_acquire_gpu(counter);
        if (v >= target) break;
        if (*reinterpret_cast<volatile int*>(err) != 0 || global_ns() - ts > budget_ns) {
          atomicOr(err, 1);
          s_stop = 1;
          break;
        }
      }
      if (mode == 1) __threadfence();
    }
    __syncthreads();
    if (s_stop) break;
    done = r;
  }
  if (threadIdx.x == 0) {
    out[2 * blockIdx.x] = global_ns() - t0;
    out[2 * blockIdx.x + 1] = static_cast<unsigned long long>(done);
  }
}

// One link of the dependent chain: lets its dependent launch at entry, then waits for
// its predecessor's completion (programmatic dependent launch; plain stream order
// without the launch attribute). CTA 0 counts the link in sink[0]; with writes > 0
// every thread then stores `writes` words (coalesced) into sink[1 + ...], the
// memory a grid's completion has to make visible.
__global__ void chain_kernel(int* sink, int writes) {
  pdl_trigger();
  pdl_wait();
  if (blockIdx.x == 0 && threadIdx.x == 0) sink[0] += 1;
  const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
  const size_t t = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  for (int w = 0; w < writes; ++w) sink[1 + w * stride + t] = w;
}

}  // namespace
}  // namespace fm

extern "C" int fm_test_grid_barrier(int ctas, int threads, int rounds, int mode, unsigned long long budget_ns,
                                    void* scratch, unsigned long long* out, void* stream) {
  if (!scratch || !out) return fm::record_error(FM_ERR_INVALID_ARG, "fm_test_grid_barrier: NULL argument");
  if (ctas < 1 || threads < 32 || threads > 1024 || threads % 32 || rounds < 1 || rounds > 1000000 || mode < 0 ||
      mode > 2 || budget_ns < 1000ull || budget_ns > 10000000000ull)
    return fm::record_error(FM_ERR_SHAPE, "fm_test_grid_barrier: argument out of range");
  if (reinterpret_cast<uintptr_t>(scratch) % 16)
    return fm::record_error(FM_ERR_ALIGN, "fm_test_grid_barrier: scratch not 16-byte aligned");
  int dev = 0, sms = 0, coop = 0, per_sm = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev) != cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fm::grid_barrier_kernel, threads, 0) != cudaSuccess)
    return fm::record_error(FM_ERR_CUDA, "fm_test_grid_barrier: device query failed");
  if (!coop) return fm::record_error(FM_ERR_UNSUPPORTED, "fm_test_grid_barrier: no cooperative launch");
  if (static_cast<long long>(per_sm) * sms < ctas)
    return fm::record_error(FM_ERR_SHAPE, "fm_test_grid_barrier: the CTAs cannot all be resident at once");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  unsigned* words = static_cast<unsigned*>(scratch);
  void* args[] = {&words, &rounds, &mode, &budget_ns, &out};
  int err = 0;
  if (cudaMemsetAsync(words, 0, 2 * sizeof(unsigned), s) != cudaSuccess ||
      cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(fm::grid_barrier_kernel), dim3(ctas), dim3(threads),
                                  args, 0, s) != cudaSuccess ||
      cudaMemcpyAsync(&err, words + 1, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return fm::record_error(FM_ERR_CUDA, "fm_test_grid_barrier: launch or copy failed");
  return err ? fm::record_error(FM_ERR_DEVICE, "fm_test_grid_barrier: a barrier wait ran out") : FM_OK;
}

extern "C" int fm_test_pdl_chain(int ctas, int threads, int kernels, int reps, int pdl, int cluster, int writes,
                                 void* scratch, size_t scratch_bytes, float* us_per_kernel) {
  if (!scratch || !us_per_kernel) return fm::record_error(FM_ERR_INVALID_ARG, "fm_test_pdl_chain: NULL argument");
  if (ctas < 1 || ctas > 65535 || threads < 32 || threads > 1024 || threads % 32 || kernels < 1 || kernels > 4096 ||
      reps < 1 || reps > 1000 || cluster < 1 || cluster > 8 || (cluster & (cluster - 1)) || ctas % cluster ||
      writes < 0 || writes > 64)
    return fm::record_error(FM_ERR_SHAPE, "fm_test_pdl_chain: argument out of range");
  if (scratch_bytes < 4 * (1 + static_cast<size_t>(ctas) * threads * writes))
    return fm::record_error(FM_ERR_WORKSPACE, "fm_test_pdl_chain: scratch smaller than 4 * (1 + ctas * threads * writes)");
  cudaStream_t s = nullptr;
  cudaGraph_t graph = nullptr;
  cudaGraphExec_t exec = nullptr;
  cudaEvent_t e0 = nullptr, e1 = nullptr;
  const char* why = nullptr;
  if (cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking) != cudaSuccess) {
    why = "fm_test_pdl_chain: stream creation failed";
  } else if (cudaMemsetAsync(scratch, 0, sizeof(int), s) != cudaSuccess ||
             cudaStreamBeginCapture(s, cudaStreamCaptureModeThreadLocal) != cudaSuccess) {
    why = "fm_test_pdl_chain: capture start failed";
  } else {
    fm::LaunchOpts lo;
    lo.stream = s;
    lo.pdl = pdl != 0;
    lo.cluster = dim3(static_cast<unsigned>(cluster), 1, 1);
    cudaError_t le = cudaSuccess;
    for (int i = 0; i < kernels && le == cudaSuccess; ++i)
      le = fm::launch(fm::chain_kernel, dim3(ctas), dim3(threads), 0, lo, static_cast<int*>(scratch), writes);
    const cudaError_t ce = cudaStreamEndCapture(s, &graph);
    if (le != cudaSuccess || ce != cudaSuccess) why = "fm_test_pdl_chain: capture failed";
  }
  float ms = 0.f;
  if (!why && (cudaGraphInstantiate(&exec, graph, 0) != cudaSuccess || cudaGraphLaunch(exec, s) != cudaSuccess ||
               cudaStreamSynchronize(s) != cudaSuccess))
    why = "fm_test_pdl_chain: graph instantiation or warm-up failed";
  if (!why && (cudaEventCreate(&e0) != cudaSuccess || cudaEventCreate(&e1) != cudaSuccess)) why = "fm_test_pdl_chain: event creation failed";
  if (!why) {
    cudaError_t e = cudaEventRecord(e0, s);
    for (int r = 0; r < reps && e == cudaSuccess; ++r) e = cudaGraphLaunch(exec, s);
    if (e == cudaSuccess) e = cudaEventRecord(e1, s);
    if (e == cudaSuccess) e = cudaEventSynchronize(e1);
    if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, e0, e1);
    if (e != cudaSuccess) why = "fm_test_pdl_chain: timed launches failed";
  }
  if (e0) cudaEventDestroy(e0);
  if (e1) cudaEventDestroy(e1);
  if (exec) cudaGraphExecDestroy(exec);
  if (graph) cudaGraphDestroy(graph);
  if (s) cudaStreamDestroy(s);
  if (why) return fm::record_error(FM_ERR_CUDA, why);
  *us_per_kernel = ms * 1000.0f / (static_cast<float>(reps) * static_cast<float>(kernels));
  return FM_OK;
}
