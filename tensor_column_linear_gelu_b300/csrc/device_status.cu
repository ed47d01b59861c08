// device_status.cu -- the library's device-side error word and the bounded-wait
// self-test.
//
// Kernels with spin-waits take the word's device address as a parameter and
// atomically OR a code into it when a bounded wait gives up (see sync.cuh).
// tp_device_status() synchronises the caller's stream, reads and clears it.
#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "sync.cuh"

namespace tpla {
namespace {

__device__ unsigned int g_device_error;

// Waits on an mbarrier that nothing ever arrives on, with a short limit; the
// wait gives up, the kernel records kErrSelftest and returns.
__global__ void bounded_wait_selftest_kernel(unsigned int* err, uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t b = smem_u32(&bar);
  if (threadIdx.x == 0) {
    mbar_init(b, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    if (!mbar_wait_bounded(b, 0, limit_ns)) report_error(err, kErrSelftest);
  }
  __syncthreads();
}

}  // namespace

// Device address of the error word on the current device.  Cached per
// device; the cache is guarded, so concurrent first calls from several host
// threads are safe.
unsigned int* device_error_word() {
  static unsigned int* cache[64] = {nullptr};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!cache[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return nullptr;
    cache[dev] = static_cast<unsigned int*>(p);
  }
  return cache[dev];
}

tp_status read_and_clear_device_error(cudaStream_t stream) {
  if (cudaStreamSynchronize(stream) != cudaSuccess) return TP_ERR_CUDA;
  unsigned int* w = device_error_word();
  if (!w) return TP_ERR_CUDA;
  unsigned int v = 0;
  if (cudaMemcpyAsync(&v, w, sizeof(v), cudaMemcpyDeviceToHost, stream) != cudaSuccess)
    return TP_ERR_CUDA;
  if (cudaMemsetAsync(w, 0, sizeof(v), stream) != cudaSuccess) return TP_ERR_CUDA;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return TP_ERR_CUDA;
  if (v & kErrIndexCheck) return TP_ERR_DEVICE_CHECK;
  return v ? TP_ERR_DEVICE_TIMEOUT : TP_OK;
}

tp_status launch_bounded_wait_selftest(int64_t limit_ns, cudaStream_t stream) {
  unsigned int* w = device_error_word();
  if (!w) return TP_ERR_CUDA;
  bounded_wait_selftest_kernel<<<1, 32, 0, stream>>>(w, (uint64_t)limit_ns);
  return cudaGetLastError() == cudaSuccess ? TP_OK : TP_ERR_CUDA;
}

}  // namespace tpla
