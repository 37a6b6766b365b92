// The library's own device error word, its query call, and a self-test of
// the bounded mbarrier wait.
//
// A kernel that skips a bad page id or sparse index, or whose pipeline wait
// runs out, ORs a QPKV_DEV_ERR_* bit into a device error word.  Callers may
// pass their own word; when they pass NULL the entry points substitute this
// library-owned one (one int32 per GPU, in a file-scope __device__ array),
// so the condition is never lost.  qpkv_error_check reads and clears it.
#include <cuda_runtime.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace qpkv {
namespace {

// [0]: the word kernels OR into; [1]: the value taken by the last check.
static __device__ __align__(16) int32_t g_error_word[4];

constexpr int kMaxDevices = 64;
int32_t* g_word_addr[kMaxDevices];
std::mutex g_word_mutex;

__global__ void take_error_word_kernel(int32_t* w) { w[1] = atomicExch(&w[0], 0); }

// One thread waits on an mbarrier whose single expected arrival nobody
// makes, with the given cycle limit; the wait returns false when the limit
// runs out and the kernel reports QPKV_DEV_ERR_TIMEOUT.  Nothing else is in
// flight (no copies, no MMAs, no tensor memory), so returning is all the
// clean-up there is.
__global__ void wait_timeout_kernel(long long limit_cycles, int32_t* err) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0 && !mbar_wait(&bar, 0, limit_cycles)) report_error(err, kDevErrTimeout);
  __syncthreads();
}

}  // namespace

int32_t* default_error_word() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_word_mutex);
  if (g_word_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_error_word) != cudaSuccess) return nullptr;
    g_word_addr[dev] = static_cast<int32_t*>(p);
  }
  return g_word_addr[dev];
}

}  // namespace qpkv

extern "C" {

qpkv_status qpkv_error_status(int32_t bits) {
  if (bits & QPKV_DEV_ERR_TIMEOUT) return QPKV_ERR_TIMEOUT;
  return bits != 0 ? QPKV_ERR_DEVICE : QPKV_OK;
}

qpkv_status qpkv_error_check(void* stream, int32_t* bits_out) {
  using namespace qpkv;
  if (bits_out != nullptr) *bits_out = 0;
  int32_t* w = default_error_word();
  if (w == nullptr) return QPKV_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  take_error_word_kernel<<<1, 1, 0, s>>>(w);
  int32_t bits = 0;
  if (cudaGetLastError() != cudaSuccess ||
      cudaMemcpyAsync(&bits, w + 1, sizeof(bits), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return QPKV_ERR_CUDA;
  if (bits_out != nullptr) *bits_out = bits;
  return qpkv_error_status(bits);
}

qpkv_status qpkv_selftest_wait_timeout(int64_t limit_cycles, int32_t* error_word, void* stream) {
  using namespace qpkv;
  if (limit_cycles < 1000 || limit_cycles > kWaitTimeoutCycles) return QPKV_ERR_INVALID_ARG;
  if (error_word == nullptr) error_word = default_error_word();
  if (error_word == nullptr) return QPKV_ERR_CUDA;
  wait_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(limit_cycles, error_word);
  return cudaGetLastError() == cudaSuccess ? QPKV_OK : QPKV_ERR_CUDA;
}

}  // extern "C"
