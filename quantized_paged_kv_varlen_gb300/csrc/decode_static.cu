// Paged FP8 decode for callers that cannot allocate device memory.
//
// Some callers have no way to call cudaMalloc: a runtime that owns every
// byte of device memory and hands out none, a plugin without an allocator
// handle, or a latency-critical loop that must never enter the allocator.
// qpkv_decode_static serves them.  It runs the same plan, split-KV attend
// and merge as qpkv_decode_plan + qpkv_decode_run, but the two workspaces
// those need live in fixed arrays compiled into this file:
//   g_int_scratch   QPKV_STATIC_INT_BYTES   the work list and split offsets
//   g_float_scratch QPKV_STATIC_FLOAT_BYTES the fp32 partial outputs and lse
// Every GPU that loads the library holds both until the process exits.  In
// host code the array names are host-side stand-ins, not device addresses,
// so the first call on each device looks the device addresses up with
// cudaGetSymbolAddress (that device current) and keeps them.  The work
// list is staged through one shared host buffer by a pageable copy, so a
// call refuses to run (QPKV_ERR_UNSUPPORTED, nothing enqueued) while its
// stream is capturing.  All calls share the arrays and
// each call rewrites everything it later reads (nothing must start at zero);
// calls whose GPU work overlaps race on them.  Batches that need more space
// are rejected on the host with QPKV_ERR_STATIC_LIMIT.  Nothing here
// allocates: no cudaMalloc, no cudaFree, no allocating library routine.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "internal.h"

namespace qpkv {
namespace {

static __device__ __align__(256) uint8_t g_int_scratch[QPKV_STATIC_INT_BYTES];
static __device__ __align__(256) uint8_t g_float_scratch[QPKV_STATIC_FLOAT_BYTES];

// Host staging of the work list: filled by the host planner, then copied
// (pageable cudaMemcpyAsync, which stages the bytes before it returns).
alignas(256) uint8_t g_host_staging[QPKV_STATIC_INT_BYTES];

constexpr int kMaxDevices = 64;
struct DeviceScratch {
  void* int_ptr = nullptr;
  void* float_ptr = nullptr;
};
DeviceScratch g_scratch[kMaxDevices];
std::mutex g_mutex;

// Device addresses of the fixed arrays on the current device (looked up once).
cudaError_t scratch_for_current_device(DeviceScratch* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  DeviceScratch& s = g_scratch[dev];
  if (s.int_ptr == nullptr || s.float_ptr == nullptr) {
    void* ip = nullptr;
    void* fp = nullptr;
    e = cudaGetSymbolAddress(&ip, g_int_scratch);
    if (e != cudaSuccess) return e;
    e = cudaGetSymbolAddress(&fp, g_float_scratch);
    if (e != cudaSuccess) return e;
    s.int_ptr = ip;
    s.float_ptr = fp;
  }
  *out = s;
  return cudaSuccess;
}

}  // namespace
}  // namespace qpkv

extern "C" qpkv_status qpkv_decode_static(const int32_t* seqlens_kv_host, int32_t batch_size,
                                          int32_t num_qo_heads, int32_t num_kv_heads,
                                          int32_t page_size, int32_t head_dim, int32_t num_sms,
                                          const void* q, const void* k_pool, const void* v_pool,
                                          const float* k_scale_pool, const float* v_scale_pool,
                                          int32_t num_pages, const int32_t* block_table,
                                          int32_t bt_stride, float sm_scale, void* o, float* lse,
                                          int32_t* error_word, void* stream) {
  using namespace qpkv;
  // host-only checks first: shapes, then the fixed-size limits
  size_t int_bytes = 0, float_bytes = 0;
  qpkv_status st = qpkv_decode_workspace_sizes(seqlens_kv_host, batch_size, num_qo_heads,
                                               num_kv_heads, head_dim, num_sms, &int_bytes,
                                               &float_bytes);
  if (st != QPKV_OK) return st;
  if (int_bytes > QPKV_STATIC_INT_BYTES || float_bytes > QPKV_STATIC_FLOAT_BYTES)
    return QPKV_ERR_STATIC_LIMIT;
  if (o == nullptr) return QPKV_ERR_INVALID_ARG;
  // The copy below reads g_host_staging when it runs; a recorded copy would
  // read whatever a later call planned there.
  cudaStreamCaptureStatus capturing = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(static_cast<cudaStream_t>(stream), &capturing) != cudaSuccess)
    return QPKV_ERR_CUDA;
  if (capturing != cudaStreamCaptureStatusNone) return QPKV_ERR_UNSUPPORTED;

  int64_t plan_info[QPKV_PLAN_INFO_LEN];
  DeviceScratch scratch;
  {
    std::lock_guard<std::mutex> lock(g_mutex);
    st = qpkv_decode_plan_host(seqlens_kv_host, batch_size, num_qo_heads, num_kv_heads,
                               page_size, head_dim, num_sms, g_host_staging,
                               sizeof(g_host_staging), plan_info);
    if (st != QPKV_OK) return st;
    if (scratch_for_current_device(&scratch) != cudaSuccess) return QPKV_ERR_CUDA;
    if (cudaMemcpyAsync(scratch.int_ptr, g_host_staging, int_bytes, cudaMemcpyHostToDevice,
                        static_cast<cudaStream_t>(stream)) != cudaSuccess)
      return QPKV_ERR_CUDA;
  }
  st = qpkv_decode_attend(plan_info, scratch.float_ptr, QPKV_STATIC_FLOAT_BYTES, scratch.int_ptr,
                          q, k_pool, v_pool, k_scale_pool, v_scale_pool, num_pages, page_size,
                          block_table, bt_stride, sm_scale, error_word, stream);
  if (st != QPKV_OK) return st;
  return qpkv_decode_merge(plan_info, scratch.float_ptr, QPKV_STATIC_FLOAT_BYTES, scratch.int_ptr,
                           o, lse, stream);
}
