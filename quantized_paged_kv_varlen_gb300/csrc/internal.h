// Host-side declarations shared between the C-ABI layer (api.cpp) and the
// kernel launchers (*.cu).  Not part of the public interface.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>

#include "../../include/qpkv.h"

namespace qpkv {

// Work item of the split-KV decode: request, kv head, token range [t0, t1),
// and the row of its partial result in the float workspace.
struct DecodeItem {
  int32_t b, hk, t0, t1, slot, pad0, pad1, pad2;
};

// Layout of the decode plan (int workspace) and the float workspace.
struct DecodePlan {
  int64_t num_items;
  int64_t chunk;
  int64_t total_splits;
  int64_t items_offset;      // bytes into the int workspace
  int64_t split_off_offset;  // bytes into the int workspace: int32 [B + 1]
  int64_t int_bytes;
  int64_t float_bytes;
  int64_t batch;
  int64_t num_qo_heads;
  int64_t num_kv_heads;
  int64_t head_dim;
  int64_t page_size;
  int64_t max_len;   // longest request; block_table rows must cover it
  int64_t kind;      // 0: one kv head per work item, 1: all kv heads per work item
  int64_t counter_offset;  // kind 1: bytes into the int workspace of 2 int32 work counters
  int64_t kv_layout;       // QPKV_KV_LAYOUT_NHD (planned) or QPKV_KV_LAYOUT_HND (set later)
  int64_t magic;
};
constexpr int64_t kPlanMagic = 0x71706b76706c616eLL;  // "qpkvplan"

cudaError_t launch_rope_table(float theta, float rope_scale, int max_pos, int rot_dim,
                              float* cos_out, float* sin_out, cudaStream_t stream);

cudaError_t launch_write_cache(const qpkv_write_params& p, cudaStream_t stream);

cudaError_t launch_decode_attend(const DecodePlan& plan, float* float_ws, void* int_ws,
                                 const void* q, const void* k_pool, const void* v_pool,
                                 const float* k_scale_pool, const float* v_scale_pool,
                                 int num_pages, int page_size, const int32_t* block_table,
                                 int bt_stride, float sm_scale, int32_t* error_word,
                                 cudaStream_t stream, int* status);

// All-heads decode (decode_heads.cu): geometry check and launcher.
bool heads_geometry(int Hq, int Hkv, int D, int page_size, int* nt, int* bt, int* nb,
                    int* max_tiles);
cudaError_t launch_decode_heads(const DecodePlan& plan, float* float_ws, void* int_ws,
                                const void* q, const void* k_pool, const void* v_pool,
                                const float* k_scale_pool, const float* v_scale_pool,
                                int num_pages, int page_size, const int32_t* block_table,
                                int bt_stride, float sm_scale, int32_t* error_word,
                                cudaStream_t stream, int* status);

cudaError_t launch_decode_merge(const DecodePlan& plan, const float* float_ws, const void* int_ws,
                                void* o, float* lse, cudaStream_t stream);

// Dense FP8 attention forward (fp8_attn.cu).
cudaError_t launch_fp8_attn(const void* q, const void* k, const void* v, int B, int Sq, int Sk,
                            int Hq, int Hkv, int D, const float* q_descale, const float* k_descale,
                            const float* v_descale, float softmax_scale, int causal, void* o,
                            float* lse, int32_t* error_word, cudaStream_t stream, int* status);

// Varlen INT8-QK paged prefill (prefill_int8.cu).
size_t prefill_workspace_bytes(int num_seqs, int num_tokens, int num_heads_q);
cudaError_t launch_prefill_int8(const qpkv_prefill_params& p, cudaStream_t stream, int* status);

// MLA-absorb sparse decode (mla_sparse.cu).
size_t mla_workspace_bytes(int num_tokens, int sparse_size);
cudaError_t launch_mla_sparse(const qpkv_mla_params& p, cudaStream_t stream, int* status);

// The library-owned device error word of the current device (errors.cu),
// used by the entry points when the caller passes no word; NULL on failure.
int32_t* default_error_word();

// cuTensorMapEncodeTiled through the runtime's driver entry point (no -lcuda).
CUresult encode_tensor_map(CUtensorMap* map, CUtensorMapDataType dtype, uint32_t rank,
                           void* base, const uint64_t* dims, const uint64_t* strides_bytes,
                           const uint32_t* box, CUtensorMapSwizzle swizzle);

}  // namespace qpkv
