// The extern "C" boundary: argument checks, the host decode planner, tensor
// maps, and dispatch to the kernel launchers.  No exception leaves this file;
// no allocation, free or synchronisation happens here.
#include <climits>
#include <cstdint>
#include <algorithm>
#include <cstring>
#include <cuda.h>
#include <cuda_runtime.h>

#include "internal.h"

namespace qpkv {

CUresult encode_tensor_map(CUtensorMap* map, CUtensorMapDataType dtype, uint32_t rank,
                           void* base, const uint64_t* dims, const uint64_t* strides_bytes,
                           const uint32_t* box, CUtensorMapSwizzle swizzle) {
  using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
  static EncodeFn fn = nullptr;
  if (fn == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || p == nullptr)
      return CUDA_ERROR_NOT_FOUND;
    fn = reinterpret_cast<EncodeFn>(p);
  }
  cuuint64_t d[5];
  cuuint64_t s[4];
  cuuint32_t bx[5], es[5];
  for (uint32_t i = 0; i < rank; ++i) {
    d[i] = dims[i];
    bx[i] = box[i];
    es[i] = 1;
    if (i + 1 < rank) s[i] = strides_bytes[i];
  }
  return fn(map, dtype, rank, base, d, s, bx, es, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool supported_decode_shape(int64_t Hq, int64_t Hkv, int64_t D) {
  if (Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0) return false;
  const int64_t G = Hq / Hkv;
  return (D == 64 || D == 128) && (G == 1 || G == 2 || G == 4 || G == 8);
}

// Per-head work items (kind 0): 512 tokens when that still gives every SM a
// few items, else 256 or 128 so that small batches spread over the GPU.
int64_t pick_chunk(const int32_t* lens, int32_t B, int64_t Hkv, int32_t num_sms) {
  const int64_t sms = num_sms > 0 ? num_sms : 148;
  for (int64_t chunk : {512, 256}) {
    int64_t items = 0;
    for (int32_t b = 0; b < B; ++b) items += (static_cast<int64_t>(lens[b]) + chunk - 1) / chunk;
    if (items * Hkv >= 4 * sms) return chunk;
  }
  return 128;
}

// All-heads work items (kind 1): the largest power-of-two number of tiles
// (up to the kernel's register budget) that still gives every SM two items.
int64_t pick_chunk_heads(const int32_t* lens, int32_t B, int nt, int max_tiles, int32_t num_sms) {
  const int64_t sms = num_sms > 0 ? num_sms : 148;
  for (int64_t tiles = max_tiles; tiles > 1; tiles /= 2) {
    const int64_t chunk = tiles * nt;
    int64_t items = 0;
    for (int32_t b = 0; b < B; ++b) items += (static_cast<int64_t>(lens[b]) + chunk - 1) / chunk;
    if (items >= 2 * sms) return chunk;
  }
  return nt;
}

// Whether the all-heads kernel handles this shape for some page size.
bool heads_shape_ok(int64_t Hq, int64_t Hkv, int64_t D) {
  int nt, bt, nb, mt;
  return Hkv > 0 && heads_geometry(static_cast<int>(Hq), static_cast<int>(Hkv), static_cast<int>(D),
                                   static_cast<int>(128 / Hkv), &nt, &bt, &nb, &mt);
}

// Plan layout for the given kind (0: per kv head, 1: all kv heads per item).
void fill_plan_layout(const int32_t* lens, int32_t B, int64_t Hq, int64_t Hkv, int64_t D,
                      int32_t num_sms, int kind, DecodePlan* p) {
  std::memset(p, 0, sizeof(*p));
  p->kind = kind;
  int64_t items_per_split = Hkv;
  int64_t head_bytes = 0;
  if (kind == 1) {
    int nt, bt, nb, mt;
    heads_geometry(static_cast<int>(Hq), static_cast<int>(Hkv), static_cast<int>(D),
                   static_cast<int>(128 / Hkv), &nt, &bt, &nb, &mt);
    p->chunk = pick_chunk_heads(lens, B, nt, mt, num_sms);
    items_per_split = 1;
    p->counter_offset = 0;
    head_bytes = 256;   // two int32 work counters, padded
  } else {
    p->chunk = pick_chunk(lens, B, Hkv, num_sms);
    p->counter_offset = -1;
  }
  int64_t splits = 0;
  for (int32_t b = 0; b < B; ++b) splits += (static_cast<int64_t>(lens[b]) + p->chunk - 1) / p->chunk;
  p->total_splits = splits;
  p->num_items = splits * items_per_split;
  p->items_offset = head_bytes;
  p->split_off_offset = static_cast<int64_t>(
      align_up(static_cast<size_t>(head_bytes + p->num_items * sizeof(DecodeItem)), 256));
  p->int_bytes = static_cast<int64_t>(
      align_up(static_cast<size_t>(p->split_off_offset) + (B + 1) * sizeof(int32_t), 256));
  p->float_bytes = static_cast<int64_t>(align_up(
      static_cast<size_t>(splits) * Hq * (D + 1) * sizeof(float), 256));
  p->batch = B;
  p->num_qo_heads = Hq;
  p->num_kv_heads = Hkv;
  p->head_dim = D;
  for (int32_t b = 0; b < B; ++b) p->max_len = lens[b] > p->max_len ? lens[b] : p->max_len;
  p->kv_layout = QPKV_KV_LAYOUT_NHD;
  p->magic = kPlanMagic;
}

static_assert(sizeof(DecodePlan) <= QPKV_PLAN_INFO_LEN * sizeof(int64_t), "plan_info too small");

bool load_plan(const int64_t* plan_info, DecodePlan* p) {
  if (plan_info == nullptr) return false;
  std::memcpy(p, plan_info, sizeof(*p));
  return p->magic == kPlanMagic && p->num_items >= 0 && p->batch > 0;
}

qpkv_status check_decode_common(const int32_t* lens, int32_t B, int32_t Hq, int32_t Hkv,
                                int32_t D) {
  if (lens == nullptr || B < 1 || Hq < 1 || Hkv < 1) return QPKV_ERR_INVALID_ARG;
  if (Hq % Hkv != 0) return QPKV_ERR_INVALID_ARG;
  for (int32_t b = 0; b < B; ++b)
    if (lens[b] < 0) return QPKV_ERR_INVALID_ARG;
  if (!supported_decode_shape(Hq, Hkv, D)) return QPKV_ERR_UNSUPPORTED;
  return QPKV_OK;
}

bool page_size_ok(int32_t ps) {
  if (ps < 16 || ps % 16 != 0) return false;
  return (256 % ps == 0) || (ps % 256 == 0);
}

qpkv_status check_run_args(const DecodePlan& plan, const void* float_ws, size_t float_ws_bytes,
                           const void* int_ws, const void* q, const void* k_pool,
                           const void* v_pool, const float* ks, const float* vs,
                           int32_t num_pages, int32_t page_size, const int32_t* bt,
                           int32_t bt_stride) {
  if (float_ws == nullptr || int_ws == nullptr || q == nullptr || k_pool == nullptr ||
      v_pool == nullptr || ks == nullptr || vs == nullptr || bt == nullptr)
    return QPKV_ERR_INVALID_ARG;
  if (!aligned16(float_ws) || !aligned16(int_ws) || !aligned16(q) || !aligned16(k_pool) ||
      !aligned16(v_pool))
    return QPKV_ERR_INVALID_ARG;
  if (num_pages < 1 || bt_stride < 1) return QPKV_ERR_INVALID_ARG;
  if (!page_size_ok(page_size)) return QPKV_ERR_UNSUPPORTED;
  if ((plan.max_len + page_size - 1) / page_size > bt_stride) return QPKV_ERR_INVALID_ARG;
  if (static_cast<int64_t>(float_ws_bytes) < plan.float_bytes) return QPKV_ERR_WORKSPACE_TOO_SMALL;
  return QPKV_OK;
}

}  // namespace
}  // namespace qpkv

using namespace qpkv;

extern "C" {

qpkv_status qpkv_decode_plan_set_kv_layout(int64_t* plan_info, int32_t kv_layout) {
  DecodePlan p;
  if (!load_plan(plan_info, &p)) return QPKV_ERR_INVALID_ARG;
  if (kv_layout != QPKV_KV_LAYOUT_NHD && kv_layout != QPKV_KV_LAYOUT_HND)
    return QPKV_ERR_INVALID_ARG;
  p.kv_layout = kv_layout;
  std::memcpy(plan_info, &p, sizeof(p));
  return QPKV_OK;
}

const char* qpkv_status_string(qpkv_status s) {
  switch (s) {
    case QPKV_OK: return "ok";
    case QPKV_ERR_INVALID_ARG: return "invalid argument";
    case QPKV_ERR_UNSUPPORTED: return "unsupported shape, dtype or mode";
    case QPKV_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case QPKV_ERR_CUDA: return "CUDA error";
    case QPKV_ERR_DEVICE: return "device error word set";
    case QPKV_ERR_TIMEOUT: return "device wait timed out";
    case QPKV_ERR_STATIC_LIMIT: return "problem exceeds the fixed scratch of qpkv_decode_static";
    default: return "unknown status";
  }
}

int32_t qpkv_version(void) { return 100; }

size_t qpkv_struct_size(int32_t which) {
  switch (which) {
    case 0: return sizeof(qpkv_write_params);
    case 1: return sizeof(qpkv_prefill_params);
    case 2: return sizeof(qpkv_mla_params);
    default: return 0;
  }
}

qpkv_status qpkv_rope_table(float theta, float rope_scale, int32_t max_pos, int32_t rot_dim,
                            float* cos_out, float* sin_out, void* stream) {
  if (cos_out == nullptr || sin_out == nullptr || max_pos < 1 || rot_dim < 2 || rot_dim % 2 ||
      !(theta > 0.f) || !(rope_scale > 0.f))
    return QPKV_ERR_INVALID_ARG;
  return launch_rope_table(theta, rope_scale, max_pos, rot_dim, cos_out, sin_out,
                           static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? QPKV_OK
             : QPKV_ERR_CUDA;
}

qpkv_status qpkv_write_cache(const qpkv_write_params* p, void* stream) {
  if (p == nullptr) return QPKV_ERR_INVALID_ARG;
  if (p->num_seqs < 1 || p->num_tokens < 0 || p->max_seqlen < 0 || p->num_heads_kv < 1 ||
      p->num_pages < 1 || p->bt_stride < 1 || p->page_size < 1)
    return QPKV_ERR_INVALID_ARG;
  if (p->cu_seqlens_q == nullptr || p->block_table == nullptr || p->k == nullptr ||
      p->k_pool == nullptr)
    return QPKV_ERR_INVALID_ARG;
  if (p->page_size % 16 != 0) return QPKV_ERR_UNSUPPORTED;
  if (!aligned16(p->k) || !aligned16(p->k_pool)) return QPKV_ERR_INVALID_ARG;
  switch (p->mode) {
    case QPKV_WRITE_FP8_TOKEN_HEAD:
      if (p->head_dim != 64 && p->head_dim != 128) return QPKV_ERR_UNSUPPORTED;
      if (p->flags & ~QPKV_WRITE_HND) return QPKV_ERR_UNSUPPORTED;
      if ((p->rope_cos == nullptr) != (p->rope_sin == nullptr)) return QPKV_ERR_INVALID_ARG;
      if (p->rope_cos != nullptr && p->rope_max_pos < 1) return QPKV_ERR_INVALID_ARG;
      if (p->q != nullptr &&
          (p->rope_cos == nullptr || p->q_out == nullptr || p->num_heads_q < 1 ||
           !aligned16(p->q) || !aligned16(p->q_out)))
        return QPKV_ERR_INVALID_ARG;
      if (p->v == nullptr || p->v_pool == nullptr || p->k_scale_pool == nullptr ||
          p->v_scale_pool == nullptr)
        return QPKV_ERR_INVALID_ARG;
      if (!aligned16(p->v) || !aligned16(p->v_pool)) return QPKV_ERR_INVALID_ARG;
      break;
    case QPKV_WRITE_INT8_BLOCK128_ROPE:
      if (p->head_dim != 128) return QPKV_ERR_UNSUPPORTED;
      if (p->num_heads_q < 1 || p->num_heads_q % p->num_heads_kv != 0) return QPKV_ERR_UNSUPPORTED;
      if (p->start_pos != nullptr) return QPKV_ERR_INVALID_ARG;
      if (p->q == nullptr || p->v == nullptr || p->v_pool == nullptr || p->q_out == nullptr ||
          p->k_block_scale == nullptr || p->q_block_scale == nullptr || p->rope_cos == nullptr ||
          p->rope_sin == nullptr)
        return QPKV_ERR_INVALID_ARG;
      if (!aligned16(p->q) || !aligned16(p->v) || !aligned16(p->v_pool) || !aligned16(p->q_out))
        return QPKV_ERR_INVALID_ARG;
      if (p->num_blocks < (p->max_seqlen + 127) / 128 || p->rope_max_pos < p->max_seqlen)
        return QPKV_ERR_INVALID_ARG;
      if (p->flags & ~(QPKV_WRITE_SMOOTH_K | QPKV_WRITE_V_FP8)) return QPKV_ERR_UNSUPPORTED;
      if ((p->flags & QPKV_WRITE_V_FP8) && p->v_channel_scale == nullptr) return QPKV_ERR_INVALID_ARG;
      if (p->flags & (QPKV_WRITE_SMOOTH_K | QPKV_WRITE_V_FP8)) {
        if ((p->flags & QPKV_WRITE_SMOOTH_K) && p->k_mean == nullptr) return QPKV_ERR_INVALID_ARG;
        if (p->workspace == nullptr || !aligned16(p->workspace)) return QPKV_ERR_INVALID_ARG;
        if (p->workspace_bytes <
            qpkv_smooth_workspace_bytes(p->num_seqs, p->num_blocks, p->num_heads_kv))
          return QPKV_ERR_WORKSPACE_TOO_SMALL;
      }
      break;
    case QPKV_WRITE_MLA_ROW:
      if (p->head_dim != 576 || p->num_heads_kv != 1 || p->flags != 0) return QPKV_ERR_UNSUPPORTED;
      if (p->rope_cos != nullptr && (p->rope_sin == nullptr || p->rope_max_pos < 1))
        return QPKV_ERR_INVALID_ARG;
      if (p->q != nullptr &&
          (p->rope_cos == nullptr || p->q_out == nullptr || p->num_heads_q < 1 ||
           !aligned16(p->q) || !aligned16(p->q_out)))
        return QPKV_ERR_INVALID_ARG;
      break;
    default:
      return QPKV_ERR_UNSUPPORTED;
  }
  qpkv_write_params w = *p;
  if (w.error_word == nullptr && (w.error_word = default_error_word()) == nullptr)
    return QPKV_ERR_CUDA;
  return launch_write_cache(w, static_cast<cudaStream_t>(stream)) == cudaSuccess ? QPKV_OK
                                                                                 : QPKV_ERR_CUDA;
}

qpkv_status qpkv_decode_workspace_sizes(const int32_t* lens, int32_t B, int32_t Hq, int32_t Hkv,
                                        int32_t D, int32_t num_sms, size_t* int_ws_bytes,
                                        size_t* float_ws_bytes) {
  const qpkv_status st = check_decode_common(lens, B, Hq, Hkv, D);
  if (st != QPKV_OK) return st;
  // the page size is not known yet: size for every layout the plan may pick
  DecodePlan p;
  fill_plan_layout(lens, B, Hq, Hkv, D, num_sms, 0, &p);
  size_t ib = static_cast<size_t>(p.int_bytes), fb = static_cast<size_t>(p.float_bytes);
  if (heads_shape_ok(Hq, Hkv, D)) {
    fill_plan_layout(lens, B, Hq, Hkv, D, num_sms, 1, &p);
    ib = ib > static_cast<size_t>(p.int_bytes) ? ib : static_cast<size_t>(p.int_bytes);
    fb = fb > static_cast<size_t>(p.float_bytes) ? fb : static_cast<size_t>(p.float_bytes);
  }
  if (int_ws_bytes) *int_ws_bytes = ib;
  if (float_ws_bytes) *float_ws_bytes = fb;
  return QPKV_OK;
}

qpkv_status qpkv_decode_plan_host(const int32_t* lens, int32_t B, int32_t Hq, int32_t Hkv,
                                  int32_t page_size, int32_t D, int32_t num_sms,
                                  void* host_int_ws, size_t host_int_bytes, int64_t* plan_info) {
  const qpkv_status st = check_decode_common(lens, B, Hq, Hkv, D);
  if (st != QPKV_OK) return st;
  if (host_int_ws == nullptr || plan_info == nullptr) return QPKV_ERR_INVALID_ARG;
  if (!page_size_ok(page_size)) return QPKV_ERR_UNSUPPORTED;
  int nt, bt, nb, mt;
  const int kind = heads_geometry(Hq, Hkv, D, page_size, &nt, &bt, &nb, &mt) ? 1 : 0;
  DecodePlan p;
  fill_plan_layout(lens, B, Hq, Hkv, D, num_sms, kind, &p);
  p.page_size = page_size;
  if (host_int_bytes < static_cast<size_t>(p.int_bytes)) return QPKV_ERR_WORKSPACE_TOO_SMALL;
  uint8_t* base = static_cast<uint8_t*>(host_int_ws);
  DecodeItem* items = reinterpret_cast<DecodeItem*>(base + p.items_offset);
  int32_t* split_off = reinterpret_cast<int32_t*>(base + p.split_off_offset);
  int64_t n = 0, s = 0;
  for (int32_t b = 0; b < B; ++b) {
    split_off[b] = static_cast<int32_t>(s);
    for (int64_t t0 = 0; t0 < lens[b]; t0 += p.chunk, ++s) {
      const int32_t t1 = static_cast<int32_t>(t0 + p.chunk < lens[b] ? t0 + p.chunk : lens[b]);
      if (kind == 1) {
        items[n++] = DecodeItem{b, 0, static_cast<int32_t>(t0), t1, static_cast<int32_t>(s), 0, 0, 0};
      } else {
        // items of one token range are adjacent across kv heads, so the CTAs
        // that share the per-token scale sectors run together
        for (int32_t h = 0; h < Hkv; ++h)
          items[n++] = DecodeItem{b, h, static_cast<int32_t>(t0), t1, static_cast<int32_t>(s), 0, 0, 0};
      }
    }
  }
  split_off[B] = static_cast<int32_t>(s);
  if (kind == 1) {
    // taken from a shared counter, largest first: full chunks, then the
    // partial last chunks of the requests from long to short
    std::stable_sort(items, items + n, [](const DecodeItem& x, const DecodeItem& y) {
      return (x.t1 - x.t0) > (y.t1 - y.t0);
    });
    int32_t* counters = reinterpret_cast<int32_t*>(base + p.counter_offset);
    counters[0] = 0;
    counters[1] = 0;
  }
  std::memset(plan_info, 0, QPKV_PLAN_INFO_LEN * sizeof(int64_t));
  std::memcpy(plan_info, &p, sizeof(p));
  return QPKV_OK;
}

qpkv_status qpkv_decode_plan(const int32_t* lens, int32_t B, int32_t Hq, int32_t Hkv,
                             int32_t page_size, int32_t D, int32_t num_sms, void* pinned_int_ws,
                             size_t pinned_bytes, void* int_ws, size_t int_ws_bytes,
                             int64_t* plan_info, void* stream) {
  if (int_ws == nullptr) return QPKV_ERR_INVALID_ARG;
  const qpkv_status st = qpkv_decode_plan_host(lens, B, Hq, Hkv, page_size, D, num_sms,
                                               pinned_int_ws, pinned_bytes, plan_info);
  if (st != QPKV_OK) return st;
  DecodePlan p;
  load_plan(plan_info, &p);
  if (int_ws_bytes < static_cast<size_t>(p.int_bytes)) return QPKV_ERR_WORKSPACE_TOO_SMALL;
  return cudaMemcpyAsync(int_ws, pinned_int_ws, static_cast<size_t>(p.int_bytes),
                         cudaMemcpyHostToDevice, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? QPKV_OK
             : QPKV_ERR_CUDA;
}

qpkv_status qpkv_decode_attend(const int64_t* plan_info, void* float_ws, size_t float_ws_bytes,
                               void* int_ws, const void* q, const void* k_pool,
                               const void* v_pool, const float* k_scale_pool,
                               const float* v_scale_pool, int32_t num_pages, int32_t page_size,
                               const int32_t* block_table, int32_t bt_stride, float sm_scale,
                               int32_t* error_word, void* stream) {
  DecodePlan p;
  if (!load_plan(plan_info, &p)) return QPKV_ERR_INVALID_ARG;
  if (page_size != p.page_size) return QPKV_ERR_INVALID_ARG;
  qpkv_status st = check_run_args(p, float_ws, float_ws_bytes, int_ws, q, k_pool, v_pool,
                                  k_scale_pool, v_scale_pool, num_pages, page_size, block_table,
                                  bt_stride);
  if (st != QPKV_OK) return st;
  if (error_word == nullptr && (error_word = default_error_word()) == nullptr) return QPKV_ERR_CUDA;
  int status = QPKV_OK;
  const cudaError_t e = launch_decode_attend(
      p, static_cast<float*>(float_ws), int_ws, q, k_pool, v_pool, k_scale_pool, v_scale_pool,
      num_pages, page_size, block_table, bt_stride, sm_scale, error_word,
      static_cast<cudaStream_t>(stream), &status);
  if (status != QPKV_OK) return status;
  return e == cudaSuccess ? QPKV_OK : QPKV_ERR_CUDA;
}

qpkv_status qpkv_decode_merge(const int64_t* plan_info, const void* float_ws,
                              size_t float_ws_bytes, const void* int_ws, void* o, float* lse,
                              void* stream) {
  DecodePlan p;
  if (!load_plan(plan_info, &p)) return QPKV_ERR_INVALID_ARG;
  if (float_ws == nullptr || int_ws == nullptr || o == nullptr) return QPKV_ERR_INVALID_ARG;
  if (!aligned16(float_ws) || !aligned16(o)) return QPKV_ERR_INVALID_ARG;
  if (static_cast<int64_t>(float_ws_bytes) < p.float_bytes) return QPKV_ERR_WORKSPACE_TOO_SMALL;
  return launch_decode_merge(p, static_cast<const float*>(float_ws), int_ws, o, lse,
                             static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? QPKV_OK
             : QPKV_ERR_CUDA;
}

qpkv_status qpkv_decode_run(const int64_t* plan_info, void* float_ws, size_t float_ws_bytes,
                            void* int_ws, const void* q, const void* k_pool,
                            const void* v_pool, const float* k_scale_pool,
                            const float* v_scale_pool, int32_t num_pages, int32_t page_size,
                            const int32_t* block_table, int32_t bt_stride, float sm_scale,
                            void* o, float* lse, int32_t* error_word, void* stream) {
  if (o == nullptr) return QPKV_ERR_INVALID_ARG;
  qpkv_status st = qpkv_decode_attend(plan_info, float_ws, float_ws_bytes, int_ws, q, k_pool,
                                      v_pool, k_scale_pool, v_scale_pool, num_pages, page_size,
                                      block_table, bt_stride, sm_scale, error_word, stream);
  if (st != QPKV_OK) return st;
  return qpkv_decode_merge(plan_info, float_ws, float_ws_bytes, int_ws, o, lse, stream);
}

qpkv_status qpkv_fp8_attn_fwd(const void* q, const void* k, const void* v, int32_t batch,
                              int32_t seqlen_q, int32_t seqlen_k, int32_t num_qo_heads,
                              int32_t num_kv_heads, int32_t head_dim, const float* q_descale,
                              const float* k_descale, const float* v_descale,
                              float softmax_scale, int32_t causal, void* o, float* lse,
                              int32_t* error_word, void* stream) {
  if (batch < 0 || seqlen_q < 0 || seqlen_k < 0) return QPKV_ERR_INVALID_ARG;
  if (num_qo_heads <= 0 || num_kv_heads <= 0) return QPKV_ERR_INVALID_ARG;
  if (head_dim != 128 || num_qo_heads % num_kv_heads != 0) return QPKV_ERR_UNSUPPORTED;
  if (batch == 0 || seqlen_q == 0) return QPKV_OK;
  if (o == nullptr || q_descale == nullptr || k_descale == nullptr || v_descale == nullptr)
    return QPKV_ERR_INVALID_ARG;
  if (seqlen_k > 0 && (q == nullptr || k == nullptr || v == nullptr)) return QPKV_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return QPKV_ERR_INVALID_ARG;
  if (error_word == nullptr && (error_word = default_error_word()) == nullptr) return QPKV_ERR_CUDA;
  int status = QPKV_OK;
  const cudaError_t e = launch_fp8_attn(q, k, v, batch, seqlen_q, seqlen_k, num_qo_heads,
                                        num_kv_heads, head_dim, q_descale, k_descale, v_descale,
                                        softmax_scale, causal, o, lse, error_word,
                                        static_cast<cudaStream_t>(stream), &status);
  if (status != QPKV_OK) return static_cast<qpkv_status>(status);
  return e == cudaSuccess ? QPKV_OK : QPKV_ERR_CUDA;
}

size_t qpkv_smooth_workspace_bytes(int32_t num_seqs, int32_t num_blocks, int32_t num_heads_kv) {
  if (num_seqs < 0 || num_blocks < 0 || num_heads_kv < 0) return 0;
  // int64 K sums, then float V channel maxima
  return static_cast<size_t>(num_seqs) * num_blocks * num_heads_kv * 128 *
         (sizeof(long long) + sizeof(float));
}

size_t qpkv_prefill_workspace_bytes(int32_t num_seqs, int32_t num_tokens, int32_t num_heads_q) {
  if (num_seqs < 0 || num_tokens < 0 || num_heads_q < 0) return 0;
  return prefill_workspace_bytes(num_seqs, num_tokens, num_heads_q);
}

qpkv_status qpkv_prefill_paged(const qpkv_prefill_params* p, void* stream) {
  if (p == nullptr) return QPKV_ERR_INVALID_ARG;
  const bool ragged = p->cu_seqlens_kv != nullptr;
  if (p->num_seqs < 0 || p->num_tokens < 0 || p->num_heads_q <= 0 || p->num_heads_kv <= 0 ||
      p->num_blocks <= 0)
    return QPKV_ERR_INVALID_ARG;
  if (ragged ? p->num_kv_tokens < 0
             : (p->num_pages <= 0 || p->bt_stride <= 0 || p->page_size <= 0))
    return QPKV_ERR_INVALID_ARG;
  const int ps = p->page_size;
  if (p->head_dim != 128 || p->num_heads_q % p->num_heads_kv != 0) return QPKV_ERR_UNSUPPORTED;
  if (!ragged && (ps % 16 != 0 || (128 % ps != 0 && ps % 128 != 0) || ps > 16384))
    return QPKV_ERR_UNSUPPORTED;
  if (p->num_heads_q > 32768) return QPKV_ERR_UNSUPPORTED;
  if (p->num_seqs == 0 || p->num_tokens == 0) return QPKV_OK;
  if (p->cu_seqlens_q == nullptr || p->q == nullptr || p->q_block_scale == nullptr ||
      p->k_block_scale == nullptr || p->o == nullptr || p->workspace == nullptr)
    return QPKV_ERR_INVALID_ARG;
  if (!ragged && (p->seqlens_kv == nullptr || p->block_table == nullptr))
    return QPKV_ERR_INVALID_ARG;
  if ((!ragged || p->num_kv_tokens > 0) && (p->k_pool == nullptr || p->v_pool == nullptr))
    return QPKV_ERR_INVALID_ARG;
  if (!aligned16(p->q) || !aligned16(p->k_pool) || !aligned16(p->v_pool) || !aligned16(p->o) ||
      !aligned16(p->workspace))
    return QPKV_ERR_INVALID_ARG;
  if (p->workspace_bytes < prefill_workspace_bytes(p->num_seqs, p->num_tokens, p->num_heads_q))
    return QPKV_ERR_WORKSPACE_TOO_SMALL;
  qpkv_prefill_params w = *p;
  if (w.error_word == nullptr && (w.error_word = default_error_word()) == nullptr)
    return QPKV_ERR_CUDA;
  int status = QPKV_OK;
  const cudaError_t e = launch_prefill_int8(w, static_cast<cudaStream_t>(stream), &status);
  if (status != QPKV_OK) return static_cast<qpkv_status>(status);
  return e == cudaSuccess ? QPKV_OK : QPKV_ERR_CUDA;
}

qpkv_status qpkv_csr_to_block_table(const int32_t* indptr, const int32_t* indices,
                                    const int32_t* last_page_len, int32_t batch,
                                    int32_t page_size, int32_t bt_stride,
                                    int32_t* block_table_out, int32_t* seqlens_out) {
  if (batch < 0 || page_size < 1 || bt_stride < 0) return QPKV_ERR_INVALID_ARG;
  if (indptr == nullptr || (batch > 0 && (last_page_len == nullptr || seqlens_out == nullptr)))
    return QPKV_ERR_INVALID_ARG;
  if (batch > 0 && bt_stride > 0 && block_table_out == nullptr) return QPKV_ERR_INVALID_ARG;
  if (indptr[0] != 0) return QPKV_ERR_INVALID_ARG;
  for (int b = 0; b < batch; ++b) {
    const int64_t n = static_cast<int64_t>(indptr[b + 1]) - indptr[b];
    if (n < 0 || n > bt_stride) return QPKV_ERR_INVALID_ARG;
    if (n > 0 && indices == nullptr) return QPKV_ERR_INVALID_ARG;
    if (n > 0 && (last_page_len[b] < 1 || last_page_len[b] > page_size)) return QPKV_ERR_INVALID_ARG;
    const int64_t len = n > 0 ? (n - 1) * page_size + last_page_len[b] : 0;
    if (len > INT32_MAX) return QPKV_ERR_INVALID_ARG;
  }
  for (int b = 0; b < batch; ++b) {
    const int n = indptr[b + 1] - indptr[b];
    for (int i = 0; i < bt_stride; ++i)
      block_table_out[static_cast<size_t>(b) * bt_stride + i] = i < n ? indices[indptr[b] + i] : -1;
    seqlens_out[b] = n > 0 ? (n - 1) * page_size + last_page_len[b] : 0;
  }
  return QPKV_OK;
}

size_t qpkv_mla_workspace_bytes(int32_t num_tokens, int32_t sparse_size) {
  if (num_tokens < 0 || sparse_size < 0) return 0;
  return mla_workspace_bytes(num_tokens, sparse_size);
}

qpkv_status qpkv_mla_sparse_decode(const qpkv_mla_params* p, void* stream) {
  if (p == nullptr) return QPKV_ERR_INVALID_ARG;
  if (p->num_seqs <= 0 || p->num_tokens < 0 || p->num_heads_q <= 0 || p->block_size <= 0 ||
      p->num_blocks <= 0 || p->bt_stride <= 0 || p->sparse_size <= 0)
    return QPKV_ERR_INVALID_ARG;
  if (p->head_dim_qk != 576 || p->head_dim_v != 512 || p->num_heads_q > 128 ||
      (p->sparse_mode != 0 && p->sparse_mode != 3) || p->sparse_block_size < 0 ||
      p->sparse_block_size > 128)
    return QPKV_ERR_UNSUPPORTED;
  const long long keys =
      static_cast<long long>(p->sparse_size) * (p->sparse_block_size > 1 ? p->sparse_block_size : 1);
  if (keys > (1ll << 24)) return QPKV_ERR_UNSUPPORTED;
  if (p->num_tokens == 0) return QPKV_OK;
  if (p->cu_seqlens_q == nullptr || p->seqlens_kv == nullptr || p->block_table == nullptr ||
      p->q == nullptr || p->kv_pool == nullptr || p->sparse_indices == nullptr || p->o == nullptr ||
      p->workspace == nullptr)
    return QPKV_ERR_INVALID_ARG;
  if (!aligned16(p->q) || !aligned16(p->kv_pool) || !aligned16(p->o) || !aligned16(p->workspace))
    return QPKV_ERR_INVALID_ARG;
  if (p->workspace_bytes < mla_workspace_bytes(p->num_tokens, static_cast<int>(keys)))
    return QPKV_ERR_WORKSPACE_TOO_SMALL;
  qpkv_mla_params w = *p;
  if (w.error_word == nullptr && (w.error_word = default_error_word()) == nullptr)
    return QPKV_ERR_CUDA;
  int status = QPKV_OK;
  const cudaError_t e = launch_mla_sparse(w, static_cast<cudaStream_t>(stream), &status);
  if (status != QPKV_OK) return static_cast<qpkv_status>(status);
  return e == cudaSuccess ? QPKV_OK : QPKV_ERR_CUDA;
}

}  // extern "C"
