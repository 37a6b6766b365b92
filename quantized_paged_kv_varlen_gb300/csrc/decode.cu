// Split-KV paged FP8 decode and its log-sum-exp merge.
//
// What is computed ("KvQuantSparseFlashAttention" README, 计算公式, with the
// per-token-head FP8 quantisation named under 功能说明):
//   O[b, h] = softmax(sm_scale * q[b, h] . Dequant(K_b)^T) . Dequant(V_b),
//   Dequant(x)[t] = e4m3(x[t]) * scale[t],
// over the L_b cached tokens of request b gathered through block_table
// (README 参数说明 row block_table; flashinfer "Batch Decode Attention
// Kernels" plan/run split).  The host plan cuts every (request, kv head)
// into work items of <= 512 tokens; each item yields an fp32 partial output
// and its log-sum-exp, and a merge kernel combines them.
//
// GB300 design: a persistent kernel, one CTA per SM, six warps.
//  * Warp 0 (producer) walks this CTA's items and streams every K and V tile
//    (128 tokens of one kv head) through a ring of shared-memory stages:
//    whole-page TMA boxes [page rows x D bytes] with 128/64-byte swizzle.
//    The page ids of an item are fetched by all 32 lanes at once.  A page
//    that is only partly inside the request is copied row by row with
//    16-byte cp.async, so bytes outside a request never reach shared memory
//    (the ring is zeroed once; every row in it is a real cache row or zero,
//    so 0 * row stays 0 in the MMA).  With each K tile the lanes also gather
//    its 128 k- and v-scales (4-byte cp.async) into a separate scale ring.
//    The ring never drains between items: HBM stays busy.
//  * Warp 1 issues the tcgen05 MMAs, FP8 operands straight from the cache
//    bytes, swap-AB so the 128 tokens fill the MMA's M:
//      S^T[128 tok x N] = K[128 tok x D] . Qt^T        (K-major A and B)
//      O^T[D x N]      += V^T[D x 128 tok] . Pt^T      (MN-major A: V as stored)
//    The bf16 query and the fp32 probabilities are not FP8 values, so each
//    is carried as three E4M3 terms with scales s, s/16, s/256 (~12
//    significant bits, more than bf16's 8); the N columns hold (term, head)
//    pairs, recombined in fp32 after the TMEM load.  No K/V element is ever
//    converted.  Tile order K(0) | K(1) V(0) | K(2) V(1) | ... lets the QK of
//    item k+1 run while item k's softmax is computed.
//  * Warps 2-5 (128 threads) split the queries into terms, run the softmax
//    (exact over an item: all its logits sit in TMEM), fold the k-scales
//    into the logits and the v-scales into the probabilities, and write the
//    partials; the epilogue of item k-1 runs after the softmax of item k.
//    TMEM accumulators and operand buffers are triple-buffered across items.
#include <cmath>

#include "common.cuh"
#include "internal.h"

namespace qpkv {
namespace {

constexpr int kTile = 128;     // tokens per MMA tile
constexpr int kMaxTiles = 4;   // tiles per work item
constexpr int kTerms = 3;
constexpr int kBufs = 3;       // items in flight in TMEM
constexpr int kOpBufs = 2;     // query / probability operand buffers
constexpr int kThreads = 192;  // producer, MMA, 4 softmax warps
constexpr int kSoftmaxThreads = 128;
constexpr int kBarSoftmax = 1;  // named barrier id of the softmax warps
constexpr int kMaxStages = 16;
constexpr int kScaleSlots = 16;  // K tiles whose scales may be in flight
constexpr int kDescRing = 8;     // item descriptors published by the producer
constexpr int kQRing = 4;        // item query rows copied by the producer

template <int D, int G>
struct Cfg {
  static constexpr int kN = ((kTerms * G + 15) / 16) * 16;
  static constexpr int kTileBytes = kTile * D;
  static constexpr uint32_t kSwz = D == 128 ? kSwizzle128B : kSwizzle64B;
  static constexpr int kSBO = 8 * D;
  static constexpr int kQBytes = ((kN * D + 1023) / 1024) * 1024;
  static constexpr int kPTileBytes = kN * kTile;
  static constexpr int kPBytes = kMaxTiles * kPTileBytes;
  static constexpr int kSlotBytes = 2 * kTile * 4;  // k-scales then v-scales
  static constexpr int kQRowBytes = G * D * 2;      // bf16 query rows of one item
  static constexpr int kFixed = kOpBufs * (kQBytes + kPBytes) + kScaleSlots * kSlotBytes +
                                kQRing * kQRowBytes + kDescRing * 32;
  static constexpr int kBudget = 224 * 1024;
  static constexpr int kStagesRaw = (kBudget - kFixed) / kTileBytes;
  static constexpr int kStages = kStagesRaw > kMaxStages ? kMaxStages : kStagesRaw;
  static constexpr int kOffQ = kStages * kTileBytes;
  static constexpr int kOffP = kOffQ + kOpBufs * kQBytes;
  static constexpr int kOffScale = kOffP + kOpBufs * kPBytes;
  static constexpr int kOffQRing = kOffScale + kScaleSlots * kSlotBytes;
  static constexpr int kOffDesc = kOffQRing + kQRing * kQRowBytes;
  static constexpr int kBytes = kOffDesc + kDescRing * 32;
  static constexpr int kSmem = kBytes + 1024;
  static constexpr int kBufCols = kMaxTiles * kN + kN;  // S tiles + O
  static constexpr int kTmemCols =
      kBufs * kBufCols <= 128 ? 128 : (kBufs * kBufCols <= 256 ? 256 : 512);
  static constexpr int kEPT =
      (G * D) / kSoftmaxThreads > 0 ? (G * D) / kSoftmaxThreads : 1;
  static constexpr int kActive = G * D / kEPT;  // softmax threads taking part in the q split
  static constexpr int kTPH = D / kEPT;          // threads per head in the q split
  // the ring must hold K(k+1) and V(k) at once, plus one stage to stream into
  static_assert(kStages >= 2 * kMaxTiles + 1, "ring too small for two items in flight");
  static_assert(kBufs * kBufCols <= 512, "TMEM");
  static_assert(kEPT <= 8, "q split: at most 8 elements per thread");
  static_assert(kQRowBytes % 16 == 0 && kQRowBytes / 16 <= 4 * 32, "q copy: <= 4 chunks a lane");
  static_assert(kSmem <= 227 * 1024, "shared memory");
};

struct DecodeArgs {
  const DecodeItem* items;
  int num_items;
  int Hq, Hkv;
  const uint16_t* q;
  const uint8_t* k_pool;
  const uint8_t* v_pool;
  const float* k_scale;
  const float* v_scale;
  const int32_t* block_table;
  int bt_stride;
  int page_size;
  int num_pages;
  float sm_scale_log2;  // sm_scale * log2(e)
  float* part_o;        // [total_splits, Hq, D]
  float* part_lse;      // [total_splits, Hq]
  int* err;
};

struct SharedState {
  uint64_t full[kMaxStages], empty[kMaxStages];
  uint64_t slot_free[kScaleSlots];
  uint64_t q_free[kQRing];
  uint64_t q_ready[kBufs], s_full[kBufs], p_ready[kBufs], o_full[kBufs], buf_free[kBufs];
  uint32_t tmem_base;
  int abort;
};

// Bounded wait that also gives up as soon as another role aborted.
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, SharedState& sh,
                                              int* err) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 64; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (*reinterpret_cast<volatile int*>(&sh.abort)) return false;
    if (clock64() - t0 > kWaitTimeoutCycles) {
      sh.abort = 1;
      report_error(err, kDevErrTimeout);
      return false;
    }
  }
}

__device__ __forceinline__ int item_tiles(const DecodeItem& it) {
  return (it.t1 - it.t0 + kTile - 1) / kTile;
}

// max over the kTPH softmax threads of one head group (power of two)
template <int TPH>
__device__ __forceinline__ float head_group_max(float v, float* red, int sw) {
  if constexpr (TPH <= 32) {
#pragma unroll
    for (int o = 1; o < TPH; o <<= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
  } else {
    v = warp_max(v);
    if ((threadIdx.x & 31) == 0) red[sw] = v;
    named_barrier(kBarSoftmax, kSoftmaxThreads);
    const int first = (sw / (TPH / 32)) * (TPH / 32);
    float m = red[first];
#pragma unroll
    for (int i = 1; i < TPH / 32; ++i) m = fmaxf(m, red[first + i]);
    named_barrier(kBarSoftmax, kSoftmaxThreads);
    return m;
  }
}

// Three-term E4M3 split of x with term scales s1, s1/16, s1/256.
__device__ __forceinline__ void split3(float x, float s1, float inv1, uint8_t& c1, uint8_t& c2,
                                      uint8_t& c3) {
  c1 = f32_to_e4m3(x * inv1);
  const float r1 = fmaf(-e4m3_to_f32(c1), s1, x);
  c2 = f32_to_e4m3(r1 * inv1 * 16.0f);
  const float r2 = fmaf(-e4m3_to_f32(c2), s1 * (1.0f / 16.0f), r1);
  c3 = f32_to_e4m3(r2 * inv1 * 256.0f);
}

// HND: K/V pools [P, Hkv, ps, D] (compile-time, so the NHD kernel carries
// no code for the other layout)
template <int D, int G, bool HND>
__global__ void __launch_bounds__(kThreads, 1)
    decode_attend_kernel(const __grid_constant__ CUtensorMap k_map,
                         const __grid_constant__ CUtensorMap v_map, const DecodeArgs a) {
  using C = Cfg<D, G>;
  constexpr int NS = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint8_t* sQ = smem + C::kOffQ;
  uint8_t* sP = smem + C::kOffP;
  float* sScale = reinterpret_cast<float*>(smem + C::kOffScale);
  uint8_t* sQRing = smem + C::kOffQRing;
  DecodeItem* sDesc = reinterpret_cast<DecodeItem*>(smem + C::kOffDesc);
  __shared__ SharedState sh;
  __shared__ float red_a[4][G], red_b[4][G], red_c[4][G];
  __shared__ float red_q[4];
  __shared__ float sig_q[kOpBufs][G];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int ps = a.page_size;
  const int R = ps < kTile ? ps : kTile;  // rows per TMA box
  const int bpt = kTile / R;              // boxes per tile

  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&sh.full[s], 1 + 32);  // producer's expect_tx + 32 lanes' cp.async
      mbar_init(&sh.empty[s], 1);      // MMA commit
    }
    for (int s = 0; s < kScaleSlots; ++s) mbar_init(&sh.slot_free[s], kSoftmaxThreads);
    for (int s = 0; s < kQRing; ++s) mbar_init(&sh.q_free[s], kSoftmaxThreads);
    for (int b = 0; b < kBufs; ++b) {
      mbar_init(&sh.q_ready[b], kSoftmaxThreads);
      mbar_init(&sh.s_full[b], 1);
      mbar_init(&sh.p_ready[b], kSoftmaxThreads);
      mbar_init(&sh.o_full[b], 1);
      mbar_init(&sh.buf_free[b], kSoftmaxThreads);
    }
    sh.abort = 0;
    fence_mbar_init();
  }
  // rows never loaded must hold finite bytes: zero the ring once
  for (int i = tid; i < NS * C::kTileBytes / 16; i += kThreads)
    reinterpret_cast<uint4*>(smem)[i] = make_uint4(0, 0, 0, 0);
  fence_proxy_async_smem();
  if (warp == 1) tmem_alloc(&sh.tmem_base, C::kTmemCols);
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = sh.tmem_base;
  const int n_my = a.num_items > static_cast<int>(blockIdx.x)
                       ? (a.num_items - 1 - static_cast<int>(blockIdx.x)) / gridDim.x + 1
                       : 0;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    tma_prefetch_desc(&k_map);
    tma_prefetch_desc(&v_map);
    auto load_desc = [&](int k) {
      DecodeItem it{};
      if (k < n_my) it = a.items[blockIdx.x + static_cast<size_t>(k) * gridDim.x];
      return it;
    };
    // box `lane` of an item: x = token row page * ps + offset (indexes the
    // scale pools), y = the K/V row of the tensor maps (x for NHD, page *
    // Hkv * ps + offset for HND); -1: none / skipped page
    auto box_rows = [&](int k, const DecodeItem& it) {
      int2 row = make_int2(-1, -1);
      if (k < n_my && lane < item_tiles(it) * bpt) {
        const int tok = it.t0 + (lane / bpt) * kTile + (lane % bpt) * R;
        if (tok < it.t1) {
          const int page =
              __ldg(a.block_table + static_cast<size_t>(it.b) * a.bt_stride + tok / ps);
          if (page >= 0 && page < a.num_pages) {
            row.x = page * ps + (tok % ps);
            row.y = HND ? page * a.Hkv * ps + (tok % ps) : row.x;
          } else {
            report_error(a.err, kDevErrBadPage);
          }
        }
      }
      return row;
    };
    int pos = 0;   // ring position (K and V tiles)
    int kq = 0;    // K tiles emitted (scale-ring position)
    auto emit = [&](int k, const DecodeItem& it, int2 rows, int j, bool is_v) -> bool {
      const int s = pos % NS;
      bool ok = true;
      if (lane == 0) ok = wait_or_abort(&sh.empty[s], ((pos / NS) & 1) ^ 1, sh, a.err);
      float* slot = sScale + (kq % kScaleSlots) * (2 * kTile);
      if (!is_v && lane == 0 && ok)
        ok = wait_or_abort(&sh.slot_free[kq % kScaleSlots], ((kq / kScaleSlots) & 1) ^ 1, sh,
                           a.err);
      // the query/descriptor entry of item k - kQRing must have been consumed
      if (!is_v && j == 0 && lane == 0 && ok)
        ok = wait_or_abort(&sh.q_free[k % kQRing], ((k / kQRing) & 1) ^ 1, sh, a.err);
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      if (!ok) return false;
      uint8_t* stage = smem + s * C::kTileBytes;
      const int tok0 = it.t0 + j * kTile;
      const int nvalid = min(kTile, it.t1 - tok0);
      const int nfull = nvalid / R;               // boxes entirely inside the item
      const int tail = nvalid - nfull * R;        // rows of the partly valid box
      const int my_row = __shfl_sync(0xffffffffu, rows.y, j * bpt + (lane < bpt ? lane : 0));
      const unsigned issue = __ballot_sync(0xffffffffu, lane < nfull && my_row >= 0);
      if (!is_v && j == 0) {
        // first tile of the item: publish its descriptor and query rows
        // under the same barrier as the tile
        if (lane == 0) sDesc[k % kDescRing] = it;
        const uint8_t* qsrc = reinterpret_cast<const uint8_t*>(
            a.q + (static_cast<size_t>(it.b) * a.Hq + static_cast<size_t>(it.hk) * G) * D);
        uint8_t* qdst = sQRing + (k % kQRing) * C::kQRowBytes;
        for (int c = lane; c < C::kQRowBytes / 16; c += 32) cp_async_16(qdst + 16 * c, qsrc + 16 * c);
      }
      if (lane == 0) mbar_arrive_expect_tx(&sh.full[s], __popc(issue) * R * D);
      __syncwarp();
      if (lane < nfull && my_row >= 0)
        tma_load_3d(stage + lane * R * D, is_v ? &v_map : &k_map, &sh.full[s], 0, it.hk, my_row);
      if (tail > 0) {
        const int row0 = __shfl_sync(0xffffffffu, rows.y, j * bpt + nfull);
        if (row0 >= 0) {
          const uint8_t* pool = is_v ? a.v_pool : a.k_pool;
          for (int i = lane; i < tail * (D / 16); i += 32) {
            const int r = i / (D / 16), c = i % (D / 16);
            const size_t kv_row = HND ? static_cast<size_t>(row0 + r) + static_cast<size_t>(it.hk) * ps
                                      : static_cast<size_t>(row0 + r) * a.Hkv + it.hk;
            cp_async_16(stage + swizzled_offset(nfull * R + r, 16 * c, D),
                        pool + kv_row * D + 16 * c);
          }
        }
      }
      if (!is_v) {
#pragma unroll
        for (int m = 0; m < kTile / 32; ++m) {
          const int t = lane + 32 * m;
          const int row0 = __shfl_sync(0xffffffffu, rows.x, j * bpt + t / R);
          if (t < nvalid && row0 >= 0) {
            const size_t e = static_cast<size_t>(row0 + t % R) * a.Hkv + it.hk;
            cp_async_4(slot + t, a.k_scale + e);
            cp_async_4(slot + kTile + t, a.v_scale + e);
          }
        }
        ++kq;
      }
      cp_async_arrive_noinc(&sh.full[s]);
      ++pos;
      return true;
    };
    // descriptors run two items ahead, page rows one item ahead
    DecodeItem d0 = load_desc(0), d1 = load_desc(1), d2 = load_desc(2);
    int2 r0 = box_rows(0, d0), r1 = box_rows(1, d1);
    bool ok = n_my > 0;
    for (int j = 0; ok && j < item_tiles(d0); ++j) ok = emit(0, d0, r0, j, false);
    for (int k = 0; ok && k < n_my; ++k) {
      const DecodeItem d3 = load_desc(k + 3);
      const int2 r2 = box_rows(k + 2, d2);
      if (k + 1 < n_my)
        for (int j = 0; ok && j < item_tiles(d1); ++j) ok = emit(k + 1, d1, r1, j, false);
      for (int j = 0; ok && j < item_tiles(d0); ++j) ok = emit(k, d0, r0, j, true);
      d0 = d1;
      d1 = d2;
      d2 = d3;
      r0 = r1;
      r1 = r2;
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA
    if (lane == 0 && n_my > 0) {
      constexpr uint32_t idesc_qk = make_idesc(kFmtE4M3, kFmtE4M3, 0, 0, 128, C::kN);
      constexpr uint32_t idesc_pv = make_idesc(kFmtE4M3, kFmtE4M3, 1, 0, 128, C::kN);
      int pos = 0;
      int nt_of[kBufs];
      auto qk = [&](int k) -> bool {
        const int b = k % kBufs;
        if (!wait_or_abort(&sh.q_ready[b], (k / kBufs) & 1, sh, a.err)) return false;
        if (k >= kBufs &&
            !wait_or_abort(&sh.buf_free[b], ((k - kBufs) / kBufs) & 1, sh, a.err))
          return false;
        // q_ready(k) implies the item's first K tile (and its descriptor) landed
        const int nt = item_tiles(sDesc[k % kDescRing]);
        nt_of[b] = nt;
        tc_fence_after_sync();
        const uint32_t s_base = tmem + b * C::kBufCols;
        const uint32_t qop = smem_u32(sQ + (k % kOpBufs) * C::kQBytes);
        for (int j = 0; j < nt; ++j) {
          const int s = pos % NS;
          if (!wait_or_abort(&sh.full[s], (pos / NS) & 1, sh, a.err)) return false;
          tc_fence_after_sync();
          const uint32_t tile = smem_u32(smem + s * C::kTileBytes);
#pragma unroll
          for (int kk = 0; kk < D / 32; ++kk) {
            const uint64_t da = make_smem_desc(tile + 32 * kk, 16, C::kSBO, C::kSwz);
            const uint64_t db = make_smem_desc(qop + 32 * kk, 16, C::kSBO, C::kSwz);
            tc_mma_f8(s_base + j * C::kN, da, db, idesc_qk, kk > 0);
          }
          tc_commit(&sh.empty[s]);
          ++pos;
        }
        tc_commit(&sh.s_full[b]);
        return true;
      };
      auto pv = [&](int k) -> bool {
        const int b = k % kBufs;
        if (!wait_or_abort(&sh.p_ready[b], (k / kBufs) & 1, sh, a.err)) return false;
        tc_fence_after_sync();
        const uint32_t o_col = tmem + b * C::kBufCols + kMaxTiles * C::kN;
        const uint8_t* pbuf = sP + (k % kOpBufs) * C::kPBytes;
        for (int j = 0; j < nt_of[b]; ++j) {
          const int s = pos % NS;
          if (!wait_or_abort(&sh.full[s], (pos / NS) & 1, sh, a.err)) return false;
          tc_fence_after_sync();
          const uint32_t tile = smem_u32(smem + s * C::kTileBytes);
          const uint32_t ptile = smem_u32(pbuf + j * C::kPTileBytes);
#pragma unroll
          for (int kk = 0; kk < kTile / 32; ++kk) {
            // MN-major A: one D-byte atom per 8 token rows; for D = 64 the
            // upper half of M re-reads the same atom (LBO 0) and is ignored
            const uint64_t da =
                make_smem_desc(tile + kk * 32 * D, D == 128 ? 16 * 1024 : 0, C::kSBO, C::kSwz);
            const uint64_t db = make_smem_desc(ptile + 32 * kk, 16, 1024, kSwizzle128B);
            tc_mma_f8(o_col, da, db, idesc_pv, (j > 0 || kk > 0) ? 1u : 0u);
          }
          tc_commit(&sh.empty[s]);
          ++pos;
        }
        tc_commit(&sh.o_full[b]);
        return true;
      };
      bool ok = qk(0);
      for (int k = 0; k < n_my && ok; ++k) {
        if (k + 1 < n_my) ok = qk(k + 1);
        if (ok) ok = pv(k);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------- softmax / epilogue
    const int sw = warp & 3;             // TMEM lane quarter of this warp
    const int tl = sw * 32 + lane;       // token row of S^T, d row of O^T
    const uint32_t lane_base = static_cast<uint32_t>(sw * 32) << 16;
    const int qg = tl / C::kTPH;
    const int qd0 = (tl % C::kTPH) * C::kEPT;
    const bool qactive = tl < C::kActive;
    // Wait for item k's first K tile (its descriptor and query rows come
    // with it), then split the query into E4M3 terms for the QK MMA.  The
    // stage cannot be recycled before this wait: its QK needs q_ready(k).
    auto fetch_and_split = [&](int k, int kpos) -> DecodeItem {
      wait_or_abort(&sh.full[kpos % NS], (kpos / NS) & 1, sh, a.err);
      const DecodeItem it = sDesc[k % kDescRing];
      const uint16_t* qrow =
          reinterpret_cast<const uint16_t*>(sQRing + (k % kQRing) * C::kQRowBytes);
      float x[C::kEPT];
      float amax = 0.f;
      if (qactive) {
#pragma unroll
        for (int e = 0; e < C::kEPT; ++e) {
          x[e] = bf16_bits_to_float(qrow[qg * D + qd0 + e]);
          amax = fmaxf(amax, fabsf(x[e]));
        }
      }
      mbar_arrive(&sh.q_free[k % kQRing]);
      amax = head_group_max<C::kTPH>(amax, red_q, sw);
      const float s1 = amax * (1.0f / 448.0f);
      const float inv1 = s1 > 0.f ? 1.0f / s1 : 0.f;
      uint8_t* dst = sQ + (k % kOpBufs) * C::kQBytes;
      if (qactive) {
        if ((tl % C::kTPH) == 0) sig_q[k % kOpBufs][qg] = s1;
#pragma unroll
        for (int e = 0; e < C::kEPT; ++e) {
          uint8_t c1, c2, c3;
          split3(x[e], s1, inv1, c1, c2, c3);
          dst[swizzled_offset(0 * G + qg, qd0 + e, D)] = c1;
          dst[swizzled_offset(1 * G + qg, qd0 + e, D)] = c2;
          dst[swizzled_offset(2 * G + qg, qd0 + e, D)] = c3;
        }
      }
      for (int i = tl; i < (C::kN - kTerms * G) * D; i += kSoftmaxThreads)
        dst[swizzled_offset(kTerms * G + i / D, i % D, D)] = 0;
      fence_proxy_async_smem();
      mbar_arrive(&sh.q_ready[k % kBufs]);
      return it;
    };
    // epilogue of item k: recombine the O terms, normalise, write the partial
    auto epilogue = [&](int k, const DecodeItem& it, const float (&mrow)[G],
                        const float (&lsum)[G], const float (&pmax)[G]) {
      const int b = k % kBufs;
      wait_or_abort(&sh.o_full[b], (k / kBufs) & 1, sh, a.err);
      __syncwarp();   // converged before the .sync.aligned TMEM loads
      tc_fence_after_sync();
      uint32_t r[C::kN];
#pragma unroll
      for (int c = 0; c < C::kN; c += 16) {
        uint32_t part[16];
        tmem_ld16(tmem + lane_base + b * C::kBufCols + kMaxTiles * C::kN + c, part);
#pragma unroll
        for (int i = 0; i < 16; ++i) r[c + i] = part[i];
      }
      tmem_ld_wait();
      tc_fence_before_sync();
      mbar_arrive(&sh.buf_free[b]);
      if (tl < D) {
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float sdot = __uint_as_float(r[g]) + __uint_as_float(r[G + g]) * (1.0f / 16.0f) +
                             __uint_as_float(r[2 * G + g]) * (1.0f / 256.0f);
          const float o = lsum[g] > 0.f ? sdot * (pmax[g] * (1.0f / 448.0f)) / lsum[g] : 0.f;
          a.part_o[(static_cast<size_t>(it.slot) * a.Hq + it.hk * G + g) * D + tl] = o;
        }
      }
      if (tl < G) {
        const float lse = lsum[tl] > 0.f ? (mrow[tl] + log2f(lsum[tl])) * kLn2 : -INFINITY;
        a.part_lse[static_cast<size_t>(it.slot) * a.Hq + it.hk * G + tl] = lse;
      }
    };

    // ring positions mirror the producer: K(0) | K(1) V(0) | K(2) V(1) | ...
    DecodeItem cur{}, prev{};
    int kpos_cur = 0, pos = 0;
    if (n_my > 0) {
      cur = fetch_and_split(0, 0);
      pos = item_tiles(cur);
    }
    float pm_prev[G], pl_prev[G], pp_prev[G];
    int kq = 0;   // K tiles consumed (scale-ring position)
    // No early exit in this loop: all 128 threads must meet every named
    // barrier.  After an abort every wait returns at once and the loop runs
    // out quickly with the error already reported.
    for (int k = 0; k < n_my; ++k) {
      const int nt = item_tiles(cur);
      const int b = k % kBufs;
      DecodeItem nxt{};
      int kpos_next = pos;
      if (k + 1 < n_my) {
        nxt = fetch_and_split(k + 1, kpos_next);
        pos += item_tiles(nxt);
      }
      pos += nt;   // V(k)

      // ---- logits with the k-scales folded in
      wait_or_abort(&sh.s_full[b], (k / kBufs) & 1, sh, a.err);
      __syncwarp();   // converged before the .sync.aligned TMEM loads
      tc_fence_after_sync();
      float l2[kMaxTiles][G];
      float vsc[kMaxTiles];
      bool valid[kMaxTiles];
#pragma unroll
      for (int j = 0; j < kMaxTiles; ++j) {
        valid[j] = false;
        vsc[j] = 0.f;
#pragma unroll
        for (int g = 0; g < G; ++g) l2[j][g] = -INFINITY;
        if (j < nt) {
          uint32_t r[C::kN];
#pragma unroll
          for (int c = 0; c < C::kN; c += 16) {
            uint32_t part[16];
            tmem_ld16(tmem + lane_base + b * C::kBufCols + j * C::kN + c, part);
#pragma unroll
            for (int i = 0; i < 16; ++i) r[c + i] = part[i];
          }
          tmem_ld_wait();
          const int q = kq + j;
          const float* slot = sScale + (q % kScaleSlots) * (2 * kTile);
          valid[j] = cur.t0 + j * kTile + tl < cur.t1;
          const float ks = valid[j] ? slot[tl] : 0.f;
          vsc[j] = valid[j] ? slot[kTile + tl] : 0.f;
          mbar_arrive(&sh.slot_free[q % kScaleSlots]);
          const float f = a.sm_scale_log2 * ks;
#pragma unroll
          for (int g = 0; g < G; ++g) {
            const float sdot = __uint_as_float(r[g]) +
                               __uint_as_float(r[G + g]) * (1.0f / 16.0f) +
                               __uint_as_float(r[2 * G + g]) * (1.0f / 256.0f);
            if (valid[j]) l2[j][g] = f * sig_q[k % kOpBufs][g] * sdot;
          }
        }
      }
      kq += nt;
      float mrow[G], lsum[G], pmax[G];
#pragma unroll
      for (int g = 0; g < G; ++g) {
        float m = l2[0][g];
#pragma unroll
        for (int j = 1; j < kMaxTiles; ++j) m = fmaxf(m, l2[j][g]);
        m = warp_max(m);
        if (lane == 0) red_a[sw][g] = m;
      }
      named_barrier(kBarSoftmax, kSoftmaxThreads);
#pragma unroll
      for (int g = 0; g < G; ++g)
        mrow[g] = fmaxf(fmaxf(red_a[0][g], red_a[1][g]), fmaxf(red_a[2][g], red_a[3][g]));

      // ---- probabilities times v-scales, as three E4M3 terms
      float p[kMaxTiles][G];
#pragma unroll
      for (int g = 0; g < G; ++g) {
        float s = 0.f, pm = 0.f;
#pragma unroll
        for (int j = 0; j < kMaxTiles; ++j) {
          const float e = valid[j] ? exp2f(l2[j][g] - mrow[g]) : 0.f;
          s += e;
          p[j][g] = e * vsc[j];
          pm = fmaxf(pm, p[j][g]);
        }
        s = warp_sum(s);
        pm = warp_max(pm);
        if (lane == 0) {
          red_b[sw][g] = s;
          red_c[sw][g] = pm;
        }
      }
      named_barrier(kBarSoftmax, kSoftmaxThreads);
#pragma unroll
      for (int g = 0; g < G; ++g) {
        lsum[g] = red_b[0][g] + red_b[1][g] + red_b[2][g] + red_b[3][g];
        pmax[g] = fmaxf(fmaxf(red_c[0][g], red_c[1][g]), fmaxf(red_c[2][g], red_c[3][g]));
      }
      uint8_t* pbuf = sP + (k % kOpBufs) * C::kPBytes;
#pragma unroll
      for (int j = 0; j < kMaxTiles; ++j) {
        if (j < nt) {
          uint8_t* dst = pbuf + j * C::kPTileBytes;
#pragma unroll
          for (int g = 0; g < G; ++g) {
            const float s1 = pmax[g] * (1.0f / 448.0f);
            const float inv1 = s1 > 0.f ? 1.0f / s1 : 0.f;
            uint8_t c1, c2, c3;
            split3(p[j][g], s1, inv1, c1, c2, c3);
            dst[swizzled_offset(0 * G + g, tl, 128)] = c1;
            dst[swizzled_offset(1 * G + g, tl, 128)] = c2;
            dst[swizzled_offset(2 * G + g, tl, 128)] = c3;
          }
#pragma unroll
          for (int n = kTerms * G; n < C::kN; ++n) dst[swizzled_offset(n, tl, 128)] = 0;
        }
      }
      fence_proxy_async_smem();
      mbar_arrive(&sh.p_ready[b]);

      // ---- the previous item's epilogue overlaps this item's PV MMAs
      if (k > 0) epilogue(k - 1, prev, pm_prev, pl_prev, pp_prev);
#pragma unroll
      for (int g = 0; g < G; ++g) {
        pm_prev[g] = mrow[g];
        pl_prev[g] = lsum[g];
        pp_prev[g] = pmax[g];
      }
      prev = cur;
      cur = nxt;
      kpos_cur = kpos_next;
    }
    (void)kpos_cur;
    if (n_my > 0) epilogue(n_my - 1, prev, pm_prev, pl_prev, pp_prev);
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

// ---------------------------------------------------------------- merge
// One warp per (request, q head); lane l owns D/32 consecutive outputs.
// The lanes load the splits' lse values together (32 per round) and reduce
// them with shuffles; the partial outputs are then read eight splits at a
// time, all loads of a group in flight before their weighted sum.
template <int D>
__global__ void __launch_bounds__(128) decode_merge_kernel(int B, int Hq,
                                                           const int32_t* __restrict__ split_off,
                                                           const float* __restrict__ part_o,
                                                           const float* __restrict__ part_lse,
                                                           uint16_t* __restrict__ o,
                                                           float* __restrict__ lse) {
  constexpr int EPL = D / 32, kGroup = 8;
  const int w = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  griddep_wait();   // the partials of the split-KV launch before this one
  if (w >= B * Hq) return;
  const int b = w / Hq, h = w % Hq;
  const int s0 = split_off[b], n = split_off[b + 1] - s0;
  float M = -INFINITY;
  for (int i = lane; i < n; i += 32) M = fmaxf(M, __ldg(part_lse + static_cast<size_t>(s0 + i) * Hq + h));
  M = warp_max(M);
  float acc[EPL];
#pragma unroll
  for (int e = 0; e < EPL; ++e) acc[e] = 0.f;
  float den = 0.f;
  if (M > -INFINITY) {
    for (int base = 0; base < n; base += 32) {
      float wgt = 0.f;
      if (base + lane < n) {
        const float ls = __ldg(part_lse + static_cast<size_t>(s0 + base + lane) * Hq + h);
        wgt = ls > -INFINITY ? __expf(ls - M) : 0.f;
      }
      den += wgt;
      const int cnt = min(32, n - base);
      for (int j = 0; j < cnt; j += kGroup) {
        float v[kGroup][EPL];
#pragma unroll
        for (int u = 0; u < kGroup; ++u) {
          const float* src =
              part_o + (static_cast<size_t>(s0 + base + j + u) * Hq + h) * D + lane * EPL;
#pragma unroll
          for (int e = 0; e < EPL; ++e) v[u][e] = 0.f;
          if (j + u < cnt) {
            if constexpr (EPL == 4) {
              const float4 x = __ldg(reinterpret_cast<const float4*>(src));
              v[u][0] = x.x; v[u][1] = x.y; v[u][2] = x.z; v[u][3] = x.w;
            } else {
              const float2 x = __ldg(reinterpret_cast<const float2*>(src));
              v[u][0] = x.x; v[u][1] = x.y;
            }
          }
        }
#pragma unroll
        for (int u = 0; u < kGroup; ++u) {
          const float wu = __shfl_sync(0xffffffffu, wgt, (j + u) & 31);
          // a split with weight 0 adds nothing, even if its partial row holds NaN
#pragma unroll
          for (int e = 0; e < EPL; ++e) acc[e] = wu > 0.f ? fmaf(wu, v[u][e], acc[e]) : acc[e];
        }
      }
    }
    den = warp_sum(den);
  }
  const float inv = den > 0.f ? 1.0f / den : 0.f;
  uint16_t out[EPL];
#pragma unroll
  for (int e = 0; e < EPL; ++e) {
    const __nv_bfloat16 bv = __float2bfloat16_rn(acc[e] * inv);
    out[e] = *reinterpret_cast<const uint16_t*>(&bv);
  }
  uint16_t* dst = o + (static_cast<size_t>(b) * Hq + h) * D + lane * EPL;
  if constexpr (EPL == 4) {
    *reinterpret_cast<uint2*>(dst) =
        make_uint2(out[0] | (static_cast<uint32_t>(out[1]) << 16),
                   out[2] | (static_cast<uint32_t>(out[3]) << 16));
  } else {
    *reinterpret_cast<uint32_t*>(dst) = out[0] | (static_cast<uint32_t>(out[1]) << 16);
  }
  if (lse != nullptr && lane == 0)
    lse[static_cast<size_t>(b) * Hq + h] = den > 0.f ? M + logf(den) : -INFINITY;
}

template <int D, int G>
cudaError_t launch_attend_t(const CUtensorMap& km, const CUtensorMap& vm, const DecodeArgs& a,
                            bool hnd, cudaStream_t stream) {
  using C = Cfg<D, G>;
  auto* kern = hnd ? decode_attend_kernel<D, G, true> : decode_attend_kernel<D, G, false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                           cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int grid = a.num_items < sms ? a.num_items : sms;
  kern<<<grid, kThreads, C::kSmem, stream>>>(km, vm, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode_attend(const DecodePlan& plan, float* float_ws, void* int_ws,
                                 const void* q, const void* k_pool, const void* v_pool,
                                 const float* k_scale_pool, const float* v_scale_pool,
                                 int num_pages, int page_size, const int32_t* block_table,
                                 int bt_stride, float sm_scale, int32_t* error_word,
                                 cudaStream_t stream, int* status) {
  *status = QPKV_OK;
  if (plan.num_items == 0) return cudaSuccess;
  if (plan.kind == 1)
    return launch_decode_heads(plan, float_ws, int_ws, q, k_pool, v_pool, k_scale_pool,
                               v_scale_pool, num_pages, page_size, block_table, bt_stride, sm_scale,
                               error_word, stream, status);
  const int D = static_cast<int>(plan.head_dim);
  const int Hkv = static_cast<int>(plan.num_kv_heads);
  const int G = static_cast<int>(plan.num_qo_heads / plan.num_kv_heads);
  const int R = page_size < kTile ? page_size : kTile;
  // pool as (d, kv head, K/V row); NHD rows are tokens (stride Hkv * D, head
  // stride D), HND rows run through each (page, head) run of ps tokens
  // (stride D, head stride ps * D)
  const bool hnd = plan.kv_layout == QPKV_KV_LAYOUT_HND;
  CUtensorMap km, vm;
  const uint64_t dims[3] = {static_cast<uint64_t>(D), static_cast<uint64_t>(Hkv),
                            static_cast<uint64_t>(num_pages) * page_size * (hnd ? Hkv : 1)};
  const uint64_t strides[2] = {hnd ? static_cast<uint64_t>(page_size) * D : static_cast<uint64_t>(D),
                               hnd ? static_cast<uint64_t>(D) : static_cast<uint64_t>(Hkv) * D};
  const uint32_t box[3] = {static_cast<uint32_t>(D), 1u, static_cast<uint32_t>(R)};
  const CUtensorMapSwizzle swz =
      D == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  if (encode_tensor_map(&km, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(k_pool), dims,
                        strides, box, swz) != CUDA_SUCCESS ||
      encode_tensor_map(&vm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(v_pool), dims,
                        strides, box, swz) != CUDA_SUCCESS) {
    *status = QPKV_ERR_CUDA;
    return cudaErrorInvalidValue;
  }
  const uint8_t* iws = static_cast<const uint8_t*>(int_ws);
  DecodeArgs a;
  a.items = reinterpret_cast<const DecodeItem*>(iws + plan.items_offset);
  a.num_items = static_cast<int>(plan.num_items);
  a.Hq = static_cast<int>(plan.num_qo_heads);
  a.Hkv = Hkv;
  a.q = static_cast<const uint16_t*>(q);
  a.k_pool = static_cast<const uint8_t*>(k_pool);
  a.v_pool = static_cast<const uint8_t*>(v_pool);
  a.k_scale = k_scale_pool;
  a.v_scale = v_scale_pool;
  a.block_table = block_table;
  a.bt_stride = bt_stride;
  a.page_size = page_size;
  a.num_pages = num_pages;
  a.sm_scale_log2 = sm_scale * kLog2e;
  a.part_o = float_ws;
  a.part_lse = float_ws + plan.total_splits * plan.num_qo_heads * plan.head_dim;
  a.err = error_word;
#define QPKV_DECODE_CASE(DD, GG) \
  if (D == DD && G == GG) return launch_attend_t<DD, GG>(km, vm, a, hnd, stream);
  QPKV_DECODE_CASE(128, 1)
  QPKV_DECODE_CASE(128, 2)
  QPKV_DECODE_CASE(128, 4)
  QPKV_DECODE_CASE(128, 8)
  QPKV_DECODE_CASE(64, 1)
  QPKV_DECODE_CASE(64, 2)
  QPKV_DECODE_CASE(64, 4)
  QPKV_DECODE_CASE(64, 8)
#undef QPKV_DECODE_CASE
  *status = QPKV_ERR_UNSUPPORTED;
  return cudaErrorInvalidValue;
}

cudaError_t launch_decode_merge(const DecodePlan& plan, const float* float_ws, const void* int_ws,
                                void* o, float* lse, cudaStream_t stream) {
  const int B = static_cast<int>(plan.batch), Hq = static_cast<int>(plan.num_qo_heads);
  const int warps = B * Hq;
  if (warps == 0) return cudaSuccess;
  const int32_t* split_off = reinterpret_cast<const int32_t*>(
      static_cast<const uint8_t*>(int_ws) + plan.split_off_offset);
  const float* part_lse = float_ws + plan.total_splits * plan.num_qo_heads * plan.head_dim;
  const int grid = (warps * 32 + 127) / 128;
  // a programmatic dependent of the split-KV launch: it is scheduled while
  // that launch drains and waits for it before reading the partials
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(128);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  uint16_t* out = static_cast<uint16_t*>(o);
  if (plan.head_dim == 128)
    return cudaLaunchKernelEx(&cfg, decode_merge_kernel<128>, B, Hq, split_off, float_ws, part_lse,
                              out, lse);
  return cudaLaunchKernelEx(&cfg, decode_merge_kernel<64>, B, Hq, split_off, float_ws, part_lse, out,
                            lse);
}

}  // namespace qpkv
