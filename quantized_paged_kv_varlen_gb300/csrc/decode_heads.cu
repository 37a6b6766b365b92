// Split-KV paged FP8 decode, all kv heads of a token range per work item.
//
// Same computation as decode.cu ("KvQuantSparseFlashAttention" README,
// 计算公式, per-token-head FP8 K/V, pages gathered through block_table;
// flashinfer "Batch Decode Attention Kernels" plan/run split), laid out for
// HBM efficiency when pages are small.  With page_size 16 a (page, kv head)
// block is only 16 rows x 128 bytes; streaming such 2 KB pieces caps the SM's
// copy engine near 4 TB/s, while whole 16 KB pages stream at the HBM rate.
//
// Geometry: 4 or 8 kv heads.  A tile is 128 (kv head, token) rows, nt =
// 128 / Hkv consecutive tokens of every kv head, fetched as one TMA box
// [D bytes x nt tokens x Hkv heads] whose dimensions are ordered so that
// shared memory comes out head-major: row r = head * nt + t.  For the
// 8-head / page-16 cache one box is one whole 16 KB page.  Each softmax warp
// owns 32 tile rows, i.e. whole kv heads (one head of 32 tokens, or two of
// 16), so every per-head reduction stays inside a warp.
//
// MMAs (tcgen05, FP8 operands straight from the cache bytes):
//   S[128 rows x N] = K_tile[128 x D] . Qt[N x D]^T,  N = 16-padded 3*Hq
// gives every row its logits against all query heads (a row keeps the 3*G
// columns of its own kv head), and
//   O[128 x D] += P[128 x 128 rows] . V_tile[128 rows x D]
// where P is block diagonal: its row for (query head, term) is nonzero only
// on the tile rows of that query head's kv head.  Queries and probabilities
// enter the FP8 MMA as three E4M3 terms (scales s, s/16, s/256).  O's TMEM
// lanes are (query head, term) rows placed in the lane quarter of the warp
// that owns the kv head, so the rare rescale of a head's O rows and the
// epilogue need no cross-warp synchronisation.
//
// The softmax is online: a query head keeps a running maximum and moves it
// only when a tile exceeds it by more than 2^8 (then that head's O rows are
// rescaled).  Probabilities are at most 2^8 and carry the per-token v-scale,
// so the item's largest v-scale fixes the probability term scale up front.
//
// Roles (one persistent CTA per SM, 12 warps):
//   warp 0  items: takes work items (the first by CTA index, then from a
//           global counter, largest first), resolves the item's pages into a
//           row table, loads its k/v-scales and fixes the probability term
//           scales;
//   warp 1  stream: lane 0 issues one TMA per tile in the order
//           K(0) K(1) | K(2) V(0) | K(3) V(1) | ... (K two tiles ahead of V,
//           at most one item ahead); the warp copies partial tail tiles row
//           by row;
//   warp 2  QK MMAs, warp 11 PV MMAs (one issuing lane each);
//   warps 3-6 softmax;
//   warps 7-10 split each item's queries into E4M3 terms (two items ahead)
//           and move finished O rows out of TMEM (the epilogue).
// The last CTA to finish re-arms the counter.
#include <cmath>

#include "common.cuh"
#include "internal.h"
#include "ring_sched.cuh"

namespace qpkv {
namespace {

constexpr int kTile = 128;        // (kv head, token) rows per tile = MMA M
constexpr int kThreads = 384;     // 12 warps
constexpr int kWarpItems = 0, kWarpStream = 1, kWarpMma = 2, kWarpSoftmax0 = 3;
constexpr int kSoftmax = 128;     // warps 3..6 (softmax), 7..10 (epilogue)
constexpr int kWarpEpi0 = 7;      // warps 7..10
constexpr int kWarpPv = 11;
constexpr int kMaxStages = 16;
constexpr int kMaxTilesItem = 16;
constexpr int kSBufs = 2;         // S accumulators in TMEM
constexpr int kOBufs = 2;         // O accumulators in TMEM (one per item in flight)
constexpr int kPBufs = 2;         // block-diagonal P operand buffers
constexpr int kMaxN = 96;         // 3 terms x 32 query heads
constexpr float kRescaleLog2 = 8.0f;   // running max moves only by more than this

template <int D>
struct HCfg {
  static constexpr int kTileBytes = kTile * D;
  static constexpr uint32_t kSwz = D == 128 ? kSwizzle128B : kSwizzle64B;
  static constexpr int kSBO = 8 * D;
  static constexpr int kQTBytes = ((kMaxN * D + 1023) / 1024) * 1024;
  static constexpr int kPBytes = kTile * kTile;                   // 128 rows x 128 tile rows
  static constexpr int kScaleBytes = kMaxTilesItem * kTile * 4;   // one item's k- or v-scales
  static constexpr int kFixed = 2 * kQTBytes + kPBufs * kPBytes + 4 * kScaleBytes;
  static constexpr int kBudget = 221 * 1024;   // + ~3.2 KB static shared state
  static constexpr int kStagesRaw = (kBudget - kFixed) / kTileBytes;
  static constexpr int kStages = kStagesRaw > kMaxStages ? kMaxStages : kStagesRaw;
  static constexpr int kOffQT = kStages * kTileBytes;
  static constexpr int kOffP = kOffQT + 2 * kQTBytes;
  static constexpr int kOffKS = kOffP + kPBufs * kPBytes;
  static constexpr int kOffVS = kOffKS + 2 * kScaleBytes;
  static constexpr int kBytes = kOffVS + 2 * kScaleBytes;
  static constexpr int kSmem = kBytes + 1024;
  static constexpr int kOCol0 = kSBufs * kMaxN;   // first O column in TMEM
  static_assert(kStages >= 6, "ring too small");
  static_assert(kSmem + 4096 <= 227 * 1024, "shared memory (dynamic + static)");
  static_assert(kOCol0 + kOBufs * D <= 512, "TMEM");
};

struct HeadsArgs {
  const DecodeItem* items;
  int num_items;
  int* counters;   // [0]: items claimed past the first wave, [1]: CTAs finished
  int Hq, Hkv;
  int N;           // QK MMA N: 16-padded 3 * Hq
  int nt;          // tokens per tile (128 / Hkv)
  const uint16_t* q;
  const uint8_t* k_pool;
  const uint8_t* v_pool;
  const float* k_scale;
  const float* v_scale;
  const int32_t* block_table;
  int bt_stride;
  int page_size;
  int num_pages;
  float sm_scale_log2;
  float* part_o;
  float* part_lse;
  int* err;
};

struct HShared {
  uint64_t full[kMaxStages], empty[kMaxStages];
  uint64_t tab_full[2];    // item's descriptor and row table written
  uint64_t scl_full[2];    // item's k/v-scales landed
  uint64_t desc_full[2];   // item completely prepared (query terms, term scales)
  uint64_t desc_free[2];   // item's shared resources released by all roles
  uint64_t s_full[kSBufs], s_free[kSBufs];
  uint64_t p_ready[kPBufs], p_free[kPBufs];
  uint64_t o_full[kOBufs], o_free[kOBufs];
  uint64_t mma_done[2];      // QK and PV issuers' MMAs complete
  uint64_t ep_ready[2];      // item's O scales written, O may be read once complete
  uint64_t q_done[2];        // item's query terms and their scales written
  DecodeItem desc[2];
  int tab[2][kMaxTilesItem];   // K/V row of each tile's box in the tensor maps, -1 if its page is bad
  float sig_q[2][32];          // query term scale per query head
  float sig_p[2][32];          // probability term scale per query head
  float ep_scale[2][kTile];   // per O row: sig_p / softmax denominator
  float ep_lse[2][kTile];     // per O row: natural-log LSE
  int ep_slot[2];             // partial-output slot, -1: stop
  uint32_t tmem_base;
  int abort;
};

// Bounded mbarrier wait; gives up when another role aborted or the limit runs out.
__device__ __forceinline__ bool hwait(uint64_t* bar, uint32_t parity, HShared& sh, int* err) {
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

// Bounded wait that ignores the abort flag: used to let this CTA's own copies
// and MMAs land before it exits.
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity, int* err) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > kWaitTimeoutCycles) {
      report_error(err, kDevErrTimeout);
      return;
    }
  }
}

// Lane 0 waits, the warp learns the outcome and is ordered after the wait.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, HShared& sh, int* err,
                                          int lane) {
  int ok = 1;
  if (lane == 0) ok = hwait(bar, parity, sh, err) ? 1 : 0;
  ok = __shfl_sync(0xffffffffu, ok, 0);
  __syncwarp();
  return ok != 0;
}

__device__ __forceinline__ int htiles(const DecodeItem& it, int nt) {
  return (it.t1 - it.t0 + nt - 1) / nt;
}

// Three-term E4M3 split with term scales s1, s1/16, s1/256, for a pair
// of values (codes: low byte = x0).
__device__ __forceinline__ void hsplit3x2(float x0, float x1, float inv1, float s1, uint16_t& c1,
                                         uint16_t& c2, uint16_t& c3) {
  c1 = f32x2_to_e4m3x2(x1 * inv1, x0 * inv1);
  const float2 d1 = e4m3x2_to_f32x2(c1);
  const float r0 = fmaf(-d1.x, s1, x0), r1 = fmaf(-d1.y, s1, x1);
  c2 = f32x2_to_e4m3x2(r1 * inv1 * 16.0f, r0 * inv1 * 16.0f);
  const float2 d2 = e4m3x2_to_f32x2(c2);
  const float s16 = s1 * (1.0f / 16.0f);
  const float q0 = fmaf(-d2.x, s16, r0), q1 = fmaf(-d2.y, s16, r1);
  c3 = f32x2_to_e4m3x2(q1 * inv1 * 256.0f, q0 * inv1 * 256.0f);
}



// HND: K/V pools [P, Hkv, ps, D] (a compile-time switch, so the NHD kernel
// carries no code for the other layout)
template <int D, int G, bool HND>
__global__ void __launch_bounds__(kThreads, 1)
    decode_heads_kernel(const __grid_constant__ CUtensorMap k_map,
                        const __grid_constant__ CUtensorMap v_map, const HeadsArgs a) {
  using C = HCfg<D>;
  constexpr int NS = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint8_t* sQT = smem + C::kOffQT;     // [2][N x D] query terms (QK B operand)
  uint8_t* sP = smem + C::kOffP;       // [kPBufs][128 x 128] block-diagonal P
  float* sKS = reinterpret_cast<float*>(smem + C::kOffKS);   // [2][16 tiles][128] k-scales
  float* sVS = reinterpret_cast<float*>(smem + C::kOffVS);   // [2][16 tiles][128] v-scales
  __shared__ HShared sh;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int Hkv = a.Hkv, Hq = a.Hq, nt = a.nt, N = a.N;
  const int ps = a.page_size;

  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&sh.full[s], 1);
      mbar_init(&sh.empty[s], 1);
    }
    for (int d = 0; d < 2; ++d) {
      mbar_init(&sh.tab_full[d], 1);
      mbar_init(&sh.scl_full[d], 1);
      mbar_init(&sh.desc_full[d], 1);
      mbar_init(&sh.desc_free[d], 1 + 1 + 1 + kSoftmax);   // QK commit, PV issuer, stream, softmax
    }
    for (int b = 0; b < kSBufs; ++b) {
      mbar_init(&sh.s_full[b], 1);
      mbar_init(&sh.s_free[b], kSoftmax);
    }
    for (int b = 0; b < kPBufs; ++b) {
      mbar_init(&sh.p_ready[b], kSoftmax);
      mbar_init(&sh.p_free[b], 1);
    }
    for (int b = 0; b < kOBufs; ++b) {
      mbar_init(&sh.o_full[b], 1);
      mbar_init(&sh.o_free[b], kSoftmax);
    }
    for (int d = 0; d < 2; ++d) {
      mbar_init(&sh.ep_ready[d], kSoftmax);
      mbar_init(&sh.q_done[d], kSoftmax);
    }
    mbar_init(&sh.mma_done[0], 1);
    mbar_init(&sh.mma_done[1], 1);
    sh.abort = 0;
    fence_mbar_init();
  }
  // Stage rows never loaded must hold finite bytes, P is zero off its
  // diagonal blocks, query-term rows past 3*Hq are zero: clear everything once.
  for (int i = tid; i < C::kBytes / 16; i += kThreads)
    reinterpret_cast<uint4*>(smem)[i] = make_uint4(0, 0, 0, 0);
  fence_proxy_async_smem();
  if (warp == kWarpMma) tmem_alloc(&sh.tmem_base, 512);
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = sh.tmem_base;

  if (warp == kWarpItems) {
    // ------------------------------------------------------------ items
    for (int o = 0;; ++o) {
      const int d = o & 1;
      int idx = static_cast<int>(blockIdx.x);
      if (o > 0) {
        int v = 0;
        if (lane == 0) v = atomicAdd(&a.counters[0], 1);
        idx = __shfl_sync(0xffffffffu, v, 0) + static_cast<int>(gridDim.x);
      }
      DecodeItem it{};
      it.b = -1;
      if (idx < a.num_items) it = a.items[idx];
      const int ntl = it.b < 0 ? 0 : htiles(it, nt);
      // lane j resolves tile j's page
      int row = -1, krow = -1;
      if (lane < ntl) {
        const int tok = it.t0 + lane * nt;
        const int page = __ldg(a.block_table + static_cast<size_t>(it.b) * a.bt_stride + tok / ps);
        if (page >= 0 && page < a.num_pages) {
          row = page * ps + tok % ps;
          krow = HND ? page * Hkv * ps + tok % ps : row;
        } else {
          report_error(a.err, kDevErrBadPage);
        }
      }
      // the resources of item o-2 must be released by every role
      if (!warp_wait(&sh.desc_free[d], ((o >> 1) & 1) ^ 1, sh, a.err, lane)) break;
      if (lane < kMaxTilesItem) sh.tab[d][lane] = krow;
      if (lane == 0) sh.desc[d] = it;
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.tab_full[d]);
      if (it.b < 0) {
        if (lane == 0) mbar_arrive(&sh.desc_full[d]);
        break;
      }
      // k- and v-scales of every tile (one 512-byte piece each)
      float* ks = sKS + d * (kMaxTilesItem * kTile);
      float* vs = sVS + d * (kMaxTilesItem * kTile);
      // the scale pools may have been written by the launch before this one
      if (o == 0) griddep_wait();
      const bool load = lane < ntl && row >= 0;
      const int total = __popc(__ballot_sync(0xffffffffu, load)) * (2 * kTile * 4);
      if (lane == 0) mbar_arrive_expect_tx(&sh.scl_full[d], total);
      __syncwarp();
      if (load) {
        bulk_load(ks + lane * kTile, a.k_scale + static_cast<size_t>(row) * Hkv, kTile * 4,
                  &sh.scl_full[d]);
        bulk_load(vs + lane * kTile, a.v_scale + static_cast<size_t>(row) * Hkv, kTile * 4,
                  &sh.scl_full[d]);
      }
      // the epilogue warps split the item's queries into E4M3 terms
      if (!warp_wait(&sh.q_done[d], (o >> 1) & 1, sh, a.err, lane)) {
        if (lane == 0) drain_wait(&sh.scl_full[d], (o >> 1) & 1, a.err);
        break;
      }
      // probability term scale per query head from its kv head's largest
      // v-scale over the item's valid tokens
      if (!warp_wait(&sh.scl_full[d], (o >> 1) & 1, sh, a.err, lane)) {
        if (lane == 0) drain_wait(&sh.scl_full[d], (o >> 1) & 1, a.err);
        break;
      }
      float m = 0.f;
      for (int i = lane; i < ntl * kTile; i += 32) {
        const int j = i / kTile, r = i % kTile;
        if (it.t0 + j * nt + r / Hkv < it.t1) m = fmaxf(m, vs[i]);
      }
      for (int off = Hkv; off < 32; off <<= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
      // probabilities are <= 2^8: P' = p * v_scale <= 2^8 * m = 448 * sig_p
      if (lane < Hkv)
        for (int g = 0; g < G; ++g) sh.sig_p[d][lane * G + g] = m * (256.0f / 448.0f);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh.desc_full[d]);
    }
  } else if (warp == kWarpStream) {
    // ------------------------------------------------------------ stream
    if (lane == 0) {
      tma_prefetch_desc(&k_map);
      tma_prefetch_desc(&v_map);
    }
    // the K/V pools may have been written by the launch before this one
    griddep_wait();
    int pos = 0;
    // one tile into the next ring stage: a whole box by TMA (lane 0), or the
    // valid rows of a partial tail tile by 16-byte copies (whole warp)
    auto emit = [&](const DecodeItem& it, int d, int j, bool is_v) -> bool {
      const int s = pos % NS;
      if (!warp_wait(&sh.empty[s], ((pos / NS) & 1) ^ 1, sh, a.err, lane)) return false;
      uint8_t* stage = smem + s * C::kTileBytes;
      const int nvalid = min(nt, it.t1 - (it.t0 + j * nt));
      const int row = sh.tab[d][j];
      if (nvalid == nt) {
        if (lane == 0) {
          if (row >= 0) {
            mbar_arrive_expect_tx(&sh.full[s], C::kTileBytes);
            tma_load_3d(stage, is_v ? &v_map : &k_map, &sh.full[s], 0, row, 0);
          } else {
            mbar_arrive(&sh.full[s]);
          }
        }
      } else {
        if (row >= 0) {
          const uint8_t* pool = is_v ? a.v_pool : a.k_pool;
          constexpr int kChunks = D / 16;
          const int per_head = nvalid * kChunks;
          for (int i = lane; i < Hkv * per_head; i += 32) {
            const int h = i / per_head, rem = i % per_head;
            const int t = rem / kChunks, c = rem % kChunks;
            const size_t kv_row = HND ? static_cast<size_t>(row + t) + static_cast<size_t>(h) * a.page_size
                                      : static_cast<size_t>(row + t) * Hkv + h;
            cp_async_16(stage + swizzled_offset(h * nt + t, 16 * c, D), pool + kv_row * D + 16 * c);
          }
          cp_async_wait_all();
          fence_proxy_async_smem();   // generic-proxy rows, read by the tensor cores
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh.full[s]);
      }
      ++pos;
      return true;
    };
    auto open = [&](int o, DecodeItem& it) -> bool {
      if (!warp_wait(&sh.tab_full[o & 1], (o >> 1) & 1, sh, a.err, lane)) return false;
      it = sh.desc[o & 1];
      return true;
    };
    DecodeItem it0{}, it1{};
    auto open_item = [&](int o) -> int {
      DecodeItem it;
      if (!open(o, it)) return -1;
      if (o & 1) it1 = it; else it0 = it;
      return it.b < 0 ? 0 : htiles(it, nt);
    };
    RingSched q{0, 0, 0, 0, 0, 0, 0, false, 2};
    q.ntl0 = open_item(0);
    if (q.ntl0 > 0) {
      while (true) {
        const int step = ring_next(q, open_item);
        if (step == kStepK) {
          if (!emit((q.ko & 1) ? it1 : it0, q.ko & 1, q.kj, false)) break;
          ++q.kj;
          ++q.lead;
        } else if (step == kStepV) {
          const bool last = q.vj == q.ntl(q.vo) - 1;
          if (!emit((q.vo & 1) ? it1 : it0, q.vo & 1, q.vj, true)) break;
          if (last && lane == 0) mbar_arrive(&sh.desc_free[q.vo & 1]);   // done with its row table
          ++q.vj;
          --q.lead;
        } else {
          break;
        }
      }
    }
    // this CTA's copies still in flight land before it exits
    if (lane == 0)
      for (int i = pos > NS ? pos - NS : 0; i < pos; ++i)
        drain_wait(&sh.full[i % NS], (i / NS) & 1, a.err);
    __syncwarp();
  } else if (warp == kWarpMma || warp == kWarpPv) {
    // ---------------------------------------------------------------- MMA
    // Lane 0 of warp 2 issues the QK MMAs, lane 0 of warp 11 the PV MMAs;
    // both walk the ring schedule and skip the other side's stages, so
    // neither waits behind the other's issue.
    const bool is_qk = warp == kWarpMma;
    if (lane == 0) {
      const uint32_t idesc_qk = make_idesc(kFmtE4M3, kFmtE4M3, 0, 0, 128, N);
      const uint32_t idesc_pv = make_idesc(kFmtE4M3, kFmtE4M3, 1, 1, 128, D);
      // operand descriptors at offset 0 of each region; an operand at byte
      // offset x adds x >> 4 to the start-address field
      const uint64_t kdesc0 = make_smem_desc(smem_u32(smem), 16, C::kSBO, C::kSwz);
      const uint64_t vdesc0 = make_smem_desc(smem_u32(smem), 0, C::kSBO, C::kSwz);
      const uint64_t qdesc0 = make_smem_desc(smem_u32(sQT), 16, C::kSBO, C::kSwz);
      const uint64_t pdesc0 = make_smem_desc(smem_u32(sP), 0, 1024, kSwizzle128B);
      int pos = 0, st = 0, pt = 0;
      auto qk = [&](int o, int j, int ntl) -> bool {
        const int sb = st % kSBufs;
        const int s = pos % NS;
        if (!hwait(&sh.s_free[sb], ((st / kSBufs) & 1) ^ 1, sh, a.err) ||
            !hwait(&sh.full[s], (pos / NS) & 1, sh, a.err))
          return false;
        tc_fence_after_sync();
        const uint64_t da0 = kdesc0 + static_cast<uint64_t>((s * C::kTileBytes) >> 4);
        const uint64_t db0 = qdesc0 + static_cast<uint64_t>(((o & 1) * C::kQTBytes) >> 4);
#pragma unroll
        for (int kk = 0; kk < D / 32; ++kk)
          tc_mma_f8(tmem + sb * kMaxN, da0 + 2 * kk, db0 + 2 * kk, idesc_qk, kk > 0);
        tc_commit(&sh.empty[s]);
        tc_commit(&sh.s_full[sb]);
        if (j == ntl - 1) tc_commit(&sh.desc_free[o & 1]);   // last read of its query terms
        ++pos;
        ++st;
        return true;
      };
      auto pv = [&](int o, int j, int ntl) -> bool {
        const int pb = pt % kPBufs;
        const int s = pos % NS;
        if (!hwait(&sh.p_ready[pb], (pt / kPBufs) & 1, sh, a.err) ||
            !hwait(&sh.full[s], (pos / NS) & 1, sh, a.err))
          return false;
        tc_fence_after_sync();
        // A = P and B = V, both stored row per tile row (MN-major, one
        // 128-byte swizzle atom wide for P); K steps of 32 tile rows
        const uint64_t da0 = pdesc0 + static_cast<uint64_t>((pb * C::kPBytes) >> 4);
        const uint64_t db0 = vdesc0 + static_cast<uint64_t>((s * C::kTileBytes) >> 4);
#pragma unroll
        for (int kk = 0; kk < kTile / 32; ++kk)
          tc_mma_f8(tmem + C::kOCol0 + (o & 1) * D, da0 + (32 * 128 / 16) * kk, db0 + (2 * D) * kk,
                    idesc_pv, (j > 0 || kk > 0) ? 1u : 0u);
        tc_commit(&sh.empty[s]);
        tc_commit(&sh.p_free[pb]);
        if (j == ntl - 1) tc_commit(&sh.o_full[o & 1]);
        ++pos;
        ++pt;
        return true;
      };
      auto open_item = [&](int o) -> int {
        if (!hwait(&sh.desc_full[o & 1], (o >> 1) & 1, sh, a.err)) return -1;
        const DecodeItem it = sh.desc[o & 1];
        if (!is_qk) mbar_arrive(&sh.desc_free[o & 1]);   // the QK side releases by commit
        return it.b < 0 ? 0 : htiles(it, nt);
      };
      RingSched q{0, 0, 0, 0, 0, 0, 0, false, 2};
      q.ntl0 = open_item(0);
      if (q.ntl0 > 0) {
        while (true) {
          const int step = ring_next(q, open_item);
          if (step == kStepK) {
            if (is_qk) {
              if (!qk(q.ko, q.kj, q.ntl(q.ko))) break;
            } else {
              ++pos;
            }
            ++q.kj;
            ++q.lead;
          } else if (step == kStepV) {
            if (!is_qk) {
              if (q.vj == 0 && !hwait(&sh.o_free[q.vo & 1], ((q.vo >> 1) & 1) ^ 1, sh, a.err)) break;
              if (!pv(q.vo, q.vj, q.ntl(q.vo))) break;
            } else {
              ++pos;
            }
            ++q.vj;
            --q.lead;
          } else {
            break;
          }
        }
      }
      // every MMA issued here completes before TMEM is released
      tc_commit(&sh.mma_done[is_qk ? 0 : 1]);
      drain_wait(&sh.mma_done[is_qk ? 0 : 1], 0, a.err);
    }
    __syncwarp();
  } else if (warp >= kWarpSoftmax0 && warp < kWarpEpi0) {
    // ---------------------------------------------------------- softmax
    constexpr int kG3 = 3 * G;
    const int sw = warp & 3;                  // TMEM lane quarter
    const int tl = sw * 32 + lane;            // tile row = S lane
    const uint32_t lane_base = static_cast<uint32_t>(sw * 32) << 16;
    const int hpw = Hkv / 4;                  // kv heads per warp
    const int my_h = tl / nt;                 // kv head of this row
    const int my_t = tl % nt;                 // token of this row within the tile
    const int sidx = my_t * Hkv + my_h;       // [token][head] scale index within a tile
    const int sel = my_h % hpw;
    const int w_h0 = sw * hpw;
    // this lane's O row (see o_lane_role); S lanes of its kv head start at src_o
    const int o_slot = lane / nt, o_within = lane % nt;
    const bool o_lane = o_within < kG3;
    const int g_o = o_within / 3;
    const int qh_o = o_lane ? (sw * hpw + o_slot) * G + g_o : 0;
    const int src_o = o_slot * nt;
    // this row's 3G probability bytes: P tile row tl, bytes r0 .. r0 + 3G - 1
    const int r0 = sw * 32 + sel * nt;
    int st = 0, pt = 0;
    for (int o = 0;; ++o) {
      const int d = o & 1;
      if (!warp_wait(&sh.desc_full[d], (o >> 1) & 1, sh, a.err, lane)) break;
      const DecodeItem cur = sh.desc[d];
      if (cur.b < 0) {
        // tell the epilogue warps to stop, once they are done with item o-2
        hwait(&sh.o_free[d], ((o >> 1) & 1) ^ 1, sh, a.err);
        if (tl == 0) sh.ep_slot[d] = -1;
        mbar_arrive(&sh.ep_ready[d]);
        break;
      }
      const int ntl = htiles(cur, nt);
      float sq[G];
#pragma unroll
      for (int g = 0; g < G; ++g) sq[g] = sh.sig_q[d][my_h * G + g] * a.sm_scale_log2;
      const float sp = sh.sig_p[d][my_h * G];
      const float spinv = sp > 0.f ? 1.0f / sp : 0.f;
      const float spo = o_lane ? sh.sig_p[d][qh_o] : 0.f;
      const float* ksb = sKS + d * (kMaxTilesItem * kTile);
      const float* vsb = sVS + d * (kMaxTilesItem * kTile);
      float m_run[G], lpart[G];
#pragma unroll
      for (int g = 0; g < G; ++g) {
        m_run[g] = -INFINITY;
        lpart[g] = 0.f;
      }
      for (int j = 0; j < ntl; ++j) {
        // ---- logits of this row against its kv head's query heads
        const int sb = st % kSBufs;
        hwait(&sh.s_full[sb], (st / kSBufs) & 1, sh, a.err);
        __syncwarp();   // converged before the .sync.aligned TMEM accesses
        tc_fence_after_sync();
        uint32_t r[32];
        tmem_ld32(tmem + lane_base + sb * kMaxN + w_h0 * kG3, r);
        tmem_ld_wait();
        tc_fence_before_sync();
        mbar_arrive(&sh.s_free[sb]);
        ++st;
        const bool valid = cur.t0 + j * nt + my_t < cur.t1;
        const float ks = ksb[j * kTile + sidx];
        const float vs = valid ? vsb[j * kTile + sidx] : 0.f;
        float l[G];
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float v0 = __uint_as_float(sel ? r[(kG3 + g) & 31] : r[g]);
          const float v1 = __uint_as_float(sel ? r[(kG3 + G + g) & 31] : r[G + g]);
          const float v2 = __uint_as_float(sel ? r[(kG3 + 2 * G + g) & 31] : r[2 * G + g]);
          const float sdot = v0 + v1 * (1.0f / 16.0f) + v2 * (1.0f / 256.0f);
          l[g] = valid ? ks * sq[g] * sdot : -INFINITY;
        }
        // ---- running maximum per query head, moved only when a tile beats it
        // by more than 2^8: a warp vote first, the tile maxima only then
        bool beat = false;
#pragma unroll
        for (int g = 0; g < G; ++g) beat |= l[g] > m_run[g] + kRescaleLog2;
        bool need = false;
        float fac[G];
#pragma unroll
        for (int g = 0; g < G; ++g) fac[g] = 1.f;
        if (__any_sync(0xffffffffu, beat)) {
          float tmx[G];
#pragma unroll
          for (int g = 0; g < G; ++g) tmx[g] = l[g];
#pragma unroll
          for (int off = 1; off < 32; off <<= 1) {
            if (off < nt) {
#pragma unroll
              for (int g = 0; g < G; ++g)
                tmx[g] = fmaxf(tmx[g], __shfl_xor_sync(0xffffffffu, tmx[g], off));
            }
          }
#pragma unroll
          for (int g = 0; g < G; ++g) {
            if (tmx[g] > m_run[g] + kRescaleLog2) {
              if (m_run[g] > -INFINITY) {
                need = true;
                fac[g] = exp2f(m_run[g] - tmx[g]);
              }
              m_run[g] = tmx[g];
            }
          }
        }
        float p[G];
#pragma unroll
        for (int g = 0; g < G; ++g) {
          p[g] = valid ? exp2f(l[g] - m_run[g]) : 0.f;
          lpart[g] = lpart[g] * fac[g] + p[g];
        }
        if (__any_sync(0xffffffffu, need)) {
          // rare: rescale this warp's O rows by their query heads' factors,
          // once the previous PV has finished writing them
          float fo = 1.f;
#pragma unroll
          for (int g = 0; g < G; ++g) {
            const float t = __shfl_sync(0xffffffffu, fac[g], src_o);
            if (g == g_o) fo = t;
          }
          if (!o_lane) fo = 1.f;
          hwait(&sh.p_free[(pt - 1) % kPBufs], ((pt - 1) / kPBufs) & 1, sh, a.err);
          __syncwarp();
          tc_fence_after_sync();
#pragma unroll 1
          for (int c = 0; c < D / 16; ++c) {
            uint32_t part[16];
            const uint32_t addr = tmem + lane_base + C::kOCol0 + d * D + 16 * c;
            tmem_ld16(addr, part);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 16; ++i) part[i] = __float_as_uint(__uint_as_float(part[i]) * fo);
            tmem_st16(addr, part);
            tmem_st_wait();
          }
          tc_fence_before_sync();
        }
        // ---- P' = p * v-scale, three E4M3 terms, into the block-diagonal P:
        // bytes (g, term) at r0 + 3g + term of row tl, packed into words
        constexpr int kWords = (kG3 + 3) / 4;
        uint32_t wd[kWords];
#pragma unroll
        for (int i = 0; i < kWords; ++i) wd[i] = 0;
#pragma unroll
        for (int g = 0; g < G; g += 2) {
          uint16_t c1, c2, c3;
          hsplit3x2(p[g] * vs, g + 1 < G ? p[g + 1] * vs : 0.f, spinv, sp, c1, c2, c3);
          const uint32_t b[6] = {c1 & 0xFFu, c2 & 0xFFu, c3 & 0xFFu,
                                 static_cast<uint32_t>(c1 >> 8), static_cast<uint32_t>(c2 >> 8),
                                 static_cast<uint32_t>(c3 >> 8)};
#pragma unroll
          for (int i = 0; i < 6; ++i) {
            const int m = 3 * g + i;
            if (m < kG3) wd[m / 4] |= b[i] << (8 * (m % 4));
          }
        }
        const int pb = pt % kPBufs;
        hwait(&sh.p_free[pb], ((pt / kPBufs) & 1) ^ 1, sh, a.err);
        uint8_t* dst = sP + pb * C::kPBytes;
#pragma unroll
        for (int i = 0; i < kWords; ++i)
          *reinterpret_cast<uint32_t*>(dst + swizzled_offset(tl, r0 + 4 * i, 128)) = wd[i];
        fence_proxy_async_smem();
        mbar_arrive(&sh.p_ready[pb]);
        ++pt;
      }
      // ---- softmax denominators and reference maxima, moved to the O lanes
      float lo = 0.f, mo = -INFINITY;
#pragma unroll
      for (int g = 0; g < G; ++g) {
        float x = lpart[g];
#pragma unroll
        for (int off = 1; off < 32; off <<= 1)
          if (off < nt) x += __shfl_xor_sync(0xffffffffu, x, off);
        const float hsum = __shfl_sync(0xffffffffu, x, src_o);
        const float hmax = __shfl_sync(0xffffffffu, m_run[g], src_o);
        if (g == g_o) {
          lo = hsum;
          mo = hmax;
        }
      }
      // hand the item to the epilogue warps (after they finished item o-2)
      hwait(&sh.o_free[d], ((o >> 1) & 1) ^ 1, sh, a.err);
      sh.ep_scale[d][tl] = lo > 0.f ? spo / lo : 0.f;
      sh.ep_lse[d][tl] = lo > 0.f ? (mo + log2f(lo)) * kLn2 : -INFINITY;
      if (tl == 0) sh.ep_slot[d] = cur.slot;
      mbar_arrive(&sh.desc_free[d]);   // done with the item's scales and descriptor
      mbar_arrive(&sh.ep_ready[d]);
    }
  } else {
    // ------------------------------------------ query split and epilogue
    // These warps split the queries of each item into E4M3 terms (two items
    // ahead) and move each finished item's O rows out of TMEM.
    const int et = tid - kWarpEpi0 * 32;      // 0..127
    const int E = (Hq * D) / kSoftmax >= 8 ? (Hq * D) / kSoftmax : 8;   // query elements per thread
    const int tph = D / E;                    // threads per query head (<= 16)
    const bool q_thread = et < Hq * tph;      // whole warps (Hq * tph is a multiple of 32)
    const int qh_s = et / tph;
    const int d0 = (et % tph) * E;
    // Query split of item o: rows h*3G + term*G + g of the QK B operand and
    // the term scale of every query head.  1: done, 0: end of work, -1: failed.
    auto qprep = [&](int o) -> int {
      const int d = o & 1;
      if (!warp_wait(&sh.tab_full[d], (o >> 1) & 1, sh, a.err, lane)) return -1;
      const DecodeItem it = sh.desc[d];
      if (it.b < 0) return 0;
      if (q_thread) {
        const uint16_t* src = a.q + (static_cast<size_t>(it.b) * Hq + qh_s) * D + d0;
        uint32_t w[16];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          if (8 * i < E) {
            const uint4 v = __ldg(reinterpret_cast<const uint4*>(src + 8 * i));
            w[4 * i] = v.x;
            w[4 * i + 1] = v.y;
            w[4 * i + 2] = v.z;
            w[4 * i + 3] = v.w;
          }
        }
        float amax = 0.f;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          if (2 * i < E) {
            amax = fmaxf(amax, fabsf(bf16_bits_to_float(static_cast<uint16_t>(w[i] & 0xFFFFu))));
            amax = fmaxf(amax, fabsf(bf16_bits_to_float(static_cast<uint16_t>(w[i] >> 16))));
          }
        }
#pragma unroll
        for (int off = 1; off < 16; off <<= 1)
          if (off < tph) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
        const float s1 = amax * (1.0f / 448.0f);
        const float inv1 = s1 > 0.f ? 1.0f / s1 : 0.f;
        if (et % tph == 0) sh.sig_q[d][qh_s] = s1;
        uint8_t* qt = sQT + d * C::kQTBytes;
        const int n0 = (qh_s / G) * 3 * G + qh_s % G;
#pragma unroll
        for (int i = 0; i < 8; ++i) {   // 4 elements -> one 32-bit word per term row
          if (4 * i < E) {
            uint16_t a1, a2, a3, b1, b2, b3;
            const uint32_t lo = w[2 * i], hi = w[2 * i + 1];
            hsplit3x2(bf16_bits_to_float(static_cast<uint16_t>(lo & 0xFFFFu)),
                      bf16_bits_to_float(static_cast<uint16_t>(lo >> 16)), inv1, s1, a1, a2, a3);
            hsplit3x2(bf16_bits_to_float(static_cast<uint16_t>(hi & 0xFFFFu)),
                      bf16_bits_to_float(static_cast<uint16_t>(hi >> 16)), inv1, s1, b1, b2, b3);
            const int k = d0 + 4 * i;
            *reinterpret_cast<uint32_t*>(qt + swizzled_offset(n0, k, D)) = a1 | (uint32_t(b1) << 16);
            *reinterpret_cast<uint32_t*>(qt + swizzled_offset(n0 + G, k, D)) = a2 | (uint32_t(b2) << 16);
            *reinterpret_cast<uint32_t*>(qt + swizzled_offset(n0 + 2 * G, k, D)) =
                a3 | (uint32_t(b3) << 16);
          }
        }
        fence_proxy_async_smem();   // generic stores, read by the tensor cores
      }
      mbar_arrive(&sh.q_done[d]);
      return 1;
    };
    int q_next = 0;
    bool q_more = true;
    auto q_step = [&]() {
      if (!q_more) return;
      const int r = qprep(q_next);
      if (r > 0) ++q_next; else q_more = false;
    };
    q_step();
    q_step();

    // epilogue: O rows -> fp32 partial output (terms combined) and lse
    const int sw = warp & 3;
    const int tl = sw * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(sw * 32) << 16;
    const int hpw = Hkv / 4;
    const int o_slot = lane / nt, o_within = lane % nt;
    const bool o_lane = o_within < 3 * G;
    const int qh_o = o_lane ? (sw * hpw + o_slot) * G + o_within / 3 : 0;
    const bool writer = o_lane && o_within % 3 == 0;
    for (int o = 0;; ++o) {
      const int d = o & 1;
      if (!warp_wait(&sh.ep_ready[d], (o >> 1) & 1, sh, a.err, lane)) break;
      const int slot = sh.ep_slot[d];
      if (slot < 0) break;
      const float so = sh.ep_scale[d][tl];
      const float lse = sh.ep_lse[d][tl];
      hwait(&sh.o_full[d], (o >> 1) & 1, sh, a.err);
      __syncwarp();
      tc_fence_after_sync();
      float* out = a.part_o + (static_cast<size_t>(slot) * Hq + qh_o) * D;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t v[32];
        tmem_ld32(tmem + lane_base + C::kOCol0 + d * D + 32 * c, v);
        tmem_ld_wait();
        float y[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float x0 = __uint_as_float(v[i]);
          const float x1 = __shfl_down_sync(0xffffffffu, x0, 1);
          const float x2 = __shfl_down_sync(0xffffffffu, x0, 2);
          y[i] = (x0 + x1 * (1.0f / 16.0f) + x2 * (1.0f / 256.0f)) * so;
        }
        if (writer) {
          float4* o4 = reinterpret_cast<float4*>(out + 32 * c);
#pragma unroll
          for (int i = 0; i < 8; ++i)
            o4[i] = make_float4(y[4 * i], y[4 * i + 1], y[4 * i + 2], y[4 * i + 3]);
        }
      }
      tc_fence_before_sync();
      mbar_arrive(&sh.o_free[d]);
      if (writer) a.part_lse[static_cast<size_t>(slot) * Hq + qh_o] = lse;
      q_step();
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  griddep_launch_dependents();   // the merge may start launching
  if (warp == kWarpMma) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, 512);
  }
  if (tid == 0) {
    // the last CTA to finish re-arms the work counter for the next launch
    __threadfence();
    if (atomicAdd(&a.counters[1], 1) == static_cast<int>(gridDim.x) - 1) {
      atomicExch(&a.counters[0], 0);
      atomicExch(&a.counters[1], 0);
    }
  }
}

template <int D, int G>
cudaError_t launch_heads_t(const CUtensorMap& km, const CUtensorMap& vm, const HeadsArgs& a,
                           bool hnd, cudaStream_t stream) {
  using C = HCfg<D>;
  auto* kern = hnd ? decode_heads_kernel<D, G, true> : decode_heads_kernel<D, G, false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int grid = a.num_items < sms ? a.num_items : sms;
  // launched as a programmatic dependent: the prologue (barriers, tensor
  // memory, the first work item's pages and queries) overlaps the end of the
  // launch before it; the K/V and scale reads wait for it
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = C::kSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, km, vm, a);
}

}  // namespace

bool heads_geometry(int Hq, int Hkv, int D, int page_size, int* nt, int* bt, int* nb,
                    int* max_tiles) {
  if (Hkv != 4 && Hkv != 8) return false;   // a warp's 32 tile rows hold whole kv heads
  if (Hq % Hkv != 0 || 3 * Hq > kMaxN) return false;
  const int G = Hq / Hkv;
  if (G != 1 && G != 2 && G != 4 && G != 8) return false;
  if (D != 64 && D != 128) return false;
  const int t = kTile / Hkv;
  if (page_size <= 0 || page_size % t != 0) return false;   // one box never crosses a page
  *nt = t;
  *bt = t;
  *nb = 1;
  *max_tiles = kMaxTilesItem;
  return true;
}

cudaError_t launch_decode_heads(const DecodePlan& plan, float* float_ws, void* int_ws,
                                const void* q, const void* k_pool, const void* v_pool,
                                const float* k_scale_pool, const float* v_scale_pool,
                                int num_pages, int page_size, const int32_t* block_table,
                                int bt_stride, float sm_scale, int32_t* error_word,
                                cudaStream_t stream, int* status) {
  *status = QPKV_OK;
  if (plan.num_items == 0) return cudaSuccess;
  const int D = static_cast<int>(plan.head_dim);
  const int Hkv = static_cast<int>(plan.num_kv_heads);
  const int Hq = static_cast<int>(plan.num_qo_heads);
  int nt, bt, nb, mt;
  if (!heads_geometry(Hq, Hkv, D, page_size, &nt, &bt, &nb, &mt)) {
    *status = QPKV_ERR_UNSUPPORTED;
    return cudaErrorInvalidValue;
  }
  // the row table holds at most kMaxTilesItem tiles per item
  if (plan.chunk <= 0 || plan.chunk % nt != 0 || plan.chunk > kMaxTilesItem * nt) {
    *status = QPKV_ERR_UNSUPPORTED;
    return cudaErrorInvalidValue;
  }
  // pool viewed as (d, token row, kv head): boxes come out head-major in smem
  // (HND: rows run through each (page, head) run of ps tokens, row stride D,
  // head stride ps * D)
  const bool hnd = plan.kv_layout == QPKV_KV_LAYOUT_HND;
  CUtensorMap km, vm;
  const uint64_t dims[3] = {static_cast<uint64_t>(D),
                            static_cast<uint64_t>(num_pages) * page_size * (hnd ? Hkv : 1),
                            static_cast<uint64_t>(Hkv)};
  const uint64_t strides[2] = {hnd ? static_cast<uint64_t>(D) : static_cast<uint64_t>(Hkv) * D,
                               hnd ? static_cast<uint64_t>(page_size) * D : static_cast<uint64_t>(D)};
  const uint32_t box[3] = {static_cast<uint32_t>(D), static_cast<uint32_t>(nt),
                           static_cast<uint32_t>(Hkv)};
  const CUtensorMapSwizzle swz = D == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  if (encode_tensor_map(&km, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(k_pool), dims,
                        strides, box, swz) != CUDA_SUCCESS ||
      encode_tensor_map(&vm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(v_pool), dims,
                        strides, box, swz) != CUDA_SUCCESS) {
    *status = QPKV_ERR_CUDA;
    return cudaErrorInvalidValue;
  }
  uint8_t* iws = static_cast<uint8_t*>(int_ws);
  HeadsArgs a;
  a.items = reinterpret_cast<const DecodeItem*>(iws + plan.items_offset);
  a.num_items = static_cast<int>(plan.num_items);
  a.counters = reinterpret_cast<int*>(iws + plan.counter_offset);
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.N = ((3 * Hq + 15) / 16) * 16;
  a.nt = nt;
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
  const int G = Hq / Hkv;
#define QPKV_HEADS_CASE(DD, GG) \
  if (D == DD && G == GG) return launch_heads_t<DD, GG>(km, vm, a, hnd, stream);
  QPKV_HEADS_CASE(128, 1)
  QPKV_HEADS_CASE(128, 2)
  QPKV_HEADS_CASE(128, 4)
  QPKV_HEADS_CASE(128, 8)
  QPKV_HEADS_CASE(64, 1)
  QPKV_HEADS_CASE(64, 2)
  QPKV_HEADS_CASE(64, 4)
  QPKV_HEADS_CASE(64, 8)
#undef QPKV_HEADS_CASE
  *status = QPKV_ERR_UNSUPPORTED;
  return cudaErrorInvalidValue;
}

}  // namespace qpkv
