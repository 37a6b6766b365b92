// Split-KV paged FP8 decode, all kv heads of a token range per work item.
//
// Same computation as decode.cu ("KvQuantSparseFlashAttention" README,
// 计算公式, per-token-head FP8 K/V, pages gathered through block_table;
// flashinfer "Batch Decode Attention Kernels" plan/run split), laid out for
// HBM efficiency when pages are small.  With page_size 16 a (page, kv head)
// block is only 16 rows x 128 bytes; streaming such 2 KB pieces caps the SM's
// copy engine near 4 TB/s, while whole 16 KB pages stream at the HBM rate.
//
// A tile is 128 (kv head, token) rows: nt = 128 / Hkv consecutive tokens of
// every kv head, fetched as TMA boxes [D bytes x bt tokens x Hkv heads] whose
// dimensions are ordered so that shared memory comes out head-major: row
// r = box * (Hkv*bt) + head * bt + t.  For the 8-head / page-16 cache one box
// is one whole 16 KB page.  The MMAs (tcgen05, FP8 operands straight from the
// cache bytes):
//   S[128 rows x N] = K_tile[128 x D] . Qt[N x D]^T,  N = 16-padded 3*Hq
// gives every row the logits against all query heads; a row keeps only the
// 3*G columns of its own kv head.  The probabilities form a block-diagonal
// P^T [N x 128 rows] (row n nonzero only on its kv head's rows), so
//   O^T[D x N] += V_tile^T[D x 128 rows] . P^T^T
// sums each query head over its own kv head's tokens.  Queries and
// probabilities enter the FP8 MMA as three E4M3 terms (s, s/16, s/256).
//
// The softmax is online, one tile at a time: a query head keeps a running
// maximum and moves it only when a tile exceeds it by more than 2^8 (then the
// item's O columns in TMEM are rescaled, which is rare); probabilities are at
// most 2^8 and are scaled by the per-token v-scale, so the item's largest
// v-scale (loaded with the item) fixes the probability term scale up front.
//
// Roles (one persistent CTA per SM, 6 warps): warp 0 takes items from a
// global counter (largest first), publishes descriptor, query rows and
// v-scales, and streams the tiles K(0) | K(1) V(0) | K(2) V(1) | ... through
// a shared-memory ring, K one tile ahead of V across item boundaries; warp 1
// issues QK(t+1) before PV(t); warps 2-5 own one tile row each and write
// P^T and the fp32 partial output.  The last CTA to finish re-arms the
// counter.
#include <cmath>

#include "common.cuh"
#include "internal.h"

namespace qpkv {
namespace {

constexpr int kTile = 128;      // (head, token) rows per tile
constexpr int kTerms = 3;
constexpr int kThreads = 192;
constexpr int kSoftmax = 128;
constexpr int kBarSoftmax = 1;
constexpr int kMaxStages = 12;
constexpr int kKSlots = 16;     // k-scale slots (one per K tile in flight)
constexpr int kMaxTilesItem = 16;
constexpr int kSBufs = 3;       // S accumulators in TMEM
constexpr int kOBufs = 2;       // O accumulators in TMEM (one per item in flight)
constexpr int kPBufs = 2;       // block-diagonal P^T operand buffers
constexpr int kMaxN = 96;       // 3 terms x 32 query heads
constexpr float kRescaleLog2 = 8.0f;   // running max moves only by more than this

template <int D, int G>
struct HCfg {
  static constexpr int kTileBytes = kTile * D;
  static constexpr uint32_t kSwz = D == 128 ? kSwizzle128B : kSwizzle64B;
  static constexpr int kSBO = 8 * D;
  static constexpr int kQTermBytes = ((kMaxN * D + 1023) / 1024) * 1024;
  static constexpr int kPTileBytes = kMaxN * kTile;
  static constexpr int kQRowBytes = 32 * D * 2;                 // bf16 rows, <= 32 query heads
  static constexpr int kVBufBytes = kMaxTilesItem * kTile * 4;  // v-scales of one item
  static constexpr int kFixed = 2 * kQTermBytes + kPBufs * kPTileBytes + kKSlots * kTile * 4 +
                                2 * kVBufBytes + 2 * kQRowBytes;
  static constexpr int kBudget = 222 * 1024;   // + ~3 KB static shared state
  static constexpr int kStagesRaw = (kBudget - kFixed) / kTileBytes;
  static constexpr int kStages = kStagesRaw > kMaxStages ? kMaxStages : kStagesRaw;
  static constexpr int kOffQT = kStages * kTileBytes;
  static constexpr int kOffP = kOffQT + 2 * kQTermBytes;
  static constexpr int kOffKS = kOffP + kPBufs * kPTileBytes;
  static constexpr int kOffVB = kOffKS + kKSlots * kTile * 4;
  static constexpr int kOffQRow = kOffVB + 2 * kVBufBytes;
  static constexpr int kBytes = kOffQRow + 2 * kQRowBytes;
  static constexpr int kSmem = kBytes + 1024;
  static_assert(kStages >= 6, "ring too small");
  static_assert(kSmem <= 227 * 1024, "shared memory");
  static_assert((kSBufs + kOBufs) * kMaxN <= 512, "TMEM");
};

struct HeadsArgs {
  const DecodeItem* items;
  int num_items;
  int* counters;   // [0]: next item, [1]: CTAs finished; both zero at launch
  int Hq, Hkv;
  int N;           // MMA N: 16-padded 3 * Hq
  int nt;          // tokens per tile (128 / Hkv)
  int bt;          // tokens per TMA box
  int nb;          // boxes per tile
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
  uint64_t kslot_free[kKSlots];
  uint64_t desc_full[2], desc_free[2];
  uint64_t q_ready[2];
  uint64_t s_full[kSBufs], s_free[kSBufs];
  uint64_t p_ready[kPBufs], p_free[kPBufs];
  uint64_t o_full[kOBufs], o_free[kOBufs];
  DecodeItem desc[2];
  float sig_q[2][32];      // query term scale per query head (per item parity)
  float sig_p[2][32];      // probability term scale per query head
  float m2[2][32], lsum[2][32];
  float red[2][8][8];      // [tile parity][16-row slot][g] tile maxima
  float redl[8][8];        // [16-row slot][g] softmax denominators
  float redq[kSoftmax];
  float vred[kSoftmax];
  float factor[32];        // O rescale factor per query head
  uint32_t tmem_base;
  int abort;
  int stop;
};

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

__device__ __forceinline__ int htiles(const DecodeItem& it, int nt) {
  return (it.t1 - it.t0 + nt - 1) / nt;
}

// Three-term E4M3 split of x with term scales s1, s1/16, s1/256.
__device__ __forceinline__ void hsplit3(float x, float inv1, float s1, uint8_t& c1, uint8_t& c2,
                                       uint8_t& c3) {
  c1 = f32_to_e4m3(x * inv1);
  const float r1 = fmaf(-e4m3_to_f32(c1), s1, x);
  c2 = f32_to_e4m3(r1 * inv1 * 16.0f);
  const float r2 = fmaf(-e4m3_to_f32(c2), s1 * (1.0f / 16.0f), r1);
  c3 = f32_to_e4m3(r2 * inv1 * 256.0f);
}

// Pick register `i` of 4 without dynamic indexing.
__device__ __forceinline__ int pick4(const int (&r)[4], int i) {
  return i == 0 ? r[0] : (i == 1 ? r[1] : (i == 2 ? r[2] : r[3]));
}

template <int D, int G>
__global__ void __launch_bounds__(kThreads, 1)
    decode_heads_kernel(const __grid_constant__ CUtensorMap k_map,
                        const __grid_constant__ CUtensorMap v_map, const HeadsArgs a) {
  using C = HCfg<D, G>;
  constexpr int NS = C::kStages;
  constexpr int kG3 = kTerms * G;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint8_t* sQT = smem + C::kOffQT;     // [2][N x D] query terms (QK B operand)
  uint8_t* sP = smem + C::kOffP;       // [kPBufs][N x 128] block-diagonal P^T
  float* sKS = reinterpret_cast<float*>(smem + C::kOffKS);   // [kKSlots][128] k-scales
  float* sVB = reinterpret_cast<float*>(smem + C::kOffVB);   // [2][16 tiles][128] v-scales
  uint8_t* sQRow = smem + C::kOffQRow; // [2][Hq x D] bf16 query rows
  __shared__ HShared sh;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int Hkv = a.Hkv, Hq = a.Hq, nt = a.nt, bt = a.bt, nb = a.nb, N = a.N;
  const int ps = a.page_size;
  const int rpb = Hkv * bt;  // rows per box

  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&sh.full[s], 1 + 32);  // expect_tx arrival + 32 lanes' cp.async arrivals
      mbar_init(&sh.empty[s], 1);
    }
    for (int s = 0; s < kKSlots; ++s) mbar_init(&sh.kslot_free[s], kSoftmax);
    for (int d = 0; d < 2; ++d) {
      mbar_init(&sh.desc_full[d], 1);
      mbar_init(&sh.desc_free[d], 1 + kSoftmax);
      mbar_init(&sh.q_ready[d], kSoftmax);
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
    sh.abort = 0;
    sh.stop = 0;
    fence_mbar_init();
  }
  // Rows never loaded must hold finite bytes, P^T is zero off its diagonal
  // blocks and the query-term rows past 3*Hq are zero: clear all three once.
  for (int i = tid; i < C::kOffKS / 16; i += kThreads)
    reinterpret_cast<uint4*>(smem)[i] = make_uint4(0, 0, 0, 0);
  fence_proxy_async_smem();
  if (warp == 1) tmem_alloc(&sh.tmem_base, 512);
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = sh.tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    tma_prefetch_desc(&k_map);
    tma_prefetch_desc(&v_map);
    int pos = 0, kq = 0;
    auto next_item = [&]() {
      int idx = 0;
      if (lane == 0) idx = atomicAdd(&a.counters[0], 1);
      idx = __shfl_sync(0xffffffffu, idx, 0);
      DecodeItem it{};
      it.b = -1;
      if (idx < a.num_items) it = a.items[idx];
      return it;
    };
    // pool rows of this item's boxes; lane l holds boxes l, l+32, l+64, l+96
    auto box_rows = [&](const DecodeItem& it, int (&rows)[4]) {
      const int nbox = it.b < 0 ? 0 : htiles(it, nt) * nb;
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        rows[m] = -1;
        const int box = lane + 32 * m;
        if (box < nbox) {
          const int tok = it.t0 + (box / nb) * nt + (box % nb) * bt;
          if (tok < it.t1) {
            const int page =
                __ldg(a.block_table + static_cast<size_t>(it.b) * a.bt_stride + tok / ps);
            if (page >= 0 && page < a.num_pages) {
              rows[m] = page * ps + (tok % ps);
            } else {
              report_error(a.err, kDevErrBadPage);
            }
          }
        }
      }
    };
    // Item o: descriptor, its query rows and all its v-scales, under desc_full.
    auto publish = [&](int o, const DecodeItem& it, const int (&rows)[4]) -> bool {
      const int d = o & 1;
      bool ok = true;
      if (lane == 0) ok = hwait(&sh.desc_free[d], ((o >> 1) & 1) ^ 1, sh, a.err);
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      if (!ok) return false;
      if (it.b < 0) {
        if (lane == 0) {
          sh.desc[d] = it;
          mbar_arrive(&sh.desc_full[d]);
        }
        return true;
      }
      int vbytes = 0;
#pragma unroll
      for (int m = 0; m < 4; ++m) vbytes += rows[m] >= 0 ? rpb * 4 : 0;
      const int total = __reduce_add_sync(0xffffffffu, vbytes) + Hq * D * 2;
      if (lane == 0) {
        sh.desc[d] = it;
        mbar_arrive_expect_tx(&sh.desc_full[d], total);
        bulk_load(sQRow + d * C::kQRowBytes, a.q + static_cast<size_t>(it.b) * Hq * D, Hq * D * 2,
                  &sh.desc_full[d]);
      }
      __syncwarp();
      float* vb = sVB + d * (kMaxTilesItem * kTile);
#pragma unroll
      for (int m = 0; m < 4; ++m)
        if (rows[m] >= 0)
          bulk_load(vb + (lane + 32 * m) * rpb, a.v_scale + static_cast<size_t>(rows[m]) * Hkv,
                    rpb * 4, &sh.desc_full[d]);
      return true;
    };
    auto emit = [&](const DecodeItem& it, const int (&rows)[4], int j, bool is_v) -> bool {
      const int s = pos % NS;
      bool ok = true;
      if (lane == 0) ok = hwait(&sh.empty[s], ((pos / NS) & 1) ^ 1, sh, a.err);
      float* kslot = sKS + (kq % kKSlots) * kTile;
      if (!is_v && lane == 0 && ok)
        ok = hwait(&sh.kslot_free[kq % kKSlots], ((kq / kKSlots) & 1) ^ 1, sh, a.err);
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      if (!ok) return false;
      uint8_t* stage = smem + s * C::kTileBytes;
      const int nvalid = min(nt, it.t1 - (it.t0 + j * nt));
      // lanes < nb own one box each: its pool row and its valid token count
      const int src = pick4(rows, (j * nb) / 32);
      const int myrow = __shfl_sync(0xffffffffu, src, (j * nb + (lane < nb ? lane : 0)) % 32);
      const int nvb = lane < nb ? max(0, min(bt, nvalid - lane * bt)) : 0;
      const bool full_box = nvb == bt && myrow >= 0;
      const bool kscale_box = !is_v && nvb > 0 && myrow >= 0;
      const int bytes = (full_box ? rpb * D : 0) + (kscale_box ? rpb * 4 : 0);
      const int total = __reduce_add_sync(0xffffffffu, bytes);
      if (lane == 0) mbar_arrive_expect_tx(&sh.full[s], total);
      __syncwarp();
      if (full_box)
        tma_load_3d(stage + lane * rpb * D, is_v ? &v_map : &k_map, &sh.full[s], 0, myrow, 0);
      if (kscale_box)
        bulk_load(kslot + lane * rpb, a.k_scale + static_cast<size_t>(myrow) * Hkv, rpb * 4,
                  &sh.full[s]);
      // a box only partly inside the item: its valid rows by 16-byte cp.async
      const uint8_t* pool = is_v ? a.v_pool : a.k_pool;
      for (int b = 0; b < nb; ++b) {
        const int pn = __shfl_sync(0xffffffffu, nvb, b);
        const int prow = __shfl_sync(0xffffffffu, myrow, b);
        if (pn > 0 && pn < bt && prow >= 0) {
          const int per_head = pn * (D / 16);
          for (int i = lane; i < Hkv * per_head; i += 32) {
            const int h = i / per_head, rem = i % per_head;
            const int t = rem / (D / 16), c = rem % (D / 16);
            cp_async_16(stage + swizzled_offset(b * rpb + h * bt + t, 16 * c, D),
                        pool + (static_cast<size_t>(prow + t) * Hkv + h) * D + 16 * c);
          }
        }
      }
      cp_async_arrive_noinc(&sh.full[s]);
      if (!is_v) ++kq;
      ++pos;
      return true;
    };

    // tile stream: K(0,0), then per step the next K tile and the current V
    // tile; items are taken (and published) when the K side reaches them
    DecodeItem pf = next_item();
    int pf_rows[4];
    box_rows(pf, pf_rows);
    DecodeItem kI = pf;
    int kr[4] = {pf_rows[0], pf_rows[1], pf_rows[2], pf_rows[3]};
    bool ok = publish(0, kI, kr);
    int o_pub = 1;
    if (ok && kI.b >= 0) {
      pf = next_item();
      box_rows(pf, pf_rows);
      ok = emit(kI, kr, 0, false);
      int kj = 1, ko = 0;
      DecodeItem vI = kI;
      int vr[4] = {kr[0], kr[1], kr[2], kr[3]};
      int vj = 0, vo = 0;
      bool kdone = false;
      while (ok) {
        if (!kdone) {
          if (kj < htiles(kI, nt)) {
            ok = emit(kI, kr, kj, false);
            ++kj;
          } else {
            ok = publish(o_pub, pf, pf_rows);
            ++o_pub;
            if (pf.b < 0) {
              kdone = true;
            } else {
              kI = pf;
#pragma unroll
              for (int m = 0; m < 4; ++m) kr[m] = pf_rows[m];
              ++ko;
              pf = next_item();
              box_rows(pf, pf_rows);
              ok = ok && emit(kI, kr, 0, false);
              kj = 1;
            }
          }
        }
        if (!ok) break;
        ok = emit(vI, vr, vj, true);
        ++vj;
        if (vj == htiles(vI, nt)) {
          if (vo == ko) break;   // the K side found no further item
          vI = kI;
#pragma unroll
          for (int m = 0; m < 4; ++m) vr[m] = kr[m];
          vo = ko;
          vj = 0;
        }
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA
    if (lane == 0) {
      const uint32_t idesc_qk = make_idesc(kFmtE4M3, kFmtE4M3, 0, 0, 128, N);
      const uint32_t idesc_pv = make_idesc(kFmtE4M3, kFmtE4M3, 1, 0, 128, N);
      int pos = 0, st = 0, pt = 0;
      auto qk = [&](int o) -> bool {
        const int sb = st % kSBufs;
        const int s = pos % NS;
        if (!hwait(&sh.s_free[sb], ((st / kSBufs) & 1) ^ 1, sh, a.err) ||
            !hwait(&sh.full[s], (pos / NS) & 1, sh, a.err))
          return false;
        tc_fence_after_sync();
        const uint32_t tile = smem_u32(smem + s * C::kTileBytes);
        const uint32_t qt = smem_u32(sQT + (o & 1) * C::kQTermBytes);
#pragma unroll
        for (int kk = 0; kk < D / 32; ++kk) {
          const uint64_t da = make_smem_desc(tile + 32 * kk, 16, C::kSBO, C::kSwz);
          const uint64_t db = make_smem_desc(qt + 32 * kk, 16, C::kSBO, C::kSwz);
          tc_mma_f8(tmem + sb * kMaxN, da, db, idesc_qk, kk > 0);
        }
        tc_commit(&sh.empty[s]);
        tc_commit(&sh.s_full[sb]);
        ++pos;
        ++st;
        return true;
      };
      auto pv = [&](int o, int j) -> bool {
        const int pb = pt % kPBufs;
        const int s = pos % NS;
        if (!hwait(&sh.p_ready[pb], (pt / kPBufs) & 1, sh, a.err) ||
            !hwait(&sh.full[s], (pos / NS) & 1, sh, a.err))
          return false;
        tc_fence_after_sync();
        const uint32_t tile = smem_u32(smem + s * C::kTileBytes);
        const uint32_t ptile = smem_u32(sP + pb * C::kPTileBytes);
#pragma unroll
        for (int kk = 0; kk < kTile / 32; ++kk) {
          // MN-major A: V rows as stored; for D = 64 the upper half of M
          // re-reads the same atom (LBO 0) and is ignored
          const uint64_t da =
              make_smem_desc(tile + kk * 32 * D, D == 128 ? 16 * 1024 : 0, C::kSBO, C::kSwz);
          const uint64_t db = make_smem_desc(ptile + 32 * kk, 16, 1024, kSwizzle128B);
          tc_mma_f8(tmem + (kSBufs + (o & 1)) * kMaxN, da, db, idesc_pv,
                    (j > 0 || kk > 0) ? 1u : 0u);
        }
        tc_commit(&sh.empty[s]);
        tc_commit(&sh.p_free[pb]);
        ++pos;
        ++pt;
        return true;
      };
      // item o's descriptor (and the go-ahead for its QK: queries split)
      auto open_item = [&](int o, DecodeItem& it) -> bool {
        if (!hwait(&sh.desc_full[o & 1], (o >> 1) & 1, sh, a.err)) return false;
        it = sh.desc[o & 1];
        mbar_arrive(&sh.desc_free[o & 1]);
        if (it.b < 0) return false;
        return hwait(&sh.q_ready[o & 1], (o >> 1) & 1, sh, a.err);
      };
      DecodeItem kI;
      bool ok = open_item(0, kI) && qk(0);
      int ko = 0, kj = 1, kntl = htiles(kI, nt);
      int vo = 0, vj = 0, vntl = kntl;
      bool kdone = false;
      while (ok) {
        if (!kdone) {
          if (kj < kntl) {
            ok = qk(ko);
            ++kj;
          } else {
            DecodeItem nI;
            if (open_item(ko + 1, nI)) {
              ++ko;
              kntl = htiles(nI, nt);
              ok = qk(ko);
              kj = 1;
            } else {
              kdone = true;
            }
          }
        }
        if (!ok) break;
        if (vj == 0 && !hwait(&sh.o_free[vo & 1], ((vo >> 1) & 1) ^ 1, sh, a.err)) break;
        ok = pv(vo, vj);
        ++vj;
        if (ok && vj == vntl) {
          tc_commit(&sh.o_full[vo & 1]);
          if (vo == ko) break;
          vo = ko;
          vntl = kntl;
          vj = 0;
        }
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------- softmax / epilogue
    const int sw = warp & 3;
    const int tl = sw * 32 + lane;            // TMEM lane = tile row (S) = d (O)
    const uint32_t lane_base = static_cast<uint32_t>(sw * 32) << 16;
    const int rbox = tl / rpb, rrem = tl % rpb;
    const int my_h = rrem / bt;               // kv head of this row
    const int my_t = rbox * bt + rrem % bt;   // token offset of this row in its tile
    const int sidx = my_t * Hkv + my_h;       // [token][head] scale index within a tile
    const int w_h0 = ((sw * 32) % rpb) / bt;  // kv head of the warp's first row
    const int sel = my_h - w_h0;              // 0 or 1 (a warp spans at most 2 heads)
    const bool owner = rbox == 0 && (rrem % bt) == 0;   // one row per kv head
    int my_slots = 0;                         // 16-row slots holding my kv head
    for (int s16 = 0; s16 < 8; ++s16)
      if (((16 * s16) % rpb) / bt == my_h) my_slots |= 1 << s16;
    int st = 0, pt = 0, kq = 0, tpar = 0;

    // Take item o: wait for its descriptor, query rows and v-scales, agree on
    // whether to stop, split the queries into E4M3 terms, fix the probability
    // term scale of every query head from its kv head's largest v-scale.
    auto take = [&](int o, DecodeItem& it) -> bool {
      const int d = o & 1;
      const bool ok = hwait(&sh.desc_full[d], (o >> 1) & 1, sh, a.err);
      it = sh.desc[d];
      named_barrier(kBarSoftmax, kSoftmax);
      if (tl == 0) sh.stop = (!ok || it.b < 0 || *reinterpret_cast<volatile int*>(&sh.abort)) ? 1 : 0;
      named_barrier(kBarSoftmax, kSoftmax);
      if (sh.stop) return false;
      const uint16_t* qrow = reinterpret_cast<const uint16_t*>(sQRow + d * C::kQRowBytes);
      uint8_t* qt = sQT + d * C::kQTermBytes;
      const int th = kSoftmax / Hq;               // threads per query head (Hq <= 32)
      const int qh = tl / th;
      const int E = D / th;                       // elements per thread
      const int d0 = (tl % th) * E;
      float amax = 0.f;
      for (int e = 0; e < E; ++e) amax = fmaxf(amax, fabsf(bf16_bits_to_float(qrow[qh * D + d0 + e])));
      sh.redq[tl] = amax;
      // v-scale maximum of this thread's kv head (tl % Hkv) over the valid tokens
      const int ntl = htiles(it, nt);
      const float* vb = sVB + d * (kMaxTilesItem * kTile);
      float vmax = 0.f;
      for (int i = 0; i < ntl; ++i)
        if (it.t0 + i * nt + tl / Hkv < it.t1) vmax = fmaxf(vmax, vb[i * kTile + tl]);
      sh.vred[tl] = vmax;
      named_barrier(kBarSoftmax, kSoftmax);
      for (int i = 0; i < th; ++i) amax = fmaxf(amax, sh.redq[qh * th + i]);
      const float s1 = amax * (1.0f / 448.0f);
      const float inv1 = s1 > 0.f ? 1.0f / s1 : 0.f;
      if ((tl % th) == 0) sh.sig_q[d][qh] = s1;
      const int row0 = (qh / G) * kG3 + (qh % G);
      for (int e = 0; e < E; ++e) {
        uint8_t c1, c2, c3;
        hsplit3(bf16_bits_to_float(qrow[qh * D + d0 + e]), inv1, s1, c1, c2, c3);
        qt[swizzled_offset(row0, d0 + e, D)] = c1;
        qt[swizzled_offset(row0 + G, d0 + e, D)] = c2;
        qt[swizzled_offset(row0 + 2 * G, d0 + e, D)] = c3;
      }
      if (tl < Hkv) {
        float m = 0.f;
        for (int i = tl; i < kSoftmax; i += Hkv) m = fmaxf(m, sh.vred[i]);
        // probabilities are <= 2^8: P' = p * v_scale <= 2^8 * m = 448 * scale
        for (int g = 0; g < G; ++g) sh.sig_p[d][tl * G + g] = m * (256.0f / 448.0f);
      }
      fence_proxy_async_smem();
      named_barrier(kBarSoftmax, kSoftmax);   // scales visible to every softmax warp
      mbar_arrive(&sh.q_ready[d]);
      return true;
    };

    DecodeItem cur;
    bool have = take(0, cur);
    for (int o = 0; have; ++o) {
      const int d = o & 1;
      const int ntl = htiles(cur, nt);
      const float sp = sh.sig_p[d][my_h * G];
      const float spinv = sp > 0.f ? 1.0f / sp : 0.f;
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
        tc_fence_after_sync();
        uint32_t r[48];
#pragma unroll
        for (int c = 0; c < 3; ++c) {
          if (c * 16 < 2 * kG3) {
            uint32_t part[16];
            tmem_ld16(tmem + lane_base + sb * kMaxN + w_h0 * kG3 + 16 * c, part);
#pragma unroll
            for (int i = 0; i < 16; ++i) r[16 * c + i] = part[i];
          }
        }
        tmem_ld_wait();
        tc_fence_before_sync();
        mbar_arrive(&sh.s_free[sb]);
        ++st;
        const float ks = sKS[(kq % kKSlots) * kTile + sidx];
        mbar_arrive(&sh.kslot_free[kq % kKSlots]);
        ++kq;
        const bool valid = cur.t0 + j * nt + my_t < cur.t1;
        const float vs = valid ? sVB[d * (kMaxTilesItem * kTile) + j * kTile + sidx] : 0.f;
        const float f = a.sm_scale_log2 * ks;
        float l[G];
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float v0 = __uint_as_float(sel ? r[kG3 + g] : r[g]);
          const float v1 = __uint_as_float(sel ? r[kG3 + G + g] : r[G + g]);
          const float v2 = __uint_as_float(sel ? r[kG3 + 2 * G + g] : r[2 * G + g]);
          const float sdot = v0 + v1 * (1.0f / 16.0f) + v2 * (1.0f / 256.0f);
          l[g] = valid ? f * sh.sig_q[d][my_h * G + g] * sdot : -INFINITY;
        }
        // ---- running maximum per query head (moved only by more than 2^8)
#pragma unroll
        for (int g = 0; g < G; ++g) {
          float x = l[g];
#pragma unroll
          for (int off = 1; off < 16; off <<= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, off));
          if ((lane & 15) == 0) sh.red[tpar][tl >> 4][g] = x;
        }
        named_barrier(kBarSoftmax, kSoftmax);
        bool need = false;
        float fac[G];
#pragma unroll
        for (int g = 0; g < G; ++g) {
          float tmax = -INFINITY;
          for (int s16 = 0; s16 < 8; ++s16)
            if ((my_slots >> s16) & 1) tmax = fmaxf(tmax, sh.red[tpar][s16][g]);
          fac[g] = 1.f;
          if (tmax > m_run[g] + kRescaleLog2) {
            if (m_run[g] > -INFINITY) {
              need = true;
              fac[g] = exp2f(m_run[g] - tmax);
            }
            m_run[g] = tmax;
          }
        }
        tpar ^= 1;
        const bool any = named_barrier_or(kBarSoftmax, kSoftmax, need);
        float p[G];
#pragma unroll
        for (int g = 0; g < G; ++g) {
          p[g] = valid ? exp2f(l[g] - m_run[g]) : 0.f;
          lpart[g] = lpart[g] * fac[g] + p[g];
        }
        if (any) {
          // rare: a head's reference maximum moved; rescale its O columns
          if (owner) {
#pragma unroll
            for (int g = 0; g < G; ++g) sh.factor[my_h * G + g] = fac[g];
          }
          named_barrier(kBarSoftmax, kSoftmax);
          hwait(&sh.p_free[(pt - 1) % kPBufs], ((pt - 1) / kPBufs) & 1, sh, a.err);
          tc_fence_after_sync();
          constexpr int kHC = kG3 <= 16 ? 16 : 32;
          for (int h = 0; h < Hkv; ++h) {
#pragma unroll
            for (int c = 0; c < kHC / 16; ++c) {
              uint32_t part[16];
              const uint32_t addr = tmem + lane_base + (kSBufs + d) * kMaxN + h * kG3 + 16 * c;
              tmem_ld16(addr, part);
              tmem_ld_wait();
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                const int col = 16 * c + i;
                if (col < kG3)
                  part[i] = __float_as_uint(__uint_as_float(part[i]) * sh.factor[h * G + col % G]);
              }
              tmem_st16(addr, part);
              tmem_st_wait();   // the next load overlaps these columns
            }
          }
          tc_fence_before_sync();
        }
        // ---- probabilities times v-scale -> block-diagonal P^T (3 terms)
        const int pb = pt % kPBufs;
        hwait(&sh.p_free[pb], ((pt / kPBufs) & 1) ^ 1, sh, a.err);
        uint8_t* dst = sP + pb * C::kPTileBytes;
#pragma unroll
        for (int g = 0; g < G; ++g) {
          uint8_t c1, c2, c3;
          hsplit3(p[g] * vs, spinv, sp, c1, c2, c3);
          const int n0 = my_h * kG3 + g;
          dst[swizzled_offset(n0, tl, 128)] = c1;
          dst[swizzled_offset(n0 + G, tl, 128)] = c2;
          dst[swizzled_offset(n0 + 2 * G, tl, 128)] = c3;
        }
        fence_proxy_async_smem();
        mbar_arrive(&sh.p_ready[pb]);
        ++pt;
      }
      // ---- softmax denominators and reference maxima of the item
#pragma unroll
      for (int g = 0; g < G; ++g) {
        float x = lpart[g];
#pragma unroll
        for (int off = 1; off < 16; off <<= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
        if ((lane & 15) == 0) sh.redl[tl >> 4][g] = x;
      }
      named_barrier(kBarSoftmax, kSoftmax);
      if (owner) {
#pragma unroll
        for (int g = 0; g < G; ++g) {
          float sum = 0.f;
          for (int s16 = 0; s16 < 8; ++s16)
            if ((my_slots >> s16) & 1) sum += sh.redl[s16][g];
          sh.lsum[d][my_h * G + g] = sum;
          sh.m2[d][my_h * G + g] = m_run[g];
        }
      }
      named_barrier(kBarSoftmax, kSoftmax);
      mbar_arrive(&sh.desc_free[d]);   // done with this item's query rows and v-scales
      // ---- the next item's queries go out before this item's epilogue
      DecodeItem nxt;
      const bool more = take(o + 1, nxt);
      // ---- epilogue: O^T columns -> fp32 partial output and lse
      hwait(&sh.o_full[d], (o >> 1) & 1, sh, a.err);
      tc_fence_after_sync();
      constexpr int kHC = kG3 <= 16 ? 16 : 32;
      for (int h = 0; h < Hkv; ++h) {
        uint32_t ov[kHC];
#pragma unroll
        for (int c = 0; c < kHC / 16; ++c) {
          uint32_t part[16];
          tmem_ld16(tmem + lane_base + (kSBufs + d) * kMaxN + h * kG3 + 16 * c, part);
#pragma unroll
          for (int i = 0; i < 16; ++i) ov[16 * c + i] = part[i];
        }
        tmem_ld_wait();
        if (tl < D) {
#pragma unroll
          for (int g = 0; g < G; ++g) {
            const int qh = h * G + g;
            const float sdot = __uint_as_float(ov[g]) + __uint_as_float(ov[G + g]) * (1.0f / 16.0f) +
                               __uint_as_float(ov[2 * G + g]) * (1.0f / 256.0f);
            const float lsum = sh.lsum[d][qh];
            const float out = lsum > 0.f ? sdot * sh.sig_p[d][qh] / lsum : 0.f;
            a.part_o[(static_cast<size_t>(cur.slot) * Hq + qh) * D + tl] = out;
          }
        }
      }
      tc_fence_before_sync();
      mbar_arrive(&sh.o_free[d]);
      if (tl < Hq) {
        const float lsum = sh.lsum[d][tl];
        a.part_lse[static_cast<size_t>(cur.slot) * Hq + tl] =
            lsum > 0.f ? (sh.m2[d][tl] + log2f(lsum)) * kLn2 : -INFINITY;
      }
      cur = nxt;
      have = more;
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
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
                           cudaStream_t stream) {
  using C = HCfg<D, G>;
  auto* kern = decode_heads_kernel<D, G>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int grid = a.num_items < sms ? a.num_items : sms;
  kern<<<grid, kThreads, C::kSmem, stream>>>(km, vm, a);
  return cudaGetLastError();
}

}  // namespace
bool heads_geometry(int Hq, int Hkv, int D, int page_size, int* nt, int* bt, int* nb,
                    int* max_tiles) {
  if (Hkv != 1 && Hkv != 2 && Hkv != 4 && Hkv != 8) return false;
  if (Hq % Hkv != 0 || 3 * Hq > kMaxN) return false;
  const int G = Hq / Hkv;
  if (G != 1 && G != 2 && G != 4 && G != 8) return false;
  if (D != 64 && D != 128) return false;
  if (Hq * D < kTile) return false;   // the query split gives every thread >= 1 element
  const int t = kTile / Hkv;
  if (page_size % 16 != 0) return false;
  if (!(page_size % t == 0 || t % page_size == 0)) return false;
  *nt = t;
  *bt = page_size < t ? page_size : t;
  *nb = t / *bt;
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
  // pool viewed as (d, token row, kv head): boxes come out head-major in smem
  CUtensorMap km, vm;
  const uint64_t dims[3] = {static_cast<uint64_t>(D), static_cast<uint64_t>(num_pages) * page_size,
                            static_cast<uint64_t>(Hkv)};
  const uint64_t strides[2] = {static_cast<uint64_t>(Hkv) * D, static_cast<uint64_t>(D)};
  const uint32_t box[3] = {static_cast<uint32_t>(D), static_cast<uint32_t>(bt),
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
  a.bt = bt;
  a.nb = nb;
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
  if (D == DD && G == GG) return launch_heads_t<DD, GG>(km, vm, a, stream);
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
