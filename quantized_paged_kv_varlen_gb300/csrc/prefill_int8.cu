// Varlen causal prefill over a paged cache: INT8 Q and K with one fp32 scale
// per (sequence, 128-token block, head), bf16 V ("[Feature] Sage Attention
// Support Varlen & write kv cache BF16/FP16", Description items 1-3;
// "KvQuantSparseFlashAttention" README, 计算公式 and 参数说明 rows
// actual_seq_lengths_query / actual_seq_lengths_kv / block_table /
// sparse_mode = 3):
//   logit(i, j) = scale * sq[b, i/128, h] * sk[b, j/128, hk] * (q8_i . k8_j)
//   O_i = sum_j softmax_j(logit(i, .)) V_j,   lse_i = logsumexp_j logit(i, j)
// Query i (0-based in its sequence) sees key j iff j < L_kv and, when
// causal, j <= i + L_kv - L_q (bottom-right aligned).
//
// The integer dot products are exact.  Q codes enter the f16 MMA as they
// are; K codes enter biased by 128 as f16 subnormals (x + 128) * 2^-24, so
// every partial sum is an integer below 2^22 times 2^-24 and the fp32
// accumulator holds S' = 2^-24 (q8 . k8 + 128 sum_d q8_d) exactly.  The
// softmax removes the row constant 128 sum_d q8_d inside the same fused
// multiply-add that applies the scales: the two block scales and the
// softmax scale multiply the logits of a tile at once (q and key tiles are
// aligned to the 128-token blocks).
//
// One persistent CTA per SM, 12 warps:
//   warps 0, 11  convert every staged int8 tile (per work item its 128-row
//              Q tile, then each key tile) into the f16 K-major SW128
//              operand layout, one 64-column half each; lane 0 of warp 0
//              issues the int8 Q and K copies (K rows of the pages a key
//              tile spans; pages past L_kv read as zeros) up to three steps
//              ahead, with the page ids fetched two tiles earlier into a
//              shared ring (IdRing)
//   warp 1     QK MMAs  S[128 q x 128 k] = Q16 . K16^T        (kind::f16)
//   warp 10    PV MMAs  O[128 q x 128 d] += P . V, and the V copies (one
//              box per page and 64-column half for bf16 V, one per page
//              for E4M3 V), one key tile ahead.  kind::f16 with P read from
//              tensor memory, where the softmax wrote it over columns
//              [0, 32) and [64, 96) of its S buffer: bf16 P against bf16 V,
//              or (the V8 instantiation, E4M3 V) f16 P against V widened
//              in place from E4M3 to f16 (exact) by this warp, with the
//              per-channel V scales applied in the epilogue
//   warps 2-9  online softmax, two threads per query row (columns [0, 64)
//              on warps 2-5, [64, 128) on warps 6-9), lazy maximum (moves
//              only by more than 2^8, then O is rescaled), and the epilogue
//              O / l -> bf16 plus the lse.
// The copy-issuing lanes do no integer division by the runtime page size
// and no error reporting: both slowed the whole pipeline (a division runs
// through the MUFU pipe the softmax keeps busy); bad page ids are flagged
// by the prep pass and read as zeros.
// TMEM: three S buffers and O (512 columns).
//
// Work: a unit is the pair of q tiles (t, n-1-t) of one (sequence, head).
// A one-block prep pass sorts the sequences by the cost of their units
// (longest first) and writes the unit table to the caller's workspace; the
// CTAs take units round-robin.  The same pass writes O = 0 and lse = -inf
// for q tiles no key is visible to.
#include <cmath>

#include "common.cuh"
#include "internal.h"

namespace qpkv {
namespace {

constexpr int kT = 128;                 // q rows per tile = keys per tile
constexpr int kD = 128;                 // head dim
constexpr int kThreads = 384;           // 12 warps
constexpr int kWarpLoad = 0, kWarpQk = 1, kWarpPv = 10, kWarpConv = 11;
constexpr int kSoftmax = 256;           // two threads per query row
constexpr int kK8Stages = 4;            // staged int8 Q / K tiles
constexpr int kK16Bufs = 2;             // converted K tiles
constexpr int kVStages = 2;             // V tiles (bf16, or E4M3 in the first half)
constexpr int kI8Tile = kT * kD;        // 16 KB
constexpr int kH16Tile = 2 * kT * kD;   // 32 KB: two 64-column halves
constexpr int kHalf = kT * 128;         // 16 KB, one half (128 rows of 128 bytes)
constexpr int kOffQ16 = 0;
constexpr int kOffK8 = kOffQ16 + kH16Tile;
constexpr int kOffK16 = kOffK8 + kK8Stages * kI8Tile;
constexpr int kOffV = kOffK16 + kK16Bufs * kH16Tile;
constexpr int kSmem = kOffV + kVStages * kH16Tile + 1024;
constexpr float kRescaleLog2 = 8.0f;
constexpr int kSBufs = 3;
constexpr uint32_t kColS = 0;           // S buffers: columns [0, 384)
constexpr uint32_t kColO = 384;         // O: columns [384, 512)

struct PArgs {
  int B, T, Hq, Hkv, G, ps, P, bt_stride, NB, causal;
  int ragged, T_kv;     // ragged K/V: rows [T_kv, Hkv, D] addressed from the unit record
  int rows_box, nbox;   // page rows per TMA box, boxes per 128-key tile
  // key tile j, box i -> block_table entry and row offset in the page, with
  // no division on the device (an integer division by a runtime value runs
  // through the MUFU pipe, which the softmax keeps busy):
  //   page_size <= 128: entry j * nbox + i, offset 0;
  //   page_size = 128 m, m > 1: entry j / m = umulhi(j, m_magic), offset
  //   (j - entry * m) * 128, m_magic = ceil(2^32 / m) (exact while j * m < 2^32)
  int m;
  unsigned m_magic;
  float scale_log2;     // softmax scale * log2(e)
  const int32_t* cu_q;  // [B] inclusive prefix sums
  const int32_t* lk;    // [B]
  const int32_t* bt;    // [B, bt_stride]
  const int8_t* q8;     // [T, Hq, D]
  const float* sv;      // FP8 V: channel scales [B, Hkv, D]
  const float* sq;      // [B, NB, Hq]
  const float* sk;      // [B, NB, Hkv]
  uint16_t* o;          // bf16 [T, Hq, D]
  float* lse;           // [T, Hq] or null
  const int32_t* ws;    // unit table: [0] units, then 4 ints per sorted sequence
  int* err;
};

// Unit-table entry of the k-th sequence in cost order.
enum : int { kWsSeq = 0, kWsCum = 1, kWsQtLo = 2, kWsNq = 3, kWsStride = 4 };

struct Shared {
  uint64_t k8_full[kK8Stages], k8_empty[kK8Stages];
  uint64_t q16_full, q16_free;
  uint64_t k16_full[kK16Bufs], k16_empty[kK16Bufs];
  uint64_t v_full[kVStages], v_empty[kVStages];
  uint64_t s_full[kSBufs], p_ready[kSBufs], pv_done[kSBufs];
  uint64_t o_full, o_free;
  uint64_t mma_done[2];
  float pair[2][kT];      // [column half][row]: a row's partial maxima / sums
  uint32_t tmem_base;
  int abort;
  int kring[6], vring[6];   // IdRing slots of the K and V copy issuers
};

// Bounded mbarrier wait: the first probe is inline, the polling loop is one
// shared out-of-line copy (the kernel's many wait sites otherwise crowd the
// instruction cache).
__device__ __noinline__ bool awaitb_slow(uint64_t* bar, uint32_t parity, Shared& sh, int* err) {
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

__device__ __forceinline__ bool awaitb(uint64_t* bar, uint32_t parity, Shared& sh, int* err) {
  return mbar_try_wait(bar, parity) || awaitb_slow(bar, parity, sh, err);
}

__device__ __noinline__ void drain(uint64_t* bar, uint32_t parity, int* err) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > kWaitTimeoutCycles) {
      report_error(err, kDevErrTimeout);
      return;
    }
  }
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// K/V tiles a q tile needs: keys [0, last] with last the final key any of
// its rows (i < L_q) sees.
__host__ __device__ __forceinline__ int kv_tiles_of(int Lq, int Lk, int qt, int causal) {
  int last = Lk - 1;
  if (causal) {
    const int row = qt * kT + kT - 1 < Lq - 1 ? qt * kT + kT - 1 : Lq - 1;
    last = last < row + Lk - Lq ? last : row + Lk - Lq;
  }
  return last < 0 ? 0 : last / kT + 1;
}

// First q tile with a visible key, and the q tile count of a sequence.
__device__ __forceinline__ void q_tile_range(int Lq, int Lk, int causal, int& qt_lo, int& nqt) {
  nqt = (Lq + kT - 1) / kT;
  if (Lk <= 0)
    qt_lo = nqt;
  else if (causal && Lq > Lk)
    qt_lo = min((Lq - Lk) / kT, nqt);
  else
    qt_lo = 0;
}

struct Tile {
  int b, h, hk, qt, begin, Lq, Lk, nkv;   // hk = h / (Hq / Hkv)
  int kvb;   // ragged K/V: the sequence's first row
};

// Workspace: int32 [0] unit count, [1, 1 + 4B) the sequences in cost order
// (kWs* fields), [1 + 4B, 1 + 5B) their costs; from byte offset
// units_offset(B) one 32-byte record per unit in that order:
//   {b, h | kv head << 16, qt_a, qt_b (-1 when the unit has one q tile),
//    begin, Lq, Lk, first K/V row (ragged K/V; 0 for a paged cache)}.
__host__ __device__ __forceinline__ size_t units_offset(int B) {
  return ((static_cast<size_t>(1 + (kWsStride + 1) * static_cast<size_t>(B)) * 4 + 15) / 16) * 16;
}

// This CTA's work items: units blockIdx.x, +grid, ... of the record list;
// each unit gives q tiles qt_a and then qt_b.  Moving to the next unit only
// issues the load of its record; the value is first used at the next
// get(), one item later, so no role waits on it at an item change.
struct Items {
  int unit, second, total;
  int4 r0, r1;   // the record of this unit (or, after advance(), its successor)
  const int4* recs;
  __device__ __forceinline__ void start(const PArgs& a) {
    recs = reinterpret_cast<const int4*>(reinterpret_cast<const uint8_t*>(a.ws) + units_offset(a.B));
    total = a.ws[0];
    unit = static_cast<int>(blockIdx.x);
    second = 0;
    load();
  }
  __device__ __forceinline__ void load() {
    if (unit < total) {
      r0 = recs[2 * unit];
      r1 = recs[2 * unit + 1];
    }
  }
  __device__ __forceinline__ bool valid() const { return unit < total; }
  __device__ __forceinline__ void get(const PArgs& a, Tile& t) const {
    t.b = r0.x;
    t.h = r0.y & 0xFFFF;
    t.hk = r0.y >> 16;
    t.qt = second ? r0.w : r0.z;
    t.begin = r1.x;
    t.Lq = r1.y;
    t.Lk = r1.z;
    t.kvb = r1.w;
    t.nkv = kv_tiles_of(t.Lq, t.Lk, t.qt, a.causal);
  }
  __device__ __forceinline__ void advance() {
    if (!second && r0.w >= 0) {
      second = 1;
    } else {
      second = 0;
      unit += static_cast<int>(gridDim.x);
      load();
    }
  }
};

// Conversion of one 64-column half of an int8 tile (128 rows of 128 codes,
// SW128 as TMA wrote it) into the f16 K-major SW128 operand (half `part`
// holds operand columns [64 part, 64 part + 64)).  Both operands place the
// codes of a 4-byte group (d0 d1 d2 d3) as the f16 pairs (d0, d2), (d1, d3):
// the same order on both sides, so the dot products are unchanged.
//   Q (exact):  f16 bits 0x6400 | (x ^ 0x80) = 1152 + x, minus 1152.
//   K (biased): f16 bits (x ^ 0x80) = (x + 128) * 2^-24, a subnormal; then
//               S' = 2^-24 (q . k + 128 sum_d q_d), all integers below 2^22,
//               and the softmax takes the row constant 128 sum_d q_d back out.
// Lane (r7, cq) takes rows 8g + r7 and source chunk 4 part + cq, so the
// eight lanes of a quarter-warp touch eight distinct 16-byte bank groups on
// both sides; for K four rows are loaded before any is stored.
template <bool kIsQ>
__device__ __forceinline__ void convert_half(const uint8_t* src, uint8_t* dst, int lane, int part) {
  const int r7 = lane & 7, c = 4 * part + (lane >> 3);
  const uint8_t* s0 = src + r7 * 128 + ((c ^ r7) << 4);
  uint8_t* d0 = dst + part * kHalf + r7 * 128;
  const int g0 = 2 * (c & 3);
  const int o0 = (g0 ^ r7) << 4, o1 = ((g0 + 1) ^ r7) << 4;
  constexpr int kBatch = kIsQ ? 1 : 4;   // Q: once per work item, kept small
#pragma unroll 1
  for (int g = 0; g < 16; g += kBatch) {
    uint4 w[kBatch];
#pragma unroll
    for (int i = 0; i < kBatch; ++i) w[i] = *reinterpret_cast<const uint4*>(s0 + (g + i) * 1024);
#pragma unroll
    for (int i = 0; i < kBatch; ++i) {
      const uint32_t ws[4] = {w[i].x ^ 0x80808080u, w[i].y ^ 0x80808080u, w[i].z ^ 0x80808080u,
                              w[i].w ^ 0x80808080u};
      uint32_t h[8];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        if (kIsQ) {
          h[2 * k] = f16x2_sub(prmt(ws[k], 0x64646464u, 0x4240u), 0x64806480u);
          h[2 * k + 1] = f16x2_sub(prmt(ws[k], 0x64646464u, 0x4341u), 0x64806480u);
        } else {
          h[2 * k] = ws[k] & 0x00FF00FFu;
          h[2 * k + 1] = (ws[k] >> 8) & 0x00FF00FFu;
        }
      }
      uint8_t* d = d0 + (g + i) * 1024;
      *reinterpret_cast<uint4*>(d + o0) = make_uint4(h[0], h[1], h[2], h[3]);
      *reinterpret_cast<uint4*>(d + o1) = make_uint4(h[4], h[5], h[6], h[7]);
    }
  }
}

// Page ids of the first two TMA boxes of key tiles j, j + 1, j + 2 of one
// walk, in a 3-slot shared-memory ring filled by 4-byte cp.async copies two
// tiles before the tile is issued, so issuing a copy never waits on a
// block_table load.  One walk per issuing thread; each fetch() closes one
// cp.async group, and a fetch is issued for every position after the first
// two of a work item, so when position j is issued only the group of j + 1
// can still be in flight.  Boxes 2..7 (pages shorter than 64 rows) are read
// directly when the tile is issued.
__device__ __forceinline__ int bt_entry(const PArgs& a, int j, int i) {
  return a.m == 1 ? j * a.nbox + i : static_cast<int>(__umulhi(static_cast<unsigned>(j), a.m_magic));
}
__device__ __forceinline__ int page_offset(const PArgs& a, int j, int e) {
  return a.m == 1 ? 0 : (j - e * a.m) * kT;
}

struct IdRing {
  int* slot;   // shared [3][2]
  __device__ __forceinline__ void fetch(const PArgs& a, const Tile& t, int j) const {
    if (!a.ragged && j < t.nkv) {
      const int32_t* row = a.bt + static_cast<size_t>(t.b) * a.bt_stride;
      const int nb = a.nbox < 2 ? a.nbox : 2;
      for (int i = 0; i < nb; ++i) {
        const int key0 = j * kT + i * a.rows_box;
        if (key0 < t.Lk) cp_async_4(slot + 2 * (j % 3) + i, row + bt_entry(a, j, i));
      }
    }
    cp_async_commit();
  }
  // the walk moved to position j of its current item (j == first: just opened)
  __device__ __forceinline__ void advanced(const PArgs& a, const Tile& t, int j, int first) const {
    if (j == first) {
      fetch(a, t, 0);
      fetch(a, t, 1);
    } else if (j >= 1) {
      fetch(a, t, j + 1);
    }
  }
};

// A walk over this CTA's work items one tile at a time: per item its q
// tile (j = -1, when with_q) and then its key tiles j = 0 .. nkv - 1.
struct TileWalk {
  Items it;
  Tile t;
  int j;
  bool live, with_q;
  __device__ __forceinline__ void start(const PArgs& a, bool q) {
    with_q = q;
    it.start(a);
    open(a);
  }
  __device__ __forceinline__ void open(const PArgs& a) {
    live = it.valid();
    if (live) {
      it.get(a, t);
      it.advance();
    }
    j = with_q ? -1 : 0;
  }
  __device__ __forceinline__ void next(const PArgs& a) {
    if (++j >= t.nkv) open(a);
  }
};

// V8: V is E4M3 with per-(sequence, head, channel) scales, widened to f16
// in shared memory, and P is f16; else V is bf16 and P bf16.
template <bool V8>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_int8_kernel(const __grid_constant__ CUtensorMap q_map,
                        const __grid_constant__ CUtensorMap k_map,
                        const __grid_constant__ CUtensorMap v_map, const PArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  __shared__ Shared sh;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    for (int s = 0; s < kK8Stages; ++s) {
      mbar_init(&sh.k8_full[s], 1);
      mbar_init(&sh.k8_empty[s], 64);
    }
    mbar_init(&sh.q16_full, 64);
    mbar_init(&sh.q16_free, 1);
    for (int s = 0; s < kK16Bufs; ++s) {
      mbar_init(&sh.k16_full[s], 64);
      mbar_init(&sh.k16_empty[s], 1);
    }
    for (int s = 0; s < kVStages; ++s) {
      mbar_init(&sh.v_full[s], 1);
      mbar_init(&sh.v_empty[s], 1);
    }
    for (int b = 0; b < kSBufs; ++b) {
      mbar_init(&sh.s_full[b], 1);
      mbar_init(&sh.p_ready[b], kSoftmax);
      mbar_init(&sh.pv_done[b], 1);
    }
    mbar_init(&sh.o_full, 1);
    mbar_init(&sh.o_free, kSoftmax);
    mbar_init(&sh.mma_done[0], 1);
    mbar_init(&sh.mma_done[1], 1);
    sh.abort = 0;
    fence_mbar_init();
  }
  if (warp == kWarpQk) tmem_alloc(&sh.tmem_base, 512);
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = sh.tmem_base;

  // pool row of box i of key tile j; keys past L_kv and bad page ids read
  // rows past the pool's end, which the copy fills with zeros
  const int oob = a.ragged ? a.T_kv : a.P * a.ps;
  // (paged: after cp_async_wait_but_one(), the ring holds tile j's ids)
  auto page_row = [&](const Tile& t, const int* ring, int i, int j) -> int {
    const int key0 = j * kT + i * a.rows_box;
    if (key0 >= t.Lk) return oob;
    if (a.ragged) return t.kvb + key0;
    const int e = bt_entry(a, j, i);
    const int id = i < 2 ? ring[2 * (j % 3) + i]
                         : __ldg(a.bt + static_cast<size_t>(t.b) * a.bt_stride + e);
    // an entry outside the pool reads zeros (the prep pass flags it)
    if (static_cast<unsigned>(id) >= static_cast<unsigned>(a.P)) return oob;
    return id * a.ps + page_offset(a, j, e);
  };

  if (warp == kWarpLoad || warp == kWarpConv) {
    // ----------------------------------- Q / K copies and int8 -> f16
    // Both warps walk the q / key tiles of the work items in order (per
    // item its Q tile, then its key tiles) and convert one 64-column half
    // each.  Lane 0 of warp 0 also issues the int8 copies, up to three
    // steps ahead of the step being converted; its only wait is for a
    // stage both warps have finished with, which needs no later step here.
    const int part = warp == kWarpLoad ? 0 : 1;
    const bool issuer = part == 0 && lane == 0;
    TileWalk cv, ld;
    const IdRing kr{sh.kring};
    cv.start(a, true);
    int kpos = 0, ipos = 0, c16 = 0;
    if (issuer) {
      tma_prefetch_desc(&q_map);
      tma_prefetch_desc(&k_map);
      ld.start(a, true);
      if (ld.live) kr.advanced(a, ld.t, ld.j, -1);
    }
    auto issue = [&](int upto) -> bool {
      while (ld.live && ipos <= upto) {
        const int s = ipos % kK8Stages;
        if (!awaitb(&sh.k8_empty[s], ((ipos / kK8Stages) & 1) ^ 1, sh, a.err)) return false;
        mbar_arrive_expect_tx(&sh.k8_full[s], kI8Tile);
        uint8_t* dst = smem + kOffK8 + s * kI8Tile;
        const Tile& t = ld.t;
        if (ld.j < 0) {
          tma_load_3d(dst, &q_map, &sh.k8_full[s], 0, t.h, t.begin + t.qt * kT);
        } else {
          cp_async_wait_but_one();
#pragma unroll 1
          for (int i = 0; i < a.nbox; ++i)
            tma_load_3d(dst + i * a.rows_box * 128, &k_map, &sh.k8_full[s], 0, t.hk,
                        page_row(ld.t, sh.kring, i, ld.j));
        }
        ++ipos;
        ld.next(a);
        if (ld.live) kr.advanced(a, ld.t, ld.j, -1);
      }
      return true;
    };
    for (int o = 0; cv.live; cv.next(a)) {
      bool ok = true;
      if (issuer) ok = issue(kpos + kK8Stages - 1);
      if (__shfl_sync(0xffffffffu, ok ? 1 : 0, 0) == 0) break;
      const bool is_q = cv.j < 0;
      const int s = kpos % kK8Stages, d = c16 % kK16Bufs;
      bool w = is_q ? awaitb(&sh.q16_free, (o & 1) ^ 1, sh, a.err)
                    : awaitb(&sh.k16_empty[d], ((c16 / kK16Bufs) & 1) ^ 1, sh, a.err);
      w = w && awaitb(&sh.k8_full[s], (kpos / kK8Stages) & 1, sh, a.err);
      if (!__all_sync(0xffffffffu, w)) break;
      const uint8_t* src = smem + kOffK8 + s * kI8Tile;
      if (is_q)
        convert_half<true>(src, smem + kOffQ16, lane, part);
      else
        convert_half<false>(src, smem + kOffK16 + d * kH16Tile, lane, part);
      fence_proxy_async_smem();   // generic writes -> tensor-core reads
      mbar_arrive(is_q ? &sh.q16_full : &sh.k16_full[d]);
      mbar_arrive(&sh.k8_empty[s]);
      ++kpos;
      if (is_q) {
        ++o;
      } else {
        ++c16;
      }
    }
    if (issuer) {
      cp_async_wait_all();
      for (int i = ipos > kK8Stages ? ipos - kK8Stages : 0; i < ipos; ++i)
        drain(&sh.k8_full[i % kK8Stages], (i / kK8Stages) & 1, a.err);
    }
    __syncwarp();
  } else if (warp == kWarpQk) {
    // ------------------------------------------------------------ QK MMA
    if (lane == 0) {
      const uint32_t idesc_qk = make_idesc(kFmtF16, kFmtF16, 0, 0, kT, kT);
      // K-major operands advance 32 bytes per K = 16 step inside a 128-byte
      // row and switch to the second 64-column half after four steps
      const uint64_t qdesc = make_smem_desc(smem_u32(smem + kOffQ16), 16, 1024, kSwizzle128B);
      const uint64_t kdesc0 = make_smem_desc(smem_u32(smem + kOffK16), 16, 1024, kSwizzle128B);
      Items it;
      it.start(a);
      int c16 = 0, st = 0;
      bool ok = true;
      for (int o = 0; ok && it.valid(); ++o) {
        Tile t;
        it.get(a, t);
        it.advance();
        if (!awaitb(&sh.q16_full, o & 1, sh, a.err)) break;
        for (int j = 0; j < t.nkv; ++j) {
          const int sb = st % kSBufs, d = c16 % kK16Bufs;
          // QK(st) overwrites the S buffer that held P(st - 3)
          ok = st < kSBufs || awaitb(&sh.pv_done[sb], ((st - kSBufs) / kSBufs) & 1, sh, a.err);
          ok = ok && awaitb(&sh.k16_full[d], (c16 / kK16Bufs) & 1, sh, a.err);
          if (!ok) break;
          tc_fence_after_sync();
          const uint64_t db = kdesc0 + static_cast<uint64_t>((d * kH16Tile) >> 4);
#pragma unroll
          for (int kk = 0; kk < kD / 16; ++kk) {
            const uint32_t off = (kk >> 2) * kHalf + (kk & 3) * 32;
            tc_mma_f16(tmem + kColS + sb * kT, qdesc + (off >> 4), db + (off >> 4), idesc_qk,
                       kk > 0 ? 1u : 0u);
          }
          tc_commit(&sh.k16_empty[d]);
          tc_commit(&sh.s_full[sb]);
          if (j == t.nkv - 1) tc_commit(&sh.q16_free);
          ++c16;
          ++st;
        }
      }
      tc_commit(&sh.mma_done[0]);
      drain(&sh.mma_done[0], 0, a.err);
    }
    __syncwarp();
  } else if (warp == kWarpPv) {
    // ------------------------------------------------------------ PV MMA
    // Lane 0 also issues the V copies: V(t + 1) once PV(t - 1) has
    // completed (two stages), before waiting for P(t).  The whole warp
    // waits; rows of a V tile past L_kv (the unwritten rest of a sequence's
    // last page, whose bits may be NaN) are zeroed first, since P = 0 there
    // does not cancel a NaN.  Lane 0 issues the MMAs.
    const uint32_t idesc_pv = V8 ? make_idesc(kFmtF16, kFmtF16, 0, 1, kT, kD)
                                 : make_idesc(kFmtBF16, kFmtBF16, 0, 1, kT, kD);
    // MN-major 16-bit V: two 64-column atoms 16 KB apart (leading byte
    // offset), 16 key rows (2 KB) per K = 16 step
    const uint64_t vdesc0 = make_smem_desc(smem_u32(smem + kOffV), kHalf, 1024, kSwizzle128B);
    Items it;
    it.start(a);
    TileWalk vw;
    const IdRing vr{sh.vring};
    int vpos = 0, pvc = 0, vis = 0;
    if (lane == 0) {
      tma_prefetch_desc(&v_map);
      vw.start(a, false);
      if (vw.live) vr.advanced(a, vw.t, vw.j, 0);
    }
    // lane 0: issue the V copies of tiles up to `upto`, waiting for a free
    // stage only when `block`; false on abort
    auto issue_v = [&](int upto, bool block) -> bool {
      while (vw.live && vis <= upto) {
        const int s = vis % kVStages;
        const uint32_t par = ((vis / kVStages) & 1) ^ 1;
        if (block) {
          if (!awaitb(&sh.v_empty[s], par, sh, a.err)) return false;
        } else if (!mbar_test_wait(&sh.v_empty[s], par)) {
          return true;
        }
        mbar_arrive_expect_tx(&sh.v_full[s], V8 ? kI8Tile : kH16Tile);
        const Tile& t = vw.t;
        cp_async_wait_but_one();
#pragma unroll 1
        for (int i = 0; i < a.nbox; ++i) {
          const int row = page_row(vw.t, sh.vring, i, vw.j);
          uint8_t* dst = smem + kOffV + s * kH16Tile + i * a.rows_box * 128;
          tma_load_3d(dst, &v_map, &sh.v_full[s], 0, t.hk, row);
          if (!V8) tma_load_3d(dst + kHalf, &v_map, &sh.v_full[s], 64, t.hk, row);
        }
        ++vis;
        vw.next(a);
        if (vw.live) vr.advanced(a, vw.t, vw.j, 0);
      }
      return true;
    };
    bool ok = true;
    for (int o = 0; ok && it.valid(); ++o) {
      Tile t;
      it.get(a, t);
      it.advance();
      for (int j = 0; j < t.nkv; ++j) {
        const int sb = pvc % kSBufs, s = vpos % kVStages;
        // O is single-buffered: item o-1's epilogue has read it
        bool w = j > 0 || awaitb(&sh.o_free, (o & 1) ^ 1, sh, a.err);
        const uint32_t ppar = (pvc / kSBufs) & 1;
        if (lane == 0) {
          // wait for P(t), issuing V copies as their stages free up (the
          // stage of V(t + 1) frees when PV(t - 1) completes); then make
          // sure V(t) itself is on its way
          const long long t0 = clock64();
          issue_v(vpos + kVStages - 1, false);
          while (w && !mbar_test_wait(&sh.p_ready[sb], ppar)) {
            issue_v(vpos + kVStages - 1, false);
            if (*reinterpret_cast<volatile int*>(&sh.abort)) {
              w = false;
            } else if (clock64() - t0 > kWaitTimeoutCycles) {
              sh.abort = 1;
              report_error(a.err, kDevErrTimeout);
              w = false;
            }
          }
          w = w && issue_v(vpos, true);
        } else {
          w = w && awaitb(&sh.p_ready[sb], ppar, sh, a.err);
        }
        w = w && awaitb(&sh.v_full[s], (vpos / kVStages) & 1, sh, a.err);
        ok = __all_sync(0xffffffffu, w);
        if (!ok) break;
        uint8_t* vt = smem + kOffV + s * kH16Tile;
        const int r0 = t.Lk - j * kT;
        if (r0 < kT) {
          constexpr int kRowChunks = V8 ? 8 : 16;   // 16-byte pieces per key row
          for (int i = lane; i < (kT - r0) * kRowChunks; i += 32) {
            const int row = r0 + i / kRowChunks, c = i % kRowChunks;
            *reinterpret_cast<uint4*>(vt + (c >> 3) * kHalf + row * 128 + (c & 7) * 16) =
                make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async_smem();
          __syncwarp();
        }
        if (V8) {
          // E4M3 [128 keys][128 bytes] in the stage's first 16 KB -> f16 in two
          // halves [128 keys][64], 128-byte swizzle.  Half 0 of key row r
          // takes exactly the bytes of source row r: each lane reads its
          // whole row into registers, the warp syncs, then every lane writes.
#pragma unroll 1
          for (int r0 = 0; r0 < kT; r0 += 32) {
            const int r = r0 + lane;
            uint4 src[8];
#pragma unroll
            for (int c = 0; c < 8; ++c)
              src[c] = *reinterpret_cast<const uint4*>(vt + r * 128 + (((c ^ r) & 7) << 4));
            __syncwarp();
#pragma unroll
            for (int c = 0; c < 8; ++c) {
              const uint32_t wv[4] = {src[c].x, src[c].y, src[c].z, src[c].w};
              uint32_t o[8];
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                o[2 * q] = e4m3x2_to_f16x2(static_cast<uint16_t>(wv[q] & 0xFFFFu));
                o[2 * q + 1] = e4m3x2_to_f16x2(static_cast<uint16_t>(wv[q] >> 16));
              }
              uint8_t* base = vt + (c >> 2) * kHalf + r * 128;
              const int c0 = 2 * (c & 3);
              *reinterpret_cast<uint4*>(base + (((c0 ^ r) & 7) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
              *reinterpret_cast<uint4*>(base + ((((c0 + 1) ^ r) & 7) << 4)) =
                  make_uint4(o[4], o[5], o[6], o[7]);
            }
            __syncwarp();
          }
          fence_proxy_async_smem();
          __syncwarp();
        }
        if (lane == 0) {
          tc_fence_after_sync();
          const uint64_t db = vdesc0 + static_cast<uint64_t>((s * kH16Tile) >> 4);
#pragma unroll
          for (int kk = 0; kk < kT / 16; ++kk)
            tc_mma_f16_tmem_a(tmem + kColO, tmem + kColS + sb * kT + (kk >> 2) * 64 + 8 * (kk & 3),
                              db + static_cast<uint64_t>((kk * 16 * 128) >> 4), idesc_pv,
                              (j > 0 || kk > 0) ? 1u : 0u);
          tc_commit(&sh.v_empty[s]);
          tc_commit(&sh.pv_done[sb]);
          if (j == t.nkv - 1) tc_commit(&sh.o_full);
        }
        __syncwarp();
        ++vpos;
        ++pvc;
      }
    }
    if (lane == 0) {
      // every MMA issued here completes before TMEM is released, every
      // copy lands before the CTA exits
      tc_commit(&sh.mma_done[1]);
      drain(&sh.mma_done[1], 0, a.err);
      cp_async_wait_all();
      for (int i = vis > kVStages ? vis - kVStages : 0; i < vis; ++i)
        drain(&sh.v_full[i % kVStages], (i / kVStages) & 1, a.err);
    }
    __syncwarp();
  } else {
    // ---------------------------------------------- softmax and epilogue
    const int sw = warp & 3;                      // TMEM lane quarter
    const int half = (warp - 2) >> 2;             // column half
    const int r = sw * 32 + lane;                 // tile row = TMEM lane
    const uint32_t bar_id = 1 + sw;
    const uint32_t lane_base = static_cast<uint32_t>(sw * 32) << 16;
    Items it;
    it.start(a);
    int st = 0;
    // this thread's half of a q row: the sum of its 64 codes (rows past the
    // packed tokens were read as zeros)
    auto row_half_load = [&](const Tile& t, uint4 (&w)[4]) {
      const int tok = t.begin + t.qt * kT + r;
      if (tok < a.T) {
        const uint4* qr = reinterpret_cast<const uint4*>(
            a.q8 + (static_cast<size_t>(tok) * a.Hq + t.h) * kD + 64 * half);
#pragma unroll
        for (int i = 0; i < 4; ++i) w[i] = __ldg(qr + i);
      } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) w[i] = make_uint4(0, 0, 0, 0);
      }
    };
    auto row_half_sum = [](const uint4 (&w)[4]) -> int {
      int acc = 0;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        acc = __dp4a(static_cast<int>(w[i].x), 0x01010101, acc);
        acc = __dp4a(static_cast<int>(w[i].y), 0x01010101, acc);
        acc = __dp4a(static_cast<int>(w[i].z), 0x01010101, acc);
        acc = __dp4a(static_cast<int>(w[i].w), 0x01010101, acc);
      }
      return acc;
    };
    int qhalf = 0;
    if (it.valid()) {
      Tile t0;
      it.get(a, t0);
      uint4 w[4];
      row_half_load(t0, w);
      qhalf = row_half_sum(w);
    }
    for (int o = 0; it.valid(); ++o) {
      Tile t;
      it.get(a, t);
      it.advance();
      const int hk = t.hk;
      const float base =
          a.scale_log2 * __ldg(a.sq + (static_cast<size_t>(t.b) * a.NB + t.qt) * a.Hq + t.h);
      const float* skp = a.sk + static_cast<size_t>(t.b) * a.NB * a.Hkv + hk;
      const int row = t.qt * kT + r;   // query index within the sequence
      const int lim = a.causal ? min(t.Lk - 1, row + t.Lk - t.Lq) : t.Lk - 1;
      // the row's 128 * sum_d q_d, which the biased key codes add to every
      // raw score of the row: the two halves' sums meet in shared memory
      sh.pair[half][r] = static_cast<float>(qhalf);
      named_barrier(bar_id, 64);
      const float corr = 128.f * (static_cast<float>(qhalf) + sh.pair[half ^ 1][r]);
      named_barrier(bar_id, 64);
      // l: the sum of the unrounded p (for the lse); lr: the sum of the
      // 16-bit P the P.V product sees (bf16, or f16 in the V8
      // instantiation), which normalises O so that P's rounding cancels
      // where one key dominates
      float m = -INFINITY, l = 0.f, lr = 0.f;
      float sk_next = __ldg(skp);
      for (int j = 0; j < t.nkv; ++j) {
        // logit multiplier of this key tile (log2 units), kept above 0 so
        // that -inf * sc stays -inf
        const float sc = fmaxf(base * sk_next, 1e-30f);
        // raw S' = 2^-24 (q . k + corr): logit (log2 units) = S' sc24 + off
        const float sc24 = sc * 16777216.f, off = -corr * sc;
        if (j + 1 < t.nkv) sk_next = __ldg(skp + static_cast<size_t>(j + 1) * a.Hkv);
        const int sb = st % kSBufs;
        awaitb(&sh.s_full[sb], (st / kSBufs) & 1, sh, a.err);
        __syncwarp();
        tc_fence_after_sync();
        const uint32_t srow = tmem + lane_base + kColS + sb * kT;
        const int climit = lim - j * kT - 64 * half;   // this half's columns c <= climit are visible
        // pass 1: the row maximum of this half's 64 raw scores, read as two
        // 32-column chunks (masked keys -inf; sc24 > 0 keeps the order)
        float xm = -INFINITY;
#pragma unroll 1
        for (int c2 = 0; c2 < 2; ++c2) {
          uint32_t v[32];
          tmem_ld32(srow + 64 * half + 32 * c2, v);
          tmem_ld_wait();
          const int lim2 = climit - 32 * c2;
#pragma unroll
          for (int i = 0; i < 32; ++i)
            xm = fmaxf(xm, i <= lim2 ? __uint_as_float(v[i]) : -INFINITY);
        }
        sh.pair[half][r] = xm;
        named_barrier(bar_id, 64);
        xm = fmaxf(xm, sh.pair[half ^ 1][r]);
        named_barrier(bar_id, 64);   // both read before either writes again
        const float mx = fmaf(xm, sc24, off);
        float f = 1.f;
        bool need = false;
        if (mx > m + kRescaleLog2) {
          if (m > -INFINITY) {
            f = exp2f(m - mx);
            l *= f;
            lr *= f;
            need = true;
          }
          m = mx;
        }
        if (__any_sync(0xffffffffu, need)) {
          awaitb(&sh.pv_done[(st - 1) % kSBufs], ((st - 1) / kSBufs) & 1, sh, a.err);
          __syncwarp();
          tc_fence_after_sync();
          const uint32_t orow = tmem + lane_base + kColO + 64 * half;
#pragma unroll 1
          for (int c2 = 0; c2 < 2; ++c2) {
            uint32_t w[32];
            tmem_ld32(orow + 32 * c2, w);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) w[i] = __float_as_uint(__uint_as_float(w[i]) * f);
            tmem_st32(orow + 32 * c2, w);
            tmem_st_wait();
          }
        }
        // pass 2: P = 2^(x sc - m) in bf16, two keys per column.  This half's
        // keys [64 half, 64 half + 64) go to its own S columns [64 half,
        // 64 half + 32), each chunk over columns it has already read.
        const float nm = (m > -INFINITY ? -m : 0.f) + off;
#pragma unroll 1
        for (int c2 = 0; c2 < 2; ++c2) {
          uint32_t v[32];
          tmem_ld32(srow + 64 * half + 32 * c2, v);
          tmem_ld_wait();
          const int lim2 = climit - 32 * c2;
          {
            uint32_t pk[16];
#pragma unroll
            for (int w = 0; w < 16; ++w) {
              const float x0 = 2 * w <= lim2 ? __uint_as_float(v[2 * w]) : -INFINITY;
              const float x1 = 2 * w + 1 <= lim2 ? __uint_as_float(v[2 * w + 1]) : -INFINITY;
              const float p0 = fast_exp2(fmaf(x0, sc24, nm));
              const float p1 = fast_exp2(fmaf(x1, sc24, nm));
              l += p0 + p1;
              if (V8) {
                // f16 pairs (11 significant bits) for the f16 P.V product
                pk[w] = f32x2_to_f16x2(p1, p0);
                lr = add_f16x2_to_f32(lr, pk[w]);
              } else {
                const __nv_bfloat162 b2 = __floats2bfloat162_rn(p0, p1);
                pk[w] = *reinterpret_cast<const uint32_t*>(&b2);
                lr += __uint_as_float(pk[w] << 16) + __uint_as_float(pk[w] & 0xFFFF0000u);
              }
            }
            tmem_st16(srow + 64 * half + 16 * c2, pk);
          }
        }
        tmem_st_wait();
        tc_fence_before_sync();
        mbar_arrive(&sh.p_ready[sb]);
        ++st;
      }
      sh.pair[half][r] = l;
      named_barrier(bar_id, 64);
      const float lt = l + sh.pair[half ^ 1][r];
      named_barrier(bar_id, 64);
      sh.pair[half][r] = lr;
      named_barrier(bar_id, 64);
      const float ln = lr + sh.pair[half ^ 1][r];   // the normaliser of O
      named_barrier(bar_id, 64);
      const float so = ln > 0.f ? 1.f / ln : 0.f;
      // the next item's q row half loads while this item's O is written
      uint4 qn[4];
      Tile tn;
      const bool more = it.valid();
      if (more) {
        it.get(a, tn);
        row_half_load(tn, qn);
      }
      awaitb(&sh.o_full, o & 1, sh, a.err);
      __syncwarp();
      tc_fence_after_sync();
      const bool write = row < t.Lq;
      const size_t orow_g = static_cast<size_t>(t.begin) + row;
      uint16_t* out = a.o + (orow_g * a.Hq + t.h) * kD + 64 * half;
      const uint32_t orow = tmem + lane_base + kColO + 64 * half;
#pragma unroll 1
      for (int c2 = 0; c2 < 2; ++c2) {
        uint32_t v[32];
        tmem_ld32(orow + 32 * c2, v);
        tmem_ld_wait();
        if (V8) {
          // the channel scales of this half's 32 columns (same for all rows)
          const float* svp = a.sv + (static_cast<size_t>(t.b) * a.Hkv + t.hk) * kD + 64 * half + 32 * c2;
#pragma unroll
          for (int i = 0; i < 32; ++i)
            v[i] = __float_as_uint(__uint_as_float(v[i]) * __ldg(svp + i));
        }
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const __nv_bfloat162 b2 =
              __floats2bfloat162_rn(__uint_as_float(v[2 * i]) * so, __uint_as_float(v[2 * i + 1]) * so);
          pk[i] = *reinterpret_cast<const uint32_t*>(&b2);
        }
        if (write) {
          uint4* o4 = reinterpret_cast<uint4*>(out + 32 * c2);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            o4[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
        }
      }
      tc_fence_before_sync();
      mbar_arrive(&sh.o_free);
      if (write && half == 0 && a.lse != nullptr)
        a.lse[orow_g * a.Hq + t.h] = lt > 0.f ? (m + log2f(lt)) * kLn2 : -INFINITY;
      if (more) qhalf = row_half_sum(qn);
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == kWarpQk) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, 512);
  }
}

struct PrepArgs {
  int B, T, Hq, G, NB, causal, ps, bt_stride, P;
  int ragged, T_kv;
  const int32_t* bt;
  const int32_t* cu_q;
  const int32_t* lk;
  const int32_t* cu_kv;   // ragged K/V: inclusive prefix sums of L_kv
  int32_t* ws;   // [0] units, [1, 1 + 4B) table, [1 + 4B, 1 + 5B) costs
  uint16_t* o;
  float* lse;
  int* err;
};

// A sequence's q tile range and whether its lengths fit the arrays the
// caller described (block scales, block_table row, packed q rows).
__device__ __forceinline__ bool seq_info(const PrepArgs& p, int b, int& begin, int& Lq, int& Lk,
                                         int& qt_lo, int& nqv) {
  begin = b > 0 ? p.cu_q[b - 1] : 0;
  const int end = p.cu_q[b];
  Lq = end - begin;
  const int kvb = p.ragged ? (b > 0 ? p.cu_kv[b - 1] : 0) : 0;
  Lk = p.ragged ? p.cu_kv[b] - kvb : p.lk[b];
  const bool kv_ok = p.ragged ? kvb >= 0 && p.cu_kv[b] <= p.T_kv
                              : static_cast<long long>(Lk) <= static_cast<long long>(p.bt_stride) * p.ps;
  const bool ok = begin >= 0 && Lq >= 0 && end <= p.T && Lk >= 0 &&
                  (Lq + kT - 1) / kT <= p.NB && (Lk + kT - 1) / kT <= p.NB && kv_ok;
  int nqt = 0;
  qt_lo = 0;
  if (ok) q_tile_range(Lq, Lk, p.causal, qt_lo, nqt);
  nqv = ok ? nqt - qt_lo : 0;
  return ok;
}

// Block 0: unit table in cost order.  Every block: O = 0, lse = -inf on
// the rows of q tiles that see no key (and of sequences rejected above);
// block_table entries of the pages holding keys [0, L_kv) outside the pool
// are flagged here, once, rather than where the copies are issued.
__global__ void __launch_bounds__(256) prefill_prep_kernel(const PrepArgs p) {
  if (blockIdx.x == 0) {
    int32_t* cost = p.ws + 1 + kWsStride * p.B;
    for (int b = threadIdx.x; b < p.B; b += blockDim.x) {
      int begin, Lq, Lk, qt_lo, nqv;
      if (!seq_info(p, b, begin, Lq, Lk, qt_lo, nqv)) report_error(p.err, kDevErrBadLength);
      // K/V tiles of the sequence's costliest unit (its first pair)
      cost[b] = nqv > 0 ? kv_tiles_of(Lq, Lk, qt_lo, p.causal) +
                              (nqv > 1 ? kv_tiles_of(Lq, Lk, qt_lo + nqv - 1, p.causal) : 0)
                        : 0;
    }
    __syncthreads();
    for (int b = threadIdx.x; b < p.B; b += blockDim.x) {
      const int cb = cost[b];
      int rank = 0;
      for (int c = 0; c < p.B; ++c) {
        const int cc = cost[c];
        rank += (cc > cb || (cc == cb && c < b)) ? 1 : 0;
      }
      int begin, Lq, Lk, qt_lo, nqv;
      seq_info(p, b, begin, Lq, Lk, qt_lo, nqv);
      int32_t* e = p.ws + 1 + rank * kWsStride;
      e[kWsSeq] = b;
      e[kWsCum] = p.Hq * ((nqv + 1) / 2);   // units; made inclusive below
      e[kWsQtLo] = qt_lo;
      e[kWsNq] = nqv;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      int run = 0;
      for (int k = 0; k < p.B; ++k) {
        run += p.ws[1 + k * kWsStride + kWsCum];
        p.ws[1 + k * kWsStride + kWsCum] = run;
      }
      p.ws[0] = run;
    }
  }
  for (int b = blockIdx.x; b < p.B; b += gridDim.x) {
    int begin, Lq, Lk, qt_lo, nqv;
    const bool ok = seq_info(p, b, begin, Lq, Lk, qt_lo, nqv);
    int rows = ok ? min(Lq, qt_lo * kT) : 0;
    if (!ok && begin >= 0 && Lq > 0 && begin + Lq <= p.T) rows = Lq;
    if (ok && !p.ragged) {
      const int npg = (Lk + p.ps - 1) / p.ps;
      const int32_t* row = p.bt + static_cast<size_t>(b) * p.bt_stride;
      for (int e = threadIdx.x; e < npg; e += blockDim.x)
        if (static_cast<unsigned>(row[e]) >= static_cast<unsigned>(p.P))
          report_error(p.err, kDevErrBadPage);
    }
    const int chunks = rows * p.Hq * (kD / 8);
    for (int i = threadIdx.x; i < chunks; i += blockDim.x) {
      const int c = i % (kD / 8), rh = i / (kD / 8);
      const size_t tok = static_cast<size_t>(begin) + rh / p.Hq;
      const int h = rh % p.Hq;
      reinterpret_cast<uint4*>(p.o + (tok * p.Hq + h) * kD)[c] = make_uint4(0, 0, 0, 0);
      if (c == 0 && p.lse != nullptr) p.lse[tok * p.Hq + h] = -INFINITY;
    }
  }
}

// One thread per unit: its record (sequence, head, q tiles, lengths).
__global__ void __launch_bounds__(256) prefill_units_kernel(const PrepArgs p) {
  const int u = static_cast<int>(blockIdx.x * blockDim.x + threadIdx.x);
  if (u >= p.ws[0]) return;
  const int32_t* tab = p.ws + 1;
  int lo = 0, hi = p.B - 1;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (tab[mid * kWsStride + kWsCum] > u) hi = mid; else lo = mid + 1;
  }
  const int32_t* e = tab + lo * kWsStride;
  const int local = u - (lo > 0 ? tab[(lo - 1) * kWsStride + kWsCum] : 0);
  const int b = e[kWsSeq], qt_lo = e[kWsQtLo], nqv = e[kWsNq];
  const int pairs = (nqv + 1) >> 1;
  const int tt = local % pairs;
  const int begin = b > 0 ? p.cu_q[b - 1] : 0;
  const int kvb = p.ragged ? (b > 0 ? p.cu_kv[b - 1] : 0) : 0;
  const int Lk = p.ragged ? p.cu_kv[b] - kvb : p.lk[b];
  int4* rec = reinterpret_cast<int4*>(reinterpret_cast<uint8_t*>(p.ws) + units_offset(p.B)) + 2 * u;
  const int h = local / pairs;
  rec[0] = make_int4(b, h | ((h / p.G) << 16), qt_lo + tt,
                     nqv - 1 - tt != tt ? qt_lo + nqv - 1 - tt : -1);
  rec[1] = make_int4(begin, p.cu_q[b] - begin, Lk, kvb);
}

// Upper bound of the unit count: sum_b ceil(ceil(L_b / 128) / 2) per head is
// at most T / 256 + B.
long long max_units(int B, int T, int Hq) {
  return static_cast<long long>(Hq) * ((static_cast<long long>(T) + 255) / 256 + B);
}

}  // namespace

size_t prefill_workspace_bytes(int num_seqs, int num_tokens, int num_heads_q) {
  return units_offset(num_seqs) +
         32 * static_cast<size_t>(max_units(num_seqs, num_tokens, num_heads_q));
}

cudaError_t launch_prefill_int8(const qpkv_prefill_params& p, cudaStream_t stream, int* status) {
  *status = QPKV_OK;
  if (p.num_seqs == 0 || p.num_tokens == 0) return cudaSuccess;
  const bool ragged = p.cu_seqlens_kv != nullptr;
  const int ps = ragged ? kT : p.page_size;
  const int rows_box = ps < kT ? ps : kT;
  PrepArgs pa;
  pa.ragged = ragged ? 1 : 0;
  pa.T_kv = p.num_kv_tokens;
  pa.cu_kv = p.cu_seqlens_kv;
  pa.B = p.num_seqs;
  pa.T = p.num_tokens;
  pa.Hq = p.num_heads_q;
  pa.G = p.num_heads_q / p.num_heads_kv;
  pa.P = p.num_pages;
  pa.bt = p.block_table;
  pa.NB = p.num_blocks;
  pa.causal = p.causal ? 1 : 0;
  pa.ps = ps;
  pa.bt_stride = p.bt_stride;
  pa.cu_q = p.cu_seqlens_q;
  pa.lk = p.seqlens_kv;
  pa.ws = static_cast<int32_t*>(p.workspace);
  pa.o = static_cast<uint16_t*>(p.o);
  pa.lse = p.lse;
  pa.err = p.error_word;
  const int prep_grid = p.num_seqs < 256 ? p.num_seqs : 256;
  prefill_prep_kernel<<<prep_grid, 256, 0, stream>>>(pa);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const long long umax = max_units(p.num_seqs, p.num_tokens, p.num_heads_q);
  prefill_units_kernel<<<static_cast<unsigned>((umax + 255) / 256), 256, 0, stream>>>(pa);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (ragged && p.num_kv_tokens == 0) return cudaSuccess;   // no keys: the prep pass wrote every row

  // q [T, Hq, D] int8, pools [P * ps, Hkv, D] (int8 K, bf16 V) as 3-D maps
  // (d, head, row); a box is 128 q rows / one page's rows of one head
  const uint64_t D = kD, T = static_cast<uint64_t>(p.num_tokens);
  const uint64_t Hq = static_cast<uint64_t>(p.num_heads_q), Hkv = static_cast<uint64_t>(p.num_heads_kv);
  const uint64_t rows = ragged ? static_cast<uint64_t>(p.num_kv_tokens)
                               : static_cast<uint64_t>(p.num_pages) * ps;
  CUtensorMap qm, km, vm;
  const uint64_t qdims[3] = {D, Hq, T}, qstr[2] = {D, Hq * D};
  const uint64_t kdims[3] = {D, Hkv, rows}, kstr[2] = {D, Hkv * D};
  const uint64_t vstr[2] = {2 * D, 2 * Hkv * D};
  const uint32_t qbox[3] = {kD, 1u, kT};
  const uint32_t kbox[3] = {kD, 1u, static_cast<uint32_t>(rows_box)};
  const uint32_t vbox[3] = {64u, 1u, static_cast<uint32_t>(rows_box)};
  // FP8 V (v_scale given): E4M3 codes shaped like K, one 128-byte box row
  const bool v8 = p.v_scale != nullptr;
  if (encode_tensor_map(&qm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(p.q), qdims, qstr,
                        qbox, CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS ||
      encode_tensor_map(&km, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(p.k_pool), kdims,
                        kstr, kbox, CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS ||
      (v8 ? encode_tensor_map(&vm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(p.v_pool),
                              kdims, kstr, kbox, CU_TENSOR_MAP_SWIZZLE_128B)
          : encode_tensor_map(&vm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(p.v_pool),
                              kdims, vstr, vbox, CU_TENSOR_MAP_SWIZZLE_128B)) != CUDA_SUCCESS) {
    *status = QPKV_ERR_CUDA;
    return cudaErrorInvalidValue;
  }
  PArgs a;
  a.B = p.num_seqs;
  a.T = p.num_tokens;
  a.q8 = static_cast<const int8_t*>(p.q);
  a.sv = p.v_scale;
  a.Hq = p.num_heads_q;
  a.Hkv = p.num_heads_kv;
  a.G = p.num_heads_q / p.num_heads_kv;
  a.ps = ps;
  a.P = p.num_pages;
  a.bt_stride = p.bt_stride;
  a.NB = p.num_blocks;
  a.causal = p.causal ? 1 : 0;
  a.ragged = ragged ? 1 : 0;
  a.T_kv = p.num_kv_tokens;
  a.rows_box = rows_box;
  a.nbox = kT / rows_box;
  a.m = ps > kT ? ps / kT : 1;
  a.m_magic = a.m > 1 ? static_cast<unsigned>(((1ull << 32) + a.m - 1) / a.m) : 0u;
  a.scale_log2 = (p.sm_scale > 0.f ? p.sm_scale : 1.0f / sqrtf(static_cast<float>(kD))) * kLog2e;
  a.cu_q = p.cu_seqlens_q;
  a.lk = p.seqlens_kv;
  a.bt = p.block_table;
  a.sq = p.q_block_scale;
  a.sk = p.k_block_scale;
  a.o = static_cast<uint16_t*>(p.o);
  a.lse = p.lse;
  a.ws = static_cast<const int32_t*>(p.workspace);
  a.err = p.error_word;
  auto* kern = v8 ? prefill_int8_kernel<true> : prefill_int8_kernel<false>;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  kern<<<sms, kThreads, kSmem, stream>>>(qm, km, vm, a);
  return cudaGetLastError();
}
}  // namespace qpkv
