// Dense FP8 attention forward with per-(batch, head) descales
// ("[Triton] FP8 with FA v3 API": flash_attn_func(q_fp8, k_fp8, v_fp8,
// softmax_scale, causal, q_descale, k_descale, v_descale)):
//   O = softmax(scale * qd * kd * Q8 K8^T + mask) * V8 * vd
// Q/K/V are E4M3 codes in BSND layout, descales fp32 [B, heads of that
// tensor], O bf16 BSND, lse (natural log) fp32 [B, Sq, Hq].  Causal masking
// is bottom-right aligned: key j is visible to query i iff j <= i + Sk - Sq.
//
// Each persistent CTA (one per SM) runs two 128-row query tiles of one
// (batch, head) side by side, tiles A = 2p and B = 2p + 1 of a pair, over
// the same stream of K/V tiles: while one tile's softmax computes its
// exponentials, the tensor core works on the other tile, and each K/V tile
// is fetched once for both.  14 warps:
//   warp 0      TMA: the pair's Q tiles (two slots), K tiles (4-stage ring),
//               V tiles (2-stage ring), K one step ahead of V; K and V
//               copies leave together from two lanes
//   warp 1      tcgen05 MMAs from one thread, per step g of the K/V stream:
//                 PV_A(g-1) QK_A(g) PV_B(g-1) QK_B(g)
//               QK: S[128 q x 128 k] = Q . K^T, E4M3 operands (kind::f8f6f4);
//               PV: O[128 q x 128 d] += P . V, f16 operands (kind::f16) with P
//               read from tensor memory and V widened from E4M3 (exact)
//   warps 2, 3, 12, 13  widen each V tile from E4M3 to f16, written in the
//               MN-major operand layout of the PV product (two 64-column
//               halves); one such warp on each scheduler
//   warps 4-7   softmax and epilogue of tile A, one thread per query row
//   warps 8-11  the same for tile B
// P is f16 (11 significant bits, range 2^-24 .. 65504): with the lazy
// running maximum below, p <= 2^8.  The softmax keeps the running maximum
// until a tile beats it by more than 2^8 (then the row's O is rescaled).
// TMEM: S_A, S_B, O_A, O_B, 128 columns each; a tile's P (two f16 per
// column) overwrites the first 64 columns of its S buffer.  The MMAs of the
// issuing thread run in issue order, so QK_X(g+1) overwrites S_X only after
// PV_X(g) has read P_X(g), and the commit behind QK_X(g+1) tells the
// softmax that PV_X(g) is done before it may rescale O_X.
//
// Work: a unit is a pair of q tiles of one (batch, head); units are taken
// in (batch, head)-major order (the CTAs running at the same time share a
// few heads' K/V through L2) and dealt to the CTAs in a snake order, which
// evens out the pairs' different causal lengths.
#include <cmath>

#include "common.cuh"
#include "internal.h"

namespace qpkv {
namespace {

constexpr int kT = 128;               // q rows per tile = keys per tile = MMA M and N
constexpr int kD = 128;               // head dim
constexpr int kThreads = 448;         // 14 warps
constexpr int kWarpLoad = 0, kWarpMma = 1, kWarpConv0 = 2, kWarpSoftA = 4, kWarpSoftB = 8,
              kWarpConv2 = 12;
constexpr int kConvThreads = 128;
constexpr int kKStages = 4;           // E4M3 K tiles, 16 KB each
constexpr int kVStages = 2;           // E4M3 V tiles, 16 KB each
constexpr int kV16Bufs = 2;           // f16 V tiles, 32 KB each
constexpr int kTile8 = kT * kD;       // 16 KB
constexpr int kTile16 = 2 * kT * kD;  // 32 KB: two halves of 64 columns
constexpr int kHalf16 = kT * 128;     // 16 KB: one half (128 rows of 128 bytes)
constexpr int kOffQ = 0;                                  // [2 slots][2 tiles] Q
constexpr int kOffK = kOffQ + 4 * kTile8;
constexpr int kOffV8 = kOffK + kKStages * kTile8;
constexpr int kOffV16 = kOffV8 + kVStages * kTile8;
constexpr int kSmem = kOffV16 + kV16Bufs * kTile16 + 1024;
constexpr float kRescaleLog2 = 8.0f;
constexpr uint32_t kColS0 = 0, kColO0 = 256;   // S_A, S_B at 0, 128; O_A, O_B at 256, 384

struct AttnArgs {
  int B, Sq, Sk, Hq, Hkv, G;
  int qt_lo, nq;      // q tiles [qt_lo, qt_lo + nq) have visible keys
  int pairs;          // units per (batch, head) = ceil(nq / 2)
  int units;          // B * Hq * pairs
  int causal;
  float scale_log2;   // softmax scale * log2(e)
  const float* qd;
  const float* kd;
  const float* vd;
  uint16_t* o;        // bf16 [B, Sq, Hq, D]
  float* lse;         // [B, Sq, Hq] or null
  int* err;
};

struct Shared {
  uint64_t q_full[2], q_free[2];
  uint64_t k_full[kKStages], k_empty[kKStages];
  uint64_t v_full[kVStages], v_empty[kVStages];
  uint64_t v16_full[kV16Bufs], v16_empty[kV16Bufs];
  uint64_t s_full[2], p_ready[2], o_full[2];   // per tile A / B
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort;
};

__device__ __forceinline__ bool awaitb(uint64_t* bar, uint32_t parity, Shared& sh, int* err) {
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

// Bounded wait that ignores the abort flag (this CTA's own copies / MMAs).
__device__ __forceinline__ void drain(uint64_t* bar, uint32_t parity, int* err) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > kWaitTimeoutCycles) {
      report_error(err, kDevErrTimeout);
      return;
    }
  }
}

// Lane 0 waits, the warp learns the outcome and is ordered after the wait.
__device__ __forceinline__ bool warp_await(uint64_t* bar, uint32_t parity, Shared& sh, int* err,
                                           int lane) {
  int ok = 1;
  if (lane == 0) ok = awaitb(bar, parity, sh, err) ? 1 : 0;
  ok = __shfl_sync(0xffffffffu, ok, 0);
  __syncwarp();
  return ok != 0;
}

// 2^x by the hardware approximation (relative error ~2^-22; -inf -> 0).
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// K/V tiles of q tile qt: keys [0, last] with last the final key any of its
// rows sees.
__device__ __forceinline__ int kv_tiles(const AttnArgs& a, int qt) {
  int last = a.Sk - 1;
  if (a.causal) last = min(last, qt * kT + kT - 1 + a.Sk - a.Sq);
  return last < 0 ? 0 : last / kT + 1;
}

// This CTA's units in order (round r takes unit r * grid + c on even
// rounds, r * grid + grid - 1 - c on odd ones) and the K/V steps of each.
struct Walk {
  int r;                // round of the current unit
  int u;                // unit index, >= a.units at the end
  int uc;               // units of this CTA before the current one
  int b, h, qt;         // qt: tile A; tile B = qt + 1 when has_b
  int has_b, na, nb, ns;
  int j;                // step within the unit
  int g;                // step of this CTA's K/V stream
  __device__ __forceinline__ void load_unit(const AttnArgs& a) {
    const int grid = static_cast<int>(gridDim.x), c = static_cast<int>(blockIdx.x);
    u = r * grid + ((r & 1) ? grid - 1 - c : c);
    if (u >= a.units) return;
    const int bh = u / a.pairs, p = u % a.pairs;
    b = bh / a.Hq;
    h = bh % a.Hq;
    qt = a.qt_lo + 2 * p;
    has_b = 2 * p + 1 < a.nq;
    na = kv_tiles(a, qt);
    nb = has_b ? kv_tiles(a, qt + 1) : 0;
    ns = has_b ? nb : na;
  }
  __device__ __forceinline__ void start(const AttnArgs& a) {
    r = 0;
    uc = 0;
    j = 0;
    g = 0;
    load_unit(a);
  }
  __device__ __forceinline__ bool valid(const AttnArgs& a) const { return u < a.units; }
  __device__ __forceinline__ bool active(int x) const { return x == 0 ? j < na : (has_b && j < nb); }
  __device__ __forceinline__ int nx(int x) const { return x == 0 ? na : nb; }
  // advance one step of the stream
  __device__ __forceinline__ void next(const AttnArgs& a) {
    ++g;
    if (++j < ns) return;
    j = 0;
    ++r;
    ++uc;
    load_unit(a);
  }
  // advance to the next step where tile x is active
  __device__ __forceinline__ void next_active(const AttnArgs& a, int x) {
    do {
      next(a);
    } while (valid(a) && !active(x));
  }
};

__global__ void __launch_bounds__(kThreads, 1)
    fp8_attn_kernel(const __grid_constant__ CUtensorMap q_map,
                    const __grid_constant__ CUtensorMap k_map,
                    const __grid_constant__ CUtensorMap v_map, const AttnArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  __shared__ Shared sh;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sh.q_full[i], 1);
      mbar_init(&sh.q_free[i], 1);
      mbar_init(&sh.s_full[i], 1);
      mbar_init(&sh.p_ready[i], 128);
      mbar_init(&sh.o_full[i], 1);
    }
    for (int s = 0; s < kKStages; ++s) {
      mbar_init(&sh.k_full[s], 1);
      mbar_init(&sh.k_empty[s], 1);
    }
    for (int s = 0; s < kVStages; ++s) {
      mbar_init(&sh.v_full[s], 1);
      mbar_init(&sh.v_empty[s], kConvThreads / 32);
    }
    for (int s = 0; s < kV16Bufs; ++s) {
      mbar_init(&sh.v16_full[s], kConvThreads / 32);
      mbar_init(&sh.v16_empty[s], 1);
    }
    mbar_init(&sh.mma_done, 1);
    sh.abort = 0;
    fence_mbar_init();
  }
  if (warp == kWarpMma) tmem_alloc(&sh.tmem_base, 512);
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = sh.tmem_base;

  if (warp == kWarpLoad) {
    // ------------------------------------------------------------- loads
    // One thread's tensor copies leave one after another (each issue holds
    // the thread for a few hundred cycles); copies of several lanes in one
    // instruction go out together.  So lane 0 issues K(g+1) while lane 1
    // issues V(g), and the unit's two Q tiles go out from lanes 0 and 1.
    if (lane == 0) {
      tma_prefetch_desc(&q_map);
      tma_prefetch_desc(&k_map);
      tma_prefetch_desc(&v_map);
    }
    Walk kw, vw;
    kw.start(a);
    vw.start(a);
    int ncopies_k = 0, ncopies_v = 0, nq_slots = 0;
    bool ok = true;
    // the Q tiles of kw's unit (at its first step)
    auto issue_q = [&]() -> bool {
      const int slot = kw.uc & 1;
      if (!warp_await(&sh.q_free[slot], ((kw.uc >> 1) & 1) ^ 1, sh, a.err, lane)) return false;
      if (lane == 0) mbar_arrive_expect_tx(&sh.q_full[slot], (1 + kw.has_b) * kTile8);
      __syncwarp();
      if (lane <= kw.has_b)
        tma_load_4d(smem + kOffQ + (slot * 2 + lane) * kTile8, &q_map, &sh.q_full[slot], 0, kw.h,
                    (kw.qt + lane) * kT, kw.b);
      __syncwarp();
      ++nq_slots;
      return true;
    };
    // K of step kw (when do_k) and V of step vw (when do_v), one instruction
    auto issue = [&](bool do_k, bool do_v) -> bool {
      const int ks = kw.g % kKStages, vs = vw.g % kVStages;
      if (do_k) {
        if (kw.j == 0 && !issue_q()) return false;
        if (!warp_await(&sh.k_empty[ks], ((kw.g / kKStages) & 1) ^ 1, sh, a.err, lane))
          return false;
      }
      if (do_v && !warp_await(&sh.v_empty[vs], ((vw.g / kVStages) & 1) ^ 1, sh, a.err, lane))
        return false;
      if ((lane == 0 && do_k) || (lane == 1 && do_v)) {
        const bool k = lane == 0;
        uint64_t* bar = k ? &sh.k_full[ks] : &sh.v_full[vs];
        const int hh = (k ? kw.h : vw.h) / a.G, jj = k ? kw.j : vw.j, bb = k ? kw.b : vw.b;
        mbar_arrive_expect_tx(bar, kTile8);
        tma_load_4d(smem + (k ? kOffK + ks * kTile8 : kOffV8 + vs * kTile8), k ? &k_map : &v_map,
                    bar, 0, hh, jj * kT, bb);
      }
      __syncwarp();
      if (do_k) {
        ++ncopies_k;
        kw.next(a);
      }
      if (do_v) {
        ++ncopies_v;
        vw.next(a);
      }
      return true;
    };
    if (kw.valid(a)) ok = issue(true, false);
    while (ok && vw.valid(a)) ok = issue(kw.valid(a), true);
    // this CTA's copies still in flight land before it exits
    if (lane == 0) {
      for (int i = ncopies_k > kKStages ? ncopies_k - kKStages : 0; i < ncopies_k; ++i)
        drain(&sh.k_full[i % kKStages], (i / kKStages) & 1, a.err);
      for (int i = ncopies_v > kVStages ? ncopies_v - kVStages : 0; i < ncopies_v; ++i)
        drain(&sh.v_full[i % kVStages], (i / kVStages) & 1, a.err);
      for (int i = nq_slots > 2 ? nq_slots - 2 : 0; i < nq_slots; ++i)
        drain(&sh.q_full[i & 1], (i >> 1) & 1, a.err);
    }
    __syncwarp();
  } else if (warp == kWarpMma) {
    // -------------------------------------------------------------- MMA
    if (lane == 0) {
      const uint32_t idesc_qk = make_idesc(kFmtE4M3, kFmtE4M3, 0, 0, kT, kT);
      const uint32_t idesc_pv = make_idesc(kFmtF16, kFmtF16, 0, 1, kT, kD);
      const uint64_t qdesc0 = make_smem_desc(smem_u32(smem + kOffQ), 16, 1024, kSwizzle128B);
      const uint64_t kdesc0 = make_smem_desc(smem_u32(smem + kOffK), 16, 1024, kSwizzle128B);
      // MN-major f16 V: two 64-column atoms 16 KB apart, 16 key rows (2 KB)
      // per K = 16 step
      const uint64_t vdesc0 = make_smem_desc(smem_u32(smem + kOffV16), kHalf16, 1024, kSwizzle128B);
      Walk w;
      w.start(a);
      int cnt_p[2] = {0, 0};    // PVs issued per tile (p_ready phases)
      // the pending PV of each tile: its step's g and j, whether it ends the
      // tile's unit, whether it is the last reader of its V buffer
      int pend_g[2] = {-1, -1}, pend_j[2] = {0, 0}, pend_last[2] = {0, 0}, pend_rel[2] = {0, 0};
      bool ok = true;
      auto pv = [&](int x) -> bool {
        const int g = pend_g[x];
        if (!awaitb(&sh.p_ready[x], cnt_p[x] & 1, sh, a.err)) return false;
        if (!awaitb(&sh.v16_full[g % kV16Bufs], (g / kV16Bufs) & 1, sh, a.err)) return false;
        tc_fence_after_sync();
        const uint64_t db = vdesc0 + static_cast<uint64_t>(((g % kV16Bufs) * kTile16) >> 4);
        const uint32_t cs = kColS0 + 128u * x, co = kColO0 + 128u * x;
#pragma unroll
        for (int kk = 0; kk < kT / 16; ++kk)
          tc_mma_f16_tmem_a(tmem + co, tmem + cs + 8 * kk,
                            db + static_cast<uint64_t>((kk * 16 * 128) >> 4), idesc_pv,
                            (pend_j[x] > 0 || kk > 0) ? 1u : 0u);
        if (pend_rel[x]) tc_commit(&sh.v16_empty[g % kV16Bufs]);
        if (pend_last[x]) tc_commit(&sh.o_full[x]);
        ++cnt_p[x];
        pend_g[x] = -1;
        return true;
      };
      auto qk = [&](int x) -> bool {
        const int slot = w.uc & 1, s = w.g % kKStages;
        if (w.j == 0 && !awaitb(&sh.q_full[slot], (w.uc >> 1) & 1, sh, a.err)) return false;
        if (!awaitb(&sh.k_full[s], (w.g / kKStages) & 1, sh, a.err)) return false;
        tc_fence_after_sync();
        const uint64_t da = qdesc0 + static_cast<uint64_t>(((slot * 2 + x) * kTile8) >> 4);
        const uint64_t db = kdesc0 + static_cast<uint64_t>((s * kTile8) >> 4);
        const uint32_t cs = kColS0 + 128u * x;
#pragma unroll
        for (int kk = 0; kk < kD / 32; ++kk)
          tc_mma_f8(tmem + cs, da + 2 * kk, db + 2 * kk, idesc_qk, kk > 0);
        tc_commit(&sh.s_full[x]);
        // the last reader of this K stage (and, at the unit's end, of the Q slot)
        const bool last_reader = x == 1 || !w.active(1);
        if (last_reader) {
          tc_commit(&sh.k_empty[s]);
          if (w.j == w.ns - 1) tc_commit(&sh.q_free[slot]);
        }
        pend_g[x] = w.g;
        pend_j[x] = w.j;
        pend_last[x] = w.j == w.nx(x) - 1;
        pend_rel[x] = last_reader;
        return true;
      };
      // step g: PV_A(pending) QK_A(g) PV_B(pending) QK_B(g)
      while (ok && w.valid(a)) {
        for (int x = 0; x < 2 && ok; ++x) {
          if (pend_g[x] >= 0) ok = pv(x);
          if (ok && w.active(x)) ok = qk(x);
        }
        if (ok) w.next(a);
      }
      for (int x = 0; x < 2 && ok; ++x)
        if (pend_g[x] >= 0) ok = pv(x);
      // every MMA issued here completes before TMEM is released
      tc_commit(&sh.mma_done);
      drain(&sh.mma_done, 0, a.err);
    }
    __syncwarp();
  } else if (warp < kWarpSoftA || warp >= kWarpConv2) {
    // ---------------------------------------- V: E4M3 -> f16 (exact)
    // Input: a TMA tile [128 keys][128 bytes], 128-byte swizzle.  Output:
    // two halves [128 keys][64 f16] (dims 0-63, 64-127), 128-byte swizzle.
    const int ct = warp < kWarpSoftA ? tid - kWarpConv0 * 32 : tid - kWarpConv2 * 32 + 64;
    Walk w;
    w.start(a);
    while (w.valid(a)) {
      const int g = w.g, s = g % kVStages, bsel = g % kV16Bufs;
      if (!warp_await(&sh.v_full[s], (g / kVStages) & 1, sh, a.err, lane)) break;
      if (!warp_await(&sh.v16_empty[bsel], ((g / kV16Bufs) & 1) ^ 1, sh, a.err, lane)) break;
      const uint8_t* src = smem + kOffV8 + s * kTile8;
      uint8_t* dst = smem + kOffV16 + bsel * kTile16;
#pragma unroll
      for (int k = 0; k < (kT * 8) / kConvThreads; ++k) {
        const int i = ct + kConvThreads * k;
        const int row = i >> 3, c = i & 7;
        const uint4 xv = *reinterpret_cast<const uint4*>(src + row * 128 + (((c ^ row) & 7) << 4));
        const uint32_t wv[4] = {xv.x, xv.y, xv.z, xv.w};
        uint32_t o[8];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          o[2 * q] = e4m3x2_to_f16x2(static_cast<uint16_t>(wv[q] & 0xFFFFu));
          o[2 * q + 1] = e4m3x2_to_f16x2(static_cast<uint16_t>(wv[q] >> 16));
        }
        uint8_t* base = dst + (c >> 2) * kHalf16 + row * 128;
        const int c0 = 2 * (c & 3);
        *reinterpret_cast<uint4*>(base + (((c0 ^ row) & 7) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
        *reinterpret_cast<uint4*>(base + ((((c0 + 1) ^ row) & 7) << 4)) =
            make_uint4(o[4], o[5], o[6], o[7]);
      }
      fence_proxy_async_smem();   // generic stores, read by the tensor core
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&sh.v_empty[s]);
        mbar_arrive(&sh.v16_full[bsel]);
      }
      w.next(a);
    }
  } else {
    // ---------------------------------------------- softmax and epilogue
    const int x = warp < kWarpSoftB ? 0 : 1;      // tile A or B
    const int r = (warp & 3) * 32 + lane;         // tile row = TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t srow = tmem + lane_base + kColS0 + 128u * x;
    const uint32_t orow = tmem + lane_base + kColO0 + 128u * x;
    Walk w;
    w.start(a);
    if (w.valid(a) && !w.active(x)) w.next_active(a, x);
    int cnt = 0, units = 0;
    float m = -INFINITY, l = 0.f;
    while (w.valid(a)) {
      const int qt = w.qt + x;
      const int row = qt * kT + r;
      const int hk = w.h / a.G;
      // last key this row sees (may be negative: none)
      const int lim = a.causal ? min(a.Sk - 1, row + a.Sk - a.Sq) : a.Sk - 1;
      if (w.j == 0) {
        m = -INFINITY;
        l = 0.f;
      }
      // logit multiplier (log2 units); kept above 0 so that -inf * sc stays -inf
      const float sc = fmaxf(a.scale_log2 * __ldg(a.qd + w.b * a.Hq + w.h) *
                                 __ldg(a.kd + w.b * a.Hkv + hk),
                             1e-30f);
      const int climit = lim - w.j * kT;          // columns c <= climit are visible
      if (!awaitb(&sh.s_full[x], cnt & 1, sh, a.err)) break;
      __syncwarp();   // converged before the .sync.aligned TMEM accesses
      tc_fence_after_sync();
      const bool whole = __all_sync(0xffffffffu, climit >= kT - 1);
      // pass 1: the row maximum of the raw scores (masked keys -inf; sc > 0
      // keeps the order)
      float xm = -INFINITY;
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t v[32];
        tmem_ld32(srow + 32 * c, v);
        tmem_ld_wait();
        float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
        if (whole) {
#pragma unroll
          for (int i = 0; i < 32; i += 2)
            m4[(i >> 1) & 3] = fmax3(m4[(i >> 1) & 3], __uint_as_float(v[i]), __uint_as_float(v[i + 1]));
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i)
            m4[i & 3] = fmaxf(m4[i & 3], 32 * c + i <= climit ? __uint_as_float(v[i]) : -INFINITY);
        }
        xm = fmax3(xm, fmax3(m4[0], m4[1], m4[2]), m4[3]);
      }
      const float mx = xm * sc;   // the row's tile maximum in log2 units
      float f = 1.f;
      bool need = false;
      if (mx > m + kRescaleLog2) {
        if (m > -INFINITY) {
          f = exp2f(m - mx);
          l *= f;
          need = true;
        }
        m = mx;
      }
      if (__any_sync(0xffffffffu, need)) {
        // the previous PV of this tile is complete (it was issued before the
        // QK whose commit the s_full wait saw); rows that keep their maximum
        // use the factor 1
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t v[32];
          tmem_ld32(orow + 32 * c, v);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * f);
          tmem_st32(orow + 32 * c, v);
          tmem_st_wait();
        }
      }
      // pass 2: P = 2^(x sc - m) as f16 pairs into the first 64 columns of S
      // (chunk c of 32 keys -> columns [16c, 16c + 16), all already read)
      const float nm = m > -INFINITY ? -m : 0.f;   // a row that sees no key gets p = 0
      // pairs of keys in packed f32x2 arithmetic: x = s sc - m, the sums
      const uint64_t sc2 = f32x2_pack(sc, sc), nm2 = f32x2_pack(nm, nm);
      uint64_t ls2 = f32x2_pack(0.f, 0.f);
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t v[32];
        tmem_ld32(srow + 32 * c, v);
        tmem_ld_wait();
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          float2 x = f32x2_unpack(
              f32x2_fma(f32x2_pack(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1])), sc2, nm2));
          if (!whole) {
            x.x = 32 * c + 2 * i <= climit ? x.x : -INFINITY;
            x.y = 32 * c + 2 * i + 1 <= climit ? x.y : -INFINITY;
          }
          const float p0 = fast_exp2(x.x), p1 = fast_exp2(x.y);
          ls2 = f32x2_add(ls2, f32x2_pack(p0, p1));
          pk[i] = f32x2_to_f16x2(p1, p0);
        }
        tmem_st16(srow + 16 * c, pk);
      }
      const float2 ls = f32x2_unpack(ls2);
      l += ls.x + ls.y;
      tmem_st_wait();
      tc_fence_before_sync();
      mbar_arrive(&sh.p_ready[x]);
      ++cnt;
      if (w.j == w.nx(x) - 1) {
        // ---- epilogue: O / l * vd -> bf16, and the lse, once the tile's
        // last PV has landed
        const float vd = __ldg(a.vd + w.b * a.Hkv + hk);
        const float so = l > 0.f ? vd / l : 0.f;
        if (!awaitb(&sh.o_full[x], units & 1, sh, a.err)) break;
        __syncwarp();
        tc_fence_after_sync();
        const bool write = row < a.Sq;
        uint16_t* out = a.o + ((static_cast<size_t>(w.b) * a.Sq + row) * a.Hq + w.h) * kD;
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t v[32];
          tmem_ld32(orow + 32 * c, v);
          tmem_ld_wait();
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const __nv_bfloat162 t2 = __floats2bfloat162_rn(__uint_as_float(v[2 * i]) * so,
                                                            __uint_as_float(v[2 * i + 1]) * so);
            pk[i] = *reinterpret_cast<const uint32_t*>(&t2);
          }
          if (write) {
            uint4* o4 = reinterpret_cast<uint4*>(out + 32 * c);
#pragma unroll
            for (int i = 0; i < 4; ++i)
              o4[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
          }
        }
        tc_fence_before_sync();
        if (write && a.lse != nullptr)
          a.lse[(static_cast<size_t>(w.b) * a.Sq + row) * a.Hq + w.h] =
              l > 0.f ? (m + log2f(l)) * kLn2 : -INFINITY;
        ++units;
      }
      w.next_active(a, x);
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, 512);
  }
}

// Rows [0, rows) of every (batch, head) see no key: O = 0, lse = -inf.
__global__ void fp8_attn_empty_rows_kernel(int B, int Sq, int Hq, int rows, uint16_t* o,
                                           float* lse) {
  const size_t n_rows = static_cast<size_t>(B) * rows * Hq;
  const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n_rows * (kD / 8);
       i += stride) {
    const size_t rix = i / (kD / 8), c = i % (kD / 8);
    const size_t h = rix % Hq, s = (rix / Hq) % rows, b = rix / (static_cast<size_t>(Hq) * rows);
    const size_t base = ((b * Sq + s) * Hq + h);
    reinterpret_cast<uint4*>(o + base * kD)[c] = make_uint4(0, 0, 0, 0);
    if (c == 0 && lse != nullptr) lse[base] = -INFINITY;
  }
}

}  // namespace

cudaError_t launch_fp8_attn(const void* q, const void* k, const void* v, int B, int Sq, int Sk,
                            int Hq, int Hkv, int D, const float* q_descale, const float* k_descale,
                            const float* v_descale, float softmax_scale, int causal, void* o,
                            float* lse, int32_t* error_word, cudaStream_t stream, int* status) {
  *status = QPKV_OK;
  if (D != kD) {
    *status = QPKV_ERR_UNSUPPORTED;
    return cudaErrorInvalidValue;
  }
  if (B == 0 || Sq == 0) return cudaSuccess;
  const int nqt = (Sq + kT - 1) / kT;
  // first q tile with a visible key: some row i of it has i + Sk - Sq >= 0
  int qt_lo = 0;
  if (Sk == 0) {
    qt_lo = nqt;
  } else if (causal && Sq - Sk - (kT - 1) > 0) {
    qt_lo = (Sq - Sk - (kT - 1) + kT - 1) / kT;
  }
  qt_lo = qt_lo > nqt ? nqt : qt_lo;
  if (qt_lo > 0) {
    const int rows = qt_lo * kT < Sq ? qt_lo * kT : Sq;
    const long long work = static_cast<long long>(B) * rows * Hq * (kD / 8);
    const int blocks = static_cast<int>(work / 256 + 1 < 4096 ? work / 256 + 1 : 4096);
    fp8_attn_empty_rows_kernel<<<blocks, 256, 0, stream>>>(B, Sq, Hq, rows,
                                                          static_cast<uint16_t*>(o), lse);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (qt_lo == nqt) return cudaSuccess;
  // BSND tensors viewed as (d, head, s, b): a box is 128 rows of one head
  CUtensorMap qm, km, vm;
  const uint32_t box[4] = {static_cast<uint32_t>(kD), 1u, static_cast<uint32_t>(kT), 1u};
  const uint64_t qdims[4] = {static_cast<uint64_t>(D), static_cast<uint64_t>(Hq),
                             static_cast<uint64_t>(Sq), static_cast<uint64_t>(B)};
  const uint64_t qstr[3] = {static_cast<uint64_t>(D), static_cast<uint64_t>(Hq) * D,
                            static_cast<uint64_t>(Sq) * Hq * D};
  const uint64_t kdims[4] = {static_cast<uint64_t>(D), static_cast<uint64_t>(Hkv),
                             static_cast<uint64_t>(Sk), static_cast<uint64_t>(B)};
  const uint64_t kstr[3] = {static_cast<uint64_t>(D), static_cast<uint64_t>(Hkv) * D,
                            static_cast<uint64_t>(Sk) * Hkv * D};
  if (encode_tensor_map(&qm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(q), qdims, qstr,
                        box, CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS ||
      encode_tensor_map(&km, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(k), kdims, kstr,
                        box, CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS ||
      encode_tensor_map(&vm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(v), kdims, kstr,
                        box, CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS) {
    *status = QPKV_ERR_CUDA;
    return cudaErrorInvalidValue;
  }
  AttnArgs a;
  a.B = B;
  a.Sq = Sq;
  a.Sk = Sk;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.G = Hq / Hkv;
  a.qt_lo = qt_lo;
  a.nq = nqt - qt_lo;
  a.pairs = (a.nq + 1) / 2;
  a.units = B * Hq * a.pairs;
  a.causal = causal ? 1 : 0;
  a.scale_log2 = (softmax_scale > 0.f ? softmax_scale : 1.0f / sqrtf(static_cast<float>(D))) * kLog2e;
  a.qd = q_descale;
  a.kd = k_descale;
  a.vd = v_descale;
  a.o = static_cast<uint16_t*>(o);
  a.lse = lse;
  a.err = error_word;
  cudaError_t e = cudaFuncSetAttribute(fp8_attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int grid = a.units < sms ? a.units : sms;
  fp8_attn_kernel<<<grid, kThreads, kSmem, stream>>>(qm, km, vm, a);
  return cudaGetLastError();
}

}  // namespace qpkv
