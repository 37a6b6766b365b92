// Dense FP8 attention forward with per-(batch, head) descales
// ("[Triton] FP8 with FA v3 API": flash_attn_func(q_fp8, k_fp8, v_fp8,
// softmax_scale, causal, q_descale, k_descale, v_descale)):
//   O = softmax(scale * qd * kd * Q8 K8^T + mask) * V8 * vd
// Q/K/V are E4M3 codes in BSND layout, descales fp32 [B, heads of that
// tensor], O bf16 BSND, lse (natural log) fp32 [B, Sq, Hq].  Causal masking
// is bottom-right aligned: key j is visible to query i iff j <= i + Sk - Sq.
//
// One persistent CTA per SM, 10 warps:
//   warp 0     TMA loads: the work item's 128-row Q tile, then its K and V
//              tiles in the ring order K(0) K(1) K(2) | V(0) K(3) | V(1) ...
//   warps 1, 10  tcgen05 MMAs, one issuing lane each (QK on warp 1, PV on
//              warp 10):
//                S[128 q x 128 k] = Q[128 x D] . K_tile[128 x D]^T   (FP8)
//                O[128 q x D]   += P[128 q x 128 k] . V_tile[128 k x D]
//              P is read straight from tensor memory, where the softmax
//              wrote it into a P buffer as two E4M3 terms hi + lo (K = 256: hi rows, then lo rows, each
//              against the same V tile), about 8 significant bits;
//   warps 2-9  online softmax, two threads per query row (TMEM lane): warps
//              2-5 take the row's keys [0, 64), warps 6-9 keys [64, 128);
//              the pair combines its maxima through shared memory at a
//              64-thread named barrier.  The running maximum moves only
//              when a tile beats it by more than 2^8, then the row's O is
//              rescaled.  At the end of a work item the same threads write
//              O / l * vd as bf16 and the lse.
// TMEM holds two S buffers, two P buffers (64 columns each) and O: QK(t)
// waits only for the softmax to have read S(t-2), and the softmax writes
// P(t) once PV(t-2) has read that P buffer, so the in-order tensor pipe
// never holds QK back behind a late PV.
//
// Work: a unit is the pair of q tiles (t, n-1-t) of one (batch, head), so
// every unit costs the same number of causal K/V tiles; units are dealt to
// the CTAs round-robin in (batch, head) order, so the CTAs running at the
// same time share a few heads' K/V through L2.
#include <cmath>

#include "common.cuh"
#include "internal.h"
#include "ring_sched.cuh"

namespace qpkv {
namespace {

constexpr int kT = 128;             // q rows per tile = keys per tile = MMA M and N
constexpr int kD = 128;             // head dim
constexpr int kThreads = 352;       // 11 warps
constexpr int kWarpLoad = 0, kWarpMma = 1, kWarpPv = 10;   // softmax + epilogue: warps 2..9
constexpr int kSoftmax = 256;       // two threads per query row
constexpr int kStages = 8;         // K/V ring, 16 KB each
constexpr int kTileBytes = kT * kD; // one E4M3 tile
constexpr int kSmem = (2 + kStages) * kTileBytes + 1024;
constexpr float kRescaleLog2 = 8.0f;
constexpr int kSBufs = 2;           // S ring in TMEM: QK(t) waits for the softmax to read S(t-2)
constexpr int kPBufs = 2;           // P ring in TMEM: P(t) waits for PV(t-2)
constexpr uint32_t kColS = 0;       // S buffers: columns [0, 128), [128, 256)
constexpr uint32_t kColP = 256;     // P buffers: columns [256, 320), [320, 384)
constexpr uint32_t kColO = 384;     // O: columns [384, 512)

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
  uint64_t full[kStages], empty[kStages];
  uint64_t q_full[2], q_free[2];
  uint64_t s_full[kSBufs], s_free[kSBufs];   // QK(t) written / read by the softmax
  uint64_t p_ready[kPBufs];
  uint64_t pv_done[kPBufs];    // PV step t completes a phase of pv_done[t % 2]
  uint64_t o_full, o_free;      // one phase per work item
  uint64_t mma_done[2];         // QK and PV issuers' MMAs complete
  float pmax[2][2][kT];        // [tile parity][column half][row] partial row maxima
  float psum[2][kT];           // [column half][row] partial softmax denominators
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

// 2^x by the hardware approximation (relative error ~2^-22; -inf -> 0).
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// This CTA's work items in order: units blockIdx.x, +grid, ...; a unit is
// q tiles t and nq-1-t (t once when they coincide) of one (batch, head).
struct Items {
  int unit, second;
  __device__ __forceinline__ void start() {
    unit = static_cast<int>(blockIdx.x);
    second = 0;
  }
  __device__ __forceinline__ bool valid(const AttnArgs& a) const { return unit < a.units; }
  __device__ __forceinline__ void get(const AttnArgs& a, int& b, int& h, int& qt) const {
    const int bh = unit / a.pairs, t = unit % a.pairs;
    b = bh / a.Hq;
    h = bh % a.Hq;
    qt = a.qt_lo + (second ? a.nq - 1 - t : t);
  }
  __device__ __forceinline__ void advance(const AttnArgs& a) {
    const int t = unit % a.pairs;
    if (!second && a.nq - 1 - t != t) {
      second = 1;
    } else {
      second = 0;
      unit += static_cast<int>(gridDim.x);
    }
  }
};

// K/V tiles of q tile qt: keys [0, last] with last the final key any of its
// rows sees.
__device__ __forceinline__ int kv_tiles(const AttnArgs& a, int qt) {
  int last = a.Sk - 1;
  if (a.causal) last = min(last, qt * kT + kT - 1 + a.Sk - a.Sq);
  return last < 0 ? 0 : last / kT + 1;
}

__global__ void __launch_bounds__(kThreads, 1)
    fp8_attn_kernel(const __grid_constant__ CUtensorMap q_map,
                    const __grid_constant__ CUtensorMap k_map,
                    const __grid_constant__ CUtensorMap v_map, const AttnArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint8_t* sQ = smem;                       // [2] Q tiles
  uint8_t* sRing = smem + 2 * kTileBytes;   // [kStages] K or V tiles
  __shared__ Shared sh;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sh.full[s], 1);
      mbar_init(&sh.empty[s], 1);
    }
    for (int d = 0; d < 2; ++d) {
      mbar_init(&sh.q_full[d], 1);
      mbar_init(&sh.q_free[d], 1);
    }
    for (int b = 0; b < kSBufs; ++b) {
      mbar_init(&sh.s_full[b], 1);
      mbar_init(&sh.s_free[b], kSoftmax);
    }
    for (int b = 0; b < kPBufs; ++b) {
      mbar_init(&sh.p_ready[b], kSoftmax);
    }
    mbar_init(&sh.o_full, 1);
    mbar_init(&sh.o_free, kSoftmax);
    for (int b = 0; b < kPBufs; ++b) mbar_init(&sh.pv_done[b], 1);
    mbar_init(&sh.mma_done[0], 1);
    mbar_init(&sh.mma_done[1], 1);
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
    if (lane == 0) {
      tma_prefetch_desc(&q_map);
      tma_prefetch_desc(&k_map);
      tma_prefetch_desc(&v_map);
      Items it;
      it.start();
      int ib0 = 0, ib1 = 0, ih0 = 0, ih1 = 0;   // batch and kv head of the items in flight
      auto open_item = [&](int o) -> int {
        if (!it.valid(a)) return 0;
        int b, h, qt;
        it.get(a, b, h, qt);
        it.advance(a);
        if (o & 1) { ib1 = b; ih1 = h / a.G; } else { ib0 = b; ih0 = h / a.G; }
        const int qb = o & 1;
        if (!awaitb(&sh.q_free[qb], ((o >> 1) & 1) ^ 1, sh, a.err)) return -1;
        mbar_arrive_expect_tx(&sh.q_full[qb], kTileBytes);
        tma_load_4d(sQ + qb * kTileBytes, &q_map, &sh.q_full[qb], 0, h, qt * kT, b);
        return kv_tiles(a, qt);
      };
      int pos = 0;
      auto emit = [&](int o, int j, bool is_v) -> bool {
        const int s = pos % kStages;
        if (!awaitb(&sh.empty[s], ((pos / kStages) & 1) ^ 1, sh, a.err)) return false;
        mbar_arrive_expect_tx(&sh.full[s], kTileBytes);
        const int b = (o & 1) ? ib1 : ib0, hk = (o & 1) ? ih1 : ih0;
        tma_load_4d(sRing + s * kTileBytes, is_v ? &v_map : &k_map, &sh.full[s], 0, hk, j * kT, b);
        ++pos;
        return true;
      };
      RingSched q{0, 0, 0, 0, 0, 0, 0, false, 3};
      q.ntl0 = open_item(0);
      if (q.ntl0 > 0) {
        while (true) {
          const int step = ring_next(q, open_item);
          if (step == kStepK) {
            if (!emit(q.ko, q.kj, false)) break;
            ++q.kj;
            ++q.lead;
          } else if (step == kStepV) {
            if (!emit(q.vo, q.vj, true)) break;
            ++q.vj;
            --q.lead;
          } else {
            break;
          }
        }
      }
      // this CTA's copies in flight land before it exits
      for (int i = pos > kStages ? pos - kStages : 0; i < pos; ++i)
        drain(&sh.full[i % kStages], (i / kStages) & 1, a.err);
    }
    __syncwarp();
  } else if (warp == kWarpMma || warp == kWarpPv) {
    // -------------------------------------------------------------- MMA
    // Lane 0 of warp 1 issues the QK MMAs, lane 0 of warp 10 the PV MMAs;
    // both walk the ring schedule and skip the other side's stages.  QK(t)
    // overwrites the S buffer that held P(t-3), so it first waits for
    // PV(t-3) to complete.
    const bool is_qk = warp == kWarpMma;
    if (lane == 0) {
      const uint32_t idesc_qk = make_idesc(kFmtE4M3, kFmtE4M3, 0, 0, kT, kT);
      const uint32_t idesc_pv = make_idesc(kFmtE4M3, kFmtE4M3, 0, 1, kT, kD);
      // descriptors at offset 0 of each region; an operand at byte offset x
      // adds x >> 4 to the start-address field
      const uint64_t qdesc0 = make_smem_desc(smem_u32(sQ), 16, 1024, kSwizzle128B);
      const uint64_t kdesc0 = make_smem_desc(smem_u32(sRing), 16, 1024, kSwizzle128B);
      const uint64_t vdesc0 = make_smem_desc(smem_u32(sRing), 0, 1024, kSwizzle128B);
      Items it;
      it.start();
      auto open_item = [&](int o) -> int {
        if (!it.valid(a)) return 0;
        int b, h, qt;
        it.get(a, b, h, qt);
        it.advance(a);
        if (is_qk && !awaitb(&sh.q_full[o & 1], (o >> 1) & 1, sh, a.err)) return -1;
        return kv_tiles(a, qt);
      };
      int pos = 0, st = 0, pvc = 0;
      auto qk = [&](int o, int j, int ntl) -> bool {
        const int sb = st % kSBufs;
        const int s = pos % kStages;
        if (st >= kSBufs &&
            !awaitb(&sh.s_free[sb], ((st - kSBufs) / kSBufs) & 1, sh, a.err))   // S(st - 2) read
          return false;
        if (!awaitb(&sh.full[s], (pos / kStages) & 1, sh, a.err)) return false;
        tc_fence_after_sync();
        const uint64_t da0 = qdesc0 + static_cast<uint64_t>(((o & 1) * kTileBytes) >> 4);
        const uint64_t db0 = kdesc0 + static_cast<uint64_t>((s * kTileBytes) >> 4);
#pragma unroll
        for (int kk = 0; kk < kD / 32; ++kk)
          tc_mma_f8(tmem + kColS + sb * kT, da0 + 2 * kk, db0 + 2 * kk, idesc_qk, kk > 0);
        tc_commit(&sh.empty[s]);
        tc_commit(&sh.s_full[sb]);
        if (j == ntl - 1) tc_commit(&sh.q_free[o & 1]);
        ++pos;
        ++st;
        return true;
      };
      auto pv = [&](int o, int j, int ntl) -> bool {
        const int sb = pvc % kPBufs;
        const int s = pos % kStages;
        // O is single-buffered: item o-1's epilogue has read it
        if (j == 0 && !awaitb(&sh.o_free, (o & 1) ^ 1, sh, a.err)) return false;
        if (!awaitb(&sh.p_ready[sb], (pvc / kPBufs) & 1, sh, a.err) ||
            !awaitb(&sh.full[s], (pos / kStages) & 1, sh, a.err))
          return false;
        tc_fence_after_sync();
        const uint64_t db0 = vdesc0 + static_cast<uint64_t>((s * kTileBytes) >> 4);
        // K = 256: the hi terms of keys 0..127, then the lo terms, both
        // against the same V rows
#pragma unroll
        for (int kk = 0; kk < 2 * kT / 32; ++kk)
          tc_mma_f8_tmem_a(tmem + kColO, tmem + kColP + sb * 64 + 8 * kk,
                           db0 + (32 * kD / 16) * (kk & 3), idesc_pv, (j > 0 || kk > 0) ? 1u : 0u);
        tc_commit(&sh.empty[s]);
        tc_commit(&sh.pv_done[sb]);
        if (j == ntl - 1) tc_commit(&sh.o_full);
        ++pos;
        ++pvc;
        return true;
      };
      RingSched q{0, 0, 0, 0, 0, 0, 0, false, 3};
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
      drain(&sh.mma_done[is_qk ? 0 : 1], 0, a.err);
    }
    __syncwarp();
  } else if (warp < kWarpPv) {
    // ---------------------------------------------- softmax and epilogue
    // Two threads per query row: warps 2-5 take columns [0, 64), warps
    // 6-9 columns [64, 128) of the same TMEM lanes; a row's pair meets at a
    // 64-thread named barrier to combine the row maximum.
    const int sw = warp & 3;                      // TMEM lane quarter
    const int half = (warp - 2) >> 2;             // column half
    const int r = sw * 32 + lane;                 // tile row = TMEM lane
    const uint32_t bar_id = 1 + sw;               // the pair's named barrier
    const uint32_t lane_base = static_cast<uint32_t>(sw * 32) << 16;
    Items it;
    it.start();
    int st = 0;
    for (int o = 0; it.valid(a); ++o) {
      int b, h, qt;
      it.get(a, b, h, qt);
      it.advance(a);
      const int nkv = kv_tiles(a, qt);
      const int hk = h / a.G;
      // logit multiplier (log2 units); kept above 0 so that -inf * sc stays -inf
      const float sc = fmaxf(a.scale_log2 * __ldg(a.qd + b * a.Hq + h) * __ldg(a.kd + b * a.Hkv + hk),
                             1e-30f);
      const int row = qt * kT + r;
      // last key this row sees (may be negative: none)
      const int lim = a.causal ? min(a.Sk - 1, row + a.Sk - a.Sq) : a.Sk - 1;
      float m = -INFINITY, l = 0.f;
      for (int j = 0; j < nkv; ++j) {
        const int sb = st % kSBufs;
        awaitb(&sh.s_full[sb], (st / kSBufs) & 1, sh, a.err);
        __syncwarp();   // converged before the .sync.aligned TMEM accesses
        tc_fence_after_sync();
        const uint32_t srow = tmem + lane_base + kColS + sb * kT;
        const int climit = lim - j * kT - 64 * half;   // this half's columns c <= climit are visible
        const bool whole = climit >= 63;
        uint32_t v0[32], v1[32];
        tmem_ld32(srow + 64 * half, v0);
        tmem_ld32(srow + 64 * half + 32, v1);
        tmem_ld_wait();
        tc_fence_before_sync();
        mbar_arrive(&sh.s_free[sb]);   // QK(st + 2) may overwrite this S buffer
        // raw logits; masked keys -inf (sc > 0, so max and order carry over)
        float x[64];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          x[i] = __uint_as_float(v0[i]);
          x[32 + i] = __uint_as_float(v1[i]);
        }
        if (!whole) {
#pragma unroll
          for (int c = 0; c < 64; ++c)
            if (c > climit) x[c] = -INFINITY;
        }
        // row maximum in eight independent chains (a single chain of 64
        // dependent max operations is latency-bound)
        float xm8[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) xm8[i] = x[i];
#pragma unroll
        for (int c = 8; c < 64; ++c) xm8[c & 7] = fmaxf(xm8[c & 7], x[c]);
        float xm = fmaxf(fmaxf(fmaxf(xm8[0], xm8[1]), fmaxf(xm8[2], xm8[3])),
                         fmaxf(fmaxf(xm8[4], xm8[5]), fmaxf(xm8[6], xm8[7])));
        sh.pmax[st & 1][half][r] = xm;
        named_barrier(bar_id, 64);
        xm = fmaxf(xm, sh.pmax[st & 1][half ^ 1][r]);
        const float mx = xm * sc;   // the row's tile maximum in log2 units
        // ---- running maximum, moved only by more than 2^8; then O is
        // rescaled.  Both threads of a row take the same decision; the
        // TMEM access is warp-wide (.sync.aligned), rows that keep their
        // maximum use the factor 1.
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
          // the previous PV of this item must have finished writing O (PV
          // step t-1 may still be in flight; t+1 cannot be done)
          awaitb(&sh.pv_done[(st - 1) % kPBufs], ((st - 1) / kPBufs) & 1, sh, a.err);
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
        // ---- P = 2^(x sc - m) as two E4M3 terms hi + lo (about 8
        // significant bits, built in f16x2), packed four keys per column
        const float nm = m > -INFINITY ? -m : 0.f;   // a row that sees no key gets p = 0
        uint32_t pk[16], pl[16];
        float ls[4] = {0.f, 0.f, 0.f, 0.f};   // four independent sum chains
#pragma unroll
        for (int wq = 0; wq < 16; ++wq) {
          float p[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            p[e] = fast_exp2(fmaf(x[4 * wq + e], sc, nm));
            ls[e] += p[e];
          }
          const uint32_t f01 = f32x2_to_f16x2(p[1], p[0]);
          const uint32_t f23 = f32x2_to_f16x2(p[3], p[2]);
          const uint16_t h01 = f16x2_to_e4m3x2(f01);
          const uint16_t h23 = f16x2_to_e4m3x2(f23);
          const uint16_t l01 = f16x2_to_e4m3x2(f16x2_sub(f01, e4m3x2_to_f16x2(h01)));
          const uint16_t l23 = f16x2_to_e4m3x2(f16x2_sub(f23, e4m3x2_to_f16x2(h23)));
          pk[wq] = h01 | (static_cast<uint32_t>(h23) << 16);
          pl[wq] = l01 | (static_cast<uint32_t>(l23) << 16);
        }
        l += (ls[0] + ls[1]) + (ls[2] + ls[3]);
        // the P buffer of step st was read by PV(st - 2)
        const int pb = st % kPBufs;
        if (st >= kPBufs) {
          awaitb(&sh.pv_done[pb], ((st - kPBufs) / kPBufs) & 1, sh, a.err);
          __syncwarp();
          tc_fence_after_sync();
        }
        const uint32_t prow = tmem + lane_base + kColP + pb * 64;
        tmem_st16(prow + 16 * half, pk);        // columns [0, 32): hi terms
        tmem_st16(prow + 32 + 16 * half, pl);   // columns [32, 64): lo terms
        tmem_st_wait();
        tc_fence_before_sync();
        mbar_arrive(&sh.p_ready[pb]);
        ++st;
      }
      // ---- the row's denominator: this half's partial sum plus the other's
      sh.psum[half][r] = l;
      named_barrier(bar_id, 64);
      const float lt = l + sh.psum[half ^ 1][r];
      named_barrier(bar_id, 64);   // psum may be rewritten at the next item
      // ---- epilogue: this half's 64 columns of O / l * vd -> bf16, and the
      // lse, once the item's last PV has landed; then O is free for item o+2
      const float vd = __ldg(a.vd + b * a.Hkv + hk);
      const float so = lt > 0.f ? vd / lt : 0.f;
      awaitb(&sh.o_full, o & 1, sh, a.err);
      __syncwarp();
      tc_fence_after_sync();
      const bool write = row < a.Sq;
      uint16_t* out = a.o + ((static_cast<size_t>(b) * a.Sq + row) * a.Hq + h) * kD + 64 * half;
      const uint32_t orow = tmem + lane_base + kColO + 64 * half;
#pragma unroll 1
      for (int c2 = 0; c2 < 2; ++c2) {
        uint32_t v[32];
        tmem_ld32(orow + 32 * c2, v);
        tmem_ld_wait();
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const __nv_bfloat162 t =
              __floats2bfloat162_rn(__uint_as_float(v[2 * i]) * so, __uint_as_float(v[2 * i + 1]) * so);
          pk[i] = *reinterpret_cast<const uint32_t*>(&t);
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
        a.lse[(static_cast<size_t>(b) * a.Sq + row) * a.Hq + h] =
            lt > 0.f ? (m + log2f(lt)) * kLn2 : -INFINITY;
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
