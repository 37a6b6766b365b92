// MLA-absorb sparse paged decode ("KvQuantSparseFlashAttention" README,
// 计算公式 and 参数说明 rows query / key / value / sparse_indices /
// block_table / actual_seq_lengths_query / actual_seq_lengths_kv /
// sparse_mode / attention_mode = 2):
//   per query token t and q head h, the keys are the tokens listed in
//   sparse_indices[t, 0, :] (valid entries first, the first -1 ends the
//   list), each a 656-byte cache row: 512 INT8 nope codes, 64 bf16 rope
//   values, 4 fp32 scales of the 128-wide nope tiles.
//   K_j = [code_j * scale_j(tile) || rope_j] (576), V_j = code_j * scale_j (512)
//   O[t, h] = softmax_j(scale * q[t, h] . K_j) . V_j,   lse = logsumexp.
//
// The 128 q heads of a token share its keys, so both products are GEMMs:
// S[128 heads x n] = Q[128 x 576] . K^T and O[128 x 512] = P . V.  An fp32
// O of 128 x 512 alone fills tensor memory, so the path runs as three
// stream-ordered kernels:
//   mla_qk       one CTA per (token, 512 keys): the group's sparse ids ->
//                pool rows (block_table lookup; -1 for ids after the first
//                -1, outside [0, L_kv), or hidden by sparse_mode 3), sorted
//                by pool row and written to the workspace for the PV stage;
//                Q and dequantised-K chunks of 64 dims stream through shared
//                memory (TMA for Q, eight converter warps gather and
//                dequantise the rows), S for the four 128-key tiles
//                accumulates in tensor memory; the epilogue (12 warps)
//                writes P_tile = 2^(x - m) as bf16 with each tile's row
//                maximum m and sum
//   mla_softmax  per (token, head) row: the row's maximum M and sum L from
//                the tile statistics, P = P_tile * 2^(m - M) / L in place,
//                and the lse
//   mla_pv       one CTA per (token, 128 output columns = one scale tile):
//                P chunks by TMA, V chunks dequantised by the converter
//                warps, O[128 x 128] in tensor memory, bf16 out.
// Dequantisation rounds code * scale (fp32 product) once to bf16.
#include <climits>
#include <cmath>

#include "common.cuh"
#include "internal.h"

namespace qpkv {
namespace {

constexpr int kQN = 128;            // q heads per token (MMA M)
constexpr int kDqk = 576, kDv = 512;
constexpr int kRow = 656;           // cache row bytes
constexpr int kScaleOff = 640;      // byte offset of the 4 fp32 tile scales
constexpr int kChunks = kDqk / 64;  // 9 chunks of 64 dims (8 nope, 1 rope)
constexpr int kKeysQk = 512;        // keys per QK CTA (4 S tiles of 128)
constexpr int kThreads = 448;       // 14 warps
constexpr int kWarpTma = 0, kWarpMma = 1, kConv0 = 2, kNConv = 8, kEpi0 = 10;
constexpr int kConvThreads = kNConv * 32;

struct MlaArgs {
  int T, QN, Sp, S;         // tokens, q heads, padded key count, sparse_indices row length
  int sbs;                  // tokens per listed id (sparse_block_size)
  int bs, P, bt_stride, B, mode;
  float scale_log2;
  const int32_t* cu_q;
  const int32_t* lk;
  const int32_t* bt;
  const int32_t* idx;       // [T, 1, S]
  const uint8_t* pool;      // [P * bs, 656]
  int32_t* rows;            // [T, Sp] pool row per key, -1 = masked
  float* stats;             // [T, 128, Sp / 128, 2] tile (max, sum)
  uint16_t* p;              // [T, 128, Sp] bf16: 2^(x - m_tile), then the normalised P
  uint16_t* o;              // [T, QN, 512] bf16
  float* lse;               // [T, QN] or null
  int* err;
};

__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, int* err) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > kWaitTimeoutCycles) {
      report_error(err, kDevErrTimeout);
      return false;
    }
  }
  return true;
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

// Four INT8 codes times a scale -> two bf16x2 words (code exact in fp32 by
// the 2^23 + 128 + code encoding, one rounding of the product, one to bf16).
__device__ __forceinline__ void dequant4(uint32_t w, float s, uint32_t& lo, uint32_t& hi) {
  const uint32_t u = w ^ 0x80808080u;
  const float bias = 8388736.0f;   // 2^23 + 128
  const float c0 = __uint_as_float(prmt(u, 0x4B000000u, 0x7540u)) - bias;
  const float c1 = __uint_as_float(prmt(u, 0x4B000000u, 0x7541u)) - bias;
  const float c2 = __uint_as_float(prmt(u, 0x4B000000u, 0x7542u)) - bias;
  const float c3 = __uint_as_float(prmt(u, 0x4B000000u, 0x7543u)) - bias;
  const __nv_bfloat162 a = __floats2bfloat162_rn(c0 * s, c1 * s);
  const __nv_bfloat162 b = __floats2bfloat162_rn(c2 * s, c3 * s);
  lo = *reinterpret_cast<const uint32_t*>(&a);
  hi = *reinterpret_cast<const uint32_t*>(&b);
}

// 16 codes (one uint4) times s -> 16 bf16 as two 16-byte pieces.
__device__ __forceinline__ void dequant16(const uint4& w, float s, uint4& p0, uint4& p1) {
  dequant4(w.x, s, p0.x, p0.y);
  dequant4(w.y, s, p0.z, p0.w);
  dequant4(w.z, s, p1.x, p1.y);
  dequant4(w.w, s, p1.z, p1.w);
}


// ---------------------------------------------------------- keys -> rows
// Key j of token t is token id * sbs + j % sbs of the listed id
// list[j / sbs] (sbs = sparse_block_size, 1 for token-wise lists) and
// becomes a pool row, or -1: past the list (the first -1 of the token's
// list ends it), a block outside the sequence (flagged), a block token at
// or past L_kv, hidden by the right-down causal rule of sparse_mode 3, or on
// a page id outside the pool (flagged).
struct TokenSeq {
  int nv;        // listed ids before the first -1
  int b;         // the token's sequence
  bool has_seq;
  int Lq, i, Lk;
};

__device__ __forceinline__ TokenSeq token_seq(const MlaArgs& a, int t, int nv) {
  int lo = 0, hi = a.B - 1;   // the sequence of token t: first b with cu[b] > t
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (a.cu_q[mid] > t) hi = mid; else lo = mid + 1;
  }
  TokenSeq q;
  q.nv = nv;
  q.b = lo;
  q.has_seq = a.cu_q[lo] > t;
  const int begin = lo > 0 ? a.cu_q[lo - 1] : 0;
  q.Lq = a.cu_q[lo] - begin;
  q.i = t - begin;
  q.Lk = a.lk[lo];
  return q;
}

__device__ __forceinline__ int key_row(const MlaArgs& a, const int32_t* ids, const TokenSeq& q,
                                       int j) {
  const int li = j / a.sbs;
  if (!q.has_seq || li >= q.nv) return -1;
  const int id = ids[li];
  const long long tok = static_cast<long long>(id) * a.sbs + (j - li * a.sbs);
  const long long rows_bt = static_cast<long long>(a.bt_stride) * a.bs;
  if (id < 0 || static_cast<long long>(id) * a.sbs >= q.Lk ||
      static_cast<long long>(id) * a.sbs >= rows_bt) {
    if (j == li * a.sbs) report_error(a.err, kDevErrBadIndex);
    return -1;
  }
  if (tok >= q.Lk || tok >= rows_bt || (a.mode == 3 && tok > q.i + q.Lk - q.Lq)) return -1;
  const int kt = static_cast<int>(tok);
  const int pg = a.bt[static_cast<size_t>(q.b) * a.bt_stride + kt / a.bs];
  if (pg < 0 || pg >= a.P) {
    report_error(a.err, kDevErrBadPage);
    return -1;
  }
  return pg * a.bs + kt % a.bs;
}

// ------------------------------------------------------------------- QK
constexpr int kQkStage = 16384 + 4 * 16384;          // Q chunk + K chunk of 4 tiles
constexpr int kQkSmem = 2 * kQkStage + 1024;

struct QkShared {
  uint64_t q_full[2], k_full[2], empty[2], s_full, mma_done;
  uint32_t tmem_base;
};

__global__ void __launch_bounds__(kThreads, 1)
    mla_qk_kernel(const __grid_constant__ CUtensorMap q_map, const MlaArgs a, int ngroups) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  __shared__ QkShared sh;
  __shared__ __align__(16) uint8_t key_ok[kKeysQk];   // key of this CTA has a pool row
  __shared__ int srt[kKeysQk];                         // the group's rows being sorted
  __shared__ int first_neg;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int t = static_cast<int>(blockIdx.x) / ngroups, g = static_cast<int>(blockIdx.x) % ngroups;
  const int key0 = g * kKeysQk;
  const int nt = min(4, (a.Sp - key0) / 128);      // S tiles of this CTA
  if (tid == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(&sh.q_full[s], 1);
      mbar_init(&sh.k_full[s], kConvThreads);
      mbar_init(&sh.empty[s], 1);
    }
    mbar_init(&sh.s_full, 1);
    mbar_init(&sh.mma_done, 1);
    fence_mbar_init();
  }
  if (warp == kWarpMma) tmem_alloc(&sh.tmem_base, 512);
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = sh.tmem_base;

  if (warp == kWarpTma) {
    if (lane == 0) {
      tma_prefetch_desc(&q_map);
      for (int c = 0; c < kChunks; ++c) {
        const int s = c & 1;
        if (!wait_bar(&sh.empty[s], ((c >> 1) & 1) ^ 1, a.err)) break;
        mbar_arrive_expect_tx(&sh.q_full[s], 16384);
        tma_load_3d(smem + s * kQkStage, &q_map, &sh.q_full[s], 64 * c, 0, t);
      }
    }
    __syncwarp();
  } else if (warp == kWarpMma) {
    if (lane == 0) {
      const uint32_t idesc = make_idesc(kFmtBF16, kFmtBF16, 0, 0, 128, 128);
      const uint64_t desc0 = make_smem_desc(smem_u32(smem), 16, 1024, kSwizzle128B);
      for (int c = 0; c < kChunks; ++c) {
        const int s = c & 1;
        if (!wait_bar(&sh.q_full[s], (c >> 1) & 1, a.err) ||
            !wait_bar(&sh.k_full[s], (c >> 1) & 1, a.err))
          break;
        tc_fence_after_sync();
        const uint64_t qd = desc0 + static_cast<uint64_t>((s * kQkStage) >> 4);
        for (int n = 0; n < nt; ++n) {
          const uint64_t kd = qd + static_cast<uint64_t>(((n + 1) * 16384) >> 4);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            tc_mma_f16(tmem + 128 * n, qd + 2 * kk, kd + 2 * kk, idesc, (c > 0 || kk > 0) ? 1u : 0u);
        }
        tc_commit(&sh.empty[s]);
      }
      tc_commit(&sh.s_full);
      tc_commit(&sh.mma_done);
      wait_bar(&sh.mma_done, 0, a.err);
    }
    __syncwarp();
  } else if (warp < kEpi0) {
    // ------------------------------------------------ gather + dequant
    // Lane j of the converter warps owns keys j and j + 256 of the group.
    // Units 0-7: the 64 nope codes of chunk u of both keys; 8, 9: the 64
    // rope values of the first / second key.  The next unit's loads are
    // in flight while a unit is converted.
    const int lj = tid - kConv0 * 32;
    const int ka = lj, kb = lj + 256;
    int32_t* rws = a.rows + static_cast<size_t>(t) * a.Sp + key0;
    // The pool rows of the group's keys (the first -1 of the token's list
    // ends it) ...
    const int32_t* ids = a.idx + static_cast<size_t>(t) * a.S;
    if (lj == 0) first_neg = a.S;
    named_barrier(2, kConvThreads);
    for (int j = lj; j < a.S; j += kConvThreads)
      if (__ldg(ids + j) == -1) atomicMin(&first_neg, j);
    named_barrier(2, kConvThreads);
    const TokenSeq tq = token_seq(a, t, first_neg);
    const int r0 = ka < 128 * nt ? key_row(a, ids, tq, key0 + ka) : -1;
    const int r1 = kb < 128 * nt ? key_row(a, ids, tq, key0 + kb) : -1;
    // ... sorted by pool row (rows of -1 last): attention does not depend on
    // the order of the keys, and the gathers then walk the pool in
    // ascending order, neighbouring lanes on neighbouring pages.  The sorted
    // rows go to the workspace for the PV stage.
    srt[ka] = r0 >= 0 ? r0 : INT_MAX;
    srt[kb] = r1 >= 0 ? r1 : INT_MAX;
    named_barrier(2, kConvThreads);
    for (int k = 2; k <= kKeysQk; k <<= 1) {
      for (int h = k >> 1; h > 0; h >>= 1) {
        const int i = (lj / h) * 2 * h + lj % h, o = i + h;   // one pair per thread
        const int x = srt[i], y = srt[o];
        if ((x > y) == ((i & k) == 0)) {
          srt[i] = y;
          srt[o] = x;
        }
        named_barrier(2, kConvThreads);
      }
    }
    const int ra = srt[ka] != INT_MAX ? srt[ka] : -1;
    const int rb = srt[kb] != INT_MAX ? srt[kb] : -1;
    if (ka < 128 * nt) rws[ka] = ra;
    if (kb < 128 * nt) rws[kb] = rb;
    key_ok[ka] = ra >= 0;
    key_ok[kb] = rb >= 0;
    const uint8_t* pa = ra >= 0 ? a.pool + static_cast<size_t>(ra) * kRow : nullptr;
    const uint8_t* pb = rb >= 0 ? a.pool + static_cast<size_t>(rb) * kRow : nullptr;
    const uint4 z = make_uint4(0, 0, 0, 0);
    const uint4 sca = pa ? __ldg(reinterpret_cast<const uint4*>(pa + kScaleOff)) : z;
    const uint4 scb = pb ? __ldg(reinterpret_cast<const uint4*>(pb + kScaleOff)) : z;
    auto load = [&](int u, uint4 (&w)[8]) {
      if (u < 8) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          w[i] = pa ? __ldg(reinterpret_cast<const uint4*>(pa + 64 * u) + i) : z;
          w[4 + i] = pb ? __ldg(reinterpret_cast<const uint4*>(pb + 64 * u) + i) : z;
        }
      } else {
        const uint8_t* pr = u == 8 ? pa : pb;
#pragma unroll
        for (int i = 0; i < 8; ++i)
          w[i] = pr ? __ldg(reinterpret_cast<const uint4*>(pr + kDv) + i) : z;
      }
    };
    // 16-byte piece q of key k's 128-byte row inside the K chunk of a stage
    auto piece = [&](uint8_t* stage, int k, int q) -> uint4* {
      const int row = k & 127;
      return reinterpret_cast<uint4*>(stage + 16384 * (1 + (k >> 7)) + row * 128 +
                                      ((q ^ (row & 7)) << 4));
    };
    uint4 cur[8], nxt[8];
    load(0, nxt);
    for (int u = 0; u < 10; ++u) {
#pragma unroll
      for (int i = 0; i < 8; ++i) cur[i] = nxt[i];
      if (u + 1 < 10) load(u + 1, nxt);
      const int c = u < 8 ? u : 8;
      const int s = c & 1;
      uint8_t* stage = smem + s * kQkStage;
      if (u <= 8 && !wait_bar(&sh.empty[s], ((c >> 1) & 1) ^ 1, a.err)) break;
      if (u < 8) {
        const float sa = u < 2 ? __uint_as_float(sca.x) : u < 4 ? __uint_as_float(sca.y)
                       : u < 6 ? __uint_as_float(sca.z) : __uint_as_float(sca.w);
        const float sb = u < 2 ? __uint_as_float(scb.x) : u < 4 ? __uint_as_float(scb.y)
                       : u < 6 ? __uint_as_float(scb.z) : __uint_as_float(scb.w);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          uint4 p0, p1;
          dequant16(cur[i], sa, p0, p1);
          *piece(stage, ka, 2 * i) = p0;
          *piece(stage, ka, 2 * i + 1) = p1;
          dequant16(cur[4 + i], sb, p0, p1);
          *piece(stage, kb, 2 * i) = p0;
          *piece(stage, kb, 2 * i + 1) = p1;
        }
      } else {
        const int k = u == 8 ? ka : kb;
#pragma unroll
        for (int i = 0; i < 8; ++i) *piece(stage, k, i) = cur[i];
      }
      if (u != 8) {
        fence_proxy_async_smem();
        mbar_arrive(&sh.k_full[s]);
      }
    }
  }
  if (warp >= kConv0) {
    // ----------------------------------------------------------- epilogue
    // Warps 2-13 (the converters join once their units are done): quarter
    // warp & 3 of the head rows, tiles {0, 3}, {1}, {2} by (warp - 2) / 4.
    // Per tile and head row: m = the row maximum of the scaled logits
    // (masked keys -inf), P_tile = 2^(x - m) in bf16 and l = sum P_tile to
    // the workspace.
    const int sw = warp & 3, part = (warp - kConv0) >> 2, r = sw * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(sw * 32) << 16;
    named_barrier(1, kThreads - kConv0 * 32);   // the converters' key_ok flags are written
    wait_bar(&sh.s_full, 0, a.err);
    __syncwarp();
    tc_fence_after_sync();
    uint16_t* prow = a.p + (static_cast<size_t>(t) * kQN + r) * a.Sp + key0;
    const int ntile = a.Sp / 128;
    for (int n = part; n < nt; n += 3) {
      float m = -INFINITY;
#pragma unroll 1
      for (int cc = 0; cc < 4; ++cc) {
        uint32_t v[32];
        tmem_ld32(tmem + lane_base + 128 * n + 32 * cc, v);
        tmem_ld_wait();
        const int kb0 = 128 * n + 32 * cc;
#pragma unroll
        for (int i = 0; i < 32; i += 4) {
          const uchar4 rr = *reinterpret_cast<const uchar4*>(key_ok + kb0 + i);
          m = fmaxf(m, fmaxf(fmaxf(rr.x ? __uint_as_float(v[i]) : -INFINITY,
                                   rr.y ? __uint_as_float(v[i + 1]) : -INFINITY),
                             fmaxf(rr.z ? __uint_as_float(v[i + 2]) : -INFINITY,
                                   rr.w ? __uint_as_float(v[i + 3]) : -INFINITY)));
        }
      }
      m = m > -INFINITY ? m * a.scale_log2 : -INFINITY;   // scale_log2 > 0 keeps the order
      const float nm = m > -INFINITY ? -m : 0.f;
      float l = 0.f;
#pragma unroll 1
      for (int cc = 0; cc < 4; ++cc) {
        uint32_t v[32];
        tmem_ld32(tmem + lane_base + 128 * n + 32 * cc, v);
        tmem_ld_wait();
        const int kb0 = 128 * n + 32 * cc;
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 32; i += 4) {
          const uchar4 rr = *reinterpret_cast<const uchar4*>(key_ok + kb0 + i);
          const float p0 = rr.x ? fast_exp2(fmaf(__uint_as_float(v[i]), a.scale_log2, nm)) : 0.f;
          const float p1 = rr.y ? fast_exp2(fmaf(__uint_as_float(v[i + 1]), a.scale_log2, nm)) : 0.f;
          const float p2 = rr.z ? fast_exp2(fmaf(__uint_as_float(v[i + 2]), a.scale_log2, nm)) : 0.f;
          const float p3 = rr.w ? fast_exp2(fmaf(__uint_as_float(v[i + 3]), a.scale_log2, nm)) : 0.f;
          l += (p0 + p1) + (p2 + p3);
          const __nv_bfloat162 b0 = __floats2bfloat162_rn(p0, p1);
          const __nv_bfloat162 b1 = __floats2bfloat162_rn(p2, p3);
          pk[i / 2] = *reinterpret_cast<const uint32_t*>(&b0);
          pk[i / 2 + 1] = *reinterpret_cast<const uint32_t*>(&b1);
        }
        uint4* dst = reinterpret_cast<uint4*>(prow + kb0);
#pragma unroll
        for (int i = 0; i < 4; ++i) dst[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
      }
      float* st = a.stats + ((static_cast<size_t>(t) * kQN + r) * ntile + (key0 / 128 + n)) * 2;
      st[0] = m;
      st[1] = l;
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, 512);
  }
}

// -------------------------------------------------------------- softmax
// One warp per (token, head) row, eight rows per block: M and L from the
// tile statistics (warp reductions), then P = P_tile * 2^(m_tile - M) / L
// in place (bf16), eight keys per lane and step, and the lse.
__global__ void __launch_bounds__(256) mla_softmax_kernel(const MlaArgs a, int nrows) {
  const int lane = threadIdx.x & 31;
  const int row = static_cast<int>(blockIdx.x) * 8 + (threadIdx.x >> 5);   // t * 128 + h
  if (row >= nrows) return;
  const int ntile = a.Sp / 128;
  const float* st = a.stats + static_cast<size_t>(row) * ntile * 2;
  float M = -INFINITY;
  for (int i = lane; i < ntile; i += 32) M = fmaxf(M, st[2 * i]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  float L = 0.f;
  if (M > -INFINITY)
    for (int i = lane; i < ntile; i += 32)
      if (st[2 * i] > -INFINITY) L += st[2 * i + 1] * exp2f(st[2 * i] - M);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
  const float inv = L > 0.f ? 1.f / L : 0.f;
  uint16_t* pr = a.p + static_cast<size_t>(row) * a.Sp;
  for (int j = 8 * lane; j < a.Sp; j += 256) {
    const float mt = st[2 * (j / 128)];
    const float f = mt > -INFINITY ? exp2f(mt - M) * inv : 0.f;
    uint4 w = *reinterpret_cast<const uint4*>(pr + j);
    uint32_t* ww = reinterpret_cast<uint32_t*>(&w);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&ww[i]));
      const __nv_bfloat162 o = __floats2bfloat162_rn(x.x * f, x.y * f);
      ww[i] = *reinterpret_cast<const uint32_t*>(&o);
    }
    *reinterpret_cast<uint4*>(pr + j) = w;
  }
  const int t = row / kQN, h = row % kQN;
  if (lane == 0 && a.lse != nullptr && h < a.QN)
    a.lse[static_cast<size_t>(t) * a.QN + h] = L > 0.f ? (M + log2f(L)) * kLn2 : -INFINITY;
}

// ------------------------------------------------------------------- PV
// Stage: P[128 heads x 128 keys] (two K-major 64-key chunks by TMA) and
// V[128 keys x 128 columns] (two MN-major 64-column atoms written by the
// converter warps).
constexpr int kPvStages = 3;
constexpr int kPvStage = 4 * 16384;
constexpr int kPvSmem = kPvStages * kPvStage + 1024;

struct PvShared {
  uint64_t p_full[kPvStages], v_full[kPvStages], empty[kPvStages], o_full, mma_done;
  uint32_t tmem_base;
};

__global__ void __launch_bounds__(kThreads, 1)
    mla_pv_kernel(const __grid_constant__ CUtensorMap p_map, const MlaArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  __shared__ PvShared sh;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int t = static_cast<int>(blockIdx.x) >> 2, q = static_cast<int>(blockIdx.x) & 3;
  const int nsteps = a.Sp / 128;
  if (tid == 0) {
    for (int s = 0; s < kPvStages; ++s) {
      mbar_init(&sh.p_full[s], 1);
      mbar_init(&sh.v_full[s], kConvThreads);
      mbar_init(&sh.empty[s], 1);
    }
    mbar_init(&sh.o_full, 1);
    mbar_init(&sh.mma_done, 1);
    fence_mbar_init();
  }
  if (warp == kWarpMma) tmem_alloc(&sh.tmem_base, 128);
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = sh.tmem_base;

  if (warp == kWarpTma) {
    if (lane == 0) {
      tma_prefetch_desc(&p_map);
      for (int i = 0; i < nsteps; ++i) {
        const int s = i % kPvStages;
        if (!wait_bar(&sh.empty[s], ((i / kPvStages) & 1) ^ 1, a.err)) break;
        mbar_arrive_expect_tx(&sh.p_full[s], 2 * 16384);
        uint8_t* dst = smem + s * kPvStage;
        tma_load_3d(dst, &p_map, &sh.p_full[s], 128 * i, 0, t);
        tma_load_3d(dst + 16384, &p_map, &sh.p_full[s], 128 * i + 64, 0, t);
      }
    }
    __syncwarp();
  } else if (warp == kWarpMma) {
    if (lane == 0) {
      const uint32_t idesc = make_idesc(kFmtBF16, kFmtBF16, 0, 1, 128, 128);
      const uint64_t pdesc0 = make_smem_desc(smem_u32(smem), 16, 1024, kSwizzle128B);
      const uint64_t vdesc0 = make_smem_desc(smem_u32(smem + 2 * 16384), 16384, 1024, kSwizzle128B);
      for (int i = 0; i < nsteps; ++i) {
        const int s = i % kPvStages;
        if (!wait_bar(&sh.p_full[s], (i / kPvStages) & 1, a.err) ||
            !wait_bar(&sh.v_full[s], (i / kPvStages) & 1, a.err))
          break;
        tc_fence_after_sync();
        const uint64_t pd = pdesc0 + static_cast<uint64_t>((s * kPvStage) >> 4);
        const uint64_t vd = vdesc0 + static_cast<uint64_t>((s * kPvStage) >> 4);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          tc_mma_f16(tmem, pd + static_cast<uint64_t>(((kk >> 2) * 16384 + (kk & 3) * 32) >> 4),
                     vd + static_cast<uint64_t>((kk * 16 * 128) >> 4), idesc,
                     (i > 0 || kk > 0) ? 1u : 0u);
        tc_commit(&sh.empty[s]);
      }
      tc_commit(&sh.o_full);
      tc_commit(&sh.mma_done);
      wait_bar(&sh.mma_done, 0, a.err);
    }
    __syncwarp();
  } else if (warp < kEpi0) {
    // ------------------------------------------------ gather + dequant
    // Lane j: key j / 2 of each 128-key step, columns [64 (j & 1), +64) of
    // this CTA's 128-column slice (one scale tile); the next step's loads
    // are in flight while a step is converted.
    const int lj = tid - kConv0 * 32;
    const int k = lj >> 1, hc = lj & 1;
    const int32_t* rws = a.rows + static_cast<size_t>(t) * a.Sp;
    const uint4 z = make_uint4(0, 0, 0, 0);
    auto load = [&](int i, uint4 (&w)[4], float& sc) {
      const int r = rws[128 * i + k];
      if (r >= 0) {
        const uint8_t* pr = a.pool + static_cast<size_t>(r) * kRow;
        const uint4* src = reinterpret_cast<const uint4*>(pr + 128 * q + 64 * hc);
#pragma unroll
        for (int e = 0; e < 4; ++e) w[e] = __ldg(src + e);
        sc = __ldg(reinterpret_cast<const float*>(pr + kScaleOff) + q);
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) w[e] = z;
        sc = 0.f;
      }
    };
    uint4 cur[4], nxt[4];
    float scur, snxt;
    if (nsteps > 0) load(0, nxt, snxt);
    for (int i = 0; i < nsteps; ++i) {
#pragma unroll
      for (int e = 0; e < 4; ++e) cur[e] = nxt[e];
      scur = snxt;
      if (i + 1 < nsteps) load(i + 1, nxt, snxt);
      const int s = i % kPvStages;
      if (!wait_bar(&sh.empty[s], ((i / kPvStages) & 1) ^ 1, a.err)) break;
      uint8_t* vrow = smem + s * kPvStage + 2 * 16384 + hc * 16384 + k * 128;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        uint4 p0, p1;
        dequant16(cur[e], scur, p0, p1);
        *reinterpret_cast<uint4*>(vrow + (((2 * e) ^ (k & 7)) << 4)) = p0;
        *reinterpret_cast<uint4*>(vrow + (((2 * e + 1) ^ (k & 7)) << 4)) = p1;
      }
      fence_proxy_async_smem();
      mbar_arrive(&sh.v_full[s]);
    }
  } else {
    // ----------------------------------------------------------- epilogue
    const int sw = warp & 3, r = sw * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(sw * 32) << 16;
    wait_bar(&sh.o_full, 0, a.err);
    __syncwarp();
    tc_fence_after_sync();
    uint16_t* out = a.o + (static_cast<size_t>(t) * a.QN + r) * kDv + 128 * q;
#pragma unroll 1
    for (int cc = 0; cc < 4; ++cc) {
      uint32_t v[32];
      tmem_ld32(tmem + lane_base + 32 * cc, v);
      tmem_ld_wait();
      uint32_t pk[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const __nv_bfloat162 b2 = __floats2bfloat162_rn(__uint_as_float(v[2 * i]),
                                                        __uint_as_float(v[2 * i + 1]));
        pk[i] = *reinterpret_cast<const uint32_t*>(&b2);
      }
      if (r < a.QN) {
        uint4* o4 = reinterpret_cast<uint4*>(out + 32 * cc);
#pragma unroll
        for (int i = 0; i < 4; ++i) o4[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
      }
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, 128);
  }
}

struct MlaLayout {
  size_t rows, stats, p, total;
};

MlaLayout mla_layout(int T, int Sp) {
  auto up = [](size_t x) { return (x + 255) / 256 * 256; };
  MlaLayout l;
  l.rows = 0;
  l.stats = up(static_cast<size_t>(T) * Sp * 4);
  l.p = l.stats + up(static_cast<size_t>(T) * kQN * (Sp / 128) * 8);
  l.total = l.p + up(static_cast<size_t>(T) * kQN * Sp * 2);
  return l;
}

int padded_sparse(int S) { return (S + 127) / 128 * 128; }

}  // namespace

size_t mla_workspace_bytes(int num_tokens, int sparse_size) {
  return mla_layout(num_tokens, padded_sparse(sparse_size)).total;
}

cudaError_t launch_mla_sparse(const qpkv_mla_params& p, cudaStream_t stream, int* status) {
  *status = QPKV_OK;
  if (p.num_tokens == 0) return cudaSuccess;
  const int sbs = p.sparse_block_size > 1 ? p.sparse_block_size : 1;
  const int T = p.num_tokens, Sp = padded_sparse(p.sparse_size * sbs);
  const MlaLayout lay = mla_layout(T, Sp);
  uint8_t* ws = static_cast<uint8_t*>(p.workspace);
  MlaArgs a;
  a.T = T;
  a.QN = p.num_heads_q;
  a.Sp = Sp;
  a.S = p.sparse_size;
  a.sbs = sbs;
  a.bs = p.block_size;
  a.P = p.num_blocks;
  a.bt_stride = p.bt_stride;
  a.B = p.num_seqs;
  a.mode = p.sparse_mode;
  a.scale_log2 = (p.scale > 0.f ? p.scale : 1.0f / sqrtf(static_cast<float>(kDqk))) * kLog2e;
  a.cu_q = p.cu_seqlens_q;
  a.lk = p.seqlens_kv;
  a.bt = p.block_table;
  a.idx = p.sparse_indices;
  a.pool = static_cast<const uint8_t*>(p.kv_pool);
  a.rows = reinterpret_cast<int32_t*>(ws + lay.rows);
  a.stats = reinterpret_cast<float*>(ws + lay.stats);
  a.p = reinterpret_cast<uint16_t*>(ws + lay.p);
  a.o = static_cast<uint16_t*>(p.o);
  a.lse = p.lse;
  a.err = p.error_word;

  CUtensorMap qm, pm;
  const uint64_t qdims[3] = {kDqk, static_cast<uint64_t>(p.num_heads_q), static_cast<uint64_t>(T)};
  const uint64_t qstr[2] = {2ull * kDqk, 2ull * kDqk * p.num_heads_q};
  const uint64_t pdims[3] = {static_cast<uint64_t>(Sp), kQN, static_cast<uint64_t>(T)};
  const uint64_t pstr[2] = {2ull * Sp, 2ull * Sp * kQN};
  const uint32_t box[3] = {64u, 128u, 1u};
  if (encode_tensor_map(&qm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(p.q), qdims, qstr,
                        box, CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS ||
      encode_tensor_map(&pm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a.p, pdims, pstr, box,
                        CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS) {
    *status = QPKV_ERR_CUDA;
    return cudaErrorInvalidValue;
  }
  cudaError_t e = cudaFuncSetAttribute(mla_qk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kQkSmem);
  if (e != cudaSuccess) return e;
  const int ngroups = (Sp + kKeysQk - 1) / kKeysQk;
  mla_qk_kernel<<<T * ngroups, kThreads, kQkSmem, stream>>>(qm, a, ngroups);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  mla_softmax_kernel<<<(T * kQN + 7) / 8, 256, 0, stream>>>(a, T * kQN);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(mla_pv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kPvSmem);
  if (e != cudaSuccess) return e;
  mla_pv_kernel<<<T * 4, kThreads, kPvSmem, stream>>>(pm, a);
  return cudaGetLastError();
}
}  // namespace qpkv
