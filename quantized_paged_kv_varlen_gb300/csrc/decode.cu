// Split-KV paged FP8 decode and its log-sum-exp merge.
//
// What is computed ("KvQuantSparseFlashAttention" README, 计算公式, with the
// per-token-head FP8 quantisation named under 功能说明):
//   O[b, h] = softmax(sm_scale * q[b, h] . Dequant(K_b)^T) . Dequant(V_b),
//   Dequant(x)[t] = e4m3(x[t]) * scale[t],
// over the L_b cached tokens of request b gathered through block_table
// (README 参数说明 row block_table; flashinfer "Batch Decode Attention
// Kernels" plan/run split).  The host plan cuts every (request, kv head)
// into work items of <= 256 tokens; one CTA handles one item and writes an
// fp32 partial output and its log-sum-exp, and a merge kernel combines them.
//
// GB300 design (one CTA = 4 warps, up to 3 CTAs per SM):
//  * Thread 0 issues TMA boxes of whole pages ([page_size rows x D bytes] of
//    one kv head, 128-byte or 64-byte swizzle) for every K and V tile of the
//    item at once: the kernel is HBM-bound and keeps 64 KiB in flight per CTA.
//  * The contraction runs on tcgen05 with FP8 operands straight from the
//    cache bytes, in swap-AB form so the 128 cache tokens fill the MMA's M:
//      S^T[128 tok x N] = K[128 tok x D] . Qt^T      (K-major A and B)
//      O^T[D x N]      += V^T[D x 128 tok] . Pt^T    (MN-major A: V as stored)
//    The bf16 query and the fp32 probabilities are not FP8 values, so each is
//    carried as three E4M3 terms with scales s, s/16, s/256 (a 3-term split
//    keeps ~12 significant bits, more than bf16's 8); the N = 16 (or 32)
//    columns hold (term, head) pairs and are recombined in fp32 after the
//    TMEM load.  No element of K or V is ever converted.
//  * The softmax over an item is exact (all 256 logits are in TMEM at once),
//    so no running rescale is needed inside an item; the merge combines items.
//  * Per-token k-scales fold into the logits, v-scales into the probabilities.
#include <cmath>

#include "common.cuh"
#include "internal.h"

namespace qpkv {
namespace {

constexpr int kTile = 128;    // tokens per MMA tile
constexpr int kMaxTiles = 2;  // tiles per work item
constexpr int kThreads = 128;
constexpr int kTerms = 3;

template <int D, int G>
struct Cfg {
  static constexpr int kN = ((kTerms * G + 15) / 16) * 16;
  static constexpr int kTileBytes = kTile * D;
  static constexpr uint32_t kSwz = D == 128 ? kSwizzle128B : kSwizzle64B;
  static constexpr int kSBO = 8 * D;
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kOffK + kMaxTiles * kTileBytes;
  static constexpr int kOffQ = kOffV + kMaxTiles * kTileBytes;
  static constexpr int kOffP = kOffQ + ((kN * D + 1023) / 1024) * 1024;
  static constexpr int kPBytes = kN * kTile;
  static constexpr int kBytes = kOffP + kMaxTiles * kPBytes;
  static constexpr int kSmem = kBytes + 1024;
  static constexpr int kTmemO = kMaxTiles * kN;
  static constexpr int kTmemCols = (kMaxTiles + 1) * kN <= 64 ? 64 : 128;
  static constexpr int kEPT = (G * D) / kThreads > 0 ? (G * D) / kThreads : 1;
  static constexpr int kActive = G * D / kEPT;  // threads taking part in the q split
  static constexpr int kTPH = D / kEPT;          // threads per head in the q split
  static_assert(kN <= 64, "head group too large");
  static_assert(kEPT <= 8, "q split: at most 8 elements per thread");
};

struct DecodeArgs {
  const DecodeItem* items;
  const int32_t* split_off;
  int chunk;
  int Hq, Hkv;
  const uint16_t* q;
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

// max over the kTPH threads of one head group (power of two); red: >= 4 floats
template <int TPH>
__device__ __forceinline__ float head_group_max(float v, float* red) {
  if constexpr (TPH <= 32) {
#pragma unroll
    for (int o = 1; o < TPH; o <<= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
  } else {
    v = warp_max(v);
    const int warp = threadIdx.x >> 5;
    if ((threadIdx.x & 31) == 0) red[warp] = v;
    __syncthreads();
    const int first = (warp / (TPH / 32)) * (TPH / 32);
    float m = red[first];
#pragma unroll
    for (int i = 1; i < TPH / 32; ++i) m = fmaxf(m, red[first + i]);
    __syncthreads();
    return m;
  }
}

template <int D, int G>
__global__ void __launch_bounds__(kThreads, 3)
    decode_attend_kernel(const __grid_constant__ CUtensorMap k_map,
                         const __grid_constant__ CUtensorMap v_map, const DecodeArgs a) {
  using C = Cfg<D, G>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint8_t* sK = smem + C::kOffK;
  uint8_t* sV = smem + C::kOffV;
  uint8_t* sQ = smem + C::kOffQ;
  uint8_t* sP = smem + C::kOffP;

  __shared__ uint64_t bar_k[kMaxTiles], bar_v[kMaxTiles], bar_s, bar_o;
  __shared__ uint32_t tmem_base;
  __shared__ float red_a[4][G], red_b[4][G], red_c[4][G];
  __shared__ float red_q[4];
  __shared__ float sig_q[G];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const DecodeItem it = a.items[blockIdx.x];
  const int n_tok = it.t1 - it.t0;
  const int ntiles = (n_tok + kTile - 1) / kTile;
  const int ps = a.page_size;
  const int32_t* bt_row = a.block_table + static_cast<size_t>(it.b) * a.bt_stride;

  if (tid == 0) {
#pragma unroll
    for (int j = 0; j < kMaxTiles; ++j) {
      mbar_init(&bar_k[j], 1);
      mbar_init(&bar_v[j], 1);
    }
    mbar_init(&bar_s, 1);
    mbar_init(&bar_o, 1);
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(&tmem_base, C::kTmemCols);
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = tmem_base;

  // ---- producer: every K and V page box of the item, issued at once
  if (tid == 0) {
    tma_prefetch_desc(&k_map);
    tma_prefetch_desc(&v_map);
    const int R = ps < kTile ? ps : kTile;  // rows per box
    for (int tensor = 0; tensor < 2; ++tensor) {
      for (int j = 0; j < ntiles; ++j) {
        const int tok0 = it.t0 + j * kTile;
        const int tok_end = min(tok0 + kTile, it.t1);
        const int nbox = (tok_end - tok0 + R - 1) / R;
        int rows[kTile / 16];
        uint32_t bytes = 0;
        for (int r = 0; r < nbox; ++r) {
          const int tok = tok0 + r * R;
          const int page = __ldg(bt_row + tok / ps);
          if (page < 0 || page >= a.num_pages) {
            report_error(a.err, kDevErrBadPage);
            rows[r] = -1;
          } else {
            rows[r] = page * ps + (tok % ps);
            bytes += R * D;
          }
        }
        uint64_t* bar = tensor == 0 ? &bar_k[j] : &bar_v[j];
        uint8_t* dst = (tensor == 0 ? sK : sV) + j * C::kTileBytes;
        mbar_arrive_expect_tx(bar, bytes);
        for (int r = 0; r < nbox; ++r) {
          if (rows[r] < 0) continue;
          tma_load_3d(dst + r * R * D, tensor == 0 ? &k_map : &v_map, bar, 0, it.hk, rows[r]);
        }
      }
    }
  }

  // ---- per-token scales of this thread's tokens (one token per tile)
  float ks[kMaxTiles], vs[kMaxTiles];
  bool valid[kMaxTiles];
#pragma unroll
  for (int j = 0; j < kMaxTiles; ++j) {
    const int tok = it.t0 + j * kTile + tid;
    valid[j] = tok < it.t1;
    ks[j] = 0.f;
    vs[j] = 0.f;
    if (valid[j]) {
      const int page = __ldg(bt_row + tok / ps);
      if (page >= 0 && page < a.num_pages) {
        const size_t row = static_cast<size_t>(page) * ps + (tok % ps);
        ks[j] = __ldg(a.k_scale + row * a.Hkv + it.hk);
        vs[j] = __ldg(a.v_scale + row * a.Hkv + it.hk);
      }
    }
  }

  // ---- query -> three E4M3 terms per element, written as the MMA's B operand
  {
    const int g = tid / C::kTPH;
    const int d0 = (tid % C::kTPH) * C::kEPT;
    const bool active = tid < C::kActive;
    float x[C::kEPT];
    float amax = 0.f;
    if (active) {
      const uint16_t* src =
          a.q + (static_cast<size_t>(it.b) * a.Hq + it.hk * G + g) * D + d0;
#pragma unroll
      for (int e = 0; e < C::kEPT; ++e) {
        x[e] = bf16_bits_to_float(src[e]);
        amax = fmaxf(amax, fabsf(x[e]));
      }
    }
    amax = head_group_max<C::kTPH>(amax, red_q);
    const float s1 = amax * (1.0f / 448.0f);
    const float inv1 = s1 > 0.f ? 1.0f / s1 : 0.f;
    if (active) {
      if ((tid % C::kTPH) == 0) sig_q[g] = s1;
#pragma unroll
      for (int e = 0; e < C::kEPT; ++e) {
        const int d = d0 + e;
        const uint8_t c1 = f32_to_e4m3(x[e] * inv1);
        const float r1 = fmaf(-e4m3_to_f32(c1), s1, x[e]);
        const uint8_t c2 = f32_to_e4m3(r1 * inv1 * 16.0f);
        const float r2 = fmaf(-e4m3_to_f32(c2), s1 * (1.0f / 16.0f), r1);
        const uint8_t c3 = f32_to_e4m3(r2 * inv1 * 256.0f);
        sQ[swizzled_offset(0 * G + g, d, D)] = c1;
        sQ[swizzled_offset(1 * G + g, d, D)] = c2;
        sQ[swizzled_offset(2 * G + g, d, D)] = c3;
      }
    }
    // unused B rows must be zero
    for (int i = tid; i < (C::kN - kTerms * G) * D; i += kThreads)
      sQ[swizzled_offset(kTerms * G + i / D, i % D, D)] = 0;
    fence_proxy_async_smem();
  }
  __syncthreads();

  // ---- QK^T: S^T_j = K_j . Qt^T
  if (tid == 0) {
    tc_fence_after_sync();
    constexpr uint32_t idesc = make_idesc(kFmtE4M3, kFmtE4M3, 0, 0, 128, C::kN);
    for (int j = 0; j < ntiles; ++j) {
      if (!mbar_wait(&bar_k[j], 0)) report_error(a.err, kDevErrTimeout);
      tc_fence_after_sync();
#pragma unroll
      for (int kk = 0; kk < D / 32; ++kk) {
        const uint64_t da = make_smem_desc(smem_u32(sK + j * C::kTileBytes) + 32 * kk, 16,
                                           C::kSBO, C::kSwz);
        const uint64_t db = make_smem_desc(smem_u32(sQ) + 32 * kk, 16, C::kSBO, C::kSwz);
        tc_mma_f8(tmem + j * C::kN, da, db, idesc, kk > 0);
      }
    }
    tc_commit(&bar_s);
  }
  __syncwarp();

  // ---- softmax over the item (exact: every logit is in TMEM)
  if (!mbar_wait(&bar_s, 0)) report_error(a.err, kDevErrTimeout);
  tc_fence_after_sync();
  float l2[kMaxTiles][G];
#pragma unroll
  for (int j = 0; j < kMaxTiles; ++j) {
    if (j < ntiles) {
      uint32_t r[C::kN];
#pragma unroll
      for (int c = 0; c < C::kN; c += 16) {
        uint32_t part[16];
        tmem_ld16(tmem + (static_cast<uint32_t>(warp * 32) << 16) + j * C::kN + c, part);
#pragma unroll
        for (int i = 0; i < 16; ++i) r[c + i] = part[i];
      }
      tmem_ld_wait();
      const float f = a.sm_scale_log2 * ks[j];
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float s = __uint_as_float(r[g]) + __uint_as_float(r[G + g]) * (1.0f / 16.0f) +
                        __uint_as_float(r[2 * G + g]) * (1.0f / 256.0f);
        l2[j][g] = valid[j] ? f * sig_q[g] * s : -INFINITY;
      }
    } else {
#pragma unroll
      for (int g = 0; g < G; ++g) l2[j][g] = -INFINITY;
    }
  }
  float mrow[G], lsum[G], pmax[G];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    float m = l2[0][g];
#pragma unroll
    for (int j = 1; j < kMaxTiles; ++j) m = fmaxf(m, l2[j][g]);
    m = warp_max(m);
    if (lane == 0) red_a[warp][g] = m;
  }
  __syncthreads();
#pragma unroll
  for (int g = 0; g < G; ++g)
    mrow[g] = fmaxf(fmaxf(red_a[0][g], red_a[1][g]), fmaxf(red_a[2][g], red_a[3][g]));
  float p[kMaxTiles][G];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    float s = 0.f, pm = 0.f;
#pragma unroll
    for (int j = 0; j < kMaxTiles; ++j) {
      const float e = valid[j] ? exp2f(l2[j][g] - mrow[g]) : 0.f;
      s += e;
      p[j][g] = e * vs[j];
      pm = fmaxf(pm, p[j][g]);
    }
    s = warp_sum(s);
    pm = warp_max(pm);
    if (lane == 0) {
      red_b[warp][g] = s;
      red_c[warp][g] = pm;
    }
  }
  __syncthreads();
#pragma unroll
  for (int g = 0; g < G; ++g) {
    lsum[g] = red_b[0][g] + red_b[1][g] + red_b[2][g] + red_b[3][g];
    pmax[g] = fmaxf(fmaxf(red_c[0][g], red_c[1][g]), fmaxf(red_c[2][g], red_c[3][g]));
  }
  // P' = p * v_scale as three E4M3 terms, column `tid` of the B operand of tile j
#pragma unroll
  for (int j = 0; j < kMaxTiles; ++j) {
    if (j < ntiles) {
      uint8_t* dst = sP + j * C::kPBytes;
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float s1 = pmax[g] * (1.0f / 448.0f);
        const float inv1 = s1 > 0.f ? 1.0f / s1 : 0.f;
        const float x = p[j][g];
        const uint8_t c1 = f32_to_e4m3(x * inv1);
        const float r1 = fmaf(-e4m3_to_f32(c1), s1, x);
        const uint8_t c2 = f32_to_e4m3(r1 * inv1 * 16.0f);
        const float r2 = fmaf(-e4m3_to_f32(c2), s1 * (1.0f / 16.0f), r1);
        const uint8_t c3 = f32_to_e4m3(r2 * inv1 * 256.0f);
        dst[swizzled_offset(0 * G + g, tid, 128)] = c1;
        dst[swizzled_offset(1 * G + g, tid, 128)] = c2;
        dst[swizzled_offset(2 * G + g, tid, 128)] = c3;
      }
#pragma unroll
      for (int n = kTerms * G; n < C::kN; ++n) dst[swizzled_offset(n, tid, 128)] = 0;
      // V rows past the item (or of a skipped page) may hold anything, NaN
      // codes included: zero them so 0 * V stays 0 in the MMA.
      if (!mbar_wait(&bar_v[j], 0)) report_error(a.err, kDevErrTimeout);
      if (!valid[j] || vs[j] == 0.f) {
        uint4* row = reinterpret_cast<uint4*>(sV + j * C::kTileBytes + tid * D);
#pragma unroll
        for (int c = 0; c < D / 16; ++c) row[c] = make_uint4(0, 0, 0, 0);
      }
    }
  }
  fence_proxy_async_smem();
  tc_fence_before_sync();
  __syncthreads();

  // ---- PV: O^T += V_j^T . Pt_j^T
  if (tid == 0) {
    tc_fence_after_sync();
    constexpr uint32_t idesc = make_idesc(kFmtE4M3, kFmtE4M3, 1, 0, 128, C::kN);
    // MN-major A: one D-byte atom per 8 token rows; for D = 64 the second
    // 64-row half of M re-reads the same atom (LBO 0) and is ignored.
    for (int j = 0; j < ntiles; ++j) {
#pragma unroll
      for (int kk = 0; kk < kTile / 32; ++kk) {
        const uint64_t da = make_smem_desc(smem_u32(sV + j * C::kTileBytes) + kk * 32 * D,
                                           D == 128 ? 16 * 1024 : 0, C::kSBO, C::kSwz);
        const uint64_t db =
            make_smem_desc(smem_u32(sP + j * C::kPBytes) + 32 * kk, 16, 1024, kSwizzle128B);
        tc_mma_f8(tmem + C::kTmemO, da, db, idesc, (j > 0 || kk > 0) ? 1u : 0u);
      }
    }
    tc_commit(&bar_o);
  }
  __syncwarp();

  // ---- epilogue: recombine the terms, normalise, write the partial
  if (!mbar_wait(&bar_o, 0)) report_error(a.err, kDevErrTimeout);
  tc_fence_after_sync();
  {
    uint32_t r[C::kN];
#pragma unroll
    for (int c = 0; c < C::kN; c += 16) {
      uint32_t part[16];
      tmem_ld16(tmem + (static_cast<uint32_t>(warp * 32) << 16) + C::kTmemO + c, part);
#pragma unroll
      for (int i = 0; i < 16; ++i) r[c + i] = part[i];
    }
    tmem_ld_wait();
    const int slot = a.split_off[it.b] + it.t0 / a.chunk;
    if (tid < D) {
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float s = __uint_as_float(r[g]) + __uint_as_float(r[G + g]) * (1.0f / 16.0f) +
                        __uint_as_float(r[2 * G + g]) * (1.0f / 256.0f);
        const float o = lsum[g] > 0.f ? s * (pmax[g] * (1.0f / 448.0f)) / lsum[g] : 0.f;
        a.part_o[(static_cast<size_t>(slot) * a.Hq + it.hk * G + g) * D + tid] = o;
      }
    }
    if (tid < G) {
      const float lse = lsum[tid] > 0.f ? (mrow[tid] + log2f(lsum[tid])) * kLn2 : -INFINITY;
      a.part_lse[static_cast<size_t>(slot) * a.Hq + it.hk * G + tid] = lse;
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

// ---------------------------------------------------------------- merge
// One warp per (request, q head); lane l owns D/32 consecutive outputs.
template <int D>
__global__ void __launch_bounds__(128) decode_merge_kernel(int B, int Hq,
                                                           const int32_t* __restrict__ split_off,
                                                           const float* __restrict__ part_o,
                                                           const float* __restrict__ part_lse,
                                                           uint16_t* __restrict__ o,
                                                           float* __restrict__ lse) {
  constexpr int EPL = D / 32;
  const int w = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (w >= B * Hq) return;
  const int b = w / Hq, h = w % Hq;
  const int s0 = split_off[b], s1 = split_off[b + 1];
  float M = -INFINITY;
  for (int s = s0; s < s1; ++s) M = fmaxf(M, part_lse[static_cast<size_t>(s) * Hq + h]);
  float acc[EPL];
#pragma unroll
  for (int e = 0; e < EPL; ++e) acc[e] = 0.f;
  float den = 0.f;
  if (M > -INFINITY) {
    for (int s = s0; s < s1; ++s) {
      const float ls = part_lse[static_cast<size_t>(s) * Hq + h];
      const float wgt = ls > -INFINITY ? __expf(ls - M) : 0.f;
      den += wgt;
      const float* src = part_o + (static_cast<size_t>(s) * Hq + h) * D + lane * EPL;
      if constexpr (EPL == 4) {
        const float4 v = *reinterpret_cast<const float4*>(src);
        acc[0] += wgt * v.x;
        acc[1] += wgt * v.y;
        acc[2] += wgt * v.z;
        acc[3] += wgt * v.w;
      } else {
        const float2 v = *reinterpret_cast<const float2*>(src);
        acc[0] += wgt * v.x;
        acc[1] += wgt * v.y;
      }
    }
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
                            int num_items, cudaStream_t stream) {
  using C = Cfg<D, G>;
  auto* kern = decode_attend_kernel<D, G>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  if (e != cudaSuccess) return e;
  kern<<<num_items, kThreads, C::kSmem, stream>>>(km, vm, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode_attend(const DecodePlan& plan, float* float_ws, const void* int_ws,
                                 const void* q, const void* k_pool, const void* v_pool,
                                 const float* k_scale_pool, const float* v_scale_pool,
                                 int num_pages, int page_size, const int32_t* block_table,
                                 int bt_stride, float sm_scale, int32_t* error_word,
                                 cudaStream_t stream, int* status) {
  *status = QPKV_OK;
  if (plan.num_items == 0) return cudaSuccess;
  const int D = static_cast<int>(plan.head_dim);
  const int Hkv = static_cast<int>(plan.num_kv_heads);
  const int G = static_cast<int>(plan.num_qo_heads / plan.num_kv_heads);
  const int R = page_size < kTile ? page_size : kTile;
  CUtensorMap km, vm;
  const uint64_t dims[3] = {static_cast<uint64_t>(D), static_cast<uint64_t>(Hkv),
                            static_cast<uint64_t>(num_pages) * page_size};
  const uint64_t strides[2] = {static_cast<uint64_t>(D), static_cast<uint64_t>(Hkv) * D};
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
  a.split_off = reinterpret_cast<const int32_t*>(iws + plan.split_off_offset);
  a.chunk = static_cast<int>(plan.chunk);
  a.Hq = static_cast<int>(plan.num_qo_heads);
  a.Hkv = Hkv;
  a.q = static_cast<const uint16_t*>(q);
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
  const int n = static_cast<int>(plan.num_items);
#define QPKV_DECODE_CASE(DD, GG) \
  if (D == DD && G == GG) return launch_attend_t<DD, GG>(km, vm, a, n, stream);
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
  if (plan.head_dim == 128)
    decode_merge_kernel<128><<<grid, 128, 0, stream>>>(B, Hq, split_off, float_ws, part_lse,
                                                       static_cast<uint16_t*>(o), lse);
  else
    decode_merge_kernel<64><<<grid, 128, 0, stream>>>(B, Hq, split_off, float_ws, part_lse,
                                                      static_cast<uint16_t*>(o), lse);
  return cudaGetLastError();
}

}  // namespace qpkv
