// Cache write: (RoPE +) quantise + page-append of new tokens.
//
// "[Feature] Sage Attention Support Varlen & write kv cache BF16/FP16",
// Description item 1 (RoPE fused into the KV-cache write) and item 2 (varlen
// quantisation: a quantisation block never crosses a sequence boundary);
// "KvQuantSparseFlashAttention" README, 参数说明 rows key / block_table
// (PA_BSND pages) and the Per-Token-Head(-Tile-128) quantisation named under
// 功能说明.  Memory-bound elementwise work with small reductions: plain SIMT
// with 16-byte vector accesses, no tensor cores.
//
// Rounding is explicit so the bytes are reproducible: IEEE float32 division
// (__fdiv_rn), nearest-even conversions, RoPE products and sums rounded
// separately (__fmul_rn / __fadd_rn / __fsub_rn, no contraction).
//
// Options: the HND K/V pool layout (FP8 mode); K smoothing and E4M3 V with
// per-channel scales (INT8 mode: a first pass writes exact per-block
// partials, int64 key sums / float channel maxima, to the caller's scratch,
// and the block write combines a sequence's partials); RoPE on the 64-wide
// rope part of MLA rows and queries.
#include "common.cuh"
#include "internal.h"

namespace qpkv {
namespace {

__device__ __forceinline__ int pool_page(const int32_t* __restrict__ bt, int bt_stride, int b,
                                         int p, int ps, int num_pages, int* err) {
  const int page = __ldg(bt + static_cast<size_t>(b) * bt_stride + p / ps);
  if (page < 0 || page >= num_pages) {
    report_error(err, kDevErrBadPage);
    return -1;
  }
  return page;
}

// ---------------------------------------------- FP8 per-(token, head) mode
// One warp per (token, kv head); lane l owns D/32 consecutive elements, so
// the rotate-half partner of lane l's elements (i + D/2) sits on lane l ^ 16.

// Rotate-half RoPE of the EPL elements x a lane owns (first element index
// i0 = lane * EPL of a D-wide head) at table row `pos`: each product and sum
// rounded to float32 separately.
template <int D, int EPL>
__device__ __forceinline__ void rope_lane(float (&x)[EPL], int lane, int pos,
                                          const float* __restrict__ cos_t,
                                          const float* __restrict__ sin_t) {
  const bool first = lane < 16;                       // elements i < D/2
  const int i0 = (lane & 15) * EPL;                   // pair index of x[0]
  const float* c = cos_t + static_cast<size_t>(pos) * (D / 2) + i0;
  const float* s = sin_t + static_cast<size_t>(pos) * (D / 2) + i0;
#pragma unroll
  for (int e = 0; e < EPL; ++e) {
    const float other = __shfl_xor_sync(0xffffffffu, x[e], 16);
    const float ce = __ldg(c + e), se = __ldg(s + e);
    x[e] = first ? __fsub_rn(__fmul_rn(x[e], ce), __fmul_rn(other, se))
                 : __fadd_rn(__fmul_rn(x[e], ce), __fmul_rn(other, se));
  }
}

template <int EPL>
__device__ __forceinline__ void load_bf16_lane(const uint16_t* src, float (&x)[EPL]) {
  if constexpr (EPL == 4) {
    const uint2 raw = *reinterpret_cast<const uint2*>(src);
    x[0] = bf16_bits_to_float(raw.x & 0xFFFF);
    x[1] = bf16_bits_to_float(raw.x >> 16);
    x[2] = bf16_bits_to_float(raw.y & 0xFFFF);
    x[3] = bf16_bits_to_float(raw.y >> 16);
  } else {
    const uint32_t raw = *reinterpret_cast<const uint32_t*>(src);
    x[0] = bf16_bits_to_float(raw & 0xFFFF);
    x[1] = bf16_bits_to_float(raw >> 16);
  }
}

template <int D>
__global__ void __launch_bounds__(256) write_fp8_token_head_kernel(
    int T, int B, int H, int ps, int num_pages, int bt_stride, const int32_t* __restrict__ cu,
    const int32_t* __restrict__ start_pos, const int32_t* __restrict__ bt,
    const uint16_t* __restrict__ k, const uint16_t* __restrict__ v, uint8_t* __restrict__ k_pool,
    uint8_t* __restrict__ v_pool, float* __restrict__ k_scale, float* __restrict__ v_scale,
    int32_t* __restrict__ slots, int hnd, const float* __restrict__ rope_cos,
    const float* __restrict__ rope_sin, int rope_max_pos, int* err) {
  constexpr int EPL = D / 32;  // 2 or 4 elements per lane
  // a programmatic dependent launch (the decode) may start its prologue now;
  // it waits for this grid to complete before it reads the pools
  griddep_launch_dependents();
  const int w = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (w >= T * H) return;
  const int t = w / H, h = w - (w / H) * H;
  const int b = seq_of_token(cu, B, t);
  const int p = (start_pos ? __ldg(start_pos + b) : 0) + (t - seq_begin(cu, b));
  if (rope_cos != nullptr && (p < 0 || p >= rope_max_pos)) {
    if (lane == 0) report_error(err, kDevErrBadLength);
    return;
  }
  const int page = pool_page(bt, bt_stride, b, p, ps, num_pages, lane == 0 ? err : nullptr);
  if (page < 0) return;
  const size_t slot = static_cast<size_t>(page) * ps + (p % ps);
  if (slots != nullptr && h == 0 && lane == 0) slots[t] = static_cast<int32_t>(slot);
  // K/V row of (token, head): NHD [P, ps, H, D], HND [P, H, ps, D]
  const size_t kv_row = hnd ? (static_cast<size_t>(page) * H + h) * ps + (p % ps) : slot * H + h;

#pragma unroll
  for (int which = 0; which < 2; ++which) {
    const uint16_t* src = (which ? v : k) + (static_cast<size_t>(t) * H + h) * D + lane * EPL;
    float x[EPL];
    load_bf16_lane<EPL>(src, x);
    if (which == 0 && rope_cos != nullptr) rope_lane<D, EPL>(x, lane, p, rope_cos, rope_sin);   // K only
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < EPL; ++i) amax = fmaxf(amax, fabsf(x[i]));
    amax = warp_max(amax);
    const float scale = __fdiv_rn(amax, 448.0f);
    uint32_t packed = 0;
    if (scale != 0.f) {
#pragma unroll
      for (int i = 0; i < EPL; ++i)
        packed |= static_cast<uint32_t>(f32_to_e4m3(__fdiv_rn(x[i], scale))) << (8 * i);
    }
    uint8_t* dst = (which ? v_pool : k_pool) + kv_row * D + lane * EPL;
    if constexpr (EPL == 4) {
      *reinterpret_cast<uint32_t*>(dst) = packed;
    } else {
      *reinterpret_cast<uint16_t*>(dst) = static_cast<uint16_t>(packed);
    }
    if (lane == 0) (which ? v_scale : k_scale)[slot * H + h] = scale;
  }
}

// The query side of the FP8-mode RoPE: one warp per (token, q head), the
// rotated values rounded to bf16 (nearest-even) into q_out (may alias q:
// each lane writes only what it read, after the whole warp has read).
template <int D>
__global__ void __launch_bounds__(256) rope_q_kernel(
    int T, int B, int Hq, const int32_t* __restrict__ cu, const int32_t* __restrict__ start_pos,
    const uint16_t* q, const float* __restrict__ rope_cos, const float* __restrict__ rope_sin,
    int rope_max_pos, uint16_t* q_out, int* err) {
  constexpr int EPL = D / 32;
  const long w = (static_cast<long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (w >= static_cast<long>(T) * Hq) return;
  const int t = static_cast<int>(w / Hq);
  const int b = seq_of_token(cu, B, t);
  const int p = (start_pos ? __ldg(start_pos + b) : 0) + (t - seq_begin(cu, b));
  if (p < 0 || p >= rope_max_pos) {
    if (lane == 0) report_error(err, kDevErrBadLength);
    return;
  }
  float x[EPL];
  load_bf16_lane<EPL>(q + w * D + lane * EPL, x);
  rope_lane<D, EPL>(x, lane, p, rope_cos, rope_sin);
  uint16_t o[EPL];
#pragma unroll
  for (int e = 0; e < EPL; ++e) {
    const __nv_bfloat16 bv = __float2bfloat16_rn(x[e]);
    o[e] = *reinterpret_cast<const uint16_t*>(&bv);
  }
  uint16_t* dst = q_out + w * D + lane * EPL;
  if constexpr (EPL == 4) {
    *reinterpret_cast<uint2*>(dst) = make_uint2(o[0] | (static_cast<uint32_t>(o[1]) << 16),
                                                o[2] | (static_cast<uint32_t>(o[3]) << 16));
  } else {
    *reinterpret_cast<uint32_t*>(dst) = o[0] | (static_cast<uint32_t>(o[1]) << 16);
  }
}

// ------------------------------- INT8 per-(sequence, 128-token block, head)
// One CTA (256 threads) per (block, head, sequence).  Thread tid owns token
// r = tid / 2 of the block and RoPE pairs i in [32*(tid%2), 32*(tid%2)+32),
// i.e. elements i and i + 64 of the 128-wide head.
constexpr int kBlk = 128;

__device__ __forceinline__ void load_bf16x8(const uint16_t* src, float (&x)[8]) {
  const uint4 raw = *reinterpret_cast<const uint4*>(src);
  const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    x[2 * j] = bf16_bits_to_float(w[j] & 0xFFFF);
    x[2 * j + 1] = bf16_bits_to_float(w[j] >> 16);
  }
}

__device__ __forceinline__ float block_max_256(float v, float* red) {
  v = warp_max(v);
  const int warp = threadIdx.x >> 5;
  if ((threadIdx.x & 31) == 0) red[warp] = v;
  __syncthreads();
  float m = red[0];
#pragma unroll
  for (int i = 1; i < 8; ++i) m = fmaxf(m, red[i]);
  __syncthreads();
  return m;
}

// Rotate, subtract the smoothing mean km (shared, 128 floats; NULL: none),
// quantise to INT8 with one block scale, and store the codes.
// Returns nothing; writes codes to dst_row (128 int8) and the scale via *scale_out.
__device__ __forceinline__ void rope_quant_block(const uint16_t* __restrict__ src_row, bool valid,
                                                 int pos, int half, const float* __restrict__ cos_t,
                                                 const float* __restrict__ sin_t, const float* km,
                                                 int8_t* dst_row, float* scale_out, float* red) {
  float y1[32], y2[32];
  float amax = 0.f;
  if (valid) {
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      float a[8], bb[8];
      load_bf16x8(src_row + half * 32 + c * 8, a);
      load_bf16x8(src_row + 64 + half * 32 + c * 8, bb);
      // this chunk's 8 cos / sin values: two 16-byte loads each
      const float4* cp = reinterpret_cast<const float4*>(cos_t + static_cast<size_t>(pos) * 64 +
                                                         half * 32 + c * 8);
      const float4* sp = reinterpret_cast<const float4*>(sin_t + static_cast<size_t>(pos) * 64 +
                                                         half * 32 + c * 8);
      const float4 c0 = __ldg(cp), c1 = __ldg(cp + 1), s0 = __ldg(sp), s1 = __ldg(sp + 1);
      const float cv[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
      const float sv[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float cs = cv[j];
        const float sn = sv[j];
        float r1 = __fsub_rn(__fmul_rn(a[j], cs), __fmul_rn(bb[j], sn));
        float r2 = __fadd_rn(__fmul_rn(bb[j], cs), __fmul_rn(a[j], sn));
        if (km != nullptr) {
          r1 = __fsub_rn(r1, km[half * 32 + c * 8 + j]);
          r2 = __fsub_rn(r2, km[64 + half * 32 + c * 8 + j]);
        }
        y1[c * 8 + j] = r1;
        y2[c * 8 + j] = r2;
        amax = fmaxf(amax, fmaxf(fabsf(r1), fabsf(r2)));
      }
    }
  }
  amax = block_max_256(amax, red);
  const float scale = __fdiv_rn(amax, 127.0f);
  if (threadIdx.x == 0) *scale_out = scale;
  if (!valid) return;
  uint32_t w1[8], w2[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    uint32_t p1 = 0, p2 = 0;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      int c1 = 0, c2 = 0;
      if (scale != 0.f) {
        c1 = min(127, max(-127, __float2int_rn(__fdiv_rn(y1[4 * j + e], scale))));
        c2 = min(127, max(-127, __float2int_rn(__fdiv_rn(y2[4 * j + e], scale))));
      }
      p1 |= (static_cast<uint32_t>(c1) & 0xFFu) << (8 * e);
      p2 |= (static_cast<uint32_t>(c2) & 0xFFu) << (8 * e);
    }
    w1[j] = p1;
    w2[j] = p2;
  }
  uint4* d1 = reinterpret_cast<uint4*>(dst_row + half * 32);
  uint4* d2 = reinterpret_cast<uint4*>(dst_row + 64 + half * 32);
  d1[0] = make_uint4(w1[0], w1[1], w1[2], w1[3]);
  d1[1] = make_uint4(w1[4], w1[5], w1[6], w1[7]);
  d2[0] = make_uint4(w2[0], w2[1], w2[2], w2[3]);
  d2[1] = make_uint4(w2[4], w2[5], w2[6], w2[7]);
}

// K smoothing, pass 1: per (sequence, 128-token block, kv head) the int64 sum
// over the block's tokens of RNE(clamp(k_rot, -2^15, 2^15) * 2^24) per dim
// (exact, so the order of the sums does not matter); two row phases of 128
// threads, thread d owns dim d.  The rotation is the one the write applies.
constexpr float kMeanClamp = 32768.0f, kMeanOne = 16777216.0f;   // 2^15, 2^24

__global__ void __launch_bounds__(256) k_block_sum_kernel(
    int Hkv, int num_blocks, int max_pos, const int32_t* __restrict__ cu,
    const uint16_t* __restrict__ k,
    const float* __restrict__ cos_t, const float* __restrict__ sin_t,
    long long* __restrict__ partial) {
  __shared__ long long part[128];
  const int blk = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int begin = seq_begin(cu, b);
  const int L = __ldg(cu + b) - begin;
  if (blk * kBlk >= L) return;
  const int d = threadIdx.x & 127, phase = threadIdx.x >> 7, i = d & 63;
  // tokens past the launched blocks or the RoPE tables are the write's to flag
  const int n = min(kBlk, min(L, max_pos) - blk * kBlk);
  long long acc = 0;
  for (int r = phase; r < n; r += 2) {
    const int pos = blk * kBlk + r;
    const uint16_t* row = k + (static_cast<size_t>(begin + pos) * Hkv + h) * 128;
    const float a = bf16_bits_to_float(__ldg(row + i)), bb = bf16_bits_to_float(__ldg(row + 64 + i));
    const float cs = __ldg(cos_t + static_cast<size_t>(pos) * 64 + i);
    const float sn = __ldg(sin_t + static_cast<size_t>(pos) * 64 + i);
    const float y = d < 64 ? __fsub_rn(__fmul_rn(a, cs), __fmul_rn(bb, sn))
                           : __fadd_rn(__fmul_rn(bb, cs), __fmul_rn(a, sn));
    acc += __float2ll_rn(fminf(fmaxf(y, -kMeanClamp), kMeanClamp) * kMeanOne);
  }
  if (phase == 1) part[d] = acc;
  __syncthreads();
  if (phase == 0)
    partial[((static_cast<size_t>(b) * num_blocks + blk) * Hkv + h) * 128 + d] = acc + part[d];
}

// FP8 V, pass 1: per (sequence, 128-token block, kv head) the largest |v|
// of each channel over the block's tokens (a maximum: order-free).
__global__ void __launch_bounds__(128) v_block_max_kernel(
    int Hkv, int num_blocks, const int32_t* __restrict__ cu, const uint16_t* __restrict__ v,
    float* __restrict__ vmax) {
  const int blk = blockIdx.x, h = blockIdx.y, b = blockIdx.z, d = threadIdx.x;
  const int begin = seq_begin(cu, b);
  const int L = __ldg(cu + b) - begin;
  if (blk * kBlk >= L) return;
  const int n = min(kBlk, L - blk * kBlk);
  float m = 0.f;
  for (int r = 0; r < n; ++r)
    m = fmaxf(m, fabsf(bf16_bits_to_float(
                     __ldg(v + (static_cast<size_t>(begin + blk * kBlk + r) * Hkv + h) * 128 + d))));
  vmax[((static_cast<size_t>(b) * num_blocks + blk) * Hkv + h) * 128 + d] = m;
}

__global__ void __launch_bounds__(256) write_int8_block128_rope_kernel(
    int B, int Hq, int Hkv, int ps, int num_pages, int bt_stride, int num_blocks,
    const int32_t* __restrict__ cu, const int32_t* __restrict__ bt,
    const uint16_t* __restrict__ q, const uint16_t* __restrict__ k,
    const uint16_t* __restrict__ v, const float* __restrict__ cos_t,
    const float* __restrict__ sin_t, int8_t* __restrict__ k_pool, uint16_t* __restrict__ v_pool,
    float* __restrict__ k_bscale, int8_t* __restrict__ q_out, float* __restrict__ q_bscale,
    int32_t* __restrict__ slots, const long long* __restrict__ partial, float* __restrict__ k_mean,
    const float* __restrict__ vmax, float* __restrict__ v_cscale, int max_pos, int* err) {
  constexpr int D = 128;
  __shared__ float red[8];
  __shared__ float km[D];
  __shared__ float vsc[D];
  const int blk = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int begin = seq_begin(cu, b);
  const int L = __ldg(cu + b) - begin;
  if (blk * kBlk >= L) return;  // block past this sequence's end
  // a sequence longer than the launch (max_seqlen) or the RoPE tables
  const int nblk = (L + kBlk - 1) / kBlk;
  if ((nblk > static_cast<int>(gridDim.x) || L > max_pos) && blk == 0 && h == 0 &&
      threadIdx.x == 0)
    report_error(err, kDevErrBadLength);
  const bool smooth = partial != nullptr && h < Hkv;
  if (smooth) {
    // K smoothing, pass 2: the sequence's mean from the exact block sums
    if (threadIdx.x < D) {
      long long sum = 0;
      const int nsum = min(nblk, static_cast<int>(gridDim.x));
      for (int j = 0; j < nsum; ++j)
        sum += partial[((static_cast<size_t>(b) * num_blocks + j) * Hkv + h) * D + threadIdx.x];
      const float m =
          __double2float_rn(__ll2double_rn(sum) / (static_cast<double>(L) * static_cast<double>(kMeanOne)));
      km[threadIdx.x] = m;
      if (blk == 0) k_mean[(static_cast<size_t>(b) * Hkv + h) * D + threadIdx.x] = m;
    }
    __syncthreads();
  }
  const bool v8 = vmax != nullptr && h < Hkv;
  if (v8) {
    // FP8 V, pass 2: the channel's absmax over the sequence -> scale / 448
    if (threadIdx.x < D) {
      float amax = 0.f;
      const int nsum = min(nblk, static_cast<int>(gridDim.x));
      for (int j = 0; j < nsum; ++j)
        amax = fmaxf(amax, vmax[((static_cast<size_t>(b) * num_blocks + j) * Hkv + h) * D + threadIdx.x]);
      const float sc = __fdiv_rn(amax, 448.0f);
      vsc[threadIdx.x] = sc;
      if (blk == 0) v_cscale[(static_cast<size_t>(b) * Hkv + h) * D + threadIdx.x] = sc;
    }
    __syncthreads();
  }
  const int r = threadIdx.x >> 1, half = threadIdx.x & 1;
  const int pos = blk * kBlk + r;
  const bool valid = pos < L && pos < max_pos;
  const int t = begin + pos;

  if (h < Hq) {
    const uint16_t* src = q + (static_cast<size_t>(t) * Hq + h) * D;
    int8_t* dst = q_out + (static_cast<size_t>(t) * Hq + h) * D;
    rope_quant_block(src, valid, pos, half, cos_t, sin_t, nullptr, dst,
                     q_bscale + (static_cast<size_t>(b) * num_blocks + blk) * Hq + h, red);
  }
  if (h < Hkv) {
    int page = 0;
    if (valid) page = pool_page(bt, bt_stride, b, pos, ps, num_pages, half == 0 ? err : nullptr);
    const bool ok = valid && page >= 0;
    const size_t slot = static_cast<size_t>(ok ? page : 0) * ps + (pos % ps);
    if (ok && slots != nullptr && h == 0 && half == 0) slots[t] = static_cast<int32_t>(slot);
    const uint16_t* src = k + (static_cast<size_t>(t) * Hkv + h) * D;
    int8_t* dst = k_pool + (slot * Hkv + h) * D;
    // the block reduction needs every thread; an invalid page only drops the store
    __shared__ __align__(16) int8_t sink[2 * D];
    rope_quant_block(src, valid, pos, half, cos_t, sin_t, smooth ? km : nullptr, ok ? dst : sink,
                     k_bscale + (static_cast<size_t>(b) * num_blocks + blk) * Hkv + h, red);
    if (ok && !v8) {
      const uint4* vs = reinterpret_cast<const uint4*>(v + (static_cast<size_t>(t) * Hkv + h) * D +
                                                       half * 64);
      uint4* vd = reinterpret_cast<uint4*>(v_pool + (slot * Hkv + h) * D + half * 64);
#pragma unroll
      for (int c = 0; c < 8; ++c) vd[c] = vs[c];
    } else if (ok) {
      // E4M3 codes of v / channel scale (float32 division), this thread's 64
      // channels; the pool holds one byte per element
      const uint16_t* vs = v + (static_cast<size_t>(t) * Hkv + h) * D + half * 64;
      uint8_t* vd = reinterpret_cast<uint8_t*>(v_pool) + (slot * Hkv + h) * D + half * 64;
#pragma unroll
      for (int g = 0; g < 4; ++g) {
        float xa[8], xb[8];
        load_bf16x8(vs + 16 * g, xa);
        load_bf16x8(vs + 16 * g + 8, xb);
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          uint32_t word = 0;
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int c = 16 * g + 4 * e + k;
            const float sc = vsc[half * 64 + c];
            const float xv = 4 * e + k < 8 ? xa[4 * e + k] : xb[4 * e + k - 8];
            const uint32_t code = sc != 0.f ? f32_to_e4m3(__fdiv_rn(xv, sc)) : 0u;
            word |= code << (8 * k);
          }
          w[e] = word;
        }
        *reinterpret_cast<uint4*>(vd + 16 * g) = make_uint4(w[0], w[1], w[2], w[3]);
      }
    }
  }
}

// ------------------------------------------------------------ MLA rows
// One warp per token: lane l quantises nope dims [16l, 16l + 16) (tile l / 8),
// lanes 0..7 copy the 64 bf16 rope values (with RoPE: lanes 0..3 rotate
// the pairs (i, i + 32), i in [8l, 8l + 8)), lanes 0/8/16/24 store the scales.
constexpr int kMlaIn = 576, kMlaRow = 656, kMlaRopeHalf = 32;

// Rotate-half RoPE of one lane's 8 pairs of the 64-wide rope part: x holds
// dims [8l, 8l + 8), y dims [32 + 8l, 32 + 8l + 8) as bf16; the float32
// results (products and sums rounded separately) are rounded to bf16.
__device__ __forceinline__ void mla_rope8(uint4& x, uint4& y, const float* __restrict__ cs,
                                          const float* __restrict__ sn) {
  float a[8], b[8];
  const uint32_t* xw = reinterpret_cast<const uint32_t*>(&x);
  const uint32_t* yw = reinterpret_cast<const uint32_t*>(&y);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    a[2 * j] = bf16_bits_to_float(xw[j] & 0xFFFF);
    a[2 * j + 1] = bf16_bits_to_float(xw[j] >> 16);
    b[2 * j] = bf16_bits_to_float(yw[j] & 0xFFFF);
    b[2 * j + 1] = bf16_bits_to_float(yw[j] >> 16);
  }
  uint32_t ox[4], oy[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    float r1[2], r2[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int k = 2 * j + e;
      const float c = __ldg(cs + k), s = __ldg(sn + k);
      r1[e] = __fsub_rn(__fmul_rn(a[k], c), __fmul_rn(b[k], s));
      r2[e] = __fadd_rn(__fmul_rn(b[k], c), __fmul_rn(a[k], s));
    }
    const __nv_bfloat162 p1 = __floats2bfloat162_rn(r1[0], r1[1]);
    const __nv_bfloat162 p2 = __floats2bfloat162_rn(r2[0], r2[1]);
    ox[j] = *reinterpret_cast<const uint32_t*>(&p1);
    oy[j] = *reinterpret_cast<const uint32_t*>(&p2);
  }
  x = make_uint4(ox[0], ox[1], ox[2], ox[3]);
  y = make_uint4(oy[0], oy[1], oy[2], oy[3]);
}

// Position of token t, or -1 (flagged) when it lies past the RoPE tables.
__device__ __forceinline__ int mla_pos(const int32_t* __restrict__ cu,
                                       const int32_t* __restrict__ start_pos, int B, int t,
                                       int max_pos, int* err) {
  const int b = seq_of_token(cu, B, t);
  const int p = (start_pos ? __ldg(start_pos + b) : 0) + (t - seq_begin(cu, b));
  if (p < 0 || p >= max_pos) {
    report_error(err, kDevErrBadLength);
    return -1;
  }
  return p;
}

__global__ void __launch_bounds__(256) write_mla_row_kernel(
    int T, int B, int ps, int num_pages, int bt_stride, const int32_t* __restrict__ cu,
    const int32_t* __restrict__ start_pos, const int32_t* __restrict__ bt,
    const uint16_t* __restrict__ kv, const float* __restrict__ rope_cos,
    const float* __restrict__ rope_sin, int rope_max_pos, uint8_t* __restrict__ pool,
    int32_t* __restrict__ slots, int* err) {
  const int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (t >= T) return;
  const int b = seq_of_token(cu, B, t);
  const int p = (start_pos ? __ldg(start_pos + b) : 0) + (t - seq_begin(cu, b));
  if (rope_cos != nullptr && (p < 0 || p >= rope_max_pos)) {
    if (lane == 0) report_error(err, kDevErrBadLength);
    return;
  }
  const int page = pool_page(bt, bt_stride, b, p, ps, num_pages, lane == 0 ? err : nullptr);
  if (page < 0) return;
  const size_t slot = static_cast<size_t>(page) * ps + (p % ps);
  if (slots != nullptr && lane == 0) slots[t] = static_cast<int32_t>(slot);
  const uint16_t* src = kv + static_cast<size_t>(t) * kMlaIn;
  uint8_t* row = pool + slot * kMlaRow;

  float a[8], c[8];
  load_bf16x8(src + lane * 16, a);
  load_bf16x8(src + lane * 16 + 8, c);
  float amax = 0.f;
#pragma unroll
  for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fmaxf(fabsf(a[j]), fabsf(c[j])));
#pragma unroll
  for (int o = 1; o < 8; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const float scale = __fdiv_rn(amax, 127.0f);
  uint32_t w[4] = {0, 0, 0, 0};
  if (scale != 0.f) {
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const float x = j < 8 ? a[j] : c[j - 8];
      const int code = min(127, max(-127, __float2int_rn(__fdiv_rn(x, scale))));
      w[j / 4] |= (static_cast<uint32_t>(code) & 0xFFu) << (8 * (j % 4));
    }
  }
  *reinterpret_cast<uint4*>(row + lane * 16) = make_uint4(w[0], w[1], w[2], w[3]);
  if (rope_cos == nullptr) {
    if (lane < 8) {
      *reinterpret_cast<uint4*>(row + 512 + lane * 16) =
          *reinterpret_cast<const uint4*>(src + 512 + lane * 8);
    }
  } else if (lane < 4) {
    uint4 x = *reinterpret_cast<const uint4*>(src + 512 + lane * 8);
    uint4 y = *reinterpret_cast<const uint4*>(src + 512 + kMlaRopeHalf + lane * 8);
    const size_t tab = static_cast<size_t>(p) * kMlaRopeHalf + lane * 8;
    mla_rope8(x, y, rope_cos + tab, rope_sin + tab);
    *reinterpret_cast<uint4*>(row + 512 + lane * 16) = x;
    *reinterpret_cast<uint4*>(row + 512 + 2 * kMlaRopeHalf + lane * 16) = y;
  }
  if ((lane & 7) == 0) *reinterpret_cast<float*>(row + 640 + 4 * (lane >> 3)) = scale;
}

// The query side of the MLA RoPE: one warp per (token, head) row of 576
// bf16; the 512 nope values are copied, the rope part rotated at the
// token's position (q_out may alias q: each lane writes what it read).
__global__ void __launch_bounds__(256) rope_mla_q_kernel(
    int T, int B, int Hq, const int32_t* __restrict__ cu, const int32_t* __restrict__ start_pos,
    const uint16_t* q, const float* __restrict__ rope_cos, const float* __restrict__ rope_sin,
    int rope_max_pos, uint16_t* q_out, int* err) {
  const long w = (static_cast<long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (w >= static_cast<long>(T) * Hq) return;
  const int t = static_cast<int>(w / Hq);
  const int p = mla_pos(cu, start_pos, B, t, rope_max_pos, lane == 0 ? err : nullptr);
  if (p < 0) return;
  const uint16_t* src = q + w * kMlaIn;
  uint16_t* dst = q_out + w * kMlaIn;
  // nope: 1024 bytes, two 16-byte pieces per lane
  const uint4 n0 = *reinterpret_cast<const uint4*>(src + lane * 8);
  const uint4 n1 = *reinterpret_cast<const uint4*>(src + 256 + lane * 8);
  uint4 x, y;
  if (lane < 4) {
    x = *reinterpret_cast<const uint4*>(src + 512 + lane * 8);
    y = *reinterpret_cast<const uint4*>(src + 512 + kMlaRopeHalf + lane * 8);
    const size_t tab = static_cast<size_t>(p) * kMlaRopeHalf + lane * 8;
    mla_rope8(x, y, rope_cos + tab, rope_sin + tab);
  }
  *reinterpret_cast<uint4*>(dst + lane * 8) = n0;
  *reinterpret_cast<uint4*>(dst + 256 + lane * 8) = n1;
  if (lane < 4) {
    *reinterpret_cast<uint4*>(dst + 512 + lane * 8) = x;
    *reinterpret_cast<uint4*>(dst + 512 + kMlaRopeHalf + lane * 8) = y;
  }
}

}  // namespace

cudaError_t launch_write_cache(const qpkv_write_params& p, cudaStream_t stream) {
  const int threads = 256;
  switch (p.mode) {
    case QPKV_WRITE_FP8_TOKEN_HEAD: {
      const long warps = static_cast<long>(p.num_tokens) * p.num_heads_kv;
      const int grid = static_cast<int>((warps * 32 + threads - 1) / threads);
      if (grid == 0) return cudaSuccess;
      auto* kern = p.head_dim == 128 ? write_fp8_token_head_kernel<128>
                                     : write_fp8_token_head_kernel<64>;
      kern<<<grid, threads, 0, stream>>>(
          p.num_tokens, p.num_seqs, p.num_heads_kv, p.page_size, p.num_pages, p.bt_stride,
          p.cu_seqlens_q, p.start_pos, p.block_table, static_cast<const uint16_t*>(p.k),
          static_cast<const uint16_t*>(p.v), static_cast<uint8_t*>(p.k_pool),
          static_cast<uint8_t*>(p.v_pool), p.k_scale_pool, p.v_scale_pool, p.slot_mapping,
          (p.flags & QPKV_WRITE_HND) ? 1 : 0, p.rope_cos, p.rope_sin, p.rope_max_pos,
          p.error_word);
      if (p.q != nullptr) {
        const long qwarps = static_cast<long>(p.num_tokens) * p.num_heads_q;
        const int qgrid = static_cast<int>((qwarps * 32 + threads - 1) / threads);
        auto* qk = p.head_dim == 128 ? rope_q_kernel<128> : rope_q_kernel<64>;
        qk<<<qgrid, threads, 0, stream>>>(p.num_tokens, p.num_seqs, p.num_heads_q, p.cu_seqlens_q,
                                          p.start_pos, static_cast<const uint16_t*>(p.q),
                                          p.rope_cos, p.rope_sin, p.rope_max_pos,
                                          static_cast<uint16_t*>(p.q_out), p.error_word);
      }
      return cudaGetLastError();
    }
    case QPKV_WRITE_INT8_BLOCK128_ROPE: {
      const int nblk = (p.max_seqlen + kBlk - 1) / kBlk;
      if (nblk == 0) return cudaSuccess;
      const int hmax = p.num_heads_q > p.num_heads_kv ? p.num_heads_q : p.num_heads_kv;
      long long* partial = nullptr;
      float* vmax = nullptr;
      if (p.flags & QPKV_WRITE_V_FP8) {
        // after the K sums in the scratch: float [B, num_blocks, Hkv, 128]
        vmax = reinterpret_cast<float*>(static_cast<uint8_t*>(p.workspace) +
                                        static_cast<size_t>(p.num_seqs) * p.num_blocks *
                                            p.num_heads_kv * 128 * sizeof(long long));
        v_block_max_kernel<<<dim3(nblk, p.num_heads_kv, p.num_seqs), 128, 0, stream>>>(
            p.num_heads_kv, p.num_blocks, p.cu_seqlens_q, static_cast<const uint16_t*>(p.v), vmax);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
      }
      if (p.flags & QPKV_WRITE_SMOOTH_K) {
        partial = static_cast<long long*>(p.workspace);
        k_block_sum_kernel<<<dim3(nblk, p.num_heads_kv, p.num_seqs), threads, 0, stream>>>(
            p.num_heads_kv, p.num_blocks, p.rope_max_pos, p.cu_seqlens_q,
            static_cast<const uint16_t*>(p.k),
            p.rope_cos, p.rope_sin, partial);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
      }
      dim3 grid(nblk, hmax, p.num_seqs);
      write_int8_block128_rope_kernel<<<grid, threads, 0, stream>>>(
          p.num_seqs, p.num_heads_q, p.num_heads_kv, p.page_size, p.num_pages, p.bt_stride,
          p.num_blocks, p.cu_seqlens_q, p.block_table, static_cast<const uint16_t*>(p.q),
          static_cast<const uint16_t*>(p.k), static_cast<const uint16_t*>(p.v), p.rope_cos,
          p.rope_sin, static_cast<int8_t*>(p.k_pool), static_cast<uint16_t*>(p.v_pool),
          p.k_block_scale, static_cast<int8_t*>(p.q_out), p.q_block_scale, p.slot_mapping,
          partial, p.k_mean, vmax, p.v_channel_scale, p.rope_max_pos, p.error_word);
      return cudaGetLastError();
    }
    case QPKV_WRITE_MLA_ROW: {
      const int grid = static_cast<int>((static_cast<long>(p.num_tokens) * 32 + threads - 1) /
                                        threads);
      if (grid == 0) return cudaSuccess;
      write_mla_row_kernel<<<grid, threads, 0, stream>>>(
          p.num_tokens, p.num_seqs, p.page_size, p.num_pages, p.bt_stride, p.cu_seqlens_q,
          p.start_pos, p.block_table, static_cast<const uint16_t*>(p.k), p.rope_cos, p.rope_sin,
          p.rope_max_pos, static_cast<uint8_t*>(p.k_pool), p.slot_mapping, p.error_word);
      cudaError_t e = cudaGetLastError();
      if (e != cudaSuccess || p.q == nullptr) return e;
      const long warps = static_cast<long>(p.num_tokens) * p.num_heads_q;
      rope_mla_q_kernel<<<static_cast<unsigned>((warps * 32 + threads - 1) / threads), threads, 0,
                          stream>>>(p.num_tokens, p.num_seqs, p.num_heads_q, p.cu_seqlens_q,
                                    p.start_pos, static_cast<const uint16_t*>(p.q), p.rope_cos,
                                    p.rope_sin, p.rope_max_pos, static_cast<uint16_t*>(p.q_out),
                                    p.error_word);
      return cudaGetLastError();
    }
    default:
      return cudaErrorInvalidValue;
  }
}

// ----------------------------------------------------------- RoPE tables
namespace {
__global__ void rope_table_kernel(double theta, double rope_scale, int max_pos, int rot_dim,
                                  float* __restrict__ cos_out, float* __restrict__ sin_out) {
  const int half = rot_dim / 2;
  const long n = static_cast<long>(max_pos) * half;
  for (long idx = blockIdx.x * static_cast<long>(blockDim.x) + threadIdx.x; idx < n;
       idx += static_cast<long>(gridDim.x) * blockDim.x) {
    const int pos = static_cast<int>(idx / half), i = static_cast<int>(idx % half);
    const double inv_freq = pow(theta, -2.0 * i / static_cast<double>(rot_dim));
    const double angle = (static_cast<double>(pos) / rope_scale) * inv_freq;
    cos_out[idx] = static_cast<float>(cos(angle));
    sin_out[idx] = static_cast<float>(sin(angle));
  }
}
}  // namespace

cudaError_t launch_rope_table(float theta, float rope_scale, int max_pos, int rot_dim,
                              float* cos_out, float* sin_out, cudaStream_t stream) {
  const long n = static_cast<long>(max_pos) * (rot_dim / 2);
  const int threads = 256;
  const int grid = static_cast<int>(n / threads + 1 < 4096 ? n / threads + 1 : 4096);
  rope_table_kernel<<<grid, threads, 0, stream>>>(theta, rope_scale, max_pos, rot_dim, cos_out,
                                                  sin_out);
  return cudaGetLastError();
}

}  // namespace qpkv
