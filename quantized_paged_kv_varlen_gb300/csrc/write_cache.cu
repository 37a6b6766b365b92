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
// Rounding is explicit so the bytes are reproducible: the codes are those
// of IEEE float32 division (__fdiv_rn, or a reciprocal product where that
// provably rounds the same way), nearest-even conversions, RoPE products
// and sums rounded separately (__fmul_rn / __fadd_rn / __fsub_rn, no
// contraction).
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
// One CTA of 1024 threads per (sequence, 128-token block, group of kWrHeads
// heads).  Thread tid owns token row r = tid / 8 of the block and the eight
// RoPE pairs i in [8j, 8j + 8), j = tid % 8: elements [8j, 8j + 8) and
// [64 + 8j, 64 + 8j + 8) of every 128-wide head.  A row's cos / sin values
// and page slot are the same for all heads, so they are read once.  The CTA
// then walks its heads: every thread copies its own 96 input bytes (Q, K
// and V) of the next head into a two-stage shared-memory ring with cp.async
// while the current head is processed.  Q and K are rotated once for their
// maxima (one block-wide barrier for both), then rotated again from the
// ring and quantised, which keeps the loop within the 64 registers a
// 1024-thread CTA allows; V is stored as it is.  A thread reads back only
// what it copied, so the ring needs no barrier.  The division by the block
// scale is a multiply by its reciprocal, with the exact division taken for
// a group of four codes when one of them sits near a rounding boundary.
constexpr int kBlk = 128;
constexpr int kWrThreads = 1024, kWrHeads = 8;
constexpr int kWrPlane = kWrThreads * 16;            // one 16-byte half of one tensor
constexpr int kWrStage = 6 * kWrPlane;               // Q, K, V halves of one head
constexpr int kWrSmem = 2 * kWrStage;
static_assert(kWrThreads == 8 * kBlk && kWrThreads / 32 == 32, "one row per 8 threads");

// 1.5 * 2^23: a float of magnitude below 2^22 plus this constant, rounded
// to float32, is the constant plus the value rounded to an integer (nearest
// even), held in the low mantissa bits.
constexpr float kRoundMagic = 12582912.0f;
// With s = float32(amax / 127) and inv = float32(127 / amax), the product
// p = float32(y * inv) lies within 3 * 2^-24 * |y / s| of y / s, and the
// correctly rounded quotient float32(y / s) within 2^-24 * |y / s|; as
// |y / s| <= 127.00001 (|y| <= amax), the two are at most 3.1e-5 apart.  A
// product further than 1e-4 from every half-integer therefore rounds to the
// same integer as the quotient; closer ones take the exact division, and so
// does every code when s lies outside [1e-30, 1e30] (1 / amax not normal).
constexpr float kNearHalf = 0.4999f;

// Fast INT8 code of y / s: returns kRoundMagic + n (n = the code), whose low
// byte is n's two's-complement byte, and folds |p - n| into dev.
__device__ __forceinline__ float int8_code_fast(float y, float inv, float& dev) {
  const float p = __fmul_rn(y, inv);
  const float f = __fadd_rn(p, kRoundMagic);
  dev = fmaxf(dev, fabsf(__fsub_rn(p, __fsub_rn(f, kRoundMagic))));
  return f;
}

// The same code from the correctly rounded float32 quotient, in the same
// encoding: clamp(RNE(y / scale), -127, 127), 0 for a zero scale.
__device__ __forceinline__ float int8_code_exact(float y, float scale) {
  const int c = scale != 0.f ? min(127, max(-127, __float2int_rn(__fdiv_rn(y, scale)))) : 0;
  return __int_as_float(__float_as_int(kRoundMagic) + c);
}

// Low bytes of four codes in kRoundMagic + n form -> one little-endian word.
__device__ __forceinline__ uint32_t low_bytes4(float a, float b, float c, float d) {
  const uint32_t lo = __byte_perm(__float_as_uint(a), __float_as_uint(b), 0x0040);
  const uint32_t hi = __byte_perm(__float_as_uint(c), __float_as_uint(d), 0x0040);
  return __byte_perm(lo, hi, 0x5410);
}

__device__ __forceinline__ void unpack_bf16x8(const uint4& raw, float (&x)[8]) {
  const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    x[2 * e] = bf16_bits_to_float(w[e] & 0xFFFF);
    x[2 * e + 1] = bf16_bits_to_float(w[e] >> 16);
  }
}

__device__ __forceinline__ void load_bf16x8(const uint16_t* src, float (&x)[8]) {
  unpack_bf16x8(*reinterpret_cast<const uint4*>(src), x);
}

// Rotate-half RoPE of one thread's 8 pairs (products and sums rounded
// separately), minus the smoothing mean km (shared, 128 floats; NULL: none);
// y[0..7] are elements 8j + e, y[8..15] elements 64 + 8j + e.  Rows outside
// the sequence come out zero: their ring bytes and cos / sin are zero and
// they pass no mean.  Returns the bits of max |y| (non-negative floats order
// like their bit patterns).
__device__ __forceinline__ uint32_t rope_row(const uint4& lo, const uint4& hi,
                                             const float (&cs)[8], const float (&sn)[8],
                                             const float* km, int j, float (&y)[16]) {
  float a[8], c[8];
  unpack_bf16x8(lo, a);
  unpack_bf16x8(hi, c);
  float amax = 0.f;
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    float r1 = __fsub_rn(__fmul_rn(a[e], cs[e]), __fmul_rn(c[e], sn[e]));
    float r2 = __fadd_rn(__fmul_rn(c[e], cs[e]), __fmul_rn(a[e], sn[e]));
    if (km != nullptr) {
      r1 = __fsub_rn(r1, km[8 * j + e]);
      r2 = __fsub_rn(r2, km[64 + 8 * j + e]);
    }
    y[e] = r1;
    y[8 + e] = r2;
    amax = fmax3(amax, fabsf(y[e]), fabsf(y[8 + e]));
  }
  return __float_as_uint(amax);
}

// Scale amax / 127 (float32 division) and the codes of y: fast path from
// 127 / amax, exact division where a product sits near a half-integer or
// the reciprocal would not be a normal float.  Stores the 16 codes at dst
// (row base + 8j; NULL: none).
__device__ __forceinline__ float quant_row(const float (&y)[16], float amax, int8_t* dst) {
  const float scale = __fdiv_rn(amax, 127.0f);
  const float inv = __fdiv_rn(127.0f, amax);
  const bool fast = scale >= 1e-30f && scale <= 1e30f;
  uint32_t w[4];
#pragma unroll
  for (int g = 0; g < 4; ++g) {
    float dev = 0.f;
    w[g] = low_bytes4(int8_code_fast(y[4 * g], inv, dev), int8_code_fast(y[4 * g + 1], inv, dev),
                      int8_code_fast(y[4 * g + 2], inv, dev), int8_code_fast(y[4 * g + 3], inv, dev));
    if (!fast || !(dev <= kNearHalf))   // rare: this group of four by division
      w[g] = low_bytes4(int8_code_exact(y[4 * g], scale), int8_code_exact(y[4 * g + 1], scale),
                        int8_code_exact(y[4 * g + 2], scale), int8_code_exact(y[4 * g + 3], scale));
  }
  if (dst != nullptr) {
    *reinterpret_cast<uint2*>(dst) = make_uint2(w[0], w[1]);
    *reinterpret_cast<uint2*>(dst + 64) = make_uint2(w[2], w[3]);
  }
  return scale;
}

// K smoothing, pass 1: per (sequence, 128-token block, kv head) the int64 sum
// over the block's tokens of RNE(clamp(k_rot, -2^15, 2^15) * 2^24) per dim
// (exact, so the order of the sums does not matter).  Thread tid takes rows
// tid / 8 + 32 i and the eight RoPE pairs of j = tid % 8 (16-byte loads, as
// in the write); the 32 row phases meet in shared memory.  The rotation is
// the one the write applies.
constexpr float kMeanClamp = 32768.0f, kMeanOne = 16777216.0f;   // 2^15, 2^24

__global__ void __launch_bounds__(256) k_block_sum_kernel(
    int Hkv, int num_blocks, int max_pos, const int32_t* __restrict__ cu,
    const uint16_t* __restrict__ k,
    const float* __restrict__ cos_t, const float* __restrict__ sin_t,
    long long* __restrict__ partial) {
  __shared__ long long part[32][128];
  const int blk = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int begin = seq_begin(cu, b);
  const int L = __ldg(cu + b) - begin;
  if (blk * kBlk >= L) return;
  const int rp = threadIdx.x >> 3, j = threadIdx.x & 7;
  // tokens past the launched blocks or the RoPE tables are the write's to flag
  const int n = min(kBlk, min(L, max_pos) - blk * kBlk);
  // all four rows' loads first (rows past the block read as zeros, which
  // add nothing), then the arithmetic
  constexpr int kRows = kBlk / 32;
  uint4 raw[kRows][2];
  float4 cv[kRows][2], sv[kRows][2];
#pragma unroll
  for (int i = 0; i < kRows; ++i) {
    const int r = rp + 32 * i, pos = blk * kBlk + r;
    raw[i][0] = raw[i][1] = make_uint4(0u, 0u, 0u, 0u);
    cv[i][0] = cv[i][1] = sv[i][0] = sv[i][1] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (r < n) {
      const uint4* row = reinterpret_cast<const uint4*>(
          k + (static_cast<size_t>(begin + pos) * Hkv + h) * 128 + 8 * j);
      raw[i][0] = __ldcs(row);
      raw[i][1] = __ldcs(row + 8);   // elements 64 + 8j
      const float4* cp = reinterpret_cast<const float4*>(cos_t + static_cast<size_t>(pos) * 64 + 8 * j);
      const float4* sp = reinterpret_cast<const float4*>(sin_t + static_cast<size_t>(pos) * 64 + 8 * j);
      cv[i][0] = __ldg(cp);
      cv[i][1] = __ldg(cp + 1);
      sv[i][0] = __ldg(sp);
      sv[i][1] = __ldg(sp + 1);
    }
  }
  long long acc[16];
#pragma unroll
  for (int e = 0; e < 16; ++e) acc[e] = 0;
#pragma unroll
  for (int i = 0; i < kRows; ++i) {
    float a[8], c[8];
    unpack_bf16x8(raw[i][0], a);
    unpack_bf16x8(raw[i][1], c);
    const float cs[8] = {cv[i][0].x, cv[i][0].y, cv[i][0].z, cv[i][0].w,
                         cv[i][1].x, cv[i][1].y, cv[i][1].z, cv[i][1].w};
    const float sn[8] = {sv[i][0].x, sv[i][0].y, sv[i][0].z, sv[i][0].w,
                         sv[i][1].x, sv[i][1].y, sv[i][1].z, sv[i][1].w};
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float y1 = __fsub_rn(__fmul_rn(a[e], cs[e]), __fmul_rn(c[e], sn[e]));
      const float y2 = __fadd_rn(__fmul_rn(c[e], cs[e]), __fmul_rn(a[e], sn[e]));
      acc[e] += __float2ll_rn(fminf(fmaxf(y1, -kMeanClamp), kMeanClamp) * kMeanOne);
      acc[8 + e] += __float2ll_rn(fminf(fmaxf(y2, -kMeanClamp), kMeanClamp) * kMeanOne);
    }
  }
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    part[rp][8 * j + e] = acc[e];
    part[rp][64 + 8 * j + e] = acc[8 + e];
  }
  __syncthreads();
  if (threadIdx.x < 128) {
    long long sum = 0;
#pragma unroll 8
    for (int p = 0; p < 32; ++p) sum += part[p][threadIdx.x];
    partial[((static_cast<size_t>(b) * num_blocks + blk) * Hkv + h) * 128 + threadIdx.x] = sum;
  }
}

// FP8 V, pass 1: per (sequence, 128-token block, kv head) the largest |v|
// of each channel over the block's tokens (a maximum: order-free); the same
// thread layout as the K sums.
__global__ void __launch_bounds__(256) v_block_max_kernel(
    int Hkv, int num_blocks, const int32_t* __restrict__ cu, const uint16_t* __restrict__ v,
    float* __restrict__ vmax) {
  __shared__ float part[32][128];
  const int blk = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int begin = seq_begin(cu, b);
  const int L = __ldg(cu + b) - begin;
  if (blk * kBlk >= L) return;
  const int rp = threadIdx.x >> 3, j = threadIdx.x & 7;
  const int n = min(kBlk, L - blk * kBlk);
  constexpr int kRows = kBlk / 32;
  uint4 raw[kRows][2];
#pragma unroll
  for (int i = 0; i < kRows; ++i) {
    const int r = rp + 32 * i;
    raw[i][0] = raw[i][1] = make_uint4(0u, 0u, 0u, 0u);   // rows past the block: zeros
    if (r < n) {
      const uint4* row = reinterpret_cast<const uint4*>(
          v + (static_cast<size_t>(begin + blk * kBlk + r) * Hkv + h) * 128 + 8 * j);
      raw[i][0] = __ldcs(row);
      raw[i][1] = __ldcs(row + 8);   // elements 64 + 8j
    }
  }
  float m[16];
#pragma unroll
  for (int e = 0; e < 16; ++e) m[e] = 0.f;
#pragma unroll
  for (int i = 0; i < kRows; ++i) {
    float a[8], c[8];
    unpack_bf16x8(raw[i][0], a);
    unpack_bf16x8(raw[i][1], c);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      m[e] = fmaxf(m[e], fabsf(a[e]));
      m[8 + e] = fmaxf(m[8 + e], fabsf(c[e]));
    }
  }
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    part[rp][8 * j + e] = m[e];
    part[rp][64 + 8 * j + e] = m[8 + e];
  }
  __syncthreads();
  if (threadIdx.x < 128) {
    float mx = 0.f;
#pragma unroll 8
    for (int p = 0; p < 32; ++p) mx = fmaxf(mx, part[p][threadIdx.x]);
    vmax[((static_cast<size_t>(b) * num_blocks + blk) * Hkv + h) * 128 + threadIdx.x] = mx;
  }
}

__global__ void __launch_bounds__(kWrThreads, 1) write_int8_block128_rope_kernel(
    int B, int Hq, int Hkv, int ps, int num_pages, int bt_stride, int num_blocks, int nblk_launch,
    const int32_t* __restrict__ cu, const int32_t* __restrict__ bt,
    const uint16_t* __restrict__ q, const uint16_t* __restrict__ k,
    const uint16_t* __restrict__ v, const float* __restrict__ cos_t,
    const float* __restrict__ sin_t, int8_t* __restrict__ k_pool, uint16_t* __restrict__ v_pool,
    float* __restrict__ k_bscale, int8_t* __restrict__ q_out, float* __restrict__ q_bscale,
    int32_t* __restrict__ slots, const long long* __restrict__ partial, float* __restrict__ k_mean,
    const float* __restrict__ vmax, float* __restrict__ v_cscale, int max_pos, int* err) {
  constexpr int D = 128;
  __shared__ uint2 red[2][32];          // per warp: max |y| bits of Q and of K
  __shared__ float km[kWrHeads][D];    // K smoothing means of the group's heads
  __shared__ float vsc[kWrHeads][D];   // FP8 V channel scales of the group's heads
  extern __shared__ __align__(16) uint8_t ring[];
  const int hmax = max(Hq, Hkv);
  const int ngroups = (hmax + kWrHeads - 1) / kWrHeads;
  const int hg = blockIdx.x % ngroups;
  const int b = (blockIdx.x / ngroups) % B, blk = blockIdx.x / ngroups / B;
  const int begin = seq_begin(cu, b);
  const int L = __ldg(cu + b) - begin;
  if (blk * kBlk >= L) return;  // block past this sequence's end
  // a sequence longer than the launch (max_seqlen) or the RoPE tables
  const int nblk = (L + kBlk - 1) / kBlk;
  if ((nblk > nblk_launch || L > max_pos) && blk == 0 && hg == 0 && threadIdx.x == 0)
    report_error(err, kDevErrBadLength);
  const int h0 = hg * kWrHeads, nh = min(kWrHeads, hmax - h0);
  const int r = threadIdx.x >> 3, j = threadIdx.x & 7;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int pos = blk * kBlk + r;
  const bool valid = pos < L && pos < max_pos;
  const size_t t = static_cast<size_t>(begin + pos);

  // ring stage s, tensor u (Q, K, V), half (elements 8j.. / 64 + 8j..):
  // planes of 16 bytes per thread, so a warp's accesses are contiguous
  auto at = [&](int s, int u, int half) {
    return ring + s * kWrStage + (2 * u + half) * kWrPlane + threadIdx.x * 16;
  };
  auto copy_in = [&](int s, int u, const uint16_t* src) {
    const uint32_t n = valid ? 16u : 0u;
    cp_async_16_zfill(at(s, u, 0), src + 8 * j, n);
    cp_async_16_zfill(at(s, u, 1), src + 64 + 8 * j, n);
  };
  auto fetch = [&](int hh) {
    if (hh < nh) {
      const int h = h0 + hh, s = hh & 1;
      const size_t row = valid ? t : 0;
      if (h < Hq) copy_in(s, 0, q + (row * Hq + h) * D);
      if (h < Hkv) {
        copy_in(s, 1, k + (row * Hkv + h) * D);
        if (valid) copy_in(s, 2, v + (row * Hkv + h) * D);
      }
    }
    cp_async_commit();
  };
  auto ring16 = [&](int s, int u, int half) { return *reinterpret_cast<const uint4*>(at(s, u, half)); };
  fetch(0);

  float cs[8], sn[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) cs[e] = sn[e] = 0.f;
  if (valid) {
    const float4* cp = reinterpret_cast<const float4*>(cos_t + static_cast<size_t>(pos) * 64 + 8 * j);
    const float4* sp = reinterpret_cast<const float4*>(sin_t + static_cast<size_t>(pos) * 64 + 8 * j);
    const float4 c0 = __ldg(cp), c1 = __ldg(cp + 1), s0 = __ldg(sp), s1 = __ldg(sp + 1);
    cs[0] = c0.x; cs[1] = c0.y; cs[2] = c0.z; cs[3] = c0.w;
    cs[4] = c1.x; cs[5] = c1.y; cs[6] = c1.z; cs[7] = c1.w;
    sn[0] = s0.x; sn[1] = s0.y; sn[2] = s0.z; sn[3] = s0.w;
    sn[4] = s1.x; sn[5] = s1.y; sn[6] = s1.z; sn[7] = s1.w;
  }
  size_t slot = 0;
  bool ok = false;
  if (valid && h0 < Hkv) {
    const int page = pool_page(bt, bt_stride, b, pos, ps, num_pages, j == 0 ? err : nullptr);
    ok = page >= 0;
    slot = static_cast<size_t>(ok ? page : 0) * ps + (pos % ps);
    if (ok && slots != nullptr && hg == 0 && j == 0) slots[t] = static_cast<int32_t>(slot);
  }

  const bool smooth = partial != nullptr, v8 = vmax != nullptr;
  if ((smooth || v8) && h0 < Hkv) {
    // pass 2 of K smoothing (the sequence's mean from the exact block sums)
    // and of FP8 V (the channel's absmax over the sequence -> scale / 448)
    const int nsum = min(nblk, nblk_launch);
    for (int idx = threadIdx.x; idx < nh * D; idx += kWrThreads) {
      const int hh = idx / D, d = idx % D, h = h0 + hh;
      if (h >= Hkv) continue;
      const size_t o = (static_cast<size_t>(b) * Hkv + h) * D + d;
      if (smooth) {
        long long sum = 0;
        for (int jb = 0; jb < nsum; ++jb)
          sum += partial[((static_cast<size_t>(b) * num_blocks + jb) * Hkv + h) * D + d];
        const float m = __double2float_rn(
            __ll2double_rn(sum) / (static_cast<double>(L) * static_cast<double>(kMeanOne)));
        km[hh][d] = m;
        if (blk == 0) k_mean[o] = m;
      }
      if (v8) {
        float amax = 0.f;
        for (int jb = 0; jb < nsum; ++jb)
          amax = fmaxf(amax, vmax[((static_cast<size_t>(b) * num_blocks + jb) * Hkv + h) * D + d]);
        const float sc = __fdiv_rn(amax, 448.0f);
        vsc[hh][d] = sc;
        if (blk == 0) v_cscale[o] = sc;
      }
    }
    __syncthreads();
  }

  for (int hh = 0; hh < nh; ++hh) {
    fetch(hh + 1);
    cp_async_wait_group<1>();   // this head's group has landed
    const int s = hh & 1, h = h0 + hh;
    const bool has_q = h < Hq, has_k = h < Hkv;   // the same for the whole CTA
    const float* kmh = smooth && valid ? km[hh] : nullptr;   // this head's K mean
    float y[16];
    uint32_t mq = 0u, mk = 0u;
    if (has_q) mq = rope_row(ring16(s, 0, 0), ring16(s, 0, 1), cs, sn, nullptr, j, y);
    if (has_k) mk = rope_row(ring16(s, 1, 0), ring16(s, 1, 1), cs, sn, kmh, j, y);
    mq = __reduce_max_sync(0xffffffffu, mq);
    mk = __reduce_max_sync(0xffffffffu, mk);
    if (lane == 0) red[hh & 1][warp] = make_uint2(mq, mk);
    __syncthreads();
    const uint2 m = red[hh & 1][lane];
    mq = __reduce_max_sync(0xffffffffu, m.x);
    mk = __reduce_max_sync(0xffffffffu, m.y);
    const size_t sb = static_cast<size_t>(b) * num_blocks + blk;
    if (has_q) {
      rope_row(ring16(s, 0, 0), ring16(s, 0, 1), cs, sn, nullptr, j, y);
      int8_t* dst = valid ? q_out + (t * Hq + h) * D + 8 * j : nullptr;
      const float sc = quant_row(y, __uint_as_float(mq), dst);
      if (threadIdx.x == 0) q_bscale[sb * Hq + h] = sc;
    }
    if (has_k) {
      rope_row(ring16(s, 1, 0), ring16(s, 1, 1), cs, sn, kmh, j, y);
      int8_t* dst = ok ? k_pool + (slot * Hkv + h) * D + 8 * j : nullptr;
      const float sc = quant_row(y, __uint_as_float(mk), dst);
      if (threadIdx.x == 0) k_bscale[sb * Hkv + h] = sc;
      if (ok && !v8) {
        uint4* vd = reinterpret_cast<uint4*>(v_pool + (slot * Hkv + h) * D + 8 * j);
        vd[0] = ring16(s, 2, 0);
        vd[8] = ring16(s, 2, 1);   // elements 64 + 8j
      } else if (ok) {
        // E4M3 codes of v / channel scale (float32 division); one byte per element
        uint8_t* vd = reinterpret_cast<uint8_t*>(v_pool) + (slot * Hkv + h) * D + 8 * j;
#pragma unroll
        for (int g = 0; g < 2; ++g) {
          float x[8];
          unpack_bf16x8(ring16(s, 2, g), x);
          uint32_t w[2] = {0u, 0u};
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const float sc = vsc[hh][64 * g + 8 * j + e];
            const uint32_t code = sc != 0.f ? f32_to_e4m3(__fdiv_rn(x[e], sc)) : 0u;
            w[e / 4] |= code << (8 * (e % 4));
          }
          *reinterpret_cast<uint2*>(vd + 64 * g) = make_uint2(w[0], w[1]);
        }
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
        v_block_max_kernel<<<dim3(nblk, p.num_heads_kv, p.num_seqs), 256, 0, stream>>>(
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
      // blocks outermost, so the heavier full blocks start first and the
      // CTAs reading one block's cos / sin rows run together
      const long ctas = static_cast<long>(nblk) * p.num_seqs * ((hmax + kWrHeads - 1) / kWrHeads);
      cudaError_t e = cudaFuncSetAttribute(write_int8_block128_rope_kernel,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, kWrSmem);
      if (e != cudaSuccess) return e;
      write_int8_block128_rope_kernel<<<static_cast<unsigned>(ctas), kWrThreads, kWrSmem, stream>>>(
          p.num_seqs, p.num_heads_q, p.num_heads_kv, p.page_size, p.num_pages, p.bt_stride,
          p.num_blocks, nblk, p.cu_seqlens_q, p.block_table, static_cast<const uint16_t*>(p.q),
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
