// Device helpers shared by the qpkv kernels: bf16 / E4M3 conversions with
// explicit rounding, warp reductions, varlen bookkeeping.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "ptx.cuh"

namespace qpkv {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

// Two float32 -> two E4M3 codes (round to nearest even, saturate to +-448);
// `hi` lands in the upper byte of the 16-bit result.
__device__ __forceinline__ uint16_t f32x2_to_e4m3x2(float hi, float lo) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ uint8_t f32_to_e4m3(float x) {
  return static_cast<uint8_t>(f32x2_to_e4m3x2(0.f, x) & 0xFF);
}

// Two E4M3 codes (low byte = element 0) -> two floats (exact).
__device__ __forceinline__ float2 e4m3x2_to_f32x2(uint16_t codes) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(codes));
  __half2 h = *reinterpret_cast<__half2*>(&h2);
  return __half22float2(h);
}

// Two float32 -> packed f16x2 (round to nearest even); `hi` in the upper half.
__device__ __forceinline__ uint32_t f32x2_to_f16x2(float hi, float lo) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Packed f16x2 -> two E4M3 codes (round to nearest even, saturate to +-448).
__device__ __forceinline__ uint16_t f16x2_to_e4m3x2(uint32_t h2) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f16x2 %0, %1;" : "=h"(r) : "r"(h2));
  return r;
}

// Two E4M3 codes -> packed f16x2 (exact).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint16_t codes) {
  uint32_t r;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(codes));
  return r;
}

// Packed f16x2 a - b (round to nearest even).
__device__ __forceinline__ uint32_t f16x2_sub(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// Packed f16x2 a + b (round to nearest even).
__device__ __forceinline__ uint32_t f16x2_add(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("add.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// acc + both f16 halves of a packed pair, each added in f32 (mixed-precision
// adds: the f16 values enter exactly).
__device__ __forceinline__ float add_f16x2_to_f32(float acc, uint32_t h2) {
  const uint16_t lo = static_cast<uint16_t>(h2 & 0xFFFFu), hi = static_cast<uint16_t>(h2 >> 16);
  asm("add.rn.f32.f16 %0, %1, %0;" : "+f"(acc) : "h"(lo));
  asm("add.rn.f32.f16 %0, %1, %0;" : "+f"(acc) : "h"(hi));
  return acc;
}

__device__ __forceinline__ float e4m3_to_f32(uint8_t code) {
  return e4m3x2_to_f32x2(static_cast<uint16_t>(code)).x;
}

// max(a, b, c) in one instruction.
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Packed pairs of float32 (one 64-bit register pair): a * b + c and a + b,
// each element rounded to nearest like fmaf / the scalar add.
__device__ __forceinline__ uint64_t f32x2_pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ float2 f32x2_unpack(uint64_t v) {
  float2 r;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
  return r;
}
__device__ __forceinline__ uint64_t f32x2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t f32x2_add(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Sequence index of a token given inclusive prefix sums cu[0..B): the
// smallest b with t < cu[b].
__device__ __forceinline__ int seq_of_token(const int32_t* __restrict__ cu, int B, int t) {
  int lo = 0, hi = B - 1;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (t < __ldg(cu + mid)) hi = mid; else lo = mid + 1;
  }
  return lo;
}

__device__ __forceinline__ int seq_begin(const int32_t* __restrict__ cu, int b) {
  return b == 0 ? 0 : __ldg(cu + b - 1);
}

}  // namespace qpkv
