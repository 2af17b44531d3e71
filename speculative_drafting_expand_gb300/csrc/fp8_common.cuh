// fp8_common.cuh -- pieces of the fp8 (e4m3) KV cache path: f16 MMA
// descriptors, f16 packing and the e4m3 conversions.
#pragma once

#include <cuda_fp16.h>

#include "pe_common.cuh"

namespace pe {

// kind::f16 with f16 A and B (format code 0 in both operand fields).
__host__ __device__ constexpr uint32_t idesc_f16_f32(int M, int N) {
  return (1u << 4) | (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}
// The same with the B operand MN-major.
__host__ __device__ constexpr uint32_t idesc_f16_f32_bmn(int M, int N) {
  return idesc_f16_f32(M, N) | (1u << 16);
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  const __half2 b = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&b);
}

// OCP FP8 E4M3 (bias 7, no infinities, 448 largest).  Two codes in the low
// 16 bits of `codes` (the lower byte is the first element) -> an f16 pair
// (the first element in the low half); every e4m3 value is an f16.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t codes) {
  uint32_t r;
  asm("{\n\t.reg .b16 c;\n\tcvt.u16.u32 c, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, c;\n\t}"
      : "=r"(r)
      : "r"(codes));
  return r;
}

// Two floats -> two e4m3 codes, rounded to nearest even and saturated to
// +-448 (lo in the low byte, hi in the high byte).
__device__ __forceinline__ uint16_t f32x2_to_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// bf16 pair -> f16 pair (through fp32; every bf16 of the activations'
// range is rounded to the nearest f16).
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t v) {
  return pack_f16x2(__uint_as_float(v << 16), __uint_as_float(v & 0xffff0000u));
}

}  // namespace pe
