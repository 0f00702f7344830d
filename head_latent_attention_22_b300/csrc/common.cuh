// Shared device-side helpers of the MLA library: the device error word and
// small conversions. Kernels never trap: a bad index or a wait that runs out
// sets a bit here and the kernel skips the access or returns.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/mla.h"

namespace mla {

enum : unsigned { ERR_BIT_BOUNDS = 1u, ERR_BIT_TIMEOUT = 2u };

// One error word per device (module scope: the whole library is one
// translation unit, so this is the only definition).
static __device__ unsigned int g_dev_error = 0;

__device__ __forceinline__ void flag_error(unsigned bit) { atomicOr(&g_dev_error, bit); }

__device__ __forceinline__ float bf16_to_f32(uint16_t h) {
  return __uint_as_float(static_cast<uint32_t>(h) << 16);
}

// Round-to-nearest-even fp32 -> bf16 bits (the hardware conversion).
__device__ __forceinline__ uint16_t f32_to_bf16_bits(float f) {
  __nv_bfloat16 h = __float2bfloat16_rn(f);
  return *reinterpret_cast<uint16_t*>(&h);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  return static_cast<uint32_t>(f32_to_bf16_bits(lo)) |
         (static_cast<uint32_t>(f32_to_bf16_bits(hi)) << 16);
}

// Two fp32 -> two E4M3 codes, round-to-nearest-even, saturating to +-448.
// Byte 0 of the result holds `lo`, byte 1 holds `hi`.
__device__ __forceinline__ uint16_t f32x2_to_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// One E4M3 code -> fp32 (exact).
__device__ __forceinline__ float e4m3_to_f32(uint8_t code) {
  uint32_t h2;
  uint16_t c = code;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(c));
  __half_raw hr;
  hr.x = static_cast<unsigned short>(h2 & 0xffffu);
  return __half2float(__half(hr));
}

template <typename T>
__device__ __forceinline__ float load_as_f32(const T* p, int64_t i);
template <>
__device__ __forceinline__ float load_as_f32<float>(const float* p, int64_t i) { return p[i]; }
template <>
__device__ __forceinline__ float load_as_f32<uint16_t>(const uint16_t* p, int64_t i) {
  return bf16_to_f32(p[i]);
}

__host__ __device__ inline size_t row_bytes_of(int cache_dtype, int d_c, int d_rope) {
  switch (cache_dtype) {
    case MLA_DTYPE_BF16: return static_cast<size_t>(d_c + d_rope) * 2;
    case MLA_DTYPE_FP32: return static_cast<size_t>(d_c + d_rope) * 4;
    case MLA_DTYPE_FP8_E4M3_B128: return static_cast<size_t>(d_c) + 4 * (d_c / 128) + 2 * d_rope;
    default: return 0;
  }
}

}  // namespace mla
