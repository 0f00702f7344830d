// mla_append kernels: latent RMSNorm (DeepSeek-V2 report, section 3.1.2),
// decoupled RoPE on the shared key (section 2.1.3) and the paged row write.
// One warp per token. The vectorised kernel covers the DeepSeek-V2 row
// (d_c = 512, d_rope = 64, bf16 inputs) with 16-byte loads and stores; the
// scalar kernel covers every other shape.
#pragma once

#include "common.cuh"

namespace mla {

// Frequencies of the decoupled RoPE: f_m = theta^(-2m/d), and under YaRN (s > 1) the
// "NTK-by-parts" rule of YaRN (Peng et al. 2023) that the DeepSeek-V2 report applies
// (section 3.1.4): a pair making r = orig_len f / (2 pi) turns over the original context
// keeps f for r >= beta, takes f / s for r <= alpha, and blends linearly in r between.
constexpr int kRopeTable = 64;   // pairs whose frequency the host computes (d_rope <= 128)

struct RopeFreq {
  double log_theta;
  double yarn_s, yarn_alpha, yarn_beta, yarn_orig_len;   // yarn_s <= 1: plain RoPE
  int n_table;                                           // pairs m < n_table take table[m]
  double table[kRopeTable];                              // f_m, computed by the host by the rule below
};

__host__ __device__ inline double rope_freq_rule(const RopeFreq& r, int m, int d_rope) {
  double f = exp(-(2.0 * m / d_rope) * r.log_theta);
  if (r.yarn_s > 1.0) {
    const double turns = r.yarn_orig_len * f / (2.0 * 3.141592653589793);
    double g = (turns - r.yarn_alpha) / (r.yarn_beta - r.yarn_alpha);
    g = g < 0.0 ? 0.0 : (g > 1.0 ? 1.0 : g);
    f = (1.0 - g) * f / r.yarn_s + g * f;
  }
  return f;
}

__device__ __forceinline__ double rope_freq(const RopeFreq& r, int m, int d_rope) {
  return m < r.n_table ? r.table[m] : rope_freq_rule(r, m, d_rope);
}

struct AppendArgs {
  const void* c_raw;
  const void* k_raw;
  const int32_t* positions;
  const int32_t* seq_idx;
  const float* gamma;
  uint8_t* pool;
  int64_t num_pages;
  const int32_t* block_table;
  int batch, max_pages, n_tokens, d_c, d_rope, page_size, cache_dtype, rope_interleaved;
  float eps;
  RopeFreq rf;
  int64_t row_bytes;
};

// Pool row of token t, or -1 (and the bounds bit) when any index is outside its array.
__device__ __forceinline__ int64_t append_slot(const AppendArgs& a, int t, int* pos_out) {
  const int pos = a.positions[t];
  const int s = a.seq_idx ? a.seq_idx[t] : t;
  if (s < 0 || s >= a.batch || pos < 0) return -1;
  const int pg = pos / a.page_size;
  if (pg >= a.max_pages) return -1;
  const int64_t page = a.block_table ? static_cast<int64_t>(a.block_table[static_cast<int64_t>(s) * a.max_pages + pg])
                                     : static_cast<int64_t>(s) * a.max_pages + pg;
  if (page < 0 || page >= a.num_pages) return -1;
  *pos_out = pos;
  return page * a.page_size + pos % a.page_size;
}

// Rotation of pair m at position pos by the angle pos * f_m, formed in fp64. For a result stored in
// bf16 (kBf16Out) the angle is reduced to [-pi, pi] in fp64 (Cody-Waite reduction by 2 pi split into
// a head and a tail) and its sine and cosine are taken in fp32: their error (a few 1e-8) is far
// below the bf16 rounding of the stored value, while fp64 sines and cosines are slow on this part.
// A result stored in fp32 keeps the fp64 sine and cosine.
template <bool kBf16Out>
__device__ __forceinline__ void rope_pair(double a, double b, int m, int d_rope, int pos,
                                          const RopeFreq& rf, double* ra, double* rb) {
  const double inv_freq = rope_freq(rf, m, d_rope);
  const double ang = static_cast<double>(pos) * inv_freq;
  if (!kBf16Out) {
    double sn, cs;
    sincos(ang, &sn, &cs);
    *ra = a * cs - b * sn;
    *rb = a * sn + b * cs;
    return;
  }
  constexpr double kTwoPiHi = 6.283185307179586;          // 2 pi rounded to fp64
  constexpr double kTwoPiLo = 2.4492935982947064e-16;     // 2 pi - kTwoPiHi
  const double k = rint(ang * (1.0 / kTwoPiHi));
  const double red = fma(-k, kTwoPiLo, fma(-k, kTwoPiHi, ang));
  float sf, cf;
  sincosf(static_cast<float>(red), &sf, &cf);
  const double sn = sf, cs = cf;
  *ra = a * cs - b * sn;
  *rb = a * sn + b * cs;
}

__device__ __forceinline__ uint16_t f64_to_bf16_bits(double d) {
  __nv_bfloat16 h = __double2bfloat16(d);  // one rounding, to nearest even
  return *reinterpret_cast<uint16_t*>(&h);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// ---------------------------------------------------------------- d_c = 512, d_rope = 64, bf16 in
// Lane l owns latent elements [16 l, 16 l + 16) and rope pair l.
template <int CACHE>  // MLA_DTYPE_BF16 or MLA_DTYPE_FP8_E4M3_B128
__global__ void __launch_bounds__(256) append_dsv2_kernel(AppendArgs a) {
  const int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (t >= a.n_tokens) return;
  int pos = 0;
  const int64_t slot = append_slot(a, t, &pos);
  if (slot < 0) {
    if (lane == 0) flag_error(ERR_BIT_BOUNDS);
    return;
  }
  uint8_t* row = a.pool + slot * a.row_bytes;

  const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.c_raw) +
                                                    static_cast<int64_t>(t) * 512 + 16 * lane);
  uint4 v0 = __ldg(src), v1 = __ldg(src + 1);
  const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
  float x[16];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    x[2 * i] = bf16_to_f32(static_cast<uint16_t>(w[i] & 0xffffu));
    x[2 * i + 1] = bf16_to_f32(static_cast<uint16_t>(w[i] >> 16));
  }
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) ss = fmaf(x[i], x[i], ss);
  ss = warp_sum(ss);
  const float inv = 1.0f / sqrtf(ss / 512.0f + a.eps);
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const float g = a.gamma ? a.gamma[16 * lane + i] : 1.0f;
    x[i] = x[i] * inv * g;
  }

  int rope_off;
  if constexpr (CACHE == MLA_DTYPE_BF16) {
    uint4 o0, o1;
    o0.x = pack_bf16x2(x[0], x[1]);   o0.y = pack_bf16x2(x[2], x[3]);
    o0.z = pack_bf16x2(x[4], x[5]);   o0.w = pack_bf16x2(x[6], x[7]);
    o1.x = pack_bf16x2(x[8], x[9]);   o1.y = pack_bf16x2(x[10], x[11]);
    o1.z = pack_bf16x2(x[12], x[13]); o1.w = pack_bf16x2(x[14], x[15]);
    uint4* dst = reinterpret_cast<uint4*>(row + 32 * lane);
    dst[0] = o0;
    dst[1] = o1;
    rope_off = 1024;
  } else {
    // block of 128 values = lanes 8k .. 8k+7
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(x[i]));
#pragma unroll
    for (int o = 4; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float s = amax == 0.f ? 1.0f : __fdiv_rn(amax, 448.0f);
    uint32_t q[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t lo = f32x2_to_e4m3x2(__fdiv_rn(x[4 * i], s), __fdiv_rn(x[4 * i + 1], s));
      const uint32_t hi = f32x2_to_e4m3x2(__fdiv_rn(x[4 * i + 2], s), __fdiv_rn(x[4 * i + 3], s));
      q[i] = lo | (hi << 16);
    }
    *reinterpret_cast<uint4*>(row + 16 * lane) = make_uint4(q[0], q[1], q[2], q[3]);
    if ((lane & 7) == 0) *reinterpret_cast<float*>(row + 512 + 4 * (lane >> 3)) = s;
    rope_off = 528;
  }

  const uint16_t* kr = static_cast<const uint16_t*>(a.k_raw) + static_cast<int64_t>(t) * 64;
  uint16_t* kdst = reinterpret_cast<uint16_t*>(row + rope_off);
  const int i0 = a.rope_interleaved ? 2 * lane : lane;
  const int i1 = a.rope_interleaved ? 2 * lane + 1 : lane + 32;
  double ra, rb;
  rope_pair<true>(bf16_to_f32(kr[i0]), bf16_to_f32(kr[i1]), lane, 64, pos, a.rf, &ra, &rb);
  if (a.rope_interleaved) {
    *reinterpret_cast<uint32_t*>(kdst + i0) =
        static_cast<uint32_t>(f64_to_bf16_bits(ra)) | (static_cast<uint32_t>(f64_to_bf16_bits(rb)) << 16);
  } else {
    kdst[i0] = f64_to_bf16_bits(ra);
    kdst[i1] = f64_to_bf16_bits(rb);
  }
}

// ---------------------------------------------------------------- any shape (scalar)
template <typename Tin>
__global__ void __launch_bounds__(256) append_generic_kernel(AppendArgs a) {
  const int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (t >= a.n_tokens) return;
  int pos = 0;
  const int64_t slot = append_slot(a, t, &pos);
  if (slot < 0) {
    if (lane == 0) flag_error(ERR_BIT_BOUNDS);
    return;
  }
  uint8_t* row = a.pool + slot * a.row_bytes;
  const Tin* c = static_cast<const Tin*>(a.c_raw) + static_cast<int64_t>(t) * a.d_c;
  const Tin* k = static_cast<const Tin*>(a.k_raw) + static_cast<int64_t>(t) * a.d_rope;

  float ss = 0.f;
  for (int i = lane; i < a.d_c; i += 32) {
    const float x = load_as_f32(c, i);
    ss = fmaf(x, x, ss);
  }
  ss = warp_sum(ss);
  const float inv = 1.0f / sqrtf(ss / static_cast<float>(a.d_c) + a.eps);
  auto cval = [&](int i) { return load_as_f32(c, i) * inv * (a.gamma ? a.gamma[i] : 1.0f); };

  int64_t rope_off = 0;
  if (a.cache_dtype == MLA_DTYPE_FP32) {
    float* dst = reinterpret_cast<float*>(row);
    for (int i = lane; i < a.d_c; i += 32) dst[i] = cval(i);
    rope_off = 4LL * a.d_c;
  } else if (a.cache_dtype == MLA_DTYPE_BF16) {
    uint16_t* dst = reinterpret_cast<uint16_t*>(row);
    for (int i = lane; i < a.d_c; i += 32) dst[i] = f32_to_bf16_bits(cval(i));
    rope_off = 2LL * a.d_c;
  } else {  // FP8_E4M3_B128
    float* scales = reinterpret_cast<float*>(row + a.d_c);
    for (int blk = 0; blk < a.d_c / 128; ++blk) {
      float amax = 0.f;
      for (int i = blk * 128 + lane; i < blk * 128 + 128; i += 32) amax = fmaxf(amax, fabsf(cval(i)));
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
      const float s = amax == 0.f ? 1.0f : __fdiv_rn(amax, 448.0f);
      for (int i = blk * 128 + lane; i < blk * 128 + 128; i += 32)
        row[i] = static_cast<uint8_t>(f32x2_to_e4m3x2(__fdiv_rn(cval(i), s), 0.f) & 0xffu);
      if (lane == 0) scales[blk] = s;
    }
    rope_off = a.d_c + 4LL * (a.d_c / 128);
  }

  const int half = a.d_rope / 2;
  for (int m = lane; m < half; m += 32) {
    const int i0 = a.rope_interleaved ? 2 * m : m;
    const int i1 = a.rope_interleaved ? 2 * m + 1 : m + half;
    double ra, rb;
    if (a.cache_dtype == MLA_DTYPE_FP32)
      rope_pair<false>(load_as_f32(k, i0), load_as_f32(k, i1), m, a.d_rope, pos, a.rf, &ra, &rb);
    else
      rope_pair<true>(load_as_f32(k, i0), load_as_f32(k, i1), m, a.d_rope, pos, a.rf, &ra, &rb);
    if (a.cache_dtype == MLA_DTYPE_FP32) {
      float* dst = reinterpret_cast<float*>(row + rope_off);
      dst[i0] = static_cast<float>(ra);
      dst[i1] = static_cast<float>(rb);
    } else {
      uint16_t* dst = reinterpret_cast<uint16_t*>(row + rope_off);
      dst[i0] = f64_to_bf16_bits(ra);
      dst[i1] = f64_to_bf16_bits(rb);
    }
  }
}

// ---------------------------------------------------------------- mla_rope_query
// q_rope[b, i, :] = RoPE(q_rope_raw[b, i, :], positions[b]) with the frequencies of
// the keys; one thread per (row, pair), so the rotation may be done in place.
struct RopeQueryArgs {
  const void* in;
  void* out;
  const int32_t* positions;
  int batch, n_heads, d_rope, rope_interleaved;
  RopeFreq rf;
};

template <typename T>
__global__ void rope_query_kernel(RopeQueryArgs a) {
  const int half = a.d_rope / 2;
  const int64_t n = static_cast<int64_t>(a.batch) * a.n_heads * half;
  for (int64_t idx = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; idx < n;
       idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int m = static_cast<int>(idx % half);
    const int64_t row = idx / half;   // b * n_heads + i
    const int pos = a.positions[row / a.n_heads];
    if (pos < 0) {
      if (m == 0) flag_error(ERR_BIT_BOUNDS);
      continue;
    }
    const int i0 = a.rope_interleaved ? 2 * m : m;
    const int i1 = a.rope_interleaved ? 2 * m + 1 : m + half;
    const T* src = static_cast<const T*>(a.in) + row * a.d_rope;
    T* dst = static_cast<T*>(a.out) + row * a.d_rope;
    double ra, rb;
    rope_pair<sizeof(T) == 2>(load_as_f32(src, i0), load_as_f32(src, i1), m, a.d_rope, pos, a.rf, &ra, &rb);
    if constexpr (sizeof(T) == 4) {
      dst[i0] = static_cast<float>(ra);
      dst[i1] = static_cast<float>(rb);
    } else {
      dst[i0] = f64_to_bf16_bits(ra);
      dst[i1] = f64_to_bf16_bits(rb);
    }
  }
}

}  // namespace mla
