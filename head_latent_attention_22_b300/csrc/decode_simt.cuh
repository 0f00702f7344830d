// CUDA-core (SIMT) MLA decode for shapes the tensor-core kernels do not
// cover (any n_heads, d_c <= 512, any d_rope/d_head, fp32 or bf16 inputs,
// fp32/bf16/fp8 cache). Same three steps as the tensor-core path, all in
// fp32 (DeepSeek-V2 report, section 2.1.2 absorbed form):
//   1. absorb : q_lat[b,i] = W_UK[i]^T q_nope[b,i]; q_rope appended
//   2. attend : per (sequence, head group, split of the tokens) an online
//               softmax over the split's cache rows -> unnormalised partial
//               o_lat, running max m (log2 domain) and sum l
//   3. combine: log-sum-exp merge of the splits, then out = W_UV[i] o_lat
#pragma once

#include "common.cuh"

namespace mla {

constexpr int kSimtHeadsPerCta = 8;   // one warp per head
constexpr int kSimtTileTokens = 16;   // cache rows staged in shared memory at a time
constexpr int kSimtMaxDc = 512;       // latent elements a lane can hold: 16 per lane

struct SimtArgs {
  const void* q_nope;
  const void* q_rope;
  const void* w_uk;
  const void* w_uv;
  const uint8_t* pool;
  int64_t num_pages;
  const int32_t* block_table;
  const int32_t* seq_lens;
  int batch, max_pages, n_heads, d_c, d_rope, d_head, page_size, cache_dtype;
  int64_t row_bytes;
  float scale_log2;   // softmax scale * log2(e)
  float* out;
  float* q_lat;       // [B, H, d_c + d_rope]
  float* part_o;      // [B, S, H, d_c]
  float* part_m;      // [B, S, H]
  float* part_l;      // [B, S, H]
  int n_splits, split_tokens;
  int max_seq_len;    // host bound the split plan covers
};

// Cache length of sequence b, clamped to the planned bound max_seq_len.
__device__ __forceinline__ int clamped_len(const SimtArgs& a, int b) {
  int L = a.seq_lens[b];
  const int cap = a.max_seq_len;
  if (L < 0 || L > cap) {
    flag_error(ERR_BIT_BOUNDS);
    L = L < 0 ? 0 : cap;
  }
  return L;
}

// Pool row of token `pos` of sequence b (-1 if its page id is outside the pool).
__device__ __forceinline__ int64_t cache_row(const SimtArgs& a, int b, int pos) {
  const int pg = pos / a.page_size;
  const int64_t page = a.block_table ? static_cast<int64_t>(a.block_table[static_cast<int64_t>(b) * a.max_pages + pg])
                                     : static_cast<int64_t>(b) * a.max_pages + pg;
  if (page < 0 || page >= a.num_pages) return -1;
  return page * a.page_size + pos % a.page_size;
}

// Element e (< d_c + d_rope) of a cache row, as fp32.
__device__ __forceinline__ float cache_elem(const SimtArgs& a, const uint8_t* row, int e) {
  switch (a.cache_dtype) {
    case MLA_DTYPE_FP32: return reinterpret_cast<const float*>(row)[e];
    case MLA_DTYPE_BF16: return bf16_to_f32(reinterpret_cast<const uint16_t*>(row)[e]);
    default: {
      if (e < a.d_c) {
        const float s = reinterpret_cast<const float*>(row + a.d_c)[e >> 7];
        return e4m3_to_f32(row[e]) * s;
      }
      const uint16_t* r = reinterpret_cast<const uint16_t*>(row + a.d_c + 4 * (a.d_c / 128));
      return bf16_to_f32(r[e - a.d_c]);
    }
  }
}

template <typename Tin>
__global__ void __launch_bounds__(128) absorb_simt_kernel(SimtArgs a) {
  extern __shared__ float q_s[];  // [d_head]
  const int i = blockIdx.x, b = blockIdx.y;
  const int D = a.d_c + a.d_rope;
  const Tin* qn = static_cast<const Tin*>(a.q_nope) + (static_cast<int64_t>(b) * a.n_heads + i) * a.d_head;
  for (int d = threadIdx.x; d < a.d_head; d += blockDim.x) q_s[d] = load_as_f32(qn, d);
  __syncthreads();
  const Tin* w = static_cast<const Tin*>(a.w_uk) + static_cast<int64_t>(i) * a.d_head * a.d_c;
  float* dst = a.q_lat + (static_cast<int64_t>(b) * a.n_heads + i) * D;
  for (int k = threadIdx.x; k < a.d_c; k += blockDim.x) {
    float acc = 0.f;
    for (int d = 0; d < a.d_head; ++d) acc = fmaf(load_as_f32(w, static_cast<int64_t>(d) * a.d_c + k), q_s[d], acc);
    dst[k] = acc;
  }
  const Tin* qr = static_cast<const Tin*>(a.q_rope) + (static_cast<int64_t>(b) * a.n_heads + i) * a.d_rope;
  for (int r = threadIdx.x; r < a.d_rope; r += blockDim.x) dst[a.d_c + r] = load_as_f32(qr, r);
}

__global__ void __launch_bounds__(32 * kSimtHeadsPerCta) attend_simt_kernel(SimtArgs a) {
  extern __shared__ float smem[];
  const int D = a.d_c + a.d_rope;
  float* q_s = smem;                                  // [heads per CTA][D]
  float* tile = smem + kSimtHeadsPerCta * D;          // [tile tokens][D]
  const int split = blockIdx.x, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.y * kSimtHeadsPerCta + warp;
  const bool head_ok = h < a.n_heads;

  for (int idx = threadIdx.x; idx < kSimtHeadsPerCta * D; idx += blockDim.x) {
    const int hh = blockIdx.y * kSimtHeadsPerCta + idx / D;
    q_s[idx] = hh < a.n_heads ? a.q_lat[(static_cast<int64_t>(b) * a.n_heads + hh) * D + idx % D] : 0.f;
  }
  const int L = clamped_len(a, b);
  const int t0 = split * a.split_tokens;
  const int t1 = min(L, t0 + a.split_tokens);

  float m = -INFINITY, l = 0.f;
  float o[kSimtMaxDc / 32];
#pragma unroll
  for (int r = 0; r < kSimtMaxDc / 32; ++r) o[r] = 0.f;
  const float* qh = q_s + warp * D;

  for (int tb = t0; tb < t1; tb += kSimtTileTokens) {
    const int n = min(kSimtTileTokens, t1 - tb);
    __syncthreads();
    for (int idx = threadIdx.x; idx < n * D; idx += blockDim.x) {
      const int j = idx / D, e = idx % D;
      const int64_t row = cache_row(a, b, tb + j);
      float v = 0.f;
      if (row >= 0) v = cache_elem(a, a.pool + row * a.row_bytes, e);
      else if (e == 0) flag_error(ERR_BIT_BOUNDS);
      tile[idx] = v;
    }
    __syncthreads();
    if (!head_ok) continue;
    float s[kSimtTileTokens];
    float smax = -INFINITY;
#pragma unroll
    for (int j = 0; j < kSimtTileTokens; ++j) {
      float acc = 0.f;
      if (j < n) {
        for (int e = lane; e < D; e += 32) acc = fmaf(qh[e], tile[j * D + e], acc);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        s[j] = acc * a.scale_log2;
      } else {
        s[j] = -INFINITY;
      }
      smax = fmaxf(smax, s[j]);
    }
    const float m_new = fmaxf(m, smax);
    const float alpha = exp2f(m - m_new);   // m = -inf on the first tile -> 0
    float psum = 0.f;
#pragma unroll
    for (int j = 0; j < kSimtTileTokens; ++j) {
      s[j] = exp2f(s[j] - m_new);
      psum += s[j];
    }
    l = l * alpha + psum;
#pragma unroll
    for (int r = 0; r < kSimtMaxDc / 32; ++r) {
      const int k = lane + 32 * r;
      if (k < a.d_c) {
        float acc = o[r] * alpha;
#pragma unroll
        for (int j = 0; j < kSimtTileTokens; ++j) acc = fmaf(s[j], tile[j * D + k], acc);
        o[r] = acc;
      }
    }
    m = m_new;
  }
  if (!head_ok) return;
  const int64_t pidx = (static_cast<int64_t>(b) * a.n_splits + split) * a.n_heads + h;
#pragma unroll
  for (int r = 0; r < kSimtMaxDc / 32; ++r) {
    const int k = lane + 32 * r;
    if (k < a.d_c) a.part_o[pidx * a.d_c + k] = o[r];
  }
  if (lane == 0) {
    a.part_m[pidx] = m;
    a.part_l[pidx] = l;
  }
}

template <typename Tin>
__global__ void __launch_bounds__(256) combine_simt_kernel(SimtArgs a) {
  extern __shared__ float olat[];  // [d_c]
  const int i = blockIdx.x, b = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t base = static_cast<int64_t>(b) * a.n_splits * a.n_heads + i;
  float M = -INFINITY;
  for (int s = 0; s < a.n_splits; ++s) M = fmaxf(M, a.part_m[base + static_cast<int64_t>(s) * a.n_heads]);
  float denom = 0.f;
  for (int s = 0; s < a.n_splits; ++s) {
    const int64_t p = base + static_cast<int64_t>(s) * a.n_heads;
    if (a.part_l[p] > 0.f) denom += exp2f(a.part_m[p] - M) * a.part_l[p];
  }
  const float inv = denom > 0.f ? 1.0f / denom : 0.f;
  for (int k = threadIdx.x; k < a.d_c; k += blockDim.x) {
    float acc = 0.f;
    for (int s = 0; s < a.n_splits; ++s) {
      const int64_t p = base + static_cast<int64_t>(s) * a.n_heads;
      if (a.part_l[p] > 0.f) acc = fmaf(exp2f(a.part_m[p] - M), a.part_o[p * a.d_c + k], acc);
    }
    olat[k] = acc * inv;
  }
  __syncthreads();
  const Tin* w = static_cast<const Tin*>(a.w_uv) + static_cast<int64_t>(i) * a.d_head * a.d_c;
  for (int d = warp; d < a.d_head; d += blockDim.x / 32) {
    float acc = 0.f;
    for (int k = lane; k < a.d_c; k += 32) acc = fmaf(load_as_f32(w, static_cast<int64_t>(d) * a.d_c + k), olat[k], acc);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (lane == 0) a.out[(static_cast<int64_t>(b) * a.n_heads + i) * a.d_head + d] = acc;
  }
}

}  // namespace mla
