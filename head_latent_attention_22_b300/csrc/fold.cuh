// W_UV folded into the output projection W_O (DeepSeek-V2 report, section
// 2.1.2: W_UV can be absorbed into W_O; section 2.1.1: the per-head outputs
// are concatenated and multiplied by W_O). With
//   W_OUV[:, i d_c .. (i+1) d_c) = W_O[:, i d_h .. (i+1) d_h) W_UV,i,
// the attention output in hidden space is u = W_OUV [o_lat,1; ...; o_lat,H],
// one GEMM over the latent-space outputs the merge step produces, with no
// per-head output in between.
//
//   fold_wo_kernel:    the fold itself, once per set of weights (plain fp32
//                      CUDA-core tiles; not on the decode path), stored as
//                      fp16: the folded products are small (|W_OUV| is about
//                      |W_O| |W_UV| sqrt(d_h)) and fp16 keeps 3 more bits than
//                      bf16 there; o_lat enters as an fp16 hi/lo pair to match.
//   out_tc_kernel:     u partials: CTA (m, g) computes rows 128 m .. of W_OUV
//                      times the o_lat hi/lo pair of every sequence over the
//                      g-th slice of the 65,536-wide contraction, on tcgen05
//                      (M = 128 hidden rows, N = batch, K = 16); the weight
//                      stream is what bounds it.
//   out_reduce_kernel: u = the sum of the slices' partials.
#pragma once

#include "common.cuh"
#include "decode_tc.cuh"
#include "tc.cuh"

namespace mla {
namespace tcd {

// ------------------------------------------------------------------ fold_wo_kernel
constexpr int kFoldTile = 64;   // output tile: 64 hidden rows x 64 latent columns of one head

// grid (hidden / 64, d_c / 64, H), 256 threads: each thread 4 x 4 outputs, the d_h = 128 contraction in two
// halves staged in shared memory.
__global__ void __launch_bounds__(256) fold_wo_kernel(const uint16_t* __restrict__ w_uv, const uint16_t* __restrict__ w_o,
                                                      uint16_t* __restrict__ w_ouv, int hidden) {
  constexpr int kK = 64;
  __shared__ float sa[kK][kFoldTile + 1];   // W_O[n0 + r, i d_h + k0 + k] as [k][r]
  __shared__ float sb[kK][kFoldTile];       // W_UV[i, k0 + k, c0 + c]
  const int n0 = blockIdx.x * kFoldTile, c0 = blockIdx.y * kFoldTile, i = blockIdx.z;
  const int t = threadIdx.x;
  const int tr = (t / 16) * 4, tcol = (t % 16) * 4;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < kDh; k0 += kK) {
    for (int e = t; e < kFoldTile * kK; e += 256) {
      const int r = e / kK, k = e % kK;
      sa[k][r] = bf16_to_f32(w_o[static_cast<int64_t>(n0 + r) * (kH * kDh) + i * kDh + k0 + k]);
      const int kb = e / kFoldTile, c = e % kFoldTile;
      sb[kb][c] = bf16_to_f32(w_uv[(static_cast<int64_t>(i) * kDh + k0 + kb) * kDc + c0 + c]);
    }
    __syncthreads();
    for (int k = 0; k < kK; ++k) {
      float av[4], bv[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        av[u] = sa[k][tr + u];
        bv[u] = sb[k][tcol + u];
      }
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int v = 0; v < 4; ++v) acc[u][v] = fmaf(av[u], bv[v], acc[u][v]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    uint16_t* dst = w_ouv + static_cast<int64_t>(n0 + tr + u) * (kH * kDc) + i * kDc + c0 + tcol;
    const uint32_t w0 = static_cast<uint32_t>(__half_as_ushort(__float2half_rn(acc[u][0]))) |
                        (static_cast<uint32_t>(__half_as_ushort(__float2half_rn(acc[u][1]))) << 16);
    const uint32_t w1 = static_cast<uint32_t>(__half_as_ushort(__float2half_rn(acc[u][2]))) |
                        (static_cast<uint32_t>(__half_as_ushort(__float2half_rn(acc[u][3]))) << 16);
    *reinterpret_cast<uint2*>(dst) = make_uint2(w0, w1);
  }
}

// ------------------------------------------------------------------ out_tc_kernel
constexpr int kOutMaxNb = 128;    // sequences per call on this path
constexpr int kOutStages = 4;
constexpr int kOutThreads = 128;

struct OutArgs {
  float* partial;   // [n_groups][batch][hidden]
  int batch, nb, hidden, n_groups;
};

__host__ __device__ constexpr size_t out_stage_bytes(int nb) { return 16384 + 2 * static_cast<size_t>(nb) * 128; }
__host__ __device__ constexpr size_t out_smem_bytes(int nb) {
  return 1024 + kOutStages * out_stage_bytes(nb) + 8 * (2 * kOutStages + 2) + 16;
}

// map_w: W_OUV [hidden, 128 * 512] fp16, boxes of 128 rows x 64 columns; map_hi / map_lo: o_lat as
// fp16 hi / lo [B, 128 * 512], boxes of nb rows x 64 columns (all 128-byte swizzle).
__global__ void __launch_bounds__(kOutThreads) out_tc_kernel(const __grid_constant__ CUtensorMap map_w,
                                                            const __grid_constant__ CUtensorMap map_hi,
                                                            const __grid_constant__ CUtensorMap map_lo, OutArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u);
  const size_t stb = out_stage_bytes(a.nb);
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + kOutStages * stb);
  uint64_t* empty = full + kOutStages;
  uint64_t* done = empty + kOutStages;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(done + 2);
  const int mt = blockIdx.x, g = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int kChunks = kH * kDc / 64;   // 1024 contraction chunks of 64
  const int c0 = static_cast<int>(static_cast<int64_t>(g) * kChunks / a.n_groups);
  const int c1 = static_cast<int>(static_cast<int64_t>(g + 1) * kChunks / a.n_groups);
  const uint32_t hb = static_cast<uint32_t>(a.nb) * 128;   // bytes of one hi (or lo) box
  if (threadIdx.x == 0) {
    for (int s = 0; s < kOutStages; ++s) {
      tc::mbar_init(&full[s], 1);
      tc::mbar_init(&empty[s], 1);
    }
    tc::mbar_init(&done[0], 1);
    tc::fence_mbar_init();
    tc::tma_prefetch_map(&map_w);
    tc::tma_prefetch_map(&map_hi);
    tc::tma_prefetch_map(&map_lo);
    // the weights do not depend on the kernels before this one: the first stages' weight boxes go now
    for (int c = c0; c < c1 && c - c0 < kOutStages; ++c) {
      uint8_t* st = sm + ((c - c0) % kOutStages) * stb;
      tc::mbar_arrive_expect_tx(&full[(c - c0) % kOutStages], 16384 + 2 * hb);
      tc::tma_load_2d(st, &map_w, 64 * c, 128 * mt, &full[(c - c0) % kOutStages]);
    }
  }
  if (warp == 1) tc::tmem_alloc<128>(tslot);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tm = *tslot;
  asm volatile("griddepcontrol.wait;" ::: "memory");   // o_lat comes from the merge kernel
  bool ok = true;
  if (warp == 0) {
    if (lane == 0) {
      for (int c = c0; c < c1 && ok; ++c) {
        const int i = c - c0, s = i % kOutStages;
        uint8_t* st = sm + s * stb;
        if (i >= kOutStages) {
          ok = tc::mbar_wait(&empty[s], ((i / kOutStages) - 1) & 1);
          if (!ok) break;
          tc::mbar_arrive_expect_tx(&full[s], 16384 + 2 * hb);
          tc::tma_load_2d(st, &map_w, 64 * c, 128 * mt, &full[s]);
        }
        tc::tma_load_2d(st + 16384, &map_hi, 64 * c, 0, &full[s]);
        tc::tma_load_2d(st + 16384 + hb, &map_lo, 64 * c, 0, &full[s]);
      }
      // copies in flight land before the CTA exits
      const int n = c1 - c0;
      for (int i = n > kOutStages ? n - kOutStages : 0; i < n; ++i) tc::mbar_wait(&full[i % kOutStages], (i / kOutStages) & 1);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // fp16 A and B (format fields 0), fp32 D, M = 128, N = nb, both K-major
      const uint32_t idesc = (1u << 4) | ((static_cast<uint32_t>(a.nb) >> 3) << 17) | ((128u >> 4) << 24);
      const uint64_t d0 = tc::sdesc_sw128(tc::smem_u32(sm), 16, 1024);
      for (int c = c0; c < c1 && ok; ++c) {
        const int i = c - c0, s = i % kOutStages;
        ok = tc::mbar_wait(&full[s], (i / kOutStages) & 1);
        if (!ok) break;
        tc::tc_fence_after();
        const uint64_t ab = d0 + static_cast<uint64_t>((s * stb) >> 4);
        const uint64_t hbd = d0 + static_cast<uint64_t>((s * stb + 16384) >> 4);
        const uint64_t lbd = d0 + static_cast<uint64_t>((s * stb + 16384 + hb) >> 4);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          tc::mma_ss(tm, ab + 2 * k, hbd + 2 * k, idesc, (i == 0 && k == 0) ? 0u : 1u);
          tc::mma_ss(tm, ab + 2 * k, lbd + 2 * k, idesc, 1u);
        }
        tc::mma_commit(&empty[s]);
      }
      tc::mma_commit(&done[0]);
    }
  }
  __syncwarp();
  // every thread: row 32 warp + lane of this CTA's 128 hidden rows, one column per sequence
  ok = tc::mbar_wait(&done[0], 0) && ok;
  tc::tc_fence_after();
  const int n = 128 * mt + 32 * warp + lane;
  for (int b0 = 0; b0 < a.nb; b0 += 16) {
    uint32_t r[16];
    tc::tmem_ld16(tc::tmem_at(tm, 32 * warp, b0), r);
    tc::tmem_ld_wait();
#pragma unroll
    for (int c = 0; c < 16; ++c)
      if (b0 + c < a.batch)
        a.partial[(static_cast<int64_t>(g) * a.batch + b0 + c) * a.hidden + n] = __uint_as_float(r[c]);
  }
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  if (warp == 1) tc::tmem_dealloc<128>(tm);
}

// out[b, n] = sum over the contraction slices g of partial[g, b, n]
__global__ void __launch_bounds__(256) out_reduce_kernel(const float* __restrict__ partial, float* __restrict__ out,
                                                         int n_groups, int64_t count) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  for (int64_t e = blockIdx.x * 256 + threadIdx.x; e < count; e += static_cast<int64_t>(gridDim.x) * 256) {
    float s = 0.f;
    for (int g = 0; g < n_groups; ++g) s += partial[g * count + e];
    out[e] = s;
  }
}

}  // namespace tcd
}  // namespace mla
