// Tensor-core (tcgen05 + TMEM + TMA) MLA decode for the DeepSeek-V2 shape:
// 128 heads of d_h = 128, latent d_c = 512, decoupled rope d_r = 64, bf16
// queries and weights; cache rows of 576 bf16 values, or 512 E4M3 codes with
// an fp32 scale per 128 values plus 64 bf16 rope values (DeepSeek-V2 report,
// section 2.1.2 absorbed form, section 2.1.3 decoupled RoPE, section 3.2.3
// quantised KV cache).
//
// Four kernels per decode:
//   absorb  : Q_lat[b,i,0:512] = W_UK[i]^T q_nope[b,i] (two CTAs per head, each
//             with its 64 KB half of the weight slice in flight at once, M = 2 x
//             128 latent rows, N = batch), q_rope copied to Q_lat[b,i,512:576];
//             one extra CTA clamps the lengths and writes the plan the other
//             kernels share (tile prefix sums, cluster shares).
//   attend  : persistent clusters of two CTAs; cluster c takes an equal share
//             of all 64-token tiles of all sequences, cut at sequence ends
//             into segments. In a pair, CTA0 owns latent columns 0..255 plus
//             the 64 rope columns and CTA1 owns latent columns 256..511: each
//             keeps its Q slice in TMEM, computes a partial score tile, swaps
//             it with its peer through distributed shared memory, runs the
//             (identical) online softmax, and accumulates its half of O_lat
//             in TMEM. Each segment ends in an unnormalised partial
//             (O half, running max m, sum l). With an FP8 cache the softmax
//             warps also dequantise the next tile into the bf16 stage.
//   merge   : one CTA per (sequence, 4 latent columns), thread = head:
//             log-sum-exp merge of the sequence's partials, o_lat written as
//             bf16 hi + lo.
//   uv      : one CTA per head: out[b,i,:] = W_UV[i] (o_hi + o_lo) on the
//             tensor cores (M = 128 output rows, N = sequences).
#pragma once

#include "common.cuh"
#include "tc.cuh"

namespace mla {
namespace tcd {

constexpr int kH = 128, kDc = 512, kDr = 64, kDh = 128, kRow = 576;
constexpr int kTile = 64;                    // tokens per attend tile
constexpr int kBlk = kTile * 128;            // one TMA box: 64 rows x 64 bf16 (128 B) = 8 KB
constexpr int kStageBytes = 4 * kBlk;        // latent boxes of one tile for one CTA: 256 columns
constexpr int kStages = 4;                   // latent ring depth (bf16 cache)
constexpr int kStagesF8 = 3;                 // latent ring depth (FP8 cache: bf16 tiles dequantised in place)
constexpr int kRopeStages = 3;               // rope ring depth (CTA0 only)
constexpr int kRawStages = 3;                // FP8 cache: ring of raw rows (codes + block scales)
constexpr int kRawCodeBytes = kTile * 256;   // this CTA's 256 E4M3 codes of 64 rows
constexpr int kRawBytes = kRawCodeBytes + kTile * 16;   // + the 4 fp32 block scales of each row
constexpr int kParts = 4;                    // softmax warps per TMEM lane quarter
constexpr int kCols = kTile / kParts;        // score columns per softmax thread
constexpr int kXvalBytes = kH * kTile * 2;   // one partial score tile as fp16
constexpr int kXbufBytes = kXvalBytes + kParts * kH * 4;   // + one power-of-two scale per (row, column part)
constexpr int kSoftmaxThreads = 128 * kParts;   // 4 TMEM lane quarters x kParts column parts
constexpr int kAttendThreads = 128 + kSoftmaxThreads;  // warp 0 TMA, warps 1-2 MMA, warps 4-19 softmax
constexpr float kRescaleThreshold = 8.0f;    // log2 units: O is rescaled only when the max grows by > 2^8

// Shared-memory carve-up of the attend kernel (after 1 KB alignment), per cache format.
template <bool kF8>
struct AttendLayout {
  static constexpr int kSt = kF8 ? kStagesF8 : kStages;
  static constexpr int kRaw = kF8 ? kRawStages : 0;
  static constexpr size_t kRopes = static_cast<size_t>(kSt) * kStageBytes;
  static constexpr size_t kRawOff = kRopes + static_cast<size_t>(kRopeStages) * kBlk;
  static constexpr size_t kXbuf = kRawOff + static_cast<size_t>(kRaw) * kRawBytes;
};

// TMEM columns of the attend kernel (512 allocated)
constexpr uint32_t kTmO = 0;     // O half: 128 lanes x 256 fp32
constexpr uint32_t kTmS = 256;   // partial / full score tile: 64 fp32
constexpr uint32_t kTmQ = 320;   // Q slice, bf16 pairs: up to 160 columns
constexpr uint32_t kTmP = 480;   // probabilities, bf16 pairs: 32 columns

// Layouts in the workspace. Both are chunk-major so that a warp holding 32
// consecutive heads touches one contiguous 512-byte line:
//   Q_lat  [B][72 chunks][128 heads][8 bf16]   chunk c = latent 8c..8c+7 (c < 64), rope 8(c-64).. (c >= 64)
//   part_o [slot][128 chunks][128 heads][4 fp32]  chunk c = latent 4c..4c+3
constexpr int kQChunks = kRow / 8;    // 72
constexpr int kOChunks = kDc / 4;     // 128

__host__ __device__ __forceinline__ int64_t qlat_index(int64_t b, int chunk, int head) {
  return ((b * kQChunks + chunk) * kH + head) * 8;
}
__host__ __device__ __forceinline__ int64_t parto_index(int64_t slot, int chunk, int head) {
  return ((slot * kOChunks + chunk) * kH + head) * 4;
}

struct Plan {
  int32_t* lens;         // [B] lengths clamped to [0, max_seq_len]
  int32_t* cum;          // [B+1] prefix sums of ceil(len / 64)
  int32_t* first_seq;    // [clusters] sequence holding the first tile of each cluster's share
  int32_t* share_start;  // [clusters + 1] first tile of each cluster's share (share c = [start[c], start[c+1]))
  int32_t* seq_c0;       // [B] first cluster whose share meets sequence b's tiles (when it has any)
  int32_t* seq_c1;       // [B] last such cluster
};

// Tile range [t0, t1) of cluster c when T tiles are split over nc clusters.
__host__ __device__ __forceinline__ int64_t share_begin(int64_t c, int64_t T, int64_t nc) { return c * T / nc; }

// The cluster whose share holds tile t (T > 0).
__host__ __device__ __forceinline__ int64_t share_owner(int64_t t, int64_t T, int64_t nc) {
  return ((t + 1) * nc - 1) / T;
}

// ================================================================== absorb (+ plan)
struct AbsorbArgs {
  const uint16_t* q_rope;     // [B, H, 64]
  const int32_t* seq_lens;    // [B]
  uint16_t* q_lat;            // chunk-major (see qlat_index), or row-major [B, H, 576] when row_major
  Plan plan;
  int batch, nb, max_seq_len, ncl;
  int row_major;
};

__host__ __device__ __forceinline__ int64_t qlat_row_index(int64_t b, int head, int k) {
  return (b * kH + head) * kRow + k;
}

constexpr int kAbsorbThreads = 128;

__device__ void plan_block(const AbsorbArgs& a) {
  __shared__ int32_t carry;
  __shared__ int32_t warp_tot[kAbsorbThreads / 32];
  if (threadIdx.x == 0) {
    carry = 0;
    a.plan.cum[0] = 0;
  }
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int base = 0; base < a.batch; base += kAbsorbThreads) {
    const int b = base + threadIdx.x;
    int n = 0;
    if (b < a.batch) {
      int L = a.seq_lens[b];
      if (L < 0 || L > a.max_seq_len) {
        flag_error(ERR_BIT_BOUNDS);
        L = L < 0 ? 0 : a.max_seq_len;
      }
      a.plan.lens[b] = L;
      n = (L + kTile - 1) / kTile;
    }
    int x = n;  // inclusive warp scan
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) warp_tot[warp] = x;
    __syncthreads();
    int off = carry;
    for (int w = 0; w < warp; ++w) off += warp_tot[w];
    if (b < a.batch) a.plan.cum[b + 1] = off + x;
    __syncthreads();
    if (threadIdx.x == kAbsorbThreads - 1) carry = off + x;
    __syncthreads();
  }
  // cluster shares: start tile and first sequence of each; clusters of each sequence
  const int64_t T = a.plan.cum[a.batch];
  for (int c = threadIdx.x; c <= a.ncl; c += kAbsorbThreads) {
    const int64_t t = share_begin(c, T, a.ncl);
    a.plan.share_start[c] = static_cast<int32_t>(t);
    if (c == a.ncl) continue;
    int lo = 0, hi = a.batch;   // cum[lo] <= t
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (a.plan.cum[mid] <= t) lo = mid; else hi = mid;
    }
    a.plan.first_seq[c] = lo;
  }
  for (int b = threadIdx.x; b < a.batch; b += kAbsorbThreads) {
    const int64_t tb0 = a.plan.cum[b], tb1 = a.plan.cum[b + 1];
    if (tb1 > tb0) {
      a.plan.seq_c0[b] = static_cast<int32_t>(share_owner(tb0, T, a.ncl));
      a.plan.seq_c1[b] = static_cast<int32_t>(share_owner(tb1 - 1, T, a.ncl));
    } else {
      a.plan.seq_c0[b] = 0;
      a.plan.seq_c1[b] = -1;
    }
  }
}

// Two CTAs per head i (blockIdx.x = 2 i + half, half = 128-row M tiles
// 2 half and 2 half + 1 of the 512 latent rows); the last CTA writes the plan.
// Each CTA streams its 64 KB of W_UK[i] with one barrier per M tile, so the
// MMAs of the first tile start while the second is still in flight; the
// weights are requested before the wait on the preceding kernel.
__global__ void __launch_bounds__(kAbsorbThreads) absorb_tc_kernel(const __grid_constant__ CUtensorMap map_wuk,
                                                                   const __grid_constant__ CUtensorMap map_qn,
                                                                   AbsorbArgs a) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (blockIdx.x == 2 * kH) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    plan_block(a);
    return;
  }
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* sA = sm;                          // 4 boxes [128 d_h rows x 64 latent] = 64 KB
  uint8_t* sB = sm + 4 * 16384;              // 2 boxes [nb rows x 64 d_h]
  uint64_t* bars = reinterpret_cast<uint64_t*>(sB + 2 * a.nb * 128);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 5);
  const int i = blockIdx.x >> 1, half = blockIdx.x & 1;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    tc::mbar_init(&bars[0], 1);  // weights of M tile 0 landed
    tc::mbar_init(&bars[1], 1);  // weights of M tile 1 landed
    tc::mbar_init(&bars[2], 1);  // queries landed (one phase per N chunk)
    tc::mbar_init(&bars[3], 1);  // MMAs done (one phase per N chunk)
    tc::fence_mbar_init();
    tc::tma_prefetch_map(&map_wuk);
    tc::tma_prefetch_map(&map_qn);
    for (int mt = 0; mt < 2; ++mt) {
      tc::mbar_arrive_expect_tx(&bars[mt], 2 * 16384);
      for (int j = 0; j < 2; ++j)
        tc::tma_load_2d(sA + (2 * mt + j) * 16384, &map_wuk, 256 * half + 128 * mt + 64 * j, i * kDh, &bars[mt]);
    }
  }
  if (warp == 0) tc::tmem_alloc<256>(tslot);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tm = *tslot;
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // q_rope -> Q_lat chunks 64..71 of head i (one of the two CTAs)
  if (half == 0) {
    for (int idx = threadIdx.x; idx < a.batch * 8; idx += kAbsorbThreads) {
      const int b = idx >> 3, c = idx & 7;
      const uint4 v = reinterpret_cast<const uint4*>(a.q_rope + (static_cast<int64_t>(b) * kH + i) * kDr)[c];
      *reinterpret_cast<uint4*>(a.q_lat + (a.row_major ? qlat_row_index(b, i, kDc + 8 * c)
                                                       : qlat_index(b, kDc / 8 + c, i))) = v;
    }
  }
  const uint32_t idesc = tc::idesc_bf16_f32(128, a.nb, 1, 0);
  bool ok = true;
  int chunk = 0;
  for (int n0 = 0; n0 < a.batch; n0 += a.nb, ++chunk) {
    if (threadIdx.x == 0) {
      tc::mbar_arrive_expect_tx(&bars[2], 2 * a.nb * 128);
      tc::tma_load_2d(sB, &map_qn, i * kDh, n0, &bars[2]);
      tc::tma_load_2d(sB + a.nb * 128, &map_qn, i * kDh + 64, n0, &bars[2]);
      ok = tc::mbar_wait(&bars[2], chunk & 1);
      for (int mt = 0; mt < 2 && ok; ++mt) {
        ok = tc::mbar_wait(&bars[mt], 0);
        tc::tc_fence_after();
        if (ok) {
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint64_t ad = tc::sdesc_sw128(tc::smem_u32(sA + (2 * mt) * 16384 + 2048 * kk), 16384, 1024);
            const uint64_t bd = tc::sdesc_sw128(tc::smem_u32(sB + (kk >> 2) * a.nb * 128 + (kk & 3) * 32), 16, 1024);
            tc::mma_ss(tm + mt * a.nb, ad, bd, idesc, kk > 0 ? 1u : 0u);
          }
        }
      }
      tc::mma_commit(&bars[3]);
    }
    __syncwarp();
    ok = tc::mbar_wait(&bars[3], chunk & 1);
    tc::tc_fence_after();
    // epilogue: lane = latent row within the M tile, columns = sequences
    for (int mt = 0; mt < 2; ++mt) {
      for (int c0 = 0; c0 < a.nb; c0 += 16) {
        uint32_t r[16];
        tc::tmem_ld16(tc::tmem_at(tm, 32 * warp, mt * a.nb + c0), r);
        tc::tmem_ld_wait();
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          const int b = n0 + c0 + c;
          const int k = 256 * half + mt * 128 + 32 * warp + lane;   // latent element
          if (b < a.batch && ok)
            a.q_lat[a.row_major ? qlat_row_index(b, i, k) : qlat_index(b, k >> 3, i) + (k & 7)] =
                f32_to_bf16_bits(__uint_as_float(r[c]));
        }
      }
    }
    tc::tc_fence_before();
    __syncthreads();  // TMEM and the query box are reused by the next chunk
  }
  if (warp == 0) tc::tmem_dealloc<256>(tm);
}

// ================================================================== attend
struct AttendArgs {
  const uint16_t* q_lat;      // chunk-major, see qlat_index
  const int32_t* block_table; // [B, max_pages] (NULL: contiguous, sequence b owns pages b*max_pages ..)
  Plan plan;
  float* part_o;              // chunk-major (see parto_index) fp32, unnormalised
  float* part_ml;             // [slots, H, 2]: running max (log2 units) and sum
  int64_t num_pages;
  int batch, max_pages, page_size;
  int rope_x;                 // column of the rope box in the rope tensor map
  float scale_log2;           // softmax scale * log2(e), > 0
};

struct AttendSmem {
  uint64_t full[kStages], empty[kStages];       // latent ring (bf16 tiles, however they were filled)
  uint64_t raw_full[kRawStages], raw_empty[kRawStages];   // FP8 cache: raw rows
  uint64_t rfull[kRopeStages], rempty[kRopeStages];  // rope ring (CTA0)
  uint64_t s_full, s_free, p_full, o_done, q_ready, o_free, drain, drain2;
  uint64_t xfull[2];          // peer partial scores landed in xbuf[0/1] (byte-counted)
  uint64_t pair_max[4][2];    // the softmax warps of a lane quarter swapped row maxima (by tile parity)
  uint64_t pair_sum[4];       // ... and row sums at a segment end
  float red[2][kParts][kH];   // per-part row maxima, by tile parity
  float redl[kParts][kH];     // per-part row sums at a segment end
  uint32_t tmem_base;
  int32_t abort_flag;
};

// Segment iterator: the (sequence, tile range) pieces of this cluster's share.
struct SegIter {
  int64_t t, t1;  // next tile (global index) and end of share
  int b;          // current sequence
  __device__ __forceinline__ bool next(const int32_t* cum, int batch, int* seq, int* j0, int* j1) {
    if (t >= t1) return false;
    while (b < batch && cum[b + 1] <= t) ++b;
    if (b >= batch) return false;
    const int64_t end = min(t1, static_cast<int64_t>(cum[b + 1]));
    *seq = b;
    *j0 = static_cast<int>(t - cum[b]);
    *j1 = static_cast<int>(end - cum[b]);
    t = end;
    return true;
  }
};

__device__ __forceinline__ SegIter seg_begin(const Plan& plan, int batch, uint32_t c, uint32_t nc) {
  (void)batch;
  (void)nc;
  SegIter it;
  it.t = plan.share_start[c];
  it.t1 = plan.share_start[c + 1];
  it.b = plan.first_seq[c];
  return it;
}

__device__ __forceinline__ bool aborted(const AttendSmem* s) {
  return *reinterpret_cast<const volatile int32_t*>(&s->abort_flag) != 0;
}

__device__ __forceinline__ void set_abort(AttendSmem* s) {
  *reinterpret_cast<volatile int32_t*>(&s->abort_flag) = 1;
}

// Score MMAs over NK steps of 16 along the contraction, B = NK/4 boxes of 8 KB
// from b0; unrolled so that no branch separates two MMAs. `first` = 1 starts
// the accumulation.
template <int NK>
__device__ __forceinline__ void issue_scores(uint32_t d, uint32_t a, uint64_t b0, uint32_t idesc, uint32_t first) {
#pragma unroll
  for (int k = 0; k < NK; ++k)
    tc::mma_ts(d, a + 8 * k, b0 + static_cast<uint64_t>(((k >> 2) * kBlk + (k & 3) * 32) >> 4), idesc,
               (k == 0 && first) ? 0u : 1u);
}

// O half [128 heads x 256] (+)= P (TMEM, 64 tokens) x V (the tile's 4 latent boxes, MN-major).
__device__ __forceinline__ void issue_pv(uint32_t d, uint32_t a, uint64_t b0, uint32_t idesc, uint32_t acc0) {
  tc::mma_ts(d, a, b0, idesc, acc0);
#pragma unroll
  for (int k = 1; k < 4; ++k) tc::mma_ts(d, a + 8 * k, b0 + static_cast<uint64_t>((k * 2048) >> 4), idesc, 1u);
}

// This part's share of the Q slice of sequence b (row h) into TMEM columns
// kTmQ.. as bf16 pairs. CTA0's slice is latent 0..255 then rope 512..575
// (40 chunks of 16 bytes), CTA1's latent 256..511 (32 chunks); part p takes
// chunks p * NCH/kParts .. (p+1) * NCH/kParts - 1.
template <int NCH>
__device__ __forceinline__ void load_q_part(const uint16_t* q_lat, int b, int h, uint32_t rank, int part,
                                            uint32_t taddr) {
  constexpr int kPer = NCH / kParts;
  uint4 v[kPer];
#pragma unroll
  for (int u = 0; u < kPer; ++u) {
    const int c = part * kPer + u;   // chunk of this CTA's slice
    const int qc = rank == 0 ? (c < 32 ? c : kDc / 8 + (c - 32)) : 32 + c;
    v[u] = *reinterpret_cast<const uint4*>(q_lat + qlat_index(b, qc, h));
  }
  const uint32_t t0 = taddr + 4 * part * kPer;
#pragma unroll
  for (int u = 0; u + 4 <= kPer; u += 4) {
    uint32_t w[16];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      w[4 * e] = v[u + e].x; w[4 * e + 1] = v[u + e].y; w[4 * e + 2] = v[u + e].z; w[4 * e + 3] = v[u + e].w;
    }
    tc::tmem_st16(t0 + 4 * u, w);
  }
  if constexpr (kPer % 4 == 2) {
    uint32_t w[8];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      w[4 * e] = v[kPer - 2 + e].x; w[4 * e + 1] = v[kPer - 2 + e].y;
      w[4 * e + 2] = v[kPer - 2 + e].z; w[4 * e + 3] = v[kPer - 2 + e].w;
    }
    tc::tmem_st8(t0 + 4 * (kPer - 2), w);
  }
  tc::tmem_st_wait();
}

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ float f16_lo(uint32_t w) { return __half2float(__ushort_as_half(static_cast<unsigned short>(w & 0xffffu))); }
__device__ __forceinline__ float f16_hi(uint32_t w) { return __half2float(__ushort_as_half(static_cast<unsigned short>(w >> 16))); }

// (f32)a.lo + (f32)b.lo and (f32)a.hi + (f32)b.hi for two fp16 pairs, on the
// fp32 pipe (mixed-precision adds convert their fp16 operand exactly); equal
// to converting both and adding, and symmetric in a and b.
__device__ __forceinline__ float2 add_f16x2_f32(uint32_t a, uint32_t b) {
  float lo, hi;
  asm("{\n\t.reg .b16 al, ah, bl, bh;\n\t.reg .f32 t0, t1;\n\t"
      "mov.b32 {al, ah}, %2;\n\t"
      "mov.b32 {bl, bh}, %3;\n\t"
      "add.rn.f32.f16 t0, bl, 0f00000000;\n\t"
      "add.rn.f32.f16 %0, al, t0;\n\t"
      "add.rn.f32.f16 t1, bh, 0f00000000;\n\t"
      "add.rn.f32.f16 %1, ah, t1;\n\t}"
      : "=f"(lo), "=f"(hi)
      : "r"(a), "r"(b));
  return make_float2(lo, hi);
}

// Partial scores travel between the two CTAs as fp16 scaled by 2^-k, with k
// chosen per (row, column half) so that the largest magnitude stays below
// 2^15: no overflow whatever the inputs, 11 significant bits. Both CTAs add
// the same rounded values, so their softmax decisions agree bit for bit.
__device__ __forceinline__ float exchange_scale(float amax, float* unscale) {
  const int e = static_cast<int>((__float_as_uint(amax) >> 23) & 0xffu) - 127;
  const int k = e > 14 ? e - 14 : 0;
  *unscale = __uint_as_float(static_cast<uint32_t>(127 + k) << 23);
  return __uint_as_float(static_cast<uint32_t>(127 - k) << 23);
}

// kF8 = false: map_lat is the bf16 pool [rows, 576], boxes of 64 x 64 (128-byte swizzle);
//              map_scale is unused.
// kF8 = true:  map_lat and map_scale are byte views of the FP8 pool [rows, 656] with unswizzled
//              boxes of 64 rows x 256 codes (this CTA's half, column 256 * rank) and of
//              64 rows x 16 bytes (the four block scales, column 512); the softmax threads
//              dequantise them into the same bf16 tile layout the TMA gives a bf16 pool.
// map_rope: the 64 rope values of each row as bf16, box 64 x 64 at column a.rope_x.
template <bool kF8>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kAttendThreads, 1)
    attend_tc_kernel(const __grid_constant__ CUtensorMap map_lat, const __grid_constant__ CUtensorMap map_scale,
                     const __grid_constant__ CUtensorMap map_rope, AttendArgs a) {
  using LY = AttendLayout<kF8>;
  constexpr int kSt = LY::kSt;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* tiles = sm;                                           // kSt x 32 KB latent boxes (bf16)
  uint8_t* ropes = sm + LY::kRopes;                              // kRopeStages x 8 KB (CTA0)
  uint8_t* rawb = sm + LY::kRawOff;                              // FP8: kRawStages x raw rows
  uint8_t* xbuf = sm + LY::kXbuf;                                // 2 x [128 heads x 64] partial scores
  AttendSmem* S = reinterpret_cast<AttendSmem*>(xbuf + 2 * kXbufBytes);

  const uint32_t rank = tc::cluster_ctarank(), peer = rank ^ 1u;
  const uint32_t cl = tc::cluster_id_x(), ncl = tc::n_clusters_x();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kSt; ++s) {
      tc::mbar_init(&S->full[s], kF8 ? kSoftmaxThreads : 1);   // FP8: every dequantising thread arrives
      tc::mbar_init(&S->empty[s], 1);
    }
    for (int s = 0; s < kRawStages; ++s) {
      tc::mbar_init(&S->raw_full[s], 1);
      tc::mbar_init(&S->raw_empty[s], kSoftmaxThreads);
    }
    for (int s = 0; s < kRopeStages; ++s) {
      tc::mbar_init(&S->rfull[s], 1);
      tc::mbar_init(&S->rempty[s], 1);
    }
    tc::mbar_init(&S->s_full, 1);
    tc::mbar_init(&S->s_free, kSoftmaxThreads);
    tc::mbar_init(&S->p_full, kSoftmaxThreads);
    tc::mbar_init(&S->o_done, 1);
    tc::mbar_init(&S->q_ready, kSoftmaxThreads);
    tc::mbar_init(&S->o_free, kSoftmaxThreads);
    tc::mbar_init(&S->drain, 1);
    tc::mbar_init(&S->drain2, 1);
    tc::mbar_init(&S->xfull[0], 1);
    tc::mbar_init(&S->xfull[1], 1);
    for (int q = 0; q < 4; ++q) {
      tc::mbar_init(&S->pair_max[q][0], 32 * kParts);
      tc::mbar_init(&S->pair_max[q][1], 32 * kParts);
      tc::mbar_init(&S->pair_sum[q], 32 * kParts);
    }
    S->abort_flag = 0;
    tc::fence_mbar_init();
    // both exchange buffers expect one partial score tile from the peer
    tc::mbar_arrive_expect_tx(&S->xfull[0], kXbufBytes);
    tc::mbar_arrive_expect_tx(&S->xfull[1], kXbufBytes);
    tc::tma_prefetch_map(&map_lat);
    if (kF8) tc::tma_prefetch_map(&map_scale);
    tc::tma_prefetch_map(&map_rope);
  }
  if (warp == 1) tc::tmem_alloc<512>(&S->tmem_base);
  tc::tc_fence_before();
  tc::cluster_sync();
  tc::tc_fence_after();
  const uint32_t tm = S->tmem_base;
  // everything below reads what the absorb kernel wrote
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int32_t* cum = a.plan.cum;

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer (whole warp walks
    // the tiles; lane l looks up the page of the l-th tile of each group of 32, lane 0 issues)
    const uint64_t policy = tc::policy_evict_first();
    SegIter si = seg_begin(a.plan, a.batch, cl, ncl);
    int b, j0, j1;
    uint32_t it = 0;
    bool ok = true;
    while (ok && si.next(cum, a.batch, &b, &j0, &j1)) {
      for (int jc = j0; jc < j1 && ok; jc += 32) {
        int32_t y_l = 0;
        const int jl = jc + lane;
        if (jl < j1) {
          const int64_t tok = static_cast<int64_t>(jl) * kTile;
          const int pg = static_cast<int>(tok / a.page_size);
          int64_t page = -1;
          if (pg < a.max_pages)
            page = a.block_table ? a.block_table[static_cast<int64_t>(b) * a.max_pages + pg]
                                 : static_cast<int64_t>(b) * a.max_pages + pg;
          if (page < 0 || page >= a.num_pages) {
            flag_error(ERR_BIT_BOUNDS);
            y_l = -2 * kTile;  // entirely outside the pool: the copy fills zeros
          } else {
            y_l = static_cast<int32_t>(page * a.page_size + tok % a.page_size);
          }
        }
        const int n = min(32, j1 - jc);
        for (int u = 0; u < n; ++u) {
          const int32_t y = __shfl_sync(0xffffffffu, y_l, u);
          if (lane == 0 && ok) {
            const int st = it % kSt, rs = it % kRopeStages, ws = it % kRawStages;
            if (kF8) {
              if (it >= kRawStages) ok = tc::mbar_wait(&S->raw_empty[ws], ((it / kRawStages) - 1) & 1);
            } else {
              if (it >= kSt) ok = tc::mbar_wait(&S->empty[st], ((it / kSt) - 1) & 1);
            }
            if (ok && rank == 0 && it >= kRopeStages) ok = tc::mbar_wait(&S->rempty[rs], ((it / kRopeStages) - 1) & 1);
            if (ok && aborted(S)) ok = false;
            if (ok) {
              if (kF8) {
                uint8_t* dst = rawb + ws * kRawBytes;
                tc::mbar_arrive_expect_tx(&S->raw_full[ws], kRawBytes);
                tc::tma_load_2d_hint(dst, &map_lat, static_cast<int>(rank) * 256, y, &S->raw_full[ws], policy);
                tc::tma_load_2d_hint(dst + kRawCodeBytes, &map_scale, kDc, y, &S->raw_full[ws], policy);
              } else {
                uint8_t* dst = tiles + st * kStageBytes;
                tc::mbar_arrive_expect_tx(&S->full[st], kStageBytes);
                for (int k = 0; k < 4; ++k)
                  tc::tma_load_2d_hint(dst + k * kBlk, &map_lat, static_cast<int>(rank) * 256 + 64 * k, y,
                                       &S->full[st], policy);
              }
              if (rank == 0) {
                tc::mbar_arrive_expect_tx(&S->rfull[rs], kBlk);
                tc::tma_load_2d_hint(ropes + rs * kBlk, &map_rope, a.rope_x, y, &S->rfull[rs], policy);
              }
              ++it;
            }
          }
          ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
          if (!ok) break;
        }
      }
    }
    it = __shfl_sync(0xffffffffu, it, 0);
    if (lane == 0) {
      if (!ok) set_abort(S);
      // drain: copies still in flight must land before the CTA exits
      if (kF8) {
        const uint32_t first = it > kRawStages ? it - kRawStages : 0;
        for (uint32_t q = first; q < it; ++q) tc::mbar_wait(&S->raw_full[q % kRawStages], (q / kRawStages) & 1);
      } else {
        const uint32_t first = it > kSt ? it - kSt : 0;
        for (uint32_t q = first; q < it; ++q) tc::mbar_wait(&S->full[q % kSt], (q / kSt) & 1);
      }
      if (rank == 0) {
        const uint32_t rfirst = it > kRopeStages ? it - kRopeStages : 0;
        for (uint32_t q = rfirst; q < it; ++q) tc::mbar_wait(&S->rfull[q % kRopeStages], (q / kRopeStages) & 1);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- score MMA issuer
    // S(it) as soon as its tile has landed and the softmax has copied S(it-1)
    // out of TMEM; the PVs go out from warp 2, so neither stream waits for the other.
    if (lane == 0) {
      const uint32_t idesc_s = tc::idesc_bf16_f32(128, kTile, 0, 0);
      const uint64_t desc0 = tc::sdesc_sw128(tc::smem_u32(tiles), 16, 1024);      // K-major tile, stage 0
      const uint64_t rdesc0 = tc::sdesc_sw128(tc::smem_u32(ropes), 16, 1024);     // K-major rope box, stage 0
      SegIter si = seg_begin(a.plan, a.batch, cl, ncl);
      int b, j0, j1;
      uint32_t it = 0, seg = 0;
      bool ok = true;
      while (ok && si.next(cum, a.batch, &b, &j0, &j1)) {
        ok = tc::mbar_wait(&S->q_ready, seg & 1);
        for (int j = j0; j < j1 && ok; ++j, ++it) {
          const uint32_t st = it % kSt, rs = it % kRopeStages;
          ok = tc::mbar_wait(&S->full[st], (it / kSt) & 1);
          if (ok && rank == 0) ok = tc::mbar_wait(&S->rfull[rs], (it / kRopeStages) & 1);
          if (ok && it > 0) ok = tc::mbar_wait(&S->s_free, (it - 1) & 1);
          if (!ok || aborted(S)) { ok = false; break; }
          tc::tc_fence_after();
          issue_scores<16>(tm + kTmS, tm + kTmQ, desc0 + static_cast<uint64_t>((st * kStageBytes) >> 4), idesc_s, 1u);
          if (rank == 0) {
            issue_scores<4>(tm + kTmS, tm + kTmQ + 128, rdesc0 + static_cast<uint64_t>((rs * kBlk) >> 4), idesc_s, 0u);
            tc::mma_commit(&S->rempty[rs]);
          }
          tc::mma_commit(&S->s_full);
        }
        ++seg;
      }
      if (!ok) set_abort(S);
      // every MMA issued so far must complete before TMEM is released
      tc::mma_commit(&S->drain);
      tc::mbar_wait(&S->drain, 0);
    }
  } else if (warp == 2) {
    // ---------------------------------------------------------------- PV MMA issuer
    if (lane == 0) {
      const uint32_t idesc_o = tc::idesc_bf16_f32(128, 256, 0, 1);
      const uint64_t vdesc0 = tc::sdesc_sw128(tc::smem_u32(tiles), kBlk, 1024);   // MN-major V, stage 0
      SegIter si = seg_begin(a.plan, a.batch, cl, ncl);
      int b, j0, j1;
      uint32_t it = 0, seg = 0;
      bool ok = true;
      while (ok && si.next(cum, a.batch, &b, &j0, &j1)) {
        for (int j = j0; j < j1 && ok; ++j, ++it) {
          // P(it) in TMEM implies S(it), hence its tile, were complete
          ok = tc::mbar_wait(&S->p_full, it & 1);
          if (ok && j == j0 && seg > 0) ok = tc::mbar_wait(&S->o_free, (seg - 1) & 1);
          if (!ok || aborted(S)) { ok = false; break; }
          tc::tc_fence_after();
          const uint32_t st = it % kSt;
          issue_pv(tm + kTmO, tm + kTmP, vdesc0 + static_cast<uint64_t>((st * kStageBytes) >> 4), idesc_o,
                   j == j0 ? 0u : 1u);
          tc::mma_commit(&S->o_done);
          tc::mma_commit(&S->empty[st]);
        }
        ++seg;
      }
      if (!ok) set_abort(S);
      tc::mma_commit(&S->drain2);
      tc::mbar_wait(&S->drain2, 0);
    }
  } else if (warp >= 4) {
    // ---------------------------------------------------------------- softmax + epilogue
    // kParts warps per TMEM lane quarter: warp w holds head rows 32 (w % 4) .. +31
    // and token columns kCols * part .. + kCols - 1 of every tile.
    const int quarter = warp & 3, part = (warp - 4) >> 2;
    const int h = 32 * quarter + lane;           // head = TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>(32 * quarter) << 16;
    const uint32_t t_s = tm + lane_base + kTmS + kCols * part;
    const uint32_t t_o = tm + lane_base + kTmO + (256 / kParts) * part;
    const uint32_t t_p = tm + lane_base + kTmP + (kCols / 2) * part;
    auto load_q = [&](int bq) {
      if (rank == 0) load_q_part<40>(a.q_lat, bq, h, rank, part, tm + lane_base + kTmQ);
      else load_q_part<32>(a.q_lat, bq, h, rank, part, tm + lane_base + kTmQ);
      tc::tc_fence_before();
      tc::mbar_arrive(&S->q_ready);
    };
    // this thread's 32 bytes of row h in the exchange buffers (16-byte chunks 2 part, 2 part + 1, swizzled)
    auto xoff = [&](int u) { return h * 128 + (((2 * part + u) ^ (h & 7)) << 4); };
    const uint32_t peer_x = tc::map_peer(xbuf, peer);
    const uint32_t peer_bar0 = tc::map_peer(&S->xfull[0], peer);
    const uint32_t peer_bar1 = tc::map_peer(&S->xfull[1], peer);
    const float sl = a.scale_log2;

    SegIter si = seg_begin(a.plan, a.batch, cl, ncl);
    int b, j0, j1;
    uint32_t it = 0;
    bool ok = true;
    bool have = si.next(cum, a.batch, &b, &j0, &j1);
    if (have) load_q(b);
    // the tile waiting for its peer half: this thread's own partial scores (scaled fp16 pairs)
    uint32_t pend[kCols / 2];
    float pend_un = 1.f;
    bool have_pend = false;
    int pend_valid = 0;
    uint32_t pend_it = 0;
    float m_used = -INFINITY, l = 0.f;
    uint32_t n_epi = 0;   // segment epilogues done (phase of pair_sum)

    // Finishes tile `q` up to its P store: full scores, online softmax.
    auto finish = [&](uint32_t q, int valid) -> bool {
      const uint32_t xb = q & 1u;
      if (!tc::mbar_wait(&S->xfull[xb], (q >> 1) & 1)) return false;
      if (h == 0 && part == 0) tc::mbar_arrive_expect_tx(&S->xfull[xb], kXbufBytes);   // arm its next use
      float s[kCols];
      {
        const uint8_t* xr = xbuf + xb * kXbufBytes;
        const float pun = reinterpret_cast<const float*>(xr + kXvalBytes)[part * kH + h];
        uint4 v[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) v[u] = *reinterpret_cast<const uint4*>(xr + xoff(u));
        const uint32_t pw[8] = {v[0].x, v[0].y, v[0].z, v[0].w, v[1].x, v[1].y, v[1].z, v[1].w};
        if (pun == 1.f && pend_un == 1.f) {   // the usual case: no rescaling of either side
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const float2 v2 = add_f16x2_f32(pend[e], pw[e]);
            s[2 * e] = v2.x;
            s[2 * e + 1] = v2.y;
          }
        } else {
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            s[2 * e] = f16_lo(pend[e]) * pend_un + f16_lo(pw[e]) * pun;
            s[2 * e + 1] = f16_hi(pend[e]) * pend_un + f16_hi(pw[e]) * pun;
          }
        }
      }
      const int vh = valid - kCols * part;        // valid columns of this thread
      if (vh < kCols) {
#pragma unroll
        for (int c = 0; c < kCols; ++c) if (c >= vh) s[c] = -INFINITY;
      }
      float mx;
      {
        float t4[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) t4[c] = fmaxf(fmaxf(s[c], s[c + 4]), fmaxf(s[c + 8], s[c + 12]));
        mx = fmaxf(fmaxf(t4[0], t4[1]), fmaxf(t4[2], t4[3]));
      }
      // row maximum over the kParts warps holding this row
      S->red[q & 1][part][h] = mx;
      tc::mbar_arrive(&S->pair_max[quarter][q & 1]);
      if (!tc::mbar_wait(&S->pair_max[quarter][q & 1], (q >> 1) & 1)) return false;
#pragma unroll
      for (int pp = 0; pp < kParts; ++pp) mx = fmaxf(mx, S->red[q & 1][pp][h]);
      mx *= sl;
      bool rescale = false;
      float alpha = 1.f;
      if (m_used == -INFINITY) {
        m_used = mx;
      } else if (mx > m_used + kRescaleThreshold) {
        alpha = tc::ex2_approx(m_used - mx);
        l *= alpha;
        m_used = mx;
        rescale = true;
      }
      const float neg_m = -m_used;
      uint32_t p[kCols / 2];
      float ps[2] = {0.f, 0.f};
#pragma unroll
      for (int c = 0; c < kCols; c += 2) {
        const uint32_t w = tc::pack_bf16(tc::ex2_approx(fmaf(s[c], sl, neg_m)), tc::ex2_approx(fmaf(s[c + 1], sl, neg_m)));
        p[c / 2] = w;
        ps[(c / 2) & 1] += bf_lo(w) + bf_hi(w);
      }
      l += ps[0] + ps[1];
      // PV of the previous tile must be done: the P buffer and O are ours
      if (q > 0 && !tc::mbar_wait(&S->o_done, (q - 1) & 1)) return false;
      tc::tc_fence_after();
      if (rescale) {
        for (int c0 = 0; c0 < 256 / kParts; c0 += 16) {
          uint32_t r[16];
          tc::tmem_ld16(t_o + c0, r);
          tc::tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < 16; ++c) r[c] = __float_as_uint(__uint_as_float(r[c]) * alpha);
          tc::tmem_st16(t_o + c0, r);
        }
      }
      tc::tmem_st8(t_p, p);   // completed by finish_commit, after this tile's send
      return true;
    };

    // FP8 cache: tile q's raw rows -> bf16 tile in the latent stage (128-byte swizzled
    // boxes of 64 latent columns), value = E4M3 code * block scale rounded to bf16.
    // 2,048 output chunks of 8 values per tile, four per softmax thread.
    auto dequant = [&](uint32_t q) -> bool {
      const uint32_t ws = q % kRawStages, st = q % kSt;
      if (!tc::mbar_wait(&S->raw_full[ws], (q / kRawStages) & 1)) return false;
      if (q >= static_cast<uint32_t>(kSt) && !tc::mbar_wait(&S->empty[st], ((q / kSt) - 1) & 1)) return false;
      const uint8_t* raw = rawb + ws * kRawBytes;
      uint8_t* stage = tiles + st * kStageBytes;
#pragma unroll
      for (int u = 0; u < (kTile * 32) / kSoftmaxThreads; ++u) {
        const int ci = static_cast<int>(threadIdx.x) - 128 + u * kSoftmaxThreads;
        const int row = ci >> 5, k = ci & 31;   // output chunk k = latent 8k..8k+7 of this CTA's 256
        const uint2 codes = *reinterpret_cast<const uint2*>(raw + row * 256 + 8 * k);
        const float sc = reinterpret_cast<const float*>(raw + kRawCodeBytes + row * 16)[2 * rank + (k >> 4)];
        const uint32_t cw[2] = {codes.x, codes.y};
        uint32_t o[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint16_t pair = static_cast<uint16_t>(cw[i >> 1] >> (16 * (i & 1)));
          uint32_t h2;
          asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(pair));
          const float2 v = add_f16x2_f32(h2, 0u);
          o[i] = tc::pack_bf16(v.x * sc, v.y * sc);
        }
        *reinterpret_cast<uint4*>(stage + (k >> 3) * kBlk + row * 128 + (((k & 7) ^ (row & 7)) << 4)) =
            make_uint4(o[0], o[1], o[2], o[3]);
      }
      tc::fence_proxy_async_smem();
      tc::mbar_arrive(&S->full[st]);
      tc::mbar_arrive(&S->raw_empty[ws]);
      return true;
    };
    const uint32_t n_share = static_cast<uint32_t>(a.plan.share_start[cl + 1] - a.plan.share_start[cl]);
    if (kF8 && n_share > 0 && !dequant(0)) ok = false;

    // Completes tile `q`: its P store, the rows past the sequence end, the hand-off to the PV warp.
    auto finish_commit = [&](uint32_t q, int valid) {
      tc::tmem_st_wait();
      // rows past the sequence end must not reach PV as NaN/Inf garbage
      if (valid < kTile) {
        uint8_t* stage = tiles + (q % kSt) * kStageBytes;
        const int nrow = kTile - valid;
        for (int idx = threadIdx.x - 128; idx < nrow * 4 * 8; idx += kSoftmaxThreads) {
          const int blk = idx / (nrow * 8), rem = idx % (nrow * 8);
          const int row = valid + rem / 8, ch = rem % 8;
          *reinterpret_cast<uint4*>(stage + blk * kBlk + row * 128 + ch * 16) = make_uint4(0, 0, 0, 0);
        }
        tc::fence_proxy_async_smem();
      }
      tc::tc_fence_before();
      tc::mbar_arrive(&S->p_full);
    };

    while (ok && have) {
      const int L = a.plan.lens[b];
      const int slot = b + static_cast<int>(cl);
      int nb_, nj0, nj1;
      SegIter si_next = si;
      const bool have_next = si_next.next(cum, a.batch, &nb_, &nj0, &nj1);
      m_used = -INFINITY;
      l = 0.f;
      for (int j = j0; j < j1 && ok; ++j, ++it) {
        // ---- own partial scores of tile it -> scaled fp16 -> the peer
        ok = tc::mbar_wait(&S->s_full, it & 1);
        if (!ok || aborted(S)) { ok = false; break; }
        tc::tc_fence_after();
        uint32_t own[kCols / 2];
        float own_un;
        {
          uint32_t r0[16];
          tc::tmem_ld16(t_s, r0);
          tc::tmem_ld_wait();
          // columns past the sequence end hold scores of whatever the pool rows contain:
          // zero them so they cannot set the scale (the softmax masks them anyway)
          const int vh = min(kTile, L - j * kTile) - kCols * part;
          if (vh < kCols) {
#pragma unroll
            for (int c = 0; c < 16; ++c) if (c >= vh) r0[c] = 0u;
          }
          float am[4];
#pragma unroll
          for (int c = 0; c < 4; ++c)
            am[c] = fmaxf(fmaxf(fabsf(__uint_as_float(r0[c])), fabsf(__uint_as_float(r0[c + 4]))),
                          fmaxf(fabsf(__uint_as_float(r0[c + 8])), fabsf(__uint_as_float(r0[c + 12]))));
          const float sc = exchange_scale(fmaxf(fmaxf(am[0], am[1]), fmaxf(am[2], am[3])), &own_un);
          if (sc != 1.f) {
#pragma unroll
            for (int c = 0; c < 16; ++c) r0[c] = __float_as_uint(__uint_as_float(r0[c]) * sc);
          }
#pragma unroll
          for (int c = 0; c < 8; ++c) own[c] = pack_f16(__uint_as_float(r0[2 * c]), __uint_as_float(r0[2 * c + 1]));
        }
        tc::tc_fence_before();
        tc::mbar_arrive(&S->s_free);
        if (kF8 && it + 1 < n_share && !dequant(it + 1)) { ok = false; break; }
        // ---- finish the previous tile of this segment (its peer half arrived while
        // this tile's scores were computed), then send this tile's half. Sending
        // only after consuming the peer's previous tile keeps two buffers safe:
        // the peer sent that tile after it had read what this CTA sent two tiles ago.
        if (have_pend) {
          ok = finish(pend_it, pend_valid);
          if (!ok) break;
        }
        {
          const uint32_t xb = it & 1u;
          const uint32_t dst = peer_x + xb * kXbufBytes;
          const uint32_t bar = xb ? peer_bar1 : peer_bar0;
#pragma unroll
          for (int u = 0; u < 2; ++u)
            tc::st_async_v4(dst + xoff(u), bar, own[4 * u], own[4 * u + 1], own[4 * u + 2], own[4 * u + 3]);
          tc::st_async_b32(dst + kXvalBytes + 4 * (part * kH + h), bar, __float_as_uint(own_un));
        }
        if (have_pend) finish_commit(pend_it, pend_valid);
        if (j == j1 - 1 && have_next) load_q(nb_);   // all score MMAs of this segment are done
#pragma unroll
        for (int c = 0; c < kCols / 2; ++c) pend[c] = own[c];
        pend_un = own_un;
        pend_valid = min(kTile, L - j * kTile);
        pend_it = it;
        have_pend = true;
      }
      if (!ok) break;
      ok = finish(pend_it, pend_valid);
      have_pend = false;
      if (!ok) break;
      finish_commit(pend_it, pend_valid);
      // ---- segment epilogue: unnormalised O (this thread's 256 / kParts columns), m and l
      ok = tc::mbar_wait(&S->o_done, (it - 1) & 1);
      if (!ok) break;
      tc::tc_fence_after();
      const int chunk0 = (rank * 256 + (256 / kParts) * part) / 4;   // first 4-float chunk of this thread's columns
      {
        uint32_t r0[16], r1[16], r2[16], r3[16];
        tc::tmem_ld16(t_o, r0);
        tc::tmem_ld16(t_o + 16, r1);
        tc::tmem_ld16(t_o + 32, r2);
        tc::tmem_ld16(t_o + 48, r3);
        tc::tmem_ld_wait();
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          *reinterpret_cast<uint4*>(a.part_o + parto_index(slot, chunk0 + u, h)) =
              make_uint4(r0[4 * u], r0[4 * u + 1], r0[4 * u + 2], r0[4 * u + 3]);
          *reinterpret_cast<uint4*>(a.part_o + parto_index(slot, chunk0 + 4 + u, h)) =
              make_uint4(r1[4 * u], r1[4 * u + 1], r1[4 * u + 2], r1[4 * u + 3]);
          *reinterpret_cast<uint4*>(a.part_o + parto_index(slot, chunk0 + 8 + u, h)) =
              make_uint4(r2[4 * u], r2[4 * u + 1], r2[4 * u + 2], r2[4 * u + 3]);
          *reinterpret_cast<uint4*>(a.part_o + parto_index(slot, chunk0 + 12 + u, h)) =
              make_uint4(r3[4 * u], r3[4 * u + 1], r3[4 * u + 2], r3[4 * u + 3]);
        }
      }
      tc::tc_fence_before();
      tc::mbar_arrive(&S->o_free);
      // l of the kParts warps of this row (all scaled by the same factors)
      S->redl[part][h] = l;
      tc::mbar_arrive(&S->pair_sum[quarter]);
      ok = tc::mbar_wait(&S->pair_sum[quarter], n_epi & 1);
      ++n_epi;
      if (!ok) break;
      if (rank == 0 && part == 0) {
        float lt = 0.f;
#pragma unroll
        for (int pp = 0; pp < kParts; ++pp) lt += S->redl[pp][h];
        float2* ml = reinterpret_cast<float2*>(a.part_ml) + static_cast<int64_t>(slot) * kH + h;
        *ml = make_float2(m_used, lt);
      }
      have = si.next(cum, a.batch, &b, &j0, &j1);
    }
    if (!ok) set_abort(S);
  }
  // ---------------------------------------------------------------- teardown
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  tc::tc_fence_before();
  __syncthreads();
  __syncwarp();
  tc::cluster_sync();  // the peer no longer writes into this CTA's shared memory
  tc::tc_fence_after();
  if (warp == 1) tc::tmem_dealloc<512>(tm);
}

// ================================================================== merge (log-sum-exp over segments)
struct MergeArgs {
  Plan plan;
  const float* part_o;   // chunk-major, see parto_index
  const float* part_ml;  // [slots, H, 2]
  uint16_t* o_hi;        // [B, H, 512] bf16: o_lat rounded
  uint16_t* o_lo;        // [B, H, 512] bf16: o_lat - o_hi rounded
  int batch, ncl;
};

constexpr int kMergeSplit = kOChunks;            // CTAs per sequence: one 4-float chunk each

// One CTA per (sequence b, 4 latent elements); thread = head. o_lat =
// sum_s w_s O_s / sum_s w_s l_s with w_s = 2^(m_s - max m) over the partials
// of b's segments (slots b + c for the clusters c whose shares meet b's
// tiles). Every load is a warp reading 32 consecutive heads of one chunk.
__global__ void __launch_bounds__(kH) merge_kernel(MergeArgs a) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int h = threadIdx.x;
  const int b = blockIdx.y;
  const int chunk = blockIdx.x;
  const int c0 = a.plan.seq_c0[b], c1 = a.plan.seq_c1[b];   // c1 < c0: no tiles, output 0
  const int32_t* start = a.plan.share_start;
  const float2* ml_all = reinterpret_cast<const float2*>(a.part_ml);
  // online log-sum-exp over the partials, eight at a time so their loads overlap
  float M = -INFINITY, den = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int cb = c0; cb <= c1; cb += 8) {
    float4 o[8];
    float2 ml[8];
    bool use[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      // the loads do not wait for the share check: a slot of an empty share (which wrote
      // no partial) is read and then ignored, so all loads are one round trip
      const int c = cb + u;
      use[u] = c <= c1 && start[c] < start[c + 1];
      if (c <= c1) {
        ml[u] = ml_all[static_cast<int64_t>(b + c) * kH + h];
        o[u] = *reinterpret_cast<const float4*>(a.part_o + parto_index(b + c, chunk, h));
      }
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      if (!use[u]) continue;
      float w = 1.f;
      if (ml[u].x > M) {
        const float r = exp2f(M - ml[u].x);   // 0 on the first partial (M = -inf)
        acc.x *= r; acc.y *= r; acc.z *= r; acc.w *= r;
        den *= r;
        M = ml[u].x;
      } else {
        w = exp2f(ml[u].x - M);
      }
      acc.x = fmaf(w, o[u].x, acc.x);
      acc.y = fmaf(w, o[u].y, acc.y);
      acc.z = fmaf(w, o[u].z, acc.z);
      acc.w = fmaf(w, o[u].w, acc.w);
      den = fmaf(w, ml[u].y, den);
    }
  }
  const float inv = den > 0.f ? 1.f / den : 0.f;
  const float v[4] = {acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv};
  uint32_t hi[2], lo[2];
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    hi[u] = tc::pack_bf16(v[2 * u], v[2 * u + 1]);
    lo[u] = tc::pack_bf16(v[2 * u] - bf16_to_f32(static_cast<uint16_t>(hi[u] & 0xffffu)),
                          v[2 * u + 1] - bf16_to_f32(static_cast<uint16_t>(hi[u] >> 16)));
  }
  const int64_t e = (static_cast<int64_t>(b) * kH + h) * kDc + 4 * chunk;
  *reinterpret_cast<uint2*>(a.o_hi + e) = make_uint2(hi[0], hi[1]);
  *reinterpret_cast<uint2*>(a.o_lo + e) = make_uint2(lo[0], lo[1]);
}

// ================================================================== W_UV
struct UvArgs {
  float* out;      // [B, H, 128]
  int batch;
};

constexpr int kUvThreads = 128;
constexpr int kUvNb = 32;   // sequences per MMA chunk
constexpr size_t kUvSmem = 8 * 16384 + 2 * 8 * kUvNb * 128 + 64;

// One CTA per head i: out[b, i, :] = W_UV[i] (o_hi[b, i, :] + o_lo[b, i, :]),
// M = 128 output rows, N = 32 sequences per chunk, K = 512 twice (hi, lo).
__global__ void __launch_bounds__(kUvThreads) uv_tc_kernel(const __grid_constant__ CUtensorMap map_wuv,
                                                           const __grid_constant__ CUtensorMap map_hi,
                                                           const __grid_constant__ CUtensorMap map_lo, UvArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* sA = sm;                                 // W_UV[i]: 8 boxes [128 rows x 64] = 128 KB
  uint8_t* sHi = sm + 8 * 16384;                    // o_hi rows: 8 boxes [32 rows x 64] = 32 KB
  uint8_t* sLo = sHi + 8 * kUvNb * 128;             // o_lo rows
  uint64_t* bars = reinterpret_cast<uint64_t*>(sLo + 8 * kUvNb * 128);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 3);
  const int i = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, t = threadIdx.x;
  if (t == 0) {
    tc::mbar_init(&bars[0], 1);   // weights landed
    tc::mbar_init(&bars[1], 1);   // o_lat rows landed (one phase per chunk)
    tc::mbar_init(&bars[2], 1);   // MMAs done (one phase per chunk)
    tc::fence_mbar_init();
    tc::tma_prefetch_map(&map_wuv);
    tc::tma_prefetch_map(&map_hi);
    tc::tma_prefetch_map(&map_lo);
    // the weights do not depend on the kernels before: start streaming them now
    tc::mbar_arrive_expect_tx(&bars[0], 8 * 16384);
    for (int j = 0; j < 8; ++j) tc::tma_load_2d(sA + j * 16384, &map_wuv, 64 * j, i * kDh, &bars[0]);
  }
  if (warp == 0) tc::tmem_alloc<32>(tslot);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tm = *tslot;
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const uint32_t idesc = tc::idesc_bf16_f32(128, kUvNb, 0, 0);
  bool ok = true;
  int chunk = 0;
  for (int n0 = 0; n0 < a.batch; n0 += kUvNb, ++chunk) {
    if (t == 0) {
      tc::mbar_arrive_expect_tx(&bars[1], 2 * 8 * kUvNb * 128);
      for (int k = 0; k < 8; ++k) {
        tc::tma_load_2d(sHi + k * kUvNb * 128, &map_hi, i * kDc + 64 * k, n0, &bars[1]);
        tc::tma_load_2d(sLo + k * kUvNb * 128, &map_lo, i * kDc + 64 * k, n0, &bars[1]);
      }
      ok = tc::mbar_wait(&bars[0], 0) && tc::mbar_wait(&bars[1], chunk & 1);
      tc::tc_fence_after();
      if (ok) {
        const uint64_t a0 = tc::sdesc_sw128(tc::smem_u32(sA), 16, 1024);
        const uint64_t h0 = tc::sdesc_sw128(tc::smem_u32(sHi), 16, 1024);
        const uint64_t l0 = tc::sdesc_sw128(tc::smem_u32(sLo), 16, 1024);
#pragma unroll
        for (int kk = 0; kk < 32; ++kk) {
          const uint64_t ad = a0 + static_cast<uint64_t>(((kk >> 2) * 16384 + (kk & 3) * 32) >> 4);
          const uint64_t bo = static_cast<uint64_t>(((kk >> 2) * (kUvNb * 128) + (kk & 3) * 32) >> 4);
          tc::mma_ss(tm, ad, h0 + bo, idesc, kk > 0 ? 1u : 0u);
          tc::mma_ss(tm, ad, l0 + bo, idesc, 1u);
        }
      }
      tc::mma_commit(&bars[2]);
    }
    __syncwarp();
    ok = tc::mbar_wait(&bars[2], chunk & 1) && ok;
    tc::tc_fence_after();
    uint32_t r0[16], r1[16];
    tc::tmem_ld16(tc::tmem_at(tm, 32 * warp, 0), r0);
    tc::tmem_ld16(tc::tmem_at(tm, 32 * warp, 16), r1);
    tc::tmem_ld_wait();
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      const int b0 = n0 + c, b1 = n0 + 16 + c;
      if (b0 < a.batch) a.out[(static_cast<int64_t>(b0) * kH + i) * kDh + 32 * warp + lane] = __uint_as_float(r0[c]);
      if (b1 < a.batch) a.out[(static_cast<int64_t>(b1) * kH + i) * kDh + 32 * warp + lane] = __uint_as_float(r1[c]);
    }
    tc::tc_fence_before();
    __syncthreads();   // the B operand and TMEM are reused by the next chunk
  }
  if (warp == 0) tc::tmem_dealloc<32>(tm);
}

}  // namespace tcd
}  // namespace mla
