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
//   attend  : persistent clusters of two CTAs (attend_pair.cuh); cluster c
//             takes an equal share of all 64-token tiles of all sequences,
//             cut at sequence ends into segments. Each CTA of a pair owns 64
//             heads; the score and PV contractions run as pair MMAs, and each
//             segment ends in an unnormalised partial (O, running max m, sum l).
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
constexpr float kRescaleThreshold = 8.0f;    // log2 units: O is rescaled only when the max grows by > 2^8

// Layout of the segment partials in the workspace, chunk-major so that a warp
// holding 32 consecutive heads touches one contiguous 512-byte line:
//   part_o [slot][128 chunks][128 heads][4 fp32]  chunk c = latent 4c..4c+3
constexpr int kOChunks = kDc / 4;     // 128

__host__ __device__ __forceinline__ int64_t parto_index(int64_t slot, int chunk, int head) {
  return ((slot * kOChunks + chunk) * kH + head) * 4;
}

// The clusters split the work in units: a sequence with tiles counts its tiles plus kSegUnits for
// the start of a segment (its queries' load, the pipeline fill and the partial's write, about three
// tiles' time), so a cluster whose share crosses into another sequence gets fewer tiles. Tile j of
// sequence b is unit cum[b] + kSegUnits + j.
constexpr int kSegUnits = 3;
// Pool rows of the first kPlanRows tiles of each share are in the plan, so that the attend kernel
// requests them as soon as the plan is ready, without walking the plan and the page table first.
constexpr int kPlanRows = 4;

struct Plan {
  int32_t* lens;         // [B] lengths clamped to [0, max_seq_len]
  int32_t* cum;          // [B+1] prefix sums of units(b) = tiles(b) + kSegUnits (0 for a sequence without tiles)
  int32_t* first_seq;    // [clusters] sequence holding the first unit of each cluster's share
  int32_t* share_start;  // [clusters + 1] first unit of each cluster's share (share c = [start[c], start[c+1]))
  int32_t* seq_c0;       // [B] first cluster whose share holds tiles of sequence b (when it has any)
  int32_t* seq_c1;       // [B] last such cluster
  int32_t* share_tiles;  // [clusters] tiles in each cluster's share
  int32_t* first_rows;   // [clusters][kPlanRows] pool rows of each share's first tiles (see cache_tile_row)
};

// Unit range [t0, t1) of cluster c when T units are split over nc clusters.
__host__ __device__ __forceinline__ int64_t share_begin(int64_t c, int64_t T, int64_t nc) { return c * T / nc; }

// The cluster whose share holds unit t (T > 0).
__host__ __device__ __forceinline__ int64_t share_owner(int64_t t, int64_t T, int64_t nc) {
  return ((t + 1) * nc - 1) / T;
}

// ================================================================== absorb (+ plan)
struct AbsorbArgs {
  const uint16_t* q_rope;     // [B, H, 64]
  const int32_t* seq_lens;    // [B]
  const int32_t* block_table; // [B, max_pages] (NULL: contiguous, sequence b owns pages b*max_pages ..)
  uint16_t* q_lat;            // row-major [B, H, 576], see qlat_row_index
  Plan plan;
  int64_t num_pages;
  int max_pages, page_size;
  int batch, nb, max_seq_len, ncl;
  int f16_lat;                // 1: the latent part of Q_lat in fp16 (the operand type of an FP8 cache's tiles)
};

__host__ __device__ __forceinline__ int64_t qlat_row_index(int64_t b, int head, int k) {
  return (b * kH + head) * kRow + k;
}

struct SegIter {
  int64_t t, t1;  // next unit (global index) and end of share
  int b;          // current sequence
  // the next (sequence, tile range [j0, j1)) with at least one tile; false at the share's end
  __host__ __device__ __forceinline__ bool next(const int32_t* cum, int batch, int* seq, int* j0, int* j1) {
    while (t < t1) {
      while (b < batch && cum[b + 1] <= t) ++b;
      if (b >= batch) return false;
      const int64_t first = cum[b] + kSegUnits;   // unit of the sequence's tile 0
      const int64_t start = t > first ? t : first;
      const int64_t end = t1 < cum[b + 1] ? t1 : static_cast<int64_t>(cum[b + 1]);
      t = end;
      if (start < end) {
        *seq = b;
        *j0 = static_cast<int>(start - first);
        *j1 = static_cast<int>(end - first);
        return true;
      }
    }
    return false;
  }
};

// Tiles in the unit range [t0, t1) whose first unit lies in sequence `first` (units less the
// segment-start units the range holds); with fb / fj, also the sequence and tile index of the
// range's first kPlanRows tiles (entries past the count are left alone).
__host__ __device__ __forceinline__ int64_t share_tile_count(const int32_t* cum, int batch, int first, int64_t t0,
                                                             int64_t t1, int* fb = nullptr, int* fj = nullptr) {
  SegIter si{t0, t1, first};
  int b, j0, j1;
  int64_t n = 0;
  while (si.next(cum, batch, &b, &j0, &j1)) {
    if (fb)
      for (int64_t k = n; k < kPlanRows && k < n + (j1 - j0); ++k) {
        fb[k] = b;
        fj[k] = j0 + static_cast<int>(k - n);
      }
    n += j1 - j0;
  }
  return n;
}

// Pool row of tile j (tokens 64 j ..) of sequence b: page block_table[b][64 j / page_size] (or
// b * max_pages + that index without a table), row 64 j mod page_size within it. A page id outside
// [0, num_pages) or a page index past max_pages flags a bounds error and gives a row outside the
// pool, which a tile load fills with zeros.
__device__ __forceinline__ int32_t cache_tile_row(const int32_t* block_table, int b, int j, int max_pages,
                                                  int page_size, int64_t num_pages) {
  const int64_t tok = static_cast<int64_t>(j) * kTile;
  const int pg = static_cast<int>(tok / page_size);
  int64_t page = -1;
  if (pg < max_pages)
    page = block_table ? block_table[static_cast<int64_t>(b) * max_pages + pg] : static_cast<int64_t>(b) * max_pages + pg;
  if (page < 0 || page >= num_pages) {
    flag_error(ERR_BIT_BOUNDS);
    return -2 * kTile;
  }
  return static_cast<int32_t>(page * page_size + tok % page_size);
}

constexpr int kAbsorbThreads = 128;

// Prefix sums the plan block keeps in shared memory (the absorb kernel's dynamic shared memory,
// unused by this block): the share searches read them there for batches below this size.
constexpr int kPlanSmemRows = 16384;

__device__ void plan_block(const AbsorbArgs& a, int32_t* cum_s) {
  const bool in_smem = a.batch < kPlanSmemRows;
  __shared__ int32_t carry;
  __shared__ int32_t warp_tot[kAbsorbThreads / 32];
  if (threadIdx.x == 0) {
    carry = 0;
    a.plan.cum[0] = 0;
    cum_s[0] = 0;
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
      if (n > 0) n += kSegUnits;
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
    if (b < a.batch) {
      a.plan.cum[b + 1] = off + x;
      if (in_smem) cum_s[b + 1] = off + x;
    }
    __syncthreads();
    if (threadIdx.x == kAbsorbThreads - 1) carry = off + x;
    __syncthreads();
  }
  // cluster shares: start tile and first sequence of each; clusters of each sequence
  const int32_t* cum = in_smem ? cum_s : a.plan.cum;
  const int64_t T = cum[a.batch];
  for (int c = threadIdx.x; c <= a.ncl; c += kAbsorbThreads) {
    const int64_t t = share_begin(c, T, a.ncl);
    a.plan.share_start[c] = static_cast<int32_t>(t);
    if (c == a.ncl) continue;
    int lo = 0, hi = a.batch;   // cum[lo] <= t
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (cum[mid] <= t) lo = mid; else hi = mid;
    }
    a.plan.first_seq[c] = lo;
    int fb[kPlanRows], fj[kPlanRows];
    const int64_t n = share_tile_count(cum, a.batch, lo, t, share_begin(c + 1, T, a.ncl), fb, fj);
    a.plan.share_tiles[c] = static_cast<int32_t>(n);
    int32_t rows[kPlanRows];
#pragma unroll
    for (int k = 0; k < kPlanRows; ++k)   // independent page-table loads
      rows[k] = k < n ? cache_tile_row(a.block_table, fb[k], fj[k], a.max_pages, a.page_size, a.num_pages) : 0;
#pragma unroll
    for (int k = 0; k < kPlanRows; ++k) a.plan.first_rows[c * kPlanRows + k] = rows[k];
  }
  for (int b = threadIdx.x; b < a.batch; b += kAbsorbThreads) {
    const int64_t tb0 = cum[b], tb1 = cum[b + 1];
    if (tb1 > tb0) {
      a.plan.seq_c0[b] = static_cast<int32_t>(share_owner(tb0 + kSegUnits, T, a.ncl));   // its first tile
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
  extern __shared__ uint8_t smem_raw[];
  if (blockIdx.x == 2 * kH) {
    // the lengths and the page table go to L2 while the kernel ahead finishes (a prefetch reads
    // nothing, so a kernel that still writes them is no hazard: L2 holds the one copy)
    const char* pl = reinterpret_cast<const char*>(a.seq_lens);
    for (int64_t o = 128 * threadIdx.x; o < 4 * static_cast<int64_t>(a.batch); o += 128 * kAbsorbThreads)
      asm volatile("prefetch.global.L2 [%0];" ::"l"(pl + o));
    if (a.block_table) {
      const char* pt = reinterpret_cast<const char*>(a.block_table);
      const int64_t nbytes = min(4 * static_cast<int64_t>(a.batch) * a.max_pages, static_cast<int64_t>(1) << 19);
      for (int64_t o = 128 * threadIdx.x; o < nbytes; o += 128 * kAbsorbThreads)
        asm volatile("prefetch.global.L2 [%0];" ::"l"(pt + o));
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");
    plan_block(a, reinterpret_cast<int32_t*>(smem_raw));
    return;
  }
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
      *reinterpret_cast<uint4*>(a.q_lat + qlat_row_index(b, i, kDc + 8 * c)) = v;
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
            a.q_lat[qlat_row_index(b, i, k)] =
                a.f16_lat ? __half_as_ushort(__float2half_rn(__uint_as_float(r[c]))) : f32_to_bf16_bits(__uint_as_float(r[c]));
        }
      }
    }
    tc::tc_fence_before();
    __syncthreads();  // TMEM and the query box are reused by the next chunk
  }
  if (warp == 0) tc::tmem_dealloc<256>(tm);
}

// ================================================================== attend (shared by the attend kernel)
struct AttendArgs {
  const uint16_t* q_lat;      // row-major [B, H, 576], see qlat_row_index
  const int32_t* block_table; // [B, max_pages] (NULL: contiguous, sequence b owns pages b*max_pages ..)
  int max_seq_len;
  Plan plan;
  float* part_o;              // chunk-major (see parto_index) fp32, unnormalised
  float* part_ml;             // [slots, H, 2]: running max (log2 units) and sum
  int64_t num_pages;
  int batch, max_pages, page_size;
  float scale_log2;           // softmax scale * log2(e), > 0
};

// Segment iterator: the (sequence, tile range) pieces of this cluster's share.

__device__ __forceinline__ SegIter seg_begin(const Plan& plan, int batch, uint32_t c, uint32_t nc) {
  (void)batch;
  (void)nc;
  SegIter it;
  it.t = plan.share_start[c];
  it.t1 = plan.share_start[c + 1];
  it.b = plan.first_seq[c];
  return it;
}

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

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

// ================================================================== merge (log-sum-exp over segments)
struct MergeArgs {
  Plan plan;
  const float* part_o;   // chunk-major, see parto_index
  const float* part_ml;  // [slots, H, 2]
  uint16_t* o_hi;        // [B, H, 512] bf16 (fp16 when f16): o_lat rounded
  uint16_t* o_lo;        // [B, H, 512] bf16 (fp16 when f16): o_lat - o_hi rounded
  int batch, ncl;
  int f16;               // 1: fp16 pair (the operand type of the folded output GEMM)
};

// One CTA per (sequence b, kG chunks of 4 latent elements); thread = head.
// o_lat = sum_s w_s O_s / sum_s w_s l_s with w_s = 2^(m_s - max m) over the
// partials of b's segments (slots b + c for the clusters c whose shares meet
// b's tiles), as an online log-sum-exp over kS slots at a time: the (m, l)
// pairs and the kG chunks of kS slots are loaded together, one round trip per
// group. Small batches take one chunk per CTA (enough CTAs to fill the GPU);
// larger ones four, so that fewer, longer CTAs do the work. Every load is a
// warp reading 32 consecutive heads of one chunk.
template <int kG, int kS>
__global__ void __launch_bounds__(kH) merge_kernel(MergeArgs a) {
  static_assert(kG == 1 || kG % 2 == 0, "chunks are stored 8 or 16 elements at a time");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int h = threadIdx.x;
  const int b = blockIdx.y;
  const int ch0 = blockIdx.x * kG;
  const int c0 = a.plan.seq_c0[b], c1 = a.plan.seq_c1[b];   // c1 < c0: no tiles, output 0
  const int32_t* start = a.plan.share_start;
  const float2* ml_all = reinterpret_cast<const float2*>(a.part_ml);
  float M = -INFINITY, den = 0.f;
  float4 acc[kG];
#pragma unroll
  for (int k = 0; k < kG; ++k) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int cb = c0; cb <= c1; cb += kS) {
    float4 o[kS][kG];
    float2 ml[kS];
    bool use[kS];
#pragma unroll
    for (int u = 0; u < kS; ++u) {
      // the loads do not wait for the share check: a slot of an empty share (which wrote
      // no partial) is read and then ignored, so all loads are one round trip
      const int c = cb + u;
      use[u] = c <= c1 && start[c] < start[c + 1];
      if (c <= c1) {
        ml[u] = ml_all[static_cast<int64_t>(b + c) * kH + h];
#pragma unroll
        for (int k = 0; k < kG; ++k)
          o[u][k] = *reinterpret_cast<const float4*>(a.part_o + parto_index(b + c, ch0 + k, h));
      }
    }
#pragma unroll
    for (int u = 0; u < kS; ++u) {
      if (!use[u]) continue;
      float w = 1.f;
      if (ml[u].x > M) {
        const float r = exp2f(M - ml[u].x);   // 0 on the first partial (M = -inf)
#pragma unroll
        for (int k = 0; k < kG; ++k) {
          acc[k].x *= r; acc[k].y *= r; acc[k].z *= r; acc[k].w *= r;
        }
        den *= r;
        M = ml[u].x;
      } else {
        w = exp2f(ml[u].x - M);
      }
#pragma unroll
      for (int k = 0; k < kG; ++k) {
        acc[k].x = fmaf(w, o[u][k].x, acc[k].x);
        acc[k].y = fmaf(w, o[u][k].y, acc[k].y);
        acc[k].z = fmaf(w, o[u][k].z, acc[k].z);
        acc[k].w = fmaf(w, o[u][k].w, acc[k].w);
      }
      den = fmaf(w, ml[u].y, den);
    }
  }
  const float inv = den > 0.f ? 1.f / den : 0.f;
  uint32_t hi[2 * kG], lo[2 * kG];
#pragma unroll
  for (int k = 0; k < kG; ++k) {
    const float v[4] = {acc[k].x * inv, acc[k].y * inv, acc[k].z * inv, acc[k].w * inv};
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      if (a.f16) {
        const __half h0 = __float2half_rn(v[2 * u]), h1 = __float2half_rn(v[2 * u + 1]);
        const __half l0 = __float2half_rn(v[2 * u] - __half2float(h0));
        const __half l1 = __float2half_rn(v[2 * u + 1] - __half2float(h1));
        hi[2 * k + u] = static_cast<uint32_t>(__half_as_ushort(h0)) | (static_cast<uint32_t>(__half_as_ushort(h1)) << 16);
        lo[2 * k + u] = static_cast<uint32_t>(__half_as_ushort(l0)) | (static_cast<uint32_t>(__half_as_ushort(l1)) << 16);
      } else {
        const uint32_t p = tc::pack_bf16(v[2 * u], v[2 * u + 1]);
        hi[2 * k + u] = p;
        lo[2 * k + u] = tc::pack_bf16(v[2 * u] - bf16_to_f32(static_cast<uint16_t>(p & 0xffffu)),
                                      v[2 * u + 1] - bf16_to_f32(static_cast<uint16_t>(p >> 16)));
      }
    }
  }
  const int64_t e = (static_cast<int64_t>(b) * kH + h) * kDc + 4 * ch0;   // 4 kG elements, 8 kG-byte aligned
  if constexpr (kG == 1) {
    *reinterpret_cast<uint2*>(a.o_hi + e) = make_uint2(hi[0], hi[1]);
    *reinterpret_cast<uint2*>(a.o_lo + e) = make_uint2(lo[0], lo[1]);
  } else {
#pragma unroll
    for (int q = 0; q < kG / 2; ++q) {
      reinterpret_cast<uint4*>(a.o_hi + e)[q] = make_uint4(hi[4 * q], hi[4 * q + 1], hi[4 * q + 2], hi[4 * q + 3]);
      reinterpret_cast<uint4*>(a.o_lo + e)[q] = make_uint4(lo[4 * q], lo[4 * q + 1], lo[4 * q + 2], lo[4 * q + 3]);
    }
  }
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
