// Attend step of the tensor-core MLA decode on a CTA pair whose MMAs are
// pair MMAs (tcgen05 cta_group::2), for a bf16 latent cache (DeepSeek-V2
// report, section 2.1.2: scores and values both read the shared latent;
// section 2.1.3: the decoupled rope key adds to the scores).
//
// Why this shape. The output accumulator O_lat of 128 heads x 512 latent
// values in fp32 fills one SM's tensor memory, so two SMs share every tile.
// Splitting the work so that each SM owns 64 heads end to end needs no
// software exchange between them: the pair MMA moves operand halves between
// the two SMs itself. Each CTA keeps half of every cache tile (its 256 latent
// columns and 32 of the 64 rope columns) and the queries of its 64 heads.
//
//   scores  S = Q K^T: one pair MMA per 16-wide step of the contraction, M = 256
//           rows (per CTA: 64 heads x the two halves of the contraction), N = 128
//           (64 tokens x the two halves), K = 288. Of each CTA's 128 x 128 result
//           only the blocks (head, half A) x (token, half A) and (head, half B) x
//           (token, half B) are used; their sum is the score. This costs twice
//           the MACs of the score but runs 18 full-rate MMAs per tile, where a
//           64-column MMA would be held up by the tensor pipe's fixed cost per
//           instruction.
//   softmax each CTA only for its 64 heads (8 warps, 16 scores per thread).
//   PV      O += P V: pair MMA, M = 128 (64 heads per CTA), N = 256 latent
//           columns per MMA (128 from each CTA's half), K = 64 tokens.
//
// Tensor memory (512 columns): two score buffers of 128 columns, then O as two
// 128-column halves (the pair-MMA layout puts row m of a CTA's 64 in lanes m and
// m + 64, each with one half of the N columns).
#pragma once

#include "common.cuh"
#include "decode_tc.cuh"
#include "tc.cuh"

namespace mla {
namespace tcd {

constexpr int kPrMaxStages = 4;                     // cache tile ring depth (bf16 cache; 3 with FP8)
constexpr int kPrBox = kTile * 128;                 // one latent TMA box: 64 rows x 64 bf16 = 8 KB (128-byte swizzle)
constexpr int kPrRopeBox = kTile * 64;              // one rope box: 64 rows x 32 bf16 = 4 KB (64-byte swizzle)
constexpr int kPrStageBytes = 4 * kPrBox + kPrRopeBox;   // this CTA's 256 latent and 32 rope columns of a tile
constexpr int kPrQBox = 128 * 128;                  // 128 rows x 64 bf16 = 16 KB
constexpr int kPrQBytes = 4 * kPrQBox + 128 * 64;   // queries of 64 heads, both contraction halves (+ 32 rope each)
constexpr int kPrPHalf = 64 * 64;                   // P of 32 tokens: 64 heads x 32 bf16 (64-byte swizzle)
// P of a tile: tokens 0..31 go into the tile's rope box (dead once its score MMAs completed),
// tokens 32..63 into one of two 4 KB buffers (by tile parity)
constexpr int kPrPBytes = 2 * kPrPHalf;
constexpr int kPrSoftmaxWarps = 8;
constexpr uint32_t kPrTmS = 0;                      // score buffers at 0 and 128
constexpr uint32_t kPrTmO = 256;                    // O: PV MMA 0 at 256, MMA 1 at 384
constexpr int kPrKSteps = 18;                       // contraction steps of 16 per half (256 latent + 32 rope)
constexpr int kPrF8Ahead = 8;                       // FP8 cache: tiles prefetched to L2 ahead of their loads

struct PairSmem {
  uint64_t full[kPrMaxStages];    // this CTA's half of a tile landed (TMA; bf16 cache)
  uint64_t empty[kPrMaxStages];   // the PV of the tile in the slot completed (pair commit)
  uint64_t ready[kPrMaxStages];   // even CTA: both halves of a tile are in their bf16 stages
  uint64_t raw_full[2];           // FP8 cache: codes, scales and rope values of a tile landed
  uint64_t raw_empty[2];          // FP8 cache: the dequantising warps are done with a raw slot
  uint64_t qfull, qfree, qready;
  uint64_t s_full[2];          // scores of a tile are in TMEM (pair commit)
  uint64_t s_free[2];          // even CTA: all softmax warps of both CTAs read them
  uint64_t p_full[2];          // even CTA, by tile parity: P written, O rescaled, tail rows cleared, in both CTAs
  uint64_t o_done[2];          // the PV of a tile of this parity completed (pair commit)
  uint64_t o_free;             // even CTA: both CTAs read O at a segment end
  uint64_t drain[3];
  union {
    float red_max[2][2][64];   // [tile parity][token half][head] row maxima of the two warps of a head
    float red_l[2][64];        // [token half][head] row sums at a segment end (after the last tile's maxima)
  };
  float alpha[2][64];          // [tile parity][head] rescale factor of O (1 when unchanged)
  uint32_t tmem_base;
  int32_t abort_flag;
};

// Per cache format: ring depths, thread count and shared-memory carve-up
// (Q | bf16 stages | FP8 raw ring | P tokens 32..63 | barriers).
template <bool kF8>
struct PairCfg {
  static constexpr int kSt = kF8 ? 3 : kPrMaxStages;
  static constexpr int kRaw = kF8 ? 2 : 0;
  static constexpr int kRawCodes = kTile * 256;                 // this CTA's 256 E4M3 codes of 64 rows
  static constexpr int kRawBytes = kRawCodes + kTile * 16;      // + the 4 fp32 block scales of each row
  static constexpr int kDequantWarps = kF8 ? 4 : 0;
  static constexpr int kThreads = 32 * (6 + kPrSoftmaxWarps + kDequantWarps);
  static constexpr size_t kRawOff = kPrQBytes + static_cast<size_t>(kSt) * kPrStageBytes;
  static constexpr size_t kPOff = kRawOff + static_cast<size_t>(kRaw) * kRawBytes;
  static constexpr size_t kSmem = 1024 + kPOff + kPrPBytes + sizeof(PairSmem);
};

__device__ __forceinline__ bool pr_aborted(const PairSmem* s) {
  return *reinterpret_cast<const volatile int32_t*>(&s->abort_flag) != 0;
}
__device__ __forceinline__ void pr_set_abort(PairSmem* s) {
  *reinterpret_cast<volatile int32_t*>(&s->abort_flag) = 1;
}

// bf16 cache (kF8 = false):
//   map_lat:   the pool [rows, 576], boxes of 64 rows x 64 columns, 128-byte swizzle.
//   map_rope:  the same pool, boxes of 64 rows x 32 columns, 64-byte swizzle.
// FP8 cache (kF8 = true; rows of 512 E4M3 codes, 4 fp32 scales, 64 bf16 rope values):
//   map_lat:   byte view of the pool [rows, 656], unswizzled boxes of 64 rows x 256 codes.
//   map_scale: the same, boxes of 64 rows x 16 bytes (the 4 block scales).
//   map_rope:  the rope values as bf16 [rows, 64] (row stride 656 bytes), boxes of 64 x 32, 64-byte swizzle.
// map_q:  Q_lat row-major [B * 128 heads, 576] bf16, boxes of 16 rows x 64 columns, 128-byte swizzle.
// map_qr: the same Q_lat, boxes of 16 rows x 32 columns, 64-byte swizzle.
// The FP8 codes are dequantised by four extra warps into the tile layout a bf16 pool gives, in fp16
// (code x block scale: the code converts exactly, one packed fp16 multiply): fp16 keeps 3 more bits
// than bf16 and costs two instructions per pair of values. The latent part of the queries (written
// by the absorb kernel) and P are then fp16 too; the rope part stays bf16 with its own MMA kind.
template <bool kF8>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(PairCfg<kF8>::kThreads, 1)
    attend_pair_kernel(const __grid_constant__ CUtensorMap map_lat, const __grid_constant__ CUtensorMap map_rope,
                       const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_qr,
                       const __grid_constant__ CUtensorMap map_scale, AttendArgs a) {
  using CF = PairCfg<kF8>;
  constexpr int kPrStages = CF::kSt;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* sQ = sm;                                   // 4 boxes [128 rows x 64], 1 box [128 rows x 32]
  uint8_t* stages = sm + kPrQBytes;                   // kPrStages x (4 boxes [64 tokens x 64], 1 [64 x 32])
  uint8_t* rawb = sm + CF::kRawOff;                   // FP8: 2 x (codes [64 x 256], scales [64 x 16])
  uint8_t* sP = sm + CF::kPOff;                       // 2 x [64 heads x 32 tokens] (P tokens 32..63)
  PairSmem* S = reinterpret_cast<PairSmem*>(sP + kPrPBytes);

  const uint32_t rank = tc::cluster_ctarank();
  const uint32_t cl = tc::cluster_id_x(), ncl = tc::n_clusters_x();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kPrStages; ++s) {
      tc::mbar_init(&S->full[s], 1);
      tc::mbar_init(&S->empty[s], 1);
      tc::mbar_init(&S->ready[s], kF8 ? 2 * CF::kDequantWarps : 2);
    }
    for (int s = 0; s < CF::kRaw; ++s) {
      tc::mbar_init(&S->raw_full[s], 1);
      tc::mbar_init(&S->raw_empty[s], CF::kDequantWarps);
    }
    tc::mbar_init(&S->qfull, 1);
    tc::mbar_init(&S->qfree, 2);   // one commit from each score issuer
    tc::mbar_init(&S->qready, 2);
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(&S->s_full[b], 1);
      tc::mbar_init(&S->s_free[b], 2 * kPrSoftmaxWarps);
    }
    tc::mbar_init(&S->p_full[0], 2 * kPrSoftmaxWarps);
    tc::mbar_init(&S->p_full[1], 2 * kPrSoftmaxWarps);
    tc::mbar_init(&S->o_done[0], 1);
    tc::mbar_init(&S->o_done[1], 1);
    tc::mbar_init(&S->o_free, 2 * kPrSoftmaxWarps);
    for (int i = 0; i < 3; ++i) tc::mbar_init(&S->drain[i], 1);
    S->abort_flag = 0;
    tc::fence_mbar_init();
    tc::tma_prefetch_map(&map_lat);
    tc::tma_prefetch_map(&map_rope);
    tc::tma_prefetch_map(&map_q);
    tc::tma_prefetch_map(&map_qr);
    if (kF8) tc::tma_prefetch_map(&map_scale);
  }
  if (warp == 1) tc::tmem_alloc_pair<512>(&S->tmem_base);
  tc::tc_fence_before();
  tc::cluster_sync();
  tc::tc_fence_after();
  const uint32_t tm = S->tmem_base;

  uint32_t n_pre = 0;
  const uint64_t policy = tc::policy_evict_first();
  auto issue_tile = [&](uint32_t it, int32_t y) {   // lane 0 of the producer warp; slots free for it < ring
    const int st = it % kPrStages;
    if (kF8) {
      uint8_t* raw = rawb + (it & 1) * CF::kRawBytes;
      uint64_t* bar = &S->raw_full[it & 1];
      tc::mbar_arrive_expect_tx(bar, CF::kRawBytes + kPrRopeBox);
      tc::tma_load_2d_hint(raw, &map_lat, static_cast<int>(rank) * 256, y, bar, policy);
      tc::tma_load_2d_hint(raw + CF::kRawCodes, &map_scale, kDc, y, bar, policy);
      tc::tma_load_2d_hint(stages + st * kPrStageBytes + 4 * kPrBox, &map_rope, 32 * static_cast<int>(rank), y, bar,
                           policy);
    } else {
      uint8_t* dst = stages + st * kPrStageBytes;
      tc::mbar_arrive_expect_tx(&S->full[st], kPrStageBytes);
      for (int k = 0; k < 4; ++k)
        tc::tma_load_2d_hint(dst + k * kPrBox, &map_lat, static_cast<int>(rank) * 256 + 64 * k, y, &S->full[st],
                             policy);
      tc::tma_load_2d_hint(dst + 4 * kPrBox, &map_rope, kDc + 32 * static_cast<int>(rank), y, &S->full[st], policy);
    }
  };
  // pool row of tile j of sequence b (or a row outside the pool, which loads zeros, for a bad page id)
  auto tile_row = [&](int b, int j) -> int32_t {
    return cache_tile_row(a.block_table, b, j, a.max_pages, a.page_size, a.num_pages);
  };

  // everything below reads what the absorb kernel wrote
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int32_t* cum = a.plan.cum;
  const uint32_t n_share = static_cast<uint32_t>(a.plan.share_tiles[cl]);

  if (warp == 0) {
    // ---------------------------------------------------------------- cache tiles (both CTAs: own half)
    SegIter si = seg_begin(a.plan, a.batch, cl, ncl);
    int b, j0, j1;
    uint32_t it = 0;
    bool ok = true;
    {
      // the share's first tiles, whose pool rows the plan holds, go out at once
      constexpr uint32_t ring = kF8 ? CF::kRaw : kPrStages;
      static_assert(ring <= kPlanRows, "the plan holds the rows of one ring of tiles");
      n_pre = min(ring, n_share);
      int32_t y = 0;
      if (lane < n_pre) y = a.plan.first_rows[cl * kPlanRows + lane];
      for (uint32_t k = 0; k < n_pre; ++k) {
        const int32_t yk = __shfl_sync(0xffffffffu, y, k);
        if (lane == 0) issue_tile(k, yk);
      }
    }
    while (ok && si.next(cum, a.batch, &b, &j0, &j1)) {
      for (int jc = j0; jc < j1 && ok; jc += 32) {
        int32_t y_l = 0;
        const int jl = jc + lane;
        if (jl < j1) y_l = tile_row(b, jl);
        const int n = min(32, j1 - jc);
        // FP8 cache: the raw ring is two tiles deep, less than HBM's latency at this tile rate, so
        // tiles go to L2 kPrF8Ahead tiles before their loads
        auto l2_tile = [&](int32_t yy) {
          tc::tma_prefetch_l2_2d(&map_lat, static_cast<int>(rank) * 256, yy);
          tc::tma_prefetch_l2_2d(&map_scale, kDc, yy);
          tc::tma_prefetch_l2_2d(&map_rope, 32 * static_cast<int>(rank), yy);
        };
        if (kF8 && lane < kPrF8Ahead && lane < n) l2_tile(y_l);
        for (int u = 0; u < n; ++u) {
          const int32_t y = __shfl_sync(0xffffffffu, y_l, u);
          const int32_t y_ahead = __shfl_sync(0xffffffffu, y_l, (u + kPrF8Ahead) & 31);
          if (kF8 && lane == 0 && u + kPrF8Ahead < n) l2_tile(y_ahead);
          if (lane == 0 && ok && it >= n_pre) {   // tiles before n_pre went out from the plan's rows
            const int st = it % kPrStages;
            if (it >= kPrStages) ok = tc::mbar_wait(&S->empty[st], ((it / kPrStages) - 1) & 1);
            if (kF8 && ok && it >= 2) ok = tc::mbar_wait(&S->raw_empty[it & 1], ((it / 2) - 1) & 1);
            if (ok && pr_aborted(S)) ok = false;
            if (ok) issue_tile(it, y);   // FP8: codes and scales into the raw ring, rope into the stage
          }
          if (lane == 0 && ok) ++it;
          ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
          if (!ok) break;
        }
      }
    }
    it = __shfl_sync(0xffffffffu, it, 0);
    if (it < n_pre) it = n_pre;   // the tiles requested from the plan's rows are in flight too
    if (lane == 0) {
      if (!ok) pr_set_abort(S);
      // copies still in flight must land before the CTA exits
      if (kF8) {
        const uint32_t first = it > 2 ? it - 2 : 0;
        for (uint32_t q = first; q < it; ++q) tc::mbar_wait(&S->raw_full[q & 1], (q / 2) & 1);
      } else {
        const uint32_t first = it > kPrStages ? it - kPrStages : 0;
        for (uint32_t q = first; q < it; ++q) tc::mbar_wait(&S->full[q % kPrStages], (q / kPrStages) & 1);
      }
    }
  } else if (warp == 1 || warp == 5) {
    // ---------------------------------------------------------------- score MMA issuers (even CTA)
    // Scores go out from two threads, warp 1 for even tiles and warp 5 for odd ones, and PVs
    // from a third: the tensor pipe stays fed while one thread waits or loops.
    if (rank == 0 && lane == 0) {
      const uint32_t mine = warp == 1 ? 0u : 1u;   // tile parity this thread issues
      const uint32_t idesc_s = tc::idesc_bf16_f32(256, 128, 0, 0);                // rope part: bf16
      // latent part: bf16, or fp16 (A and B format fields 0) with an FP8 cache
      const uint32_t idesc_l = kF8 ? ((1u << 4) | ((128u >> 3) << 17) | ((256u >> 4) << 24)) : idesc_s;
      const uint64_t qdesc0 = tc::sdesc_sw128(tc::smem_u32(sQ), 16, 1024);       // K-major Q, 128 rows
      const uint64_t kdesc0 = tc::sdesc_sw128(tc::smem_u32(stages), 16, 1024);   // K-major tile, 64 rows
      const uint64_t qrdesc0 = tc::sdesc_sw64(tc::smem_u32(sQ + 4 * kPrQBox), 16, 512);        // rope part of Q
      const uint64_t krdesc0 = tc::sdesc_sw64(tc::smem_u32(stages + 4 * kPrBox), 16, 512);     // rope box, stage 0
      SegIter si = seg_begin(a.plan, a.batch, cl, ncl);
      int b, j0, j1;
      uint32_t it = 0, seg = 0;
      bool ok = true;
      while (ok && si.next(cum, a.batch, &b, &j0, &j1)) {
        ok = tc::mbar_wait(&S->qready, seg & 1);
        for (int j = j0; j < j1 && ok; ++j, ++it) {
          if ((it & 1u) != mine) continue;
          const uint32_t st = it % kPrStages;
          ok = tc::mbar_wait(&S->ready[st], (it / kPrStages) & 1);
          if (ok && it >= 2) ok = tc::mbar_wait(&S->s_free[it & 1], ((it - 2) >> 1) & 1);
          if (!ok || pr_aborted(S)) { ok = false; break; }
          tc::tc_fence_after();
          const uint32_t d = tm + kPrTmS + 128 * (it & 1);
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            const int box = k >> 2, off = (k & 3) * 32;
            const uint64_t ad = qdesc0 + static_cast<uint64_t>((box * kPrQBox + off) >> 4);
            const uint64_t bd = kdesc0 + static_cast<uint64_t>((st * kPrStageBytes + box * kPrBox + off) >> 4);
            tc::mma_ss_pair(d, ad, bd, idesc_l, k > 0 ? 1u : 0u);
          }
#pragma unroll
          for (int k = 0; k < kPrKSteps - 16; ++k) {
            const uint64_t ad = qrdesc0 + static_cast<uint64_t>((k * 32) >> 4);
            const uint64_t bd = krdesc0 + static_cast<uint64_t>((st * kPrStageBytes + k * 32) >> 4);
            tc::mma_ss_pair(d, ad, bd, idesc_s, 1u);
          }
          tc::mma_commit_pair(&S->s_full[it & 1]);
        }
        // the queries may be replaced once both threads' score MMAs of the segment completed
        if (ok) tc::mma_commit_pair(&S->qfree);
        ++seg;
      }
      if (!ok) pr_set_abort(S);
      // every MMA issued so far must complete before TMEM is released
      tc::mma_commit_pair(&S->drain[mine]);
      tc::mbar_wait(&S->drain[mine], 0);
    }
  } else if (warp == 2) {
    // ---------------------------------------------------------------- PV MMA issuer (even CTA)
    if (rank == 0 && lane == 0) {
      // P x V: bf16, or fp16 with an FP8 cache
      const uint32_t idesc_o =
          kF8 ? ((1u << 4) | (1u << 16) | ((256u >> 3) << 17) | ((128u >> 4) << 24)) : tc::idesc_bf16_f32(128, 256, 0, 1);
      const uint64_t vdesc0 = tc::sdesc_sw128(tc::smem_u32(stages), kPrBox, 1024);   // MN-major V
      const uint64_t plo0 = tc::sdesc_sw64(tc::smem_u32(stages + 4 * kPrBox), 16, 512);   // P tokens 0..31, stage 0
      const uint64_t phi0 = tc::sdesc_sw64(tc::smem_u32(sP), 16, 512);                    // P tokens 32..63, buffer 0
      SegIter si = seg_begin(a.plan, a.batch, cl, ncl);
      int b, j0, j1;
      uint32_t it = 0, seg = 0;
      bool ok = true;
      while (ok && si.next(cum, a.batch, &b, &j0, &j1)) {
        for (int j = j0; j < j1 && ok; ++j, ++it) {
          // one barrier per tile parity: the softmax may finish tile it + 1 before this thread
          // has seen tile it complete, but not tile it + 2 (its P buffer is read by PV(it))
          ok = tc::mbar_wait(&S->p_full[it & 1], (it >> 1) & 1);
          if (ok && j == j0 && seg > 0) ok = tc::mbar_wait(&S->o_free, (seg - 1) & 1);
          if (!ok || pr_aborted(S)) { ok = false; break; }
          tc::tc_fence_after();
          const uint32_t st = it % kPrStages;
#pragma unroll
          for (int h = 0; h < 2; ++h) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t ad = kk < 2 ? plo0 + static_cast<uint64_t>((st * kPrStageBytes + kk * 32) >> 4)
                                         : phi0 + static_cast<uint64_t>(((it & 1) * kPrPHalf + (kk - 2) * 32) >> 4);
              const uint64_t bd =
                  vdesc0 + static_cast<uint64_t>((st * kPrStageBytes + 2 * h * kPrBox + kk * 2048) >> 4);
              tc::mma_ss_pair(tm + kPrTmO + 128 * h, ad, bd, idesc_o, (j == j0 && kk == 0) ? 0u : 1u);
            }
          }
          tc::mma_commit_pair(&S->o_done[it & 1]);
          tc::mma_commit_pair(&S->empty[st]);
        }
        ++seg;
      }
      if (!ok) pr_set_abort(S);
      tc::mma_commit_pair(&S->drain[2]);
      tc::mbar_wait(&S->drain[2], 0);
    }
  } else if (warp == 4) {
    // ---------------------------------------------------------------- tile forwarder (both CTAs, bf16)
    // tells the even CTA's MMA issuer that this CTA's half of a tile has landed
    if (!kF8 && lane == 0) {
      const uint32_t ready0 = tc::map_peer(&S->ready[0], 0);
      for (uint32_t it = 0; it < n_share; ++it) {
        const uint32_t st = it % kPrStages;
        if (!tc::mbar_wait(&S->full[st], (it / kPrStages) & 1) || pr_aborted(S)) {
          pr_set_abort(S);
          break;
        }
        tc::mbar_arrive_cluster(ready0 + 8u * st);
      }
    }
  } else if (warp == 3) {
    // ---------------------------------------------------------------- queries of this CTA's 64 heads
    // row r = 32 q + i of each box: head 16 q + (i mod 16), contraction half i / 16 (half A: latent
    // 0..255 and rope 0..31, the even CTA's columns; half B: latent 256..511 and rope 32..63)
    if (lane == 0) {
      const uint32_t qready = tc::map_peer(&S->qready, 0);
      SegIter si = seg_begin(a.plan, a.batch, cl, ncl);
      int b, j0, j1;
      uint32_t seg = 0;
      bool ok = true;
      while (ok && si.next(cum, a.batch, &b, &j0, &j1)) {
        if (seg > 0) ok = tc::mbar_wait(&S->qfree, (seg - 1) & 1);
        if (!ok || pr_aborted(S)) { ok = false; break; }
        tc::mbar_arrive_expect_tx(&S->qfull, kPrQBytes);
        const int row0 = b * kH + 64 * static_cast<int>(rank);
        for (int q = 0; q < 4; ++q)
          for (int half = 0; half < 2; ++half) {
            const int r = 32 * q + 16 * half;   // first of the 16 rows of (quarter q, contraction half)
            for (int k = 0; k < 4; ++k)
              tc::tma_load_2d(sQ + k * kPrQBox + r * 128, &map_q, 256 * half + 64 * k, row0 + 16 * q, &S->qfull);
            tc::tma_load_2d(sQ + 4 * kPrQBox + r * 64, &map_qr, kDc + 32 * half, row0 + 16 * q, &S->qfull);
          }
        ok = tc::mbar_wait(&S->qfull, seg & 1);
        if (!ok) break;
        tc::mbar_arrive_cluster(qready);
        ++seg;
      }
      if (!ok) pr_set_abort(S);
    }
  } else if (kF8 && warp >= 6 + kPrSoftmaxWarps) {
    // ---------------------------------------------------------------- FP8: dequantise (both CTAs)
    // tile it's raw rows -> its bf16 stage: value = E4M3 code x block scale, rounded to bf16,
    // written in the 128-byte swizzled layout of a bf16 tile; 2,048 chunks of 8 values per tile
    const int dt = static_cast<int>(threadIdx.x) - 32 * (6 + kPrSoftmaxWarps);   // 0 .. 127
    const uint32_t ready0 = tc::map_peer(&S->ready[0], 0);
    for (uint32_t it = 0; it < n_share; ++it) {
      const uint32_t st = it % kPrStages;
      if (!tc::mbar_wait(&S->raw_full[it & 1], (it / 2) & 1) || pr_aborted(S)) {
        pr_set_abort(S);
        break;
      }
      const uint8_t* raw = rawb + (it & 1) * CF::kRawBytes;
      uint8_t* stage = stages + st * kPrStageBytes;
#pragma unroll 4
      for (int u = 0; u < (kF8 ? (kTile * 32) / (32 * CF::kDequantWarps + (kF8 ? 0 : 1)) : 0); ++u) {
        const int ci = dt + u * 32 * CF::kDequantWarps;
        const int row = ci >> 5, k = ci & 31;   // chunk k = latent 8k .. 8k + 7 of this CTA's 256
        const uint2 codes = *reinterpret_cast<const uint2*>(raw + row * 256 + 8 * k);
        const float sc = reinterpret_cast<const float*>(raw + CF::kRawCodes + row * 16)[2 * rank + (k >> 4)];
        uint32_t sc2;   // the block scale in both halves of an fp16 pair
        asm("cvt.rn.f16x2.f32 %0, %1, %1;" : "=r"(sc2) : "f"(sc));
        const uint32_t cw[2] = {codes.x, codes.y};
        uint32_t o[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint16_t pair = static_cast<uint16_t>(cw[i >> 1] >> (16 * (i & 1)));
          uint32_t h2;
          asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(pair));
          asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(o[i]) : "r"(h2), "r"(sc2));
        }
        *reinterpret_cast<uint4*>(stage + (k >> 3) * kPrBox + row * 128 + (((k & 7) ^ (row & 7)) << 4)) =
            make_uint4(o[0], o[1], o[2], o[3]);
      }
      tc::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        tc::mbar_arrive(&S->raw_empty[it & 1]);
        tc::mbar_arrive_cluster(ready0 + 8u * st);
      }
    }
  } else {
    // ---------------------------------------------------------------- softmax + segment epilogue
    const int q = warp & 3, w2 = (warp - 6) >> 2;     // lane quarter; token half (32 w2 .. 32 w2 + 31)
    const int hl = 16 * q + (lane & 15);              // this CTA's head whose scores this thread finishes
    const int part = lane >> 4;                       // which 16 of the warp's 32 tokens it finishes
    const uint32_t lane_base = static_cast<uint32_t>(32 * q) << 16;
    const uint32_t s_free0 = tc::map_peer(&S->s_free[0], 0);
    const uint32_t p_full0 = tc::map_peer(&S->p_full[0], 0);
    const uint32_t o_free = tc::map_peer(&S->o_free, 0);
    const float sl = a.scale_log2;
    // O lanes this thread reads or rescales: lane 32 q + lane holds head (32 q + lane) mod 64 of this
    // CTA, latent columns (lane >= 64 ? 256 : 0) + 128 w2 .. + 127 in TMEM columns kPrTmO + 128 w2 ..
    const int o_head = (32 * q + lane) & 63;
    const int o_lat0 = (32 * q + lane >= 64 ? 256 : 0) + 128 * w2;
    const uint32_t t_o = tm + lane_base + kPrTmO + 128 * w2;

    // Every barrier below is passed by all softmax threads the same number of times: a wait
    // that runs out only marks the tile bad, and the threads leave together after a vote.
    SegIter si = seg_begin(a.plan, a.batch, cl, ncl);
    int b, j0, j1;
    uint32_t it = 0;
    bool ok = true;
    while (ok && si.next(cum, a.batch, &b, &j0, &j1)) {
      const int L = a.plan.lens[b];
      const int slot = b + static_cast<int>(cl);
      float m_used = -INFINITY, l = 0.f;
      for (int j = j0; j < j1 && ok; ++j, ++it) {
        const int valid = min(kTile, L - j * kTile);
        bool good = tc::mbar_wait(&S->s_full[it & 1], (it >> 1) & 1) && !pr_aborted(S);
        tc::tc_fence_after();
        float s[16];
        {
          uint32_t ra[32], rb[32];
          const uint32_t t_s = tm + lane_base + kPrTmS + 128 * (it & 1) + 32 * w2;
          tc::tmem_ld32(t_s, ra);        // lanes of half A: this head's half-A scores of 32 tokens
          tc::tmem_ld32(t_s + 64, rb);   // lanes of half B: its half-B scores of the same tokens
          tc::tmem_ld_wait();
          tc::tc_fence_before();
          __syncwarp();
          if (lane == 0) tc::mbar_arrive_cluster_relaxed(s_free0 + 8u * (it & 1));
          // the two halves of a head sit in lanes i and i + 16 of the warp: swap the 16 tokens
          // each of them finishes
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) {
            const uint32_t send = part ? rb[jj] : ra[16 + jj];
            const float r = __uint_as_float(__shfl_xor_sync(0xffffffffu, send, 16));
            s[jj] = __uint_as_float(part ? rb[16 + jj] : ra[jj]) + r;
          }
        }
        const int vt = valid - (32 * w2 + 16 * part);   // valid tokens among this thread's 16
        if (vt < 16) {
#pragma unroll
          for (int jj = 0; jj < 16; ++jj)
            if (jj >= vt) s[jj] = -INFINITY;
        }
        float mx;
        {
          float t4[4];
#pragma unroll
          for (int c = 0; c < 4; ++c) t4[c] = fmaxf(fmaxf(s[c], s[c + 4]), fmaxf(s[c + 8], s[c + 12]));
          mx = fmaxf(fmaxf(t4[0], t4[1]), fmaxf(t4[2], t4[3]));
        }
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
        S->red_max[it & 1][w2][hl] = mx;
        tc::named_sync(1 + q, 64);   // the two warps holding this quarter's heads
        mx = fmaxf(S->red_max[it & 1][0][hl], S->red_max[it & 1][1][hl]) * sl;
        bool resc = false;
        float alpha = 1.f;
        if (m_used == -INFINITY) {
          m_used = mx;
        } else if (mx > m_used + kRescaleThreshold) {
          alpha = tc::ex2_approx(m_used - mx);
          l *= alpha;
          m_used = mx;
          resc = true;
        }
        const float neg_m = -m_used;
        uint32_t p[8];
        float ps[2] = {0.f, 0.f};
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const float e0 = tc::ex2_approx(fmaf(s[2 * c], sl, neg_m)), e1 = tc::ex2_approx(fmaf(s[2 * c + 1], sl, neg_m));
          // l sums the values the PV multiplies: P after its rounding to the MMA type
          if (kF8) {
            const __half2 h = __floats2half2_rn(e0, e1);
            p[c] = *reinterpret_cast<const uint32_t*>(&h);
            const float2 f = __half22float2(h);
            ps[c & 1] += f.x + f.y;
          } else {
            const uint32_t w = tc::pack_bf16(e0, e1);
            p[c] = w;
            ps[c & 1] += bf_lo(w) + bf_hi(w);
          }
        }
        l += ps[0] + ps[1];
        if (lane < 16) S->alpha[it & 1][hl] = alpha;
        // the second half of P goes into the buffer the PV two tiles back read
        if (it > 1) good = tc::mbar_wait(&S->o_done[it & 1], ((it - 2) >> 1) & 1) && good;
        tc::tc_fence_after();
        if (tc::named_sync_or(5, 32 * kPrSoftmaxWarps, resc)) {
          // O must not be in use: the PV of the previous tile completes first
          if (it > 0) good = tc::mbar_wait(&S->o_done[(it - 1) & 1], ((it - 1) >> 1) & 1) && good;
          tc::tc_fence_after();
          // a head's O rows are lanes h and h + 64: the threads on those lanes rescale them
          const float f = S->alpha[it & 1][o_head];
          if (__any_sync(0xffffffffu, f != 1.f)) {
#pragma unroll 1
            for (int c0 = 0; c0 < 128; c0 += 32) {
              uint32_t r[32];
              tc::tmem_ld32(t_o + c0, r);
              tc::tmem_ld_wait();
#pragma unroll
              for (int c = 0; c < 32; ++c) r[c] = __float_as_uint(__uint_as_float(r[c]) * f);
              tc::tmem_st32(t_o + c0, r);
            }
            tc::tmem_st_wait();
          }
        }
        {
          // 64-byte rows, 64-byte swizzle: chunk c of row r sits at chunk c ^ ((r >> 1) & 3)
          uint8_t* prow = (w2 == 0 ? stages + (it % kPrStages) * kPrStageBytes + 4 * kPrBox
                                   : sP + (it & 1) * kPrPHalf) + hl * 64;
          const int c0 = 2 * part, x = (hl >> 1) & 3;   // 16-byte chunks of the row: 8 tokens each
          *reinterpret_cast<uint4*>(prow + ((c0 ^ x) << 4)) = make_uint4(p[0], p[1], p[2], p[3]);
          *reinterpret_cast<uint4*>(prow + (((c0 + 1) ^ x) << 4)) = make_uint4(p[4], p[5], p[6], p[7]);
        }
        // rows past the sequence end must not reach PV as NaN/Inf garbage
        if (valid < kTile) {
          uint8_t* stage = stages + (it % kPrStages) * kPrStageBytes;
          const int nrow = kTile - valid;
          for (int idx = threadIdx.x - 192; idx < nrow * 4 * 8; idx += 32 * kPrSoftmaxWarps) {
            const int box = idx / (nrow * 8), rem = idx % (nrow * 8);
            const int row = valid + rem / 8, ch = rem % 8;
            *reinterpret_cast<uint4*>(stage + box * kPrBox + row * 128 + ch * 16) = make_uint4(0, 0, 0, 0);
          }
        }
        tc::fence_proxy_async_smem();
        tc::tc_fence_before();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive_cluster(p_full0 + 8u * (it & 1));
        ok = tc::named_sync_and(5, 32 * kPrSoftmaxWarps, good);
      }
      if (!ok) break;
      // ---- segment epilogue: unnormalised O of this CTA's 64 heads, m and l
      bool good = tc::mbar_wait(&S->o_done[(it - 1) & 1], ((it - 1) >> 1) & 1);
      tc::tc_fence_after();
      {
        const int gh = 64 * static_cast<int>(rank) + o_head;
#pragma unroll 1
        for (int c0 = 0; c0 < 128; c0 += 32) {
          uint32_t r[32];
          tc::tmem_ld32(t_o + c0, r);
          tc::tmem_ld_wait();
#pragma unroll
          for (int u = 0; u < 8; ++u)
            *reinterpret_cast<uint4*>(a.part_o + parto_index(slot, (o_lat0 + c0) / 4 + u, gh)) =
                make_uint4(r[4 * u], r[4 * u + 1], r[4 * u + 2], r[4 * u + 3]);
        }
      }
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive_cluster(o_free);
      const float lw = l + __shfl_xor_sync(0xffffffffu, l, 16);
      S->red_l[w2][hl] = lw;
      tc::named_sync(1 + q, 64);
      if (w2 == 0 && part == 0) {
        float2* ml = reinterpret_cast<float2*>(a.part_ml) + static_cast<int64_t>(slot) * kH +
                     64 * static_cast<int>(rank) + hl;
        *ml = make_float2(m_used, S->red_l[0][hl] + S->red_l[1][hl]);
      }
      ok = tc::named_sync_and(5, 32 * kPrSoftmaxWarps, good);
    }
    if (!ok) pr_set_abort(S);
  }
  // ---------------------------------------------------------------- teardown
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  tc::tc_fence_before();
  __syncthreads();
  tc::cluster_sync();   // no pair MMA, remote arrive or TMEM access of the other CTA is left
  tc::tc_fence_after();
  if (warp == 1) tc::tmem_dealloc_pair<512>(tm);
}

}  // namespace tcd
}  // namespace mla
