// Prefill of MLA over a paged latent cache in the non-absorbed form
// (DeepSeek-V2 report, section 2.1.2: keys and values are up-projections of
// the cached latent, k_{j,i} = W_UK,i c_j and v_{j,i} = W_UV,i c_j;
// section 2.1.3: the full key is [k_{j,i} ; k^R_j], the full query
// [q^C_i ; q^R_i]; section 2.1.1: causal softmax attention per head).
//
// A prompt token attends to every row of its sequence up to its own
// position, so a prompt of n tokens costs n^2/2 score dot products per head:
// the work is a dense contraction, not a stream of cache bytes. The
// per-head keys and values are therefore materialised once per prompt
// (d_h + d_h values per head and token, 2 x 128 x 128 x 2 bytes = 64 KB per
// token for the DeepSeek-V2 shape), then read by a causal attention kernel
// whose scores have the contraction width d_h + d_h^R = 192 instead of the
// 576 of the absorbed form the decode uses.
//
//   kv_up_kernel:        [rows x 512] latent tiles (gathered from the pages) x
//                        [W_UK ; W_UV]^T ([512 x 32768]) -> K_nope (bf16, the
//                        query's type, for the score MMA) and V (fp16)
//                        [B * L_pad, 128 heads x 128]. Pair MMAs on two CTAs
//                        (M = 256 rows, N = 256, K = 16); fp32 accumulators in
//                        TMEM, two of them so the epilogue of one column
//                        tile overlaps the MMAs of the next.
//   prefill_attn_kernel: per (sequence, head, 256 query rows) on a CTA pair:
//                        S = Q K^T (pair MMA, M = 256, N = 128 keys,
//                        K = 192, bf16), online softmax with a causal mask,
//                        O += P V (pair MMA, M = 256, N = 128, K = 128 keys,
//                        fp16, P from TMEM), out = O / l in fp32.
//
// V and P are fp16 rather than bf16: with few keys (the first tokens of a
// prompt) a weighted sum does not average the rounding of its terms away,
// and fp16's 11 significant bits keep that rounding 8x smaller. Both stay in
// range: P <= 2^8 (the lazy rescale bound) and V = W_UV c is of the order of
// the latent's unit RMS times the weights' norm.
#pragma once

#include "common.cuh"
#include "decode_tc.cuh"
#include "tc.cuh"

namespace mla {
namespace tcd {

// Instruction descriptor of tcgen05.mma kind::f16 with fp16 A and B and an fp32 D (the A and B
// format fields are 0 for fp16); M x N tile, a_mn / b_mn select MN-major operands.
__host__ __device__ constexpr uint32_t idesc_f16_f32(uint32_t M, uint32_t N, uint32_t a_mn, uint32_t b_mn) {
  return (1u << 4) | (a_mn << 15) | (b_mn << 16) | ((N >> 3) << 17) | ((M >> 4) << 24);
}

// Two fp32 values -> fp16x2 (round to nearest even), `lo` in the low half.
__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Starts bringing the box at (x, y) of a tensor into L2 (no shared memory, no completion).
__device__ __forceinline__ void pf_prefetch_2d(const CUtensorMap* map, int32_t x, int32_t y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y)
               : "memory");
}

constexpr int kPfRows = 128;              // query rows and key rows per tile
constexpr int kPfBox = kPfRows * 128;     // one TMA box: 128 rows x 64 bf16 (128-byte swizzle) = 16 KB
constexpr int kPfHalfBox = 64 * 128;      // 64 rows x 64 bf16 = 8 KB
constexpr int kPfWidthKV = 2 * kH * kDh;  // columns of [K_nope | V] per token: 32768

// ------------------------------------------------------------------ kv_up_kernel
// A cluster of two CTAs computes two 128-row tiles (CTA r: row tile 2 p + r) against the same
// 256 weight rows with pair MMAs (M = 256, N = 256): each CTA streams only its 128 of the 256 weight
// rows, 16 KB per 64-column chunk where a CTA working alone would stream 32 KB; the weight stream
// is what one SM's tensor-memory-access unit (about 34 bytes per cycle) could not keep up with.
constexpr int kKvNt = 256;                            // weight rows (output columns) per pair MMA tile
constexpr int kKvTilesPerItem = 16;                   // column tiles a work item covers
constexpr int kKvGroups = kPfWidthKV / kKvNt / kKvTilesPerItem;   // 8 items per pair of row tiles
constexpr int kKvStages = 4;                          // weight chunk ring: 128 rows x 64 columns = 16 KB each
constexpr int kKvABytes = 8 * kPfBox;                 // latent tile: 8 boxes of 128 rows x 64 columns = 128 KB
constexpr int kKvBBytes = (kKvNt / 2) * 128;          // 16 KB
constexpr int kKvThreads = 32 * 7;                    // producer, MMA issuer, 4 epilogue warps, forwarder

struct KvUpSmem {
  uint64_t a_full, a_empty, a_ready;
  uint64_t b_full[kKvStages], b_empty[kKvStages], b_ready[kKvStages];
  uint64_t d_full[2], d_free[2];
  uint64_t drain;
  uint32_t tmem_base;
  int32_t abort_flag;
};
constexpr size_t kKvSmem = 1024 + kKvABytes + static_cast<size_t>(kKvStages) * kKvBBytes + sizeof(KvUpSmem);

struct KvUpArgs {
  const int32_t* block_table;   // [B, max_pages] or NULL (contiguous pages b * max_pages + p)
  const int32_t* seq_lens;      // [B]
  const uint16_t* pool;         // [num_pages * page_size, 576] bf16
  uint16_t* k_buf;              // [B * lpad, 128 * 128] bf16
  uint16_t* v_buf;              // same, fp16
  uint16_t* kr_buf;             // [B * lpad, 64] bf16: the shared rope key of every row
  int64_t num_pages;
  int batch, max_pages, page_size, max_seq_len, lpad;
};

__device__ __forceinline__ int clamp_len(int L, int max_len) { return L < 0 ? 0 : (L > max_len ? max_len : L); }

// Pool row of the 64 rows of sequence b that start at token `tok` (a multiple of 64), or a
// coordinate outside the pool (the TMA then fills zeros) when the rows lie past the
// sequence's length; a page id outside the pool for rows the sequence holds is flagged.
__device__ __forceinline__ int32_t pf_pool_row(const int32_t* block_table, int64_t num_pages, int max_pages,
                                               int page_size, int b, int64_t tok, int L) {
  if (tok >= L) return -4 * kPfRows;
  const int pg = static_cast<int>(tok / page_size);
  int64_t page = -1;
  if (pg < max_pages)
    page = block_table ? block_table[static_cast<int64_t>(b) * max_pages + pg]
                       : static_cast<int64_t>(b) * max_pages + pg;
  if (page < 0 || page >= num_pages) {
    flag_error(ERR_BIT_BOUNDS);
    return -4 * kPfRows;
  }
  return static_cast<int32_t>(page * page_size + tok % page_size);
}

__device__ __forceinline__ bool kv_aborted(const KvUpSmem* s) {
  return *reinterpret_cast<const volatile int32_t*>(&s->abort_flag) != 0;
}
__device__ __forceinline__ void kv_set_abort(KvUpSmem* s) { *reinterpret_cast<volatile int32_t*>(&s->abort_flag) = 1; }

// Work item i: row tiles 2 p and 2 p + 1 (row tile t: rows 128 (t / B) .. of sequence t mod B),
// column tiles [16 g, 16 g + 16). A row tile past its sequence's length is dead: its CTA still takes
// part in the pair MMAs (its half of the weights) but loads zeros and writes nothing; an item whose
// two tiles are both dead is skipped.
struct KvItem {
  int b, r, g;
  bool live, any;
};
__device__ __forceinline__ KvItem kv_item(const KvUpArgs& a, int64_t i, uint32_t rank) {
  const int64_t n_rt = static_cast<int64_t>(a.batch) * (a.lpad / kPfRows);
  KvItem it;
  it.g = static_cast<int>(i % kKvGroups);
  const int64_t p = i / kKvGroups;
  it.any = false;
  it.b = 0;
  it.r = 0;
  it.live = false;
  for (uint32_t q = 0; q < 2; ++q) {
    const int64_t rt = 2 * p + q;
    if (rt >= n_rt) continue;
    const int b = static_cast<int>(rt % a.batch), r = static_cast<int>(rt / a.batch);
    const bool lv = static_cast<int64_t>(r) * kPfRows < clamp_len(a.seq_lens[b], a.max_seq_len);
    it.any = it.any || lv;
    if (q == rank) {
      it.b = b;
      it.r = r;
      it.live = lv;
    }
  }
  return it;
}

// map_lat: the pool [rows, 576] bf16, boxes of 64 rows x 64 columns, 128-byte swizzle.
// map_wuk / map_wuv: W_UK / W_UV as [128 * 128, 512] bf16, boxes of 128 rows x 64 columns.
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kKvThreads, 1)
    kv_up_kernel(const __grid_constant__ CUtensorMap map_lat, const __grid_constant__ CUtensorMap map_wuk,
                 const __grid_constant__ CUtensorMap map_wuv, KvUpArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* sA = sm;
  uint8_t* sB = sm + kKvABytes;
  KvUpSmem* S = reinterpret_cast<KvUpSmem*>(sB + kKvStages * kKvBBytes);
  const uint32_t rank = tc::cluster_ctarank();
  const uint32_t cl = tc::cluster_id_x(), ncl = tc::n_clusters_x();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    tc::mbar_init(&S->a_full, 1);
    tc::mbar_init(&S->a_empty, 1);
    tc::mbar_init(&S->a_ready, 2);
    for (int s = 0; s < kKvStages; ++s) {
      tc::mbar_init(&S->b_full[s], 1);
      tc::mbar_init(&S->b_empty[s], 1);
      tc::mbar_init(&S->b_ready[s], 2);
    }
    for (int d = 0; d < 2; ++d) {
      tc::mbar_init(&S->d_full[d], 1);
      tc::mbar_init(&S->d_free[d], 8);   // the 4 epilogue warps of both CTAs
    }
    tc::mbar_init(&S->drain, 1);
    S->abort_flag = 0;
    tc::fence_mbar_init();
    tc::tma_prefetch_map(&map_lat);
    tc::tma_prefetch_map(&map_wuk);
    tc::tma_prefetch_map(&map_wuv);
  }
  if (warp == 1) tc::tmem_alloc_pair<512>(&S->tmem_base);
  tc::tc_fence_before();
  tc::cluster_sync();
  tc::tc_fence_after();
  const uint32_t tm = S->tmem_base;
  // the pool rows and the lengths come from the kernels ahead of this one on the stream
  asm volatile("griddepcontrol.wait;" ::: "memory");

  const int64_t n_items = ((static_cast<int64_t>(a.lpad / kPfRows) * a.batch + 1) / 2) * kKvGroups;
  if (warp == 0) {
    // ------------------------------------------------------------ producer (both CTAs: own tile, own weight half)
    if (lane == 0) {
      uint32_t n = 0, c = 0;   // items and weight chunks loaded
      bool ok = true;
      for (int64_t i = cl; i < n_items && ok; i += ncl) {
        const KvItem it = kv_item(a, i, rank);
        if (!it.any) continue;
        if (n > 0) ok = tc::mbar_wait(&S->a_empty, (n - 1) & 1);
        if (!ok || kv_aborted(S)) { ok = false; break; }
        const int L = it.live ? clamp_len(a.seq_lens[it.b], a.max_seq_len) : 0;
        tc::mbar_arrive_expect_tx(&S->a_full, kKvABytes);
        for (int h = 0; h < 2; ++h) {
          const int64_t tok = static_cast<int64_t>(it.r) * kPfRows + 64 * h;
          const int32_t y = pf_pool_row(a.block_table, a.num_pages, a.max_pages, a.page_size, it.b, tok, L);
          for (int k = 0; k < 8; ++k)
            tc::tma_load_2d(sA + k * kPfBox + h * kPfHalfBox, &map_lat, 64 * k, y, &S->a_full);
        }
        ++n;
        for (int t = 0; t < kKvTilesPerItem && ok; ++t) {
          const int n0 = (it.g * kKvTilesPerItem + t) * kKvNt + (kKvNt / 2) * static_cast<int>(rank);
          const CUtensorMap* mw = n0 < kH * kDh ? &map_wuk : &map_wuv;
          const int row = n0 < kH * kDh ? n0 : n0 - kH * kDh;
          for (int kc = 0; kc < 8; ++kc, ++c) {
            const int st = c % kKvStages;
            if (c >= kKvStages) ok = tc::mbar_wait(&S->b_empty[st], ((c / kKvStages) - 1) & 1);
            if (!ok) break;
            tc::mbar_arrive_expect_tx(&S->b_full[st], kKvBBytes);
            tc::tma_load_2d(sB + st * kKvBBytes, mw, 64 * kc, row, &S->b_full[st]);
          }
        }
      }
      if (!ok) kv_set_abort(S);
      // copies in flight land before the CTA exits
      if (n > 0) tc::mbar_wait(&S->a_full, (n - 1) & 1);
      const uint32_t first = c > kKvStages ? c - kKvStages : 0;
      for (uint32_t q = first; q < c; ++q) tc::mbar_wait(&S->b_full[q % kKvStages], (q / kKvStages) & 1);
    }
  } else if (warp == 6) {
    // ------------------------------------------------------------ forwarder (both CTAs)
    // tells the even CTA's MMA issuer when this CTA's tile and weight chunks have landed, in the
    // order the producer requested them
    if (lane == 0) {
      const uint32_t a_ready0 = tc::map_peer(&S->a_ready, 0);
      const uint32_t b_ready0 = tc::map_peer(&S->b_ready[0], 0);
      uint32_t n = 0, c = 0;
      bool ok = true;
      for (int64_t i = cl; i < n_items && ok; i += ncl) {
        const KvItem it = kv_item(a, i, rank);
        if (!it.any) continue;
        ok = tc::mbar_wait(&S->a_full, n & 1);
        if (!ok || kv_aborted(S)) { ok = false; break; }
        tc::mbar_arrive_cluster(a_ready0);
        ++n;
        for (int q = 0; q < kKvTilesPerItem * 8 && ok; ++q, ++c) {
          const int st = c % kKvStages;
          ok = tc::mbar_wait(&S->b_full[st], (c / kKvStages) & 1);
          if (!ok || kv_aborted(S)) { ok = false; break; }
          tc::mbar_arrive_cluster(b_ready0 + 8u * st);
        }
      }
      if (!ok) kv_set_abort(S);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (even CTA)
    if (rank == 0 && lane == 0) {
      const uint32_t idesc = tc::idesc_bf16_f32(256, kKvNt, 0, 0);
      const uint64_t adesc0 = tc::sdesc_sw128(tc::smem_u32(sA), 16, 1024);
      const uint64_t bdesc0 = tc::sdesc_sw128(tc::smem_u32(sB), 16, 1024);
      uint32_t n = 0, c = 0, d = 0;   // items, weight chunks, column tiles
      bool ok = true;
      for (int64_t i = cl; i < n_items && ok; i += ncl) {
        const KvItem it = kv_item(a, i, rank);
        if (!it.any) continue;
        ok = tc::mbar_wait(&S->a_ready, n & 1);
        for (int t = 0; t < kKvTilesPerItem && ok; ++t, ++d) {
          const uint32_t buf = d & 1;
          if (d >= 2) ok = tc::mbar_wait(&S->d_free[buf], ((d >> 1) - 1) & 1);
          for (int kc = 0; kc < 8 && ok; ++kc, ++c) {
            const int st = c % kKvStages;
            ok = tc::mbar_wait(&S->b_ready[st], (c / kKvStages) & 1);
            if (!ok || kv_aborted(S)) { ok = false; break; }
            tc::tc_fence_after();
#pragma unroll
            for (int k = 0; k < 4; ++k)
              tc::mma_ss_pair(tm + 256 * buf, adesc0 + static_cast<uint64_t>((kc * kPfBox + 32 * k) >> 4),
                              bdesc0 + static_cast<uint64_t>((st * kKvBBytes + 32 * k) >> 4), idesc,
                              (kc == 0 && k == 0) ? 0u : 1u);
            tc::mma_commit_pair(&S->b_empty[st]);
          }
          if (ok) tc::mma_commit_pair(&S->d_full[buf]);
        }
        if (ok) tc::mma_commit_pair(&S->a_empty);
        ++n;
      }
      if (!ok) kv_set_abort(S);
      tc::mma_commit_pair(&S->drain);
      tc::mbar_wait(&S->drain, 0);
    }
  } else {
    // ------------------------------------------------------------ epilogue (both CTAs): TMEM -> K_nope / V rows
    const int q = warp & 3;   // TMEM lane quarter of this warp
    const int row = 32 * q + lane;
    const uint32_t d_free0 = tc::map_peer(&S->d_free[0], 0);
    uint32_t d = 0;
    bool ok = true;
    for (int64_t i = cl; i < n_items && ok; i += ncl) {
      const KvItem it = kv_item(a, i, rank);
      if (!it.any) continue;
      const int L = it.live ? clamp_len(a.seq_lens[it.b], a.max_seq_len) : 0;
      const bool valid = static_cast<int64_t>(it.r) * kPfRows + row < L;   // rows past L are written as zeros
      const int64_t grow = static_cast<int64_t>(it.b) * a.lpad + static_cast<int64_t>(it.r) * kPfRows + row;
      if (it.g == 0 && it.live) {
        // the row's rope key, copied beside K_nope so that the attention kernel reads whole
        // 128-row tiles without page lookups (zeros past the sequence's length)
        uint4 rv[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) rv[u] = make_uint4(0u, 0u, 0u, 0u);
        const int64_t tok0 = static_cast<int64_t>(it.r) * kPfRows + (row & ~63);
        const int32_t prow =
            valid ? pf_pool_row(a.block_table, a.num_pages, a.max_pages, a.page_size, it.b, tok0, L) : -1;
        if (prow >= 0) {
          const uint4* src = reinterpret_cast<const uint4*>(a.pool + static_cast<int64_t>(prow + (row & 63)) * kRow + kDc);
#pragma unroll
          for (int u = 0; u < 8; ++u) rv[u] = src[u];
        }
        uint4* dr = reinterpret_cast<uint4*>(a.kr_buf + grow * kDr);
#pragma unroll
        for (int u = 0; u < 8; ++u) dr[u] = rv[u];
      }
      for (int t = 0; t < kKvTilesPerItem; ++t, ++d) {
        const uint32_t buf = d & 1;
        bool good = tc::mbar_wait(&S->d_full[buf], (d >> 1) & 1);
        good = __all_sync(0xffffffffu, good);
        if (!good) { ok = false; break; }
        tc::tc_fence_after();
        if (it.live) {
          const int n0 = (it.g * kKvTilesPerItem + t) * kKvNt;
          uint16_t* dst = (n0 < kH * kDh ? a.k_buf + n0 : a.v_buf + (n0 - kH * kDh)) + grow * (kH * kDh);
#pragma unroll 1
          for (int c0 = 0; c0 < kKvNt; c0 += 32) {
            uint32_t r[32];
            tc::tmem_ld32(tm + (static_cast<uint32_t>(32 * q) << 16) + 256 * buf + c0, r);
            tc::tmem_ld_wait();
            uint32_t w[16];
            if (n0 < kH * kDh) {
#pragma unroll
              for (int u = 0; u < 16; ++u)
                w[u] = valid ? tc::pack_bf16(__uint_as_float(r[2 * u]), __uint_as_float(r[2 * u + 1])) : 0u;
            } else {
#pragma unroll
              for (int u = 0; u < 16; ++u)
                w[u] = valid ? pack_f16(__uint_as_float(r[2 * u]), __uint_as_float(r[2 * u + 1])) : 0u;
            }
            uint4* o = reinterpret_cast<uint4*>(dst + c0);
#pragma unroll
            for (int u = 0; u < 4; ++u) o[u] = make_uint4(w[4 * u], w[4 * u + 1], w[4 * u + 2], w[4 * u + 3]);
          }
        }
        tc::tc_fence_before();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive_cluster(d_free0 + 8u * buf);
      }
    }
    if (!ok) kv_set_abort(S);
  }
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  tc::tc_fence_before();
  __syncthreads();
  tc::cluster_sync();   // no pair MMA, remote arrive or TMEM access of the other CTA is left
  tc::tc_fence_after();
  if (warp == 1) tc::tmem_dealloc_pair<512>(tm);
}

// ------------------------------------------------------------------ prefill_attn_kernel
// A cluster of two CTAs works on 256 query rows of one (sequence, head): CTA r holds rows
// 128 r .. 128 r + 127 and issues nothing; the even CTA issues pair MMAs (tcgen05 cta_group::2) for
// both. In the score MMA each CTA supplies half of the key tile's rows (64 keys) and in the PV MMA
// half of the value columns (64 of d_h), so a CTA loads 40 KB per 128-key tile where one CTA
// working alone loads 80 KB: a tile load is then shorter than the tile's MMAs (one SM's tensor
// memory access pipe moves about 34 bytes per cycle).
constexpr int kPaKStages = 4;                         // ring depth of key tiles
constexpr int kPaVStages = 4;                         // ring depth of value tiles
constexpr int kPaQBytes = 3 * kPfBox;                 // this CTA's 128 query rows: q_nope (2 boxes), q_rope
constexpr int kPaKBytes = 3 * kPfHalfBox;             // this CTA's 64 keys: k_nope (2 boxes), rope key (1 box)
constexpr int kPaVBytes = kPfBox;                     // all 128 keys x this CTA's 64 value columns
constexpr int kPaSoftmaxWarps = 8;
constexpr int kPaL2Ahead = 4;                         // tiles a key/value tile is prefetched to L2 ahead of its load
constexpr int kPaThreads = 32 * (kPaSoftmaxWarps + 4);   // softmax 0-7, producer 8, S MMAs 9, forwarder 10, PV MMAs 11
constexpr uint32_t kPaTmS = 0;     // score buffers: columns 0 and 128
constexpr uint32_t kPaTmP = 256;   // P buffers (fp16 pairs): columns 256 and 320
constexpr uint32_t kPaTmO = 384;   // O: 128 columns

struct PaSmem {
  uint64_t q_full, q_empty, q_ready;
  uint64_t k_full[kPaKStages], k_empty[kPaKStages], k_ready[kPaKStages];
  uint64_t v_full[kPaVStages], v_empty[kPaVStages], v_ready[kPaVStages];
  uint64_t s_full[2], s_free[2], p_full[2], o_done[2];
  uint64_t drain[2];
  float red_max[2][2][kPfRows];   // [tile parity][column half][row]
  float red_l[2][kPfRows];        // [column half][row]
  uint32_t tmem_base;
  int32_t abort_flag;
};
constexpr size_t kPaSmem = 1024 + kPaQBytes + static_cast<size_t>(kPaKStages) * kPaKBytes +
                           static_cast<size_t>(kPaVStages) * kPaVBytes + sizeof(PaSmem);

// Pair MMA with A (P) in tensor memory: each CTA's rows at the same TMEM address.
__device__ __forceinline__ void mma_ts_pair(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

struct PrefillArgs {
  const int32_t* block_table;
  const int32_t* seq_lens;   // [B] rows of each sequence in the cache, its new tokens included
  const int32_t* q_start;    // [B + 1] new tokens of sequence b are rows q_start[b] .. q_start[b+1]-1
  float* out;                // [T, 128, 128] fp32
  int64_t num_pages;
  int batch, max_pages, page_size, max_seq_len, lpad, n_tokens, qp_max;
  float scale_log2;
};

// Unit u: query rows 256 t .. 256 t + 255 of (sequence b, head). Units of one (sequence, head) are
// consecutive (longest first), so the clusters working at one time share a few heads' K and V in L2.
struct PaUnit {
  int b, t, head, nk, n, p0, q0;   // q0: first query row of the pair (this CTA adds 128 rank)
  bool live;
};
__device__ __forceinline__ PaUnit pa_unit(const PrefillArgs& a, int64_t u) {
  PaUnit x;
  const int64_t grp = u / a.qp_max;
  x.t = a.qp_max - 1 - static_cast<int>(u % a.qp_max);
  x.b = static_cast<int>(grp / kH);
  x.head = static_cast<int>(grp % kH);
  const int L = clamp_len(a.seq_lens[x.b], a.max_seq_len);
  const int s0 = a.q_start[x.b], s1 = a.q_start[x.b + 1];
  x.n = s1 - s0;
  x.q0 = s0 + 2 * kPfRows * x.t;
  x.p0 = L - x.n;
  x.live = x.n > 0 && x.n <= L && s0 >= 0 && s1 <= a.n_tokens && 2 * kPfRows * x.t < x.n;
  if (!x.live) {
    if (x.t == 0 && x.head == 0 && (x.n < 0 || x.n > L || s0 < 0 || s1 > a.n_tokens)) flag_error(ERR_BIT_BOUNDS);
    x.nk = 0;
    return x;
  }
  const int last = x.p0 + min(x.n, 2 * kPfRows * (x.t + 1)) - 1;   // position of the pair's last query row
  x.nk = last / kPfRows + 1;
  return x;
}

__device__ __forceinline__ bool pa_aborted(const PaSmem* s) {
  return *reinterpret_cast<const volatile int32_t*>(&s->abort_flag) != 0;
}
__device__ __forceinline__ void pa_set_abort(PaSmem* s) { *reinterpret_cast<volatile int32_t*>(&s->abort_flag) = 1; }

// map_qn: q_nope [T, 128 * 128] bf16 and map_qr: q_rope [T, 128 * 64], boxes of 128 rows; map_k: K_nope
// [B * lpad, 128 * 128] bf16 and map_kr: the rope keys [B * lpad, 64], boxes of 64 rows; map_v: V (fp16)
// [B * lpad, 128 * 128], boxes of 128 rows. Every box is 64 columns wide with the 128-byte swizzle.
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kPaThreads, 1)
    prefill_attn_kernel(const __grid_constant__ CUtensorMap map_qn, const __grid_constant__ CUtensorMap map_qr,
                        const __grid_constant__ CUtensorMap map_k, const __grid_constant__ CUtensorMap map_v,
                        const __grid_constant__ CUtensorMap map_kr, PrefillArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* sQ = sm;
  uint8_t* kst0 = sm + kPaQBytes;                      // key tiles (this CTA's 64 keys)
  uint8_t* vst0 = kst0 + kPaKStages * kPaKBytes;       // value tiles (this CTA's 64 columns)
  PaSmem* S = reinterpret_cast<PaSmem*>(vst0 + kPaVStages * kPaVBytes);
  const uint32_t rank = tc::cluster_ctarank();
  const uint32_t cl = tc::cluster_id_x(), ncl = tc::n_clusters_x();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    tc::mbar_init(&S->q_full, 1);
    tc::mbar_init(&S->q_empty, 1);
    tc::mbar_init(&S->q_ready, 2);
    for (int s = 0; s < kPaKStages; ++s) {
      tc::mbar_init(&S->k_full[s], 1);
      tc::mbar_init(&S->k_empty[s], 1);
      tc::mbar_init(&S->k_ready[s], 2);
    }
    for (int s = 0; s < kPaVStages; ++s) {
      tc::mbar_init(&S->v_full[s], 1);
      tc::mbar_init(&S->v_empty[s], 1);
      tc::mbar_init(&S->v_ready[s], 2);
    }
    for (int s = 0; s < 2; ++s) {
      tc::mbar_init(&S->s_full[s], 1);
      tc::mbar_init(&S->s_free[s], 2 * kPaSoftmaxWarps);
      tc::mbar_init(&S->p_full[s], 2 * kPaSoftmaxWarps);
      tc::mbar_init(&S->o_done[s], 1);
    }
    tc::mbar_init(&S->drain[0], 1);
    tc::mbar_init(&S->drain[1], 1);
    S->abort_flag = 0;
    tc::fence_mbar_init();
    tc::tma_prefetch_map(&map_qn);
    tc::tma_prefetch_map(&map_qr);
    tc::tma_prefetch_map(&map_k);
    tc::tma_prefetch_map(&map_v);
    tc::tma_prefetch_map(&map_kr);
  }
  if (warp == kPaSoftmaxWarps + 1) tc::tmem_alloc_pair<512>(&S->tmem_base);
  tc::tc_fence_before();
  tc::cluster_sync();
  tc::tc_fence_after();
  const uint32_t tm = S->tmem_base;
  // K_nope, V and the rope keys come from the kv_up kernel ahead of this one
  asm volatile("griddepcontrol.wait;" ::: "memory");

  const int64_t n_units = static_cast<int64_t>(a.batch) * kH * a.qp_max;
  const int row_off = kPfRows * static_cast<int>(rank);   // this CTA's first row within the pair's 256
  if (warp == kPaSoftmaxWarps) {
    // ------------------------------------------------------------ producer (both CTAs: own halves)
    // key tile g goes out as soon as the score MMA of tile g - kPaKStages completed; value tile
    // g - 1 after it, once the PV of tile g - 1 - kPaVStages completed
    if (lane == 0) {
      uint32_t n = 0, g = 0, gv = 0;   // units, key tiles and value tiles loaded
      int32_t pend_y = 0, pend_x = 0;  // value tile waiting to go out (when gv < g)
      bool ok = true;
      auto load_v = [&]() -> bool {
        const int st = gv % kPaVStages;
        if (gv >= kPaVStages && !tc::mbar_wait(&S->v_empty[st], ((gv / kPaVStages) - 1) & 1)) return false;
        tc::mbar_arrive_expect_tx(&S->v_full[st], kPaVBytes);
        tc::tma_load_2d(vst0 + st * kPaVBytes, &map_v, pend_x, pend_y, &S->v_full[st]);
        ++gv;
        return true;
      };
      for (int64_t u = cl; u < n_units && ok; u += ncl) {
        const PaUnit x = pa_unit(a, u);
        if (!x.live) continue;
        if (n > 0) ok = tc::mbar_wait(&S->q_empty, (n - 1) & 1);
        if (!ok || pa_aborted(S)) { ok = false; break; }
        const int qrow = x.q0 + row_off;
        tc::mbar_arrive_expect_tx(&S->q_full, kPaQBytes);
        tc::tma_load_2d(sQ, &map_qn, x.head * kDh, qrow, &S->q_full);
        tc::tma_load_2d(sQ + kPfBox, &map_qn, x.head * kDh + 64, qrow, &S->q_full);
        tc::tma_load_2d(sQ + 2 * kPfBox, &map_qr, x.head * kDr, qrow, &S->q_full);
        ++n;
        PaUnit y;   // this cluster's next unit: its queries and first tiles go to L2 early
        y.live = false;
        for (int64_t w = u + ncl; w < n_units; w += ncl) {
          y = pa_unit(a, w);
          if (!y.live) continue;
          pf_prefetch_2d(&map_qn, y.head * kDh, y.q0 + row_off);
          pf_prefetch_2d(&map_qn, y.head * kDh + 64, y.q0 + row_off);
          pf_prefetch_2d(&map_qr, y.head * kDr, y.q0 + row_off);
          break;
        }
        auto l2_tile = [&](const PaUnit& z, int jj) {
          const int64_t r0 = static_cast<int64_t>(z.b) * a.lpad + static_cast<int64_t>(jj) * kPfRows;
          pf_prefetch_2d(&map_k, z.head * kDh, static_cast<int32_t>(r0 + 64 * rank));
          pf_prefetch_2d(&map_k, z.head * kDh + 64, static_cast<int32_t>(r0 + 64 * rank));
          pf_prefetch_2d(&map_kr, 0, static_cast<int32_t>(r0 + 64 * rank));
          pf_prefetch_2d(&map_v, z.head * kDh + 64 * static_cast<int>(rank), static_cast<int32_t>(r0));
        };
        if (n == 1)
          for (int jj = 0; jj < kPaL2Ahead && jj < x.nk; ++jj) l2_tile(x, jj);
        const int64_t krow0 = static_cast<int64_t>(x.b) * a.lpad;
        for (int j = 0; j < x.nk && ok; ++j, ++g) {
          if (j + kPaL2Ahead < x.nk)
            l2_tile(x, j + kPaL2Ahead);
          else if (y.live && j + kPaL2Ahead - x.nk < y.nk)
            l2_tile(y, j + kPaL2Ahead - x.nk);
          const int st = g % kPaKStages;
          if (g >= kPaKStages) ok = tc::mbar_wait(&S->k_empty[st], ((g / kPaKStages) - 1) & 1);
          if (!ok) break;
          uint8_t* kst = kst0 + st * kPaKBytes;
          const int32_t yk = static_cast<int32_t>(krow0 + static_cast<int64_t>(j) * kPfRows + 64 * rank);
          tc::mbar_arrive_expect_tx(&S->k_full[st], kPaKBytes);
          tc::tma_load_2d(kst, &map_k, x.head * kDh, yk, &S->k_full[st]);
          tc::tma_load_2d(kst + kPfHalfBox, &map_k, x.head * kDh + 64, yk, &S->k_full[st]);
          tc::tma_load_2d(kst + 2 * kPfHalfBox, &map_kr, 0, yk, &S->k_full[st]);
          if (gv < g) ok = load_v();
          pend_x = x.head * kDh + 64 * static_cast<int>(rank);
          pend_y = static_cast<int32_t>(krow0 + static_cast<int64_t>(j) * kPfRows);
        }
      }
      if (ok && gv < g) ok = load_v();
      if (!ok) pa_set_abort(S);
      if (n > 0) tc::mbar_wait(&S->q_full, (n - 1) & 1);
      for (uint32_t q = g > kPaKStages ? g - kPaKStages : 0; q < g; ++q)
        tc::mbar_wait(&S->k_full[q % kPaKStages], (q / kPaKStages) & 1);
      for (uint32_t q = gv > kPaVStages ? gv - kPaVStages : 0; q < gv; ++q)
        tc::mbar_wait(&S->v_full[q % kPaVStages], (q / kPaVStages) & 1);
    }
  } else if (warp == kPaSoftmaxWarps + 2) {
    // ------------------------------------------------------------ forwarder (both CTAs)
    // tells the even CTA's MMA issuer when this CTA's queries, key half and value half have landed,
    // in the order the producer requested them
    if (lane == 0) {
      const uint32_t q_ready0 = tc::map_peer(&S->q_ready, 0);
      const uint32_t k_ready0 = tc::map_peer(&S->k_ready[0], 0);
      const uint32_t v_ready0 = tc::map_peer(&S->v_ready[0], 0);
      uint32_t n = 0, g = 0, gv = 0;
      bool ok = true;
      auto fwd_v = [&]() -> bool {
        const int st = gv % kPaVStages;
        if (!tc::mbar_wait(&S->v_full[st], (gv / kPaVStages) & 1)) return false;
        tc::mbar_arrive_cluster(v_ready0 + 8u * st);
        ++gv;
        return true;
      };
      for (int64_t u = cl; u < n_units && ok; u += ncl) {
        const PaUnit x = pa_unit(a, u);
        if (!x.live) continue;
        ok = tc::mbar_wait(&S->q_full, n & 1);
        if (!ok || pa_aborted(S)) { ok = false; break; }
        tc::mbar_arrive_cluster(q_ready0);
        ++n;
        for (int j = 0; j < x.nk && ok; ++j, ++g) {
          const int st = g % kPaKStages;
          ok = tc::mbar_wait(&S->k_full[st], (g / kPaKStages) & 1);
          if (!ok || pa_aborted(S)) { ok = false; break; }
          tc::mbar_arrive_cluster(k_ready0 + 8u * st);
          if (gv < g) ok = fwd_v();
        }
      }
      if (ok && gv < g) ok = fwd_v();
      if (!ok) pa_set_abort(S);
    }
  } else if (warp == kPaSoftmaxWarps + 1) {
    // ------------------------------------------------------------ score MMA issuer (even CTA)
    // Scores and PVs go out from two threads, so that the tensor pipe stays fed while one of them
    // waits for its next operands.
    if (rank == 0 && lane == 0) {
      const uint32_t idesc_s = tc::idesc_bf16_f32(256, 128, 0, 0);
      const uint64_t qdesc0 = tc::sdesc_sw128(tc::smem_u32(sQ), 16, 1024);         // K-major Q, 128 rows
      const uint64_t kdesc0 = tc::sdesc_sw128(tc::smem_u32(kst0), 16, 1024);       // K-major keys, 64 rows
      uint32_t n = 0, g = 0;
      bool ok = true;
      for (int64_t u = cl; u < n_units && ok; u += ncl) {
        const PaUnit x = pa_unit(a, u);
        if (!x.live) continue;
        ok = tc::mbar_wait(&S->q_ready, n & 1);
        for (int j = 0; j < x.nk && ok; ++j, ++g) {
          const uint32_t s = g & 1, st = g % kPaKStages;
          ok = tc::mbar_wait(&S->k_ready[st], (g / kPaKStages) & 1);
          if (ok && g >= 2) ok = tc::mbar_wait(&S->s_free[s], ((g - 2) >> 1) & 1);
          if (!ok || pa_aborted(S)) { ok = false; break; }
          tc::tc_fence_after();
#pragma unroll
          for (int k = 0; k < 12; ++k) {
            const uint32_t qoff = (k >> 2) * kPfBox + (k & 3) * 32;
            const uint32_t koff = st * kPaKBytes + (k >> 2) * kPfHalfBox + (k & 3) * 32;
            tc::mma_ss_pair(tm + kPaTmS + 128 * s, qdesc0 + static_cast<uint64_t>(qoff >> 4),
                            kdesc0 + static_cast<uint64_t>(koff >> 4), idesc_s, k > 0 ? 1u : 0u);
          }
          tc::mma_commit_pair(&S->s_full[s]);
          tc::mma_commit_pair(&S->k_empty[st]);
          if (j == x.nk - 1) tc::mma_commit_pair(&S->q_empty);
        }
        ++n;
      }
      if (!ok) pa_set_abort(S);
      tc::mma_commit_pair(&S->drain[0]);
      tc::mbar_wait(&S->drain[0], 0);
    }
  } else if (warp == kPaSoftmaxWarps + 3) {
    // ------------------------------------------------------------ PV MMA issuer (even CTA)
    if (rank == 0 && lane == 0) {
      const uint32_t idesc_o = idesc_f16_f32(256, 128, 0, 1);
      const uint64_t vdesc0 = tc::sdesc_sw128(tc::smem_u32(vst0), kPfBox, 1024);   // MN-major V, 64 columns
      uint32_t g = 0;
      bool ok = true;
      for (int64_t u = cl; u < n_units && ok; u += ncl) {
        const PaUnit x = pa_unit(a, u);
        if (!x.live) continue;
        for (int j = 0; j < x.nk && ok; ++j, ++g) {
          // O (+)= P V of key tile g (P from TMEM, 16 keys per MMA); the first of a unit starts O afresh,
          // after the softmax warps (whose P it waits for) have read the previous unit's O
          const uint32_t s = g & 1, st = g % kPaVStages;
          ok = tc::mbar_wait(&S->v_ready[st], (g / kPaVStages) & 1);
          if (ok) ok = tc::mbar_wait(&S->p_full[s], (g >> 1) & 1);
          if (!ok || pa_aborted(S)) { ok = false; break; }
          tc::tc_fence_after();
#pragma unroll
          for (int k = 0; k < 8; ++k)
            mma_ts_pair(tm + kPaTmO, tm + kPaTmP + 64 * s + 8 * k,
                        vdesc0 + static_cast<uint64_t>((st * kPaVBytes + 2048 * k) >> 4), idesc_o,
                        (j == 0 && k == 0) ? 0u : 1u);
          tc::mma_commit_pair(&S->o_done[s]);
          tc::mma_commit_pair(&S->v_empty[st]);
        }
      }
      if (!ok) pa_set_abort(S);
      tc::mma_commit_pair(&S->drain[1]);
      tc::mbar_wait(&S->drain[1], 0);
    }
  } else {
    // ------------------------------------------------------------ softmax (warps 0-7, both CTAs)
    // warp w: TMEM lane quarter w & 3 (query rows 32 (w & 3) .. + 31 of this CTA), key columns
    // 64 (w >> 2) .. + 63 of each tile and O columns 64 (w >> 2) .. + 63
    const int q4 = warp & 3, hc = warp >> 2;
    const int row = 32 * q4 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(32 * q4) << 16;
    const uint32_t s_free0 = tc::map_peer(&S->s_free[0], 0), p_full0 = tc::map_peer(&S->p_full[0], 0);
    const float sl = a.scale_log2;
    uint32_t g = 0;
    bool ok = true;
    for (int64_t u = cl; u < n_units && ok; u += ncl) {
      const PaUnit x = pa_unit(a, u);
      if (!x.live) continue;
      const int qp = x.p0 + 2 * kPfRows * x.t + row_off + row;   // position of this row's token
      float m_used = -INFINITY, l = 0.f;
      // a wait that runs out stops this warp's waiting for the rest of the unit; the warps vote at
      // its end and leave together
      bool alive = true;
      for (int j = 0; j < x.nk; ++j, ++g) {
        const uint32_t s = g & 1;
        if (alive) alive = __all_sync(0xffffffffu, tc::mbar_wait(&S->s_full[s], (g >> 1) & 1));
        tc::tc_fence_after();
        float v[64];
        {
          uint32_t r0[32], r1[32];
          tc::tmem_ld32(tm + lane_base + kPaTmS + 128 * s + 64 * hc, r0);
          tc::tmem_ld32(tm + lane_base + kPaTmS + 128 * s + 64 * hc + 32, r1);
          tc::tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            v[i] = __uint_as_float(r0[i]);
            v[32 + i] = __uint_as_float(r1[i]);
          }
        }
        tc::tc_fence_before();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive_cluster_relaxed(s_free0 + 8u * s);   // only TMEM was read
        // causal mask: key position k0 + i is visible to this row iff k0 + i <= qp
        const int k0 = kPfRows * j + 64 * hc;
        if (k0 + 63 > qp) {
#pragma unroll
          for (int i = 0; i < 64; ++i)
            if (k0 + i > qp) v[i] = -INFINITY;
        }
        float m4[4] = {v[0], v[1], v[2], v[3]};
#pragma unroll
        for (int i = 4; i < 64; i += 4)
#pragma unroll
          for (int k = 0; k < 4; ++k) m4[k] = fmaxf(m4[k], v[i + k]);
        S->red_max[s][hc][row] = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
        tc::named_sync(1 + q4, 64);
        const float mt = fmaxf(S->red_max[s][0][row], S->red_max[s][1][row]) * sl;
        if (j == 0) {
          m_used = mt;
        } else {
          const bool need = mt > m_used + static_cast<float>(kRescaleThreshold);
          if (__any_sync(0xffffffffu, need)) {
            // the O rows a rescale touches: the previous tile's PV must have completed
            if (alive) alive = __all_sync(0xffffffffu, tc::mbar_wait(&S->o_done[s ^ 1u], ((g - 1) >> 1) & 1));
            tc::tc_fence_after();
            const float f = need ? tc::ex2_approx(m_used - mt) : 1.f;
            if (need) {
              m_used = mt;
              l *= f;
            }
#pragma unroll 1
            for (int c0 = 0; c0 < 64; c0 += 32) {
              uint32_t r[32];
              tc::tmem_ld32(tm + lane_base + kPaTmO + 64 * hc + c0, r);
              tc::tmem_ld_wait();
#pragma unroll
              for (int c = 0; c < 32; ++c) r[c] = __float_as_uint(__uint_as_float(r[c]) * f);
              tc::tmem_st32(tm + lane_base + kPaTmO + 64 * hc + c0, r);
            }
          }
        }
        {
          const float neg_m = -m_used;
          uint32_t pk[32];
          float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const float e0 = tc::ex2_approx(fmaf(v[2 * i], sl, neg_m));
            const float e1 = tc::ex2_approx(fmaf(v[2 * i + 1], sl, neg_m));
            ls[i & 3] += e0 + e1;
            pk[i] = pack_f16(e0, e1);
          }
          l += (ls[0] + ls[1]) + (ls[2] + ls[3]);
          // this P buffer was last read by the PV of tile g - 2
          if (g >= 2 && alive) alive = __all_sync(0xffffffffu, tc::mbar_wait(&S->o_done[s], ((g - 2) >> 1) & 1));
          tc::tc_fence_after();
          tc::tmem_st32(tm + lane_base + kPaTmP + 64 * s + 32 * hc, pk);
          tc::tmem_st_wait();
        }
        tc::tc_fence_before();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive_cluster(p_full0 + 8u * s);
      }
      // ---- epilogue: out = O / l for the rows that are this unit's tokens
      if (alive) alive = __all_sync(0xffffffffu, tc::mbar_wait(&S->o_done[(g - 1) & 1], ((g - 1) >> 1) & 1));
      tc::tc_fence_after();
      S->red_l[hc][row] = l;
      tc::named_sync(1 + q4, 64);
      const float inv = 1.f / (S->red_l[0][row] + S->red_l[1][row]);
      const bool valid = 2 * kPfRows * x.t + row_off + row < x.n;
      float* dst = a.out + (static_cast<int64_t>(x.q0 + row_off + row) * kH + x.head) * kDh + 64 * hc;
      {
        uint32_t r0[32], r1[32];
        tc::tmem_ld32(tm + lane_base + kPaTmO + 64 * hc, r0);
        tc::tmem_ld32(tm + lane_base + kPaTmO + 64 * hc + 32, r1);
        tc::tmem_ld_wait();
        if (valid) {
#pragma unroll
          for (int c = 0; c < 32; c += 4) {
            *reinterpret_cast<float4*>(dst + c) =
                make_float4(__uint_as_float(r0[c]) * inv, __uint_as_float(r0[c + 1]) * inv,
                            __uint_as_float(r0[c + 2]) * inv, __uint_as_float(r0[c + 3]) * inv);
            *reinterpret_cast<float4*>(dst + 32 + c) =
                make_float4(__uint_as_float(r1[c]) * inv, __uint_as_float(r1[c + 1]) * inv,
                            __uint_as_float(r1[c + 2]) * inv, __uint_as_float(r1[c + 3]) * inv);
          }
        }
      }
      ok = tc::named_sync_and(5, 32 * kPaSoftmaxWarps, alive);
    }
    if (!ok) pa_set_abort(S);
  }
  // ---------------------------------------------------------------- teardown
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  tc::tc_fence_before();
  __syncthreads();
  tc::cluster_sync();   // no pair MMA, remote arrive or TMEM access of the other CTA is left
  tc::tc_fence_after();
  if (warp == kPaSoftmaxWarps + 1) tc::tmem_dealloc_pair<512>(tm);
}

}  // namespace tcd
}  // namespace mla
