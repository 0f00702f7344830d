// Tensor-core (tcgen05 + TMEM + TMA) MLA decode for the DeepSeek-V2 shape:
// 128 heads of d_h = 128, latent d_c = 512, decoupled rope d_r = 64, bf16
// queries and weights, bf16 cache rows of 576 values (DeepSeek-V2 report,
// section 2.1.2 absorbed form, section 2.1.3 decoupled RoPE).
//
// Three kernels per decode:
//   absorb  : Q_lat[b,i,0:512] = W_UK[i]^T q_nope[b,i] (one CTA per head, the
//             whole 128 KB weight slice in flight at once, M = 4 x 128 latent
//             rows, N = batch), q_rope copied to Q_lat[b,i,512:576]; one
//             extra CTA clamps the lengths and writes the per-sequence tile
//             prefix sums the other two kernels share.
//   attend  : persistent clusters of two CTAs; cluster c takes an equal share
//             of all 64-token tiles of all sequences, cut at sequence ends
//             into segments. In a pair, CTA0 owns latent columns 0..255 plus
//             the 64 rope columns and CTA1 owns latent columns 256..511: each
//             keeps its Q slice in TMEM, computes a partial score tile, swaps
//             it with its peer through distributed shared memory, runs the
//             (identical) online softmax, and accumulates its half of O_lat
//             in TMEM. Each segment ends in an unnormalised partial
//             (O half, running max m, sum l).
//   combine : one CTA per head: log-sum-exp merge of the partials of every
//             sequence, o_lat split into bf16 hi + lo, then
//             out[b,i,:] = W_UV[i] (o_hi + o_lo) on the tensor cores.
#pragma once

#include "common.cuh"
#include "tc.cuh"

namespace mla {
namespace tcd {

constexpr int kH = 128, kDc = 512, kDr = 64, kDh = 128, kRow = 576;
constexpr int kTile = 64;                    // tokens per attend tile
constexpr int kBlk = kTile * 128;            // one TMA box: 64 rows x 64 bf16 (128 B) = 8 KB
constexpr int kStageBlks = 5;                // CTA0: 4 latent boxes + 1 rope box; CTA1: 4 latent boxes
constexpr int kStageBytes = kStageBlks * kBlk;
constexpr int kStages = 4;
constexpr int kXbufBytes = kH * kTile * 4;   // one partial score tile, fp32
constexpr int kAttendThreads = 256;          // warp 0 TMA, warp 1 MMA, warps 4-7 softmax/epilogue
constexpr float kRescaleThreshold = 8.0f;    // log2 units: O is rescaled only when the max grows by > 2^8

// TMEM columns of the attend kernel (512 allocated)
constexpr uint32_t kTmO = 0;     // O half: 128 lanes x 256 fp32
constexpr uint32_t kTmS = 256;   // partial / full score tile: 64 fp32
constexpr uint32_t kTmQ = 320;   // Q slice, bf16 pairs: up to 160 columns
constexpr uint32_t kTmP = 480;   // probabilities, bf16 pairs: 32 columns

struct Plan {
  int32_t* lens;   // [B] lengths clamped to [0, max_seq_len]
  int32_t* cum;    // [B+1] prefix sums of ceil(len / 64)
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
  uint16_t* q_lat;            // [B, H, 576]
  Plan plan;
  int batch, nb, max_seq_len;
};

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
}

// One CTA per head i (blockIdx.x < H); CTA H writes the plan.
__global__ void __launch_bounds__(kAbsorbThreads) absorb_tc_kernel(const __grid_constant__ CUtensorMap map_wuk,
                                                                   const __grid_constant__ CUtensorMap map_qn,
                                                                   AbsorbArgs a) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (blockIdx.x == kH) {
    plan_block(a);
    return;
  }
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* sA = sm;                          // 8 boxes [128 d_h rows x 64 latent] = 128 KB
  uint8_t* sB = sm + 8 * 16384;              // 2 boxes [nb rows x 64 d_h]
  uint64_t* bars = reinterpret_cast<uint64_t*>(sB + 2 * a.nb * 128);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 4);
  const int i = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    tc::mbar_init(&bars[0], 1);  // weights landed
    tc::mbar_init(&bars[1], 1);  // queries landed (one phase per N chunk)
    tc::mbar_init(&bars[2], 1);  // MMAs done (one phase per N chunk)
    tc::fence_mbar_init();
    tc::tma_prefetch_map(&map_wuk);
    tc::tma_prefetch_map(&map_qn);
  }
  if (warp == 0) tc::tmem_alloc<512>(tslot);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tm = *tslot;
  if (threadIdx.x == 0) {
    tc::mbar_arrive_expect_tx(&bars[0], 8 * 16384);
    for (int j = 0; j < 8; ++j) tc::tma_load_2d(sA + j * 16384, &map_wuk, 64 * j, i * kDh, &bars[0]);
  }
  // q_rope -> Q_lat[:, i, 512:576]
  for (int idx = threadIdx.x; idx < a.batch * 8; idx += kAbsorbThreads) {
    const int b = idx >> 3, c = idx & 7;
    const uint4 v = reinterpret_cast<const uint4*>(a.q_rope + (static_cast<int64_t>(b) * kH + i) * kDr)[c];
    reinterpret_cast<uint4*>(a.q_lat + (static_cast<int64_t>(b) * kH + i) * kRow + kDc)[c] = v;
  }
  const uint32_t idesc = tc::idesc_bf16_f32(128, a.nb, 1, 0);
  bool ok = true;
  int chunk = 0;
  for (int n0 = 0; n0 < a.batch; n0 += a.nb, ++chunk) {
    if (threadIdx.x == 0) {
      tc::mbar_arrive_expect_tx(&bars[1], 2 * a.nb * 128);
      tc::tma_load_2d(sB, &map_qn, i * kDh, n0, &bars[1]);
      tc::tma_load_2d(sB + a.nb * 128, &map_qn, i * kDh + 64, n0, &bars[1]);
      ok = tc::mbar_wait(&bars[0], 0) && tc::mbar_wait(&bars[1], chunk & 1);
      tc::tc_fence_after();
      if (ok) {
        for (int mt = 0; mt < 4; ++mt) {
          for (int kk = 0; kk < 8; ++kk) {
            const uint64_t ad = tc::sdesc_sw128(tc::smem_u32(sA + (2 * mt) * 16384 + 2048 * kk), 16384, 1024);
            const uint64_t bd = tc::sdesc_sw128(tc::smem_u32(sB + (kk >> 2) * a.nb * 128 + (kk & 3) * 32), 16, 1024);
            tc::mma_ss(tm + mt * a.nb, ad, bd, idesc, kk > 0);
          }
        }
      }
      tc::mma_commit(&bars[2]);
    }
    __syncwarp();
    ok = tc::mbar_wait(&bars[2], chunk & 1);
    tc::tc_fence_after();
    // epilogue: lane = latent row within the M tile, columns = sequences
    for (int mt = 0; mt < 4; ++mt) {
      for (int c0 = 0; c0 < a.nb; c0 += 16) {
        uint32_t r[16];
        tc::tmem_ld16(tc::tmem_at(tm, 32 * warp, mt * a.nb + c0), r);
        tc::tmem_ld_wait();
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          const int b = n0 + c0 + c;
          if (b < a.batch && ok)
            a.q_lat[(static_cast<int64_t>(b) * kH + i) * kRow + mt * 128 + 32 * warp + lane] =
                f32_to_bf16_bits(__uint_as_float(r[c]));
        }
      }
    }
    tc::tc_fence_before();
    __syncthreads();  // TMEM and the query box are reused by the next chunk
  }
  if (warp == 0) tc::tmem_dealloc<512>(tm);
}

// ================================================================== attend
struct AttendArgs {
  const uint16_t* q_lat;      // [B, H, 576]
  const int32_t* block_table; // [B, max_pages] (NULL: contiguous, sequence b owns pages b*max_pages ..)
  Plan plan;
  float* part_o;              // [slots, H, 512] fp32, unnormalised
  float* part_ml;             // [slots, H, 2]: running max (log2 units) and sum
  int64_t num_pages;
  int batch, max_pages, page_size;
  float scale_log2;
};

struct AttendSmem {
  uint64_t full[kStages], empty[kStages];
  uint64_t s_full, s_free, p_full, o_done, q_ready, o_free, xfull, xempty, drain;
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

__device__ __forceinline__ SegIter seg_begin(const int32_t* cum, int batch, uint32_t c, uint32_t nc) {
  const int64_t T = cum[batch];
  SegIter it;
  it.t = share_begin(c, T, nc);
  it.t1 = share_begin(c + 1, T, nc);
  // first sequence whose tiles reach past t: binary search on cum
  int lo = 0, hi = batch;  // cum[lo] <= t < cum[hi] when t < T
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (cum[mid] <= it.t) lo = mid; else hi = mid;
  }
  it.b = lo;
  return it;
}

__device__ __forceinline__ bool aborted(const AttendSmem* s) {
  return *reinterpret_cast<const volatile int32_t*>(&s->abort_flag) != 0;
}

__device__ __forceinline__ void set_abort(AttendSmem* s) {
  *reinterpret_cast<volatile int32_t*>(&s->abort_flag) = 1;
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kAttendThreads, 1)
    attend_tc_kernel(const __grid_constant__ CUtensorMap map_pool, AttendArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* tiles = sm;
  float* xbuf = reinterpret_cast<float*>(sm + kStages * kStageBytes);
  AttendSmem* S = reinterpret_cast<AttendSmem*>(sm + kStages * kStageBytes + kXbufBytes);

  const uint32_t rank = tc::cluster_ctarank(), peer = rank ^ 1u;
  const uint32_t cl = tc::cluster_id_x(), ncl = tc::n_clusters_x();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_blk = rank == 0 ? 5 : 4;          // boxes per tile for this CTA
  const int n_k = n_blk * 4;                    // K steps of 16 in the score MMA

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      tc::mbar_init(&S->full[s], 1);
      tc::mbar_init(&S->empty[s], 1);
    }
    tc::mbar_init(&S->s_full, 1);
    tc::mbar_init(&S->s_free, 128);
    tc::mbar_init(&S->p_full, 128);
    tc::mbar_init(&S->o_done, 1);
    tc::mbar_init(&S->q_ready, 128);
    tc::mbar_init(&S->o_free, 128);
    tc::mbar_init(&S->xfull, 128);
    tc::mbar_init(&S->xempty, 128);
    tc::mbar_init(&S->drain, 1);
    S->abort_flag = 0;
    tc::fence_mbar_init();
    tc::tma_prefetch_map(&map_pool);
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
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0) {
      const uint64_t policy = tc::policy_evict_first();
      SegIter si = seg_begin(cum, a.batch, cl, ncl);
      int b, j0, j1;
      uint32_t it = 0;
      bool ok = true;
      while (ok && si.next(cum, a.batch, &b, &j0, &j1)) {
        for (int j = j0; j < j1 && ok; ++j, ++it) {
          const int st = it % kStages;
          if (it >= kStages) ok = tc::mbar_wait(&S->empty[st], ((it / kStages) - 1) & 1);
          if (!ok || aborted(S)) { ok = false; break; }
          const int64_t tok = static_cast<int64_t>(j) * kTile;
          const int pg = static_cast<int>(tok / a.page_size);
          int64_t page = -1;
          if (pg < a.max_pages)
            page = a.block_table ? a.block_table[static_cast<int64_t>(b) * a.max_pages + pg]
                                 : static_cast<int64_t>(b) * a.max_pages + pg;
          int32_t y;
          if (page < 0 || page >= a.num_pages) {
            flag_error(ERR_BIT_BOUNDS);
            y = -2 * kTile;  // entirely outside the pool: the copy fills zeros
          } else {
            y = static_cast<int32_t>(page * a.page_size + tok % a.page_size);
          }
          uint8_t* dst = tiles + st * kStageBytes;
          tc::mbar_arrive_expect_tx(&S->full[st], n_blk * kBlk);
          for (int k = 0; k < 4; ++k)
            tc::tma_load_2d_hint(dst + k * kBlk, &map_pool, static_cast<int>(rank) * 256 + 64 * k, y, &S->full[st],
                                 policy);
          if (rank == 0) tc::tma_load_2d_hint(dst + 4 * kBlk, &map_pool, kDc, y, &S->full[st], policy);
        }
      }
      if (!ok) set_abort(S);
      // drain: copies still in flight must land before the CTA exits
      const uint32_t first = it > kStages ? it - kStages : 0;
      for (uint32_t q = first; q < it; ++q) tc::mbar_wait(&S->full[q % kStages], (q / kStages) & 1);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t idesc_s = tc::idesc_bf16_f32(128, kTile, 0, 0);
      const uint32_t idesc_o = tc::idesc_bf16_f32(128, 256, 0, 1);
      SegIter si = seg_begin(cum, a.batch, cl, ncl);
      int b, j0, j1;
      uint32_t it = 0, seg = 0;
      bool ok = true;
      // lagged PV of the previous tile
      bool have_prev = false, prev_first = false;
      uint32_t prev_stage = 0, prev_seg = 0;
      auto issue_pv = [&](uint32_t q) -> bool {
        if (!tc::mbar_wait(&S->p_full, q & 1)) return false;
        if (prev_first && prev_seg > 0 && !tc::mbar_wait(&S->o_free, (prev_seg - 1) & 1)) return false;
        tc::tc_fence_after();
        const uint32_t base = tc::smem_u32(tiles + prev_stage * kStageBytes);
        for (int k = 0; k < 4; ++k) {
          const uint64_t bd = tc::sdesc_sw128(base + k * 2048, kBlk, 1024);
          tc::mma_ts(tm + kTmO, tm + kTmP + 8 * k, bd, idesc_o, (k > 0 || !prev_first) ? 1u : 0u);
        }
        tc::mma_commit(&S->o_done);
        tc::mma_commit(&S->empty[prev_stage]);
        return true;
      };
      while (ok && si.next(cum, a.batch, &b, &j0, &j1)) {
        ok = tc::mbar_wait(&S->q_ready, seg & 1);
        for (int j = j0; j < j1 && ok; ++j, ++it) {
          const uint32_t st = it % kStages;
          ok = tc::mbar_wait(&S->full[st], (it / kStages) & 1);
          if (ok && it > 0) ok = tc::mbar_wait(&S->s_free, (it - 1) & 1);
          if (!ok || aborted(S)) { ok = false; break; }
          tc::tc_fence_after();
          const uint32_t base = tc::smem_u32(tiles + st * kStageBytes);
          for (int k = 0; k < n_k; ++k) {
            const uint64_t bd = tc::sdesc_sw128(base + (k >> 2) * kBlk + (k & 3) * 32, 16, 1024);
            tc::mma_ts(tm + kTmS, tm + kTmQ + 8 * k, bd, idesc_s, k > 0 ? 1u : 0u);
          }
          tc::mma_commit(&S->s_full);
          if (have_prev) ok = issue_pv(it - 1);
          have_prev = true;
          prev_first = (j == j0);
          prev_stage = st;
          prev_seg = seg;
        }
        ++seg;
      }
      if (ok && have_prev) ok = issue_pv(it - 1);
      if (!ok) set_abort(S);
      // every MMA issued so far must complete before TMEM is released
      tc::mma_commit(&S->drain);
      tc::mbar_wait(&S->drain, 0);
    }
  } else if (warp >= 4) {
    // ---------------------------------------------------------------- softmax + epilogue
    const int h = threadIdx.x - 128;             // head = TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>(32 * (warp & 3)) << 16;
    const int q_words = n_blk * 32;              // bf16 pairs of this CTA's Q slice
    auto load_q = [&](int b) {
      const uint16_t* q = a.q_lat + (static_cast<int64_t>(b) * kH + h) * kRow;
      for (int w0 = 0; w0 < q_words; w0 += 16) {
        // words w0..w0+15 = K elements 2*w0 .. 2*w0+31
        const int k0 = 2 * w0;
        const int col = rank == 0 ? (k0 < 256 ? k0 : kDc + (k0 - 256)) : 256 + k0;
        const uint4* src = reinterpret_cast<const uint4*>(q + col);
        uint32_t v[16];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const uint4 x = src[u];
          v[4 * u] = x.x; v[4 * u + 1] = x.y; v[4 * u + 2] = x.z; v[4 * u + 3] = x.w;
        }
        tc::tmem_st16(tm + lane_base + kTmQ + w0, v);
      }
      tc::tmem_st_wait();
      tc::tc_fence_before();
      tc::mbar_arrive(&S->q_ready);
    };

    SegIter si = seg_begin(cum, a.batch, cl, ncl);
    int b, j0, j1;
    uint32_t it = 0, seg = 0;
    bool ok = true;
    bool have = si.next(cum, a.batch, &b, &j0, &j1);
    if (have) load_q(b);
    while (ok && have) {
      const int L = a.plan.lens[b];
      const int slot = b + static_cast<int>(cl);
      int nb_, nj0, nj1;
      SegIter si_next = si;
      const bool have_next = si_next.next(cum, a.batch, &nb_, &nj0, &nj1);
      float m_used = -INFINITY, l = 0.f;
      for (int j = j0; j < j1 && ok; ++j, ++it) {
        // ---- own partial scores
        ok = tc::mbar_wait(&S->s_full, it & 1);
        if (!ok || aborted(S)) { ok = false; break; }
        tc::tc_fence_after();
        float s[kTile];
#pragma unroll
        for (int c0 = 0; c0 < kTile; c0 += 16) {
          uint32_t r[16];
          tc::tmem_ld16(tm + lane_base + kTmS + c0, r);
          tc::tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < 16; ++c) s[c0 + c] = __uint_as_float(r[c]);
        }
        tc::tc_fence_before();
        tc::mbar_arrive(&S->s_free);
        if (j == j1 - 1 && have_next) load_q(nb_);   // all score MMAs of this segment are done
        // ---- swap partial scores with the peer CTA
        if (it > 0) ok = tc::mbar_wait<true>(&S->xempty, (it - 1) & 1);
        if (!ok) break;
#pragma unroll
        for (int q = 0; q < 16; ++q) {
          const int chunk = q ^ (h & 15);
          tc::st_cluster_v4(tc::map_peer(xbuf + h * kTile + chunk * 4, peer), __float_as_uint(s[4 * q]),
                            __float_as_uint(s[4 * q + 1]), __float_as_uint(s[4 * q + 2]),
                            __float_as_uint(s[4 * q + 3]));
        }
        tc::mbar_arrive_remote(&S->xfull, peer);
        ok = tc::mbar_wait<true>(&S->xfull, it & 1);
        if (!ok) break;
#pragma unroll
        for (int q = 0; q < 16; ++q) {
          const int chunk = q ^ (h & 15);
          const float4 v = *reinterpret_cast<const float4*>(xbuf + h * kTile + chunk * 4);
          s[4 * q] += v.x; s[4 * q + 1] += v.y; s[4 * q + 2] += v.z; s[4 * q + 3] += v.w;
        }
        tc::mbar_arrive_remote(&S->xempty, peer);
        // ---- online softmax (base 2), identical in both CTAs
        const int valid = min(kTile, L - j * kTile);
        float mx = -INFINITY;
#pragma unroll
        for (int c = 0; c < kTile; ++c) {
          s[c] = c < valid ? s[c] * a.scale_log2 : -INFINITY;
          mx = fmaxf(mx, s[c]);
        }
        bool rescale = false;
        float alpha = 1.f;
        if (m_used == -INFINITY) {
          m_used = mx;
        } else if (mx > m_used + kRescaleThreshold) {
          alpha = exp2f(m_used - mx);
          l *= alpha;
          m_used = mx;
          rescale = true;
        }
        uint32_t p[kTile / 2];
        float psum = 0.f;
#pragma unroll
        for (int c = 0; c < kTile; c += 2) {
          const uint32_t w = tc::pack_bf16(exp2f(s[c] - m_used), exp2f(s[c + 1] - m_used));
          p[c / 2] = w;
          psum += bf16_to_f32(static_cast<uint16_t>(w & 0xffffu)) + bf16_to_f32(static_cast<uint16_t>(w >> 16));
        }
        l += psum;
        // ---- PV of the previous tile must be done: P buffer and O are ours
        if (it > 0) ok = tc::mbar_wait(&S->o_done, (it - 1) & 1);
        if (!ok) break;
        tc::tc_fence_after();
        if (rescale) {
          for (int c0 = 0; c0 < 256; c0 += 16) {
            uint32_t r[16];
            tc::tmem_ld16(tm + lane_base + kTmO + c0, r);
            tc::tmem_ld_wait();
#pragma unroll
            for (int c = 0; c < 16; ++c) r[c] = __float_as_uint(__uint_as_float(r[c]) * alpha);
            tc::tmem_st16(tm + lane_base + kTmO + c0, r);
          }
        }
        {
          uint32_t w0[16], w1[16];
#pragma unroll
          for (int c = 0; c < 16; ++c) { w0[c] = p[c]; w1[c] = p[16 + c]; }
          tc::tmem_st16(tm + lane_base + kTmP, w0);
          tc::tmem_st16(tm + lane_base + kTmP + 16, w1);
        }
        tc::tmem_st_wait();
        // ---- rows past the sequence end must not reach PV as NaN/Inf garbage
        if (valid < kTile) {
          uint8_t* stage = tiles + (it % kStages) * kStageBytes;
          const int nrow = kTile - valid;
          for (int idx = h; idx < nrow * 4 * 8; idx += 128) {
            const int blk = idx / (nrow * 8), rem = idx % (nrow * 8);
            const int row = valid + rem / 8, ch = rem % 8;
            *reinterpret_cast<uint4*>(stage + blk * kBlk + row * 128 + ch * 16) = make_uint4(0, 0, 0, 0);
          }
          tc::fence_proxy_async_smem();
        }
        tc::tc_fence_before();
        tc::mbar_arrive(&S->p_full);
      }
      if (!ok) break;
      // ---- segment epilogue: unnormalised O half, m and l
      ok = tc::mbar_wait(&S->o_done, (it - 1) & 1);
      if (!ok) break;
      tc::tc_fence_after();
      float* dst = a.part_o + (static_cast<int64_t>(slot) * kH + h) * kDc + rank * 256;
      for (int c0 = 0; c0 < 256; c0 += 16) {
        uint32_t r[16];
        tc::tmem_ld16(tm + lane_base + kTmO + c0, r);
        tc::tmem_ld_wait();
#pragma unroll
        for (int u = 0; u < 4; ++u)
          reinterpret_cast<uint4*>(dst + c0)[u] = make_uint4(r[4 * u], r[4 * u + 1], r[4 * u + 2], r[4 * u + 3]);
      }
      tc::tc_fence_before();
      tc::mbar_arrive(&S->o_free);
      if (rank == 0) {
        float2* ml = reinterpret_cast<float2*>(a.part_ml) + static_cast<int64_t>(slot) * kH + h;
        *ml = make_float2(m_used, l);
      }
      ++seg;
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

// ================================================================== combine + W_UV
struct CombineArgs {
  Plan plan;
  const float* part_o;
  const float* part_ml;
  float* out;          // [B, H, 128]
  int batch, ncl;
};

constexpr int kCombineThreads = 128;
constexpr int kCombineNb = 32;        // sequences per MMA chunk
constexpr int kCombineMaxSlots = 512; // partial slots one chunk may touch: kCombineNb + clusters

// Dynamic shared memory of the combine kernel (after 1 KB alignment).
constexpr size_t kCombineSmem = 8 * 16384 + 2 * 8 * kCombineNb * 128 + kCombineMaxSlots * 4 + 2 * kCombineNb * 4 + 64;

__global__ void __launch_bounds__(kCombineThreads) combine_tc_kernel(const __grid_constant__ CUtensorMap map_wuv,
                                                                     CombineArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* sA = sm;                                   // W_UV[i]: 8 boxes [128 rows x 64] = 128 KB
  uint8_t* sHi = sm + 8 * 16384;                      // o_lat hi: 8 blocks [32 rows x 64] = 32 KB
  uint8_t* sLo = sHi + 8 * kCombineNb * 128;          // o_lat lo
  float* wts = reinterpret_cast<float*>(sLo + 8 * kCombineNb * 128);   // merge weight per slot of the chunk
  int32_t* seg_first = reinterpret_cast<int32_t*>(wts + kCombineMaxSlots);
  int32_t* seg_count = seg_first + kCombineNb;
  uint64_t* bars = reinterpret_cast<uint64_t*>(seg_count + kCombineNb);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 2);
  const int i = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, t = threadIdx.x;
  if (t == 0) {
    tc::mbar_init(&bars[0], 1);
    tc::mbar_init(&bars[1], 1);
    tc::fence_mbar_init();
    tc::tma_prefetch_map(&map_wuv);
    // the weights do not depend on the attend kernel: start streaming them now
    tc::mbar_arrive_expect_tx(&bars[0], 8 * 16384);
    for (int j = 0; j < 8; ++j) tc::tma_load_2d(sA + j * 16384, &map_wuv, 64 * j, i * kDh, &bars[0]);
  }
  if (warp == 0) tc::tmem_alloc<32>(tslot);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tm = *tslot;
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int64_t T = a.plan.cum[a.batch];
  const uint32_t idesc = tc::idesc_bf16_f32(128, kCombineNb, 0, 0);
  const float2* ml_all = reinterpret_cast<const float2*>(a.part_ml);
  bool ok = true;
  int chunk = 0;
  for (int n0 = 0; n0 < a.batch; n0 += kCombineNb, ++chunk) {
    // ---- pass 1 (one thread per sequence): merge weights of its partials.
    // Sequence b's partials sit in slots b + c for the clusters c whose
    // shares meet its tiles; in a chunk those slots form one contiguous run.
    const int64_t slot0 = (T > 0 && n0 < a.batch) ? n0 + share_owner(a.plan.cum[n0] < T ? a.plan.cum[n0] : T - 1, T, a.ncl) : 0;
    if (t < kCombineNb) {
      const int b = n0 + t;
      int first = 0, count = 0;
      if (b < a.batch && T > 0) {
        const int64_t tb0 = a.plan.cum[b], tb1 = a.plan.cum[b + 1];
        if (tb1 > tb0) {
          const int64_t c0 = share_owner(tb0, T, a.ncl), c1 = share_owner(tb1 - 1, T, a.ncl);
          float M = -INFINITY;
          for (int64_t c = c0; c <= c1; ++c)
            if (share_begin(c, T, a.ncl) < share_begin(c + 1, T, a.ncl)) M = fmaxf(M, ml_all[(b + c) * kH + i].x);
          float den = 0.f;
          for (int64_t c = c0; c <= c1; ++c) {
            float w = 0.f;
            if (share_begin(c, T, a.ncl) < share_begin(c + 1, T, a.ncl)) {
              const float2 ml = ml_all[(b + c) * kH + i];
              w = exp2f(ml.x - M);
              den += w * ml.y;
            }
            wts[b + c - slot0] = w;
          }
          const float inv = den > 0.f ? 1.f / den : 0.f;
          for (int64_t c = c0; c <= c1; ++c) wts[b + c - slot0] *= inv;
          first = static_cast<int>(b + c0 - slot0);
          count = static_cast<int>(c1 - c0 + 1);
        }
      }
      seg_first[t] = first;
      seg_count[t] = count;
    }
    __syncthreads();
    // ---- pass 2: o_lat rows, thread t owns latent elements 4t .. 4t+3 of every row
    for (int n = 0; n < kCombineNb; ++n) {
      const int first = seg_first[n], count = seg_count[n];
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
      for (int u = 0; u < count; ++u) {
        const float w = wts[first + u];
        if (w == 0.f) continue;   // a cluster with an empty share wrote nothing into this slot
        const float4 o = reinterpret_cast<const float4*>(a.part_o + ((slot0 + first + u) * kH + i) * kDc)[t];
        acc.x += w * o.x; acc.y += w * o.y; acc.z += w * o.z; acc.w += w * o.w;
      }
      // hi/lo bf16 split into the K-major 128-byte-swizzled B operand: row n, K = 4t..4t+3
      const float v[4] = {acc.x, acc.y, acc.z, acc.w};
      uint32_t hi[2], lo[2];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const uint32_t hw = tc::pack_bf16(v[2 * u], v[2 * u + 1]);
        hi[u] = hw;
        lo[u] = tc::pack_bf16(v[2 * u] - bf16_to_f32(static_cast<uint16_t>(hw & 0xffffu)),
                              v[2 * u + 1] - bf16_to_f32(static_cast<uint16_t>(hw >> 16)));
      }
      const int k = 4 * t, kb = k >> 6, kin = k & 63;
      const int off = kb * (kCombineNb * 128) + n * 128 + ((((kin >> 3) ^ (n & 7)) << 4)) + (kin & 7) * 2;
      *reinterpret_cast<uint2*>(sHi + off) = make_uint2(hi[0], hi[1]);
      *reinterpret_cast<uint2*>(sLo + off) = make_uint2(lo[0], lo[1]);
    }
    tc::fence_proxy_async_smem();
    tc::tc_fence_before();
    __syncthreads();
    if (t == 0) {
      tc::tc_fence_after();
      ok = tc::mbar_wait(&bars[0], 0);
      if (ok) {
        for (int kk = 0; kk < 32; ++kk) {
          const uint64_t ad = tc::sdesc_sw128(tc::smem_u32(sA + (kk >> 2) * 16384 + (kk & 3) * 32), 16, 1024);
          const uint32_t boff = (kk >> 2) * (kCombineNb * 128) + (kk & 3) * 32;
          tc::mma_ss(tm, ad, tc::sdesc_sw128(tc::smem_u32(sHi + boff), 16, 1024), idesc, kk > 0);
          tc::mma_ss(tm, ad, tc::sdesc_sw128(tc::smem_u32(sLo + boff), 16, 1024), idesc, 1);
        }
      }
      tc::mma_commit(&bars[1]);
    }
    __syncwarp();
    ok = tc::mbar_wait(&bars[1], chunk & 1) && ok;
    tc::tc_fence_after();
    for (int c0 = 0; c0 < kCombineNb; c0 += 16) {
      uint32_t r[16];
      tc::tmem_ld16(tc::tmem_at(tm, 32 * warp, c0), r);
      tc::tmem_ld_wait();
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        const int b = n0 + c0 + c;
        if (b < a.batch) a.out[(static_cast<int64_t>(b) * kH + i) * kDh + 32 * warp + lane] = __uint_as_float(r[c]);
      }
    }
    tc::tc_fence_before();
    __syncthreads();   // the B operand, the weights and TMEM are reused by the next chunk
  }
  if (warp == 0) tc::tmem_dealloc<32>(tm);
}

}  // namespace tcd
}  // namespace mla
