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
//   kv_up_kernel:        [rows x 512] latent tile (gathered from the pages) x
//                        [W_UK ; W_UV]^T ([512 x 32768]) -> K_nope (bf16, the
//                        query's type, for the score MMA) and V (fp16)
//                        [B * L_pad, 128 heads x 128]. tcgen05 MMA
//                        M = 128 rows, N = 256, K = 16; fp32 accumulators in
//                        TMEM, two of them so the epilogue of one column
//                        tile overlaps the MMAs of the next.
//   prefill_attn_kernel: per (sequence, head, 128-row query tile): S = Q K^T
//                        (M = N = 128, K = 192, bf16), online softmax with a
//                        causal mask, O += P V (M = N = 128, K = 128, fp16,
//                        P from TMEM), out = O / l in fp32.
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
constexpr int kKvNt = 256;                            // weight rows (output columns) per MMA tile
constexpr int kKvTilesPerItem = 16;                   // column tiles a work item covers
constexpr int kKvGroups = kPfWidthKV / kKvNt / kKvTilesPerItem;   // 8 items per row tile
constexpr int kKvStages = 3;                          // weight chunk ring: 256 rows x 64 columns = 32 KB each
constexpr int kKvABytes = 8 * kPfBox;                 // latent tile: 8 boxes of 128 rows x 64 columns = 128 KB
constexpr int kKvBBytes = kKvNt * 128;                // 32 KB
constexpr int kKvThreads = 32 * 6;                    // producer, MMA, 4 epilogue warps

struct KvUpSmem {
  uint64_t a_full, a_empty;
  uint64_t b_full[kKvStages], b_empty[kKvStages];
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

// Work item i: row tile r of sequence b, column tiles [16 g, 16 g + 16). Items whose rows lie past
// the sequence's length are empty.
struct KvItem {
  int b, r, g;
  bool live;
};
__device__ __forceinline__ KvItem kv_item(const KvUpArgs& a, int64_t i) {
  KvItem it;
  it.g = static_cast<int>(i % kKvGroups);
  const int64_t rb = i / kKvGroups;
  it.b = static_cast<int>(rb % a.batch);
  it.r = static_cast<int>(rb / a.batch);
  const int L = clamp_len(a.seq_lens[it.b], a.max_seq_len);
  it.live = static_cast<int64_t>(it.r) * kPfRows < L;
  return it;
}

// map_lat: the pool [rows, 576] bf16, boxes of 64 rows x 64 columns, 128-byte swizzle.
// map_wuk / map_wuv: W_UK / W_UV as [128 * 128, 512] bf16, boxes of 256 rows x 64 columns.
__global__ void __launch_bounds__(kKvThreads, 1)
    kv_up_kernel(const __grid_constant__ CUtensorMap map_lat, const __grid_constant__ CUtensorMap map_wuk,
                 const __grid_constant__ CUtensorMap map_wuv, KvUpArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* sA = sm;
  uint8_t* sB = sm + kKvABytes;
  KvUpSmem* S = reinterpret_cast<KvUpSmem*>(sB + kKvStages * kKvBBytes);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    tc::mbar_init(&S->a_full, 1);
    tc::mbar_init(&S->a_empty, 1);
    for (int s = 0; s < kKvStages; ++s) {
      tc::mbar_init(&S->b_full[s], 1);
      tc::mbar_init(&S->b_empty[s], 1);
    }
    for (int d = 0; d < 2; ++d) {
      tc::mbar_init(&S->d_full[d], 1);
      tc::mbar_init(&S->d_free[d], 4);
    }
    tc::mbar_init(&S->drain, 1);
    S->abort_flag = 0;
    tc::fence_mbar_init();
    tc::tma_prefetch_map(&map_lat);
    tc::tma_prefetch_map(&map_wuk);
    tc::tma_prefetch_map(&map_wuv);
  }
  if (warp == 1) tc::tmem_alloc<512>(&S->tmem_base);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tm = S->tmem_base;
  // the pool rows and the lengths come from the kernels ahead of this one on the stream
  asm volatile("griddepcontrol.wait;" ::: "memory");

  const int64_t n_items = static_cast<int64_t>((a.lpad / kPfRows)) * a.batch * kKvGroups;
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t n = 0, c = 0;   // items and weight chunks loaded
      bool ok = true;
      for (int64_t i = blockIdx.x; i < n_items && ok; i += gridDim.x) {
        const KvItem it = kv_item(a, i);
        if (!it.live) continue;
        if (n > 0) ok = tc::mbar_wait(&S->a_empty, (n - 1) & 1);
        if (!ok || kv_aborted(S)) { ok = false; break; }
        const int L = clamp_len(a.seq_lens[it.b], a.max_seq_len);
        tc::mbar_arrive_expect_tx(&S->a_full, kKvABytes);
        for (int h = 0; h < 2; ++h) {
          const int64_t tok = static_cast<int64_t>(it.r) * kPfRows + 64 * h;
          const int32_t y = pf_pool_row(a.block_table, a.num_pages, a.max_pages, a.page_size, it.b, tok, L);
          for (int k = 0; k < 8; ++k)
            tc::tma_load_2d(sA + k * kPfBox + h * kPfHalfBox, &map_lat, 64 * k, y, &S->a_full);
        }
        ++n;
        for (int t = 0; t < kKvTilesPerItem && ok; ++t) {
          const int n0 = (it.g * kKvTilesPerItem + t) * kKvNt;
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
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = tc::idesc_bf16_f32(128, kKvNt, 0, 0);
      const uint64_t adesc0 = tc::sdesc_sw128(tc::smem_u32(sA), 16, 1024);
      const uint64_t bdesc0 = tc::sdesc_sw128(tc::smem_u32(sB), 16, 1024);
      uint32_t n = 0, c = 0, d = 0;   // items, weight chunks, column tiles
      bool ok = true;
      for (int64_t i = blockIdx.x; i < n_items && ok; i += gridDim.x) {
        const KvItem it = kv_item(a, i);
        if (!it.live) continue;
        ok = tc::mbar_wait(&S->a_full, n & 1);
        for (int t = 0; t < kKvTilesPerItem && ok; ++t, ++d) {
          const uint32_t buf = d & 1;
          if (d >= 2) ok = tc::mbar_wait(&S->d_free[buf], ((d >> 1) - 1) & 1);
          for (int kc = 0; kc < 8 && ok; ++kc, ++c) {
            const int st = c % kKvStages;
            ok = tc::mbar_wait(&S->b_full[st], (c / kKvStages) & 1);
            if (!ok || kv_aborted(S)) { ok = false; break; }
            tc::tc_fence_after();
#pragma unroll
            for (int k = 0; k < 4; ++k)
              tc::mma_ss(tm + 256 * buf, adesc0 + static_cast<uint64_t>((kc * kPfBox + 32 * k) >> 4),
                         bdesc0 + static_cast<uint64_t>((st * kKvBBytes + 32 * k) >> 4), idesc,
                         (kc == 0 && k == 0) ? 0u : 1u);
            tc::mma_commit(&S->b_empty[st]);
          }
          if (ok) tc::mma_commit(&S->d_full[buf]);
        }
        if (ok) tc::mma_commit(&S->a_empty);
        ++n;
      }
      if (!ok) kv_set_abort(S);
      tc::mma_commit(&S->drain);
      tc::mbar_wait(&S->drain, 0);
    }
  } else {
    // ------------------------------------------------------------ epilogue: TMEM -> bf16 rows of K_nope / V
    const int q = warp & 3;   // TMEM lane quarter of this warp
    const int row = 32 * q + lane;
    uint32_t d = 0;
    bool ok = true;
    for (int64_t i = blockIdx.x; i < n_items && ok; i += gridDim.x) {
      const KvItem it = kv_item(a, i);
      if (!it.live) continue;
      const int L = clamp_len(a.seq_lens[it.b], a.max_seq_len);
      const bool valid = static_cast<int64_t>(it.r) * kPfRows + row < L;   // rows past L are written as zeros
      const int64_t grow = static_cast<int64_t>(it.b) * a.lpad + static_cast<int64_t>(it.r) * kPfRows + row;
      if (it.g == 0) {
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
        tc::tc_fence_before();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&S->d_free[buf]);
      }
    }
    if (!ok) kv_set_abort(S);
  }
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  if (warp == 1) tc::tmem_dealloc<512>(tm);
}

// ------------------------------------------------------------------ prefill_attn_kernel
constexpr int kPaStages = 2;                          // ring depth of key tiles and of value tiles
constexpr int kPaQBytes = 3 * kPfBox;                 // q_nope (2 boxes) and q_rope (1 box) of 128 rows: 48 KB
constexpr int kPaKBytes = 3 * kPfBox;                 // k_nope (2 boxes) and the shared rope key (1 box)
constexpr int kPaVBytes = 2 * kPfBox;                 // V: 2 boxes of 128 rows x 64 columns
constexpr int kPaSoftmaxWarps = 8;
constexpr int kPaThreads = 32 * (kPaSoftmaxWarps + 2);
constexpr uint32_t kPaTmS = 0;     // score buffers: columns 0 and 128
constexpr uint32_t kPaTmP = 256;   // P buffers (bf16 pairs): columns 256 and 320
constexpr uint32_t kPaTmO = 384;   // O: 128 columns

struct PaSmem {
  uint64_t q_full, q_empty;
  uint64_t k_full[kPaStages], k_empty[kPaStages], v_full[kPaStages], v_empty[kPaStages];
  uint64_t s_full[2], s_free[2], p_full[2], o_done[2];
  uint64_t drain;
  float red_max[2][2][kPfRows];   // [tile parity][column half][row]
  float red_l[2][kPfRows];        // [column half][row]
  uint32_t tmem_base;
  int32_t abort_flag;
};
constexpr size_t kPaSmem =
    1024 + kPaQBytes + static_cast<size_t>(kPaStages) * (kPaKBytes + kPaVBytes) + sizeof(PaSmem);

struct PrefillArgs {
  const int32_t* block_table;
  const int32_t* seq_lens;   // [B] rows of each sequence in the cache, its new tokens included
  const int32_t* q_start;    // [B + 1] new tokens of sequence b are rows q_start[b] .. q_start[b+1]-1
  float* out;                // [T, 128, 128] fp32
  int64_t num_pages;
  int batch, max_pages, page_size, max_seq_len, lpad, n_tokens, qt_max;
  float scale_log2;
};

// Unit u: query tile t of (sequence b, head). Units of one (sequence, head) are consecutive
// (longest tile first), so the CTAs working at one time share a few heads' K and V in L2.
struct PaUnit {
  int b, t, head, nk, n, p0, q0;
  bool live;
};
__device__ __forceinline__ PaUnit pa_unit(const PrefillArgs& a, int64_t u) {
  PaUnit x;
  const int64_t grp = u / a.qt_max;
  x.t = a.qt_max - 1 - static_cast<int>(u % a.qt_max);
  x.b = static_cast<int>(grp / kH);
  x.head = static_cast<int>(grp % kH);
  const int L = clamp_len(a.seq_lens[x.b], a.max_seq_len);
  const int s0 = a.q_start[x.b], s1 = a.q_start[x.b + 1];
  x.n = s1 - s0;
  x.q0 = s0 + kPfRows * x.t;
  x.p0 = L - x.n;
  x.live = x.n > 0 && x.n <= L && s0 >= 0 && s1 <= a.n_tokens && kPfRows * x.t < x.n;
  if (!x.live) {
    if (x.t == 0 && x.head == 0 && (x.n < 0 || x.n > L || s0 < 0 || s1 > a.n_tokens)) flag_error(ERR_BIT_BOUNDS);
    x.nk = 0;
    return x;
  }
  const int last = x.p0 + min(x.n, kPfRows * (x.t + 1)) - 1;   // position of the tile's last query row
  x.nk = last / kPfRows + 1;
  return x;
}

__device__ __forceinline__ bool pa_aborted(const PaSmem* s) {
  return *reinterpret_cast<const volatile int32_t*>(&s->abort_flag) != 0;
}
__device__ __forceinline__ void pa_set_abort(PaSmem* s) { *reinterpret_cast<volatile int32_t*>(&s->abort_flag) = 1; }

// map_qn: q_nope [T, 128 * 128] bf16; map_qr: q_rope [T, 128 * 64]; map_k / map_v: K_nope (bf16) /
// V (fp16) [B * lpad, 128 * 128]; map_kr: the rope keys [B * lpad, 64]. All boxes are 128 rows x 64
// columns with the 128-byte swizzle.
__global__ void __launch_bounds__(kPaThreads, 1)
    prefill_attn_kernel(const __grid_constant__ CUtensorMap map_qn, const __grid_constant__ CUtensorMap map_qr,
                        const __grid_constant__ CUtensorMap map_k, const __grid_constant__ CUtensorMap map_v,
                        const __grid_constant__ CUtensorMap map_kr, PrefillArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* sQ = sm;
  uint8_t* kst0 = sm + kPaQBytes;                      // key tiles
  uint8_t* vst0 = kst0 + kPaStages * kPaKBytes;        // value tiles
  PaSmem* S = reinterpret_cast<PaSmem*>(vst0 + kPaStages * kPaVBytes);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    tc::mbar_init(&S->q_full, 1);
    tc::mbar_init(&S->q_empty, 1);
    for (int s = 0; s < kPaStages; ++s) {
      tc::mbar_init(&S->k_full[s], 1);
      tc::mbar_init(&S->k_empty[s], 1);
      tc::mbar_init(&S->v_full[s], 1);
      tc::mbar_init(&S->v_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      tc::mbar_init(&S->s_full[s], 1);
      tc::mbar_init(&S->s_free[s], kPaSoftmaxWarps);
      tc::mbar_init(&S->p_full[s], kPaSoftmaxWarps);
      tc::mbar_init(&S->o_done[s], 1);
    }
    tc::mbar_init(&S->drain, 1);
    S->abort_flag = 0;
    tc::fence_mbar_init();
    tc::tma_prefetch_map(&map_qn);
    tc::tma_prefetch_map(&map_qr);
    tc::tma_prefetch_map(&map_k);
    tc::tma_prefetch_map(&map_v);
    tc::tma_prefetch_map(&map_kr);
  }
  if (warp == kPaSoftmaxWarps + 1) tc::tmem_alloc<512>(&S->tmem_base);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tm = S->tmem_base;
  // K_nope and V come from the kv_up kernel ahead of this one
  asm volatile("griddepcontrol.wait;" ::: "memory");

  const int64_t n_units = static_cast<int64_t>(a.batch) * kH * a.qt_max;
  if (warp == kPaSoftmaxWarps) {
    // ------------------------------------------------------------ producer
    // key tile g goes out as soon as the score MMA of tile g - 2 completed; value tile g - 1 after
    // it (its PV comes after the softmax of tile g - 1), once the PV of tile g - 3 completed
    if (lane == 0) {
      uint32_t n = 0, g = 0, gv = 0;   // units, key tiles and value tiles loaded
      int32_t pend_y = 0, pend_x = 0;  // value tile waiting to go out (when gv < g)
      bool ok = true;
      auto load_v = [&]() -> bool {
        const int st = gv % kPaStages;
        if (gv >= kPaStages && !tc::mbar_wait(&S->v_empty[st], ((gv / kPaStages) - 1) & 1)) return false;
        uint8_t* dst = vst0 + st * kPaVBytes;
        tc::mbar_arrive_expect_tx(&S->v_full[st], kPaVBytes);
        tc::tma_load_2d(dst, &map_v, pend_x, pend_y, &S->v_full[st]);
        tc::tma_load_2d(dst + kPfBox, &map_v, pend_x + 64, pend_y, &S->v_full[st]);
        ++gv;
        return true;
      };
      for (int64_t u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
        const PaUnit x = pa_unit(a, u);
        if (!x.live) continue;
        if (n > 0) ok = tc::mbar_wait(&S->q_empty, (n - 1) & 1);
        if (!ok || pa_aborted(S)) { ok = false; break; }
        tc::mbar_arrive_expect_tx(&S->q_full, kPaQBytes);
        tc::tma_load_2d(sQ, &map_qn, x.head * kDh, x.q0, &S->q_full);
        tc::tma_load_2d(sQ + kPfBox, &map_qn, x.head * kDh + 64, x.q0, &S->q_full);
        tc::tma_load_2d(sQ + 2 * kPfBox, &map_qr, x.head * kDr, x.q0, &S->q_full);
        ++n;
        // the next unit's queries into L2 while this unit runs
        for (int64_t w = u + gridDim.x; w < n_units; w += gridDim.x) {
          const PaUnit y = pa_unit(a, w);
          if (!y.live) continue;
          pf_prefetch_2d(&map_qn, y.head * kDh, y.q0);
          pf_prefetch_2d(&map_qn, y.head * kDh + 64, y.q0);
          pf_prefetch_2d(&map_qr, y.head * kDr, y.q0);
          break;
        }
        const int64_t krow0 = static_cast<int64_t>(x.b) * a.lpad;
        for (int j = 0; j < x.nk && ok; ++j, ++g) {
          const int st = g % kPaStages;
          if (g >= kPaStages) ok = tc::mbar_wait(&S->k_empty[st], ((g / kPaStages) - 1) & 1);
          if (!ok) break;
          uint8_t* kst = kst0 + st * kPaKBytes;
          const int32_t yk = static_cast<int32_t>(krow0 + static_cast<int64_t>(j) * kPfRows);
          tc::mbar_arrive_expect_tx(&S->k_full[st], kPaKBytes);
          tc::tma_load_2d(kst, &map_k, x.head * kDh, yk, &S->k_full[st]);
          tc::tma_load_2d(kst + kPfBox, &map_k, x.head * kDh + 64, yk, &S->k_full[st]);
          tc::tma_load_2d(kst + 2 * kPfBox, &map_kr, 0, yk, &S->k_full[st]);
          if (gv < g) ok = load_v();
          pend_x = x.head * kDh;
          pend_y = yk;
        }
      }
      if (ok && gv < g) ok = load_v();
      if (!ok) pa_set_abort(S);
      if (n > 0) tc::mbar_wait(&S->q_full, (n - 1) & 1);
      for (uint32_t q = g > kPaStages ? g - kPaStages : 0; q < g; ++q)
        tc::mbar_wait(&S->k_full[q % kPaStages], (q / kPaStages) & 1);
      for (uint32_t q = gv > kPaStages ? gv - kPaStages : 0; q < gv; ++q)
        tc::mbar_wait(&S->v_full[q % kPaStages], (q / kPaStages) & 1);
    }
  } else if (warp == kPaSoftmaxWarps + 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc_s = tc::idesc_bf16_f32(128, 128, 0, 0);
      const uint32_t idesc_o = idesc_f16_f32(128, 128, 0, 1);
      const uint64_t qdesc0 = tc::sdesc_sw128(tc::smem_u32(sQ), 16, 1024);         // K-major Q
      const uint64_t kdesc0 = tc::sdesc_sw128(tc::smem_u32(kst0), 16, 1024);       // K-major keys, stage 0
      const uint64_t vdesc0 = tc::sdesc_sw128(tc::smem_u32(vst0), kPfBox, 1024);   // MN-major V, stage 0
      uint32_t n = 0, g = 0;
      bool ok = true;
      // O (+)= P V of key tile gg (P from TMEM, 16 keys per MMA)
      auto issue_pv = [&](uint32_t gg, bool first) -> bool {
        const uint32_t s = gg & 1;
        bool good = tc::mbar_wait(&S->v_full[gg % kPaStages], (gg / kPaStages) & 1);
        if (good) good = tc::mbar_wait(&S->p_full[s], (gg >> 1) & 1);
        if (!good || pa_aborted(S)) return false;
        tc::tc_fence_after();
#pragma unroll
        for (int k = 0; k < 8; ++k)
          tc::mma_ts(tm + kPaTmO, tm + kPaTmP + 64 * s + 8 * k,
                     vdesc0 + static_cast<uint64_t>(((gg % kPaStages) * kPaVBytes + 2048 * k) >> 4), idesc_o,
                     (first && k == 0) ? 0u : 1u);
        tc::mma_commit(&S->o_done[s]);
        tc::mma_commit(&S->v_empty[gg % kPaStages]);
        return true;
      };
      for (int64_t u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
        const PaUnit x = pa_unit(a, u);
        if (!x.live) continue;
        ok = tc::mbar_wait(&S->q_full, n & 1);
        for (int j = 0; j < x.nk && ok; ++j, ++g) {
          const uint32_t s = g & 1;
          ok = tc::mbar_wait(&S->k_full[g % kPaStages], (g / kPaStages) & 1);
          if (ok && g >= 2) ok = tc::mbar_wait(&S->s_free[s], ((g - 2) >> 1) & 1);
          if (!ok || pa_aborted(S)) { ok = false; break; }
          tc::tc_fence_after();
          const uint32_t kst = (g % kPaStages) * kPaKBytes;
#pragma unroll
          for (int k = 0; k < 12; ++k) {
            const uint32_t off = (k >> 2) * kPfBox + (k & 3) * 32;
            tc::mma_ss(tm + kPaTmS + 128 * s, qdesc0 + static_cast<uint64_t>(off >> 4),
                       kdesc0 + static_cast<uint64_t>((kst + off) >> 4), idesc_s, k > 0 ? 1u : 0u);
          }
          tc::mma_commit(&S->s_full[s]);
          tc::mma_commit(&S->k_empty[g % kPaStages]);
          if (j == x.nk - 1) tc::mma_commit(&S->q_empty);
          if (j >= 1) ok = issue_pv(g - 1, j == 1);
        }
        if (ok) ok = issue_pv(g - 1, x.nk == 1);
        ++n;
      }
      if (!ok) pa_set_abort(S);
      tc::mma_commit(&S->drain);
      tc::mbar_wait(&S->drain, 0);
    }
  } else {
    // ------------------------------------------------------------ softmax (warps 0-7)
    // warp w: TMEM lane quarter w & 3 (query rows 32 (w & 3) .. + 31), key columns 64 (w >> 2) .. + 63
    // of each tile and O columns 64 (w >> 2) .. + 63
    const int q4 = warp & 3, hc = warp >> 2;
    const int row = 32 * q4 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(32 * q4) << 16;
    const float sl = a.scale_log2;
    uint32_t g = 0;
    bool ok = true;
    for (int64_t u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
      const PaUnit x = pa_unit(a, u);
      if (!x.live) continue;
      const int qp = x.p0 + kPfRows * x.t + row;   // position of this row's token
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
        if (lane == 0) tc::mbar_arrive(&S->s_free[s]);
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
        if (lane == 0) tc::mbar_arrive(&S->p_full[s]);
      }
      // ---- epilogue: out = O / l for the rows that are this unit's tokens
      if (alive) alive = __all_sync(0xffffffffu, tc::mbar_wait(&S->o_done[(g - 1) & 1], ((g - 1) >> 1) & 1));
      tc::tc_fence_after();
      S->red_l[hc][row] = l;
      tc::named_sync(1 + q4, 64);
      const float inv = 1.f / (S->red_l[0][row] + S->red_l[1][row]);
      const bool valid = kPfRows * x.t + row < x.n;
      float* dst = a.out + (static_cast<int64_t>(x.q0 + row) * kH + x.head) * kDh + 64 * hc;
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
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  if (warp == kPaSoftmaxWarps + 1) tc::tmem_dealloc<512>(tm);
}

}  // namespace tcd
}  // namespace mla
