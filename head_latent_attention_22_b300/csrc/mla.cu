// Host side of the MLA C ABI (include/mla.h): argument checks, planning of
// the split over sequence blocks, workspace layout and kernel launches. The
// whole library is this one translation unit.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <mutex>
#include <string>

#include "append.cuh"
#include "attend_pair.cuh"
#include "common.cuh"
#include "decode_simt.cuh"
#include "decode_tc.cuh"
#include "fold.cuh"
#include "prefill.cuh"
#include "tmap.cuh"

namespace mla {
namespace {

thread_local std::string g_last_error;

// Optional per-kernel timing events (see mla_set_stage_events).
struct StageEvents {
  cudaEvent_t ev[8];
  int n = 0;
};
thread_local StageEvents g_stage;

inline void stage_mark(int k, cudaStream_t st) {
  if (k < g_stage.n) cudaEventRecord(g_stage.ev[k], st);
}

mla_status fail(mla_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}

mla_status cuda_fail(cudaError_t e, const char* what) {
  return fail(MLA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

mla_status check_config(const mla_config* c) {
  if (!c) return fail(MLA_ERR_INVALID_ARG, "cfg is NULL");
  if (c->n_heads < 1 || c->d_c < 1 || c->d_rope < 2 || (c->d_rope & 1) || c->d_head < 1 || c->page_size < 1)
    return fail(MLA_ERR_INVALID_ARG, "bad sizes: n_heads=%d d_c=%d d_rope=%d d_head=%d page_size=%d",
                c->n_heads, c->d_c, c->d_rope, c->d_head, c->page_size);
  if (c->io_dtype != MLA_DTYPE_BF16 && c->io_dtype != MLA_DTYPE_FP32)
    return fail(MLA_ERR_INVALID_ARG, "io_dtype must be BF16 or FP32");
  if (c->cache_dtype != MLA_DTYPE_BF16 && c->cache_dtype != MLA_DTYPE_FP32 &&
      c->cache_dtype != MLA_DTYPE_FP8_E4M3_B128)
    return fail(MLA_ERR_INVALID_ARG, "unknown cache_dtype %d", c->cache_dtype);
  if (c->cache_dtype == MLA_DTYPE_FP8_E4M3_B128 && (c->d_c % 128) != 0)
    return fail(MLA_ERR_INVALID_ARG, "FP8 cache needs d_c %% 128 == 0 (d_c=%d)", c->d_c);
  if (!(c->eps >= 0.f) || !(c->rope_theta > 0.f) || !std::isfinite(c->scale))
    return fail(MLA_ERR_INVALID_ARG, "bad eps/rope_theta/scale");
  if (c->yarn_factor > 1.f &&
      (!std::isfinite(c->yarn_factor) || !(c->yarn_beta > c->yarn_alpha) || !std::isfinite(c->yarn_alpha) ||
       !std::isfinite(c->yarn_beta) || !std::isfinite(c->yarn_mscale) || c->yarn_orig_len < 1))
    return fail(MLA_ERR_INVALID_ARG, "bad YaRN fields: factor=%g alpha=%g beta=%g mscale=%g orig_len=%d",
                c->yarn_factor, c->yarn_alpha, c->yarn_beta, c->yarn_mscale, c->yarn_orig_len);
  return MLA_OK;
}

bool yarn_on(const mla_config* c) { return c->yarn_factor > 1.f; }

// RoPE frequencies of cfg (plain, or YaRN-scaled), as the kernels take them.
RopeFreq rope_freq_of(const mla_config* c) {
  RopeFreq r{};
  r.log_theta = std::log(static_cast<double>(c->rope_theta));
  if (yarn_on(c)) {
    r.yarn_s = c->yarn_factor;
    r.yarn_alpha = c->yarn_alpha;
    r.yarn_beta = c->yarn_beta;
    r.yarn_orig_len = c->yarn_orig_len;
  }
  r.n_table = 0;
  if (c->d_rope / 2 <= kRopeTable) {
    for (int m = 0; m < c->d_rope / 2; ++m) r.table[m] = rope_freq_rule(r, m, c->d_rope);
    r.n_table = c->d_rope / 2;
  }
  return r;
}

// Softmax scale of the decode: cfg->scale (1/sqrt(d_head + d_rope) when it is
// not positive: the width of the full key [k_C ; k_R]), times YaRN's logit
// factor (mscale ln s + 1)^2.
float softmax_scale(const mla_config* c) {
  const double base = c->scale > 0.f ? static_cast<double>(c->scale)
                                     : 1.0 / std::sqrt(static_cast<double>(c->d_head + c->d_rope));
  if (!yarn_on(c)) return static_cast<float>(base);
  const double m = static_cast<double>(c->yarn_mscale) * std::log(static_cast<double>(c->yarn_factor)) + 1.0;
  return static_cast<float>(base * m * m);
}

cudaStream_t as_stream(void* s) { return static_cast<cudaStream_t>(s); }

int current_sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 148;
  return n;
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Virtual sequences of mla_decode_multi: v = b * q_len + k sees the first
// seq_lens[b] - (q_len - 1 - k) rows of sequence b, through sequence b's pages.
__global__ void expand_multi_kernel(const int32_t* seq_lens, const int32_t* block_table, int32_t* lens_v,
                                    int32_t* table_v, int batch, int q_len, int max_pages) {
  const int64_t n = static_cast<int64_t>(batch) * q_len * max_pages;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int p = static_cast<int>(i % max_pages);
    const int64_t v = i / max_pages;
    const int b = static_cast<int>(v / q_len), k = static_cast<int>(v % q_len);
    table_v[i] = block_table ? block_table[static_cast<int64_t>(b) * max_pages + p]
                             : static_cast<int32_t>(static_cast<int64_t>(b) * max_pages + p);
    if (p == 0) {
      const int L = seq_lens[b] - (q_len - 1 - k);
      lens_v[v] = L > 0 ? L : 0;
    }
  }
}

size_t multi_prefix_bytes(int32_t batch, int32_t q_len, int32_t max_pages) {
  const size_t nv = static_cast<size_t>(batch) * q_len;
  return align_up(nv * 4, 256) + align_up(nv * static_cast<size_t>(max_pages) * 4, 256);
}

// ------------------------------------------------------------------ SIMT decode plan
struct SimtPlan {
  int n_splits, split_tokens;
  size_t off_qlat, off_o, off_m, off_l, bytes;
};

SimtPlan simt_plan(const mla_config* c, int batch, int max_seq_len) {
  SimtPlan p{};
  const int L = max_seq_len < 1 ? 1 : max_seq_len;
  int splits = (L + 511) / 512;
  if (splits > 64) splits = 64;
  if (splits < 1) splits = 1;
  int per = (L + splits - 1) / splits;
  per = (per + kSimtTileTokens - 1) / kSimtTileTokens * kSimtTileTokens;
  splits = (L + per - 1) / per;
  p.n_splits = splits;
  p.split_tokens = per;
  const size_t BH = static_cast<size_t>(batch) * c->n_heads;
  size_t off = 0;
  p.off_qlat = off;
  off = align_up(off + BH * (c->d_c + c->d_rope) * 4, 256);
  p.off_o = off;
  off = align_up(off + BH * splits * c->d_c * 4, 256);
  p.off_m = off;
  off = align_up(off + BH * splits * 4, 256);
  p.off_l = off;
  off = align_up(off + BH * splits * 4, 256);
  p.bytes = off;
  return p;
}

mla_status decode_simt(const mla_config* c, const void* q_nope, const void* q_rope, const void* w_uk,
                       const void* w_uv, const void* pool, int64_t num_pages, const int32_t* block_table,
                       const int32_t* seq_lens, int batch, int max_pages, int max_seq_len, float* out,
                       void* workspace, size_t workspace_bytes, cudaStream_t st) {
  if (c->d_c > kSimtMaxDc) return fail(MLA_ERR_UNSUPPORTED, "CUDA-core decode supports d_c <= %d", kSimtMaxDc);
  const SimtPlan p = simt_plan(c, batch, max_seq_len);
  if (workspace_bytes < p.bytes)
    return fail(MLA_ERR_INVALID_ARG, "workspace too small: %zu < %zu", workspace_bytes, p.bytes);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  SimtArgs a{};
  a.q_nope = q_nope; a.q_rope = q_rope; a.w_uk = w_uk; a.w_uv = w_uv;
  a.pool = static_cast<const uint8_t*>(pool);
  a.num_pages = num_pages; a.block_table = block_table; a.seq_lens = seq_lens;
  a.batch = batch; a.max_pages = max_pages; a.n_heads = c->n_heads; a.d_c = c->d_c;
  a.d_rope = c->d_rope; a.d_head = c->d_head; a.page_size = c->page_size;
  a.cache_dtype = c->cache_dtype;
  a.row_bytes = static_cast<int64_t>(row_bytes_of(c->cache_dtype, c->d_c, c->d_rope));
  a.scale_log2 = softmax_scale(c) * 1.4426950408889634f;
  a.out = out;
  a.q_lat = reinterpret_cast<float*>(ws + p.off_qlat);
  a.part_o = reinterpret_cast<float*>(ws + p.off_o);
  a.part_m = reinterpret_cast<float*>(ws + p.off_m);
  a.part_l = reinterpret_cast<float*>(ws + p.off_l);
  a.n_splits = p.n_splits;
  a.split_tokens = p.split_tokens;
  a.max_seq_len = max_seq_len;

  const int D = c->d_c + c->d_rope;
  const size_t smem_att = static_cast<size_t>(kSimtHeadsPerCta + kSimtTileTokens) * D * 4;
  if (smem_att > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(attend_simt_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem_att));
    if (e != cudaSuccess) return cuda_fail(e, "attend_simt smem attribute");
  }
  const dim3 g_abs(c->n_heads, batch);
  stage_mark(0, st);
  if (c->io_dtype == MLA_DTYPE_BF16)
    absorb_simt_kernel<uint16_t><<<g_abs, 128, c->d_head * 4, st>>>(a);
  else
    absorb_simt_kernel<float><<<g_abs, 128, c->d_head * 4, st>>>(a);
  stage_mark(1, st);
  const dim3 g_att(p.n_splits, (c->n_heads + kSimtHeadsPerCta - 1) / kSimtHeadsPerCta, batch);
  attend_simt_kernel<<<g_att, 32 * kSimtHeadsPerCta, smem_att, st>>>(a);
  stage_mark(2, st);
  if (c->io_dtype == MLA_DTYPE_BF16)
    combine_simt_kernel<uint16_t><<<g_abs, 256, c->d_c * 4, st>>>(a);
  else
    combine_simt_kernel<float><<<g_abs, 256, c->d_c * 4, st>>>(a);
  stage_mark(3, st);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "decode (CUDA-core) launch");
  return MLA_OK;
}

// ------------------------------------------------------------------ tensor-core decode
// The tcgen05 kernels cover the DeepSeek-V2 shape with bf16 queries, weights
// and cache, and pages holding whole 64-token tiles.
bool tc_supported(const mla_config* c) {
  return c->n_heads == tcd::kH && c->d_c == tcd::kDc && c->d_rope == tcd::kDr && c->d_head == tcd::kDh &&
         c->io_dtype == MLA_DTYPE_BF16 &&
         (c->cache_dtype == MLA_DTYPE_BF16 || c->cache_dtype == MLA_DTYPE_FP8_E4M3_B128) &&
         c->page_size % tcd::kTile == 0;
}

// Clusters the workspace is sized for; a launch never uses more.
constexpr int kMaxClusters = 128;

struct TcPlan {
  int nb, slots;
  size_t off_qlat, off_lens, off_cum, off_first, off_start, off_c0, off_c1, off_tiles, off_rows, off_ml, off_o, off_hi,
      off_lo, bytes;
};

TcPlan tc_plan(int batch) {
  TcPlan p{};
  p.nb = batch >= 128 ? 128 : (batch + 15) / 16 * 16;
  p.slots = batch + kMaxClusters - 1;
  size_t off = 0;
  p.off_qlat = off;
  off = align_up(off + static_cast<size_t>(batch) * tcd::kH * tcd::kRow * 2, 256);
  p.off_lens = off;
  off = align_up(off + static_cast<size_t>(batch) * 4, 256);
  p.off_cum = off;
  off = align_up(off + static_cast<size_t>(batch + 1) * 4, 256);
  p.off_first = off;
  off = align_up(off + static_cast<size_t>(kMaxClusters) * 4, 256);
  p.off_start = off;
  off = align_up(off + static_cast<size_t>(kMaxClusters + 1) * 4, 256);
  p.off_c0 = off;
  off = align_up(off + static_cast<size_t>(batch) * 4, 256);
  p.off_c1 = off;
  off = align_up(off + static_cast<size_t>(batch) * 4, 256);
  p.off_tiles = off;
  off = align_up(off + static_cast<size_t>(kMaxClusters) * 4, 256);
  p.off_rows = off;
  off = align_up(off + static_cast<size_t>(kMaxClusters) * tcd::kPlanRows * 4, 256);
  p.off_ml = off;
  off = align_up(off + static_cast<size_t>(p.slots) * tcd::kH * 8, 256);
  p.off_o = off;
  off = align_up(off + static_cast<size_t>(p.slots) * tcd::kH * tcd::kDc * 4, 256);
  p.off_hi = off;
  off = align_up(off + static_cast<size_t>(batch) * tcd::kH * tcd::kDc * 2, 256);
  p.off_lo = off;
  off = align_up(off + static_cast<size_t>(batch) * tcd::kH * tcd::kDc * 2, 256);
  p.bytes = off;
  return p;
}

static_assert(tcd::PairCfg<false>::kSmem <= 232448, "attend kernel shared memory exceeds the 227 KB a CTA may use");
static_assert(tcd::PairCfg<true>::kSmem <= 232448, "attend kernel (FP8 cache) shared memory exceeds 227 KB");
constexpr size_t kUvSmem = 1024 + tcd::kUvSmem;
size_t absorb_smem(int nb) { return 1024 + 4 * 16384 + 2 * static_cast<size_t>(nb) * 128 + 64; }
static_assert(4 * static_cast<size_t>(tcd::kPlanSmemRows) <= 1024 + 4 * 16384,
              "the plan block's prefix sums fit the absorb kernel's shared memory");

struct TcDeviceState {
  bool ready = false;
  int clusters[2] = {0, 0};   // bf16 cache (pair kernel), FP8 cache
};
std::mutex g_tc_mu;
TcDeviceState g_tc_state[64];

// Number of two-CTA clusters of attend kernel `fn` (threads, shared memory) that fit on the GPU at once.
mla_status cluster_count(const void* fn, int threads, size_t smem, int* clusters) {
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return cuda_fail(e, "attend smem attribute");
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(2 * kMaxClusters);
  lc.blockDim = dim3(threads);
  lc.dynamicSmemBytes = smem;
  int n = 0;
  if ((e = cudaOccupancyMaxActiveClusters(&n, fn, &lc)) != cudaSuccess || n < 1)
    return cuda_fail(e == cudaSuccess ? cudaErrorInvalidConfiguration : e, "attend cluster occupancy");
  const int half_sms = current_sm_count() / 2;
  n = n < half_sms ? n : half_sms;
  *clusters = n < kMaxClusters ? n : kMaxClusters;
  return MLA_OK;
}

// Per device, once: shared-memory limits of the kernels and the number of
// two-CTA clusters of each attend kernel that fit on the GPU at once.
// clusters[0]: bf16 cache, clusters[1]: FP8 cache.
mla_status tc_device_setup(int* clusters) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= 64) return fail(MLA_ERR_UNSUPPORTED, "device %d beyond 64 devices", dev);
  std::lock_guard<std::mutex> lock(g_tc_mu);
  TcDeviceState& st = g_tc_state[dev];
  if (!st.ready) {
    if ((e = cudaFuncSetAttribute(tcd::absorb_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  static_cast<int>(absorb_smem(128)))) != cudaSuccess)
      return cuda_fail(e, "absorb smem attribute");
    if ((e = cudaFuncSetAttribute(tcd::uv_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  static_cast<int>(kUvSmem))) != cudaSuccess)
      return cuda_fail(e, "uv smem attribute");
    mla_status s = cluster_count(reinterpret_cast<const void*>(tcd::attend_pair_kernel<false>),
                                 tcd::PairCfg<false>::kThreads, tcd::PairCfg<false>::kSmem, &st.clusters[0]);
    if (s != MLA_OK) return s;
    if ((s = cluster_count(reinterpret_cast<const void*>(tcd::attend_pair_kernel<true>), tcd::PairCfg<true>::kThreads,
                           tcd::PairCfg<true>::kSmem, &st.clusters[1])) != MLA_OK)
      return s;
    st.ready = true;
  }
  clusters[0] = st.clusters[0];
  clusters[1] = st.clusters[1];
  return MLA_OK;
}

mla_status launch_pdl(const void* fn, dim3 grid, dim3 block, size_t smem, cudaStream_t st, void** args) {
  cudaLaunchConfig_t lc = {};
  lc.gridDim = grid;
  lc.blockDim = block;
  lc.dynamicSmemBytes = smem;
  lc.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = attr;
  lc.numAttrs = g_stage.n > 0 ? 0 : 1;   // per-kernel timing wants the kernels apart
  cudaError_t e = cudaLaunchKernelExC(&lc, fn, args);
  if (e != cudaSuccess) return cuda_fail(e, "tensor-core decode launch");
  return MLA_OK;
}

// Split of the hidden-output GEMM's 65,536-wide contraction: about two waves of two CTAs per SM.
int out_groups(int hidden) {
  const int m_tiles = hidden / 128;
  const int want = (4 * current_sm_count() + m_tiles - 1) / m_tiles;
  return want < 1 ? 1 : (want > 64 ? 64 : want);
}

size_t out_partial_bytes(int batch, int hidden) {
  return align_up(static_cast<size_t>(out_groups(hidden)) * batch * hidden * 4, 256);
}

// w_ouv == NULL: the per-head outputs out[B, H, d_h] (W_UV after the merge). Otherwise W_UV folded into
// W_O: out[B, hidden] = W_OUV o_lat.
mla_status decode_tc(const mla_config* c, const void* q_nope, const void* q_rope, const void* w_uk, const void* w_uv,
                     const void* pool, int64_t num_pages, const int32_t* block_table, const int32_t* seq_lens,
                     int batch, int max_pages, int max_seq_len, float* out, void* workspace, size_t workspace_bytes,
                     cudaStream_t st, const void* w_ouv = nullptr, int hidden = 0) {
  const TcPlan p = tc_plan(batch);
  const size_t need = p.bytes + (w_ouv ? out_partial_bytes(batch, hidden) : 0);
  if (workspace_bytes < need)
    return fail(MLA_ERR_INVALID_ARG, "workspace too small: %zu < %zu", workspace_bytes, need);
  const int64_t pool_rows = num_pages * static_cast<int64_t>(c->page_size);
  if (pool_rows >= (static_cast<int64_t>(1) << 31))
    return fail(MLA_ERR_UNSUPPORTED, "pool of %lld rows exceeds the 2^31 rows a tile coordinate can address",
                static_cast<long long>(pool_rows));
  const bool f8 = c->cache_dtype == MLA_DTYPE_FP8_E4M3_B128;
  int ncl2[2] = {0, 0};
  mla_status s = tc_device_setup(ncl2);
  if (s != MLA_OK) return s;
  const int ncl = ncl2[f8 ? 1 : 0];
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  tcd::Plan plan{reinterpret_cast<int32_t*>(ws + p.off_lens), reinterpret_cast<int32_t*>(ws + p.off_cum),
                 reinterpret_cast<int32_t*>(ws + p.off_first), reinterpret_cast<int32_t*>(ws + p.off_start),
                 reinterpret_cast<int32_t*>(ws + p.off_c0), reinterpret_cast<int32_t*>(ws + p.off_c1),
                 reinterpret_cast<int32_t*>(ws + p.off_tiles), reinterpret_cast<int32_t*>(ws + p.off_rows)};
  uint16_t* q_lat = reinterpret_cast<uint16_t*>(ws + p.off_qlat);

  CUtensorMap m_lat, m_scale, m_rope, m_wuk, m_wuv, m_qn, m_hi, m_lo, m_q, m_qr;
  uint16_t* o_hi = reinterpret_cast<uint16_t*>(ws + p.off_hi);
  uint16_t* o_lo = reinterpret_cast<uint16_t*>(ws + p.off_lo);
  const CUtensorMapDataType BF = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const CUtensorMapSwizzle SW = CU_TENSOR_MAP_SWIZZLE_128B;
  const CUtensorMapSwizzle SW64 = CU_TENSOR_MAP_SWIZZLE_64B;
  bool maps_ok;
  if (f8) {
    // FP8 row: 512 E4M3 codes, 4 fp32 block scales, 64 bf16 rope values (656 bytes)
    const uint64_t rb = tcd::kDc + 4 * (tcd::kDc / 128) + 2 * tcd::kDr;
    const CUtensorMapDataType U8 = CU_TENSOR_MAP_DATA_TYPE_UINT8;
    const CUtensorMapSwizzle NS = CU_TENSOR_MAP_SWIZZLE_NONE;
    const uint8_t* rope_base = static_cast<const uint8_t*>(pool) + tcd::kDc + 4 * (tcd::kDc / 128);
    maps_ok = make_map_2d(&m_lat, pool, U8, rb, static_cast<uint64_t>(pool_rows), rb, 256, tcd::kTile, NS) &&
              make_map_2d(&m_scale, pool, U8, rb, static_cast<uint64_t>(pool_rows), rb, 16, tcd::kTile, NS) &&
              make_map_2d(&m_rope, rope_base, BF, tcd::kDr, static_cast<uint64_t>(pool_rows), rb, 32, tcd::kTile,
                          SW64);
  } else {
    maps_ok = make_map_2d(&m_lat, pool, BF, tcd::kRow, static_cast<uint64_t>(pool_rows), tcd::kRow * 2, 64, tcd::kTile,
                          SW) &&
              make_map_2d(&m_rope, pool, BF, tcd::kRow, static_cast<uint64_t>(pool_rows), tcd::kRow * 2, 32,
                          tcd::kTile, SW64);
    m_scale = m_lat;   // unused with a bf16 pool
  }
  // Q_lat row-major [B * 128, 576], read in boxes of 16 heads x 64 values (latent) and 16 heads x 32 (rope)
  maps_ok = maps_ok &&
            make_map_2d(&m_q, q_lat, BF, tcd::kRow, static_cast<uint64_t>(batch) * tcd::kH, tcd::kRow * 2, 64, 16,
                        SW) &&
            make_map_2d(&m_qr, q_lat, BF, tcd::kRow, static_cast<uint64_t>(batch) * tcd::kH, tcd::kRow * 2, 32, 16,
                        SW64);
  const int out_nb = (batch + 15) / 16 * 16;
  const CUtensorMapDataType F16 = CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  CUtensorMap m_wouv, m_ohi, m_olo;
  if (w_ouv)
    maps_ok = maps_ok &&
              make_map_2d(&m_wouv, w_ouv, F16, static_cast<uint64_t>(tcd::kH) * tcd::kDc, static_cast<uint64_t>(hidden),
                          static_cast<uint64_t>(tcd::kH) * tcd::kDc * 2, 64, 128, SW) &&
              make_map_2d(&m_ohi, o_hi, F16, tcd::kH * tcd::kDc, static_cast<uint64_t>(batch), tcd::kH * tcd::kDc * 2, 64,
                          static_cast<uint32_t>(out_nb), SW) &&
              make_map_2d(&m_olo, o_lo, F16, tcd::kH * tcd::kDc, static_cast<uint64_t>(batch), tcd::kH * tcd::kDc * 2, 64,
                          static_cast<uint32_t>(out_nb), SW);
  else
    maps_ok = maps_ok && make_map_2d(&m_wuv, w_uv, BF, tcd::kDc, tcd::kH * tcd::kDh, tcd::kDc * 2, 64, tcd::kDh, SW);
  if (!maps_ok ||
      !make_map_2d(&m_wuk, w_uk, BF, tcd::kDc, tcd::kH * tcd::kDh, tcd::kDc * 2, 64, tcd::kDh, SW) ||
      !make_map_2d(&m_qn, q_nope, BF, tcd::kH * tcd::kDh, static_cast<uint64_t>(batch), tcd::kH * tcd::kDh * 2, 64,
                   static_cast<uint32_t>(p.nb), SW) ||
      !make_map_2d(&m_hi, o_hi, BF, tcd::kH * tcd::kDc, static_cast<uint64_t>(batch), tcd::kH * tcd::kDc * 2, 64,
                   tcd::kUvNb, SW) ||
      !make_map_2d(&m_lo, o_lo, BF, tcd::kH * tcd::kDc, static_cast<uint64_t>(batch), tcd::kH * tcd::kDc * 2, 64,
                   tcd::kUvNb, SW))
    return fail(MLA_ERR_CUDA, "cuTensorMapEncodeTiled refused a tensor description (or the driver entry point is missing)");

  tcd::AbsorbArgs aa{};
  aa.q_rope = static_cast<const uint16_t*>(q_rope);
  aa.seq_lens = seq_lens;
  aa.block_table = block_table;
  aa.num_pages = num_pages;
  aa.max_pages = max_pages;
  aa.page_size = c->page_size;
  aa.q_lat = q_lat;
  aa.plan = plan;
  aa.batch = batch;
  aa.nb = p.nb;
  aa.max_seq_len = max_seq_len;
  aa.ncl = ncl;
  aa.f16_lat = f8 ? 1 : 0;

  tcd::AttendArgs ta{};
  ta.q_lat = q_lat;
  ta.block_table = block_table;
  ta.max_seq_len = max_seq_len;
  ta.plan = plan;
  ta.part_o = reinterpret_cast<float*>(ws + p.off_o);
  ta.part_ml = reinterpret_cast<float*>(ws + p.off_ml);
  ta.num_pages = num_pages;
  ta.batch = batch;
  ta.max_pages = max_pages;
  ta.page_size = c->page_size;
  ta.scale_log2 = softmax_scale(c) * 1.4426950408889634f;

  tcd::MergeArgs ma{};
  ma.plan = plan;
  ma.part_o = ta.part_o;
  ma.part_ml = ta.part_ml;
  ma.o_hi = o_hi;
  ma.o_lo = o_lo;
  ma.batch = batch;
  ma.ncl = ncl;
  ma.f16 = w_ouv ? 1 : 0;

  tcd::UvArgs ua{};
  ua.out = out;
  ua.batch = batch;

  stage_mark(0, st);
  void* absorb_args[] = {&m_wuk, &m_qn, &aa};
  s = launch_pdl(reinterpret_cast<const void*>(tcd::absorb_tc_kernel), dim3(2 * tcd::kH + 1), dim3(tcd::kAbsorbThreads),
                 absorb_smem(p.nb), st, absorb_args);
  if (s != MLA_OK) return s;
  stage_mark(1, st);
  void* attend_args[] = {&m_lat, &m_rope, &m_q, &m_qr, &m_scale, &ta};
  if (f8)
    s = launch_pdl(reinterpret_cast<const void*>(tcd::attend_pair_kernel<true>), dim3(2 * ncl),
                   dim3(tcd::PairCfg<true>::kThreads), tcd::PairCfg<true>::kSmem, st, attend_args);
  else
    s = launch_pdl(reinterpret_cast<const void*>(tcd::attend_pair_kernel<false>), dim3(2 * ncl),
                   dim3(tcd::PairCfg<false>::kThreads), tcd::PairCfg<false>::kSmem, st, attend_args);
  if (s != MLA_OK) return s;
  stage_mark(2, st);
  void* merge_args[] = {&ma};
  // four chunks per CTA once that still gives two CTAs per SM (2 ncl SMs), else one
  if (static_cast<int64_t>(batch) * (tcd::kOChunks / 4) >= 4 * static_cast<int64_t>(ncl))
    s = launch_pdl(reinterpret_cast<const void*>(tcd::merge_kernel<4, 8>), dim3(tcd::kOChunks / 4, batch),
                   dim3(tcd::kH), 0, st, merge_args);
  else
    s = launch_pdl(reinterpret_cast<const void*>(tcd::merge_kernel<1, 16>), dim3(tcd::kOChunks, batch), dim3(tcd::kH),
                   0, st, merge_args);
  if (s != MLA_OK) return s;
  stage_mark(3, st);
  if (w_ouv) {
    tcd::OutArgs oa{};
    oa.partial = reinterpret_cast<float*>(ws + p.bytes);
    oa.batch = batch;
    oa.nb = out_nb;
    oa.hidden = hidden;
    oa.n_groups = out_groups(hidden);
    const size_t osm = tcd::out_smem_bytes(out_nb);
    cudaError_t e = cudaFuncSetAttribute(tcd::out_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(osm));
    if (e != cudaSuccess) return cuda_fail(e, "out_tc smem attribute");
    void* out_args[] = {&m_wouv, &m_ohi, &m_olo, &oa};
    s = launch_pdl(reinterpret_cast<const void*>(tcd::out_tc_kernel), dim3(hidden / 128, oa.n_groups),
                   dim3(tcd::kOutThreads), osm, st, out_args);
    if (s != MLA_OK) return s;
    stage_mark(4, st);
    const float* part = oa.partial;
    int groups = oa.n_groups;
    int64_t count = static_cast<int64_t>(batch) * hidden;
    void* red_args[] = {&part, &out, &groups, &count};
    const int64_t want = (count + 255) / 256;
    s = launch_pdl(reinterpret_cast<const void*>(tcd::out_reduce_kernel), dim3(static_cast<unsigned>(want < 1184 ? want : 1184)),
                   dim3(256), 0, st, red_args);
    if (s != MLA_OK) return s;
    stage_mark(5, st);
    return MLA_OK;
  }
  void* uv_args[] = {&m_wuv, &m_hi, &m_lo, &ua};
  s = launch_pdl(reinterpret_cast<const void*>(tcd::uv_tc_kernel), dim3(tcd::kH), dim3(tcd::kUvThreads), kUvSmem, st,
                 uv_args);
  if (s != MLA_OK) return s;
  stage_mark(4, st);
  return MLA_OK;
}

// ------------------------------------------------------------------ prefill (tensor cores)
// Workspace: K_nope (bf16) and V (fp16) of every row of every sequence, [B * lpad, 128 * 128] each, and
// the rows' rope keys [B * lpad, 64] bf16, with lpad = max_seq_len rounded up to whole 128-row tiles.
struct PfPlan {
  int lpad;
  size_t off_k, off_v, off_kr, bytes;
};

PfPlan pf_plan(int batch, int max_seq_len) {
  PfPlan p{};
  const int L = max_seq_len > 0 ? max_seq_len : 1;
  p.lpad = (L + tcd::kPfRows - 1) / tcd::kPfRows * tcd::kPfRows;
  const size_t kv = static_cast<size_t>(batch) * p.lpad * tcd::kH * tcd::kDh * 2;
  p.off_k = 0;
  p.off_v = align_up(kv, 256);
  p.off_kr = p.off_v + align_up(kv, 256);
  p.bytes = p.off_kr + align_up(static_cast<size_t>(batch) * p.lpad * tcd::kDr * 2, 256);
  return p;
}

static_assert(tcd::kKvSmem <= 232448, "kv_up kernel shared memory exceeds the 227 KB a CTA may use");
static_assert(tcd::kPaSmem <= 232448, "prefill attention kernel shared memory exceeds 227 KB");

bool g_pf_ready[64] = {};

mla_status prefill_tc(const mla_config* c, const void* q_nope, const void* q_rope, const void* w_uk, const void* w_uv,
                      const void* pool, int64_t num_pages, const int32_t* block_table, const int32_t* seq_lens,
                      const int32_t* q_start, int batch, int max_pages, int max_seq_len, int n_tokens, float* out,
                      void* workspace, size_t workspace_bytes, cudaStream_t st) {
  const PfPlan p = pf_plan(batch, max_seq_len);
  if (workspace_bytes < p.bytes)
    return fail(MLA_ERR_INVALID_ARG, "workspace too small: %zu < %zu", workspace_bytes, p.bytes);
  const int64_t pool_rows = num_pages * static_cast<int64_t>(c->page_size);
  const int64_t kv_rows = static_cast<int64_t>(batch) * p.lpad;
  if (pool_rows >= (static_cast<int64_t>(1) << 31) || kv_rows >= (static_cast<int64_t>(1) << 31))
    return fail(MLA_ERR_UNSUPPORTED, "pool or key rows exceed the 2^31 rows a tile coordinate can address");
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= 64) return fail(MLA_ERR_UNSUPPORTED, "device %d beyond 64 devices", dev);
  {
    std::lock_guard<std::mutex> lock(g_tc_mu);
    if (!g_pf_ready[dev]) {
      if ((e = cudaFuncSetAttribute(tcd::kv_up_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    static_cast<int>(tcd::kKvSmem))) != cudaSuccess)
        return cuda_fail(e, "kv_up smem attribute");
      if ((e = cudaFuncSetAttribute(tcd::prefill_attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    static_cast<int>(tcd::kPaSmem))) != cudaSuccess)
        return cuda_fail(e, "prefill attention smem attribute");
      g_pf_ready[dev] = true;
    }
  }
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  uint16_t* k_buf = reinterpret_cast<uint16_t*>(ws + p.off_k);
  uint16_t* v_buf = reinterpret_cast<uint16_t*>(ws + p.off_v);
  uint16_t* kr_buf = reinterpret_cast<uint16_t*>(ws + p.off_kr);
  const CUtensorMapDataType BF = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const CUtensorMapSwizzle SW = CU_TENSOR_MAP_SWIZZLE_128B;
  const uint64_t wkv = static_cast<uint64_t>(tcd::kH) * tcd::kDh;
  CUtensorMap m_lat, m_wuk, m_wuv, m_qn, m_qr, m_k, m_v, m_kr;
  if (!make_map_2d(&m_lat, pool, BF, tcd::kRow, static_cast<uint64_t>(pool_rows), tcd::kRow * 2, 64, 64, SW) ||
      !make_map_2d(&m_wuk, w_uk, BF, tcd::kDc, wkv, tcd::kDc * 2, 64, tcd::kKvNt / 2, SW) ||
      !make_map_2d(&m_wuv, w_uv, BF, tcd::kDc, wkv, tcd::kDc * 2, 64, tcd::kKvNt / 2, SW) ||
      !make_map_2d(&m_qn, q_nope, BF, wkv, static_cast<uint64_t>(n_tokens), wkv * 2, 64, tcd::kPfRows, SW) ||
      !make_map_2d(&m_qr, q_rope, BF, static_cast<uint64_t>(tcd::kH) * tcd::kDr, static_cast<uint64_t>(n_tokens),
                   static_cast<uint64_t>(tcd::kH) * tcd::kDr * 2, 64, tcd::kPfRows, SW) ||
      !make_map_2d(&m_k, k_buf, BF, wkv, static_cast<uint64_t>(kv_rows), wkv * 2, 64, 64, SW) ||
      !make_map_2d(&m_v, v_buf, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, wkv, static_cast<uint64_t>(kv_rows), wkv * 2, 64,
                   tcd::kPfRows, SW) ||
      !make_map_2d(&m_kr, kr_buf, BF, tcd::kDr, static_cast<uint64_t>(kv_rows), tcd::kDr * 2, 64, 64, SW))
    return fail(MLA_ERR_CUDA, "cuTensorMapEncodeTiled refused a tensor description (or the driver entry point is missing)");

  tcd::KvUpArgs ka{};
  ka.block_table = block_table;
  ka.seq_lens = seq_lens;
  ka.pool = static_cast<const uint16_t*>(pool);
  ka.k_buf = k_buf;
  ka.v_buf = v_buf;
  ka.kr_buf = kr_buf;
  ka.num_pages = num_pages;
  ka.batch = batch;
  ka.max_pages = max_pages;
  ka.page_size = c->page_size;
  ka.max_seq_len = max_seq_len;
  ka.lpad = p.lpad;

  tcd::PrefillArgs pa{};
  pa.block_table = block_table;
  pa.seq_lens = seq_lens;
  pa.q_start = q_start;
  pa.out = out;
  pa.num_pages = num_pages;
  pa.batch = batch;
  pa.max_pages = max_pages;
  pa.page_size = c->page_size;
  pa.max_seq_len = max_seq_len;
  pa.lpad = p.lpad;
  pa.n_tokens = n_tokens;
  pa.qp_max = (p.lpad + 2 * tcd::kPfRows - 1) / (2 * tcd::kPfRows);
  pa.scale_log2 = softmax_scale(c) * 1.4426950408889634f;

  const int sms = current_sm_count();
  const int64_t items = ((static_cast<int64_t>(p.lpad / tcd::kPfRows) * batch + 1) / 2) * tcd::kKvGroups;
  int kv_clusters = 0;
  mla_status ks = cluster_count(reinterpret_cast<const void*>(tcd::kv_up_kernel), tcd::kKvThreads, tcd::kKvSmem,
                                &kv_clusters);
  if (ks != MLA_OK) return ks;
  if (items < kv_clusters) kv_clusters = static_cast<int>(items);
  const int64_t units = static_cast<int64_t>(batch) * tcd::kH * pa.qp_max;
  int pa_clusters = 0;
  mla_status cs = cluster_count(reinterpret_cast<const void*>(tcd::prefill_attn_kernel), tcd::kPaThreads, tcd::kPaSmem,
                                &pa_clusters);
  if (cs != MLA_OK) return cs;
  if (units < pa_clusters) pa_clusters = static_cast<int>(units);
  stage_mark(0, st);
  void* kv_args[] = {&m_lat, &m_wuk, &m_wuv, &ka};
  mla_status s = launch_pdl(reinterpret_cast<const void*>(tcd::kv_up_kernel), dim3(2 * kv_clusters),
                            dim3(tcd::kKvThreads), tcd::kKvSmem, st, kv_args);
  if (s != MLA_OK) return s;
  stage_mark(1, st);
  void* pa_args[] = {&m_qn, &m_qr, &m_k, &m_v, &m_kr, &pa};
  s = launch_pdl(reinterpret_cast<const void*>(tcd::prefill_attn_kernel), dim3(2 * pa_clusters),
                 dim3(tcd::kPaThreads), tcd::kPaSmem, st, pa_args);
  if (s != MLA_OK) return s;
  stage_mark(2, st);
  return MLA_OK;
}

// ------------------------------------------------------------------ fixed scratch
// Scratch of mla_decode_static_scratch: one array per device, for callers
// that cannot allocate. Host code must not use the symbol as an address; the
// device address comes from cudaGetSymbolAddress. It is looked up on every
// call (the lookup allocates nothing), so a module reloaded after a device
// reset is never used through a stale address.
static __device__ __align__(256) unsigned char g_static_scratch[MLA_STATIC_SCRATCH_BYTES];

mla_status static_scratch_address(void** addr) {
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_static_scratch);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(static scratch)");
  *addr = p;
  return MLA_OK;
}

}  // namespace
}  // namespace mla

using namespace mla;

extern "C" {

size_t mla_cache_row_bytes(const mla_config* cfg) {
  if (check_config(cfg) != MLA_OK) return 0;
  return row_bytes_of(cfg->cache_dtype, cfg->d_c, cfg->d_rope);
}

mla_status mla_append(const mla_config* cfg, const void* c_kv_raw, const void* k_rope_raw,
                      const int32_t* positions, const int32_t* seq_idx, const float* gamma, void* pool,
                      int64_t num_pages, const int32_t* block_table, int32_t batch, int32_t max_pages,
                      int32_t n_tokens, void* stream) {
  mla_status s = check_config(cfg);
  if (s != MLA_OK) return s;
  if (n_tokens < 0 || batch < 1 || max_pages < 1 || num_pages < 1)
    return fail(MLA_ERR_INVALID_ARG, "bad sizes: n_tokens=%d batch=%d max_pages=%d num_pages=%lld", n_tokens,
                batch, max_pages, static_cast<long long>(num_pages));
  if (n_tokens == 0) return MLA_OK;
  if (!c_kv_raw || !k_rope_raw || !positions || !pool)
    return fail(MLA_ERR_INVALID_ARG, "c_kv_raw, k_rope_raw, positions and pool must be non-NULL");
  if (!aligned16(c_kv_raw) || !aligned16(k_rope_raw) || !aligned16(pool))
    return fail(MLA_ERR_INVALID_ARG, "c_kv_raw, k_rope_raw and pool must be 16-byte aligned");
  AppendArgs a{};
  a.c_raw = c_kv_raw; a.k_raw = k_rope_raw; a.positions = positions; a.seq_idx = seq_idx; a.gamma = gamma;
  a.pool = static_cast<uint8_t*>(pool); a.num_pages = num_pages; a.block_table = block_table;
  a.batch = batch; a.max_pages = max_pages; a.n_tokens = n_tokens; a.d_c = cfg->d_c; a.d_rope = cfg->d_rope;
  a.page_size = cfg->page_size; a.cache_dtype = cfg->cache_dtype; a.rope_interleaved = cfg->rope_interleaved;
  a.eps = cfg->eps; a.rf = rope_freq_of(cfg);
  a.row_bytes = static_cast<int64_t>(row_bytes_of(cfg->cache_dtype, cfg->d_c, cfg->d_rope));
  const cudaStream_t st = as_stream(stream);
  const int threads = 256, warps = threads / 32;
  const int blocks = (n_tokens + warps - 1) / warps;
  const bool dsv2 = cfg->io_dtype == MLA_DTYPE_BF16 && cfg->d_c == 512 && cfg->d_rope == 64 &&
                    (cfg->cache_dtype == MLA_DTYPE_BF16 || cfg->cache_dtype == MLA_DTYPE_FP8_E4M3_B128);
  if (dsv2 && cfg->cache_dtype == MLA_DTYPE_BF16)
    append_dsv2_kernel<MLA_DTYPE_BF16><<<blocks, threads, 0, st>>>(a);
  else if (dsv2)
    append_dsv2_kernel<MLA_DTYPE_FP8_E4M3_B128><<<blocks, threads, 0, st>>>(a);
  else if (cfg->io_dtype == MLA_DTYPE_BF16)
    append_generic_kernel<uint16_t><<<blocks, threads, 0, st>>>(a);
  else
    append_generic_kernel<float><<<blocks, threads, 0, st>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "append launch");
  return MLA_OK;
}

size_t mla_decode_workspace_size(const mla_config* cfg, int32_t batch, int32_t max_seq_len) {
  if (check_config(cfg) != MLA_OK || batch < 1) return 0;
  if (tc_supported(cfg)) return tc_plan(batch).bytes;
  return simt_plan(cfg, batch, max_seq_len).bytes;
}

mla_status mla_rope_query(const mla_config* cfg, const void* q_rope_raw, const int32_t* positions, void* q_rope,
                          int32_t batch, void* stream) {
  mla_status s = check_config(cfg);
  if (s != MLA_OK) return s;
  if (batch < 0) return fail(MLA_ERR_INVALID_ARG, "batch=%d", batch);
  if (batch == 0) return MLA_OK;
  if (!q_rope_raw || !positions || !q_rope) return fail(MLA_ERR_INVALID_ARG, "NULL argument");
  RopeQueryArgs a{};
  a.in = q_rope_raw;
  a.out = q_rope;
  a.positions = positions;
  a.batch = batch;
  a.n_heads = cfg->n_heads;
  a.d_rope = cfg->d_rope;
  a.rope_interleaved = cfg->rope_interleaved;
  a.rf = rope_freq_of(cfg);
  const int64_t n = static_cast<int64_t>(batch) * cfg->n_heads * (cfg->d_rope / 2);
  const int threads = 256;
  const int64_t want = (n + threads - 1) / threads;
  const int blocks = static_cast<int>(want < 4096 ? want : 4096);
  const cudaStream_t st = as_stream(stream);
  if (cfg->io_dtype == MLA_DTYPE_BF16)
    rope_query_kernel<uint16_t><<<blocks, threads, 0, st>>>(a);
  else
    rope_query_kernel<float><<<blocks, threads, 0, st>>>(a);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "rope_query launch");
  return MLA_OK;
}

size_t mla_decode_multi_workspace_size(const mla_config* cfg, int32_t batch, int32_t q_len, int32_t max_pages,
                                       int32_t max_seq_len) {
  if (check_config(cfg) != MLA_OK || batch < 1 || q_len < 1 || max_pages < 1 || max_seq_len < 0) return 0;
  return multi_prefix_bytes(batch, q_len, max_pages) + mla_decode_workspace_size(cfg, batch * q_len, max_seq_len);
}

mla_status mla_decode_multi(const mla_config* cfg, const void* q_nope, const void* q_rope, const void* w_uk,
                            const void* w_uv, const void* pool, int64_t num_pages, const int32_t* block_table,
                            const int32_t* seq_lens, int32_t batch, int32_t q_len, int32_t max_pages,
                            int32_t max_seq_len, float* out, void* workspace, size_t workspace_bytes,
                            void* stream) {
  mla_status s = check_config(cfg);
  if (s != MLA_OK) return s;
  if (batch < 1 || q_len < 1 || max_pages < 1 || static_cast<int64_t>(batch) * q_len > (1 << 20))
    return fail(MLA_ERR_INVALID_ARG, "bad sizes: batch=%d q_len=%d max_pages=%d", batch, q_len, max_pages);
  if (!seq_lens || !workspace) return fail(MLA_ERR_INVALID_ARG, "seq_lens and workspace must be non-NULL");
  if (!aligned16(workspace)) return fail(MLA_ERR_INVALID_ARG, "workspace must be 16-byte aligned");
  const size_t pre = multi_prefix_bytes(batch, q_len, max_pages);
  const size_t need = mla_decode_multi_workspace_size(cfg, batch, q_len, max_pages, max_seq_len);
  if (need == 0 || workspace_bytes < need)
    return fail(MLA_ERR_INVALID_ARG, "workspace too small: %zu < %zu", workspace_bytes, need);
  const int nv = batch * q_len;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int32_t* lens_v = reinterpret_cast<int32_t*>(ws);
  int32_t* table_v = reinterpret_cast<int32_t*>(ws + align_up(static_cast<size_t>(nv) * 4, 256));
  const int64_t n = static_cast<int64_t>(nv) * max_pages;
  const int threads = 256;
  const int64_t want = (n + threads - 1) / threads;
  const int blocks = static_cast<int>(want < 4096 ? want : 4096);
  expand_multi_kernel<<<blocks, threads, 0, as_stream(stream)>>>(seq_lens, block_table, lens_v, table_v, batch, q_len,
                                                                  max_pages);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "decode_multi expand launch");
  return mla_decode(cfg, q_nope, q_rope, w_uk, w_uv, pool, num_pages, table_v, lens_v, nv, max_pages, max_seq_len,
                    out, ws + pre, workspace_bytes - pre, stream);
}

int32_t mla_decode_path(const mla_config* cfg) {
  if (check_config(cfg) != MLA_OK) return 0;
  return tc_supported(cfg) ? 1 : 0;
}

mla_status mla_decode(const mla_config* cfg, const void* q_nope, const void* q_rope, const void* w_uk,
                      const void* w_uv, const void* pool, int64_t num_pages, const int32_t* block_table,
                      const int32_t* seq_lens, int32_t batch, int32_t max_pages, int32_t max_seq_len,
                      float* out, void* workspace, size_t workspace_bytes, void* stream) {
  mla_status s = check_config(cfg);
  if (s != MLA_OK) return s;
  if (batch < 1 || max_pages < 1 || num_pages < 1 || max_seq_len < 0)
    return fail(MLA_ERR_INVALID_ARG, "bad sizes: batch=%d max_pages=%d num_pages=%lld max_seq_len=%d", batch,
                max_pages, static_cast<long long>(num_pages), max_seq_len);
  if (static_cast<int64_t>(max_seq_len) > static_cast<int64_t>(max_pages) * cfg->page_size)
    return fail(MLA_ERR_INVALID_ARG, "max_seq_len %d exceeds max_pages * page_size", max_seq_len);
  if (!q_nope || !q_rope || !w_uk || !w_uv || !pool || !seq_lens || !out || !workspace)
    return fail(MLA_ERR_INVALID_ARG, "a required pointer is NULL");
  if (!aligned16(q_nope) || !aligned16(q_rope) || !aligned16(w_uk) || !aligned16(w_uv) || !aligned16(pool) ||
      !aligned16(out) || !aligned16(workspace))
    return fail(MLA_ERR_INVALID_ARG, "q_nope, q_rope, w_uk, w_uv, pool, out and workspace must be 16-byte aligned");
  if (tc_supported(cfg))
    return decode_tc(cfg, q_nope, q_rope, w_uk, w_uv, pool, num_pages, block_table, seq_lens, batch, max_pages,
                     max_seq_len, out, workspace, workspace_bytes, as_stream(stream));
  return decode_simt(cfg, q_nope, q_rope, w_uk, w_uv, pool, num_pages, block_table, seq_lens, batch, max_pages,
                     max_seq_len, out, workspace, workspace_bytes, as_stream(stream));
}

mla_status mla_decode_static_scratch(const mla_config* cfg, const void* q_nope, const void* q_rope,
                                     const void* w_uk, const void* w_uv, const void* pool, int64_t num_pages,
                                     const int32_t* block_table, const int32_t* seq_lens, int32_t batch,
                                     int32_t max_pages, int32_t max_seq_len, float* out, void* stream) {
  mla_status s = check_config(cfg);
  if (s != MLA_OK) return s;
  if (batch < 1 || max_seq_len < 0) return fail(MLA_ERR_INVALID_ARG, "bad sizes: batch=%d max_seq_len=%d", batch, max_seq_len);
  const size_t need = mla_decode_workspace_size(cfg, batch, max_seq_len);
  if (need > MLA_STATIC_SCRATCH_BYTES)
    return fail(MLA_ERR_INVALID_ARG, "this decode needs %zu bytes of scratch; the fixed array holds %zu", need,
                static_cast<size_t>(MLA_STATIC_SCRATCH_BYTES));
  void* scratch = nullptr;
  s = static_scratch_address(&scratch);
  if (s != MLA_OK) return s;
  return mla_decode(cfg, q_nope, q_rope, w_uk, w_uv, pool, num_pages, block_table, seq_lens, batch, max_pages,
                    max_seq_len, out, scratch, MLA_STATIC_SCRATCH_BYTES, stream);
}

mla_status mla_fold_output_weight(const mla_config* cfg, const void* w_uv, const void* w_o, int32_t hidden,
                                  void* w_ouv, void* stream) {
  mla_status s = check_config(cfg);
  if (s != MLA_OK) return s;
  if (!tc_supported(cfg))
    return fail(MLA_ERR_UNSUPPORTED, "the folded output projection runs the DeepSeek-V2 shape with bf16 weights");
  if (hidden < 128 || hidden % 128 != 0) return fail(MLA_ERR_INVALID_ARG, "hidden must be a positive multiple of 128");
  if (!w_uv || !w_o || !w_ouv) return fail(MLA_ERR_INVALID_ARG, "a required pointer is NULL");
  if (!aligned16(w_uv) || !aligned16(w_o) || !aligned16(w_ouv))
    return fail(MLA_ERR_INVALID_ARG, "w_uv, w_o and w_ouv must be 16-byte aligned");
  tcd::fold_wo_kernel<<<dim3(hidden / tcd::kFoldTile, tcd::kDc / tcd::kFoldTile, tcd::kH), 256, 0, as_stream(stream)>>>(
      static_cast<const uint16_t*>(w_uv), static_cast<const uint16_t*>(w_o), static_cast<uint16_t*>(w_ouv), hidden);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "fold launch");
  return MLA_OK;
}

size_t mla_decode_hidden_workspace_size(const mla_config* cfg, int32_t batch, int32_t max_seq_len, int32_t hidden) {
  if (check_config(cfg) != MLA_OK || !tc_supported(cfg) || batch < 1 || batch > tcd::kOutMaxNb || max_seq_len < 0 ||
      hidden < 128 || hidden % 128 != 0)
    return 0;
  return tc_plan(batch).bytes + out_partial_bytes(batch, hidden);
}

mla_status mla_decode_hidden(const mla_config* cfg, const void* q_nope, const void* q_rope, const void* w_uk,
                             const void* w_ouv, const void* pool, int64_t num_pages, const int32_t* block_table,
                             const int32_t* seq_lens, int32_t batch, int32_t max_pages, int32_t max_seq_len,
                             int32_t hidden, float* out, void* workspace, size_t workspace_bytes, void* stream) {
  mla_status s = check_config(cfg);
  if (s != MLA_OK) return s;
  if (!tc_supported(cfg))
    return fail(MLA_ERR_UNSUPPORTED, "the folded output projection runs the DeepSeek-V2 shape with bf16 weights");
  if (batch < 1 || batch > tcd::kOutMaxNb || max_pages < 1 || num_pages < 1 || max_seq_len < 0 || hidden < 128 ||
      hidden % 128 != 0)
    return fail(MLA_ERR_INVALID_ARG, "bad sizes: batch=%d (1..%d) max_pages=%d num_pages=%lld max_seq_len=%d hidden=%d",
                batch, tcd::kOutMaxNb, max_pages, static_cast<long long>(num_pages), max_seq_len, hidden);
  if (static_cast<int64_t>(max_seq_len) > static_cast<int64_t>(max_pages) * cfg->page_size)
    return fail(MLA_ERR_INVALID_ARG, "max_seq_len %d exceeds max_pages * page_size", max_seq_len);
  if (!q_nope || !q_rope || !w_uk || !w_ouv || !pool || !seq_lens || !out || !workspace)
    return fail(MLA_ERR_INVALID_ARG, "a required pointer is NULL");
  if (!aligned16(q_nope) || !aligned16(q_rope) || !aligned16(w_uk) || !aligned16(w_ouv) || !aligned16(pool) ||
      !aligned16(out) || !aligned16(workspace))
    return fail(MLA_ERR_INVALID_ARG, "q_nope, q_rope, w_uk, w_ouv, pool, out and workspace must be 16-byte aligned");
  return decode_tc(cfg, q_nope, q_rope, w_uk, nullptr, pool, num_pages, block_table, seq_lens, batch, max_pages,
                   max_seq_len, out, workspace, workspace_bytes, as_stream(stream), w_ouv, hidden);
}

size_t mla_prefill_workspace_size(const mla_config* cfg, int32_t batch, int32_t max_seq_len) {
  if (check_config(cfg) != MLA_OK || batch < 1 || max_seq_len < 0 || !tc_supported(cfg) ||
      cfg->cache_dtype != MLA_DTYPE_BF16)
    return 0;
  return pf_plan(batch, max_seq_len).bytes;
}

mla_status mla_prefill(const mla_config* cfg, const void* q_nope, const void* q_rope, const void* w_uk,
                       const void* w_uv, const void* pool, int64_t num_pages, const int32_t* block_table,
                       const int32_t* seq_lens, const int32_t* q_start, int32_t batch, int32_t max_pages,
                       int32_t max_seq_len, int32_t n_tokens, float* out, void* workspace, size_t workspace_bytes,
                       void* stream) {
  mla_status s = check_config(cfg);
  if (s != MLA_OK) return s;
  if (!tc_supported(cfg) || cfg->cache_dtype != MLA_DTYPE_BF16)
    return fail(MLA_ERR_UNSUPPORTED,
                "prefill runs the DeepSeek-V2 shape (128 heads, d_c 512, d_rope 64, d_head 128) with bf16 "
                "queries, weights and cache, and pages of a multiple of 64 tokens");
  if (batch < 1 || max_pages < 1 || num_pages < 1 || max_seq_len < 0 || n_tokens < 0)
    return fail(MLA_ERR_INVALID_ARG, "bad sizes: batch=%d max_pages=%d num_pages=%lld max_seq_len=%d n_tokens=%d",
                batch, max_pages, static_cast<long long>(num_pages), max_seq_len, n_tokens);
  if (static_cast<int64_t>(max_seq_len) > static_cast<int64_t>(max_pages) * cfg->page_size)
    return fail(MLA_ERR_INVALID_ARG, "max_seq_len %d exceeds max_pages * page_size", max_seq_len);
  if (static_cast<int64_t>(n_tokens) > static_cast<int64_t>(batch) * max_seq_len)
    return fail(MLA_ERR_INVALID_ARG, "n_tokens %d exceeds batch * max_seq_len", n_tokens);
  if (n_tokens == 0) return MLA_OK;
  if (!q_nope || !q_rope || !w_uk || !w_uv || !pool || !seq_lens || !q_start || !out || !workspace)
    return fail(MLA_ERR_INVALID_ARG, "a required pointer is NULL");
  if (!aligned16(q_nope) || !aligned16(q_rope) || !aligned16(w_uk) || !aligned16(w_uv) || !aligned16(pool) ||
      !aligned16(out) || !aligned16(workspace))
    return fail(MLA_ERR_INVALID_ARG, "q_nope, q_rope, w_uk, w_uv, pool, out and workspace must be 16-byte aligned");
  return prefill_tc(cfg, q_nope, q_rope, w_uk, w_uv, pool, num_pages, block_table, seq_lens, q_start, batch,
                    max_pages, max_seq_len, n_tokens, out, workspace, workspace_bytes, as_stream(stream));
}

mla_status mla_check_device_errors(void* stream) {
  cudaError_t e = cudaStreamSynchronize(as_stream(stream));
  if (e != cudaSuccess) return cuda_fail(e, "stream synchronize");
  unsigned int word = 0, zero = 0;
  e = cudaMemcpyFromSymbol(&word, g_dev_error, sizeof(word));
  if (e != cudaSuccess) return cuda_fail(e, "read device error word");
  if (word == 0) return MLA_OK;
  e = cudaMemcpyToSymbol(g_dev_error, &zero, sizeof(zero));
  if (e != cudaSuccess) return cuda_fail(e, "clear device error word");
  if (word & ERR_BIT_TIMEOUT) return fail(MLA_ERR_TIMEOUT, "a device-side wait ran out (word=0x%x)", word);
  return fail(MLA_ERR_BOUNDS, "a device-side index was out of range (word=0x%x)", word);
}

const char* mla_decode_stage_names(const mla_config* cfg) {
  if (cfg && check_config(cfg) == MLA_OK && tc_supported(cfg)) return "absorb_tc,attend_tc,merge,uv_tc";
  return "absorb_simt,attend_simt,combine_simt";
}

mla_status mla_set_stage_events(void* const* events, int32_t n_events) {
  if (n_events < 0 || n_events > 8) return fail(MLA_ERR_INVALID_ARG, "n_events must be in [0, 8]");
  if (!events) n_events = 0;
  for (int i = 0; i < n_events; ++i) {
    if (!events[i]) return fail(MLA_ERR_INVALID_ARG, "event %d is NULL", i);
    g_stage.ev[i] = static_cast<cudaEvent_t>(events[i]);
  }
  g_stage.n = n_events;
  return MLA_OK;
}

const char* mla_last_error(void) { return g_last_error.c_str(); }

}  // extern "C"
