/*
 * mla.h - C ABI of the B300 (sm_103a) MLA decode library (libmla.so).
 *
 * Multi-head Latent Attention decode over a paged latent KV cache, as the
 * DeepSeek-V2 report (translated page) states it in section 2.1:
 *   - 2.1.2 low-rank joint KV compression: only a d_c-wide latent c_j is
 *     cached per token; keys and values are its up-projections W_UK c_j and
 *     W_UV c_j, and because W_UK can be absorbed into the query and W_UV
 *     into the output, no per-head key or value is ever formed;
 *   - 2.1.3 decoupled RoPE: a d_rope-wide key k^R_j = RoPE(k_raw_j), shared by
 *     all heads, is cached beside c_j, so a row holds (d_c + d_rope) values;
 *   - 3.1.2 an RMSNorm follows the compressed latent.
 * Page tables (fixed-size pages of cache rows, a per-sequence list of page
 * ids) are this library's storage layout; the report does not describe one.
 *
 * Conventions for every call:
 *   - Every pointer argument is DEVICE memory owned by the caller, unless
 *     stated otherwise. The library allocates no device memory and keeps no
 *     pointer after a call returns.
 *   - Arrays are dense, row-major, innermost dimension contiguous; base
 *     pointers of the pool, the raw inputs, the queries, the weights, `out`
 *     and `workspace` must be 16-byte aligned.
 *   - Calls are asynchronous on `stream` (a cudaStream_t, NULL = legacy
 *     default stream). The returned status covers host-side argument checks
 *     and launch errors only. Errors found on the device (a page id outside
 *     the pool, a position beyond the page table, a bounded wait that ran
 *     out) skip the offending access and set a per-device error word, which
 *     mla_check_device_errors() reads and clears.
 *   - On any status other than MLA_OK, mla_last_error() returns a message
 *     (thread-local; valid until the next call on the same thread).
 */
#ifndef MLA_H_
#define MLA_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MLA_API __attribute__((visibility("default")))
#else
#define MLA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MLA_OK = 0,
  MLA_ERR_INVALID_ARG = 1,  /* a null/misaligned pointer, a bad size or config */
  MLA_ERR_UNSUPPORTED = 2,  /* a config no kernel here implements */
  MLA_ERR_CUDA = 3,         /* a CUDA runtime call or launch failed */
  MLA_ERR_TIMEOUT = 4,      /* a device-side bounded wait ran out */
  MLA_ERR_BOUNDS = 5        /* a device-side index fell outside its array */
} mla_status;

typedef enum {
  MLA_DTYPE_BF16 = 0,
  MLA_DTYPE_FP32 = 1,
  /* cache only: per row, d_c E4M3 codes, then d_c/128 fp32 scales (one per
     128-value block: value = code * scale), then d_rope bf16 rope values */
  MLA_DTYPE_FP8_E4M3_B128 = 2
} mla_dtype;

typedef struct {
  int32_t n_heads;          /* n_h, query heads */
  int32_t d_c;              /* latent width (KV compression dim) */
  int32_t d_rope;           /* decoupled rope width d_h^R (even) */
  int32_t d_head;           /* d_h, width of q_nope and of each head's output */
  int32_t page_size;        /* tokens per cache page */
  int32_t io_dtype;         /* mla_dtype of queries, weights, raw latents/keys: BF16 or FP32 */
  int32_t cache_dtype;      /* mla_dtype of the pool rows */
  float scale;              /* softmax scale applied to q.k; <= 0 selects 1/sqrt(d_head + d_rope), the
                               width of the full key [k_C ; k_R] (report sections 2.1.1, 2.1.3) */
  float eps;                /* RMSNorm epsilon */
  float rope_theta;         /* RoPE base; pair m turns by pos * theta^(-2m/d_rope) */
  int32_t rope_interleaved; /* 1: pairs (2m, 2m+1) (RoFormer); 0: pairs (m, m + d_rope/2) */
  /* YaRN extension of the decoupled RoPE (report section 3.1.4; there s = 40,
     alpha = 1, beta = 32 over a 4K context, mscale 0.0707). yarn_factor s > 1
     turns it on; <= 1 means plain RoPE and the other yarn fields are ignored.
     Pair m's frequency f = rope_theta^(-2m/d_rope) makes r = yarn_orig_len f / (2 pi)
     turns over the original context and becomes (1 - g) f / s + g f with
     g = clamp((r - yarn_alpha) / (yarn_beta - yarn_alpha), 0, 1) in mla_append and
     mla_rope_query; mla_decode multiplies the logits by (yarn_mscale ln s + 1)^2
     on top of `scale`. */
  float yarn_factor;
  float yarn_alpha;
  float yarn_beta;
  float yarn_mscale;
  int32_t yarn_orig_len;
} mla_config;

/* Bytes of one cache row for `cfg` (0 if cfg is invalid):
   BF16 (d_c + d_rope) * 2; FP32 (d_c + d_rope) * 4;
   FP8_E4M3_B128 d_c + 4 * d_c / 128 + 2 * d_rope. */
MLA_API size_t mla_cache_row_bytes(const mla_config* cfg);

/*
 * mla_append - write n_tokens new tokens into the paged latent cache.
 *
 * Computes, per token t (report sections 3.1.2 and 2.1.3):
 *   c  = c_kv_raw[t] / sqrt(mean(c_kv_raw[t]^2) + eps) * gamma   (fp32 math)
 *   kR = RoPE(k_rope_raw[t], positions[t])   (angle and rotation in fp64)
 * and stores (c, kR), converted to the cache format, as the row
 *   slot = block_table[s * max_pages + positions[t] / page_size] * page_size
 *          + positions[t] % page_size,   s = seq_idx ? seq_idx[t] : t.
 * Conversion is round-to-nearest-even (bf16) or, for FP8_E4M3_B128, per
 * 128-value block scale = amax / 448 (1 if amax == 0) and code =
 * E4M3_satfinite_RNE(c / scale) with an IEEE fp32 division.
 *
 *   c_kv_raw   [n_tokens, d_c]    io_dtype
 *   k_rope_raw [n_tokens, d_rope] io_dtype
 *   positions  [n_tokens] int32   0-based position in its sequence
 *   seq_idx    [n_tokens] int32 or NULL (token t belongs to sequence t)
 *   gamma      [d_c] fp32 RMSNorm gain, or NULL (all ones)
 *   pool       [num_pages, page_size, row_bytes] bytes, written
 *   block_table[batch, max_pages] int32, or NULL: sequence s then owns pages
 *              s*max_pages .. s*max_pages + max_pages-1 (contiguous layout)
 * A token whose sequence, position or page id falls outside these arrays is
 * not written and sets MLA_ERR_BOUNDS in the device error word. Two tokens
 * given the same slot in one call race.
 */
MLA_API mla_status mla_append(const mla_config* cfg, const void* c_kv_raw, const void* k_rope_raw,
                      const int32_t* positions, const int32_t* seq_idx, const float* gamma,
                      void* pool, int64_t num_pages, const int32_t* block_table,
                      int32_t batch, int32_t max_pages, int32_t n_tokens, void* stream);

/*
 * Bytes of scratch memory mla_decode needs for `batch` sequences whose
 * lengths are at most max_seq_len, on the current device. The caller
 * allocates it (any contents; 256-byte alignment).
 */
MLA_API size_t mla_decode_workspace_size(const mla_config* cfg, int32_t batch, int32_t max_seq_len);

/*
 * mla_decode - one decode step of MLA over the paged latent cache.
 *
 * For each sequence b < batch and head i < n_heads (report section 2.1.2,
 * absorbed form; section 2.1.3 decoupled RoPE):
 *   q_lat   = W_UK[i]^T q_nope[b,i]                       (d_c)
 *   s_j     = scale * (q_lat . c_j + q_rope[b,i] . kR_j),  j < seq_lens[b]
 *   p       = softmax_j(s)
 *   out[b,i]= W_UV[i] (sum_j p_j c_j)                     (d_head, fp32)
 * where (c_j, kR_j) is cache row j of sequence b, found through block_table
 * as in mla_append. seq_lens[b] == 0 gives zeros.
 *
 *   q_nope  [batch, n_heads, d_head] io_dtype
 *   q_rope  [batch, n_heads, d_rope] io_dtype, already rotated
 *   w_uk    [n_heads, d_head, d_c]   io_dtype  (head i = rows i*d_head.. of W_UK)
 *   w_uv    [n_heads, d_head, d_c]   io_dtype
 *   pool, num_pages, block_table, max_pages: as in mla_append (read only)
 *   seq_lens[batch] int32 (device)
 *   max_seq_len  host-side upper bound of seq_lens (plans the split over
 *                sequence blocks; a larger device value sets MLA_ERR_BOUNDS
 *                and is clamped)
 *   out     [batch, n_heads, d_head] fp32, written
 *   workspace, workspace_bytes: at least mla_decode_workspace_size() bytes
 * Pages of a sequence are processed in independent splits whose partial
 * results are merged by a log-sum-exp combine before W_UV is applied.
 *
 * Kernels: n_heads 128, d_c 512, d_rope 64, d_head 128 with bf16 queries and
 * weights, a bf16 or FP8_E4M3_B128 cache and page_size a multiple of 64 run
 * on the tensor cores (tcgen05/TMEM/TMA, mla_decode_path() == 1; an FP8 cache
 * is dequantised to fp16 in shared memory before the MMAs); every other valid
 * config runs on CUDA cores. On the tensor-core path the kernels are chained
 * with programmatic dependent launch:
 *   - the first one may start reading W_UK before the kernel that precedes
 *     mla_decode on `stream` has finished, so that kernel must not write the
 *     weights;
 *   - every other input (q_nope, q_rope, seq_lens, block_table, the pool) is
 *     read only after the preceding kernel completes.
 */
MLA_API mla_status mla_decode(const mla_config* cfg, const void* q_nope, const void* q_rope,
                      const void* w_uk, const void* w_uv, const void* pool, int64_t num_pages,
                      const int32_t* block_table, const int32_t* seq_lens, int32_t batch,
                      int32_t max_pages, int32_t max_seq_len, float* out, void* workspace,
                      size_t workspace_bytes, void* stream);

/*
 * mla_decode_multi - decode q_len new tokens of each sequence at once (the
 * draft tokens of multi-token prediction, verified together; DeepSeek-V3
 * summary, section 3). The cache already holds all q_len new tokens as the
 * last rows of each sequence; new token k (0-based) of sequence b attends
 * causally to the first seq_lens[b] - (q_len - 1 - k) rows (none if that is
 * not positive):
 *   q_nope [batch, q_len, n_heads, d_head], q_rope [batch, q_len, n_heads, d_rope]
 *   out    [batch, q_len, n_heads, d_head] fp32
 * Other arguments as mla_decode; the workspace is
 * mla_decode_multi_workspace_size(cfg, batch, q_len, max_pages, max_seq_len)
 * bytes (0 for invalid arguments).
 * Each new token is decoded as a sequence of its own over the pages of its
 * sequence, so the q_len of them read the same pages while those are in L2.
 */
MLA_API size_t mla_decode_multi_workspace_size(const mla_config* cfg, int32_t batch, int32_t q_len,
                                               int32_t max_pages, int32_t max_seq_len);
MLA_API mla_status mla_decode_multi(const mla_config* cfg, const void* q_nope, const void* q_rope,
                                    const void* w_uk, const void* w_uv, const void* pool, int64_t num_pages,
                                    const int32_t* block_table, const int32_t* seq_lens, int32_t batch,
                                    int32_t q_len, int32_t max_pages, int32_t max_seq_len, float* out,
                                    void* workspace, size_t workspace_bytes, void* stream);

/*
 * mla_decode_static_scratch - mla_decode that allocates nothing and takes no
 * workspace argument. The paper has no counterpart to this call; it exists
 * for callers of this library that cannot allocate device memory at the
 * point where they decode, e.g. a plugin running inside a host program that
 * owns all device memory and offers it no allocator, or a serving loop whose
 * memory plan is fixed up front and which must not call cudaMalloc (that
 * call can synchronise the device and stall other streams).
 *
 * Arguments, results and errors are those of mla_decode, minus workspace.
 * The scratch is one device array inside the library of
 * MLA_STATIC_SCRATCH_BYTES (48 MiB); every GPU that loads the library holds
 * it until the process exits. A request needing more scratch than that
 * (mla_decode_workspace_size() > MLA_STATIC_SCRATCH_BYTES) is refused with
 * MLA_ERR_INVALID_ARG before anything is launched; nothing is allocated.
 *
 * Every call looks up the array's device address on the current device
 * with cudaGetSymbolAddress (which allocates nothing); the first call on a
 * device also loads the library's device code there, so make that first call
 * before any stream capture. For the DeepSeek-V2 shape on the tensor-core
 * path (128 heads, d_c 512, d_rope 64, d_head 128) the array holds the
 * scratch of a batch of at most 25 sequences, whatever their lengths. All calls on a device share the one array, so
 * two calls whose kernels overlap on the GPU (different streams, or threads
 * without ordering) race on it and both results are undefined; serialise
 * them. The array keeps the last call's contents; the decode writes every
 * scratch location before reading it, so nothing needs clearing between calls.
 */
#define MLA_STATIC_SCRATCH_BYTES ((size_t)48 << 20)
MLA_API mla_status mla_decode_static_scratch(const mla_config* cfg, const void* q_nope, const void* q_rope,
                                             const void* w_uk, const void* w_uv, const void* pool,
                                             int64_t num_pages, const int32_t* block_table,
                                             const int32_t* seq_lens, int32_t batch, int32_t max_pages,
                                             int32_t max_seq_len, float* out, void* stream);

/*
 * W_UV folded into the output projection W_O (DeepSeek-V2 report, section
 * 2.1.2: W_UV can be absorbed into W_O; section 2.1.1: u = W_O [o_1; ...; o_H]).
 *
 * mla_fold_output_weight - once per set of weights:
 *   w_ouv[:, i d_c .. (i+1) d_c) = w_o[:, i d_h .. (i+1) d_h) w_uv[i]   (fp32 sums, rounded to io_dtype)
 *   w_uv  [n_heads, d_head, d_c], w_o [hidden, n_heads * d_head] (row-major) in io_dtype;
 *   w_ouv [hidden, n_heads * d_c] written in fp16 (IEEE binary16, round to nearest even): the folded
 *   products are of the order |W_O| |W_UV| sqrt(d_head), where fp16 keeps 3 more bits than bf16.
 *   hidden a positive multiple of 128 (5120 for DeepSeek-V2). Runs on CUDA cores (not a decode step).
 *
 * mla_decode_hidden - mla_decode with the output taken to the hidden size:
 *   out[b, :] = w_ouv [o_lat(b, 1); ...; o_lat(b, H)]  (= W_O [o(b, 1); ...; o(b, H)]), fp32 [batch, hidden]
 * where o_lat(b, i) is head i's attention-weighted latent; one GEMM over the 65,536-wide latent outputs
 * replaces the W_UV step and the caller's W_O GEMM. Arguments as mla_decode, with w_ouv in place of w_uv;
 * the workspace is mla_decode_hidden_workspace_size() bytes (0 for an unsupported config or size).
 * Supported: the tensor-core decode path's configs, batch 1 .. 128. As with W_UK, the GEMM may start
 * reading w_ouv before the kernel that precedes the call on `stream` has finished, so that kernel must
 * not write it.
 */
MLA_API mla_status mla_fold_output_weight(const mla_config* cfg, const void* w_uv, const void* w_o, int32_t hidden,
                                          void* w_ouv, void* stream);
MLA_API size_t mla_decode_hidden_workspace_size(const mla_config* cfg, int32_t batch, int32_t max_seq_len,
                                                int32_t hidden);
MLA_API mla_status mla_decode_hidden(const mla_config* cfg, const void* q_nope, const void* q_rope, const void* w_uk,
                                     const void* w_ouv, const void* pool, int64_t num_pages,
                                     const int32_t* block_table, const int32_t* seq_lens, int32_t batch,
                                     int32_t max_pages, int32_t max_seq_len, int32_t hidden, float* out,
                                     void* workspace, size_t workspace_bytes, void* stream);

/*
 * mla_prefill - attention of whole prompts (or prompt chunks) over the
 * paged latent cache, in the non-absorbed form of the DeepSeek-V2 report,
 * section 2.1.2 (per-head keys k_{j,i} = W_UK,i c_j and values
 * v_{j,i} = W_UV,i c_j materialised from the cached latents) with the
 * decoupled rope key of section 2.1.3 and causal softmax attention
 * (section 2.1.1). The new tokens must already be in the cache (mla_append):
 * sequence b holds seq_lens[b] rows, of which the last
 * n_b = q_start[b+1] - q_start[b] are its new tokens, at positions
 * seq_lens[b] - n_b .. seq_lens[b] - 1; new token k attends to rows
 * 0 .. seq_lens[b] - n_b + k (a full prompt has n_b = seq_lens[b]; a chunk
 * of a longer prompt attends to the rows cached before it too).
 *   q_nope [n_tokens, n_heads, d_head] io_dtype, q_rope [n_tokens, n_heads,
 *            d_rope] (rotated at each token's position, e.g. by mla_rope_query)
 *   w_uk, w_uv [n_heads, d_head, d_c]
 *   pool, num_pages, block_table, max_pages: as in mla_append (read only)
 *   seq_lens [batch] int32 (device), q_start [batch + 1] int32 (device),
 *            non-decreasing, q_start[0] = 0, q_start[batch] = n_tokens
 *   max_seq_len  host-side upper bound of seq_lens (sizes the workspace)
 *   out    [n_tokens, n_heads, d_head] fp32: row q_start[b] + k is new token k
 *          of sequence b, out = sum_j softmax_j(scale q.k_j) v_j per head
 *   workspace, workspace_bytes: at least mla_prefill_workspace_size() bytes
 *          (the per-head keys and values, 2 * batch * ceil(max_seq_len/128)
 *          * 128 * n_heads * d_head bf16 values)
 * Supported: the DeepSeek-V2 shape with bf16 queries, weights and cache and
 * page_size a multiple of 64 (MLA_ERR_UNSUPPORTED otherwise; the workspace
 * size is then 0). A sequence with n_b < 0, n_b > seq_lens[b] or q_start
 * outside [0, n_tokens] sets MLA_ERR_BOUNDS and is skipped; a page id outside
 * the pool for a row the sequence holds sets MLA_ERR_BOUNDS and reads zeros.
 * Kernels: kv_up (tcgen05 GEMM of the latent rows against [W_UK ; W_UV]) and
 * prefill_attn (tcgen05 causal attention, P kept in tensor memory), chained
 * with programmatic dependent launch: the preceding kernel on `stream` must
 * have finished writing the pool, block_table and seq_lens (an ordinary
 * kernel always has).
 */
MLA_API size_t mla_prefill_workspace_size(const mla_config* cfg, int32_t batch, int32_t max_seq_len);
MLA_API mla_status mla_prefill(const mla_config* cfg, const void* q_nope, const void* q_rope, const void* w_uk,
                               const void* w_uv, const void* pool, int64_t num_pages, const int32_t* block_table,
                               const int32_t* seq_lens, const int32_t* q_start, int32_t batch, int32_t max_pages,
                               int32_t max_seq_len, int32_t n_tokens, float* out, void* workspace,
                               size_t workspace_bytes, void* stream);

/*
 * Waits for `stream`, then returns and clears the current device's error
 * word: MLA_OK, MLA_ERR_BOUNDS or MLA_ERR_TIMEOUT (timeout wins if both).
 */
MLA_API mla_status mla_check_device_errors(void* stream);

/*
 * mla_rope_query - rotate the rope part of the decode queries (report section
 * 2.1.3: q^R = RoPE(W_QR c^Q)) with the frequencies mla_append gives the keys,
 * YaRN included:
 *   q_rope[b, i, :] = RoPE(q_rope_raw[b, i, :], positions[b])
 * angle and rotation in fp64, the result rounded to nearest even in io_dtype.
 *   q_rope_raw, q_rope [batch, n_heads, d_rope] io_dtype (may be the same array)
 *   positions          [batch] int32, the position of each sequence's query token
 * A negative position skips the sequence's rows and sets MLA_ERR_BOUNDS.
 */
MLA_API mla_status mla_rope_query(const mla_config* cfg, const void* q_rope_raw, const int32_t* positions,
                                  void* q_rope, int32_t batch, void* stream);

/* Which kernels mla_decode would use for cfg on the current device:
   1 = tcgen05/TMA tensor-core path, 0 = CUDA-core (SIMT) path. */
MLA_API int32_t mla_decode_path(const mla_config* cfg);

/* Kernel names of one mla_decode call for cfg, in launch order, comma
   separated (e.g. "absorb,attend,combine"); static storage. */
MLA_API const char* mla_decode_stage_names(const mla_config* cfg);

/*
 * Timing hook. After this call, every mla_decode on the calling thread
 * records events[0] on its stream before its first kernel and events[k]
 * after its k-th kernel, for k < n_events (cudaEvent_t handles owned by the
 * caller). n_events = 0 (or events = NULL) turns the hook off. At most 8.
 */
MLA_API mla_status mla_set_stage_events(void* const* events, int32_t n_events);

/* Thread-local message describing the last non-OK status. */
MLA_API const char* mla_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* MLA_H_ */
