/*
 * mla.h - C ABI of the B300 (sm_103a) Multi-head Latent Attention decode library.
 *
 * The library computes one MLA attention layer at decode time over a paged
 * cache that holds, per token, only the latent c_KV (d_c values) and the
 * decoupled RoPE key k_R (d_rope values).  Per-head keys and values are never
 * formed: the key up-projection is folded into the query and the value
 * up-projection is applied after the weighted sum.
 *
 * Sources (cited by title and section):
 *   [KJ] "What does Multi-head Latent Attention compress, and how is that
 *        different from quantizing the cache?" (katajob.com)
 *   [ZQ] "How does DeepSeek's Multi-Latent Attention (MLA) compress the KV
 *        cache below GQA?" (zenaique.com)
 *   [BB] "Multi-head Latent Attention (MLA)" (bembew.net)
 *   [TM] "Multi-head Latent Attention" card mla-attention (talentme)
 *   [SC] "What Is Multi-head Latent Attention—and How Does It Shrink AI's
 *        Memory?" (satishkchoudhary.com)
 *
 * Conventions shared by every call
 *   - All pointers named d_* or documented as "device" are device pointers on
 *     the current CUDA device; the caller allocates and owns them.  The
 *     library never allocates device memory; every compute call takes a
 *     caller-owned workspace whose size the matching *_workspace_bytes()
 *     returns (0 means the configuration is invalid or unsupported).
 *   - Every workspace begins with a 256-byte header whose first 32-bit word is
 *     the device status word of the calls made with that workspace.  A new
 *     workspace must start with that word at zero (e.g. cudaMemsetAsync of its
 *     first 4 bytes); calls only OR flags into it and mla_get_device_status()
 *     clears it.  Calls that share a workspace share its word; calls with
 *     different workspaces (on different streams, say) never see each
 *     other's flags.
 *   - Every call is asynchronous on `stream` (a cudaStream_t; NULL is the
 *     legacy default stream).  Argument errors are detected on the host and
 *     returned before anything is launched.
 *   - Storage dtype (mla_config.dtype) applies to activations, weights, the
 *     cache, queries and outputs alike; accumulation is always fp32.  bf16
 *     results are rounded to nearest even.
 *   - bf16 runs on the sm_103a tensor-core kernels, which cover the
 *     DeepSeek-V2 head shapes (128 heads, d_c = 512, d_rope = 64, 64-token
 *     blocks, projection widths that are multiples of 64); any other bf16
 *     shape returns MLA_ERR_UNSUPPORTED.  fp32 runs on CUDA-core kernels at
 *     any shape (tensor cores cannot hold fp32 operands at fp32 accuracy).
 *   - Weights are stored row-major as [out_features][in_features]; the
 *     per-head up-projections as [n_heads][out][d_c].
 *   - Device pointers must be 16-byte aligned.
 *   - Device-side index problems (a block-table entry outside the pool, a
 *     position outside a sequence's blocks, a sequence index outside the
 *     batch) never fault: the offending access is skipped and a flag is set
 *     in the call's status word.  Every wait inside a kernel is bounded (about
 *     2 s); one that runs out sets a timeout flag and the kernel returns.
 */
#ifndef MLA_H_
#define MLA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st* mla_stream_t;

typedef enum {
  MLA_OK = 0,
  MLA_ERR_INVALID_ARG = 1,   /* null/misaligned pointer, bad size, inconsistent config        */
  MLA_ERR_UNSUPPORTED = 2,   /* valid but not implemented (odd d_rope, bf16 outside the tensor-core shapes) */
  MLA_ERR_CUDA = 3,          /* a CUDA runtime call or launch failed                         */
  MLA_ERR_TIMEOUT = 4,       /* device: a bounded wait gave up (reported by get_device_status) */
  MLA_ERR_DEVICE_INDEX = 5,  /* device: an out-of-range index was skipped                    */
  MLA_ERR_WORKSPACE = 6      /* workspace pointer null or smaller than required              */
} mla_status;

typedef enum { MLA_F32 = 0, MLA_BF16 = 1 } mla_dtype;

/* Layer shape.  d_rope is the width of both k_R and each head's rotated query
 * part (qk_rope).  softmax_scale <= 0 selects 1/sqrt(qk_nope + d_rope). */
typedef struct {
  int d_model;
  int n_heads;
  int qk_nope;
  int d_rope;
  int v_head;
  int d_c;
  int block_size;      /* tokens per cache block; 64 */
  float softmax_scale;
  int dtype;           /* mla_dtype */
  int cache_fp8;       /* 0: cache rows in dtype; 1: reduced-precision cache (bf16 only, see below) */
  int rope_per_head;   /* 0: one positional key per token shared by all heads; 1: one per head (below) */
} mla_config;

/* Paged latent cache.  Each token's row is [c_KV || k_R], d_c + d_rope values
 * ([ZQ "What MLA caches..."]: the latent is the only content written to the
 * cache; [SC]: plus the small positional component).  Logical position p of
 * sequence b lives in physical block
 *   k = block_table[b * max_blocks_per_seq + p / block_size]
 * at offset o = p % block_size, and each block is stored transposed:
 *   pool: [num_blocks][d_c + d_rope][block_size] of dtype, element e of that
 *   token at pool[(k * (d_c + d_rope) + e) * block_size + o].
 * (Element-major blocks let the decode kernel fetch whole contiguous runs of a
 * block per copy and feed them to the tensor cores as either operand layout.)
 *
 * Per-head positional keys (rope_per_head = 1, dtype bf16, cache_fp8 = 0; [ZQ]
 * "a small per-head RoPE-carrying key", the alternative to the shared key of
 * [TM]/[SC]): a token's row is [c_KV (d_c) || k_R^1 (d_rope) || ... || k_R^H],
 * row width d_c + n_heads * d_rope, each k_R^h = RoPE(W_KR^h x, pos) with the
 * rotation frequencies restarting for every head; W_KR is then
 * [n_heads * d_rope][d_model].  Supported by mla_compress_append and the
 * explicit form (mla_prefill_attention); mla_decode_attention returns
 * MLA_ERR_UNSUPPORTED (the absorbed kernel shares one key across heads as an
 * MMA operand; per-head keys are a per-head dot product, not an MMA).
 *
 * Reduced-precision cache (cache_fp8 = 1, dtype bf16; [KJ "Compression as
 * architecture versus compression as post-processing"]: a latent can itself be
 * stored in a reduced-precision format).  The format is this library's (the
 * pages name none): the latent of a token is stored as FP8 E4M3 codes of
 * c_t / s_t, s_t the smallest power of two with max|c_t| / s_t <= 448 (1 for
 * an all-zero row), rounded to nearest even; the positional key as bf16 values
 * of k_R,t / s_t (exact: s_t is a power of two); s_t as fp32.  A block holds
 * block_size * (d_c + 2 d_rope + 4) bytes, element-major per part:
 *   codes  [d_c][block_size] bytes at block offset 0,
 *   k_R/s  [d_rope][block_size] bf16 at block offset d_c * block_size,
 *   s      [block_size] fp32 at block offset (d_c + 2 d_rope) * block_size.
 * The reduced-precision cache takes block_size 64, d_c a multiple of 64 and
 * d_rope <= 64; for other shapes every call returns MLA_ERR_UNSUPPORTED and
 * the size queries return 0. */
typedef struct {
  void* pool;                   /* device */
  int num_blocks;
  const int32_t* block_table;   /* device, [batch][max_blocks_per_seq]; unused entries may hold -1 */
  int max_blocks_per_seq;
  int batch;                    /* rows of block_table */
} mla_paged_cache;

/* RoPE cos/sin table: [max_pos][d_rope/2][2] fp32 (cos, sin of pos * base^(-2i/d_rope)). */
typedef struct {
  const float* cos_sin;         /* device */
  int max_pos;
} mla_rope_table;

/* Bytes one token occupies in the cache: (d_c + d_rope) * sizeof(dtype), or
 * d_c + 2 d_rope + 4 for the reduced-precision cache (644 at the DeepSeek-V2 shape),
 * or (d_c + n_heads * d_rope) * 2 with per-head positional keys.
 * [TM "Key Problems Solved"]: the per-token cache shrinks from 2*H*d to the
 * latent; [SC]: plus the positional part.  Returns 0 for an invalid config. */
size_t mla_cache_bytes_per_token(const mla_config* cfg);

/* Fill a RoPE table on the device for positions [0, max_pos):
 *   cos_sin[p][i] = (cos(p * base^(-2i/d_rope)), sin(...)), computed in double
 * precision and rounded to fp32.  Pairs (2i, 2i+1) are rotated together
 * ([BB "2. Decoupling RoPE from Compression"]; interleaved-pair reading).
 * d_cos_sin: device, max_pos * d_rope floats. */
mla_status mla_rope_table_create(const mla_config* cfg, float base, int max_pos, float* d_cos_sin,
                                 mla_stream_t stream);

/* Workspace bytes mla_compress_append needs for T tokens. */
size_t mla_compress_workspace_bytes(const mla_config* cfg, int T);

/* Down-project T tokens and write their cache rows.
 *   c_t   = W_DKV x_t                    ([KJ "The mechanism"]; [BB "1. Low-Rank
 *                                          Decomposition" and "Implementation Logic" step 1])
 *   k_R,t = RoPE(W_KR x_t, pos_t)        ([BB "Implementation Logic" steps 3-4];
 *                                          [TM "Core Definition"] k_t^R)
 * and store [c_t || k_R,t] at logical position pos[t] of sequence seq_idx[t].
 *   x      device [T][d_model]
 *   W_DKV  device [d_c][d_model];  W_KR device [d_rope][d_model]
 *   seq_idx, pos  device int32 [T]
 *   rope   table covering every pos[t]
 *   cache  the paged cache; only the T addressed rows are written
 * With cache_fp8 the row is quantised as described above (one scale per token,
 * from the row's fp32 values).
 * A token whose seq_idx, pos or block id is out of range is skipped and
 * flagged (MLA_ERR_DEVICE_INDEX via mla_get_device_status). */
mla_status mla_compress_append(const mla_config* cfg, const void* x, const void* W_DKV, const void* W_KR,
                               const int32_t* seq_idx, const int32_t* pos, const mla_rope_table* rope,
                               const mla_paged_cache* cache, int T,
                               void* workspace, size_t workspace_bytes, mla_stream_t stream);

/* Workspace bytes mla_absorb_query needs for N query tokens. */
size_t mla_absorb_workspace_bytes(const mla_config* cfg, int N);

/* Project N query tokens and fold the key up-projection into them:
 *   q_nope^h = W_Q^h x,  q_R^h = RoPE(W_QR^h x, q_pos),  q_abs^h = W_UK^h^T q_nope^h
 * ([KJ "Why it is not just extra work at decode time"]: the key up-projection
 * is absorbed into the query projection).
 *   x      device [N][d_model];  q_pos device int32 [N]
 *   W_Q    device [n_heads*qk_nope][d_model];  W_QR device [n_heads*d_rope][d_model]
 *   W_UK   device [n_heads][qk_nope][d_c]
 *   q_out  device [N][n_heads][d_c + d_rope] = [q_abs^h || q_R^h] */
mla_status mla_absorb_query(const mla_config* cfg, const void* x, const void* W_Q, const void* W_QR,
                            const void* W_UK, const int32_t* q_pos, const mla_rope_table* rope,
                            void* q_out, int N, void* workspace, size_t workspace_bytes,
                            mla_stream_t stream);

/* Workspace bytes mla_decode_attention needs for `batch` sequences of n_q
 * queries whose block tables have max_blocks_per_seq entries. */
size_t mla_decode_workspace_bytes(const mla_config* cfg, int batch, int n_q, int max_blocks_per_seq);

/* Softmax attention of every query over the latent cache, accumulated in latent space:
 *   s_t^h   = scale * (q_abs^h . c_t + q_R^h . k_R,t)   for t < vis_j
 *   o_lat^h = sum_t softmax(s^h)_t c_t
 * with vis_j = kv_len[b] - (n_q - 1 - j) for query j of sequence b (causal
 * among the n_q queries).  Every visible token is attended ([SC]: every prior
 * token keeps an entry; [ZQ]: decode streams the entire cache from HBM).
 * Long sequences are split across CTAs and merged by log-sum-exp inside this call.
 *   q       device [batch][n_q][n_heads][d_c + d_rope] (mla_absorb_query output)
 *   kv_len  device int32 [batch]; must not exceed max_blocks_per_seq * block_size
 *   o_lat   device [batch][n_q][n_heads][d_c]
 *   lse     optional device fp32 [batch][n_q][n_heads] (natural log of the
 *           softmax normaliser of the scaled scores; -inf when nothing is
 *           visible), or NULL
 * A query with no visible token gets o_lat = 0.
 * With cache_fp8 the call first expands the visited blocks of every sequence
 * into bf16 rows (codes * s, (k_R / s) * s: exact) in the workspace and then
 * attends over them; the workspace grows by batch * max_blocks_per_seq bf16
 * blocks.
 * Reproducibility: on the tensor-core path each 128-token score tile sums its
 * six 96-element slices in a fixed order, so repeated calls on the same inputs
 * and GPU give the same bits; another SM count or batch moves the split points
 * and changes results only by fp32 rounding. */
mla_status mla_decode_attention(const mla_config* cfg, const void* q, const mla_paged_cache* cache,
                                const int32_t* kv_len, int batch, int n_q, void* o_lat, float* lse,
                                void* workspace, size_t workspace_bytes, mla_stream_t stream);

/* Workspace bytes mla_output_project needs for N query tokens. */
size_t mla_output_workspace_bytes(const mla_config* cfg, int N);

/* Apply the value up-projection and the output projection:
 *   o^h = W_UV^h o_lat^h,  out = W_O concat_h(o^h)
 * ([KJ "Why it is not just extra work at decode time"]: the value
 * up-projection is absorbed on the output side).
 *   o_lat  device [N][n_heads][d_c];  W_UV device [n_heads][v_head][d_c]
 *   W_O    device [d_model][n_heads*v_head];  out device [N][d_model] */
mla_status mla_output_project(const mla_config* cfg, const void* o_lat, const void* W_UV, const void* W_O,
                              void* out, int N, void* workspace, size_t workspace_bytes,
                              mla_stream_t stream);

/* ---- Explicit form: prefill of a prompt (keys and values rebuilt per head) ----
 * At prefill every prompt token is a query.  Rebuilding the per-head keys and
 * values from the cached latent ([TM] point 4: K/V recomputed from the latent at
 * prefill; [KJ "The mechanism"]: up-projections expand the latent into per-head
 * keys and values) costs 2 (qk_nope + d_rope + v_head) FLOP per (query, key,
 * head) against 2 (2 d_c + d_rope) for the absorbed form, so long prompts take
 * this path: mla_project_query, mla_prefill_attention, mla_head_output_project.
 * bf16 only, on the tensor-core shapes above; fp32 returns MLA_ERR_UNSUPPORTED. */

/* Workspace bytes mla_project_query needs for N query tokens. */
size_t mla_project_workspace_bytes(const mla_config* cfg, int N);

/* Project N query tokens without absorbing W_UK:
 *   q_nope^h = W_Q^h x,  q_R^h = RoPE(W_QR^h x, q_pos)
 *   x      device [N][d_model];  q_pos device int32 [N]
 *   W_Q    device [n_heads*qk_nope][d_model];  W_QR device [n_heads*d_rope][d_model]
 *   q_out  device [N][n_heads][qk_nope + d_rope] = [q_nope^h || q_R^h]
 * A q_pos outside the RoPE table skips that token's rotated part and is flagged. */
mla_status mla_project_query(const mla_config* cfg, const void* x, const void* W_Q, const void* W_QR,
                             const int32_t* q_pos, const mla_rope_table* rope, void* q_out, int N,
                             void* workspace, size_t workspace_bytes, mla_stream_t stream);

/* Workspace bytes mla_prefill_attention needs for a sequence of kv_len cached
 * tokens: the 256-byte header, the sequence's cache rows gathered in 64-element
 * column chunks (kv_len * row bf16, row = d_c + d_rope, or d_c + n_heads * d_rope
 * with per-head keys) and its rebuilt keys and values
 * (kv_len * n_heads * (qk_nope + v_head) bf16, 64 KB per token at the
 * DeepSeek-V2 shape). */
size_t mla_prefill_workspace_bytes(const mla_config* cfg, int kv_len);

/* Causal attention of the last T tokens of sequence `seq` over its first kv_len
 * cached tokens, in the explicit form:
 *   k_t^h = [W_UK^h c_t || k_R,t],  v_t^h = W_UV^h c_t                 ([BB "1. Low-Rank
 *                                     Decomposition"], names read as up-projections)
 *   s_t^h = scale * (q_nope^h . W_UK^h c_t + q_R^h . k_R,t)  for t <= pos_j
 *   o^h   = sum_t softmax(s^h)_t v_t^h
 * Query j (0 <= j < T) has position pos_j = kv_len - T + j and sees tokens 0..pos_j
 * ([SC]: every prior token keeps an entry).  Its rows must already be in the
 * cache (mla_compress_append of the prompt).
 *   q      device [T][n_heads][qk_nope + d_rope] (mla_project_query output)
 *   cache  the paged cache; seq < cache->batch; kv_len <= max_blocks_per_seq * block_size
 *   W_UK   device [n_heads][qk_nope][d_c];  W_UV device [n_heads][v_head][d_c]
 *   o      device [T][n_heads][v_head]
 *   lse    optional device fp32 [T][n_heads] (natural log of the softmax
 *          normaliser of the scaled scores), or NULL
 * 1 <= T <= kv_len.  Block-table entries outside the pool read as zero rows
 * and are flagged.  With cache_fp8 the gather expands the rows to bf16.
 * Three launches: the latent gather, the K/V GEMM, the attention kernel. */
mla_status mla_prefill_attention(const mla_config* cfg, const void* q, const mla_paged_cache* cache, int seq,
                                 int kv_len, int T, const void* W_UK, const void* W_UV, void* o, float* lse,
                                 void* workspace, size_t workspace_bytes, mla_stream_t stream);

/* Workspace bytes mla_head_output_project needs for N tokens. */
size_t mla_head_output_workspace_bytes(const mla_config* cfg, int N);

/* The output projection of per-head outputs: out = W_O concat_h(o^h).
 *   o    device [N][n_heads][v_head];  W_O device [d_model][n_heads*v_head]
 *   out  device [N][d_model] */
mla_status mla_head_output_project(const mla_config* cfg, const void* o, const void* W_O, void* out, int N,
                                   void* workspace, size_t workspace_bytes, mla_stream_t stream);

/* Synchronise `stream`, then read and clear the status word of `workspace`
 * (the word in its header), or, when workspace is NULL, the library's own word
 * on the current device, which only mla_compress_append_noalloc writes.
 * Returns MLA_OK, MLA_ERR_DEVICE_INDEX or MLA_ERR_TIMEOUT (index takes
 * precedence); *flags (if not NULL) receives the raw bit set (bit 0 index,
 * bit 1 timeout).  Order the read after the calls it should cover: pass the
 * stream they ran on. */
mla_status mla_get_device_status(const void* workspace, mla_stream_t stream, uint32_t* flags);

/* Self-check of the failure detection (no counterpart on the pages): launch one
 * thread that waits on an mbarrier nothing ever completes, using the same
 * bounded-wait routine as every kernel of the library but with a limit of
 * `limit_cycles` SM cycles (10^4 .. 2*10^8, i.e. at most ~0.1 s) instead of
 * ~2 s.  The wait gives up, sets the timeout flag in the workspace's status
 * word and the kernel returns, leaving the context usable;
 * mla_get_device_status(workspace, ...) then reports MLA_ERR_TIMEOUT.
 * workspace: at least the 256-byte header, its status word zero. */
mla_status mla_selftest_wait_timeout(void* workspace, size_t workspace_bytes, uint32_t limit_cycles,
                                     mla_stream_t stream);

/* mla_compress_append without a workspace argument.  No counterpart on the pages:
 * an interface for callers that cannot allocate device memory, for example code
 * that runs where every device allocation is owned by a fixed pool or arena
 * set up at start-up (inference servers, embedded runtimes, other languages'
 * runtimes holding only raw device pointers), or that may not call cudaMalloc
 * on the decode path because it would synchronise the device.
 * Same operation and arguments as mla_compress_append, and the same argument
 * checks in the same order, except:
 *   - the fp32 scratch lives in one fixed 16 MiB array inside the library
 *     (every GPU that loads the library holds it until the process exits);
 *     a call whose scratch would exceed it (mla_compress_workspace_bytes(cfg, T)
 *     minus the 256-byte header > 16 MiB) returns MLA_ERR_WORKSPACE without
 *     touching the GPU; with the DeepSeek-V2 shape on a 148-SM B300 every call
 *     of up to 1024 tokens fits;
 *   - device-side flags go to the library's own status word, read with
 *     mla_get_device_status(NULL, stream, ...);
 *   - the first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress); make that first call before capturing a stream;
 *   - all calls on a device share the array and it keeps the last call's
 *     contents (nothing in it has to start at zero: each call writes every
 *     element it reads), so calls that overlap on the GPU (e.g. on two
 *     streams at once) race; order them on one stream.
 * The function allocates nothing: no cudaMalloc, cudaFree or allocating library call. */
mla_status mla_compress_append_noalloc(const mla_config* cfg, const void* x, const void* W_DKV, const void* W_KR,
                                       const int32_t* seq_idx, const int32_t* pos, const mla_rope_table* rope,
                                       const mla_paged_cache* cache, int T, mla_stream_t stream);

/* Number of kernels this library has launched in this process (all devices).
 * For accounting in benchmarks; no counterpart on the pages. */
uint64_t mla_kernel_launches(void);

/* Static string naming a status code. */
const char* mla_status_string(mla_status status);

#ifdef __cplusplus
}
#endif

#endif /* MLA_H_ */
