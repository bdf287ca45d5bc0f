// extern "C" entry points of the MLA decode library: argument validation,
// workspace carving and kernel dispatch.  The operations themselves are
// documented in include/mla.h.
#include <math.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

#include "mla_common.cuh"
#include "mla_tc.cuh"

namespace mla {

// Device-side error word of calls that take no workspace (bit 0: index skipped, bit 1: bounded wait
// gave up).  Calls with a workspace keep their word in the workspace's header instead.
static __device__ uint32_t g_status_word;

static std::atomic<uint64_t> g_launches{0};
void count_launch(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }

namespace {
struct SmemLimit {
  const void* kernel;
  int device;
  int bytes;
};
std::mutex g_smem_mutex;
SmemLimit g_smem_limits[256];
int g_smem_count = 0;
}  // namespace

cudaError_t ensure_smem_limit(const void* kernel, int bytes, int device) {
  std::lock_guard<std::mutex> lock(g_smem_mutex);
  for (int i = 0; i < g_smem_count; ++i) {
    SmemLimit& l = g_smem_limits[i];
    if (l.kernel == kernel && l.device == device) {
      if (l.bytes >= bytes) return cudaSuccess;
      const cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
      if (e == cudaSuccess) l.bytes = bytes;
      return e;
    }
  }
  const cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && g_smem_count < 256) g_smem_limits[g_smem_count++] = {kernel, device, bytes};
  return e;
}

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_dev_mutex;
uint32_t* g_status_ptr[kMaxDevices] = {};
int g_sm_count[kMaxDevices] = {};

// Per-device constants, resolved once with that device current.  Device-side flags of the call go
// to the status word in the header of `status_ws` (a caller workspace), or to the library's own
// word when it is null.
mla_status device_ctx(cudaStream_t stream, void* status_ws, Ctx* out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MLA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_dev_mutex);
  if (!g_status_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return MLA_ERR_CUDA;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return MLA_ERR_CUDA;
    g_status_ptr[dev] = static_cast<uint32_t*>(p);
    g_sm_count[dev] = sms;
  }
  out->stream = stream;
  out->status = status_ws ? static_cast<uint32_t*>(status_ws) : g_status_ptr[dev];
  out->sm_count = g_sm_count[dev];
  out->device = dev;
  return MLA_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool ok_ptr(const void* p) { return p != nullptr && aligned16(p); }
size_t elem_size(int dtype) { return dtype == MLA_BF16 ? 2 : 4; }
size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

mla_status check_cfg(const mla_config* c) {
  if (!c) return MLA_ERR_INVALID_ARG;
  if (c->d_model <= 0 || c->n_heads <= 0 || c->qk_nope <= 0 || c->d_rope <= 0 || c->v_head <= 0 || c->d_c <= 0 ||
      c->block_size <= 0)
    return MLA_ERR_INVALID_ARG;
  if (c->dtype != MLA_F32 && c->dtype != MLA_BF16) return MLA_ERR_INVALID_ARG;
  if (c->cache_fp8 != 0 && c->cache_fp8 != 1) return MLA_ERR_INVALID_ARG;
  if (c->cache_fp8 && c->dtype != MLA_BF16) return MLA_ERR_UNSUPPORTED;
  // the reduced-precision format's kernels: 64-token blocks, latent in 64-column groups, one warp lane
  // per positional pair
  if (c->cache_fp8 && (c->block_size != 64 || c->d_c % 64 || c->d_rope > 64)) return MLA_ERR_UNSUPPORTED;
  if (c->rope_per_head != 0 && c->rope_per_head != 1) return MLA_ERR_INVALID_ARG;
  if (c->rope_per_head && (c->dtype != MLA_BF16 || c->cache_fp8)) return MLA_ERR_UNSUPPORTED;
  if (c->d_rope % 2) return MLA_ERR_UNSUPPORTED;
  if (c->d_c > 512 || c->d_c + c->d_rope > 2048) return MLA_ERR_UNSUPPORTED;
  return MLA_OK;
}

mla_status check_cache(const mla_paged_cache* k) {
  if (!k || !ok_ptr(k->pool) || !ok_ptr(k->block_table)) return MLA_ERR_INVALID_ARG;
  if (k->num_blocks <= 0 || k->max_blocks_per_seq <= 0 || k->batch <= 0) return MLA_ERR_INVALID_ARG;
  return MLA_OK;
}

mla_status check_rope(const mla_rope_table* r) {
  if (!r || !ok_ptr(r->cos_sin) || r->max_pos <= 0) return MLA_ERR_INVALID_ARG;
  return MLA_OK;
}

float resolve_scale(const mla_config* c) {
  return c->softmax_scale > 0.f ? c->softmax_scale : 1.0f / sqrtf((float)(c->qk_nope + c->d_rope));
}

// Bump allocator over the caller's workspace.
struct Carve {
  char* base;
  size_t used = 0;
  template <typename P> P* take(size_t bytes) {
    P* p = reinterpret_cast<P*>(base ? base + used : nullptr);
    used = align_up(used + bytes, 256);
    return p;
  }
};

// Split plan of the general decode path: enough CTAs to fill the GPU twice.
void simt_split_plan(const mla_config* c, int batch, int n_q, int max_blocks, int sm_count, int* splits,
                     int* tokens_per_split) {
  const long long cap = (long long)max_blocks * c->block_size;
  const long long ctas = (long long)batch * n_q * ((c->n_heads + 3) / 4);
  long long s = ctas > 0 ? (2LL * sm_count + ctas - 1) / ctas : 1;
  const long long max_s = (cap + 255) / 256;
  if (s > max_s) s = max_s;
  if (s < 1) s = 1;
  long long tps = (cap + s - 1) / s;
  tps = (tps + 31) / 32 * 32;
  if (tps < 32) tps = 32;
  *tokens_per_split = (int)tps;
  *splits = (int)((cap + tps - 1) / tps);
}

size_t simt_decode_ws(const mla_config* c, int batch, int n_q, int max_blocks, int sm_count) {
  int splits = 1, tps = 0;
  simt_split_plan(c, batch, n_q, max_blocks, sm_count, &splits, &tps);
  if (splits <= 1) return 0;
  const size_t items = (size_t)batch * n_q;
  Carve cv{nullptr};
  cv.take<float>(items * splits * c->n_heads * c->d_c * sizeof(float));
  cv.take<float>(items * splits * c->n_heads * sizeof(float));
  return cv.used;
}

int current_sm_count() {
  Ctx ctx;
  if (device_ctx(nullptr, nullptr, &ctx) != MLA_OK) return 148;
  return ctx.sm_count;
}

// Every workspace starts with this header; its first word is the status word of the calls that use
// the workspace.
constexpr size_t kWsHeader = kWorkspaceHeaderBytes;

// Workspace check shared by every call: at least `need` bytes (header included), 16-byte aligned.
mla_status check_workspace(const void* ws, size_t bytes, size_t need) {
  if (need == 0) return MLA_ERR_UNSUPPORTED;
  if (bytes < need || !ok_ptr(ws)) return MLA_ERR_WORKSPACE;
  return MLA_OK;
}

char* ws_body(void* ws) { return static_cast<char*>(ws) + kWsHeader; }

#define MLA_TRY(expr)                    \
  do {                                   \
    mla_status _s = (expr);              \
    if (_s != MLA_OK) return _s;         \
  } while (0)
#define MLA_CUDA(expr)                          \
  do {                                          \
    if ((expr) != cudaSuccess) return MLA_ERR_CUDA; \
  } while (0)

}  // namespace
}  // namespace mla

namespace mla {

mla_status validate_append(const mla_config* cfg, const void* x, const void* W_DKV, const void* W_KR,
                           const int32_t* seq_idx, const int32_t* pos, const mla_rope_table* rope,
                           const mla_paged_cache* cache, int T) {
  MLA_TRY(check_cfg(cfg));
  if (T < 0) return MLA_ERR_INVALID_ARG;
  if (T == 0) return MLA_OK;
  if (!ok_ptr(x) || !ok_ptr(W_DKV) || !ok_ptr(W_KR) || !ok_ptr(seq_idx) || !ok_ptr(pos)) return MLA_ERR_INVALID_ARG;
  MLA_TRY(check_rope(rope));
  MLA_TRY(check_cache(cache));
  if (cfg->dtype == MLA_BF16 && !tc_compress_supported(cfg, T)) return MLA_ERR_UNSUPPORTED;
  return MLA_OK;
}

size_t append_scratch_bytes(const mla_config* cfg, int T) {
  if (check_cfg(cfg) != MLA_OK || T < 0) return 0;
  if (cfg->dtype == MLA_BF16) return tc_compress_supported(cfg, T) ? tc_compress_workspace_bytes(cfg, T, current_sm_count()) : 0;
  return align_up((size_t)T * (cfg->d_c + cfg->d_rope) * sizeof(float), 256);
}

mla_status run_append(const mla_config* cfg, const void* x, const void* W_DKV, const void* W_KR,
                      const int32_t* seq_idx, const int32_t* pos, const mla_rope_table* rope,
                      const mla_paged_cache* cache, int T, void* scratch, void* status_ws, cudaStream_t stream) {
  Ctx ctx;
  MLA_TRY(device_ctx(stream, status_ws, &ctx));
  if (cfg->dtype == MLA_BF16) {
    MLA_CUDA(tc_compress_append(ctx, cfg, x, W_DKV, W_KR, seq_idx, pos, *rope, *cache, T, scratch));
    return MLA_OK;
  }
  const int d_c = cfg->d_c, d_r = cfg->d_rope, width = d_c + d_r;
  float* Y = static_cast<float*>(scratch);
  GemmDesc g{};
  g.X = x; g.x_rs = cfg->d_model; g.x_gs = 0; g.x_f32 = 0;
  g.W = W_DKV; g.w_ms = cfg->d_model; g.w_ks = 1; g.w_gs = 0;
  g.Y = Y; g.y_rs = width; g.y_gs = 0; g.y_f32 = 1;
  g.R = T; g.M = d_c; g.K = cfg->d_model; g.G = 1;
  MLA_CUDA(simt_gemm(ctx, cfg->dtype, g));
  g.W = W_KR; g.Y = Y + d_c; g.M = d_r;
  MLA_CUDA(simt_gemm(ctx, cfg->dtype, g));
  MLA_CUDA(simt_compress_epilogue(ctx, cfg->dtype, Y, T, d_c, d_r, seq_idx, pos, *rope, *cache, cfg->block_size));
  return MLA_OK;
}

}  // namespace mla

using namespace mla;

extern "C" {

uint64_t mla_kernel_launches(void) { return g_launches.load(std::memory_order_relaxed); }

const char* mla_status_string(mla_status s) {
  switch (s) {
    case MLA_OK: return "MLA_OK";
    case MLA_ERR_INVALID_ARG: return "MLA_ERR_INVALID_ARG";
    case MLA_ERR_UNSUPPORTED: return "MLA_ERR_UNSUPPORTED";
    case MLA_ERR_CUDA: return "MLA_ERR_CUDA";
    case MLA_ERR_TIMEOUT: return "MLA_ERR_TIMEOUT";
    case MLA_ERR_DEVICE_INDEX: return "MLA_ERR_DEVICE_INDEX";
    case MLA_ERR_WORKSPACE: return "MLA_ERR_WORKSPACE";
  }
  return "MLA_ERR_UNKNOWN";
}

size_t mla_cache_bytes_per_token(const mla_config* cfg) {
  if (check_cfg(cfg) != MLA_OK) return 0;
  if (cfg->cache_fp8) return (size_t)cfg->d_c + 2 * (size_t)cfg->d_rope + 4;
  if (cfg->rope_per_head) return ((size_t)cfg->d_c + (size_t)cfg->n_heads * cfg->d_rope) * 2;
  return (size_t)(cfg->d_c + cfg->d_rope) * elem_size(cfg->dtype);
}

mla_status mla_rope_table_create(const mla_config* cfg, float base, int max_pos, float* d_cos_sin,
                                 mla_stream_t stream) {
  MLA_TRY(check_cfg(cfg));
  if (!ok_ptr(d_cos_sin) || max_pos <= 0 || !(base > 1.0f)) return MLA_ERR_INVALID_ARG;
  Ctx ctx;
  MLA_TRY(device_ctx(stream, nullptr, &ctx));
  MLA_CUDA(rope_table_fill(ctx, base, max_pos, cfg->d_rope, d_cos_sin));
  return MLA_OK;
}

size_t mla_compress_workspace_bytes(const mla_config* cfg, int T) {
  if (check_cfg(cfg) != MLA_OK || T < 0) return 0;
  if (T == 0) return kWsHeader;
  const size_t body = append_scratch_bytes(cfg, T);
  return body ? kWsHeader + body : 0;
}

mla_status mla_compress_append(const mla_config* cfg, const void* x, const void* W_DKV, const void* W_KR,
                               const int32_t* seq_idx, const int32_t* pos, const mla_rope_table* rope,
                               const mla_paged_cache* cache, int T, void* workspace, size_t workspace_bytes,
                               mla_stream_t stream) {
  MLA_TRY(validate_append(cfg, x, W_DKV, W_KR, seq_idx, pos, rope, cache, T));
  if (T == 0) return MLA_OK;
  MLA_TRY(check_workspace(workspace, workspace_bytes, mla_compress_workspace_bytes(cfg, T)));
  return run_append(cfg, x, W_DKV, W_KR, seq_idx, pos, rope, cache, T, ws_body(workspace), workspace, stream);
}

size_t mla_absorb_workspace_bytes(const mla_config* cfg, int N) {
  if (check_cfg(cfg) != MLA_OK || N < 0) return 0;
  if (cfg->dtype == MLA_BF16) {
    if (N == 0) return kWsHeader;
    return tc_absorb_supported(cfg, N) ? kWsHeader + tc_absorb_workspace_bytes(cfg, N, current_sm_count()) : 0;
  }
  const size_t H = cfg->n_heads;
  Carve cv{nullptr};
  cv.take<float>((size_t)N * H * cfg->qk_nope * sizeof(float));
  cv.take<float>((size_t)N * H * cfg->d_rope * sizeof(float));
  cv.take<float>((size_t)N * H * cfg->d_c * sizeof(float));
  return kWsHeader + cv.used;
}

mla_status mla_absorb_query(const mla_config* cfg, const void* x, const void* W_Q, const void* W_QR,
                            const void* W_UK, const int32_t* q_pos, const mla_rope_table* rope, void* q_out, int N,
                            void* workspace, size_t workspace_bytes, mla_stream_t stream) {
  MLA_TRY(check_cfg(cfg));
  if (N < 0) return MLA_ERR_INVALID_ARG;
  if (N == 0) return MLA_OK;
  if (!ok_ptr(x) || !ok_ptr(W_Q) || !ok_ptr(W_QR) || !ok_ptr(W_UK) || !ok_ptr(q_pos) || !ok_ptr(q_out))
    return MLA_ERR_INVALID_ARG;
  MLA_TRY(check_rope(rope));
  if (cfg->dtype == MLA_BF16 && !tc_absorb_supported(cfg, N)) return MLA_ERR_UNSUPPORTED;
  MLA_TRY(check_workspace(workspace, workspace_bytes, mla_absorb_workspace_bytes(cfg, N)));
  Ctx ctx;
  MLA_TRY(device_ctx(stream, workspace, &ctx));
  if (cfg->dtype == MLA_BF16) {
    MLA_CUDA(tc_absorb_query(ctx, cfg, x, W_Q, W_QR, W_UK, q_pos, *rope, q_out, N, ws_body(workspace)));
    return MLA_OK;
  }
  const int H = cfg->n_heads, qn = cfg->qk_nope, d_r = cfg->d_rope, d_c = cfg->d_c;
  Carve cv{ws_body(workspace)};
  float* Yn = cv.take<float>((size_t)N * H * qn * sizeof(float));
  float* Yr = cv.take<float>((size_t)N * H * d_r * sizeof(float));
  float* Ya = cv.take<float>((size_t)N * H * d_c * sizeof(float));
  GemmDesc g{};
  // q_nope = W_Q x   and   q_rope (unrotated) = W_QR x
  g.X = x; g.x_rs = cfg->d_model; g.x_f32 = 0;
  g.W = W_Q; g.w_ms = cfg->d_model; g.w_ks = 1;
  g.Y = Yn; g.y_rs = (long long)H * qn; g.y_f32 = 1;
  g.R = N; g.M = H * qn; g.K = cfg->d_model; g.G = 1;
  MLA_CUDA(simt_gemm(ctx, cfg->dtype, g));
  g.W = W_QR; g.Y = Yr; g.y_rs = (long long)H * d_r; g.M = H * d_r;
  MLA_CUDA(simt_gemm(ctx, cfg->dtype, g));
  // q_abs^h[c] = sum_i q_nope^h[i] W_UK[h][i][c]   (batched over heads)
  GemmDesc a{};
  a.X = Yn; a.x_rs = (long long)H * qn; a.x_gs = qn; a.x_f32 = 1;
  a.W = W_UK; a.w_ms = 1; a.w_ks = d_c; a.w_gs = (long long)qn * d_c;
  a.Y = Ya; a.y_rs = (long long)H * d_c; a.y_gs = d_c; a.y_f32 = 1;
  a.R = N; a.M = d_c; a.K = qn; a.G = H;
  MLA_CUDA(simt_gemm(ctx, cfg->dtype, a));
  MLA_CUDA(simt_query_epilogue(ctx, cfg->dtype, Ya, Yr, N, H, d_c, d_r, q_pos, *rope, q_out));
  return MLA_OK;
}

size_t mla_decode_workspace_bytes(const mla_config* cfg, int batch, int n_q, int max_blocks_per_seq) {
  if (check_cfg(cfg) != MLA_OK || batch < 0 || n_q <= 0 || max_blocks_per_seq <= 0) return 0;
  if (batch == 0) return kWsHeader;
  const int sms = current_sm_count();
  if (cfg->dtype == MLA_BF16) {
    if (!tc_decode_supported(cfg, batch, n_q)) return 0;
    return kWsHeader + align_up(tc_decode_workspace_bytes(cfg, batch, n_q, max_blocks_per_seq, sms), 256) +
           (cfg->cache_fp8 ? fp8_expand_bytes(cfg, batch, max_blocks_per_seq) : 0);
  }
  return kWsHeader + simt_decode_ws(cfg, batch, n_q, max_blocks_per_seq, sms);
}

mla_status mla_decode_attention(const mla_config* cfg, const void* q, const mla_paged_cache* cache,
                                const int32_t* kv_len, int batch, int n_q, void* o_lat, float* lse, void* workspace,
                                size_t workspace_bytes, mla_stream_t stream) {
  MLA_TRY(check_cfg(cfg));
  if (batch < 0 || n_q <= 0) return MLA_ERR_INVALID_ARG;
  if (batch == 0) return MLA_OK;
  if (!ok_ptr(q) || !ok_ptr(kv_len) || !ok_ptr(o_lat) || (lse && !aligned16(lse))) return MLA_ERR_INVALID_ARG;
  MLA_TRY(check_cache(cache));
  if (cache->batch < batch) return MLA_ERR_INVALID_ARG;
  if (cfg->dtype == MLA_BF16 && !tc_decode_supported(cfg, batch, n_q)) return MLA_ERR_UNSUPPORTED;
  MLA_TRY(check_workspace(workspace, workspace_bytes,
                          mla_decode_workspace_bytes(cfg, batch, n_q, cache->max_blocks_per_seq)));
  Ctx ctx;
  MLA_TRY(device_ctx(stream, workspace, &ctx));
  const float scale = resolve_scale(cfg);
  if (cfg->dtype == MLA_BF16) {
    if (cfg->cache_fp8) {
      // the visited blocks expanded to bf16 rows in the workspace, then the same attention kernel
      char* scratch = ws_body(workspace) +
                      align_up(tc_decode_workspace_bytes(cfg, batch, n_q, cache->max_blocks_per_seq, ctx.sm_count), 256);
      mla_paged_cache expanded;
      MLA_CUDA(launch_expand_fp8(ctx, cfg, *cache, kv_len, batch, scratch, &expanded));
      MLA_CUDA(tc_decode_attention(ctx, cfg, q, expanded, kv_len, batch, n_q, scale, o_lat, lse, ws_body(workspace)));
      return MLA_OK;
    }
    MLA_CUDA(tc_decode_attention(ctx, cfg, q, *cache, kv_len, batch, n_q, scale, o_lat, lse, ws_body(workspace)));
    return MLA_OK;
  }
  int splits = 1, tps = 0;
  simt_split_plan(cfg, batch, n_q, cache->max_blocks_per_seq, ctx.sm_count, &splits, &tps);
  const size_t items = (size_t)batch * n_q;
  Carve cv{ws_body(workspace)};
  float* part_o = nullptr;
  float* part_lse = nullptr;
  if (splits > 1) {
    part_o = cv.take<float>(items * splits * cfg->n_heads * cfg->d_c * sizeof(float));
    part_lse = cv.take<float>(items * splits * cfg->n_heads * sizeof(float));
  }
  MLA_CUDA(simt_decode(ctx, cfg->dtype, q, *cache, cfg->block_size, kv_len, batch, n_q, cfg->n_heads, cfg->d_c,
                       cfg->d_rope, scale, splits, tps, part_o, part_lse, o_lat, lse));
  if (splits > 1)
    MLA_CUDA(combine_partials(ctx, cfg->dtype, part_o, part_lse, (int)items, splits, cfg->n_heads, cfg->d_c, o_lat,
                              lse));
  return MLA_OK;
}

size_t mla_output_workspace_bytes(const mla_config* cfg, int N) {
  if (check_cfg(cfg) != MLA_OK || N < 0) return 0;
  if (cfg->dtype == MLA_BF16) {
    if (N == 0) return kWsHeader;
    return tc_output_supported(cfg, N) ? kWsHeader + tc_output_workspace_bytes(cfg, N, current_sm_count()) : 0;
  }
  return kWsHeader + align_up((size_t)N * cfg->n_heads * cfg->v_head * sizeof(float), 256);
}

mla_status mla_output_project(const mla_config* cfg, const void* o_lat, const void* W_UV, const void* W_O, void* out,
                              int N, void* workspace, size_t workspace_bytes, mla_stream_t stream) {
  MLA_TRY(check_cfg(cfg));
  if (N < 0) return MLA_ERR_INVALID_ARG;
  if (N == 0) return MLA_OK;
  if (!ok_ptr(o_lat) || !ok_ptr(W_UV) || !ok_ptr(W_O) || !ok_ptr(out)) return MLA_ERR_INVALID_ARG;
  if (cfg->dtype == MLA_BF16 && !tc_output_supported(cfg, N)) return MLA_ERR_UNSUPPORTED;
  MLA_TRY(check_workspace(workspace, workspace_bytes, mla_output_workspace_bytes(cfg, N)));
  Ctx ctx;
  MLA_TRY(device_ctx(stream, workspace, &ctx));
  if (cfg->dtype == MLA_BF16) {
    MLA_CUDA(tc_output_project(ctx, cfg, o_lat, W_UV, W_O, out, N, ws_body(workspace)));
    return MLA_OK;
  }
  const int H = cfg->n_heads, v = cfg->v_head, d_c = cfg->d_c;
  float* Yo = reinterpret_cast<float*>(ws_body(workspace));
  // o^h[v] = sum_c W_UV[h][v][c] o_lat^h[c]   (batched over heads)
  GemmDesc a{};
  a.X = o_lat; a.x_rs = (long long)H * d_c; a.x_gs = d_c; a.x_f32 = 0;
  a.W = W_UV; a.w_ms = d_c; a.w_ks = 1; a.w_gs = (long long)v * d_c;
  a.Y = Yo; a.y_rs = (long long)H * v; a.y_gs = v; a.y_f32 = 1;
  a.R = N; a.M = v; a.K = d_c; a.G = H;
  MLA_CUDA(simt_gemm(ctx, cfg->dtype, a));
  // out = W_O concat_h o^h
  GemmDesc g{};
  g.X = Yo; g.x_rs = (long long)H * v; g.x_f32 = 1;
  g.W = W_O; g.w_ms = (long long)H * v; g.w_ks = 1;
  g.Y = out; g.y_rs = cfg->d_model; g.y_f32 = 0;
  g.R = N; g.M = cfg->d_model; g.K = H * v; g.G = 1;
  MLA_CUDA(simt_gemm(ctx, cfg->dtype, g));
  return MLA_OK;
}

mla_status mla_get_device_status(const void* workspace, mla_stream_t stream, uint32_t* flags) {
  if (workspace && !aligned16(workspace)) return MLA_ERR_INVALID_ARG;
  Ctx ctx;
  MLA_TRY(device_ctx(stream, const_cast<void*>(workspace), &ctx));
  uint32_t word = 0;
  MLA_CUDA(cudaMemcpyAsync(&word, ctx.status, sizeof(word), cudaMemcpyDeviceToHost, stream));
  MLA_CUDA(cudaMemsetAsync(ctx.status, 0, sizeof(uint32_t), stream));
  MLA_CUDA(cudaStreamSynchronize(stream));
  if (flags) *flags = word;
  if (word & kFlagIndex) return MLA_ERR_DEVICE_INDEX;
  if (word & kFlagTimeout) return MLA_ERR_TIMEOUT;
  return MLA_OK;
}

mla_status mla_selftest_wait_timeout(void* workspace, size_t workspace_bytes, uint32_t limit_cycles,
                                     mla_stream_t stream) {
  if (limit_cycles < 10000u || limit_cycles > 200000000u) return MLA_ERR_INVALID_ARG;
  MLA_TRY(check_workspace(workspace, workspace_bytes, kWsHeader));
  Ctx ctx;
  MLA_TRY(device_ctx(stream, workspace, &ctx));
  MLA_CUDA(launch_wait_timeout_check(ctx, (long long)limit_cycles));
  return MLA_OK;
}

// ------------------------------------------------------------------ explicit form (prefill)
size_t mla_project_workspace_bytes(const mla_config* cfg, int N) {
  if (check_cfg(cfg) != MLA_OK || N < 0 || cfg->dtype != MLA_BF16) return 0;
  if (N == 0) return kWsHeader;
  return tc_project_supported(cfg, N) ? kWsHeader + tc_project_workspace_bytes(cfg, N, current_sm_count()) : 0;
}

mla_status mla_project_query(const mla_config* cfg, const void* x, const void* W_Q, const void* W_QR,
                             const int32_t* q_pos, const mla_rope_table* rope, void* q_out, int N, void* workspace,
                             size_t workspace_bytes, mla_stream_t stream) {
  MLA_TRY(check_cfg(cfg));
  if (N < 0) return MLA_ERR_INVALID_ARG;
  if (N == 0) return MLA_OK;
  if (!ok_ptr(x) || !ok_ptr(W_Q) || !ok_ptr(W_QR) || !ok_ptr(q_pos) || !ok_ptr(q_out)) return MLA_ERR_INVALID_ARG;
  MLA_TRY(check_rope(rope));
  if (cfg->dtype != MLA_BF16 || !tc_project_supported(cfg, N)) return MLA_ERR_UNSUPPORTED;
  MLA_TRY(check_workspace(workspace, workspace_bytes, mla_project_workspace_bytes(cfg, N)));
  Ctx ctx;
  MLA_TRY(device_ctx(stream, workspace, &ctx));
  MLA_CUDA(tc_project_query(ctx, cfg, x, W_Q, W_QR, q_pos, *rope, q_out, N, ws_body(workspace)));
  return MLA_OK;
}

size_t mla_prefill_workspace_bytes(const mla_config* cfg, int kv_len) {
  if (check_cfg(cfg) != MLA_OK || kv_len <= 0 || cfg->dtype != MLA_BF16) return 0;
  const size_t body = tc_prefill_workspace_bytes(cfg, kv_len);
  return body ? kWsHeader + body : 0;
}

mla_status mla_prefill_attention(const mla_config* cfg, const void* q, const mla_paged_cache* cache, int seq,
                                 int kv_len, int T, const void* W_UK, const void* W_UV, void* o, float* lse,
                                 void* workspace, size_t workspace_bytes, mla_stream_t stream) {
  MLA_TRY(check_cfg(cfg));
  if (!ok_ptr(q) || !ok_ptr(W_UK) || !ok_ptr(W_UV) || !ok_ptr(o) || (lse && !aligned16(lse)))
    return MLA_ERR_INVALID_ARG;
  MLA_TRY(check_cache(cache));
  if (seq < 0 || seq >= cache->batch || T < 1 || kv_len < T ||
      (long long)kv_len > (long long)cache->max_blocks_per_seq * cfg->block_size)
    return MLA_ERR_INVALID_ARG;
  if (cfg->dtype != MLA_BF16 || !tc_prefill_supported(cfg)) return MLA_ERR_UNSUPPORTED;
  MLA_TRY(check_workspace(workspace, workspace_bytes, mla_prefill_workspace_bytes(cfg, kv_len)));
  Ctx ctx;
  MLA_TRY(device_ctx(stream, workspace, &ctx));
  MLA_CUDA(tc_prefill_attention(ctx, cfg, q, *cache, seq, kv_len, T, W_UK, W_UV, resolve_scale(cfg), o, lse,
                                ws_body(workspace)));
  return MLA_OK;
}

size_t mla_head_output_workspace_bytes(const mla_config* cfg, int N) {
  if (check_cfg(cfg) != MLA_OK || N < 0 || cfg->dtype != MLA_BF16) return 0;
  if (N == 0) return kWsHeader;
  return tc_head_output_supported(cfg, N) ? kWsHeader + tc_head_output_workspace_bytes(cfg, N, current_sm_count())
                                          : 0;
}

mla_status mla_head_output_project(const mla_config* cfg, const void* o, const void* W_O, void* out, int N,
                                   void* workspace, size_t workspace_bytes, mla_stream_t stream) {
  MLA_TRY(check_cfg(cfg));
  if (N < 0) return MLA_ERR_INVALID_ARG;
  if (N == 0) return MLA_OK;
  if (!ok_ptr(o) || !ok_ptr(W_O) || !ok_ptr(out)) return MLA_ERR_INVALID_ARG;
  if (cfg->dtype != MLA_BF16 || !tc_head_output_supported(cfg, N)) return MLA_ERR_UNSUPPORTED;
  MLA_TRY(check_workspace(workspace, workspace_bytes, mla_head_output_workspace_bytes(cfg, N)));
  Ctx ctx;
  MLA_TRY(device_ctx(stream, workspace, &ctx));
  MLA_CUDA(tc_head_output_project(ctx, cfg, o, W_O, out, N, ws_body(workspace)));
  return MLA_OK;
}

}  // extern "C"
