// Tensor-core (tcgen05 / TMEM / TMA) kernels for the bf16 DeepSeek-V2-shaped layer.
#pragma once

#include "mla_common.cuh"

namespace mla {

bool tc_decode_supported(const mla_config* cfg, int batch, int n_q);
size_t tc_decode_workspace_bytes(const mla_config* cfg, int batch, int n_q, int max_blocks, int sm_count);
cudaError_t tc_decode_attention(const Ctx& ctx, const mla_config* cfg, const void* q, const mla_paged_cache& cache,
                                const int32_t* kv_len, int batch, int n_q, float scale, void* o_lat, float* lse,
                                void* workspace);

bool tc_compress_supported(const mla_config* cfg, int T);
size_t tc_compress_workspace_bytes(const mla_config* cfg, int T, int sm_count);
cudaError_t tc_compress_append(const Ctx& ctx, const mla_config* cfg, const void* x, const void* W_DKV,
                               const void* W_KR, const int32_t* seq_idx, const int32_t* pos,
                               const mla_rope_table& rope, const mla_paged_cache& cache, int T, void* workspace);

bool tc_absorb_supported(const mla_config* cfg, int N);
size_t tc_absorb_workspace_bytes(const mla_config* cfg, int N, int sm_count);
cudaError_t tc_absorb_query(const Ctx& ctx, const mla_config* cfg, const void* x, const void* W_Q, const void* W_QR,
                            const void* W_UK, const int32_t* q_pos, const mla_rope_table& rope, void* q_out, int N,
                            void* workspace);

bool tc_output_supported(const mla_config* cfg, int N);
size_t tc_output_workspace_bytes(const mla_config* cfg, int N, int sm_count);
cudaError_t tc_output_project(const Ctx& ctx, const mla_config* cfg, const void* o_lat, const void* W_UV,
                              const void* W_O, void* out, int N, void* workspace);

// Self-check of the bounded waits: one thread waits on an mbarrier nothing completes, gives up after
// limit_cycles and sets the timeout flag in ctx.status.
cudaError_t launch_wait_timeout_check(const Ctx& ctx, long long limit_cycles);

}  // namespace mla
