// Tensor-core (tcgen05 / TMEM / TMA) kernels for the bf16 DeepSeek-V2-shaped layer.
#pragma once

#include <cuda.h>

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

// Explicit form (prefill): query projection without absorption, per-head K / V rebuilt from the latent,
// causal attention per head, and the output projection of per-head outputs.
bool tc_project_supported(const mla_config* cfg, int N);
size_t tc_project_workspace_bytes(const mla_config* cfg, int N, int sm_count);
cudaError_t tc_project_query(const Ctx& ctx, const mla_config* cfg, const void* x, const void* W_Q, const void* W_QR,
                             const int32_t* q_pos, const mla_rope_table& rope, void* q_out, int N, void* workspace);
cudaError_t tc_reconstruct_kv(const Ctx& ctx, const mla_config* cfg, const void* lat, int L, const void* W_UK,
                              const void* W_UV, void* kv);
bool tc_prefill_supported(const mla_config* cfg);
size_t tc_prefill_workspace_bytes(const mla_config* cfg, int kv_len);
cudaError_t tc_prefill_attention(const Ctx& ctx, const mla_config* cfg, const void* q, const mla_paged_cache& cache,
                                 int seq, int kv_len, int T, const void* W_UK, const void* W_UV, float scale, void* o,
                                 float* lse, void* workspace);
bool tc_head_output_supported(const mla_config* cfg, int N);
size_t tc_head_output_workspace_bytes(const mla_config* cfg, int N, int sm_count);
cudaError_t tc_head_output_project(const Ctx& ctx, const mla_config* cfg, const void* o, const void* W_O, void* out,
                                   int N, void* workspace);

// Reduced-precision latent cache (FP8 E4M3 codes with a power-of-two scale per token).
// The append's epilogue from the k-split partials of the stacked W_DKV / W_KR GEMM.
cudaError_t launch_compress_reduce_fp8(const Ctx& ctx, const float* part, int splits, int T, int d_c, int d_r,
                                       const int32_t* seq_idx, const int32_t* pos, const mla_rope_table& rope,
                                       const mla_paged_cache& cache, int block_size);
// Scratch for the decode: batch * max_blocks bf16 blocks and their block table.
size_t fp8_expand_bytes(const mla_config* cfg, int batch, int max_blocks);
// Expand the visited blocks of every sequence into bf16 blocks in `scratch`; *expanded describes them
// as a bf16 paged cache (block b * max_blocks + k holds logical block k of sequence b).
cudaError_t launch_expand_fp8(const Ctx& ctx, const mla_config* cfg, const mla_paged_cache& cache,
                              const int32_t* kv_len, int batch, void* scratch, mla_paged_cache* expanded);
// Prefill: sequence seq's first L rows expanded to bf16 into the chunk-major lat[(d_c + d_rope) / 64][L][64].
cudaError_t launch_gather_latent_fp8(const Ctx& ctx, const mla_config* cfg, const mla_paged_cache& cache, int seq,
                                     int L, void* lat);

// bf16 tensor map of rank 1..5 with the 128-byte swizzle: dims[0] innermost, strides[i] the byte
// stride of dimension i + 1, box the copied extent per dimension.
bool encode_map_bf16(CUtensorMap* m, const void* base, int rank, const uint64_t* dims, const uint64_t* strides,
                     const uint32_t* box);

// Self-check of the bounded waits: one thread waits on an mbarrier nothing completes, gives up after
// limit_cycles and sets the timeout flag in ctx.status.
cudaError_t launch_wait_timeout_check(const Ctx& ctx, long long limit_cycles);

}  // namespace mla
