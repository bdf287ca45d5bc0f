// Shared device helpers and internal launcher declarations for the MLA library.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "mla.h"

namespace mla {

enum : uint32_t { kFlagIndex = 1u, kFlagTimeout = 2u };

// Every caller workspace starts with a header of this many bytes; its first 32-bit word is the
// device status word of the calls that use the workspace.
constexpr size_t kWorkspaceHeaderBytes = 256;

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

using bf16 = __nv_bfloat16;

template <typename T> __device__ __forceinline__ float to_f32(T v);
template <> __device__ __forceinline__ float to_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ float to_f32<bf16>(bf16 v) { return __bfloat162float(v); }

template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ bf16 from_f32<bf16>(float v) { return __float2bfloat16_rn(v); }

// Host-side count of kernel launches (see mla_kernel_launches()).
void count_launch(int n = 1);

// Raise a kernel's dynamic shared-memory limit to `bytes` on `device`, calling the runtime only when
// the limit grows (so that launches made while a stream is being captured into a graph do not).
cudaError_t ensure_smem_limit(const void* kernel, int bytes, int device);

__device__ __forceinline__ void flag_error(uint32_t* status, uint32_t bit) { atomicOr(status, bit); }

// Physical block holding logical position `pos` of sequence b, or -1 when any index is out of range.
// The pool stores each block transposed, [row element][block_size tokens]: element e of the token at
// offset o of block k lives at ((k * row_width + e) * block_size + o).
__device__ __forceinline__ int cache_block(const int32_t* table, int max_blocks, int num_blocks, int block_size,
                                           int b, int pos) {
  if (pos < 0 || pos >= max_blocks * block_size) return -1;
  const int blk = table[(long long)b * max_blocks + pos / block_size];
  return (blk < 0 || blk >= num_blocks) ? -1 : blk;
}

// ------------------------------------------------------------------ programmatic dependent launch
// Every kernel of the decode step lets the next kernel in its stream be scheduled as soon as it starts
// (pdl_trigger), and reads or writes global memory only after the kernel before it has completed
// (pdl_wait, placed after the CTA's own set-up: barrier init, TMEM allocation, tensor-map prefetch).
// A kernel's set-up thus overlaps the previous kernel's tail; since every kernel waits before it
// completes, completion stays ordered along the stream.  Without the launch attribute both are no-ops.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ------------------------------------------------------------------ launch plumbing
struct Ctx {
  cudaStream_t stream;
  uint32_t* status;   // device error word of this call (its workspace header, or the library's word)
  int sm_count;
  int device;
};

// Argument checks of the cache append shared by the allocating and the allocation-free entry points,
// in the order they are applied (no workspace check).
mla_status validate_append(const mla_config* cfg, const void* x, const void* W_DKV, const void* W_KR,
                           const int32_t* seq_idx, const int32_t* pos, const mla_rope_table* rope,
                           const mla_paged_cache* cache, int T);
// Scratch bytes the append of T tokens needs beyond the workspace header (0: unsupported).
size_t append_scratch_bytes(const mla_config* cfg, int T);
// The append after validation: `scratch` holds append_scratch_bytes(cfg, T) bytes; device-side
// flags go to the status word in the header of `status_ws`, or to the library's word when null.
// Launch `kernel` as a programmatic dependent of the previous kernel in `stream` (see pdl_wait).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args&&... args) {
  cudaLaunchConfig_t lc = {};
  lc.gridDim = grid;
  lc.blockDim = block;
  lc.dynamicSmemBytes = smem;
  lc.stream = stream;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = at;
  lc.numAttrs = 1;
  return cudaLaunchKernelEx(&lc, kernel, static_cast<KArgs>(args)...);
}

mla_status run_append(const mla_config* cfg, const void* x, const void* W_DKV, const void* W_KR,
                      const int32_t* seq_idx, const int32_t* pos, const mla_rope_table* rope,
                      const mla_paged_cache* cache, int T, void* scratch, void* status_ws, cudaStream_t stream);

// Generic strided GEMM description: Y[g][r][m] = sum_k X[g][r][k] * W[g][m][k]
// where W is addressed as W + g*w_gs + m*w_ms + k*w_ks (so both [m][k] and
// [k][m] weight layouts are expressible).
struct GemmDesc {
  const void* X; long long x_rs, x_gs; int x_f32;   // X element type: fp32 or the storage dtype
  const void* W; long long w_ms, w_ks, w_gs;
  void* Y; long long y_rs, y_gs; int y_f32;         // Y element type: fp32 or the storage dtype
  int R, M, K, G;
};

// SIMT kernels (any shape, fp32 or bf16 storage).
cudaError_t simt_gemm(const Ctx&, int dtype, const GemmDesc&);
cudaError_t simt_compress_epilogue(const Ctx&, int dtype, const float* Y, int T, int d_c, int d_r,
                                   const int32_t* seq_idx, const int32_t* pos, const mla_rope_table& rope,
                                   const mla_paged_cache& cache, int block_size);
cudaError_t simt_query_epilogue(const Ctx&, int dtype, const float* Y_abs, const float* Y_rope, int N, int H,
                                int d_c, int d_r, const int32_t* q_pos, const mla_rope_table& rope, void* q_out);
cudaError_t simt_decode(const Ctx&, int dtype, const void* q, const mla_paged_cache& cache, int block_size,
                        const int32_t* kv_len, int B, int n_q, int H, int d_c, int d_r, float scale,
                        int splits, int tokens_per_split, float* part_o, float* part_lse, void* o_lat,
                        float* lse_out);
cudaError_t combine_partials(const Ctx&, int dtype, const float* part_o, const float* part_lse, int items,
                             int splits, int H, int d_c, void* o_lat, float* lse_out);
cudaError_t rope_table_fill(const Ctx&, float base, int max_pos, int d_rope, float* cos_sin);

}  // namespace mla
