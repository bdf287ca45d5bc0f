// General SIMT (CUDA-core, fp32 arithmetic) kernels for every MLA decode step.
//
// These serve fp32 storage at any layer shape: tensor cores cannot hold fp32
// operands at fp32 accuracy.  bf16 storage runs only on the tcgen05 kernels
// (mla_decode_tc.cu, mla_gemm_tc.cu); these entry points refuse it.  The math
// of each step is documented in include/mla.h.
#include <math.h>

#include "mla_common.cuh"

namespace mla {
namespace {

// ------------------------------------------------------------------ GEMM
constexpr int kBR = 64, kBM = 64, kBK = 16;

template <typename T, typename XT, typename YT>
__global__ void __launch_bounds__(256) simt_gemm_kernel(GemmDesc d) {
  __shared__ float xs[kBK][kBR + 4];
  __shared__ float ws[kBK][kBM + 4];
  const int g = blockIdx.z;
  const int r0 = blockIdx.y * kBR, m0 = blockIdx.x * kBM;
  const XT* X = reinterpret_cast<const XT*>(d.X) + (long long)g * d.x_gs;
  const T* W = reinterpret_cast<const T*>(d.W) + (long long)g * d.w_gs;
  YT* Y = reinterpret_cast<YT*>(d.Y) + (long long)g * d.y_gs;
  const int tid = threadIdx.x, tx = tid % 16, ty = tid / 16;
  float acc[4][4] = {};
  const bool w_k_contig = (d.w_ks == 1);
  for (int k0 = 0; k0 < d.K; k0 += kBK) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      int e = tid + i * 256;
      int r = e / kBK, k = e % kBK;
      float v = 0.f;
      if (r0 + r < d.R && k0 + k < d.K) v = to_f32<XT>(X[(long long)(r0 + r) * d.x_rs + k0 + k]);
      xs[k][r] = v;
      int m, kk;
      if (w_k_contig) { m = e / kBK; kk = e % kBK; } else { kk = e / kBM; m = e % kBM; }
      float w = 0.f;
      if (m0 + m < d.M && k0 + kk < d.K) w = to_f32<T>(W[(long long)(m0 + m) * d.w_ms + (long long)(k0 + kk) * d.w_ks]);
      ws[kk][m] = w;
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < kBK; ++k) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) { a[i] = xs[k][ty * 4 + i]; b[i] = ws[k][tx * 4 + i]; }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    int r = r0 + ty * 4 + i;
    if (r >= d.R) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      int m = m0 + tx * 4 + j;
      if (m < d.M) Y[(long long)r * d.y_rs + m] = from_f32<YT>(acc[i][j]);
    }
  }
}

template <typename T>
cudaError_t gemm_typed(const Ctx& c, const GemmDesc& d) {
  dim3 grid((d.M + kBM - 1) / kBM, (d.R + kBR - 1) / kBR, d.G);
  if (d.x_f32 && d.y_f32) simt_gemm_kernel<T, float, float><<<grid, 256, 0, c.stream>>>(d);
  else if (d.x_f32) simt_gemm_kernel<T, float, T><<<grid, 256, 0, c.stream>>>(d);
  else if (d.y_f32) simt_gemm_kernel<T, T, float><<<grid, 256, 0, c.stream>>>(d);
  else simt_gemm_kernel<T, T, T><<<grid, 256, 0, c.stream>>>(d);
  count_launch();
  return cudaGetLastError();
}

// ------------------------------------------------------------------ RoPE helpers
// Rotate the pair (a, b) by the tabulated angle: (a cos - b sin, a sin + b cos).
__device__ __forceinline__ void rope_pair(float a, float b, const float* cs, float& o0, float& o1) {
  const float cosv = cs[0], sinv = cs[1];
  o0 = a * cosv - b * sinv;
  o1 = a * sinv + b * cosv;
}

template <typename T>
__global__ void compress_epilogue_kernel(const float* __restrict__ Y, int T_, int d_c, int d_r,
                                         const int32_t* __restrict__ seq_idx, const int32_t* __restrict__ pos,
                                         const float* __restrict__ rope, int rope_max, T* pool, int num_blocks,
                                         const int32_t* __restrict__ table, int max_blocks, int batch,
                                         int block_size, uint32_t* status) {
  const int t = blockIdx.x;
  const int b = seq_idx[t], p = pos[t];
  int blk = -1;
  if (b >= 0 && b < batch && p < rope_max) blk = cache_block(table, max_blocks, num_blocks, block_size, b, p);
  if (blk < 0) {
    if (threadIdx.x == 0) flag_error(status, kFlagIndex);
    return;
  }
  const int width = d_c + d_r;
  const float* y = Y + (long long)t * width;
  // element e of this token: pool[(blk * width + e) * block_size + p % block_size]
  T* dst = pool + (long long)blk * width * block_size + p % block_size;
  for (int i = threadIdx.x; i < d_c; i += blockDim.x) dst[(long long)i * block_size] = from_f32<T>(y[i]);
  for (int i = threadIdx.x; i < d_r / 2; i += blockDim.x) {
    float o0, o1;
    rope_pair(y[d_c + 2 * i], y[d_c + 2 * i + 1], rope + ((long long)p * (d_r / 2) + i) * 2, o0, o1);
    dst[(long long)(d_c + 2 * i) * block_size] = from_f32<T>(o0);
    dst[(long long)(d_c + 2 * i + 1) * block_size] = from_f32<T>(o1);
  }
}

template <typename T>
__global__ void query_epilogue_kernel(const float* __restrict__ Y_abs, const float* __restrict__ Y_rope, int H,
                                      int d_c, int d_r, const int32_t* __restrict__ q_pos,
                                      const float* __restrict__ rope, int rope_max, T* q_out, uint32_t* status) {
  const int n = blockIdx.x, h = blockIdx.y;
  const int p = q_pos[n];
  const int width = d_c + d_r;
  T* dst = q_out + ((long long)n * H + h) * width;
  const float* ya = Y_abs + ((long long)n * H + h) * d_c;
  for (int i = threadIdx.x; i < d_c; i += blockDim.x) dst[i] = from_f32<T>(ya[i]);
  if (p < 0 || p >= rope_max) {
    if (threadIdx.x == 0) flag_error(status, kFlagIndex);
    return;
  }
  const float* yr = Y_rope + ((long long)n * H + h) * d_r;
  for (int i = threadIdx.x; i < d_r / 2; i += blockDim.x) {
    float o0, o1;
    rope_pair(yr[2 * i], yr[2 * i + 1], rope + ((long long)p * (d_r / 2) + i) * 2, o0, o1);
    dst[d_c + 2 * i] = from_f32<T>(o0);
    dst[d_c + 2 * i + 1] = from_f32<T>(o1);
  }
}

// ------------------------------------------------------------------ decode attention
constexpr int kChunk = 32;      // tokens per smem tile (one per lane when scoring)
constexpr int kHeadsPerCta = 4; // one warp per head
constexpr int kMaxPerLane = 16; // d_c <= 512

template <typename T>
__global__ void __launch_bounds__(128) simt_decode_kernel(
    const T* __restrict__ q, const T* __restrict__ pool, const int32_t* __restrict__ table, int max_blocks,
    int num_blocks, int block_size, const int32_t* __restrict__ kv_len, int n_q, int H, int d_c, int d_r,
    float scale_log2, int splits, int tokens_per_split, float* part_o, float* part_lse, T* o_lat,
    float* lse_out, uint32_t* status) {
  extern __shared__ float smem[];
  const int width = d_c + d_r, stride = width + 1;
  float* qs = smem;                              // [kHeadsPerCta][width]
  float* tile = smem + kHeadsPerCta * width;     // [kChunk][stride]
  const int item = blockIdx.x;                   // b * n_q + j
  const int b = item / n_q, j = item % n_q;
  const int h0 = blockIdx.y * kHeadsPerCta;
  const int split = blockIdx.z;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int h = h0 + warp;

  int kv = kv_len[b];
  const int cap = max_blocks * block_size;
  if (kv < 0 || kv > cap) {
    if (threadIdx.x == 0) flag_error(status, kFlagIndex);
    kv = kv < 0 ? 0 : cap;
  }
  int vis = kv - (n_q - 1 - j);
  if (vis < 0) vis = 0;
  const int t_begin = split * tokens_per_split;
  int t_end = t_begin + tokens_per_split;
  if (t_end > vis) t_end = vis;

  for (int i = threadIdx.x; i < kHeadsPerCta * width; i += blockDim.x) {
    int hh = h0 + i / width;
    qs[i] = hh < H ? to_f32<T>(q[((long long)item * H + hh) * width + i % width]) : 0.f;
  }
  float m = -INFINITY, l = 0.f;
  float acc[kMaxPerLane];
#pragma unroll
  for (int i = 0; i < kMaxPerLane; ++i) acc[i] = 0.f;
  const int per_lane = (d_c + 31) / 32;

  __shared__ int tile_blk[kChunk];
  for (int t0 = t_begin; t0 < t_end; t0 += kChunk) {
    const int count = min(kChunk, t_end - t0);
    __syncthreads();
    if (threadIdx.x < count) {
      const int blk = cache_block(table, max_blocks, num_blocks, block_size, b, t0 + threadIdx.x);
      if (blk < 0) flag_error(status, kFlagIndex);
      tile_blk[threadIdx.x] = blk;
    }
    __syncthreads();
    // element i of token r: pool[(blk * width + i) * block_size + (t0 + r) % block_size]
    for (int idx = threadIdx.x; idx < count * width; idx += blockDim.x) {
      const int i = idx / count, r = idx % count;
      const int blk = tile_blk[r];
      tile[r * stride + i] =
          blk < 0 ? 0.f
                  : to_f32<T>(pool[((long long)blk * width + i) * block_size + (t0 + r) % block_size]);
    }
    __syncthreads();
    if (h >= H) continue;
    const float* qh = qs + warp * width;
    float s = -INFINITY;
    if (lane < count) {
      const float* kt = tile + lane * stride;
      float dot = 0.f;
      for (int i = 0; i < width; ++i) dot = fmaf(qh[i], kt[i], dot);
      s = dot * scale_log2;
    }
    float cmax = s;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) cmax = fmaxf(cmax, __shfl_xor_sync(0xffffffffu, cmax, o));
    const float m_new = fmaxf(m, cmax);
    const float alpha = (m == -INFINITY) ? 0.f : exp2f(m - m_new);
    const float p = (lane < count) ? exp2f(s - m_new) : 0.f;
    float psum = p;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) psum += __shfl_xor_sync(0xffffffffu, psum, o);
    l = l * alpha + psum;
    m = m_new;
#pragma unroll
    for (int i = 0; i < kMaxPerLane; ++i) acc[i] *= alpha;
    for (int t = 0; t < count; ++t) {
      const float pt = __shfl_sync(0xffffffffu, p, t);
      const float* vt = tile + t * stride;
#pragma unroll
      for (int i = 0; i < kMaxPerLane; ++i)
        if (i < per_lane && lane + 32 * i < d_c) acc[i] = fmaf(pt, vt[lane + 32 * i], acc[i]);
    }
  }
  if (h >= H) return;
  const float inv = l > 0.f ? 1.f / l : 0.f;
  const float lse = l > 0.f ? (m + log2f(l)) * kLn2 : -INFINITY;
  if (splits == 1) {
    T* dst = o_lat + ((long long)item * H + h) * d_c;
#pragma unroll
    for (int i = 0; i < kMaxPerLane; ++i)
      if (i < per_lane && lane + 32 * i < d_c) dst[lane + 32 * i] = from_f32<T>(acc[i] * inv);
    if (lse_out && lane == 0) lse_out[(long long)item * H + h] = lse;
  } else {
    const long long slot = ((long long)item * splits + split) * H + h;
    float* dst = part_o + slot * d_c;
#pragma unroll
    for (int i = 0; i < kMaxPerLane; ++i)
      if (i < per_lane && lane + 32 * i < d_c) dst[lane + 32 * i] = acc[i] * inv;
    if (lane == 0) part_lse[slot] = lse;
  }
}

// o = sum_s exp(lse_s - lse) o_s,  lse = log sum_s exp(lse_s); partials laid out [item][split][H][d_c].
template <typename T>
__global__ void combine_kernel(const float* __restrict__ part_o, const float* __restrict__ part_lse, int splits,
                               int H, int d_c, T* o_lat, float* lse_out) {
  const int item = blockIdx.x, h = blockIdx.y;
  float mx = -INFINITY;
  for (int s = 0; s < splits; ++s) mx = fmaxf(mx, part_lse[((long long)item * splits + s) * H + h]);
  float z = 0.f;
  for (int s = 0; s < splits; ++s) {
    float ls = part_lse[((long long)item * splits + s) * H + h];
    z += (ls == -INFINITY) ? 0.f : expf(ls - mx);
  }
  const float inv = z > 0.f ? 1.f / z : 0.f;
  T* dst = o_lat + ((long long)item * H + h) * d_c;
  for (int i = threadIdx.x; i < d_c; i += blockDim.x) {
    float acc = 0.f;
    for (int s = 0; s < splits; ++s) {
      const long long slot = ((long long)item * splits + s) * H + h;
      float ls = part_lse[slot];
      if (ls != -INFINITY) acc = fmaf(expf(ls - mx), part_o[slot * d_c + i], acc);
    }
    dst[i] = from_f32<T>(acc * inv);
  }
  if (lse_out && threadIdx.x == 0) lse_out[(long long)item * H + h] = z > 0.f ? mx + logf(z) : -INFINITY;
}

__global__ void rope_table_kernel(double base, int max_pos, int d_rope, float* cos_sin) {
  const int half = d_rope / 2;
  const long long n = (long long)max_pos * half;
  for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < n; e += (long long)gridDim.x * blockDim.x) {
    const int p = (int)(e / half), i = (int)(e % half);
    const double theta = pow(base, -2.0 * i / d_rope);
    double sv, cv;
    sincos((double)p * theta, &sv, &cv);
    cos_sin[2 * e] = (float)cv;
    cos_sin[2 * e + 1] = (float)sv;
  }
}

}  // namespace

cudaError_t simt_gemm(const Ctx& c, int dtype, const GemmDesc& d) {
  if (dtype != MLA_F32) return cudaErrorNotSupported;
  if (d.R == 0 || d.M == 0 || d.G == 0) return cudaSuccess;
  return gemm_typed<float>(c, d);
}

cudaError_t simt_compress_epilogue(const Ctx& c, int dtype, const float* Y, int T_, int d_c, int d_r,
                                   const int32_t* seq_idx, const int32_t* pos, const mla_rope_table& rope,
                                   const mla_paged_cache& cache, int block_size) {
  if (dtype != MLA_F32) return cudaErrorNotSupported;
  if (T_ == 0) return cudaSuccess;
  compress_epilogue_kernel<float><<<T_, 128, 0, c.stream>>>(Y, T_, d_c, d_r, seq_idx, pos, rope.cos_sin, rope.max_pos,
                                                              (float*)cache.pool, cache.num_blocks, cache.block_table,
                                                              cache.max_blocks_per_seq, cache.batch, block_size, c.status);
  count_launch();
  return cudaGetLastError();
}

cudaError_t simt_query_epilogue(const Ctx& c, int dtype, const float* Y_abs, const float* Y_rope, int N, int H,
                                int d_c, int d_r, const int32_t* q_pos, const mla_rope_table& rope, void* q_out) {
  if (dtype != MLA_F32) return cudaErrorNotSupported;
  if (N == 0) return cudaSuccess;
  dim3 grid(N, H);
  query_epilogue_kernel<float><<<grid, 128, 0, c.stream>>>(Y_abs, Y_rope, H, d_c, d_r, q_pos, rope.cos_sin,
                                                             rope.max_pos, (float*)q_out, c.status);
  count_launch();
  return cudaGetLastError();
}

cudaError_t simt_decode(const Ctx& c, int dtype, const void* q, const mla_paged_cache& cache, int block_size,
                        const int32_t* kv_len, int B, int n_q, int H, int d_c, int d_r, float scale, int splits,
                        int tokens_per_split, float* part_o, float* part_lse, void* o_lat, float* lse_out) {
  if (dtype != MLA_F32) return cudaErrorNotSupported;
  if (B == 0) return cudaSuccess;
  const int width = d_c + d_r;
  const size_t smem = sizeof(float) * (kHeadsPerCta * width + kChunk * (width + 1));
  dim3 grid(B * n_q, (H + kHeadsPerCta - 1) / kHeadsPerCta, splits);
  const float scale_log2 = scale * kLog2e;
  {
    auto k = simt_decode_kernel<float>;
    const cudaError_t ea = ensure_smem_limit((const void*)k, (int)smem, c.device);
    if (ea != cudaSuccess) return ea;
    k<<<grid, 128, smem, c.stream>>>((const float*)q, (const float*)cache.pool, cache.block_table,
                                     cache.max_blocks_per_seq, cache.num_blocks, block_size, kv_len, n_q, H, d_c, d_r,
                                     scale_log2, splits, tokens_per_split, part_o, part_lse, (float*)o_lat, lse_out,
                                     c.status);
  }
  count_launch();
  return cudaGetLastError();
}

cudaError_t combine_partials(const Ctx& c, int dtype, const float* part_o, const float* part_lse, int items,
                             int splits, int H, int d_c, void* o_lat, float* lse_out) {
  if (dtype != MLA_F32) return cudaErrorNotSupported;
  if (items == 0) return cudaSuccess;
  dim3 grid(items, H);
  combine_kernel<float><<<grid, 128, 0, c.stream>>>(part_o, part_lse, splits, H, d_c, (float*)o_lat, lse_out);
  count_launch();
  return cudaGetLastError();
}

cudaError_t rope_table_fill(const Ctx& c, float base, int max_pos, int d_rope, float* cos_sin) {
  long long n = (long long)max_pos * (d_rope / 2);
  int blocks = (int)((n + 255) / 256);
  if (blocks > 4096) blocks = 4096;
  if (blocks < 1) blocks = 1;
  rope_table_kernel<<<blocks, 256, 0, c.stream>>>((double)base, max_pos, d_rope, cos_sin);
  count_launch();
  return cudaGetLastError();
}

}  // namespace mla
