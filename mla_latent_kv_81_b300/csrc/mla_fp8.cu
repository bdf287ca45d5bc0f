// The reduced-precision latent cache ("What does Multi-head Latent Attention compress...", "Compression
// as architecture versus compression as post-processing": a latent representation can itself be stored
// in a reduced-precision format).  The format (the pages name none): per token, FP8 E4M3 codes of
// c_t / s_t with s_t the smallest power of two for which max|c_t| / s_t <= 448 (1 for an all-zero row),
// rounded to nearest even; the positional key as bf16 k_R,t / s_t (exact, s_t a power of two); s_t as
// fp32.  Per block of B tokens, element-major: codes [d_c][B] bytes, k_R / s [d_rope][B] bf16, s [B].
//
//   compress_reduce_fp8_kernel  the append's epilogue: sums the k-split partials of the stacked W_DKV /
//                               W_KR GEMM, rotates k_R, picks s_t and writes the quantised row;
//   expand_fp8_blocks_kernel    decode: the visited blocks of every sequence expanded to bf16 rows
//                               (codes * s and (k_R / s) * s, both exact) for the attention kernel;
//   gather_latent_fp8_kernel    prefill: one sequence's rows expanded into the chunk-major buffer the
//                               K/V GEMM and the attention kernel read.
#include <cuda_fp16.h>

#include "mla_tc.cuh"

namespace mla {
namespace {

constexpr float kE4M3Max = 448.f;

// Smallest k with m <= 448 * 2^k (m > 0, finite): exact comparisons of fp32 powers of two times 448.
__device__ __forceinline__ int fp8_scale_exponent(float m) {
  if (!(m > 0.f)) return 0;
  int k = ilogbf(m) - 10;
  while (m > ldexpf(kE4M3Max, k)) ++k;
  return k;
}

// Two fp32 values to two E4M3 codes (round to nearest even, saturating to +-448): lo in bits 0-7.
__device__ __forceinline__ uint16_t to_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Two E4M3 codes (lo in bits 0-7) to two floats (exact).
__device__ __forceinline__ float2 from_e4m3x2(uint16_t v) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(v));
  return __half22float2(*reinterpret_cast<const __half2*>(&h2));
}

// Warp = token t0 + warp of the block; lane l holds the latent columns 2l + 64 i, 2l + 64 i + 1
// (i < d_c / 64) and the positional pair d_c + 2l, d_c + 2l + 1 (l < d_r / 2).
constexpr int kFp8Tok = 8;
constexpr int kMaxLatPerLane = 16;   // d_c <= 512

__global__ void __launch_bounds__(256) compress_reduce_fp8_kernel(
    const float* part, int splits, int T, int d_c, int d_r, const int32_t* seq_idx, const int32_t* pos,
    const float* rope, int rope_max, uint8_t* pool, int num_blocks, const int32_t* table, int max_blocks,
    int batch, int block_size, uint32_t* status) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * kFp8Tok + warp;
  if (t >= T) return;
  const int width = d_c + d_r;
  const int b = seq_idx[t], p_t = pos[t];
  int blk = -1;
  if (b >= 0 && b < batch && p_t >= 0 && p_t < rope_max)
    blk = cache_block(table, max_blocks, num_blocks, block_size, b, p_t);
  if (blk < 0) {
    if (lane == 0) flag_error(status, kFlagIndex);
    return;
  }
  const long long sstride = (long long)T * width, row = (long long)t * width;
  auto sum2 = [&](int col) {
    float2 acc = make_float2(0.f, 0.f);
    for (int sp = 0; sp < splits; ++sp) {
      const float2 w = *reinterpret_cast<const float2*>(part + sp * sstride + row + col);
      acc.x += w.x;
      acc.y += w.y;
    }
    return acc;
  };
  // the latent values of this lane and the row maximum of |c|
  float2 c[kMaxLatPerLane / 2];
  float mx = 0.f;
  const int nlat = d_c / 64;
#pragma unroll
  for (int i = 0; i < kMaxLatPerLane / 2; ++i) {
    if (i < nlat) {
      c[i] = sum2(64 * i + 2 * lane);
      mx = fmaxf(mx, fmaxf(fabsf(c[i].x), fabsf(c[i].y)));
    }
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  const int k = fp8_scale_exponent(mx);
  const long long bbytes = (long long)block_size * (d_c + 2 * d_r + 4);
  uint8_t* base = pool + blk * bbytes;
  const int off = p_t % block_size;
#pragma unroll
  for (int i = 0; i < kMaxLatPerLane / 2; ++i) {
    if (i < nlat) {
      const uint16_t q = to_e4m3x2(ldexpf(c[i].x, -k), ldexpf(c[i].y, -k));
      const int e = 64 * i + 2 * lane;
      base[(long long)e * block_size + off] = (uint8_t)(q & 0xFF);
      base[(long long)(e + 1) * block_size + off] = (uint8_t)(q >> 8);
    }
  }
  // the positional key: rotate the pair, divide by the token's scale, round to bf16
  if (2 * lane < d_r) {
    const float2 v = sum2(d_c + 2 * lane);
    const float* cs = rope + ((long long)p_t * (d_r / 2) + lane) * 2;
    const float o0 = v.x * cs[0] - v.y * cs[1], o1 = v.x * cs[1] + v.y * cs[0];
    bf16* kr = reinterpret_cast<bf16*>(base + (long long)d_c * block_size);
    kr[(long long)(2 * lane) * block_size + off] = __float2bfloat16_rn(ldexpf(o0, -k));
    kr[(long long)(2 * lane + 1) * block_size + off] = __float2bfloat16_rn(ldexpf(o1, -k));
  }
  if (lane == 0)
    reinterpret_cast<float*>(base + (long long)(d_c + 2 * d_r) * block_size)[off] = ldexpf(1.f, k);
}

// Expand one 64-token block of the reduced-precision format into bf16 [d_c + d_r][64] at dst.
// 256 threads; thread = (row, 8-token group).  src == nullptr writes zeros.
__device__ __forceinline__ void expand_block(const uint8_t* src, bf16* dst, int d_c, int d_r) {
  constexpr int kB = 64;
  __shared__ float sc[kB];
  if (threadIdx.x < kB) sc[threadIdx.x] = src ? reinterpret_cast<const float*>(src + (d_c + 2 * d_r) * kB)[threadIdx.x] : 0.f;
  __syncthreads();
  const int rows = d_c + d_r;
  for (int w = threadIdx.x; w < rows * (kB / 8); w += blockDim.x) {
    const int e = w >> 3, t0 = (w & 7) * 8;
    float v[8];
    if (!src) {
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] = 0.f;
    } else if (e < d_c) {
      const uint2 raw = *reinterpret_cast<const uint2*>(src + (long long)e * kB + t0);
      const uint32_t wds[2] = {raw.x, raw.y};
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const float2 a = from_e4m3x2((uint16_t)(wds[j] & 0xFFFF)), b2 = from_e4m3x2((uint16_t)(wds[j] >> 16));
        v[4 * j] = a.x; v[4 * j + 1] = a.y; v[4 * j + 2] = b2.x; v[4 * j + 3] = b2.y;
      }
    } else {
      const uint4 raw = *reinterpret_cast<const uint4*>(src + (long long)d_c * kB + ((long long)(e - d_c) * kB + t0) * 2);
      const uint32_t wds[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const __nv_bfloat162 h = *reinterpret_cast<const __nv_bfloat162*>(&wds[j]);
        v[2 * j] = __low2float(h);
        v[2 * j + 1] = __high2float(h);
      }
    }
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * j] * sc[t0 + 2 * j], v[2 * j + 1] * sc[t0 + 2 * j + 1]);
      o[j] = *reinterpret_cast<const uint32_t*>(&h);
    }
    *reinterpret_cast<uint4*>(dst + (long long)e * kB + t0) = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// Block (k, b): logical block k of sequence b, if it holds a visible token, expanded into dst block
// b * max_blocks + k; the table entry of that block is written to out_table.
__global__ void __launch_bounds__(256) expand_fp8_blocks_kernel(const uint8_t* pool, int num_blocks,
                                                                const int32_t* table, int max_blocks,
                                                                const int32_t* kv_len, int d_c, int d_r,
                                                                bf16* out, int32_t* out_table, uint32_t* status) {
  constexpr int kB = 64;
  const int k = blockIdx.x, b = blockIdx.y;
  const int d = b * max_blocks + k;
  if (threadIdx.x == 0) out_table[d] = d;
  int L = kv_len[b];
  if (L < 0 || L > max_blocks * kB) L = L < 0 ? 0 : max_blocks * kB;   // the attention kernel flags it
  if (k * kB >= L) return;
  const int blk = table[(long long)b * max_blocks + k];
  const bool ok = blk >= 0 && blk < num_blocks;
  if (!ok && threadIdx.x == 0) flag_error(status, kFlagIndex);
  const long long bbytes = (long long)kB * (d_c + 2 * d_r + 4);
  expand_block(ok ? pool + blk * bbytes : nullptr, out + (long long)d * (d_c + d_r) * kB, d_c, d_r);
}

// Block (k, chunk): rows of logical block k of sequence seq, 64-element chunk `chunk`, into
// lat[chunk][pos][64] for pos < L (bf16).
__global__ void __launch_bounds__(256) gather_latent_fp8_kernel(const uint8_t* pool, const int32_t* table,
                                                                int max_blocks, int num_blocks, int seq, int L,
                                                                int d_c, int d_r, bf16* lat, uint32_t* status) {
  constexpr int kB = 64;
  __shared__ float sc[kB];
  __shared__ uint16_t tile[64][65];
  const int bt = blockIdx.x, chunk = blockIdx.y;
  int blk = bt < max_blocks ? table[(long long)seq * max_blocks + bt] : -1;
  if (blk < 0 || blk >= num_blocks) {
    if (threadIdx.x == 0 && chunk == 0) flag_error(status, kFlagIndex);
    blk = -1;
  }
  const long long bbytes = (long long)kB * (d_c + 2 * d_r + 4);
  const uint8_t* src = blk >= 0 ? pool + blk * bbytes : nullptr;
  if (threadIdx.x < kB) sc[threadIdx.x] = src ? reinterpret_cast<const float*>(src + (d_c + 2 * d_r) * kB)[threadIdx.x] : 0.f;
  __syncthreads();
  for (int i = threadIdx.x; i < 64 * 64; i += blockDim.x) {
    const int e = i >> 6, t = i & 63, el = chunk * 64 + e;
    float v = 0.f;
    if (src) {
      if (el < d_c) {
        const uint8_t c = src[(long long)el * kB + t];
        v = from_e4m3x2((uint16_t)c).x;
      } else {
        v = __bfloat162float(reinterpret_cast<const bf16*>(src + (long long)d_c * kB)[(long long)(el - d_c) * kB + t]);
      }
      v *= sc[t];
    }
    const bf16 h = __float2bfloat16_rn(v);
    tile[e][t] = *reinterpret_cast<const uint16_t*>(&h);
  }
  __syncthreads();
  uint16_t* dst = reinterpret_cast<uint16_t*>(lat);
  for (int i = threadIdx.x; i < 64 * 64; i += blockDim.x) {
    const int t = i >> 6, e = i & 63;
    const int p = bt * kB + t;
    if (p < L) dst[((long long)chunk * L + p) * 64 + e] = tile[e][t];
  }
}

}  // namespace

cudaError_t launch_compress_reduce_fp8(const Ctx& ctx, const float* part, int splits, int T, int d_c, int d_r,
                                       const int32_t* seq_idx, const int32_t* pos, const mla_rope_table& rope,
                                       const mla_paged_cache& cache, int block_size) {
  if (d_c % 64 || d_c > 64 * kMaxLatPerLane / 2 || d_r > 64 || d_r % 2) return cudaErrorInvalidValue;
  compress_reduce_fp8_kernel<<<(T + kFp8Tok - 1) / kFp8Tok, 256, 0, ctx.stream>>>(
      part, splits, T, d_c, d_r, seq_idx, pos, rope.cos_sin, rope.max_pos, static_cast<uint8_t*>(cache.pool),
      cache.num_blocks, cache.block_table, cache.max_blocks_per_seq, cache.batch, block_size, ctx.status);
  count_launch();
  return cudaGetLastError();
}

size_t fp8_expand_bytes(const mla_config* cfg, int batch, int max_blocks) {
  const size_t blocks = (size_t)batch * max_blocks;
  const size_t pool = blocks * (cfg->d_c + cfg->d_rope) * cfg->block_size * 2;
  return (pool + 255) / 256 * 256 + (blocks * 4 + 255) / 256 * 256;
}

cudaError_t launch_expand_fp8(const Ctx& ctx, const mla_config* cfg, const mla_paged_cache& cache,
                              const int32_t* kv_len, int batch, void* scratch, mla_paged_cache* expanded) {
  if (cfg->block_size != 64) return cudaErrorInvalidValue;
  const size_t blocks = (size_t)batch * cache.max_blocks_per_seq;
  const size_t pool = (blocks * (cfg->d_c + cfg->d_rope) * 64 * 2 + 255) / 256 * 256;
  bf16* out = static_cast<bf16*>(scratch);
  int32_t* out_table = reinterpret_cast<int32_t*>(static_cast<char*>(scratch) + pool);
  expand_fp8_blocks_kernel<<<dim3(cache.max_blocks_per_seq, batch), 256, 0, ctx.stream>>>(
      static_cast<const uint8_t*>(cache.pool), cache.num_blocks, cache.block_table, cache.max_blocks_per_seq, kv_len,
      cfg->d_c, cfg->d_rope, out, out_table, ctx.status);
  count_launch();
  expanded->pool = out;
  expanded->num_blocks = (int)blocks;
  expanded->block_table = out_table;
  expanded->max_blocks_per_seq = cache.max_blocks_per_seq;
  expanded->batch = batch;
  return cudaGetLastError();
}

cudaError_t launch_gather_latent_fp8(const Ctx& ctx, const mla_config* cfg, const mla_paged_cache& cache, int seq,
                                     int L, void* lat) {
  if (cfg->block_size != 64 || (cfg->d_c + cfg->d_rope) % 64) return cudaErrorInvalidValue;
  const dim3 grid((L + 63) / 64, (cfg->d_c + cfg->d_rope) / 64);
  gather_latent_fp8_kernel<<<grid, 256, 0, ctx.stream>>>(static_cast<const uint8_t*>(cache.pool), cache.block_table,
                                                         cache.max_blocks_per_seq, cache.num_blocks, seq, L, cfg->d_c,
                                                         cfg->d_rope, static_cast<bf16*>(lat), ctx.status);
  count_launch();
  return cudaGetLastError();
}

}  // namespace mla
