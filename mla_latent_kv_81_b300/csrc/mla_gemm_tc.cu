// Projection GEMMs on tcgen05 tensor cores, and the bf16 projection paths built on them.
//
// One persistent kernel computes, for a batch of G independent problems,
//   D[g][n][m] = sum_k A[g][m][k] * B[g][n][k]
// with A the weights (M = output features, streamed once) and B the
// activations (N = tokens, re-read from L2).  The weights are the M = 128 rows
// of each MMA, so the narrow token count of decode (N = 16..256) costs no
// padding of M.  A may be stored K-major ([M][K], as W) or M-major ([K][M], as
// the transposed key up-projection).  Work units are (g, m-tile, n-tile,
// k-split); a split writes fp32 partials that a small kernel sums, and an
// unsplit unit may store bf16 directly.
//
// The decode-step projections ("What does Multi-head Latent Attention
// compress...", "Why it is not just extra work at decode time": query
// projection, key up-projection folded into the query, value up-projection
// and output projection applied after the weighted sum; "The mechanism":
// down-projection of each token into the latent) are chains of such GEMMs
// plus elementwise epilogues (RoPE, bf16 rounding, paged-cache scatter).
#include <math.h>

#include <mutex>

#include "mla_sm100.cuh"
#include "mla_tc.cuh"

namespace mla {
namespace {
using namespace sm100;

constexpr int kGThreads = 256;       // warp 0 TMA, warp 1 MMA, warp 2 TMEM, warps 4-7 epilogue
constexpr int kGRingBytes = 196608;  // 192 KB of A/B stages
constexpr int kGCtrl = 1024;
constexpr int kGSmem = kGCtrl + kGRingBytes + 1024;
constexpr int kGMaxStages = 12;
constexpr int kATileBytes = 128 * 64 * 2;   // [128 rows x 64 k] bf16

struct GemmArgs {
  int M, N, K, G;
  int m_tiles, n_tiles, splits, kb;   // kb = K / 64
  int n_tile;                         // tokens per tile (multiple of 16, <= 256)
  int a_mn;                           // A stored [K][M] (M contiguous)
  int a_k_period;                     // > 0: A's k coordinate wraps every a_k_period (B = [hi || lo] split)
  int m_tiles1;                       // m-tiles taken from the first A map; later ones from the second
  int units;                          // G * m_tiles * n_tiles * splits
  int stages, stage_bytes;
  float* partial;                     // [splits][G][N][M] fp32, or null
  bf16* out;                          // direct bf16 output when partial == null
  long long out_ld, out_g;            // out[g * out_g + n * out_ld + m]
  long long out_mc;                   // > 0: out stored chunk-major, out[(m / 64) * out_mc + n * 64 + m % 64]
  int b_kchunk;                       // B stored chunk-major [K / 64][N][64] (one contiguous box per k-block)
  uint32_t* status;
};

struct GCtrl {
  uint64_t full[kGMaxStages], empty[kGMaxStages];
  uint64_t acc_full[2], acc_empty[2];
  uint32_t tmem_base;
  int abort_flag;
};

__device__ __forceinline__ void unit_coords(const GemmArgs& a, int u, int& g, int& mt, int& nt, int& sp) {
  sp = u % a.splits;
  u /= a.splits;
  nt = u % a.n_tiles;
  u /= a.n_tiles;
  mt = u % a.m_tiles;
  g = u / a.m_tiles;
}

__device__ __forceinline__ void split_range(const GemmArgs& a, int sp, int& k0, int& k1) {
  k0 = (int)((long long)sp * a.kb / a.splits);
  k1 = (int)((long long)(sp + 1) * a.kb / a.splits);
}

// AMN: A stored [K][M] (M contiguous).  A template parameter so that every MMA operand offset between
// the MMAs of a k-block is a compile-time constant (runtime arithmetic there stalls their issue).
template <bool AMN>
__global__ void __launch_bounds__(kGThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap a_map, const __grid_constant__ CUtensorMap a_map2,
                   const __grid_constant__ CUtensorMap b_map, GemmArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  GCtrl* ctrl = reinterpret_cast<GCtrl*>(smem);
  uint8_t* ring = smem + kGCtrl;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  volatile int* abort_flag = &ctrl->abort_flag;
  pdl_trigger();

  if (tid == 0) {
    for (int i = 0; i < a.stages; ++i) { mbar_init(&ctrl->full[i], 1); mbar_init(&ctrl->empty[i], 1); }
    for (int i = 0; i < 2; ++i) { mbar_init(&ctrl->acc_full[i], 1); mbar_init(&ctrl->acc_empty[i], 128); }
    ctrl->abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 2) {
    tmem_alloc(&ctrl->tmem_base, 512);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&a_map);
    if (a.m_tiles1 < a.m_tiles) prefetch_tmap(&a_map2);
    prefetch_tmap(&b_map);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  pdl_wait();
  const uint32_t tmem = ctrl->tmem_base;
  const uint32_t ring_base = smem_u32(ring);
  const uint32_t b_bytes = (uint32_t)a.n_tile * 128;

  if (warp == 0) {
    if (lane == 0) {
      // producer: A tile [128 x 64] and B tile [n_tile x 64] per k-block
      int st = 0;
      uint32_t ph = 0;
      for (int u = blockIdx.x; u < a.units; u += gridDim.x) {
        int g, mt, nt, sp, k0, k1;
        unit_coords(a, u, g, mt, nt, sp);
        split_range(a, sp, k0, k1);
        for (int kb = k0; kb < k1; ++kb) {
          if (!mbar_wait(&ctrl->empty[st], ph ^ 1, a.status, abort_flag)) goto done;
          uint8_t* sa = ring + st * a.stage_bytes;
          uint8_t* sb = sa + kATileBytes;
          mbar_arrive_expect_tx(&ctrl->full[st], kATileBytes + b_bytes);
          const int ka = a.a_k_period > 0 ? (kb * 64) % a.a_k_period : kb * 64;
          const bool second = mt >= a.m_tiles1;
          const CUtensorMap* am = second ? &a_map2 : &a_map;
          const int ma = (second ? mt - a.m_tiles1 : mt) * 128;
          if (AMN) {
            // A^T stored [K][M]: two [64 k x 64 m] boxes cover the 128 rows of the tile
            tma_load_3d(sa, am, &ctrl->full[st], ma, ka, g);
            tma_load_3d(sa + kATileBytes / 2, am, &ctrl->full[st], ma + 64, ka, g);
          } else {
            tma_load_3d(sa, am, &ctrl->full[st], ka, ma, g);
          }
          if (a.b_kchunk)
            tma_load_3d(sb, &b_map, &ctrl->full[st], 0, nt * a.n_tile, kb);
          else
            tma_load_3d(sb, &b_map, &ctrl->full[st], kb * 64, nt * a.n_tile, g);
          if (++st == a.stages) { st = 0; ph ^= 1; }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16(128, a.n_tile, AMN, false);
      const uint64_t ring_a = AMN ? desc_sw128(ring_base, kATileBytes / 2, 1024) : desc_sw128(ring_base, 16, 1024);
      const uint64_t ring_b = desc_sw128(ring_base + kATileBytes, 16, 1024);
      const uint64_t stage_step = (uint64_t)(a.stage_bytes >> 4);
      int st = 0, acc = 0;
      uint32_t ph = 0, acc_ph = 0;
      for (int u = blockIdx.x; u < a.units; u += gridDim.x) {
        int g, mt, nt, sp, k0, k1;
        unit_coords(a, u, g, mt, nt, sp);
        split_range(a, sp, k0, k1);
        if (!mbar_wait(&ctrl->acc_empty[acc], acc_ph ^ 1, a.status, abort_flag)) goto done;
        tc_fence_after();
        const uint32_t d = tmem + acc * 256;
        uint32_t first = 0;   // 0: the unit's first k-block overwrites the accumulator
        for (int kb = k0; kb < k1; ++kb) {
          if (!mbar_wait(&ctrl->full[st], ph, a.status, abort_flag)) goto done;
          tc_fence_after();
          const uint64_t ad = ring_a + st * stage_step, bd = ring_b + st * stage_step;
          // K-major operands step 32 B along the swizzled row; an M-major A steps 16 rows of 128 B
          constexpr uint64_t kAStep = AMN ? (2048 >> 4) : 2;
          mma_ss(d, ad, bd, idesc, first);
          mma_ss(d, ad + kAStep, bd + 2, idesc, 1u);
          mma_ss(d, ad + 2 * kAStep, bd + 4, idesc, 1u);
          mma_ss(d, ad + 3 * kAStep, bd + 6, idesc, 1u);
          first = 1;
          mma_commit(&ctrl->empty[st]);
          if (++st == a.stages) { st = 0; ph ^= 1; }
        }
        mma_commit(&ctrl->acc_full[acc]);
        if (++acc == 2) { acc = 0; acc_ph ^= 1; }
      }
    }
  } else if (warp >= 4) {
    // epilogue: thread owns accumulator row m (TMEM lane), writes token columns
    const int q4 = warp & 3;
    const int row = q4 * 32 + lane;
    const uint32_t lane_base = tmem + ((uint32_t)(q4 * 32) << 16);
    int acc = 0;
    uint32_t acc_ph = 0;
    for (int u = blockIdx.x; u < a.units; u += gridDim.x) {
      int g, mt, nt, sp;
      unit_coords(a, u, g, mt, nt, sp);
      const bool ok = mbar_wait(&ctrl->acc_full[acc], acc_ph, a.status, abort_flag);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();
      const int m = mt * 128 + row;
      const int n0 = nt * a.n_tile;
      for (int c = 0; c < a.n_tile; c += 32) {
        uint32_t r[32];
        tmem_ld32(lane_base + acc * 256 + c, r);
        tmem_ld_wait();
        if (m < a.M) {
          if (a.partial) {
            float* dst = a.partial + (((long long)sp * a.G + g) * a.N) * a.M + m;
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const int n = n0 + c + i;
              if (n < a.N) dst[(long long)n * a.M] = __uint_as_float(r[i]);
            }
          } else {
            const long long ld = a.out_mc ? 64 : a.out_ld;
            bf16* dst = a.out + (a.out_mc ? (long long)(m >> 6) * a.out_mc + (m & 63) : (long long)g * a.out_g + m);
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const int n = n0 + c + i;
              if (n < a.N) dst[(long long)n * ld] = __float2bfloat16_rn(__uint_as_float(r[i]));
            }
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&ctrl->acc_empty[acc]);
      if (++acc == 2) { acc = 0; acc_ph ^= 1; }
    }
  }
done:
  tc_fence_before();
  __syncthreads();
  if (*abort_flag && warp == 0 && lane == 0) {
    const long long t0 = clock64();
    while (clock64() - t0 < 2000000LL) { }
  }
  tc_fence_after();
  if (warp == 2) tmem_dealloc(tmem, 512);
}

// ------------------------------------------------------------------ elementwise epilogues
// Rotate the pair (a, b) by the tabulated angle: (a cos - b sin, a sin + b cos).
__device__ __forceinline__ void rope2(float a, float b, const float* cs, float& o0, float& o1) {
  o0 = a * cs[0] - b * cs[1];
  o1 = a * cs[1] + b * cs[0];
}

__device__ __forceinline__ float4 sum_splits4(const float* part, int splits, long long split_stride, long long idx) {
  float4 v = *reinterpret_cast<const float4*>(part + idx);
  for (int s = 1; s < splits; ++s) {
    const float4 w = *reinterpret_cast<const float4*>(part + s * split_stride + idx);
    v.x += w.x; v.y += w.y; v.z += w.z; v.w += w.w;
  }
  return v;
}

// From the k-split partials [splits][N][H*qk + H*d_r] of the fused W_Q / W_QR GEMM:
// q_nope as two bf16 parts ([n][h][hi(qk) || lo(qk)]) and the rotated query part of q_out.
// One thread per 4 consecutive columns.
__global__ void absorb_reduce_kernel(const float* part, int splits, int N, int H, int qk, int d_r, int d_c,
                                     const int32_t* q_pos, const float* rope, int rope_max, bf16* q_nope,
                                     bf16* q_out, uint32_t* status) {
  pdl_trigger();
  pdl_wait();
  const int Mt = H * (qk + d_r);
  const long long total4 = (long long)N * Mt / 4, stride = (long long)N * Mt;
  for (long long e4 = blockIdx.x * (long long)blockDim.x + threadIdx.x; e4 < total4;
       e4 += (long long)gridDim.x * blockDim.x) {
    const long long e = e4 * 4;
    const int n = (int)(e / Mt), col = (int)(e % Mt);
    const float4 v = sum_splits4(part, splits, stride, e);
    if (col < H * qk) {
      const int h = col / qk, i = col % qk;
      bf16* hi = q_nope + ((long long)n * H + h) * 2 * qk + i;
      const float vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const bf16 a = __float2bfloat16_rn(vv[j]);
        hi[j] = a;
        hi[qk + j] = __float2bfloat16_rn(vv[j] - __bfloat162float(a));
      }
    } else {
      const int c = col - H * qk, h = c / d_r, r = c % d_r;   // r even: two rotated pairs
      const int p = q_pos[n];
      if (p < 0 || p >= rope_max) {
        flag_error(status, kFlagIndex);
        continue;
      }
      const float* cs = rope + ((long long)p * (d_r / 2) + r / 2) * 2;
      float o0, o1, o2, o3;
      rope2(v.x, v.y, cs, o0, o1);
      rope2(v.z, v.w, cs + 2, o2, o3);
      __nv_bfloat162* dst =
          reinterpret_cast<__nv_bfloat162*>(q_out + ((long long)n * H + h) * (d_c + d_r) + d_c + r);
      dst[0] = __floats2bfloat162_rn(o0, o1);
      dst[1] = __floats2bfloat162_rn(o2, o3);
    }
  }
}

// The explicit-form query from the same partials: q_out[n][h] = [q_nope^h (bf16) || RoPE(q_R^h) (bf16)].
// One thread per 4 consecutive columns.
__global__ void query_reduce_kernel(const float* part, int splits, int N, int H, int qk, int d_r, const int32_t* q_pos,
                                    const float* rope, int rope_max, bf16* q_out, uint32_t* status) {
  pdl_trigger();
  pdl_wait();
  const int Mt = H * (qk + d_r);
  const long long total4 = (long long)N * Mt / 4, stride = (long long)N * Mt;
  for (long long e4 = blockIdx.x * (long long)blockDim.x + threadIdx.x; e4 < total4;
       e4 += (long long)gridDim.x * blockDim.x) {
    const long long e = e4 * 4;
    const int n = (int)(e / Mt), col = (int)(e % Mt);
    const float4 v = sum_splits4(part, splits, stride, e);
    __nv_bfloat162* dst;
    float o0 = v.x, o1 = v.y, o2 = v.z, o3 = v.w;
    if (col < H * qk) {
      const int h = col / qk, i = col % qk;
      dst = reinterpret_cast<__nv_bfloat162*>(q_out + ((long long)n * H + h) * (qk + d_r) + i);
    } else {
      const int c = col - H * qk, h = c / d_r, r = c % d_r;   // r even: two rotated pairs
      const int p = q_pos[n];
      if (p < 0 || p >= rope_max) {
        flag_error(status, kFlagIndex);
        continue;
      }
      const float* cs = rope + ((long long)p * (d_r / 2) + r / 2) * 2;
      rope2(v.x, v.y, cs, o0, o1);
      rope2(v.z, v.w, cs + 2, o2, o3);
      dst = reinterpret_cast<__nv_bfloat162*>(q_out + ((long long)n * H + h) * (qk + d_r) + qk + r);
    }
    dst[0] = __floats2bfloat162_rn(o0, o1);
    dst[1] = __floats2bfloat162_rn(o2, o3);
  }
}

// Cache rows [c || RoPE(k_R)] from the k-split partials [splits][T][d_c + d_r] of the fused
// W_DKV / W_KR GEMM, scattered into the paged pool, which stores each block transposed
// ([d_c + d_r][block_size]).  Block (8-token group, 64-column group), warp w = token t0 + w: the partials
// are read token by token (coalesced, all splits in flight at once), summed, rotated and rounded, then
// transposed through shared memory so that tokens at consecutive positions of one block write
// contiguous bytes of each element row.
constexpr int kAppTok = 8, kAppCols = 64;

__global__ void __launch_bounds__(256) compress_reduce_kernel(const float* part, int splits, int T, int d_c, int d_r,
                                                              int d_rh,
                                                              const int32_t* seq_idx, const int32_t* pos,
                                                              const float* rope, int rope_max, bf16* pool,
                                                              int num_blocks, const int32_t* table, int max_blocks,
                                                              int batch, int block_size, uint32_t* status) {
  __shared__ bf16 tile[kAppCols][kAppTok];
  __shared__ long long dst_base[kAppTok];   // pool offset of column 0 of each token, or -1 (skipped)
  pdl_trigger();
  pdl_wait();
  const int t0 = blockIdx.x * kAppTok, c0 = blockIdx.y * kAppCols;
  const int width = d_c + d_r;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = t0 + warp;
  // lane l holds columns c0 + 2l and c0 + 2l + 1 of token t (a RoPE pair when in the k_R part)
  const int col = c0 + 2 * lane;
  int p_t = 0;
  long long base = -1;
  if (t < T) {
    const int b = seq_idx[t];
    p_t = pos[t];
    int blk = -1;
    if (b >= 0 && b < batch && p_t >= 0 && p_t < rope_max)
      blk = cache_block(table, max_blocks, num_blocks, block_size, b, p_t);
    if (blk < 0) {
      if (blockIdx.y == 0 && lane == 0) flag_error(status, kFlagIndex);
    } else {
      base = (long long)blk * width * block_size + p_t % block_size;
    }
  }
  if (lane == 0) dst_base[warp] = base;
  if (base >= 0 && col < width) {
    const long long idx = (long long)t * width + col, sstride = (long long)T * width;
    float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
    int sp = 0;
    for (; sp + 4 <= splits; sp += 4) {
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const float2 w = *reinterpret_cast<const float2*>(part + (sp + u) * sstride + idx);
        acc[u].x += w.x;
        acc[u].y += w.y;
      }
    }
    for (; sp < splits; ++sp) {
      const float2 w = *reinterpret_cast<const float2*>(part + sp * sstride + idx);
      acc[0].x += w.x;
      acc[0].y += w.y;
    }
    float2 v = make_float2((acc[0].x + acc[1].x) + (acc[2].x + acc[3].x), (acc[0].y + acc[1].y) + (acc[2].y + acc[3].y));
    if (col >= d_c) {
      // rotation frequencies restart in every head's key when the keys are per head (d_rh < d_r)
      const float* cs = rope + ((long long)p_t * (d_rh / 2) + ((col - d_c) % d_rh) / 2) * 2;
      float o0, o1;
      rope2(v.x, v.y, cs, o0, o1);
      v = make_float2(o0, o1);
    }
    tile[2 * lane][warp] = __float2bfloat16_rn(v.x);
    tile[2 * lane + 1][warp] = __float2bfloat16_rn(v.y);
  }
  __syncthreads();
  // thread (r, j): element row c0 + r of token t0 + j
#pragma unroll
  for (int k = 0; k < kAppCols * kAppTok / 256; ++k) {
    const int e = threadIdx.x + k * 256, r = e / kAppTok, j = e % kAppTok;
    const long long bj = dst_base[j];
    if (t0 + j < T && bj >= 0 && c0 + r < width) pool[bj + (long long)(c0 + r) * block_size] = tile[r][j];
  }
}

// bf16 output from k-split partials ([splits][count]), 4 elements per thread.
__global__ void sum_to_bf16_kernel(const float* part, int splits, long long count, bf16* out) {
  pdl_trigger();
  pdl_wait();
  for (long long e4 = blockIdx.x * (long long)blockDim.x + threadIdx.x; e4 < count / 4;
       e4 += (long long)gridDim.x * blockDim.x) {
    const float4 v = sum_splits4(part, splits, count, e4 * 4);
    __nv_bfloat162* dst = reinterpret_cast<__nv_bfloat162*>(out + e4 * 4);
    dst[0] = __floats2bfloat162_rn(v.x, v.y);
    dst[1] = __floats2bfloat162_rn(v.z, v.w);
  }
}

// ------------------------------------------------------------------ host planning
using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                              const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                              CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
std::mutex g_gmutex;
EncodeFn g_genc = nullptr;

EncodeFn encoder() {
  std::lock_guard<std::mutex> lock(g_gmutex);
  if (!g_genc) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    g_genc = reinterpret_cast<EncodeFn>(fn);
  }
  return g_genc;
}

// 3-D bf16 tensor map: dims {inner, d1, d2}, byte strides of d1 and d2, box {64, box1, 1}, 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t d1, uint64_t d2, uint64_t s1, uint64_t s2,
              uint32_t box1) {
  EncodeFn enc = encoder();
  if (!enc) return false;
  const cuuint64_t dims[3] = {inner, d1, d2};
  const cuuint64_t strides[2] = {s1, s2};
  const cuuint32_t box[3] = {64, box1, 1}, es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

// bf16 tensor map of any rank with the 128-byte swizzle (declared in mla_tc.cuh).
bool encode_map_bf16(CUtensorMap* m, const void* base, int rank, const uint64_t* dims, const uint64_t* strides,
                     const uint32_t* box) {
  EncodeFn enc = encoder();
  if (!enc || rank < 1 || rank > 5) return false;
  cuuint64_t d[5], st[4];
  cuuint32_t b[5], es[5];
  for (int i = 0; i < rank; ++i) { d[i] = dims[i]; b[i] = box[i]; es[i] = 1; }
  for (int i = 0; i + 1 < rank; ++i) st[i] = strides[i];
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (cuuint32_t)rank, const_cast<void*>(base), d, st, b, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

namespace {

struct GemmPlan {
  GemmArgs args;
  int grid;
};

// Tile and split a problem so that the SMs are covered about four units deep
// (direct = no k-split: the GEMM stores bf16 itself).
constexpr int kMinKbPerSplit = 8;   // 512 of K: 128 KB of a 128-row bf16 weight tile per split

GemmPlan plan_gemm(int M, int N, int K, int G, bool a_mn, bool direct, int sm_count) {
  GemmPlan p{};
  GemmArgs& a = p.args;
  a.M = M; a.N = N; a.K = K; a.G = G;
  a.a_mn = a_mn ? 1 : 0;
  a.n_tile = N >= 256 ? 256 : ((N + 15) / 16) * 16;
  if (a.n_tile < 16) a.n_tile = 16;
  a.m_tiles = (M + 127) / 128;
  a.n_tiles = (N + a.n_tile - 1) / a.n_tile;
  a.m_tiles1 = a.m_tiles;
  a.kb = K / 64;
  const long long base = (long long)G * a.m_tiles * a.n_tiles;
  // the fewest k-splits whose units fill the waves of SMs at least 90%, but no split shallower than
  // kMinKbPerSplit k-blocks: a thinner split costs more in fp32 partials and their reduction than its
  // extra parallelism saves on a small weight
  int splits = 1;
  if (!direct) {
    double best = 0.0;
    const int max_splits = a.kb / kMinKbPerSplit > 1 ? a.kb / kMinKbPerSplit : 1;
    for (int s = 1; s <= max_splits && s <= 64; ++s) {
      const long long u = base * s;
      const double eff = (double)u / ((double)sm_count * ((u + sm_count - 1) / sm_count));
      if (eff > best + 1e-9) { best = eff; splits = s; }
      if (eff >= 0.9) break;
    }
  }
  a.splits = splits;
  a.units = (int)(base * splits);
  a.stage_bytes = kATileBytes + a.n_tile * 128;
  a.stages = kGRingBytes / a.stage_bytes;
  if (a.stages > kGMaxStages) a.stages = kGMaxStages;
  p.grid = a.units < sm_count ? a.units : sm_count;
  return p;
}

size_t partial_bytes(const GemmPlan& p) {
  return (size_t)p.args.splits * p.args.G * p.args.N * p.args.M * sizeof(float);
}

cudaError_t launch_gemm(const Ctx& ctx, const CUtensorMap& am, const CUtensorMap& am2, const CUtensorMap& bm,
                        GemmPlan& p) {
  p.args.status = ctx.status;
  const void* kern = p.args.a_mn ? (const void*)gemm_tc_kernel<true> : (const void*)gemm_tc_kernel<false>;
  cudaError_t e = ensure_smem_limit(kern, kGSmem, ctx.device);
  if (e != cudaSuccess) return e;
  if (p.args.units == 0) return cudaSuccess;
  e = cudaSuccess;
  if (p.args.a_mn)
    e = launch_pdl(gemm_tc_kernel<true>, dim3(p.grid), dim3(kGThreads), kGSmem, ctx.stream, am, am2, bm, p.args);
  else
    e = launch_pdl(gemm_tc_kernel<false>, dim3(p.grid), dim3(kGThreads), kGSmem, ctx.stream, am, am2, bm, p.args);
  count_launch();
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

size_t align256(size_t v) { return (v + 255) / 256 * 256; }

bool shapes_ok(const mla_config* cfg) {
  return cfg->dtype == MLA_BF16 && cfg->d_model % 64 == 0 && cfg->qk_nope % 64 == 0 && cfg->d_c % 128 == 0 &&
         cfg->d_c % 64 == 0 && cfg->d_rope % 2 == 0 && (cfg->n_heads * cfg->v_head) % 64 == 0 &&
         cfg->d_rope <= 128 && cfg->v_head % 16 == 0;
}

}  // namespace

// ------------------------------------------------------------------ compress_append
namespace {
// Plan for [W_A; W_B] x over tokens: the m-tiles of W_A (M_a a multiple of 128) then those of W_B.
GemmPlan plan_stacked(int M_a, int M_b, int N, int K, int sm_count) {
  GemmPlan p = plan_gemm(M_a + M_b, N, K, 1, false, false, sm_count);
  p.args.m_tiles1 = M_a / 128;
  return p;
}
bool stack_ok(int M_a) { return M_a % 128 == 0; }
int launch_blocks(long long work, int threads, int sm_count) {
  long long b = (work + threads - 1) / threads;
  if (b > 8LL * sm_count) b = 8LL * sm_count;
  return b < 1 ? 1 : (int)b;
}
}  // namespace

bool tc_compress_supported(const mla_config* cfg, int T) {
  return shapes_ok(cfg) && T > 0 && stack_ok(cfg->d_c) && (cfg->d_c + cfg->d_rope) % 4 == 0;
}

size_t tc_compress_workspace_bytes(const mla_config* cfg, int T, int sm_count) {
  if (!tc_compress_supported(cfg, T)) return 0;
  const int d_r = cfg->rope_per_head ? cfg->n_heads * cfg->d_rope : cfg->d_rope;
  return align256(partial_bytes(plan_stacked(cfg->d_c, d_r, T, cfg->d_model, sm_count)));
}

cudaError_t tc_compress_append(const Ctx& ctx, const mla_config* cfg, const void* x, const void* W_DKV,
                               const void* W_KR, const int32_t* seq_idx, const int32_t* pos,
                               const mla_rope_table& rope, const mla_paged_cache& cache, int T, void* workspace) {
  const int D = cfg->d_model, d_c = cfg->d_c, d_rh = cfg->d_rope;
  const int d_r = cfg->rope_per_head ? cfg->n_heads * d_rh : d_rh;   // positional columns of a row
  GemmPlan pl = plan_stacked(d_c, d_r, T, D, ctx.sm_count);
  pl.args.partial = static_cast<float*>(workspace);
  CUtensorMap a1, a2, b;
  if (!make_map(&a1, W_DKV, D, d_c, 1, (uint64_t)D * 2, (uint64_t)D * 2 * d_c, 128) ||
      !make_map(&a2, W_KR, D, d_r, 1, (uint64_t)D * 2, (uint64_t)D * 2 * d_r, 128) ||
      !make_map(&b, x, D, T, 1, (uint64_t)D * 2, (uint64_t)D * 2 * T, pl.args.n_tile))
    return cudaErrorInvalidValue;
  cudaError_t e = launch_gemm(ctx, a1, a2, b, pl);
  if (e != cudaSuccess) return e;
  if (cfg->cache_fp8)
    return launch_compress_reduce_fp8(ctx, pl.args.partial, pl.args.splits, T, d_c, d_r, seq_idx, pos, rope, cache,
                                      cfg->block_size);
  const int width = d_c + d_r;
  dim3 grid((T + kAppTok - 1) / kAppTok, (width + kAppCols - 1) / kAppCols);
  e = launch_pdl(compress_reduce_kernel, grid, dim3(256), 0, ctx.stream, pl.args.partial, pl.args.splits, T, d_c, d_r,
                 d_rh, seq_idx, pos, rope.cos_sin, rope.max_pos, (bf16*)cache.pool, cache.num_blocks, cache.block_table,
                 cache.max_blocks_per_seq, cache.batch, cfg->block_size, ctx.status);
  count_launch();
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// ------------------------------------------------------------------ absorb_query
bool tc_absorb_supported(const mla_config* cfg, int N) {
  return shapes_ok(cfg) && N > 0 && stack_ok(cfg->n_heads * cfg->qk_nope) && cfg->d_rope % 4 == 0;
}

namespace {
struct AbsorbLayout {
  GemmPlan pqr, pa;
  size_t off_nope, total;
};
AbsorbLayout absorb_layout(const mla_config* cfg, int N, int sm_count) {
  AbsorbLayout l;
  const int H = cfg->n_heads;
  l.pqr = plan_stacked(H * cfg->qk_nope, H * cfg->d_rope, N, cfg->d_model, sm_count);
  // K = 2 * qk_nope: the same W_UK^T tile multiplies the high and low bf16 parts of q_nope
  l.pa = plan_gemm(cfg->d_c, N, 2 * cfg->qk_nope, H, true, true, sm_count);
  l.pa.args.a_k_period = cfg->qk_nope;
  l.off_nope = align256(partial_bytes(l.pqr));
  l.total = l.off_nope + align256((size_t)N * H * cfg->qk_nope * 2 * 2);
  return l;
}
}  // namespace

size_t tc_absorb_workspace_bytes(const mla_config* cfg, int N, int sm_count) {
  if (!tc_absorb_supported(cfg, N)) return 0;
  return absorb_layout(cfg, N, sm_count).total;
}

cudaError_t tc_absorb_query(const Ctx& ctx, const mla_config* cfg, const void* x, const void* W_Q, const void* W_QR,
                            const void* W_UK, const int32_t* q_pos, const mla_rope_table& rope, void* q_out, int N,
                            void* workspace) {
  const int D = cfg->d_model, H = cfg->n_heads, qk = cfg->qk_nope, d_r = cfg->d_rope, d_c = cfg->d_c;
  AbsorbLayout l = absorb_layout(cfg, N, ctx.sm_count);
  char* ws = static_cast<char*>(workspace);
  l.pqr.args.partial = reinterpret_cast<float*>(ws);
  bf16* q_nope = reinterpret_cast<bf16*>(ws + l.off_nope);
  CUtensorMap aq, ar, bx, auk, bn;
  if (!make_map(&aq, W_Q, D, (uint64_t)H * qk, 1, (uint64_t)D * 2, (uint64_t)D * 2 * H * qk, 128) ||
      !make_map(&ar, W_QR, D, (uint64_t)H * d_r, 1, (uint64_t)D * 2, (uint64_t)D * 2 * H * d_r, 128) ||
      !make_map(&bx, x, D, N, 1, (uint64_t)D * 2, (uint64_t)D * 2 * N, l.pqr.args.n_tile) ||
      // W_UK^h^T: stored [h][i][c] (c contiguous) = an M-major A with M = d_c, K = qk_nope
      !make_map(&auk, W_UK, d_c, qk, H, (uint64_t)d_c * 2, (uint64_t)d_c * 2 * qk, 64) ||
      // q_nope^h: [n][h][hi || lo], rows n with stride H * 2 * qk
      !make_map(&bn, q_nope, 2 * qk, N, H, (uint64_t)H * 2 * qk * 2, (uint64_t)2 * qk * 2, l.pa.args.n_tile))
    return cudaErrorInvalidValue;
  cudaError_t e = launch_gemm(ctx, aq, ar, bx, l.pqr);
  if (e != cudaSuccess) return e;
  const long long work = (long long)N * H * (qk + d_r) / 4;
  e = launch_pdl(absorb_reduce_kernel, dim3(launch_blocks(work, 256, ctx.sm_count)), dim3(256), 0, ctx.stream,
                 l.pqr.args.partial, l.pqr.args.splits, N, H, qk, d_r, d_c, q_pos, rope.cos_sin, rope.max_pos, q_nope,
                 (bf16*)q_out, ctx.status);
  count_launch();
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // q_abs^h = W_UK^h^T q_nope^h, written straight into q_out[n][h][0:d_c]
  l.pa.args.partial = nullptr;
  l.pa.args.out = static_cast<bf16*>(q_out);
  l.pa.args.out_ld = (long long)H * (d_c + d_r);
  l.pa.args.out_g = d_c + d_r;
  return launch_gemm(ctx, auk, auk, bn, l.pa);
}

// ------------------------------------------------------------------ output_project
bool tc_output_supported(const mla_config* cfg, int N) { return shapes_ok(cfg) && N > 0 && cfg->d_model % 4 == 0; }

namespace {
struct OutputLayout {
  GemmPlan pv, po;
  size_t off_o, off_part, total;
};
OutputLayout output_layout(const mla_config* cfg, int N, int sm_count) {
  OutputLayout l;
  const int H = cfg->n_heads;
  l.pv = plan_gemm(cfg->v_head, N, cfg->d_c, H, false, true, sm_count);
  l.po = plan_gemm(cfg->d_model, N, H * cfg->v_head, 1, false, false, sm_count);
  l.off_o = 0;
  l.off_part = align256((size_t)N * H * cfg->v_head * 2);
  l.total = l.off_part + align256(partial_bytes(l.po));
  return l;
}
}  // namespace

size_t tc_output_workspace_bytes(const mla_config* cfg, int N, int sm_count) {
  if (!tc_output_supported(cfg, N)) return 0;
  return output_layout(cfg, N, sm_count).total;
}

cudaError_t tc_output_project(const Ctx& ctx, const mla_config* cfg, const void* o_lat, const void* W_UV,
                              const void* W_O, void* out, int N, void* workspace) {
  const int D = cfg->d_model, H = cfg->n_heads, v = cfg->v_head, d_c = cfg->d_c;
  OutputLayout l = output_layout(cfg, N, ctx.sm_count);
  char* ws = static_cast<char*>(workspace);
  bf16* o = reinterpret_cast<bf16*>(ws + l.off_o);
  l.po.args.partial = reinterpret_cast<float*>(ws + l.off_part);
  CUtensorMap auv, bl, awo, bo;
  if (!make_map(&auv, W_UV, d_c, v, H, (uint64_t)d_c * 2, (uint64_t)d_c * 2 * v, 128) ||
      // o_lat^h: [n][h][c], rows n with stride H * d_c
      !make_map(&bl, o_lat, d_c, N, H, (uint64_t)H * d_c * 2, (uint64_t)d_c * 2, l.pv.args.n_tile) ||
      !make_map(&awo, W_O, (uint64_t)H * v, D, 1, (uint64_t)H * v * 2, (uint64_t)H * v * 2 * D, 128) ||
      !make_map(&bo, o, (uint64_t)H * v, N, 1, (uint64_t)H * v * 2, (uint64_t)H * v * 2 * N, l.po.args.n_tile))
    return cudaErrorInvalidValue;
  // o^h = W_UV^h o_lat^h, bf16 into o[n][h][v]
  l.pv.args.partial = nullptr;
  l.pv.args.out = o;
  l.pv.args.out_ld = (long long)H * v;
  l.pv.args.out_g = v;
  cudaError_t e = launch_gemm(ctx, auv, auv, bl, l.pv);
  if (e != cudaSuccess) return e;
  e = launch_gemm(ctx, awo, awo, bo, l.po);
  if (e != cudaSuccess) return e;
  const long long count = (long long)N * D;
  e = launch_pdl(sum_to_bf16_kernel, dim3(launch_blocks(count / 4, 256, ctx.sm_count)), dim3(256), 0, ctx.stream,
                 l.po.args.partial, l.po.args.splits, count, static_cast<bf16*>(out));
  count_launch();
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}


// ------------------------------------------------------------------ explicit form (prefill)
// Query projection without absorption: q_out[n][h] = [W_Q^h x_n || RoPE(W_QR^h x_n, q_pos_n)].
bool tc_project_supported(const mla_config* cfg, int N) {
  return shapes_ok(cfg) && N > 0 && stack_ok(cfg->n_heads * cfg->qk_nope) && cfg->d_rope % 4 == 0 &&
         cfg->qk_nope % 4 == 0;
}

size_t tc_project_workspace_bytes(const mla_config* cfg, int N, int sm_count) {
  if (!tc_project_supported(cfg, N)) return 0;
  const int H = cfg->n_heads;
  return align256(partial_bytes(plan_stacked(H * cfg->qk_nope, H * cfg->d_rope, N, cfg->d_model, sm_count)));
}

cudaError_t tc_project_query(const Ctx& ctx, const mla_config* cfg, const void* x, const void* W_Q, const void* W_QR,
                             const int32_t* q_pos, const mla_rope_table& rope, void* q_out, int N, void* workspace) {
  const int D = cfg->d_model, H = cfg->n_heads, qk = cfg->qk_nope, d_r = cfg->d_rope;
  GemmPlan pl = plan_stacked(H * qk, H * d_r, N, D, ctx.sm_count);
  pl.args.partial = static_cast<float*>(workspace);
  CUtensorMap aq, ar, bx;
  if (!make_map(&aq, W_Q, D, (uint64_t)H * qk, 1, (uint64_t)D * 2, (uint64_t)D * 2 * H * qk, 128) ||
      !make_map(&ar, W_QR, D, (uint64_t)H * d_r, 1, (uint64_t)D * 2, (uint64_t)D * 2 * H * d_r, 128) ||
      !make_map(&bx, x, D, N, 1, (uint64_t)D * 2, (uint64_t)D * 2 * N, pl.args.n_tile))
    return cudaErrorInvalidValue;
  cudaError_t e = launch_gemm(ctx, aq, ar, bx, pl);
  if (e != cudaSuccess) return e;
  const long long work = (long long)N * H * (qk + d_r) / 4;
  query_reduce_kernel<<<launch_blocks(work, 256, ctx.sm_count), 256, 0, ctx.stream>>>(
      pl.args.partial, pl.args.splits, N, H, qk, d_r, q_pos, rope.cos_sin, rope.max_pos, (bf16*)q_out, ctx.status);
  count_launch();
  return cudaGetLastError();
}

// Per-head keys and values rebuilt from the latent rows, stored chunk-major lat[(d_c + d_rope) / 64][L][64]
// (the first d_c / 64 chunks are read): row m of the stacked up-projections [W_UK (all heads); W_UV (all
// heads)] times c_t goes to kv[m / 64][t][m % 64], bf16.  Both layouts make every TMA box one contiguous
// run.  One GEMM, stored directly (K = d_c needs no k-split).
cudaError_t tc_reconstruct_kv(const Ctx& ctx, const mla_config* cfg, const void* lat, int L, const void* W_UK,
                              const void* W_UV, void* kv) {
  const int H = cfg->n_heads, qk = cfg->qk_nope, v = cfg->v_head, d_c = cfg->d_c, row = cfg->d_c + cfg->d_rope;
  if (qk % 64 || v % 64 || row % 64) return cudaErrorInvalidValue;
  GemmPlan pl = plan_gemm(H * qk + H * v, L, d_c, 1, false, true, ctx.sm_count);
  pl.args.m_tiles1 = H * qk / 128;
  pl.args.partial = nullptr;
  pl.args.out = static_cast<bf16*>(kv);
  pl.args.out_ld = 64;
  pl.args.out_g = 0;
  pl.args.out_mc = (long long)L * 64;
  pl.args.b_kchunk = 1;
  CUtensorMap a1, a2, b;
  if (!make_map(&a1, W_UK, d_c, (uint64_t)H * qk, 1, (uint64_t)d_c * 2, (uint64_t)d_c * 2 * H * qk, 128) ||
      !make_map(&a2, W_UV, d_c, (uint64_t)H * v, 1, (uint64_t)d_c * 2, (uint64_t)d_c * 2 * H * v, 128) ||
      !make_map(&b, lat, 64, L, row / 64, 128, (uint64_t)L * 128, pl.args.n_tile))
    return cudaErrorInvalidValue;
  return launch_gemm(ctx, a1, a2, b, pl);
}

// out = W_O concat_h(o^h) for head outputs o[N][H][v_head] (bf16).
bool tc_head_output_supported(const mla_config* cfg, int N) {
  return shapes_ok(cfg) && N > 0 && cfg->d_model % 4 == 0;
}

size_t tc_head_output_workspace_bytes(const mla_config* cfg, int N, int sm_count) {
  if (!tc_head_output_supported(cfg, N)) return 0;
  return align256(partial_bytes(plan_gemm(cfg->d_model, N, cfg->n_heads * cfg->v_head, 1, false, false, sm_count)));
}

cudaError_t tc_head_output_project(const Ctx& ctx, const mla_config* cfg, const void* o, const void* W_O, void* out,
                                   int N, void* workspace) {
  const int D = cfg->d_model, Hv = cfg->n_heads * cfg->v_head;
  GemmPlan po = plan_gemm(D, N, Hv, 1, false, false, ctx.sm_count);
  po.args.partial = static_cast<float*>(workspace);
  CUtensorMap awo, bo;
  if (!make_map(&awo, W_O, (uint64_t)Hv, D, 1, (uint64_t)Hv * 2, (uint64_t)Hv * 2 * D, 128) ||
      !make_map(&bo, o, (uint64_t)Hv, N, 1, (uint64_t)Hv * 2, (uint64_t)Hv * 2 * N, po.args.n_tile))
    return cudaErrorInvalidValue;
  cudaError_t e = launch_gemm(ctx, awo, awo, bo, po);
  if (e != cudaSuccess) return e;
  const long long count = (long long)N * D;
  sum_to_bf16_kernel<<<launch_blocks(count / 4, 256, ctx.sm_count), 256, 0, ctx.stream>>>(
      po.args.partial, po.args.splits, count, static_cast<bf16*>(out));
  count_launch();
  return cudaGetLastError();
}

}  // namespace mla
