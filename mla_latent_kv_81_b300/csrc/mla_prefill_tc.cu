// Prefill attention in the explicit form, on tcgen05 tensor cores.
//
// Every token of a prompt whose latent rows are already in the paged cache is a query attending
// causally to the prompt.  At prefill the pages recompute per-head keys and values from the cached
// latent instead of keeping them ("Multi-head Latent Attention" card mla-attention, point 4: K/V
// recomputed from the latent at prefill; "What does Multi-head Latent Attention compress...", "The
// mechanism": up-projections expand the latent into per-head keys and values).  For a long prompt
// this form costs 2 (qk_nope + d_rope + v_head) FLOP per (query, key, head), against
// 2 (d_c + d_rope + d_c) for the absorbed form, so the keys and values are rebuilt once:
//   1. gather_latent_kernel: the sequence's rows, stored element-major per cache block, into one
//      token-major buffer lat[L][d_c + d_rope];
//   2. tc_reconstruct_kv (projection GEMM): kv[t] = [W_UK^h c_t for all h || W_UV^h c_t for all h];
//   3. prefill_attn_kernel: per (head, 128-query tile) unit, scores S = Q K^T over 128-key tiles with
//      K = [W_UK^h c_t || k_R,t] (the positional key shared by all heads, taken from lat; its score
//      added to the content score, "Multi-head Latent Attention (MLA)" Implementation Logic step 5,
//      reading c2), causal online softmax, O += P V, O = softmax . V^h.
//
// Kernel layout (one CTA per SM, persistent over units, 256 threads):
//   warp 0: TMA producer; warp 1: MMA issuer (one thread); warp 2: TMEM allocation;
//   warps 4-7: softmax, one thread per query row (TMEM lane), then the epilogue.
//   TMEM: S double-buffered in columns [0, 256), O in [256, 384), the query in [384, 480)
//   (copied from shared memory with tcgen05.cp, the A operand of the score MMAs).
//   Shared memory: a ring of 48 KB slots for the query (3 chunks of 64 elements) and the key tiles
//   (K_nope: 2 chunks, k_R: 1 chunk, each [128 tokens][128 B] with the 128-byte swizzle); a ring of
//   32 KB value slots ([2 chunks of 64 dims][128 tokens][128 B], an MN-major B operand); one 32 KB
//   buffer of P (bf16, K-major A operand of the P V MMAs).
#include <math.h>

#include "mla_sm100.cuh"
#include "mla_tc.cuh"

namespace mla {
namespace {
using namespace sm100;

constexpr int kH = 128, kQK = 128, kDR = 64, kVH = 128, kDC = 512, kRowW = kDC + kDR;
constexpr int kQW = kQK + kDR;            // query row [q_nope || q_R]
constexpr int kFT = 128;                  // queries per tile, keys per tile
constexpr int kFBlk = 64;                 // cache block size the kernel is built for
constexpr int kChunk = kFT * 128;         // [128 rows][64 bf16] = 16 KB
constexpr int kSSlot = 3 * kChunk;        // query, or K_nope (2 chunks) + k_R (1 chunk)
constexpr int kVSlot = 2 * kChunk;        // V (2 chunks of 64 dims)
constexpr int kSRing = 2, kVRing = 2;
constexpr int kFThreads = 256;
constexpr int kOffSRing = 1024;
constexpr int kOffVRing = kOffSRing + kSRing * kSSlot;
constexpr int kOffP = kOffVRing + kVRing * kVSlot;
constexpr int kFSmem = kOffP + 2 * kChunk + 1024;   // + alignment slack of the dynamic base
constexpr uint32_t kColS = 0, kColO = 256, kColQ = 384;
constexpr float kFLazy = 8.f;                        // the running max moves when it grows by > 2^8

static_assert(kFSmem <= 232448, "shared memory of one CTA");
static_assert(kQW == 3 * 64 && kQK == 2 * 64 && kVH == 2 * 64, "64-element chunks");

struct FCtrl {
  uint64_t k_full[kSRing], k_empty[kSRing], v_full[kVRing], v_empty[kVRing];
  uint64_t s_full[2], s_empty[2], p_full, pv_done, o_free;
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(FCtrl) <= kOffSRing, "control block");

struct FParams {
  int T, L, q0;       // queries, keys (cached prompt rows), position of query 0 (= L - T)
  int H, qtiles, units;
  float scale_log2;
  bf16* o;            // [T][H][v_head]
  float* lse;         // [T][H] or null
  uint32_t* status;
};

// Unit u: head h and query tile qt (the longest query tiles of a head first); p0 = position of the
// tile's first query; n = key tiles up to the tile's last valid query.
__device__ __forceinline__ void unit_of(const FParams& p, int u, int& h, int& qt, int& n, int& p0) {
  h = u / p.qtiles;
  qt = p.qtiles - 1 - u % p.qtiles;
  p0 = p.q0 + qt * kFT;
  const int last = p.q0 + min(qt * kFT + kFT, p.T) - 1;
  n = last / kFT + 1;
}

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, uint32_t* status, volatile int* abort_flag) {
  const bool ok = mbar_wait_cta(bar, parity, status, abort_flag);
  return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ void tmem_cp_128x256b(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.128x256b [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

// ------------------------------------------------------------------ gather
// lat[t][e] = element e of the token at position t of sequence `seq`, for t < L.  Block (64-token
// cache block, 64-element group): the block's element rows (64 tokens, contiguous) are read, transposed
// through shared memory and written token-major.  Out-of-range block-table entries flag an index
// error and give zero rows.
__global__ void __launch_bounds__(256) gather_latent_kernel(const bf16* pool, const int32_t* table, int max_blocks,
                                                            int num_blocks, int seq, int L, bf16* lat,
                                                            uint32_t* status) {
  __shared__ uint16_t tile[64][65];
  const int bt = blockIdx.x, e0 = blockIdx.y * 64;
  int blk = bt < max_blocks ? table[(long long)seq * max_blocks + bt] : -1;
  if (blk < 0 || blk >= num_blocks) {
    if (threadIdx.x == 0 && blockIdx.y == 0) flag_error(status, kFlagIndex);
    blk = -1;
  }
  const uint16_t* src = reinterpret_cast<const uint16_t*>(pool);
  for (int i = threadIdx.x; i < 64 * 64; i += 256) {
    const int e = i >> 6, t = i & 63;
    tile[e][t] = blk >= 0 ? src[((long long)blk * kRowW + e0 + e) * kFBlk + t] : (uint16_t)0;
  }
  __syncthreads();
  uint16_t* dst = reinterpret_cast<uint16_t*>(lat);
  for (int i = threadIdx.x; i < 64 * 64; i += 256) {
    const int t = i >> 6, e = i & 63;
    const int pos = bt * kFBlk + t;
    if (pos < L) dst[(long long)pos * kRowW + e0 + e] = tile[e][t];
  }
}

// ------------------------------------------------------------------ attention
// mapq: q [T][H][192] as {192, H, T}; mapkv: kv [L][2H][128] as {128, 2H, L} (heads H.. are V);
// mapr: lat [L][576] as {576, L}.  Boxes of 64 elements x 128 rows, out-of-range rows read as zero.
__global__ void __launch_bounds__(kFThreads, 1)
    prefill_attn_kernel(const __grid_constant__ CUtensorMap mapq, const __grid_constant__ CUtensorMap mapkv,
                        const __grid_constant__ CUtensorMap mapr, FParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  FCtrl* ctrl = reinterpret_cast<FCtrl*>(smem);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  volatile int* abort_flag = &ctrl->abort_flag;

  if (tid == 0) {
    for (int i = 0; i < kSRing; ++i) { mbar_init(&ctrl->k_full[i], 1); mbar_init(&ctrl->k_empty[i], 1); }
    for (int i = 0; i < kVRing; ++i) { mbar_init(&ctrl->v_full[i], 1); mbar_init(&ctrl->v_empty[i], 1); }
    for (int i = 0; i < 2; ++i) { mbar_init(&ctrl->s_full[i], 1); mbar_init(&ctrl->s_empty[i], 128); }
    mbar_init(&ctrl->p_full, 128);
    mbar_init(&ctrl->pv_done, 1);
    mbar_init(&ctrl->o_free, 128);
    ctrl->abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 2) {
    tmem_alloc(&ctrl->tmem_base, 512);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&mapq);
    prefetch_tmap(&mapkv);
    prefetch_tmap(&mapr);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctrl->tmem_base;
  const uint32_t sbase = smem_u32(smem);

  if (warp == 0) {
    if (lane == 0) {
      // producer, in the order the MMA thread consumes: the query, K(0), then K(j), V(j-1) for
      // j = 1..n-1, then V(n-1)
      int kr = 0, vr = 0;
      uint32_t kph = 0, vph = 0;
      for (int u = blockIdx.x; u < p.units; u += gridDim.x) {
        int h, qt, n, p0;
        unit_of(p, u, h, qt, n, p0);
        if (!mbar_wait_cta(&ctrl->k_empty[kr], kph ^ 1, p.status, abort_flag)) goto done;
        {
          uint8_t* dst = smem + kOffSRing + kr * kSSlot;
          mbar_arrive_expect_tx(&ctrl->k_full[kr], kSSlot);
#pragma unroll
          for (int c = 0; c < 3; ++c) tma_load_3d(dst + c * kChunk, &mapq, &ctrl->k_full[kr], c * 64, h, qt * kFT);
        }
        if (++kr == kSRing) { kr = 0; kph ^= 1; }
        for (int j = 0; j <= n; ++j) {
          if (j < n) {
            if (!mbar_wait_cta(&ctrl->k_empty[kr], kph ^ 1, p.status, abort_flag)) goto done;
            uint8_t* dst = smem + kOffSRing + kr * kSSlot;
            mbar_arrive_expect_tx(&ctrl->k_full[kr], kSSlot);
            tma_load_3d(dst, &mapkv, &ctrl->k_full[kr], 0, h, j * kFT);
            tma_load_3d(dst + kChunk, &mapkv, &ctrl->k_full[kr], 64, h, j * kFT);
            tma_load_2d(dst + 2 * kChunk, &mapr, &ctrl->k_full[kr], kDC, j * kFT);
            if (++kr == kSRing) { kr = 0; kph ^= 1; }
          }
          if (j >= 1) {
            if (!mbar_wait_cta(&ctrl->v_empty[vr], vph ^ 1, p.status, abort_flag)) goto done;
            uint8_t* dst = smem + kOffVRing + vr * kVSlot;
            mbar_arrive_expect_tx(&ctrl->v_full[vr], kVSlot);
            tma_load_3d(dst, &mapkv, &ctrl->v_full[vr], 0, p.H + h, (j - 1) * kFT);
            tma_load_3d(dst + kChunk, &mapkv, &ctrl->v_full[vr], 64, p.H + h, (j - 1) * kFT);
            if (++vr == kVRing) { vr = 0; vph ^= 1; }
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // S (128 queries x 128 keys) = Q K^T: A = the query in TMEM (8 columns per 16-element K-step),
      // B = the key slot (K-major, 32 B per K-step).  O (128 x 128) += P V: A = P (K-major, two
      // 64-key chunks), B = the value slot (MN-major: 64-dim chunks kChunk apart, 2048 B per 16 keys).
      const uint32_t idesc_s = idesc_bf16(128, kFT, false, false);
      const uint32_t idesc_pv = idesc_bf16(128, kVH, false, true);
      const uint64_t kdesc0 = desc_sw128(sbase + kOffSRing, 16, 1024);
      const uint64_t vdesc0 = desc_sw128(sbase + kOffVRing, kChunk, 1024);
      const uint64_t pdesc0 = desc_sw128(sbase + kOffP, 16, 1024);
      const uint32_t tq = tmem + kColQ, to = tmem + kColO;
      int kr = 0, vr = 0, g = 0, nu = 0;
      uint32_t kph = 0, vph = 0;
      for (int u = blockIdx.x; u < p.units; u += gridDim.x, ++nu) {
        int h, qt, n, p0;
        unit_of(p, u, h, qt, n, p0);
        // the unit's query into TMEM: this thread's tcgen05 operations run in issue order, so the copies
        // land only after the previous unit's score MMAs have read the old query
        if (!mbar_wait_cta(&ctrl->k_full[kr], kph, p.status, abort_flag)) goto done;
        tc_fence_after();
        {
          const uint64_t qd = kdesc0 + (uint64_t)(kr * (kSSlot >> 4));
#pragma unroll
          for (int c = 0; c < 3; ++c)
#pragma unroll
            for (int k = 0; k < 4; ++k)
              tmem_cp_128x256b(tq + c * 32 + k * 8, qd + (uint64_t)(c * (kChunk >> 4) + k * 2));
        }
        mma_commit(&ctrl->k_empty[kr]);
        if (++kr == kSRing) { kr = 0; kph ^= 1; }
        for (int j = 0; j <= n; ++j) {
          if (j < n) {
            const int gs = g + j, buf = gs & 1;
            if (!mbar_wait_cta(&ctrl->s_empty[buf], ((gs >> 1) & 1) ^ 1, p.status, abort_flag)) goto done;
            if (!mbar_wait_cta(&ctrl->k_full[kr], kph, p.status, abort_flag)) goto done;
            tc_fence_after();
            const uint64_t kd = kdesc0 + (uint64_t)(kr * (kSSlot >> 4));
            const uint32_t d = tmem + kColS + buf * kFT;
#pragma unroll
            for (int c = 0; c < 3; ++c)
#pragma unroll
              for (int k = 0; k < 4; ++k)
                mma_ts(d, tq + c * 32 + k * 8, kd + (uint64_t)(c * (kChunk >> 4) + k * 2), idesc_s,
                       (c | k) ? 1u : 0u);
            mma_commit(&ctrl->k_empty[kr]);
            mma_commit(&ctrl->s_full[buf]);
            if (++kr == kSRing) { kr = 0; kph ^= 1; }
          }
          if (j >= 1) {
            const int gp = g + j - 1;
            if (!mbar_wait_cta(&ctrl->p_full, gp & 1, p.status, abort_flag)) goto done;
            // the first P V of a unit overwrites O: the previous unit's epilogue must have read it
            if (j == 1 && !mbar_wait_cta(&ctrl->o_free, (nu & 1) ^ 1, p.status, abort_flag)) goto done;
            if (!mbar_wait_cta(&ctrl->v_full[vr], vph, p.status, abort_flag)) goto done;
            tc_fence_after();
            const uint64_t vd = vdesc0 + (uint64_t)(vr * (kVSlot >> 4));
#pragma unroll
            for (int k = 0; k < 8; ++k)
              mma_ss(to, pdesc0 + (uint64_t)((k >> 2) * (kChunk >> 4) + (k & 3) * 2), vd + (uint64_t)(k * 128),
                     idesc_pv, (j > 1 || k > 0) ? 1u : 0u);
            mma_commit(&ctrl->v_empty[vr]);
            mma_commit(&ctrl->pv_done);
            if (++vr == kVRing) { vr = 0; vph ^= 1; }
          }
        }
        g += n;
      }
    }
  } else if (warp >= 4) {
    // softmax: thread = query row r of the unit's tile (TMEM lane r)
    const int q4 = warp & 3, r = q4 * 32 + lane;
    const uint32_t lane_base = tmem + ((uint32_t)(q4 * 32) << 16);
    uint8_t* prow = smem + kOffP + r * 128;
    const int sw = r & 7;
    int g = 0;
    for (int u = blockIdx.x; u < p.units; u += gridDim.x) {
      int h, qt, n, p0;
      unit_of(p, u, h, qt, n, p0);
      const int pos = p0 + r;   // this query's position: it sees keys 0..pos
      float m = -INFINITY, l = 0.f;
      for (int j = 0; j < n; ++j, ++g) {
        const int buf = g & 1;
        if (!warp_wait(&ctrl->s_full[buf], (g >> 1) & 1, p.status, abort_flag)) goto done;
        tc_fence_after();
        uint32_t s[4][32];
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32(lane_base + kColS + buf * kFT + c * 32, s[c]);
        tmem_ld_wait();
        tc_fence_before();
        mbar_arrive(&ctrl->s_empty[buf]);
        if (j * kFT + kFT - 1 > p0) {
          // a tile holding keys after some query of the tile: causal mask
          const int lim = pos - j * kFT;
#pragma unroll
          for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (c * 32 + i > lim) s[c][i] = __float_as_uint(-INFINITY);
        }
        float mx = -INFINITY;
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int i = 0; i < 32; ++i) mx = fmaxf(mx, __uint_as_float(s[c][i]));
        mx *= p.scale_log2;   // the positive scale commutes with the maximum
        float alpha = 1.f;
        if (j == 0) {
          m = mx;
        } else if (mx > m + kFLazy) {
          alpha = ex2(m - mx);
          l *= alpha;
          m = mx;
        }
        // the row sum adds the bf16 weights the P V MMAs use, so that the weights of the output are
        // normalised exactly: with the lazy maximum the largest weight is up to 2^8, not 1, and an fp32
        // sum of the unrounded weights would scale a row dominated by one token by its rounding error
        uint32_t pk[64];
        float sum0 = 0.f, sum1 = 0.f;
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float e0 = ex2(fmaf(__uint_as_float(s[c][2 * i]), p.scale_log2, -m));
            const float e1 = ex2(fmaf(__uint_as_float(s[c][2 * i + 1]), p.scale_log2, -m));
            const uint32_t w = pack_bf16x2(e0, e1);
            sum0 += __uint_as_float(w << 16);
            sum1 += __uint_as_float(w & 0xFFFF0000u);
            pk[c * 16 + i] = w;
          }
        l += sum0 + sum1;
        // the previous P V has read the P buffer and finished accumulating O
        if (g >= 1 && !warp_wait(&ctrl->pv_done, (g - 1) & 1, p.status, abort_flag)) goto done;
        tc_fence_after();
        if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
          for (int c = 0; c < 4; ++c) {
            uint32_t o[32];
            tmem_ld32(lane_base + kColO + c * 32, o);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
            tmem_st32(lane_base + kColO + c * 32, o);
          }
          tmem_st_wait();
        }
        // P row r: keys 64 ch .. 64 ch + 63 in chunk ch, 16-byte unit uu (keys 8 uu .. 8 uu + 7) at the
        // 128-byte swizzled position uu ^ (r & 7)
#pragma unroll
        for (int ch = 0; ch < 2; ++ch)
#pragma unroll
          for (int uu = 0; uu < 8; ++uu)
            *reinterpret_cast<uint4*>(prow + ch * kChunk + ((uu ^ sw) << 4)) =
                make_uint4(pk[ch * 32 + 4 * uu], pk[ch * 32 + 4 * uu + 1], pk[ch * 32 + 4 * uu + 2],
                           pk[ch * 32 + 4 * uu + 3]);
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(&ctrl->p_full);
      }
      // epilogue: O / l in bf16, and the log-sum-exp of the row
      if (!warp_wait(&ctrl->pv_done, (g - 1) & 1, p.status, abort_flag)) goto done;
      tc_fence_after();
      {
        const float inv = l > 0.f ? 1.f / l : 0.f;
        const int q = qt * kFT + r;
        uint4* dst = reinterpret_cast<uint4*>(p.o + ((long long)q * p.H + h) * kVH);
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t o[32];
          tmem_ld32(lane_base + kColO + c * 32, o);
          tmem_ld_wait();
          if (q < p.T) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              uint32_t w[4];
#pragma unroll
              for (int k = 0; k < 4; ++k)
                w[k] = pack_bf16x2(__uint_as_float(o[8 * i + 2 * k]) * inv, __uint_as_float(o[8 * i + 2 * k + 1]) * inv);
              dst[c * 4 + i] = make_uint4(w[0], w[1], w[2], w[3]);
            }
          }
        }
        if (q < p.T && p.lse) p.lse[(long long)q * p.H + h] = l > 0.f ? (m + __log2f(l)) * kLn2 : -INFINITY;
      }
      tc_fence_before();
      mbar_arrive(&ctrl->o_free);
    }
  }

done:
  tc_fence_before();
  __syncthreads();
  if (*abort_flag && warp == 0 && lane == 0) {
    // let any copy still in flight land before the CTA's shared memory goes away
    const long long t0 = clock64();
    while (clock64() - t0 < 2000000LL) { }
  }
  tc_fence_after();
  if (warp == 2) tmem_dealloc(tmem, 512);
}

struct PrefillLayout {
  size_t lat, kv, total;
};
PrefillLayout prefill_layout(int L) {
  PrefillLayout w;
  auto a256 = [](size_t v) { return (v + 255) / 256 * 256; };
  w.lat = 0;
  w.kv = a256((size_t)L * kRowW * 2);
  w.total = w.kv + a256((size_t)L * 2 * kH * kQK * 2);
  return w;
}

}  // namespace

bool tc_prefill_supported(const mla_config* cfg) {
  return cfg->dtype == MLA_BF16 && cfg->n_heads == kH && cfg->qk_nope == kQK && cfg->d_rope == kDR &&
         cfg->v_head == kVH && cfg->d_c == kDC && cfg->block_size == kFBlk && cfg->d_model % 64 == 0;
}

size_t tc_prefill_workspace_bytes(const mla_config* cfg, int kv_len) {
  if (!tc_prefill_supported(cfg) || kv_len <= 0) return 0;
  return prefill_layout(kv_len).total;
}

cudaError_t tc_prefill_attention(const Ctx& ctx, const mla_config* cfg, const void* q, const mla_paged_cache& cache,
                                 int seq, int kv_len, int T, const void* W_UK, const void* W_UV, float scale, void* o,
                                 float* lse, void* workspace) {
  const int L = kv_len, H = kH;
  const PrefillLayout w = prefill_layout(L);
  char* base = static_cast<char*>(workspace);
  bf16* lat = reinterpret_cast<bf16*>(base + w.lat);
  bf16* kv = reinterpret_cast<bf16*>(base + w.kv);
  const dim3 gg((L + kFBlk - 1) / kFBlk, kRowW / 64);
  gather_latent_kernel<<<gg, 256, 0, ctx.stream>>>(static_cast<const bf16*>(cache.pool), cache.block_table,
                                                   cache.max_blocks_per_seq, cache.num_blocks, seq, L, lat,
                                                   ctx.status);
  count_launch();
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  e = tc_reconstruct_kv(ctx, cfg, lat, L, W_UK, W_UV, kv);
  if (e != cudaSuccess) return e;
  CUtensorMap mapq, mapkv, mapr;
  const uint64_t dq[3] = {(uint64_t)kQW, (uint64_t)H, (uint64_t)T}, sq[2] = {(uint64_t)kQW * 2, (uint64_t)H * kQW * 2};
  const uint64_t dkv[3] = {(uint64_t)kQK, (uint64_t)2 * H, (uint64_t)L},
                 skv[2] = {(uint64_t)kQK * 2, (uint64_t)2 * H * kQK * 2};
  const uint64_t dr[2] = {(uint64_t)kRowW, (uint64_t)L}, sr[1] = {(uint64_t)kRowW * 2};
  const uint32_t box3[3] = {64, 1, kFT}, box2[2] = {64, kFT};
  if (!encode_map_bf16(&mapq, q, 3, dq, sq, box3) || !encode_map_bf16(&mapkv, kv, 3, dkv, skv, box3) ||
      !encode_map_bf16(&mapr, lat, 2, dr, sr, box2))
    return cudaErrorInvalidValue;
  FParams fp;
  fp.T = T;
  fp.L = L;
  fp.q0 = L - T;
  fp.H = H;
  fp.qtiles = (T + kFT - 1) / kFT;
  fp.units = H * fp.qtiles;
  fp.scale_log2 = scale * kLog2e;
  fp.o = static_cast<bf16*>(o);
  fp.lse = lse;
  fp.status = ctx.status;
  e = ensure_smem_limit((const void*)prefill_attn_kernel, kFSmem, ctx.device);
  if (e != cudaSuccess) return e;
  const int grid = fp.units < ctx.sm_count ? fp.units : ctx.sm_count;
  prefill_attn_kernel<<<grid, kFThreads, kFSmem, ctx.stream>>>(mapq, mapkv, mapr, fp);
  count_launch();
  return cudaGetLastError();
}

}  // namespace mla
