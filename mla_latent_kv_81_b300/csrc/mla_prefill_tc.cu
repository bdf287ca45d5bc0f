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
//      chunk-major buffer lat[row / 64][L][64] (row = d_c + d_rope, or d_c + H d_rope with per-head
//      positional keys, head h's key then in chunk d_c / 64 + h);
//   2. tc_reconstruct_kv (projection GEMM): per-head keys W_UK^h c_t and values W_UV^h c_t, chunk-major
//      kv[4H][L][64] (64-element chunk 2h + c of head h's key, 2H + 2h + c of its value);
//   Every TMA box of the GEMM and of the attention kernel over these buffers is one contiguous run
//   (rows of 128 B 1 KB or more apart had held a box to a fraction of the per-SM copy rate).
//   3. prefill_attn_kernel: per (head, 128-query tile) unit, scores S = Q K^T over 128-key tiles with
//      K = [W_UK^h c_t || k_R,t] (the positional key shared by all heads, taken from lat; its score
//      added to the content score, "Multi-head Latent Attention (MLA)" Implementation Logic step 5,
//      reading c2), causal online softmax, O += P V, O = softmax . V^h.
//
// Kernel layout (one CTA per SM, persistent over units, 256 threads):
//   warp 0: TMA producer of the key ring; warp 3: TMA producer of the value ring; warp 1: MMA issuer
//   (one thread); warp 2: TMEM allocation;
//   warps 4-11: softmax and epilogue, two threads per query row (TMEM lane): warps 4-7 take key columns
//   0-63 of S and value columns 0-63 of O, warps 8-11 columns 64-127; the two halves of a row exchange
//   their maxima (and, at the end of a unit, their row sums) through shared memory and a bounded
//   mbarrier.
//   TMEM: S double-buffered in columns [0, 256), O in [256, 384), the query in [384, 480)
//   (copied from shared memory with tcgen05.cp, the A operand of the score MMAs).  P (bf16) is written
//   over the first 64 columns of its own S buffer and read from there as the A operand of P V.
//   Shared memory: a ring of nine 16 KB chunk slots for the query chunks and the key tiles (K_nope: 2
//   chunks, k_R: 1 chunk, each [128 tokens][128 B] with the 128-byte swizzle), three key tiles deep;
//   a ring of two 32 KB value slots ([2 chunks of 64 dims][128 tokens][128 B], an MN-major B operand).
//   The loads run up to three tiles ahead: the kernel's pace is otherwise set by the latency of the
//   copies (bytes in flight per SM), not by the tensor cores or the softmax.
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
constexpr int kKSlots = 9;                // K ring: 16 KB chunk slots (query chunks, then 3 per key tile)
constexpr int kVSlot = 2 * kChunk;        // V ring slot: the tile's two 64-dim chunks, adjacent
constexpr int kVRing = 2;
constexpr int kFThreads = 384;
constexpr int kOffKRing = 4096;
constexpr int kOffVRing = kOffKRing + kKSlots * kChunk;
constexpr int kFSmem = kOffVRing + kVRing * kVSlot + 1024;   // + alignment slack of the dynamic base
constexpr uint32_t kColS = 0, kColO = 256, kColQ = 384;
constexpr float kFLazy = 8.f;                        // the running max moves when it grows by > 2^8

static_assert(kFSmem <= 232448, "shared memory of one CTA");
static_assert(kQW == 3 * 64 && kQK == 2 * 64 && kVH == 2 * 64, "64-element chunks");

struct FCtrl {
  uint64_t k_full[kKSlots], k_empty[kKSlots], v_full[kVRing], v_empty[kVRing];
  uint64_t s_full[2], p_full[2], pv_done[2], o_free;   // one s_full / p_full / pv_done per S buffer
  uint64_t xch[2];                 // exchanges between the two halves of each row (alternating)
  uint32_t tmem_base;
  int abort_flag;
  float xval[2][2][128];           // [exchange parity][half][row]: half-row maxima, or partial row sums
};
static_assert(sizeof(FCtrl) <= kOffKRing, "control block");

struct FParams {
  int T, L, q0;       // queries, keys (cached prompt rows), position of query 0 (= L - T)
  int H, qtiles, units;
  int rope_chunk, rope_step;   // chunk of lat holding head h's positional key: rope_chunk + h * rope_step
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
// lat[e / 64][t][e % 64] = element e of the token at position t of sequence `seq`, for t < L.  Block
// (64-token cache block, 64-element chunk): the block's element rows (64 tokens, contiguous) are read,
// transposed through shared memory and written as 64 rows of 128 B (one contiguous 8 KB run).
// Out-of-range block-table entries flag an index error and give zero rows.
__global__ void __launch_bounds__(256) gather_latent_kernel(const bf16* pool, int row_w, const int32_t* table,
                                                            int max_blocks, int num_blocks, int seq, int L, bf16* lat,
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
    tile[e][t] = blk >= 0 ? src[((long long)blk * row_w + e0 + e) * kFBlk + t] : (uint16_t)0;
  }
  __syncthreads();
  uint16_t* dst = reinterpret_cast<uint16_t*>(lat);
  for (int i = threadIdx.x; i < 64 * 64; i += 256) {
    const int t = i >> 6, e = i & 63;
    const int pos = bt * kFBlk + t;
    if (pos < L) dst[((long long)blockIdx.y * L + pos) * 64 + e] = tile[e][t];
  }
}

// ------------------------------------------------------------------ attention
// mapq: q [T][H][192] as {192, H, T}, box {64, 1, 128}; mapkv: kv [4H][L][64] as {64, L, 4H} and mapr:
// lat [9][L][64] as {64, L, 9}, boxes {64, 128, 1}.  Out-of-range rows read as zero.
__global__ void __launch_bounds__(kFThreads, 1)
    prefill_attn_kernel(const __grid_constant__ CUtensorMap mapq, const __grid_constant__ CUtensorMap mapkv,
                        const __grid_constant__ CUtensorMap mapr, FParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  FCtrl* ctrl = reinterpret_cast<FCtrl*>(smem);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  volatile int* abort_flag = &ctrl->abort_flag;

  if (tid == 0) {
    for (int i = 0; i < kKSlots; ++i) { mbar_init(&ctrl->k_full[i], 1); mbar_init(&ctrl->k_empty[i], 1); }
    for (int i = 0; i < kVRing; ++i) { mbar_init(&ctrl->v_full[i], 1); mbar_init(&ctrl->v_empty[i], 1); }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&ctrl->s_full[i], 1);
      mbar_init(&ctrl->p_full[i], 256);
      mbar_init(&ctrl->pv_done[i], 1);
      mbar_init(&ctrl->xch[i], 256);
    }
    mbar_init(&ctrl->o_free, 256);
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
      // key producer, in the order the MMA thread consumes the key ring: the query's 3 chunks, then the
      // 3 chunks of each key tile.  One 16 KB chunk per slot.
      int kr = 0;
      uint32_t kph = 0;
      auto load_chunk = [&](const CUtensorMap* map, int c0, int c1, int c2) -> bool {
        if (!mbar_wait_cta(&ctrl->k_empty[kr], kph ^ 1, p.status, abort_flag)) return false;
        mbar_arrive_expect_tx(&ctrl->k_full[kr], kChunk);
        tma_load_3d(smem + kOffKRing + kr * kChunk, map, &ctrl->k_full[kr], c0, c1, c2);
        if (++kr == kKSlots) { kr = 0; kph ^= 1; }
        return true;
      };
      for (int u = blockIdx.x; u < p.units; u += gridDim.x) {
        int h, qt, n, p0;
        unit_of(p, u, h, qt, n, p0);
        for (int c = 0; c < 3; ++c)
          if (!load_chunk(&mapq, c * 64, h, qt * kFT)) goto done;
        for (int j = 0; j < n; ++j)
          if (!load_chunk(&mapkv, 0, j * kFT, 2 * h) || !load_chunk(&mapkv, 0, j * kFT, 2 * h + 1) ||
              !load_chunk(&mapr, 0, j * kFT, p.rope_chunk + h * p.rope_step))
            goto done;
      }
    }
  } else if (warp == 3) {
    if (lane == 0) {
      // value producer: one tile of V per slot.  Its own thread, so that a full value ring never holds
      // back the key loads (the copies take microseconds under load: the key ring must run ahead)
      int vr = 0;
      uint32_t vph = 0;
      for (int u = blockIdx.x; u < p.units; u += gridDim.x) {
        int h, qt, n, p0;
        unit_of(p, u, h, qt, n, p0);
        for (int j = 0; j < n; ++j) {
          if (!mbar_wait_cta(&ctrl->v_empty[vr], vph ^ 1, p.status, abort_flag)) goto done;
          uint8_t* dst = smem + kOffVRing + vr * kVSlot;
          mbar_arrive_expect_tx(&ctrl->v_full[vr], kVSlot);
          tma_load_3d(dst, &mapkv, &ctrl->v_full[vr], 0, j * kFT, 2 * p.H + 2 * h);
          tma_load_3d(dst + kChunk, &mapkv, &ctrl->v_full[vr], 0, j * kFT, 2 * p.H + 2 * h + 1);
          if (++vr == kVRing) { vr = 0; vph ^= 1; }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // S (128 queries x 128 keys) = Q K^T: A = the query in TMEM (8 columns per 16-element K-step),
      // B = a key chunk slot (K-major, 32 B per K-step).  O (128 x 128) += P V: A = P, written by the
      // softmax over the first 64 columns of its own S buffer (bf16 pairs, 8 columns per 16 keys),
      // B = the value slot (MN-major: 64-dim chunks kChunk apart, 2048 B per 16 keys).
      const uint32_t idesc_s = idesc_bf16(128, kFT, false, false);
      const uint32_t idesc_pv = idesc_bf16(128, kVH, false, true);
      const uint64_t kdesc0 = desc_sw128(sbase + kOffKRing, 16, 1024);
      const uint64_t vdesc0 = desc_sw128(sbase + kOffVRing, kChunk, 1024);
      const uint32_t tq = tmem + kColQ, to = tmem + kColO;
      int kr = 0, vr = 0, g = 0, nu = 0;
      uint32_t kph = 0, vph = 0;
      for (int u = blockIdx.x; u < p.units; u += gridDim.x, ++nu) {
        int h, qt, n, p0;
        unit_of(p, u, h, qt, n, p0);
        // the unit's query into TMEM: this thread's tcgen05 operations run in issue order, so the copies
        // land only after the previous unit's score MMAs have read the old query
        for (int c = 0; c < 3; ++c) {
          if (!mbar_wait_cta(&ctrl->k_full[kr], kph, p.status, abort_flag)) goto done;
          tc_fence_after();
          const uint64_t qd = kdesc0 + (uint64_t)(kr * (kChunk >> 4));
#pragma unroll
          for (int k = 0; k < 4; ++k) tmem_cp_128x256b(tq + c * 32 + k * 8, qd + (uint64_t)(k * 2));
          mma_commit(&ctrl->k_empty[kr]);
          if (++kr == kKSlots) { kr = 0; kph ^= 1; }
        }
        for (int j = 0; j <= n; ++j) {
          if (j < n) {
            const int gs = g + j, buf = gs & 1;
            // S buffer buf last held P(gs - 2), read by P V(gs - 2): that MMA was issued by this thread
            // before, and tcgen05 operations of one thread run in issue order, so S(gs) may be queued now
            const uint32_t d = tmem + kColS + buf * kFT;
#pragma unroll
            for (int c = 0; c < 3; ++c) {
              if (!mbar_wait_cta(&ctrl->k_full[kr], kph, p.status, abort_flag)) goto done;
              tc_fence_after();
              const uint64_t kd = kdesc0 + (uint64_t)(kr * (kChunk >> 4));
#pragma unroll
              for (int k = 0; k < 4; ++k)
                mma_ts(d, tq + c * 32 + k * 8, kd + (uint64_t)(k * 2), idesc_s, (c | k) ? 1u : 0u);
              mma_commit(&ctrl->k_empty[kr]);
              if (++kr == kKSlots) { kr = 0; kph ^= 1; }
            }
            mma_commit(&ctrl->s_full[buf]);
            // P V(gs - 2) done before anything later: every wait on a pv_done barrier (this one, the
            // softmax's before a rescale, the epilogue's) then finds its barrier at most one phase short
            // of the completion it names (the barriers are per S buffer because at a unit's first tile
            // P V(gs - 1) has already been issued)
            if (gs >= 2 && !mbar_wait_cta(&ctrl->pv_done[buf], ((gs >> 1) & 1) ^ 1, p.status, abort_flag)) goto done;
          }
          if (j >= 1) {
            const int gp = g + j - 1;
            // one barrier per S buffer: the softmax may write P(gp + 1) before this wait, so a single
            // barrier could run two phases ahead of it
            if (!mbar_wait_cta(&ctrl->p_full[gp & 1], (gp >> 1) & 1, p.status, abort_flag)) goto done;
            // the first P V of a unit overwrites O: the previous unit's epilogue must have read it
            if (j == 1 && !mbar_wait_cta(&ctrl->o_free, (nu & 1) ^ 1, p.status, abort_flag)) goto done;
            if (!mbar_wait_cta(&ctrl->v_full[vr], vph, p.status, abort_flag)) goto done;
            tc_fence_after();
            const uint64_t vd = vdesc0 + (uint64_t)(vr * (kVSlot >> 4));
            const uint32_t pa = tmem + kColS + (gp & 1) * kFT;
#pragma unroll
            for (int k = 0; k < 8; ++k)
              mma_ts(to, pa + k * 8, vd + (uint64_t)(k * 128), idesc_pv, (j > 1 || k > 0) ? 1u : 0u);
            mma_commit(&ctrl->v_empty[vr]);
            mma_commit(&ctrl->pv_done[gp & 1]);
            if (++vr == kVRing) { vr = 0; vph ^= 1; }
          }
        }
        g += n;
      }
    }
  } else if (warp >= 4) {
    // softmax: thread = (query row r of the unit's tile = TMEM lane r, half hf of the columns)
    const int q4 = warp & 3, r = q4 * 32 + lane, hf = (warp - 4) >> 2;
    const uint32_t lane_base = tmem + ((uint32_t)(q4 * 32) << 16);
    int g = 0, nx = 0;
    // exchange v with the other half of the row; returns the other half's value
    auto exchange = [&](float v, float& other) -> bool {
      const int b = nx & 1;
      ctrl->xval[b][hf][r] = v;
      mbar_arrive(&ctrl->xch[b]);
      const bool ok = warp_wait(&ctrl->xch[b], (nx >> 1) & 1, p.status, abort_flag);
      other = ctrl->xval[b][hf ^ 1][r];
      ++nx;
      return ok;
    };
    for (int u = blockIdx.x; u < p.units; u += gridDim.x) {
      int h, qt, n, p0;
      unit_of(p, u, h, qt, n, p0);
      const int pos = p0 + r;   // this query's position: it sees keys 0..pos
      float m = -INFINITY, l = 0.f;
      for (int j = 0; j < n; ++j, ++g) {
        const int buf = g & 1;
        if (!warp_wait(&ctrl->s_full[buf], (g >> 1) & 1, p.status, abort_flag)) goto done;
        tc_fence_after();
        uint32_t s[2][32];
        tmem_ld32(lane_base + kColS + buf * kFT + hf * 64, s[0]);
        tmem_ld32(lane_base + kColS + buf * kFT + hf * 64 + 32, s[1]);
        tmem_ld_wait();
        if (j * kFT + kFT - 1 > p0) {
          // a tile holding keys after some query of the tile: causal mask
          const int lim = pos - j * kFT - hf * 64;
#pragma unroll
          for (int c = 0; c < 2; ++c)
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (c * 32 + i > lim) s[c][i] = __float_as_uint(-INFINITY);
        }
        // eight independent partial maxima, then the other half's maximum
        float mp[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) mp[k] = -INFINITY;
#pragma unroll
        for (int c = 0; c < 2; ++c)
#pragma unroll
          for (int i = 0; i < 32; ++i) mp[i & 7] = fmaxf(mp[i & 7], __uint_as_float(s[c][i]));
        float mx = fmaxf(fmaxf(fmaxf(mp[0], mp[1]), fmaxf(mp[2], mp[3])), fmaxf(fmaxf(mp[4], mp[5]), fmaxf(mp[6], mp[7])));
        float mo;
        if (!exchange(mx, mo)) goto done;
        mx = fmaxf(mx, mo) * p.scale_log2;   // the positive scale commutes with the maximum
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
        uint32_t pk[32];
        float sp[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) sp[k] = 0.f;
#pragma unroll
        for (int c = 0; c < 2; ++c)
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float e0 = ex2(fmaf(__uint_as_float(s[c][2 * i]), p.scale_log2, -m));
            const float e1 = ex2(fmaf(__uint_as_float(s[c][2 * i + 1]), p.scale_log2, -m));
            const uint32_t w = pack_bf16x2(e0, e1);
            sp[(2 * i) & 7] += __uint_as_float(w << 16);
            sp[(2 * i + 1) & 7] += __uint_as_float(w & 0xFFFF0000u);
            pk[c * 16 + i] = w;
          }
        l += ((sp[0] + sp[1]) + (sp[2] + sp[3])) + ((sp[4] + sp[5]) + (sp[6] + sp[7]));
        // a larger maximum: O is rescaled once the previous P V has finished accumulating into it
        if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
          if (!warp_wait(&ctrl->pv_done[(g - 1) & 1], ((g - 1) >> 1) & 1, p.status, abort_flag)) goto done;
          tc_fence_after();
#pragma unroll 1
          for (int c = 0; c < 2; ++c) {
            uint32_t o[32];
            tmem_ld32(lane_base + kColO + hf * 64 + c * 32, o);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
            tmem_st32(lane_base + kColO + hf * 64 + c * 32, o);
          }
          tmem_st_wait();
        }
        // P row r, keys 64 hf .. 64 hf + 63, as bf16 pairs into columns 32 hf .. 32 hf + 31 of this tile's
        // S buffer (the exchange above ordered it after both halves' loads of S)
        tmem_st32(lane_base + kColS + buf * kFT + hf * 32, pk);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&ctrl->p_full[buf]);
      }
      // epilogue: the full row sum, then O / l in bf16 (this half's 64 columns) and the log-sum-exp
      {
        float lo;
        if (!exchange(l, lo)) goto done;
        l += lo;
      }
      if (!warp_wait(&ctrl->pv_done[(g - 1) & 1], ((g - 1) >> 1) & 1, p.status, abort_flag)) goto done;
      tc_fence_after();
      {
        const float inv = l > 0.f ? 1.f / l : 0.f;
        const int q = qt * kFT + r;
        uint4* dst = reinterpret_cast<uint4*>(p.o + ((long long)q * p.H + h) * kVH + hf * 64);
#pragma unroll 1
        for (int c = 0; c < 2; ++c) {
          uint32_t o[32];
          tmem_ld32(lane_base + kColO + hf * 64 + c * 32, o);
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
        if (hf == 0 && q < p.T && p.lse) p.lse[(long long)q * p.H + h] = l > 0.f ? (m + __log2f(l)) * kLn2 : -INFINITY;
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
// Width of a cache row: the latent and one positional key, or one positional key per head.
int row_width(const mla_config* cfg) { return cfg->d_c + (cfg->rope_per_head ? cfg->n_heads : 1) * cfg->d_rope; }

PrefillLayout prefill_layout(int L, int row_w) {
  PrefillLayout w;
  auto a256 = [](size_t v) { return (v + 255) / 256 * 256; };
  w.lat = 0;
  w.kv = a256((size_t)L * row_w * 2);
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
  return prefill_layout(kv_len, row_width(cfg)).total;
}

cudaError_t tc_prefill_attention(const Ctx& ctx, const mla_config* cfg, const void* q, const mla_paged_cache& cache,
                                 int seq, int kv_len, int T, const void* W_UK, const void* W_UV, float scale, void* o,
                                 float* lse, void* workspace) {
  const int L = kv_len, H = kH, row_w = row_width(cfg);
  const PrefillLayout w = prefill_layout(L, row_w);
  char* base = static_cast<char*>(workspace);
  bf16* lat = reinterpret_cast<bf16*>(base + w.lat);
  bf16* kv = reinterpret_cast<bf16*>(base + w.kv);
  cudaError_t e;
  if (cfg->cache_fp8) {
    e = launch_gather_latent_fp8(ctx, cfg, cache, seq, L, lat);
  } else {
    const dim3 gg((L + kFBlk - 1) / kFBlk, row_w / 64);
    gather_latent_kernel<<<gg, 256, 0, ctx.stream>>>(static_cast<const bf16*>(cache.pool), row_w, cache.block_table,
                                                     cache.max_blocks_per_seq, cache.num_blocks, seq, L, lat,
                                                     ctx.status);
    count_launch();
    e = cudaGetLastError();
  }
  if (e != cudaSuccess) return e;
  e = tc_reconstruct_kv(ctx, cfg, lat, L, W_UK, W_UV, kv);
  if (e != cudaSuccess) return e;
  CUtensorMap mapq, mapkv, mapr;
  const uint64_t dq[3] = {(uint64_t)kQW, (uint64_t)H, (uint64_t)T}, sq[2] = {(uint64_t)kQW * 2, (uint64_t)H * kQW * 2};
  const uint64_t dkv[3] = {64, (uint64_t)L, (uint64_t)4 * H}, skv[2] = {128, (uint64_t)L * 128};
  const uint64_t dr[3] = {64, (uint64_t)L, (uint64_t)row_w / 64}, sr[2] = {128, (uint64_t)L * 128};
  const uint32_t boxq[3] = {64, 1, kFT}, boxc[3] = {64, kFT, 1};
  if (!encode_map_bf16(&mapq, q, 3, dq, sq, boxq) || !encode_map_bf16(&mapkv, kv, 3, dkv, skv, boxc) ||
      !encode_map_bf16(&mapr, lat, 3, dr, sr, boxc))
    return cudaErrorInvalidValue;
  FParams fp;
  fp.T = T;
  fp.L = L;
  fp.q0 = L - T;
  fp.H = H;
  fp.qtiles = (T + kFT - 1) / kFT;
  fp.units = H * fp.qtiles;
  fp.rope_chunk = kDC / 64;
  fp.rope_step = cfg->rope_per_head ? kDR / 64 : 0;
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
