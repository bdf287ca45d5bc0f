// Decode attention over the paged latent cache on tcgen05 tensor cores.
//
// Specialised for the DeepSeek-V2 head shapes: 128 heads, d_c = 512,
// d_rope = 64, bf16 storage, 64-token cache blocks.  All heads of a query
// share one pass over the latent cache: heads are the M = 128 rows of every
// MMA, the cached rows are the shared operand ("Why it is not just extra work
// at decode time": attention runs in the latent space after the key
// up-projection is folded into the query).
//
// A full fp32 accumulator O (128 heads x 512) fills all of one SM's tensor
// memory, so each unit of work runs on a cluster of two CTAs:
//   * the score CTA (rank 0) keeps the absorbed query Q [128 x 576] in TMEM,
//     streams [64 tokens x 576] tiles with TMA, computes S = Q K^T (A from
//     TMEM), and runs the online softmax with two threads per head row; it
//     pushes bf16 P (and the per-row rescale factor) into the value CTA's
//     shared memory with st.async;
//   * the value CTA (rank 1) streams the [64 x 512] latent part of the same
//     tiles and accumulates O += P V in all 512 TMEM columns; two warpgroups
//     rescale O when the running maximum jumps (rarely) and write the result.
// The cached tokens of all queries are cut into equal tile ranges, one per
// cluster (split-KV); ranges that cover part of a query write fp32 partials
// that a second kernel merges by log-sum-exp.
#include <math.h>

#include <mutex>

#include "mla_sm100.cuh"
#include "mla_tc.cuh"

namespace mla {
namespace {
using namespace sm100;

constexpr int kH = 128, kDC = 512, kDR = 64, kRow = 576, kBlk = 64;
constexpr int kThreads = 512;  // warps 0-3: TMA, MMA, TMEM, spare; 4-11: two warpgroups; 12-15: P sender
constexpr int kBoxBytes = 64 * 64 * 2;             // one swizzled [64 tokens x 64 elements] chunk
constexpr int kChunks = kRow / 64;                  // 9 chunks per cached row: 8 latent + 1 positional
constexpr int kKStageBytes = kChunks * kBoxBytes;   // score CTA: whole rows (73,728 B)
constexpr int kVStageBytes = 8 * kBoxBytes;         // value CTA: latent part (65,536 B)
constexpr int kKStages = 3;
constexpr int kKSplit = 5;                          // a score stage loads and frees as chunks 0-4 and chunks 5-8
constexpr int kVStages = 2;
constexpr int kPSlots = 3;
constexpr int kSlotBytes = 18432;                   // P 16 KB | alpha | l (cols 0-31) | l (cols 32-63) | m
constexpr int kSlotAlpha = 16384, kSlotL0 = 16896, kSlotL1 = 17408, kSlotM = 17920;
constexpr int kCtrlBytes = 4096;
constexpr int kOffStages = kCtrlBytes;                               // both roles
constexpr int kOffSlots = kOffStages + kVStages * kVStageBytes;     // value CTA
constexpr int kSmemScore = kOffStages + kKStages * kKStageBytes;
constexpr int kSmemValue = kOffSlots + kPSlots * kSlotBytes;
constexpr int kSmemBytes = (kSmemScore > kSmemValue ? kSmemScore : kSmemValue) + 1024;  // + alignment slack
constexpr uint32_t kTxTile = 16384 + 512;
constexpr uint32_t kTxLast = kTxTile + 1536;
// score CTA TMEM columns: S buffers at 0 and 64, Q at 128..415, two staged P tiles at 416 and 448
// (64 bf16 per row packed in 32 columns), per-row alpha / l (two halves) / m of each staged tile at 480 + 4*slot
constexpr int kSCol = 0, kQCol = 128, kPStageCol = 416, kPExtraCol = 480;
constexpr float kRescaleThreshold = 8.0f;            // log2 units: rescale O only when the max grows by 2^8

enum : int { kCmdRescale = 1, kCmdEpilogue = 2, kCmdExit = 3 };

struct Piece {
  int item;     // b * n_q + j
  int t_begin;  // first token (multiple of 64)
  int t_end;    // one past the last token
  int slot;     // partial slot, or -1 when the piece is the whole query
};

struct Ctrl {
  uint64_t k_full[kKStages][2], k_empty[kKStages][2];   // [stage][chunks 0-4 | chunks 5-8]
  uint64_t s_full[2], s_empty[2];
  uint64_t q_ready;
  uint64_t xch[2];
  uint64_t p_staged[2], p_free[2];
  uint64_t p_empty[kPSlots];
  uint64_t v_full[kVStages], v_empty[kVStages];
  uint64_t p_full[kPSlots];
  uint64_t mma_idle, work, done;
  uint32_t tmem_base;
  int abort_flag;
  int cmd, cmd_slot, cmd_piece;
  float l_buf[kH];
  float m_buf[kH];
  float half_max[2][2][kH];   // [tile parity][column half][row]
};
static_assert(sizeof(Ctrl) <= kCtrlBytes, "control block too large");

struct Params {
  const bf16* q;
  const int32_t* table;
  int max_blocks, num_blocks;
  int n_q;
  const Piece* pieces;
  const int2* cluster_range;
  bf16* o_lat;
  float* lse_out;
  float* part_o;
  float* part_lse;
  float scale_log2;
  uint32_t* status;
};

__device__ __forceinline__ int ceil_div(int a, int b) { return (a + b - 1) / b; }

// Walks the tiles of a cluster's pieces in order.
struct TileCursor {
  int pi, end, t, t_end, b;
  __device__ void start(const Piece* pieces, int first, int last, int n_q) {
    pi = first - 1;
    end = last;
    t = t_end = 0;
    b = 0;
    next_piece(pieces, n_q);
  }
  __device__ void next_piece(const Piece* pieces, int n_q) {
    while (++pi < end) {
      const Piece pc = pieces[pi];
      if (pc.t_end > pc.t_begin) {
        t = pc.t_begin;
        t_end = pc.t_end;
        b = pc.item / n_q;
        return;
      }
    }
  }
  __device__ bool valid() const { return pi < end; }
  __device__ void advance(const Piece* pieces, int n_q) {
    t += kBlk;
    if (t >= t_end) next_piece(pieces, n_q);
  }
};

constexpr int kLookahead = 4;   // block-table entries read this many tiles before their loads

// Physical block of the cursor's tile (0 and a flag when the table entry is out of range), or -1 past the end.
__device__ __forceinline__ int block_of(const TileCursor& c, const int32_t* table, int max_blocks, int num_blocks,
                                        uint32_t* status, bool flag) {
  if (!c.valid()) return -1;
  int blk = __ldg(table + (long long)c.b * max_blocks + c.t / kBlk);
  if (blk < 0 || blk >= num_blocks) {
    if (flag) flag_error(status, kFlagIndex);
    blk = 0;
  }
  return blk;
}

// A wait whose outcome is the same for every lane of the warp (tcgen05 loads and
// stores that follow are warp-collective).
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, uint32_t* status, volatile int* abort_flag) {
  const bool ok = mbar_wait(bar, parity, status, abort_flag);
  return __all_sync(0xffffffffu, ok);
}

// ------------------------------------------------------------------ planner
// One CTA of 1024 threads.  Cuts the visible tiles of all queries into C
// equal contiguous ranges (cluster c gets global tiles [c*T/C, (c+1)*T/C))
// and lists the resulting pieces in global tile order.
constexpr int kPlanThreads = 1024;

__device__ int block_scan_excl(int v, int* sh, int& total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) sh[wid] = x;
  __syncthreads();
  if (wid == 0) {
    int w = sh[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    sh[lane] = w;
  }
  __syncthreads();
  const int excl = x - v + (wid > 0 ? sh[wid - 1] : 0);
  total = sh[31];
  __syncthreads();
  return excl;
}

__device__ __forceinline__ int visible_tokens(const int32_t* kv_len, int item, int n_q, int cap, uint32_t* status,
                                              bool flag) {
  const int b = item / n_q, j = item % n_q;
  int kv = kv_len[b];
  if (kv < 0 || kv > cap) {
    if (flag) flag_error(status, kFlagIndex);
    kv = kv < 0 ? 0 : cap;
  }
  const int vis = kv - (n_q - 1 - j);
  return vis > 0 ? vis : 0;
}

__device__ __forceinline__ int cluster_of(long long x, long long T, int C) {
  return (int)(((x + 1) * C + T - 1) / T) - 1;
}

__global__ void __launch_bounds__(kPlanThreads) plan_kernel(const int32_t* kv_len, int items, int n_q, int cap, int C,
                                                            int* prefix, int2* item_range, int* slot_off,
                                                            int2* cluster_range, Piece* pieces, uint32_t* status) {
  __shared__ int sh[32];
  // pass 1: exclusive prefix of visible tiles
  int carry = 0;
  for (int base = 0; base < items; base += kPlanThreads) {
    const int i = base + threadIdx.x;
    const int tiles = i < items ? ceil_div(visible_tokens(kv_len, i, n_q, cap, status, true), kBlk) : 0;
    int tot;
    const int ex = block_scan_excl(tiles, sh, tot);
    if (i < items) prefix[i] = carry + ex;
    carry += tot;
  }
  const long long T = carry;
  if (threadIdx.x == 0) prefix[items] = carry;
  for (int c = threadIdx.x; c < C; c += kPlanThreads) cluster_range[c] = make_int2(0, 0);
  // with fewer tiles than clusters, use one cluster per tile so that no cluster's range is empty
  if (T < C) C = (int)T;
  __syncthreads();
  // pass 2: pieces per query and partial slots
  int carry_p = 0, carry_s = 0;
  for (int base = 0; base < items; base += kPlanThreads) {
    const int i = base + threadIdx.x;
    int np = 0;
    if (i < items) {
      const int P0 = prefix[i], P1 = prefix[i + 1];
      if (P1 > P0) np = cluster_of(P1 - 1, T, C) - cluster_of(P0, T, C) + 1;
    }
    int tp, ts;
    const int ex_p = block_scan_excl(np, sh, tp);
    const int ex_s = block_scan_excl(np > 1 ? np : 0, sh, ts);
    if (i < items) {
      item_range[i] = make_int2(carry_p + ex_p, np);
      slot_off[i] = carry_s + ex_s;
    }
    carry_p += tp;
    carry_s += ts;
  }
  __syncthreads();
  // pass 3: write the pieces and each cluster's [first, end) range
  for (int i = threadIdx.x; i < items; i += kPlanThreads) {
    const int2 r = item_range[i];
    if (r.y == 0) continue;
    const long long P0 = prefix[i], P1 = prefix[i + 1];
    const int vis = visible_tokens(kv_len, i, n_q, cap, status, false);
    const int c0 = cluster_of(P0, T, C);
    for (int k = 0; k < r.y; ++k) {
      const int c = c0 + k;
      const long long lo = (long long)c * T / C, hi = (long long)(c + 1) * T / C;
      const long long a = lo > P0 ? lo : P0, e = hi < P1 ? hi : P1;
      Piece pc;
      pc.item = i;
      pc.t_begin = (int)(a - P0) * kBlk;
      pc.t_end = (int)(e - P0) * kBlk;
      if (pc.t_end > vis) pc.t_end = vis;
      pc.slot = r.y > 1 ? slot_off[i] + k : -1;
      const int idx = r.x + k;
      pieces[idx] = pc;
      if (lo >= P0) cluster_range[c].x = idx;
      if (hi <= P1) cluster_range[c].y = idx + 1;
    }
  }
}

// ------------------------------------------------------------------ attention kernel
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    decode_tc_kernel(const __grid_constant__ CUtensorMap map5, const __grid_constant__ CUtensorMap map4, Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  Ctrl* ctrl = reinterpret_cast<Ctrl*>(smem);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_ctarank();
  const int cid = (int)cluster_id_x();
  volatile int* abort_flag = &ctrl->abort_flag;

  if (tid == 0) {
    for (int i = 0; i < kKStages; ++i)
      for (int j = 0; j < 2; ++j) { mbar_init(&ctrl->k_full[i][j], 1); mbar_init(&ctrl->k_empty[i][j], 1); }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&ctrl->s_full[i], 1);
      mbar_init(&ctrl->s_empty[i], 256);
      mbar_init(&ctrl->xch[i], 256);
      mbar_init(&ctrl->p_staged[i], 256);
      mbar_init(&ctrl->p_free[i], 128);
    }
    mbar_init(&ctrl->q_ready, 256);
    for (int i = 0; i < kPSlots; ++i) { mbar_init(&ctrl->p_empty[i], 1); mbar_init(&ctrl->p_full[i], 1); }
    for (int i = 0; i < kVStages; ++i) { mbar_init(&ctrl->v_full[i], 1); mbar_init(&ctrl->v_empty[i], 1); }
    mbar_init(&ctrl->mma_idle, 1);
    mbar_init(&ctrl->work, 1);
    mbar_init(&ctrl->done, 256);
    ctrl->abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 2) {
    tmem_alloc(&ctrl->tmem_base, 512);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&map5);
    prefetch_tmap(&map4);
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem = ctrl->tmem_base;
  const int2 range = p.cluster_range[cid];
  const uint32_t smem_base = smem_u32(smem);
  // warpgroup lanes: warps 4..11, quarter q = TMEM lane group, half = which 32 columns / 256 O columns
  const int q4 = warp & 3, half = (warp - 4) >> 2;
  const int h = q4 * 32 + lane;

  if (rank == 0) {
    // =========================== score CTA ===========================
    if (warp == 0) {
      if (lane == 0) {
        // block-table entries are read kLookahead tiles ahead so their latency overlaps the stage waits
        int stage = 0;
        uint32_t phase = 0;
        TileCursor ahead;
        ahead.start(p.pieces, range.x, range.y, p.n_q);
        int nb[kLookahead];
#pragma unroll
        for (int i = 0; i < kLookahead; ++i) {
          nb[i] = block_of(ahead, p.table, p.max_blocks, p.num_blocks, p.status, true);
          if (ahead.valid()) ahead.advance(p.pieces, p.n_q);
        }
        bool more = nb[0] >= 0;
        while (more) {
#pragma unroll
          for (int u = 0; u < kLookahead; ++u) {
            const int blk = nb[u];
            if (blk < 0) { more = false; break; }
            nb[u] = block_of(ahead, p.table, p.max_blocks, p.num_blocks, p.status, true);
            if (ahead.valid()) ahead.advance(p.pieces, p.n_q);
            uint8_t* dst = smem + kOffStages + stage * kKStageBytes;
            if (!mbar_wait(&ctrl->k_empty[stage][0], phase ^ 1, p.status, abort_flag)) goto score_done;
            mbar_arrive_expect_tx(&ctrl->k_full[stage][0], kKSplit * kBoxBytes);
            tma_load_4d(dst, &map5, &ctrl->k_full[stage][0], 0, 0, 0, blk);
            if (!mbar_wait(&ctrl->k_empty[stage][1], phase ^ 1, p.status, abort_flag)) goto score_done;
            mbar_arrive_expect_tx(&ctrl->k_full[stage][1], (kChunks - kKSplit) * kBoxBytes);
            tma_load_4d(dst + kKSplit * kBoxBytes, &map4, &ctrl->k_full[stage][1], 0, 0, kKSplit, blk);
            if (++stage == kKStages) { stage = 0; phase ^= 1; }
          }
        }
      }
    } else if (warp == 1) {
      if (lane == 0) {
        const uint32_t idesc = idesc_bf16(128, 64, false, false);
        const uint64_t kdesc0 = desc_sw128(smem_base + kOffStages, 16, 1024);
        int stage = 0, sbuf = 0;
        uint32_t kphase = 0, sphase = 0, qphase = 0;
        for (int pi = range.x; pi < range.y; ++pi) {
          const Piece pc = p.pieces[pi];
          if (pc.t_end <= pc.t_begin) continue;
          if (!mbar_wait(&ctrl->q_ready, qphase, p.status, abort_flag)) goto score_done;
          qphase ^= 1;
          for (int t = pc.t_begin; t < pc.t_end; t += kBlk) {
            if (!mbar_wait(&ctrl->s_empty[sbuf], sphase ^ 1, p.status, abort_flag)) goto score_done;
            const uint64_t kd = kdesc0 + (uint64_t)(stage * (kKStageBytes >> 4));
            const uint32_t d = tmem + kSCol + sbuf * 64;
            // 36 K-steps of 16: chunk s/4 (8 KB apart), 32 B within the 128-B swizzled row;
            // each half of the stage is released as soon as its MMAs complete
            if (!mbar_wait(&ctrl->k_full[stage][0], kphase, p.status, abort_flag)) goto score_done;
            tc_fence_after();
#pragma unroll
            for (int s = 0; s < 4 * kKSplit; ++s)
              mma_ts(d, tmem + kQCol + s * 8, kd + (uint64_t)((s >> 2) * (kBoxBytes >> 4) + (s & 3) * 2), idesc,
                     s > 0 ? 1u : 0u);
            mma_commit(&ctrl->k_empty[stage][0]);
            if (!mbar_wait(&ctrl->k_full[stage][1], kphase, p.status, abort_flag)) goto score_done;
            tc_fence_after();
#pragma unroll
            for (int s = 4 * kKSplit; s < kRow / 16; ++s)
              mma_ts(d, tmem + kQCol + s * 8, kd + (uint64_t)((s >> 2) * (kBoxBytes >> 4) + (s & 3) * 2), idesc, 1u);
            mma_commit(&ctrl->k_empty[stage][1]);
            mma_commit(&ctrl->s_full[sbuf]);
            if (++stage == kKStages) { stage = 0; kphase ^= 1; }
            if (++sbuf == 2) { sbuf = 0; sphase ^= 1; }
          }
        }
      }
    } else if (warp >= 4 && warp < 12) {
      // softmax: head row h, columns [32*half, 32*half + 32) of each tile
      const uint32_t lane_base = tmem + ((uint32_t)(q4 * 32) << 16);
      int sbuf = 0, tile = 0;
      uint32_t sphase = 0;
      for (int pi = range.x; pi < range.y; ++pi) {
        const Piece pc = p.pieces[pi];
        if (pc.t_end <= pc.t_begin) continue;
        {
          // absorbed query row h -> TMEM columns [kQCol, kQCol + 288); chunks 0-4 / 5-8 per half
          const uint4* src = reinterpret_cast<const uint4*>(p.q + ((size_t)pc.item * kH + h) * kRow);
#pragma unroll 1
          for (int c = half * 5; c < (half ? 9 : 5); ++c) {
            uint32_t r[32];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const uint4 v = __ldg(src + c * 8 + i);
              r[4 * i] = v.x; r[4 * i + 1] = v.y; r[4 * i + 2] = v.z; r[4 * i + 3] = v.w;
            }
            tmem_st32(lane_base + kQCol + c * 32, r);
          }
          tmem_st_wait();
          tc_fence_before();
          mbar_arrive(&ctrl->q_ready);
        }
        float m = -INFINITY, lpart = 0.f;
        for (int t = pc.t_begin; t < pc.t_end; t += kBlk, ++tile) {
          const int valid = min(kBlk, pc.t_end - t) - half * 32;   // valid columns in this half (may be <= 0)
          const bool first = (t == pc.t_begin), last = (t + kBlk >= pc.t_end);
          if (!warp_wait(&ctrl->s_full[sbuf], sphase, p.status, abort_flag)) goto score_done;
          tc_fence_after();
          uint32_t sr[32];
          tmem_ld32(lane_base + kSCol + sbuf * 64 + half * 32, sr);
          tmem_ld_wait();
          tc_fence_before();
          mbar_arrive(&ctrl->s_empty[sbuf]);
          if (++sbuf == 2) { sbuf = 0; sphase ^= 1; }
          float x[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) x[i] = i < valid ? __uint_as_float(sr[i]) * p.scale_log2 : -INFINITY;
          float mx8[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) mx8[i] = fmaxf(fmaxf(x[i], x[i + 8]), fmaxf(x[i + 16], x[i + 24]));
          const float hmax = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                                   fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
          // exchange the half-row maxima with the partner thread of the other warpgroup
          ctrl->half_max[tile & 1][half][h] = hmax;
          mbar_arrive(&ctrl->xch[tile & 1]);
          if (!warp_wait(&ctrl->xch[tile & 1], (tile >> 1) & 1, p.status, abort_flag)) goto score_done;
          const float mx = fmaxf(ctrl->half_max[tile & 1][0][h], ctrl->half_max[tile & 1][1][h]);
          float alpha = 1.f;
          if (first) {
            m = mx;
          } else if (mx > m + kRescaleThreshold) {
            alpha = ex2(m - mx);
            lpart *= alpha;
            m = mx;
          }
          uint32_t pk[16];
          float ps[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float p0 = ex2(x[2 * i] - m), p1 = ex2(x[2 * i + 1] - m);
            ps[i & 3] += p0 + p1;
            pk[i] = pack_bf16x2(p0, p1);
          }
          lpart += (ps[0] + ps[1]) + (ps[2] + ps[3]);
          // stage P and the row statistics in TMEM; the sender warpgroup pushes them to the value CTA
          const int st = tile & 1;
          if (!warp_wait(&ctrl->p_free[st], ((tile >> 1) & 1) ^ 1, p.status, abort_flag)) goto score_done;
          tc_fence_after();
          tmem_st16(lane_base + kPStageCol + st * 32 + half * 16, pk);
          if (half == 0) {
            tmem_st1(lane_base + kPExtraCol + st * 4 + 0, __float_as_uint(alpha));
            tmem_st1(lane_base + kPExtraCol + st * 4 + 1, __float_as_uint(lpart));
            tmem_st1(lane_base + kPExtraCol + st * 4 + 3, __float_as_uint(m));
          } else {
            tmem_st1(lane_base + kPExtraCol + st * 4 + 2, __float_as_uint(lpart));
          }
          tmem_st_wait();
          tc_fence_before();
          mbar_arrive(&ctrl->p_staged[st]);
        }
      }
    } else if (warp >= 12) {
      // P sender: TMEM-staged tiles -> value CTA slots (st.async), row h = lane of this warp's quarter
      const int hs = (warp & 3) * 32 + lane;
      const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) * 32) << 16);
      const uint32_t peer_slots = mapa(smem_base + kOffSlots, 1);
      int pslot = 0, tile = 0;
      uint32_t pphase = 0;
      for (int pi = range.x; pi < range.y; ++pi) {
        const Piece pc = p.pieces[pi];
        if (pc.t_end <= pc.t_begin) continue;
        for (int t = pc.t_begin; t < pc.t_end; t += kBlk, ++tile) {
          const bool last = (t + kBlk >= pc.t_end);
          const int st = tile & 1;
          if (!warp_wait(&ctrl->p_staged[st], (tile >> 1) & 1, p.status, abort_flag)) goto score_done;
          tc_fence_after();
          uint32_t pk[32], ex[4];
          tmem_ld32(lane_base + kPStageCol + st * 32, pk);
          tmem_ld4(lane_base + kPExtraCol + st * 4, ex);
          tmem_ld_wait();
          tc_fence_before();
          mbar_arrive(&ctrl->p_free[st]);
          if (!warp_wait(&ctrl->p_empty[pslot], pphase ^ 1, p.status, abort_flag)) goto score_done;
          const uint32_t slot = peer_slots + pslot * kSlotBytes;
          const uint32_t rbar = mapa(smem_u32(&ctrl->p_full[pslot]), 1);
#pragma unroll
          for (int c = 0; c < 8; ++c)
            st_async_v4(slot + hs * 128 + ((c ^ (hs & 7)) << 4), pk[4 * c], pk[4 * c + 1], pk[4 * c + 2],
                        pk[4 * c + 3], rbar);
          st_async_b32(slot + kSlotAlpha + 4 * hs, ex[0], rbar);
          if (last) {
            st_async_b32(slot + kSlotL0 + 4 * hs, ex[1], rbar);
            st_async_b32(slot + kSlotL1 + 4 * hs, ex[2], rbar);
            st_async_b32(slot + kSlotM + 4 * hs, ex[3], rbar);
          }
          if (++pslot == kPSlots) { pslot = 0; pphase ^= 1; }
        }
      }
    }
  score_done:;
  } else {
    // =========================== value CTA ===========================
    if (warp == 0) {
      if (lane == 0) {
        int stage = 0;
        uint32_t phase = 0;
        TileCursor ahead;
        ahead.start(p.pieces, range.x, range.y, p.n_q);
        int nb[kLookahead];
#pragma unroll
        for (int i = 0; i < kLookahead; ++i) {
          nb[i] = block_of(ahead, p.table, p.max_blocks, p.num_blocks, p.status, false);
          if (ahead.valid()) ahead.advance(p.pieces, p.n_q);
        }
        bool more = nb[0] >= 0;
        while (more) {
#pragma unroll
          for (int u = 0; u < kLookahead; ++u) {
            const int blk = nb[u];
            if (blk < 0) { more = false; break; }
            nb[u] = block_of(ahead, p.table, p.max_blocks, p.num_blocks, p.status, false);
            if (ahead.valid()) ahead.advance(p.pieces, p.n_q);
            if (!mbar_wait(&ctrl->v_empty[stage], phase ^ 1, p.status, abort_flag)) goto value_done;
            mbar_arrive_expect_tx(&ctrl->v_full[stage], kVStageBytes);
            tma_load_4d(smem + kOffStages + stage * kVStageBytes, &map4, &ctrl->v_full[stage], 0, 0, 0, blk);
            tma_load_4d(smem + kOffStages + stage * kVStageBytes + 4 * kBoxBytes, &map4, &ctrl->v_full[stage], 0, 0, 4,
                        blk);
            if (++stage == kVStages) { stage = 0; phase ^= 1; }
          }
        }
      }
    } else if (warp == 1) {
      // MMA warp: lane 0 issues, the whole warp waits and zeroes tail rows
      const uint32_t idesc = idesc_bf16(128, 256, false, true);
      const uint64_t pdesc0 = desc_sw128(smem_base + kOffSlots, 16, 1024);
      const uint64_t vdesc0 = desc_sw128(smem_base + kOffStages, kBoxBytes, 1024);
      int vstage = 0, pslot = 0;
      uint32_t vphase = 0, pphase = 0, idle_phase = 0, done_phase = 0;
      for (int pi = range.x; pi < range.y; ++pi) {
        const Piece pc = p.pieces[pi];
        if (pc.t_end <= pc.t_begin) continue;
        for (int t = pc.t_begin; t < pc.t_end; t += kBlk) {
          const int valid = min(kBlk, pc.t_end - t);
          const bool first = (t == pc.t_begin), last = (t + kBlk >= pc.t_end);
          if (!warp_wait(&ctrl->v_full[vstage], vphase, p.status, abort_flag)) goto value_mma_exit;
          if (lane == 0) mbar_arrive_expect_tx(&ctrl->p_full[pslot], last ? kTxLast : kTxTile);
          __syncwarp();
          if (!warp_wait(&ctrl->p_full[pslot], pphase, p.status, abort_flag)) goto value_mma_exit;
          uint8_t* vst = smem + kOffStages + vstage * kVStageBytes;
          uint8_t* slot = smem + kOffSlots + pslot * kSlotBytes;
          if (valid < kBlk) {
            // tokens past the end of the sequence: zero their rows so 0 * garbage cannot reach O
            const int nrow = kBlk - valid;
            for (int e = lane; e < nrow * 64; e += 32) {
              const int box = e / (nrow * 8), rem = e % (nrow * 8);
              const int row = valid + rem / 8, ch = rem % 8;
              *reinterpret_cast<uint4*>(vst + box * kBoxBytes + row * 128 + ch * 16) = make_uint4(0, 0, 0, 0);
            }
          }
          // does any row's running max jump on this tile?
          const float* alphas = reinterpret_cast<const float*>(slot + kSlotAlpha);
          const bool flag = __any_sync(0xffffffffu, alphas[lane] != 1.f || alphas[lane + 32] != 1.f ||
                                                        alphas[lane + 64] != 1.f || alphas[lane + 96] != 1.f);
          if (last) {
            const float* l0 = reinterpret_cast<const float*>(slot + kSlotL0);
            const float* l1 = reinterpret_cast<const float*>(slot + kSlotL1);
            const float* mm = reinterpret_cast<const float*>(slot + kSlotM);
            for (int i = lane; i < kH; i += 32) {
              ctrl->l_buf[i] = l0[i] + l1[i];
              ctrl->m_buf[i] = mm[i];
            }
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (flag && !first) {
            // the running max jumped: O must be rescaled before this tile accumulates
            if (lane == 0) mma_commit(&ctrl->mma_idle);
            __syncwarp();
            if (!warp_wait(&ctrl->mma_idle, idle_phase, p.status, abort_flag)) goto value_mma_exit;
            idle_phase ^= 1;
            if (lane == 0) {
              ctrl->cmd = kCmdRescale;
              ctrl->cmd_slot = pslot;
              mbar_arrive(&ctrl->work);
            }
            if (!warp_wait(&ctrl->done, done_phase, p.status, abort_flag)) goto value_mma_exit;
            done_phase ^= 1;
          }
          tc_fence_after();
          if (lane == 0) {
            const uint64_t pd = pdesc0 + (uint64_t)(pslot * (kSlotBytes >> 4));
            const uint64_t vd = vdesc0 + (uint64_t)(vstage * (kVStageBytes >> 4));
#pragma unroll
            for (int s = 0; s < 4; ++s)
#pragma unroll
              for (int nh = 0; nh < 2; ++nh)
                mma_ss(tmem + nh * 256, pd + (uint64_t)(s * 2),
                       vd + (uint64_t)(nh * 4 * (kBoxBytes >> 4) + s * (2048 >> 4)), idesc,
                       (!first || s > 0) ? 1u : 0u);
            mma_commit(&ctrl->v_empty[vstage]);
            mma_commit_multicast(&ctrl->p_empty[pslot], 0x1);
          }
          __syncwarp();
          if (++vstage == kVStages) { vstage = 0; vphase ^= 1; }
          if (++pslot == kPSlots) { pslot = 0; pphase ^= 1; }
        }
        // piece finished: wait for the last accumulation, then hand O to the epilogue
        if (lane == 0) mma_commit(&ctrl->mma_idle);
        __syncwarp();
        if (!warp_wait(&ctrl->mma_idle, idle_phase, p.status, abort_flag)) goto value_mma_exit;
        idle_phase ^= 1;
        if (lane == 0) {
          ctrl->cmd = kCmdEpilogue;
          ctrl->cmd_piece = pi;
          mbar_arrive(&ctrl->work);
        }
        if (!warp_wait(&ctrl->done, done_phase, p.status, abort_flag)) goto value_mma_exit;
        done_phase ^= 1;
      }
    value_mma_exit:
      if (lane == 0) {
        ctrl->cmd = kCmdExit;
        mbar_arrive(&ctrl->work);
      }
    } else if (warp >= 4 && warp < 12) {
      // rescale / epilogue: O row h, columns [256*half, 256*half + 256)
      const uint32_t lane_base = tmem + ((uint32_t)(q4 * 32) << 16) + half * 256;
      uint32_t wphase = 0;
      while (true) {
        if (!warp_wait(&ctrl->work, wphase, p.status, abort_flag)) break;
        wphase ^= 1;
        const int cmd = *reinterpret_cast<volatile int*>(&ctrl->cmd);
        if (cmd == kCmdExit) break;
        tc_fence_after();
        if (cmd == kCmdRescale) {
          const float alpha =
              reinterpret_cast<const float*>(smem + kOffSlots + ctrl->cmd_slot * kSlotBytes + kSlotAlpha)[h];
          const bool need = __any_sync(0xffffffffu, alpha != 1.f);
          if (need) {
#pragma unroll 1
            for (int c = 0; c < 8; ++c) {
              uint32_t r[32];
              tmem_ld32(lane_base + c * 32, r);
              tmem_ld_wait();
#pragma unroll
              for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
              tmem_st32(lane_base + c * 32, r);
            }
            tmem_st_wait();
          }
        } else {
          const Piece pc = p.pieces[ctrl->cmd_piece];
          const float l = ctrl->l_buf[h], mrow = ctrl->m_buf[h];
          const float inv = l > 0.f ? 1.f / l : 0.f;
          const float lse = l > 0.f ? (mrow + __log2f(l)) * kLn2 : -INFINITY;
          if (pc.slot < 0) {
            uint4* dst = reinterpret_cast<uint4*>(p.o_lat + ((size_t)pc.item * kH + h) * kDC + half * 256);
#pragma unroll 1
            for (int c = 0; c < 8; ++c) {
              uint32_t r[32];
              tmem_ld32(lane_base + c * 32, r);
              tmem_ld_wait();
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                uint4 v;
                v.x = pack_bf16x2(__uint_as_float(r[8 * i + 0]) * inv, __uint_as_float(r[8 * i + 1]) * inv);
                v.y = pack_bf16x2(__uint_as_float(r[8 * i + 2]) * inv, __uint_as_float(r[8 * i + 3]) * inv);
                v.z = pack_bf16x2(__uint_as_float(r[8 * i + 4]) * inv, __uint_as_float(r[8 * i + 5]) * inv);
                v.w = pack_bf16x2(__uint_as_float(r[8 * i + 6]) * inv, __uint_as_float(r[8 * i + 7]) * inv);
                dst[c * 4 + i] = v;
              }
            }
            if (p.lse_out && half == 0) p.lse_out[(size_t)pc.item * kH + h] = lse;
          } else {
            float4* dst = reinterpret_cast<float4*>(p.part_o + ((size_t)pc.slot * kH + h) * kDC + half * 256);
#pragma unroll 1
            for (int c = 0; c < 8; ++c) {
              uint32_t r[32];
              tmem_ld32(lane_base + c * 32, r);
              tmem_ld_wait();
#pragma unroll
              for (int i = 0; i < 8; ++i)
                dst[c * 8 + i] = make_float4(__uint_as_float(r[4 * i]) * inv, __uint_as_float(r[4 * i + 1]) * inv,
                                             __uint_as_float(r[4 * i + 2]) * inv, __uint_as_float(r[4 * i + 3]) * inv);
            }
            if (half == 0) p.part_lse[(size_t)pc.slot * kH + h] = lse;
          }
        }
        tc_fence_before();
        mbar_arrive(&ctrl->done);
      }
    }
  value_done:;
  }

  // ------------------------------------------------------------------ teardown
  tc_fence_before();
  __syncthreads();
  if (*abort_flag && warp == 0 && lane == 0) {
    // let any copy still in flight land before the CTA's shared memory goes away
    const long long t0 = clock64();
    while (clock64() - t0 < 2000000LL) { }
  }
  cluster_sync();
  tc_fence_after();
  if (warp == 2) tmem_dealloc(tmem, 512);
}

// ------------------------------------------------------------------ split merge
__global__ void __launch_bounds__(128) merge_kernel(const Piece* pieces, const int2* item_range, const float* part_o,
                                                    const float* part_lse, bf16* o_lat, float* lse_out) {
  const int item = blockIdx.x;
  const int2 r = item_range[item];
  if (r.y == 1) return;  // written directly by the attention kernel
  const int h = blockIdx.y * 4 + threadIdx.x / 32, lane = threadIdx.x & 31;
  bf16* dst = o_lat + ((size_t)item * kH + h) * kDC;
  if (r.y == 0) {
    for (int i = lane; i < kDC; i += 32) dst[i] = __float2bfloat16_rn(0.f);
    if (lse_out && lane == 0) lse_out[(size_t)item * kH + h] = -INFINITY;
    return;
  }
  float mx = -INFINITY;
  for (int k = 0; k < r.y; ++k) mx = fmaxf(mx, part_lse[(size_t)pieces[r.x + k].slot * kH + h]);
  float z = 0.f;
  float acc[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) acc[i] = 0.f;
  for (int k = 0; k < r.y; ++k) {
    const int slot = pieces[r.x + k].slot;
    const float w = expf(part_lse[(size_t)slot * kH + h] - mx);
    z += w;
    const float4* src = reinterpret_cast<const float4*>(part_o + ((size_t)slot * kH + h) * kDC);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float4 v = src[lane + 32 * i];
      acc[4 * i] = fmaf(w, v.x, acc[4 * i]);
      acc[4 * i + 1] = fmaf(w, v.y, acc[4 * i + 1]);
      acc[4 * i + 2] = fmaf(w, v.z, acc[4 * i + 2]);
      acc[4 * i + 3] = fmaf(w, v.w, acc[4 * i + 3]);
    }
  }
  const float inv = 1.f / z;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int e = 4 * (lane + 32 * i);
    __nv_bfloat162* d2 = reinterpret_cast<__nv_bfloat162*>(dst + e);
    d2[0] = __floats2bfloat162_rn(acc[4 * i] * inv, acc[4 * i + 1] * inv);
    d2[1] = __floats2bfloat162_rn(acc[4 * i + 2] * inv, acc[4 * i + 3] * inv);
  }
  if (lse_out && lane == 0) lse_out[(size_t)item * kH + h] = mx + logf(z);
}

// ------------------------------------------------------------------ host side
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

std::mutex g_mutex;
EncodeTiledFn g_encode = nullptr;
int g_clusters[64] = {};

EncodeTiledFn encode_fn() {
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  }
  return g_encode;
}

// Number of clusters that can be resident at once (one CTA per SM).
int cluster_count(int device, int sm_count) {
  {
    std::lock_guard<std::mutex> lock(g_mutex);
    if (device >= 0 && device < 64 && g_clusters[device] > 0) return g_clusters[device];
  }
  int n = sm_count / 2;
  if (ensure_smem_limit((const void*)decode_tc_kernel, kSmemBytes, device) == cudaSuccess) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * n, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = kSmemBytes;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = 2;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int k = 0;
    if (cudaOccupancyMaxActiveClusters(&k, decode_tc_kernel, &cfg) == cudaSuccess && k > 0 && k < n) n = k;
  }
  cudaGetLastError();
  std::lock_guard<std::mutex> lock(g_mutex);
  if (device >= 0 && device < 64) g_clusters[device] = n;
  return n;
}

struct WsLayout {
  size_t prefix, item_range, slot_off, cluster_range, pieces, part_o, part_lse, total;
};

WsLayout ws_layout(int items, int C) {
  WsLayout w;
  size_t o = 0;
  auto take = [&](size_t bytes) { size_t r = o; o = (o + bytes + 255) / 256 * 256; return r; };
  w.prefix = take(sizeof(int) * (items + 1));
  w.item_range = take(sizeof(int2) * items);
  w.slot_off = take(sizeof(int) * items);
  w.cluster_range = take(sizeof(int2) * C);
  w.pieces = take(sizeof(Piece) * (items + C));
  w.part_o = take(sizeof(float) * (size_t)2 * C * kH * kDC);
  w.part_lse = take(sizeof(float) * (size_t)2 * C * kH);
  w.total = o;
  return w;
}

}  // namespace

bool tc_decode_supported(const mla_config* cfg, int batch, int n_q) {
  return cfg->dtype == MLA_BF16 && cfg->n_heads == kH && cfg->d_c == kDC && cfg->d_rope == kDR &&
         cfg->block_size == kBlk && batch > 0 && n_q > 0 && (long long)batch * n_q < (1LL << 24);
}

size_t tc_decode_workspace_bytes(const mla_config* cfg, int batch, int n_q, int max_blocks, int sm_count) {
  if (!tc_decode_supported(cfg, batch, n_q)) return 0;
  (void)max_blocks;
  return ws_layout(batch * n_q, sm_count / 2).total;
}

cudaError_t tc_decode_attention(const Ctx& ctx, const mla_config* cfg, const void* q, const mla_paged_cache& cache,
                                const int32_t* kv_len, int batch, int n_q, float scale, void* o_lat, float* lse,
                                void* workspace) {
  EncodeTiledFn encode = encode_fn();
  if (!encode) return cudaErrorNotSupported;
  const int C = cluster_count(ctx.device, ctx.sm_count);
  const int items = batch * n_q;
  const WsLayout w = ws_layout(items, ctx.sm_count / 2);
  char* ws = static_cast<char*>(workspace);
  int* prefix = reinterpret_cast<int*>(ws + w.prefix);
  int2* item_range = reinterpret_cast<int2*>(ws + w.item_range);
  int* slot_off = reinterpret_cast<int*>(ws + w.slot_off);
  int2* cluster_range = reinterpret_cast<int2*>(ws + w.cluster_range);
  Piece* pieces = reinterpret_cast<Piece*>(ws + w.pieces);

  // The pool viewed as [block][64-element chunk][token][element]; a box of 5 or 4 chunks lands
  // as [chunk][token][128 B] with the 128-byte swizzle the MMA descriptors expect.
  CUtensorMap map5, map4;
  const cuuint64_t dims[4] = {64, (cuuint64_t)kBlk, (cuuint64_t)kChunks, (cuuint64_t)cache.num_blocks};
  const cuuint64_t strides[3] = {(cuuint64_t)kRow * 2, 128, (cuuint64_t)kBlk * kRow * 2};
  const cuuint32_t box5[4] = {64, (cuuint32_t)kBlk, (cuuint32_t)kKSplit, 1};
  const cuuint32_t box4[4] = {64, (cuuint32_t)kBlk, 4, 1};
  const cuuint32_t estride[4] = {1, 1, 1, 1};
  if (encode(&map5, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, cache.pool, dims, strides, box5, estride,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS ||
      encode(&map4, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, cache.pool, dims, strides, box4, estride,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;

  const int cap = cache.max_blocks_per_seq * kBlk;
  plan_kernel<<<1, kPlanThreads, 0, ctx.stream>>>(kv_len, items, n_q, cap, C, prefix, item_range, slot_off,
                                                 cluster_range, pieces, ctx.status);
  count_launch();
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;

  Params prm;
  prm.q = static_cast<const bf16*>(q);
  prm.table = cache.block_table;
  prm.max_blocks = cache.max_blocks_per_seq;
  prm.num_blocks = cache.num_blocks;
  prm.n_q = n_q;
  prm.pieces = pieces;
  prm.cluster_range = cluster_range;
  prm.o_lat = static_cast<bf16*>(o_lat);
  prm.lse_out = lse;
  prm.part_o = reinterpret_cast<float*>(ws + w.part_o);
  prm.part_lse = reinterpret_cast<float*>(ws + w.part_lse);
  prm.scale_log2 = scale * kLog2e;
  prm.status = ctx.status;
  e = ensure_smem_limit((const void*)decode_tc_kernel, kSmemBytes, ctx.device);
  if (e != cudaSuccess) return e;
  decode_tc_kernel<<<2 * C, kThreads, kSmemBytes, ctx.stream>>>(map5, map4, prm);
  count_launch();
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;

  merge_kernel<<<dim3(items, kH / 4), 128, 0, ctx.stream>>>(pieces, item_range, prm.part_o, prm.part_lse,
                                                            prm.o_lat, lse);
  count_launch();
  return cudaGetLastError();
}

}  // namespace mla

