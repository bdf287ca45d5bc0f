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
//   * the score CTA (rank 0) keeps the latent part of the absorbed query in
//     TMEM and its positional part in shared memory, streams the cache in
//     128-token tiles (two blocks) through a ring of 16 KB chunk slots with
//     TMA, computes S = Q K^T with N = 128 MMAs (the tensor core runs N = 64
//     at about 60% of its rate), and runs the online softmax with two threads
//     per head row (one per 64-token half); each half is one unit of bf16 P,
//     staged with its per-row rescale factor in shared memory and shipped to
//     the value CTA's shared memory by one bulk copy;
//   * the value CTA (rank 1) streams the [64 x 512] latent part of every block
//     as two 32 KB halves and accumulates O += P V in all 512 TMEM columns;
//     two warpgroups rescale O when the running maximum jumps (rarely) and
//     write the result.
// The cached tokens of all queries are cut into equal ranges of 128-token
// tiles, one per cluster (split-KV); ranges that cover part of a query write
// fp32 partials that a second kernel merges by log-sum-exp.
#include <math.h>

#include <mutex>

#include "mla_sm100.cuh"
#include "mla_tc.cuh"

namespace mla {
namespace {
using namespace sm100;

constexpr int kH = 128, kDC = 512, kDR = 64, kRow = 576, kBlk = 64;
constexpr int kTile = 2 * kBlk;                     // tokens per score tile: N of the score MMAs
constexpr int kThreads = 384;                       // warps 0-3: TMA, MMA, TMEM, spare; 4-11: two warpgroups
constexpr int kBoxBytes = 64 * 64 * 2;              // one swizzled [64 tokens x 64 elements] box
constexpr int kChunks = kRow / 64;                  // 9 chunks per cached row: 8 latent + 1 positional
constexpr int kSlotK = 2 * kBoxBytes;               // score ring slot: one chunk of a 128-token tile
constexpr int kRing = 10;
constexpr int kSlotV = 4 * kBoxBytes;               // value ring slot: four latent chunks of one block
constexpr int kVRing = 5;
constexpr int kPSlots = 3;                          // P units (64 tokens) in flight to the value CTA
constexpr int kSlotBytes = 18432;                   // P 16 KB | alpha | l (tokens 0-63) | l (64-127) | m
constexpr int kSlotAlpha = 16384, kSlotL0 = 16896, kSlotL1 = 17408, kSlotM = 17920;
constexpr int kCtrlBytes = 4096;
constexpr int kOffQR = kCtrlBytes;                  // score CTA: positional part of Q, [128 rows x 128 B]
constexpr int kOffRing = kOffQR + kH * 128;
constexpr int kOffV = kCtrlBytes;                   // value CTA
constexpr int kOffSlots = kOffV + kVRing * kSlotV;
constexpr int kOffStage = kOffRing + kRing * kSlotK;  // score CTA: each warpgroup's unit of P, laid out as a slot
constexpr int kSmemScore = kOffStage + 2 * kSlotBytes;
constexpr int kSmemValue = kOffSlots + kPSlots * kSlotBytes;
constexpr int kSmemBytes = (kSmemScore > kSmemValue ? kSmemScore : kSmemValue) + 1024;  // + alignment slack
static_assert(kOffRing % 1024 == 0 && kOffSlots % 1024 == 0 && kOffStage % 1024 == 0 && kSlotBytes % 1024 == 0,
              "swizzle alignment");
static_assert(kSmemBytes <= 232448, "shared memory");
constexpr uint32_t kTxUnit = 16384 + 512;
constexpr uint32_t kTxLast = kTxUnit + 1536;
// score CTA TMEM columns: S buffers at 0 and 128, latent Q at 256..511 (64 bf16 per 32 columns)
constexpr int kSCol = 0, kQCol = 256;
constexpr float kRescaleThreshold = 8.0f;            // log2 units: rescale O only when the max grows by 2^8

enum : int { kCmdRescale = 1, kCmdEpilogue = 2, kCmdExit = 3 };

struct Piece {
  int item;     // b * n_q + j
  int t_begin;  // first token (multiple of 128)
  int t_end;    // one past the last token
  int slot;     // partial slot, or -1 when the piece is the whole query
};

struct Ctrl {
  uint64_t k_full[kRing], k_empty[kRing];
  uint64_t s_full[2], s_empty[2];
  uint64_t q_ready;
  uint64_t stage_free[2], stage_full[2];   // per warpgroup: its P staging buffer may be written / is written
  uint64_t xch[2];
  uint64_t p_empty[kPSlots];
  uint64_t v_full[kVRing], v_empty[kVRing];
  uint64_t p_full[kPSlots];
  uint64_t mma_idle, work, done;
  uint32_t tmem_base;
  int abort_flag;
  int cmd, cmd_slot, cmd_piece;
  float l_buf[kH];
  float m_buf[kH];
  float half_max[2][2][kH];   // [tile parity][token half][row]
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

// Maximum of three floats in one instruction.
__device__ __forceinline__ float max3f(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

__device__ __forceinline__ int ceil_div(int a, int b) { return (a + b - 1) / b; }

// Walks a cluster's pieces in steps of `step` tokens.
struct TileCursor {
  int pi, end, t, t_end, b, step;
  __device__ void start(const Piece* pieces, int first, int last, int n_q, int step_) {
    pi = first - 1;
    end = last;
    t = t_end = 0;
    b = 0;
    step = step_;
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
    t += step;
    if (t >= t_end) next_piece(pieces, n_q);
  }
};

// Block-table entries are loaded this many steps before their TMA loads and checked only when used,
// so the latency of the table read never sits in front of a load.
constexpr int kLookahead = 4;

// Table entry `idx` of sequence b, loaded but not yet checked.
__device__ __forceinline__ int table_raw(const Params& p, int b, int idx) {
  return __ldg(p.table + (long long)b * p.max_blocks + idx);
}
// A loaded entry as a physical block (0 and a flag when it is out of range).
__device__ __forceinline__ int checked_block(const Params& p, int blk, bool flag) {
  if (blk < 0 || blk >= p.num_blocks) {
    if (flag) flag_error(p.status, kFlagIndex);
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

// The same for barriers that only this CTA completes (cheaper CTA-scope acquire).
__device__ __forceinline__ bool warp_wait_cta(uint64_t* bar, uint32_t parity, uint32_t* status,
                                              volatile int* abort_flag) {
  const bool ok = mbar_wait_cta(bar, parity, status, abort_flag);
  return __all_sync(0xffffffffu, ok);
}

// ------------------------------------------------------------------ planner
// One CTA of 1024 threads.  Cuts the visible 128-token tiles of all queries into C
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
    const int tiles = i < items ? ceil_div(visible_tokens(kv_len, i, n_q, cap, status, true), kTile) : 0;
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
      pc.t_begin = (int)(a - P0) * kTile;
      pc.t_end = (int)(e - P0) * kTile;
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
    decode_tc_kernel(const __grid_constant__ CUtensorMap map1, const __grid_constant__ CUtensorMap map4, Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  Ctrl* ctrl = reinterpret_cast<Ctrl*>(smem);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_ctarank();
  const int cid = (int)cluster_id_x();
  volatile int* abort_flag = &ctrl->abort_flag;

  if (tid == 0) {
    for (int i = 0; i < kRing; ++i) { mbar_init(&ctrl->k_full[i], 1); mbar_init(&ctrl->k_empty[i], 1); }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&ctrl->s_full[i], 1);
      mbar_init(&ctrl->s_empty[i], 256);
      mbar_init(&ctrl->xch[i], 256);
    }
    mbar_init(&ctrl->q_ready, 256);
    for (int i = 0; i < 2; ++i) { mbar_init(&ctrl->stage_free[i], 1); mbar_init(&ctrl->stage_full[i], 128); }
    for (int i = 0; i < kPSlots; ++i) { mbar_init(&ctrl->p_empty[i], 1); mbar_init(&ctrl->p_full[i], 1); }
    for (int i = 0; i < kVRing; ++i) { mbar_init(&ctrl->v_full[i], 1); mbar_init(&ctrl->v_empty[i], 1); }
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
    prefetch_tmap(&map1);
    prefetch_tmap(&map4);
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem = ctrl->tmem_base;
  const int2 range = p.cluster_range[cid];
  const uint32_t smem_base = smem_u32(smem);
  // warpgroup lanes: warps 4..11, quarter q4 = TMEM lane group, half = which 64 tokens / 256 O columns
  const int q4 = warp & 3, half = (warp - 4) >> 2;
  const int h = q4 * 32 + lane;

  if (rank == 0) {
    // =========================== score CTA ===========================
    if (warp == 0) {
      if (lane == 0) {
        // ring slot = one 64-element chunk of a 128-token tile: chunk c of the tile's first block at +0,
        // of its second block at +8 KB (absent in a one-block tail tile)
        int r = 0;
        uint32_t phase = 0;
        TileCursor ahead;
        ahead.start(p.pieces, range.x, range.y, p.n_q, kTile);
        // raw entries of the next kLookahead tiles; bit u of `live` / `two`: tile u exists / has a second block
        int raw0[kLookahead], raw1[kLookahead];
        uint32_t live = 0, two = 0;
#pragma unroll
        for (int u = 0; u < kLookahead; ++u) {
          raw0[u] = raw1[u] = 0;
          if (ahead.valid()) {
            live |= 1u << u;
            raw0[u] = table_raw(p, ahead.b, ahead.t / kBlk);
            if (ahead.t + kBlk < ahead.t_end) { two |= 1u << u; raw1[u] = table_raw(p, ahead.b, ahead.t / kBlk + 1); }
            ahead.advance(p.pieces, p.n_q);
          }
        }
        while (live & 1u) {
#pragma unroll
          for (int u = 0; u < kLookahead; ++u) {
            if (!(live & (1u << u))) break;
            const int b0 = checked_block(p, raw0[u], true);
            const int b1 = (two & (1u << u)) ? checked_block(p, raw1[u], true) : -1;
            live &= ~(1u << u);
            two &= ~(1u << u);
            if (ahead.valid()) {   // refill this entry with the tile kLookahead steps ahead
              live |= 1u << u;
              raw0[u] = table_raw(p, ahead.b, ahead.t / kBlk);
              if (ahead.t + kBlk < ahead.t_end) { two |= 1u << u; raw1[u] = table_raw(p, ahead.b, ahead.t / kBlk + 1); }
              ahead.advance(p.pieces, p.n_q);
            }
#pragma unroll 1
            for (int c = 0; c < kChunks; ++c) {
              if (!mbar_wait_cta(&ctrl->k_empty[r], phase ^ 1, p.status, abort_flag)) goto score_done;
              uint8_t* dst = smem + kOffRing + r * kSlotK;
              mbar_arrive_expect_tx(&ctrl->k_full[r], b1 >= 0 ? 2 * kBoxBytes : kBoxBytes);
              tma_load_4d(dst, &map1, &ctrl->k_full[r], 0, 0, c, b0);
              if (b1 >= 0) tma_load_4d(dst + kBoxBytes, &map1, &ctrl->k_full[r], 0, 0, c, b1);
              if (++r == kRing) { r = 0; phase ^= 1; }
            }
          }
        }
      }
    } else if (warp == 1) {
      if (lane == 0) {
        // S[128 heads x 128 tokens] = Q K^T over 9 chunks of 4 K-steps; latent chunks take A from TMEM,
        // the positional chunk from shared memory; every chunk's slot is released when its MMAs complete
        const uint32_t idesc = idesc_bf16(128, kTile, false, false);
        const uint64_t ring0 = desc_sw128(smem_base + kOffRing, 16, 1024);
        const uint64_t qr0 = desc_sw128(smem_base + kOffQR, 16, 1024);
        int r = 0, sbuf = 0;
        uint32_t kphase = 0, sphase = 0, qphase = 0;
        for (int pi = range.x; pi < range.y; ++pi) {
          const Piece pc = p.pieces[pi];
          if (pc.t_end <= pc.t_begin) continue;
          if (!mbar_wait(&ctrl->q_ready, qphase, p.status, abort_flag)) goto score_done;
          qphase ^= 1;
          for (int t = pc.t_begin; t < pc.t_end; t += kTile) {
            if (!mbar_wait_cta(&ctrl->s_empty[sbuf], sphase ^ 1, p.status, abort_flag)) goto score_done;
            const uint32_t d = tmem + kSCol + sbuf * kTile;
            // the tile's 9 chunks are accumulated in the order they land (their loads complete out of
            // order), so a late chunk does not hold the slots of the chunks behind it
            uint32_t pending = (1u << kChunks) - 1;
            uint32_t acc = 0;
            const long long t0 = clock64();
            while (pending) {
              bool progress = false;
#pragma unroll
              for (int c = 0; c < kChunks; ++c) {
                if (!(pending & (1u << c))) continue;
                int rc = r + c;
                uint32_t ph = kphase;
                if (rc >= kRing) { rc -= kRing; ph ^= 1; }
                if (!mbar_poll_cta(smem_u32(&ctrl->k_full[rc]), ph)) continue;
                tc_fence_after();
                const uint64_t kd = ring0 + (uint64_t)(rc * (kSlotK >> 4));
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                  if (c < kChunks - 1)
                    mma_ts(d, tmem + kQCol + c * 32 + k * 8, kd + (uint64_t)(k * 2), idesc, (acc | k) ? 1u : 0u);
                  else
                    mma_ss(d, qr0 + (uint64_t)(k * 2), kd + (uint64_t)(k * 2), idesc, (acc | k) ? 1u : 0u);
                }
                acc = 1;
                mma_commit(&ctrl->k_empty[rc]);
                pending &= ~(1u << c);
                progress = true;
              }
              if (!progress) {
                // nothing landed: doze on the oldest outstanding chunk for a moment
                int rc = r + __ffs(pending) - 1;
                uint32_t ph = kphase;
                if (rc >= kRing) { rc -= kRing; ph ^= 1; }
                mbar_test_sleep(smem_u32(&ctrl->k_full[rc]), ph, 200u);
                if (*abort_flag) goto score_done;
                if (clock64() - t0 > kTimeoutCycles) {
                  atomicOr(p.status, kFlagTimeout);
                  *abort_flag = 1;
                  goto score_done;
                }
              }
            }
            r += kChunks;
            if (r >= kRing) { r -= kRing; kphase ^= 1; }
            mma_commit(&ctrl->s_full[sbuf]);
            if (++sbuf == 2) { sbuf = 0; sphase ^= 1; }
          }
        }
      }
    } else if (warp >= 4 && warp < 12) {
      // softmax: head row h, tokens [64*half, 64*half + 64) of each tile, which form one unit of P
      const uint32_t lane_base = tmem + ((uint32_t)(q4 * 32) << 16);
      const uint32_t peer_slots = mapa(smem_base + kOffSlots, 1);
      int sbuf = 0, tile = 0, unit = 0;
      uint32_t sphase = 0, stage_phase = 0;
      for (int pi = range.x; pi < range.y; ++pi) {
        const Piece pc = p.pieces[pi];
        if (pc.t_end <= pc.t_begin) continue;
        {
          // absorbed query row h: latent chunks 4*half .. 4*half+3 -> TMEM; the positional part -> the
          // swizzled shared-memory rows the MMA reads as A
          const uint4* src = reinterpret_cast<const uint4*>(p.q + ((size_t)pc.item * kH + h) * kRow);
#pragma unroll 1
          for (int c = 4 * half; c < 4 * half + 4; ++c) {
            uint32_t r[32];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const uint4 v = __ldg(src + c * 8 + i);
              r[4 * i] = v.x; r[4 * i + 1] = v.y; r[4 * i + 2] = v.z; r[4 * i + 3] = v.w;
            }
            tmem_st32(lane_base + kQCol + c * 32, r);
          }
          if (half == 1) {
            uint8_t* qr = smem + kOffQR + h * 128;
#pragma unroll
            for (int u = 0; u < 8; ++u) *reinterpret_cast<uint4*>(qr + ((u ^ (h & 7)) << 4)) = __ldg(src + 64 + u);
            fence_proxy_async_smem();
          }
          tmem_st_wait();
          tc_fence_before();
          mbar_arrive(&ctrl->q_ready);
        }
        float m = -INFINITY, lpart = 0.f;
        for (int t = pc.t_begin; t < pc.t_end; t += kTile, ++tile) {
          const int ntok = min(kTile, pc.t_end - t);
          const int nunits = ntok > kBlk ? 2 : 1;
          const int valid = ntok - half * kBlk;   // valid columns of this half (may be <= 0)
          const bool first = (t == pc.t_begin), last = (t + kTile >= pc.t_end);
          if (!warp_wait_cta(&ctrl->s_full[sbuf], sphase, p.status, abort_flag)) goto score_done;
          tc_fence_after();
          uint32_t sa[32], sb[32];   // columns 0-31 and 32-63 of this half
          tmem_ld32(lane_base + kSCol + sbuf * kTile + half * kBlk, sa);
          tmem_ld32(lane_base + kSCol + sbuf * kTile + half * kBlk + 32, sb);
          tmem_ld_wait();
          tc_fence_before();
          mbar_arrive(&ctrl->s_empty[sbuf]);
          if (++sbuf == 2) { sbuf = 0; sphase ^= 1; }
          if (valid < kBlk) {
            // columns past the end of the piece (only in its last tile)
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              if (i >= valid) sa[i] = __float_as_uint(-INFINITY);
              if (i + 32 >= valid) sb[i] = __float_as_uint(-INFINITY);
            }
          }
          float mx8[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float t1 = max3f(__uint_as_float(sa[i]), __uint_as_float(sa[i + 8]), __uint_as_float(sa[i + 16]));
            const float t2 = max3f(__uint_as_float(sb[i]), __uint_as_float(sb[i + 8]), __uint_as_float(sb[i + 16]));
            mx8[i] = max3f(max3f(t1, t2, __uint_as_float(sa[i + 24])), __uint_as_float(sb[i + 24]), t1);
          }
          const float hmax = max3f(max3f(mx8[0], mx8[1], mx8[2]), max3f(mx8[3], mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7]));
          // exchange the half-row maxima with the partner thread of the other warpgroup
          ctrl->half_max[tile & 1][half][h] = hmax;
          mbar_arrive(&ctrl->xch[tile & 1]);
          if (!warp_wait_cta(&ctrl->xch[tile & 1], (tile >> 1) & 1, p.status, abort_flag)) goto score_done;
          // raw scores: the positive scale commutes with the maximum
          const float mx = fmaxf(ctrl->half_max[tile & 1][0][h], ctrl->half_max[tile & 1][1][h]) * p.scale_log2;
          float alpha = 1.f;
          if (first) {
            m = mx;
          } else if (mx > m + kRescaleThreshold) {
            alpha = ex2(m - mx);
            lpart *= alpha;
            m = mx;
          }
          uint32_t pk[32];
          // paired fp32 arithmetic: one instruction per two columns for the scaling and the row sum
          const float2 sc2 = make_float2(p.scale_log2, p.scale_log2), nm2 = make_float2(-m, -m);
          float2 ps2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float2 xa = __ffma2_rn(make_float2(__uint_as_float(sa[2 * i]), __uint_as_float(sa[2 * i + 1])), sc2, nm2);
            const float2 xb = __ffma2_rn(make_float2(__uint_as_float(sb[2 * i]), __uint_as_float(sb[2 * i + 1])), sc2, nm2);
            const float2 pa = make_float2(ex2(xa.x), ex2(xa.y)), pb = make_float2(ex2(xb.x), ex2(xb.y));
            ps2[i & 1] = __fadd2_rn(ps2[i & 1], __fadd2_rn(pa, pb));
            pk[i] = pack_bf16x2(pa.x, pa.y);
            pk[16 + i] = pack_bf16x2(pb.x, pb.y);
          }
          lpart += (ps2[0].x + ps2[0].y) + (ps2[1].x + ps2[1].y);
          // this half's unit of P (with its rescale factor and, on a piece's last tile, the row
          // statistics) is written to the warpgroup's staging buffer in the value CTA's slot layout and
          // shipped by one bulk copy: a few large DMA transfers instead of thousands of remote stores,
          // which would hold up the MMA warp's tcgen05 instructions behind them
          uint8_t* stage = smem + kOffStage + half * kSlotBytes;
          const bool leader = (warp & 3) == 0 && lane == 0;
          if (leader) {
            bulk_wait_read_all();            // the previous tile's copies have read the buffer
            mbar_arrive(&ctrl->stage_free[half]);
          }
          if (!warp_wait_cta(&ctrl->stage_free[half], stage_phase, p.status, abort_flag)) goto score_done;
          if (half < nunits) {
#pragma unroll
            for (int c = 0; c < 8; ++c)
              *reinterpret_cast<uint4*>(stage + h * 128 + ((c ^ (h & 7)) << 4)) =
                  make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
            reinterpret_cast<float*>(stage + kSlotAlpha)[h] = half == 0 ? alpha : 1.f;
          }
          if (last) {
            reinterpret_cast<float*>(stage + (half ? kSlotL1 : kSlotL0))[h] = lpart;
            if (half == 0) reinterpret_cast<float*>(stage + kSlotM)[h] = m;
          }
          fence_proxy_async_smem();
          mbar_arrive(&ctrl->stage_full[half]);
          if (leader) {
            if (!mbar_wait_cta(&ctrl->stage_full[half], stage_phase, p.status, abort_flag)) goto score_done;
            if (half < nunits) {
              const int u = unit + half, slot = u % kPSlots;
              if (!mbar_wait(&ctrl->p_empty[slot], ((u / kPSlots) & 1) ^ 1, p.status, abort_flag)) goto score_done;
              bulk_copy_to_peer(peer_slots + slot * kSlotBytes, stage, kSlotAlpha + kH * 4,
                                mapa(smem_u32(&ctrl->p_full[slot]), 1));
            }
            if (last) {
              const int u = unit + nunits - 1, slot = u % kPSlots;
              if (!mbar_wait(&ctrl->p_empty[slot], ((u / kPSlots) & 1) ^ 1, p.status, abort_flag)) goto score_done;
              const uint32_t rbar = mapa(smem_u32(&ctrl->p_full[slot]), 1);
              const int lo = half ? kSlotL1 : kSlotL0;
              bulk_copy_to_peer(peer_slots + slot * kSlotBytes + lo, stage + lo, kH * 4, rbar);
              if (half == 0) bulk_copy_to_peer(peer_slots + slot * kSlotBytes + kSlotM, stage + kSlotM, kH * 4, rbar);
            }
            bulk_commit_group();
          }
          stage_phase ^= 1;
          unit += nunits;
        }
      }
      // the staging buffers must outlive the copies reading them
      if ((warp & 3) == 0 && lane == 0) bulk_wait_all();
    }
  score_done:;
  } else {
    // =========================== value CTA ===========================
    if (warp == 0) {
      if (lane == 0) {
        // ring slot = latent chunks 0-3 or 4-7 of one 64-token block
        int r = 0;
        uint32_t phase = 0;
        TileCursor ahead;
        ahead.start(p.pieces, range.x, range.y, p.n_q, kBlk);
        constexpr int kLA = 2 * kLookahead;   // blocks ahead
        int raw[kLA];
        uint32_t live = 0;
#pragma unroll
        for (int u = 0; u < kLA; ++u) {
          raw[u] = 0;
          if (ahead.valid()) {
            live |= 1u << u;
            raw[u] = table_raw(p, ahead.b, ahead.t / kBlk);
            ahead.advance(p.pieces, p.n_q);
          }
        }
        while (live & 1u) {
#pragma unroll
          for (int u = 0; u < kLA; ++u) {
            if (!(live & (1u << u))) break;
            const int blk = checked_block(p, raw[u], false);
            live &= ~(1u << u);
            if (ahead.valid()) {
              live |= 1u << u;
              raw[u] = table_raw(p, ahead.b, ahead.t / kBlk);
              ahead.advance(p.pieces, p.n_q);
            }
#pragma unroll 1
            for (int nh = 0; nh < 2; ++nh) {
              if (!mbar_wait_cta(&ctrl->v_empty[r], phase ^ 1, p.status, abort_flag)) goto value_done;
              mbar_arrive_expect_tx(&ctrl->v_full[r], kSlotV);
              tma_load_4d(smem + kOffV + r * kSlotV, &map4, &ctrl->v_full[r], 0, 0, 4 * nh, blk);
              if (++r == kVRing) { r = 0; phase ^= 1; }
            }
          }
        }
      }
    } else if (warp == 1) {
      // MMA warp: lane 0 issues, the whole warp waits and zeroes tail rows
      const uint32_t idesc = idesc_bf16(128, 256, false, true);
      const uint64_t pdesc0 = desc_sw128(smem_base + kOffSlots, 16, 1024);
      const uint64_t vdesc0 = desc_sw128(smem_base + kOffV, kBoxBytes, 1024);
      int r = 0, pslot = 0;
      uint32_t vphase = 0, pphase = 0, idle_phase = 0, done_phase = 0;
      for (int pi = range.x; pi < range.y; ++pi) {
        const Piece pc = p.pieces[pi];
        if (pc.t_end <= pc.t_begin) continue;
        for (int t = pc.t_begin; t < pc.t_end; t += kBlk) {
          const int valid = min(kBlk, pc.t_end - t);
          const bool first = (t == pc.t_begin), last = (t + kBlk >= pc.t_end);
          if (lane == 0) mbar_arrive_expect_tx(&ctrl->p_full[pslot], last ? kTxLast : kTxUnit);
          __syncwarp();
          if (!warp_wait(&ctrl->p_full[pslot], pphase, p.status, abort_flag)) goto value_mma_exit;
          uint8_t* slot = smem + kOffSlots + pslot * kSlotBytes;
          // does any row's running max jump on this unit?
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
          __syncwarp();
          if (flag && !first) {
            // the running max jumped: O must be rescaled before this unit accumulates
            if (lane == 0) mma_commit(&ctrl->mma_idle);
            __syncwarp();
            if (!warp_wait_cta(&ctrl->mma_idle, idle_phase, p.status, abort_flag)) goto value_mma_exit;
            idle_phase ^= 1;
            if (lane == 0) {
              ctrl->cmd = kCmdRescale;
              ctrl->cmd_slot = pslot;
              mbar_arrive(&ctrl->work);
            }
            if (!warp_wait_cta(&ctrl->done, done_phase, p.status, abort_flag)) goto value_mma_exit;
            done_phase ^= 1;
          }
#pragma unroll 1
          for (int nh = 0; nh < 2; ++nh) {
            if (!warp_wait_cta(&ctrl->v_full[r], vphase, p.status, abort_flag)) goto value_mma_exit;
            if (valid < kBlk) {
              // tokens past the end of the sequence: zero their rows so 0 * garbage cannot reach O
              uint8_t* vst = smem + kOffV + r * kSlotV;
              const int nrow = kBlk - valid;
              for (int e = lane; e < nrow * 32; e += 32) {
                const int box = e / (nrow * 8), rem = e % (nrow * 8);
                const int row = valid + rem / 8, ch = rem % 8;
                *reinterpret_cast<uint4*>(vst + box * kBoxBytes + row * 128 + ch * 16) = make_uint4(0, 0, 0, 0);
              }
              fence_proxy_async_smem();
              __syncwarp();
            }
            tc_fence_after();
            if (lane == 0) {
              const uint64_t pd = pdesc0 + (uint64_t)(pslot * (kSlotBytes >> 4));
              const uint64_t vd = vdesc0 + (uint64_t)(r * (kSlotV >> 4));
#pragma unroll
              for (int s = 0; s < 4; ++s)
                mma_ss(tmem + nh * 256, pd + (uint64_t)(s * 2), vd + (uint64_t)(s * (2048 >> 4)), idesc,
                       (!first || s > 0) ? 1u : 0u);
              mma_commit(&ctrl->v_empty[r]);
            }
            __syncwarp();
            if (++r == kVRing) { r = 0; vphase ^= 1; }
          }
          if (lane == 0) mma_commit_multicast(&ctrl->p_empty[pslot], 0x1);
          __syncwarp();
          if (++pslot == kPSlots) { pslot = 0; pphase ^= 1; }
        }
        // piece finished: wait for the last accumulation, then hand O to the epilogue
        if (lane == 0) mma_commit(&ctrl->mma_idle);
        __syncwarp();
        if (!warp_wait_cta(&ctrl->mma_idle, idle_phase, p.status, abort_flag)) goto value_mma_exit;
        idle_phase ^= 1;
        if (lane == 0) {
          ctrl->cmd = kCmdEpilogue;
          ctrl->cmd_piece = pi;
          mbar_arrive(&ctrl->work);
        }
        if (!warp_wait_cta(&ctrl->done, done_phase, p.status, abort_flag)) goto value_mma_exit;
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
        if (!warp_wait_cta(&ctrl->work, wphase, p.status, abort_flag)) break;
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
            // partial layout [slot][column / 4][row][4]: each store of a warp fills 512 contiguous bytes
            float4* dst = reinterpret_cast<float4*>(p.part_o) + ((size_t)pc.slot * (kDC / 4) + half * 64) * kH + h;
#pragma unroll 1
            for (int c = 0; c < 8; ++c) {
              uint32_t r[32];
              tmem_ld32(lane_base + c * 32, r);
              tmem_ld_wait();
#pragma unroll
              for (int i = 0; i < 8; ++i)
                dst[(size_t)(c * 8 + i) * kH] =
                    make_float4(__uint_as_float(r[4 * i]) * inv, __uint_as_float(r[4 * i + 1]) * inv,
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
// Block (item, g) merges columns [16 g, 16 g + 16) of all 128 heads; thread = head row.
constexpr int kMergeGroups = kDC / 16;

__global__ void __launch_bounds__(kH) merge_kernel(const Piece* pieces, const int2* item_range, const float* part_o,
                                                   const float* part_lse, bf16* o_lat, float* lse_out) {
  const int item = blockIdx.x, g = blockIdx.y, h = threadIdx.x;
  const int2 r = item_range[item];
  if (r.y == 1) return;  // written directly by the attention kernel
  uint4* dst = reinterpret_cast<uint4*>(o_lat + ((size_t)item * kH + h) * kDC + g * 16);
  if (r.y == 0) {
#pragma unroll
    for (int i = 0; i < 2; ++i) dst[i] = make_uint4(0, 0, 0, 0);
    if (lse_out && g == 0) lse_out[(size_t)item * kH + h] = -INFINITY;
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
    // partial layout [slot][column / 4][row][4]
    const float4* src = reinterpret_cast<const float4*>(part_o) + ((size_t)slot * (kDC / 4) + g * 4) * kH + h;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float4 v = src[(size_t)j * kH];
      acc[4 * j] = fmaf(w, v.x, acc[4 * j]);
      acc[4 * j + 1] = fmaf(w, v.y, acc[4 * j + 1]);
      acc[4 * j + 2] = fmaf(w, v.z, acc[4 * j + 2]);
      acc[4 * j + 3] = fmaf(w, v.w, acc[4 * j + 3]);
    }
  }
  const float inv = 1.f / z;
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    uint4 v;
    v.x = pack_bf16x2(acc[8 * i] * inv, acc[8 * i + 1] * inv);
    v.y = pack_bf16x2(acc[8 * i + 2] * inv, acc[8 * i + 3] * inv);
    v.z = pack_bf16x2(acc[8 * i + 4] * inv, acc[8 * i + 5] * inv);
    v.w = pack_bf16x2(acc[8 * i + 6] * inv, acc[8 * i + 7] * inv);
    dst[i] = v;
  }
  if (lse_out && g == 0) lse_out[(size_t)item * kH + h] = mx + logf(z);
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

  // The pool viewed as [block][64-element chunk][token][element]; a box of 1 or 4 chunks lands
  // as [chunk][token][128 B] with the 128-byte swizzle the MMA descriptors expect.
  CUtensorMap map1, map4;
  const cuuint64_t dims[4] = {64, (cuuint64_t)kBlk, (cuuint64_t)kChunks, (cuuint64_t)cache.num_blocks};
  const cuuint64_t strides[3] = {(cuuint64_t)kRow * 2, 128, (cuuint64_t)kBlk * kRow * 2};
  const cuuint32_t box1[4] = {64, (cuuint32_t)kBlk, 1, 1};
  const cuuint32_t box4[4] = {64, (cuuint32_t)kBlk, 4, 1};
  const cuuint32_t estride[4] = {1, 1, 1, 1};
  if (encode(&map1, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, cache.pool, dims, strides, box1, estride,
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
  decode_tc_kernel<<<2 * C, kThreads, kSmemBytes, ctx.stream>>>(map1, map4, prm);
  count_launch();
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;

  merge_kernel<<<dim3(items, kMergeGroups), kH, 0, ctx.stream>>>(pieces, item_range, prm.part_o, prm.part_lse,
                                                            prm.o_lat, lse);
  count_launch();
  return cudaGetLastError();
}

}  // namespace mla

