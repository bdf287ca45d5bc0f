// Decode attention over the paged latent cache on tcgen05 tensor cores.
//
// Specialised for the DeepSeek-V2 head shapes: 128 heads, d_c = 512,
// d_rope = 64, bf16 storage, 64-token cache blocks.  All heads of a query
// share one pass over the latent cache: heads are the M = 128 rows of every
// MMA, the cached rows are the shared operand ("Why it is not just extra work
// at decode time": attention runs in the latent space after the key
// up-projection is folded into the query).
//
// The pool stores every block transposed, [576 elements][64 tokens], so one TMA
// box carries a contiguous run of element rows of a block, and the rows serve
// as either MMA operand layout: tokens-contiguous (MN-major) B for the scores,
// K-major B for the values.
//
// A full fp32 accumulator O (128 heads x 512) fills all of one SM's tensor
// memory, so each unit of work runs on a cluster of two CTAs:
//   * the score CTA (rank 0) streams the cache in 128-token tiles (two blocks,
//     joined through the B descriptor's leading byte offset) through a ring of
//     24 KB slots and computes S = Q K^T with N = 128 MMAs issued from
//     compile-time operand offsets; the absorbed query of each piece arrives by
//     TMA through the same ring and is copied into tensor memory with
//     tcgen05.cp behind the previous piece's MMAs (its positional part goes to
//     shared memory, gated by a free/full barrier pair); two threads per head
//     row run the online softmax, and each 64-token unit of bf16 P is staged
//     with its rescale factor and shipped to the value CTA by one bulk copy;
//   * the value CTA (rank 1) streams the 512 latent rows of every block as two
//     32 KB boxes and accumulates O += P V in all 512 TMEM columns; two
//     warpgroups rescale O when the running maximum jumps (rarely) and write
//     the result.
// Every cluster plans its own work in its prologue: the visible 128-token tiles
// of all queries are cut into equal contiguous ranges, one per cluster
// (split-KV); ranges that cover part of a query write fp32 partials that a
// second kernel, launched as a programmatic dependent, merges by log-sum-exp.
#include <cuda_fp16.h>
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
// The pool stores each block transposed, [576 elements][64 tokens] (128 B per element row), so a TMA box
// of whole element rows is one contiguous run of the block.
constexpr int kE = 96;                              // elements per score-ring box: 6 boxes cover a block
constexpr int kSlotsPerTile = kRow / kE;            // ring slots per 128-token tile
constexpr int kBoxK = kE * 128;                     // one block's kE element rows (12 KB)
constexpr int kSlotK = 2 * kBoxK;                   // score ring slot: the same rows of the tile's two blocks
constexpr int kRing = 7;
constexpr int kVRows = 256;                         // latent rows per value box: the N of one P.V MMA group
constexpr int kSlotV = kVRows * 128;                // value ring slot (32 KB)
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
static_assert(kRow % kE == 0 && kE % 16 == 0 && kDC % 16 == 0, "score slots hold whole K-steps");
static_assert(kOffRing % 1024 == 0 && kOffSlots % 1024 == 0 && kOffStage % 1024 == 0 && kSlotBytes % 1024 == 0 &&
                  kBoxK % 1024 == 0 && kSlotV % 1024 == 0,
              "swizzle alignment");
static_assert(kSmemBytes <= 232448, "shared memory");
constexpr uint32_t kTxUnit = 16384 + 512;
constexpr uint32_t kTxLast = kTxUnit + 1536;
// score CTA TMEM columns: S buffers at 0 and 128, latent Q at 256..511 (64 bf16 per 32 columns)
constexpr int kSCol = 0, kQCol = 256;
constexpr float kRescaleThreshold = 8.0f;            // log2 units: rescale O only when the max grows by 2^8

constexpr int kQChunks = kDC / 64;                  // latent query chunks of 64 columns per piece
constexpr uint32_t kQChunkBytes = kH * 128;          // one chunk: [128 heads][64 bf16] (16 KB)
static_assert(kQChunkBytes <= (uint32_t)kSlotK, "a query chunk travels in one score-ring slot");

enum : int { kCmdRescale = 1, kCmdEpilogue = 2, kCmdZero = 3, kCmdExit = 4 };

// A contiguous range of one query's visible tokens processed by one cluster.
struct Piece {
  int item;     // b * n_q + j
  int t_begin;  // first token (multiple of 128)
  int t_end;    // one past the last token (== t_begin: the query sees nothing)
  int slot;     // partial slot, or -1 when the piece is the whole query
};

struct Ctrl {
  uint64_t k_full[kRing], k_empty[kRing];
  uint64_t s_full[2], s_empty[2];
  uint64_t qr_full, qr_free;               // positional query part in shared memory: loaded / free again
  uint64_t stage_free[2], stage_full[2];   // per warpgroup: its P staging buffer may be written / is written
  uint64_t xch[2];
  uint64_t p_empty[kPSlots];
  uint64_t v_full[kVRing], v_empty[kVRing];
  uint64_t p_full[kPSlots];
  uint64_t mma_idle, work, done;
  uint32_t tmem_base;
  int abort_flag;
  int cmd, cmd_slot;
  Piece cmd_piece;
  // this cluster's share of the tiles, [lo, hi), and where its scan of the queries starts
  int plan_lo, plan_hi, plan_item, plan_prefix, plan_total, plan_last;
  float l_buf[kH];
  float m_buf[kH];
  float half_max[2][2][kH];   // [tile parity][token half][row]
};
static_assert(sizeof(Ctrl) <= kCtrlBytes, "control block too large");

struct Params {
  const bf16* q;
  const int32_t* table;
  const int32_t* kv_len;
  int max_blocks, num_blocks;
  int n_q, items, cap;        // cap = max_blocks * block size
  int* prefix;                // [items + 1]: exclusive prefix of visible tiles (written by CTA 0)
  bf16* o_lat;
  float* lse_out;
  __half* part_o;               // [2 clusters][kDC / 8][kH][8] fp16
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

// ------------------------------------------------------------------ work plan
// The visible 128-token tiles of all queries, in query order, are cut into C equal contiguous ranges,
// one per cluster: cluster c takes global tiles [c T / C, (c + 1) T / C) (C = min(clusters, T)).  A
// query with nothing visible belongs to the cluster whose range holds its position in that order (the
// last cluster when it sits at the end).  A piece that covers part of a query writes a partial into
// slot 2c when it continues a query begun by an earlier cluster, else into slot 2c + 1.

__device__ __forceinline__ int visible_tokens(const Params& p, int item, bool flag) {
  const int b = item / p.n_q, j = item - b * p.n_q;
  int kv = __ldg(p.kv_len + b);
  if (kv < 0 || kv > p.cap) {
    if (flag) flag_error(p.status, kFlagIndex);
    kv = kv < 0 ? 0 : p.cap;
  }
  const int vis = kv - (p.n_q - 1 - j);
  return vis > 0 ? vis : 0;
}

__device__ __forceinline__ int cluster_of(long long x, long long T, int C) {
  return (int)(((x + 1) * C + T - 1) / T) - 1;
}

// Inclusive prefix sum across the warp.
__device__ __forceinline__ int warp_scan_incl(int v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += y;
  }
  return v;
}

// One warp of every CTA: the cluster's tile range and the first query it deals with.  CTA 0 also
// publishes the tile prefix for the merge kernel.
__device__ void plan_cluster(const Params& p, Ctrl* ctrl, int cid, int clusters) {
  const int lane = threadIdx.x & 31;
  const bool writer = blockIdx.x == 0;
  int carry = 0;
  for (int base = 0; base < p.items; base += 32) {
    const int i = base + lane;
    const int tiles = i < p.items ? ceil_div(visible_tokens(p, i, writer), kTile) : 0;
    const int x = warp_scan_incl(tiles);
    if (writer && i < p.items) p.prefix[i] = carry + x - tiles;
    carry += __shfl_sync(0xffffffffu, x, 31);
  }
  const int T = carry;
  if (writer && lane == 0) p.prefix[p.items] = T;
  const int Ce = max(1, min(clusters, T));
  int lo = T + 1, hi = T + 1, item = p.items, prefix = T;
  if (cid < Ce) {
    lo = (int)((long long)cid * T / Ce);
    hi = (int)((long long)(cid + 1) * T / Ce);
    int run = 0;
    for (int base = 0; base < p.items; base += 32) {
      const int i = base + lane;
      const int tiles = i < p.items ? ceil_div(visible_tokens(p, i, false), kTile) : 0;
      const int x = warp_scan_incl(tiles);
      const int P = run + x - tiles;
      const bool mine = i < p.items && (tiles > 0 ? P + tiles > lo : P >= lo);
      const uint32_t m = __ballot_sync(0xffffffffu, mine);
      if (m) {
        const int l0 = __ffs(m) - 1;
        item = base + l0;
        prefix = __shfl_sync(0xffffffffu, P, l0);
        break;
      }
      run += __shfl_sync(0xffffffffu, x, 31);
    }
  }
  if (lane == 0) {
    ctrl->plan_lo = lo;
    ctrl->plan_hi = hi;
    ctrl->plan_item = item;
    ctrl->plan_prefix = prefix;
    ctrl->plan_total = T;
    ctrl->plan_last = cid == Ce - 1;
  }
}

// Walks the pieces of this cluster in order; each role of the kernel runs its own copy.
struct PieceIter {
  int item, prefix, lo, hi, T, cid;
  bool last;
  __device__ void init(const Ctrl* c, int cid_) {
    item = c->plan_item;
    prefix = c->plan_prefix;
    lo = c->plan_lo;
    hi = c->plan_hi;
    T = c->plan_total;
    last = c->plan_last != 0;
    cid = cid_;
  }
  // The next piece, including queries with nothing visible (t_end == t_begin).
  __device__ bool next(const Params& p, Piece& pc) {
    while (item < p.items) {
      const int vis = visible_tokens(p, item, false);
      const int tiles = ceil_div(vis, kTile);
      const int P = prefix;
      if (P >= hi && !(last && P == T)) return false;
      const int i = item;
      ++item;
      prefix += tiles;
      if (tiles == 0) {
        if (P >= lo) {
          pc.item = i;
          pc.t_begin = pc.t_end = 0;
          pc.slot = -1;
          return true;
        }
        continue;
      }
      const int a = max(lo, P), e = min(hi, P + tiles);
      if (e <= a) continue;
      pc.item = i;
      pc.t_begin = (a - P) * kTile;
      pc.t_end = min(vis, (e - P) * kTile);
      pc.slot = (a > P || e < P + tiles) ? 2 * cid + (a > P ? 0 : 1) : -1;
      return true;
    }
    return false;
  }
  __device__ bool next_nonempty(const Params& p, Piece& pc) {
    while (next(p, pc))
      if (pc.t_end > pc.t_begin) return true;
    return false;
  }
};

// Copy a [128 rows x 32 B] slice of a shared-memory matrix (descriptor) into 8 TMEM columns.
__device__ __forceinline__ void tmem_cp_128x256b(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.128x256b [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

// ------------------------------------------------------------------ epilogue stores
// 32 fp32 columns of an O row, normalised, as 4 x 16 bytes of bf16.
__device__ __forceinline__ void store_bf16_chunk(uint4* dst, const uint32_t (&r)[32], float inv) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint4 v;
    v.x = pack_bf16x2(__uint_as_float(r[8 * i + 0]) * inv, __uint_as_float(r[8 * i + 1]) * inv);
    v.y = pack_bf16x2(__uint_as_float(r[8 * i + 2]) * inv, __uint_as_float(r[8 * i + 3]) * inv);
    v.z = pack_bf16x2(__uint_as_float(r[8 * i + 4]) * inv, __uint_as_float(r[8 * i + 5]) * inv);
    v.w = pack_bf16x2(__uint_as_float(r[8 * i + 6]) * inv, __uint_as_float(r[8 * i + 7]) * inv);
    dst[i] = v;
  }
}
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
// The same columns as fp16 in the partial layout [column / 8][row][8] (dst at this row's first group): a
// partial is a normalised weighted mean of cached values, well inside fp16 range, and 11 significant
// bits keep its rounding far below the bf16 rounding of the final output.
__device__ __forceinline__ void store_f16_chunk(uint4* dst, const uint32_t (&r)[32], float inv) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint4 v;
    v.x = pack_f16x2(__uint_as_float(r[8 * i + 0]) * inv, __uint_as_float(r[8 * i + 1]) * inv);
    v.y = pack_f16x2(__uint_as_float(r[8 * i + 2]) * inv, __uint_as_float(r[8 * i + 3]) * inv);
    v.z = pack_f16x2(__uint_as_float(r[8 * i + 4]) * inv, __uint_as_float(r[8 * i + 5]) * inv);
    v.w = pack_f16x2(__uint_as_float(r[8 * i + 6]) * inv, __uint_as_float(r[8 * i + 7]) * inv);
    dst[(size_t)i * kH] = v;
  }
}

// ------------------------------------------------------------------ score MMAs
// The kE / 16 K-steps of ring slot S of a score tile, each an M = 128 (heads), N = 128 (tokens), K = 16
// MMA into d: K-step elements e = S * kE + 16 k.  Latent elements take A from the query's TMEM columns
// (32 columns per 64 bf16 elements, 8 per K-step), positional elements from the shared-memory rows
// (32 B per K-step); B advances 16 element rows (2048 B) per K-step.
template <int S>
__device__ __forceinline__ void score_slot_mmas_t(uint32_t d, uint32_t tq, uint64_t qr0, uint64_t bd, uint32_t idesc) {
#pragma unroll
  for (int k = 0; k < kE / 16; ++k) {
    const int e = S * kE + k * 16;
    const uint32_t acc = (S > 0 || k > 0) ? 1u : 0u;
    if (e < kDC)
      mma_ts(d, tq + (e / 64) * 32 + ((e % 64) / 16) * 8, bd + (uint64_t)(k * 128), idesc, acc);
    else
      mma_ss(d, qr0 + (uint64_t)(((e - kDC) / 16) * 2), bd + (uint64_t)(k * 128), idesc, acc);
  }
}

// Dispatch on a slot index that is a compile-time constant wherever the caller's loop is unrolled.
__device__ __forceinline__ void score_slot_mmas(int sl, uint32_t d, uint32_t tq, uint64_t qr0, uint64_t bd,
                                                uint32_t idesc) {
  static_assert(kSlotsPerTile <= 6, "dispatch covers six slots");
  switch (sl) {
    case 0: score_slot_mmas_t<0>(d, tq, qr0, bd, idesc); break;
    case 1: score_slot_mmas_t<(1 < kSlotsPerTile ? 1 : 0)>(d, tq, qr0, bd, idesc); break;
    case 2: score_slot_mmas_t<(2 < kSlotsPerTile ? 2 : 0)>(d, tq, qr0, bd, idesc); break;
    case 3: score_slot_mmas_t<(3 < kSlotsPerTile ? 3 : 0)>(d, tq, qr0, bd, idesc); break;
    case 4: score_slot_mmas_t<(4 < kSlotsPerTile ? 4 : 0)>(d, tq, qr0, bd, idesc); break;
    default: score_slot_mmas_t<(5 < kSlotsPerTile ? 5 : 0)>(d, tq, qr0, bd, idesc); break;
  }
}

// ------------------------------------------------------------------ attention kernel
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    decode_tc_kernel(const __grid_constant__ CUtensorMap mapk, const __grid_constant__ CUtensorMap mapv,
                     const __grid_constant__ CUtensorMap mapq, Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  Ctrl* ctrl = reinterpret_cast<Ctrl*>(smem);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_ctarank();
  const int cid = (int)cluster_id_x();
  volatile int* abort_flag = &ctrl->abort_flag;

  // the next kernel (the merge) may be scheduled now; it waits for this grid before touching memory
  pdl_trigger();
  if (tid == 0) {
    for (int i = 0; i < kRing; ++i) { mbar_init(&ctrl->k_full[i], 1); mbar_init(&ctrl->k_empty[i], 1); }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&ctrl->s_full[i], 1);
      mbar_init(&ctrl->s_empty[i], 256);
      mbar_init(&ctrl->xch[i], 256);
    }
    mbar_init(&ctrl->qr_full, 1);
    mbar_init(&ctrl->qr_free, 1);
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
    prefetch_tmap(&mapk);
    prefetch_tmap(&mapv);
    prefetch_tmap(&mapq);
  }
  // everything below reads what earlier kernels of the stream wrote (queries, appended rows)
  pdl_wait();
  if (warp == 3) plan_cluster(p, ctrl, cid, (int)num_clusters_x());
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem = ctrl->tmem_base;
  const uint32_t smem_base = smem_u32(smem);
  // warpgroup lanes: warps 4..11, quarter q4 = TMEM lane group, half = which 64 tokens / 256 O columns
  const int q4 = warp & 3, half = (warp - 4) >> 2;
  const int h = q4 * 32 + lane;
  PieceIter it;
  it.init(ctrl, cid);
  Piece pc;

  if (rank == 0) {
    // =========================== score CTA ===========================
    if (warp == 0) {
      if (lane == 0) {
        // per piece: the 8 latent query chunks (16 KB each, through the ring), the positional query chunk
        // (into QR once the previous piece's MMAs are done with it), then the tiles.  A tile slot holds
        // element rows [sl * kE, sl * kE + kE) of the tile's first block at +0 and of its second block at
        // +kBoxK (absent in a one-block tail tile).  Block-table entries are read one tile ahead.
        int r = 0, npiece = 0;
        uint32_t phase = 0;
        while (it.next_nonempty(p, pc)) {
          const int32_t* trow = p.table + (long long)(pc.item / p.n_q) * p.max_blocks;
          int raw0 = __ldg(trow + pc.t_begin / kBlk);
          int raw1 = pc.t_begin + kBlk < pc.t_end ? __ldg(trow + pc.t_begin / kBlk + 1) : 0;
#pragma unroll 1
          for (int c = 0; c < kQChunks; ++c) {
            if (!mbar_wait_cta(&ctrl->k_empty[r], phase ^ 1, p.status, abort_flag)) goto score_done;
            mbar_arrive_expect_tx(&ctrl->k_full[r], kQChunkBytes);
            tma_load_3d(smem + kOffRing + r * kSlotK, &mapq, &ctrl->k_full[r], c * 64, 0, pc.item);
            if (++r == kRing) { r = 0; phase ^= 1; }
          }
          if (!mbar_wait_cta(&ctrl->qr_free, (npiece & 1) ^ 1, p.status, abort_flag)) goto score_done;
          mbar_arrive_expect_tx(&ctrl->qr_full, kQChunkBytes);
          tma_load_3d(smem + kOffQR, &mapq, &ctrl->qr_full, kDC, 0, pc.item);
          for (int t = pc.t_begin; t < pc.t_end; t += kTile) {
            const bool two = t + kBlk < pc.t_end;
            const int b0 = checked_block(p, raw0, true);
            const int b1 = two ? checked_block(p, raw1, true) : -1;
            const int tn = t + kTile;
            if (tn < pc.t_end) {
              raw0 = __ldg(trow + tn / kBlk);
              if (tn + kBlk < pc.t_end) raw1 = __ldg(trow + tn / kBlk + 1);
            }
#pragma unroll 1
            for (int sl = 0; sl < kSlotsPerTile; ++sl) {
              if (!mbar_wait_cta(&ctrl->k_empty[r], phase ^ 1, p.status, abort_flag)) goto score_done;
              uint8_t* dst = smem + kOffRing + r * kSlotK;
              mbar_arrive_expect_tx(&ctrl->k_full[r], two ? kSlotK : kBoxK);
              tma_load_3d(dst, &mapk, &ctrl->k_full[r], 0, sl * kE, b0);
              if (two) tma_load_3d(dst + kBoxK, &mapk, &ctrl->k_full[r], 0, sl * kE, b1);
              if (++r == kRing) { r = 0; phase ^= 1; }
            }
          }
          ++npiece;
        }
      }
    } else if (warp == 1) {
      if (lane == 0) {
        // S[128 heads x 128 tokens] = Q K^T: the cached rows are the MN-major B operand (tokens contiguous),
        // the tile's two blocks one box apart (leading byte offset kBoxK), 8-element groups 1024 B apart;
        // latent K-steps take A from TMEM, positional K-steps from shared memory
        const uint32_t idesc = idesc_bf16(128, kTile, false, true);
        const uint64_t ring0 = desc_sw128(smem_base + kOffRing, kBoxK, 1024);
        const uint64_t qr0 = desc_sw128(smem_base + kOffQR, 16, 1024);
        const uint64_t qchunk0 = desc_sw128(smem_base + kOffRing, 16, 1024);
        const uint32_t tq = tmem + kQCol;
        int r = 0, sbuf = 0, npiece = 0;
        uint32_t kphase = 0, sphase = 0;
        while (it.next_nonempty(p, pc)) {
          // the piece's latent query into TMEM: tcgen05 operations of this thread run in issue order, so
          // the copies land only after the previous piece's MMAs have read the old query
#pragma unroll 1
          for (int c = 0; c < kQChunks; ++c) {
            if (!mbar_wait_cta(&ctrl->k_full[r], kphase, p.status, abort_flag)) goto score_done;
            tc_fence_after();
            const uint64_t sd = qchunk0 + (uint64_t)(r * (kSlotK >> 4));
#pragma unroll
            for (int k = 0; k < 4; ++k) tmem_cp_128x256b(tq + c * 32 + k * 8, sd + (uint64_t)(k * 2));
            mma_commit(&ctrl->k_empty[r]);
            if (++r == kRing) { r = 0; kphase ^= 1; }
          }
          for (int t = pc.t_begin; t < pc.t_end; t += kTile) {
            if (!mbar_wait_cta(&ctrl->s_empty[sbuf], sphase ^ 1, p.status, abort_flag)) goto score_done;
            tc_fence_after();
            const uint32_t d = tmem + kSCol + sbuf * kTile;
#pragma unroll
            for (int sl = 0; sl < kSlotsPerTile; ++sl) {
              if (!mbar_wait_cta(&ctrl->k_full[r], kphase, p.status, abort_flag)) goto score_done;
              if (sl == kSlotsPerTile - 1 && t == pc.t_begin) {
                // the positional query part of this piece (read by the last slot's K-steps)
                if (!mbar_wait_cta(&ctrl->qr_full, npiece & 1, p.status, abort_flag)) goto score_done;
              }
              tc_fence_after();
              // every MMA operand of the slot is a compile-time offset from two base registers: any runtime
              // arithmetic between the MMAs of a slot stalls their issue
              score_slot_mmas(sl, d, tq, qr0, ring0 + (uint64_t)(r * (kSlotK >> 4)), idesc);
              mma_commit(&ctrl->k_empty[r]);
              if (++r == kRing) { r = 0; kphase ^= 1; }
            }
            mma_commit(&ctrl->s_full[sbuf]);
            if (++sbuf == 2) { sbuf = 0; sphase ^= 1; }
          }
          // QR (and the TMEM query) may be replaced once this piece's MMAs complete
          mma_commit(&ctrl->qr_free);
          ++npiece;
        }
      }
    } else if (warp >= 4 && warp < 12) {
      // softmax: head row h, tokens [64*half, 64*half + 64) of each tile, which form one unit of P
      const uint32_t lane_base = tmem + ((uint32_t)(q4 * 32) << 16);
      const uint32_t peer_slots = mapa(smem_base + kOffSlots, 1);
      int sbuf = 0, tile = 0, unit = 0;
      uint32_t sphase = 0, stage_phase = 0;
      while (it.next_nonempty(p, pc)) {
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
        // ring slot = latent element rows [0, 256) or [256, 512) of one 64-token block; block-table entries
        // are read one block ahead
        int r = 0;
        uint32_t phase = 0;
        while (it.next_nonempty(p, pc)) {
          const int32_t* trow = p.table + (long long)(pc.item / p.n_q) * p.max_blocks;
          int raw = __ldg(trow + pc.t_begin / kBlk);
          for (int t = pc.t_begin; t < pc.t_end; t += kBlk) {
            const int blk = checked_block(p, raw, false);
            if (t + kBlk < pc.t_end) raw = __ldg(trow + (t + kBlk) / kBlk);
#pragma unroll 1
            for (int nh = 0; nh < 2; ++nh) {
              if (!mbar_wait_cta(&ctrl->v_empty[r], phase ^ 1, p.status, abort_flag)) goto value_done;
              mbar_arrive_expect_tx(&ctrl->v_full[r], kSlotV);
              tma_load_3d(smem + kOffV + r * kSlotV, &mapv, &ctrl->v_full[r], 0, kVRows * nh, blk);
              if (++r == kVRing) { r = 0; phase ^= 1; }
            }
          }
        }
      }
    } else if (warp == 1) {
      // MMA warp: lane 0 issues, the whole warp waits and zeroes tail tokens.  O[:, 256 nh .. +256] +=
      // P (A: [heads][64 tokens], K-major) . V (B: the slot's 256 latent rows of 64 tokens, K-major)
      const uint32_t idesc = idesc_bf16(128, kVRows, false, false);
      const uint64_t pdesc0 = desc_sw128(smem_base + kOffSlots, 16, 1024);
      const uint64_t vdesc0 = desc_sw128(smem_base + kOffV, 16, 1024);
      int r = 0, pslot = 0;
      uint32_t vphase = 0, pphase = 0, idle_phase = 0, done_phase = 0;
      while (it.next(p, pc)) {
        if (pc.t_end <= pc.t_begin) {
          // a query with nothing visible: the epilogue writes its zero output
          if (lane == 0) {
            ctrl->cmd = kCmdZero;
            ctrl->cmd_piece = pc;
            mbar_arrive(&ctrl->work);
          }
          if (!warp_wait_cta(&ctrl->done, done_phase, p.status, abort_flag)) goto value_mma_exit;
          done_phase ^= 1;
          continue;
        }
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
              // tokens past the end of the sequence: zero their columns so 0 * garbage cannot reach O.
              // Row e holds tokens 8u..8u+7 in 16-byte unit u, stored at unit u ^ (e & 7) (128-byte swizzle)
              uint8_t* vst = smem + kOffV + r * kSlotV;
              const int u_full = (valid + 7) >> 3, u_part = valid >> 3, j0 = valid & 7;
              for (int e = lane; e < kVRows; e += 32) {
                uint8_t* row = vst + e * 128;
                for (int u = u_full; u < 8; ++u)
                  *reinterpret_cast<uint4*>(row + ((u ^ (e & 7)) << 4)) = make_uint4(0, 0, 0, 0);
                if (j0) {
                  uint16_t* unit = reinterpret_cast<uint16_t*>(row + ((u_part ^ (e & 7)) << 4));
                  for (int j = j0; j < 8; ++j) unit[j] = 0;
                }
              }
              fence_proxy_async_smem();
              __syncwarp();
            }
            tc_fence_after();
            if (lane == 0) {
              const uint64_t pd = pdesc0 + (uint64_t)(pslot * (kSlotBytes >> 4));
              const uint64_t vd = vdesc0 + (uint64_t)(r * (kSlotV >> 4));
#pragma unroll
              for (int s = 0; s < 4; ++s)   // K-steps of 16 tokens: 32 B along both operands' rows
                mma_ss(tmem + nh * kVRows, pd + (uint64_t)(s * 2), vd + (uint64_t)(s * 2), idesc,
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
          ctrl->cmd_piece = pc;
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
        } else if (cmd == kCmdZero) {
          const Piece pz = ctrl->cmd_piece;
          uint4* dst = reinterpret_cast<uint4*>(p.o_lat + ((size_t)pz.item * kH + h) * kDC + half * 256);
#pragma unroll
          for (int i = 0; i < 32; ++i) dst[i] = make_uint4(0, 0, 0, 0);
          if (p.lse_out && half == 0) p.lse_out[(size_t)pz.item * kH + h] = -INFINITY;
        } else {
          const Piece pc = ctrl->cmd_piece;
          const float l = ctrl->l_buf[h], mrow = ctrl->m_buf[h];
          const float inv = l > 0.f ? 1.f / l : 0.f;
          const float lse = l > 0.f ? (mrow + __log2f(l)) * kLn2 : -INFINITY;
          // eight 32-column chunks of the row, each TMEM load in flight while the previous chunk is stored
          uint32_t ra[32], rb[32];
          tmem_ld32(lane_base, ra);
          tmem_ld_wait();
          if (pc.slot < 0) {
            uint4* dst = reinterpret_cast<uint4*>(p.o_lat + ((size_t)pc.item * kH + h) * kDC + half * 256);
#pragma unroll 1
            for (int c = 0; c < 8; c += 2) {
              tmem_ld32(lane_base + (c + 1) * 32, rb);
              store_bf16_chunk(dst + c * 4, ra, inv);
              tmem_ld_wait();
              if (c + 2 < 8) tmem_ld32(lane_base + (c + 2) * 32, ra);
              store_bf16_chunk(dst + (c + 1) * 4, rb, inv);
              tmem_ld_wait();
            }
            if (p.lse_out && half == 0) p.lse_out[(size_t)pc.item * kH + h] = lse;
          } else {
            // partial layout [slot][column / 8][row][8] (fp16): each store of a warp fills 512 contiguous bytes
            uint4* dst = reinterpret_cast<uint4*>(p.part_o) + ((size_t)pc.slot * (kDC / 8) + half * 32) * kH + h;
#pragma unroll 1
            for (int c = 0; c < 8; c += 2) {
              tmem_ld32(lane_base + (c + 1) * 32, rb);
              store_f16_chunk(dst + (size_t)c * 4 * kH, ra, inv);
              tmem_ld_wait();
              if (c + 2 < 8) tmem_ld32(lane_base + (c + 2) * 32, ra);
              store_f16_chunk(dst + (size_t)(c + 1) * 4 * kH, rb, inv);
              tmem_ld_wait();
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
// Block (item, g) merges columns [16 g, 16 g + 16) of all 128 heads; thread = head row.  Launched as a
// programmatic dependent of the attention kernel: it waits for that grid (and its writes) to complete.
// A query's pieces lie in clusters c0..c1 (from the published tile prefix); the piece in c0 wrote
// slot 2 c0 + 1, the one in each later cluster c slot 2 c.  Queries held by one cluster, or with
// nothing visible, were written by the attention kernel itself.
constexpr int kMergeGroups = kDC / 16;

__global__ void __launch_bounds__(kH) merge_kernel(const int* prefix, int items, int clusters, const __half* part_o,
                                                   const float* part_lse, bf16* o_lat, float* lse_out) {
  pdl_trigger();
  pdl_wait();
  const int item = blockIdx.x, g = blockIdx.y, h = threadIdx.x;
  const int T = prefix[items];
  const int P0 = prefix[item], P1 = prefix[item + 1];
  if (P1 <= P0) return;
  const int Ce = max(1, min(clusters, T));
  const int c0 = cluster_of(P0, T, Ce), c1 = cluster_of(P1 - 1, T, Ce);
  if (c1 == c0) return;
  float mx = -INFINITY;
  for (int c = c0; c <= c1; ++c) mx = fmaxf(mx, part_lse[(size_t)(c == c0 ? 2 * c + 1 : 2 * c) * kH + h]);
  float z = 0.f;
  float acc[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) acc[i] = 0.f;
  for (int c = c0; c <= c1; ++c) {
    const int slot = c == c0 ? 2 * c + 1 : 2 * c;
    const float w = expf(part_lse[(size_t)slot * kH + h] - mx);
    z += w;
    // partial layout [slot][column / 8][row][8] (fp16)
    const uint4* src = reinterpret_cast<const uint4*>(part_o) + ((size_t)slot * (kDC / 8) + g * 2) * kH + h;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const uint4 v = src[(size_t)j * kH];
      const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&wv[q]));
        acc[8 * j + 2 * q] = fmaf(w, f.x, acc[8 * j + 2 * q]);
        acc[8 * j + 2 * q + 1] = fmaf(w, f.y, acc[8 * j + 2 * q + 1]);
      }
    }
  }
  const float inv = 1.f / z;
  uint4* dst = reinterpret_cast<uint4*>(o_lat + ((size_t)item * kH + h) * kDC + g * 16);
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
  size_t prefix, part_o, part_lse, total;
};

WsLayout ws_layout(int items, int C) {
  WsLayout w;
  size_t o = 0;
  auto take = [&](size_t bytes) { size_t r = o; o = (o + bytes + 255) / 256 * 256; return r; };
  w.prefix = take(sizeof(int) * (items + 1));
  w.part_o = take(sizeof(__half) * (size_t)2 * C * kH * kDC);
  w.part_lse = take(sizeof(float) * (size_t)2 * C * kH);
  w.total = o;
  return w;
}

}  // namespace

bool tc_decode_supported(const mla_config* cfg, int batch, int n_q) {
  // one positional key shared by all heads: it is the B operand of the positional K-steps
  return cfg->dtype == MLA_BF16 && !cfg->rope_per_head && cfg->n_heads == kH && cfg->d_c == kDC &&
         cfg->d_rope == kDR && cfg->block_size == kBlk && batch > 0 && n_q > 0 && (long long)batch * n_q < (1LL << 24);
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

  // The pool viewed as [block][element row][token] (each block stored transposed); a box of whole element
  // rows lands as [row][64 tokens = 128 B] with the 128-byte swizzle the MMA descriptors expect.  The
  // queries viewed as [item][head][element]; a box of 64 elements of all 128 heads lands as the K-major
  // [head][128 B] layout of an MMA A operand.
  CUtensorMap mapk, mapv, mapq;
  const cuuint64_t dims[3] = {(cuuint64_t)kBlk, (cuuint64_t)kRow, (cuuint64_t)cache.num_blocks};
  const cuuint64_t strides[2] = {(cuuint64_t)kBlk * 2, (cuuint64_t)kBlk * kRow * 2};
  const cuuint32_t boxk[3] = {(cuuint32_t)kBlk, (cuuint32_t)kE, 1};
  const cuuint32_t boxv[3] = {(cuuint32_t)kBlk, (cuuint32_t)kVRows, 1};
  const cuuint64_t qdims[3] = {(cuuint64_t)kRow, (cuuint64_t)kH, (cuuint64_t)items};
  const cuuint64_t qstrides[2] = {(cuuint64_t)kRow * 2, (cuuint64_t)kH * kRow * 2};
  const cuuint32_t boxq[3] = {64, (cuuint32_t)kH, 1};
  const cuuint32_t estride[3] = {1, 1, 1};
  if (encode(&mapk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, cache.pool, dims, strides, boxk, estride,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS ||
      encode(&mapv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, cache.pool, dims, strides, boxv, estride,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS ||
      encode(&mapq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q), qdims, qstrides, boxq, estride,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;

  Params prm;
  prm.q = static_cast<const bf16*>(q);
  prm.table = cache.block_table;
  prm.kv_len = kv_len;
  prm.max_blocks = cache.max_blocks_per_seq;
  prm.num_blocks = cache.num_blocks;
  prm.n_q = n_q;
  prm.items = items;
  prm.cap = cache.max_blocks_per_seq * kBlk;
  prm.prefix = reinterpret_cast<int*>(ws + w.prefix);
  prm.o_lat = static_cast<bf16*>(o_lat);
  prm.lse_out = lse;
  prm.part_o = reinterpret_cast<__half*>(ws + w.part_o);
  prm.part_lse = reinterpret_cast<float*>(ws + w.part_lse);
  prm.scale_log2 = scale * kLog2e;
  prm.status = ctx.status;
  cudaError_t e = ensure_smem_limit((const void*)decode_tc_kernel, kSmemBytes, ctx.device);
  if (e != cudaSuccess) return e;
  e = launch_pdl(decode_tc_kernel, dim3(2 * C), dim3(kThreads), kSmemBytes, ctx.stream, mapk, mapv, mapq, prm);
  count_launch();
  if (e != cudaSuccess) return e;
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;

  // the merge is a programmatic dependent of the attention grid: it may be scheduled while that grid
  // runs and waits (griddepcontrol.wait) for it to complete
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(items, kMergeGroups, 1);
  lc.blockDim = dim3(kH, 1, 1);
  lc.dynamicSmemBytes = 0;
  lc.stream = ctx.stream;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = at;
  lc.numAttrs = 1;
  e = cudaLaunchKernelEx(&lc, merge_kernel, (const int*)prm.prefix, items, C, (const __half*)prm.part_o,
                         (const float*)prm.part_lse, prm.o_lat, lse);
  count_launch();
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace mla
