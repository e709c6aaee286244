// Absorbed MLA decode on the 5th-generation tensor cores (sm_103a).
//
// Math ("MLA, dim by dim" 4.2 and 5.2; "From Vanilla Transformers to Modern
// LLMs -- Part 3" 3.o-3.p): per (sequence b, query slot i) and head h,
//   s_j  = (q_lat[h] . c_j + q_rope[h] . kR_j) * scale      (j visible)
//   o_lat[h] = sum_j softmax(s)_j c_j ,  lse[h] = ln sum_j exp(s_j)
// with heads as the MMA M dimension (128 rows) and 64 cached tokens (one
// page) per tile as N, so one tile read from HBM serves every head.
//
// A cluster of two CTAs (a "pair", two SMs) splits the work by role, because
// one SM's tensor memory (512 fp32 columns x 128 lanes) holds either the full
// latent accumulator O (128 heads x 512) or the full query, not both:
//   * the S-CTA (cluster rank 1) keeps the item's query [q_lat ; q_rope]
//     (128 x 576 bf16 = 288 columns) in TMEM as the A operand of
//     S = Q C^T (M=128, N=64, K=576, three S buffers in the other 192
//     columns), runs the online softmax and ships P (bf16) to its peer;
//   * the V-CTA (rank 0) keeps O (512 columns) in TMEM and accumulates
//     O += P C (M=128, N=2x256, K=64) from P in its shared memory.
// Every cache tile is loaded once from HBM: each CTA issues half of the
// latent boxes with TMA multicast to both CTAs (the S-CTA also loads the
// RoPE box for itself), so the two CTAs see the same 64 x 512 latent tile at
// the same shared-memory offset.  A stage is refilled only when both the
// QK^T of the S-CTA and the PV of the V-CTA that read it have completed
// (tcgen05.commit multicast to both CTAs' "empty" barriers).
//
// Messages from the S-CTA to the V-CTA travel by st.async into the V-CTA's
// shared memory, each counted by an mbarrier: per tile the P tile (16 KB,
// already in the 128B-swizzled K-major layout of the MMA), the per-row
// rescale factor and four per-warp rescale flags; per segment the row
// statistics (running max and sum) the epilogue needs.
//
// Online softmax in base 2 with lazy rescaling: the running maximum moves
// (and O is rescaled by the V-CTA's correction warps) only when a tile's
// maximum exceeds it by more than 8 (a factor 256); otherwise P is taken
// against the stale maximum, which leaves o = O / l exact.
//
// Split-KV: the visible tiles of all (sequence, slot) items are laid end to
// end and cut into equal ranges, one per co-resident pair.  Pieces of items
// cut by a range boundary write fp32 partials (O/l and lse) that
// combine_tc_kernel merges with log-sum-exp weights; whole items are written
// directly.  The plan is computed on the device from seqlens (no host sync).
//
// Warp roles (192 threads per CTA): warp 0 TMA producer, warp 1 TMEM owner
// and MMA issuer, warps 2-5 softmax (S-CTA) or rescale / epilogue (V-CTA);
// warp w of 2-5 owns TMEM lanes (rows) 32*(w%4) .. 32*(w%4)+31.
//
// Every wait is bounded; a lost wait records MLA_ERR_TIMEOUT in the
// workspace, tells the peer CTA to stop, and the CTA unwinds (no trap).
#include <math.h>

#include "internal.cuh"
#include "ptx.cuh"
#include "tc.cuh"
#include "tmap.cuh"

namespace mla {
namespace {

constexpr int kMaxPairs = kNumSMs / 2;  // 74 clusters of 2 CTAs
constexpr int kTile = 64;               // tokens per tile = block size
constexpr int kDc = 512, kDr = 64, kD = kDc + kDr;
constexpr int kStages = 3;
constexpr int kMaxItems = 1024;  // B * Hq limit of this path
constexpr int kPrefetchTiles = 6;  // L2 prefetch distance (tiles)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2(256)

constexpr uint32_t kRankV = 0, kRankS = 1;
constexpr uint16_t kMaskBoth = 0x3, kMaskS = 1u << kRankS;

// ---- shared memory (offsets from the dynamic base, identical in both CTAs)
constexpr uint32_t kBox = 64 * 128;                   // 64 rows x 128 B, 128B swizzle
constexpr uint32_t kLatStage = 8 * kBox;              // 64 tokens x 512 latent
constexpr uint32_t kOffLat = 0;                       // both: [kStages][8 boxes]
constexpr uint32_t kOffRope = kStages * kLatStage;    // S: [kStages] RoPE boxes
constexpr uint32_t kOffPrefix = kOffRope + kStages * kBox;  // S: tiles prefix [W+1]
constexpr uint32_t kOffP = kStages * kLatStage;       // V: [2] P tiles
constexpr uint32_t kPBytes = 128 * 128;               // 128 rows x 64 bf16
constexpr uint32_t kOffAlpha = kOffP + 2 * kPBytes;   // V: [2][128] f32
constexpr uint32_t kOffFlags = kOffAlpha + 2 * 128 * 4;  // V: [2][4] u32
constexpr uint32_t kOffStats = kOffFlags + 2 * 16;    // V: m[128], l[128]
constexpr uint32_t kOffBars = kOffStats + 2 * 128 * 4;
constexpr uint32_t kMsgBytes = kPBytes + 128 * 4 + 16;  // one P message
constexpr uint32_t kStatsBytes = 2 * 128 * 4;
static_assert(kOffPrefix + (kMaxItems + 1) * 4 <= kOffAlpha, "S-CTA prefix overlaps");

struct Bars {
  uint64_t full[kStages], empty[kStages];
  uint64_t s_full[3], s_free[3];   // S: score buffers
  uint64_t p_full[2];              // V: P messages arrived
  uint64_t p_free[2];              // S: V-CTA done with a P buffer
  uint64_t q_full, q_free;         // S: query in TMEM / QK^T of a segment done
  uint64_t stats_full;             // V: row statistics arrived
  uint64_t stats_free;             // S: V-CTA read the statistics
  uint64_t o_full, pv_done;        // V: accumulator complete
  uint64_t ev_full, ev_done;       // V: MMA warp <-> correction warps
  uint64_t drain;
};

struct Misc {
  uint32_t tmem;
  int abort;
  int ev_type;  // kEvRescale | buffer << 4, kEvEpilogue, kEvDone
  int per, t_begin, t_end, w0, t_total;
  int bad_smem;
};
constexpr int kEvRescale = 1, kEvEpilogue = 2, kEvDone = 3;

constexpr uint32_t kOffMisc = kOffBars + ((sizeof(Bars) + 15) / 16) * 16;
constexpr uint32_t kSmemBytes = kOffMisc + ((sizeof(Misc) + 15) / 16) * 16;
static_assert(kSmemBytes <= 232448, "over the 227 KB shared-memory limit");

// TMEM columns
constexpr uint32_t kTmemQ = 0;    // S: 288 columns of packed bf16 query
constexpr uint32_t kTmemS = 320;  // S: + 64 * buffer (3 buffers)
constexpr uint32_t kTmemO = 0;    // V: 512 columns

struct DecodeArgs {
  const __nv_bfloat16 *q_lat;   // [W*H][512]
  const __nv_bfloat16 *q_rope;  // [W*H][64]
  const int32_t *block_table;
  const int32_t *seqlens;
  int B, Hq, H, max_blocks, max_seqlen, num_blocks, npairs;
  float scale_log2;
  __nv_bfloat16 *o_lat;
  float *lse;
  float *o_part;    // [2 * kMaxPairs][128][512]
  float *lse_part;  // [2 * kMaxPairs][128]
  int *plan;        // [0] = tiles per pair, [1..W+1] = prefix of tiles per item
  int *err;
};

__device__ __forceinline__ int visible_len(const DecodeArgs &a, int w, bool *bad) {
  const int b = w / a.Hq, slot = w % a.Hq;
  const int sl = a.seqlens[b];
  if (sl < 0 || sl > a.max_seqlen || sl > a.max_blocks * kTile) {
    *bad = true;
    return 0;
  }
  const int n = sl - a.Hq + slot + 1;
  return n > 0 ? n : 0;
}

__device__ __forceinline__ bool wait_bar(uint64_t *bar, uint32_t parity, volatile int *abort) {
  return ptx::mbar_wait<false>(bar, parity, abort);
}
__device__ __forceinline__ bool wait_bar_cl(uint64_t *bar, uint32_t parity, volatile int *abort) {
  return ptx::mbar_wait<true>(bar, parity, abort);
}
// One answer for the whole warp (warp-collective code follows every wait).
__device__ __forceinline__ bool wait_bar_warp(uint64_t *bar, uint32_t parity, volatile int *abort,
                                              bool cluster_scope = false) {
  const bool ok = cluster_scope ? wait_bar_cl(bar, parity, abort) : wait_bar(bar, parity, abort);
  return __all_sync(0xffffffffu, ok);
}

// Prefix of tiles per item, read from the S-CTA's shared memory (locally or
// through distributed shared memory).
struct Prefix {
  const int *local;
  uint32_t remote;
  __device__ int operator()(int i) const {
    return local ? local[i] : ptx::ld_cluster_s32(remote + 4u * (uint32_t)i);
  }
};

// The segments of one pair: consecutive (item, tile range) pieces of its
// range [t_begin, t_end) of the global tile order, starting at item w0.
struct SegIter {
  Prefix pre;
  int W, t_begin, t_end, w;
  __device__ void init(Prefix p, int W_, int tb, int te, int w0) {
    pre = p;
    W = W_;
    t_begin = tb;
    t_end = te;
    w = w0;
  }
  // next non-empty segment: item, first and end local tile; false when done
  __device__ bool next(int *item, int *lt0, int *lt1, bool *whole) {
    while (w < W) {
      const int s = pre(w), e = pre(w + 1);
      if (s >= t_end) return false;
      const int cur = w++;
      if (e <= s || e <= t_begin) continue;
      const int g0 = s > t_begin ? s : t_begin;
      const int g1 = e < t_end ? e : t_end;
      *item = cur;
      *lt0 = g0 - s;
      *lt1 = g1 - s;
      *whole = (g0 == s) && (g1 == e);
      return true;
    }
    return false;
  }
};

// Block-table entries of one sequence, 32 at a time in a warp register
// (lane i holds entry base + i); warp-collective.
struct TableWindow {
  const int32_t *tbl;
  int lt1, base;
  int v;
  __device__ void reset(const int32_t *t, int end) {
    tbl = t;
    lt1 = end;
    base = -1;
    v = 0;
  }
  __device__ int at(int lt, int lane) {
    const int b = lt & ~31;
    if (b != base) {
      base = b;
      v = (b + lane < lt1) ? tbl[b + lane] : 0;
    }
    return __shfl_sync(0xffffffffu, v, lt & 31);
  }
};

__device__ __forceinline__ void signal_abort(Misc *misc, uint32_t peer) {
  atomicExch(&misc->abort, 1);
  ptx::st_cluster_s32(ptx::map_to_rank(&misc->abort, peer), 1);
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(192, 1)
    decode_tc_kernel(const __grid_constant__ CUtensorMap tm_cache, DecodeArgs a) {
  extern __shared__ __align__(1024) uint8_t smem[];
  Bars *bars = reinterpret_cast<Bars *>(smem + kOffBars);
  Misc *misc = reinterpret_cast<Misc *>(smem + kOffMisc);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = ptx::cluster_ctarank();
  const uint32_t peer = rank ^ 1u;
  const bool isS = rank == kRankS;
  const int pair = blockIdx.x >> 1;
  const int W = a.B * a.Hq;
  volatile int *abort = &misc->abort;
  int *s_prefix = reinterpret_cast<int *>(smem + kOffPrefix);

  // ---- setup: barriers, TMEM, tile plan ----
  if (threadIdx.x == 0) {
    misc->abort = 0;
    misc->ev_type = 0;
    // the swizzled tiles need a 1024-byte aligned base; refuse to run otherwise
    misc->bad_smem = (ptx::smem_u32(smem) & 1023u) != 0;
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(&bars->full[s], 1);
      ptx::mbar_init(&bars->empty[s], 2);
    }
    for (int s = 0; s < 3; ++s) {
      ptx::mbar_init(&bars->s_full[s], 1);
      ptx::mbar_init(&bars->s_free[s], 128);
    }
    for (int s = 0; s < 2; ++s) {
      ptx::mbar_init(&bars->p_full[s], 1);
      ptx::mbar_init(&bars->p_free[s], 1);
    }
    ptx::mbar_init(&bars->q_full, 128);
    ptx::mbar_init(&bars->q_free, 1);
    ptx::mbar_init(&bars->stats_full, 1);
    ptx::mbar_init(&bars->stats_free, 4);
    ptx::mbar_init(&bars->o_full, 1);
    ptx::mbar_init(&bars->pv_done, 1);
    ptx::mbar_init(&bars->ev_full, 1);
    ptx::mbar_init(&bars->ev_done, 128);
    ptx::mbar_init(&bars->drain, 1);
    ptx::fence_mbar_init();
    if (!isS) {  // arm the first message phases the S-CTA will fill
      ptx::mbar_arrive_expect_tx(&bars->p_full[0], kMsgBytes);
      ptx::mbar_arrive_expect_tx(&bars->p_full[1], kMsgBytes);
      ptx::mbar_arrive_expect_tx(&bars->stats_full, kStatsBytes);
    }
  }
  if (warp == 0 && lane == 0) ptx::tma_prefetch_desc(&tm_cache);
  if (warp == 1) ptx::tmem_alloc(&misc->tmem, 512);
  if (isS) {
    // tiles per item -> s_prefix[w + 1], then an inclusive scan
    bool any_bad = false;
    for (int w = threadIdx.x; w < W; w += blockDim.x) {
      bool bad = false;
      const int n = visible_len(a, w, &bad);
      any_bad |= bad;
      s_prefix[w + 1] = (n + kTile - 1) / kTile;
    }
    if (any_bad && pair == 0) set_device_error(a.err, kDevBounds);
    __syncthreads();
    if (warp == 0) {
      int running = 0;
      for (int base = 0; base < W; base += 32) {
        const int idx = base + lane;
        int v = idx < W ? s_prefix[idx + 1] : 0;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const int u = __shfl_up_sync(0xffffffffu, v, off);
          if (lane >= off) v += u;
        }
        if (idx < W) s_prefix[idx + 1] = running + v;
        running += __shfl_sync(0xffffffffu, v, 31);
      }
      if (lane == 0) s_prefix[0] = 0;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      const int t_total = s_prefix[W];
      const int per = (t_total + a.npairs - 1) / a.npairs;
      const int tb = min(t_total, pair * per);
      const int te = min(t_total, tb + per);
      // first item whose tile range ends after tb
      int lo = 0, hi = W;
      while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (s_prefix[mid + 1] <= tb) lo = mid + 1;
        else hi = mid;
      }
      misc->per = per;
      misc->t_begin = tb;
      misc->t_end = te;
      misc->w0 = lo;
      misc->t_total = t_total;
    }
    if (blockIdx.x == 1) {  // the S-CTA of pair 0 publishes the plan for the combine
      if (threadIdx.x == 0) a.plan[0] = (s_prefix[W] + a.npairs - 1) / a.npairs;
      for (int w = threadIdx.x; w <= W; w += blockDim.x) a.plan[1 + w] = s_prefix[w];
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_sync();  // both CTAs started, barriers initialised, plan computed
  ptx::tc_fence_after();

  const uint32_t tmem = misc->tmem;
  const bool bad_smem = misc->bad_smem != 0;
  Prefix pre;
  pre.local = isS ? s_prefix : nullptr;
  pre.remote = isS ? 0u : ptx::map_to_rank(s_prefix, kRankS);
  // this pair's tile range (the V-CTA reads the S-CTA's values)
  int t_begin, t_end, w0;
  if (isS) {
    t_begin = misc->t_begin;
    t_end = misc->t_end;
    w0 = misc->w0;
  } else {
    t_begin = ptx::ld_cluster_s32(ptx::map_to_rank(&misc->t_begin, kRankS));
    t_end = ptx::ld_cluster_s32(ptx::map_to_rank(&misc->t_end, kRankS));
    w0 = ptx::ld_cluster_s32(ptx::map_to_rank(&misc->w0, kRankS));
  }

  if (bad_smem) {
    if (threadIdx.x == 0) set_device_error(a.err, kDevTimeout);
  } else if (warp == 0) {
    // ===================== TMA producer (both CTAs) =====================
    SegIter it;
    it.init(pre, W, t_begin, t_end, w0);
    int item, lt0, lt1, g = 0;
    bool whole;
    TableWindow cur, ahead;
    const uint32_t tx_bytes = isS ? kLatStage + kBox : kLatStage;
    const int box0 = isS ? 4 : 0;
    while (!*abort && it.next(&item, &lt0, &lt1, &whole)) {
      const int b = item / a.Hq;
      const int32_t *tbl = a.block_table + (size_t)b * a.max_blocks;
      cur.reset(tbl, lt1);
      ahead.reset(tbl, lt1);
      if (isS && lane == 0) {  // the query the softmax warps load next
        const size_t row0 = (size_t)item * a.H;
        const int nrows = a.H < 128 ? a.H : 128;
        ptx::prefetch_l2(a.q_lat + row0 * kDc, (uint32_t)nrows * kDc * 2);
        ptx::prefetch_l2(a.q_rope + row0 * kDr, (uint32_t)nrows * kDr * 2);
      }
      bool failed = false;
      for (int lt = lt0; lt < lt1; ++lt, ++g) {
        const int st = g % kStages;
        if (g >= kStages &&
            !wait_bar_warp(&bars->empty[st], ((g / kStages) - 1) & 1, abort)) {
          failed = true;
          break;
        }
        int blk = cur.at(lt, lane);
        if (blk < 0 || blk >= a.num_blocks) blk = 0;  // reported by the softmax warps
        if (lane == 0) {
          uint8_t *dst = smem + kOffLat + st * kLatStage;
          ptx::mbar_arrive_expect_tx(&bars->full[st], tx_bytes);
          for (int k = 0; k < 4; ++k)
            ptx::tma_load_2d_mc(dst + (box0 + k) * kBox, &tm_cache, &bars->full[st],
                                (box0 + k) * 64, blk * kTile, kMaskBoth);
          if (isS)
            ptx::tma_load_2d(smem + kOffRope + st * kBox, &tm_cache, &bars->full[st], kDc,
                             blk * kTile);
        }
        const int lp = lt + kPrefetchTiles;
        if (lp < lt1) {
          int pblk = ahead.at(lp, lane);
          if (lane == 0 && pblk >= 0 && pblk < a.num_blocks) {
            for (int k = 0; k < 4; ++k) ptx::tma_prefetch_2d(&tm_cache, (box0 + k) * 64, pblk * kTile);
            if (isS) ptx::tma_prefetch_2d(&tm_cache, kDc, pblk * kTile);
          }
        }
      }
      if (failed) {
        signal_abort(misc, peer);
        break;
      }
    }
    // Leave only when both CTAs are done with every stage this CTA filled:
    // all loads have landed and no multicast commit is still on its way.
    if (!*abort)
      for (int k = g - kStages < 0 ? 0 : g - kStages; k < g; ++k)
        wait_bar_warp(&bars->empty[k % kStages], (k / kStages) & 1, abort);
  } else if (warp == 1) {
    if (isS) {
      // ===================== S-CTA: QK^T issuer =====================
      if (lane == 0) {
        const uint32_t idesc = ptx::idesc_bf16(128, kTile, false, false);
        const uint32_t lat_addr = ptx::smem_u32(smem + kOffLat);
        const uint32_t rope_addr = ptx::smem_u32(smem + kOffRope);
        SegIter it;
        it.init(pre, W, t_begin, t_end, w0);
        int item, lt0, lt1, seg = 0, g = 0;
        bool whole, failed = false;
        while (!failed && it.next(&item, &lt0, &lt1, &whole)) {
          if (!wait_bar(&bars->q_full, seg & 1, abort)) { failed = true; break; }
          ptx::tc_fence_after();
          for (int lt = lt0; lt < lt1; ++lt, ++g) {
            const int st = g % kStages, sb = g % 3;
            if (!wait_bar(&bars->full[st], (g / kStages) & 1, abort)) { failed = true; break; }
            if (g >= 3 && !wait_bar(&bars->s_free[sb], ((g / 3) - 1) & 1, abort)) { failed = true; break; }
            ptx::tc_fence_after();
            const uint32_t d = tmem + kTmemS + sb * kTile;
            const uint32_t lat = lat_addr + st * kLatStage;
#pragma unroll
            for (int kk = 0; kk < 32; ++kk) {  // latent: 8 boxes x 4 k-steps of 16
              const uint64_t bd =
                  ptx::smem_desc(lat + (kk >> 2) * kBox + (kk & 3) * 32, 16, 1024, ptx::kSw128);
              ptx::mma_bf16_ts(d, tmem + kTmemQ + kk * 8, bd, idesc, kk != 0);
            }
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {  // RoPE: one box, 4 k-steps
              const uint64_t bd =
                  ptx::smem_desc(rope_addr + st * kBox + kk * 32, 16, 1024, ptx::kSw128);
              ptx::mma_bf16_ts(d, tmem + kTmemQ + 256 + kk * 8, bd, idesc, 1u);
            }
            ptx::mma_commit(&bars->s_full[sb]);
            ptx::mma_commit_mc(&bars->empty[st], kMaskBoth);
          }
          if (failed) break;
          ptx::mma_commit(&bars->q_free);
          ++seg;
        }
        ptx::mma_commit(&bars->drain);
        ptx::mbar_wait(&bars->drain, 0);
        if (failed) signal_abort(misc, peer);
      }
    } else {
      // ===================== V-CTA: PV issuer =====================
      if (lane == 0) {
        const uint32_t idesc = ptx::idesc_bf16(128, 256, false, true);
        const uint32_t lat_addr = ptx::smem_u32(smem + kOffLat);
        const uint32_t p_addr = ptx::smem_u32(smem + kOffP);
        const uint32_t *flags = reinterpret_cast<const uint32_t *>(smem + kOffFlags);
        SegIter it;
        it.init(pre, W, t_begin, t_end, w0);
        int item, lt0, lt1, seg = 0, g = 0, nev = 0, npv = 0;
        bool whole, failed = false;
        auto post = [&](int type) -> bool {
          misc->ev_type = type;
          ptx::mbar_arrive(&bars->ev_full);
          const bool ok = wait_bar(&bars->ev_done, nev & 1, abort);
          ++nev;
          return ok;
        };
        while (!failed && it.next(&item, &lt0, &lt1, &whole)) {
          for (int lt = lt0; lt < lt1; ++lt, ++g) {
            const int st = g % kStages, pb = g & 1;
            if (!wait_bar(&bars->full[st], (g / kStages) & 1, abort)) { failed = true; break; }
            if (!wait_bar_cl(&bars->p_full[pb], (g >> 1) & 1, abort)) { failed = true; break; }
            const volatile uint32_t *f = flags + 4 * pb;
            const bool resc = lt != lt0 && ((f[0] | f[1] | f[2] | f[3]) != 0);
            if (resc) {
              // O *= alpha (per row) once the previous PV has accumulated
              ptx::mma_commit(&bars->pv_done);
              if (!wait_bar(&bars->pv_done, npv & 1, abort)) { failed = true; break; }
              ++npv;
              if (!post(kEvRescale | (pb << 4))) { failed = true; break; }
            }
            // the next message into this buffer comes after the PV below
            ptx::mbar_arrive_expect_tx(&bars->p_full[pb], kMsgBytes);
            ptx::fence_proxy_async_smem();  // P was written by st.async
            ptx::tc_fence_after();
            const uint32_t lat = lat_addr + st * kLatStage;
#pragma unroll
            for (int kk = 0; kk < kTile / 16; ++kk) {
              const uint64_t ad =
                  ptx::smem_desc(p_addr + pb * kPBytes + kk * 32, 16, 1024, ptx::kSw128);
#pragma unroll
              for (int h = 0; h < 2; ++h) {
                const uint64_t bd =
                    ptx::smem_desc(lat + h * 4 * kBox + kk * 2048, 4 * 2048, 1024, ptx::kSw128);
                ptx::mma_bf16(tmem + kTmemO + h * 256, ad, bd, idesc,
                              (lt == lt0 && kk == 0) ? 0u : 1u);
              }
            }
            ptx::mma_commit_mc(&bars->p_free[pb], kMaskS);
            ptx::mma_commit_mc(&bars->empty[st], kMaskBoth);
          }
          if (failed) break;
          ptx::mma_commit(&bars->o_full);
          if (!wait_bar(&bars->o_full, seg & 1, abort)) { failed = true; break; }
          if (!post(kEvEpilogue)) { failed = true; break; }
          ++seg;
        }
        misc->ev_type = kEvDone;
        ptx::mbar_arrive(&bars->ev_full);
        ptx::mma_commit(&bars->drain);
        ptx::mbar_wait(&bars->drain, 0);
        if (failed) signal_abort(misc, peer);
      }
    }
  } else if (isS) {
    // ===================== S-CTA: softmax (warps 2-5) =====================
    const int row = 32 * (warp & 3) + lane;
    const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
    SegIter it;
    it.init(pre, W, t_begin, t_end, w0);
    int item, lt0, lt1, seg = 0, g = 0;
    bool whole, failed = false;
    // remote (V-CTA) addresses of the message buffers and their barriers
    const uint32_t rP = ptx::map_to_rank(smem + kOffP, kRankV);
    const uint32_t rAlpha = ptx::map_to_rank(smem + kOffAlpha, kRankV);
    const uint32_t rFlags = ptx::map_to_rank(smem + kOffFlags, kRankV);
    const uint32_t rStats = ptx::map_to_rank(smem + kOffStats, kRankV);
    const uint32_t rPFull0 = ptx::map_to_rank(&bars->p_full[0], kRankV);
    const uint32_t rPFull1 = ptx::map_to_rank(&bars->p_full[1], kRankV);
    const uint32_t rStatsFull = ptx::map_to_rank(&bars->stats_full, kRankV);
    const float c = a.scale_log2;
    while (!failed && it.next(&item, &lt0, &lt1, &whole)) {
      bool dummy = false;
      const int n_vis = visible_len(a, item, &dummy);
      const int b = item / a.Hq;
      // block-table entries this segment reads (each warp on its own)
      bool seg_bad;
      {
        const int32_t *tbl = a.block_table + (size_t)b * a.max_blocks;
        bool bad = false;
        for (int lt = lt0 + lane; lt < lt1; lt += 32) {
          const int blk = tbl[lt];
          bad |= (blk < 0 || blk >= a.num_blocks);
        }
        seg_bad = __any_sync(0xffffffffu, bad);
      }
      // -- this item's query -> TMEM (row = lane), once the previous
      //    segment's QK^T no longer reads it --
      if (seg > 0 && !wait_bar_warp(&bars->q_free, (seg - 1) & 1, abort)) { failed = true; break; }
      ptx::tc_fence_after();
      {
        const bool valid = row < a.H;
        const size_t grow = (size_t)item * a.H + row;
        const uint4 *ql = reinterpret_cast<const uint4 *>(a.q_lat + grow * kDc);
        const uint4 *qr = reinterpret_cast<const uint4 *>(a.q_rope + grow * kDr);
#pragma unroll
        for (int half = 0; half < 2; ++half) {  // 2 x 9 chunks of 16 columns
          uint32_t v[9][16];
#pragma unroll
          for (int cc = 0; cc < 9; ++cc) {
            const int chunk = half * 9 + cc;  // 0..15 latent, 16..17 RoPE
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              uint4 x = make_uint4(0, 0, 0, 0);
              if (valid) x = chunk < 16 ? __ldg(ql + chunk * 4 + q) : __ldg(qr + (chunk - 16) * 4 + q);
              v[cc][4 * q] = x.x;
              v[cc][4 * q + 1] = x.y;
              v[cc][4 * q + 2] = x.z;
              v[cc][4 * q + 3] = x.w;
            }
          }
#pragma unroll
          for (int cc = 0; cc < 9; ++cc)
            ptx::tmem_st16_nc(tmem + lane_base + kTmemQ + (half * 9 + cc) * 16, v[cc]);
        }
        ptx::tmem_st_wait();
      }
      ptx::tc_fence_before();
      ptx::mbar_arrive(&bars->q_full);

      float m_run = -INFINITY, l_run = 0.f;
      for (int lt = lt0; lt < lt1; ++lt, ++g) {
        const int sb = g % 3, pb = g & 1;
        if (!wait_bar_warp(&bars->s_full[sb], (g / 3) & 1, abort)) { failed = true; break; }
        ptx::tc_fence_after();
        float s[64];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          float v[16];
          ptx::tmem_ld16(tmem + lane_base + kTmemS + sb * kTile + q * 16, v);
#pragma unroll
          for (int i = 0; i < 16; ++i) s[q * 16 + i] = v[i];
        }
        ptx::tmem_ld_wait();
        ptx::tc_fence_before();
        ptx::mbar_arrive(&bars->s_free[sb]);
        const int tok0 = lt * kTile;
        if (tok0 + kTile > n_vis) {
#pragma unroll
          for (int j = 0; j < 64; ++j)
            if (tok0 + j >= n_vis) s[j] = -INFINITY;
        }
        float mx = s[0];
#pragma unroll
        for (int j = 1; j < 64; ++j) mx = fmaxf(mx, s[j]);
        const float mt = mx * c;
        float m_use = m_run, alpha = 1.f;
        bool resc = false;
        if (lt == lt0) {
          m_use = mt;
        } else if (mt > m_run + kRescaleThreshold) {
          m_use = mt;
          alpha = ptx::ex2(m_run - mt);
          resc = true;
        }
        uint32_t pk[32];
        float lsum = 0.f;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float p0 = ptx::ex2(fmaf(s[2 * i], c, -m_use));
          const float p1 = ptx::ex2(fmaf(s[2 * i + 1], c, -m_use));
          lsum += p0 + p1;
          pk[i] = ptx::pack_bf16x2(p0, p1);
        }
        l_run = l_run * alpha + lsum;
        m_run = m_use;
        // P buffer pb was last read by the V-CTA's PV of tile g-2
        if (g >= 2 && !wait_bar_warp(&bars->p_free[pb], ((g >> 1) - 1) & 1, abort, true)) {
          failed = true;
          break;
        }
        const uint32_t rbar = pb ? rPFull1 : rPFull0;
        const uint32_t prow = rP + pb * kPBytes + row * 128;
#pragma unroll
        for (int cc = 0; cc < 8; ++cc)
          ptx::st_async_v4(prow + ((cc ^ (row & 7)) << 4), pk[4 * cc], pk[4 * cc + 1],
                           pk[4 * cc + 2], pk[4 * cc + 3], rbar);
        ptx::st_async_b32(rAlpha + (pb * 128 + row) * 4, __float_as_uint(alpha), rbar);
        const uint32_t wflag = __ballot_sync(0xffffffffu, resc);
        if (lane == 0) ptx::st_async_b32(rFlags + (pb * 4 + (warp & 3)) * 4, wflag, rbar);
      }
      if (failed) break;
      // -- row statistics of the segment -> V-CTA epilogue --
      if (seg > 0 && !wait_bar_warp(&bars->stats_free, (seg - 1) & 1, abort, true)) { failed = true; break; }
      ptx::st_async_b32(rStats + row * 4, __float_as_uint(m_run), rStatsFull);
      ptx::st_async_b32(rStats + (128 + row) * 4, __float_as_uint(seg_bad ? -1.f : l_run),
                        rStatsFull);
      ++seg;
    }
    if (failed) {
      signal_abort(misc, peer);
    } else {
      // the V-CTA's last remote arrivals land before this CTA may exit
      if (seg > 0) wait_bar_warp(&bars->stats_free, (seg - 1) & 1, abort, true);
      for (int k = g - 2 < 0 ? 0 : g - 2; k < g; ++k)
        wait_bar_warp(&bars->p_free[k & 1], (k >> 1) & 1, abort, true);
    }
    // items with nothing visible (or an invalid length): o = 0, lse = -inf
    for (int w = pair; w < W; w += a.npairs) {
      if (s_prefix[w + 1] != s_prefix[w]) continue;
      if (row < a.H) {
        const size_t r = (size_t)w * a.H + row;
        uint4 *d4 = reinterpret_cast<uint4 *>(a.o_lat + r * kDc);
        for (int i = 0; i < kDc * 2 / 16; ++i) d4[i] = make_uint4(0, 0, 0, 0);
        a.lse[r] = -INFINITY;
      }
    }
  } else {
    // ============ V-CTA: rescale and epilogue (warps 2-5) ============
    const int row = 32 * (warp & 3) + lane;
    const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
    const float *alpha_buf = reinterpret_cast<const float *>(smem + kOffAlpha);
    const float *stats = reinterpret_cast<const float *>(smem + kOffStats);
    const uint32_t rStatsFree = ptx::map_to_rank(&bars->stats_free, kRankS);
    SegIter it;
    it.init(pre, W, t_begin, t_end, w0);
    int item, lt0, lt1, seg = 0, nev = 0;
    bool whole, failed = false;
    for (;;) {
      if (!wait_bar_warp(&bars->ev_full, nev & 1, abort)) { failed = true; break; }
      ++nev;
      const int ev = *reinterpret_cast<volatile int *>(&misc->ev_type);
      if ((ev & 15) == kEvDone) break;
      if ((ev & 15) == kEvRescale) {
        const int pb = ev >> 4;
        // the factors arrived by st.async from the peer (seen through the
        // MMA warp's cluster-scope wait)
        asm volatile("fence.acq_rel.cluster;" ::: "memory");
        const float al = alpha_buf[pb * 128 + row];
        ptx::tc_fence_after();
        if (al != 1.f) {
#pragma unroll 1
          for (int q = 0; q < 512 / 16; ++q) {
            float v[16];
            ptx::tmem_ld16(tmem + lane_base + kTmemO + q * 16, v);
            ptx::tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 16; ++i) v[i] *= al;
            ptx::tmem_st16(tmem + lane_base + kTmemO + q * 16, v);
          }
          ptx::tmem_st_wait();
        }
        ptx::tc_fence_before();
        ptx::mbar_arrive(&bars->ev_done);
        continue;
      }
      // epilogue of the next segment
      if (!it.next(&item, &lt0, &lt1, &whole)) { failed = true; break; }
      if (!wait_bar_warp(&bars->o_full, seg & 1, abort) ||
          !wait_bar_warp(&bars->stats_full, seg & 1, abort, true)) {
        failed = true;
        break;
      }
      ptx::tc_fence_after();
      const float m = stats[row], l = stats[128 + row];
      __syncwarp();
      if (warp == 2 && lane == 0)  // next segment's statistics phase
        ptx::mbar_arrive_expect_tx(&bars->stats_full, kStatsBytes);
      if (lane == 0) ptx::mbar_arrive_remote(&bars->stats_free, kRankS);
      (void)rStatsFree;
      const bool seg_bad = l < 0.f;
      const bool write_row = row < a.H;
      const float inv_l = l > 0.f ? 1.f / l : 0.f;
      const float lse_val = l > 0.f ? (m + log2f(l)) * kLn2 : -INFINITY;
      const size_t grow = (size_t)item * a.H + row;
      if (whole) {
        __nv_bfloat16 *dst = a.o_lat + grow * kDc;
#pragma unroll 1
        for (int q = 0; q < kDc / 32; ++q) {
          float v0[16], v1[16];
          ptx::tmem_ld16(tmem + lane_base + kTmemO + q * 32, v0);
          ptx::tmem_ld16(tmem + lane_base + kTmemO + q * 32 + 16, v1);
          ptx::tmem_ld_wait();
          if (write_row) {
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              pk[i] = seg_bad ? 0u : ptx::pack_bf16x2(v0[2 * i] * inv_l, v0[2 * i + 1] * inv_l);
              pk[8 + i] = seg_bad ? 0u : ptx::pack_bf16x2(v1[2 * i] * inv_l, v1[2 * i + 1] * inv_l);
            }
            uint4 *d4 = reinterpret_cast<uint4 *>(dst + q * 32);
#pragma unroll
            for (int i = 0; i < 4; ++i) d4[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
          }
        }
        if (write_row) a.lse[grow] = seg_bad ? -INFINITY : lse_val;
      } else {
        // partial slot: 2*pair for the range's first segment, 2*pair+1 for its last
        const int slot_idx = 2 * pair + ((lt0 == 0) ? 1 : 0);
        float *dst = a.o_part + ((size_t)slot_idx * 128 + row) * kDc;
#pragma unroll 1
        for (int q = 0; q < kDc / 32; ++q) {
          float v0[16], v1[16];
          ptx::tmem_ld16(tmem + lane_base + kTmemO + q * 32, v0);
          ptx::tmem_ld16(tmem + lane_base + kTmemO + q * 32 + 16, v1);
          ptx::tmem_ld_wait();
          if (write_row) {
            float4 *d4 = reinterpret_cast<float4 *>(dst + q * 32);
#pragma unroll
            for (int i = 0; i < 4; ++i)
              d4[i] = make_float4(v0[4 * i] * inv_l, v0[4 * i + 1] * inv_l, v0[4 * i + 2] * inv_l,
                                  v0[4 * i + 3] * inv_l);
#pragma unroll
            for (int i = 0; i < 4; ++i)
              d4[4 + i] = make_float4(v1[4 * i] * inv_l, v1[4 * i + 1] * inv_l,
                                      v1[4 * i + 2] * inv_l, v1[4 * i + 3] * inv_l);
          }
        }
        if (write_row)
          a.lse_part[(size_t)slot_idx * 128 + row] =
              seg_bad ? __int_as_float(0x7fc00000) : lse_val;  // NaN poisons the item
      }
      if (seg_bad && row == 0) set_device_error(a.err, kDevBounds);
      ptx::tc_fence_before();
      ptx::mbar_arrive(&bars->ev_done);
      ++seg;
    }
    if (failed) signal_abort(misc, peer);
  }

  // ---- teardown ----
  __syncwarp();
  ptx::tc_fence_before();
  __syncthreads();
  if (misc->abort) {
    if (threadIdx.x == 0) set_device_error(a.err, kDevTimeout);
    __nanosleep(20000);  // copies the peer issued before it stopped have landed
  }
  ptx::cluster_sync();  // the peer no longer touches this CTA's shared memory
  ptx::tc_fence_after();
  if (warp == 1) ptx::tmem_dealloc(tmem, 512);
}

// Merge the partial pieces of every item that was cut between pairs.
// grid (W items, H / 16 row groups); 128 threads; non-split items exit.
__global__ void __launch_bounds__(128) combine_tc_kernel(DecodeArgs a) {
  const int w = blockIdx.x;
  const int per = a.plan[0];
  const int s = a.plan[1 + w], e = a.plan[2 + w];
  if (e <= s || per <= 0) return;
  const int p0 = s / per, p1 = (e - 1) / per;
  if (p0 == p1) return;  // written directly by its pair
  const int h0 = blockIdx.y * 16;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int hh = warp; hh < 16; hh += 4) {
    const int h = h0 + hh;
    if (h >= a.H) break;
    float mx = -INFINITY;
    bool poison = false;
    for (int p = p0; p <= p1; ++p) {
      const int slot = 2 * p + ((s < p * per) ? 0 : 1);
      const float v = a.lse_part[(size_t)slot * 128 + h];
      poison |= isnan(v);
      mx = fmaxf(mx, v);
    }
    const int row = w * a.H + h;
    __nv_bfloat16 *dst = a.o_lat + (size_t)row * kDc;
    if (poison || mx == -INFINITY) {
      for (int c = lane; c < kDc; c += 32) dst[c] = __float2bfloat16_rn(0.f);
      if (lane == 0) a.lse[row] = -INFINITY;
      continue;
    }
    float sum = 0.f;
    for (int p = p0; p <= p1; ++p) {
      const int slot = 2 * p + ((s < p * per) ? 0 : 1);
      sum += expf(a.lse_part[(size_t)slot * 128 + h] - mx);
    }
    const float inv = 1.f / sum;
    for (int c4 = lane; c4 < kDc / 4; c4 += 32) {
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int p = p0; p <= p1; ++p) {
        const int slot = 2 * p + ((s < p * per) ? 0 : 1);
        const float wgt = expf(a.lse_part[(size_t)slot * 128 + h] - mx) * inv;
        const float4 v = reinterpret_cast<const float4 *>(a.o_part + ((size_t)slot * 128 + h) * kDc)[c4];
        acc.x = fmaf(wgt, v.x, acc.x);
        acc.y = fmaf(wgt, v.y, acc.y);
        acc.z = fmaf(wgt, v.z, acc.z);
        acc.w = fmaf(wgt, v.w, acc.w);
      }
      uint2 pk;
      pk.x = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(acc.x)) |
             ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(acc.y)) << 16);
      pk.y = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(acc.z)) |
             ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(acc.w)) << 16);
      reinterpret_cast<uint2 *>(dst)[c4] = pk;
    }
    if (lane == 0) a.lse[row] = mx + logf(sum);
  }
}

size_t part_bytes() { return align_up((size_t)2 * kMaxPairs * 128 * kDc * sizeof(float), 256); }
size_t lse_part_bytes() { return align_up((size_t)2 * kMaxPairs * 128 * sizeof(float), 256); }

// Co-resident clusters of two CTAs for this kernel (some GPCs may not fit a
// whole number of pairs), capped at 74; looked up once per device.
int pairs_for_device() {
  static int cached[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (cached[dev] > 0) return cached[dev];
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * kMaxPairs, 1, 1);
  cfg.blockDim = dim3(192, 1, 1);
  cfg.dynamicSmemBytes = kSmemBytes;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, decode_tc_kernel, &cfg) != cudaSuccess || n <= 0) {
    cudaGetLastError();
    n = kMaxPairs;
  }
  if (n > kMaxPairs) n = kMaxPairs;
  cached[dev] = n;
  return n;
}

}  // namespace

bool tc_decode_supported(const mla_dims &d) {
  return d.dtype == MLA_BF16 && d.d_c == kDc && d.d_r == kDr && d.block_size == kTile &&
         d.H <= 128;
}

size_t tc_decode_workspace_bytes(int B, int Hq, const mla_dims &) {
  const size_t W = (size_t)B * Hq;
  return kWsHeader + part_bytes() + lse_part_bytes() + align_up((W + 2) * sizeof(int), 256);
}

cudaError_t launch_decode_tc(const void *q_lat, const void *q_rope, const void *cache,
                             int num_blocks, const int32_t *block_table, int max_blocks,
                             const int32_t *seqlens, int max_seqlen, int B, int Hq,
                             const mla_dims &d, float scale, void *o_lat, float *lse,
                             void *workspace, cudaStream_t st) {
  if ((long)B * Hq > kMaxItems) return cudaErrorNotSupported;
  CUtensorMap tm_cache;
  if (!make_tmap_2d_bf16(&tm_cache, cache, kD, (uint64_t)num_blocks * kTile, kD * 2, 64, 64,
                         CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(decode_tc_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)kSmemBytes);
  if (e != cudaSuccess) return e;
  const int npairs = pairs_for_device();
  if (npairs <= 0) return cudaErrorInvalidDevice;
  char *ws = static_cast<char *>(workspace);
  DecodeArgs a;
  a.q_lat = static_cast<const __nv_bfloat16 *>(q_lat);
  a.q_rope = static_cast<const __nv_bfloat16 *>(q_rope);
  a.block_table = block_table;
  a.seqlens = seqlens;
  a.B = B;
  a.Hq = Hq;
  a.H = d.H;
  a.max_blocks = max_blocks;
  a.max_seqlen = max_seqlen;
  a.num_blocks = num_blocks;
  a.npairs = npairs;
  a.scale_log2 = scale * kLog2e;
  a.o_lat = static_cast<__nv_bfloat16 *>(o_lat);
  a.lse = lse;
  a.err = reinterpret_cast<int *>(ws);
  a.o_part = reinterpret_cast<float *>(ws + kWsHeader);
  a.lse_part = reinterpret_cast<float *>(ws + kWsHeader + part_bytes());
  a.plan = reinterpret_cast<int *>(ws + kWsHeader + part_bytes() + lse_part_bytes());
  decode_tc_kernel<<<2 * npairs, 192, kSmemBytes, st>>>(tm_cache, a);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  dim3 cgrid(B * Hq, (d.H + 15) / 16);
  combine_tc_kernel<<<cgrid, 128, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace mla
