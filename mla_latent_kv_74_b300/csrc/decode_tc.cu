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
//     S = Q C^T (M=128, N=64, K=576; three 64-column score buffers, one
//     per tile in flight, in the other columns), runs the online softmax and
//     ships P (bf16) to its peer;
//   * the V-CTA (rank 0) keeps O (512 columns) in TMEM and accumulates
//     O += P C (M=128, N=2x256, K=64) with P in its shared memory.
// Each CTA streams the cache through its own ring of shared-memory stages,
// one 3-D TMA copy per stage: the S-CTA loads [c_KV ; k_R] tiles (HBM) and
// frees a stage as soon as its QK^T is done; the V-CTA loads the latent part
// of the same tiles a little later (L2 hits, issued evict-first: it is the
// lines' last read) and frees a stage after its PV.  Decoupling the rings
// keeps the long HBM latency off the softmax -> PV chain.  Each segment's query reaches the S-CTA through its ring too (two
// stages ahead of the segment's tiles), copied into TMEM by a softmax group.
// Two warps of the S-CTA issue QK^T on alternate tiles, all 36 k-steps of a
// tile into its score buffer (one thread issues an N = 64 MMA only every
// ~80 cycles; two interleaved chains reach ~45).
//
// P goes straight into the V-CTA's shared memory by st.async (distributed
// shared memory, counted on the destination mbarrier), already in the
// 128B-swizzled K-major layout of the MMA operand, with the rows' rescale
// factors and four per-warp rescale flags; one P buffer per tile parity.
// Each half (32 tokens) leaves as soon as its exponentials are done.  Two
// groups of four softmax warps take alternate tiles, so one group's
// transfer overlaps the other's exponentials.  The groups agree on the
// running maximum through shared memory (a tile's maximum is published
// before its exponentials, so the next tile waits only for that), keep
// their own row sums, and merge them at each segment end before the row
// statistics go to the V-CTA (st.async).  The V-CTA's correction warps apply
// the rare O rescales and run each segment's epilogue, staging O through the
// last tile's P buffer and writing whole 128-byte row pieces.
//
// Online softmax in base 2 with lazy rescaling: the running maximum moves
// (and O is rescaled by the V-CTA's correction warps) only when a tile's
// maximum exceeds it by more than 8 (a factor 256); otherwise P is taken
// against the stale maximum, which leaves o = O / l exact.
//
// Split-KV: the visible tiles of all (sequence, slot) items are laid end to
// end and cut into equal ranges, one per co-resident pair.  Pieces of items
// cut by a range boundary write partials (bf16 O/l, stored evict-last so
// they stay in L2, and fp32 lse) that combine_tc_kernel merges with
// log-sum-exp weights; whole items are written directly.  The plan is computed on the device from seqlens (no host sync).
// With several query slots per sequence the items are laid out slot by slot
// and each slot gets its own equal share of the pairs, so pair j of every
// slot walks the same sequences' pages at the same time: the slots after the
// first find each page in L2 (or merge with its miss in flight) instead of
// reading the cache from HBM again.
//
// Warp roles (352 threads per CTA): warp 0 TMA producer, warp 1 TMEM owner
// and MMA issuer; S-CTA: warp 6 the second QK^T issuer (warp 1 takes the
// even tiles, warp 6 the odd ones), warps 2-5 and 7-10 the two softmax
// groups (even / odd tiles); V-CTA: warps 2-5 rescale and epilogue.  A warp w that touches TMEM owns lanes 32*(w%4) .. 32*(w%4)+31.
// The kernel is launched as a programmatic dependent of the previous kernel
// in the stream and waits for it only after its barrier and TMEM setup.
//
// Every wait is bounded; a lost wait records MLA_ERR_TIMEOUT in the
// workspace, tells the peer CTA to stop, and the CTA unwinds (no trap).
//
// With at most 16 heads (the DeepSeek-V2-Lite shape) decode_sh_kernel
// replaces the pair: O kept transposed fits one SM's TMEM next to the
// query, so every SM streams its own tiles (see its own comment below).
#include <math.h>

#include <atomic>

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
constexpr int kThreads = 352;
// B * Hq limit of this path: the plan's per-item scan uses the (still idle)
// ring as scratch, 4 bytes per item
constexpr int kMaxItems = 8192;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2(256)
// The split plan charges each item's start (its query load and, for the pair
// that also ends an item there, an epilogue: about 9 us against 1.2 us per
// tile, measured) as this many extra tiles, so pairs that cross an item
// boundary get fewer tiles (6 balanced the pairs' end times best: at 7 the
// pairs without a boundary ended last).
constexpr int kItemCost = 6;
// The same for the few-heads kernel (one CTA per SM), whose item start costs
// about one tile: the query takes one ring stage and the epilogue of the
// previous item delays the next item's first PV.
constexpr int kShItemCost = 2;

constexpr uint32_t kRankV = 0, kRankS = 1;
constexpr uint16_t kMaskS = 1u << kRankS;

// ---- shared memory (offsets from the 1024-aligned dynamic base)
constexpr uint32_t kBox = 64 * 128;                // 64 rows x 128 B, 128B swizzle
constexpr uint32_t kOffRing = 0;
// S-CTA: [kStages] x (8 latent boxes + 1 RoPE box), the published running
// maximum, one group's row statistics at a segment end.  The ring also
// carries each segment's query: two stages of 64 rows x [q_lat ; q_rope]
// (exactly 2 x 72 KB) ahead of the segment's tiles.
constexpr uint32_t kSStage = 9 * kBox;
constexpr uint32_t kOffMDec = kStages * kSStage;  // m[128] f32
constexpr uint32_t kOffLM = kOffMDec + 128 * 4;           // m[128], l[128] f32
constexpr uint32_t kSEnd = kOffLM + 2 * 128 * 4;
// V-CTA: [kStages] x 8 latent boxes, P buffer per tile parity, their rescale
// factors and flags, row statistics
constexpr uint32_t kVStage = 8 * kBox;
constexpr uint32_t kOffP = kStages * kVStage;
constexpr uint32_t kPBytes = 128 * 128;            // 128 rows x 64 bf16
constexpr uint32_t kAuxBytes = 128 * 4 + 16;       // alpha[128] f32, flags[4] u32
constexpr uint32_t kOffAux = kOffP + 2 * kPBytes;
constexpr uint32_t kOffStats = kOffAux + 2 * kAuxBytes;  // m[128], l[128]
constexpr uint32_t kStatsBytes = 2 * 128 * 4;
constexpr uint32_t kVEnd = kOffStats + kStatsBytes;
// A P tile travels as two messages, tokens 0-31 (with the rescale factors
// and flags) and tokens 32-63, so the PV can start on the first half while
// the second is in flight and each half-buffer is freed after its k-steps.
constexpr uint32_t kMsgBytesA = kPBytes / 2 + kAuxBytes;
constexpr uint32_t kMsgBytesB = kPBytes / 2;
// both
constexpr uint32_t kOffBars = kSEnd > kVEnd ? kSEnd : kVEnd;
static_assert(kOffP % 1024 == 0, "P buffers must be 1024-byte aligned");

struct Bars {
  uint64_t full[kStages], empty[kStages];  // each CTA's own ring (V: full)
  // S: per tile g, barrier g % 6 (stage g % 3, issuer and softmax group
  // g % 2), so each barrier has one waiter that never falls a phase behind
  uint64_t sfull[6];                       // S: tile data landed
  // S: scores of tile g (TMEM buffer g % 3) ready / read: index g % 6
  uint64_t s_full[6], s_free[6];
  uint64_t q_full, q_free;                 // S: query in TMEM / QK^T of a segment done
  uint64_t qfull[2];                       // S: query rows 64h..64h+63 landed in the ring
  uint64_t m_ready[2];                     // S: group i published its tile's maximum
  uint64_t seg_sync[2];                    // S: both softmax groups at a segment end
  uint64_t p_free[4];                      // S: V-CTA done with half h of P buffer i (2i+h)
  uint64_t stats_free;                     // S: V-CTA read the statistics
  uint64_t p_full[4];                      // V: half h of P message i arrived (2i+h)
  uint64_t stats_full;                     // V: row statistics arrived
  uint64_t o_full, pv_done;                // V: accumulator complete
  uint64_t ev_full, ev_done;               // V: MMA warp <-> correction warps
  uint64_t drain[2];
};

struct Misc {
  uint32_t tmem;
  int abort;
  int ev_type;  // kEvRescale | buffer << 4, kEvEpilogue | buffer << 4, kEvDone
  int t_begin, t_end, w0, s0, t_total;
  int bad_smem;
};
constexpr int kEvRescale = 1, kEvEpilogue = 2, kEvDone = 3;

constexpr uint32_t kOffMisc = kOffBars + ((sizeof(Bars) + 15) / 16) * 16;
constexpr uint32_t kSmemBytes = kOffMisc + ((sizeof(Misc) + 15) / 16) * 16;
static_assert(kSmemBytes <= 232448, "over the 227 KB shared-memory limit");
static_assert((kMaxItems + 2) * 4 <= kStages * kSStage, "plan scan does not fit the ring");

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
  // the call covers the tokens [tok0, tok0 + tok_len) of every sequence
  // (0 and INT_MAX: all of them); block_table then starts at the range's
  // first block, so tile i of an item is the range's i-th block
  int tok0, tok_len;
  float scale_log2;
  __nv_bfloat16 *o_lat;
  float *lse;
  __nv_bfloat16 *o_part;  // [2 * pairs or CTAs][128][512] (O / l of split pieces)
  float *lse_part;  // [2 * pairs or CTAs][128]
  // plan: [0] = number of slot groups G (1 or Hq), [1+g] = units per pair of
  // group g, [1+Hq+u] = prefix of units per item in plan order u (u = slot *
  // B + b for item b * Hq + slot), u = 0..W
  int *plan;
  int *err;
};

#ifdef MLA_TRACE
// Developer tracing (built only with -DMLA_TRACE): %globaltimer stamps per
// tile and role for two pairs (the first and the middle one), read back
// with mla_debug_read_trace.  Events: 0 S: tile maximum agreed / V: producer issued the tile's loads, 1 MMA warp
// saw the tile's data, 2 S: QK^T issued / V: first P half arrived, 3 S:
// softmax exponentials done / V: PV issued, 4 S: softmax saw S / V: first
// half's MMAs issued, 5 S: P buffer free, 6 S: P sent, 7 per segment: S query
// loaded / V epilogue done, 8 S producer issued the tile's load, 9 S issuer
// passed its score-buffer wait.
constexpr int kTraceTiles = 512, kTraceEvents = 10, kTracePairs = 2;
__device__ unsigned long long g_trace[kTracePairs][2][kTraceEvents][kTraceTiles];
// per CTA: kernel entry, range start (after setup), end of work
__device__ unsigned long long g_trace_cta[2 * kMaxPairs][3];
// first start and last end of the combine kernel's blocks
__device__ unsigned long long g_trace_comb[2] = {~0ull, 0ull};
#define MLA_TRACE_CTA(k) \
  do { if (threadIdx.x == 0) g_trace_cta[blockIdx.x][k] = ptx::globaltimer_ns(); } while (0)
__device__ __forceinline__ void trace_ev(int pair, int npairs, uint32_t rank, int ev, int g) {
  const int slot = pair == 0 ? 0 : (pair == npairs / 2 ? 1 : -1);
  if (slot >= 0 && g >= 0 && g < kTraceTiles) g_trace[slot][rank][ev][g] = ptx::globaltimer_ns();
}
#define MLA_TRACE_EV(ev, g) trace_ev(pair, a.npairs, rank, (ev), (g))
#define SH_TRACE_EV(side, ev, g) trace_ev(cta, a.npairs, (side), (ev), (g))
#else
#define SH_TRACE_EV(side, ev, g) ((void)0)
#define MLA_TRACE_EV(ev, g) ((void)0)
#define MLA_TRACE_CTA(k) ((void)0)
#endif

__device__ __forceinline__ int visible_len(const DecodeArgs &a, int w, bool *bad) {
  const int b = w / a.Hq, slot = w % a.Hq;
  const int sl = a.seqlens[b];
  if (sl < 0 || sl > a.max_seqlen || sl > a.max_blocks * kTile) {
    *bad = true;
    return 0;
  }
  int n = sl - a.Hq + slot + 1 - a.tok0;  // visible tokens from the range start
  if (n > a.tok_len) n = a.tok_len;
  return n > 0 ? n : 0;
}

__device__ __forceinline__ int item_tiles(const DecodeArgs &a, int w) {
  bool bad = false;
  return (visible_len(a, w, &bad) + kTile - 1) / kTile;
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

// The segments of one pair: consecutive (item, tile range) pieces of its
// range [t_begin, t_end) of the plan's order, walked from item w0 (whose
// span starts at s0); tile counts come from seqlens.  In the plan's order an
// item with n > 0 tiles spans kCost + n units, the first kCost standing for
// its start-up cost and holding no tile: unit u of the span is tile
// u - kCost.
// Item of plan position u.  With one query slot the plan follows the items;
// with several (kSlotMajor) it lists every sequence's slot 0, then every
// sequence's slot 1, and so on.
template <bool kSlotMajor>
__device__ __forceinline__ int item_at(const DecodeArgs &a, int u) {
  return kSlotMajor ? (u % a.B) * a.Hq + u / a.B : u;
}

template <bool kSlotMajor, int kCost = kItemCost>
struct SegIter {
  const DecodeArgs *a;
  int W, t_begin, t_end, w, s;  // w: item (walked in plan order)
  // w0: the item at the start of the range (W if none), s0: its first unit
  __device__ void init(const DecodeArgs *args, int W_, int tb, int te, int w0, int s0) {
    a = args;
    W = W_;
    t_begin = tb;
    t_end = te;
    w = w0;
    s = s0;
  }
  // next non-empty segment: item, first and end local tile, visible length
  __device__ bool next(int *item, int *lt0, int *lt1, bool *whole, int *n_vis) {
    while (w < W && s < t_end) {
      bool bad = false;
      const int n = visible_len(*a, w, &bad);
      const int nt = (n + kTile - 1) / kTile;
      const int st = s, e = nt > 0 ? s + kCost + nt : s;
      const int cur = w;
      if (kSlotMajor) {
        // the same slot of the next sequence; past the last sequence, the
        // next slot's first sequence (or the end after the last slot)
        w += a->Hq;
        if (w >= W) {
          w -= W - 1;
          if (w >= a->Hq) w = W;
        }
      } else {
        ++w;
      }
      s = e;
      if (e <= st || e <= t_begin) continue;
      const int g0 = st > t_begin ? st : t_begin;
      const int g1 = e < t_end ? e : t_end;
      const int l0 = g0 - st - kCost > 0 ? g0 - st - kCost : 0;
      const int l1 = g1 - st - kCost > 0 ? g1 - st - kCost : 0;
      if (l1 <= l0) continue;  // only start-up units of this item here
      *item = cur;
      *lt0 = l0;
      *lt1 = l1;
      *whole = (l0 == 0) && (l1 == nt);
      *n_vis = n;
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

template <bool kSlotMajor>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    decode_tc_kernel(const __grid_constant__ CUtensorMap tm_cache,
                     const __grid_constant__ CUtensorMap tm_cache_v,
                     const __grid_constant__ CUtensorMap tm_qlat,
                     const __grid_constant__ CUtensorMap tm_qrope, DecodeArgs a) {
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
  MLA_TRACE_CTA(0);

  // ---- setup: barriers, TMEM, this pair's tile range ----
  if (threadIdx.x == 0) {
    misc->abort = 0;
    misc->ev_type = 0;
    // the swizzled tiles need a 1024-byte aligned base; refuse to run otherwise
    misc->bad_smem = (ptx::smem_u32(smem) & 1023u) != 0;
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(&bars->full[s], 1);
      ptx::mbar_init(&bars->empty[s], 1);
    }
    for (int s = 0; s < 6; ++s) {
      ptx::mbar_init(&bars->s_full[s], 1);
      ptx::mbar_init(&bars->s_free[s], 128);
    }
    for (int s = 0; s < 6; ++s) ptx::mbar_init(&bars->sfull[s], 1);
    ptx::mbar_init(&bars->q_full, 128);
    ptx::mbar_init(&bars->q_free, 2);
    ptx::mbar_init(&bars->qfull[0], 1);
    ptx::mbar_init(&bars->qfull[1], 1);
    for (int s = 0; s < 2; ++s) {
      ptx::mbar_init(&bars->m_ready[s], 128);
      ptx::mbar_init(&bars->seg_sync[s], 256);
      ptx::mbar_init(&bars->p_free[2 * s], 1);
      ptx::mbar_init(&bars->p_free[2 * s + 1], 1);
      ptx::mbar_init(&bars->p_full[2 * s], 1);
      ptx::mbar_init(&bars->p_full[2 * s + 1], 1);
      ptx::mbar_init(&bars->drain[s], 1);
    }
    ptx::mbar_init(&bars->stats_free, 4);
    ptx::mbar_init(&bars->stats_full, 1);
    ptx::mbar_init(&bars->o_full, 1);
    ptx::mbar_init(&bars->pv_done, 1);
    ptx::mbar_init(&bars->ev_full, 1);
    ptx::mbar_init(&bars->ev_done, 128);
    ptx::fence_mbar_init();
    if (!isS) {  // the first message phases the S-CTA fills
      for (int i = 0; i < 2; ++i) {
        ptx::mbar_arrive_expect_tx(&bars->p_full[2 * i], kMsgBytesA);
        ptx::mbar_arrive_expect_tx(&bars->p_full[2 * i + 1], kMsgBytesB);
      }
      ptx::mbar_arrive_expect_tx(&bars->stats_full, kStatsBytes);
    }
  }
  if (warp == 0 && lane == 0) {
    ptx::tma_prefetch_desc(isS ? &tm_cache : &tm_cache_v);
    if (isS) {
      ptx::tma_prefetch_desc(&tm_qlat);
      ptx::tma_prefetch_desc(&tm_qrope);
    }
  }
  if (warp == 1) ptx::tmem_alloc(&misc->tmem, 512);
  // Launched as a programmatic dependent: everything above overlaps the tail
  // of the previous kernel in the stream; its outputs (queries, and possibly
  // lengths or the cache) are read only after this wait.  Every CTA of this
  // grid is resident once all pass here, so the combine kernel may launch.
  ptx::grid_dependency_wait();
  ptx::launch_dependents();
  if (isS) {
    // tiles per item -> scan (scratch in the ring) -> this pair's range
    int *pre = reinterpret_cast<int *>(smem + kOffRing);
    bool any_bad = false;
    for (int u = threadIdx.x; u < W; u += blockDim.x) {
      bool bad = false;
      const int n = visible_len(a, item_at<kSlotMajor>(a, u), &bad);
      any_bad |= bad;
      const int nt = (n + kTile - 1) / kTile;
      pre[u + 1] = nt > 0 ? nt + kItemCost : 0;
    }
    if (any_bad && pair == 0) set_device_error(a.err, kDevBounds);
    __syncthreads();
    if (warp == 0) {
      int running = 0;
      for (int base = 0; base < W; base += 32) {
        const int idx = base + lane;
        int v = idx < W ? pre[idx + 1] : 0;
  #pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const int u = __shfl_up_sync(0xffffffffu, v, off);
          if (lane >= off) v += u;
        }
        if (idx < W) pre[idx + 1] = running + v;
        running += __shfl_sync(0xffffffffu, v, 31);
      }
      if (lane == 0) pre[0] = 0;
    }
    __syncthreads();
    if constexpr (kSlotMajor) {
      // slot groups: each query slot's items over its own share of the pairs
#ifdef MLA_FORCE_ONE_GROUP
      const int ngroups = 1;
#else
      const int ngroups = a.npairs >= a.Hq ? a.Hq : 1;
#endif
      const int pairs_per_group = a.npairs / ngroups;
      if (threadIdx.x == 0) {
        const int t_total = pre[W];
        const int g = pair / pairs_per_group, j = pair % pairs_per_group;
        const int g0 = g < ngroups ? pre[g * (W / ngroups)] : t_total;
        const int g1 = g < ngroups ? pre[(g + 1) * (W / ngroups)] : t_total;
        const int per = (g1 - g0 + pairs_per_group - 1) / pairs_per_group;
        const int tb = min(g1, g0 + j * per);
        const int te = min(g1, tb + per);
        int lo = 0, hi = W;  // first plan position whose tile range ends after tb
        while (lo < hi) {
          const int mid = (lo + hi) >> 1;
          if (pre[mid + 1] <= tb) lo = mid + 1;
          else hi = mid;
        }
        misc->t_begin = tb;
        misc->t_end = te;
        misc->w0 = lo < W ? item_at<true>(a, lo) : W;  // the SegIter walks items
        misc->s0 = lo < W ? pre[lo] : t_total;
        misc->t_total = t_total;
        if (pair == 0) {
          a.plan[0] = ngroups;
          for (int gg = 0; gg < ngroups; ++gg) {
            const int span = pre[(gg + 1) * (W / ngroups)] - pre[gg * (W / ngroups)];
            a.plan[1 + gg] = (span + pairs_per_group - 1) / pairs_per_group;
          }
        }
      }
      if (pair == 0)  // the plan of the combine kernel
        for (int u = threadIdx.x; u <= W; u += blockDim.x) a.plan[1 + a.Hq + u] = pre[u];
    } else {
      if (threadIdx.x == 0) {
        const int t_total = pre[W];
        const int per = (t_total + a.npairs - 1) / a.npairs;
        const int tb = min(t_total, pair * per);
        const int te = min(t_total, tb + per);
        int lo = 0, hi = W;  // first item whose tile range ends after tb
        while (lo < hi) {
          const int mid = (lo + hi) >> 1;
          if (pre[mid + 1] <= tb) lo = mid + 1;
          else hi = mid;
        }
        misc->t_begin = tb;
        misc->t_end = te;
        misc->w0 = lo;
        misc->s0 = lo < W ? pre[lo] : t_total;
        misc->t_total = t_total;
        if (pair == 0) a.plan[0] = per;
      }
      if (pair == 0)  // the plan of the combine kernel
        for (int w = threadIdx.x; w <= W; w += blockDim.x) a.plan[1 + w] = pre[w];
    }
    __syncthreads();  // the scratch is the ring: read before the first load
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_sync();  // both CTAs started, barriers initialised, range computed
  ptx::tc_fence_after();

  const uint32_t tmem = misc->tmem;
  const bool bad_smem = misc->bad_smem != 0;
  MLA_TRACE_CTA(1);
  int t_begin, t_end, w0, s0;
  if (isS) {
    t_begin = misc->t_begin;
    t_end = misc->t_end;
    w0 = misc->w0;
    s0 = misc->s0;
  } else {  // the V-CTA reads the S-CTA's values
    t_begin = ptx::ld_cluster_s32(ptx::map_to_rank(&misc->t_begin, kRankS));
    t_end = ptx::ld_cluster_s32(ptx::map_to_rank(&misc->t_end, kRankS));
    w0 = ptx::ld_cluster_s32(ptx::map_to_rank(&misc->w0, kRankS));
    s0 = ptx::ld_cluster_s32(ptx::map_to_rank(&misc->s0, kRankS));
  }

  if (bad_smem) {
    if (threadIdx.x == 0) set_device_error(a.err, kDevTimeout);
  } else if (warp == 0) {
    // ===================== TMA producer (each CTA its own ring) =====================
    SegIter<kSlotMajor> it;
    it.init(&a, W, t_begin, t_end, w0, s0);
    int item, lt0, lt1, n_vis, g = 0;
    bool whole, failed = false;
    TableWindow cur;
    const uint64_t evict_first = ptx::l2_policy_evict_first();
    const uint32_t stage_bytes = isS ? kSStage : kVStage;
    const int nbox = isS ? 9 : 8;
    int r = 0;  // ring position (tiles, plus two query stages per S segment)
    while (!failed && !*abort && it.next(&item, &lt0, &lt1, &whole, &n_vis)) {
      const int b = item / a.Hq;
      cur.reset(a.block_table + (size_t)b * a.max_blocks, lt1);
      if (isS) {  // the segment's query: rows 0-63 and 64-127 of the item
        for (int h = 0; h < 2; ++h, ++r) {
          const int st = r % kStages;
          if (r >= kStages && !wait_bar_warp(&bars->empty[st], ((r / kStages) - 1) & 1, abort)) {
            failed = true;
            break;
          }
          if (lane == 0) {
            uint8_t *dst = smem + kOffRing + st * kSStage;
            const int row0 = item * a.H + 64 * h;
            ptx::mbar_arrive_expect_tx(&bars->qfull[h], 9 * kBox);
            ptx::tma_load_3d(dst, &tm_qlat, &bars->qfull[h], 0, row0, 0);  // 8 latent boxes
            ptx::tma_load_2d(dst + 8 * kBox, &tm_qrope, &bars->qfull[h], 0, row0);
          }
        }
        if (failed) break;
      }
      for (int lt = lt0; lt < lt1; ++lt, ++g, ++r) {
        const int st = r % kStages;
        if (r >= kStages && !wait_bar_warp(&bars->empty[st], ((r / kStages) - 1) & 1, abort)) {
          failed = true;
          break;
        }
        int blk = cur.at(lt, lane);
        if (blk < 0 || blk >= a.num_blocks) blk = 0;  // reported by the softmax warps
        if (lane == 0) {
          if (!isS) MLA_TRACE_EV(0, g); else MLA_TRACE_EV(8, g);
          uint8_t *dst = smem + kOffRing + st * stage_bytes;
          uint64_t *fb = isS ? &bars->sfull[g % 6] : &bars->full[st];
          // the whole stage in one copy: nbox boxes of 64 rows x 128 B; the
          // V-CTA's copy is the last read of these lines, so it marks them
          // first to be evicted from L2
          ptx::mbar_arrive_expect_tx(fb, nbox * kBox);
          if (isS)
            ptx::tma_load_3d(dst, &tm_cache, fb, 0, blk * kTile, 0);
          else
            ptx::tma_load_3d_hint(dst, &tm_cache_v, fb, 0, blk * kTile, 0, evict_first);
        }
      }
    }
    if (failed) signal_abort(misc, peer);
    // leave only after this CTA's consumers released every stage it filled
    if (!*abort)
      for (int k = r - kStages < 0 ? 0 : r - kStages; k < r; ++k)
        wait_bar_warp(&bars->empty[k % kStages], (k / kStages) & 1, abort);
  } else if (isS && (warp == 1 || warp == 6)) {
    // ========== S-CTA: QK^T issuers ==========
    // The two issuers take alternate tiles (warp 1 even, warp 6 odd), each
    // all 36 k-steps of its tile into score buffer g % 3.  One thread alone
    // cannot issue N=64 MMAs at the tensor pipe's rate; two interleaved
    // whole-tile chains come closer than two half-K chains into separate
    // partial buffers, and the softmax reads one buffer per tile.
    if (lane == 0) {
      const int mine = warp == 1 ? 0 : 1;
      const uint32_t idesc = ptx::idesc_bf16(128, kTile, false, false);
      const uint64_t ring_desc = ptx::smem_desc(ptx::smem_u32(smem + kOffRing), 16, 1024, ptx::kSw128);
      SegIter<kSlotMajor> it;
      it.init(&a, W, t_begin, t_end, w0, s0);
      int item, lt0, lt1, n_vis, seg = 0, g = 0, r = 0;
      bool whole, failed = false;
      while (!failed && it.next(&item, &lt0, &lt1, &whole, &n_vis)) {
        if (!wait_bar(&bars->q_full, seg & 1, abort)) { failed = true; break; }
        ptx::tc_fence_after();
        r += 2;  // the segment's query stages
        for (int lt = lt0; lt < lt1; ++lt, ++g, ++r) {
          if ((g & 1) != mine) continue;
          const int st = r % kStages, sb = g % 3;
          if (!wait_bar(&bars->sfull[g % 6], (g / 6) & 1, abort)) { failed = true; break; }
          MLA_TRACE_EV(1, g);
          // buffer sb last held tile g-3 (the other issuer's, read by the
          // other softmax group)
          const int gp = g - 3;
          if (gp >= 0 && !wait_bar(&bars->s_free[gp % 6], (gp / 6) & 1, abort)) {
            failed = true;
            break;
          }
          MLA_TRACE_EV(9, g);
          ptx::tc_fence_after();
          const uint32_t d = tmem + kTmemS + sb * kTile;
          const uint64_t bs = ring_desc + (uint64_t)((st * kSStage) >> 4);
#pragma unroll
          for (int kk = 0; kk < 36; ++kk)  // 9 boxes (8 latent + RoPE) x 4 k-steps of 16
            ptx::mma_bf16_ts(d, tmem + kTmemQ + kk * 8,
                             bs + (uint64_t)((((kk >> 2) * kBox) + (kk & 3) * 32) >> 4), idesc,
                             kk != 0);
          ptx::mma_commit(&bars->s_full[g % 6]);
          ptx::mma_commit(&bars->empty[st]);
          MLA_TRACE_EV(2, g);
        }
        if (failed) break;
        ptx::mma_commit(&bars->q_free);
        ++seg;
      }
      uint64_t *dr = &bars->drain[mine];
      ptx::mma_commit(dr);
      ptx::mbar_wait(dr, 0);
      if (failed) signal_abort(misc, peer);
    }
  } else if (!isS && warp == 1) {
    // ===================== V-CTA: PV issuer =====================
    if (lane == 0) {
      const uint32_t idesc = ptx::idesc_bf16(128, 256, false, true);
      const uint64_t p_desc = ptx::smem_desc(ptx::smem_u32(smem + kOffP), 16, 1024, ptx::kSw128);
      const uint64_t ring_desc =
          ptx::smem_desc(ptx::smem_u32(smem + kOffRing), 4 * 2048, 1024, ptx::kSw128);
      const uint8_t *aux = smem + kOffAux;
      SegIter<kSlotMajor> it;
      it.init(&a, W, t_begin, t_end, w0, s0);
      int item, lt0, lt1, n_vis, seg = 0, g = 0, nev = 0, npv = 0;
      bool whole, failed = false;
      auto post = [&](int type) -> bool {
        misc->ev_type = type;
        ptx::mbar_arrive(&bars->ev_full);
        const bool ok = wait_bar(&bars->ev_done, nev & 1, abort);
        ++nev;
        return ok;
      };
      while (!failed && it.next(&item, &lt0, &lt1, &whole, &n_vis)) {
        for (int lt = lt0; lt < lt1; ++lt, ++g) {
          const int st = g % kStages, pb = g & 1;
          if (!wait_bar(&bars->full[st], (g / kStages) & 1, abort)) { failed = true; break; }
          MLA_TRACE_EV(1, g);
          if (!wait_bar_cl(&bars->p_full[2 * pb], (g >> 1) & 1, abort)) { failed = true; break; }
          MLA_TRACE_EV(2, g);
          const volatile uint32_t *fl =
              reinterpret_cast<const volatile uint32_t *>(aux + pb * kAuxBytes + 512);
          const uint32_t any = fl[0] | fl[1] | fl[2] | fl[3];
          if (lt != lt0 && any != 0) {
            // O *= alpha (per row) once every PV so far has accumulated
            ptx::mma_commit(&bars->pv_done);
            if (!wait_bar(&bars->pv_done, npv & 1, abort)) { failed = true; break; }
            ++npv;
            if (!post(kEvRescale | (pb << 4))) { failed = true; break; }
          }
          const uint64_t ad0 = p_desc + (uint64_t)((pb * kPBytes) >> 4);
          const uint64_t bd0 = ring_desc + (uint64_t)((st * kVStage) >> 4);
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            if (half == 1 &&
                !wait_bar_cl(&bars->p_full[2 * pb + 1], (g >> 1) & 1, abort)) {
              failed = true;
              break;
            }
            // the next message into this half-buffer comes after the MMAs below
            ptx::mbar_arrive_expect_tx(&bars->p_full[2 * pb + half],
                                       half ? kMsgBytesB : kMsgBytesA);
            ptx::fence_proxy_async_smem();  // P arrived by st.async (generic proxy)
            ptx::tc_fence_after();
#pragma unroll
            for (int k2 = 0; k2 < 2; ++k2) {
              const int kk = 2 * half + k2;
#pragma unroll
              for (int h = 0; h < 2; ++h)
                ptx::mma_bf16(tmem + kTmemO + h * 256, ad0 + (uint64_t)((kk * 32) >> 4),
                              bd0 + (uint64_t)((h * 4 * kBox + kk * 2048) >> 4), idesc,
                              (lt == lt0 && kk == 0) ? 0u : 1u);
            }
            // the last tile's P buffer becomes the epilogue's staging
            if (lt != lt1 - 1) ptx::mma_commit_mc(&bars->p_free[2 * pb + half], kMaskS);
            if (half == 0) MLA_TRACE_EV(4, g);
          }
          if (failed) break;
          ptx::mma_commit(&bars->empty[st]);
          MLA_TRACE_EV(3, g);
        }
        if (failed) break;
        ptx::mma_commit(&bars->o_full);
        if (!wait_bar(&bars->o_full, seg & 1, abort)) { failed = true; break; }
        const int last_pb = (g - 1) & 1;
        MLA_TRACE_EV(7, 256 + seg);
        if (!post(kEvEpilogue | (last_pb << 4))) { failed = true; break; }
        ptx::mbar_arrive_remote(&bars->p_free[2 * last_pb], kRankS);  // staging handed back
        ptx::mbar_arrive_remote(&bars->p_free[2 * last_pb + 1], kRankS);
        ++seg;
      }
      misc->ev_type = kEvDone;
      ptx::mbar_arrive(&bars->ev_full);
      ptx::mma_commit(&bars->drain[0]);
      ptx::mbar_wait(&bars->drain[0], 0);
      if (failed) signal_abort(misc, peer);
    }
  } else if (isS && ((warp >= 2 && warp <= 5) || (warp >= 7 && warp <= 10))) {
    // ====== S-CTA: softmax, group 0 (warps 2-5) even tiles, group 1 (7-10) odd ======
    const int grp = warp >= 7 ? 1 : 0;
    const int wq = warp & 3;
    const int row = 32 * wq + lane;
    const uint32_t lane_base = (uint32_t)(32 * wq) << 16;
    const int gtid = threadIdx.x - (grp ? 224 : 64);  // 0..127 within the group
    float *m_dec = reinterpret_cast<float *>(smem + kOffMDec);
    float *lm = reinterpret_cast<float *>(smem + kOffLM);
    const uint32_t rP = ptx::map_to_rank(smem + kOffP + grp * kPBytes, kRankV);
    const uint32_t rAux = ptx::map_to_rank(smem + kOffAux + grp * kAuxBytes, kRankV);
    const uint32_t rPFullA = ptx::map_to_rank(&bars->p_full[2 * grp], kRankV);
    const uint32_t rPFullB = ptx::map_to_rank(&bars->p_full[2 * grp + 1], kRankV);
    const uint32_t rStats = ptx::map_to_rank(smem + kOffStats, kRankV);
    const uint32_t rStatsFull = ptx::map_to_rank(&bars->stats_full, kRankV);
    const float c = a.scale_log2;
    (void)gtid;
    SegIter<kSlotMajor> it;
    it.init(&a, W, t_begin, t_end, w0, s0);
    int item, lt0, lt1, n_vis, seg = 0, g = 0, r_pos = 0;
    bool whole, failed = false;
    // both softmax groups meet twice per segment end (bounded waits, one
    // phase per segment on each barrier)
    auto group_bar = [&](int which) -> bool {
      ptx::mbar_arrive(&bars->seg_sync[which]);
      return wait_bar_warp(&bars->seg_sync[which], seg & 1, abort);
    };
    while (!failed && it.next(&item, &lt0, &lt1, &whole, &n_vis)) {
      const int b = item / a.Hq;
      const int g_first = g, g_last = g + (lt1 - lt0) - 1;
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
      // -- this item's query -> TMEM: the producer put its 128 rows in the
      //    two ring stages before the segment's tiles; the group owning the
      //    first tile copies them once the previous segment's QK^T is done,
      //    then hands the stages back --
      const int rq = r_pos;
      r_pos += 2 + (lt1 - lt0);
      if (seg > 0 && !wait_bar_warp(&bars->q_free, (seg - 1) & 1, abort)) { failed = true; break; }
      if ((g_first & 1) == grp) {
        // only the owner waits: the next query cannot land before this one's
        // stages are returned below, so it is never two phases behind
        if (!wait_bar_warp(&bars->qfull[0], seg & 1, abort) ||
            !wait_bar_warp(&bars->qfull[1], seg & 1, abort)) {
          failed = true;
          break;
        }
        ptx::tc_fence_after();
        const bool real = row < a.H;  // rows past the heads read as zero
        // row = lane of this thread: stage (rq + row/64), box k holds columns
        // 64k..64k+63 as 128-byte rows, 16-byte chunk c at (c ^ row%8)
        const uint8_t *qrow = smem + kOffRing + ((rq + (row >> 6)) % kStages) * kSStage +
                              (row & 63) * 128;
#pragma unroll
        for (int k = 0; k < 9; ++k) {
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            uint32_t v[16];
#pragma unroll
            for (int c2 = 0; c2 < 4; ++c2) {
              const int c = 4 * hh + c2;
              uint4 x = *reinterpret_cast<const uint4 *>(qrow + k * kBox + ((c ^ (row & 7)) << 4));
              if (!real) x = make_uint4(0, 0, 0, 0);
              v[4 * c2] = x.x;
              v[4 * c2 + 1] = x.y;
              v[4 * c2 + 2] = x.z;
              v[4 * c2 + 3] = x.w;
            }
            ptx::tmem_st16_nc(tmem + lane_base + kTmemQ + k * 32 + hh * 16, v);
          }
        }
        ptx::tmem_st_wait();
        ptx::tc_fence_before();
        ptx::mbar_arrive(&bars->q_full);
        if (lane == 0 && wq == 0) MLA_TRACE_EV(7, seg);
        // every row is copied once q_full completes: the stages go back
        if (threadIdx.x == (grp ? 224 : 64)) {
          if (wait_bar(&bars->q_full, seg & 1, abort)) {
            ptx::mbar_arrive(&bars->empty[rq % kStages]);
            ptx::mbar_arrive(&bars->empty[(rq + 1) % kStages]);
          }
        }
      }

      // this group's row sum over its tiles of the segment, relative to m_mine
      float m_mine = -INFINITY, l_mine = 0.f;
      // A tile's maximum is published as soon as its scores are read; its P
      // leaves in two halves, each right after its 32 exponentials, so the
      // first half is in flight while the second is computed.
      uint32_t pk[32];
      float alpha_tx = 1.f;  // the tile in flight: its rescale factor, flag and index
      bool resc_tx = false;
      int gt = -1;           // -1 once both halves have left
      auto send_half = [&](int half) -> bool {
        if (gt < 0) return true;
        const uint32_t prow = rP + row * 128;
        const int ph = ((gt >> 1) - 1) & 1;
        // each half of buffer grp was last read by the V-CTA's PV of tile gt-2
        if (gt >= 2 && !wait_bar_warp(&bars->p_free[2 * grp + half], ph, abort, true)) return false;
        if (half == 1) {  // tokens 32-63
#pragma unroll
          for (int cc = 4; cc < 8; ++cc)
            ptx::st_async_v4(prow + ((cc ^ (lane & 7)) << 4), pk[4 * cc], pk[4 * cc + 1],
                             pk[4 * cc + 2], pk[4 * cc + 3], rPFullB);
          if (lane == 0 && wq == 0) MLA_TRACE_EV(6, gt);
          gt = -1;
          return true;
        }
        // half 0 (tokens 0-31) with the rescale factors and flags
        if (lane == 0 && wq == 0) MLA_TRACE_EV(5, gt);
#pragma unroll
        for (int cc = 0; cc < 4; ++cc)
          ptx::st_async_v4(prow + ((cc ^ (lane & 7)) << 4), pk[4 * cc], pk[4 * cc + 1],
                           pk[4 * cc + 2], pk[4 * cc + 3], rPFullA);
        {  // the warp's 32 factors as 8 vector stores (lanes 0-7)
          float a4[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) a4[j] = __shfl_sync(0xffffffffu, alpha_tx, (4 * lane + j) & 31);
          if (lane < 8)
            ptx::st_async_v4(rAux + (32 * wq + 4 * lane) * 4, __float_as_uint(a4[0]),
                             __float_as_uint(a4[1]), __float_as_uint(a4[2]), __float_as_uint(a4[3]),
                             rPFullA);
        }
        const uint32_t wflag = __ballot_sync(0xffffffffu, resc_tx);
        if (lane == 0) ptx::st_async_b32(rAux + 512 + wq * 4, wflag, rPFullA);
        return true;
      };
      for (int lt = lt0; lt < lt1; ++lt, ++g) {
        if ((g & 1) != grp) continue;
        const int sb = g % 3;
        if (!wait_bar_warp(&bars->s_full[g % 6], (g / 6) & 1, abort)) { failed = true; break; }
        if (lane == 0 && wq == 0) MLA_TRACE_EV(4, g);
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
        ptx::mbar_arrive(&bars->s_free[g % 6]);  // the buffer goes back to tile g+3
        const int tok0 = lt * kTile;
        if (tok0 + kTile > n_vis) {
#pragma unroll
          for (int j = 0; j < 64; ++j)
            if (tok0 + j >= n_vis) s[j] = -INFINITY;
        }
        float mx4[4] = {s[0], s[1], s[2], s[3]};
#pragma unroll
        for (int j = 4; j < 64; ++j) mx4[j & 3] = fmaxf(mx4[j & 3], s[j]);
        const float mt = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3])) * c;
        // the previous tile's maximum (published by the other group)
        if (g > 0 && !wait_bar_warp(&bars->m_ready[grp ^ 1], ((g - 1) >> 1) & 1, abort)) { failed = true; break; }
        float m_use = mt, alpha = 1.f;
        bool resc = false;
        if (lt != lt0) {
          const float m_prev = m_dec[row];
          if (mt > m_prev + kRescaleThreshold) {
            alpha = ptx::ex2(m_prev - mt);
            resc = true;
          } else {
            m_use = m_prev;
          }
        }
        m_dec[row] = m_use;
        ptx::mbar_arrive(&bars->m_ready[grp]);
        if (lane == 0 && wq == 0) MLA_TRACE_EV(0, g);
        float ls[2] = {0.f, 0.f};
        bool sent = true;
        alpha_tx = alpha;
        resc_tx = resc;
        gt = g;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
#pragma unroll
          for (int i = 16 * half; i < 16 * half + 16; ++i) {
            const float p0 = ptx::ex2(fmaf(s[2 * i], c, -m_use));
            const float p1 = ptx::ex2(fmaf(s[2 * i + 1], c, -m_use));
            ls[i & 1] += p0 + p1;
            pk[i] = ptx::pack_bf16x2(p0, p1);
          }
          sent = sent && send_half(half);
        }
        if (!sent) { failed = true; break; }
        const float lsum = ls[0] + ls[1];
        if (m_use != m_mine) {  // the maximum moved since this group's last tile
          l_mine = (m_mine == -INFINITY) ? 0.f : l_mine * ptx::ex2(m_mine - m_use);
          m_mine = m_use;
        }
        l_mine += lsum;
        if (lane == 0 && wq == 0) MLA_TRACE_EV(3, g);
      }
      // Nothing is pending here (both halves of every tile left inside the
      // loop), so this returns at once; without the call the compiler's
      // allocation spills registers in the loop above.
      if (!failed && !(send_half(0) && send_half(1))) failed = true;
      if (failed) break;
      // -- segment end: merge the two groups' row sums, statistics -> V-CTA --
      if (seg > 0 && !wait_bar_warp(&bars->stats_free, (seg - 1) & 1, abort, true)) { failed = true; break; }
      const bool owner = (g_last & 1) == grp;
      if (!owner) {
        lm[row] = m_mine;
        lm[128 + row] = l_mine;
      }
      if (!group_bar(0)) { failed = true; break; }
      if (owner) {
        const float mo = lm[row], lo = lm[128 + row];
        const float l = l_mine + ((lo > 0.f) ? lo * ptx::ex2(mo - m_mine) : 0.f);
        ptx::st_async_b32(rStats + row * 4, __float_as_uint(m_mine), rStatsFull);
        ptx::st_async_b32(rStats + (128 + row) * 4, __float_as_uint(seg_bad ? -1.f : l),
                          rStatsFull);
        if (lane == 0 && wq == 0) MLA_TRACE_EV(7, 128 + seg);
      }
      if (!group_bar(1)) { failed = true; break; }
      ++seg;
    }
    if (failed) {
      signal_abort(misc, peer);
    } else {
      // the V-CTA's last remote arrivals land before this CTA may exit
      if (seg > 0) wait_bar_warp(&bars->stats_free, (seg - 1) & 1, abort, true);
      const int gl = g - 1 - ((g - 1 - grp) & 1);  // this group's last tile
      if (gl >= 0) {
        wait_bar_warp(&bars->p_free[2 * grp], (gl >> 1) & 1, abort, true);
        wait_bar_warp(&bars->p_free[2 * grp + 1], (gl >> 1) & 1, abort, true);
      }
    }
    // items with nothing visible (or an invalid length): o = 0, lse = -inf
    if (grp == 0) {
      for (int w = pair; w < W; w += a.npairs) {
        if (item_tiles(a, w) != 0) continue;
        if (row < a.H) {
          const size_t r = (size_t)w * a.H + row;
          uint4 *d4 = reinterpret_cast<uint4 *>(a.o_lat + r * kDc);
          for (int i = 0; i < kDc * 2 / 16; ++i) d4[i] = make_uint4(0, 0, 0, 0);
          a.lse[r] = -INFINITY;
        }
      }
    }
  } else if (!isS && warp >= 2 && warp <= 5) {
    // ============ V-CTA: rescale and epilogue (warps 2-5) ============
    const int wq = warp & 3;
    const int row = 32 * wq + lane;
    const uint32_t lane_base = (uint32_t)(32 * wq) << 16;
    const uint8_t *aux = smem + kOffAux;
    const float *stats = reinterpret_cast<const float *>(smem + kOffStats);
    SegIter<kSlotMajor> it;
    it.init(&a, W, t_begin, t_end, w0, s0);
    int item, lt0, lt1, n_vis, seg = 0, nev = 0;
    bool whole, failed = false;
    for (;;) {
      if (!wait_bar_warp(&bars->ev_full, nev & 1, abort)) { failed = true; break; }
      ++nev;
      const int ev = *reinterpret_cast<volatile int *>(&misc->ev_type);
      if ((ev & 15) == kEvDone) break;
      const int pb = ev >> 4;
      if ((ev & 15) == kEvRescale) {
        // the factors arrived by st.async (seen through the MMA warp's wait)
        asm volatile("fence.acq_rel.cluster;" ::: "memory");
        const float al = *reinterpret_cast<const volatile float *>(aux + pb * kAuxBytes + row * 4);
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
      // epilogue of the next segment; P buffer pb is free staging
      if (!it.next(&item, &lt0, &lt1, &whole, &n_vis)) { failed = true; break; }
      if (!wait_bar_warp(&bars->o_full, seg & 1, abort) ||
          !wait_bar_warp(&bars->stats_full, seg & 1, abort, true)) {
        failed = true;
        break;
      }
      ptx::tc_fence_after();
      if (lane == 0 && wq == 0) MLA_TRACE_EV(7, 128 + seg);
      const float m = stats[row], l = stats[128 + row];
      __syncwarp();
      if (wq == 0 && lane == 0)  // next segment's statistics phase
        ptx::mbar_arrive_expect_tx(&bars->stats_full, kStatsBytes);
      if (lane == 0) ptx::mbar_arrive_remote(&bars->stats_free, kRankS);
      const bool seg_bad = l < 0.f;
      const float inv_l = (l > 0.f && !seg_bad) ? 1.f / l : 0.f;
      const float lse_val = l > 0.f ? (m + log2f(l)) * kLn2 : -INFINITY;
      const size_t grow = (size_t)item * a.H + row;
      // O rows leave through this warp's 4 KB of the P buffer pb (free staging):
      // each thread writes its row's 128-byte chunk (128B-swizzled, no bank
      // conflicts), then each instruction stores four whole 128-byte row
      // pieces to global memory.
      uint8_t *stg = smem + kOffP + pb * kPBytes + wq * 4096;  // 32 rows x 128 B
      const int slot_idx = 2 * pair + ((lt0 == 0) ? 1 : 0);    // partial slot
      // whole items: rows of o_lat; split pieces: rows of o_part (both bf16)
      uint8_t *dst_base = whole
          ? reinterpret_cast<uint8_t *>(a.o_lat + ((size_t)item * a.H + 32 * wq) * kDc)
          : reinterpret_cast<uint8_t *>(a.o_part + ((size_t)slot_idx * 128 + 32 * wq) * kDc);
      const size_t dst_row_bytes = kDc * 2;
      const int rows_here = whole ? min(32, a.H - 32 * wq) : 32;  // rows of this item
      // one staged 128-byte piece per row: thread = row in, lane = 16 B out
      auto flush_piece = [&](const uint32_t (&pk)[32], size_t byte_off) {
        __syncwarp();  // the previous piece's reads of the staging are done
#pragma unroll
        for (int cc = 0; cc < 8; ++cc)
          *reinterpret_cast<uint4 *>(stg + lane * 128 + ((cc ^ (lane & 7)) << 4)) =
              make_uint4(pk[4 * cc], pk[4 * cc + 1], pk[4 * cc + 2], pk[4 * cc + 3]);
        __syncwarp();
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int r = 4 * i + (lane >> 3), k = lane & 7;
          if (r < rows_here) {
            const uint4 x = *reinterpret_cast<const uint4 *>(stg + r * 128 + ((k ^ (r & 7)) << 4));
            *reinterpret_cast<uint4 *>(dst_base + r * dst_row_bytes + byte_off + k * 16) = x;
          }
        }
      };
      // the same for a split piece, stored with an evict-last L2 hint so the
      // combine kernel finds it in L2 after the rest of the cache stream
      auto flush_piece_keep = [&](const uint32_t (&pk)[32], size_t byte_off) {
        __syncwarp();
#pragma unroll
        for (int cc = 0; cc < 8; ++cc)
          *reinterpret_cast<uint4 *>(stg + lane * 128 + ((cc ^ (lane & 7)) << 4)) =
              make_uint4(pk[4 * cc], pk[4 * cc + 1], pk[4 * cc + 2], pk[4 * cc + 3]);
        __syncwarp();
        const uint64_t keep = ptx::l2_policy_evict_last();
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int r = 4 * i + (lane >> 3), k = lane & 7;
          if (r < rows_here) {
            const uint4 x = *reinterpret_cast<const uint4 *>(stg + r * 128 + ((k ^ (r & 7)) << 4));
            ptx::st_global_v4_hint(dst_base + r * dst_row_bytes + byte_off + k * 16, x, keep);
          }
        }
      };
      // the next 64 columns load from TMEM while this piece is stored
      float v[64];
      auto load64 = [&](int q) {
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          float t16[16];
          ptx::tmem_ld16(tmem + lane_base + kTmemO + q * 64 + u * 16, t16);
#pragma unroll
          for (int i = 0; i < 16; ++i) v[u * 16 + i] = t16[i];
        }
      };
      load64(0);
      ptx::tmem_ld_wait();
#pragma unroll 1
      for (int q = 0; q < kDc / 64; ++q) {
        uint32_t pk[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) pk[i] = ptx::pack_bf16x2(v[2 * i] * inv_l, v[2 * i + 1] * inv_l);
        if (q + 1 < kDc / 64) load64(q + 1);
        if (whole)
          flush_piece(pk, (size_t)q * 128);
        else
          flush_piece_keep(pk, (size_t)q * 128);
        ptx::tmem_ld_wait();
      }
      if (whole) {
        if (row < a.H) a.lse[grow] = seg_bad ? -INFINITY : lse_val;
      } else {
        if (row < a.H)
          a.lse_part[(size_t)slot_idx * 128 + row] =
              seg_bad ? __int_as_float(0x7fc00000) : lse_val;  // NaN poisons the item
      }
      if (seg_bad && row == 0) set_device_error(a.err, kDevBounds);
      __syncwarp();
      ptx::tc_fence_before();
      ptx::mbar_arrive(&bars->ev_done);
      if (lane == 0 && wq == 0) MLA_TRACE_EV(7, seg);
      ++seg;
    }
    if (failed) signal_abort(misc, peer);
  }

  // ---- teardown ----
  __syncwarp();
  ptx::tc_fence_before();
  __syncthreads();
  MLA_TRACE_CTA(2);
  if (misc->abort) {
    if (threadIdx.x == 0) set_device_error(a.err, kDevTimeout);
    __nanosleep(20000);  // copies the peer issued before it stopped have landed
  }
  ptx::cluster_sync();  // the peer no longer touches this CTA's shared memory
  ptx::tc_fence_after();
  if (warp == 1) ptx::tmem_dealloc(tmem, 512);
}

// ---------------------------------------------------------------------------
// Few heads (H <= 16, the DeepSeek-V2-Lite shape): one CTA per SM, no pair.
//
// The pair exists because O (128 rows x 512 fp32 columns) and the query do
// not fit one SM's TMEM together.  With at most 16 heads O fits once it is
// kept transposed: O^T = C^T P^T with M = 128 latent columns per MMA (four
// MMAs cover d_c = 512), N = 16 head columns and K = 64 tokens, so O^T takes
// 4 x 16 TMEM columns next to the query (288) and two 64-column score
// buffers.  Every SM then streams its own range of tiles from HBM; nothing
// crosses DSMEM.  The scores are computed as in the pair kernel (S = Q C^T,
// M = 128 rows of which the first H are heads, N = 64 tokens, A = query in
// TMEM); P (16 rows x 64 tokens, bf16) goes to shared memory as the K-major
// B operand of the PV MMAs, whose A operand is the same ring stage read
// MN-major (latent contiguous).  The plan, the pieces and the combine are
// the pair kernel's, with one CTA in the place of a pair and an item start
// charged as kShItemCost tiles.
//
// Warp roles (288 threads): warp 0 TMA producer; warps 1 and 2 QK^T issuers
// (even / odd tiles); warp 3 TMEM owner and PV issuer; warps 4-7 rescale
// O^T and run the segment epilogues (TMEM lanes 32*(w%4)...); warp 8 the
// online softmax, one head row per lane (TMEM lanes 0-31).
namespace sh {
constexpr int kThreads = 288;
constexpr int kRows = 16;                          // head rows (H <= 16)
constexpr uint32_t kQBox = kRows * 128;            // 16 rows x 128 B
constexpr uint32_t kQBytes = 9 * kQBox;            // one item's [q_lat ; q_rope]
constexpr uint32_t kOffP = kStages * kSStage;      // two P buffers
constexpr uint32_t kPBytes = kRows * 128;          // 16 rows x 64 bf16
constexpr uint32_t kOffAux = kOffP + 2 * kPBytes;  // per P buffer: alpha[16], flag
constexpr uint32_t kAuxBytes = 80;
constexpr uint32_t kOffStats = kOffAux + 2 * kAuxBytes;  // m[16], l[16]
constexpr uint32_t kOffBars = kOffStats + 2 * kRows * 4;
struct Bars {
  uint64_t full[6], empty[kStages], qfull[2];
  uint64_t q_full, q_free, s_full[2], s_free[2], p_full[2], p_free[2];
  uint64_t pv_done, ev_full, ev_done, o_full, stats_full, stats_free, drain[3];
};
constexpr uint32_t kOffMisc = kOffBars + ((sizeof(Bars) + 15) / 16) * 16;
constexpr uint32_t kSmemBytes = kOffMisc + ((sizeof(Misc) + 15) / 16) * 16;
static_assert(kSmemBytes <= 232448, "over the 227 KB shared-memory limit");
static_assert(kOffP % 1024 == 0, "P buffers must be 1024-byte aligned");
static_assert(kQBytes <= kSStage, "an item's query fits one ring stage");
// TMEM columns: query 0-287, score buffers 320 + 64 b, O^T chunk q at 448 + 16 q
constexpr uint32_t kTmemQ = 0, kTmemS = 320, kTmemO = 448;
}  // namespace sh

__global__ void __launch_bounds__(sh::kThreads, 1)
    decode_sh_kernel(const __grid_constant__ CUtensorMap tm_cache,
                     const __grid_constant__ CUtensorMap tm_qlat,
                     const __grid_constant__ CUtensorMap tm_qrope, DecodeArgs a) {
  extern __shared__ __align__(1024) uint8_t smem[];
  sh::Bars *bars = reinterpret_cast<sh::Bars *>(smem + sh::kOffBars);
  Misc *misc = reinterpret_cast<Misc *>(smem + sh::kOffMisc);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cta = blockIdx.x;
  const int W = a.B * a.Hq;
  volatile int *abort = &misc->abort;
  MLA_TRACE_CTA(0);

  // ---- setup: barriers, TMEM, this CTA's tile range ----
  if (threadIdx.x == 0) {
    misc->abort = 0;
    misc->ev_type = 0;
    misc->bad_smem = (ptx::smem_u32(smem) & 1023u) != 0;
    for (int s = 0; s < 6; ++s) ptx::mbar_init(&bars->full[s], 1);
    for (int s = 0; s < kStages; ++s) ptx::mbar_init(&bars->empty[s], 1);
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(&bars->qfull[i], 1);
      ptx::mbar_init(&bars->s_full[i], 1);
      ptx::mbar_init(&bars->s_free[i], 32);
      ptx::mbar_init(&bars->p_full[i], 32);
      ptx::mbar_init(&bars->p_free[i], 1);
    }
    ptx::mbar_init(&bars->q_full, 32);
    ptx::mbar_init(&bars->q_free, 2);
    ptx::mbar_init(&bars->pv_done, 1);
    ptx::mbar_init(&bars->ev_full, 1);
    ptx::mbar_init(&bars->ev_done, 128);
    ptx::mbar_init(&bars->o_full, 1);
    ptx::mbar_init(&bars->stats_full, 32);
    ptx::mbar_init(&bars->stats_free, 128);
    for (int i = 0; i < 3; ++i) ptx::mbar_init(&bars->drain[i], 1);
    ptx::fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    ptx::tma_prefetch_desc(&tm_cache);
    ptx::tma_prefetch_desc(&tm_qlat);
    ptx::tma_prefetch_desc(&tm_qrope);
  }
  if (warp == 3) ptx::tmem_alloc(&misc->tmem, 512);
  ptx::grid_dependency_wait();
  ptx::launch_dependents();
  {
    // tiles per item -> scan (scratch in the ring) -> this CTA's range
    int *pre = reinterpret_cast<int *>(smem);
    bool any_bad = false;
    for (int u = threadIdx.x; u < W; u += blockDim.x) {
      bool bad = false;
      const int n = visible_len(a, u, &bad);
      any_bad |= bad;
      const int nt = (n + kTile - 1) / kTile;
      pre[u + 1] = nt > 0 ? nt + kShItemCost : 0;
    }
    if (any_bad && cta == 0) set_device_error(a.err, kDevBounds);
    __syncthreads();
    if (warp == 0) {
      int running = 0;
      for (int base = 0; base < W; base += 32) {
        const int idx = base + lane;
        int v = idx < W ? pre[idx + 1] : 0;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const int u = __shfl_up_sync(0xffffffffu, v, off);
          if (lane >= off) v += u;
        }
        if (idx < W) pre[idx + 1] = running + v;
        running += __shfl_sync(0xffffffffu, v, 31);
      }
      if (lane == 0) pre[0] = 0;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      const int t_total = pre[W];
      const int per = (t_total + a.npairs - 1) / a.npairs;
      const int tb = min(t_total, cta * per);
      const int te = min(t_total, tb + per);
      int lo = 0, hi = W;  // first item whose tile range ends after tb
      while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (pre[mid + 1] <= tb) lo = mid + 1;
        else hi = mid;
      }
      misc->t_begin = tb;
      misc->t_end = te;
      misc->w0 = lo;
      misc->s0 = lo < W ? pre[lo] : t_total;
      misc->t_total = t_total;
      if (cta == 0) a.plan[0] = per;
    }
    if (cta == 0)  // the plan of the combine kernel
      for (int w = threadIdx.x; w <= W; w += blockDim.x) a.plan[1 + w] = pre[w];
  }
  ptx::tc_fence_before();
  __syncthreads();  // the scratch is the ring: read before the first load
  ptx::tc_fence_after();
  const uint32_t tmem = misc->tmem;
  const bool bad_smem = misc->bad_smem != 0;
  const int t_begin = misc->t_begin, t_end = misc->t_end, w0 = misc->w0, s0 = misc->s0;
  MLA_TRACE_CTA(1);
  SegIter<false, kShItemCost> it;
  it.init(&a, W, t_begin, t_end, w0, s0);
  int item, lt0, lt1, n_vis;
  bool whole;

  if (bad_smem) {
    if (threadIdx.x == 0) set_device_error(a.err, kDevTimeout);
  } else if (warp == 0) {
    // ===================== TMA producer =====================
    // ring position r: one stage for each segment's query, then its tiles
    int g = 0, r = 0, seg = 0;
    bool failed = false;
    TableWindow cur;
    while (!failed && !*abort && it.next(&item, &lt0, &lt1, &whole, &n_vis)) {
      const int b = item / a.Hq;
      cur.reset(a.block_table + (size_t)b * a.max_blocks, lt1);
      {
        const int st = r % kStages;
        if (r >= kStages && !wait_bar_warp(&bars->empty[st], ((r / kStages) - 1) & 1, abort)) {
          failed = true;
          break;
        }
        if (lane == 0) {
          uint8_t *dst = smem + st * kSStage;
          uint64_t *qb = &bars->qfull[seg & 1];
          ptx::mbar_arrive_expect_tx(qb, sh::kQBytes);
          ptx::tma_load_3d(dst, &tm_qlat, qb, 0, item * a.H, 0);  // 8 latent boxes
          ptx::tma_load_2d(dst + 8 * sh::kQBox, &tm_qrope, qb, 0, item * a.H);
        }
        ++r;
      }
      for (int lt = lt0; lt < lt1; ++lt, ++g, ++r) {
        const int st = r % kStages;
        if (r >= kStages && !wait_bar_warp(&bars->empty[st], ((r / kStages) - 1) & 1, abort)) {
          failed = true;
          break;
        }
        int blk = cur.at(lt, lane);
        if (blk < 0 || blk >= a.num_blocks) blk = 0;  // reported by the softmax warp
        if (lane == 0) {
          SH_TRACE_EV(1, 8, g);
          uint64_t *fb = &bars->full[g % 6];
          ptx::mbar_arrive_expect_tx(fb, 9 * kBox);
          ptx::tma_load_3d(smem + st * kSStage, &tm_cache, fb, 0, blk * kTile, 0);
        }
      }
      ++seg;
    }
    if (failed) atomicExch(&misc->abort, 1);
    // leave only after every stage this CTA filled was released
    if (!*abort)
      for (int k = r - kStages < 0 ? 0 : r - kStages; k < r; ++k)
        wait_bar_warp(&bars->empty[k % kStages], (k / kStages) & 1, abort);
  } else if (warp == 1 || warp == 2) {
    // ========== QK^T issuers: warp 1 even tiles, warp 2 odd ==========
    if (lane == 0) {
      const int mine = warp - 1;
      const uint32_t idesc = ptx::idesc_bf16(128, kTile, false, false);
      const uint64_t ring_desc = ptx::smem_desc(ptx::smem_u32(smem), 16, 1024, ptx::kSw128);
      int g = 0, r = 0, seg = 0;
      bool failed = false;
      while (!failed && it.next(&item, &lt0, &lt1, &whole, &n_vis)) {
        if (!wait_bar(&bars->q_full, seg & 1, abort)) { failed = true; break; }
        ptx::tc_fence_after();
        ++r;  // the segment's query stage
        for (int lt = lt0; lt < lt1; ++lt, ++g, ++r) {
          if ((g & 1) != mine) continue;
          const int st = r % kStages, sb = g & 1;
          if (!wait_bar(&bars->full[g % 6], (g / 6) & 1, abort)) { failed = true; break; }
          SH_TRACE_EV(1, 1, g);
          // buffer sb last held tile g-2, read by the softmax warp
          if (g >= 2 && !wait_bar(&bars->s_free[sb], ((g - 2) >> 1) & 1, abort)) {
            failed = true;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t d = tmem + sh::kTmemS + sb * kTile;
          const uint64_t bs = ring_desc + (uint64_t)((st * kSStage) >> 4);
#pragma unroll
          for (int kk = 0; kk < 36; ++kk)  // 9 boxes (8 latent + RoPE) x 4 k-steps of 16
            ptx::mma_bf16_ts(d, tmem + sh::kTmemQ + kk * 8,
                             bs + (uint64_t)((((kk >> 2) * kBox) + (kk & 3) * 32) >> 4), idesc,
                             kk != 0);
          ptx::mma_commit(&bars->s_full[sb]);
          SH_TRACE_EV(1, 2, g);
        }
        if (failed) break;
        ptx::mma_commit(&bars->q_free);
        ++seg;
      }
      uint64_t *dr = &bars->drain[mine];
      ptx::mma_commit(dr);
      ptx::mbar_wait(dr, 0);
      if (failed) atomicExch(&misc->abort, 1);
    }
  } else if (warp == 3) {
    // ===================== PV issuer: O^T += C^T P^T =====================
    if (lane == 0) {
      const uint32_t idesc = ptx::idesc_bf16(128, sh::kRows, true, false);
      // A: the stage's latent boxes MN-major (64 latent columns per 128-byte
      // row, boxes 8 KB apart, 8 tokens per 1 KB); B: P, K-major
      const uint64_t ring_desc = ptx::smem_desc(ptx::smem_u32(smem), kBox, 1024, ptx::kSw128);
      const uint64_t p_desc =
          ptx::smem_desc(ptx::smem_u32(smem + sh::kOffP), 16, 1024, ptx::kSw128);
      const uint8_t *aux = smem + sh::kOffAux;
      int g = 0, r = 0, seg = 0, nev = 0, npv = 0;
      bool failed = false;
      auto post = [&](int type) -> bool {
        misc->ev_type = type;
        ptx::mbar_arrive(&bars->ev_full);
        const bool ok = wait_bar(&bars->ev_done, nev & 1, abort);
        ++nev;
        return ok;
      };
      while (!failed && it.next(&item, &lt0, &lt1, &whole, &n_vis)) {
        ++r;  // the segment's query stage
        for (int lt = lt0; lt < lt1; ++lt, ++g, ++r) {
          const int st = r % kStages, pb = g & 1;
          if (!wait_bar(&bars->full[g % 6], (g / 6) & 1, abort) ||
              !wait_bar(&bars->p_full[pb], (g >> 1) & 1, abort)) {
            failed = true;
            break;
          }
          SH_TRACE_EV(0, 1, g);
          const uint32_t flag =
              *reinterpret_cast<const volatile uint32_t *>(aux + pb * sh::kAuxBytes + 64);
          if (lt != lt0 && flag != 0) {
            // O^T *= alpha (per head column) once every PV so far has accumulated
            ptx::mma_commit(&bars->pv_done);
            if (!wait_bar(&bars->pv_done, npv & 1, abort)) { failed = true; break; }
            ++npv;
            if (!post(kEvRescale | (pb << 4))) { failed = true; break; }
          }
          ptx::tc_fence_after();
          const uint64_t ad = ring_desc + (uint64_t)((st * kSStage) >> 4);
          const uint64_t bd = p_desc + (uint64_t)((pb * sh::kPBytes) >> 4);
#pragma unroll
          for (int kk = 0; kk < kTile / 16; ++kk)
#pragma unroll
            for (int q = 0; q < kDc / 128; ++q)
              ptx::mma_bf16(tmem + sh::kTmemO + q * sh::kRows,
                            ad + (uint64_t)((2 * q * kBox + kk * 2048) >> 4),
                            bd + (uint64_t)((kk * 32) >> 4), idesc,
                            (lt == lt0 && kk == 0) ? 0u : 1u);
          ptx::mma_commit(&bars->p_free[pb]);
          ptx::mma_commit(&bars->empty[st]);
          SH_TRACE_EV(0, 3, g);
        }
        if (failed) break;
        ptx::mma_commit(&bars->o_full);
        if (!wait_bar(&bars->o_full, seg & 1, abort)) { failed = true; break; }
        SH_TRACE_EV(0, 7, seg);
        if (!post(kEvEpilogue)) { failed = true; break; }
        SH_TRACE_EV(0, 7, 128 + seg);
        ++seg;
      }
      misc->ev_type = kEvDone;
      ptx::mbar_arrive(&bars->ev_full);
      ptx::mma_commit(&bars->drain[2]);
      ptx::mbar_wait(&bars->drain[2], 0);
      if (failed) atomicExch(&misc->abort, 1);
    }
  } else if (warp >= 4 && warp <= 7) {
    // ============ O^T rescale and segment epilogues ============
    // lane of TMEM = latent column c within each 128-column chunk
    const int wq = warp & 3;
    const int cl = 32 * wq + lane;
    const uint32_t lane_base = (uint32_t)(32 * wq) << 16;
    const uint8_t *aux = smem + sh::kOffAux;
    const float *stats = reinterpret_cast<const float *>(smem + sh::kOffStats);
    int seg = 0, nev = 0;
    bool failed = false;
    for (;;) {
      if (!wait_bar_warp(&bars->ev_full, nev & 1, abort)) { failed = true; break; }
      ++nev;
      const int ev = *reinterpret_cast<volatile int *>(&misc->ev_type);
      if ((ev & 15) == kEvDone) break;
      if ((ev & 15) == kEvRescale) {
        const float *al = reinterpret_cast<const float *>(aux + (ev >> 4) * sh::kAuxBytes);
        float f[sh::kRows];
#pragma unroll
        for (int h = 0; h < sh::kRows; ++h) f[h] = al[h];
        ptx::tc_fence_after();
#pragma unroll 1
        for (int q = 0; q < kDc / 128; ++q) {
          float v[16];
          ptx::tmem_ld16(tmem + lane_base + sh::kTmemO + q * sh::kRows, v);
          ptx::tmem_ld_wait();
#pragma unroll
          for (int h = 0; h < 16; ++h) v[h] *= f[h];
          ptx::tmem_st16(tmem + lane_base + sh::kTmemO + q * sh::kRows, v);
        }
        ptx::tmem_st_wait();
        ptx::tc_fence_before();
        ptx::mbar_arrive(&bars->ev_done);
        continue;
      }
      // epilogue of the next segment (its PVs are complete)
      if (!it.next(&item, &lt0, &lt1, &whole, &n_vis)) { failed = true; break; }
      if (!wait_bar_warp(&bars->stats_full, seg & 1, abort)) { failed = true; break; }
      ptx::tc_fence_after();
      float inv_l[sh::kRows];
      bool seg_bad = false;
#pragma unroll
      for (int h = 0; h < sh::kRows; ++h) {
        const float l = stats[sh::kRows + h];
        seg_bad |= l < 0.f;
        inv_l[h] = l > 0.f ? 1.f / l : 0.f;
      }
      const float m_me = stats[lane & 15], l_me = stats[sh::kRows + (lane & 15)];
      ptx::mbar_arrive(&bars->stats_free);
      if (seg_bad) {
#pragma unroll
        for (int h = 0; h < sh::kRows; ++h) inv_l[h] = 0.f;
      }
      const int slot_idx = 2 * cta + ((lt0 == 0) ? 1 : 0);  // partial slot
      __nv_bfloat16 *dst = whole ? a.o_lat + (size_t)item * a.H * kDc
                                 : a.o_part + (size_t)slot_idx * 128 * kDc;
#pragma unroll 1
      for (int q = 0; q < kDc / 128; ++q) {
        float v[16];
        ptx::tmem_ld16(tmem + lane_base + sh::kTmemO + q * sh::kRows, v);
        ptx::tmem_ld_wait();
#pragma unroll
        for (int h = 0; h < sh::kRows; ++h)
          if (h < a.H) dst[(size_t)h * kDc + q * 128 + cl] = __float2bfloat16_rn(v[h] * inv_l[h]);
      }
      if (wq == 0 && lane < a.H) {
        const float lse_val = l_me > 0.f ? (m_me + log2f(l_me)) * kLn2 : -INFINITY;
        if (whole)
          a.lse[(size_t)item * a.H + lane] = seg_bad ? -INFINITY : lse_val;
        else  // NaN poisons the item in the combine
          a.lse_part[(size_t)slot_idx * 128 + lane] = seg_bad ? __int_as_float(0x7fc00000) : lse_val;
      }
      if (seg_bad && wq == 0 && lane == 0) set_device_error(a.err, kDevBounds);
      __syncwarp();
      ptx::tc_fence_before();
      ptx::mbar_arrive(&bars->ev_done);
      ++seg;
    }
    if (failed) atomicExch(&misc->abort, 1);
  } else if (warp == 8) {
    // ============ online softmax: lane = head row (TMEM lanes 0-31) ============
    const int row = lane;
    const bool real = row < a.H;
    const float c = a.scale_log2;
    float *stats = reinterpret_cast<float *>(smem + sh::kOffStats);
    uint8_t *aux = smem + sh::kOffAux;
    int g = 0, r = 0, seg = 0;
    bool failed = false;
    while (!failed && it.next(&item, &lt0, &lt1, &whole, &n_vis)) {
      const int b = item / a.Hq;
      bool seg_bad;
      {  // block-table entries this segment reads
        const int32_t *tbl = a.block_table + (size_t)b * a.max_blocks;
        bool bad = false;
        for (int lt = lt0 + lane; lt < lt1; lt += 32) {
          const int blk = tbl[lt];
          bad |= (blk < 0 || blk >= a.num_blocks);
        }
        seg_bad = __any_sync(0xffffffffu, bad);
      }
      // -- the item's query -> TMEM, once the previous segment's QK^T is done --
      const int rq = r;
      r += 1 + (lt1 - lt0);
      if (seg > 0 && !wait_bar_warp(&bars->q_free, (seg - 1) & 1, abort)) { failed = true; break; }
      if (!wait_bar_warp(&bars->qfull[seg & 1], (seg >> 1) & 1, abort)) { failed = true; break; }
      ptx::tc_fence_after();
      {
        // box k holds columns 64k..64k+63 of the 16 rows as 128-byte rows,
        // 16-byte chunk c of row h at (c ^ h%8)
        const uint8_t *qrow = smem + (rq % kStages) * kSStage + (row & 15) * 128;
#pragma unroll
        for (int k = 0; k < 9; ++k) {
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            uint32_t v[16];
#pragma unroll
            for (int c2 = 0; c2 < 4; ++c2) {
              const int cc = 4 * hh + c2;
              uint4 x = *reinterpret_cast<const uint4 *>(qrow + k * sh::kQBox + ((cc ^ (row & 7)) << 4));
              if (!real) x = make_uint4(0, 0, 0, 0);
              v[4 * c2] = x.x;
              v[4 * c2 + 1] = x.y;
              v[4 * c2 + 2] = x.z;
              v[4 * c2 + 3] = x.w;
            }
            ptx::tmem_st16_nc(tmem + sh::kTmemQ + k * 32 + hh * 16, v);
          }
        }
      }
      ptx::tmem_st_wait();
      ptx::tc_fence_before();
      ptx::mbar_arrive(&bars->q_full);
      if (lane == 0) SH_TRACE_EV(1, 7, seg);
      __syncwarp();  // every lane has read the stage
      if (lane == 0) ptx::mbar_arrive(&bars->empty[rq % kStages]);

      float m_run = -INFINITY, l_run = 0.f;
      for (int lt = lt0; lt < lt1; ++lt, ++g) {
        const int sb = g & 1;
        if (!wait_bar_warp(&bars->s_full[sb], (g >> 1) & 1, abort)) { failed = true; break; }
        if (lane == 0) SH_TRACE_EV(1, 4, g);
        ptx::tc_fence_after();
        float s[64];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          float v[16];
          ptx::tmem_ld16(tmem + sh::kTmemS + sb * kTile + q * 16, v);
#pragma unroll
          for (int i = 0; i < 16; ++i) s[q * 16 + i] = v[i];
        }
        ptx::tmem_ld_wait();
        ptx::tc_fence_before();
        ptx::mbar_arrive(&bars->s_free[sb]);  // the buffer goes back to tile g+2
        const int tok0 = lt * kTile;
        if (tok0 + kTile > n_vis) {
#pragma unroll
          for (int j = 0; j < 64; ++j)
            if (tok0 + j >= n_vis) s[j] = -INFINITY;
        }
        float mx4[4] = {s[0], s[1], s[2], s[3]};
#pragma unroll
        for (int j = 4; j < 64; ++j) mx4[j & 3] = fmaxf(mx4[j & 3], s[j]);
        const float mt = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3])) * c;
        float m_use = mt, alpha = 1.f;
        bool resc = false;
        if (lt != lt0) {
          if (mt > m_run + kRescaleThreshold) {
            alpha = ptx::ex2(m_run - mt);
            resc = true;
          } else {
            m_use = m_run;
          }
        }
        uint32_t pk[32];
        float ls[2] = {0.f, 0.f};
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float p0 = ptx::ex2(fmaf(s[2 * i], c, -m_use));
          const float p1 = ptx::ex2(fmaf(s[2 * i + 1], c, -m_use));
          ls[i & 1] += p0 + p1;
          pk[i] = ptx::pack_bf16x2(p0, p1);
        }
        l_run = (lt == lt0) ? ls[0] + ls[1] : l_run * alpha + (ls[0] + ls[1]);
        m_run = m_use;
        // P buffer sb was last read by the PV of tile g-2
        if (g >= 2 && !wait_bar_warp(&bars->p_free[sb], ((g - 2) >> 1) & 1, abort)) {
          failed = true;
          break;
        }
        if (row < sh::kRows) {
          uint8_t *prow = smem + sh::kOffP + sb * sh::kPBytes + row * 128;
#pragma unroll
          for (int cc = 0; cc < 8; ++cc)
            *reinterpret_cast<uint4 *>(prow + ((cc ^ (row & 7)) << 4)) =
                real ? make_uint4(pk[4 * cc], pk[4 * cc + 1], pk[4 * cc + 2], pk[4 * cc + 3])
                     : make_uint4(0, 0, 0, 0);
          reinterpret_cast<float *>(aux + sb * sh::kAuxBytes)[row] = real ? alpha : 1.f;
        }
        const uint32_t flag = __ballot_sync(0xffffffffu, resc && real);
        if (lane == 0) *reinterpret_cast<uint32_t *>(aux + sb * sh::kAuxBytes + 64) = flag;
        ptx::fence_proxy_async_smem();  // P is read by the tensor core (async proxy)
        ptx::mbar_arrive(&bars->p_full[sb]);
        if (lane == 0) SH_TRACE_EV(1, 3, g);
      }
      if (failed) break;
      // -- segment end: the row statistics for the epilogue --
      if (seg > 0 && !wait_bar_warp(&bars->stats_free, (seg - 1) & 1, abort)) { failed = true; break; }
      if (row < sh::kRows) {
        stats[row] = m_run;
        stats[sh::kRows + row] = (seg_bad && real) ? -1.f : l_run;
      }
      ptx::mbar_arrive(&bars->stats_full);
      ++seg;
    }
    if (failed) atomicExch(&misc->abort, 1);
    // items with nothing visible (or an invalid length): o = 0, lse = -inf
    for (int w = cta; w < W; w += a.npairs) {
      if (item_tiles(a, w) != 0) continue;
      if (real) {
        const size_t rr = (size_t)w * a.H + row;
        uint4 *d4 = reinterpret_cast<uint4 *>(a.o_lat + rr * kDc);
        for (int i = 0; i < kDc * 2 / 16; ++i) d4[i] = make_uint4(0, 0, 0, 0);
        a.lse[rr] = -INFINITY;
      }
    }
  }

  // ---- teardown ----
  __syncwarp();
  ptx::tc_fence_before();
  __syncthreads();
  MLA_TRACE_CTA(2);
  if (misc->abort) {
    if (threadIdx.x == 0) set_device_error(a.err, kDevTimeout);
    __nanosleep(20000);  // copies issued before the stop have landed
  }
  ptx::tc_fence_after();
  if (warp == 3) ptx::tmem_dealloc(tmem, 512);
}

// Merge the partial pieces of every item that was cut between pairs
// (log-sum-exp weights): one warp per output row (item w, head h), eight rows
// per block.  Lane i weighs piece p0 + i (pieces of one item <= 32 per round),
// then each lane accumulates 16 consecutive columns over the pieces, so every
// piece row is read as 2 KB of coalesced loads.  Rows of items written
// directly by their pair return at once.
constexpr int kCombineRows = 8;

// Columns 16 lane .. 16 lane + 15 of one bf16 piece row, as fp32.
__device__ __forceinline__ void load_piece16(const __nv_bfloat16 *row, int lane, float (&v)[16]) {
  const uint4 *src = reinterpret_cast<const uint4 *>(row) + lane * 2;
  const uint4 x0 = src[0], x1 = src[1];
  const uint32_t w[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    v[2 * i] = __uint_as_float(w[i] << 16);
    v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}
template <bool kSlotMajor, int kCost = kItemCost>
__global__ void __launch_bounds__(32 * kCombineRows) combine_tc_kernel(DecodeArgs a) {
  // launched early, behind the decode grid: its pieces are complete and
  // visible only after this wait; the next kernel may launch after it
  ptx::grid_dependency_wait();
  ptx::launch_dependents();
#ifdef MLA_TRACE
  if (threadIdx.x == 0) atomicMin(&g_trace_comb[0], ptx::globaltimer_ns());
  struct CombEnd {
    __device__ ~CombEnd() {
      __syncthreads();
      if (threadIdx.x == 0) atomicMax(&g_trace_comb[1], ptx::globaltimer_ns());
    }
  } comb_end;
#endif
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long rowg = (long)blockIdx.x * kCombineRows + warp;
  const int W = a.B * a.Hq;
  if (rowg >= (long)W * a.H) return;
  const int w = (int)(rowg / a.H), h = (int)(rowg % a.H);
  int per, f, e, grp_pair0;  // the item's tiles are units f .. e - 1 of its group
  if constexpr (kSlotMajor) {
    // the item's plan position and slot group (as in decode_tc_kernel)
    const int u = (w % a.Hq) * a.B + w / a.Hq;
    const int ngroups = a.plan[0];
    const int grp = ngroups > 1 ? w % a.Hq : 0;
    const int *pre = a.plan + 1 + a.Hq;
    const int base = pre[grp * (W / ngroups)];
    per = a.plan[1 + grp];
    const int s = pre[u] - base;
    e = pre[u + 1] - base;
    if (e <= s) return;
    f = s + kCost;
    grp_pair0 = grp * (a.npairs / ngroups);
  } else {
    per = a.plan[0];
    const int s = a.plan[1 + w];
    e = a.plan[2 + w];
    if (e <= s) return;
    f = s + kCost;
    grp_pair0 = 0;
  }
  if (per <= 0) return;
  const int p0 = f / per, p1 = (e - 1) / per;
  if (p0 == p1) return;  // written directly by its pair
  auto slot_of = [&](int p) { return 2 * (grp_pair0 + p) + ((f < p * per) ? 0 : 1); };
  __nv_bfloat16 *dst = a.o_lat + (size_t)rowg * kDc;
  if (p1 == p0 + 1) {
    // two pieces (an item cut once): every load in flight at once
    const int s0 = slot_of(p0), s1 = slot_of(p1);
    const float l0 = a.lse_part[(size_t)s0 * 128 + h], l1 = a.lse_part[(size_t)s1 * 128 + h];
    float v0[16], v1[16];
    load_piece16(a.o_part + ((size_t)s0 * 128 + h) * kDc, lane, v0);
    load_piece16(a.o_part + ((size_t)s1 * 128 + h) * kDc, lane, v1);
    const float mx2 = fmaxf(l0, l1);
    if (isnan(l0) || isnan(l1) || mx2 == -INFINITY) {
      reinterpret_cast<uint4 *>(dst)[lane] = make_uint4(0, 0, 0, 0);
      reinterpret_cast<uint4 *>(dst)[lane + 32] = make_uint4(0, 0, 0, 0);
      if (lane == 0) a.lse[rowg] = -INFINITY;
      return;
    }
    const float w0 = expf(l0 - mx2), w1 = expf(l1 - mx2);
    const float inv2 = 1.f / (w0 + w1), a0 = w0 * inv2, a1 = w1 * inv2;
    uint32_t pk[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
      pk[i] = ptx::pack_bf16x2(fmaf(a1, v1[2 * i], a0 * v0[2 * i]),
                               fmaf(a1, v1[2 * i + 1], a0 * v0[2 * i + 1]));
    uint4 *d4 = reinterpret_cast<uint4 *>(dst) + lane * 2;
    d4[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
    d4[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
    if (lane == 0) a.lse[rowg] = mx2 + logf(w0 + w1);
    return;
  }
  // maximum and sum of exp(lse) over the pieces
  float mx = -INFINITY;
  bool poison = false;
  for (int p = p0 + lane; p <= p1; p += 32) {
    const float v = a.lse_part[(size_t)slot_of(p) * 128 + h];
    poison |= isnan(v);
    mx = fmaxf(mx, v);
  }
#pragma unroll
  for (int off = 16; off; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
  poison = __any_sync(0xffffffffu, poison);
  if (poison || mx == -INFINITY) {
    reinterpret_cast<uint4 *>(dst)[lane] = make_uint4(0, 0, 0, 0);
    reinterpret_cast<uint4 *>(dst)[lane + 32] = make_uint4(0, 0, 0, 0);
    if (lane == 0) a.lse[rowg] = -INFINITY;
    return;
  }
  float sum = 0.f;
  for (int p = p0 + lane; p <= p1; p += 32)
    sum += expf(a.lse_part[(size_t)slot_of(p) * 128 + h] - mx);
#pragma unroll
  for (int off = 16; off; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
  const float inv = 1.f / sum;
  float acc[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) acc[i] = 0.f;
  for (int base = p0; base <= p1; base += 32) {
    const int p_l = base + lane;
    const float wl = p_l <= p1 ? expf(a.lse_part[(size_t)slot_of(p_l) * 128 + h] - mx) * inv : 0.f;
    const int n = min(32, p1 - base + 1);
    int j = 0;
    for (; j + 4 <= n; j += 4) {  // four pieces' loads in flight at once
      uint4 x[4][2];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const uint4 *src = reinterpret_cast<const uint4 *>(
                               a.o_part + ((size_t)slot_of(base + j + u) * 128 + h) * kDc) +
                           lane * 2;
        x[u][0] = src[0];
        x[u][1] = src[1];
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const float wgt = __shfl_sync(0xffffffffu, wl, j + u);
        const uint32_t wd[8] = {x[u][0].x, x[u][0].y, x[u][0].z, x[u][0].w,
                                x[u][1].x, x[u][1].y, x[u][1].z, x[u][1].w};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          acc[2 * i] = fmaf(wgt, __uint_as_float(wd[i] << 16), acc[2 * i]);
          acc[2 * i + 1] = fmaf(wgt, __uint_as_float(wd[i] & 0xffff0000u), acc[2 * i + 1]);
        }
      }
    }
    for (; j < n; ++j) {
      const float wgt = __shfl_sync(0xffffffffu, wl, j);
      float v[16];
      load_piece16(a.o_part + ((size_t)slot_of(base + j) * 128 + h) * kDc, lane, v);
#pragma unroll
      for (int i = 0; i < 16; ++i) acc[i] = fmaf(wgt, v[i], acc[i]);
    }
  }
  uint32_t pk[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) pk[i] = ptx::pack_bf16x2(acc[2 * i], acc[2 * i + 1]);
  uint4 *d4 = reinterpret_cast<uint4 *>(dst) + lane * 2;
  d4[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
  d4[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
  if (lane == 0) a.lse[rowg] = mx + logf(sum);
}

// Two piece slots of 128 rows per pair, or per CTA of the few-heads kernel.
size_t piece_slots(int H) { return (size_t)2 * (H <= sh::kRows ? kNumSMs : kMaxPairs); }
size_t part_bytes(int H) {
  return align_up(piece_slots(H) * 128 * kDc * sizeof(__nv_bfloat16), 256);
}
size_t lse_part_bytes(int H) { return align_up(piece_slots(H) * 128 * sizeof(float), 256); }
size_t plan_bytes(int B, int Hq) {
  return align_up(((size_t)B * Hq + 2 + Hq) * sizeof(int), 256);
}

// Test hook: at most this many CTA pairs take part in the split plan (0:
// no limit).  Set through mla_debug_set_decode_pairs.
std::atomic<int> g_pairs_limit{0};

// Co-resident clusters of two CTAs for this kernel (some GPCs may not fit a
// whole number of pairs), capped at 74; looked up once per device.
int pairs_on_device() {
  static int cached[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (cached[dev] > 0) return cached[dev];
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * kMaxPairs, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmemBytes;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, decode_tc_kernel<false>, &cfg) != cudaSuccess ||
      n <= 0) {
    cudaGetLastError();
    n = kMaxPairs;
  }
  if (n > kMaxPairs) n = kMaxPairs;
  cached[dev] = n;
  return n;
}

int pairs_for_device() {
  const int n = pairs_on_device();
  const int limit = g_pairs_limit.load(std::memory_order_relaxed);
  return (limit > 0 && limit < n) ? limit : n;
}

// CTAs of the few-heads kernel: one per SM (at most 148), or the test
// hook's limit.
int ctas_for_device() {
  static int cached[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (cached[dev] <= 0) {
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      return 0;
    }
    cached[dev] = sms < kNumSMs ? sms : kNumSMs;
  }
  const int limit = g_pairs_limit.load(std::memory_order_relaxed);
  return (limit > 0 && limit < cached[dev]) ? limit : cached[dev];
}

// Log-sum-exp merge of P pieces of the same rows (the outputs of calls over
// disjoint block ranges): one thread per 8 columns of an output row, four
// pieces' loads in flight at a time.  A piece with lse = -inf (nothing
// visible in its range) weighs nothing; rows with nothing visible in any
// piece get o = 0, lse = -inf.
__global__ void __launch_bounds__(256) combine_pieces_kernel(const __nv_bfloat16 *o_pieces,
                                                             const float *lse_pieces, int P,
                                                             long rows, __nv_bfloat16 *o_lat,
                                                             float *lse) {
  const long t = (long)blockIdx.x * 256 + threadIdx.x;
  const long row = t / (kDc / 8);
  const int c8 = (int)(t % (kDc / 8));
  if (row >= rows) return;
  uint4 *dst = reinterpret_cast<uint4 *>(o_lat + (size_t)row * kDc) + c8;
  float mx = -INFINITY;
  for (int p = 0; p < P; ++p) mx = fmaxf(mx, lse_pieces[(size_t)p * rows + row]);
  if (!(mx > -INFINITY)) {  // nothing visible (or a NaN)
    *dst = make_uint4(0, 0, 0, 0);
    if (c8 == 0) lse[row] = -INFINITY;
    return;
  }
  float sum = 0.f, acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.f;
#pragma unroll 4
  for (int p = 0; p < P; ++p) {
    const float wgt = expf(lse_pieces[(size_t)p * rows + row] - mx);
    const uint4 x = reinterpret_cast<const uint4 *>(o_pieces + ((size_t)p * rows + row) * kDc)[c8];
    const uint32_t wd[4] = {x.x, x.y, x.z, x.w};
    sum += wgt;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      acc[2 * i] = fmaf(wgt, __uint_as_float(wd[i] << 16), acc[2 * i]);
      acc[2 * i + 1] = fmaf(wgt, __uint_as_float(wd[i] & 0xffff0000u), acc[2 * i + 1]);
    }
  }
  const float inv = 1.f / sum;
  *dst = make_uint4(ptx::pack_bf16x2(acc[0] * inv, acc[1] * inv),
                    ptx::pack_bf16x2(acc[2] * inv, acc[3] * inv),
                    ptx::pack_bf16x2(acc[4] * inv, acc[5] * inv),
                    ptx::pack_bf16x2(acc[6] * inv, acc[7] * inv));
  if (c8 == 0) lse[row] = mx + logf(sum);
}

}  // namespace

#ifdef MLA_TRACE
extern "C" __attribute__((visibility("default"))) int mla_debug_read_trace(void *host,
                                                                          size_t bytes) {
  if (bytes < sizeof(g_trace) + sizeof(g_trace_cta) + sizeof(g_trace_comb)) return -1;
  if (cudaMemcpyFromSymbol(host, g_trace, sizeof(g_trace)) != cudaSuccess) return -1;
  if (cudaMemcpyFromSymbol(static_cast<char *>(host) + sizeof(g_trace), g_trace_cta,
                           sizeof(g_trace_cta)) != cudaSuccess)
    return -1;
  return cudaMemcpyFromSymbol(static_cast<char *>(host) + sizeof(g_trace) + sizeof(g_trace_cta),
                              g_trace_comb, sizeof(g_trace_comb)) == cudaSuccess ? 0 : -1;
}
#endif

extern "C" __attribute__((visibility("default"))) int mla_debug_set_decode_pairs(int pairs) {
  return g_pairs_limit.exchange(pairs > 0 ? pairs : 0);
}

bool tc_decode_supported(const mla_dims &d, int B, int Hq) {
  return d.dtype == MLA_BF16 && d.d_c == kDc && d.d_r == kDr && d.block_size == kTile &&
         d.H <= 128 && (long)B * Hq <= kMaxItems;
}

size_t tc_decode_workspace_bytes(int B, int Hq, const mla_dims &d) {
  return kWsHeader + part_bytes(d.H) + lse_part_bytes(d.H) + plan_bytes(B, Hq);
}

cudaError_t launch_decode_tc(const void *q_lat, const void *q_rope, const void *cache,
                             int num_blocks, const int32_t *block_table, int max_blocks,
                             const int32_t *seqlens, int max_seqlen, int B, int Hq,
                             int first_block, int end_block, const mla_dims &d, float scale,
                             void *o_lat, float *lse, void *workspace, cudaStream_t st) {
  char *ws = static_cast<char *>(workspace);
  __nv_bfloat16 *o_part = reinterpret_cast<__nv_bfloat16 *>(ws + kWsHeader);
  const uint64_t rows = (uint64_t)B * Hq * d.H;
  // The cache and q_lat as [column block of 64][row][64]: one copy moves a
  // whole stage, box k of it (columns 64k..64k+63) 8 KB after box k-1, each
  // box 64 rows x 128 B in the 128-byte swizzle.
  CUtensorMap tm_cache, tm_cache_v, tm_qlat, tm_qrope;
  const uint64_t cache_rows = (uint64_t)num_blocks * kTile;
  if (!make_tmap_3d(&tm_cache, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, cache, 64, cache_rows, kD / 64,
                    kD * 2, 128, 64, 64, kD / 64, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tmap_3d(&tm_cache_v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, cache, 64, cache_rows, kD / 64,
                    kD * 2, 128, 64, 64, kDc / 64, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tmap_3d(&tm_qlat, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, q_lat, 64, rows, kDc / 64,
                    kDc * 2, 128, 64, 64, kDc / 64, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tmap_2d_bf16(&tm_qrope, q_rope, kDr, rows, kDr * 2, 64, 64,
                         CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  // few heads: one CTA per SM, items in order; else pairs, and with several
  // query slots the slot-major plan (each slot over its own share of the
  // pairs)
  const bool few_heads = d.H <= sh::kRows;
  const bool slot_major = !few_heads && Hq > 1;
  auto combine_kernel = few_heads    ? combine_tc_kernel<false, kShItemCost>
                        : slot_major ? combine_tc_kernel<true>
                                     : combine_tc_kernel<false>;
  const int npairs = few_heads ? ctas_for_device() : pairs_for_device();
  if (npairs <= 0) return cudaErrorInvalidDevice;
  DecodeArgs a;
  a.q_lat = static_cast<const __nv_bfloat16 *>(q_lat);
  a.q_rope = static_cast<const __nv_bfloat16 *>(q_rope);
  // a block range starts the table at its first block (no item has a tile
  // when that is past the table's end, so the pointer is then never read)
  a.block_table = block_table + (first_block < max_blocks ? first_block : max_blocks);
  a.seqlens = seqlens;
  a.B = B;
  a.Hq = Hq;
  a.H = d.H;
  a.max_blocks = max_blocks;
  a.max_seqlen = max_seqlen;
  a.num_blocks = num_blocks;
  a.npairs = npairs;
  {  // the range in tokens, clamped to the table (no sequence reaches past it)
    const long b0 = first_block < max_blocks ? first_block : max_blocks;
    const long b1 = end_block < max_blocks ? end_block : max_blocks;
    const long t0 = b0 * kTile, tl = (b1 - b0) * kTile;
    a.tok0 = t0 > INT_MAX ? INT_MAX : (int)t0;
    a.tok_len = tl > INT_MAX ? INT_MAX : (int)tl;
  }
  a.scale_log2 = scale * kLog2e;
  a.o_lat = static_cast<__nv_bfloat16 *>(o_lat);
  a.lse = lse;
  a.err = reinterpret_cast<int *>(ws);
  a.o_part = o_part;
  a.lse_part = reinterpret_cast<float *>(ws + kWsHeader + part_bytes(d.H));
  a.plan = reinterpret_cast<int *>(ws + kWsHeader + part_bytes(d.H) + lse_part_bytes(d.H));
#ifdef MLA_TRACE
  {
    const unsigned long long init[2] = {~0ull, 0ull};
    cudaMemcpyToSymbolAsync(g_trace_comb, init, sizeof(init), 0, cudaMemcpyHostToDevice, st);
  }
#endif
  // both kernels are programmatic dependents of their predecessor in the
  // stream (each waits on it in-kernel before reading its outputs)
  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.stream = st;
  cfg.attrs = pdl;
  cfg.numAttrs = 1;
  cudaError_t e;
  if (few_heads) {
    // the query as 16-row boxes: one copy of 8 latent boxes and one RoPE box
    CUtensorMap tm_q16, tm_r16;
    if (!make_tmap_3d(&tm_q16, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, q_lat, 64, rows, kDc / 64,
                      kDc * 2, 128, 64, sh::kRows, kDc / 64, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_tmap_2d_bf16(&tm_r16, q_rope, kDr, rows, kDr * 2, 64, sh::kRows,
                           CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
    e = cudaFuncSetAttribute(decode_sh_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)sh::kSmemBytes);
    if (e != cudaSuccess) return e;
    cfg.gridDim = dim3(npairs, 1, 1);
    cfg.blockDim = dim3(sh::kThreads, 1, 1);
    cfg.dynamicSmemBytes = sh::kSmemBytes;
    e = cudaLaunchKernelEx(&cfg, decode_sh_kernel, tm_cache, tm_q16, tm_r16, a);
  } else {
    auto decode_kernel = slot_major ? decode_tc_kernel<true> : decode_tc_kernel<false>;
    e = cudaFuncSetAttribute(decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    cfg.gridDim = dim3(2 * npairs, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = kSmemBytes;
    e = cudaLaunchKernelEx(&cfg, decode_kernel, tm_cache, tm_cache_v, tm_qlat, tm_qrope, a);
  }
  if (e != cudaSuccess) return e;
  const long rows_total = (long)B * Hq * d.H;
  cfg.gridDim = dim3((unsigned)((rows_total + kCombineRows - 1) / kCombineRows), 1, 1);
  cfg.blockDim = dim3(32 * kCombineRows, 1, 1);
  cfg.dynamicSmemBytes = 0;
  return cudaLaunchKernelEx(&cfg, combine_kernel, a);
}

cudaError_t launch_combine_pieces_tc(const void *o_pieces, const float *lse_pieces, int P,
                                     long rows, void *o_lat, float *lse, cudaStream_t st) {
  if (rows <= 0) return cudaSuccess;
  const long threads = rows * (kDc / 8);
  combine_pieces_kernel<<<(unsigned)((threads + 255) / 256), 256, 0, st>>>(
      static_cast<const __nv_bfloat16 *>(o_pieces), lse_pieces, P, rows,
      static_cast<__nv_bfloat16 *>(o_lat), lse);
  return cudaGetLastError();
}

}  // namespace mla
