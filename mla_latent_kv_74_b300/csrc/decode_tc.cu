// Absorbed MLA decode on the 5th-generation tensor cores (sm_103a).
//
// Math ("MLA, dim by dim" 4.2 and 5.2; "From Vanilla Transformers to Modern
// LLMs -- Part 3" 3.o-3.p): per (sequence b, query slot i) and head h,
//   s_j  = (q_lat[h] . c_j + q_rope[h] . kR_j) * scale      (j visible)
//   o_lat[h] = sum_j softmax(s)_j c_j ,  lse[h] = ln sum_j exp(s_j)
// with heads as the MMA M dimension (128 rows), 64 cached tokens per tile as
// N, so one latent tile read from HBM serves every head of the sequence.
//
// Layout of the work
//   * A cluster of two CTAs (a "pair") splits the latent width: CTA r owns
//     latent columns [256r, 256r+256) and RoPE columns [32r, 32r+32).  Each
//     CTA loads only its 288-column half of every cache tile (no byte is read
//     twice from HBM), computes partial scores S_r = Q_r C_r^T (M=128, N=64,
//     K=288) into TMEM, and the pair swaps the fp32 partials through
//     distributed shared memory: S = S_0 + S_1 is then bit-identical in both
//     CTAs, so both run the same online softmax and each accumulates its own
//     half of O = P C (M=128, N=256, K=64) in TMEM.
//   * TMEM (512 columns): O half [0,256), two score buffers [256,320),
//     [320,384).  Shared memory: Q half (72 KB), two cache stages (36 KB each),
//     two P tiles (16 KB each), one 32 KB receive buffer for the peer's scores.
//   * Split-KV: the visible tiles of all (sequence, slot) items are laid end to
//     end and cut into 74 equal ranges, one per pair (148 SMs).  A range can
//     start or end inside an item; such pieces write fp32 partials
//     (O/l and lse) that the combine kernel merges with log-sum-exp weights,
//     all other items are written directly.
//   * Roles: warps 0-3 (128 threads, thread t = head row t = TMEM lane t) do
//     the score exchange, softmax, O rescaling and the epilogue; warp 4 issues
//     TMA loads (paged: the tile's row coordinate comes from the block table);
//     warp 5 owns TMEM and issues tcgen05.mma.
//   * Online softmax in base 2 with lazy rescaling: the running maximum is
//     only moved (and O rescaled) when a tile's maximum exceeds it by more
//     than 8 (a factor 256); otherwise P is taken against the stale maximum,
//     which leaves o = O / l exact.
//
// Every wait is bounded; a lost wait records MLA_ERR_TIMEOUT in the
// workspace and the CTA unwinds (waits for its own copies and MMAs, frees
// TMEM, meets its peer at the final cluster barrier).
#include <math.h>

#include "internal.cuh"
#include "ptx.cuh"
#include "tc.cuh"
#include "tmap.cuh"

namespace mla {
namespace {

constexpr int kPairs = kNumSMs / 2;  // 74 clusters of 2 CTAs
constexpr int kTile = 64;            // tokens per tile = block size
constexpr int kDc = 512, kDr = 64, kD = kDc + kDr;
constexpr int kHalfC = 256, kHalfR = 32;
constexpr int kMaxItems = 1024;      // B * Hq limit of this path
constexpr int kStages = 2;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2(256)

// shared-memory map (offsets from a 1024-aligned base)
constexpr uint32_t kQLatBytes = 4 * 128 * 128;       // 4 boxes of 128 rows x 128 B
constexpr uint32_t kQRopeBytes = 128 * 64;           // 128 rows x 64 B
constexpr uint32_t kQBytes = kQLatBytes + kQRopeBytes;  // 73728
constexpr uint32_t kKvLatBytes = 4 * 64 * 128;       // 4 boxes of 64 rows x 128 B
constexpr uint32_t kKvRopeBytes = 64 * 64;
constexpr uint32_t kKvBytes = kKvLatBytes + kKvRopeBytes;  // 36864
constexpr uint32_t kPBytes = 128 * 128;               // 128 rows x 64 bf16
constexpr uint32_t kRecvBytes = 128 * 64 * 4;         // 128 rows x 64 fp32
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffKv = kOffQ + kQBytes;
constexpr uint32_t kOffP = kOffKv + kStages * kKvBytes;
constexpr uint32_t kOffRecv = kOffP + 2 * kPBytes;
constexpr uint32_t kSmemBytes = kOffRecv + kRecvBytes + 1024;  // + alignment slack

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 0;
constexpr uint32_t kTmemS = 256;  // + 64 * buffer

struct DecodeArgs {
  const int32_t *block_table;
  const int32_t *seqlens;
  int B, Hq, H, max_blocks, max_seqlen, num_blocks;
  float scale_log2;
  __nv_bfloat16 *o_lat;
  float *lse;
  float *o_part;    // [2 * kPairs][128][512]
  float *lse_part;  // [2 * kPairs][128]
  int *plan;        // [0] = tiles per pair, [1..W+1] = prefix of tiles per item
  int *err;
};

struct Bars {
  uint64_t q_full, q_free;
  uint64_t kv_full[kStages], kv_empty[kStages];
  uint64_t s_full[2], s_free[2];
  uint64_t p_full[2], pv_done[2];
  uint64_t o_full, o_free;
  uint64_t recv_full, peer_free;  // exchange with the other CTA of the pair
  uint64_t drain;
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

// Bounded wait that also gives up when another role already aborted.
__device__ __forceinline__ bool wait_bar(uint64_t *bar, uint32_t parity, volatile int *abort,
                                         bool cluster_scope = false) {
  return cluster_scope ? ptx::mbar_wait<true>(bar, parity, abort)
                       : ptx::mbar_wait<false>(bar, parity, abort);
}

// The same, with one answer for the whole warp (the softmax warps run
// warp-collective tcgen05 loads and shuffles after every wait).
__device__ __forceinline__ bool wait_bar_warp(uint64_t *bar, uint32_t parity, volatile int *abort,
                                              bool cluster_scope = false) {
  const bool ok = wait_bar(bar, parity, abort, cluster_scope);
  return __all_sync(0xffffffffu, ok);
}

// The segments of one pair: consecutive (item, tile range) pieces of its
// range [t_begin, t_end) of the global tile order.
struct SegIter {
  const int *prefix;
  int W, t_begin, t_end;
  int w;  // current item
  __device__ void init(const int *p, int W_, int tb, int te) {
    prefix = p;
    W = W_;
    t_begin = tb;
    t_end = te;
    // first item whose range ends after t_begin
    int lo = 0, hi = W;
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (prefix[mid + 1] <= t_begin) lo = mid + 1;
      else hi = mid;
    }
    w = lo;
  }
  // next non-empty segment: item, first and end local tile; false when done
  __device__ bool next(int *item, int *lt0, int *lt1, bool *whole) {
    while (w < W && prefix[w] < t_end) {
      const int s = prefix[w], e = prefix[w + 1];
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

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(192, 1)
    decode_tc_kernel(const __grid_constant__ CUtensorMap tm_qlat,
                     const __grid_constant__ CUtensorMap tm_qrope,
                     const __grid_constant__ CUtensorMap tm_cache,
                     const __grid_constant__ CUtensorMap tm_cache_rope, DecodeArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ Bars bars;
  __shared__ int s_prefix[kMaxItems + 1];
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = ptx::cluster_ctarank();
  const uint32_t peer = rank ^ 1u;
  const int pair = blockIdx.x >> 1;
  const int W = a.B * a.Hq;
  volatile int *abort = &s_abort;

  // ---- setup: barriers, TMEM, tile plan ----
  if (threadIdx.x == 0) {
    ptx::mbar_init(&bars.q_full, 1);
    ptx::mbar_init(&bars.q_free, 1);
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(&bars.kv_full[s], 1);
      ptx::mbar_init(&bars.kv_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      ptx::mbar_init(&bars.s_full[s], 1);
      ptx::mbar_init(&bars.s_free[s], 128);
      ptx::mbar_init(&bars.p_full[s], 128);
      ptx::mbar_init(&bars.pv_done[s], 1);
    }
    ptx::mbar_init(&bars.o_full, 1);
    ptx::mbar_init(&bars.o_free, 128);
    ptx::mbar_init(&bars.recv_full, 128);
    ptx::mbar_init(&bars.peer_free, 128);
    ptx::mbar_init(&bars.drain, 1);
    ptx::fence_mbar_init();
    s_abort = 0;
  }
  if (warp == 4 && lane == 0) {
    ptx::tma_prefetch_desc(&tm_qlat);
    ptx::tma_prefetch_desc(&tm_qrope);
    ptx::tma_prefetch_desc(&tm_cache);
    ptx::tma_prefetch_desc(&tm_cache_rope);
  }
  if (warp == 5) ptx::tmem_alloc(&s_tmem, kTmemCols);
  // tiles per item -> s_prefix[w + 1]
  bool any_bad = false;
  for (int w = threadIdx.x; w < W; w += blockDim.x) {
    bool bad = false;
    const int n = visible_len(a, w, &bad);
    any_bad |= bad;
    s_prefix[w + 1] = (n + kTile - 1) / kTile;
  }
  if (any_bad && rank == 0 && pair == 0) set_device_error(a.err, kDevBounds);
  __syncthreads();
  if (warp == 0) {  // inclusive scan, 32 items per round
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
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  ptx::cluster_sync();  // the peer's barriers are initialised before any remote arrive

  const uint32_t tmem = s_tmem;
  const int t_total = s_prefix[W];
  const int per = (t_total + kPairs - 1) / kPairs;
  const int t_begin = min(t_total, pair * per);
  const int t_end = min(t_total, t_begin + per);
  if (blockIdx.x == 0 && threadIdx.x <= W) {
    if (threadIdx.x == 0) a.plan[0] = per;
  }
  if (blockIdx.x == 0)
    for (int w = threadIdx.x; w <= W; w += blockDim.x) a.plan[1 + w] = s_prefix[w];

  uint8_t *sQ = smem + kOffQ;
  uint8_t *sKv = smem + kOffKv;
  uint8_t *sP = smem + kOffP;
  float *sRecv = reinterpret_cast<float *>(smem + kOffRecv);

  if (warp == 4) {
    // ===================== TMA producer =====================
    if (lane == 0) {
      SegIter it;
      it.init(s_prefix, W, t_begin, t_end);
      int item, lt0, lt1, seg = 0, g = 0;
      bool whole;
      int q_issued = 0;
      while (!*abort && it.next(&item, &lt0, &lt1, &whole)) {
        if (seg > 0 && !wait_bar(&bars.q_free, (seg - 1) & 1, abort)) break;
        const int row0 = item * a.H;
        ptx::mbar_arrive_expect_tx(&bars.q_full, kQBytes);
        for (int k = 0; k < 4; ++k)
          ptx::tma_load_2d(sQ + k * 16384, &tm_qlat, &bars.q_full, rank * kHalfC + k * 64, row0);
        ptx::tma_load_2d(sQ + kQLatBytes, &tm_qrope, &bars.q_full, rank * kHalfR, row0);
        ++q_issued;
        const int b = item / a.Hq;
        const int32_t *tbl = a.block_table + (size_t)b * a.max_blocks;
        for (int lt = lt0; lt < lt1; ++lt, ++g) {
          const int st = g % kStages;
          if (g >= kStages && !wait_bar(&bars.kv_empty[st], ((g / kStages) - 1) & 1, abort)) break;
          int blk = tbl[lt];
          if (blk < 0 || blk >= a.num_blocks) blk = 0;  // reported by the softmax warps
          uint8_t *dst = sKv + st * kKvBytes;
          ptx::mbar_arrive_expect_tx(&bars.kv_full[st], kKvBytes);
          for (int k = 0; k < 4; ++k)
            ptx::tma_load_2d(dst + k * 8192, &tm_cache, &bars.kv_full[st],
                             rank * kHalfC + k * 64, blk * kTile);
          ptx::tma_load_2d(dst + kKvLatBytes, &tm_cache_rope, &bars.kv_full[st],
                           kDc + rank * kHalfR, blk * kTile);
        }
        ++seg;
      }
      // never leave with copies in flight: the last load into each buffer
      // must have landed (a no-op when the consumer already saw it)
      if (q_issued > 0) ptx::mbar_wait(&bars.q_full, (q_issued - 1) & 1);
      for (int k = g - kStages < 0 ? 0 : g - kStages; k < g; ++k)
        ptx::mbar_wait(&bars.kv_full[k % kStages], (k / kStages) & 1);
    }
  } else if (warp == 5) {
    // ===================== MMA issuer =====================
    if (lane == 0) {
      const uint32_t idesc_qk = ptx::idesc_bf16(128, kTile, false, false);
      const uint32_t idesc_pv = ptx::idesc_bf16(128, kHalfC, false, true);
      const uint32_t q_addr = ptx::smem_u32(sQ);
      const uint32_t kv_addr = ptx::smem_u32(sKv);
      const uint32_t p_addr = ptx::smem_u32(sP);
      SegIter it;
      it.init(s_prefix, W, t_begin, t_end);
      int item, lt0, lt1, seg = 0, g = 0;
      bool whole;
      bool failed = false;
      auto issue_pv = [&](int gg, bool first_of_seg) -> bool {
        const int pb = gg & 1;
        if (first_of_seg && seg > 0 && !wait_bar(&bars.o_free, (seg - 1) & 1, abort)) return false;
        if (!wait_bar(&bars.p_full[pb], (gg >> 1) & 1, abort)) return false;
        ptx::tc_fence_after();
        const uint32_t st_addr = kv_addr + (gg % kStages) * kKvBytes;
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk) {
          const uint64_t ad = ptx::smem_desc(p_addr + pb * kPBytes + kk * 32, 16, 1024, ptx::kSw128);
          const uint64_t bd = ptx::smem_desc(st_addr + kk * 2048, 8192, 1024, ptx::kSw128);
          ptx::mma_bf16(tmem + kTmemO, ad, bd, idesc_pv, (first_of_seg && kk == 0) ? 0u : 1u);
        }
        ptx::mma_commit(&bars.pv_done[pb]);
        ptx::mma_commit(&bars.kv_empty[gg % kStages]);
        return true;
      };
      while (!failed && it.next(&item, &lt0, &lt1, &whole)) {
        if (!wait_bar(&bars.q_full, seg & 1, abort)) { failed = true; break; }
        const int g_first = g;
        for (int lt = lt0; lt < lt1; ++lt, ++g) {
          const int st = g % kStages, sb = g & 1;
          if (!wait_bar(&bars.kv_full[st], (g / kStages) & 1, abort)) { failed = true; break; }
          if (g >= 2 && !wait_bar(&bars.s_free[sb], ((g >> 1) - 1) & 1, abort)) { failed = true; break; }
          ptx::tc_fence_after();
          const uint32_t st_addr = kv_addr + st * kKvBytes;
          const uint32_t d_s = tmem + kTmemS + sb * kTile;
#pragma unroll
          for (int kk = 0; kk < 16; ++kk) {  // latent: 4 boxes x 4 k-steps of 16
            const uint64_t ad = ptx::smem_desc(q_addr + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024, ptx::kSw128);
            const uint64_t bd = ptx::smem_desc(st_addr + (kk >> 2) * 8192 + (kk & 3) * 32, 16, 1024, ptx::kSw128);
            ptx::mma_bf16(d_s, ad, bd, idesc_qk, kk != 0);
          }
#pragma unroll
          for (int kk = 0; kk < 2; ++kk) {  // RoPE: one 64-byte-swizzled box, 2 k-steps
            const uint64_t ad = ptx::smem_desc(q_addr + kQLatBytes + kk * 32, 16, 512, ptx::kSw64);
            const uint64_t bd = ptx::smem_desc(st_addr + kKvLatBytes + kk * 32, 16, 512, ptx::kSw64);
            ptx::mma_bf16(d_s, ad, bd, idesc_qk, 1u);
          }
          ptx::mma_commit(&bars.s_full[sb]);
          if (lt == lt1 - 1) ptx::mma_commit(&bars.q_free);
          if (g > g_first && !issue_pv(g - 1, g - 1 == g_first)) { failed = true; break; }
        }
        if (failed) break;
        if (!issue_pv(g - 1, g - 1 == g_first)) { failed = true; break; }
        ptx::mma_commit(&bars.o_full);
        ++seg;
      }
      // drain: every MMA issued above has completed before TMEM is freed
      ptx::mma_commit(&bars.drain);
      ptx::mbar_wait(&bars.drain, 0);
      if (failed) atomicExch(&s_abort, 1);
    }
  } else {
    // ===================== softmax / epilogue (warps 0-3) =====================
    const int t = threadIdx.x;  // head row == TMEM lane
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    SegIter it;
    it.init(s_prefix, W, t_begin, t_end);
    int item, lt0, lt1, seg = 0, g = 0;
    bool whole;
    bool failed = false;
    float *recv_row_base = sRecv;  // [16][128][4]
    while (!failed && it.next(&item, &lt0, &lt1, &whole)) {
      const int b = item / a.Hq, slot = item % a.Hq;
      bool dummy = false;
      const int n_vis = visible_len(a, item, &dummy);
      // validate the block-table entries this segment reads (each warp on
      // its own, so no cross-warp barrier is needed)
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
      float m_run = -INFINITY, l_run = 0.f;
      const int g_first = g;
      for (int lt = lt0; lt < lt1; ++lt, ++g) {
        const int sb = g & 1;
        // -- partial scores of this CTA --
        if (!wait_bar_warp(&bars.s_full[sb], (g >> 1) & 1, abort)) { failed = true; break; }
        ptx::tc_fence_after();
        float s[64];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          float v[16];
          ptx::tmem_ld16(tmem + lane_base + kTmemS + sb * kTile + c * 16, v);
#pragma unroll
          for (int i = 0; i < 16; ++i) s[c * 16 + i] = v[i];
        }
        ptx::tmem_ld_wait();
        ptx::tc_fence_before();
        ptx::mbar_arrive(&bars.s_free[sb]);
        // -- swap partials with the peer CTA --
        if (g > 0 && !wait_bar_warp(&bars.peer_free, (g - 1) & 1, abort, true)) { failed = true; break; }
#pragma unroll
        for (int c = 0; c < 16; ++c)
          ptx::st_cluster_v4(recv_row_base + (c * 128 + t) * 4, peer, s[4 * c], s[4 * c + 1],
                             s[4 * c + 2], s[4 * c + 3]);
        ptx::mbar_arrive_remote(&bars.recv_full, peer);
        if (!wait_bar_warp(&bars.recv_full, g & 1, abort, true)) { failed = true; break; }
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          const float4 p4 = *reinterpret_cast<const float4 *>(recv_row_base + (c * 128 + t) * 4);
          s[4 * c] += p4.x;
          s[4 * c + 1] += p4.y;
          s[4 * c + 2] += p4.z;
          s[4 * c + 3] += p4.w;
        }
        ptx::mbar_arrive_remote(&bars.peer_free, peer);
        // -- online softmax (base 2) --
        const int tok0 = lt * kTile;
        float mt = -INFINITY;
#pragma unroll
        for (int j = 0; j < 64; ++j) {
          s[j] = (tok0 + j < n_vis) ? s[j] * a.scale_log2 : -INFINITY;
          mt = fmaxf(mt, s[j]);
        }
        const bool first = (g == g_first);
        float m_use = m_run, alpha = 1.f;
        bool rescale = false;
        if (first) {
          m_use = mt;
        } else if (mt > m_run + kRescaleThreshold) {
          m_use = mt;
          alpha = exp2f(m_run - mt);
          rescale = true;
        }
        // P tile (bf16) in the 128B-swizzled K-major layout of the MMA
        const int pb = g & 1;
        // P buffer pb was last read by PV(g-2)
        if (g >= 2 && !wait_bar_warp(&bars.pv_done[pb], ((g >> 1) - 1) & 1, abort)) { failed = true; break; }
        if (__any_sync(0xffffffffu, rescale)) {
          // O row t *= alpha once PV(g-1) has finished accumulating
          if (!wait_bar_warp(&bars.pv_done[(g - 1) & 1], ((g - 1) >> 1) & 1, abort)) { failed = true; break; }
          ptx::tc_fence_after();
#pragma unroll 1
          for (int c = 0; c < kHalfC / 16; ++c) {
            float v[16];
            ptx::tmem_ld16(tmem + lane_base + kTmemO + c * 16, v);
            ptx::tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 16; ++i) v[i] *= alpha;
            ptx::tmem_st16(tmem + lane_base + kTmemO + c * 16, v);
          }
          ptx::tmem_st_wait();
        }
        float lsum = 0.f;
        uint8_t *prow = sP + pb * kPBytes + t * 128;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          uint32_t packed[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const __nv_bfloat16 lo = __float2bfloat16_rn(exp2f(s[c * 8 + 2 * i] - m_use));
            const __nv_bfloat16 hi = __float2bfloat16_rn(exp2f(s[c * 8 + 2 * i + 1] - m_use));
            lsum += __bfloat162float(lo) + __bfloat162float(hi);
            packed[i] = (uint32_t)__bfloat16_as_ushort(lo) | ((uint32_t)__bfloat16_as_ushort(hi) << 16);
          }
          *reinterpret_cast<uint4 *>(prow + ((c ^ (t & 7)) << 4)) =
              make_uint4(packed[0], packed[1], packed[2], packed[3]);
        }
        l_run = l_run * alpha + lsum;
        m_run = m_use;
        ptx::fence_proxy_async_smem();
        ptx::tc_fence_before();
        ptx::mbar_arrive(&bars.p_full[pb]);
      }
      if (failed) break;
      // -- epilogue: O half of row t -> output --
      if (!wait_bar_warp(&bars.o_full, seg & 1, abort)) { failed = true; break; }
      ptx::tc_fence_after();
      const int row = item * a.H + t;
      const bool write_row = t < a.H;
      const float inv_l = l_run > 0.f ? 1.f / l_run : 0.f;
      const float lse_val = l_run > 0.f ? (m_run + log2f(l_run)) * kLn2 : -INFINITY;
      if (whole) {
        __nv_bfloat16 *dst = a.o_lat + (size_t)row * kDc + rank * kHalfC;
#pragma unroll 1
        for (int c = 0; c < kHalfC / 16; ++c) {
          float v[16];
          ptx::tmem_ld16(tmem + lane_base + kTmemO + c * 16, v);
          ptx::tmem_ld_wait();
          if (write_row) {
            uint32_t pk[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const float x0 = seg_bad ? 0.f : v[2 * i] * inv_l;
              const float x1 = seg_bad ? 0.f : v[2 * i + 1] * inv_l;
              pk[i] = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(x0)) |
                      ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(x1)) << 16);
            }
            uint4 *d4 = reinterpret_cast<uint4 *>(dst + c * 16);
            d4[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
            d4[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
          }
        }
        if (write_row && rank == 0) a.lse[row] = seg_bad ? -INFINITY : lse_val;
      } else {
        // partial slot: 2*pair for the range's first segment, 2*pair+1 for its last
        const int slot_idx = 2 * pair + ((lt0 == 0) ? 1 : 0);
        float *dst = a.o_part + ((size_t)slot_idx * 128 + t) * kDc + rank * kHalfC;
#pragma unroll 1
        for (int c = 0; c < kHalfC / 16; ++c) {
          float v[16];
          ptx::tmem_ld16(tmem + lane_base + kTmemO + c * 16, v);
          ptx::tmem_ld_wait();
          if (write_row) {
            float4 *d4 = reinterpret_cast<float4 *>(dst + c * 16);
#pragma unroll
            for (int i = 0; i < 4; ++i)
              d4[i] = make_float4(v[4 * i] * inv_l, v[4 * i + 1] * inv_l, v[4 * i + 2] * inv_l,
                                  v[4 * i + 3] * inv_l);
          }
        }
        if (write_row && rank == 0)
          a.lse_part[(size_t)slot_idx * 128 + t] =
              seg_bad ? __int_as_float(0x7fc00000) : lse_val;  // NaN poisons the item
      }
      if (seg_bad && t == 0) set_device_error(a.err, kDevBounds);
      ptx::tc_fence_before();
      ptx::mbar_arrive(&bars.o_free);
      ++seg;
      (void)slot;
    }
    if (failed) atomicExch(&s_abort, 1);
    // items with nothing visible (or an invalid length): o = 0, lse = -inf
    for (int w = pair; w < W; w += kPairs) {
      if (s_prefix[w + 1] != s_prefix[w]) continue;
      if (t < a.H) {
        const int row = w * a.H + t;
        uint4 *d4 = reinterpret_cast<uint4 *>(a.o_lat + (size_t)row * kDc + rank * kHalfC);
        for (int i = 0; i < kHalfC * 2 / 16; ++i) d4[i] = make_uint4(0, 0, 0, 0);
        if (rank == 0) a.lse[row] = -INFINITY;
      }
    }
  }

  // ---- teardown ----
  __syncwarp();
  ptx::tc_fence_before();
  __syncthreads();
  if (s_abort && threadIdx.x == 0) set_device_error(a.err, kDevTimeout);
  ptx::cluster_sync();  // the peer no longer touches this CTA's shared memory
  ptx::tc_fence_after();
  if (warp == 5) ptx::tmem_dealloc(tmem, kTmemCols);
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

size_t part_bytes() { return align_up((size_t)2 * kPairs * 128 * kDc * sizeof(float), 256); }
size_t lse_part_bytes() { return align_up((size_t)2 * kPairs * 128 * sizeof(float), 256); }

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
  const uint64_t rows = (uint64_t)B * Hq * d.H;
  CUtensorMap tm_qlat, tm_qrope, tm_cache;
  if (!make_tmap_2d_bf16(&tm_qlat, q_lat, kDc, rows, kDc * 2, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tmap_2d_bf16(&tm_qrope, q_rope, kDr, rows, kDr * 2, 32, 128, CU_TENSOR_MAP_SWIZZLE_64B) ||
      !make_tmap_2d_bf16(&tm_cache, cache, kD, (uint64_t)num_blocks * kTile, kD * 2, 64, 64,
                         CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  // the RoPE box of the cache is 32 columns wide with a 64-byte swizzle
  CUtensorMap tm_cache_rope;
  if (!make_tmap_2d_bf16(&tm_cache_rope, cache, kD, (uint64_t)num_blocks * kTile, kD * 2, 32, 64,
                         CU_TENSOR_MAP_SWIZZLE_64B))
    return cudaErrorInvalidValue;
  char *ws = static_cast<char *>(workspace);
  DecodeArgs a;
  a.block_table = block_table;
  a.seqlens = seqlens;
  a.B = B;
  a.Hq = Hq;
  a.H = d.H;
  a.max_blocks = max_blocks;
  a.max_seqlen = max_seqlen;
  a.num_blocks = num_blocks;
  a.scale_log2 = scale * kLog2e;
  a.o_lat = static_cast<__nv_bfloat16 *>(o_lat);
  a.lse = lse;
  a.err = reinterpret_cast<int *>(ws);
  a.o_part = reinterpret_cast<float *>(ws + kWsHeader);
  a.lse_part = reinterpret_cast<float *>(ws + kWsHeader + part_bytes());
  a.plan = reinterpret_cast<int *>(ws + kWsHeader + part_bytes() + lse_part_bytes());
  cudaError_t e = cudaFuncSetAttribute(decode_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)kSmemBytes);
  if (e != cudaSuccess) return e;
  decode_tc_kernel<<<2 * kPairs, 192, kSmemBytes, st>>>(tm_qlat, tm_qrope, tm_cache, tm_cache_rope, a);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  dim3 cgrid(B * Hq, (d.H + 15) / 16);
  combine_tc_kernel<<<cgrid, 128, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace mla
