// MLA prefill in the standard order on the 5th-generation tensor cores
// (sm_103a): keys and values are rebuilt from the latents first, then causal
// attention runs over d_k = d_h + d_r and d_v = d_h.
//
// Math ("MLA, dim by dim" 4.1; "MLA Explained", training and prefill): per
// packed sequence and head h,
//   K = [C W_UK[h]^T ; k_R]   (T x 192),   V = C W_UV[h]^T   (T x 128)
//   S = [q_nope ; q_rope] K^T * scale,   causal row softmax,   out = P V
// with lse the natural log-sum-exp of the scaled scores.  Absorbing W_UK and
// W_UV here would move the T^2 contractions from 192 / 128 onto d_c = 512,
// so unlike decode the up-projections run first: kv_rebuild_kernel writes
// [K_nope | V] per (token, head) into the workspace, and prefill_attn_kernel
// reads it.
//
// The attention kernel is persistent: one CTA per SM takes (128-query tile,
// head, prompt) items from a work list in the workspace (a counter the
// rebuild kernel zeroes).  Items are numbered with the query tiles of one
// head adjacent (heaviest first), so the CTAs at work at any time share a
// few heads' K and V in L2; each CTA loads the next item's query and first
// key tiles, and computes its first scores, while it finishes the current
// one.
//
// Queries are the MMA M dimension (128 rows = TMEM lanes), keys come in
// tiles of 128:
//   S  = Q K^T    M=128, N=128, K=192  A = Q (TMEM), B = K tile (smem)
//   O += P V      M=128, N=128, K=128  A = P (TMEM, bf16), B = V tile (smem,
//                                       MN-major)
// TMEM (512 columns): the 128-column score tile, the 128-column output
// accumulator, two 64-column buffers of packed bf16 probabilities and the
// query (96 columns).  Shared memory: a ring of three K stages (48 KB: the
// two halves of K_nope and k_R) whose first fill is the query tile on its
// way into TMEM, and a ring of two V stages (32 KB), all 128-byte swizzled
// and loaded by TMA.  Keeping the query out of shared memory buys the third
// K stage, which hides the L2 latency of the next key tile.
//
// Warp roles (384 threads): warp 0 runs the work list and loads the query
// and K tiles, warp 10 loads the V tiles, warp 1 owns TMEM and issues
// Q K^T, warp 11 issues P V, warps 2-9 run the online softmax and the
// epilogue: thread = query row = TMEM lane, warps w and w+4 on lanes
// 32*(w%4).. (one SM sub-partition), each taking half of a tile's 128 key
// columns; the pair agrees on the row maximum through shared memory and an
// mbarrier.  As soon as the softmax has read a score tile the next Q K^T
// goes into the same columns, so the next scores are ready when the softmax
// finishes; the P V of each tile follows its softmax.
//
// Online softmax in base 2 with lazy rescaling: the running maximum moves,
// and the warp's rows of O are rescaled in TMEM, only when a tile's maximum
// exceeds it by more than 8 (a factor of 256); otherwise the probabilities
// are taken against the stale maximum, which leaves O / l exact.
//
// Every wait is bounded; a lost wait records MLA_ERR_TIMEOUT in the
// workspace's error word and the CTA drains its copies and MMAs, frees TMEM
// and returns.
#include <math.h>

#include "internal.cuh"
#include "ptx.cuh"
#include "tc.cuh"
#include "tmap.cuh"

namespace mla {
namespace {

constexpr int kQT = 128;  // queries per item (the MMA M dimension)
constexpr int kKT = 128;  // keys per tile
constexpr int kDh = 128, kDr = 64, kDc = 512;
constexpr int kThreads = 384;   // attention: two TMA warps, two MMA warps, eight softmax warps
constexpr int kRThreads = 192;  // rebuild: TMA, MMA, four epilogue warps
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2(256)

// ---- shared memory (offsets from the 1024-aligned dynamic base)
constexpr uint32_t kBox = 128 * 128;  // 128 rows x 64 bf16 (128 B), 128B swizzle
// K ring: stage = boxes k_nope[0:64], k_nope[64:128], k_R.  The query tile
// (boxes q_nope[0:64], q_nope[64:128], q_rope) is the ring's first fill, on
// its way into TMEM.
constexpr int kKStages = 3;
constexpr uint32_t kKStage = 3 * kBox;
constexpr uint32_t kOffK = 0;
// V ring: stage = boxes v[0:64], v[64:128]
constexpr int kVStages = 2;
constexpr uint32_t kVStage = 2 * kBox;
constexpr uint32_t kOffV = kOffK + kKStages * kKStage;
// softmax pair exchange: row maxima [tile parity][column half][128], row
// sums [column half][128]
constexpr uint32_t kOffRed = kOffV + kVStages * kVStage;
constexpr uint32_t kOffBars = kOffRed + 6 * 128 * 4;

// One unit of work: a 128-query tile of one head of one prompt (n key tiles;
// n == 0 ends the list).
struct Item {
  int tok0, T, q0, h, n;
};
// roles that take each published item: the V producer, the two MMA issuers
// (one thread each) and the eight softmax warps (one arrival per warp)
constexpr uint32_t kItemTakers = 3 + 8;

struct Bars {
  uint64_t k_full[kKStages], k_empty[kKStages];  // K ring: per item the query, then its key tiles
  uint64_t v_full[kVStages], v_empty[kVStages];  // V ring
  uint64_t q_tmem;      // the query copied into TMEM (one arrival per softmax warp)
  uint64_t s_full;      // scores of the current tile ready
  uint64_t s_free;      // ... and read (one arrival per softmax warp)
  uint64_t p_full[2];   // probabilities of tile j in buffer j % 2 (one arrival per warp)
  uint64_t pv_done[2];  // P(j) V accumulated (buffer j % 2 free again)
  uint64_t o_done;    // the item's last P V accumulated
  uint64_t drain[2];  // each MMA issuer's last MMAs done
  // softmax pairs: row maxima of tile j exchanged (per row quarter and tile
  // parity), row sums exchanged at the end; 64 arrivals each
  uint64_t pair_max[4][2], pair_sum[4];
  uint64_t o_free;  // the epilogue has read O (one arrival per softmax warp)
  // the work list: warp 0 publishes each item, every other role takes it
  uint64_t item_full[2], item_empty[2];
  Item items[2];
  uint32_t tmem;
  int fail;
};
constexpr uint32_t kSmemBytes = 1024 + kOffBars + ((sizeof(Bars) + 15) / 16) * 16;
static_assert(kSmemBytes <= 232448, "over the 227 KB shared-memory limit");

// TMEM columns
constexpr uint32_t kTmemS = 0;    // 128 fp32 scores
constexpr uint32_t kTmemO = 128;  // 128 fp32 output accumulator
constexpr uint32_t kTmemP = 256;  // 2 x 64 (128 bf16 probabilities each, two per column)
constexpr uint32_t kTmemQ = 384;  // 96 (the 192 bf16 query elements of a row)
struct PrefillArgs {
  const int32_t *cu_seqlens;  // [B + 1]
  int B, H, max_seqlen, total;
  int nq;                           // query tiles per prompt at max_seqlen
  unsigned long long total_items;   // B * H * nq
  unsigned long long *next_item;    // work-list counter, zeroed by the rebuild kernel
  float scale_log2;
  __nv_bfloat16 *out;  // [total][H][128]
  float *lse;          // [total][H]
  int *err;
};

__device__ __forceinline__ bool wait_warp(uint64_t *bar, uint32_t parity, volatile int *fail) {
  return __all_sync(0xffffffffu, ptx::mbar_wait(bar, parity, fail));
}

__global__ void __launch_bounds__(kThreads, 1)
    prefill_attn_kernel(const __grid_constant__ CUtensorMap tm_q,   // q_nope [total][H*128]
                        const __grid_constant__ CUtensorMap tm_qr,  // q_rope [total][H*64]
                        const __grid_constant__ CUtensorMap tm_kv,  // [K_nope | V] [H*4][total][64]
                        const __grid_constant__ CUtensorMap tm_kr,  // k_R [total][64]
                        PrefillArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Bars *bars = reinterpret_cast<Bars *>(smem + kOffBars);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kKStages; ++i) {
      ptx::mbar_init(&bars->k_full[i], 1);
      ptx::mbar_init(&bars->k_empty[i], 1);
    }
    for (int i = 0; i < kVStages; ++i) {
      ptx::mbar_init(&bars->v_full[i], 1);
      ptx::mbar_init(&bars->v_empty[i], 1);
    }
    ptx::mbar_init(&bars->q_tmem, 8);
    ptx::mbar_init(&bars->s_full, 1);
    ptx::mbar_init(&bars->s_free, 8);
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(&bars->p_full[i], 8);
      ptx::mbar_init(&bars->pv_done[i], 1);
      ptx::mbar_init(&bars->item_full[i], 1);
      ptx::mbar_init(&bars->item_empty[i], kItemTakers);
    }
    ptx::mbar_init(&bars->o_done, 1);
    ptx::mbar_init(&bars->o_free, 8);
    ptx::mbar_init(&bars->drain[0], 1);
    ptx::mbar_init(&bars->drain[1], 1);
    for (int i = 0; i < 4; ++i) {
      ptx::mbar_init(&bars->pair_max[i][0], 64);
      ptx::mbar_init(&bars->pair_max[i][1], 64);
      ptx::mbar_init(&bars->pair_sum[i], 64);
    }
    bars->fail = 0;
    ptx::fence_mbar_init();
    ptx::tma_prefetch_desc(&tm_q);
    ptx::tma_prefetch_desc(&tm_qr);
    ptx::tma_prefetch_desc(&tm_kv);
    ptx::tma_prefetch_desc(&tm_kr);
  }
  if (warp == 1) ptx::tmem_alloc(&bars->tmem, 512);
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = bars->tmem;
  volatile int *fail = &bars->fail;
  auto set_fail = [&]() { atomicExch(const_cast<int *>(fail), 1); };
  // item k of this CTA's list, for the single-thread roles
  auto take_item = [&](int k, Item *it) -> bool {
    if (!ptx::mbar_wait(&bars->item_full[k & 1], (k >> 1) & 1, fail)) return false;
    *it = bars->items[k & 1];
    ptx::mbar_arrive(&bars->item_empty[k & 1]);
    return true;
  };

  if (warp == 0) {
    // ======== work list and TMA producer: the query, then the K tiles ========
    if (lane == 0) {
      int f = 0;  // fills of the K ring (all items)
      auto fill_wait = [&](int ff) -> bool {
        return ff < kKStages ||
               ptx::mbar_wait(&bars->k_empty[ff % kKStages], ((ff / kKStages) - 1) & 1, fail);
      };
      bool ok = true;
      for (int k = 0; ok; ++k) {
        if (k >= 2 && !ptx::mbar_wait(&bars->item_empty[k & 1], ((k >> 1) - 1) & 1, fail)) {
          ok = false;
          break;
        }
        // the next non-empty (query tile, head, prompt), query tiles of one
        // head adjacent and heaviest first, so the CTAs at work at any time
        // share a few heads' K and V in L2
        Item it = {0, 0, 0, 0, 0};
        for (;;) {
          const unsigned long long i = atomicAdd(a.next_item, 1ull);
          if (i >= a.total_items) break;
          const int qr = (int)(i % (unsigned long long)a.nq);
          const unsigned long long rest = i / (unsigned long long)a.nq;
          const int h = (int)(rest % (unsigned long long)a.H);
          const int b = (int)(rest / (unsigned long long)a.H);
          const int tok0 = a.cu_seqlens[b];
          const int T = a.cu_seqlens[b + 1] - tok0;
          if (tok0 < 0 || T < 0 || T > a.max_seqlen || tok0 > a.total - T) {
            set_device_error(a.err, kDevBounds);
            continue;
          }
          const int qt = a.nq - 1 - qr;
          if (qt * kQT >= T) continue;
          // key tiles 0 .. qt: the tile's first query sees key 128 qt, so
          // every tile holds a visible key for every row
          it = Item{tok0, T, qt * kQT, h, qt + 1};
          break;
        }
        bars->items[k & 1] = it;
        ptx::mbar_arrive(&bars->item_full[k & 1]);
        if (it.n == 0) break;
        if (!fill_wait(f)) {
          ok = false;
          break;
        }
        uint8_t *qd = smem + kOffK + (f % kKStages) * kKStage;
        uint64_t *qb = &bars->k_full[f % kKStages];
        ptx::mbar_arrive_expect_tx(qb, kKStage);
        ptx::tma_load_2d(qd, &tm_q, qb, it.h * kDh, it.tok0 + it.q0);
        ptx::tma_load_2d(qd + kBox, &tm_q, qb, it.h * kDh + 64, it.tok0 + it.q0);
        ptx::tma_load_2d(qd + 2 * kBox, &tm_qr, qb, it.h * kDr, it.tok0 + it.q0);
        ++f;
        const int zk = it.h * 4;  // the head's K_nope chunks
        for (int j = 0; j < it.n; ++j, ++f) {
          if (!fill_wait(f)) {
            ok = false;
            break;
          }
          uint8_t *kd = smem + kOffK + (f % kKStages) * kKStage;
          uint64_t *kb = &bars->k_full[f % kKStages];
          const int y = it.tok0 + j * kKT;
          ptx::mbar_arrive_expect_tx(kb, kKStage);
          ptx::tma_load_3d(kd, &tm_kv, kb, 0, y, zk);
          ptx::tma_load_3d(kd + kBox, &tm_kv, kb, 0, y, zk + 1);
          ptx::tma_load_2d(kd + 2 * kBox, &tm_kr, kb, 0, y);
        }
      }
      if (!ok) set_fail();
      // never leave with copies in flight: the ring's last fills have landed
      for (int i = f - kKStages < 0 ? 0 : f - kKStages; i < f; ++i)
        ptx::mbar_wait(&bars->k_full[i % kKStages], (i / kKStages) & 1);
    }
  } else if (warp == 10) {
    // ================= TMA producer: the V tiles =================
    if (lane == 0) {
      int fv = 0;
      bool ok = true;
      for (int k = 0; ok; ++k) {
        Item it;
        if (!take_item(k, &it)) {
          ok = false;
          break;
        }
        if (it.n == 0) break;
        const int zv = it.h * 4 + 2;  // the head's V chunks
        for (int j = 0; j < it.n; ++j, ++fv) {
          const int st = fv % kVStages;
          if (fv >= kVStages &&
              !ptx::mbar_wait(&bars->v_empty[st], ((fv / kVStages) - 1) & 1, fail)) {
            ok = false;
            break;
          }
          uint8_t *vd = smem + kOffV + st * kVStage;
          ptx::mbar_arrive_expect_tx(&bars->v_full[st], kVStage);
          ptx::tma_load_3d(vd, &tm_kv, &bars->v_full[st], 0, it.tok0 + j * kKT, zv);
          ptx::tma_load_3d(vd + kBox, &tm_kv, &bars->v_full[st], 0, it.tok0 + j * kKT, zv + 1);
        }
      }
      if (!ok) set_fail();
      for (int i = fv - kVStages < 0 ? 0 : fv - kVStages; i < fv; ++i)
        ptx::mbar_wait(&bars->v_full[i % kVStages], (i / kVStages) & 1);
    }
  } else if (warp == 1 || warp == 11) {
    // ======== MMA issuers: warp 1 Q K^T (and TMEM owner), warp 11 P V ========
    // One thread cannot issue these MMAs at the tensor pipe's rate (its issue
    // stalls while earlier MMAs execute); two threads, each waiting only on
    // its own operands, keep the pipe fed.
    if (lane == 0) {
      bool ok = true;
      if (warp == 1) {
        const uint32_t idesc_s = ptx::idesc_bf16(kQT, kKT, false, false);
        const uint64_t kdesc =
            ptx::smem_desc(ptx::smem_u32(smem + kOffK), 16, 1024, ptx::kSw128);
        int f = 0, g = 0;  // K-ring fills, score tiles (all items)
        for (int k = 0; ok; ++k) {
          Item it;
          if (!take_item(k, &it)) {
            ok = false;
            break;
          }
          if (it.n == 0) break;
          // the item's query is in TMEM: its ring stage goes back
          if (!ptx::mbar_wait(&bars->q_tmem, k & 1, fail)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          ptx::mbar_arrive(&bars->k_empty[f % kKStages]);
          ++f;
          // S = Q K^T per key tile, A = the query in TMEM, once the softmax
          // has read the previous tile's scores
          for (int j = 0; j < it.n; ++j, ++f, ++g) {
            const int st = f % kKStages;
            if ((g > 0 && !ptx::mbar_wait(&bars->s_free, (g - 1) & 1, fail)) ||
                !ptx::mbar_wait(&bars->k_full[st], (f / kKStages) & 1, fail)) {
              ok = false;
              break;
            }
            ptx::tc_fence_after();
            const uint64_t kd = kdesc + (uint64_t)((st * kKStage) >> 4);
#pragma unroll
            for (int kk = 0; kk < 12; ++kk) {  // 3 boxes x 4 k-steps of 16
              const uint32_t off = (kk >> 2) * kBox + (kk & 3) * 32;
              ptx::mma_bf16_ts(tmem + kTmemS, tmem + kTmemQ + kk * 8, kd + (uint64_t)(off >> 4),
                               idesc_s, kk != 0);
            }
            ptx::mma_commit(&bars->s_full);
            ptx::mma_commit(&bars->k_empty[st]);
          }
        }
      } else {
        const uint32_t idesc_o = ptx::idesc_bf16(kQT, kDh, false, true);
        // V is MN-major: the two 64-wide d_v blocks are one box (kBox) apart
        const uint64_t vdesc =
            ptx::smem_desc(ptx::smem_u32(smem + kOffV), kBox, 1024, ptx::kSw128);
        int g = 0;  // tiles (all items); V-ring fill = tile
        for (int k = 0; ok; ++k) {
          Item it;
          if (!take_item(k, &it)) {
            ok = false;
            break;
          }
          if (it.n == 0) break;
          // O += P(j) V(j) once the softmax has written P(j); the item's first
          // tile starts O afresh once the previous item's epilogue read it
          for (int j = 0; j < it.n; ++j, ++g) {
            const int pb = g & 1, vs = g % kVStages;
            if ((j == 0 && k > 0 && !ptx::mbar_wait(&bars->o_free, (k - 1) & 1, fail)) ||
                !ptx::mbar_wait(&bars->p_full[pb], (g >> 1) & 1, fail) ||
                !ptx::mbar_wait(&bars->v_full[vs], (g / kVStages) & 1, fail)) {
              ok = false;
              break;
            }
            ptx::tc_fence_after();
            const uint64_t vd = vdesc + (uint64_t)((vs * kVStage) >> 4);
#pragma unroll
            for (int kk = 0; kk < kKT / 16; ++kk)
              ptx::mma_bf16_ts(tmem + kTmemO, tmem + kTmemP + pb * 64 + kk * 8,
                               vd + (uint64_t)((kk * 2048) >> 4), idesc_o, (j | kk) != 0);
            ptx::mma_commit(&bars->pv_done[pb]);
            ptx::mma_commit(&bars->v_empty[vs]);
          }
          if (ok) ptx::mma_commit(&bars->o_done);
        }
      }
      if (!ok) set_fail();
      // every MMA this thread issued has completed before TMEM is freed
      uint64_t *dr = &bars->drain[warp == 1 ? 0 : 1];
      ptx::mma_commit(dr);
      ptx::mbar_wait(dr, 0);
    }
  } else {
    // ============ softmax and epilogue (warps 2-9, a pair per row quarter) ============
    // warps w and w+4 share TMEM lanes 32*(w%4).. (one SM sub-partition) and
    // split the 128 key columns of a tile, then the 128 output columns
    const int wq = warp & 3;
    const int ch = (warp - 2) >> 2;  // column half
    const int row = wq * 32 + lane;  // query row of the tile = TMEM lane
    const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
    float *red = reinterpret_cast<float *>(smem + kOffRed);
    // both warps of the pair arrive (release: the value written before is
    // visible), then wait with a bounded wait
    auto pair_exchange = [&](uint64_t *bar, uint32_t parity) -> bool {
      ptx::mbar_arrive(bar);
      return wait_warp(bar, parity, fail);
    };
    auto take = [&](int k, Item *it) -> bool {
      if (!wait_warp(&bars->item_full[k & 1], (k >> 1) & 1, fail)) return false;
      *it = bars->items[k & 1];
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&bars->item_empty[k & 1]);
      return true;
    };
    // the query rows of the item whose query is ring fill f, into TMEM (A
    // operand of Q K^T): box b holds elements 64b.., its 16-byte chunk c of
    // row r at (c ^ r%8); this warp takes three of the six 64-element
    // halves-of-boxes
    auto load_query = [&](int f) -> bool {
      if (!wait_warp(&bars->k_full[f % kKStages], (f / kKStages) & 1, fail)) return false;
      const uint8_t *qrow = smem + kOffK + (f % kKStages) * kKStage + row * 128;
#pragma unroll
      for (int gq = 0; gq < 3; ++gq) {
        const int part = 3 * ch + gq, bx = part >> 1, hh = part & 1;
        uint32_t v[16];
#pragma unroll
        for (int c2 = 0; c2 < 4; ++c2) {
          const int c = 4 * hh + c2;
          const uint4 u = *reinterpret_cast<const uint4 *>(qrow + bx * kBox + ((c ^ (row & 7)) << 4));
          v[4 * c2] = u.x;
          v[4 * c2 + 1] = u.y;
          v[4 * c2 + 2] = u.z;
          v[4 * c2 + 3] = u.w;
        }
        ptx::tmem_st16_nc(tmem + lane_base + kTmemQ + bx * 32 + hh * 16, v);
      }
      ptx::tmem_st_wait();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&bars->q_tmem);
      return true;
    };
    int f = 0, g = 0;  // K-ring fills, score tiles (all items)
    Item it;
    bool ok = take(0, &it) && (it.n == 0 || load_query(f));
    for (int k = 0; ok && it.n > 0; ++k) {
      const int n = it.n;
      const int q = it.q0 + row;                    // position in the prompt
      const int qlim = q < it.T ? q : it.T - 1;     // last visible key (rows past T: all keys)
      float m_used = -INFINITY, l = 0.f;  // m_used in scaled base-2 units
      for (int j = 0; j < n && ok; ++j, ++g) {
        const int s = g & 1;
        if (!wait_warp(&bars->s_full, g & 1, fail)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        float x[64];
#pragma unroll
        for (int c = 0; c < 64; c += 16) {
          float v[16];
          ptx::tmem_ld16(tmem + lane_base + kTmemS + ch * 64 + c, v);
#pragma unroll
          for (int i = 0; i < 16; ++i) x[c + i] = v[i];
        }
        ptx::tmem_ld_wait();
        // the score columns may take the next tile now
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&bars->s_free);
        if (j == n - 1) {
          // the diagonal tile: keys past this row's position are masked
          // (every key of an earlier tile precedes every query of the item)
          const int lim = qlim - j * kKT - ch * 64;
#pragma unroll
          for (int c = 0; c < 64; ++c) x[c] = c <= lim ? x[c] : -INFINITY;
        }
        float m4[4] = {x[0], x[1], x[2], x[3]};
#pragma unroll
        for (int c = 4; c < 64; c += 4)
#pragma unroll
          for (int i = 0; i < 4; ++i) m4[i] = fmaxf(m4[i], x[c + i]);
        float mt = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
        // the pair's row maxima meet in shared memory (one buffer per tile
        // parity, so a fast warp cannot overwrite a value its partner has
        // yet to read)
        red[(s * 2 + ch) * 128 + row] = mt;
        if (!pair_exchange(&bars->pair_max[wq][s], (g >> 1) & 1)) {
          ok = false;
          break;
        }
        mt = fmaxf(mt, red[(s * 2 + (ch ^ 1)) * 128 + row]) * a.scale_log2;
        const bool grow = mt > m_used + kRescaleThreshold;
        float alpha = 1.f;
        if (grow) {
          alpha = ptx::ex2(m_used - mt);  // 0 on the item's first tile (m_used = -inf)
          m_used = mt;
        }
        l *= alpha;
        if (j > 0 && __any_sync(0xffffffffu, grow)) {
          // O holds the item's tiles before this one: rescale this warp's
          // rows and columns once the previous P V is in (both warps of the
          // pair take the same decision)
          if (!wait_warp(&bars->pv_done[(g - 1) & 1], ((g - 1) >> 1) & 1, fail)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
#pragma unroll
          for (int c = 0; c < 64; c += 16) {
            float v[16];
            ptx::tmem_ld16(tmem + lane_base + kTmemO + ch * 64 + c, v);
            ptx::tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 16; ++i) v[i] *= alpha;
            ptx::tmem_st16(tmem + lane_base + kTmemO + ch * 64 + c, v);
          }
        }
        // P buffer s was last read by the P V of tile g - 2
        if (g >= 2 && !wait_warp(&bars->pv_done[s], ((g - 2) >> 1) & 1, fail)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const float nm = -m_used;
        float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int c = 0; c < 64; c += 32) {
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float p0 = ptx::ex2(fmaf(x[c + 2 * i], a.scale_log2, nm));
            const float p1 = ptx::ex2(fmaf(x[c + 2 * i + 1], a.scale_log2, nm));
            ls[i & 3] += p0 + p1;
            pk[i] = ptx::pack_bf16x2(p0, p1);
          }
          ptx::tmem_st16_nc(tmem + lane_base + kTmemP + s * 64 + ch * 32 + c / 2, pk);
        }
        l += (ls[0] + ls[1]) + (ls[2] + ls[3]);
        ptx::tmem_st_wait();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&bars->p_full[s]);
      }
      if (!ok) break;
      // the pair's row sums
      red[(4 + ch) * 128 + row] = l;
      if (!pair_exchange(&bars->pair_sum[wq], k & 1)) {
        ok = false;
        break;
      }
      l += red[(4 + (ch ^ 1)) * 128 + row];
      // the next item's query goes into TMEM before this item's epilogue (every
      // Q K^T of this item has completed), so its first Q K^T overlaps it
      f += n + 1;
      Item nx;
      if (!take(k + 1, &nx) || (nx.n > 0 && !load_query(f))) {
        ok = false;
        break;
      }
      if (!wait_warp(&bars->o_done, k & 1, fail)) {
        ok = false;
        break;
      }
      ptx::tc_fence_after();
      const bool store = q < it.T;
      const float inv = 1.f / l;
      const size_t orow = (size_t)(it.tok0 + (store ? q : 0)) * a.H + it.h;
#pragma unroll
      for (int c = 0; c < 64; c += 16) {
        float v[16];
        ptx::tmem_ld16(tmem + lane_base + kTmemO + ch * 64 + c, v);
        ptx::tmem_ld_wait();
        uint32_t pk[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) pk[i] = ptx::pack_bf16x2(v[2 * i] * inv, v[2 * i + 1] * inv);
        if (store) {
          uint4 *d4 = reinterpret_cast<uint4 *>(a.out + orow * kDh + ch * 64 + c);
          d4[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
          d4[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
        }
      }
      if (store && ch == 0) a.lse[orow] = (m_used + log2f(l)) * kLn2;
      // O may take the next item
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&bars->o_free);
      it = nx;
    }
    if (!ok) set_fail();
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 512);
  }
  if (threadIdx.x == 0 && bars->fail) set_device_error(a.err, kDevTimeout);
}

// ---- keys and values rebuilt from the latents ----
//
// [W_UK[h] c_t ; W_UV[h] c_t] (256 columns, stored as four 64-column chunks
// kv[h][c][t][64], token-minor) for a tile of 128 tokens and kRebuildHeads
// consecutive heads per CTA:
//   D[t][n] = sum_c C[t][c] W[n][c]   M = 128 tokens, N = 256 (W_UK[h] rows
//   then W_UV[h] rows), K = d_c = 512
// The latent tile (128 x 512, 128 KB) is loaded once and stays in shared
// memory; the weights stream through a ring of 64-wide K chunks (W_UK and
// W_UV boxes side by side: one 256-row K-major operand).  Two TMEM
// accumulators (256 columns each) let the epilogue of one head overlap the
// MMAs of the next.  Thread = token row = TMEM lane: each thread writes its
// token's 128-byte row of each chunk, and a warp's 32 consecutive tokens
// fill 4 KB of contiguous memory.
constexpr int kRebuildHeads = 8;
constexpr int kRStages = 3;
constexpr uint32_t kRBoxA = 128 * 128;       // 128 tokens x 64 latents
constexpr uint32_t kROffA = 0;                // 8 boxes: latents 0-63, 64-127, ...
constexpr uint32_t kROffB = 8 * kRBoxA;       // ring of [W_UK chunk ; W_UV chunk]
constexpr uint32_t kRStage = 2 * 128 * 128;   // 256 rows x 128 B
constexpr uint32_t kROffBars = kROffB + kRStages * kRStage;

struct RBars {
  uint64_t a_full;
  uint64_t b_full[kRStages], b_empty[kRStages];
  uint64_t acc_full[2], acc_empty[2];
  uint64_t drain;
  uint32_t tmem;
  int fail;
};
constexpr uint32_t kRSmemBytes = 1024 + kROffBars + ((sizeof(RBars) + 15) / 16) * 16;
static_assert(kRSmemBytes <= 232448, "over the 227 KB shared-memory limit");

struct RebuildArgs {
  int T, H;
  __nv_bfloat16 *kv;  // [H][4][T][64]: 64-column chunks of [K_nope | V], token-minor
  int *err;
  unsigned long long *next_item;  // the attention kernel's work-list counter, zeroed here
};

__global__ void __launch_bounds__(kRThreads, 1)
    kv_rebuild_kernel(const __grid_constant__ CUtensorMap tm_c,    // c_kv [T][512]
                      const __grid_constant__ CUtensorMap tm_wuk,  // W_UK [H*128][512]
                      const __grid_constant__ CUtensorMap tm_wuv,  // W_UV [H*128][512]
                      RebuildArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  RBars *bars = reinterpret_cast<RBars *>(smem + kROffBars);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t0 = blockIdx.x * 128;
  const int h0 = blockIdx.y * kRebuildHeads;
  const int nh = a.H - h0 < kRebuildHeads ? a.H - h0 : kRebuildHeads;
  constexpr int kChunks = kDc / 64;
  // the attention kernel that follows in the stream starts its work list at 0
  if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) *a.next_item = 0;

  if (threadIdx.x == 0) {
    ptx::mbar_init(&bars->a_full, 1);
    for (int i = 0; i < kRStages; ++i) {
      ptx::mbar_init(&bars->b_full[i], 1);
      ptx::mbar_init(&bars->b_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(&bars->acc_full[i], 1);
      ptx::mbar_init(&bars->acc_empty[i], 4);
    }
    ptx::mbar_init(&bars->drain, 1);
    bars->fail = 0;
    ptx::fence_mbar_init();
    ptx::tma_prefetch_desc(&tm_c);
    ptx::tma_prefetch_desc(&tm_wuk);
    ptx::tma_prefetch_desc(&tm_wuv);
  }
  if (warp == 1) ptx::tmem_alloc(&bars->tmem, 512);
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = bars->tmem;
  volatile int *fail = &bars->fail;

  if (warp == 0) {
    // ================= TMA producer =================
    if (lane == 0) {
      ptx::mbar_arrive_expect_tx(&bars->a_full, 8 * kRBoxA);
      for (int k = 0; k < kChunks; ++k)
        ptx::tma_load_2d(smem + kROffA + k * kRBoxA, &tm_c, &bars->a_full, k * 64, t0);
      const int nf = nh * kChunks;
      int f = 0;
      for (; f < nf; ++f) {
        const int s = f % kRStages, h = h0 + f / kChunks, k = f % kChunks;
        if (f >= kRStages &&
            !ptx::mbar_wait(&bars->b_empty[s], ((f / kRStages) - 1) & 1, fail)) {
          atomicExch(const_cast<int *>(fail), 1);
          break;
        }
        uint8_t *dst = smem + kROffB + s * kRStage;
        ptx::mbar_arrive_expect_tx(&bars->b_full[s], kRStage);
        ptx::tma_load_2d(dst, &tm_wuk, &bars->b_full[s], k * 64, h * kDh);
        ptx::tma_load_2d(dst + kRStage / 2, &tm_wuv, &bars->b_full[s], k * 64, h * kDh);
      }
      // never leave with copies in flight
      ptx::mbar_wait(&bars->a_full, 0);
      for (int i = f - kRStages < 0 ? 0 : f - kRStages; i < f; ++i)
        ptx::mbar_wait(&bars->b_full[i % kRStages], (i / kRStages) & 1);
    }
  } else if (warp == 1) {
    // ================= MMA issuer =================
    if (lane == 0) {
      const uint32_t idesc = ptx::idesc_bf16(128, 256, false, false);
      const uint64_t adesc = ptx::smem_desc(ptx::smem_u32(smem + kROffA), 16, 1024, ptx::kSw128);
      const uint64_t bdesc = ptx::smem_desc(ptx::smem_u32(smem + kROffB), 16, 1024, ptx::kSw128);
      bool ok = ptx::mbar_wait(&bars->a_full, 0, fail);
      ptx::tc_fence_after();
      for (int g = 0; g < nh && ok; ++g) {
        const int buf = g & 1;
        if (g >= 2 && !ptx::mbar_wait(&bars->acc_empty[buf], ((g - 2) >> 1) & 1, fail)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        for (int k = 0; k < kChunks; ++k) {
          const int f = g * kChunks + k, s = f % kRStages;
          if (!ptx::mbar_wait(&bars->b_full[s], (f / kRStages) & 1, fail)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint64_t ad = adesc + (uint64_t)((k * kRBoxA) >> 4);
          const uint64_t bd = bdesc + (uint64_t)((s * kRStage) >> 4);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            ptx::mma_bf16(tmem + buf * 256, ad + (uint64_t)((kk * 32) >> 4),
                          bd + (uint64_t)((kk * 32) >> 4), idesc, (k | kk) != 0);
          ptx::mma_commit(&bars->b_empty[s]);
        }
        if (ok) ptx::mma_commit(&bars->acc_full[buf]);
      }
      if (!ok) atomicExch(const_cast<int *>(fail), 1);
      ptx::mma_commit(&bars->drain);
      ptx::mbar_wait(&bars->drain, 0);
    }
  } else {
    // ================= epilogue (warps 2-5) =================
    const int wq = warp & 3;
    const int row = wq * 32 + lane;
    const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
    const bool store = t0 + row < a.T;
    for (int g = 0; g < nh; ++g) {
      const int buf = g & 1;
      if (!wait_warp(&bars->acc_full[buf], (g >> 1) & 1, fail)) {
        atomicExch(const_cast<int *>(fail), 1);
        break;
      }
      ptx::tc_fence_after();
      // the 64-column chunk c (0-1 K_nope, 2-3 V) of head h0 + g for token t
      // lives at kv[((h0 + g) * 4 + c) * T + t][64]: a warp's 32 consecutive
      // tokens fill 4 KB of contiguous rows
      __nv_bfloat16 *dst = a.kv + ((size_t)(h0 + g) * 4 * a.T + (store ? t0 + row : 0)) * 64;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        float v[8][16];
#pragma unroll
        for (int i = 0; i < 8; ++i)
          ptx::tmem_ld16(tmem + lane_base + buf * 256 + half * 128 + i * 16, v[i]);
        ptx::tmem_ld_wait();
        if (store) {
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            uint32_t pk[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) pk[e] = ptx::pack_bf16x2(v[i][2 * e], v[i][2 * e + 1]);
            // 32 bytes per lane in one store (chunk rows are 128-byte aligned)
            asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(
                             dst + (size_t)(2 * half + (i >> 2)) * a.T * 64 + (i & 3) * 16),
                         "r"(pk[0]), "r"(pk[1]), "r"(pk[2]), "r"(pk[3]), "r"(pk[4]), "r"(pk[5]),
                         "r"(pk[6]), "r"(pk[7])
                         : "memory");
          }
        }
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&bars->acc_empty[buf]);
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 512);
  }
  if (threadIdx.x == 0 && bars->fail) set_device_error(a.err, kDevTimeout);
}

cudaError_t launch_kv_rebuild(const void *c_kv, const void *W_UK, const void *W_UV, void *kv,
                              int T, const mla_dims &d, int *err,
                              unsigned long long *next_item, cudaStream_t st) {
  const uint64_t rows = (uint64_t)d.H * kDh;
  CUtensorMap tm_c, tm_wuk, tm_wuv;
  if (!make_tmap_2d_bf16(&tm_c, c_kv, kDc, T, kDc * 2, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tmap_2d_bf16(&tm_wuk, W_UK, kDc, rows, kDc * 2, 64, 128,
                         CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tmap_2d_bf16(&tm_wuv, W_UV, kDc, rows, kDc * 2, 64, 128,
                         CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(kv_rebuild_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)kRSmemBytes);
  if (e != cudaSuccess) return e;
  RebuildArgs a;
  a.T = T;
  a.H = d.H;
  a.kv = static_cast<__nv_bfloat16 *>(kv);
  a.err = err;
  a.next_item = next_item;
  const dim3 grid((T + 127) / 128, (d.H + kRebuildHeads - 1) / kRebuildHeads);
  kv_rebuild_kernel<<<grid, kRThreads, kRSmemBytes, st>>>(tm_c, tm_wuk, tm_wuv, a);
  return cudaGetLastError();
}

}  // namespace

bool tc_prefill_supported(const mla_dims &d) {
  return d.dtype == MLA_BF16 && d.d_h == kDh && d.d_c == kDc && d.d_r == kDr;
}

size_t prefill_workspace_bytes(int total, const mla_dims &d) {
  return kWsHeader + align_up((size_t)total * d.H * 2 * kDh * sizeof(__nv_bfloat16), 256);
}

cudaError_t launch_prefill_tc(const void *q_nope, const void *q_rope, const void *c_kv,
                              const void *k_r, const void *W_UK, const void *W_UV,
                              const int32_t *cu_seqlens, int B, int max_seqlen, int total,
                              const mla_dims &d, float scale, void *out, float *lse,
                              void *workspace, cudaStream_t st) {
  char *ws = static_cast<char *>(workspace);
  void *kv = ws + kWsHeader;
  // [K_nope | V] of every (token, head): [total][H][256]
  // workspace header: the error word at byte 0, the work-list counter at 8
  unsigned long long *next_item = reinterpret_cast<unsigned long long *>(ws + 8);
  cudaError_t e = launch_kv_rebuild(c_kv, W_UK, W_UV, kv, total, d, reinterpret_cast<int *>(ws),
                                    next_item, st);
  if (e != cudaSuccess) return e;
  const uint64_t H = (uint64_t)d.H;
  CUtensorMap tm_q, tm_qr, tm_kv, tm_kr;
  if (!make_tmap_2d_bf16(&tm_q, q_nope, H * kDh, total, H * kDh * 2, 64, kQT,
                         CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tmap_2d_bf16(&tm_qr, q_rope, H * kDr, total, H * kDr * 2, 64, kQT,
                         CU_TENSOR_MAP_SWIZZLE_128B) ||
      // [K_nope | V] as [H * 4 chunks][total][64]: boxes of 128 tokens x 64
      // columns, the same shared-memory tiles as a row-major view would give
      !make_tmap_3d(&tm_kv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, kv, 64, total, (uint64_t)H * 4,
                    128, (uint64_t)total * 128, 64, kKT, 1, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tmap_2d_bf16(&tm_kr, k_r, kDr, total, kDr * 2, 64, kKT, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  e = cudaFuncSetAttribute(prefill_attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)kSmemBytes);
  if (e != cudaSuccess) return e;
  PrefillArgs a;
  a.cu_seqlens = cu_seqlens;
  a.B = B;
  a.H = d.H;
  a.max_seqlen = max_seqlen;
  a.total = total;
  a.scale_log2 = scale * kLog2e;
  a.out = static_cast<__nv_bfloat16 *>(out);
  a.lse = lse;
  a.err = reinterpret_cast<int *>(ws);
  a.nq = (max_seqlen + kQT - 1) / kQT;
  a.total_items = (unsigned long long)B * d.H * a.nq;
  a.next_item = next_item;
  // persistent: one CTA per SM (shared memory and TMEM admit one), each
  // taking (query tile, head, prompt) items from the work list
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
    return cudaErrorInvalidDevice;
  const unsigned grid =
      (unsigned)(a.total_items < (unsigned long long)sms ? a.total_items : (unsigned long long)sms);
  prefill_attn_kernel<<<grid, kThreads, kSmemBytes, st>>>(tm_q, tm_qr, tm_kv, tm_kr, a);
  return cudaGetLastError();
}

}  // namespace mla
