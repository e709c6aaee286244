// Per-head batched GEMMs of the decode step on the 5th-generation tensor
// cores (TMA -> shared memory -> tcgen05.mma -> TMEM -> registers -> global).
//
//   absorb   ("From Vanilla Transformers to Modern LLMs -- Part 3" 3.e.2):
//     q_lat[r,h,c] = sum_a W_UK[h,a,c] q_nope[r,h,a]
//     computed transposed, D[c][r] = A[c][a] B[r][a]: M = c (128 per CTA),
//     N = query rows r, K = d_h.  A = W_UK[h] read MN-major (c contiguous).
//   out_proj ("From Vanilla Transformers to Modern LLMs -- Part 3" 3.g):
//     out[r,h,a] = sum_c W_UV[h,a,c] o_lat[r,h,c]
//     D[a][r] = A[a][c] B[r][c]: M = a (d_h = 128), N = r, K = d_c.
//     Both operands K-major.
//
//   project  ("Multi-Head Latent Attention: Low-Rank KV Compression, Decoupled
//   RoPE, and Matrix Absorption", the latent and RoPE-key projections;
//   "From Vanilla Transformers to Modern LLMs -- Part 3" 3.b, 3.k):
//     [c ; k] [t, m] = sum_x [W_DKV ; W_KR][m, x] h[t, x]
//     D[m][t] = A[m][x] B[t][x]: M = output features, N = new tokens,
//     K = d_model, split over the grid's y axis into fp32 partial sums that
//     proj_finalize_kernel adds, rotates (RoPE on k) and scatters into the
//     paged cache.
//
// The weights are the large operand (16.8 MB per matrix at H = 128) and are
// read exactly once; query rows (N <= 256 per CTA) are the small one.  One
// CTA per (128-wide M tile, head or K split, N tile); 4 warps: warp 0 issues
// TMA, warp 1 issues MMAs, warp 2 owns the TMEM allocation, all 4 drain the
// accumulator (warp w reads TMEM lanes 32w..32w+31).  K is streamed in
// 64-wide chunks through a ring of shared-memory stages (full / empty
// mbarriers).
//
// The kernels are launched as programmatic dependents of the previous kernel
// in the stream.  The producer first issues the weight tiles of every stage
// (no kernel of this library writes weights), then waits for the previous
// kernel to complete before it reads the activations, so the weight stream
// overlaps the tail of the previous kernel; it lets the next kernel launch
// only after that wait.
#include "internal.cuh"
#include "ptx.cuh"
#include "tc.cuh"
#include "tmap.cuh"

namespace mla {
namespace {

__device__ int g_gemm_error = 0;

constexpr int kM = 128;
constexpr int kKChunk = 64;  // one 128-byte swizzle span of bf16
constexpr int kMaxStages = 8;
constexpr uint32_t kABytes = kM * kKChunk * 2;  // 16 KB per chunk

struct GemmArgs {
  int num_k_chunks;  // K / 64
  int rows;          // N extent (query rows)
  int Nt;            // N per CTA (multiple of 16, <= 256)
  int H;
  int M_total;      // output width per head: d_c (absorb) or d_h (out_proj)
  int a_rows_per_head;  // rows of the 2-D weight view per head (d_h)
  int a_cols_per_head;  // K offset of the weight view per y index (split-K)
  int b_cols_per_head;  // columns of the 2-D activation view per head (K)
  int stages;
  __nv_bfloat16 *out;
  // split-K mode (part != nullptr): fp32 partial sums part[y][n][m_ofs + m]
  // of width M_total, rows m_ofs + m >= M_total dropped
  float *part;
  int m_ofs;
  // M tiles from a_tiles on read their A rows from tmA2, from row 0
  int a_tiles;
};

template <bool kAMnMajor>
__global__ void __launch_bounds__(128, 1)
    head_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                     const __grid_constant__ CUtensorMap tmA2,
                     const __grid_constant__ CUtensorMap tmB, GemmArgs g) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // 1024-byte alignment of every operand tile (128B swizzle atoms).
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t b_bytes = g.Nt * 128;
  const uint32_t stage_bytes = kABytes + b_bytes;
  __shared__ uint64_t full[kMaxStages], empty[kMaxStages], done;
  __shared__ uint32_t tmem_base;
  __shared__ int fail;

  const int warp = threadIdx.x >> 5;
  const int m0 = blockIdx.x * kM;
  const int npre = g.num_k_chunks < g.stages ? g.num_k_chunks : g.stages;
  const int h = blockIdx.y;
  const int n0 = blockIdx.z * g.Nt;
  const uint32_t ncols = g.Nt <= 32 ? 32 : (g.Nt <= 64 ? 64 : (g.Nt <= 128 ? 128 : 256));

  if (threadIdx.x == 0) {
    for (int s = 0; s < g.stages; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&empty[s], 1);
    }
    ptx::mbar_init(&done, 1);
    ptx::fence_mbar_init();
    fail = 0;
    ptx::tma_prefetch_desc(&tmA);
    ptx::tma_prefetch_desc(&tmA2);
    ptx::tma_prefetch_desc(&tmB);
  }
  if (warp == 2) ptx::tmem_alloc(&tmem_base, ncols);
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = tmem_base;

  if (warp == 0 && ptx::elect_lane0()) {
    // ---- TMA producer ----
    const bool second = (int)blockIdx.x >= g.a_tiles;
    const CUtensorMap *ta = second ? &tmA2 : &tmA;
    const int am0 = second ? ((int)blockIdx.x - g.a_tiles) * kM : m0;
    auto load_a = [&](int k, int s) {
      uint8_t *a_dst = smem + s * stage_bytes;
      if (kAMnMajor) {
        // two 64(M) x 64(K) boxes: M block j at +8 KB
        ptx::tma_load_2d(a_dst, ta, &full[s], am0, h * g.a_rows_per_head + k * kKChunk);
        ptx::tma_load_2d(a_dst + 8192, ta, &full[s], am0 + 64,
                         h * g.a_rows_per_head + k * kKChunk);
      } else {
        ptx::tma_load_2d(a_dst, ta, &full[s], h * g.a_cols_per_head + k * kKChunk,
                         h * g.a_rows_per_head + am0);
      }
    };
    auto load_b = [&](int k, int s) {
      ptx::tma_load_2d(smem + s * stage_bytes + kABytes, &tmB, &full[s],
                       h * g.b_cols_per_head + k * kKChunk, n0);
    };
    // the weights of the first stages do not depend on the previous kernel
    for (int k = 0; k < npre; ++k) {
      ptx::mbar_arrive_expect_tx(&full[k], stage_bytes);  // A now, B below
      load_a(k, k);
    }
    ptx::grid_dependency_wait();  // the activations may come from the previous kernel
    ptx::launch_dependents();
    for (int k = 0; k < npre; ++k) load_b(k, k);
    int issued = npre;
    for (int k = npre; k < g.num_k_chunks; ++k) {
      const int s = k % g.stages;
      if (!ptx::mbar_wait(&empty[s], ((k / g.stages) - 1) & 1, &fail)) {
        atomicExch(&fail, 1);
        break;
      }
      ptx::mbar_arrive_expect_tx(&full[s], stage_bytes);
      load_a(k, s);
      load_b(k, s);
      ++issued;
    }
    // never leave with copies in flight
    for (int k = issued - g.stages < 0 ? 0 : issued - g.stages; k < issued; ++k)
      if (!ptx::mbar_wait(&full[k % g.stages], (k / g.stages) & 1)) atomicExch(&fail, 1);
  } else if (warp == 1 && ptx::elect_lane0()) {
    // ---- MMA issuer ----
    const uint32_t idesc = ptx::idesc_bf16(kM, g.Nt, kAMnMajor, false);
    for (int k = 0; k < g.num_k_chunks; ++k) {
      const int s = k % g.stages;
      if (!ptx::mbar_wait(&full[s], (k / g.stages) & 1, &fail)) {
        atomicExch(&fail, 1);
        break;
      }
      ptx::tc_fence_after();
      const uint32_t a_addr = ptx::smem_u32(smem + s * stage_bytes);
      const uint32_t b_addr = a_addr + kABytes;
#pragma unroll
      for (int kk = 0; kk < kKChunk / 16; ++kk) {
        const uint64_t adesc =
            kAMnMajor ? ptx::smem_desc(a_addr + kk * 2048, 8192, 1024, ptx::kSw128)
                      : ptx::smem_desc(a_addr + kk * 32, 16, 1024, ptx::kSw128);
        const uint64_t bdesc = ptx::smem_desc(b_addr + kk * 32, 16, 1024, ptx::kSw128);
        ptx::mma_bf16(tmem, adesc, bdesc, idesc, (k | kk) != 0);
      }
      ptx::mma_commit(&empty[s]);
    }
    ptx::mma_commit(&done);
  }
  __syncwarp();

  // ---- epilogue: TMEM -> bf16 global, all 4 warps ----
  const bool ok = ptx::mbar_wait(&done, 0);
  ptx::tc_fence_after();
  if (!ok) atomicExch(&fail, 1);
  if (ok && g.part) {
    const int m = g.m_ofs + m0 + warp * 32 + (threadIdx.x & 31);
    float *dst = g.part + (size_t)h * g.rows * g.M_total + m;
    for (int c0 = 0; c0 < g.Nt; c0 += 16) {
      float v[16];
      ptx::tmem_ld16(tmem + ((uint32_t)(warp * 32) << 16) + c0, v);
      ptx::tmem_ld_wait();
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int n = n0 + c0 + i;
        if (n < g.rows && m < g.M_total) dst[(size_t)n * g.M_total] = v[i];
      }
    }
  } else if (ok) {
    const int m_local = warp * 32 + (threadIdx.x & 31);
    const size_t row_stride = (size_t)g.H * g.M_total;
    __nv_bfloat16 *dst = g.out + (size_t)h * g.M_total + m0 + m_local;
    for (int c0 = 0; c0 < g.Nt; c0 += 16) {
      float v[16];
      ptx::tmem_ld16(tmem + ((uint32_t)(warp * 32) << 16) + c0, v);
      ptx::tmem_ld_wait();
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int n = n0 + c0 + i;
        if (n < g.rows) dst[(size_t)n * row_stride] = __float2bfloat16_rn(v[i]);
      }
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 2) ptx::tmem_dealloc(tmem, ncols);
  if (threadIdx.x == 0 && fail) atomicCAS(&g_gemm_error, 0, kDevTimeout);
}

int pick_nt(int rows) {
  const int r16 = (rows + 15) / 16 * 16;
  return r16 > 256 ? 256 : r16;
}

// Launch as a programmatic dependent of the previous kernel in the stream.
// max_stages bounds the ring (the per-head decode GEMMs keep all of K in
// flight, the split-K projections four stages and two CTAs per SM).
template <bool kAMnMajor>
cudaError_t launch_head_gemm(const CUtensorMap &tmA, const CUtensorMap &tmA2,
                             const CUtensorMap &tmB, GemmArgs g, int m_tiles, cudaStream_t st,
                             int max_stages = 4) {
  const size_t stage_bytes = kABytes + (size_t)g.Nt * 128;
  const int fit = (int)((200u << 10) / stage_bytes);  // leave room below 227 KB
  int stages = g.num_k_chunks < max_stages ? g.num_k_chunks : max_stages;
  if (stages > fit) stages = fit;
  if (stages > kMaxStages) stages = kMaxStages;
  g.stages = stages < 1 ? 1 : stages;
  const size_t smem = 1024 + (size_t)g.stages * stage_bytes;
  auto kern = head_gemm_kernel<kAMnMajor>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(m_tiles, g.H, (g.rows + g.Nt - 1) / g.Nt);
  cfg.blockDim = dim3(128, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = pdl;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, tmA, tmA2, tmB, g);
}

}  // namespace

bool tc_gemm_supported(const mla_dims &d) {
  return d.dtype == MLA_BF16 && d.d_h == 128 && d.d_c == 512;
}

int read_and_clear_gemm_error() {
  int v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_gemm_error, sizeof(int)) != cudaSuccess) return -1;
  if (v != 0) cudaMemcpyToSymbol(g_gemm_error, &zero, sizeof(int));
  return v;
}

// ---- absorb and out-proj: one CTA per (head, row tile), whole operands ----
//
// Each per-head GEMM of the decode step is small (a 128 x 512 weight, at most
// a few hundred query rows), so a CTA takes a whole head: the weight arrives
// in ONE 3-D TMA copy (8 column blocks of 64, 128 KB) and the head's query
// rows in one more.  One SM completes only about two copies per microsecond,
// so the copy count, not the bytes, set the time of the chunked version.
//   absorb:   D[c][r] = W_UK[h][a][c] q_nope[r][h][a]: four M = 128 tiles of
//             c, N = query rows, K = a (d_h = 128); A read MN-major.
//   out_proj: D[a][r] = W_UV[h][a][c] o_lat[r][h][c]: M = a (128), N = rows,
//             K = c (d_c = 512); both operands K-major.
// The weight copy is issued before waiting for the previous kernel (no kernel
// of this library writes weights); the rows are read after the wait.

namespace {

constexpr uint32_t kWholeA = 128 * 512 * 2;  // one head's weight, 128 KB
constexpr int kWholeThreads = 256;

template <bool kAbsorb>
__global__ void __launch_bounds__(kWholeThreads, 1)
    head_whole_kernel(const __grid_constant__ CUtensorMap tmA,
                      const __grid_constant__ CUtensorMap tmB, __nv_bfloat16 *out, int rows,
                      int Nt, int H) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t *sA = smem, *sB = smem + kWholeA;
  __shared__ uint64_t full, done;
  __shared__ uint32_t tmem_base;
  __shared__ int fail;
  constexpr int kMTiles = kAbsorb ? 4 : 1;       // M tiles of 128
  constexpr int kBBlocks = kAbsorb ? 2 : 8;      // 64-wide K blocks of B
  constexpr int kKSteps = kAbsorb ? 8 : 32;      // K-steps of 16
  const int warp = threadIdx.x >> 5;
  const int h = blockIdx.x, n0 = blockIdx.y * Nt;
  const uint32_t b_bytes = (uint32_t)kBBlocks * Nt * 128;
  const int cols = kMTiles * Nt;  // TMEM: a power of two >= 32
  const uint32_t ncols = cols <= 32 ? 32 : cols <= 64 ? 64 : cols <= 128 ? 128 : cols <= 256 ? 256 : 512;

  if (threadIdx.x == 0) {
    ptx::mbar_init(&full, 1);
    ptx::mbar_init(&done, 1);
    ptx::fence_mbar_init();
    fail = 0;
  }
  if (warp == 2) ptx::tmem_alloc(&tmem_base, ncols);
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = tmem_base;

  if (warp == 0 && ptx::elect_lane0()) {
    ptx::mbar_arrive_expect_tx(&full, kWholeA + b_bytes);
    // the weight: [64-column block][128 rows][64], one copy
    ptx::tma_load_3d(sA, &tmA, &full, 0, h * 128, 0);
    ptx::grid_dependency_wait();  // the rows may come from the previous kernel
    ptx::launch_dependents();
    ptx::tma_load_3d(sB, &tmB, &full, 0, n0, h * kBBlocks);
  } else if (warp == 1 && ptx::elect_lane0()) {
    const uint32_t idesc = ptx::idesc_bf16(128, Nt, kAbsorb, false);
    if (!ptx::mbar_wait(&full, 0, &fail)) {
      atomicExch(&fail, 1);
    } else {
      ptx::tc_fence_after();
      const uint32_t a_addr = ptx::smem_u32(sA), b_addr = ptx::smem_u32(sB);
#pragma unroll
      for (int m = 0; m < kMTiles; ++m) {
#pragma unroll
        for (int kk = 0; kk < kKSteps; ++kk) {
          // A: absorb MN-major (c blocks 2m, 2m+1 of 128 a-rows, 16 KB apart;
          // 16 a-rows per K-step); out-proj K-major (K-step kk in block kk/4)
          const uint64_t adesc =
              kAbsorb ? ptx::smem_desc(a_addr + 2 * m * 16384 + kk * 2048, 16384, 1024, ptx::kSw128)
                      : ptx::smem_desc(a_addr + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024,
                                       ptx::kSw128);
          const uint64_t bdesc = ptx::smem_desc(b_addr + (kk >> 2) * (Nt * 128) + (kk & 3) * 32,
                                                16, 1024, ptx::kSw128);
          ptx::mma_bf16(tmem + m * Nt, adesc, bdesc, idesc, kk != 0);
        }
      }
    }
    ptx::mma_commit(&done);
  }
  __syncwarp();

  // ---- epilogue: TMEM -> bf16 global ----
  // Lane = output column (c or a), TMEM column = query row.  Each M tile is
  // transposed through the weight's (now idle) shared memory into [row][128]
  // bf16, then every row leaves as 256 contiguous bytes (16-byte stores).
  const bool ok = ptx::mbar_wait(&done, 0);
  ptx::tc_fence_after();
  if (!ok || fail) atomicExch(&fail, 1);
  __syncthreads();  // every thread has seen `fail`; the MMAs are done with sA
  if (!fail) {
    const int width = kAbsorb ? 512 : 128;
    const size_t row_stride = (size_t)H * width;
    const int lane = threadIdx.x & 31, quad = warp & 3, half = warp >> 2;
    const int nchunks = Nt / 16;  // 16 query rows per TMEM load
    for (int m = 0; m < kMTiles; ++m) {
      __nv_bfloat16 *stage = reinterpret_cast<__nv_bfloat16 *>(sA) + (size_t)m * Nt * 128;
      // warps q and q + 4 share TMEM lanes 32q..32q+31 and take alternate
      // 16-row chunks, four loads in flight per wait
      for (int j0 = half; j0 < nchunks; j0 += 8) {
        float v[4][16];
#pragma unroll
        for (int u = 0; u < 4; ++u)
          if (j0 + 2 * u < nchunks)
            ptx::tmem_ld16(tmem + ((uint32_t)(quad * 32) << 16) + m * Nt + (j0 + 2 * u) * 16, v[u]);
        ptx::tmem_ld_wait();
#pragma unroll
        for (int u = 0; u < 4; ++u)
          if (j0 + 2 * u < nchunks)
#pragma unroll
            for (int i = 0; i < 16; ++i)
              stage[(size_t)((j0 + 2 * u) * 16 + i) * 128 + quad * 32 + lane] =
                  __float2bfloat16_rn(v[u][i]);
      }
    }
    __syncthreads();
    // thread t stores 16-byte piece t % 16 of rows t / 16, t / 16 + 16, ...
    const int nrows = min(Nt, rows - n0), k = threadIdx.x & 15;
    for (int m = 0; m < kMTiles; ++m)
      for (int r = threadIdx.x >> 4; r < nrows; r += kWholeThreads / 16) {
        const uint4 x = reinterpret_cast<const uint4 *>(sA)[((size_t)m * Nt + r) * 16 + k];
        __nv_bfloat16 *dst = out + (size_t)(n0 + r) * row_stride + (size_t)h * width + m * 128;
        reinterpret_cast<uint4 *>(dst)[k] = x;
      }
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 2) ptx::tmem_dealloc(tmem, ncols);
  if (threadIdx.x == 0 && fail) atomicCAS(&g_gemm_error, 0, kDevTimeout);
}

template <bool kAbsorb>
cudaError_t launch_head_whole(const CUtensorMap &tmA, const CUtensorMap &tmB, void *out,
                              int rows, int Nt, int H, cudaStream_t st) {
  const int kBBlocks = kAbsorb ? 2 : 8;
  const size_t smem = 1024 + kWholeA + (size_t)kBBlocks * Nt * 128;
  auto kern = head_whole_kernel<kAbsorb>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(H, (rows + Nt - 1) / Nt, 1);
  cfg.blockDim = dim3(kWholeThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = pdl;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, tmA, tmB, static_cast<__nv_bfloat16 *>(out), rows, Nt,
                            H);
}

// Query rows per CTA: a multiple of 16, at most `cap` (TMEM columns of the
// absorb's four accumulators, shared memory of the out-proj's rows).
int pick_rows_tile(int rows, int cap) {
  const int r16 = (rows + 15) / 16 * 16;
  return r16 > cap ? cap : r16;
}

}  // namespace

cudaError_t launch_absorb_tc(const void *q_nope, const void *W_UK, void *q_lat, int rows,
                             const mla_dims &d, cudaStream_t st) {
  CUtensorMap tmA, tmB;
  const int Nt = pick_rows_tile(rows, 128);
  // W_UK [H*d_h][d_c] as [column block of 64][row][64]: one box per head,
  // 8 blocks x 128 rows
  if (!make_tmap_3d(&tmA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, W_UK, 64, (uint64_t)d.H * d.d_h,
                    d.d_c / 64, (uint64_t)d.d_c * 2, 128, 64, 128, d.d_c / 64,
                    CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  // q_nope [rows][H*d_h] as [block of 64][row][64]: two blocks of one head
  if (!make_tmap_3d(&tmB, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, q_nope, 64, rows,
                    (uint64_t)d.H * d.d_h / 64, (uint64_t)d.H * d.d_h * 2, 128, 64, Nt, 2,
                    CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  return launch_head_whole<true>(tmA, tmB, q_lat, rows, Nt, d.H, st);
}

cudaError_t launch_out_proj_tc(const void *o_lat, const void *W_UV, void *out, int rows,
                               const mla_dims &d, cudaStream_t st) {
  CUtensorMap tmA, tmB;
  const int Nt = pick_rows_tile(rows, 64);
  // W_UV [H*d_h][d_c] as [column block of 64][row][64]: one box per head
  if (!make_tmap_3d(&tmA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, W_UV, 64, (uint64_t)d.H * d.d_h,
                    d.d_c / 64, (uint64_t)d.d_c * 2, 128, 64, 128, d.d_c / 64,
                    CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  // o_lat [rows][H*d_c] as [block of 64][row][64]: eight blocks of one head
  if (!make_tmap_3d(&tmB, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, o_lat, 64, rows,
                    (uint64_t)d.H * d.d_c / 64, (uint64_t)d.H * d.d_c * 2, 128, 64, Nt,
                    d.d_c / 64, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  return launch_head_whole<false>(tmA, tmB, out, rows, Nt, d.H, st);
}

// ---- fused latent / RoPE-key projection into the paged cache ----

namespace {

// RoPE frequencies theta_j = base^(-2j/d_r), j < d_r/2, formed on the host in
// double precision and passed by value.
struct RopeTable {
  double theta[64];
};

RopeTable rope_table(double base, int d_r) {
  RopeTable t = {};
  for (int j = 0; j < d_r / 2 && j < 64; ++j) t.theta[j] = pow(base, -2.0 * j / d_r);
  return t;
}

// cos and sin of pos * theta: the angle is formed in double precision and
// brought into [-pi, pi] by subtracting the nearest multiple of 2 pi (2 pi
// split into a double head and tail), then evaluated in fp32.
__device__ __forceinline__ void rope_cos_sin(int pos, double theta, float *c, float *s) {
  constexpr double kTwoPiHi = 6.283185307179586;       // 2 pi rounded to double
  constexpr double kTwoPiLo = 2.4492935982947064e-16;  // 2 pi minus kTwoPiHi
  const double ang = (double)pos * theta;
  const double k = rint(ang * (1.0 / kTwoPiHi));
  const double r = fma(-k, kTwoPiLo, fma(-k, kTwoPiHi, ang));
  sincosf((float)r, s, c);
}

// Sums the K-split partials of one new token's [c ; k_R] row, rotates the
// k_R pairs (adjacent coordinates (2p, 2p+1), angle pos * base^(-2p/d_r),
// x cos + rotate_half(x) sin; "MLA, dim by dim" 3), and writes the row into
// the paged cache at the token's position.  One CTA per token, one thread
// per coordinate pair.
__global__ void __launch_bounds__(512) proj_finalize_kernel(
    const float *__restrict__ part, int splits, int T, int d_c, int d_r, RopeTable rope,
    __nv_bfloat16 *__restrict__ cache, int num_blocks, const int32_t *__restrict__ block_table,
    int max_blocks, const int32_t *__restrict__ seqlens, int n_new, int bs) {
  ptx::grid_dependency_wait();  // the partial sums of the GEMM just before
  const int t = blockIdx.x;  // token = b * n_new + i
  const int b = t / n_new, i = t % n_new;
  const int pos = seqlens[b] - n_new + i;
  if (pos < 0) return;
  const int lb = pos / bs;
  if (lb >= max_blocks) return;
  const int blk = block_table[(size_t)b * max_blocks + lb];
  if (blk < 0 || blk >= num_blocks) return;  // reported by mla_decode
  const int D = d_c + d_r;
  const int j = threadIdx.x;  // coordinate pair 2j, 2j+1
  if (2 * j >= D) return;
  // eight splits' loads in flight at a time
  const float *src = part + (size_t)t * D + 2 * j;
  const size_t split_stride = (size_t)T * D;
  float a0[8], a1[8];
#pragma unroll
  for (int u = 0; u < 8; ++u) a0[u] = a1[u] = 0.f;
  int s = 0;
  for (; s + 8 <= splits; s += 8) {
    float2 v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) v[u] = *reinterpret_cast<const float2 *>(src + (s + u) * split_stride);
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      a0[u] += v[u].x;
      a1[u] += v[u].y;
    }
  }
  for (; s < splits; ++s) {
    const float2 v = *reinterpret_cast<const float2 *>(src + s * split_stride);
    a0[0] += v.x;
    a1[0] += v.y;
  }
  float x0 = 0.f, x1 = 0.f;
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    x0 += a0[u];
    x1 += a1[u];
  }
  if (2 * j >= d_c) {  // a RoPE pair
    float c, s;
    rope_cos_sin(pos, rope.theta[j - d_c / 2], &c, &s);
    const float r0 = x0 * c - x1 * s, r1 = x1 * c + x0 * s;
    x0 = r0;
    x1 = r1;
  }
  __nv_bfloat162 o;
  o.x = __float2bfloat16_rn(x0);
  o.y = __float2bfloat16_rn(x1);
  *reinterpret_cast<__nv_bfloat162 *>(cache + ((size_t)blk * bs + pos % bs) * D + 2 * j) = o;
}

constexpr int kProjMTiles = 5;  // d_c = 512 (4 tiles) + d_r = 64 (1 tile)

// K chunks per split so that the M tiles x splits CTAs about fill the SMs.
void proj_split(int d_model, int *chunks_per_split, int *splits) {
  const int kchunks = d_model / kKChunk;
  int cps = (kchunks * kProjMTiles + kNumSMs - 1) / kNumSMs;
  if (cps < 1) cps = 1;
  *chunks_per_split = cps;
  *splits = (kchunks + cps - 1) / cps;
}

}  // namespace

bool tc_project_supported(const mla_dims &d, int d_model) {
  return d.dtype == MLA_BF16 && d.d_c == 512 && d.d_r == 64 && d_model > 0 &&
         d_model % kKChunk == 0;
}

size_t project_workspace_bytes(int T, int d_model, const mla_dims &d) {
  int cps, splits;
  proj_split(d_model, &cps, &splits);
  return (size_t)splits * T * (d.d_c + d.d_r) * sizeof(float);
}

cudaError_t launch_project_append_tc(const void *h, const void *W_DKV, const void *W_KR,
                                     int d_model, double rope_base, void *cache, int num_blocks,
                                     const int32_t *block_table, int max_blocks,
                                     const int32_t *seqlens, int B, int n_new,
                                     const mla_dims &d, void *workspace, cudaStream_t st) {
  const int T = B * n_new;
  int cps, splits;
  proj_split(d_model, &cps, &splits);
  const int Nt = pick_nt(T);
  CUtensorMap tmDKV, tmKR, tmH;
  // the weights as [rows][d_model], boxes of 64 x 128 rows (W_KR's 64 rows
  // read as one tile whose upper half is out of range: zeros)
  if (!make_tmap_2d_bf16(&tmDKV, W_DKV, d_model, d.d_c, (uint64_t)d_model * 2, 64, 128,
                         CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tmap_2d_bf16(&tmKR, W_KR, d_model, d.d_r, (uint64_t)d_model * 2, 64, 128,
                         CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tmap_2d_bf16(&tmH, h, d_model, T, (uint64_t)d_model * 2, 64, Nt,
                         CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  GemmArgs g;
  g.num_k_chunks = cps;
  g.rows = T;
  g.Nt = Nt;
  g.H = splits;
  g.M_total = d.d_c + d.d_r;
  g.a_rows_per_head = 0;
  g.a_cols_per_head = cps * kKChunk;
  g.b_cols_per_head = cps * kKChunk;
  g.out = nullptr;
  g.part = static_cast<float *>(workspace);
  g.m_ofs = 0;
  g.a_tiles = d.d_c / kM;  // tiles 0-3 from W_DKV, tile 4 from W_KR
  cudaError_t e = launch_head_gemm<false>(tmDKV, tmKR, tmH, g, kProjMTiles, st);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(T, 1, 1);
  cfg.blockDim = dim3((d.d_c + d.d_r) / 2, 1, 1);
  cfg.stream = st;
  cfg.attrs = pdl;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, proj_finalize_kernel, static_cast<const float *>(workspace),
                            splits, T, d.d_c, d.d_r, rope_table(rope_base, d.d_r),
                            static_cast<__nv_bfloat16 *>(cache), num_blocks, block_table,
                            max_blocks, seqlens, n_new, d.block_size);
}

// ---- output projection over the concatenated heads ----

namespace {

// u[t, :] = bf16(sum over K splits of the fp32 partials); one thread per
// pair of outputs, eight splits' loads in flight at a time.
__global__ void __launch_bounds__(256) splitk_sum_kernel(const float *__restrict__ part,
                                                         int splits, int T, int N,
                                                         __nv_bfloat16 *__restrict__ u) {
  ptx::grid_dependency_wait();  // the partial sums of the GEMM just before
  const int t = blockIdx.y;
  const int j = blockIdx.x * blockDim.x + threadIdx.x;  // output pair 2j, 2j+1
  if (2 * j >= N) return;
  const float *src = part + (size_t)t * N + 2 * j;
  const size_t split_stride = (size_t)T * N;
  float a0[8], a1[8];
#pragma unroll
  for (int q = 0; q < 8; ++q) a0[q] = a1[q] = 0.f;
  int s = 0;
  for (; s + 8 <= splits; s += 8) {
    float2 v[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) v[q] = *reinterpret_cast<const float2 *>(src + (s + q) * split_stride);
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      a0[q] += v[q].x;
      a1[q] += v[q].y;
    }
  }
  for (; s < splits; ++s) {
    const float2 v = *reinterpret_cast<const float2 *>(src + s * split_stride);
    a0[0] += v.x;
    a1[0] += v.y;
  }
  float x0 = 0.f, x1 = 0.f;
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    x0 += a0[q];
    x1 += a1[q];
  }
  __nv_bfloat162 o;
  o.x = __float2bfloat16_rn(x0);
  o.y = __float2bfloat16_rn(x1);
  *reinterpret_cast<__nv_bfloat162 *>(u + (size_t)t * N + 2 * j) = o;
}

// K split of a weight-streaming GEMM with T rows and M outputs.  Each CTA
// streams its chunks at a latency-bound rate (measured: about 1.1 us per
// 16 KB chunk with two ~100 KB CTAs per SM), and every split adds T x M fp32
// partials written and read back (taken at 6 TB/s).  Estimated time:
// (waves of 2 x 148 CTAs) x (chunks per CTA) x 1.1 us + splits x T x M x 8 B
// / 6 TB/s; take the split that minimises it.
void choose_split(int kchunks, int m_tiles, int T, int M, int *chunks_per_split, int *splits) {
  const int slots = 2 * kNumSMs;
  const double partial_us = (double)T * M * 8.0 / 6e6;
  int best_s = 1;
  double best = -1.0;
  for (int s = 1; s <= kchunks; ++s) {
    const int cps = (kchunks + s - 1) / s;
    if ((kchunks + cps - 1) / cps != s) continue;  // same as a smaller split
    const long waves = ((long)m_tiles * s + slots - 1) / slots;
    const double cost = (double)waves * cps * 1.1 + s * partial_us;
    if (best < 0.0 || cost < best) {
      best = cost;
      best_s = s;
    }
  }
  *chunks_per_split = (kchunks + best_s - 1) / best_s;
  *splits = best_s;
}

void oproj_split(int K, int d_model, int T, int *chunks_per_split, int *splits) {
  choose_split(K / kKChunk, (d_model + kM - 1) / kM, T, d_model, chunks_per_split, splits);
}

}  // namespace

bool tc_oproj_supported(const mla_dims &d, int d_model) {
  return d.dtype == MLA_BF16 && d.d_h == 128 && d_model > 0 && d_model % 2 == 0;
}

size_t oproj_workspace_bytes(int T, int d_model, const mla_dims &d) {
  int cps, splits;
  oproj_split(d.H * d.d_h, d_model, T, &cps, &splits);
  return (size_t)splits * T * d_model * sizeof(float);
}

cudaError_t launch_oproj_tc(const void *out, const void *W_O, void *u, int T, int d_model,
                            const mla_dims &d, void *workspace, cudaStream_t st) {
  const int K = d.H * d.d_h;
  int cps, splits;
  oproj_split(K, d_model, T, &cps, &splits);
  const int Nt = pick_nt(T);
  CUtensorMap tmA, tmB;
  // W_O as [d_model rows][H*d_h], boxes of 64 x 128 rows; out as [T][H*d_h]
  if (!make_tmap_2d_bf16(&tmA, W_O, K, d_model, (uint64_t)K * 2, 64, 128,
                         CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tmap_2d_bf16(&tmB, out, K, T, (uint64_t)K * 2, 64, Nt, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  GemmArgs g;
  g.num_k_chunks = cps;
  g.rows = T;
  g.Nt = Nt;
  g.H = splits;
  g.M_total = d_model;
  g.a_rows_per_head = 0;
  g.a_cols_per_head = cps * kKChunk;
  g.b_cols_per_head = cps * kKChunk;
  g.out = nullptr;
  g.part = static_cast<float *>(workspace);
  g.m_ofs = 0;
  g.a_tiles = 1 << 30;
  cudaError_t e = launch_head_gemm<false>(tmA, tmA, tmB, g, (d_model + kM - 1) / kM, st);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((d_model / 2 + 255) / 256), T, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.stream = st;
  cfg.attrs = pdl;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, splitk_sum_kernel, static_cast<const float *>(workspace),
                            splits, T, d_model, static_cast<__nv_bfloat16 *>(u));
}

// ---- query projections ----

namespace {

// q_nope = bf16(sum of partials) for features < H*d_h; q_rope = the RoPE'd
// rest, head by head (pairs (2j, 2j+1) of each head's d_r, angle
// pos * base^(-2j/d_r)).  Query slot i of sequence b sits at position
// seqlens[b] - Hq + i.  One thread per feature pair.
__global__ void __launch_bounds__(256) qproj_finalize_kernel(
    const float *__restrict__ part, int splits, int T, int Hd, int Hr, int d_r,
    RopeTable rope, const int32_t *__restrict__ seqlens, int Hq,
    __nv_bfloat16 *__restrict__ q_nope, __nv_bfloat16 *__restrict__ q_rope) {
  ptx::grid_dependency_wait();  // the partial sums of the GEMM just before
  const int t = blockIdx.y;
  const int M = Hd + Hr;
  const int j = blockIdx.x * blockDim.x + threadIdx.x;  // feature pair 2j, 2j+1
  if (2 * j >= M) return;
  const float *src = part + (size_t)t * M + 2 * j;
  const size_t split_stride = (size_t)T * M;
  float x0 = 0.f, x1 = 0.f;
  for (int s = 0; s < splits; ++s) {
    const float2 v = *reinterpret_cast<const float2 *>(src + s * split_stride);
    x0 += v.x;
    x1 += v.y;
  }
  __nv_bfloat162 o;
  if (2 * j < Hd) {
    o.x = __float2bfloat16_rn(x0);
    o.y = __float2bfloat16_rn(x1);
    *reinterpret_cast<__nv_bfloat162 *>(q_nope + (size_t)t * Hd + 2 * j) = o;
    return;
  }
  const int f = 2 * j - Hd;               // feature within the RoPE part
  const int p = (f % d_r) / 2;            // pair within the head
  const int b = t / Hq, i = t % Hq;
  const int pos = seqlens[b] - Hq + i;
  float c, sv;
  rope_cos_sin(pos, rope.theta[p], &c, &sv);
  o.x = __float2bfloat16_rn(x0 * c - x1 * sv);
  o.y = __float2bfloat16_rn(x1 * c + x0 * sv);
  *reinterpret_cast<__nv_bfloat162 *>(q_rope + (size_t)t * Hr + f) = o;
}

void qproj_split(int d_model, int m_tiles, int T, int M, int *chunks_per_split, int *splits) {
  choose_split(d_model / kKChunk, m_tiles, T, M, chunks_per_split, splits);
}

int qproj_m_tiles(const mla_dims &d) {
  return (d.H * d.d_h) / kM + (d.H * d.d_r + kM - 1) / kM;
}

}  // namespace

bool tc_qproj_supported(const mla_dims &d, int d_model) {
  return d.dtype == MLA_BF16 && d.d_h == 128 && d.d_r > 0 && d.d_r <= 128 && d.d_r % 2 == 0 &&
         d_model > 0 &&
         d_model % kKChunk == 0;
}

size_t qproj_workspace_bytes(int T, int d_model, const mla_dims &d) {
  int cps, splits;
  qproj_split(d_model, qproj_m_tiles(d), T, d.H * (d.d_h + d.d_r), &cps, &splits);
  return (size_t)splits * T * d.H * (d.d_h + d.d_r) * sizeof(float);
}

cudaError_t launch_qproj_tc(const void *h, const void *W_Q, const void *W_QR, int d_model,
                            double rope_base, const int32_t *seqlens, int B, int Hq,
                            const mla_dims &d, void *q_nope, void *q_rope, void *workspace,
                            cudaStream_t st) {
  const int T = B * Hq, Hd = d.H * d.d_h, Hr = d.H * d.d_r;
  int cps, splits;
  qproj_split(d_model, qproj_m_tiles(d), T, Hd + Hr, &cps, &splits);
  const int Nt = pick_nt(T);
  CUtensorMap tmQ, tmQR, tmH;
  if (!make_tmap_2d_bf16(&tmQ, W_Q, d_model, Hd, (uint64_t)d_model * 2, 64, 128,
                         CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tmap_2d_bf16(&tmQR, W_QR, d_model, Hr, (uint64_t)d_model * 2, 64, 128,
                         CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tmap_2d_bf16(&tmH, h, d_model, T, (uint64_t)d_model * 2, 64, Nt,
                         CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  GemmArgs g;
  g.num_k_chunks = cps;
  g.rows = T;
  g.Nt = Nt;
  g.H = splits;
  g.M_total = Hd + Hr;
  g.a_rows_per_head = 0;
  g.a_cols_per_head = cps * kKChunk;
  g.b_cols_per_head = cps * kKChunk;
  g.out = nullptr;
  g.part = static_cast<float *>(workspace);
  g.m_ofs = 0;
  g.a_tiles = Hd / kM;  // W_Q rows, then W_QR rows
  cudaError_t e = launch_head_gemm<false>(tmQ, tmQR, tmH, g, qproj_m_tiles(d), st);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(((Hd + Hr) / 2 + 255) / 256), T, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.stream = st;
  cfg.attrs = pdl;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, qproj_finalize_kernel, static_cast<const float *>(workspace),
                            splits, T, Hd, Hr, d.d_r, rope_table(rope_base, d.d_r), seqlens, Hq,
                            static_cast<__nv_bfloat16 *>(q_nope),
                            static_cast<__nv_bfloat16 *>(q_rope));
}

}  // namespace mla


