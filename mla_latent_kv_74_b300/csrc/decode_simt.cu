// CUDA-core absorbed MLA decode (any supported shape, fp32 or bf16) and the
// log-sum-exp combine of split-KV partials.
//
// Math ("MLA, dim by dim" 5.2; "From Vanilla Transformers to Modern LLMs --
// Part 3" 3.o-3.p): for one row (sequence b, query slot i, head h)
//   s_j = (q_lat . c_j + q_rope . kR_j) * scale
//   o_lat = sum_j softmax(s)_j c_j,  lse = ln sum_j exp(s_j)
// evaluated with a running maximum (online softmax) in base 2: scores are
// pre-multiplied by log2(e) so every exponential is one exp2f.
//
// Layout of the work: one warp per (row, split).  A lane holds the query
// dimensions lane, lane+32, ... (at most 18 of them for d_c + d_r <= 576);
// per cached token the warp reduces the dot product with shuffles and
// rescales its d_c/32 accumulators.  Each split writes o_part = O/l and
// lse_part = m + ln l; the combine merges splits with weights exp(lse_s - lse).
#include <math.h>

#include "internal.cuh"

namespace mla {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr int kQPerLane = kMaxD / 32;    // 18
constexpr int kAccPerLane = kMaxDc / 32;  // 16
constexpr int kWarps = 4;

struct SimtArgs {
  const void *q_lat, *q_rope, *cache;
  const int32_t *block_table, *seqlens;
  int num_blocks, max_blocks, max_seqlen, Hq, H, d_c, d_r, bs, chunk;
  float scale_log2;  // scale * log2(e)
  float *o_part, *lse_part;
  int *err;
};

template <typename T>
__global__ void __launch_bounds__(kWarps * 32) decode_simt_kernel(SimtArgs a) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.x * kWarps + warp;
  if (h >= a.H) return;
  const int item = blockIdx.y;  // b * Hq + slot
  const int split = blockIdx.z;
  const int b = item / a.Hq, slot = item % a.Hq;
  const int rows = gridDim.y * a.H;
  const int row = item * a.H + h;
  const int D = a.d_c + a.d_r;

  const int seqlen = a.seqlens[b];
  bool bad = seqlen < 0 || seqlen > a.max_seqlen || seqlen > a.max_blocks * a.bs;
  const int n = bad ? 0 : max(0, seqlen - a.Hq + slot + 1);
  const int j0 = split * a.chunk;
  const int j1 = min(n, j0 + a.chunk);

  const T *ql = static_cast<const T *>(a.q_lat) + (size_t)row * a.d_c;
  const T *qr = a.d_r ? static_cast<const T *>(a.q_rope) + (size_t)row * a.d_r : nullptr;
  float q[kQPerLane];
#pragma unroll
  for (int i = 0; i < kQPerLane; ++i) {
    const int dd = lane + 32 * i;
    q[i] = dd < a.d_c ? to_f32(ql[dd]) : (dd < D ? to_f32(qr[dd - a.d_c]) : 0.f);
  }
  float acc[kAccPerLane];
#pragma unroll
  for (int i = 0; i < kAccPerLane; ++i) acc[i] = 0.f;
  float m = -INFINITY, l = 0.f;

  const T *cache = static_cast<const T *>(a.cache);
  for (int j = j0; j < j1; ++j) {
    const int blk = a.block_table[(size_t)b * a.max_blocks + j / a.bs];
    if (blk < 0 || blk >= a.num_blocks) {
      bad = true;
      break;
    }
    const T *r = cache + ((size_t)blk * a.bs + j % a.bs) * D;
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < kQPerLane; ++i) {
      const int dd = lane + 32 * i;
      if (dd < D) s = fmaf(q[i], to_f32(r[dd]), s);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    s *= a.scale_log2;
    const float m_new = fmaxf(m, s);
    const float alpha = exp2f(m - m_new);  // 0 on the first token (m = -inf)
    const float p = exp2f(s - m_new);
    l = fmaf(l, alpha, p);
#pragma unroll
    for (int i = 0; i < kAccPerLane; ++i) {
      const int dd = lane + 32 * i;
      if (dd < a.d_c) acc[i] = fmaf(acc[i], alpha, p * to_f32(r[dd]));
    }
    m = m_new;
  }

  float *op = a.o_part + ((size_t)split * rows + row) * a.d_c;
  if (bad) {
    set_device_error(a.err, kDevBounds);
    // NaN marks the row as poisoned; the combine writes it as 0 / -inf.
    if (lane == 0) a.lse_part[(size_t)split * rows + row] = __int_as_float(0x7fc00000);
#pragma unroll
    for (int i = 0; i < kAccPerLane; ++i) {
      const int dd = lane + 32 * i;
      if (dd < a.d_c) op[dd] = 0.f;
    }
    return;
  }
  const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
  for (int i = 0; i < kAccPerLane; ++i) {
    const int dd = lane + 32 * i;
    if (dd < a.d_c) op[dd] = acc[i] * inv;
  }
  if (lane == 0)
    a.lse_part[(size_t)split * rows + row] = l > 0.f ? (m + log2f(l)) * kLn2 : -INFINITY;
}

template <typename T>
__global__ void __launch_bounds__(128) combine_kernel(const float *__restrict__ o_part,
                                                      const float *__restrict__ lse_part,
                                                      int nsplit, int rows, int d_c,
                                                      T *__restrict__ o_lat,
                                                      float *__restrict__ lse) {
  const int row = blockIdx.x;
  __shared__ float w_s[256];
  __shared__ float s_lse;
  __shared__ int s_state;  // 0 normal, 1 empty, 2 poisoned
  if (threadIdx.x == 0) {
    float mx = -INFINITY;
    bool poison = false;
    for (int s = 0; s < nsplit; ++s) {
      const float v = lse_part[(size_t)s * rows + row];
      if (isnan(v)) poison = true;
      mx = fmaxf(mx, v);
    }
    if (poison) {
      s_state = 2;
    } else if (mx == -INFINITY) {
      s_state = 1;
    } else {
      float sum = 0.f;
      for (int s = 0; s < nsplit; ++s) sum += expf(lse_part[(size_t)s * rows + row] - mx);
      const float inv = 1.f / sum;
      for (int s = 0; s < nsplit; ++s)
        w_s[s] = expf(lse_part[(size_t)s * rows + row] - mx) * inv;
      s_lse = mx + logf(sum);
      s_state = 0;
    }
  }
  __syncthreads();
  const int st = s_state;
  for (int dd = threadIdx.x; dd < d_c; dd += blockDim.x) {
    float o = 0.f;
    if (st == 0)
      for (int s = 0; s < nsplit; ++s) o = fmaf(w_s[s], o_part[((size_t)s * rows + row) * d_c + dd], o);
    o_lat[(size_t)row * d_c + dd] = from_f32<T>(o);
  }
  if (threadIdx.x == 0) lse[row] = st == 0 ? s_lse : -INFINITY;
}

}  // namespace

SimtPlan simt_plan(int B, int Hq, int max_seqlen, const mla_dims &d) {
  SimtPlan p;
  const long ctas = (long)((d.H + kWarps - 1) / kWarps) * B * Hq;
  const long target = 4L * kNumSMs * 4;  // ~4 waves of 4-warp CTAs
  int ns = ctas > 0 ? (int)((target + ctas - 1) / ctas) : 1;
  const int max_ns = max(1, (max_seqlen + 255) / 256);  // >= 256 tokens per split
  ns = max(1, min(ns, min(max_ns, 256)));
  p.nsplit = ns;
  p.chunk = max(1, (max_seqlen + ns - 1) / ns);
  return p;
}

size_t simt_workspace_bytes(int B, int Hq, int max_seqlen, const mla_dims &d) {
  const SimtPlan p = simt_plan(B, Hq, max_seqlen, d);
  const size_t rows = (size_t)B * Hq * d.H;
  return kWsHeader + align_up(p.nsplit * rows * d.d_c * sizeof(float), 256) +
         align_up(p.nsplit * rows * sizeof(float), 256);
}

cudaError_t launch_combine(const float *o_part, const float *lse_part, int nsplit, int rows,
                           int d_c, mla_dtype dtype, void *o_lat, float *lse,
                           cudaStream_t st) {
  if (rows == 0) return cudaSuccess;
  if (dtype == MLA_BF16)
    combine_kernel<__nv_bfloat16><<<rows, 128, 0, st>>>(o_part, lse_part, nsplit, rows, d_c,
                                                        (__nv_bfloat16 *)o_lat, lse);
  else
    combine_kernel<float><<<rows, 128, 0, st>>>(o_part, lse_part, nsplit, rows, d_c,
                                                (float *)o_lat, lse);
  return cudaGetLastError();
}

cudaError_t launch_decode_simt(const void *q_lat, const void *q_rope, const void *cache,
                               int num_blocks, const int32_t *block_table, int max_blocks,
                               const int32_t *seqlens, int max_seqlen, int B, int Hq,
                               const mla_dims &d, float scale, void *o_lat, float *lse,
                               void *workspace, cudaStream_t st) {
  const int rows = B * Hq * d.H;
  if (rows == 0) return cudaSuccess;
  const SimtPlan p = simt_plan(B, Hq, max_seqlen, d);
  char *ws = static_cast<char *>(workspace);
  SimtArgs a;
  a.q_lat = q_lat;
  a.q_rope = q_rope;
  a.cache = cache;
  a.block_table = block_table;
  a.seqlens = seqlens;
  a.num_blocks = num_blocks;
  a.max_blocks = max_blocks;
  a.max_seqlen = max_seqlen;
  a.Hq = Hq;
  a.H = d.H;
  a.d_c = d.d_c;
  a.d_r = d.d_r;
  a.bs = d.block_size;
  a.chunk = p.chunk;
  a.scale_log2 = scale * kLog2e;
  a.err = reinterpret_cast<int *>(ws);
  a.o_part = reinterpret_cast<float *>(ws + kWsHeader);
  a.lse_part = reinterpret_cast<float *>(
      ws + kWsHeader + align_up((size_t)p.nsplit * rows * d.d_c * sizeof(float), 256));
  dim3 grid((d.H + kWarps - 1) / kWarps, B * Hq, p.nsplit);
  if (d.dtype == MLA_BF16)
    decode_simt_kernel<__nv_bfloat16><<<grid, kWarps * 32, 0, st>>>(a);
  else
    decode_simt_kernel<float><<<grid, kWarps * 32, 0, st>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_combine(a.o_part, a.lse_part, p.nsplit, rows, d.d_c, d.dtype, o_lat, lse, st);
}

}  // namespace mla
