// CUDA-core per-head batched GEMMs for shapes outside the tensor-core path.
//
//   absorb:   q_lat[r,h,c] = sum_a q_nope[r,h,a] * W_UK[h,a,c]
//             ("From Vanilla Transformers to Modern LLMs -- Part 3" 3.e.2)
//   out_proj: out[r,h,a]   = sum_c W_UV[h,a,c] * o_lat[r,h,c]
//             ("From Vanilla Transformers to Modern LLMs -- Part 3" 3.g)
//
// r runs over the B*Hq query rows.  fp32 accumulation, rounded to the
// tensor dtype on store.
#include "internal.cuh"

namespace mla {
namespace {

constexpr int kRowsPerCta = 16;

// grid (ceil(d_c/128), H, ceil(rows/16)); thread = one latent column c.
template <typename T>
__global__ void __launch_bounds__(128) absorb_simt_kernel(const T *__restrict__ q_nope,
                                                          const T *__restrict__ W_UK,
                                                          T *__restrict__ q_lat, int rows,
                                                          int H, int d_h, int d_c) {
  __shared__ float qs[kRowsPerCta][kMaxDh];
  const int h = blockIdx.y;
  const int r0 = blockIdx.z * kRowsPerCta;
  const int nr = min(kRowsPerCta, rows - r0);
  for (int e = threadIdx.x; e < nr * d_h; e += blockDim.x) {
    const int r = e / d_h, a = e % d_h;
    qs[r][a] = to_f32(q_nope[((size_t)(r0 + r) * H + h) * d_h + a]);
  }
  __syncthreads();
  const int c = blockIdx.x * 128 + threadIdx.x;
  if (c >= d_c) return;
  float acc[kRowsPerCta];
#pragma unroll
  for (int r = 0; r < kRowsPerCta; ++r) acc[r] = 0.f;
  const T *w = W_UK + (size_t)h * d_h * d_c + c;
  for (int a = 0; a < d_h; ++a) {
    const float wv = to_f32(w[(size_t)a * d_c]);
#pragma unroll
    for (int r = 0; r < kRowsPerCta; ++r) acc[r] = fmaf(qs[r][a], wv, acc[r]);
  }
  for (int r = 0; r < nr; ++r) q_lat[((size_t)(r0 + r) * H + h) * d_c + c] = from_f32<T>(acc[r]);
}

// grid (H, ceil(rows/16)); 4 warps; warp w computes outputs a = w, w+4, ...
// with lanes striding the latent axis, then reduces with shuffles.
template <typename T>
__global__ void __launch_bounds__(128) out_proj_simt_kernel(const T *__restrict__ o_lat,
                                                            const T *__restrict__ W_UV,
                                                            T *__restrict__ out, int rows,
                                                            int H, int d_h, int d_c) {
  __shared__ float os[kRowsPerCta][kMaxDc];
  const int h = blockIdx.x;
  const int r0 = blockIdx.y * kRowsPerCta;
  const int nr = min(kRowsPerCta, rows - r0);
  for (int e = threadIdx.x; e < kRowsPerCta * d_c; e += blockDim.x) {
    const int r = e / d_c, c = e % d_c;
    os[r][c] = r < nr ? to_f32(o_lat[((size_t)(r0 + r) * H + h) * d_c + c]) : 0.f;
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int a = warp; a < d_h; a += 4) {
    const T *w = W_UV + ((size_t)h * d_h + a) * d_c;
    float acc[kRowsPerCta];
#pragma unroll
    for (int r = 0; r < kRowsPerCta; ++r) acc[r] = 0.f;
    for (int c = lane; c < d_c; c += 32) {
      const float wv = to_f32(w[c]);
#pragma unroll
      for (int r = 0; r < kRowsPerCta; ++r) acc[r] = fmaf(wv, os[r][c], acc[r]);
    }
#pragma unroll
    for (int r = 0; r < kRowsPerCta; ++r) {
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) acc[r] += __shfl_xor_sync(0xffffffffu, acc[r], off);
    }
    if (lane < nr) {
      float v = 0.f;
#pragma unroll
      for (int r = 0; r < kRowsPerCta; ++r)
        if (r == lane) v = acc[r];
      out[((size_t)(r0 + lane) * H + h) * d_h + a] = from_f32<T>(v);
    }
  }
}

}  // namespace

cudaError_t launch_absorb_simt(const void *q_nope, const void *W_UK, void *q_lat, int rows,
                               const mla_dims &d, cudaStream_t st) {
  if (rows == 0) return cudaSuccess;
  dim3 grid((d.d_c + 127) / 128, d.H, (rows + kRowsPerCta - 1) / kRowsPerCta);
  if (d.dtype == MLA_BF16)
    absorb_simt_kernel<__nv_bfloat16><<<grid, 128, 0, st>>>(
        (const __nv_bfloat16 *)q_nope, (const __nv_bfloat16 *)W_UK, (__nv_bfloat16 *)q_lat,
        rows, d.H, d.d_h, d.d_c);
  else
    absorb_simt_kernel<float><<<grid, 128, 0, st>>>((const float *)q_nope, (const float *)W_UK,
                                                    (float *)q_lat, rows, d.H, d.d_h, d.d_c);
  return cudaGetLastError();
}

cudaError_t launch_out_proj_simt(const void *o_lat, const void *W_UV, void *out, int rows,
                                 const mla_dims &d, cudaStream_t st) {
  if (rows == 0) return cudaSuccess;
  dim3 grid(d.H, (rows + kRowsPerCta - 1) / kRowsPerCta);
  if (d.dtype == MLA_BF16)
    out_proj_simt_kernel<__nv_bfloat16><<<grid, 128, 0, st>>>(
        (const __nv_bfloat16 *)o_lat, (const __nv_bfloat16 *)W_UV, (__nv_bfloat16 *)out, rows,
        d.H, d.d_h, d.d_c);
  else
    out_proj_simt_kernel<float><<<grid, 128, 0, st>>>((const float *)o_lat, (const float *)W_UV,
                                                      (float *)out, rows, d.H, d.d_h, d.d_c);
  return cudaGetLastError();
}

}  // namespace mla
