// Internal declarations shared by the library's translation units.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/mla.h"

namespace mla {

constexpr int kMaxD = 576;    // d_c + d_r limit of the CUDA-core decode
constexpr int kMaxDc = 512;   // d_c limit
constexpr int kMaxDr = 64;    // d_r limit
constexpr int kMaxDh = 128;   // d_h limit
constexpr int kMaxH = 256;    // head limit
constexpr int kNumSMs = 148;  // B300
// B * Hq limit of mla_decode: the CUDA-core kernel's grid has one y index
// per (sequence, query slot) item
constexpr long kMaxDecodeItems = 65535;

// Device error word values (the first int of the decode workspace).
constexpr int kDevOk = 0;
constexpr int kDevBounds = 1;
constexpr int kDevTimeout = 2;

// Workspace header: error word plus padding to 256 bytes.
constexpr size_t kWsHeader = 256;

__host__ __device__ inline size_t align_up(size_t x, size_t a) {
  return (x + a - 1) / a * a;
}

template <typename T> __device__ __forceinline__ float to_f32(T x);
template <> __device__ __forceinline__ float to_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) {
  return __bfloat162float(x);
}
template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

__device__ __forceinline__ void set_device_error(int *err, int code) {
  if (err) atomicCAS(err, kDevOk, code);
}

inline size_t elem_size(mla_dtype t) { return t == MLA_BF16 ? 2 : 4; }

// ---- launchers (each returns cudaGetLastError() of its launch) ----------

cudaError_t launch_append(void *cache, int num_blocks, const int32_t *block_table,
                          int max_blocks, const int32_t *seqlens, const void *c_kv,
                          const void *k_r, int B, int n_new, const mla_dims &d,
                          cudaStream_t st);

// CUDA-core split-KV decode: writes partials, then the combine merges them.
struct SimtPlan {
  int nsplit;
  int chunk;  // tokens per split
};
SimtPlan simt_plan(int B, int Hq, int max_seqlen, const mla_dims &d);
size_t simt_workspace_bytes(int B, int Hq, int max_seqlen, const mla_dims &d);
cudaError_t launch_decode_simt(const void *q_lat, const void *q_rope, const void *cache,
                               int num_blocks, const int32_t *block_table, int max_blocks,
                               const int32_t *seqlens, int max_seqlen, int B, int Hq,
                               const mla_dims &d, float scale, void *o_lat, float *lse,
                               void *workspace, cudaStream_t st);

cudaError_t launch_absorb_simt(const void *q_nope, const void *W_UK, void *q_lat, int rows,
                               const mla_dims &d, cudaStream_t st);
cudaError_t launch_out_proj_simt(const void *o_lat, const void *W_UV, void *out, int rows,
                                 const mla_dims &d, cudaStream_t st);

// LSE combine of split partials: o_part [nsplit, rows, d_c] fp32,
// lse_part [nsplit, rows] fp32 -> o_lat [rows, d_c] (dtype), lse [rows].
cudaError_t launch_combine(const float *o_part, const float *lse_part, int nsplit, int rows,
                           int d_c, mla_dtype dtype, void *o_lat, float *lse,
                           cudaStream_t st);

}  // namespace mla
