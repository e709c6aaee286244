// mla_append_cache: scatter the newest tokens' [c_KV ; k_R] rows into the
// paged latent cache ("MLA Explained", decode step 5; "From Vanilla
// Transformers to Modern LLMs -- Part 3" 3.q -- k_R is cached already
// rotated, next to the latent).
//
// One CTA per (new token, sequence).  The row is d_c + d_r elements; when
// both halves are 16-byte multiples (bf16 d_c=512, d_r=64: 1024 + 128 bytes)
// the copy moves 16-byte vectors, otherwise scalars.
#include "internal.cuh"

namespace mla {
namespace {

template <typename T>
__global__ void __launch_bounds__(128) append_kernel(T *__restrict__ cache, int num_blocks,
                                                     const int32_t *__restrict__ block_table,
                                                     int max_blocks,
                                                     const int32_t *__restrict__ seqlens,
                                                     const T *__restrict__ c_kv,
                                                     const T *__restrict__ k_r, int n_new,
                                                     int d_c, int d_r, int bs, bool vec) {
  // the next kernel of the step may launch now: it waits for this grid's
  // completion before it reads anything this grid writes
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int i = blockIdx.x;  // new-token index
  const int b = blockIdx.y;
  const int pos = seqlens[b] - n_new + i;
  if (pos < 0) return;
  const int lb = pos / bs;
  if (lb >= max_blocks) return;
  const int blk = block_table[(size_t)b * max_blocks + lb];
  if (blk < 0 || blk >= num_blocks) return;  // reported by mla_decode
  const int D = d_c + d_r;
  T *dst = cache + ((size_t)blk * bs + pos % bs) * D;
  const T *src_c = c_kv + ((size_t)b * n_new + i) * d_c;
  const T *src_r = k_r ? k_r + ((size_t)b * n_new + i) * d_r : nullptr;
  if (vec) {
    constexpr int kPer = 16 / sizeof(T);
    const int nc = d_c / kPer, nr = d_r / kPer;
    for (int v = threadIdx.x; v < nc + nr; v += blockDim.x) {
      const uint4 x = v < nc ? reinterpret_cast<const uint4 *>(src_c)[v]
                             : reinterpret_cast<const uint4 *>(src_r)[v - nc];
      reinterpret_cast<uint4 *>(dst)[v] = x;
    }
  } else {
    for (int e = threadIdx.x; e < D; e += blockDim.x)
      dst[e] = e < d_c ? src_c[e] : src_r[e - d_c];
  }
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

}  // namespace

cudaError_t launch_append(void *cache, int num_blocks, const int32_t *block_table,
                          int max_blocks, const int32_t *seqlens, const void *c_kv,
                          const void *k_r, int B, int n_new, const mla_dims &d,
                          cudaStream_t st) {
  if (B == 0 || n_new == 0) return cudaSuccess;
  dim3 grid(n_new, B);
  const size_t es = elem_size(d.dtype);
  const bool vec = (d.d_c * es) % 16 == 0 && (d.d_r * es) % 16 == 0 && aligned16(cache) &&
                   aligned16(c_kv) && (d.d_r == 0 || aligned16(k_r)) &&
                   ((d.d_c + d.d_r) * es) % 16 == 0;
  if (d.dtype == MLA_BF16)
    append_kernel<__nv_bfloat16><<<grid, 128, 0, st>>>(
        (__nv_bfloat16 *)cache, num_blocks, block_table, max_blocks, seqlens,
        (const __nv_bfloat16 *)c_kv, (const __nv_bfloat16 *)k_r, n_new, d.d_c, d.d_r,
        d.block_size, vec);
  else
    append_kernel<float><<<grid, 128, 0, st>>>((float *)cache, num_blocks, block_table,
                                               max_blocks, seqlens, (const float *)c_kv,
                                               (const float *)k_r, n_new, d.d_c, d.d_r,
                                               d.block_size, vec);
  return cudaGetLastError();
}

}  // namespace mla
