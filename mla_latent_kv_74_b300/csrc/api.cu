// C-ABI entry points: host-side validation, path selection and launches.
// Every entry point checks its arguments before launching anything; the
// device kernels never allocate and never synchronise.
#include <math.h>

#include <climits>

#include "internal.cuh"
#include "tc.cuh"

#define MLA_API extern "C" __attribute__((visibility("default")))

namespace mla {
namespace {

bool dims_ok(const mla_dims *d) {
  if (!d) return false;
  if (d->dtype != MLA_BF16 && d->dtype != MLA_FP32) return false;
  return d->H >= 1 && d->H <= kMaxH && d->d_h >= 1 && d->d_h <= kMaxDh && d->d_c >= 1 &&
         d->d_c <= kMaxDc && d->d_r >= 0 && d->d_r <= kMaxDr && d->block_size >= 1 &&
         d->block_size <= 1024 && isfinite(d->scale);
}

bool al(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

float eff_scale(const mla_dims *d) {
  return d->scale > 0.f ? d->scale : 1.0f / sqrtf((float)(d->d_h + d->d_r));
}

mla_status cuda_status(cudaError_t e) { return e == cudaSuccess ? MLA_OK : MLA_ERR_CUDA; }

}  // namespace
}  // namespace mla

using namespace mla;

MLA_API const char *mla_status_string(mla_status s) {
  switch (s) {
    case MLA_OK: return "MLA_OK";
    case MLA_ERR_INVALID_ARG: return "MLA_ERR_INVALID_ARG: bad pointer, alignment or size";
    case MLA_ERR_UNSUPPORTED: return "MLA_ERR_UNSUPPORTED: dims or dtype not supported";
    case MLA_ERR_WORKSPACE: return "MLA_ERR_WORKSPACE: workspace missing or too small";
    case MLA_ERR_CUDA: return "MLA_ERR_CUDA: a CUDA call or kernel launch failed";
    case MLA_ERR_DEVICE_BOUNDS: return "MLA_ERR_DEVICE_BOUNDS: block index or length out of range";
    case MLA_ERR_TIMEOUT: return "MLA_ERR_TIMEOUT: a bounded device wait gave up";
  }
  return "unknown mla_status";
}

MLA_API mla_status mla_absorb_query(const void *q_nope, const void *W_UK, void *q_lat, int B,
                                    int Hq, const mla_dims *dims, mla_stream_t stream) {
  if (!dims_ok(dims)) return dims ? MLA_ERR_UNSUPPORTED : MLA_ERR_INVALID_ARG;
  if (B < 0 || Hq < 1) return MLA_ERR_INVALID_ARG;
  if (B == 0) return MLA_OK;
  if (!q_nope || !W_UK || !q_lat || !al(q_nope, 16) || !al(W_UK, 16) || !al(q_lat, 16))
    return MLA_ERR_INVALID_ARG;
  const int rows = B * Hq;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (tc_gemm_supported(*dims))
    return cuda_status(launch_absorb_tc(q_nope, W_UK, q_lat, rows, *dims, st));
  return cuda_status(launch_absorb_simt(q_nope, W_UK, q_lat, rows, *dims, st));
}

MLA_API mla_status mla_out_proj(const void *o_lat, const void *W_UV, void *out, int B, int Hq,
                                const mla_dims *dims, mla_stream_t stream) {
  if (!dims_ok(dims)) return dims ? MLA_ERR_UNSUPPORTED : MLA_ERR_INVALID_ARG;
  if (B < 0 || Hq < 1) return MLA_ERR_INVALID_ARG;
  if (B == 0) return MLA_OK;
  if (!o_lat || !W_UV || !out || !al(o_lat, 16) || !al(W_UV, 16) || !al(out, 16))
    return MLA_ERR_INVALID_ARG;
  const int rows = B * Hq;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (tc_gemm_supported(*dims))
    return cuda_status(launch_out_proj_tc(o_lat, W_UV, out, rows, *dims, st));
  return cuda_status(launch_out_proj_simt(o_lat, W_UV, out, rows, *dims, st));
}

MLA_API mla_status mla_append_cache(void *cache, int num_blocks, const int32_t *block_table,
                                    int max_blocks, const int32_t *seqlens, const void *c_kv,
                                    const void *k_r, int B, int n_new, const mla_dims *dims,
                                    mla_stream_t stream) {
  if (!dims_ok(dims)) return dims ? MLA_ERR_UNSUPPORTED : MLA_ERR_INVALID_ARG;
  if (B < 0 || n_new < 0 || num_blocks < 1 || max_blocks < 1) return MLA_ERR_INVALID_ARG;
  if (B == 0 || n_new == 0) return MLA_OK;
  if (!cache || !block_table || !seqlens || !c_kv || (dims->d_r > 0 && !k_r))
    return MLA_ERR_INVALID_ARG;
  if (!al(cache, 16) || !al(block_table, 4) || !al(seqlens, 4) || !al(c_kv, 16) ||
      (k_r && !al(k_r, 16)))
    return MLA_ERR_INVALID_ARG;
  return cuda_status(launch_append(cache, num_blocks, block_table, max_blocks, seqlens, c_kv,
                                   k_r, B, n_new, *dims,
                                   reinterpret_cast<cudaStream_t>(stream)));
}

MLA_API mla_status mla_project_append_workspace_size(int B, int n_new, int d_model,
                                                     const mla_dims *dims, size_t *bytes) {
  if (!bytes) return MLA_ERR_INVALID_ARG;
  if (!dims_ok(dims)) return dims ? MLA_ERR_UNSUPPORTED : MLA_ERR_INVALID_ARG;
  if (B < 0 || n_new < 0 || d_model < 1) return MLA_ERR_INVALID_ARG;
  if (!tc_project_supported(*dims, d_model)) return MLA_ERR_UNSUPPORTED;
  *bytes = project_workspace_bytes(B * n_new, d_model, *dims);
  return MLA_OK;
}

MLA_API mla_status mla_project_append(const void *h, const void *W_DKV, const void *W_KR,
                                      int d_model, float rope_base, void *cache, int num_blocks,
                                      const int32_t *block_table, int max_blocks,
                                      const int32_t *seqlens, int B, int n_new,
                                      const mla_dims *dims, void *workspace,
                                      size_t workspace_bytes, mla_stream_t stream) {
  if (!dims_ok(dims)) return dims ? MLA_ERR_UNSUPPORTED : MLA_ERR_INVALID_ARG;
  if (B < 0 || n_new < 0 || d_model < 1 || num_blocks < 1 || max_blocks < 1 ||
      !(rope_base > 0.f))
    return MLA_ERR_INVALID_ARG;
  if (!tc_project_supported(*dims, d_model)) return MLA_ERR_UNSUPPORTED;
  if (B == 0 || n_new == 0) return MLA_OK;
  if (!h || !W_DKV || !W_KR || !cache || !block_table || !seqlens) return MLA_ERR_INVALID_ARG;
  if (!al(h, 16) || !al(W_DKV, 16) || !al(W_KR, 16) || !al(cache, 16) || !al(block_table, 4) ||
      !al(seqlens, 4))
    return MLA_ERR_INVALID_ARG;
  if (!workspace || !al(workspace, 256) ||
      workspace_bytes < project_workspace_bytes(B * n_new, d_model, *dims))
    return MLA_ERR_WORKSPACE;
  return cuda_status(launch_project_append_tc(
      h, W_DKV, W_KR, d_model, (double)rope_base, cache, num_blocks, block_table, max_blocks,
      seqlens, B, n_new, *dims, workspace, reinterpret_cast<cudaStream_t>(stream)));
}

MLA_API mla_status mla_o_proj_workspace_size(int B, int Hq, int d_model, const mla_dims *dims,
                                             size_t *bytes) {
  if (!bytes) return MLA_ERR_INVALID_ARG;
  if (!dims_ok(dims)) return dims ? MLA_ERR_UNSUPPORTED : MLA_ERR_INVALID_ARG;
  if (B < 0 || Hq < 1 || d_model < 1) return MLA_ERR_INVALID_ARG;
  if (!tc_oproj_supported(*dims, d_model)) return MLA_ERR_UNSUPPORTED;
  *bytes = oproj_workspace_bytes(B * Hq, d_model, *dims);
  return MLA_OK;
}

MLA_API mla_status mla_o_proj(const void *out, const void *W_O, void *u, int B, int Hq,
                              int d_model, const mla_dims *dims, void *workspace,
                              size_t workspace_bytes, mla_stream_t stream) {
  if (!dims_ok(dims)) return dims ? MLA_ERR_UNSUPPORTED : MLA_ERR_INVALID_ARG;
  if (B < 0 || Hq < 1 || d_model < 1) return MLA_ERR_INVALID_ARG;
  if (!tc_oproj_supported(*dims, d_model)) return MLA_ERR_UNSUPPORTED;
  if (B == 0) return MLA_OK;
  if (!out || !W_O || !u || !al(out, 16) || !al(W_O, 16) || !al(u, 16))
    return MLA_ERR_INVALID_ARG;
  if (!workspace || !al(workspace, 256) ||
      workspace_bytes < oproj_workspace_bytes(B * Hq, d_model, *dims))
    return MLA_ERR_WORKSPACE;
  return cuda_status(launch_oproj_tc(out, W_O, u, B * Hq, d_model, *dims, workspace,
                                     reinterpret_cast<cudaStream_t>(stream)));
}

MLA_API mla_status mla_project_query_workspace_size(int B, int Hq, int d_model,
                                                    const mla_dims *dims, size_t *bytes) {
  if (!bytes) return MLA_ERR_INVALID_ARG;
  if (!dims_ok(dims)) return dims ? MLA_ERR_UNSUPPORTED : MLA_ERR_INVALID_ARG;
  if (B < 0 || Hq < 1 || d_model < 1) return MLA_ERR_INVALID_ARG;
  if (!tc_qproj_supported(*dims, d_model)) return MLA_ERR_UNSUPPORTED;
  *bytes = qproj_workspace_bytes(B * Hq, d_model, *dims);
  return MLA_OK;
}

MLA_API mla_status mla_project_query(const void *h, const void *W_Q, const void *W_QR,
                                     int d_model, float rope_base, const int32_t *seqlens, int B,
                                     int Hq, const mla_dims *dims, void *q_nope, void *q_rope,
                                     void *workspace, size_t workspace_bytes,
                                     mla_stream_t stream) {
  if (!dims_ok(dims)) return dims ? MLA_ERR_UNSUPPORTED : MLA_ERR_INVALID_ARG;
  if (B < 0 || Hq < 1 || d_model < 1 || !(rope_base > 0.f)) return MLA_ERR_INVALID_ARG;
  if (!tc_qproj_supported(*dims, d_model)) return MLA_ERR_UNSUPPORTED;
  if (B == 0) return MLA_OK;
  if (!h || !W_Q || !W_QR || !seqlens || !q_nope || !q_rope) return MLA_ERR_INVALID_ARG;
  if (!al(h, 16) || !al(W_Q, 16) || !al(W_QR, 16) || !al(seqlens, 4) || !al(q_nope, 16) ||
      !al(q_rope, 16))
    return MLA_ERR_INVALID_ARG;
  if (!workspace || !al(workspace, 256) ||
      workspace_bytes < qproj_workspace_bytes(B * Hq, d_model, *dims))
    return MLA_ERR_WORKSPACE;
  return cuda_status(launch_qproj_tc(h, W_Q, W_QR, d_model, (double)rope_base, seqlens, B, Hq,
                                     *dims, q_nope, q_rope, workspace,
                                     reinterpret_cast<cudaStream_t>(stream)));
}

MLA_API mla_status mla_decode_workspace_size(int B, int Hq, int max_seqlen, const mla_dims *dims,
                                             size_t *bytes) {
  if (!bytes) return MLA_ERR_INVALID_ARG;
  if (!dims_ok(dims)) return dims ? MLA_ERR_UNSUPPORTED : MLA_ERR_INVALID_ARG;
  if (B < 0 || Hq < 1 || max_seqlen < 0) return MLA_ERR_INVALID_ARG;
  if ((long)B * Hq > kMaxDecodeItems) return MLA_ERR_UNSUPPORTED;
  // only the path mla_decode takes for this problem
  *bytes = tc_decode_supported(*dims, B, Hq) ? tc_decode_workspace_bytes(B, Hq, *dims)
                                              : simt_workspace_bytes(B, Hq, max_seqlen, *dims);
  return MLA_OK;
}

namespace {

// mla_decode and mla_decode_blocks: the same checks, then one launch.
mla_status decode_call(const void *q_lat, const void *q_rope, const void *cache, int num_blocks,
                       const int32_t *block_table, int max_blocks, const int32_t *seqlens,
                       int max_seqlen, int B, int Hq, int first_block, int end_block,
                       bool ranged, const mla_dims *dims, void *o_lat, float *lse,
                       void *workspace, size_t workspace_bytes, mla_stream_t stream) {
  if (!dims_ok(dims)) return dims ? MLA_ERR_UNSUPPORTED : MLA_ERR_INVALID_ARG;
  if (B < 0 || Hq < 1 || max_seqlen < 0 || num_blocks < 1 || max_blocks < 1 ||
      first_block < 0 || end_block < first_block)
    return MLA_ERR_INVALID_ARG;
  if ((long)B * Hq > kMaxDecodeItems) return MLA_ERR_UNSUPPORTED;
  if (ranged && !tc_decode_supported(*dims, B, Hq)) return MLA_ERR_UNSUPPORTED;
  if (B == 0) return MLA_OK;
  if (!q_lat || !cache || !block_table || !seqlens || !o_lat || !lse ||
      (dims->d_r > 0 && !q_rope))
    return MLA_ERR_INVALID_ARG;
  if (!al(q_lat, 16) || (q_rope && !al(q_rope, 16)) || !al(cache, 128) || !al(o_lat, 16) ||
      !al(lse, 4) || !al(block_table, 4) || !al(seqlens, 4))
    return MLA_ERR_INVALID_ARG;
  if (!workspace || !al(workspace, 256)) return MLA_ERR_WORKSPACE;
  size_t need = 0;
  mla_decode_workspace_size(B, Hq, max_seqlen, dims, &need);
  if (workspace_bytes < need) return MLA_ERR_WORKSPACE;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const float scale = eff_scale(dims);
  if (tc_decode_supported(*dims, B, Hq))
    return cuda_status(launch_decode_tc(q_lat, q_rope, cache, num_blocks, block_table,
                                        max_blocks, seqlens, max_seqlen, B, Hq, first_block,
                                        end_block, *dims, scale, o_lat, lse, workspace, st));
  return cuda_status(launch_decode_simt(q_lat, q_rope, cache, num_blocks, block_table,
                                        max_blocks, seqlens, max_seqlen, B, Hq, *dims, scale,
                                        o_lat, lse, workspace, st));
}

}  // namespace

MLA_API mla_status mla_decode(const void *q_lat, const void *q_rope, const void *cache,
                              int num_blocks, const int32_t *block_table, int max_blocks,
                              const int32_t *seqlens, int max_seqlen, int B, int Hq,
                              const mla_dims *dims, void *o_lat, float *lse, void *workspace,
                              size_t workspace_bytes, mla_stream_t stream) {
  return decode_call(q_lat, q_rope, cache, num_blocks, block_table, max_blocks, seqlens,
                     max_seqlen, B, Hq, 0, INT_MAX, false, dims, o_lat, lse, workspace,
                     workspace_bytes, stream);
}

MLA_API mla_status mla_decode_blocks(const void *q_lat, const void *q_rope, const void *cache,
                                     int num_blocks, const int32_t *block_table, int max_blocks,
                                     const int32_t *seqlens, int max_seqlen, int B, int Hq,
                                     int first_block, int end_block, const mla_dims *dims,
                                     void *o_lat, float *lse, void *workspace,
                                     size_t workspace_bytes, mla_stream_t stream) {
  return decode_call(q_lat, q_rope, cache, num_blocks, block_table, max_blocks, seqlens,
                     max_seqlen, B, Hq, first_block, end_block, true, dims, o_lat, lse,
                     workspace, workspace_bytes, stream);
}

MLA_API mla_status mla_combine_pieces(const void *o_pieces, const float *lse_pieces, int P,
                                      int B, int Hq, const mla_dims *dims, void *o_lat,
                                      float *lse, mla_stream_t stream) {
  if (!dims_ok(dims)) return dims ? MLA_ERR_UNSUPPORTED : MLA_ERR_INVALID_ARG;
  if (P < 1 || B < 0 || Hq < 1) return MLA_ERR_INVALID_ARG;
  if ((long)B * Hq > kMaxDecodeItems || !tc_decode_supported(*dims, B, Hq))
    return MLA_ERR_UNSUPPORTED;
  if (B == 0) return MLA_OK;
  if (!o_pieces || !lse_pieces || !o_lat || !lse || !al(o_pieces, 16) || !al(lse_pieces, 4) ||
      !al(o_lat, 16) || !al(lse, 4))
    return MLA_ERR_INVALID_ARG;
  const long rows = (long)B * Hq * dims->H;
  return cuda_status(launch_combine_pieces_tc(o_pieces, lse_pieces, P, rows, o_lat, lse,
                                              reinterpret_cast<cudaStream_t>(stream)));
}

MLA_API mla_status mla_prefill_workspace_size(int total_tokens, const mla_dims *dims,
                                              size_t *bytes) {
  if (!bytes) return MLA_ERR_INVALID_ARG;
  if (!dims_ok(dims)) return dims ? MLA_ERR_UNSUPPORTED : MLA_ERR_INVALID_ARG;
  if (total_tokens < 0) return MLA_ERR_INVALID_ARG;
  if (!tc_prefill_supported(*dims)) return MLA_ERR_UNSUPPORTED;
  *bytes = prefill_workspace_bytes(total_tokens, *dims);
  return MLA_OK;
}

MLA_API mla_status mla_prefill(const void *q_nope, const void *q_rope, const void *c_kv,
                               const void *k_r, const void *W_UK, const void *W_UV,
                               const int32_t *cu_seqlens, int B, int max_seqlen,
                               int total_tokens, const mla_dims *dims, void *out, float *lse,
                               void *workspace, size_t workspace_bytes, mla_stream_t stream) {
  if (!dims_ok(dims)) return dims ? MLA_ERR_UNSUPPORTED : MLA_ERR_INVALID_ARG;
  if (B < 0 || B > 65535 || max_seqlen < 0 || total_tokens < 0) return MLA_ERR_INVALID_ARG;
  if ((max_seqlen + 127) / 128 > 65535) return MLA_ERR_INVALID_ARG;
  if (!tc_prefill_supported(*dims)) return MLA_ERR_UNSUPPORTED;
  if (B == 0 || total_tokens == 0) return MLA_OK;
  if (max_seqlen == 0) return MLA_ERR_INVALID_ARG;  // tokens, but no sequence may hold one
  if (!q_nope || !q_rope || !c_kv || !k_r || !W_UK || !W_UV || !cu_seqlens || !out || !lse)
    return MLA_ERR_INVALID_ARG;
  if (!al(q_nope, 16) || !al(q_rope, 16) || !al(c_kv, 16) || !al(k_r, 16) || !al(W_UK, 16) ||
      !al(W_UV, 16) || !al(cu_seqlens, 4) || !al(out, 16) || !al(lse, 4))
    return MLA_ERR_INVALID_ARG;
  if (!workspace || !al(workspace, 256) ||
      workspace_bytes < prefill_workspace_bytes(total_tokens, *dims))
    return MLA_ERR_WORKSPACE;
  return cuda_status(launch_prefill_tc(q_nope, q_rope, c_kv, k_r, W_UK, W_UV, cu_seqlens, B,
                                       max_seqlen, total_tokens, *dims, eff_scale(dims), out,
                                       lse, workspace, reinterpret_cast<cudaStream_t>(stream)));
}

MLA_API mla_status mla_get_error(void *workspace, mla_stream_t stream) {
  if (!workspace || !al(workspace, 256)) return MLA_ERR_WORKSPACE;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  int word = 0;
  if (cudaMemcpyAsync(&word, workspace, sizeof(int), cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return MLA_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return MLA_ERR_CUDA;
  if (word != kDevOk) {
    if (cudaMemsetAsync(workspace, 0, sizeof(int), st) != cudaSuccess) return MLA_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return MLA_ERR_CUDA;
  }
  const int gemm_word = read_and_clear_gemm_error();
  if (gemm_word < 0) return MLA_ERR_CUDA;
  if (word == kDevBounds) return MLA_ERR_DEVICE_BOUNDS;
  if (word == kDevTimeout || gemm_word == kDevTimeout) return MLA_ERR_TIMEOUT;
  return MLA_OK;
}
