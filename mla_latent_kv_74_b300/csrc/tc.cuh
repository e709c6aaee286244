// Tensor-core (tcgen05 / TMA) paths: shape predicates and launchers.
#pragma once

#include "internal.cuh"

namespace mla {

// bf16, d_h = 128, d_c = 512 (per-head GEMMs on tcgen05).
bool tc_gemm_supported(const mla_dims &d);
// bf16, d_c = 512, d_r = 64, block_size = 64, H <= 128 and at most 8192
// (sequence, query slot) items (paged TMA decode on tcgen05).
bool tc_decode_supported(const mla_dims &d, int B, int Hq);
size_t tc_decode_workspace_bytes(int B, int Hq, const mla_dims &d);

cudaError_t launch_absorb_tc(const void *q_nope, const void *W_UK, void *q_lat, int rows,
                             const mla_dims &d, cudaStream_t st);
cudaError_t launch_out_proj_tc(const void *o_lat, const void *W_UV, void *out, int rows,
                               const mla_dims &d, cudaStream_t st);
// Attention over the logical cache blocks [first_block, end_block) of every
// sequence (0 and INT_MAX: the whole visible length).
cudaError_t launch_decode_tc(const void *q_lat, const void *q_rope, const void *cache,
                             int num_blocks, const int32_t *block_table, int max_blocks,
                             const int32_t *seqlens, int max_seqlen, int B, int Hq,
                             int first_block, int end_block, const mla_dims &d, float scale,
                             void *o_lat, float *lse, void *workspace, cudaStream_t st);
// Log-sum-exp merge of P pieces [P][rows][512] bf16 + [P][rows] fp32.
cudaError_t launch_combine_pieces_tc(const void *o_pieces, const float *lse_pieces, int P,
                                     long rows, void *o_lat, float *lse, cudaStream_t st);

// bf16, d_c = 512, d_r = 64, d_model a multiple of 64 (fused latent / RoPE-key
// projection into the paged cache on tcgen05).
bool tc_project_supported(const mla_dims &d, int d_model);
size_t project_workspace_bytes(int T, int d_model, const mla_dims &d);
cudaError_t launch_project_append_tc(const void *h, const void *W_DKV, const void *W_KR,
                                     int d_model, double rope_base, void *cache, int num_blocks,
                                     const int32_t *block_table, int max_blocks,
                                     const int32_t *seqlens, int B, int n_new,
                                     const mla_dims &d, void *workspace, cudaStream_t st);

// bf16, d_h = 128, even d_model (output projection over the concatenated
// heads on tcgen05, K split into fp32 partials).
bool tc_oproj_supported(const mla_dims &d, int d_model);
size_t oproj_workspace_bytes(int T, int d_model, const mla_dims &d);
cudaError_t launch_oproj_tc(const void *out, const void *W_O, void *u, int T, int d_model,
                            const mla_dims &d, void *workspace, cudaStream_t st);

// bf16, d_h = 128, even d_r, d_model a multiple of 64 (query projections
// q_nope = W_Q h and q_rope = RoPE(W_QR h) on tcgen05).
bool tc_qproj_supported(const mla_dims &d, int d_model);
size_t qproj_workspace_bytes(int T, int d_model, const mla_dims &d);
cudaError_t launch_qproj_tc(const void *h, const void *W_Q, const void *W_QR, int d_model,
                            double rope_base, const int32_t *seqlens, int B, int Hq,
                            const mla_dims &d, void *q_nope, void *q_rope, void *workspace,
                            cudaStream_t st);

// bf16, d_h = 128, d_c = 512, d_r = 64 (prefill in the standard order:
// [K_nope | V] per token and head rebuilt on tcgen05 into the workspace,
// then causal attention on tcgen05).
bool tc_prefill_supported(const mla_dims &d);
size_t prefill_workspace_bytes(int total, const mla_dims &d);
cudaError_t launch_prefill_tc(const void *q_nope, const void *q_rope, const void *c_kv,
                              const void *k_r, const void *W_UK, const void *W_UV,
                              const int32_t *cu_seqlens, int B, int max_seqlen, int total,
                              const mla_dims &d, float scale, void *out, float *lse,
                              void *workspace, cudaStream_t st);

// Read and clear the error word of the GEMM kernels (they take no workspace);
// returns the device error code, or -1 if it could not be read.
int read_and_clear_gemm_error();

}  // namespace mla
