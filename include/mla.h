/*
 * mla.h -- C ABI of the MLA decode library (Multi-head Latent Attention with
 * matrix absorption), built for NVIDIA B300 (sm_103a).
 *
 * One decode step is four stream-ordered calls:
 *
 *   mla_append_cache   write the new tokens' [c_KV ; k_R] rows into the cache
 *   mla_absorb_query   q_lat = W_UK^T q_nope            (per head)
 *   mla_decode         softmax((q_lat.c_j + q_rope.k_R_j) * scale) over the
 *                      cached latents, accumulated in latent space:
 *                      o_lat = sum_j p_j c_j, plus lse
 *   mla_out_proj       out = W_UV o_lat                  (per head)
 *
 * mla_project_query produces q_nope and q_rope from the hidden states.
 * mla_o_proj applies W^O to the concatenated head outputs of mla_out_proj.
 * mla_project_append can replace mla_append_cache when the caller holds the
 * new tokens' hidden states: it computes c = W_DKV h and k_R = RoPE(W_KR h)
 * and writes them straight into the cache.
 * mla_prefill runs attention for whole prompts in the standard (un-absorbed)
 * order, the one that is cheaper when every token is a query.
 *
 * The per-head keys W_UK c_j and values W_UV c_j of cached tokens are never
 * formed.  Sources (page title, section):
 *   - "Multi-Head Latent Attention: Low-Rank KV Compression, Decoupled RoPE,
 *     and Matrix Absorption": MLA (k = W^UK c, v = W^UV c, W in R^{d_h x d_c})
 *     and Matrix Absorption.
 *   - "MLA, dim by dim" 4.2 (decode order: absorb the query, contract the
 *     cache last, expand with W_UV after the latent sum) and 5.2 (decoupled
 *     RoPE: score = content + positional term, joint scale 1/sqrt(d_k+d_r),
 *     one rotated k_R per token shared by all heads).
 *   - "From Vanilla Transformers to Modern LLMs -- Part 3" 3.e.2 (absorbed
 *     query), 3.g/3.p (values in latent space), 3.o (scale), 3.q (cache).
 *   - "Mathematical Prerequisites for DeepSeek-V2" 6 (bilinear identity) and
 *     7 (linearity): why the absorbed order gives the same result.
 *
 * Conventions for every call
 *   - Every tensor pointer is DEVICE memory owned by the caller; the library
 *     never allocates, frees or keeps a pointer after the call returns.
 *   - Tensors are dense, row-major, in the layouts written beside each
 *     argument.  Element type is dims->dtype (bf16 or fp32) unless stated.
 *     Pointers must be 16-byte aligned; the cache pointer 128-byte aligned.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *     default stream).  No call synchronises except mla_get_error.
 *   - Argument errors are detected on the host before anything is launched;
 *     the call then returns MLA_ERR_INVALID_ARG or MLA_ERR_UNSUPPORTED and
 *     leaves every buffer untouched.  A failed launch returns MLA_ERR_CUDA.
 *   - Errors found on the device are recorded in the decode workspace's
 *     error word; read it with mla_get_error.  A block-table entry outside
 *     [0,num_blocks) or a sequence length above max_seqlen or the table's
 *     capacity (MLA_ERR_DEVICE_BOUNDS) leaves the affected rows written as
 *     o_lat = 0, lse = -inf.  A bounded wait that expired (MLA_ERR_TIMEOUT)
 *     stops the kernel early: rows it had not finished are left unwritten.
 *   - Positions start at 0.  seqlens[b] counts tokens AFTER the current Hq
 *     tokens were appended.  Query slot i (0 <= i < Hq) of sequence b sits
 *     at position seqlens[b]-Hq+i and sees positions 0..seqlens[b]-Hq+i
 *     (causal between slots).  A row that sees no position gets o_lat = 0
 *     and lse = -inf.
 */
#ifndef MLA_H_
#define MLA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same handle as cudaStream_t. */
typedef struct CUstream_st *mla_stream_t;

typedef enum {
  MLA_OK = 0,
  MLA_ERR_INVALID_ARG = 1,   /* null/misaligned pointer, bad size            */
  MLA_ERR_UNSUPPORTED = 2,   /* dims or dtype outside what the library runs */
  MLA_ERR_WORKSPACE = 3,     /* workspace missing or too small              */
  MLA_ERR_CUDA = 4,          /* a CUDA runtime call or launch failed        */
  MLA_ERR_DEVICE_BOUNDS = 5, /* device: block index / length out of range   */
  MLA_ERR_TIMEOUT = 6        /* device: a bounded wait gave up              */
} mla_status;

typedef enum { MLA_BF16 = 0, MLA_FP32 = 1 } mla_dtype;

/* Model dimensions.  H heads of width d_h; latent width d_c; decoupled RoPE
 * width d_r (the cache row is d_c + d_r wide); block_size cache rows per
 * physical block.  scale <= 0 selects 1/sqrt(d_h + d_r) ("MLA, dim by dim"
 * 5.2).  Supported: 1 <= H <= 256, 1 <= d_h <= 128, 1 <= d_c <= 512,
 * 0 <= d_r <= 64, 1 <= block_size <= 1024; both dtypes.  The tensor-core
 * paths run bf16 with d_h = 128, d_c = 512, d_r = 64, block_size = 64; every
 * other supported shape runs on CUDA-core kernels. */
typedef struct {
  int H, d_h, d_c, d_r, block_size;
  mla_dtype dtype;
  float scale;
} mla_dims;

/* Absorb W_UK into the query: q_lat[b,i,h,:] = W_UK[h]^T q_nope[b,i,h,:].
 * ("From Vanilla Transformers to Modern LLMs -- Part 3" 3.e.2;
 *  "MLA, dim by dim" 5.2, the bracketed left factor of the cached-decode score.)
 *   q_nope [B, Hq, H, d_h]   input
 *   W_UK   [H, d_h, d_c]     input, row-major per head (d_h rows of d_c)
 *   q_lat  [B, Hq, H, d_c]   output (fp32 accumulation, rounded to dtype)
 * B >= 0, Hq >= 1.  B == 0 is a no-op. */
mla_status mla_absorb_query(const void *q_nope, const void *W_UK, void *q_lat,
                            int B, int Hq, const mla_dims *dims,
                            mla_stream_t stream);

/* Append the n_new newest tokens of every sequence to the paged cache.
 * Token i (0 <= i < n_new) of sequence b goes to position
 * p = seqlens[b] - n_new + i: physical block block_table[b*max_blocks +
 * p/block_size], row p % block_size, as [c_kv[b,i,:] ; k_r[b,i,:]].
 * ("MLA Explained", decode step 5; "From Vanilla Transformers to Modern
 *  LLMs -- Part 3" 3.q: k_R is stored already rotated.)
 *   cache       [num_blocks, block_size, d_c + d_r]  in/out
 *   block_table [B, max_blocks] int32                input
 *   seqlens     [B] int32, lengths after the append  input
 *   c_kv        [B, n_new, d_c]                      input
 *   k_r         [B, n_new, d_r] (pre-rotated)        input (may be NULL iff d_r == 0)
 * Positions p < 0 and block entries outside [0, num_blocks) are skipped
 * (mla_decode reports the latter when it reads them). */
mla_status mla_append_cache(void *cache, int num_blocks,
                            const int32_t *block_table, int max_blocks,
                            const int32_t *seqlens, const void *c_kv,
                            const void *k_r, int B, int n_new,
                            const mla_dims *dims, mla_stream_t stream);

/* Bytes of device workspace mla_project_append needs (its K-split fp32
 * partial sums: about 4 MB for 64 tokens at d_model = 5120).  Returns
 * MLA_ERR_UNSUPPORTED for shapes mla_project_append does not take. */
mla_status mla_project_append_workspace_size(int B, int n_new, int d_model,
                                             const mla_dims *dims, size_t *bytes);

/* Fused down-projection, RoPE and append: for token i (0 <= i < n_new) of
 * sequence b at position p = seqlens[b] - n_new + i,
 *   c   = W_DKV h[b,i,:]                       (d_c)
 *   k   = W_KR h[b,i,:], then each adjacent pair (2j, 2j+1) of k rotated by
 *         the angle p * rope_base^(-2j/d_r):  k' = k cos + rotate_half(k) sin
 *         with rotate_half(x0, x1) = (-x1, x0)
 * and [c ; k'] is written to the cache row of position p exactly as
 * mla_append_cache writes it.  ("Multi-Head Latent Attention: Low-Rank KV
 * Compression, Decoupled RoPE, and Matrix Absorption": c = W^DKV h and the
 * shared RoPE key; "MLA, dim by dim" 3 (RoPE on adjacent pairs) and 5.2;
 * "From Vanilla Transformers to Modern LLMs -- Part 3" 3.b, 3.k, 3.q.)
 *   h           [B, n_new, d_model] bf16                 input
 *   W_DKV       [d_c, d_model] bf16 (row m gives c[m])   input
 *   W_KR        [d_r, d_model] bf16 (one k_R for all heads) input
 *   cache, block_table, seqlens: as in mla_append_cache
 *   workspace   >= mla_project_append_workspace_size bytes, 256-byte
 *               aligned, caller-owned scratch (no zeroing needed)
 * Supported: bf16, d_c = 512, d_r = 64, d_model a multiple of 64 (else
 * MLA_ERR_UNSUPPORTED).  Products accumulate in fp32; the rotation angle is
 * formed in double precision; the row is rounded to bf16 once.  Positions
 * p < 0 and block entries outside [0, num_blocks) are skipped. */
mla_status mla_project_append(const void *h, const void *W_DKV, const void *W_KR,
                              int d_model, float rope_base, void *cache,
                              int num_blocks, const int32_t *block_table,
                              int max_blocks, const int32_t *seqlens, int B,
                              int n_new, const mla_dims *dims, void *workspace,
                              size_t workspace_bytes, mla_stream_t stream);

/* Bytes of device workspace mla_project_query needs (its K-split fp32
 * partial sums: about 19 MB for 64 rows at H = 128, d_model = 5120).  Returns
 * MLA_ERR_UNSUPPORTED for shapes mla_project_query does not take. */
mla_status mla_project_query_workspace_size(int B, int Hq, int d_model,
                                            const mla_dims *dims, size_t *bytes);

/* The query side of the step, before mla_absorb_query (no query
 * compression, as in DeepSeek-V2-Lite): for query slot i of sequence b at
 * position p = seqlens[b] - Hq + i,
 *   q_nope[b,i,:,:] = W_Q h[b,i,:]                     (H * d_h)
 *   q_rope[b,i,h,:] = RoPE((W_QR h[b,i,:])[h*d_r .. h*d_r+d_r-1], p)
 * with RoPE as in mla_project_append (pairs (2j, 2j+1) of each head's d_r,
 * angle p * rope_base^(-2j/d_r)).  ("Multi-Head Latent Attention: Low-Rank
 * KV Compression, Decoupled RoPE, and Matrix Absorption": the query and its
 * per-head RoPE part; "From Vanilla Transformers to Modern LLMs -- Part 3"
 * 3.d, 3.l; "MLA, dim by dim" 3, 5.2.)
 *   h       [B, Hq, d_model] bf16                      input
 *   W_Q     [H * d_h, d_model] bf16 (row m gives q[m])  input
 *   W_QR    [H * d_r, d_model] bf16                    input
 *   q_nope  [B, Hq, H, d_h], q_rope [B, Hq, H, d_r]   output (the inputs of
 *           mla_absorb_query and mla_decode)
 *   workspace >= mla_project_query_workspace_size bytes, 256-byte aligned
 * Supported: bf16, d_h = 128, even d_r, d_model a multiple of 64.  Products
 * accumulate in fp32, the angle is formed in double precision, outputs are
 * rounded to bf16 once. */
mla_status mla_project_query(const void *h, const void *W_Q, const void *W_QR,
                             int d_model, float rope_base,
                             const int32_t *seqlens, int B, int Hq,
                             const mla_dims *dims, void *q_nope, void *q_rope,
                             void *workspace, size_t workspace_bytes,
                             mla_stream_t stream);

/* Bytes of device workspace mla_o_proj needs (its K-split fp32 partial sums:
 * about 9 MB for 64 rows at d_model = 5120, H = 128).  Returns
 * MLA_ERR_UNSUPPORTED for shapes mla_o_proj does not take. */
mla_status mla_o_proj_workspace_size(int B, int Hq, int d_model,
                                     const mla_dims *dims, size_t *bytes);

/* Output projection over the concatenated heads, the step after
 * mla_out_proj:  u[b,i,:] = W_O [out[b,i,0,:] ; ... ; out[b,i,H-1,:]]
 * ("Multi-Head Latent Attention: Low-Rank KV Compression, Decoupled RoPE,
 *  and Matrix Absorption", the head outputs concatenated and multiplied by
 *  W^O; "From Vanilla Transformers to Modern LLMs -- Part 3" 3.h, 3.p: u_t).
 *   out         [B, Hq, H, d_h]                         input
 *   W_O         [d_model, H * d_h] (row m gives u[m])   input
 *   u           [B, Hq, d_model]                        output
 *   workspace   >= mla_o_proj_workspace_size bytes, 256-byte aligned,
 *               caller-owned scratch (no zeroing needed)
 * Supported: bf16, d_h = 128, even d_model (else MLA_ERR_UNSUPPORTED).
 * Products accumulate in fp32 (K split across the SMs, partials summed in
 * fp32); u is rounded to bf16 once. */
mla_status mla_o_proj(const void *out, const void *W_O, void *u, int B, int Hq,
                      int d_model, const mla_dims *dims, void *workspace,
                      size_t workspace_bytes, mla_stream_t stream);

/* Bytes of device workspace mla_decode needs for this problem size.  The
 * workspace holds the split-KV partials, the split plan and the error word.
 * It must be zero-filled once before its first use; after that it may be
 * reused by consecutive calls on one stream.  max_seqlen is an upper bound
 * on seqlens[].  The size is that of the path mla_decode takes for these
 * arguments (see mla_decode).  B * Hq above 65535 returns
 * MLA_ERR_UNSUPPORTED. */
mla_status mla_decode_workspace_size(int B, int Hq, int max_seqlen,
                                     const mla_dims *dims, size_t *bytes);

/* Absorbed MLA decode over the paged latent cache, split across the SMs
 * along the sequence and merged by a log-sum-exp combine.
 * For every b, query slot i, head h, with n = seqlens[b] - Hq + i + 1:
 *   s_j   = (q_lat[b,i,h,:] . c_j + q_rope[b,i,h,:] . kR_j) * scale, j < n
 *   p_j   = softmax_j(s_j)
 *   o_lat[b,i,h,:] = sum_j p_j c_j          ("MLA, dim by dim" 4.2, 5.2)
 *   lse[b,i,h]     = ln sum_j exp(s_j)      (natural log, scaled units)
 * where row j of the sequence is cache[block_table[b][j/bs]][j%bs] =
 * [c_j (d_c) ; kR_j (d_r)].
 *   q_lat       [B, Hq, H, d_c]                    input
 *   q_rope      [B, Hq, H, d_r] (pre-rotated)      input (NULL iff d_r == 0)
 *   cache       [num_blocks, block_size, d_c+d_r]  input
 *   block_table [B, max_blocks] int32              input
 *   seqlens     [B] int32                          input
 *   o_lat       [B, Hq, H, d_c]                    output (dtype)
 *   lse         [B, Hq, H] float32                 output
 *   workspace   >= mla_decode_workspace_size bytes, 256-byte aligned
 * Consecutive calls that share a workspace must be ordered on one stream.
 * Paths: bf16 with d_c = 512, d_r = 64, block_size = 64, H <= 128 and
 * B * Hq <= 8192 runs on the tensor cores; every other supported problem
 * with B * Hq <= 65535 on CUDA cores; B * Hq > 65535 returns
 * MLA_ERR_UNSUPPORTED before anything is launched. */
mla_status mla_decode(const void *q_lat, const void *q_rope, const void *cache,
                      int num_blocks, const int32_t *block_table,
                      int max_blocks, const int32_t *seqlens, int max_seqlen,
                      int B, int Hq, const mla_dims *dims, void *o_lat,
                      float *lse, void *workspace, size_t workspace_bytes,
                      mla_stream_t stream);

/* mla_decode restricted to the logical cache blocks [first_block, end_block)
 * of every sequence: the keys j with first_block*block_size <= j <
 * end_block*block_size (and j < n as above).  o_lat and lse are then the
 * softmax-weighted latent and the log-sum-exp over those keys alone (o_lat
 * = 0, lse = -inf where none is visible), i.e. one piece of a split-KV
 * computation; pieces over disjoint ranges that cover [0, n) merge into
 * mla_decode's result with mla_combine_pieces.  This is how one very long
 * sequence is split across GPUs: each GPU decodes the blocks it holds and
 * the pieces are gathered to one of them.  block_table rows keep their
 * full width (entries before first_block are not read).  Arguments, layouts
 * and workspace as for mla_decode; first_block < 0 or end_block <
 * first_block returns MLA_ERR_INVALID_ARG.  Only the tensor-core path
 * takes block ranges (other problems return MLA_ERR_UNSUPPORTED). */
mla_status mla_decode_blocks(const void *q_lat, const void *q_rope, const void *cache,
                             int num_blocks, const int32_t *block_table, int max_blocks,
                             const int32_t *seqlens, int max_seqlen, int B, int Hq,
                             int first_block, int end_block, const mla_dims *dims,
                             void *o_lat, float *lse, void *workspace, size_t workspace_bytes,
                             mla_stream_t stream);

/* Log-sum-exp merge of P pieces of the same rows, each the output of
 * mla_decode_blocks over one range of a partition of the keys:
 *   lse = ln sum_p exp(lse_p),   o_lat = sum_p exp(lse_p - lse) o_p
 * (the softmax over the union of the ranges, "Part 3" 2.a and 3.f, written
 * as a weighted mean of the per-range means).  Pieces with lse_p = -inf
 * weigh nothing; rows with every lse_p = -inf (or a NaN) get o_lat = 0,
 * lse = -inf.
 *   o_pieces   [P, B, Hq, H, d_c] bf16   input (pieces stacked, 16-byte aligned)
 *   lse_pieces [P, B, Hq, H] float32     input
 *   o_lat      [B, Hq, H, d_c] bf16      output
 *   lse        [B, Hq, H] float32        output
 * Supported: the tensor-core decode shapes (bf16, d_c = 512); others return
 * MLA_ERR_UNSUPPORTED.  Asynchronous on `stream`; needs no workspace. */
mla_status mla_combine_pieces(const void *o_pieces, const float *lse_pieces, int P, int B,
                              int Hq, const mla_dims *dims, void *o_lat, float *lse,
                              mla_stream_t stream);

/* Expand the latent output through W_UV: out[b,i,h,:] = W_UV[h] o_lat[b,i,h,:].
 * ("From Vanilla Transformers to Modern LLMs -- Part 3" 3.g; "MLA, dim by
 *  dim" 4.2, the value chain contracted left to right.)
 *   o_lat [B, Hq, H, d_c]   input
 *   W_UV  [H, d_h, d_c]     input
 *   out   [B, Hq, H, d_h]   output (fp32 accumulation, rounded to dtype) */
mla_status mla_out_proj(const void *o_lat, const void *W_UV, void *out, int B,
                        int Hq, const mla_dims *dims, mla_stream_t stream);

/* Bytes of device workspace mla_prefill needs: the error word plus the
 * rebuilt keys and values, 512 bytes per (token, head) in bf16 (about
 * 268 MB for 4096 tokens at H = 128).  Returns MLA_ERR_UNSUPPORTED for
 * shapes mla_prefill does not take. */
mla_status mla_prefill_workspace_size(int total_tokens, const mla_dims *dims,
                                      size_t *bytes);

/* MLA prefill in the standard order ("MLA, dim by dim" 4.1; "MLA
 * Explained", training and prefill): the per-head keys and values are
 * rebuilt from the latents first, then causal attention runs over
 * d_k = d_h + d_r and d_v = d_h (absorption would put the T^2 contractions
 * on d_c instead).  Sequences are packed end to end: sequence b is tokens
 * cu_seqlens[b] .. cu_seqlens[b+1]-1, and token t of it (0-based) attends to
 * tokens 0..t of the same sequence.  For every such token t and head h:
 *   K_j = [W_UK[h] c_j ; kR_j],  V_j = W_UV[h] c_j
 *   s_j = [q_nope[t,h,:] ; q_rope[t,h,:]] . K_j * scale,  j <= t
 *   out[t,h,:] = sum_j softmax_j(s_j) V_j,   lse[t,h] = ln sum_j exp(s_j)
 * (scores as in mla_decode, so a sequence's last row equals a decode of it).
 *   q_nope      [total_tokens, H, d_h]             input
 *   q_rope      [total_tokens, H, d_r] (rotated)   input
 *   c_kv        [total_tokens, d_c]                input
 *   k_r         [total_tokens, d_r]   (rotated)    input
 *   W_UK, W_UV  [H, d_h, d_c]                      input
 *   cu_seqlens  [B + 1] int32, cu_seqlens[0] = 0, non-decreasing,
 *               cu_seqlens[B] = total_tokens       input (device)
 *   max_seqlen  >= every sequence length (sizes the grid)
 *   out         [total_tokens, H, d_h]             output
 *   lse         [total_tokens, H] float32          output
 *   workspace   >= mla_prefill_workspace_size bytes, 256-byte aligned; its
 *               first word is the error word that mla_get_error reads, its
 *               bytes 8-15 the attention kernel's work-list counter (reset
 *               by every call), the rest the rebuilt K and V
 * Supported: bf16, d_h = 128, d_c = 512, d_r = 64 (else MLA_ERR_UNSUPPORTED);
 * B <= 65535.  K and V are rounded to bf16 once after their fp32
 * accumulation; scores and the softmax are fp32, P is rounded to bf16 for
 * the P V product, out is rounded to bf16 once.  A sequence whose
 * cu_seqlens entries are out of range (negative length, longer than
 * max_seqlen, past total_tokens) is skipped: its rows are not written and
 * MLA_ERR_DEVICE_BOUNDS is recorded in the error word. */
mla_status mla_prefill(const void *q_nope, const void *q_rope, const void *c_kv,
                       const void *k_r, const void *W_UK, const void *W_UV,
                       const int32_t *cu_seqlens, int B, int max_seqlen,
                       int total_tokens, const mla_dims *dims, void *out,
                       float *lse, void *workspace, size_t workspace_bytes,
                       mla_stream_t stream);

/* Synchronise `stream`, read and clear the workspace's device error word,
 * together with the library-wide word of the tensor-core GEMMs
 * (mla_absorb_query, mla_out_proj, mla_project_append, mla_project_query,
 * mla_o_proj, and the key / value rebuild of mla_prefill), whose bounded
 * waits record MLA_ERR_TIMEOUT there.
 * Returns MLA_OK, MLA_ERR_DEVICE_BOUNDS, MLA_ERR_TIMEOUT or MLA_ERR_CUDA. */
mla_status mla_get_error(void *workspace, mla_stream_t stream);

/* Self-test of the failure path (no counterpart on the pages): one kernel
 * waits, through the library's bounded wait, on an mbarrier phase that
 * nothing completes.  The wait gives up after its limit (2 s) and the kernel
 * records MLA_ERR_TIMEOUT in the workspace's error word, as a real lost wait
 * in mla_decode or mla_prefill would.  mla_get_error then returns
 * MLA_ERR_TIMEOUT and clears the word; the context stays usable.
 *   workspace   any workspace of this library (>= 256 bytes, 256-byte
 *               aligned); only its error word is written
 * Returns MLA_ERR_WORKSPACE for a missing or misaligned workspace,
 * MLA_ERR_CUDA if the launch fails. */
mla_status mla_selftest_lost_wait(void *workspace, mla_stream_t stream);

/* Static, human-readable name of a status code. */
const char *mla_status_string(mla_status status);

/* Bytes of the scratch array built into the library for mla_decode_noalloc.
 * Every GPU that loads the library holds this much device memory until the
 * process exits. */
#define MLA_NOALLOC_SCRATCH_BYTES ((size_t)48 << 20)

/* mla_decode for callers that cannot allocate device memory.
 * The paper has no counterpart to this call: it exists for deployment only.
 * mla_decode needs a workspace that the caller allocates; some callers cannot
 * call cudaMalloc (a plugin inside a host application that owns all device
 * memory and exposes no allocator, or a serving loop that must never block on
 * an allocation).  This variant takes the workspace from a fixed array of
 * MLA_NOALLOC_SCRATCH_BYTES compiled into the library and allocates nothing:
 * no cudaMalloc, no cudaFree, no allocating library routine.
 *   Arguments, layouts and results are those of mla_decode, minus the
 *   workspace.  The caller still provides every input and output.
 *   - A problem whose workspace (mla_decode_workspace_size) exceeds
 *     MLA_NOALLOC_SCRATCH_BYTES is rejected with MLA_ERR_WORKSPACE before
 *     anything is launched.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current) and caches it; make
 *     that first call before any stream capture.
 *   - The array's device address is looked up (cudaGetSymbolAddress, with
 *     the caller's device current) on every call; the lookup allocates
 *     nothing.  The first call on a device, and the first after a device
 *     reset, also loads the library onto that device: make it before any
 *     stream capture.
 *   - All calls share the one array, which keeps the last call's contents;
 *     each call clears the part that must start at zero (the error word)
 *     before its kernels run.  Calls that overlap on the GPU (different
 *     streams, or different host threads without ordering) race on the array
 *     and give undefined results: order them on one stream.
 *   - Device-side errors go to the array's error word, with the effects
 *     described for mla_decode; read them with mla_decode_noalloc_get_error
 *     before the next call, which clears the word. */
mla_status mla_decode_noalloc(const void *q_lat, const void *q_rope,
                              const void *cache, int num_blocks,
                              const int32_t *block_table, int max_blocks,
                              const int32_t *seqlens, int max_seqlen, int B,
                              int Hq, const mla_dims *dims, void *o_lat,
                              float *lse, mla_stream_t stream);

/* mla_get_error for mla_decode_noalloc (no counterpart in the paper either):
 * synchronise `stream`, then read and clear the error word of the built-in
 * array (and the GEMMs' library-wide word, as mla_get_error does).  Returns
 * MLA_OK, MLA_ERR_DEVICE_BOUNDS, MLA_ERR_TIMEOUT or MLA_ERR_CUDA.  It
 * allocates nothing. */
mla_status mla_decode_noalloc_get_error(mla_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MLA_H_ */
