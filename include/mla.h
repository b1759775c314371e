/*
 * mla.h -- C ABI of the GB300 (sm_103a) MLA decode library.
 *
 * DeepSeek Multi-Head Latent Attention decode with matrix absorption over a
 * paged latent KV cache. One decode step is
 *
 *   mla_cache_append  : write the step's new tokens (c_KV, RoPE(k_R)) into the pages
 *   mla_absorb_q      : q_lat[t,h,:]  = W_UK[h]^T q_nope[t,h,:]         (128 -> 512)
 *   mla_decode_paged  : s = (q_lat.c_KV + q_rope.k_R)/sqrt(192), online softmax,
 *                       u[t,h,:] = sum_j p_j c_KV[j]  (split-KV + log-sum-exp combine)
 *   mla_out_proj      : o[t,h,:]     = W_UV[h] u[t,h,:]                 (512 -> 128)
 *
 * (mla_decode_out_proj runs the last two as one call, merging the KV splits
 * inside the projection kernel), or, with W_UV folded into the output projection W_O once at load time
 * (mla_fuse_out_weights), in place of mla_out_proj:
 *
 *   mla_out_proj_fused: y[t,:] = sum_h W~[:,h,:] u[t,h,:]     (H*512 -> d_model)
 *
 * and before the step, from the layer's hidden states (mla_decode_front):
 *
 *   h -> q_nope, q_rope (rotated), c_kv, k_r   (RMSNorm'ed low-rank projections)
 *
 * mla_linear is the generic y = x W^T these projections run on.
 *
 * Sources (page titles):
 *   [P1] "Model Architecture Driving Inference Systems: From MHA/GQA to DeepSeek
 *        MLA Matrix Absorption and Memory Minimalism" (dev.to)
 *   [P2] "Multi-Head Latent Attention (MLA): Mathematical Foundations, Low-Rank KV
 *        Compression, Decoupled Rotary Positional Embeddings, and Inference Matrix
 *        Absorption" (llms.blog)
 *   [P5] "Tech Radar: DeepSeek-V3 Multi-Head Latent Attention (MLA) Architecture &
 *        KV Cache Compression" (tanhdev.com)
 *
 * Conventions for every entry point:
 *   - Ownership: the caller owns every buffer. The library never allocates or
 *     frees memory on these paths; scratch space is passed in (workspace).
 *   - Pointers: device pointers unless stated otherwise, to contiguous row-major
 *     arrays with the layouts given below, 16-byte aligned.
 *   - Asynchrony: every call only enqueues work on `stream` (a cudaStream_t, NULL
 *     for the legacy default stream) and returns without synchronising, except
 *     mla_read_device_error, which synchronises the stream.
 *   - Errors: argument checks (shapes, dtypes, alignment, sizes) fail
 *     synchronously with MLA_ERR_INVALID_ARG / MLA_ERR_UNSUPPORTED /
 *     MLA_ERR_WORKSPACE_TOO_SMALL and enqueue nothing. A failed launch returns
 *     MLA_ERR_CUDA. Faults that depend on device data (a block-table entry
 *     outside the pool, a bad seq_len, slot or position) never trap: the
 *     kernel skips the affected work, writes zeros (and lse = -inf) there, and
 *     ORs an MLA_DEVERR_* bit into *dev_error (if dev_error is not NULL).
 *   - No C++ exception crosses this boundary.
 *   - Dimensions: d_nope = d_v = 128, d_c = 512, d_rope = 64; num_heads in
 *     [1, 128]. A cached row is 576 values: [0,512) c_KV, [512,576) RoPE(k_R).
 */
#ifndef MLA_GB300_MLA_H
#define MLA_GB300_MLA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MLA_OK = 0,
  MLA_ERR_INVALID_ARG = 1,
  MLA_ERR_UNSUPPORTED = 2,
  MLA_ERR_CUDA = 3,
  MLA_ERR_WORKSPACE_TOO_SMALL = 4,
  MLA_ERR_DEVICE_FLAG = 5
} mla_status_t;

/* Element types. MLA_E4M3 (OCP FP8 E4M3FN) is a cache type only. */
typedef enum { MLA_F32 = 0, MLA_BF16 = 1, MLA_E4M3 = 2 } mla_dtype_t;

typedef struct {
  int32_t num_heads; /* H, 1..128                                  */
  int32_t d_nope;    /* 128: per-head content query / key width     */
  int32_t d_c;       /* 512: latent width                           */
  int32_t d_rope;    /* 64: decoupled RoPE width                    */
  int32_t d_v;       /* 128: per-head value width                   */
} mla_dims_t;

typedef void *mla_stream_t; /* cudaStream_t */

/* Bits ORed into *dev_error by kernels. */
#define MLA_DEVERR_BAD_PAGE 1     /* block_table entry outside [0, num_pages)  */
#define MLA_DEVERR_BAD_SEQLEN 2   /* seq_len < q_len or > max_pages*page_size   */
#define MLA_DEVERR_BAD_SLOT 4     /* slot_mapping entry outside the pool        */
#define MLA_DEVERR_BAD_POSITION 8 /* position outside [0, max_pos)              */
#define MLA_DEVERR_TIMEOUT 16     /* a kernel-internal wait ran out of time; the
                                     affected work item's outputs are written as
                                     for an empty one (zeros, lse -inf) where
                                     the kernel can, else left unspecified      */

/* E4M3 cache: one fp32 scale per token per group; groups of the 576-value row
 * are [0,128) [128,256) [256,384) [384,512) [512,576). */
#define MLA_E4M3_GROUPS 5

/* Human-readable name of a status code (static string, never NULL). */
const char *mla_status_string(mla_status_t status);

/* Library ABI version (major*10000 + minor*100 + patch). */
int32_t mla_version(void);

/*
 * mla_rope_table -- HOST function. Fills cos_out/sin_out [max_pos][d_rope/2]
 * (host fp32 arrays owned by the caller) with cos/sin of pos*theta_i,
 * theta_i = base^(-(2i)/d_rope), each evaluated in double precision by the C
 * library and rounded once to fp32. [P1] §2.3 / [P2] "The Decoupled RoPE
 * Solution": k_R = RoPE(W_KR h) with standard rotary frequencies.
 * Returns MLA_ERR_INVALID_ARG for max_pos < 1, odd or non-positive d_rope, a
 * non-positive base or NULL outputs.
 */
mla_status_t mla_rope_table(int32_t max_pos, int32_t d_rope, double base, float *cos_out,
                            float *sin_out);

/*
 * mla_cache_append -- write n_tokens new tokens into the paged latent cache.
 * [P2] forward_decode_absorbed, step 2 (the token is cached before attending);
 * [P1] §2.4 (row = 512 c_KV + 64 k_R); [P2] "High-Throughput Serving Kernels"
 * (FP8 E4M3 cache with per-block scaling factors).
 *
 *   c_kv        [n_tokens][512]  in_dtype (MLA_F32 or MLA_BF16)
 *   k_r         [n_tokens][64]   in_dtype, BEFORE rotation
 *   positions   [n_tokens] int32, 0-based absolute position of each token
 *   slot_mapping[n_tokens] int64, row of the pool: page * page_size + offset
 *   rope_cos, rope_sin [max_pos][32] fp32 (from mla_rope_table, copied to device)
 *   cache       [num_pages][page_size][576] cache_dtype
 *   scales      [num_pages][page_size][5] fp32 when cache_dtype == MLA_E4M3, else NULL
 *
 * Row values: c_KV rounded (nearest-even) to the cache type; k_R rotated in
 * fp32 as adjacent pairs, r0 = x0*c - x1*s, r1 = x0*s + x1*c with each product
 * and sum rounded separately, then rounded to the cache type. For MLA_E4M3 the
 * fp32 row (c_KV exact, rotated k_R unrounded) is quantised per group:
 * scale = fl32(amax/448) (1 if amax == 0), byte = E4M3(fl32(x/scale)) with
 * round-to-nearest-even and saturation to +-448. The result is bit-identical
 * to that definition. Tokens with a bad slot or position are skipped and
 * flagged (MLA_DEVERR_BAD_SLOT / MLA_DEVERR_BAD_POSITION).
 */
mla_status_t mla_cache_append(const void *c_kv, const void *k_r, const int32_t *positions,
                              const int64_t *slot_mapping, const float *rope_cos,
                              const float *rope_sin, int32_t n_tokens, int32_t max_pos,
                              void *cache, float *scales, int64_t num_pages, int32_t page_size,
                              mla_dtype_t in_dtype, mla_dtype_t cache_dtype, int32_t *dev_error,
                              mla_stream_t stream);

/*
 * mla_absorb_q -- absorbed query, q_lat[t][h][:] = W_UK[h]^T q_nope[t][h][:].
 * [P1] §3.1 (absorbed query, computed once per query token); [P2] "Attention
 * Logit Matrix Absorption" and einsum('bthd,hdc->bhtc') with W_UK viewed as
 * [n_heads][d_head][d_c].
 *
 *   q_nope [n_tokens][H][128] act, w_uk [H][128][512] act, q_lat [n_tokens][H][512] act
 * act is MLA_F32 or MLA_BF16; fp32 accumulation; q_lat rounded to act.
 * n_tokens = batch * q_len, token-major; n_tokens == 0 is a no-op.
 */
mla_status_t mla_absorb_q(const void *q_nope, const void *w_uk, void *q_lat, int32_t n_tokens,
                          mla_dims_t dims, mla_dtype_t act, mla_stream_t stream);

/*
 * Number of KV splits mla_decode_paged will use for these arguments
 * (num_splits > 0 is returned clamped to [1, max_pages_per_seq]; 0 selects
 * the library's policy for the current device). Returns < 1 on bad arguments.
 */
int32_t mla_decode_num_splits(int32_t batch, int32_t q_len, int32_t max_pages_per_seq,
                              int32_t page_size, int32_t num_splits, mla_dims_t dims,
                              mla_dtype_t cache_dtype);

/*
 * Bytes of workspace mla_decode_paged needs for these arguments: the split-KV
 * partials, [batch][q_len][splits][H][512] fp32 latent outputs plus
 * [batch][q_len][splits][H] fp32 log-sum-exps, each 256-byte aligned.
 * 0 when a single split is used.
 */
size_t mla_decode_workspace_size(int32_t batch, int32_t q_len, int32_t max_pages_per_seq,
                                 int32_t page_size, int32_t num_splits, mla_dims_t dims,
                                 mla_dtype_t cache_dtype);

/*
 * mla_decode_paged -- latent-space attention over the paged cache.
 * [P1] §3.1 score S = ((q^C)^T k^C + (q^R)^T k^R)/sqrt(d_h + d_R) with
 * (q^C)^T k^C = q_lat . c_KV; [P1] §3.2 latent sum u = sum_j P_j c_KV[j];
 * [P5] §2 score formula; [P1] §4.1 paged cache with block size 64,
 * variable-length batch.
 *
 *   q_lat       [batch][q_len][H][512] act (from mla_absorb_q)
 *   q_rope      [batch][q_len][H][64]  act, already rotated
 *   cache, scales: as written by mla_cache_append
 *   block_table [batch][max_pages_per_seq] int32: physical page of logical page i
 *   seq_lens    [batch] int32: cached tokens of each sequence INCLUDING the
 *               step's q_len new ones; query j (0-based) attends to logical
 *               tokens 0 .. seq_len - q_len + j (causal within the step)
 *   softmax_scale: multiplies q.k (1/sqrt(192) for DeepSeek dimensions)
 *   num_splits  : KV splits per (sequence, query); 0 = library policy
 *   workspace   : workspace_bytes >= mla_decode_workspace_size(...)
 *   u_out       [batch][q_len][H][512] act, normalised latent output
 *   lse_out     [batch][q_len][H] fp32 natural-log log-sum-exp of the scaled
 *               scores, or NULL
 *   dev_error   : device int32 that bad data is reported into, or NULL
 *
 * Rows past seq_len in a sequence's last page are never read into the result
 * (they may hold anything, NaN included). act is MLA_F32 or MLA_BF16;
 * cache_dtype is act, or MLA_E4M3 with act == MLA_BF16. An E4M3 value is
 * defined as decode(byte) * scale; the tensor-core kernel multiplies it as
 * fl32(code * scale) rounded to bf16 (within 2^-8 relative), the operand type
 * of the bf16 activations it pairs with.
 * Which kernel runs: the tensor-core kernel for bf16 activations, 128 heads,
 * page sizes that are multiples of 64 and pools of fewer than 2^31 rows (when
 * the driver's tensor-map encoder is available); else the CUDA-core kernel.
 * mla_decode_kernel_path reports which one a call with these arguments takes.
 */
mla_status_t mla_decode_paged(const void *q_lat, const void *q_rope, const void *cache,
                              const float *scales, const int32_t *block_table,
                              const int32_t *seq_lens, int32_t batch, int32_t q_len,
                              int32_t max_pages_per_seq, int64_t num_pages, int32_t page_size,
                              float softmax_scale, int32_t num_splits, void *workspace,
                              size_t workspace_bytes, void *u_out, float *lse_out,
                              int32_t *dev_error, mla_dims_t dims, mla_dtype_t act,
                              mla_dtype_t cache_dtype, mla_stream_t stream);

/*
 * mla_decode_kernel_path -- which decode kernel mla_decode_paged runs for a
 * cache at `cache` of num_pages pages of page_size tokens with these dims and
 * types: *path_out = MLA_DECODE_PATH_TENSOR_CORE (tcgen05, TMA) or
 * MLA_DECODE_PATH_CUDA_CORE. Host only; reads no device memory. The pages
 * describe no such call: it makes the kernel choice visible to a caller.
 * Errors: MLA_ERR_INVALID_ARG for a NULL path_out or invalid dims / sizes.
 */
#define MLA_DECODE_PATH_TENSOR_CORE 1
#define MLA_DECODE_PATH_CUDA_CORE 2
mla_status_t mla_decode_kernel_path(const void *cache, const float *scales, int64_t num_pages,
                                    int32_t page_size, mla_dims_t dims, mla_dtype_t act,
                                    mla_dtype_t cache_dtype, int32_t *path_out);

/*
 * mla_decode_out_proj -- mla_decode_paged followed by mla_out_proj, as one
 * call: u = the latent attention output, then o[t][h][:] = W_UV[h] u[t][h][:]
 * ([P1] §3.1-3.2: latent scores and sum, then the value up-projection; [P1]
 * §4.1: split KV with a log-sum-exp combine). Arguments are mla_decode_paged's
 * plus
 *   w_uv  [H][128][512] act (as for mla_out_proj)
 *   o_out [batch][q_len][H][128] act
 * u_out and lse_out are written as by mla_decode_paged. When the tensor-core
 * decode runs with 2 to 4 splits, the split merge happens inside the
 * projection kernel (one kernel fewer; W_UV is requested before that kernel
 * waits for the decode), with the same arithmetic as the merge kernel, so u,
 * lse and o are bit-identical to mla_decode_paged + mla_out_proj. Otherwise the
 * two calls run as they are. Errors: those of the two calls.
 */
mla_status_t mla_decode_out_proj(const void *q_lat, const void *q_rope, const void *cache,
                                 const float *scales, const int32_t *block_table,
                                 const int32_t *seq_lens, int32_t batch, int32_t q_len,
                                 int32_t max_pages_per_seq, int64_t num_pages, int32_t page_size,
                                 float softmax_scale, int32_t num_splits, void *workspace,
                                 size_t workspace_bytes, const void *w_uv, void *u_out,
                                 float *lse_out, void *o_out, int32_t *dev_error, mla_dims_t dims,
                                 mla_dtype_t act, mla_dtype_t cache_dtype, mla_stream_t stream);

/*
 * mla_decode_paged_static_scratch -- mla_decode_paged without a caller
 * workspace. The pages describe no such call: it exists for callers that
 * cannot allocate device memory or pass it in at call time. The split-KV
 * partials go to one device array of MLA_STATIC_SCRATCH_BYTES bytes that the
 * library holds for each device from module load on; the call allocates and
 * frees nothing.
 *
 * Arguments and results are those of mla_decode_paged (minus workspace and
 * workspace_bytes); the same kernels run, so outputs are identical to
 * mla_decode_paged's for the same inputs and split count.
 * Errors: those of mla_decode_paged, plus MLA_ERR_WORKSPACE_TOO_SMALL when
 * mla_decode_workspace_size(...) for these arguments exceeds
 * MLA_STATIC_SCRATCH_BYTES (nothing is enqueued; use fewer splits, a smaller
 * batch, or mla_decode_paged with a workspace), and MLA_ERR_CUDA if the
 * array's address cannot be obtained.
 * Errors are checked in mla_decode_paged's order (the argument errors first),
 * then the scratch size.
 * Set-up: every call looks up the array's address on the current device
 * (cudaGetSymbolAddress); the first call on a device may load the module, so
 * make it before any stream capture on that device.
 * Sharing: all calls on a device share the array. Calls that may run
 * concurrently on the device (unordered streams, several host threads) race on
 * it and corrupt each other's results; order them. Nothing in the array has to
 * start at zero: every partial the combine reads was written by the same call
 * (a work item that gave up on a wait writes -inf log-sum-exps, so its
 * partials are skipped; the timeout bit in dev_error reports it).
 */
#define MLA_STATIC_SCRATCH_BYTES ((size_t)32 << 20)
mla_status_t mla_decode_paged_static_scratch(const void *q_lat, const void *q_rope, const void *cache,
                                             const float *scales, const int32_t *block_table,
                                             const int32_t *seq_lens, int32_t batch, int32_t q_len,
                                             int32_t max_pages_per_seq, int64_t num_pages,
                                             int32_t page_size, float softmax_scale, int32_t num_splits,
                                             void *u_out, float *lse_out, int32_t *dev_error,
                                             mla_dims_t dims, mla_dtype_t act, mla_dtype_t cache_dtype,
                                             mla_stream_t stream);

/*
 * mla_prefill_mha -- prefill in the MHA form: causal attention of the last
 * n_queries positions of one sequence over all its n_tokens cached rows, with
 * the per-head keys and values expanded from the latent rows.
 * "DeepSeek's attention evolution - [MLA]" §2.5 (the latent expanded back into
 * per-head K and V: multi-head attention for prefill); "Model Architecture
 * Driving Inference Systems" FAQ Q2 (prefill runs uncompressed; absorption is
 * for decode) and §2.3 (k = [k^C ; k^R], the RoPE key shared by all heads).
 *
 *   K_h[t] = [W_UK[h] c_KV[t] ; k_R[t]] (192),  V_h[t] = W_UV[h] c_KV[t] (128)
 *   o[j][h] = sum_{t <= n_tokens - n_queries + j} softmax_t(q[j][h] . K_h[t] * scale) V_h[t]
 * with q[j][h] = [q_nope[j][h] ; q_rope[j][h]].
 *
 *   q_nope  [n_queries][H][128] bf16, q_rope [n_queries][H][64] bf16 (rotated)
 *   rows    [n_tokens][576] bf16: c_KV (512) and the rotated k_R (64) of every
 *           token, the layout of a cache row
 *   w_uk, w_uv [H][128][512] bf16
 *   workspace : >= mla_prefill_workspace_size(n_tokens, dims) bytes, 16-byte
 *           aligned (the expanded K and V; its contents are overwritten)
 *   o_out   [n_queries][H][128] bf16; lse_out [n_queries][H] fp32 or NULL
 *   dev_error : device int32 for MLA_DEVERR_TIMEOUT, or NULL
 * The expansion runs on the tensor cores (fp32 accumulation, K and V rounded
 * to bf16), then the attention (fp32 scores and sums, P rounded to bf16 for
 * the PV product). Asynchronous on `stream`.
 * Errors: MLA_ERR_INVALID_ARG (dims, sizes with 1 <= n_queries <= n_tokens <=
 * 2^20, NULL or misaligned pointers, non-finite scale), MLA_ERR_UNSUPPORTED
 * (act other than MLA_BF16, or no tensor-map encoder in the driver),
 * MLA_ERR_WORKSPACE_TOO_SMALL, MLA_ERR_CUDA (launch).
 */
size_t mla_prefill_workspace_size(int32_t n_tokens, mla_dims_t dims);
mla_status_t mla_prefill_mha(const void *q_nope, const void *q_rope, const void *rows,
                             const void *w_uk, const void *w_uv, int32_t n_tokens,
                             int32_t n_queries, float softmax_scale, void *workspace,
                             size_t workspace_bytes, void *o_out, float *lse_out,
                             int32_t *dev_error, mla_dims_t dims, mla_dtype_t act,
                             mla_stream_t stream);

/*
 * mla_out_proj -- per-head value up-projection, o[t][h][:] = W_UV[h] u[t][h][:].
 * [P1] §3.2 (W_UV moved after the attention-weighted sum); [P2] "Value Output
 * Matrix Absorption" with W_UV viewed as [n_heads][d_head][d_c].
 *
 *   u [n_tokens][H][512] act, w_uv [H][128][512] act, o [n_tokens][H][128] act
 * fp32 accumulation, o rounded to act.
 */
mla_status_t mla_out_proj(const void *u, const void *w_uv, void *o, int32_t n_tokens,
                          mla_dims_t dims, mla_dtype_t act, mla_stream_t stream);

/*
 * mla_fuse_out_weights -- fold the value up-projection into the output
 * projection, once, when the weights are loaded:
 *   W~[m][h][c] = sum_e W_O[m][h][e] W_UV[h][e][c]
 * [P1] §3.2 (pre-fused W~^O_i = W^O_i W^UV_i in R^{d x d_c}) and §4.2 (the
 * fusion is done at model load time); [P2] "Value Output Matrix Absorption"
 * (W_O^i W_UV,i is a static matrix computed at initialisation).
 *
 *   w_o     [d_model][H][128] act: W_O in R^{d_model x (H*128)}, row-major,
 *           whose column block h (128 columns) belongs to head h
 *   w_uv    [H][128][512] act
 *   w_fused [d_model][H][512] act, written
 *   d_model : 1 .. 65536
 * Each output is a 128-term dot product accumulated in fp32 and rounded once
 * to act. Not part of the per-step path.
 */
mla_status_t mla_fuse_out_weights(const void *w_o, const void *w_uv, void *w_fused, int32_t d_model,
                                  mla_dims_t dims, mla_dtype_t act, mla_stream_t stream);

/*
 * Bytes of workspace mla_out_proj_fused needs for these arguments on the
 * current device: the fp32 partial sums of a K split, [splits][n_tokens][d_model],
 * 256-byte aligned; 0 when K is not split.
 */
size_t mla_out_proj_fused_workspace_size(int32_t n_tokens, int32_t d_model, mla_dims_t dims,
                                         mla_dtype_t act);

/*
 * mla_out_proj_fused -- the attention block's output in the model dimension
 * straight from the latent outputs, through the fused weight:
 *   y[t][m] = sum_h sum_c W~[m][h][c] u[t][h][c]
 * [P1] §3.2 (the 512-dimensional latent sum multiplied by the pre-fused
 * matrix); [P2] "Value Output Matrix Absorption" (the final projection goes
 * from latent space directly to the hidden dimension).
 *
 *   u         [n_tokens][H][512] act (the u_out of mla_decode_paged)
 *   w_fused   [d_model][H][512] act (from mla_fuse_out_weights)
 *   y         [n_tokens][d_model] act, written
 *   workspace : workspace_bytes >= mla_out_proj_fused_workspace_size(...)
 *               (may be NULL when that is 0); nothing in it has to start at zero
 * This is mla_linear with n_out = d_model and n_in = 512 H (W~ viewed as
 * [d_model][512 H]); its accumulation, determinism and workspace are those of
 * mla_linear.
 */
mla_status_t mla_out_proj_fused(const void *u, const void *w_fused, void *y, int32_t n_tokens,
                                int32_t d_model, void *workspace, size_t workspace_bytes,
                                mla_dims_t dims, mla_dtype_t act, mla_stream_t stream);

/*
 * mla_linear -- y[t][o] = sum_i W[o][i] x[t][i], the linear layer of a decode
 * step (nn.Linear layout, no bias): the fused output projection and the
 * front end's projections are instances of it; so is an unfused W_O applied to
 * the concatenated per-head outputs ([P2] "Value Output Matrix Absorption",
 * W_O in R^{d x (H d_v)}).
 *
 *   x [n_tokens][n_in] act, w [n_out][n_in] act, y [n_tokens][n_out] act (written)
 *   n_out, n_in: 1 .. 2^20; n_tokens: 0 .. 2^20
 *   workspace : workspace_bytes >= mla_linear_workspace_size(...) (may be NULL
 *               when that is 0); nothing in it has to start at zero
 * fp32 accumulation. bf16 with n_in % 64 == 0 runs on the tensor cores, with K
 * split across CTAs when there are too few rows of W to occupy every SM; the
 * fp32 partial sums are then added in split order by a second kernel, so the
 * result does not depend on timing. Other shapes and fp32 run on CUDA cores.
 */
size_t mla_linear_workspace_size(int32_t n_tokens, int32_t n_out, int32_t n_in, mla_dtype_t act);
mla_status_t mla_linear(const void *x, const void *w, void *y, int32_t n_tokens, int32_t n_out,
                        int32_t n_in, void *workspace, size_t workspace_bytes, mla_dtype_t act,
                        mla_stream_t stream);

/*
 * mla_decode_front -- the decode layer's front end: from the hidden states of
 * the step's new tokens to the inputs of mla_cache_append and mla_absorb_q /
 * mla_decode_paged. [P2] "PyTorch Reference Implementation"
 * (forward_decode_absorbed, steps 1 and 2); [P1] §2.1 (c^KV = W^DKV h), §2.3
 * (decoupled RoPE queries and keys).
 *
 *   c_q    = RMSNorm(W_DQ h) * g_q            RMSNorm(v) = v / sqrt(mean(v^2) + eps)
 *   q_nope = W_UQ c_q   per head 128
 *   q_rope = RoPE_pos(W_QR c_q)   per head 64, adjacent pairs, the angle and
 *            rounding conventions of mla_cache_append (cos/sin tables)
 *   c_kv   = RMSNorm(W_DKV h) * g_kv
 *   k_r    = W_KR h   (not rotated: mla_cache_append rotates it)
 *
 *   h         [n_tokens][d_model] act
 *   w_dqkv    [d_cq + 512 + 64][d_model] act: rows [0, d_cq) W_DQ, then 512
 *             rows of W_DKV, then 64 rows of W_KR (nn.Linear layouts, stacked)
 *   g_q [d_cq], g_kv [512] act: the RMSNorm gains
 *   w_uqr     [H*128 + H*64][d_cq] act: rows [0, H*128) W_UQ (row 128 h + d is
 *             head h, feature d), then H*64 rows of W_QR (row 64 h + r)
 *   positions [n_tokens] int32: each token's position (that of its cache row)
 *   rope_cos, rope_sin [max_pos][32] fp32 (mla_rope_table)
 *   eps       >= 0 (torch's nn.RMSNorm default in fp32 is 2^-23)
 *   q_nope [n_tokens][H][128], q_rope [n_tokens][H][64], c_kv [n_tokens][512],
 *   k_r [n_tokens][64] act, written
 *   workspace : workspace_bytes >= mla_decode_front_workspace_size(...); holds
 *             the fp32 sums of both products and c_q; nothing in it has to
 *             start at zero
 * The products accumulate in fp32; the norms and the rotation are computed in
 * fp32 from the fp32 sums; c_q is rounded to act once, before W_UQ and W_QR.
 * A position outside [0, max_pos) writes a zero q_rope for that token and ORs
 * MLA_DEVERR_BAD_POSITION into *dev_error.
 */
size_t mla_decode_front_workspace_size(int32_t n_tokens, int32_t d_model, int32_t d_cq,
                                       mla_dims_t dims, mla_dtype_t act);
mla_status_t mla_decode_front(const void *h, const void *w_dqkv, const void *g_q, const void *g_kv,
                              const void *w_uqr, const int32_t *positions, const float *rope_cos,
                              const float *rope_sin, int32_t max_pos, float eps, int32_t n_tokens,
                              int32_t d_model, int32_t d_cq, void *q_nope, void *q_rope, void *c_kv,
                              void *k_r, void *workspace, size_t workspace_bytes,
                              int32_t *dev_error, mla_dims_t dims, mla_dtype_t act,
                              mla_stream_t stream);

/*
 * mla_read_device_error -- synchronise `stream`, copy *dev_error (device) to
 * *code_out (host) and return MLA_ERR_DEVICE_FLAG if it is non-zero, MLA_OK
 * otherwise. Does not clear the flag.
 */
mla_status_t mla_read_device_error(const int32_t *dev_error, mla_stream_t stream,
                                   int32_t *code_out);

#ifdef __cplusplus
}
#endif

#endif /* MLA_GB300_MLA_H */
