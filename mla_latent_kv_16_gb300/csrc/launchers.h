// Internal launchers behind the C ABI (mla.h). Arguments are already validated.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <utility>

#include "mla.h"

namespace mla {

// Every kernel of the library is launched with programmatic stream
// serialization: it may start while the previous kernel in the stream is still
// running, does only work that touches no data an earlier kernel writes
// (barrier set-up, TMEM allocation, static weights), and executes
// griddepcontrol.wait (pdl_wait) before anything else. Each kernel triggers its
// own dependents at entry (pdl_trigger). A kernel the caller launched before
// ours never triggers early, so our kernels start early only behind our own.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

struct AppendArgs {
  const void* c_kv;
  const void* k_r;
  const int32_t* positions;
  const int64_t* slots;
  const float* cos_t;
  const float* sin_t;
  int32_t n_tokens;
  int32_t max_pos;
  void* cache;
  float* scales;
  int64_t n_rows;  // num_pages * page_size
  mla_dtype_t in_dtype;
  mla_dtype_t cache_dtype;
  int32_t* dev_error;
};
cudaError_t launch_append(const AppendArgs& a, cudaStream_t s);

struct ProjArgs {
  const void* x;  // q_nope [n][H][128] (absorb) or u [n][H][512] (out_proj)
  const void* w;  // [H][128][512]
  void* y;        // q_lat [n][H][512] or o [n][H][128]
  int32_t n_tokens;
  int32_t heads;
  mla_dtype_t act;
};
cudaError_t launch_absorb_simt(const ProjArgs& a, cudaStream_t s);
cudaError_t launch_out_proj_simt(const ProjArgs& a, cudaStream_t s);
// tcgen05 versions (bf16 only). Return cudaErrorNotSupported when not applicable.
cudaError_t launch_absorb_tc(const ProjArgs& a, cudaStream_t s);
cudaError_t launch_out_proj_tc(const ProjArgs& a, cudaStream_t s);

// The split merge of a decode and the value up-projection in one kernel
// (proj_tc.cu): u[t,h,:] merged from the decode's fp32 split partials, then
// o[t,h,:] = W_UV[h] u[t,h,:]. bf16, 128 heads, 2..4 splits.
struct MergeProjArgs {
  const float* part_u;    // [n][S][H][512] fp32, as the decode wrote them
  const float* part_lse;  // [n][S][H]
  int32_t num_splits;
  const void* w;          // W_UV [H][128][512] bf16
  void* u_out;            // [n][H][512] bf16: the merged latent output
  float* lse_out;         // [n][H] or nullptr
  void* o;                // [n][H][128] bf16
  int32_t n_tokens;       // n = batch * q_len
  int32_t heads;
};
bool out_proj_merge_supported(int32_t heads, int32_t splits, mla_dtype_t act);
cudaError_t launch_out_proj_merge_tc(const MergeProjArgs& a, cudaStream_t s);

struct FuseWeightsArgs {
  const void* w_o;   // [d][H][128]
  const void* w_uv;  // [H][128][512]
  void* w_fused;     // [d][H][512]
  int32_t d_model;
  int32_t heads;
  mla_dtype_t act;
};
cudaError_t launch_fuse_weights(const FuseWeightsArgs& a, cudaStream_t s);

// Generic linear layer y[t][o] = sum_i W[o][i] x[t][i] (linear.cu).
struct LinearArgs {
  const void* x;     // [n][n_in]
  const void* w;     // [n_out][n_in]
  void* y;           // [n][n_out] act (written when part is null, or by the split sum)
  float* part;       // [k_splits][n][n_out] fp32 sums, or null (then k_splits == 1, y written directly)
  int32_t n_tokens;
  int32_t n_out;
  int32_t n_in;
  int32_t k_splits;  // from linear_splits
  mla_dtype_t act;
  int32_t w_static;  // 1: no kernel still running before this one writes W (its
                     // first ring may be requested before griddepcontrol.wait)
  int64_t x_stride;  // elements between consecutive rows of x; 0 = n_in (the
                     // tensor-core path only, a multiple of 8)
};
// K splits for these sizes on the current device (1 on the CUDA-core path),
// and the bytes of their fp32 sums [splits][n][n_out], 256-byte aligned.
int32_t linear_splits(int32_t n_tokens, int32_t n_out, int32_t n_in, mla_dtype_t act);
size_t linear_partial_bytes(int32_t n_tokens, int32_t n_out, int32_t n_in, mla_dtype_t act);
// reduce: with part set, also add the splits into y (otherwise the caller
// consumes the fp32 sums itself).
cudaError_t launch_linear(const LinearArgs& a, cudaStream_t s, bool reduce);

// Prefill in the MHA form (prefill.cu): K_nope and V expanded from the latent
// rows by the linear layer, then causal attention per head on tcgen05.
struct PrefillArgs {
  const void* q_nope;  // [Tq][H][128] bf16
  const void* q_rope;  // [Tq][H][64] bf16, rotated
  const void* rows;    // [T][576] bf16: c_KV and the rotated k_R of every token
  const void* w_uk;    // [H][128][512] bf16
  const void* w_uv;    // [H][128][512] bf16
  void* k_nope;        // workspace [T][H][128] bf16
  void* v;             // workspace [T][H][128] bf16
  void* o;             // [Tq][H][128] bf16
  float* lse;          // [Tq][H] fp32 or nullptr
  int32_t* dev_error;
  int32_t n_tokens;    // T
  int32_t n_queries;   // Tq: the last Tq positions of the sequence
  int32_t heads;
  float softmax_scale;
};
size_t prefill_workspace_bytes(int32_t n_tokens, int32_t heads);
bool prefill_supported();
cudaError_t launch_prefill(const PrefillArgs& a, cudaStream_t s);

// Decode-layer front end (front.cu).
struct FrontArgs {
  const void* h;       // [n][d_model]
  const void* w_dqkv;  // [d_cq + 512 + 64][d_model]
  const void* g_q;     // [d_cq]
  const void* g_kv;    // [512]
  const void* w_uqr;   // [H*128 + H*64][d_cq]
  const int32_t* positions;
  const float* cos_t;
  const float* sin_t;
  int32_t max_pos;
  float eps;
  int32_t n_tokens;
  int32_t d_model;
  int32_t d_cq;
  int32_t heads;
  void* q_nope;  // [n][H][128]
  void* q_rope;  // [n][H][64]
  void* c_kv;    // [n][512]
  void* k_r;     // [n][64]
  void* workspace;
  int32_t* dev_error;
  mla_dtype_t act;
};
size_t front_workspace_bytes(int32_t n_tokens, int32_t d_model, int32_t d_cq, int32_t heads, mla_dtype_t act);
cudaError_t launch_front(const FrontArgs& f, cudaStream_t s);

struct DecodeArgs {
  const void* q_lat;
  const void* q_rope;
  const void* cache;
  const float* scales;
  const int32_t* block_table;
  const int32_t* seq_lens;
  int32_t batch;
  int32_t q_len;
  int32_t max_pages;
  int64_t num_pages;
  int32_t page_size;
  float softmax_scale;
  int32_t num_splits;     // resolved, >= 1
  int32_t pages_per_split;
  float* part_u;          // [B][Lq][S][H][512] fp32 (S > 1)
  float* part_lse;        // [B][Lq][S][H] fp32 (S > 1)
  void* u_out;            // [B][Lq][H][512] act
  float* lse_out;         // [B][Lq][H] or nullptr
  int32_t* dev_error;
  int32_t heads;
  mla_dtype_t act;
  mla_dtype_t cache_dtype;
};
cudaError_t launch_decode_simt(const DecodeArgs& a, cudaStream_t s);
cudaError_t launch_decode_tc(const DecodeArgs& a, cudaStream_t s);
bool decode_tc_supported(const DecodeArgs& a);
cudaError_t launch_combine(const DecodeArgs& a, cudaStream_t s);
// Argument checks, split count and workspace size of a decode call (api.cu),
// shared by mla_decode_paged and mla_decode_paged_static_scratch so that both
// return the same errors; fills *out except the workspace pointers.
mla_status_t decode_prepare(const void* q_lat, const void* q_rope, const void* cache, const float* scales,
                            const int32_t* block_table, const int32_t* seq_lens, int32_t batch, int32_t q_len,
                            int32_t max_pages_per_seq, int64_t num_pages, int32_t page_size, float softmax_scale,
                            int32_t num_splits, void* u_out, float* lse_out, int32_t* dev_error, mla_dims_t dims,
                            mla_dtype_t act, mla_dtype_t cache_dtype, DecodeArgs* out, size_t* workspace_need);
// Sets the workspace pointers (workspace: at least the size decode_prepare
// reported, 16-byte aligned; may be null when that size is 0) and launches the
// decode kernel, then (merge) the split merge kernel; without merge the split
// partials are left in the workspace for a caller that merges them itself.
mla_status_t decode_run(DecodeArgs& a, void* workspace, cudaStream_t s, bool merge = true);

int device_sm_count();

}  // namespace mla
