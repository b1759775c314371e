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

struct FuseWeightsArgs {
  const void* w_o;   // [d][H][128]
  const void* w_uv;  // [H][128][512]
  void* w_fused;     // [d][H][512]
  int32_t d_model;
  int32_t heads;
  mla_dtype_t act;
};
cudaError_t launch_fuse_weights(const FuseWeightsArgs& a, cudaStream_t s);

struct FusedOutArgs {
  const void* u;     // [n][H][512]
  const void* w;     // W~ [d][H][512]
  void* y;           // [n][d]
  float* part;       // [k_splits][n][d] fp32 partial sums (k_splits > 1)
  int32_t n_tokens;
  int32_t d_model;
  int32_t heads;
  int32_t k_splits;  // from out_fused_splits
  mla_dtype_t act;
};
// K splits of the fused output projection for these sizes on the current
// device (1 on the CUDA-core path), and the workspace bytes they need.
int32_t out_fused_splits(int32_t n_tokens, int32_t d_model, int32_t heads, mla_dtype_t act);
size_t out_fused_workspace_bytes(int32_t n_tokens, int32_t d_model, int32_t heads, mla_dtype_t act);
cudaError_t launch_out_fused(const FusedOutArgs& a, cudaStream_t s);

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

int device_sm_count();

}  // namespace mla
