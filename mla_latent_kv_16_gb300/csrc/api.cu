// C ABI entry points (include/mla.h): argument validation, split policy and
// dispatch to the sm_103a kernels. No allocation happens here; every buffer is
// the caller's.
#include <cmath>
#include <cstdint>
#include <cstring>

#include "launchers.h"
#include "mla.h"

namespace mla {

int device_sm_count() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    cached[dev] = n;
  }
  return cached[dev];
}

namespace {

constexpr int32_t kMaxTokens = 1 << 20;
constexpr int32_t kMaxBatchQ = 65535;
constexpr int32_t kMaxDModel = 1 << 16;
constexpr int32_t kMaxLinearDim = 1 << 20;
constexpr int32_t kMaxPrefillTokens = 1 << 20;

bool dims_ok(const mla_dims_t& d) {
  return d.d_nope == 128 && d.d_c == 512 && d.d_rope == 64 && d.d_v == 128 && d.num_heads >= 1 &&
         d.num_heads <= 128;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

mla_status_t from_cuda(cudaError_t e) { return e == cudaSuccess ? MLA_OK : MLA_ERR_CUDA; }

bool use_tc_decode(int32_t heads, int32_t page_size, mla_dtype_t act, mla_dtype_t cache_dtype) {
  return heads == 128 && act == MLA_BF16 && (cache_dtype == MLA_BF16 || cache_dtype == MLA_E4M3) &&
         page_size % 64 == 0;
}

// Work items of one split: the SIMT kernel runs ceil(H/8) CTAs per (b, j, split);
// the tcgen05 kernel one CTA pair.
int32_t resolve_splits(int32_t batch, int32_t q_len, int32_t max_pages, int32_t page_size,
                       int32_t requested, const mla_dims_t& d, mla_dtype_t cache_dtype) {
  if (batch < 0 || q_len < 1 || max_pages < 1 || page_size < 1 || requested < 0 || !dims_ok(d)) return 0;
  if (requested > 0) return requested > max_pages ? max_pages : requested;
  const bool tc = use_tc_decode(d.num_heads, page_size, MLA_BF16, cache_dtype);
  const int sms = device_sm_count();
  const int64_t slots = tc ? sms / 2 : sms * 2;            // concurrent work items
  const int64_t per_item = tc ? 1 : (d.num_heads + 7) / 8;
  const int64_t items0 = static_cast<int64_t>(batch > 0 ? batch : 1) * q_len * per_item;
  // Cost in the time one work item takes per page (measured on GB300 for the
  // tensor-core kernel: ~1.6 us per 64-token bf16 page, ~1.9x that for E4M3, and
  // ~8 us = 5 pages of set-up and epilogue per item):
  //   waves x (pages per split + item overhead)
  //   + the split partials' HBM traffic, written by the decode and read by the
  //     merge (B Lq S H 513 x 4 bytes each way), at 6.8 TB/s
  const double item_cost = tc ? 5.0 : 0.5;
  const double page_us =
      tc ? 1.6 * (page_size / 64.0) * (cache_dtype == MLA_E4M3 ? 1.9 : 1.0) : 1.0;
  const double part_bytes_per_split =
      2.0 * static_cast<double>(batch > 0 ? batch : 1) * q_len * d.num_heads * (512 + 1) * 4.0;  // u (512 fp32) + lse
  int32_t best = 1;
  double best_cost = 1e300;
  const int32_t smax = max_pages < 256 ? max_pages : 256;
  for (int32_t s = 1; s <= smax; ++s) {
    const int64_t pps = (max_pages + s - 1) / s;
    const int32_t s_eff = static_cast<int32_t>((max_pages + pps - 1) / pps);
    if (s_eff != s) continue;
    const int64_t waves = (items0 * s + slots - 1) / slots;
    const double part_pages = s > 1 ? part_bytes_per_split * s / 6.8e6 / page_us : 0.0;
    const double cost = static_cast<double>(waves) * (static_cast<double>(pps) + item_cost) + part_pages;
    if (cost < best_cost - 1e-9) {
      best_cost = cost;
      best = s;
    }
  }
  return best;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

size_t workspace_bytes_for(int32_t batch, int32_t q_len, int32_t splits, int32_t heads) {
  if (splits <= 1) return 0;
  const size_t rows = static_cast<size_t>(batch) * q_len * splits * heads;
  return align256(rows * 512 * sizeof(float)) + align256(rows * sizeof(float));
}

}  // namespace

mla_status_t decode_prepare(const void* q_lat, const void* q_rope, const void* cache, const float* scales,
                            const int32_t* block_table, const int32_t* seq_lens, int32_t batch, int32_t q_len,
                            int32_t max_pages_per_seq, int64_t num_pages, int32_t page_size, float softmax_scale,
                            int32_t num_splits, void* u_out, float* lse_out, int32_t* dev_error, mla_dims_t dims,
                            mla_dtype_t act, mla_dtype_t cache_dtype, DecodeArgs* out, size_t* workspace_need) {
  if (!dims_ok(dims) || batch < 0 || q_len < 1 || static_cast<int64_t>(batch) * q_len > kMaxBatchQ ||
      max_pages_per_seq < 1 || num_pages < 1 || page_size < 1 || num_splits < 0 || !std::isfinite(softmax_scale))
    return MLA_ERR_INVALID_ARG;
  if (act != MLA_F32 && act != MLA_BF16) return MLA_ERR_UNSUPPORTED;
  if (!(cache_dtype == act || (cache_dtype == MLA_E4M3 && act == MLA_BF16))) return MLA_ERR_UNSUPPORTED;
  if ((cache_dtype == MLA_E4M3) != (scales != nullptr)) return MLA_ERR_INVALID_ARG;
  if (static_cast<int64_t>(max_pages_per_seq) * page_size > (int64_t(1) << 30)) return MLA_ERR_INVALID_ARG;
  *workspace_need = 0;
  if (batch == 0) return MLA_OK;
  if (q_lat == nullptr || q_rope == nullptr || cache == nullptr || block_table == nullptr || seq_lens == nullptr ||
      u_out == nullptr)
    return MLA_ERR_INVALID_ARG;
  if (!aligned16(q_lat) || !aligned16(q_rope) || !aligned16(cache) || !aligned16(u_out))
    return MLA_ERR_INVALID_ARG;
  const int32_t S = resolve_splits(batch, q_len, max_pages_per_seq, page_size, num_splits, dims, cache_dtype);
  if (S < 1) return MLA_ERR_INVALID_ARG;
  DecodeArgs& a = *out;
  a = DecodeArgs{};
  a.q_lat = q_lat;
  a.q_rope = q_rope;
  a.cache = cache;
  a.scales = scales;
  a.block_table = block_table;
  a.seq_lens = seq_lens;
  a.batch = batch;
  a.q_len = q_len;
  a.max_pages = max_pages_per_seq;
  a.num_pages = num_pages;
  a.page_size = page_size;
  a.softmax_scale = softmax_scale;
  a.num_splits = S;
  a.pages_per_split = (max_pages_per_seq + S - 1) / S;
  a.u_out = u_out;
  a.lse_out = lse_out;
  a.dev_error = dev_error;
  a.heads = dims.num_heads;
  a.act = act;
  a.cache_dtype = cache_dtype;
  *workspace_need = workspace_bytes_for(batch, q_len, S, dims.num_heads);
  return MLA_OK;
}

mla_status_t decode_run(DecodeArgs& a, void* workspace, cudaStream_t s, bool merge) {
  const size_t rows = static_cast<size_t>(a.batch) * a.q_len * a.num_splits * a.heads;
  a.part_u = workspace != nullptr ? static_cast<float*>(workspace) : nullptr;
  a.part_lse = workspace != nullptr
                   ? reinterpret_cast<float*>(static_cast<char*>(workspace) + align256(rows * 512 * sizeof(float)))
                   : nullptr;
  cudaError_t e;
  if (use_tc_decode(a.heads, a.page_size, a.act, a.cache_dtype) && decode_tc_supported(a))
    e = launch_decode_tc(a, s);
  else
    e = launch_decode_simt(a, s);
  if (e != cudaSuccess) return MLA_ERR_CUDA;
  if (!merge) return MLA_OK;
  return from_cuda(launch_combine(a, s));
}

}  // namespace mla

using namespace mla;

extern "C" {

const char* mla_status_string(mla_status_t s) {
  switch (s) {
    case MLA_OK: return "MLA_OK";
    case MLA_ERR_INVALID_ARG: return "MLA_ERR_INVALID_ARG";
    case MLA_ERR_UNSUPPORTED: return "MLA_ERR_UNSUPPORTED";
    case MLA_ERR_CUDA: return "MLA_ERR_CUDA";
    case MLA_ERR_WORKSPACE_TOO_SMALL: return "MLA_ERR_WORKSPACE_TOO_SMALL";
    case MLA_ERR_DEVICE_FLAG: return "MLA_ERR_DEVICE_FLAG";
  }
  return "MLA_ERR_UNKNOWN";
}

int32_t mla_version(void) { return 100; }

mla_status_t mla_rope_table(int32_t max_pos, int32_t d_rope, double base, float* cos_out, float* sin_out) {
  if (max_pos < 1 || d_rope < 2 || (d_rope & 1) || !(base > 0.0) || cos_out == nullptr || sin_out == nullptr)
    return MLA_ERR_INVALID_ARG;
  const int half = d_rope / 2;
  for (int i = 0; i < half; ++i) {
    const double theta = std::pow(base, -(2.0 * i) / static_cast<double>(d_rope));
    for (int32_t p = 0; p < max_pos; ++p) {
      const double ang = static_cast<double>(p) * theta;
      cos_out[static_cast<int64_t>(p) * half + i] = static_cast<float>(std::cos(ang));
      sin_out[static_cast<int64_t>(p) * half + i] = static_cast<float>(std::sin(ang));
    }
  }
  return MLA_OK;
}

mla_status_t mla_cache_append(const void* c_kv, const void* k_r, const int32_t* positions,
                              const int64_t* slot_mapping, const float* rope_cos, const float* rope_sin,
                              int32_t n_tokens, int32_t max_pos, void* cache, float* scales, int64_t num_pages,
                              int32_t page_size, mla_dtype_t in_dtype, mla_dtype_t cache_dtype,
                              int32_t* dev_error, mla_stream_t stream) {
  if (n_tokens < 0 || n_tokens > kMaxTokens || max_pos < 1 || num_pages < 1 || page_size < 1)
    return MLA_ERR_INVALID_ARG;
  if (in_dtype != MLA_F32 && in_dtype != MLA_BF16) return MLA_ERR_UNSUPPORTED;
  if (cache_dtype != MLA_F32 && cache_dtype != MLA_BF16 && cache_dtype != MLA_E4M3) return MLA_ERR_UNSUPPORTED;
  if ((cache_dtype == MLA_E4M3) != (scales != nullptr)) return MLA_ERR_INVALID_ARG;
  if (cache == nullptr || rope_cos == nullptr || rope_sin == nullptr) return MLA_ERR_INVALID_ARG;
  if (n_tokens > 0 && (c_kv == nullptr || k_r == nullptr || positions == nullptr || slot_mapping == nullptr))
    return MLA_ERR_INVALID_ARG;
  if (!aligned16(c_kv) || !aligned16(k_r) || !aligned16(cache) || (reinterpret_cast<uintptr_t>(k_r) & 7))
    return MLA_ERR_INVALID_ARG;
  AppendArgs a{c_kv, k_r, positions, slot_mapping, rope_cos, rope_sin, n_tokens, max_pos, cache, scales,
               num_pages * static_cast<int64_t>(page_size), in_dtype, cache_dtype, dev_error};
  return from_cuda(launch_append(a, static_cast<cudaStream_t>(stream)));
}

mla_status_t mla_absorb_q(const void* q_nope, const void* w_uk, void* q_lat, int32_t n_tokens, mla_dims_t dims,
                          mla_dtype_t act, mla_stream_t stream) {
  if (!dims_ok(dims) || n_tokens < 0 || n_tokens > kMaxTokens) return MLA_ERR_INVALID_ARG;
  if (act != MLA_F32 && act != MLA_BF16) return MLA_ERR_UNSUPPORTED;
  if (n_tokens == 0) return MLA_OK;
  if (q_nope == nullptr || w_uk == nullptr || q_lat == nullptr) return MLA_ERR_INVALID_ARG;
  if (!aligned16(q_nope) || !aligned16(w_uk) || !aligned16(q_lat)) return MLA_ERR_INVALID_ARG;
  ProjArgs a{q_nope, w_uk, q_lat, n_tokens, dims.num_heads, act};
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (act == MLA_BF16) {
    cudaError_t e = launch_absorb_tc(a, s);
    if (e != cudaErrorNotSupported) return from_cuda(e);
  }
  return from_cuda(launch_absorb_simt(a, s));
}

mla_status_t mla_out_proj(const void* u, const void* w_uv, void* o, int32_t n_tokens, mla_dims_t dims,
                          mla_dtype_t act, mla_stream_t stream) {
  if (!dims_ok(dims) || n_tokens < 0 || n_tokens > kMaxTokens) return MLA_ERR_INVALID_ARG;
  if (act != MLA_F32 && act != MLA_BF16) return MLA_ERR_UNSUPPORTED;
  if (n_tokens == 0) return MLA_OK;
  if (u == nullptr || w_uv == nullptr || o == nullptr) return MLA_ERR_INVALID_ARG;
  if (!aligned16(u) || !aligned16(w_uv) || !aligned16(o)) return MLA_ERR_INVALID_ARG;
  ProjArgs a{u, w_uv, o, n_tokens, dims.num_heads, act};
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (act == MLA_BF16) {
    cudaError_t e = launch_out_proj_tc(a, s);
    if (e != cudaErrorNotSupported) return from_cuda(e);
  }
  return from_cuda(launch_out_proj_simt(a, s));
}

mla_status_t mla_fuse_out_weights(const void* w_o, const void* w_uv, void* w_fused, int32_t d_model,
                                  mla_dims_t dims, mla_dtype_t act, mla_stream_t stream) {
  if (!dims_ok(dims) || d_model < 1 || d_model > kMaxDModel) return MLA_ERR_INVALID_ARG;
  if (act != MLA_F32 && act != MLA_BF16) return MLA_ERR_UNSUPPORTED;
  if (w_o == nullptr || w_uv == nullptr || w_fused == nullptr) return MLA_ERR_INVALID_ARG;
  if (!aligned16(w_o) || !aligned16(w_uv) || !aligned16(w_fused)) return MLA_ERR_INVALID_ARG;
  FuseWeightsArgs a{w_o, w_uv, w_fused, d_model, dims.num_heads, act};
  return from_cuda(launch_fuse_weights(a, static_cast<cudaStream_t>(stream)));
}

size_t mla_linear_workspace_size(int32_t n_tokens, int32_t n_out, int32_t n_in, mla_dtype_t act) {
  if (n_tokens < 1 || n_tokens > kMaxTokens || n_out < 1 || n_out > kMaxLinearDim || n_in < 1 ||
      n_in > kMaxLinearDim)
    return 0;
  if (act != MLA_F32 && act != MLA_BF16) return 0;
  if (linear_splits(n_tokens, n_out, n_in, act) <= 1) return 0;
  return linear_partial_bytes(n_tokens, n_out, n_in, act);
}

mla_status_t mla_linear(const void* x, const void* w, void* y, int32_t n_tokens, int32_t n_out, int32_t n_in,
                        void* workspace, size_t workspace_bytes, mla_dtype_t act, mla_stream_t stream) {
  if (n_tokens < 0 || n_tokens > kMaxTokens || n_out < 1 || n_out > kMaxLinearDim || n_in < 1 ||
      n_in > kMaxLinearDim)
    return MLA_ERR_INVALID_ARG;
  if (act != MLA_F32 && act != MLA_BF16) return MLA_ERR_UNSUPPORTED;
  if (n_tokens == 0) return MLA_OK;
  if (x == nullptr || w == nullptr || y == nullptr) return MLA_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(w) || !aligned16(y)) return MLA_ERR_INVALID_ARG;
  const int32_t splits = linear_splits(n_tokens, n_out, n_in, act);
  const size_t need = splits > 1 ? linear_partial_bytes(n_tokens, n_out, n_in, act) : 0;
  if (need > 0 && (workspace == nullptr || workspace_bytes < need)) return MLA_ERR_WORKSPACE_TOO_SMALL;
  if (need > 0 && !aligned16(workspace)) return MLA_ERR_INVALID_ARG;
  // W may be the output of mla_fuse_out_weights just before: nothing is read before the wait
  LinearArgs a{x, w, y, need > 0 ? static_cast<float*>(workspace) : nullptr, n_tokens, n_out, n_in, splits, act, 0};
  return from_cuda(launch_linear(a, static_cast<cudaStream_t>(stream), true));
}

size_t mla_out_proj_fused_workspace_size(int32_t n_tokens, int32_t d_model, mla_dims_t dims, mla_dtype_t act) {
  if (!dims_ok(dims) || d_model > kMaxDModel) return 0;
  return mla_linear_workspace_size(n_tokens, d_model, dims.num_heads * dims.d_c, act);
}

mla_status_t mla_out_proj_fused(const void* u, const void* w_fused, void* y, int32_t n_tokens, int32_t d_model,
                                void* workspace, size_t workspace_bytes, mla_dims_t dims, mla_dtype_t act,
                                mla_stream_t stream) {
  if (!dims_ok(dims) || d_model < 1 || d_model > kMaxDModel) return MLA_ERR_INVALID_ARG;
  return mla_linear(u, w_fused, y, n_tokens, d_model, dims.num_heads * dims.d_c, workspace, workspace_bytes, act,
                    stream);
}

size_t mla_decode_front_workspace_size(int32_t n_tokens, int32_t d_model, int32_t d_cq, mla_dims_t dims,
                                       mla_dtype_t act) {
  if (!dims_ok(dims) || n_tokens < 1 || n_tokens > kMaxTokens || d_model < 1 || d_model > kMaxDModel ||
      d_cq < 1 || d_cq > kMaxDModel)
    return 0;
  if (act != MLA_F32 && act != MLA_BF16) return 0;
  return front_workspace_bytes(n_tokens, d_model, d_cq, dims.num_heads, act);
}

mla_status_t mla_decode_front(const void* h, const void* w_dqkv, const void* g_q, const void* g_kv,
                              const void* w_uqr, const int32_t* positions, const float* rope_cos,
                              const float* rope_sin, int32_t max_pos, float eps, int32_t n_tokens, int32_t d_model,
                              int32_t d_cq, void* q_nope, void* q_rope, void* c_kv, void* k_r, void* workspace,
                              size_t workspace_bytes, int32_t* dev_error, mla_dims_t dims, mla_dtype_t act,
                              mla_stream_t stream) {
  if (!dims_ok(dims) || n_tokens < 0 || n_tokens > kMaxTokens || d_model < 1 || d_model > kMaxDModel || d_cq < 1 ||
      d_cq > kMaxDModel || max_pos < 1 || !std::isfinite(eps) || eps < 0.0f)
    return MLA_ERR_INVALID_ARG;
  if (act != MLA_F32 && act != MLA_BF16) return MLA_ERR_UNSUPPORTED;
  if (n_tokens == 0) return MLA_OK;
  const void* ptrs[] = {h, w_dqkv, g_q, g_kv, w_uqr, positions, rope_cos, rope_sin, q_nope, q_rope, c_kv, k_r};
  for (const void* p : ptrs)
    if (p == nullptr) return MLA_ERR_INVALID_ARG;
  const void* aligned[] = {h, w_dqkv, w_uqr, q_nope, q_rope, c_kv, k_r};
  for (const void* p : aligned)
    if (!aligned16(p)) return MLA_ERR_INVALID_ARG;
  const size_t need = front_workspace_bytes(n_tokens, d_model, d_cq, dims.num_heads, act);
  if (workspace == nullptr || workspace_bytes < need) return MLA_ERR_WORKSPACE_TOO_SMALL;
  if (!aligned16(workspace)) return MLA_ERR_INVALID_ARG;
  FrontArgs f{h, w_dqkv, g_q, g_kv, w_uqr, positions, rope_cos, rope_sin, max_pos, eps, n_tokens, d_model, d_cq,
              dims.num_heads, q_nope, q_rope, c_kv, k_r, workspace, dev_error, act};
  return from_cuda(launch_front(f, static_cast<cudaStream_t>(stream)));
}

int32_t mla_decode_num_splits(int32_t batch, int32_t q_len, int32_t max_pages_per_seq, int32_t page_size,
                              int32_t num_splits, mla_dims_t dims, mla_dtype_t cache_dtype) {
  return resolve_splits(batch, q_len, max_pages_per_seq, page_size, num_splits, dims, cache_dtype);
}

size_t mla_decode_workspace_size(int32_t batch, int32_t q_len, int32_t max_pages_per_seq, int32_t page_size,
                                 int32_t num_splits, mla_dims_t dims, mla_dtype_t cache_dtype) {
  const int32_t s = resolve_splits(batch, q_len, max_pages_per_seq, page_size, num_splits, dims, cache_dtype);
  if (s < 1 || batch < 0) return 0;
  return workspace_bytes_for(batch, q_len, s, dims.num_heads);
}

mla_status_t mla_decode_paged(const void* q_lat, const void* q_rope, const void* cache, const float* scales,
                              const int32_t* block_table, const int32_t* seq_lens, int32_t batch, int32_t q_len,
                              int32_t max_pages_per_seq, int64_t num_pages, int32_t page_size, float softmax_scale,
                              int32_t num_splits, void* workspace, size_t workspace_bytes, void* u_out,
                              float* lse_out, int32_t* dev_error, mla_dims_t dims, mla_dtype_t act,
                              mla_dtype_t cache_dtype, mla_stream_t stream) {
  DecodeArgs a{};
  size_t need = 0;
  const mla_status_t st = decode_prepare(q_lat, q_rope, cache, scales, block_table, seq_lens, batch, q_len,
                                         max_pages_per_seq, num_pages, page_size, softmax_scale, num_splits, u_out,
                                         lse_out, dev_error, dims, act, cache_dtype, &a, &need);
  if (st != MLA_OK || batch == 0) return st;
  if (need > 0 && (workspace == nullptr || workspace_bytes < need)) return MLA_ERR_WORKSPACE_TOO_SMALL;
  if (need > 0 && !aligned16(workspace)) return MLA_ERR_INVALID_ARG;
  return decode_run(a, need > 0 ? workspace : nullptr, static_cast<cudaStream_t>(stream));
}

mla_status_t mla_decode_out_proj(const void* q_lat, const void* q_rope, const void* cache, const float* scales,
                                 const int32_t* block_table, const int32_t* seq_lens, int32_t batch, int32_t q_len,
                                 int32_t max_pages_per_seq, int64_t num_pages, int32_t page_size,
                                 float softmax_scale, int32_t num_splits, void* workspace, size_t workspace_bytes,
                                 const void* w_uv, void* u_out, float* lse_out, void* o_out, int32_t* dev_error,
                                 mla_dims_t dims, mla_dtype_t act, mla_dtype_t cache_dtype, mla_stream_t stream) {
  DecodeArgs a{};
  size_t need = 0;
  const mla_status_t st = decode_prepare(q_lat, q_rope, cache, scales, block_table, seq_lens, batch, q_len,
                                         max_pages_per_seq, num_pages, page_size, softmax_scale, num_splits, u_out,
                                         lse_out, dev_error, dims, act, cache_dtype, &a, &need);
  if (st != MLA_OK || batch == 0) return st;
  if (w_uv == nullptr || o_out == nullptr || !aligned16(w_uv) || !aligned16(o_out)) return MLA_ERR_INVALID_ARG;
  if (need > 0 && (workspace == nullptr || workspace_bytes < need)) return MLA_ERR_WORKSPACE_TOO_SMALL;
  if (need > 0 && !aligned16(workspace)) return MLA_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int32_t n = batch * q_len;
  // the split merge inside the projection when the decode runs on the tensor cores with 2..4 splits
  const bool fused = a.num_splits >= 2 && use_tc_decode(a.heads, a.page_size, a.act, a.cache_dtype) &&
                     decode_tc_supported(a) && out_proj_merge_supported(a.heads, a.num_splits, act);
  const mla_status_t sd = decode_run(a, need > 0 ? workspace : nullptr, s, !fused);
  if (sd != MLA_OK) return sd;
  if (fused) {
    const MergeProjArgs m{a.part_u, a.part_lse, a.num_splits, w_uv, u_out, lse_out, o_out, n, a.heads};
    return from_cuda(launch_out_proj_merge_tc(m, s));
  }
  return mla_out_proj(u_out, w_uv, o_out, n, dims, act, stream);
}

mla_status_t mla_decode_kernel_path(const void* cache, const float* scales, int64_t num_pages, int32_t page_size,
                                    mla_dims_t dims, mla_dtype_t act, mla_dtype_t cache_dtype, int32_t* path_out) {
  if (path_out == nullptr || !dims_ok(dims) || num_pages < 1 || page_size < 1) return MLA_ERR_INVALID_ARG;
  DecodeArgs a{};
  a.cache = cache;
  a.scales = scales;
  a.num_pages = num_pages;
  a.page_size = page_size;
  a.heads = dims.num_heads;
  a.act = act;
  a.cache_dtype = cache_dtype;
  *path_out = (use_tc_decode(dims.num_heads, page_size, act, cache_dtype) && decode_tc_supported(a))
                  ? MLA_DECODE_PATH_TENSOR_CORE
                  : MLA_DECODE_PATH_CUDA_CORE;
  return MLA_OK;
}

size_t mla_prefill_workspace_size(int32_t n_tokens, mla_dims_t dims) {
  if (!dims_ok(dims) || n_tokens < 1 || n_tokens > kMaxPrefillTokens) return 0;
  return prefill_workspace_bytes(n_tokens, dims.num_heads);
}

mla_status_t mla_prefill_mha(const void* q_nope, const void* q_rope, const void* rows, const void* w_uk,
                             const void* w_uv, int32_t n_tokens, int32_t n_queries, float softmax_scale,
                             void* workspace, size_t workspace_bytes, void* o_out, float* lse_out,
                             int32_t* dev_error, mla_dims_t dims, mla_dtype_t act, mla_stream_t stream) {
  if (!dims_ok(dims) || n_tokens < 1 || n_tokens > kMaxPrefillTokens || n_queries < 1 || n_queries > n_tokens ||
      !std::isfinite(softmax_scale))
    return MLA_ERR_INVALID_ARG;
  if (act != MLA_BF16) return MLA_ERR_UNSUPPORTED;
  const void* ptrs[] = {q_nope, q_rope, rows, w_uk, w_uv, o_out, workspace};
  for (const void* p : ptrs)
    if (p == nullptr) return p == workspace ? MLA_ERR_WORKSPACE_TOO_SMALL : MLA_ERR_INVALID_ARG;
  for (const void* p : ptrs)
    if (!aligned16(p)) return MLA_ERR_INVALID_ARG;
  const size_t need = prefill_workspace_bytes(n_tokens, dims.num_heads);
  if (workspace_bytes < need) return MLA_ERR_WORKSPACE_TOO_SMALL;
  if (!prefill_supported()) return MLA_ERR_UNSUPPORTED;
  PrefillArgs a{};
  a.q_nope = q_nope;
  a.q_rope = q_rope;
  a.rows = rows;
  a.w_uk = w_uk;
  a.w_uv = w_uv;
  a.k_nope = workspace;
  a.v = static_cast<char*>(workspace) + need / 2;
  a.o = o_out;
  a.lse = lse_out;
  a.dev_error = dev_error;
  a.n_tokens = n_tokens;
  a.n_queries = n_queries;
  a.heads = dims.num_heads;
  a.softmax_scale = softmax_scale;
  return from_cuda(launch_prefill(a, static_cast<cudaStream_t>(stream)));
}

mla_status_t mla_read_device_error(const int32_t* dev_error, mla_stream_t stream, int32_t* code_out) {
  if (dev_error == nullptr || code_out == nullptr) return MLA_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t v = 0;
  if (cudaMemcpyAsync(&v, dev_error, sizeof(int32_t), cudaMemcpyDeviceToHost, s) != cudaSuccess) return MLA_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MLA_ERR_CUDA;
  *code_out = v;
  return v != 0 ? MLA_ERR_DEVICE_FLAG : MLA_OK;
}

}  // extern "C"
