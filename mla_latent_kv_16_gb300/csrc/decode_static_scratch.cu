// mla_decode_paged_static_scratch: the paged decode with its split-KV scratch
// in a fixed device array of this library instead of a caller workspace.
//
// Some callers cannot hand over device memory at call time: a host runtime
// that owns no allocator of its own (a plain C or Fortran host with no CUDA
// memory pool), or code that must not allocate once serving has started
// because an allocation can synchronise the device and stall every stream.
// This entry point serves them: the fp32 partial outputs and log-sum-exps of
// the split-KV path live in one file-scope __device__ array created when the
// library's module is loaded, so the call itself allocates and frees nothing.
//
// Set-up: the first call on each device (with that device current) looks up
// the array's device address with cudaGetSymbolAddress and caches it for the
// device; later calls reuse the cached address. Make that first call before
// any stream capture begins on the device, because the look-up may load the
// module.
//
// Sharing: every call on a device uses the same array. Calls whose kernels can
// overlap in time (different streams without ordering, or different host
// threads) race on it and corrupt each other's partials; callers must order
// them (one stream, or events). Nothing in the array needs to start at zero:
// each call writes every partial log-sum-exp it later reads (-inf for an empty
// split), and reads a partial output only where its log-sum-exp is finite, so
// stale contents from an earlier call are never used.
#include <atomic>
#include <cstdint>

#include <cuda_runtime.h>

#include "mla.h"

namespace {

constexpr size_t kScratchBytes = MLA_STATIC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_decode_scratch[kScratchBytes];

std::atomic<void*> g_scratch_ptr[kMaxDevices];

// Device address of g_decode_scratch on the current device (looked up once).
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  void* p = g_scratch_ptr[dev].load(std::memory_order_acquire);
  if (p == nullptr) {
    e = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev].store(p, std::memory_order_release);
  }
  *out = p;
  return cudaSuccess;
}

}  // namespace

extern "C" {

mla_status_t mla_decode_paged_static_scratch(const void* q_lat, const void* q_rope, const void* cache,
                                             const float* scales, const int32_t* block_table,
                                             const int32_t* seq_lens, int32_t batch, int32_t q_len,
                                             int32_t max_pages_per_seq, int64_t num_pages, int32_t page_size,
                                             float softmax_scale, int32_t num_splits, void* u_out,
                                             float* lse_out, int32_t* dev_error, mla_dims_t dims,
                                             mla_dtype_t act, mla_dtype_t cache_dtype, mla_stream_t stream) {
  // Same argument checks as mla_decode_paged, done there; only the scratch
  // size is decided here, before any device work.
  if (mla_decode_num_splits(batch, q_len, max_pages_per_seq, page_size, num_splits, dims, cache_dtype) < 1)
    return MLA_ERR_INVALID_ARG;
  const size_t need =
      mla_decode_workspace_size(batch, q_len, max_pages_per_seq, page_size, num_splits, dims, cache_dtype);
  if (need > kScratchBytes) return MLA_ERR_WORKSPACE_TOO_SMALL;
  void* scratch = nullptr;
  if (scratch_address(&scratch) != cudaSuccess) return MLA_ERR_CUDA;
  return mla_decode_paged(q_lat, q_rope, cache, scales, block_table, seq_lens, batch, q_len, max_pages_per_seq,
                          num_pages, page_size, softmax_scale, num_splits, scratch, need > 0 ? kScratchBytes : 0,
                          u_out, lse_out, dev_error, dims, act, cache_dtype, stream);
}

}  // extern "C"
