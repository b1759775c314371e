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
// Address: every call looks up the array's device address on the current
// device with cudaGetSymbolAddress (cheap once the module is loaded), so the
// address stays right if the context is torn down and recreated. The first
// call on a device may load the module; make it before any stream capture
// begins on that device.
//
// Sharing: every call on a device uses the same array. Calls whose kernels can
// overlap in time (different streams without ordering, or different host
// threads) race on it and corrupt each other's partials; callers must order
// them (one stream, or events). Nothing in the array needs to start at zero:
// each call writes every partial log-sum-exp it later reads (-inf for an empty
// split, and for every split of a work item whose kernel gave up on a wait and
// raised the timeout flag), and reads a partial output only where its
// log-sum-exp is finite, so stale contents from an earlier call are never used.
#include <cstdint>

#include <cuda_runtime.h>

#include "launchers.h"
#include "mla.h"

namespace {

constexpr size_t kScratchBytes = MLA_STATIC_SCRATCH_BYTES;

__device__ __align__(256) unsigned char g_decode_scratch[kScratchBytes];

}  // namespace

extern "C" {

mla_status_t mla_decode_paged_static_scratch(const void* q_lat, const void* q_rope, const void* cache,
                                             const float* scales, const int32_t* block_table,
                                             const int32_t* seq_lens, int32_t batch, int32_t q_len,
                                             int32_t max_pages_per_seq, int64_t num_pages, int32_t page_size,
                                             float softmax_scale, int32_t num_splits, void* u_out,
                                             float* lse_out, int32_t* dev_error, mla_dims_t dims,
                                             mla_dtype_t act, mla_dtype_t cache_dtype, mla_stream_t stream) {
  // The same argument checks as mla_decode_paged, first, so that both entry
  // points return the same errors; then the scratch size, before any device work.
  mla::DecodeArgs a{};
  size_t need = 0;
  const mla_status_t st =
      mla::decode_prepare(q_lat, q_rope, cache, scales, block_table, seq_lens, batch, q_len, max_pages_per_seq,
                          num_pages, page_size, softmax_scale, num_splits, u_out, lse_out, dev_error, dims, act,
                          cache_dtype, &a, &need);
  if (st != MLA_OK || batch == 0) return st;
  if (need > kScratchBytes) return MLA_ERR_WORKSPACE_TOO_SMALL;
  void* scratch = nullptr;
  if (need > 0 && cudaGetSymbolAddress(&scratch, g_decode_scratch) != cudaSuccess) return MLA_ERR_CUDA;
  return mla::decode_run(a, scratch, static_cast<cudaStream_t>(stream));
}

}  // extern "C"
