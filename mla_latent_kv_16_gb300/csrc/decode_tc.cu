// tcgen05 paged decode (bf16 / E4M3 cache, 128 heads). Placeholder.
#include "launchers.h"

namespace mla {
bool decode_tc_supported(const DecodeArgs&) { return false; }
cudaError_t launch_decode_tc(const DecodeArgs&, cudaStream_t) { return cudaErrorNotSupported; }
}  // namespace mla
