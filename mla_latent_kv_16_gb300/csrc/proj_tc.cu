// tcgen05 per-head absorption contractions (bf16). Placeholder: reports
// "not supported" so the CUDA-core kernels run.
#include "launchers.h"

namespace mla {
cudaError_t launch_absorb_tc(const ProjArgs&, cudaStream_t) { return cudaErrorNotSupported; }
cudaError_t launch_out_proj_tc(const ProjArgs&, cudaStream_t) { return cudaErrorNotSupported; }
}  // namespace mla
