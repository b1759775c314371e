// Per-head absorption contractions on CUDA cores (fp32 accumulate).
//
//   absorb  : q_lat[t,h,c] = sum_d q_nope[t,h,d] W_UK[h,d,c]   ("Model Architecture
//             Driving Inference Systems" §3.1, absorbed query (W_UK)^T q)
//   out_proj: o[t,h,d]     = sum_c u[t,h,c] W_UV[h,d,c]       (same page, §3.2)
//
// These are the general-dtype kernels (fp32 activations, any head count). The
// bf16 path uses the tcgen05 kernels in proj_tc.cu.
#include "common.cuh"
#include "launchers.h"

namespace mla {
namespace {

constexpr int kAbsorbTok = 32;  // tokens per CTA
constexpr int kOutTok = 16;

// grid (512/128, H, ceil(n/32)), block 128: thread = one latent column c.
template <typename T>
__global__ void __launch_bounds__(128) absorb_simt_kernel(ProjArgs a) {
  pdl_trigger();
  pdl_wait();
  __shared__ float qs[kAbsorbTok][kDNope];
  const int c = blockIdx.x * 128 + threadIdx.x;
  const int h = blockIdx.y;
  const int t0 = blockIdx.z * kAbsorbTok;
  const T* q = static_cast<const T*>(a.x);
  const T* w = static_cast<const T*>(a.w) + static_cast<int64_t>(h) * kDNope * kDC;
  for (int i = threadIdx.x; i < kAbsorbTok * kDNope; i += 128) {
    const int t = i / kDNope, d = i % kDNope;
    qs[t][d] = (t0 + t < a.n_tokens)
                   ? ActIO<T>::load(q + (static_cast<int64_t>(t0 + t) * a.heads + h) * kDNope + d)
                   : 0.0f;
  }
  __syncthreads();
  float acc[kAbsorbTok];
#pragma unroll
  for (int t = 0; t < kAbsorbTok; ++t) acc[t] = 0.0f;
  // 16 rows of W_UK requested at once: 8 memory round trips per thread, not 128
  for (int d0 = 0; d0 < kDNope; d0 += 16) {
    float wv[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) wv[i] = ActIO<T>::load(w + (d0 + i) * kDC + c);
#pragma unroll
    for (int i = 0; i < 16; ++i)
#pragma unroll
      for (int t = 0; t < kAbsorbTok; ++t) acc[t] = fmaf(qs[t][d0 + i], wv[i], acc[t]);
  }
  T* y = static_cast<T*>(a.y);
#pragma unroll
  for (int t = 0; t < kAbsorbTok; ++t)
    if (t0 + t < a.n_tokens) ActIO<T>::store(y + (static_cast<int64_t>(t0 + t) * a.heads + h) * kDC + c, acc[t]);
}

// grid (H, ceil(n/16)), block 128 (4 warps). Warp w computes rows d = w, w+4, ...
// Lane l owns latent columns l + 32 i.
template <typename T>
__global__ void __launch_bounds__(128) out_proj_simt_kernel(ProjArgs a) {
  pdl_trigger();
  pdl_wait();
  __shared__ float us[kOutTok][kDC];
  const int h = blockIdx.x;
  const int t0 = blockIdx.y * kOutTok;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const T* u = static_cast<const T*>(a.x);
  const T* w = static_cast<const T*>(a.w) + static_cast<int64_t>(h) * kDV * kDC;
  for (int i = threadIdx.x; i < kOutTok * kDC; i += 128) {
    const int t = i / kDC, c = i % kDC;
    us[t][c] = (t0 + t < a.n_tokens)
                   ? ActIO<T>::load(u + (static_cast<int64_t>(t0 + t) * a.heads + h) * kDC + c)
                   : 0.0f;
  }
  __syncthreads();
  T* y = static_cast<T*>(a.y);
  // four rows of W_UV per warp requested at once (64 loads in flight per lane)
  for (int d0 = warp; d0 < kDV; d0 += 16) {
    float wr[4][16];
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int i = 0; i < 16; ++i) wr[r][i] = ActIO<T>::load(w + (d0 + 4 * r) * kDC + lane + 32 * i);
    for (int t = 0; t < kOutTok && t0 + t < a.n_tokens; ++t) {
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        float p = 0.0f;
#pragma unroll
        for (int i = 0; i < 16; ++i) p = fmaf(wr[r][i], us[t][lane + 32 * i], p);
        p = warp_sum(p);
        if (lane == 0) ActIO<T>::store(y + (static_cast<int64_t>(t0 + t) * a.heads + h) * kDV + d0 + 4 * r, p);
      }
    }
  }
}

}  // namespace

cudaError_t launch_absorb_simt(const ProjArgs& a, cudaStream_t s) {
  if (a.n_tokens == 0) return cudaSuccess;
  dim3 grid(kDC / 128, a.heads, (a.n_tokens + kAbsorbTok - 1) / kAbsorbTok);
  if (a.act == MLA_F32) return launch_pdl(absorb_simt_kernel<float>, grid, dim3(128), 0, s, a);
  return launch_pdl(absorb_simt_kernel<__nv_bfloat16>, grid, dim3(128), 0, s, a);
}

cudaError_t launch_out_proj_simt(const ProjArgs& a, cudaStream_t s) {
  if (a.n_tokens == 0) return cudaSuccess;
  dim3 grid(a.heads, (a.n_tokens + kOutTok - 1) / kOutTok);
  if (a.act == MLA_F32) return launch_pdl(out_proj_simt_kernel<float>, grid, dim3(128), 0, s, a);
  return launch_pdl(out_proj_simt_kernel<__nv_bfloat16>, grid, dim3(128), 0, s, a);
}

}  // namespace mla
