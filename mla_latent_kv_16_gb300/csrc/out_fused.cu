// Load-time fold of the value up-projection into the output projection
// ("Model Architecture Driving Inference Systems" §3.2, pre-fused
// W~^O_i = W^O_i W^UV_i, and §4.2, fused when the model is loaded;
// "Multi-Head Latent Attention (MLA)" page, "Value Output Matrix Absorption"):
//
//   W~[m][h][c] = sum_e W_O[m][h][e] W_UV[h][e][c]
//
// Run once, on CUDA cores; the per-step product y = W~ u is the generic linear
// layer of linear.cu.
#include "common.cuh"
#include "launchers.h"

namespace mla {
namespace {

// ------------------------------------------------------------------ fold (load time)

// grid (512/64, ceil(d/64), H), block 256: a 64 (m) x 64 (c) tile of W~ for
// head h, each thread 4 x 4 outputs, the 128-long e dimension in 4 steps of 32.
template <typename T>
__global__ void __launch_bounds__(256) fuse_weights_kernel(FuseWeightsArgs a) {
  pdl_trigger();
  pdl_wait();
  __shared__ float as[32][65];  // [e][m]: W_O[m0 + m][h][e0 + e]
  __shared__ float bs[32][64];  // [e][c]: W_UV[h][e0 + e][c0 + c]
  const int c0 = blockIdx.x * 64, m0 = blockIdx.y * 64, h = blockIdx.z;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const T* w_o = static_cast<const T*>(a.w_o);
  const T* w_uv = static_cast<const T*>(a.w_uv);
  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.0f;
  for (int e0 = 0; e0 < kDV; e0 += 32) {
    for (int i = threadIdx.x; i < 64 * 32; i += 256) {
      const int m = i >> 5, e = i & 31;
      const int mm = m0 + m;
      as[e][m] = mm < a.d_model ? ActIO<T>::load(w_o + (static_cast<int64_t>(mm) * a.heads + h) * kDV + e0 + e)
                                : 0.0f;
    }
    for (int i = threadIdx.x; i < 32 * 64; i += 256) {
      const int e = i >> 6, c = i & 63;
      bs[e][c] = ActIO<T>::load(w_uv + (static_cast<int64_t>(h) * kDV + e0 + e) * kDC + c0 + c);
    }
    __syncthreads();
#pragma unroll 8
    for (int e = 0; e < 32; ++e) {
      float av[4], bv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) av[i] = as[e][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) bv[j] = bs[e][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
    }
    __syncthreads();
  }
  T* out = static_cast<T*>(a.w_fused);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int mm = m0 + ty * 4 + i;
    if (mm >= a.d_model) continue;
    T* row = out + (static_cast<int64_t>(mm) * a.heads + h) * kDC + c0 + tx * 4;
#pragma unroll
    for (int j = 0; j < 4; ++j) ActIO<T>::store(row + j, acc[i][j]);
  }
}

}  // namespace

cudaError_t launch_fuse_weights(const FuseWeightsArgs& a, cudaStream_t s) {
  const dim3 grid(kDC / 64, (a.d_model + 63) / 64, a.heads);
  if (a.act == MLA_F32) return launch_pdl(fuse_weights_kernel<float>, grid, dim3(256), 0, s, a);
  return launch_pdl(fuse_weights_kernel<__nv_bfloat16>, grid, dim3(256), 0, s, a);
}

}  // namespace mla
