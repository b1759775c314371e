// mla_cache_append: write new tokens into the paged latent cache.
//
// One warp per token. Lane l owns c_KV elements [16l, 16l+16) and the RoPE
// pair l, i.e. row elements (512+2l, 513+2l). The rotation is the adjacent-pair
// rotation of the decoupled RoPE key (k_R = RoPE(W_KR h), "Model Architecture
// Driving Inference Systems" §2.3; pair layout of the complex view in "MLA:
// Mathematical Foundations", PyTorch Reference Implementation, apply_rope),
// with each product and sum rounded separately so that the stored bytes are a
// pure function of the inputs and the fp32 cos/sin tables.
//
// E4M3 rows (FP8 cache with per-block scaling factors, "MLA: Mathematical
// Foundations", High-Throughput Serving Kernels) are quantised per 128-value
// group (the 64-value RoPE tail is its own group): scale = amax/448 correctly
// rounded, byte = satfinite-RNE E4M3 of x/scale correctly rounded.
#include "common.cuh"
#include "launchers.h"

namespace mla {
namespace {

enum CacheKind { kCacheF32 = 0, kCacheBF16 = 1, kCacheE4M3 = 2 };

template <typename InT>
__device__ __forceinline__ void load_c16(const InT* p, float (&c)[16]);

template <>
__device__ __forceinline__ void load_c16<float>(const float* p, float (&c)[16]) {
  const float4* v = reinterpret_cast<const float4*>(p);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float4 x = v[i];
    c[4 * i] = x.x;
    c[4 * i + 1] = x.y;
    c[4 * i + 2] = x.z;
    c[4 * i + 3] = x.w;
  }
}

template <>
__device__ __forceinline__ void load_c16<__nv_bfloat16>(const __nv_bfloat16* p, float (&c)[16]) {
  const uint4* v = reinterpret_cast<const uint4*>(p);
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    uint4 x = v[i];
    uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      c[8 * i + 2 * k] = bf16_bits_to_f32(w[k] & 0xffffu);
      c[8 * i + 2 * k + 1] = bf16_bits_to_f32(w[k] >> 16);
    }
  }
}

template <typename InT>
__device__ __forceinline__ float2 load_pair(const InT* p);
template <>
__device__ __forceinline__ float2 load_pair<float>(const float* p) {
  return *reinterpret_cast<const float2*>(p);
}
template <>
__device__ __forceinline__ float2 load_pair<__nv_bfloat16>(const __nv_bfloat16* p) {
  uint32_t w = *reinterpret_cast<const uint32_t*>(p);
  return make_float2(bf16_bits_to_f32(w & 0xffffu), bf16_bits_to_f32(w >> 16));
}

__device__ __forceinline__ float quant_scale(float amax) {
  return amax == 0.0f ? 1.0f : __fdiv_rn(amax, kE4M3Max);
}

__device__ __forceinline__ uint32_t e4m3x2(float a, float b) {
  // a -> low byte, b -> high byte; round to nearest even, saturate to +-448
  return static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3));
}

template <typename InT, int kCache>
__global__ void __launch_bounds__(256) append_kernel(AppendArgs a) {
  pdl_trigger();
  pdl_wait();  // the previous step's readers of the cache are done
  const int token = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (token >= a.n_tokens) return;
  const int64_t slot = a.slots[token];
  const int32_t pos = a.positions[token];
  const bool bad_slot = slot < 0 || slot >= a.n_rows;
  const bool bad_pos = pos < 0 || pos >= a.max_pos;
  if (bad_slot || bad_pos) {
    if (lane == 0)
      flag_error(a.dev_error, (bad_slot ? MLA_DEVERR_BAD_SLOT : 0) | (bad_pos ? MLA_DEVERR_BAD_POSITION : 0));
    return;
  }
  const InT* c_in = static_cast<const InT*>(a.c_kv) + static_cast<int64_t>(token) * kDC + 16 * lane;
  const InT* k_in = static_cast<const InT*>(a.k_r) + static_cast<int64_t>(token) * kDRope + 2 * lane;
  float c[16];
  load_c16<InT>(c_in, c);
  const float2 x = load_pair<InT>(k_in);
  const float co = a.cos_t[static_cast<int64_t>(pos) * (kDRope / 2) + lane];
  const float si = a.sin_t[static_cast<int64_t>(pos) * (kDRope / 2) + lane];
  const float r0 = __fsub_rn(__fmul_rn(x.x, co), __fmul_rn(x.y, si));
  const float r1 = __fadd_rn(__fmul_rn(x.x, si), __fmul_rn(x.y, co));

  if constexpr (kCache == kCacheF32) {
    float* row = static_cast<float*>(a.cache) + slot * kRow;
    float4* dst = reinterpret_cast<float4*>(row + 16 * lane);
#pragma unroll
    for (int i = 0; i < 4; ++i) dst[i] = make_float4(c[4 * i], c[4 * i + 1], c[4 * i + 2], c[4 * i + 3]);
    *reinterpret_cast<float2*>(row + kDC + 2 * lane) = make_float2(r0, r1);
  } else if constexpr (kCache == kCacheBF16) {
    uint16_t* row = static_cast<uint16_t*>(a.cache) + slot * kRow;
    uint32_t w[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) w[i] = pack_bf16x2(c[2 * i], c[2 * i + 1]);
    uint4* dst = reinterpret_cast<uint4*>(row + 16 * lane);
    dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
    dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
    *reinterpret_cast<uint32_t*>(row + kDC + 2 * lane) = pack_bf16x2(r0, r1);
  } else {
    // group amax: lanes 8g..8g+7 hold latent group g; the RoPE group spans all lanes
    float am = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) am = fmaxf(am, fabsf(c[i]));
    am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 1));
    am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 2));
    am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 4));
    const float ar = warp_max(fmaxf(fabsf(r0), fabsf(r1)));
    const float sc = quant_scale(am);
    const float sr = quant_scale(ar);
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint32_t lo = e4m3x2(__fdiv_rn(c[4 * i], sc), __fdiv_rn(c[4 * i + 1], sc));
      uint32_t hi = e4m3x2(__fdiv_rn(c[4 * i + 2], sc), __fdiv_rn(c[4 * i + 3], sc));
      w[i] = lo | (hi << 16);
    }
    uint8_t* row = static_cast<uint8_t*>(a.cache) + slot * kRow;
    *reinterpret_cast<uint4*>(row + 16 * lane) = make_uint4(w[0], w[1], w[2], w[3]);
    *reinterpret_cast<uint16_t*>(row + kDC + 2 * lane) =
        static_cast<uint16_t>(e4m3x2(__fdiv_rn(r0, sr), __fdiv_rn(r1, sr)));
    float* srow = a.scales + slot * kGroups;
    if ((lane & 7) == 0) srow[lane >> 3] = sc;
    if (lane == 0) srow[4] = sr;
  }
}

template <typename InT>
cudaError_t launch_in(const AppendArgs& a, cudaStream_t s) {
  const int threads = 256;
  const int blocks = (a.n_tokens + 7) / 8;
  switch (a.cache_dtype) {
    case MLA_F32:
      return launch_pdl(append_kernel<InT, kCacheF32>, dim3(blocks), dim3(threads), 0, s, a);
    case MLA_BF16:
      return launch_pdl(append_kernel<InT, kCacheBF16>, dim3(blocks), dim3(threads), 0, s, a);
    default:
      return launch_pdl(append_kernel<InT, kCacheE4M3>, dim3(blocks), dim3(threads), 0, s, a);
  }
}

}  // namespace

cudaError_t launch_append(const AppendArgs& a, cudaStream_t s) {
  if (a.n_tokens == 0) return cudaSuccess;
  if (a.in_dtype == MLA_F32) return launch_in<float>(a, s);
  return launch_in<__nv_bfloat16>(a, s);
}

}  // namespace mla
