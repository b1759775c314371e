// Device helpers shared by the MLA decode kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "mla.h"

namespace mla {

constexpr int kDNope = 128;  // per-head content query/key width
constexpr int kDC = 512;     // latent width
constexpr int kDRope = 64;   // decoupled RoPE width
constexpr int kDV = 128;     // per-head value width
constexpr int kRow = kDC + kDRope;  // 576 values per cached token
constexpr int kGroups = MLA_E4M3_GROUPS;
constexpr float kE4M3Max = 448.0f;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Programmatic dependent launch (see launch_pdl): let the next kernel in the
// stream start, and wait until every earlier kernel has completed and its
// writes are visible.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ void flag_error(int32_t* flag, int32_t bits) {
  if (flag != nullptr) atomicOr(flag, bits);
}

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t b16) { return __uint_as_float(b16 << 16); }

// Round-to-nearest-even fp32 -> bf16 bits.
__device__ __forceinline__ uint16_t f32_to_bf16_bits(float x) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(x));
}

// Two fp32 -> bf16 (round to nearest even), lo in the low half: one paired conversion.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// Exact E4M3FN -> fp32 decode of one byte (bias 7, subnormals, no inf).
__device__ __forceinline__ float e4m3_to_f32(uint32_t byte) {
  __nv_fp8_e4m3 v;
  v.__x = static_cast<__nv_fp8_storage_t>(byte);
  return static_cast<float>(v);
}

template <typename T>
struct ActIO;
template <>
struct ActIO<float> {
  __device__ __forceinline__ static float load(const float* p) { return *p; }
  __device__ __forceinline__ static void store(float* p, float v) { *p = v; }
};
template <>
struct ActIO<__nv_bfloat16> {
  __device__ __forceinline__ static float load(const __nv_bfloat16* p) { return __bfloat162float(*p); }
  __device__ __forceinline__ static void store(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }
};

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// sum over s = 0 .. splits-1 of part[s * stride + i], added left to right in
// split order; the loads are issued four at a time so that they overlap.
__device__ __forceinline__ float split_sum(const float* part, int64_t i, int64_t stride, int splits) {
  float a = part[i];
  int s = 1;
  for (; s + 3 < splits; s += 4) {
    const float b0 = part[s * stride + i], b1 = part[(s + 1) * stride + i];
    const float b2 = part[(s + 2) * stride + i], b3 = part[(s + 3) * stride + i];
    a = (((a + b0) + b1) + b2) + b3;
  }
  for (; s < splits; ++s) a += part[s * stride + i];
  return a;
}

// L2 residency hints for data written by one kernel and read once by the
// next (split-KV partials): stored with evict_last so that a concurrent stream
// of evict_first loads does not push them out to HBM first, and read with
// evict_first, since nothing reads them again.
__device__ __forceinline__ uint64_t l2_evict_last_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ void st_global_v4_hint(void* ptr, uint4 v, uint64_t pol) {
  asm volatile("st.global.L2::cache_hint.v4.b32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(ptr), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w), "l"(pol)
               : "memory");
}
__device__ __forceinline__ float4 ld_global_v4_hint(const void* ptr, uint64_t pol) {
  float4 v;
  asm volatile("ld.global.L2::cache_hint.v4.f32 {%0, %1, %2, %3}, [%4], %5;"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "l"(ptr), "l"(pol)
               : "memory");
  return v;
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

}  // namespace mla
