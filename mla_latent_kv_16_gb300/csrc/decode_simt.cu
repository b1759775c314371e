// Paged latent-space decode attention on CUDA cores, plus the split-KV
// log-sum-exp combine.
//
// Score per head h and cached token j ("Model Architecture Driving Inference
// Systems" §3.1; "Tech Radar: DeepSeek-V3 MLA" §2):
//   s_j = (q_lat[h] . c_KV[j] + q_rope[h] . k_R[j]) * softmax_scale
// latent output (§3.2): u[h] = sum_j softmax(s)_j c_KV[j], computed with a
// running max / running sum over token tiles so that no score leaves the chip.
//
// This kernel handles every dtype and head count (fp32 tiny decode, any H); the
// bf16/E4M3 128-head path is the tcgen05 kernel in decode_tc.cu.
//
// CTA = 8 warps = 8 heads of one (sequence, query, split); warp lane = token
// inside a 32-token tile. Rows are decoded to fp32 in shared memory (rows past
// the visible range are zero-filled, so poisoned page tails never enter).
#include <math_constants.h>

#include "common.cuh"
#include "launchers.h"

namespace mla {
namespace {

constexpr int kTile = 32;
constexpr int kHG = 8;                // heads per CTA
constexpr int kRowPad = kRow + 1;     // bank-conflict-free row stride (floats)
constexpr size_t kSimtSmem = (size_t(kTile) * kRowPad + size_t(kHG) * kRow) * sizeof(float);

template <typename T>
__device__ __forceinline__ float ld_act(const void* base, int64_t idx) {
  return ActIO<T>::load(static_cast<const T*>(base) + idx);
}

// One cached row (576 values) as 16-byte chunks: 144 of fp32, 72 of bf16, 36 of E4M3.
template <int kCache>
struct RowChunks {
  static constexpr int kBytes = kCache == MLA_F32 ? 4 : (kCache == MLA_BF16 ? 2 : 1);
  static constexpr int kPer = 16 / kBytes;   // values per chunk
  static constexpr int kN = kRow / kPer;     // chunks per row
  static constexpr int kK = (kN + 31) / 32;  // chunks per lane
};

// Rows of one tile into fp32 shared memory, warp w taking rows w, w + 8, ...:
// every 16-byte load of the warp's rows is issued before any is used, so a
// tile costs one memory round trip instead of one per load. Rows past the
// visible range are zero-filled (poisoned page tails never enter).
template <int kCache>
__device__ __forceinline__ void load_tile_rows(const DecodeArgs& a, const int32_t* bt, int t0, int end, float* rs,
                                               int warp, int lane) {
  using RC = RowChunks<kCache>;
  constexpr int kRowsPerWarp = kTile / 8;
  uint4 v[kRowsPerWarp][RC::kK];
  int64_t slot[kRowsPerWarp];
#pragma unroll
  for (int r = 0; r < kRowsPerWarp; ++r) {
    const int tok = t0 + warp + 8 * r;
    slot[r] = tok < end ? static_cast<int64_t>(bt[tok / a.page_size]) * a.page_size + tok % a.page_size : -1;
    const uint4* row = reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(a.cache) +
                                                      (slot[r] < 0 ? 0 : slot[r]) * (kRow * RC::kBytes));
#pragma unroll
    for (int k = 0; k < RC::kK; ++k) {
      const int c = lane + 32 * k;
      v[r][k] = (slot[r] >= 0 && c < RC::kN) ? row[c] : make_uint4(0, 0, 0, 0);
    }
  }
#pragma unroll
  for (int r = 0; r < kRowsPerWarp; ++r) {
    float* dst = rs + (warp + 8 * r) * kRowPad;
    const float* sc = kCache == MLA_E4M3 && slot[r] >= 0 ? a.scales + slot[r] * kGroups : nullptr;
#pragma unroll
    for (int k = 0; k < RC::kK; ++k) {
      const int c = lane + 32 * k;
      if (c >= RC::kN) continue;
      const uint32_t w[4] = {v[r][k].x, v[r][k].y, v[r][k].z, v[r][k].w};
      const int k0 = c * RC::kPer;
      if constexpr (kCache == MLA_F32) {
#pragma unroll
        for (int e = 0; e < 4; ++e) dst[k0 + e] = __uint_as_float(w[e]);
      } else if constexpr (kCache == MLA_BF16) {
#pragma unroll
        for (int e = 0; e < 8; ++e) dst[k0 + e] = bf16_bits_to_f32(static_cast<uint16_t>(w[e >> 1] >> (16 * (e & 1))));
      } else {
        // dequantised value rounded to the bf16 operand type the E4M3 cache pairs with
        const float s = sc != nullptr ? sc[k0 >> 7] : 0.0f;  // a chunk lies in one 128-wide group
#pragma unroll
        for (int e = 0; e < 16; ++e)
          dst[k0 + e] = bf16_bits_to_f32(
              f32_to_bf16_bits(e4m3_to_f32(static_cast<uint8_t>(w[e >> 2] >> (8 * (e & 3)))) * s));
      }
    }
  }
}

template <typename T, int kCache>
__global__ void __launch_bounds__(256) decode_simt_kernel(DecodeArgs a) {
  pdl_trigger();
  pdl_wait();
  extern __shared__ float smem[];
  float* rs = smem;                          // [kTile][kRowPad]
  float* qs = smem + kTile * kRowPad;        // [kHG][kRow]
  const int split = blockIdx.x;
  const int h0 = blockIdx.y * kHG;
  const int bj = blockIdx.z;
  const int b = bj / a.q_len, j = bj % a.q_len;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = h0 + warp;
  const bool head_ok = h < a.heads;

  const int L = a.seq_lens[b];
  const int P = a.page_size;
  int n_vis = L - a.q_len + j + 1;
  bool bad = false;
  if (L < a.q_len || static_cast<int64_t>(L) > static_cast<int64_t>(a.max_pages) * P) {
    if (threadIdx.x == 0) flag_error(a.dev_error, MLA_DEVERR_BAD_SEQLEN);
    bad = true;
    n_vis = 0;
  }
  const int tok_begin = split * a.pages_per_split * P;
  const int tok_end = min(n_vis, (split + 1) * a.pages_per_split * P);
  const int32_t* bt = a.block_table + static_cast<int64_t>(b) * a.max_pages;
  // validate every page this split touches
  if (tok_begin < tok_end) {
    const int pg0 = tok_begin / P, pg1 = (tok_end - 1) / P;
    int local_bad = 0;
    for (int pg = pg0 + threadIdx.x; pg <= pg1; pg += blockDim.x) {
      const int32_t pp = bt[pg];
      if (pp < 0 || pp >= a.num_pages) local_bad = 1;
    }
    if (__syncthreads_or(local_bad)) {
      if (threadIdx.x == 0) flag_error(a.dev_error, MLA_DEVERR_BAD_PAGE);
      bad = true;
    }
  }

  // this warp's query, pre-scaled into the log2 domain
  const float qscale = a.softmax_scale * kLog2e;
  if (head_ok) {
    const int64_t qi = (static_cast<int64_t>(bj) * a.heads + h);
    for (int k = lane; k < kRow; k += 32) {
      const float v = k < kDC ? ld_act<T>(a.q_lat, qi * kDC + k) : ld_act<T>(a.q_rope, qi * kDRope + (k - kDC));
      qs[warp * kRow + k] = v * qscale;
    }
  }

  float m = -CUDART_INF_F, l = 0.0f;
  float acc[kDC / 32];
#pragma unroll
  for (int i = 0; i < kDC / 32; ++i) acc[i] = 0.0f;

  const int end = bad ? tok_begin : tok_end;
  for (int t0 = tok_begin; t0 < end; t0 += kTile) {
    __syncthreads();
    load_tile_rows<kCache>(a, bt, t0, end, rs, warp, lane);
    __syncthreads();
    if (head_ok) {
      const float* qh = qs + warp * kRow;
      const float* rr = rs + lane * kRowPad;
      float s4[4] = {0.0f, 0.0f, 0.0f, 0.0f};  // four chains (summed in a fixed order)
#pragma unroll 8
      for (int k = 0; k < kRow; k += 4) {
        s4[0] = fmaf(qh[k], rr[k], s4[0]);
        s4[1] = fmaf(qh[k + 1], rr[k + 1], s4[1]);
        s4[2] = fmaf(qh[k + 2], rr[k + 2], s4[2]);
        s4[3] = fmaf(qh[k + 3], rr[k + 3], s4[3]);
      }
      float s = (s4[0] + s4[1]) + (s4[2] + s4[3]);
      if (t0 + lane >= end) s = -CUDART_INF_F;
      const float m_new = fmaxf(m, warp_max(s));
      const float alpha = fast_exp2(m - m_new);   // m = -inf on the first tile -> 0
      const float p = fast_exp2(s - m_new);
      l = l * alpha + warp_sum(p);
      m = m_new;
#pragma unroll
      for (int i = 0; i < kDC / 32; ++i) acc[i] *= alpha;
      for (int t = 0; t < kTile; ++t) {
        const float pt = __shfl_sync(0xffffffffu, p, t);
        const float* rt = rs + t * kRowPad + lane;
#pragma unroll
        for (int i = 0; i < kDC / 32; ++i) acc[i] = fmaf(pt, rt[32 * i], acc[i]);
      }
    }
  }
  if (!head_ok) return;

  const bool empty = !(l > 0.0f);
  const float inv_l = empty ? 0.0f : 1.0f / l;
  const float lse = empty ? -CUDART_INF_F : (m + log2f(l)) * kLn2;
  const int64_t row = static_cast<int64_t>(bj) * a.heads + h;
  if (a.num_splits == 1) {
    T* u = static_cast<T*>(a.u_out) + row * kDC;
#pragma unroll
    for (int i = 0; i < kDC / 32; ++i) ActIO<T>::store(u + lane + 32 * i, acc[i] * inv_l);
    if (a.lse_out != nullptr && lane == 0) a.lse_out[row] = lse;
  } else {
    const int64_t prow = (static_cast<int64_t>(bj) * a.num_splits + split) * a.heads + h;
    float* pu = a.part_u + prow * kDC;
#pragma unroll
    for (int i = 0; i < kDC / 32; ++i) pu[lane + 32 * i] = acc[i] * inv_l;
    if (lane == 0) a.part_lse[prow] = lse;
  }
}

constexpr int kFewSplits = 4;
constexpr int kCombineWarps = 16;  // heads per CTA of the split merge

// The merged row of (query bj, head h): this lane's 16 columns of u = acc / sum,
// and lse = mx + log(sum) (lane 0).
template <typename T>
__device__ __forceinline__ void combine_store(const DecodeArgs& a, int bj, int h, int lane, const float (&acc)[16],
                                              bool none, float mx, float sum) {
  const float inv = none ? 0.0f : 1.0f / sum;
  const int64_t row = static_cast<int64_t>(bj) * a.heads + h;
  T* u = static_cast<T*>(a.u_out) + row * kDC + lane * 16;
  if constexpr (sizeof(T) == 2) {
    uint32_t w[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) w[k] = pack_bf16x2(acc[2 * k] * inv, acc[2 * k + 1] * inv);
    uint4* d = reinterpret_cast<uint4*>(u);
    d[0] = make_uint4(w[0], w[1], w[2], w[3]);
    d[1] = make_uint4(w[4], w[5], w[6], w[7]);
  } else {
    float4* d = reinterpret_cast<float4*>(u);
#pragma unroll
    for (int v = 0; v < 4; ++v)
      d[v] = make_float4(acc[4 * v] * inv, acc[4 * v + 1] * inv, acc[4 * v + 2] * inv, acc[4 * v + 3] * inv);
  }
  if (lane == 0 && a.lse_out != nullptr) a.lse_out[row] = none ? -CUDART_INF_F : mx + logf(sum);
}

// Split-KV merge ("Model Architecture Driving Inference Systems" §4.1, split
// KV with a log-sum-exp combine): u = sum_s e^(lse_s - lse*) u_s / sum_s
// e^(lse_s - lse*), lse = lse* + log sum_s e^(lse_s - lse*). One warp per
// (query, head): the lanes reduce the split log-sum-exps with shuffles, then
// each lane merges 16 consecutive columns of the 512 with 16-byte loads.
// kCombineWarps heads per CTA: few CTAs, so that the whole grid is resident
// (and has let the next kernel launch) within a fraction of a microsecond.
//
// Few splits (kS = S <= kFewSplits, the common case): every split's
// log-sum-exp and partial columns are requested at once, so the merge costs
// one memory round trip; with kS a compile-time count the registers hold just
// those splits, and two CTAs fit an SM at kS = 2 (one wave of CTAs for the
// DeepSeek-V3-shaped batch). A split whose lse is -inf is selected out, never
// multiplied (its partial may hold anything).
template <typename T, int kS>
__global__ void __launch_bounds__(32 * kCombineWarps, kS <= 2 ? 2 : 1) combine_few_kernel(DecodeArgs a) {
  pdl_trigger();
  pdl_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.x * kCombineWarps + warp, bj = blockIdx.y;
  if (h >= a.heads) return;
  const uint64_t pol = l2_evict_first_policy();  // the partials are read once
  const float* lse_s = a.part_lse + static_cast<int64_t>(bj) * kS * a.heads + h;  // stride a.heads
  float ls[kS];
  float4 x[kS][4];
#pragma unroll
  for (int s = 0; s < kS; ++s) {
    ls[s] = lse_s[static_cast<int64_t>(s) * a.heads];
    const float4* src = reinterpret_cast<const float4*>(
        a.part_u + ((static_cast<int64_t>(bj) * kS + s) * a.heads + h) * kDC + lane * 16);
#pragma unroll
    for (int v = 0; v < 4; ++v) x[s][v] = ld_global_v4_hint(src + v, pol);
  }
  float mx = ls[0];
#pragma unroll
  for (int s = 1; s < kS; ++s) mx = fmaxf(mx, ls[s]);
  const bool none = (mx == -CUDART_INF_F);
  float sum = 0.0f;
  float acc[16];
#pragma unroll
  for (int k = 0; k < 16; ++k) acc[k] = 0.0f;
#pragma unroll
  for (int s = 0; s < kS; ++s) {
    const bool use = !none && ls[s] != -CUDART_INF_F;
    const float wv = use ? fast_exp2((ls[s] - mx) * kLog2e) : 0.0f;
    sum += wv;
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      acc[4 * v] = use ? fmaf(wv, x[s][v].x, acc[4 * v]) : acc[4 * v];
      acc[4 * v + 1] = use ? fmaf(wv, x[s][v].y, acc[4 * v + 1]) : acc[4 * v + 1];
      acc[4 * v + 2] = use ? fmaf(wv, x[s][v].z, acc[4 * v + 2]) : acc[4 * v + 2];
      acc[4 * v + 3] = use ? fmaf(wv, x[s][v].w, acc[4 * v + 3]) : acc[4 * v + 3];
    }
  }
  combine_store<T>(a, bj, h, lane, acc, none, mx, sum);
}

// More splits (kFewSplits < S <= kManySplits), the same merge and grid.
template <typename T>
__global__ void __launch_bounds__(32 * kCombineWarps) combine_kernel(DecodeArgs a) {
  pdl_trigger();
  pdl_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.x * kCombineWarps + warp, bj = blockIdx.y;
  if (h >= a.heads) return;
  const uint64_t pol = l2_evict_first_policy();  // the partials are read once
  const int S = a.num_splits;
  const float* lse_s = a.part_lse + static_cast<int64_t>(bj) * S * a.heads + h;  // stride a.heads
  // Many splits: the maximum log-sum-exp first (lane s holds split s's for
  // S <= 32), then the splits in groups of kFewSplits whose partial columns are
  // all requested at once: 1 + ceil(S / kFewSplits) memory round trips.
  const float ls_lane = lane < S ? lse_s[static_cast<int64_t>(lane) * a.heads] : -CUDART_INF_F;
  float mx = ls_lane;
  for (int s = lane + 32; s < S; s += 32) mx = fmaxf(mx, lse_s[static_cast<int64_t>(s) * a.heads]);
  mx = warp_max(mx);
  const bool none = (mx == -CUDART_INF_F);
  float sum = 0.0f;
  float acc[16];
#pragma unroll
  for (int k = 0; k < 16; ++k) acc[k] = 0.0f;
  for (int s0 = 0; !none && s0 < S; s0 += kFewSplits) {
    float ls[kFewSplits];
    float4 x[kFewSplits][4];
#pragma unroll
    for (int u = 0; u < kFewSplits; ++u) {
      const int s = s0 + u;  // uniform across the warp
      if (s < S) {
        ls[u] = S <= 32 ? __shfl_sync(0xffffffffu, ls_lane, s) : lse_s[static_cast<int64_t>(s) * a.heads];
        const float4* src = reinterpret_cast<const float4*>(
            a.part_u + ((static_cast<int64_t>(bj) * S + s) * a.heads + h) * kDC + lane * 16);
#pragma unroll
        for (int v = 0; v < 4; ++v) x[u][v] = ld_global_v4_hint(src + v, pol);
      } else {
        ls[u] = -CUDART_INF_F;
      }
    }
#pragma unroll
    for (int u = 0; u < kFewSplits; ++u) {
      const bool use = ls[u] != -CUDART_INF_F;  // a -inf split is selected out, never multiplied
      const float wv = use ? fast_exp2((ls[u] - mx) * kLog2e) : 0.0f;
      sum += wv;
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        acc[4 * v] = use ? fmaf(wv, x[u][v].x, acc[4 * v]) : acc[4 * v];
        acc[4 * v + 1] = use ? fmaf(wv, x[u][v].y, acc[4 * v + 1]) : acc[4 * v + 1];
        acc[4 * v + 2] = use ? fmaf(wv, x[u][v].z, acc[4 * v + 2]) : acc[4 * v + 2];
        acc[4 * v + 3] = use ? fmaf(wv, x[u][v].w, acc[4 * v + 3]) : acc[4 * v + 3];
      }
    }
  }
  combine_store<T>(a, bj, h, lane, acc, none, mx, sum);
}

// The same merge for many splits (S > kManySplits): one CTA of eight warps per
// (query, head) row. Every warp finds the row's maximum log-sum-exp itself (so
// all weights share one reference and no rescaling between warps is needed),
// merges the groups of four splits 4w, 4w + 32, ... with their partials all
// requested at once, and the eight sums and 512-column rows are added in
// shared memory in warp order. Each row then costs ceil(S / 32) + 1 round
// trips instead of ceil(S / 4) + 1, with eight times the loads in flight.
constexpr int kManySplits = 8;

template <typename T>
__global__ void __launch_bounds__(256) combine_many_kernel(DecodeArgs a) {
  pdl_trigger();
  pdl_wait();
  __shared__ float4 red[8][kDC / 4];
  __shared__ float red_sum[8];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.x, bj = blockIdx.y;
  const int S = a.num_splits;
  const uint64_t pol = l2_evict_first_policy();  // the partials are read once
  const float* lse_s = a.part_lse + static_cast<int64_t>(bj) * S * a.heads + h;  // stride a.heads
  float mx = -CUDART_INF_F;
  for (int s = lane; s < S; s += 32) mx = fmaxf(mx, lse_s[static_cast<int64_t>(s) * a.heads]);
  mx = warp_max(mx);
  const bool none = (mx == -CUDART_INF_F);
  float sum = 0.0f;
  float acc[16];
#pragma unroll
  for (int k = 0; k < 16; ++k) acc[k] = 0.0f;
  for (int s0 = kFewSplits * warp; !none && s0 < S; s0 += 8 * kFewSplits) {
    float ls[kFewSplits];
    float4 x[kFewSplits][4];
#pragma unroll
    for (int u = 0; u < kFewSplits; ++u) {
      const int s = s0 + u;  // uniform across the warp
      if (s < S) {
        ls[u] = lse_s[static_cast<int64_t>(s) * a.heads];
        const float4* src = reinterpret_cast<const float4*>(
            a.part_u + ((static_cast<int64_t>(bj) * S + s) * a.heads + h) * kDC + lane * 16);
#pragma unroll
        for (int v = 0; v < 4; ++v) x[u][v] = ld_global_v4_hint(src + v, pol);
      } else {
        ls[u] = -CUDART_INF_F;
      }
    }
#pragma unroll
    for (int u = 0; u < kFewSplits; ++u) {
      const bool use = ls[u] != -CUDART_INF_F;  // a -inf split is selected out, never multiplied
      const float wv = use ? fast_exp2((ls[u] - mx) * kLog2e) : 0.0f;
      sum += wv;
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        acc[4 * v] = use ? fmaf(wv, x[u][v].x, acc[4 * v]) : acc[4 * v];
        acc[4 * v + 1] = use ? fmaf(wv, x[u][v].y, acc[4 * v + 1]) : acc[4 * v + 1];
        acc[4 * v + 2] = use ? fmaf(wv, x[u][v].z, acc[4 * v + 2]) : acc[4 * v + 2];
        acc[4 * v + 3] = use ? fmaf(wv, x[u][v].w, acc[4 * v + 3]) : acc[4 * v + 3];
      }
    }
  }
#pragma unroll
  for (int v = 0; v < 4; ++v)
    red[warp][lane * 4 + v] = make_float4(acc[4 * v], acc[4 * v + 1], acc[4 * v + 2], acc[4 * v + 3]);
  if (lane == 0) red_sum[warp] = sum;
  __syncthreads();
  if (warp != 0) return;
  float tot = 0.0f;
#pragma unroll
  for (int k = 0; k < 16; ++k) acc[k] = 0.0f;
#pragma unroll
  for (int w = 0; w < 8; ++w) {
    tot += red_sum[w];
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      const float4 y = red[w][lane * 4 + v];
      acc[4 * v] += y.x;
      acc[4 * v + 1] += y.y;
      acc[4 * v + 2] += y.z;
      acc[4 * v + 3] += y.w;
    }
  }
  combine_store<T>(a, bj, h, lane, acc, none, mx, tot);
}

// Opt the kernel into its dynamic shared memory once per device (a host call
// that costs microseconds, kept out of every launch).
template <typename K>
cudaError_t ensure_smem(K kernel, size_t bytes, int& done_for) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || done_for == dev) return e;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
  if (e == cudaSuccess) done_for = dev;
  return e;
}

template <typename T, int kCache>
cudaError_t launch_decode_c(const DecodeArgs& a, cudaStream_t s) {
  static int done_for = -1;
  const cudaError_t e = ensure_smem(decode_simt_kernel<T, kCache>, kSimtSmem, done_for);
  if (e != cudaSuccess) return e;
  dim3 grid(a.num_splits, (a.heads + kHG - 1) / kHG, a.batch * a.q_len);
  return launch_pdl(decode_simt_kernel<T, kCache>, grid, dim3(256), kSimtSmem, s, a);
}

template <typename T>
cudaError_t launch_decode_t(const DecodeArgs& a, cudaStream_t s) {
  switch (a.cache_dtype) {
    case MLA_F32: return launch_decode_c<T, MLA_F32>(a, s);
    case MLA_BF16: return launch_decode_c<T, MLA_BF16>(a, s);
    default: return launch_decode_c<T, MLA_E4M3>(a, s);
  }
}

}  // namespace

cudaError_t launch_decode_simt(const DecodeArgs& a, cudaStream_t s) {
  if (a.batch == 0) return cudaSuccess;
  if (a.act == MLA_F32) return launch_decode_t<float>(a, s);
  return launch_decode_t<__nv_bfloat16>(a, s);
}

cudaError_t launch_combine(const DecodeArgs& a, cudaStream_t s) {
  if (a.batch == 0 || a.num_splits == 1) return cudaSuccess;
  if (a.num_splits > kManySplits) {
    const dim3 grid(a.heads, a.batch * a.q_len);
    if (a.act == MLA_F32) return launch_pdl(combine_many_kernel<float>, grid, dim3(256), 0, s, a);
    return launch_pdl(combine_many_kernel<__nv_bfloat16>, grid, dim3(256), 0, s, a);
  }
  const dim3 grid((a.heads + kCombineWarps - 1) / kCombineWarps, a.batch * a.q_len), block(32 * kCombineWarps);
  static_assert(kFewSplits == 4, "few-split instances for 2..4 splits");
  if (a.act == MLA_F32) {
    switch (a.num_splits) {
      case 2: return launch_pdl(combine_few_kernel<float, 2>, grid, block, 0, s, a);
      case 3: return launch_pdl(combine_few_kernel<float, 3>, grid, block, 0, s, a);
      case 4: return launch_pdl(combine_few_kernel<float, 4>, grid, block, 0, s, a);
      default: return launch_pdl(combine_kernel<float>, grid, block, 0, s, a);
    }
  }
  switch (a.num_splits) {
    case 2: return launch_pdl(combine_few_kernel<__nv_bfloat16, 2>, grid, block, 0, s, a);
    case 3: return launch_pdl(combine_few_kernel<__nv_bfloat16, 3>, grid, block, 0, s, a);
    case 4: return launch_pdl(combine_few_kernel<__nv_bfloat16, 4>, grid, block, 0, s, a);
    default: return launch_pdl(combine_kernel<__nv_bfloat16>, grid, block, 0, s, a);
  }
}

}  // namespace mla
