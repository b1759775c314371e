// Per-head absorption contractions on tcgen05 (bf16 in, fp32 accumulate).
//
//   absorb  : q_lat[t,h,c] = sum_d W_UK[h,d,c] q_nope[t,h,d]   ("Model Architecture
//             Driving Inference Systems" §3.1: absorbed query (W_UK)^T q, computed
//             once per query token)
//   out_proj: o[t,h,d]     = sum_c W_UV[h,d,c] u[t,h,c]       (same page, §3.2)
//
// Both are computed transposed, Y_h^T = W_h' X_h^T, so that the 128 rows of a
// weight slice are the MMA M dimension and the (few) tokens are N:
//   absorb  : M = 128 latent columns c (one of 4 slices), K = 128 (d), A = W_UK[h]
//             as an MN-major operand (c contiguous), B = q_nope[:, h, :] (K-major)
//   out_proj: M = 128 (d), K = 512 (c) in 8 chunks through a TMA ring, A = W_UV[h]
//             (K-major), B = u[:, h, :] (K-major)
// One CTA per (head, M slice, token tile of up to 256). The accumulator lives
// in TMEM; the epilogue reads it back with each thread owning one output
// feature and writes tokens with coalesced bf16 stores. These GEMMs read every
// weight byte exactly once per token tile, so at decode batch sizes they are
// bound by the weight stream from HBM.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <math_constants.h>

#include "common.cuh"
#include "launchers.h"
#include "tc_ptx.cuh"

namespace mla {
namespace {

using namespace tc;

constexpr int kThreads = 128;
constexpr int kMaxTok = 256;  // tokens per CTA (MMA N)
constexpr int kChunkK = 64;   // K elements per TMA box (128 bytes of bf16)

// Shared memory: a ring of K chunks (A box of 128 rows x 128 B, then a B box of
// up to 256 token rows x 128 B), followed by this control block.
struct ProjCtl {
  uint64_t full[8];
  uint64_t empty[8];
  uint64_t done;
  uint32_t tmem_base;
  int32_t abort_flag;
};

constexpr int kABytes = 128 * 128;

// kind: 0 = absorb (A MN-major, K = 128), 1 = out_proj (A K-major, K = 512)
template <int kKind>
__global__ void __launch_bounds__(kThreads) proj_tc_kernel(const __grid_constant__ CUtensorMap amap,
                                                           const __grid_constant__ CUtensorMap bmap, ProjArgs p,
                                                           int n_tile, int stages, uint32_t tmem_cols) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int b_bytes = n_tile * 128;
  const int stage_bytes = kABytes + ((b_bytes + 1023) & ~1023);
  ProjCtl* ctl = reinterpret_cast<ProjCtl*>(base + stages * stage_bytes);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.x;
  const int mslice = blockIdx.y;  // absorb: which 128 of the 512 latent columns
  const int t0 = blockIdx.z * kMaxTok;
  const int n_tok = min(kMaxTok, p.n_tokens - t0);
  constexpr int kK = kKind == 0 ? kDNope : kDC;
  constexpr int kChunks = kK / kChunkK;
  pdl_trigger();

  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(smem_u32(&ctl->full[s]), 1);
      mbar_init(smem_u32(&ctl->empty[s]), 1);
    }
    mbar_init(smem_u32(&ctl->done), 1);
    ctl->abort_flag = 0;
    fence_mbar_init_cluster();
    prefetch_tmap(&amap);
    prefetch_tmap(&bmap);
  }
  if (warp == 0) tmem_alloc(smem_u32(&ctl->tmem_base), tmem_cols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;
  volatile int32_t* abort_flag = &ctl->abort_flag;

  // Chunk k of the weight slice (A) and of the activations (B) into stage s,
  // one barrier for both. The weights are static, so the first stages' A
  // boxes are requested before waiting for the previous kernels; the
  // activations they produced only after.
  auto load_a = [&](int k, int s) {
    const uint32_t a_dst = smem_u32(base + s * stage_bytes);
    const uint32_t bar = smem_u32(&ctl->full[s]);
    mbar_arrive_expect_tx(bar, kABytes + b_bytes);
    if constexpr (kKind == 0) {
      // W_UK[h] rows d in [64k, 64k+64), columns c in [128 m, 128 m + 128): two 64-column boxes
      tma_load_2d_nohint(a_dst, &amap, bar, 128 * mslice, h * kDNope + kChunkK * k);
      tma_load_2d_nohint(a_dst + kABytes / 2, &amap, bar, 128 * mslice + 64, h * kDNope + kChunkK * k);
    } else {
      // W_UV[h] rows d in [0,128), columns c in [64k, 64k+64)
      tma_load_2d_nohint(a_dst, &amap, bar, kChunkK * k, h * kDV);
    }
  };
  auto load_b = [&](int k, int s) {
    const uint32_t b_dst = smem_u32(base + s * stage_bytes) + kABytes;
    const uint32_t bar = smem_u32(&ctl->full[s]);
    // X[:, h, 64k : 64k+64] for tokens t0 .. t0+n_tile (rows past n_tokens read as zero)
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(
            b_dst),
        "l"(reinterpret_cast<uint64_t>(&bmap)), "r"(bar), "r"(kChunkK * k), "r"(h), "r"(t0)
        : "memory");
  };
  const int pre = min(stages, kChunks);
  if (threadIdx.x == 0)
    for (int k = 0; k < pre; ++k) load_a(k, k);
  pdl_wait();

  if (threadIdx.x == 0) {
    const uint32_t idesc = idesc_bf16_f32(128, n_tile, kKind == 0, false);
    for (int k = 0; k < pre; ++k) load_b(k, k);
    bool ok = true;
    for (int k = 0; k < kChunks && ok; ++k) {
      const int s = k % stages;
      if (!mbar_wait<2>(smem_u32(&ctl->full[s]), (k / stages) & 1, abort_flag, nullptr)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t a0 = smem_u32(base + s * stage_bytes);
      const uint64_t db = sdesc_sw128(a0 + kABytes, 16, 1024);
#pragma unroll
      for (int kk = 0; kk < kChunkK / 16; ++kk) {
        uint64_t da;
        if constexpr (kKind == 0)  // MN-major A: 16 K rows of 128 B per step; 64-column blocks 8 KB apart
          da = sdesc_sw128(a0 + kk * 16 * 128, kABytes / 2, 1024);
        else  // K-major A: 32 bytes of K per step inside the 128-byte rows
          da = sdesc_sw128(a0 + kk * 32, 16, 1024);
        mma_ss(tmem, da, db + ((kk * 32) >> 4), idesc, (k > 0 || kk > 0) ? 1u : 0u);
      }
      mma_commit(smem_u32(&ctl->empty[s]));
      if (k + stages < kChunks) {
        if (!mbar_wait<2>(smem_u32(&ctl->empty[s]), (k / stages) & 1, abort_flag, nullptr)) {
          ok = false;
          break;
        }
        load_a(k + stages, s);
        load_b(k + stages, s);
      }
    }
    mma_commit(smem_u32(&ctl->done));
    if (!ok) {
      // let every issued copy land before the CTA exits
      for (int k = 0; k < kChunks; ++k) {
        volatile int32_t never = 0;
        mbar_wait<2>(smem_u32(&ctl->full[k % stages]), (k / stages) & 1, &never, nullptr);
      }
    }
  }
  __syncwarp();
  // epilogue: thread = output feature (TMEM lane), columns = tokens
  volatile int32_t never = 0;
  const bool ok = __all_sync(0xffffffffu, mbar_wait<0>(smem_u32(&ctl->done), 0, &never, nullptr));
  tc_fence_after();
  if (ok) {
    const uint32_t lanes = static_cast<uint32_t>(warp * 32) << 16;
    const int feat = warp * 32 + lane;
    __nv_bfloat16* y = static_cast<__nv_bfloat16*>(p.y);
    for (int c = 0; c < n_tile; c += 32) {
      float v[32];
      tmem_ld32_sync(tmem + lanes + c, v);
#pragma unroll
      for (int k = 0; k < 32; ++k) {
        const int t = c + k;
        if (t < n_tok) {
          if constexpr (kKind == 0)
            y[(static_cast<int64_t>(t0 + t) * p.heads + h) * kDC + 128 * mslice + feat] = __float2bfloat16_rn(v[k]);
          else
            y[(static_cast<int64_t>(t0 + t) * p.heads + h) * kDV + feat] = __float2bfloat16_rn(v[k]);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, tmem_cols);
  }
}

// ------------------------------------------------------------------ merge + out_proj
//
// The step's tail in one kernel: the decode leaves S fp32 partial rows and
// log-sum-exps per (token, head); here each CTA (head h, up to kMpTok tokens)
// merges them ("Model Architecture Driving Inference Systems" §4.1, split KV
// with a log-sum-exp combine, the split merge kernel's arithmetic and order),
// writes u, and stages u in bf16 as the B operand of o^T = W_UV[h] u^T
// (§3.2). W_UV[h] (128 KB) is requested before the wait for the decode, so its
// stream from HBM overlaps the decode's tail and the merge. Sixteen warps merge
// (at two splits, two tokens each in flight per lane: the 32 tokens of a
// DeepSeek-V3 batch in one round trip); warps 0-3 read the accumulator back.
constexpr int kMpThreads = 512;
constexpr int kMpTok = 64;  // tokens per CTA (MMA N)

struct MergeProjCtl {
  uint64_t a_full;
  uint64_t done;
  uint32_t tmem_base;
  int32_t abort_flag;
};

template <int kS>
__global__ void __launch_bounds__(kMpThreads) out_proj_merge_kernel(const __grid_constant__ CUtensorMap amap,
                                                                   MergeProjArgs p, int n_tile, uint32_t tmem_cols) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  constexpr int kChunks = kDC / kChunkK;  // 8 K chunks of 64 latent columns
  uint8_t* a_s = base;                              // W_UV[h] chunk k at k * kABytes
  uint8_t* b_s = base + kChunks * kABytes;          // u chunk k at k * n_tile * 128 (token rows of 128 B)
  const int b_bytes = n_tile * 128;
  MergeProjCtl* ctl = reinterpret_cast<MergeProjCtl*>(b_s + kChunks * b_bytes);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.x;
  const int t0 = blockIdx.z * kMpTok;
  const int n_tok = min(kMpTok, p.n_tokens - t0);
  pdl_trigger();

  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&ctl->a_full), 1);
    mbar_init(smem_u32(&ctl->done), 1);
    ctl->abort_flag = 0;
    fence_mbar_init_cluster();
    prefetch_tmap(&amap);
  }
  if (warp == 0) tmem_alloc(smem_u32(&ctl->tmem_base), tmem_cols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;
  volatile int32_t* abort_flag = &ctl->abort_flag;
  if (threadIdx.x == 0) {
    // the weights are static: W_UV[h] rows d in [0, 128), all 512 columns, before the wait
    mbar_arrive_expect_tx(smem_u32(&ctl->a_full), kChunks * kABytes);
    for (int k = 0; k < kChunks; ++k)
      tma_load_2d_nohint(smem_u32(a_s + k * kABytes), &amap, smem_u32(&ctl->a_full), kChunkK * k, h * kDV);
  }
  pdl_wait();

  // ---- merge: warp w takes tokens w, w + 16, ... of the tile, kQ at a time;
  // lane = latent columns [16 lane, 16 lane + 16), i.e. K chunk lane / 4,
  // 16-byte chunks 2 (lane mod 4) and 2 (lane mod 4) + 1 of its 128-byte rows
  const uint64_t pol = l2_evict_first_policy();  // the partials are read once
  const int kc = lane >> 2, j0 = 2 * (lane & 3);
  constexpr int kQ = kS <= 2 ? 2 : 1;  // tokens in flight per lane (registers)
  for (int tp = warp; tp < n_tile; tp += kQ * (kMpThreads / 32)) {
    float ls[kQ][kS];
    float4 x[kQ][kS][4];
#pragma unroll
    for (int q = 0; q < kQ; ++q) {
      const int t = tp + q * (kMpThreads / 32);
      if (t < n_tok) {
        const int64_t bj = t0 + t;
#pragma unroll
        for (int s = 0; s < kS; ++s) {
          const int64_t row = (bj * kS + s) * p.heads + h;
          ls[q][s] = p.part_lse[row];
          const float4* src = reinterpret_cast<const float4*>(p.part_u + row * kDC + lane * 16);
#pragma unroll
          for (int v = 0; v < 4; ++v) x[q][s][v] = ld_global_v4_hint(src + v, pol);
        }
      }
    }
#pragma unroll
    for (int q = 0; q < kQ; ++q) {
      const int t = tp + q * (kMpThreads / 32);
      if (t >= n_tile) continue;
      uint32_t w[8];
      if (t < n_tok) {
        float mx = ls[q][0];
#pragma unroll
        for (int s = 1; s < kS; ++s) mx = fmaxf(mx, ls[q][s]);
        const bool none = (mx == -CUDART_INF_F);
        float sum = 0.0f;
        float acc[16];
#pragma unroll
        for (int k = 0; k < 16; ++k) acc[k] = 0.0f;
#pragma unroll
        for (int s = 0; s < kS; ++s) {
          const bool use = !none && ls[q][s] != -CUDART_INF_F;  // a -inf split is selected out, never multiplied
          const float wv = use ? fast_exp2((ls[q][s] - mx) * kLog2e) : 0.0f;
          sum += wv;
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            acc[4 * v] = use ? fmaf(wv, x[q][s][v].x, acc[4 * v]) : acc[4 * v];
            acc[4 * v + 1] = use ? fmaf(wv, x[q][s][v].y, acc[4 * v + 1]) : acc[4 * v + 1];
            acc[4 * v + 2] = use ? fmaf(wv, x[q][s][v].z, acc[4 * v + 2]) : acc[4 * v + 2];
            acc[4 * v + 3] = use ? fmaf(wv, x[q][s][v].w, acc[4 * v + 3]) : acc[4 * v + 3];
          }
        }
        const float inv = none ? 0.0f : 1.0f / sum;
#pragma unroll
        for (int k = 0; k < 8; ++k) w[k] = pack_bf16x2(acc[2 * k] * inv, acc[2 * k + 1] * inv);
        const int64_t orow = static_cast<int64_t>(t0 + t) * p.heads + h;
        uint4* ud = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.u_out) + orow * kDC + lane * 16);
        ud[0] = make_uint4(w[0], w[1], w[2], w[3]);
        ud[1] = make_uint4(w[4], w[5], w[6], w[7]);
        if (lane == 0 && p.lse_out != nullptr) p.lse_out[orow] = none ? -CUDART_INF_F : mx + logf(sum);
      } else {
#pragma unroll
        for (int k = 0; k < 8; ++k) w[k] = 0u;  // token rows past n: zero (their outputs are not written)
      }
      // the same bf16 values as the B operand, 128-byte swizzled token rows
      uint8_t* brow = b_s + kc * b_bytes + t * 128;
      *reinterpret_cast<uint4*>(brow + ((j0 ^ (t & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
      *reinterpret_cast<uint4*>(brow + (((j0 + 1) ^ (t & 7)) << 4)) = make_uint4(w[4], w[5], w[6], w[7]);
    }
  }
  fence_proxy_async_smem();  // generic writes of B, before the tensor core reads them
  __syncthreads();

  if (threadIdx.x == 0) {
    const uint32_t idesc = idesc_bf16_f32(128, n_tile, false, false);
    bool ok = mbar_wait<2>(smem_u32(&ctl->a_full), 0, abort_flag, nullptr);
    if (ok) {
      tc_fence_after();
      for (int k = 0; k < kChunks; ++k) {
        const uint32_t a0 = smem_u32(a_s + k * kABytes);
        const uint64_t db = sdesc_sw128(smem_u32(b_s + k * b_bytes), 16, 1024);
#pragma unroll
        for (int kk = 0; kk < kChunkK / 16; ++kk)
          mma_ss(tmem, sdesc_sw128(a0 + kk * 32, 16, 1024), db + ((kk * 32) >> 4), idesc, (k > 0 || kk > 0) ? 1u : 0u);
      }
    } else {
      // let W_UV's copies land before the CTA exits
      volatile int32_t never = 0;
      mbar_wait<2>(smem_u32(&ctl->a_full), 0, &never, nullptr);
    }
    mma_commit(smem_u32(&ctl->done));
  }
  __syncwarp();
  // epilogue (warps 0-3): thread = output feature d (TMEM lane), columns = tokens
  if (warp < 4) {
    volatile int32_t never = 0;
    const bool ok =
        __all_sync(0xffffffffu, mbar_wait<0>(smem_u32(&ctl->done), 0, &never, nullptr)) && *abort_flag == 0;
    tc_fence_after();
    const uint32_t lanes = static_cast<uint32_t>(warp * 32) << 16;
    const int feat = warp * 32 + lane;
    __nv_bfloat16* y = static_cast<__nv_bfloat16*>(p.o);
    for (int c = 0; c < n_tile; c += 32) {
      float v[32];
      tmem_ld32_sync(tmem + lanes + c, v);
#pragma unroll
      for (int k = 0; k < 32; ++k) {
        const int t = c + k;
        if (t < n_tok)  // an aborted call writes NaN, never stale values
          y[(static_cast<int64_t>(t0 + t) * p.heads + h) * kDV + feat] = __float2bfloat16_rn(ok ? v[k] : CUDART_NAN_F);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, tmem_cols);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

// 2D map over a [rows][cols] bf16 matrix with boxes of 64 columns x box_rows.
bool encode_2d(CUtensorMap* m, const void* ptr, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {64, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return encoder()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3D map over X[tokens][heads][width] bf16: boxes of 64 features x 1 head x box_tok tokens.
bool encode_3d(CUtensorMap* m, const void* ptr, uint64_t tokens, uint64_t heads, uint64_t width, uint32_t box_tok) {
  const cuuint64_t dims[3] = {width, heads, tokens};
  const cuuint64_t strides[2] = {width * 2, heads * width * 2};
  const cuuint32_t box[3] = {64, 1, box_tok};
  const cuuint32_t estr[3] = {1, 1, 1};
  return encoder()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int kKind>
cudaError_t launch_proj(const ProjArgs& a, cudaStream_t s) {
  if (a.act != MLA_BF16 || encoder() == nullptr) return cudaErrorNotSupported;
  if (a.n_tokens == 0) return cudaSuccess;
  const int n_tile = a.n_tokens >= kMaxTok ? kMaxTok : ((a.n_tokens + 15) / 16) * 16;
  uint32_t cols = 32;
  while (static_cast<int>(cols) < n_tile) cols <<= 1;
  const int b_bytes = ((n_tile * 128 + 1023) / 1024) * 1024;
  const int stage_bytes = kABytes + b_bytes;
  constexpr int kChunks = (kKind == 0 ? kDNope : kDC) / kChunkK;
  int stages = kChunks;
  while (stages > 2 && stages * stage_bytes > 160 * 1024) --stages;
  const size_t smem = 1024 + static_cast<size_t>(stages) * stage_bytes + sizeof(ProjCtl);
  CUtensorMap am, bm;
  bool ok;
  if constexpr (kKind == 0)
    ok = encode_2d(&am, a.w, static_cast<uint64_t>(a.heads) * kDNope, kDC, kChunkK) &&
         encode_3d(&bm, a.x, a.n_tokens, a.heads, kDNope, n_tile);
  else
    ok = encode_2d(&am, a.w, static_cast<uint64_t>(a.heads) * kDV, kDC, 128) &&
         encode_3d(&bm, a.x, a.n_tokens, a.heads, kDC, n_tile);
  if (!ok) return cudaErrorInvalidValue;
  static int attr_dev = -1;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (attr_dev != dev) {
    e = cudaFuncSetAttribute(proj_tc_kernel<kKind>, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
    if (e != cudaSuccess) return e;
    attr_dev = dev;
  }
  const dim3 grid(a.heads, kKind == 0 ? kDC / 128 : 1, (a.n_tokens + kMaxTok - 1) / kMaxTok);
  return launch_pdl(proj_tc_kernel<kKind>, grid, dim3(kThreads), smem, s, am, bm, a, n_tile, stages, cols);
}

}  // namespace

cudaError_t launch_absorb_tc(const ProjArgs& a, cudaStream_t s) { return launch_proj<0>(a, s); }
cudaError_t launch_out_proj_tc(const ProjArgs& a, cudaStream_t s) { return launch_proj<1>(a, s); }

bool out_proj_merge_supported(int32_t heads, int32_t splits, mla_dtype_t act) {
  return act == MLA_BF16 && heads >= 1 && splits >= 2 && splits <= 4 && encoder() != nullptr;
}

cudaError_t launch_out_proj_merge_tc(const MergeProjArgs& a, cudaStream_t s) {
  if (!out_proj_merge_supported(a.heads, a.num_splits, MLA_BF16)) return cudaErrorNotSupported;
  if (a.n_tokens == 0) return cudaSuccess;
  const int n_tile = a.n_tokens >= kMpTok ? kMpTok : ((a.n_tokens + 15) / 16) * 16;
  uint32_t cols = 32;
  while (static_cast<int>(cols) < n_tile) cols <<= 1;
  const size_t smem = 1024 + static_cast<size_t>(kDC / kChunkK) * (kABytes + n_tile * 128) + sizeof(MergeProjCtl);
  CUtensorMap am;
  if (!encode_2d(&am, a.w, static_cast<uint64_t>(a.heads) * kDV, kDC, 128)) return cudaErrorInvalidValue;
  static int attr_dev = -1;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (attr_dev != dev) {
    for (auto fn : {out_proj_merge_kernel<2>, out_proj_merge_kernel<3>, out_proj_merge_kernel<4>}) {
      e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
      if (e != cudaSuccess) return e;
    }
    attr_dev = dev;
  }
  const dim3 grid(a.heads, 1, (a.n_tokens + kMpTok - 1) / kMpTok);
  switch (a.num_splits) {
    case 2: return launch_pdl(out_proj_merge_kernel<2>, grid, dim3(kMpThreads), smem, s, am, a, n_tile, cols);
    case 3: return launch_pdl(out_proj_merge_kernel<3>, grid, dim3(kMpThreads), smem, s, am, a, n_tile, cols);
    default: return launch_pdl(out_proj_merge_kernel<4>, grid, dim3(kMpThreads), smem, s, am, a, n_tile, cols);
  }
}

}  // namespace mla
