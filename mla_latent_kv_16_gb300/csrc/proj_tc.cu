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

}  // namespace mla
