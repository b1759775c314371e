// Generic linear layer y[t][o] = sum_i W[o][i] x[t][i] for the few tokens of
// a decode step (nn.Linear layout: W is [n_out][n_in], row-major). At decode
// batch sizes this is a stream of W from HBM and nothing else matters.
//
// The tcgen05 kernel (bf16, n_in % 64 == 0) takes 128 rows of W as the MMA M
// dimension and up to 256 tokens as N, and splits the n_in (K) dimension so
// that there are enough work units (row tile x K split x token tile) for every
// SM. It is persistent, one CTA per SM: a producer warp streams all of the
// CTA's units through one TMA ring of 64-wide K chunks (a 128 x 64 box of W
// and an n x 64 box of x, both 128-byte swizzled) without a break between
// units, an MMA warp accumulates each unit in one of two TMEM buffers, and four
// epilogue warps empty the other. Rows of W past n_out read as zero and are
// not written. With many tokens (512 or more, n_out % 8 == 0: a prefill's
// expansion of the latent rows) the roles swap: 128 tokens are M and 256 rows
// of W are N, K whole, so that each epilogue thread writes one token's 256
// outputs as 16-byte vectors. With a K split (or when the caller asks for fp32 sums) the
// partial sums go to an fp32 workspace and a second kernel adds them in split
// order, so results do not depend on timing. Other types and shapes run on
// CUDA cores.
//
// Users: the fused output projection ("Model Architecture Driving Inference
// Systems" §3.2, y = W~^O u over all heads) and the decode-layer front end's
// projections ("Multi-Head Latent Attention (MLA)" page, "PyTorch Reference
// Implementation": W_DQ, W_DKV, W_KR on h; W_UQ, W_QR on c_q).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <math_constants.h>

#include "common.cuh"
#include "launchers.h"
#include "tc_ptx.cuh"

namespace mla {
namespace {

using namespace tc;

constexpr int kThreads = 192;      // producer warp, MMA warp, four epilogue warps
constexpr int kMaxTok = 256;       // tokens per unit (MMA N)
constexpr int kChunkK = 64;        // K elements per TMA box (128 bytes of bf16)
constexpr int kABytes = 128 * 128;  // one W box: 128 rows x 64 bf16
constexpr int kMaxStages = 12;
constexpr int kMaxSplits = 32;
constexpr int kRingBudget = 200 * 1024;  // shared memory for the TMA ring
// Many tokens (a prefill's expansion of the latent rows): the roles swap, 128
// tokens are the MMA M dimension and 256 rows of W are N, so that a thread of
// the epilogue holds 256 consecutive outputs of one token and writes them as
// 16-byte vectors (with rows of W as M, a warp's store covers 32 outputs x 2
// bytes of one token).
constexpr int kTmMinTok = 512;
constexpr int kTmOut = 256;
// Epilogue staging with tokens as M: each epilogue warp's 32 tokens x 64
// outputs (bf16, 4 KB), so that its stores cover whole 128-byte row segments.
constexpr int kEpiStageBytes = 4 * 4096;

struct LinearCtl {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  uint64_t acc_full[2];
  uint64_t acc_empty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int32_t abort_flag;
};

// ------------------------------------------------------------------ CUDA cores

// grid (ceil(n_out/8), min(ceil(n/8), 65535)), block 256: warp = one row o of W
// against 8 tokens at a time (token tiles strided by the grid's y extent);
// lanes stride K. Writes y, or fp32 sums to part[0] when part is set.
template <typename T>
__global__ void __launch_bounds__(256) linear_simt_kernel(LinearArgs p) {
  pdl_trigger();
  pdl_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int o = blockIdx.x * 8 + warp;
  if (o >= p.n_out) return;
  const int64_t K = p.n_in;
  const T* w = static_cast<const T*>(p.w) + static_cast<int64_t>(o) * K;
  for (int t0 = blockIdx.y * 8; t0 < p.n_tokens; t0 += gridDim.y * 8) {
    const int nt = min(8, p.n_tokens - t0);
    const T* x = static_cast<const T*>(p.x) + static_cast<int64_t>(t0) * K;
    float acc[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[j] = 0.0f;
    for (int64_t k = lane; k < K; k += 32) {
      const float wv = ActIO<T>::load(w + k);
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (j < nt) acc[j] = fmaf(wv, ActIO<T>::load(x + j * K + k), acc[j]);
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float s = warp_sum(acc[j]);
      if (lane == 0 && j < nt) {
        const int64_t idx = static_cast<int64_t>(t0 + j) * p.n_out + o;
        if (p.part != nullptr)
          p.part[idx] = s;
        else
          ActIO<T>::store(static_cast<T*>(p.y) + idx, s);
      }
    }
  }
}

// ------------------------------------------------------------------ tcgen05

// A work unit is (128 rows of W, K split, token tile). The unit's coordinates.
struct Unit {
  int o0, split, t0, c_lo, nc;
};

__device__ __forceinline__ Unit unit_at(const LinearArgs& p, int u, int o_tiles, int chunks, bool tm) {
  Unit r;
  if (tm) {
    // tokens as M: 128 tokens x 256 rows of W, K whole
    const int ot = (p.n_out + kTmOut - 1) / kTmOut;
    r.o0 = (u % ot) * kTmOut;
    r.t0 = (u / ot) * 128;
    r.split = 0;
    r.c_lo = 0;
    r.nc = chunks;
    return r;
  }
  const int rest = u / o_tiles;
  r.o0 = (u - rest * o_tiles) * 128;
  r.split = rest % p.k_splits;
  r.t0 = (rest / p.k_splits) * kMaxTok;
  r.c_lo = static_cast<int>(static_cast<int64_t>(r.split) * chunks / p.k_splits);
  r.nc = static_cast<int>(static_cast<int64_t>(r.split + 1) * chunks / p.k_splits) - r.c_lo;
  return r;
}

// Persistent: grid = min(units, SMs), one CTA per SM, CTA c takes units c, c + G,
// c + 2G, ... Warp 0 (one lane) streams every chunk of those units through the
// TMA ring without a break between units; warp 1 (one lane) issues the MMAs
// into one of two TMEM accumulators; warps 2-5 read back the other (warp w owns
// TMEM lanes 32 (w % 4) .. +32, thread = row of W) and write the unit's output.
__global__ void __launch_bounds__(kThreads, 1) linear_tc_kernel(const __grid_constant__ CUtensorMap amap,
                                                                const __grid_constant__ CUtensorMap bmap,
                                                                LinearArgs p, int n_tile, int stages,
                                                                uint32_t acc_cols, int units, int tm_flag) {
  const bool tm = tm_flag != 0;  // tokens as M (x in the A slot, W in the B slot of each stage)
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int b_bytes = n_tile * 128;
  const int stage_bytes = kABytes + ((b_bytes + 1023) & ~1023);
  uint8_t* epi_stage = base + stages * stage_bytes;  // tokens as M: the epilogue warps' staging
  LinearCtl* ctl = reinterpret_cast<LinearCtl*>(epi_stage + (tm ? kEpiStageBytes : 0));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int o_tiles = (p.n_out + 127) / 128;
  const int chunks = p.n_in / kChunkK;
  pdl_trigger();

  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(smem_u32(&ctl->full[s]), 1);
      mbar_init(smem_u32(&ctl->empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&ctl->acc_full[b]), 1);
      mbar_init(smem_u32(&ctl->acc_empty[b]), 4);  // the four epilogue warps
    }
    mbar_init(smem_u32(&ctl->drain), 1);
    ctl->abort_flag = 0;
    fence_mbar_init_cluster();
    prefetch_tmap(&amap);
    prefetch_tmap(&bmap);
  }
  if (warp == 0) tmem_alloc(smem_u32(&ctl->tmem_base), 2 * acc_cols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;
  volatile int32_t* abort_flag = &ctl->abort_flag;
  // Everything below reads or writes data of earlier kernels, except W when the
  // caller vouches that no kernel still running writes it (w_static): then the
  // producer requests the first ring of W before its wait.
  const bool producer = warp == 0 && lane == 0;
  if (!producer) pdl_wait();

  if (warp == 0) {
    if (lane == 0) {
      // ---- TMA producer. W is read once when all tokens fit one tile (x then stays in L2).
      const bool once = p.n_tokens <= kMaxTok;
      const uint64_t pol = l2_policy_evict_first();
      auto load_w = [&](uint32_t dst, uint32_t bar, int32_t xk, int32_t o0) {
        if (once)
          tma_load_2d(dst, &amap, bar, xk, o0, pol);  // rows past n_out read as zero
        else
          tma_load_2d_nohint(dst, &amap, bar, xk, o0);
      };
      uint32_t pre = 0;  // chunks whose W box was requested before the wait
      if (p.w_static && !tm) {
        for (int u = blockIdx.x; u < units && pre < static_cast<uint32_t>(stages); u += gridDim.x) {
          const Unit w = unit_at(p, u, o_tiles, chunks, tm);
          for (int k = 0; k < w.nc && pre < static_cast<uint32_t>(stages); ++k, ++pre) {
            const uint32_t bar = smem_u32(&ctl->full[pre]);
            mbar_arrive_expect_tx(bar, kABytes + b_bytes);
            load_w(smem_u32(base + pre * stage_bytes), bar, (w.c_lo + k) * kChunkK, w.o0);
          }
        }
      }
      pdl_wait();
      uint32_t g = 0;  // chunks issued so far, over all of this CTA's units
      bool ok = true;
      for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
        const Unit w = unit_at(p, u, o_tiles, chunks, tm);
        for (int k = 0; k < w.nc; ++k, ++g) {
          const int s = static_cast<int>(g % stages);
          const uint32_t dst = smem_u32(base + s * stage_bytes);
          const uint32_t bar = smem_u32(&ctl->full[s]);
          const int32_t xk = (w.c_lo + k) * kChunkK;
          if (g >= pre) {
            if (g >= static_cast<uint32_t>(stages) &&
                !mbar_wait<2>(smem_u32(&ctl->empty[s]), ((g / stages) & 1) ^ 1, abort_flag, nullptr)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(bar, kABytes + b_bytes);
            if (tm)
              tma_load_2d_nohint(dst + kABytes, &amap, bar, xk, w.o0);  // 256 rows of W as B (past n_out: zero)
            else
              load_w(dst, bar, xk, w.o0);
          }
          if (tm)
            tma_load_2d_nohint(dst, &bmap, bar, xk, w.t0);  // 128 tokens of x as A (past n: zero)
          else
            tma_load_2d_nohint(dst + kABytes, &bmap, bar, xk, w.t0);  // token rows past n read as zero
        }
      }
      if (!ok) {
        // after an abort nobody consumes: let the last copy issued into each slot land
        volatile int32_t never = 0;
        const uint32_t first = g > static_cast<uint32_t>(stages) ? g - stages : 0;
        for (uint32_t q = first; q < g; ++q)
          mbar_wait<2>(smem_u32(&ctl->full[q % stages]), (q / stages) & 1, &never, nullptr);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---- MMA issuer
      const uint32_t idesc = idesc_bf16_f32(128, n_tile, false, false);
      uint32_t g = 0;
      bool ok = true;
      int i = 0;
      for (int u = blockIdx.x; u < units && ok; u += gridDim.x, ++i) {
        const Unit w = unit_at(p, u, o_tiles, chunks, tm);
        const int b = i & 1;
        if (i >= 2 && !mbar_wait<2>(smem_u32(&ctl->acc_empty[b]), ((i >> 1) - 1) & 1, abort_flag, nullptr)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem + static_cast<uint32_t>(b) * acc_cols;
        for (int k = 0; k < w.nc; ++k, ++g) {
          const int s = static_cast<int>(g % stages);
          if (!mbar_wait<2>(smem_u32(&ctl->full[s]), (g / stages) & 1, abort_flag, nullptr)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_u32(base + s * stage_bytes);
          const uint64_t db = sdesc_sw128(a0 + kABytes, 16, 1024);
#pragma unroll
          for (int kk = 0; kk < kChunkK / 16; ++kk)
            mma_ss(d, sdesc_sw128(a0 + kk * 32, 16, 1024), db + ((kk * 32) >> 4), idesc,
                   (k > 0 || kk > 0) ? 1u : 0u);
          mma_commit(smem_u32(&ctl->empty[s]));
        }
        if (ok) mma_commit(smem_u32(&ctl->acc_full[b]));
      }
      // every MMA this thread issued completes before the TMEM is freed
      mma_commit(smem_u32(&ctl->drain));
      volatile int32_t never = 0;
      mbar_wait<2>(smem_u32(&ctl->drain), 0, &never, nullptr);
    }
  } else {
    // ---- epilogue (warps 2-5)
    const int q = warp & 3;
    const uint32_t lanes = static_cast<uint32_t>(q * 32) << 16;
    bool ok = true;
    int i = 0;
    for (int u = blockIdx.x; u < units; u += gridDim.x, ++i) {
      const Unit w = unit_at(p, u, o_tiles, chunks, tm);
      const int b = i & 1;
      const bool got =
          __all_sync(0xffffffffu, ok && mbar_wait<0>(smem_u32(&ctl->acc_full[b]), (i >> 1) & 1, abort_flag, nullptr));
      ok = got;
      tc_fence_after();
      if (tm) {
        // thread = token (TMEM lane) while reading TMEM, 64 outputs at a time. bf16
        // outputs are staged in shared memory (16-byte chunk j of token row r at
        // chunk j ^ (r mod 8), against bank conflicts) and stored as whole 128-byte
        // row segments, four tokens per warp-wide store; a warp storing one 16-byte
        // vector per token instead touched 32 rows per store. n_out % 8 == 0: a
        // chunk of 8 outputs is all in or all out.
        uint8_t* st = epi_stage + (warp - 2) * 4096;
        const int tok0 = w.t0 + q * 32;
        for (int c = 0; c < kTmOut; c += 64) {
          float v[64];
          if (got) {
            tmem_ld64_sync(tmem + static_cast<uint32_t>(b) * acc_cols + lanes + c, v);
          } else {
#pragma unroll
            for (int k = 0; k < 64; ++k) v[k] = CUDART_NAN_F;  // an aborted unit reads as NaN
          }
          if (p.part == nullptr) {
#pragma unroll
            for (int j = 0; j < 8; ++j)
              *reinterpret_cast<uint4*>(st + lane * 128 + ((j ^ (lane & 7)) << 4)) =
                  make_uint4(pack_bf16x2(v[8 * j], v[8 * j + 1]), pack_bf16x2(v[8 * j + 2], v[8 * j + 3]),
                             pack_bf16x2(v[8 * j + 4], v[8 * j + 5]), pack_bf16x2(v[8 * j + 6], v[8 * j + 7]));
            __syncwarp();
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              const int row = 4 * k + (lane >> 3), j = lane & 7;
              const int tok = tok0 + row, o = w.o0 + c + 8 * j;
              const uint4 x = *reinterpret_cast<const uint4*>(st + row * 128 + ((j ^ (row & 7)) << 4));
              if (tok < p.n_tokens && o < p.n_out)
                *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.y) + static_cast<int64_t>(tok) * p.n_out + o) = x;
            }
            __syncwarp();  // the staging area is rewritten by the next 64 outputs
          } else {
            const int tok = tok0 + lane;  // fp32 sums, thread = token
            if (tok >= p.n_tokens) continue;
#pragma unroll
            for (int g8 = 0; g8 < 8; ++g8) {
              const int o = w.o0 + c + 8 * g8;
              if (o >= p.n_out) break;
              float4* d = reinterpret_cast<float4*>(p.part + static_cast<int64_t>(tok) * p.n_out + o);
              d[0] = make_float4(v[8 * g8], v[8 * g8 + 1], v[8 * g8 + 2], v[8 * g8 + 3]);
              d[1] = make_float4(v[8 * g8 + 4], v[8 * g8 + 5], v[8 * g8 + 6], v[8 * g8 + 7]);
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (got && lane == 0) mbar_arrive(smem_u32(&ctl->acc_empty[b]));
        continue;
      }
      const int n_tok = min(kMaxTok, p.n_tokens - w.t0);
      const int o = w.o0 + q * 32 + lane;
      for (int c = 0; c < n_tile; c += 32) {
        float v[32];
        if (got) {
          tmem_ld32_sync(tmem + static_cast<uint32_t>(b) * acc_cols + lanes + c, v);
        } else {
#pragma unroll
          for (int k = 0; k < 32; ++k) v[k] = 0.0f;
        }
        if (o >= p.n_out) continue;
#pragma unroll
        for (int k = 0; k < 32; ++k) {
          const int t = c + k;
          if (t >= n_tok) break;
          const float val = got ? v[k] : CUDART_NAN_F;  // an aborted unit reads as NaN, never as stale data
          const int64_t row = w.t0 + t;
          if (p.part == nullptr)
            static_cast<__nv_bfloat16*>(p.y)[row * p.n_out + o] = __float2bfloat16_rn(val);
          else
            p.part[(static_cast<int64_t>(w.split) * p.n_tokens + row) * p.n_out + o] = val;
        }
      }
      tc_fence_before();
      __syncwarp();
      if (got && lane == 0) mbar_arrive(smem_u32(&ctl->acc_empty[b]));
    }
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 2 * acc_cols);
  }
}

// y = sum over splits s = 0, 1, ... of part[s], one output per thread.
template <typename T>
__global__ void __launch_bounds__(256) linear_reduce_kernel(LinearArgs p) {
  pdl_trigger();
  pdl_wait();
  const int64_t n = static_cast<int64_t>(p.n_tokens) * p.n_out;
  const int64_t i = static_cast<int64_t>(blockIdx.x) * 256 + threadIdx.x;
  if (i >= n) return;
  ActIO<T>::store(static_cast<T*>(p.y) + i, split_sum(p.part, i, n, p.k_splits));
}

// ------------------------------------------------------------------ host side

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

// 2D map over a [rows][cols] bf16 matrix (row stride `stride` elements, 0 =
// cols), boxes of 64 columns x box_rows.
bool encode_2d(CUtensorMap* m, const void* ptr, uint64_t rows, uint64_t cols, uint32_t box_rows,
               uint64_t stride = 0) {
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {(stride != 0 ? stride : cols) * 2};
  const cuuint32_t box[2] = {64, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return encoder()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool use_tc(int32_t n_in, mla_dtype_t act) { return act == MLA_BF16 && n_in % kChunkK == 0; }

struct LinearPlan {
  int n_tile;         // MMA N (tokens per unit, multiple of 16)
  int tok_tiles;      // units along the tokens
  int stages;         // TMA ring depth
  int splits;         // units along K
  int units;          // row tiles x splits x token tiles
  int grid;           // persistent CTAs: min(units, SMs)
  size_t smem;        // dynamic shared memory per CTA
  uint32_t acc_cols;  // TMEM columns of one of the two accumulators
  bool tm;            // tokens as M (many tokens)
};

// Tile shape, ring depth and K split of the persistent tcgen05 kernel. One CTA
// per SM streams its units back to back, so the split count minimises the
// chunks the busiest CTA streams: units per CTA (rounded up) x (chunks per unit
// + about one chunk's worth of partial-sum traffic).
LinearPlan plan_tc(int32_t n_tokens, int32_t n_out, int32_t n_in) {
  LinearPlan p{};
  if (n_tokens >= kTmMinTok && n_out % 8 == 0) {
    // tokens as M: units of 128 tokens x 256 rows of W, K whole
    p.tm = true;
    p.n_tile = kTmOut;
    p.tok_tiles = (n_tokens + 127) / 128;
    const int stage = kABytes + kTmOut * 128;
    p.stages = kRingBudget / stage;
    if (p.stages > kMaxStages) p.stages = kMaxStages;
    p.smem = 1024 + static_cast<size_t>(p.stages) * stage + kEpiStageBytes + sizeof(LinearCtl);
    p.acc_cols = kTmOut;
    p.splits = 1;
    const int64_t units = static_cast<int64_t>(p.tok_tiles) * ((n_out + kTmOut - 1) / kTmOut);
    const int64_t sms = device_sm_count();
    p.units = static_cast<int>(units);
    p.grid = static_cast<int>(units < sms ? units : sms);
    return p;
  }
  p.n_tile = n_tokens >= kMaxTok ? kMaxTok : ((n_tokens + 15) / 16) * 16;
  p.tok_tiles = (n_tokens + kMaxTok - 1) / kMaxTok;
  const int stage = kABytes + ((p.n_tile * 128 + 1023) & ~1023);
  p.stages = kRingBudget / stage;
  if (p.stages > kMaxStages) p.stages = kMaxStages;
  p.smem = 1024 + static_cast<size_t>(p.stages) * stage + sizeof(LinearCtl);
  p.acc_cols = 32;
  while (static_cast<int>(p.acc_cols) < p.n_tile) p.acc_cols <<= 1;
  const int chunks = n_in / kChunkK;
  const int64_t tiles = static_cast<int64_t>((n_out + 127) / 128) * p.tok_tiles;
  const int64_t sms = device_sm_count();
  double best = 1e300;
  p.splits = 1;
  for (int s = 1; s <= kMaxSplits && s <= chunks; ++s) {
    const int per = (chunks + s - 1) / s;
    if (s > 1 && per < 8) break;
    const int64_t per_cta = (tiles * s + sms - 1) / sms;
    const double cost = static_cast<double>(per_cta) * (per + (s > 1 ? 1.0 : 0.0));
    if (cost < best - 1e-9) {
      best = cost;
      p.splits = s;
    }
  }
  const int64_t units = tiles * p.splits;
  p.units = static_cast<int>(units);
  p.grid = static_cast<int>(units < sms ? units : sms);
  return p;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace

int32_t linear_splits(int32_t n_tokens, int32_t n_out, int32_t n_in, mla_dtype_t act) {
  if (n_tokens < 1 || n_out < 1 || n_in < 1 || !use_tc(n_in, act)) return 1;
  return plan_tc(n_tokens, n_out, n_in).splits;
}

size_t linear_partial_bytes(int32_t n_tokens, int32_t n_out, int32_t n_in, mla_dtype_t act) {
  return align256(static_cast<size_t>(linear_splits(n_tokens, n_out, n_in, act)) * n_tokens * n_out *
                  sizeof(float));
}

cudaError_t launch_linear(const LinearArgs& a, cudaStream_t s, bool reduce) {
  if (a.n_tokens == 0) return cudaSuccess;
  if (a.x_stride != 0 && a.x_stride != a.n_in && (!use_tc(a.n_in, a.act) || a.x_stride < a.n_in || a.x_stride % 8))
    return cudaErrorInvalidValue;
  if (!use_tc(a.n_in, a.act)) {
    if (a.k_splits != 1) return cudaErrorInvalidValue;
    const int tok_tiles = (a.n_tokens + 7) / 8;
    const dim3 grid((a.n_out + 7) / 8, tok_tiles < 65535 ? tok_tiles : 65535);
    if (a.act == MLA_F32) return launch_pdl(linear_simt_kernel<float>, grid, dim3(256), 0, s, a);
    return launch_pdl(linear_simt_kernel<__nv_bfloat16>, grid, dim3(256), 0, s, a);
  }
  if (encoder() == nullptr) return cudaErrorNotSupported;
  const LinearPlan pl = plan_tc(a.n_tokens, a.n_out, a.n_in);
  if (pl.splits != a.k_splits || (pl.splits > 1 && a.part == nullptr)) return cudaErrorInvalidValue;
  CUtensorMap am, bm;
  // boxes: W rows 128 (as A) or 256 (as B, tokens as M); x rows n_tile (as B) or 128 (as A)
  if (!encode_2d(&am, a.w, static_cast<uint64_t>(a.n_out), static_cast<uint64_t>(a.n_in), pl.tm ? kTmOut : 128) ||
      !encode_2d(&bm, a.x, static_cast<uint64_t>(a.n_tokens), static_cast<uint64_t>(a.n_in),
                 pl.tm ? 128u : static_cast<uint32_t>(pl.n_tile), static_cast<uint64_t>(a.x_stride)))
    return cudaErrorInvalidValue;
  static int attr_dev = -1;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (attr_dev != dev) {
    e = cudaFuncSetAttribute(linear_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 220 * 1024);
    if (e != cudaSuccess) return e;
    attr_dev = dev;
  }
  e = launch_pdl(linear_tc_kernel, dim3(pl.grid), dim3(kThreads), pl.smem, s, am, bm, a, pl.n_tile, pl.stages,
                 pl.acc_cols, pl.units, pl.tm ? 1 : 0);
  if (e != cudaSuccess || a.part == nullptr || !reduce) return e;
  const int64_t n = static_cast<int64_t>(a.n_tokens) * a.n_out;
  if ((n + 255) / 256 > 0x7fffffff) return cudaErrorInvalidConfiguration;
  return launch_pdl(linear_reduce_kernel<__nv_bfloat16>, dim3(static_cast<unsigned>((n + 255) / 256)), dim3(256),
                    0, s, a);
}

}  // namespace mla
