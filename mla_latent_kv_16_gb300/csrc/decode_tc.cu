// Paged MLA decode on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
// What is computed ("Model Architecture Driving Inference Systems" §3.1-3.2;
// "Tech Radar: DeepSeek-V3 MLA" §2): for every head h of one query position,
//   s_t = (q_lat[h] . c_KV[t] + q_rope[h] . k_R[t]) * softmax_scale
//   u[h] = sum_t softmax(s)_t c_KV[t]
// In the decode ("MQA") form all 128 heads share the same 576-wide cached rows
// ("DeepSeek's attention evolution - [MLA]" §2.5), so the heads are the MMA M
// dimension: S[128 x 64] = Q[128 x 576] * C^T per 64-token tile, and
// O[128 x 512] += P[128 x 64] * C[64 x 512].
//
// GB300 mapping. O alone (128 x 512 fp32) fills a whole SM's TMEM, and Q
// (128 x 576 bf16) would fill most of its shared memory, so each work item is
// a cluster of two CTAs that split the row by columns:
//   CTA rank 0: latent columns [0, 256)          -> K slice of S, O[:, 0:256]
//   CTA rank 1: latent [256, 512) + RoPE [512, 576) -> K slice of S, O[:, 256:512]
// Each CTA TMA-loads only its own columns of every page (HBM is read once),
// keeps its Q slice in TMEM (A operand), computes a partial S, and the pair
// exchange partial S through distributed shared memory. Both then hold the
// same full S (fp32 addition is commutative), run the same online softmax
// and feed P (bf16, in TMEM) into their own half of the PV product.
//
// Warp roles (192 threads): warp 0 issues TMA loads (3-stage ring), warp 1
// allocates TMEM and issues the MMAs, warps 2-5 own TMEM lanes 0-127 (= heads)
// and run the exchange, the online softmax (running max with lazy rescale of
// O), the tail masking and the epilogue.
//
// Every wait is bounded: on a timeout the CTA raises an error bit, stops, waits
// for its own copies and MMAs, leaves the cluster barrier and frees TMEM.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <math_constants.h>

#include "common.cuh"
#include "launchers.h"
#include "tc_ptx.cuh"

namespace mla {
namespace {

using namespace tc;

constexpr int kThreads = 192;
constexpr int kTileTok = 64;
constexpr int kStages = 3;
constexpr int kBoxBytes = kTileTok * 128;  // 64 rows x 64 bf16, 128-byte swizzled
constexpr int kMaxBoxes = 5;
constexpr int kStageBytes = kMaxBoxes * kBoxBytes;
constexpr uint32_t kTmemCols = 512;
// TMEM column map (fp32 columns)
constexpr uint32_t kTmO = 0;    // O half: 256 columns
constexpr uint32_t kTmS = 256;  // S tile: 64 columns
constexpr uint32_t kTmP = 320;  // P tile: 64 bf16 = 32 columns
constexpr uint32_t kTmQ = 352;  // Q slice: 256 (+64) bf16 = 128 (+32) columns
// Lazy rescale: keep a stale row max until the new one exceeds it by 2^8.
constexpr float kRescaleLog2 = 8.0f;

struct __align__(1024) Smem {
  uint8_t stage[kStages][kStageBytes];
  float4 xbuf[2][kTileTok / 4][128];  // partial-S exchange slots: [slot][t/4][head]
  uint64_t kv_full[kStages];
  uint64_t kv_empty[kStages];
  uint64_t s_full, s_empty, p_full, pv_done, q_ready, drain;
  uint64_t x_full[2], x_empty[2];
  uint32_t tmem_base;
  int32_t abort_flag;
};

constexpr size_t kSmemBytes = sizeof(Smem) + 1024;

__device__ __forceinline__ void tmem_ld32_sync(uint32_t taddr, uint32_t (&r)[32]) {
  tmem_ld32(taddr, r);
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                 "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                 "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]),
                 "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]),
                 "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
               :
               : "memory");
}

// Wait bounded only by time (teardown: our own copies / MMAs must land).
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, int32_t* dev_error) {
  volatile int32_t never = 0;
  mbar_wait<false>(bar, parity, &never, dev_error);
}

// Outputs of a work item with nothing to attend to (or rejected data).
__device__ void write_empty(const DecodeArgs& a, int64_t row0, int bj, int split, uint32_t rank) {
  const int S = a.num_splits;
  if (S == 1) {
    uint4* u = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.u_out) + row0 * kDC + rank * 256);
    for (int i = threadIdx.x; i < 128 * 32; i += blockDim.x) u[(i >> 5) * (kDC / 8) + (i & 31)] = make_uint4(0, 0, 0, 0);
    if (rank == 0 && a.lse_out != nullptr)
      for (int h = threadIdx.x; h < 128; h += blockDim.x) a.lse_out[row0 + h] = -CUDART_INF_F;
  } else if (rank == 0) {
    for (int h = threadIdx.x; h < 128; h += blockDim.x)
      a.part_lse[(static_cast<int64_t>(bj) * S + split) * 128 + h] = -CUDART_INF_F;
  }
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    decode_tc_kernel(const __grid_constant__ CUtensorMap tmap, const DecodeArgs a) {
  extern __shared__ uint8_t smem_raw[];
  Smem* sm = reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const uint32_t peer = rank ^ 1u;

  // ---- work item: (sequence b, query j, split) -- identical in both CTAs
  const int item = blockIdx.x >> 1;
  const int Lq = a.q_len, S = a.num_splits, P = a.page_size;
  const int j = item % Lq;
  const int split = (item / Lq) % S;
  const int b = item / (Lq * S);
  const int bj = b * Lq + j;
  const int64_t row0 = static_cast<int64_t>(bj) * 128;
  const int L = a.seq_lens[b];
  const bool bad_len = (L < Lq) || (static_cast<int64_t>(L) > static_cast<int64_t>(a.max_pages) * P);
  if (bad_len && rank == 0 && threadIdx.x == 0) flag_error(a.dev_error, MLA_DEVERR_BAD_SEQLEN);
  const int n_vis = bad_len ? 0 : L - Lq + j + 1;
  const int tok_begin = split * a.pages_per_split * P;
  const int tok_end = min(n_vis, (split + 1) * a.pages_per_split * P);
  const int32_t* bt = a.block_table + static_cast<int64_t>(b) * a.max_pages;
  int n_tiles = 0;
  if (tok_begin < tok_end) {
    int local_bad = 0;
    for (int pg = tok_begin / P + static_cast<int>(threadIdx.x); pg <= (tok_end - 1) / P; pg += kThreads) {
      const int32_t pp = bt[pg];
      local_bad |= (pp < 0 || pp >= a.num_pages) ? 1 : 0;
    }
    if (__syncthreads_or(local_bad)) {
      if (rank == 0 && threadIdx.x == 0) flag_error(a.dev_error, MLA_DEVERR_BAD_PAGE);
    } else {
      n_tiles = (tok_end - tok_begin + kTileTok - 1) / kTileTok;
    }
  }
  if (n_tiles == 0) {
    write_empty(a, row0, bj, split, rank);
    return;
  }

  const uint32_t nbox = rank == 0 ? 4u : 5u;  // 64-column boxes this CTA loads
  const uint32_t col0 = rank * 256u;
  const uint32_t nk = nbox * 4u;             // K=16 MMA steps of the S slice

  // ---- set-up
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&sm->kv_full[s]), 1);
      mbar_init(smem_u32(&sm->kv_empty[s]), 1);
    }
    mbar_init(smem_u32(&sm->s_full), 1);
    mbar_init(smem_u32(&sm->s_empty), 128);
    mbar_init(smem_u32(&sm->p_full), 128);
    mbar_init(smem_u32(&sm->pv_done), 1);
    mbar_init(smem_u32(&sm->q_ready), 128);
    mbar_init(smem_u32(&sm->drain), 1);
    for (int x = 0; x < 2; ++x) {
      mbar_init(smem_u32(&sm->x_full[x]), 4);
      mbar_init(smem_u32(&sm->x_empty[x]), 4);
    }
    sm->abort_flag = 0;
    fence_mbar_init_cluster();
  }
  if (warp == 0 && lane == 0) prefetch_tmap(&tmap);
  if (warp == 1) tmem_alloc(smem_u32(&sm->tmem_base), kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cluster_sync();  // the peer's barriers exist before anything remote happens
  const uint32_t tmem = sm->tmem_base;
  volatile int32_t* abort_flag = &sm->abort_flag;

  if (warp == 0) {
    // ================= TMA producer
    if (lane == 0) {
      const uint64_t pol = l2_policy_evict_first();
      int issued = 0;
      for (int i = 0; i < n_tiles; ++i) {
        const int st = i % kStages;
        if (!mbar_wait<false>(smem_u32(&sm->kv_empty[st]), ((i / kStages) & 1) ^ 1, abort_flag, a.dev_error)) break;
        const int tok = tok_begin + i * kTileTok;
        const int32_t y = bt[tok / P] * P + (tok % P);
        const uint32_t bar = smem_u32(&sm->kv_full[st]);
        mbar_arrive_expect_tx(bar, nbox * kBoxBytes);
        const uint32_t dst = smem_u32(sm->stage[st]);
        for (uint32_t k = 0; k < nbox; ++k)
          tma_load_2d(dst + k * kBoxBytes, &tmap, bar, static_cast<int32_t>(col0 + 64u * k), y, pol);
        issued = i + 1;
      }
      for (int i = max(0, issued - kStages); i < issued; ++i)
        drain_wait(smem_u32(&sm->kv_full[i % kStages]), (i / kStages) & 1, a.dev_error);
    }
  } else if (warp == 1) {
    // ================= MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdQK = idesc_bf16_f32(128, kTileTok, false, false);
      constexpr uint32_t kIdPV = idesc_bf16_f32(128, 256, false, true);
      auto issue_pv = [&](int i) {
        const int st = i % kStages;
        const uint32_t base = smem_u32(sm->stage[st]);
#pragma unroll
        for (uint32_t kk = 0; kk < kTileTok / 16; ++kk)
          mma_ts(tmem + kTmO, tmem + kTmP + kk * 8u, sdesc_sw128(base + kk * 16u * 128u, kBoxBytes, 1024), kIdPV,
                 (i > 0 || kk > 0) ? 1u : 0u);
        mma_commit(smem_u32(&sm->kv_empty[st]));
        mma_commit(smem_u32(&sm->pv_done));
      };
      bool ok = mbar_wait<false>(smem_u32(&sm->q_ready), 0, abort_flag, a.dev_error);
      tc_fence_after();
      for (int i = 0; ok && i < n_tiles; ++i) {
        const int st = i % kStages;
        if (!mbar_wait<false>(smem_u32(&sm->kv_full[st]), (i / kStages) & 1, abort_flag, a.dev_error) ||
            (i > 0 && !mbar_wait<false>(smem_u32(&sm->s_empty), (i - 1) & 1, abort_flag, a.dev_error))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t base = smem_u32(sm->stage[st]);
        for (uint32_t kk = 0; kk < nk; ++kk)
          mma_ts(tmem + kTmS, tmem + kTmQ + kk * 8u,
                 sdesc_sw128(base + (kk >> 2) * kBoxBytes + (kk & 3u) * 32u, 16, 1024), kIdQK, kk > 0 ? 1u : 0u);
        mma_commit(smem_u32(&sm->s_full));
        if (i > 0) {
          if (!mbar_wait<false>(smem_u32(&sm->p_full), (i - 1) & 1, abort_flag, a.dev_error)) {
            ok = false;
            break;
          }
          tc_fence_after();
          issue_pv(i - 1);
        }
      }
      if (ok && mbar_wait<false>(smem_u32(&sm->p_full), (n_tiles - 1) & 1, abort_flag, a.dev_error)) {
        tc_fence_after();
        issue_pv(n_tiles - 1);
      }
      mma_commit(smem_u32(&sm->drain));
      drain_wait(smem_u32(&sm->drain), 0, a.dev_error);
    }
  } else {
    // ================= softmax / exchange / epilogue (thread = head = TMEM lane)
    const uint32_t q4 = static_cast<uint32_t>(warp & 3);
    const int h = static_cast<int>(q4 * 32u) + lane;
    const uint32_t lanes = (q4 * 32u) << 16;
    const uint32_t tS = tmem + lanes + kTmS, tP = tmem + lanes + kTmP, tO = tmem + lanes + kTmO;
    const uint32_t tQ = tmem + lanes + kTmQ;
    auto wwait = [&](uint64_t* bar, uint32_t par) {
      return __all_sync(0xffffffffu, mbar_wait<false>(smem_u32(bar), par, abort_flag, a.dev_error));
    };
    auto wwait_cluster = [&](uint64_t* bar, uint32_t par) {
      return __all_sync(0xffffffffu, mbar_wait<true>(smem_u32(bar), par, abort_flag, a.dev_error));
    };
    // Q slice of this head into TMEM (bf16 pairs, lower K index in the low half)
    {
      const uint4* ql = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.q_lat) + (row0 + h) * kDC + col0);
      uint32_t r[32];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
#pragma unroll
        for (int v = 0; v < 8; ++v) {
          const uint4 x = ql[c * 8 + v];
          r[4 * v] = x.x;
          r[4 * v + 1] = x.y;
          r[4 * v + 2] = x.z;
          r[4 * v + 3] = x.w;
        }
        tmem_st32(tQ + c * 32u, r);
      }
      if (rank == 1) {
        const uint4* qr = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.q_rope) + (row0 + h) * kDRope);
#pragma unroll
        for (int v = 0; v < 8; ++v) {
          const uint4 x = qr[v];
          r[4 * v] = x.x;
          r[4 * v + 1] = x.y;
          r[4 * v + 2] = x.z;
          r[4 * v + 3] = x.w;
        }
        tmem_st32(tQ + 128u, r);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(smem_u32(&sm->q_ready));
    }
    const float c2 = a.softmax_scale * kLog2e;  // scores in log2 units
    float m = -CUDART_INF_F, l = 0.0f;
    const uint32_t xbuf_peer = map_to_rank(smem_u32(&sm->xbuf[0][0][0]), peer);
    bool ok = true;
    for (int i = 0; i < n_tiles; ++i) {
      if (!wwait(&sm->s_full, i & 1)) { ok = false; break; }
      tc_fence_after();
      float s[64];
      {
        uint32_t r[32];
        tmem_ld32_sync(tS, r);
#pragma unroll
        for (int k = 0; k < 32; ++k) s[k] = __uint_as_float(r[k]);
        tmem_ld32_sync(tS + 32u, r);
#pragma unroll
        for (int k = 0; k < 32; ++k) s[32 + k] = __uint_as_float(r[k]);
      }
      tc_fence_before();
      mbar_arrive(smem_u32(&sm->s_empty));

      // ---- exchange partial scores with the peer CTA
      const int xs = i & 1;
      const uint32_t xph = (i >> 1) & 1;
      if (!wwait(&sm->x_empty[xs], xph ^ 1u)) { ok = false; break; }
#pragma unroll
      for (int q = 0; q < 16; ++q)
        st_cluster_v4(xbuf_peer + static_cast<uint32_t>(((xs * 16 + q) * 128 + h) * 16), s[4 * q], s[4 * q + 1],
                      s[4 * q + 2], s[4 * q + 3]);
      fence_acq_rel_cluster();
      __syncwarp();
      if (lane == 0) mbar_arrive_remote(map_to_rank(smem_u32(&sm->x_full[xs]), peer));
      if (!wwait_cluster(&sm->x_full[xs], xph)) { ok = false; break; }
#pragma unroll
      for (int q = 0; q < 16; ++q) {
        const float4 v = sm->xbuf[xs][q][h];
        s[4 * q] += v.x;
        s[4 * q + 1] += v.y;
        s[4 * q + 2] += v.z;
        s[4 * q + 3] += v.w;
      }
      fence_acq_rel_cluster();
      __syncwarp();
      if (lane == 0) mbar_arrive_remote(map_to_rank(smem_u32(&sm->x_empty[xs]), peer));

      // ---- online softmax over this tile (identical in both CTAs)
      const int tok0 = tok_begin + i * kTileTok;
      const int valid = min(kTileTok, tok_end - tok0);
      float mx = -CUDART_INF_F;
#pragma unroll
      for (int t = 0; t < 64; ++t) {
        if (t >= valid) s[t] = -CUDART_INF_F;
        mx = fmaxf(mx, s[t]);
      }
      const bool first = (i == 0);
      const float m_new = fmaxf(m, mx * c2);
      const bool resc = !first && (m_new > m + kRescaleLog2);
      const float m_use = (first || resc) ? m_new : m;
      const float alpha = resc ? fast_exp2(m - m_use) : 1.0f;
      float rs = 0.0f;
      uint32_t pw[32];
#pragma unroll
      for (int t = 0; t < 32; ++t) {
        const float p0 = fast_exp2(fmaf(s[2 * t], c2, -m_use));
        const float p1 = fast_exp2(fmaf(s[2 * t + 1], c2, -m_use));
        rs += p0 + p1;
        pw[t] = pack_bf16x2(p0, p1);
      }
      l = l * alpha + rs;
      m = m_use;
      if (!first) {
        if (!wwait(&sm->pv_done, (i - 1) & 1)) { ok = false; break; }
        tc_fence_after();
      }
      if (__any_sync(0xffffffffu, resc)) {
        for (int c = 0; c < 8; ++c) {
          uint32_t r[32];
          tmem_ld32_sync(tO + c * 32u, r);
#pragma unroll
          for (int k = 0; k < 32; ++k) r[k] = __float_as_uint(__uint_as_float(r[k]) * alpha);
          tmem_st32(tO + c * 32u, r);
        }
        tmem_wait_st();
      }
      if (valid < kTileTok) {
        // rows past the sequence end may hold anything (NaN): zero them in the
        // V columns so that 0 * row stays 0 in the PV product
        uint4* base = reinterpret_cast<uint4*>(sm->stage[i % kStages]);
        const int rows = kTileTok - valid;
        for (int e = h; e < rows * 4 * 8; e += 128) {
          const int box = e / (rows * 8), rem = e % (rows * 8);
          base[(box * kBoxBytes + (valid + rem / 8) * 128) / 16 + (rem % 8)] = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
        __syncwarp();
      }
      tmem_st32(tP, pw);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(smem_u32(&sm->p_full));
    }
    // ---- epilogue: u = O / l (this CTA's 256 columns), lse
    if (ok && wwait(&sm->pv_done, (n_tiles - 1) & 1)) {
      tc_fence_after();
      const float inv_l = 1.0f / l;
      const float lse = (m + log2f(l)) * kLn2;
      if (S == 1) {
        uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.u_out) + (row0 + h) * kDC + col0);
        for (int c = 0; c < 8; ++c) {
          uint32_t r[32];
          tmem_ld32_sync(tO + c * 32u, r);
          uint32_t w[16];
#pragma unroll
          for (int k = 0; k < 16; ++k)
            w[k] = pack_bf16x2(__uint_as_float(r[2 * k]) * inv_l, __uint_as_float(r[2 * k + 1]) * inv_l);
#pragma unroll
          for (int v = 0; v < 4; ++v) dst[c * 4 + v] = make_uint4(w[4 * v], w[4 * v + 1], w[4 * v + 2], w[4 * v + 3]);
        }
        if (rank == 0 && a.lse_out != nullptr) a.lse_out[row0 + h] = lse;
      } else {
        const int64_t prow = (static_cast<int64_t>(bj) * S + split) * 128 + h;
        float4* dst = reinterpret_cast<float4*>(a.part_u + prow * kDC + col0);
        for (int c = 0; c < 8; ++c) {
          uint32_t r[32];
          tmem_ld32_sync(tO + c * 32u, r);
#pragma unroll
          for (int v = 0; v < 8; ++v)
            dst[c * 8 + v] = make_float4(__uint_as_float(r[4 * v]) * inv_l, __uint_as_float(r[4 * v + 1]) * inv_l,
                                         __uint_as_float(r[4 * v + 2]) * inv_l,
                                         __uint_as_float(r[4 * v + 3]) * inv_l);
        }
        if (rank == 0) a.part_lse[prow] = lse;
      }
    }
  }

  // ---- teardown: both CTAs are done with each other's shared memory
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

}  // namespace

bool decode_tc_supported(const DecodeArgs& a) {
  return a.heads == 128 && a.act == MLA_BF16 && a.cache_dtype == MLA_BF16 && a.page_size % kTileTok == 0 &&
         (reinterpret_cast<uintptr_t>(a.cache) & 15u) == 0 &&
         a.num_pages * static_cast<int64_t>(a.page_size) < (int64_t(1) << 31) && tensor_map_encoder() != nullptr;
}

cudaError_t launch_decode_tc(const DecodeArgs& a, cudaStream_t s) {
  CUtensorMap map;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(kRow), static_cast<cuuint64_t>(a.num_pages * a.page_size)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(kRow) * 2};
  const cuuint32_t box[2] = {64, kTileTok};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = tensor_map_encoder()(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(a.cache), dims,
                                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(decode_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kSmemBytes));
  if (e != cudaSuccess) return e;
  const int64_t items = static_cast<int64_t>(a.batch) * a.q_len * a.num_splits;
  decode_tc_kernel<<<dim3(static_cast<unsigned>(2 * items)), kThreads, kSmemBytes, s>>>(map, a);
  return cudaGetLastError();
}

}  // namespace mla
