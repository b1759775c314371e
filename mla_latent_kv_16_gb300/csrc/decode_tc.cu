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
// GB300 mapping. O alone (128 x 512 fp32) fills a whole SM's TMEM, so every
// work item (sequence, query, KV split) runs on two CTAs, one per half of the
// latent output: CTA "half" r accumulates O[:, 256r : 256r+256] in TMEM. Both
// CTAs compute the full score tile (the QK product is duplicated: exchanging
// 32 KB of fp32 partial scores per page between SMs would cost more than the
// MMAs it saves), so the pair never communicates. Q (128 x 576 bf16) is split
// between TMEM (latent 0-255 and RoPE 512-575: 160 columns, the A operand of
// those MMAs) and shared memory (latent 256-511, 64 KB). The two CTAs of a
// pair form a cluster so they run together and read each page from L2 once.
//
// Per CTA: warp 0 issues TMA loads of whole 576-wide pages (2-stage ring);
// warp 1 allocates TMEM and issues MMAs from an event loop (QK of a page as
// soon as its data and the score buffer are free, PV as soon as P is
// written); warps 2-9 own TMEM lanes 0-127 (= heads), two warps per lane
// quarter, each covering 32 of the 64 tokens of a page: online softmax with a
// lazily rescaled running max, P to TMEM in bf16, tail masking, epilogue.
//
// Every wait is bounded: on a timeout the CTA raises an error bit, stops, waits
// for its own copies and MMAs and frees TMEM.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <math_constants.h>

#include "common.cuh"
#include "launchers.h"
#include "tc_ptx.cuh"

namespace mla {
namespace {

using namespace tc;

constexpr int kSmxWarps = 8;
constexpr int kSmxThreads = kSmxWarps * 32;
constexpr int kThreads = 64 + kSmxThreads;
constexpr int kTileTok = 64;
constexpr int kStages = 2;
constexpr int kBoxBytes = kTileTok * 128;      // 64 rows x 64 bf16, 128-byte swizzled
constexpr int kBoxes = kRow / 64;              // 9 boxes per 576-wide page
constexpr int kStageBytes = kBoxes * kBoxBytes;
constexpr int kQBoxBytes = 128 * 128;          // Q in smem: 128 heads x 64 bf16
constexpr uint32_t kTmemCols = 512;
// TMEM column map (fp32 columns)
constexpr uint32_t kTmO = 0;    // O half: 256 columns
constexpr uint32_t kTmS = 256;  // S tile: 64 columns
constexpr uint32_t kTmP = 320;  // P tile: 64 bf16 = 32 columns
constexpr uint32_t kTmQ = 352;  // Q latent [0,256) + RoPE [512,576): 128 + 32 columns
// Lazy rescale: keep a stale row max until the new one exceeds it by 2^8.
constexpr float kRescaleLog2 = 8.0f;

struct __align__(1024) Smem {
  uint8_t stage[kStages][kStageBytes];  // whole pages, 9 boxes of 64 columns
  uint8_t q[4][kQBoxBytes];             // Q latent [256,512): 4 boxes of 64 columns
  float red[2][2][128];                 // row-max halves per page parity: [parity][half][head]
  float lsum[2][128];                   // row-sum halves for the epilogue
  // Each stage is two groups of boxes: "A" = the boxes only the QK product
  // reads (the other latent half and RoPE), released as soon as QK's first
  // part is done; "B" = this CTA's latent half, also read by PV.
  uint64_t full_a[kStages], full_b[kStages];
  uint64_t empty_a[kStages], empty_b[kStages];
  uint64_t s_full, s_empty, p_full, pv_done, q_ready, drain;
  uint64_t q_smem_full;  // TMA of Q latent [256,512) into shared memory landed
  uint64_t q_tm_full;    // TMA of Q latent [0,256) into stage 1 (staging for TMEM) landed
  uint64_t red_bar[2];  // softmax warps: row-max halves written (per page parity)
  uint64_t sum_bar;     // softmax warps: row-sum halves written (epilogue)
  uint32_t tmem_base;
  int32_t abort_flag;
};

constexpr size_t kSmemBytes = sizeof(Smem) + 1024;
constexpr int kPlain = 0, kSleep = 2;  // mbar_wait modes

// Wait bounded only by time (teardown: our own copies / MMAs must land).
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, int32_t* dev_error) {
  volatile int32_t never = 0;
  mbar_wait<kSleep>(bar, parity, &never, dev_error);
}

// Outputs of a work item with nothing to attend to (or rejected data).
__device__ void write_empty(const DecodeArgs& a, int64_t row0, int bj, int split, uint32_t half) {
  const int S = a.num_splits;
  if (S == 1) {
    uint4* u = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.u_out) + row0 * kDC + half * 256);
    for (int i = threadIdx.x; i < 128 * 32; i += blockDim.x) u[(i >> 5) * (kDC / 8) + (i & 31)] = make_uint4(0, 0, 0, 0);
    if (half == 0 && a.lse_out != nullptr)
      for (int h = threadIdx.x; h < 128; h += blockDim.x) a.lse_out[row0 + h] = -CUDART_INF_F;
  } else if (half == 0) {
    for (int h = threadIdx.x; h < 128; h += blockDim.x)
      a.part_lse[(static_cast<int64_t>(bj) * S + split) * 128 + h] = -CUDART_INF_F;
  }
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    decode_tc_kernel(const __grid_constant__ CUtensorMap tmap, const __grid_constant__ CUtensorMap qmap,
                     const DecodeArgs a) {
  extern __shared__ uint8_t smem_raw[];
  Smem* sm = reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t ohalf = blockIdx.x & 1u;  // which latent half of O this CTA owns

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
  if (bad_len && ohalf == 0 && threadIdx.x == 0) flag_error(a.dev_error, MLA_DEVERR_BAD_SEQLEN);
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
      if (ohalf == 0 && threadIdx.x == 0) flag_error(a.dev_error, MLA_DEVERR_BAD_PAGE);
    } else {
      n_tiles = (tok_end - tok_begin + kTileTok - 1) / kTileTok;
    }
  }
  if (n_tiles == 0) {
    write_empty(a, row0, bj, split, ohalf);
    return;
  }
  const uint32_t col0 = ohalf * 256u;  // first latent column of this CTA's O half

  // ---- set-up
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&sm->full_a[s]), 1);
      mbar_init(smem_u32(&sm->full_b[s]), 1);
      mbar_init(smem_u32(&sm->empty_a[s]), 1);
      mbar_init(smem_u32(&sm->empty_b[s]), 1);
    }
    mbar_init(smem_u32(&sm->s_full), 1);
    mbar_init(smem_u32(&sm->s_empty), kSmxWarps);
    mbar_init(smem_u32(&sm->p_full), kSmxWarps);
    mbar_init(smem_u32(&sm->pv_done), 1);
    mbar_init(smem_u32(&sm->q_ready), kSmxWarps);
    mbar_init(smem_u32(&sm->drain), 1);
    mbar_init(smem_u32(&sm->q_smem_full), 1);
    mbar_init(smem_u32(&sm->q_tm_full), 1);
    for (int x = 0; x < 2; ++x) mbar_init(smem_u32(&sm->red_bar[x]), kSmxWarps);
    mbar_init(smem_u32(&sm->sum_bar), kSmxWarps);
    sm->abort_flag = 0;
    fence_mbar_init_cluster();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmap);
    prefetch_tmap(&qmap);
  }
  if (warp == 1) tmem_alloc(smem_u32(&sm->tmem_base), kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm->tmem_base;
  volatile int32_t* abort_flag = &sm->abort_flag;

  // box groups of this CTA: B = its latent half (boxes 4*ohalf .. +3), A = the rest
  const int a_first = ohalf == 0 ? 4 : 0;  // A = boxes a_first..a_first+3 and box 8
  const int b_first = ohalf == 0 ? 0 : 4;
  if (warp == 0) {
    // ================= TMA producer
    if (lane == 0) {
      // Q latent [256,512) -> shared memory (A operand); latent [0,256) -> stage 1,
      // from where the softmax warps copy it into TMEM before page 1 is loaded
      mbar_arrive_expect_tx(smem_u32(&sm->q_smem_full), 4 * kQBoxBytes);
      for (int k = 0; k < 4; ++k)
        tma_load_2d_nohint(smem_u32(sm->q[k]), &qmap, smem_u32(&sm->q_smem_full), 256 + 64 * k,
                           static_cast<int32_t>(row0));
      mbar_arrive_expect_tx(smem_u32(&sm->q_tm_full), 4 * kQBoxBytes);
      for (int k = 0; k < 4; ++k)
        tma_load_2d_nohint(smem_u32(sm->stage[1]) + k * kQBoxBytes, &qmap, smem_u32(&sm->q_tm_full), 64 * k,
                           static_cast<int32_t>(row0));
      const uint64_t pol = l2_policy_evict_first();
      auto y_of = [&](int t) {  // pool row of tile t
        const int tok = tok_begin + t * kTileTok;
        return bt[tok / P] * P + (tok % P);
      };
      // pages kPrefetch tiles ahead are pulled into L2 so that a stage refill
      // (issued only when the stage frees) is an L2 hit
      constexpr int kPrefetch = 2;
      for (int t = 0; t < min(n_tiles, kPrefetch); ++t) {
        const int32_t yp = y_of(t);
        for (int k = 0; k < kBoxes; ++k) tma_prefetch_l2_2d(&tmap, 64 * k, yp);
      }
      int issued_a = 0, issued_b = 0;
      int32_t y_next = y_of(0);
      for (int i = 0; i < n_tiles; ++i) {
        const int st = i % kStages;
        const uint32_t ph = ((i / kStages) & 1) ^ 1;
        const int32_t y = y_next;
        if (i + 1 < n_tiles) y_next = y_of(i + 1);
        if (i + kPrefetch < n_tiles) {
          const int32_t yp = y_of(i + kPrefetch);
          for (int k = 0; k < kBoxes; ++k) tma_prefetch_l2_2d(&tmap, 64 * k, yp);
        }
        if (i == 1 && !mbar_wait<kSleep>(smem_u32(&sm->q_ready), 0, abort_flag, a.dev_error)) break;
        const uint32_t dst = smem_u32(sm->stage[st]);
        if (!mbar_wait<kSleep>(smem_u32(&sm->empty_a[st]), ph, abort_flag, a.dev_error)) break;
        mbar_arrive_expect_tx(smem_u32(&sm->full_a[st]), 5 * kBoxBytes);
        for (int k = 0; k < 4; ++k)
          tma_load_2d(dst + (a_first + k) * kBoxBytes, &tmap, smem_u32(&sm->full_a[st]), 64 * (a_first + k), y, pol);
        tma_load_2d(dst + 8 * kBoxBytes, &tmap, smem_u32(&sm->full_a[st]), 512, y, pol);
        issued_a = i + 1;
        if (!mbar_wait<kSleep>(smem_u32(&sm->empty_b[st]), ph, abort_flag, a.dev_error)) break;
        mbar_arrive_expect_tx(smem_u32(&sm->full_b[st]), 4 * kBoxBytes);
        for (int k = 0; k < 4; ++k)
          tma_load_2d(dst + (b_first + k) * kBoxBytes, &tmap, smem_u32(&sm->full_b[st]), 64 * (b_first + k), y, pol);
        issued_b = i + 1;
      }
      for (int i = max(0, issued_a - kStages); i < issued_a; ++i)
        drain_wait(smem_u32(&sm->full_a[i % kStages]), (i / kStages) & 1, a.dev_error);
      for (int i = max(0, issued_b - kStages); i < issued_b; ++i)
        drain_wait(smem_u32(&sm->full_b[i % kStages]), (i / kStages) & 1, a.dev_error);
      drain_wait(smem_u32(&sm->q_smem_full), 0, a.dev_error);
      drain_wait(smem_u32(&sm->q_tm_full), 0, a.dev_error);
    }
  } else if (warp == 1) {
    // ================= MMA issuer: event loop over QK part 1 (A boxes), QK part 2
    // (B boxes) and PV of successive pages
    if (lane == 0) {
      constexpr uint32_t kIdQK = idesc_bf16_f32(128, kTileTok, false, false);
      constexpr uint32_t kIdPV = idesc_bf16_f32(128, 256, false, true);
      // descriptor start addresses advance in 16-byte units in the low bits
      const uint64_t dPV0 = sdesc_sw128(smem_u32(sm->stage[0]) + ohalf * 4 * kBoxBytes, kBoxBytes, 1024);
      const uint64_t dKB0 = sdesc_sw128(smem_u32(sm->stage[0]), 16, 1024);  // page as K-major B
      const uint64_t dQA0 = sdesc_sw128(smem_u32(sm->q[0]), 16, 1024);      // Q latent [256,512) as A
      constexpr uint64_t kStageDesc = kStageBytes >> 4;
      // latent [0,256): A = Q from TMEM, B = page boxes 0-3
      auto qk_low = [&](uint64_t db, uint32_t first_acc) {
#pragma unroll
        for (uint32_t kk = 0; kk < 16; ++kk)
          mma_ts(tmem + kTmS, tmem + kTmQ + kk * 8u, db + (((kk >> 2) * kBoxBytes + (kk & 3u) * 32u) >> 4), kIdQK,
                 (kk > 0 || first_acc) ? 1u : 0u);
      };
      // latent [256,512): A = Q from shared memory, B = page boxes 4-7
      auto qk_high = [&](uint64_t db, uint32_t first_acc) {
#pragma unroll
        for (uint32_t kk = 0; kk < 16; ++kk)
          mma_ss(tmem + kTmS, dQA0 + (((kk >> 2) * kQBoxBytes + (kk & 3u) * 32u) >> 4),
                 db + (((4 + (kk >> 2)) * kBoxBytes + (kk & 3u) * 32u) >> 4), kIdQK, (kk > 0 || first_acc) ? 1u : 0u);
      };
      // RoPE [512,576): A = Q from TMEM, B = page box 8
      auto qk_rope = [&](uint64_t db) {
#pragma unroll
        for (uint32_t kk = 0; kk < 4; ++kk)
          mma_ts(tmem + kTmS, tmem + kTmQ + 128u + kk * 8u, db + ((8 * kBoxBytes + kk * 32u) >> 4), kIdQK, 1u);
      };
      bool ok = mbar_wait<kSleep>(smem_u32(&sm->q_ready), 0, abort_flag, a.dev_error) &&
                mbar_wait<kSleep>(smem_u32(&sm->q_smem_full), 0, abort_flag, a.dev_error);
      tc_fence_after();
      int q1 = 0, q2 = 0, pv = 0;  // next page for QK part 1, QK part 2, PV
      long long idle_since = 0;
      while (ok && pv < n_tiles) {
        bool did = false;
        if (pv < q2 && mbar_test_wait(smem_u32(&sm->p_full), pv & 1)) {
          tc_fence_after();
          const uint64_t d0 = dPV0 + static_cast<uint64_t>(pv % kStages) * kStageDesc;
#pragma unroll
          for (uint32_t kk = 0; kk < kTileTok / 16; ++kk)
            mma_ts(tmem + kTmO, tmem + kTmP + kk * 8u, d0 + kk * (16u * 128u >> 4), kIdPV,
                   (pv > 0 || kk > 0) ? 1u : 0u);
          mma_commit(smem_u32(&sm->empty_b[pv % kStages]));
          mma_commit(smem_u32(&sm->pv_done));
          ++pv;
          did = true;
        }
        if (q2 < q1 && mbar_test_wait(smem_u32(&sm->full_b[q2 % kStages]), (q2 / kStages) & 1)) {
          tc_fence_after();
          const uint64_t db = dKB0 + static_cast<uint64_t>(q2 % kStages) * kStageDesc;
          if (ohalf == 0) qk_low(db, 1u); else qk_high(db, 1u);
          mma_commit(smem_u32(&sm->s_full));
          ++q2;
          did = true;
        }
        // S(q1) may be written once S(q1-1) has been read out of TMEM
        if (q1 == q2 && q1 < n_tiles && mbar_test_wait(smem_u32(&sm->full_a[q1 % kStages]), (q1 / kStages) & 1) &&
            (q1 == 0 || mbar_test_wait(smem_u32(&sm->s_empty), (q1 - 1) & 1))) {
          tc_fence_after();
          const uint64_t db = dKB0 + static_cast<uint64_t>(q1 % kStages) * kStageDesc;
          if (ohalf == 0) qk_high(db, 0u); else qk_low(db, 0u);
          qk_rope(db);
          mma_commit(smem_u32(&sm->empty_a[q1 % kStages]));
          ++q1;
          did = true;
        }
        if (did) {
          idle_since = 0;
        } else {
          const long long now = clock64();
          if (idle_since == 0) idle_since = now;
          if (*abort_flag) ok = false;
          if (now - idle_since > kWaitTimeoutCycles) {
            *abort_flag = 1;
            flag_error(a.dev_error, kDevErrTimeout);
            ok = false;
          }
        }
      }
      mma_commit(smem_u32(&sm->drain));
      drain_wait(smem_u32(&sm->drain), 0, a.dev_error);
    }
  } else {
    // ================= softmax / epilogue
    // thread = (head h = TMEM lane, half of the page's 64 tokens)
    const uint32_t q4 = static_cast<uint32_t>(warp & 3);
    const int half = (warp - 2) >> 2;
    const int h = static_cast<int>(q4 * 32u) + lane;
    const uint32_t lanes = (q4 * 32u) << 16;
    const uint32_t tS = tmem + lanes + kTmS + half * 32, tP = tmem + lanes + kTmP + half * 16;
    const uint32_t tO = tmem + lanes + kTmO + half * 128, tQ = tmem + lanes + kTmQ;
    auto wwait = [&](uint64_t* bar, uint32_t par) {
      return __all_sync(0xffffffffu, mbar_wait<kPlain>(smem_u32(bar), par, abort_flag, a.dev_error));
    };
    // Q of this head into TMEM (bf16 pairs, lower K index in the low half). The
    // producer staged latent [0,256) in stage 1 (four 128 x 64 boxes, 128-byte
    // swizzle: 16-byte chunk c of row h sits at chunk c ^ (h mod 8)); half 0
    // copies latent [0,128) and the RoPE part (from global memory), half 1
    // latent [128,256). Latent [256,512) stays in shared memory (A operand).
    {
      uint4 xr[8];
      if (half == 0) {
        const uint4* qr = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.q_rope) + (row0 + h) * kDRope);
#pragma unroll
        for (int v = 0; v < 8; ++v) xr[v] = qr[v];
      }
      const bool qok = wwait(&sm->q_tm_full, 0);
      if (qok) {
        uint32_t r[32];
#pragma unroll
        for (int bb = 0; bb < 2; ++bb) {
          const uint8_t* box = sm->stage[1] + (half * 2 + bb) * kQBoxBytes + h * 128;
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const uint4 x = *reinterpret_cast<const uint4*>(box + ((c ^ (h & 7)) << 4));
            r[4 * c] = x.x;
            r[4 * c + 1] = x.y;
            r[4 * c + 2] = x.z;
            r[4 * c + 3] = x.w;
          }
          tmem_st32(tQ + static_cast<uint32_t>((half * 2 + bb) * 32), r);
        }
        if (half == 0) {
#pragma unroll
          for (int v = 0; v < 8; ++v) {
            r[4 * v] = xr[v].x;
            r[4 * v + 1] = xr[v].y;
            r[4 * v + 2] = xr[v].z;
            r[4 * v + 3] = xr[v].w;
          }
          tmem_st32(tQ + 128u, r);
        }
        tmem_wait_st();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sm->q_ready));  // also frees stage 1 for page 1
    }
    const float c2 = a.softmax_scale * kLog2e;  // scores in log2 units
    float m = -CUDART_INF_F, l = 0.0f;          // l: this thread's half of the row sum
    bool ok = true;
    for (int i = 0; ok && i < n_tiles; ++i) {
      if (!wwait(&sm->s_full, i & 1)) { ok = false; break; }
      tc_fence_after();
      float s[32];
      tmem_ld32_sync(tS, s);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sm->s_empty));  // S may be overwritten by QK(i+1)

      // ---- online softmax over this tile
      const int tok0 = tok_begin + i * kTileTok + half * 32;
      const int valid = min(32, tok_end - tok0);  // may be <= 0 for the upper half
      if (valid < 32) {
#pragma unroll
        for (int t = 0; t < 32; ++t)
          if (t >= valid) s[t] = -CUDART_INF_F;
      }
      float mx;
      {
        float t16[16];
#pragma unroll
        for (int t = 0; t < 16; ++t) t16[t] = fmaxf(s[t], s[t + 16]);
#pragma unroll
        for (int w = 8; w >= 1; w >>= 1)
#pragma unroll
          for (int t = 0; t < w; ++t) t16[t] = fmaxf(t16[t], t16[t + w]);
        mx = t16[0];
      }
      // row max over both token halves (the other half lives in another warp);
      // an mbarrier rather than bar.sync, so that an aborting warp cannot hang the rest
      sm->red[i & 1][half][h] = mx;
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sm->red_bar[i & 1]));
      if (!wwait(&sm->red_bar[i & 1], (i >> 1) & 1)) { ok = false; break; }
      mx = fmaxf(mx, sm->red[i & 1][half ^ 1][h]);
      const bool first = (i == 0);
      const float m_new = fmaxf(m, mx * c2);
      const bool resc = !first && (m_new > m + kRescaleLog2);
      const float m_use = (first || resc) ? m_new : m;
      const float alpha = resc ? fast_exp2(m - m_use) : 1.0f;
      float rsum[4] = {0.0f, 0.0f, 0.0f, 0.0f};
      uint32_t pw[16];
#pragma unroll
      for (int t = 0; t < 16; ++t) {
        const float p0 = fast_exp2(fmaf(s[2 * t], c2, -m_use));
        const float p1 = fast_exp2(fmaf(s[2 * t + 1], c2, -m_use));
        pw[t] = pack_bf16x2(p0, p1);
        // normalise by the weights the PV product actually uses (bf16-rounded)
        rsum[t & 3] += __uint_as_float(pw[t] << 16) + __uint_as_float(pw[t] & 0xffff0000u);
      }
      l = l * alpha + ((rsum[0] + rsum[1]) + (rsum[2] + rsum[3]));
      m = m_use;
      if (!first) {
        if (!wwait(&sm->pv_done, (i - 1) & 1)) { ok = false; break; }
        tc_fence_after();
      }
      if (__any_sync(0xffffffffu, resc)) {
        for (int c = 0; c < 4; ++c) {
          float o[32];
          tmem_ld32_sync(tO + c * 32u, o);
          uint32_t r[32];
#pragma unroll
          for (int k = 0; k < 32; ++k) r[k] = __float_as_uint(o[k] * alpha);
          tmem_st32(tO + c * 32u, r);
        }
        tmem_wait_st();
      }
      const int page_valid = min(kTileTok, tok_end - (tok_begin + i * kTileTok));
      if (page_valid < kTileTok) {
        // rows past the sequence end may hold anything (NaN): zero them in this
        // CTA's V columns so that 0 * row stays 0 in the PV product
        uint4* base = reinterpret_cast<uint4*>(sm->stage[i % kStages] + ohalf * 4 * kBoxBytes);
        const int rows = kTileTok - page_valid;
        const int t_id = half * 128 + h;
        for (int e = t_id; e < rows * 4 * 8; e += kSmxThreads) {
          const int box = e / (rows * 8), rem = e % (rows * 8);
          base[(box * kBoxBytes + (page_valid + rem / 8) * 128) / 16 + (rem % 8)] = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
        __syncwarp();
      }
      tmem_st16(tP, pw);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sm->p_full));
    }
    // ---- epilogue: u = O / l (this CTA's 256 columns; this thread's 128), lse
    sm->lsum[half][h] = l;
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&sm->sum_bar));
    if (ok && !wwait(&sm->sum_bar, 0)) ok = false;
    const float l_row = sm->lsum[0][h] + sm->lsum[1][h];
    if (ok && wwait(&sm->pv_done, (n_tiles - 1) & 1)) {
      tc_fence_after();
      const float inv_l = 1.0f / l_row;
      const float lse = (m + log2f(l_row)) * kLn2;
      const uint32_t c_out = col0 + half * 128;
      if (S == 1) {
        uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.u_out) + (row0 + h) * kDC + c_out);
        for (int c = 0; c < 4; ++c) {
          float o[32];
          tmem_ld32_sync(tO + c * 32u, o);
          uint32_t w[16];
#pragma unroll
          for (int k = 0; k < 16; ++k) w[k] = pack_bf16x2(o[2 * k] * inv_l, o[2 * k + 1] * inv_l);
#pragma unroll
          for (int v = 0; v < 4; ++v) dst[c * 4 + v] = make_uint4(w[4 * v], w[4 * v + 1], w[4 * v + 2], w[4 * v + 3]);
        }
        if (ohalf == 0 && half == 0 && a.lse_out != nullptr) a.lse_out[row0 + h] = lse;
      } else {
        const int64_t prow = (static_cast<int64_t>(bj) * S + split) * 128 + h;
        float4* dst = reinterpret_cast<float4*>(a.part_u + prow * kDC + c_out);
        for (int c = 0; c < 4; ++c) {
          float o[32];
          tmem_ld32_sync(tO + c * 32u, o);
#pragma unroll
          for (int v = 0; v < 8; ++v)
            dst[c * 8 + v] = make_float4(o[4 * v] * inv_l, o[4 * v + 1] * inv_l, o[4 * v + 2] * inv_l,
                                         o[4 * v + 3] * inv_l);
        }
        if (ohalf == 0 && half == 0) a.part_lse[prow] = lse;
      }
    }
  }

  // ---- teardown
  __syncwarp();
  tc_fence_before();
  __syncthreads();
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

// Tensor maps are plain host structures; encoding one costs host time on every
// call, so the last few are kept (keyed by base pointer and shape). get()
// copies the map out, so a later miss that recycles a slot cannot change a map
// already handed to a launch.
struct MapCache {
  static constexpr int kSlots = 8;
  struct Entry {
    const void* ptr = nullptr;
    uint64_t rows = 0;
    uint32_t cols = 0, box_rows = 0;
    CUtensorMap map;
  } e[kSlots];
  int next = 0;
  bool get(const void* ptr, uint64_t rows, uint32_t cols, uint32_t box_rows, CUtensorMap* out) {
    for (auto& x : e)
      if (x.ptr == ptr && x.rows == rows && x.cols == cols && x.box_rows == box_rows) {
        *out = x.map;
        return true;
      }
    Entry& n = e[next];
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
    const cuuint32_t box[2] = {64, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    if (tensor_map_encoder()(&n.map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box,
                             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS) {
      n.ptr = nullptr;
      return false;
    }
    n.ptr = ptr;
    n.rows = rows;
    n.cols = cols;
    n.box_rows = box_rows;
    next = (next + 1) % kSlots;
    *out = n.map;
    return true;
  }
};

cudaError_t launch_decode_tc(const DecodeArgs& a, cudaStream_t s) {
  static MapCache cache;  // host-side; calls on one process are expected from one thread at a time
  static int attr_set_for_device = -1;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
  if (attr_set_for_device != dev) {
    const cudaError_t e = cudaFuncSetAttribute(decode_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               static_cast<int>(kSmemBytes));
    if (e != cudaSuccess) return e;
    attr_set_for_device = dev;
  }
  CUtensorMap map, qmap;
  // cache as [num_pages*page_size rows][576] bf16, 64 x 64 boxes; q_lat as
  // [batch*q_len*128 rows][512] bf16, 128 x 64 boxes
  if (!cache.get(a.cache, static_cast<uint64_t>(a.num_pages) * a.page_size, kRow, kTileTok, &map) ||
      !cache.get(a.q_lat, static_cast<uint64_t>(a.batch) * a.q_len * 128, kDC, 128, &qmap))
    return cudaErrorInvalidValue;
  const int64_t items = static_cast<int64_t>(a.batch) * a.q_len * a.num_splits;
  decode_tc_kernel<<<dim3(static_cast<unsigned>(2 * items)), kThreads, kSmemBytes, s>>>(map, qmap, a);
  return cudaGetLastError();
}

}  // namespace mla
