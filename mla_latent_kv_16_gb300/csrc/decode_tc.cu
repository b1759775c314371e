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
//   CTA rank 0: latent columns [0, 256)             -> K slice of S, O[:, 0:256]
//   CTA rank 1: latent [256, 512) + RoPE [512, 576) -> K slice of S, O[:, 256:512]
// Each CTA TMA-loads only its own columns of every page (HBM is read once),
// keeps its Q slice in TMEM (A operand), computes a partial S, and the pair
// exchange partial S through distributed shared memory with asynchronous
// stores that complete on the receiver's mbarrier. Both then hold the same
// full S (fp32 addition is commutative), run the same online softmax and feed
// P (bf16, in TMEM) into their own half of the PV product.
//
// Warp roles (320 threads): warp 0 issues TMA loads (3-stage ring); warp 1
// allocates TMEM and issues MMAs from an event loop (QK of a page as soon as
// its data and the S buffer are free, PV as soon as P is written); warps 2-9
// own TMEM lanes 0-127 (= heads), two warps per lane quarter, each covering 32
// of the 64 tokens of a page. Page i+1's partial scores are sent to the peer
// before page i is softmaxed, so the exchange overlaps the softmax.
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

constexpr int kSmxWarps = 8;
constexpr int kSmxThreads = kSmxWarps * 32;
constexpr int kThreads = 64 + kSmxThreads;
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
  // partial-S exchange slots: [slot][region = softmax warp][token group of 4][lane]
  float4 xbuf[2][kSmxWarps][8][32];
  float red[2][2][128];               // row-max halves per page parity: [parity][half][head]
  float lsum[2][128];                 // row-sum halves for the epilogue
  uint64_t kv_full[kStages];
  uint64_t kv_empty[kStages];
  uint64_t s_full, s_empty, p_full, pv_done, q_ready, drain;
  uint64_t x_full[2][kSmxWarps];  // receiver: peer's page landed in a region (arming + tx bytes)
  uint64_t x_empty[2];  // sender side: the peer has consumed its slot
  uint64_t red_bar[2];  // softmax warps: row-max halves written (per page parity)
  uint64_t sum_bar;     // softmax warps: row-sum halves written (epilogue)
  uint32_t tmem_base;
  int32_t abort_flag;
};

constexpr size_t kSmemBytes = sizeof(Smem) + 1024;
constexpr uint32_t kXBytes = 32 * 32 * 4;                 // one region of one page of partial scores
constexpr int kPlain = 0, kAcqCluster = 1, kSleep = 2;    // mbar_wait modes

// Wait bounded only by time (teardown: our own copies / MMAs must land).
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, int32_t* dev_error) {
  volatile int32_t never = 0;
  mbar_wait<kSleep>(bar, parity, &never, dev_error);
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

  // ---- set-up
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&sm->kv_full[s]), 1);
      mbar_init(smem_u32(&sm->kv_empty[s]), 1);
    }
    mbar_init(smem_u32(&sm->s_full), 1);
    mbar_init(smem_u32(&sm->s_empty), kSmxWarps);
    mbar_init(smem_u32(&sm->p_full), kSmxWarps);
    mbar_init(smem_u32(&sm->pv_done), 1);
    mbar_init(smem_u32(&sm->q_ready), kSmxWarps);
    mbar_init(smem_u32(&sm->drain), 1);
    for (int x = 0; x < 2; ++x) {
      for (int r = 0; r < kSmxWarps; ++r) mbar_init(smem_u32(&sm->x_full[x][r]), 1);  // arming (+ peer bytes)
      mbar_init(smem_u32(&sm->x_empty[x]), kSmxWarps);  // one remote arrival per peer warp
    }
    for (int x = 0; x < 2; ++x) mbar_init(smem_u32(&sm->red_bar[x]), kSmxWarps);
    mbar_init(smem_u32(&sm->sum_bar), kSmxWarps);
    sm->abort_flag = 0;
    fence_mbar_init_cluster();
    for (int x = 0; x < 2; ++x)
      for (int r = 0; r < kSmxWarps; ++r) mbar_arrive_expect_tx(smem_u32(&sm->x_full[x][r]), kXBytes);
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
      // the page of tile i+1 is fetched while tile i waits for its stage
      int32_t page_next = bt[tok_begin / P];
      for (int i = 0; i < n_tiles; ++i) {
        const int st = i % kStages;
        const int tok = tok_begin + i * kTileTok;
        const int32_t page = page_next;
        if (i + 1 < n_tiles) page_next = bt[(tok + kTileTok) / P];
        if (!mbar_wait<kSleep>(smem_u32(&sm->kv_empty[st]), ((i / kStages) & 1) ^ 1, abort_flag, a.dev_error)) break;
        const int32_t y = page * P + (tok % P);
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
    // ================= MMA issuer: event loop over "QK of page qk" and "PV of page pv"
    if (lane == 0) {
      constexpr uint32_t kIdQK = idesc_bf16_f32(128, kTileTok, false, false);
      constexpr uint32_t kIdPV = idesc_bf16_f32(128, 256, false, true);
      // descriptor start addresses advance in 16-byte units in the low bits
      const uint64_t dPV0 = sdesc_sw128(smem_u32(sm->stage[0]), kBoxBytes, 1024);
      const uint64_t dQK0 = sdesc_sw128(smem_u32(sm->stage[0]), 16, 1024);
      constexpr uint64_t kStageDesc = kStageBytes >> 4;
      const bool rope = (nbox == 5);
      bool ok = mbar_wait<kSleep>(smem_u32(&sm->q_ready), 0, abort_flag, a.dev_error);
      tc_fence_after();
      int qk = 0, pv = 0;
      long long idle_since = 0;
      while (ok && pv < n_tiles) {
        bool did = false;
        // S(qk) may be written once S(qk-1) has been read out of TMEM
        if (qk < n_tiles && mbar_test_wait(smem_u32(&sm->kv_full[qk % kStages]), (qk / kStages) & 1) &&
            (qk == 0 || mbar_test_wait(smem_u32(&sm->s_empty), (qk - 1) & 1))) {
          tc_fence_after();
          const uint64_t d0 = dQK0 + static_cast<uint64_t>(qk % kStages) * kStageDesc;
#pragma unroll
          for (uint32_t kk = 0; kk < 16; ++kk)
            mma_ts(tmem + kTmS, tmem + kTmQ + kk * 8u, d0 + (((kk >> 2) * kBoxBytes + (kk & 3u) * 32u) >> 4), kIdQK,
                   kk > 0 ? 1u : 0u);
          if (rope) {
#pragma unroll
            for (uint32_t kk = 16; kk < 20; ++kk)
              mma_ts(tmem + kTmS, tmem + kTmQ + kk * 8u, d0 + (((kk >> 2) * kBoxBytes + (kk & 3u) * 32u) >> 4),
                     kIdQK, 1u);
          }
          mma_commit(smem_u32(&sm->s_full));
          ++qk;
          did = true;
        }
        if (pv < qk && mbar_test_wait(smem_u32(&sm->p_full), pv & 1)) {
          tc_fence_after();
          const uint64_t d0 = dPV0 + static_cast<uint64_t>(pv % kStages) * kStageDesc;
#pragma unroll
          for (uint32_t kk = 0; kk < kTileTok / 16; ++kk)
            mma_ts(tmem + kTmO, tmem + kTmP + kk * 8u, d0 + kk * (16u * 128u >> 4), kIdPV,
                   (pv > 0 || kk > 0) ? 1u : 0u);
          mma_commit(smem_u32(&sm->kv_empty[pv % kStages]));
          mma_commit(smem_u32(&sm->pv_done));
          ++pv;
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
    // ================= softmax / exchange / epilogue
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
    auto wwait_cluster = [&](uint64_t* bar, uint32_t par) {
      return __all_sync(0xffffffffu, mbar_wait<kAcqCluster>(smem_u32(bar), par, abort_flag, a.dev_error));
    };
    // Q slice of this head into TMEM (bf16 pairs, lower K index in the low half).
    // Chunks of 32 columns: half 0 writes chunks 0-1, half 1 chunks 2-3 (+4 = RoPE).
    {
      const uint4* ql = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.q_lat) + (row0 + h) * kDC + col0);
      const uint4* qr = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.q_rope) + (row0 + h) * kDRope);
      const bool do_rope = (half == 1 && rank == 1);
      uint4 x[24];  // every load in flight at once: one memory round trip
#pragma unroll
      for (int v = 0; v < 16; ++v) x[v] = ql[half * 16 + v];
      if (do_rope) {
#pragma unroll
        for (int v = 0; v < 8; ++v) x[16 + v] = qr[v];
      }
      uint32_t r[32];
#pragma unroll
      for (int c = 0; c < 3; ++c) {
        if (c == 2 && !do_rope) break;
#pragma unroll
        for (int v = 0; v < 8; ++v) {
          r[4 * v] = x[c * 8 + v].x;
          r[4 * v + 1] = x[c * 8 + v].y;
          r[4 * v + 2] = x[c * 8 + v].z;
          r[4 * v + 3] = x[c * 8 + v].w;
        }
        tmem_st32(tQ + (c == 2 ? 128u : static_cast<uint32_t>(half * 64 + c * 32)), r);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sm->q_ready));
    }
    const float c2 = a.softmax_scale * kLog2e;  // scores in log2 units
    float m = -CUDART_INF_F, l = 0.0f;          // l: this thread's half of the row sum
    const int region = half * 4 + static_cast<int>(q4);  // this warp's exchange region
    const uint32_t xbuf_peer = map_to_rank(smem_u32(&sm->xbuf[0][region][0][lane]), peer);
    const uint32_t xfull_peer[2] = {map_to_rank(smem_u32(&sm->x_full[0][region]), peer),
                                    map_to_rank(smem_u32(&sm->x_full[1][region]), peer)};
    const uint32_t xempty_peer[2] = {map_to_rank(smem_u32(&sm->x_empty[0]), peer),
                                     map_to_rank(smem_u32(&sm->x_empty[1]), peer)};
    bool ok = true;
    // Own partial scores of page i (s) and page i+1 (sn), this thread's 32 tokens.
    float s[32], sn[32];
    auto load_and_send = [&](int pg, float (&dst)[32]) -> bool {
      if (!wwait(&sm->s_full, pg & 1)) return false;
      tc_fence_after();
      tmem_ld32_sync(tS, dst);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sm->s_empty));  // S may be overwritten by QK(pg+1)
      // asynchronous stores into the peer's slot pg&1, counted on its barrier,
      // once the peer has consumed page pg-2 from that slot
      const int xs = pg & 1;
      if (!wwait_cluster(&sm->x_empty[xs], ((pg >> 1) & 1) ^ 1)) return false;
#pragma unroll
      for (int q = 0; q < 8; ++q)
        st_async_v4(xbuf_peer + static_cast<uint32_t>((xs * kSmxWarps * 8 * 32 + q * 32) * 16), dst[4 * q],
                    dst[4 * q + 1], dst[4 * q + 2], dst[4 * q + 3], xfull_peer[xs]);
      return true;
    };
    if (!load_and_send(0, s)) ok = false;
    for (int i = 0; ok && i < n_tiles; ++i) {
      if (i + 1 < n_tiles && !load_and_send(i + 1, sn)) { ok = false; break; }
      const int xs = i & 1;
      if (!wwait_cluster(&sm->x_full[xs][region], (i >> 1) & 1)) { ok = false; break; }
      // re-arm this region for page i+2 (its phase for page i has completed)
      if (lane == 0) mbar_arrive_expect_tx(smem_u32(&sm->x_full[xs][region]), kXBytes);
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const float4 v = sm->xbuf[xs][region][q][lane];
        s[4 * q] += v.x;
        s[4 * q + 1] += v.y;
        s[4 * q + 2] += v.z;
        s[4 * q + 3] += v.w;
      }
      // slot consumed (and re-armed): the peer may send page i+2 into it. The
      // warp barrier orders every lane's reads before lane 0's release.
      __syncwarp();
      if (lane == 0) mbar_arrive_remote(xempty_peer[xs]);

      // ---- online softmax over this tile (identical in both CTAs)
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
      // row max over both halves (the other half lives in another warp)
      // (an mbarrier, not bar.sync, so that an aborting warp cannot hang the rest)
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
        // rows past the sequence end may hold anything (NaN): zero them in the
        // V columns so that 0 * row stays 0 in the PV product
        uint4* base = reinterpret_cast<uint4*>(sm->stage[i % kStages]);
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
#pragma unroll
      for (int t = 0; t < 32; ++t) s[t] = sn[t];
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
        if (rank == 0 && half == 0 && a.lse_out != nullptr) a.lse_out[row0 + h] = lse;
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
        if (rank == 0 && half == 0) a.part_lse[prow] = lse;
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
