// Paged MLA decode on the 5th-generation tensor cores (tcgen05 + TMEM + TMA),
// one CTA pair (cluster of 2) per work item, each CTA doing half of the work.
//
// What is computed ("Model Architecture Driving Inference Systems" §3.1-3.2;
// "Tech Radar: DeepSeek-V3 MLA" §2): for every head h of one query position,
//   s_t = (q_lat[h] . c_KV[t] + q_rope[h] . k_R[t]) * softmax_scale
//   u[h] = sum_t softmax(s)_t c_KV[t]
// In the decode ("MQA") form all 128 heads share the same 576-wide cached rows
// ("DeepSeek's attention evolution - [MLA]" §2.5), so the heads are the MMA M
// dimension: S[128 x 64] = Q[128 x 576] * C^T per 64-token page, and
// O[128 x 512] += P[128 x 64] * C[64 x 512].
//
// GB300 mapping. O (128 x 512 fp32) alone fills one SM's TMEM, so the pair
// splits it: CTA r owns latent half r (columns [256r, 256r+256)) for all 128
// heads. Each CTA reads only its own latent half of every page (plus the RoPE
// columns of every other page) and computes a PARTIAL score over it:
// S_r = Q[:, half r] * C[:, half r]^T (+ the RoPE term on pages i = r mod 2),
// S = S_0 + S_1. The softmax is split by heads: CTA r owns heads
// [64r, 64r+64). Per page each CTA
//   1. sends the peer the partial scores of the peer's 64 heads (16 KB, DSMEM),
//   2. adds the peer's partial to its own for its heads, runs the online
//      softmax (running max with lazy rescale, row sums) and
//   3. writes P (bf16) of its heads into its own and the peer's P tile (8 KB
//      each way) together with the rescale factors of its heads,
// after which both CTAs run the PV MMAs for their O half. Nothing is computed
// twice, and each page crosses the SM boundary only as scores and weights.
//
// TMEM (512 columns): O half [0,256), two score buffers [256,320) and
// [320,384), Q's own latent half as bf16 pairs [384,512) (A of the QK MMAs).
// The rows (TMEM lanes) of Q, S, P and O are heads in an order rotated by 64
// in one CTA, so that each CTA's own heads occupy the same two lane quarters.
// Shared memory: a 4-deep ring of page halves (4 boxes of 64 tokens x 64
// columns, 128-byte swizzle), a RoPE box, Q's RoPE part, two P tiles
// (A of the PV MMAs), two inboxes for the peer's partial scores.
//
// Warps: 0 = TMA producer; 1 = TMEM allocation and MMA issue (PV of a page as
// soon as its P is complete, else the next page's QK as soon as its score
// buffer has been read and its data landed); 2-9 = two warps per TMEM lane
// quarter. On the quarters of this CTA's heads both run the softmax of every
// page, warp t over the tokens [32t, 32t+32); on the other quarters one
// forwards the peer's partial scores as soon as they are written (so that the
// score buffer is released early) and the other receives the peer's P rows and
// applies its rescale factors to those O rows. In the epilogue each warp
// normalises one half of the O columns of its quarter.
//
// Distributed shared memory carries the partial scores and P. Both land
// chunk-major ([16-byte chunk][head]) so that every warp-wide st.async writes
// 512 contiguous bytes; scattered 16-byte pieces cost twice their size on the
// link and several times the time.
//
// E4M3 cache ("Multi-Head Latent Attention (MLA): ..." "High-Throughput Serving
// Kernels": FP8 latent cache with per-block scales): the TMA brings each page
// half as bytes into the upper half of its slot, and six more warps decode it
// in place to bf16 x (per-token, per-group) scale in the same swizzled layout
// before the slot is marked full; everything after that is the bf16 path.
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

// Warps: 0 = TMA, 1 = TMEM allocation + MMA issue, then (E4M3 cache only) the
// converter warps, then eight softmax / forwarding warps (two per TMEM lane
// quarter; warp w may access lane quarter w mod 4).
constexpr int kSmxWarps = 8;
constexpr int kCvtWarps = 6;  // E4M3 -> bf16 converter warps (E4M3 cache)
__host__ __device__ constexpr int smx_warp0(bool fp8) { return 2 + (fp8 ? kCvtWarps : 0); }
__host__ __device__ constexpr int threads_for(bool fp8) { return 32 * (smx_warp0(fp8) + kSmxWarps); }
// (E4M3: 16 warps, so at most 128 registers per thread; the softmax code then
// spills a few bytes, less than a per-warpgroup register split would.)
constexpr int kFp8BoxBytes = 64 * 64;  // 64 rows x 64 bytes of E4M3
constexpr int kTileTok = 64;
constexpr int kStages = 4;                  // ring of page halves
constexpr int kBoxBytes = kTileTok * 128;   // 64 rows x 64 bf16, 128-byte swizzled
constexpr int kHalfBytes = 4 * kBoxBytes;   // one page, one latent half
constexpr int kQBoxBytes = 128 * 128;       // 128 heads x 64 bf16
constexpr int kPTileBytes = 128 * 128;      // P: 128 heads x 64 tokens bf16
constexpr uint32_t kSinBytes = 64 * 64 * 4; // payload of one score inbox
constexpr uint32_t kPinBytes = 64 * 128 + 64 * 4;  // peer's P rows + rescale factors
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmO = 0;    // O half: 256 columns
constexpr uint32_t kTmS = 256;  // two partial-score buffers of 64 columns
constexpr uint32_t kTmQ = 384;  // Q's own latent half: 128 columns of bf16 pairs
// Lazy rescale: keep a stale row max until the new one exceeds it by 2^8.
constexpr float kRescaleLog2 = 8.0f;
// The lane quarters (2*kOwnQ, 2*kOwnQ + 1) that hold a CTA's own heads, in both
// CTAs of the pair (the head order in TMEM is rotated by 64 where needed). Warp
// w runs on SM sub-partition w mod 4, and the softmax warps of the own heads
// are the busiest: they go where nothing else heavy runs. bf16 cache: quarters
// 2-3, away from the TMA (warp 0) and MMA (warp 1) issuers. E4M3 cache:
// quarters 0-1, whose sub-partitions hold one converter warp each (warps 4,
// 5) where quarters 2-3 hold two (warps 2, 6 and 3, 7).
template <bool kFp8>
constexpr uint32_t kOwnQ = kFp8 ? 0u : 1u;

struct __align__(1024) Smem {
  uint8_t kv[kStages][kHalfBytes];  // own latent half of page i in slot i % 4; slots 1-2 first stage Q
  uint8_t rope[kBoxBytes];          // RoPE box of this CTA's next RoPE page (i = r mod 2)
  uint8_t qr[kQBoxBytes];           // Q RoPE part (A of the RoPE MMAs)
  uint8_t pt[2][kPTileBytes];       // P tile per page parity (A of the PV MMAs)
  // the peer's partial scores for this CTA's 64 heads, chunk-major: 16-byte chunk v
  // (tokens 4v .. 4v+3) of head hl at sin[buffer][v][hl], so that a warp-wide
  // store or load of one chunk of 32 heads covers 512 contiguous bytes
  float4 sin[2][16][64];
  float alpha_in[2][64];            // peer's rescale factors for the peer's heads
  float mx_part[2][2][64];          // page i's row max over the token half t of each own head, in [i & 1][t]
  float lsum[2][64];                // each softmax warp's row sum, for the epilogue
  float mlast[2][64];               // the max each softmax warp's row sum refers to
  float l_in[64];                   // peer's row sums for the peer's heads
  uint64_t full_kv[kStages], empty_kv[kStages];
  uint64_t full_rope, empty_rope;
  uint64_t q_smem_full, q_tm_full, q_ready;
  uint64_t s_full[2], s_free[2];    // partial scores in TMEM: written / read by all 8 warps
  uint64_t s_in[2], rs_free[2];     // score inbox: filled by the peer / the peer's inbox is free
  uint64_t p_in[2], rp_free[2];     // P rows from the peer landed / the peer's P tile is free
  uint64_t pt_free[2];              // PV of the page that last used P tile x is done
  uint64_t p_full[2];               // P of page i complete in tile i & 1 and O rescaled (4 warps)
  uint64_t o_done, sum_bar, l_bar, drain;
  uint64_t raw_full[kStages], raw_rope_full;  // E4M3 bytes landed (TMA)
  uint64_t cvt_bar;                           // every converter warp has read its chunks of the page
  uint32_t tmem_base;
  int32_t abort_flag;
  int32_t peer_abort;  // the peer's abort flag, stored here by the peer at teardown
};
constexpr size_t kSmemBytes = sizeof(Smem) + 1024;  // + realignment slack
static_assert(kSmemBytes <= 232448, "shared memory budget of one CTA");
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

template <bool kFp8>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(threads_for(kFp8), 1)
    decode_tc_kernel(const __grid_constant__ CUtensorMap tmap, const __grid_constant__ CUtensorMap qmap,
                     const __grid_constant__ CUtensorMap rmap, const __grid_constant__ CUtensorMap pmap,
                     const DecodeArgs a) {
  extern __shared__ uint8_t smem_raw[];
  Smem* sm = reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t r = cluster_ctarank();  // latent half of O and head half of the softmax this CTA owns
  const uint32_t peer = r ^ 1u;
  // TMEM lane L (row of Q, S, P and O) holds head (L + rot) mod 128, so that in
  // both CTAs the own heads [64r, 64r+64) sit in lane quarters 2*kOwnQ and
  // 2*kOwnQ+1, i.e. on the same two SM sub-partitions (see kOwnQ).
  const uint32_t rot = 64u * (r ^ kOwnQ<kFp8>);

  // ---- work item: (sequence b, query j, split) -- identical in both CTAs
  const int item = blockIdx.x >> 1;
  const int Lq = a.q_len, S = a.num_splits, P = a.page_size;
  const int j = item % Lq;
  const int split = (item / Lq) % S;
  const int b = item / (Lq * S);
  const int bj = b * Lq + j;
  const int64_t row0 = static_cast<int64_t>(bj) * 128;
  const int32_t col_half = static_cast<int32_t>(256u * r);  // first latent column of this CTA's half

  // ---- set-up that reads no data of the previous kernels (it may run while
  // they finish: programmatic dependent launch), then the wait for them
  pdl_trigger();
  if (threadIdx.x == 0) {
    // E4M3: the converter warps complete full_kv / full_rope, the TMA raw_full
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&sm->full_kv[s]), kFp8 ? kCvtWarps : 1);
      mbar_init(smem_u32(&sm->empty_kv[s]), 1);
      mbar_init(smem_u32(&sm->raw_full[s]), 1);
    }
    mbar_init(smem_u32(&sm->raw_rope_full), 1);
    mbar_init(smem_u32(&sm->cvt_bar), kCvtWarps);
    mbar_init(smem_u32(&sm->full_rope), kFp8 ? kCvtWarps : 1);
    mbar_init(smem_u32(&sm->empty_rope), 1);
    for (int x = 0; x < 2; ++x) {
      mbar_init(smem_u32(&sm->s_full[x]), 1);
      mbar_init(smem_u32(&sm->s_free[x]), 6);  // 4 softmax + 2 forwarding warps
      mbar_init(smem_u32(&sm->s_in[x]), 1);
      mbar_init(smem_u32(&sm->rs_free[x]), 4);  // the peer's 4 softmax warps
      mbar_init(smem_u32(&sm->p_in[x]), 1);
      mbar_init(smem_u32(&sm->rp_free[x]), 1);
      mbar_init(smem_u32(&sm->pt_free[x]), 1);
      mbar_init(smem_u32(&sm->p_full[x]), 6);  // 4 softmax + 2 P-path warps
    }
    mbar_init(smem_u32(&sm->q_smem_full), 1);
    mbar_init(smem_u32(&sm->q_tm_full), 1);
    mbar_init(smem_u32(&sm->q_ready), kSmxWarps);
    mbar_init(smem_u32(&sm->o_done), 1);
    mbar_init(smem_u32(&sm->sum_bar), 4);
    mbar_init(smem_u32(&sm->l_bar), 1);
    mbar_init(smem_u32(&sm->drain), 1);
    sm->abort_flag = 0;
    sm->peer_abort = 0;
    fence_mbar_init_cluster();
    prefetch_tmap(&tmap);
    prefetch_tmap(&qmap);
    prefetch_tmap(&rmap);
  }
  if (warp == 1) tmem_alloc(smem_u32(&sm->tmem_base), kTmemCols);
  pdl_wait();

  if (threadIdx.x == 0) {
    // Q's RoPE part -> qr; Q's own latent half -> slots 1-2, from where the
    // softmax warps copy it into TMEM before pages 1 and 2 are loaded there
    // (two 64-row boxes: smem rows [64x, 64x+64) take heads (64x + rot) mod 128)
    mbar_arrive_expect_tx(smem_u32(&sm->q_smem_full), kQBoxBytes);
    for (uint32_t x = 0; x < 2; ++x)
      tma_load_2d_nohint(smem_u32(sm->qr) + x * (kQBoxBytes / 2), &rmap, smem_u32(&sm->q_smem_full), 0,
                         static_cast<int32_t>(row0 + ((64u * x + rot) & 127u)));
    mbar_arrive_expect_tx(smem_u32(&sm->q_tm_full), 4 * kQBoxBytes);
    for (int k = 0; k < 4; ++k)
      tma_load_2d_nohint(smem_u32(sm->kv[1]) + k * kQBoxBytes, &qmap, smem_u32(&sm->q_tm_full), col_half + 64 * k,
                         static_cast<int32_t>(row0));
  }

  // The split's first page depends only on the split, so its block-table
  // entries are read together with seq_lens, and thread 0 issues the TMA load
  // of the first page before the work item's bounds are known. An entry that
  // later proves bad (or a split past the sequence end) only moves that box out
  // of the pool, where TMA reads the fill value; the load is drained on every path.
  const int32_t* bt = a.block_table + static_cast<int64_t>(b) * a.max_pages;
  const int pg_lo = split * a.pages_per_split;
  const int pg_hi = min(a.max_pages, pg_lo + a.pages_per_split);
  const int my_pg = pg_lo + static_cast<int>(threadIdx.x);
  const int32_t my_entry = my_pg < pg_hi ? bt[my_pg] : 0;
  bool spec0 = false;  // thread 0: page 0 of the split already requested
  if (threadIdx.x == 0 && pg_lo < pg_hi) {
    const int64_t yl = static_cast<int64_t>(my_entry) * P;
    const int32_t y0 = (yl < 0 || yl >= a.num_pages * static_cast<int64_t>(P)) ? -kTileTok : static_cast<int32_t>(yl);
    if constexpr (kFp8) {
      mbar_arrive_expect_tx(smem_u32(&sm->raw_full[0]), 4 * kFp8BoxBytes);
      for (int k = 0; k < 4; ++k)
        tma_load_2d_nohint(smem_u32(sm->kv[0]) + kHalfBytes / 2 + k * kFp8BoxBytes, &tmap, smem_u32(&sm->raw_full[0]),
                           col_half + 64 * k, y0);
      if (r == 0) {
        mbar_arrive_expect_tx(smem_u32(&sm->raw_rope_full), kFp8BoxBytes);
        tma_load_2d_nohint(smem_u32(sm->rope) + kBoxBytes / 2, &tmap, smem_u32(&sm->raw_rope_full), 512, y0);
      }
    } else {
      mbar_arrive_expect_tx(smem_u32(&sm->full_kv[0]), kHalfBytes);
      for (int k = 0; k < 4; ++k)
        tma_load_2d_nohint(smem_u32(sm->kv[0]) + k * kBoxBytes, &tmap, smem_u32(&sm->full_kv[0]), col_half + 64 * k,
                           y0);
      if (r == 0) {
        mbar_arrive_expect_tx(smem_u32(&sm->full_rope), kBoxBytes);
        tma_load_2d_nohint(smem_u32(sm->rope), &tmap, smem_u32(&sm->full_rope), 512, y0);
      }
    }
    spec0 = true;
  }

  const int L = a.seq_lens[b];
  const bool bad_len = (L < Lq) || (static_cast<int64_t>(L) > static_cast<int64_t>(a.max_pages) * P);
  if (bad_len && r == 0 && threadIdx.x == 0) flag_error(a.dev_error, MLA_DEVERR_BAD_SEQLEN);
  const int n_vis = bad_len ? 0 : L - Lq + j + 1;
  const int tok_begin = pg_lo * P;
  const int tok_end = min(n_vis, (split + 1) * a.pages_per_split * P);
  int n_tiles = 0;
  {
    int local_bad = 0;
    if (tok_begin < tok_end)
      for (int pg = my_pg; pg <= (tok_end - 1) / P; pg += threads_for(kFp8)) {
        const int32_t pp = pg == my_pg ? my_entry : bt[pg];
        local_bad |= (pp < 0 || pp >= a.num_pages) ? 1 : 0;
      }
    if (__syncthreads_or(local_bad)) {
      if (r == 0 && threadIdx.x == 0) flag_error(a.dev_error, MLA_DEVERR_BAD_PAGE);
    } else if (tok_begin < tok_end) {
      n_tiles = (tok_end - tok_begin + kTileTok - 1) / kTileTok;
    }
  }
  if (threadIdx.x == 0) {
    // the inboxes' first phases: expect the peer's bytes
    for (int x = 0; x < 2 && x < n_tiles; ++x) {
      mbar_arrive_expect_tx(smem_u32(&sm->s_in[x]), kSinBytes);
      mbar_arrive_expect_tx(smem_u32(&sm->p_in[x]), kPinBytes);
    }
    mbar_arrive_expect_tx(smem_u32(&sm->l_bar), 64 * 4);
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // the peer's barriers are initialised before any remote traffic
  tc_fence_after();
  const uint32_t tmem = sm->tmem_base;
  volatile int32_t* abort_flag = &sm->abort_flag;

  if (n_tiles == 0) {
    // nothing to attend to (or rejected data; both CTAs of the pair agree):
    // let Q's loads land, write the empty outputs, tear down
    if (threadIdx.x == 0) {
      drain_wait(smem_u32(&sm->q_smem_full), 0, a.dev_error);
      drain_wait(smem_u32(&sm->q_tm_full), 0, a.dev_error);
      if (spec0) {
        drain_wait(smem_u32(kFp8 ? &sm->raw_full[0] : &sm->full_kv[0]), 0, a.dev_error);
        if (r == 0) drain_wait(smem_u32(kFp8 ? &sm->raw_rope_full : &sm->full_rope), 0, a.dev_error);
      }
    }
    write_empty(a, row0, bj, split, r);
  } else if (warp == 0) {
    // ================= TMA producer
    if (lane == 0) {
      const uint64_t pol = l2_policy_evict_first();
      auto y_of = [&](int t) {  // pool row of tile t
        const int tok = tok_begin + t * kTileTok;
        return bt[tok / P] * P + (tok % P);
      };
      auto prefetch = [&](int t) {
        const int32_t yp = y_of(t);
        for (int k = 0; k < 4; ++k) tma_prefetch_l2_2d(&tmap, col_half + 64 * k, yp);
        if ((t & 1) == static_cast<int>(r)) tma_prefetch_l2_2d(&tmap, 512, yp);
      };
      constexpr int kPrefetch = 3;
      // Two independent streams: the KV half of page i into ring slot i % 4 once
      // PV(i-4) has released it, and this CTA's RoPE boxes (pages i = r mod 2)
      // into the single RoPE buffer once QK of the previous one has read it.
      int ik = spec0 ? 1 : 0;                             // next page whose KV half to load
      int ir = (spec0 && r == 0) ? 2 : static_cast<int>(r);  // next RoPE page of this CTA
      if (spec0)
        for (int t = 1; t <= kPrefetch && t < n_tiles; ++t) prefetch(t);
      bool q_in = false;  // Q has left slots 1-2 (they may take pages)
      long long idle_since = 0;
      bool ok = true;
      while (ok && (ik < n_tiles || ir < n_tiles)) {
        bool did = false;
        if (ik < n_tiles) {
          const int slot = ik % kStages;
          if (ik == 1 && !q_in) q_in = mbar_test_wait(smem_u32(&sm->q_ready), 0);
          if ((ik != 1 || q_in) &&
              mbar_test_wait(smem_u32(&sm->empty_kv[slot]), ((ik / kStages) & 1) ^ 1)) {
            const int32_t y = y_of(ik);
            if constexpr (kFp8) {
              // E4M3 bytes into the upper half of the slot
              mbar_arrive_expect_tx(smem_u32(&sm->raw_full[slot]), 4 * kFp8BoxBytes);
              for (int k = 0; k < 4; ++k)
                tma_load_2d(smem_u32(sm->kv[slot]) + kHalfBytes / 2 + k * kFp8BoxBytes, &tmap,
                            smem_u32(&sm->raw_full[slot]), col_half + 64 * k, y, pol);
            } else {
              mbar_arrive_expect_tx(smem_u32(&sm->full_kv[slot]), kHalfBytes);
              for (int k = 0; k < 4; ++k)
                tma_load_2d(smem_u32(sm->kv[slot]) + k * kBoxBytes, &tmap, smem_u32(&sm->full_kv[slot]),
                            col_half + 64 * k, y, pol);
            }
            // pages ahead are pulled into L2 once this page's load is on its way
            for (int t = (ik == 0 ? 1 : ik + kPrefetch); t <= ik + kPrefetch && t < n_tiles; ++t) prefetch(t);
            ++ik;
            did = true;
          }
        }
        if (ir < n_tiles && mbar_test_wait(smem_u32(&sm->empty_rope), ((ir >> 1) & 1) ^ 1)) {
          const int32_t y = y_of(ir);
          if constexpr (kFp8) {
            mbar_arrive_expect_tx(smem_u32(&sm->raw_rope_full), kFp8BoxBytes);
            tma_load_2d(smem_u32(sm->rope) + kBoxBytes / 2, &tmap, smem_u32(&sm->raw_rope_full), 512, y, pol);
          } else {
            mbar_arrive_expect_tx(smem_u32(&sm->full_rope), kBoxBytes);
            tma_load_2d(smem_u32(sm->rope), &tmap, smem_u32(&sm->full_rope), 512, y, pol);
          }
          ir += 2;
          did = true;
        }
        if (did) {
          idle_since = 0;
        } else {
          // nothing to issue: suspend briefly on the next ring slot (or the RoPE buffer)
          if (ik < n_tiles)
            (void)mbar_try_wait_ns<200>(smem_u32(&sm->empty_kv[ik % kStages]), ((ik / kStages) & 1) ^ 1);
          else
            (void)mbar_try_wait_ns<200>(smem_u32(&sm->empty_rope), ((ir >> 1) & 1) ^ 1);
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
      // our own loads must land before the CTA tears down
      for (int i = max(0, ik - kStages); i < ik; ++i)
        drain_wait(smem_u32(kFp8 ? &sm->raw_full[i % kStages] : &sm->full_kv[i % kStages]), (i / kStages) & 1,
                   a.dev_error);
      if (ir - 2 >= 0)
        drain_wait(smem_u32(kFp8 ? &sm->raw_rope_full : &sm->full_rope), ((ir - 2) >> 1) & 1, a.dev_error);
      drain_wait(smem_u32(&sm->q_smem_full), 0, a.dev_error);
      drain_wait(smem_u32(&sm->q_tm_full), 0, a.dev_error);
    }
  } else if (warp == 1) {
    // ================= MMA issuer: PV(k) as soon as P(k) is complete, QK(k) as soon
    // as score buffer k & 1 has been read out and page k has landed
    if (lane == 0) {
      constexpr uint32_t kIdQK = idesc_bf16_f32(128, kTileTok, false, false);
      constexpr uint32_t kIdPV = idesc_bf16_f32(128, 256, false, true);
      // descriptor start addresses advance in 16-byte units in the low bits
      const uint64_t dKV0 = sdesc_sw128(smem_u32(sm->kv[0]), 16, 1024);          // K-major B: page rows = N
      const uint64_t dV0 = sdesc_sw128(smem_u32(sm->kv[0]), kBoxBytes, 1024);    // MN-major B: V
      const uint64_t dRope0 = sdesc_sw128(smem_u32(sm->rope), 16, 1024);
      const uint64_t dQR = sdesc_sw128(smem_u32(sm->qr), 16, 1024);              // A: Q RoPE
      const uint64_t dP0 = sdesc_sw128(smem_u32(sm->pt[0]), 16, 1024);           // A: P (K-major)
      // A barrier test costs a shared-memory round trip (hundreds of cycles under
      // load), so every test of a polling round is issued unconditionally and
      // the results are combined afterwards: their latencies overlap instead of
      // adding up. Testing a barrier that does not apply is harmless.
      auto ready = [&](uint64_t* bar, uint32_t par) { return mbar_test_wait(smem_u32(bar), par); };
      auto qk_ready = [&](int i) {
        const bool f = ready(&sm->s_free[i & 1], ((i - 2) >> 1) & 1);
        const bool k = ready(&sm->full_kv[i % kStages], (i / kStages) & 1);
        const bool q = ready(&sm->full_rope, (i >> 1) & 1);
        return (f | (i < 2)) & k & (q | ((i & 1) != static_cast<int>(r)));
      };
      auto issue_qk = [&](int i) {
        const uint32_t dS = tmem + kTmS + static_cast<uint32_t>(i & 1) * 64u;
        const uint64_t db = dKV0 + static_cast<uint64_t>(((i % kStages) * kHalfBytes) >> 4);
#pragma unroll
        for (uint32_t kk = 0; kk < 16; ++kk)
          mma_ts<kIdQK>(dS, tmem + kTmQ + kk * 8u, db + (((kk >> 2) * kBoxBytes + (kk & 3u) * 32u) >> 4),
                        kk > 0 ? 1u : 0u);
        if ((i & 1) == static_cast<int>(r)) {
#pragma unroll
          for (uint32_t kk = 0; kk < 4; ++kk)
            mma_ss(dS, dQR + ((kk * 32u) >> 4), dRope0 + ((kk * 32u) >> 4), kIdQK, 1u);
          mma_commit(smem_u32(&sm->empty_rope));
        }
        mma_commit(smem_u32(&sm->s_full[i & 1]));
      };
      auto issue_pv = [&](int i) {
        const int slot = i % kStages;
        const uint64_t dv = dV0 + static_cast<uint64_t>((slot * kHalfBytes) >> 4);
        const uint64_t dp = dP0 + static_cast<uint64_t>(((i & 1) * kPTileBytes) >> 4);
#pragma unroll
        for (uint32_t kk = 0; kk < kTileTok / 16; ++kk)
          mma_ss(tmem + kTmO, dp + ((kk * 32u) >> 4), dv + ((kk * 16u * 128u) >> 4), kIdPV, (i > 0 || kk > 0) ? 1u : 0u);
        mma_commit(smem_u32(&sm->empty_kv[slot]));
        mma_commit(smem_u32(&sm->pt_free[i & 1]));
        if (i == n_tiles - 1) mma_commit(smem_u32(&sm->o_done));
      };
      bool ok = mbar_wait<kPlain>(smem_u32(&sm->q_ready), 0, abort_flag, a.dev_error) &&
                mbar_wait<kPlain>(smem_u32(&sm->q_smem_full), 0, abort_flag, a.dev_error);
      tc_fence_after();
      int nq = 0, np = 0;  // next QK, next PV
      long long idle_since = 0;
      while (ok && np < n_tiles) {
        bool did = false;
        const bool pv_ok = ready(&sm->p_full[np & 1], (np >> 1) & 1) & (np < nq);
        const bool qk_ok = qk_ready(min(nq, n_tiles - 1)) & (nq < n_tiles);
        if (pv_ok) {
          tc_fence_after();
          issue_pv(np++);
          did = true;
        } else if (qk_ok) {
          tc_fence_after();
          issue_qk(nq++);
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
  } else if (kFp8 && warp < smx_warp0(kFp8)) {
    // ================= E4M3 -> bf16 (x scale) in place
    // The raw bytes of box k (64 rows x 64 B, unswizzled) sit at kHalfBytes/2 +
    // k * 4 KB of the slot: 1,024 chunks of 16 bytes, chunk g in box g / 256,
    // row (g / 4) mod 64, column chunk g mod 4 (the RoPE box's 256 chunks the
    // same way). Converter thread c (0..191) takes the chunks g = c + 192 j, so
    // every warp-wide load reads 512 contiguous bytes (no bank conflicts). Each
    // chunk has one scale: (its token row, group 2r + box / 2), or the RoPE group.
    constexpr int kCvtThreads = kCvtWarps * 32;
    constexpr int kLatChunks = 4 * kFp8BoxBytes / 16, kRopeChunks = kFp8BoxBytes / 16;
    constexpr int kJLat = (kLatChunks + kCvtThreads - 1) / kCvtThreads;
    constexpr int kJRope = (kRopeChunks + kCvtThreads - 1) / kCvtThreads;
    const int c = (warp - 2) * 32 + lane;
    const float* scales = a.scales;
    bool ok = true;
    // (x, y) * sc with one packed fp32 multiply (each product rounded once, as two
    // separate multiplies would), packed to bf16x2
    auto pack_bf16x2_scaled = [](float2 v, float sc) -> uint32_t {
      uint64_t p;
      asm("{\n\t.reg .b64 a, b;\n\tmov.b64 a, {%1, %2};\n\tmov.b64 b, {%3, %3};\n\t"
          "mul.rn.f32x2 %0, a, b;\n\t}"
          : "=l"(p)
          : "f"(v.x), "f"(v.y), "f"(sc));
      return pack_bf16x2(__uint_as_float(static_cast<uint32_t>(p)), __uint_as_float(static_cast<uint32_t>(p >> 32)));
    };
    // 16 E4M3 values (one uint4) x scale -> 16 bf16, written as two 16-byte
    // chunks of the 128-byte swizzled row at dst_row
    auto convert16 = [&](const uint4& x, float sc, uint8_t* dst_row, int rr, int ch) {
      const uint32_t wds[4] = {x.x, x.y, x.z, x.w};
      uint32_t outw[8];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const uint16_t pair = static_cast<uint16_t>(wds[q] >> (16 * hh));
          uint32_t h2;
          asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(pair));
          const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h2));
          outw[2 * q + hh] = pack_bf16x2_scaled(f, sc);
        }
      }
      *reinterpret_cast<uint4*>(dst_row + (((2 * ch) ^ (rr & 7)) << 4)) = make_uint4(outw[0], outw[1], outw[2], outw[3]);
      *reinterpret_cast<uint4*>(dst_row + (((2 * ch + 1) ^ (rr & 7)) << 4)) =
          make_uint4(outw[4], outw[5], outw[6], outw[7]);
    };
    for (int i = 0; ok && i < n_tiles; ++i) {
      const int slot = i % kStages;
      const bool rope_page = (i & 1) == static_cast<int>(r);
      const int tok = tok_begin + i * kTileTok;
      const int64_t y0 = static_cast<int64_t>(bt[tok / P]) * P + (tok % P);  // pool row of page row 0
      // this thread's scales, fetched before the page lands
      float sc_lat[kJLat], sc_rope[kJRope];
#pragma unroll
      for (int j = 0; j < kJLat; ++j) {
        const int g = c + kCvtThreads * j;
        sc_lat[j] = g < kLatChunks ? scales[(y0 + ((g >> 2) & 63)) * MLA_E4M3_GROUPS + 2 * r + (g >> 9)] : 0.0f;
      }
#pragma unroll
      for (int j = 0; j < kJRope; ++j) {
        const int g = c + kCvtThreads * j;
        sc_rope[j] = (rope_page && g < kRopeChunks) ? scales[(y0 + (g >> 2)) * MLA_E4M3_GROUPS + 4] : 0.0f;
      }
      if (!__all_sync(0xffffffffu, mbar_wait<kPlain>(smem_u32(&sm->raw_full[slot]), (i / kStages) & 1, abort_flag,
                                                      a.dev_error))) { ok = false; break; }
      if (rope_page && !__all_sync(0xffffffffu, mbar_wait<kPlain>(smem_u32(&sm->raw_rope_full), (i >> 1) & 1,
                                                                   abort_flag, a.dev_error))) { ok = false; break; }
      // read every chunk first: the bf16 output overlaps the raw bytes of other chunks
      uint8_t* kvs = sm->kv[slot];
      uint4 raw[kJLat], rraw[kJRope];
#pragma unroll
      for (int j = 0; j < kJLat; ++j) {
        const int g = c + kCvtThreads * j;
        if (g < kLatChunks) raw[j] = *reinterpret_cast<const uint4*>(kvs + kHalfBytes / 2 + g * 16);
      }
      if (rope_page) {
#pragma unroll
        for (int j = 0; j < kJRope; ++j) {
          const int g = c + kCvtThreads * j;
          if (g < kRopeChunks) rraw[j] = *reinterpret_cast<const uint4*>(sm->rope + kBoxBytes / 2 + g * 16);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sm->cvt_bar));
      if (!__all_sync(0xffffffffu, mbar_wait<kPlain>(smem_u32(&sm->cvt_bar), i & 1, abort_flag, a.dev_error))) {
        ok = false;
        break;
      }
#pragma unroll
      for (int j = 0; j < kJLat; ++j) {
        const int g = c + kCvtThreads * j;
        if (g < kLatChunks) {
          const int k = g >> 8, rr = (g >> 2) & 63;  // box, row
          convert16(raw[j], sc_lat[j], kvs + k * kBoxBytes + rr * 128, rr, g & 3);
        }
      }
      if (rope_page) {
#pragma unroll
        for (int j = 0; j < kJRope; ++j) {
          const int g = c + kCvtThreads * j;
          if (g < kRopeChunks) convert16(rraw[j], sc_rope[j], sm->rope + (g >> 2) * 128, g >> 2, g & 3);
        }
      }
      fence_proxy_async_smem();  // generic writes -> the MMAs' operand reads
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(smem_u32(&sm->full_kv[slot]));
        if (rope_page) mbar_arrive(smem_u32(&sm->full_rope));
      }
    }
  } else {
    // ================= softmax (own heads) / forwarding (peer's heads), epilogue
    const uint32_t q4 = static_cast<uint32_t>(warp & 3);  // TMEM lane quarter
    const int t = (warp - smx_warp0(kFp8)) >> 2;          // token half of a page; O column half
    const bool own = (q4 >> 1) == kOwnQ<kFp8>;            // rows of this CTA's heads
    const int h = static_cast<int>(q4 * 32u) + lane;      // TMEM lane (row of Q, S, P, O)
    const int hd = (h + static_cast<int>(rot)) & 127;     // the head it holds
    const int hl = h & 63;                                // index among the owner's 64 heads
    const uint32_t lanes = (q4 * 32u) << 16;
    const uint32_t tO = tmem + lanes + kTmO + t * 128, tQ = tmem + lanes + kTmQ;
    auto wwait = [&](uint64_t* bar, uint32_t par) {
      return __all_sync(0xffffffffu, mbar_wait<kPlain>(smem_u32(bar), par, abort_flag, a.dev_error));
    };
    // Barriers the peer completes: by the complete_tx of its st.async stores or
    // bulk copies (their bytes have landed in this CTA's shared memory once the
    // phase completes, like TMA data) or by a relaxed "buffer free" arrive that
    // carries no data; a CTA-scope wait suffices for both.
    auto wwait_cl = [&](uint64_t* bar, uint32_t par) {
      return __all_sync(0xffffffffu, mbar_wait<kPlain>(smem_u32(bar), par, abort_flag, a.dev_error));
    };
    // Q's own latent half of this head into TMEM (bf16 pairs, lower K index in
    // the low half). Staged in slots 1-2 as four 128 x 64 boxes with 128-byte
    // swizzle (16-byte chunk c of row h at chunk c ^ (h mod 8)); token half t
    // copies boxes 2t, 2t+1.
    {
      const bool qok = wwait(&sm->q_tm_full, 0);
      if (qok) {
        uint32_t rq[32];
#pragma unroll
        for (int bb = 0; bb < 2; ++bb) {
          const uint8_t* box = sm->kv[1] + (t * 2 + bb) * kQBoxBytes + hd * 128;  // (hd & 7 == h & 7)
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const uint4 x = *reinterpret_cast<const uint4*>(box + ((c ^ (h & 7)) << 4));
            rq[4 * c] = x.x;
            rq[4 * c + 1] = x.y;
            rq[4 * c + 2] = x.z;
            rq[4 * c + 3] = x.w;
          }
          tmem_st32(tQ + static_cast<uint32_t>((t * 2 + bb) * 32), rq);
        }
        tmem_wait_st();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sm->q_ready));  // also frees slots 1-2
    }
    // cluster addresses of the peer's inboxes
    const uint32_t peer_sin = map_to_rank(smem_u32(&sm->sin[0][0][0]), peer);  // chunk-major inbox
    const uint32_t peer_s_in = map_to_rank(smem_u32(&sm->s_in[0]), peer);
    const uint32_t peer_rs_free = map_to_rank(smem_u32(&sm->rs_free[0]), peer);
    const uint32_t peer_pt = map_to_rank(smem_u32(sm->pt[0]), peer);
    const uint32_t peer_alpha = map_to_rank(smem_u32(&sm->alpha_in[0][0]), peer);
    const uint32_t peer_p_in = map_to_rank(smem_u32(&sm->p_in[0]), peer);
    const uint32_t peer_rp_free = map_to_rank(smem_u32(&sm->rp_free[0]), peer);
    const uint32_t peer_l_in = map_to_rank(smem_u32(&sm->l_in[0]), peer);
    const uint32_t peer_l_bar = map_to_rank(smem_u32(&sm->l_bar), peer);

    const float c2 = a.softmax_scale * kLog2e;  // scores in log2 units
    float m = -CUDART_INF_F, l = 0.0f;          // own rows: running max (log2 units), half row sum
    bool ok = true;
    auto rescale_o = [&](float alpha, int first_col, int ncols) {
      for (int c = first_col; c < first_col + ncols; c += 32) {
        float o[32];
        tmem_ld32_sync(tmem + lanes + kTmO + static_cast<uint32_t>(c), o);
        uint32_t w32[32];
#pragma unroll
        for (int k = 0; k < 32; ++k) w32[k] = __float_as_uint(o[k] * alpha);
        tmem_st32(tmem + lanes + kTmO + static_cast<uint32_t>(c), w32);
      }
      tmem_wait_st();
    };
    if (own) {
      // ================= softmax of this CTA's heads. Both warps of the quarter
      // take every page, warp t the token columns [32t, 32t+32). They meet twice
      // per page on a named barrier that also ANDs their status: for the page's
      // row max (each then derives the same running max, so no state passes
      // between pages) and once both halves of the P rows are written (before the
      // bulk copy to the peer). A failed (timed-out) wait is carried to the next
      // meeting, so both warps leave the loop together.
      const int qo = static_cast<int>(q4 & 1);
      // named barriers 1, 2 (row max) for own quarters 0, 1
      auto meet = [&](int, bool v) -> bool { return qo == 0 ? bar_red_and<1, 64>(v) : bar_red_and<2, 64>(v); };
      const bool armer = (lane == 0) && (qo == 0) && (t == 0);
      for (int i = 0; i < n_tiles; ++i) {
        const int sb = i & 1;
        const uint32_t ph2 = (i >> 1) & 1;  // phase parity of the per-parity barriers for page i
        const int page_valid = min(kTileTok, tok_end - (tok_begin + i * kTileTok));
        bool good = ok && wwait(&sm->s_full[sb], ph2);
        float s[32];
        if (good) {
          tc_fence_after();
          tmem_ld32_sync(tmem + lanes + kTmS + static_cast<uint32_t>(sb) * 64u + t * 32u, s);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&sm->s_free[sb]));
        }
        // ---- full scores of this CTA's heads: own partial + the peer's
        good = good && wwait_cl(&sm->s_in[sb], ph2);
        if (good) {
          if (armer && i + 2 < n_tiles) mbar_arrive_expect_tx(smem_u32(&sm->s_in[sb]), kSinBytes);
#pragma unroll
          for (int v = 0; v < 8; ++v) {
            const float4 x = sm->sin[sb][8 * t + v][hl];
            s[4 * v] += x.x;
            s[4 * v + 1] += x.y;
            s[4 * v + 2] += x.z;
            s[4 * v + 3] += x.w;
          }
          __syncwarp();
          if (lane == 0) mbar_arrive_remote_relaxed(peer_rs_free + sb * 8);  // the peer may refill this inbox
          // ---- online softmax over this page
          if (page_valid < kTileTok) {
#pragma unroll
            for (int x = 0; x < 32; ++x)
              if (32 * t + x >= page_valid) s[x] = -CUDART_INF_F;
          }
          float t16[16];
#pragma unroll
          for (int x = 0; x < 16; ++x) t16[x] = fmaxf(s[x], s[x + 16]);
#pragma unroll
          for (int w = 8; w >= 1; w >>= 1)
#pragma unroll
            for (int x = 0; x < w; ++x) t16[x] = fmaxf(t16[x], t16[x + w]);
          sm->mx_part[sb][t][hl] = t16[0];
        }
        if (!meet(0, good)) { ok = false; break; }
        const float mx = fmaxf(sm->mx_part[sb][0][hl], sm->mx_part[sb][1][hl]);
        const bool first = (i == 0);
        const float m_prev = m;
        const float m_new = fmaxf(m_prev, mx * c2);
        const bool resc = !first && (m_new > m_prev + kRescaleLog2);
        const float m_use = (first || resc) ? m_new : m_prev;
        const float alpha = resc ? fast_exp2(m_prev - m_use) : 1.0f;  // for O, relative to page i-1
        float rsum[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        uint32_t pw[16];
#pragma unroll
        for (int x = 0; x < 16; ++x) {
          const float p0 = fast_exp2(fmaf(s[2 * x], c2, -m_use));
          const float p1 = fast_exp2(fmaf(s[2 * x + 1], c2, -m_use));
          pw[x] = pack_bf16x2(p0, p1);
          // fp32 row sum of the weights before their bf16 rounding for PV (the two
          // differ by at most one bf16 rounding; the rounded values cost more instructions)
          rsum[x & 3] += p0 + p1;
        }
        // this warp's row sum over its columns, carried to the new max
        l = (first ? 0.0f : l * fast_exp2(m_prev - m_use)) + ((rsum[0] + rsum[1]) + (rsum[2] + rsum[3]));
        m = m_use;
        const bool resc_any = __any_sync(0xffffffffu, resc);
        // ---- P of this head (this warp's 32 tokens) and the rescale factor. Tile
        // sb was last used for page i-2: by this CTA's PV(i-2) and, once the
        // peer's PV(i-2) is done, no longer by the peer.
        good = i < 2 || (wwait(&sm->pt_free[sb], ((i - 2) >> 1) & 1) && wwait_cl(&sm->rp_free[sb], ((i - 2) >> 1) & 1));
        if (!good) ok = false;  // carried to the next meeting
        if (good) {
          // P into this CTA's tile (128-byte swizzled rows, the PV operand) and into
          // the peer's: there the same 4 KB of this quarter's rows take the chunks
          // chunk-major ([16-byte chunk][32 rows]), so that each warp-wide st.async
          // writes 512 contiguous bytes; the peer's P-path warp swizzles them in place.
          uint8_t* prow = sm->pt[sb] + h * 128;
          // (in the peer these heads sit in the other pair of lane quarters, q4 ^ 2)
          const uint32_t remote =
              peer_pt + static_cast<uint32_t>(sb * kPTileBytes) + (q4 ^ 2u) * 32u * 128u + lane * 16u;
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const int ch = 4 * t + c;
            *reinterpret_cast<uint4*>(prow + ((ch ^ (h & 7)) << 4)) =
                make_uint4(pw[4 * c], pw[4 * c + 1], pw[4 * c + 2], pw[4 * c + 3]);
            st_async_v4(remote + static_cast<uint32_t>(ch * 32 * 16), __uint_as_float(pw[4 * c]),
                        __uint_as_float(pw[4 * c + 1]), __uint_as_float(pw[4 * c + 2]), __uint_as_float(pw[4 * c + 3]),
                        peer_p_in + sb * 8);
          }
          if (t == 0)
            st_async_b32(peer_alpha + static_cast<uint32_t>((sb * 64 + qo * 32 + lane) * 4), __float_as_uint(alpha),
                         peer_p_in + sb * 8);
          fence_proxy_async_smem();  // generic writes -> the MMAs' reads
        }
        // O rows of this CTA's heads (this warp's 128 of the 256 columns) may be
        // rescaled only after PV(i-1), which completes phase (i-1) >> 1 of
        // pt_free[(i-1) & 1]. (PV(i+1) cannot run before this page's P is complete,
        // so that barrier is at most one phase behind and its wait cannot alias.)
        if (resc_any) {
          if (wwait(&sm->pt_free[(i - 1) & 1], ((i - 1) >> 1) & 1)) {
            tc_fence_after();
            rescale_o(alpha, 128 * t, 128);
          } else {
            ok = false;  // carried to the next meeting
          }
        }
        if (ok) {
          if (page_valid < kTileTok) {
            // rows past the sequence end may hold anything (NaN): zero them in this
            // CTA's V half so that 0 * row stays 0 in the PV product
            uint4* base = reinterpret_cast<uint4*>(sm->kv[i % kStages]);
            const int rows = kTileTok - page_valid;
            for (int e = qo * 64 + t * 32 + lane; e < rows * 4 * 8; e += 128) {
              const int box = e / (rows * 8), rem = e % (rows * 8);
              base[(box * kBoxBytes + (page_valid + rem / 8) * 128) / 16 + (rem % 8)] = make_uint4(0, 0, 0, 0);
            }
            fence_proxy_async_smem();
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&sm->p_full[sb]));
        }
      }
      sm->mlast[t][hl] = m;
    } else {
      // ================= forwarding: warp t == 0 sends each page's partial scores
      // of the peer's heads (all 64 columns) to its inbox, as soon as they are
      // written, so that the score buffer is released early; warp t == 1 receives
      // the peer's P rows and applies its rescale factors
      if (t == 0) {
        for (int i = 0; ok && i < n_tiles; ++i) {
          const int sb = i & 1;
          if (!wwait(&sm->s_full[sb], (i >> 1) & 1)) { ok = false; break; }
          tc_fence_after();
          float sv[64];
          tmem_ld64_sync(tmem + lanes + kTmS + static_cast<uint32_t>(sb) * 64u, sv);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&sm->s_free[sb]));
          if (i >= 2 && !wwait_cl(&sm->rs_free[sb], ((i - 2) >> 1) & 1)) { ok = false; break; }
          const uint32_t dst = peer_sin + static_cast<uint32_t>((sb * 16 * 64 + hl) * 16);
          const uint32_t sbar = peer_s_in + sb * 8;
#pragma unroll
          for (int v = 0; v < 16; ++v)
            st_async_v4(dst + v * (64 * 16), sv[4 * v], sv[4 * v + 1], sv[4 * v + 2], sv[4 * v + 3], sbar);
        }
      } else {
        const bool armer = (lane == 0) && ((q4 & 1) == 0);
        for (int i = 0; ok && i < n_tiles; ++i) {
          const int sb = i & 1;
          if (!wwait_cl(&sm->p_in[sb], (i >> 1) & 1)) { ok = false; break; }
          if (armer && i + 2 < n_tiles) mbar_arrive_expect_tx(smem_u32(&sm->p_in[sb]), kPinBytes);
          {
            // the peer sent this quarter's P rows chunk-major; into the MMA's layout in place
            uint8_t* qbase = sm->pt[sb] + q4 * 32u * 128u;
            uint4 x[8];
#pragma unroll
            for (int c = 0; c < 8; ++c) x[c] = *reinterpret_cast<const uint4*>(qbase + (c * 32 + lane) * 16);
            __syncwarp();
#pragma unroll
            for (int c = 0; c < 8; ++c) *reinterpret_cast<uint4*>(qbase + lane * 128 + ((c ^ (h & 7)) << 4)) = x[c];
            fence_proxy_async_smem();  // generic writes -> the MMAs' reads
          }
          const float alpha = sm->alpha_in[sb][hl];
          // PV(i-1) done (P tile (i-1) & 1 free): needed before a rescale of these
          // O rows, and to let the peer refill that tile. pt_free advances once per
          // two pages and this warp waits on it in page order, so it cannot alias.
          bool signalled = (i == 0);
          auto tile_free = [&]() -> bool {
            if (signalled) return true;
            if (!wwait(&sm->pt_free[(i - 1) & 1], ((i - 1) >> 1) & 1)) return false;
            tc_fence_after();
            if (armer) mbar_arrive_remote_relaxed(peer_rp_free + ((i - 1) & 1) * 8);
            signalled = true;
            return true;
          };
          if (__any_sync(0xffffffffu, alpha != 1.0f)) {
            if (!tile_free()) { ok = false; break; }
            rescale_o(alpha, 0, 256);
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&sm->p_full[sb]));
          if (!tile_free()) { ok = false; break; }
        }
      }
    }
    // ---- epilogue: u = O / l (this CTA's 256 columns; this warp's 128), lse
    float l_row = 1.0f;
    if (own) {
      sm->lsum[t][hl] = l;  // (a warp that saw no page keeps l = 0 and m_mine = -inf)
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sm->sum_bar));
      if (ok && !wwait(&sm->sum_bar, 0)) ok = false;
      // both warps' sums (over their token halves) at the final max m
      l_row = 0.0f;
      for (int x = 0; x < 2; ++x)
        if (sm->mlast[x][hl] != -CUDART_INF_F) l_row += sm->lsum[x][hl] * fast_exp2(sm->mlast[x][hl] - m);
      if (t == 0) st_async_b32(peer_l_in + hl * 4, __float_as_uint(l_row), peer_l_bar);
      const float lse = (m + log2f(l_row)) * kLn2;
      if (t == 0 && ok) {
        if (S == 1) {
          if (a.lse_out != nullptr) a.lse_out[row0 + hd] = lse;
        } else {
          a.part_lse[(static_cast<int64_t>(bj) * S + split) * 128 + hd] = lse;
        }
      }
    } else {
      if (ok && !wwait_cl(&sm->l_bar, 0)) ok = false;
      l_row = sm->l_in[hl];
    }
    if (ok && wwait(&sm->o_done, 0)) {
      tc_fence_after();
      const float inv_l = 1.0f / l_row;
      const uint32_t c_out = static_cast<uint32_t>(col_half) + t * 128;
      const int head0 = static_cast<int>((q4 * 32u + rot) & 127u);  // first head of this warp's 32 rows
      // The page ring is idle once O is complete: each warp stages its 32 rows x
      // 128 columns there (16-byte chunks XOR-swizzled by row against bank
      // conflicts) and copies them out with consecutive lanes on consecutive
      // addresses, instead of one row per lane.
      const int wl = warp - smx_warp0(kFp8);
      if (S == 1) {
        uint8_t* stage = sm->kv[0] + wl * (32 * 256);
        for (int c = 0; c < 4; ++c) {
          float o[32];
          tmem_ld32_sync(tO + c * 32u, o);
          uint32_t w[16];
#pragma unroll
          for (int k = 0; k < 16; ++k) w[k] = pack_bf16x2(o[2 * k] * inv_l, o[2 * k + 1] * inv_l);
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            const int cc = c * 4 + v;
            *reinterpret_cast<uint4*>(stage + lane * 256 + ((cc ^ (lane & 15)) << 4)) =
                make_uint4(w[4 * v], w[4 * v + 1], w[4 * v + 2], w[4 * v + 3]);
          }
        }
        __syncwarp();
        uint8_t* u = reinterpret_cast<uint8_t*>(static_cast<__nv_bfloat16*>(a.u_out) + (row0 + head0) * kDC + c_out);
#pragma unroll 4
        for (int k = 0; k < 16; ++k) {
          const int row = k * 2 + (lane >> 4), ch = lane & 15;
          *reinterpret_cast<uint4*>(u + static_cast<size_t>(row) * kDC * 2 + ch * 16) =
              *reinterpret_cast<const uint4*>(stage + row * 256 + ((ch ^ (row & 15)) << 4));
        }
      } else {
        // fp32 partial rows of this split: four boxes of 32 rows x 32 columns
        // (128-byte rows, 16-byte chunk v of row r at v ^ (r mod 8)), stored by
        // TMA; the CTA goes on while they drain, and they stay in L2 (evict-last)
        // for the split merge that reads them next
        uint8_t* stage = sm->kv[0] + wl * (32 * 512);
        for (int c = 0; c < 4; ++c) {
          float o[32];
          tmem_ld32_sync(tO + c * 32u, o);
#pragma unroll
          for (int v = 0; v < 8; ++v)
            *reinterpret_cast<float4*>(stage + c * 4096 + lane * 128 + ((v ^ (lane & 7)) << 4)) =
                make_float4(o[4 * v] * inv_l, o[4 * v + 1] * inv_l, o[4 * v + 2] * inv_l, o[4 * v + 3] * inv_l);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          const int32_t prow0 = static_cast<int32_t>((static_cast<int64_t>(bj) * S + split) * 128 + head0);
          const uint64_t pol = l2_evict_last_policy();
          for (int c = 0; c < 4; ++c)
            tma_store_2d(&pmap, smem_u32(stage + c * 4096), static_cast<int32_t>(c_out) + 32 * c, prow0, pol);
          bulk_commit_group();
          bulk_wait_group_read0();  // the staging area has been read before the CTA tears down
        }
      }
    }
  }

  // ---- teardown: nothing of this CTA may still be in flight towards the peer.
  // If either CTA of the pair gave up on a wait (timeout), the work item's
  // outputs are incomplete: both then write them as for an empty item (zeros,
  // lse -inf), so that the combine skips this split instead of reading partials
  // an earlier call left behind.
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0) st_cluster_u32(map_to_rank(smem_u32(&sm->peer_abort), peer), *abort_flag != 0 ? 1u : 0u);
  cluster_sync();
  if (n_tiles > 0 && (*abort_flag != 0 || sm->peer_abort != 0)) write_empty(a, row0, bj, split, r);
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
  return a.heads == 128 && a.act == MLA_BF16 &&
         (a.cache_dtype == MLA_BF16 || (a.cache_dtype == MLA_E4M3 && a.scales != nullptr)) &&
         a.page_size % kTileTok == 0 &&
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
    bool bytes = false;
    bool f32 = false;
    CUtensorMap map;
  } e[kSlots];
  int next = 0;
  // bf16 elements, 64 x box_rows boxes, 128-byte swizzle; or (bytes) uint8
  // elements, 64-byte x box_rows boxes, no swizzle; or (f32) fp32 elements,
  // 32 x box_rows boxes, 128-byte swizzle
  bool get(const void* ptr, uint64_t rows, uint32_t cols, uint32_t box_rows, CUtensorMap* out, bool bytes = false,
           bool f32 = false) {
    for (auto& x : e)
      if (x.ptr == ptr && x.rows == rows && x.cols == cols && x.box_rows == box_rows && x.bytes == bytes &&
          x.f32 == f32) {
        *out = x.map;
        return true;
      }
    Entry& n = e[next];
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * (bytes ? 1 : (f32 ? 4 : 2))};
    const cuuint32_t box[2] = {f32 ? 32u : 64u, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    const CUtensorMapDataType dt =
        bytes ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : (f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16);
    if (tensor_map_encoder()(&n.map, dt, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                             CU_TENSOR_MAP_INTERLEAVE_NONE,
                             bytes ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B,
                             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS) {
      n.ptr = nullptr;
      return false;
    }
    n.ptr = ptr;
    n.rows = rows;
    n.cols = cols;
    n.box_rows = box_rows;
    n.bytes = bytes;
    n.f32 = f32;
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
    cudaError_t e = cudaFuncSetAttribute(decode_tc_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kSmemBytes));
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(decode_tc_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(kSmemBytes));
    if (e != cudaSuccess) return e;
    attr_set_for_device = dev;
  }
  const bool fp8 = a.cache_dtype == MLA_E4M3;
  CUtensorMap map, qmap, rmap, pmap;
  const uint64_t q_rows = static_cast<uint64_t>(a.batch) * a.q_len * 128;
  // cache as [num_pages*page_size rows][576] bf16, 64 x 64 boxes; q_lat as
  // [batch*q_len*128 rows][512] (128 x 64 boxes) and q_rope as [..][64] (64 x 64 boxes)
  if (!cache.get(a.cache, static_cast<uint64_t>(a.num_pages) * a.page_size, kRow, kTileTok, &map, fp8) ||
      !cache.get(a.q_lat, q_rows, kDC, 128, &qmap) || !cache.get(a.q_rope, q_rows, kDRope, 64, &rmap))
    return cudaErrorInvalidValue;
  // split partials [batch*q_len*splits*128 rows][512] fp32, stored as 32 x 32 boxes (a single split
  // writes u directly and never uses the map: q_lat's stands in)
  if (a.num_splits > 1) {
    if (a.part_u == nullptr || !cache.get(a.part_u, q_rows * a.num_splits, kDC, 32, &pmap, false, true))
      return cudaErrorInvalidValue;
  } else {
    pmap = qmap;
  }
  const int64_t items = static_cast<int64_t>(a.batch) * a.q_len * a.num_splits;
  const dim3 grid(static_cast<unsigned>(2 * items));
  if (fp8)
    return launch_pdl(decode_tc_kernel<true>, grid, dim3(threads_for(true)), kSmemBytes, s, map, qmap, rmap, pmap, a);
  return launch_pdl(decode_tc_kernel<false>, grid, dim3(threads_for(false)), kSmemBytes, s, map, qmap, rmap, pmap, a);
}

}  // namespace mla
