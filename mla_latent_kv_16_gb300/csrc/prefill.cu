// Prefill in the MHA form on the 5th-generation tensor cores.
//
// What is computed ("DeepSeek's attention evolution - [MLA]" §2.5: for a long
// prompt the shared latent is expanded back into per-head keys and values and
// ordinary multi-head attention runs; "Model Architecture Driving Inference
// Systems" FAQ Q2: prefill runs uncompressed, matrix absorption is for decode):
// for the T cached rows (c_KV[t] in R^512, rotated k_R[t] in R^64) of one
// sequence and the queries of its last Tq positions,
//   K_h[t] = [W_UK[h] c_KV[t] ; k_R[t]] (192),  V_h[t] = W_UV[h] c_KV[t] (128)
//   o_h[j] = sum_t softmax_t(q_h[j] . K_h[t] * scale) V_h[t]   over t <= T - Tq + j
// with q_h[j] = [q_nope ; q_rope] (192).
//
// Two steps. (1) The expansion is one product per weight, [T x 512] x
// [512 x H*128], on the persistent tcgen05 linear layer (the rows' c_KV part
// read with their 576-element stride), into a caller workspace. (2) A causal
// flash-attention kernel, one CTA per (head, tile of 128 queries):
//   S = Q K^T  : M = 128 queries, N = 128 keys, K = 192 (12 MMAs), S in TMEM
//   O += P V   : M = 128 queries, N = 128 (d_v), K = 128 keys (8 MMAs), with P
//                (bf16) in TMEM as the A operand and V an MN-major operand
// Warp 0 streams K and V tiles through TMA rings of two, warp 1 issues the
// QK products and warp 10 the PV products, each as soon as its inputs are
// ready (two issuing threads: the tensor pipe interleaves their MMAs, and the
// softmax of one tile overlaps the products of the others), warps 2-9 (two per TMEM lane quarter, thread
// = query row, each warp half of the tile's keys) run the online softmax:
// running max with a lazy rescale of O
// (only when the max grows by more than 2^8), fp32 row sums of the weights
// (before their bf16 rounding for the PV product: the two differ by at most one
// bf16 rounding, and summing the rounded values cost the softmax 1.5 more
// instructions per weight). Tiles past the query's position are not visited; the
// diagonal ones are masked per element. Every wait is bounded; on a timeout
// the CTA raises MLA_DEVERR_TIMEOUT, lets its own copies and MMAs land, writes
// NaN outputs for its rows and frees TMEM.
//
// TMEM (512 columns): two S buffers [0,128) [128,256), O [256,384), two P
// buffers [384,448) [448,512) (bf16 pairs). Shared memory: the Q tile (three
// 128 x 64 boxes: nope 0-63, nope 64-127, rope), two K stages (same three
// boxes) and two V stages (two boxes, d 0-63 and 64-127), 128-byte swizzled.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <math_constants.h>

#include "common.cuh"
#include "launchers.h"
#include "tc_ptx.cuh"

namespace mla {
namespace {

using namespace tc;

// TMA warp, QK-issue warp, eight softmax warps (two per TMEM lane quarter), PV-issue warp
constexpr int kPfThreads = 352;
constexpr int kPvWarp = 10;
constexpr int kRowsTile = 128;    // queries per CTA and keys per tile
constexpr int kBox = 128 * 128;   // 128 rows x 64 bf16
constexpr int kStagesK = 2, kStagesV = 2;
constexpr uint32_t kTmS = 0, kTmO = 256, kTmP = 384;
constexpr float kRescaleLog2 = 8.0f;
constexpr int kHeadGroup = 16;

struct __align__(1024) PfSmem {
  uint8_t q[3][kBox];
  uint8_t k[kStagesK][3][kBox];
  uint8_t v[kStagesV][2][kBox];
  uint64_t q_full;
  uint64_t k_full[kStagesK], k_empty[kStagesK];
  uint64_t v_full[kStagesV], v_empty[kStagesV];
  uint64_t s_full[2], s_free[2];  // S of tile j in buffer j & 1: written by QK / read by the 8 softmax warps
  uint64_t p_full[2];             // P of tile j in buffer j & 1 (and any O rescale) complete: 8 warps
  uint64_t p_free[2];             // PV of the tile that last used P buffer x is done
  uint64_t o_done, drain, drain_pv;
  float mx_part[2][2][128];       // tile j's row max over key half t, in [j & 1][t]
  float lsum[2][128];             // each softmax warp's row sum, for the epilogue
  uint32_t tmem_base;
  int32_t abort_flag;
};
constexpr size_t kPfSmemBytes = sizeof(PfSmem) + 1024;
static_assert(kPfSmemBytes <= 232448, "shared memory budget of one CTA");

struct PfMaps {
  CUtensorMap q, qr, k, kr, v;
};

__device__ __forceinline__ void pf_drain(uint32_t bar, uint32_t parity, int32_t* dev_error) {
  volatile int32_t never = 0;
  mbar_wait<2>(bar, parity, &never, dev_error);
}

__global__ void __launch_bounds__(kPfThreads, 1) prefill_attn_kernel(const __grid_constant__ PfMaps maps,
                                                                      const PrefillArgs a) {
  extern __shared__ uint8_t smem_raw[];
  PfSmem* sm = reinterpret_cast<PfSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int H = a.heads, T = a.n_tokens, Tq = a.n_queries;
  const int n_qt = (Tq + kRowsTile - 1) / kRowsTile;
  // Heads go in groups of up to 16, whose K and V (2 MB per head at 4096
  // tokens) stay in L2 while every query tile of the group reads them; within
  // a group the longest (last) query tiles go first.
  const int G = min(kHeadGroup, H);
  const int grp = static_cast<int>(blockIdx.x / static_cast<unsigned>(G * n_qt));
  const int gh = min(G, H - grp * G);  // heads in this group (fewer in a last, partial one)
  const int r_in = static_cast<int>(blockIdx.x) - grp * G * n_qt;
  const int h = grp * G + r_in % gh;
  const int qt = n_qt - 1 - r_in / gh;
  const int q0 = qt * kRowsTile;
  const int pos0 = T - Tq + q0;                              // position of the tile's first query
  const int pos_last = min(T - 1, pos0 + kRowsTile - 1);     // of its last real query
  const int n_kt = pos_last / kRowsTile + 1;                 // key tiles it sees

  pdl_trigger();
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&sm->q_full), 1);
    for (int s = 0; s < kStagesK; ++s) {
      mbar_init(smem_u32(&sm->k_full[s]), 1);
      mbar_init(smem_u32(&sm->k_empty[s]), 1);
    }
    for (int s = 0; s < kStagesV; ++s) {
      mbar_init(smem_u32(&sm->v_full[s]), 1);
      mbar_init(smem_u32(&sm->v_empty[s]), 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(smem_u32(&sm->s_full[x]), 1);
      mbar_init(smem_u32(&sm->s_free[x]), 8);
      mbar_init(smem_u32(&sm->p_full[x]), 8);
      mbar_init(smem_u32(&sm->p_free[x]), 1);
    }
    mbar_init(smem_u32(&sm->o_done), 1);
    mbar_init(smem_u32(&sm->drain), 1);
    mbar_init(smem_u32(&sm->drain_pv), 1);
    sm->abort_flag = 0;
    fence_mbar_init_cluster();
    prefetch_tmap(&maps.q);
    prefetch_tmap(&maps.qr);
    prefetch_tmap(&maps.k);
    prefetch_tmap(&maps.kr);
    prefetch_tmap(&maps.v);
    // The queries are the caller's data, which no kernel of ours writes: they
    // may be requested before the wait for the expansion that writes K and V.
    mbar_arrive_expect_tx(smem_u32(&sm->q_full), 3 * kBox);
    tma_load_2d_nohint(smem_u32(sm->q[0]), &maps.q, smem_u32(&sm->q_full), h * 128, q0);
    tma_load_2d_nohint(smem_u32(sm->q[1]), &maps.q, smem_u32(&sm->q_full), h * 128 + 64, q0);
    tma_load_2d_nohint(smem_u32(sm->q[2]), &maps.qr, smem_u32(&sm->q_full), h * 64, q0);
  }
  if (warp == 1) tmem_alloc(smem_u32(&sm->tmem_base), 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  pdl_wait();
  const uint32_t tmem = sm->tmem_base;
  volatile int32_t* abort_flag = &sm->abort_flag;

  if (warp == 0) {
    // ================= TMA producer: K(0), then K(j + 1) before V(j)
    if (lane == 0) {
      int ik = 0, iv = 0;
      bool ok = true;
      auto load_k = [&](int j) -> bool {
        const int s = j % kStagesK;
        if (j >= kStagesK && !mbar_wait<2>(smem_u32(&sm->k_empty[s]), ((j / kStagesK) & 1) ^ 1, abort_flag,
                                           a.dev_error))
          return false;
        const uint32_t bar = smem_u32(&sm->k_full[s]);
        mbar_arrive_expect_tx(bar, 3 * kBox);
        tma_load_2d_nohint(smem_u32(sm->k[s][0]), &maps.k, bar, h * 128, j * kRowsTile);
        tma_load_2d_nohint(smem_u32(sm->k[s][1]), &maps.k, bar, h * 128 + 64, j * kRowsTile);
        tma_load_2d_nohint(smem_u32(sm->k[s][2]), &maps.kr, bar, 512, j * kRowsTile);
        return true;
      };
      auto load_v = [&](int j) -> bool {
        const int s = j % kStagesV;
        if (j >= kStagesV && !mbar_wait<2>(smem_u32(&sm->v_empty[s]), ((j / kStagesV) & 1) ^ 1, abort_flag,
                                           a.dev_error))
          return false;
        const uint32_t bar = smem_u32(&sm->v_full[s]);
        mbar_arrive_expect_tx(bar, 2 * kBox);
        tma_load_2d_nohint(smem_u32(sm->v[s][0]), &maps.v, bar, h * 128, j * kRowsTile);
        tma_load_2d_nohint(smem_u32(sm->v[s][1]), &maps.v, bar, h * 128 + 64, j * kRowsTile);
        return true;
      };
      ok = load_k(0);
      if (ok) ik = 1;
      for (int j = 0; ok && j < n_kt; ++j) {
        if (j + 1 < n_kt) {
          ok = load_k(j + 1);
          if (!ok) break;
          ik = j + 2;
        }
        ok = load_v(j);
        if (!ok) break;
        iv = j + 1;
      }
      // our own loads land before the CTA tears down
      for (int j = max(0, ik - kStagesK); j < ik; ++j)
        pf_drain(smem_u32(&sm->k_full[j % kStagesK]), (j / kStagesK) & 1, a.dev_error);
      for (int j = max(0, iv - kStagesV); j < iv; ++j)
        pf_drain(smem_u32(&sm->v_full[j % kStagesV]), (j / kStagesV) & 1, a.dev_error);
      pf_drain(smem_u32(&sm->q_full), 0, a.dev_error);
    }
  } else if (warp == 1) {
    // ================= QK issue: S(j) = Q K(j)^T as soon as K(j) has landed and
    // score buffer j & 1 has been read out. The PV products are issued by
    // another warp: an issuing thread stays busy while the tensor pipe takes
    // its MMAs, so with one thread for both a ready PV waited behind the next
    // QK's issue, and the next QK behind the PV.
    if (lane == 0) {
      constexpr uint32_t kIdQK = idesc_bf16_f32(128, 128, false, false);
      const uint64_t dQ = sdesc_sw128(smem_u32(sm->q[0]), 16, 1024);
      const uint64_t dK = sdesc_sw128(smem_u32(sm->k[0][0]), 16, 1024);
      bool ok = mbar_wait<2>(smem_u32(&sm->q_full), 0, abort_flag, a.dev_error);
      for (int j = 0; ok && j < n_kt; ++j) {
        const int s = j % kStagesK, sb = j & 1;
        ok = mbar_wait<2>(smem_u32(&sm->k_full[s]), (j / kStagesK) & 1, abort_flag, a.dev_error);
        if (ok && j >= 2) ok = mbar_wait<2>(smem_u32(&sm->s_free[sb]), ((j - 2) >> 1) & 1, abort_flag, a.dev_error);
        if (!ok) break;
        tc_fence_after();
        const uint32_t d = tmem + kTmS + static_cast<uint32_t>(sb) * 128u;
        const uint64_t dk = dK + static_cast<uint64_t>((s * 3 * kBox) >> 4);
#pragma unroll
        for (uint32_t kk = 0; kk < 12; ++kk) {
          const uint32_t off = ((kk >> 2) * kBox + (kk & 3u) * 32u) >> 4;
          mma_ss(d, dQ + off, dk + off, kIdQK, kk > 0 ? 1u : 0u);
        }
        mma_commit(smem_u32(&sm->k_empty[s]));
        mma_commit(smem_u32(&sm->s_full[sb]));
      }
      mma_commit(smem_u32(&sm->drain));
      pf_drain(smem_u32(&sm->drain), 0, a.dev_error);
    }
  } else if (warp == kPvWarp) {
    // ================= PV issue: O += P(j) V(j) once P(j) is complete (P in TMEM)
    if (lane == 0) {
      constexpr uint32_t kIdPV = idesc_bf16_f32(128, 128, false, true);
      const uint64_t dV = sdesc_sw128(smem_u32(sm->v[0][0]), kBox, 1024);  // MN-major: boxes of 64 d apart
      bool ok = true;
      for (int j = 0; ok && j < n_kt; ++j) {
        const int s = j % kStagesV, pb = j & 1;
        ok = mbar_wait<2>(smem_u32(&sm->p_full[pb]), (j >> 1) & 1, abort_flag, a.dev_error) &&
             mbar_wait<2>(smem_u32(&sm->v_full[s]), (j / kStagesV) & 1, abort_flag, a.dev_error);
        if (!ok) break;
        tc_fence_after();
        const uint64_t dv = dV + static_cast<uint64_t>((s * 2 * kBox) >> 4);
#pragma unroll
        for (uint32_t kk = 0; kk < 8; ++kk)
          mma_ts<kIdPV>(tmem + kTmO, tmem + kTmP + static_cast<uint32_t>(pb) * 64u + kk * 8u,
                        dv + ((kk * 16u * 128u) >> 4), (j > 0 || kk > 0) ? 1u : 0u);
        mma_commit(smem_u32(&sm->v_empty[s]));
        mma_commit(smem_u32(&sm->p_free[pb]));
        if (j == n_kt - 1) mma_commit(smem_u32(&sm->o_done));
      }
      mma_commit(smem_u32(&sm->drain_pv));
      pf_drain(smem_u32(&sm->drain_pv), 0, a.dev_error);
    }
  } else {
    // ================= softmax (warps 2-9): two warps per TMEM lane quarter,
    // thread = query row, warp t the key columns [64t, 64t+64) of every tile.
    // The two warps of a quarter meet once per tile on a named barrier that also
    // ANDs their status, to combine their halves' row maxima (each then derives
    // the same running max); a failed wait is carried to the next meeting, so
    // both leave the loop together.
    const uint32_t q4 = static_cast<uint32_t>(warp & 3);
    const int t = (warp - 2) >> 2;
    const int row = static_cast<int>(q4 * 32u) + lane;
    const int qpos = pos0 + row;  // this query's position in the sequence
    const uint32_t lanes = (q4 * 32u) << 16;
    const float c2 = a.softmax_scale * kLog2e;
    const float masked = c2 >= 0.0f ? -CUDART_INF_F : CUDART_INF_F;  // raw score whose scaled value is -inf
    auto wwait = [&](uint64_t* bar, uint32_t par) {
      return __all_sync(0xffffffffu, mbar_wait<0>(smem_u32(bar), par, abort_flag, a.dev_error));
    };
    auto meet = [&](bool v) -> bool {
      switch (q4) {
        case 0: return bar_red_and<1, 64>(v);
        case 1: return bar_red_and<2, 64>(v);
        case 2: return bar_red_and<3, 64>(v);
        default: return bar_red_and<4, 64>(v);
      }
    };
    float m = -CUDART_INF_F, l = 0.0f;
    bool ok = true;
    for (int j = 0; j < n_kt; ++j) {
      const int sb = j & 1;
      bool good = ok && wwait(&sm->s_full[sb], (j >> 1) & 1);
      float s[64];
      if (good) {
        tc_fence_after();
        // this warp's 64 key columns in one TMEM load (one round trip)
        // raw scores; the scale into log2 units is folded into each exponent's FMA below
        tmem_ld64_sync(tmem + lanes + kTmS + static_cast<uint32_t>(sb) * 128u + static_cast<uint32_t>(64 * t), s);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&sm->s_free[sb]));
        // causal mask: key k0 + x is visible to this query if k0 + x <= qpos
        // (keys past the sequence end are past every query, so masked too); a
        // masked score is the one whose scaled value is -inf
        const int k0 = j * kRowsTile + 64 * t;
        if (k0 + 63 > pos0) {
#pragma unroll
          for (int x = 0; x < 64; ++x)
            if (k0 + x > qpos) s[x] = masked;
        }
        // the largest scaled score: the raw maximum (or minimum, for a negative scale) times c2
        float mx4[4] = {s[0], s[1], s[2], s[3]};
        if (c2 >= 0.0f) {
#pragma unroll
          for (int x = 4; x < 64; ++x) mx4[x & 3] = fmaxf(mx4[x & 3], s[x]);
          sm->mx_part[sb][t][row] = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3])) * c2;
        } else {
#pragma unroll
          for (int x = 4; x < 64; ++x) mx4[x & 3] = fminf(mx4[x & 3], s[x]);
          sm->mx_part[sb][t][row] = fminf(fminf(mx4[0], mx4[1]), fminf(mx4[2], mx4[3])) * c2;
        }
      }
      if (!meet(good)) { ok = false; break; }
      const float mx = fmaxf(sm->mx_part[sb][0][row], sm->mx_part[sb][1][row]);
      const bool first = (j == 0);
      const float m_prev = m;
      const float m_new = fmaxf(m_prev, mx);
      const bool resc = !first && (m_new > m_prev + kRescaleLog2);
      const float m_use = (first || resc) ? m_new : m_prev;
      uint32_t pw[32];
      float rsum[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
      for (int x = 0; x < 32; ++x) {
        const float p0 = fast_exp2(fmaf(s[2 * x], c2, -m_use)), p1 = fast_exp2(fmaf(s[2 * x + 1], c2, -m_use));
        pw[x] = pack_bf16x2(p0, p1);
        rsum[x & 3] += p0 + p1;
      }
      l = (first ? 0.0f : l * fast_exp2(m_prev - m_use)) + ((rsum[0] + rsum[1]) + (rsum[2] + rsum[3]));
      m = m_use;
      const bool resc_any = __any_sync(0xffffffffu, resc);
      const float alpha = resc ? fast_exp2(m_prev - m_use) : 1.0f;
      // P of this tile: the buffer was last read by PV(j - 2); this warp's 64
      // keys are its columns [32t, 32t+32) (bf16 pairs)
      if (j >= 2 && !wwait(&sm->p_free[sb], ((j - 2) >> 1) & 1)) { ok = false; continue; }
      tc_fence_after();
      tmem_st32(tmem + lanes + kTmP + static_cast<uint32_t>(sb) * 64u + static_cast<uint32_t>(32 * t), pw);
      // O rows (this warp's 64 of the 128 columns) rescale only after PV(j - 1)
      // (phase (j - 1) >> 1 of p_free[(j - 1) & 1])
      if (resc_any) {
        if (!wwait(&sm->p_free[(j - 1) & 1], ((j - 1) >> 1) & 1)) { ok = false; continue; }
        tc_fence_after();
        for (int c = 64 * t; c < 64 * t + 64; c += 32) {
          float o[32];
          tmem_ld32_sync(tmem + lanes + kTmO + static_cast<uint32_t>(c), o);
          uint32_t w32[32];
#pragma unroll
          for (int k = 0; k < 32; ++k) w32[k] = __float_as_uint(o[k] * alpha);
          tmem_st32(tmem + lanes + kTmO + static_cast<uint32_t>(c), w32);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sm->p_full[sb]));
    }
    // ---- epilogue: o = O / l (bf16), lse; an aborted CTA writes NaN. Both warps
    // of a quarter hold the same running max, so the row sum is the sum of theirs.
    sm->lsum[t][row] = l;
    const bool done = meet(ok && wwait(&sm->o_done, 0));
    tc_fence_after();
    const float l_row = sm->lsum[0][row] + sm->lsum[1][row];
    const int q = q0 + row;
    const float inv_l = 1.0f / l_row;
    // stage this warp's 32 rows x 128 bytes (its 64 columns) in the (idle) Q
    // tile, then copy them out with consecutive lanes on consecutive addresses
    uint8_t* stage = sm->q[0] + (warp - 2) * (32 * 128);
    for (int c = 0; c < 2; ++c) {
      float o[32];
      if (done) {
        tmem_ld32_sync(tmem + lanes + kTmO + static_cast<uint32_t>(64 * t + 32 * c), o);
      } else {
#pragma unroll
        for (int k = 0; k < 32; ++k) o[k] = CUDART_NAN_F;
      }
      uint32_t w[16];
#pragma unroll
      for (int k = 0; k < 16; ++k) w[k] = pack_bf16x2(o[2 * k] * inv_l, o[2 * k + 1] * inv_l);
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        const int cc = c * 4 + v;
        *reinterpret_cast<uint4*>(stage + lane * 128 + ((cc ^ (lane & 7)) << 4)) =
            make_uint4(w[4 * v], w[4 * v + 1], w[4 * v + 2], w[4 * v + 3]);
      }
    }
    __syncwarp();
    uint8_t* out = static_cast<uint8_t*>(a.o);
    for (int k = 0; k < 8; ++k) {
      const int r = k * 4 + (lane >> 3), ch = lane & 7;
      const int qr = q0 + static_cast<int>(q4 * 32u) + r;
      if (qr < Tq)
        *reinterpret_cast<uint4*>(out + (static_cast<int64_t>(qr) * H + h) * 256 + t * 128 + ch * 16) =
            *reinterpret_cast<const uint4*>(stage + r * 128 + ((ch ^ (r & 7)) << 4));
    }
    if (t == 0 && a.lse != nullptr && q < Tq)
      a.lse[static_cast<int64_t>(q) * H + h] = done ? (m + log2f(l_row)) * kLn2 : CUDART_NAN_F;
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 pf_encoder() {
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

// [rows][cols] bf16 with row stride `stride` elements, 64 x 128 boxes, 128-byte swizzle
bool pf_map(CUtensorMap* m, const void* ptr, uint64_t rows, uint64_t cols, uint64_t stride) {
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {stride * 2};
  const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(kRowsTile)};
  const cuuint32_t estr[2] = {1, 1};
  return pf_encoder()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                      CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

size_t prefill_workspace_bytes(int32_t n_tokens, int32_t heads) {
  const size_t one = (static_cast<size_t>(n_tokens) * heads * 128 * 2 + 255) & ~size_t(255);
  return 2 * one;
}

bool prefill_supported() { return pf_encoder() != nullptr; }

cudaError_t launch_prefill(const PrefillArgs& a, cudaStream_t s) {
  const int64_t T = a.n_tokens, H = a.heads;
  // (1) expansion: K_nope = C W_UK^T, V = C W_UV^T with C = rows[:, :512]
  LinearArgs lk{a.rows, a.w_uk, a.k_nope, nullptr, a.n_tokens, static_cast<int32_t>(H * 128), 512, 1, MLA_BF16, 0, 576};
  LinearArgs lv{a.rows, a.w_uv, a.v, nullptr, a.n_tokens, static_cast<int32_t>(H * 128), 512, 1, MLA_BF16, 0, 576};
  if (linear_splits(a.n_tokens, lk.n_out, 512, MLA_BF16) != 1) return cudaErrorNotSupported;
  cudaError_t e = launch_linear(lk, s, false);
  if (e == cudaSuccess) e = launch_linear(lv, s, false);
  if (e != cudaSuccess) return e;
  // (2) causal attention
  PfMaps maps;
  if (!pf_map(&maps.q, a.q_nope, static_cast<uint64_t>(a.n_queries), static_cast<uint64_t>(H * 128),
              static_cast<uint64_t>(H * 128)) ||
      !pf_map(&maps.qr, a.q_rope, static_cast<uint64_t>(a.n_queries), static_cast<uint64_t>(H * 64),
              static_cast<uint64_t>(H * 64)) ||
      !pf_map(&maps.k, a.k_nope, static_cast<uint64_t>(T), static_cast<uint64_t>(H * 128),
              static_cast<uint64_t>(H * 128)) ||
      !pf_map(&maps.kr, a.rows, static_cast<uint64_t>(T), 576, 576) ||
      !pf_map(&maps.v, a.v, static_cast<uint64_t>(T), static_cast<uint64_t>(H * 128), static_cast<uint64_t>(H * 128)))
    return cudaErrorInvalidValue;
  static int attr_dev = -1;
  int dev = 0;
  e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (attr_dev != dev) {
    e = cudaFuncSetAttribute(prefill_attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kPfSmemBytes));
    if (e != cudaSuccess) return e;
    attr_dev = dev;
  }
  const int64_t n_qt = (a.n_queries + kRowsTile - 1) / kRowsTile;
  const int64_t blocks = n_qt * H;
  if (blocks > 0x7fffffff) return cudaErrorInvalidConfiguration;
  return launch_pdl(prefill_attn_kernel, dim3(static_cast<unsigned>(blocks)), dim3(kPfThreads), kPfSmemBytes, s, maps,
                    a);
}

}  // namespace mla
