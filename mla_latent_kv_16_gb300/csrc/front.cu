// Decode-layer front end: from the hidden states h of the step's new tokens to
// the inputs of the attention step ("Multi-Head Latent Attention (MLA)" page,
// "PyTorch Reference Implementation", forward_decode_absorbed steps 1 and 2;
// "Model Architecture Driving Inference Systems" §2.1, §2.3):
//
//   [c_q' ; c_kv' ; k_r] = W_DQKV h        (W_DQ, W_DKV, W_KR stacked row-wise)
//   c_q  = RMSNorm(c_q') * g_q,  c_kv = RMSNorm(c_kv') * g_kv
//   [q_nope ; q_r] = W_UQR c_q             (W_UQ, W_QR stacked row-wise)
//   q_rope = RoPE_pos(q_r)                 (adjacent pairs, the cache's convention)
//
// Both products are the generic linear layer (linear.cu) writing fp32 sums;
// two small kernels finish each: the split sum, the RMS norms and the output
// rounding after the first, the split sum and the query rotation after the
// second. k_r leaves unrotated: mla_cache_append rotates it.
#include <math_constants.h>

#include "common.cuh"
#include "launchers.h"

namespace mla {
namespace {

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

struct FrontLayout {
  int32_t ma, mb;              // rows of W_DQKV and of W_UQR
  int32_t splits_a, splits_b;  // their K splits
  size_t off_cq, off_b, total;
};

FrontLayout front_layout(int32_t n, int32_t d_model, int32_t d_cq, int32_t heads, mla_dtype_t act) {
  FrontLayout l{};
  l.ma = d_cq + kDC + kDRope;
  l.mb = heads * (kDNope + kDRope);
  l.splits_a = linear_splits(n, l.ma, d_model, act);
  l.splits_b = linear_splits(n, l.mb, d_cq, act);
  const size_t esz = act == MLA_F32 ? 4 : 2;
  l.off_cq = linear_partial_bytes(n, l.ma, d_model, act);
  l.off_b = l.off_cq + align256(static_cast<size_t>(n) * d_cq * esz);
  l.total = l.off_b + linear_partial_bytes(n, l.mb, d_cq, act);
  return l;
}

constexpr int kFinishThreads = 1024;

// grid (n), block 1024: token t's 1536 + 512 + 64 sums; the two mean squares in
// a first pass over the (L2-resident) partials, the outputs in a second.
template <typename T>
__global__ void __launch_bounds__(kFinishThreads) front_finish_a_kernel(FrontArgs f, const float* part, int splits,
                                                                        T* c_q) {
  pdl_trigger();
  pdl_wait();
  __shared__ float red[2][kFinishThreads / 32];
  const int t = blockIdx.x;
  const int ma = f.d_cq + kDC + kDRope;
  const int64_t stride = static_cast<int64_t>(f.n_tokens) * ma;
  const int64_t row = static_cast<int64_t>(t) * ma;
  float sq_q = 0.0f, sq_kv = 0.0f;
  for (int i = threadIdx.x; i < f.d_cq + kDC; i += kFinishThreads) {
    const float v = split_sum(part, row + i, stride, splits);
    if (i < f.d_cq)
      sq_q = fmaf(v, v, sq_q);
    else
      sq_kv = fmaf(v, v, sq_kv);
  }
  sq_q = warp_sum(sq_q);
  sq_kv = warp_sum(sq_kv);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) {
    red[0][warp] = sq_q;
    red[1][warp] = sq_kv;
  }
  __syncthreads();
  float tq = 0.0f, tkv = 0.0f;
#pragma unroll
  for (int w = 0; w < kFinishThreads / 32; ++w) {
    tq += red[0][w];
    tkv += red[1][w];
  }
  const float inv_q = 1.0f / sqrtf(tq / static_cast<float>(f.d_cq) + f.eps);
  const float inv_kv = 1.0f / sqrtf(tkv / static_cast<float>(kDC) + f.eps);
  const T* g_q = static_cast<const T*>(f.g_q);
  const T* g_kv = static_cast<const T*>(f.g_kv);
  for (int i = threadIdx.x; i < ma; i += kFinishThreads) {
    const float v = split_sum(part, row + i, stride, splits);
    if (i < f.d_cq) {
      ActIO<T>::store(c_q + static_cast<int64_t>(t) * f.d_cq + i, v * inv_q * ActIO<T>::load(g_q + i));
    } else if (i < f.d_cq + kDC) {
      const int j = i - f.d_cq;
      ActIO<T>::store(static_cast<T*>(f.c_kv) + static_cast<int64_t>(t) * kDC + j, v * inv_kv * ActIO<T>::load(g_kv + j));
    } else {
      ActIO<T>::store(static_cast<T*>(f.k_r) + static_cast<int64_t>(t) * kDRope + (i - f.d_cq - kDC), v);
    }
  }
}

// grid (n, ceil(mb / 512)), block 256: one adjacent pair of outputs per thread.
// Pairs in the first H*128 rows are q_nope; the rest are q_r, rotated by the
// token's position in fp32 with every product and sum rounded separately, as
// the cache append rotates k_R.
template <typename T>
__global__ void __launch_bounds__(256) front_finish_b_kernel(FrontArgs f, const float* part, int splits) {
  pdl_trigger();
  pdl_wait();
  const int t = blockIdx.x;
  const int mb = f.heads * (kDNope + kDRope);
  const int o = 2 * (blockIdx.y * 256 + threadIdx.x);
  if (o >= mb) return;
  const int64_t stride = static_cast<int64_t>(f.n_tokens) * mb;
  const int64_t row = static_cast<int64_t>(t) * mb;
  const float v0 = split_sum(part, row + o, stride, splits);
  const float v1 = split_sum(part, row + o + 1, stride, splits);
  const int n_nope = f.heads * kDNope;
  if (o < n_nope) {
    T* q = static_cast<T*>(f.q_nope) + static_cast<int64_t>(t) * n_nope + o;
    ActIO<T>::store(q, v0);
    ActIO<T>::store(q + 1, v1);
    return;
  }
  const int r = o - n_nope;  // head r / 64, element r % 64 (even)
  T* q = static_cast<T*>(f.q_rope) + static_cast<int64_t>(t) * (f.heads * kDRope) + r;
  const int32_t pos = f.positions[t];
  if (pos < 0 || pos >= f.max_pos) {
    if (r == 0) flag_error(f.dev_error, MLA_DEVERR_BAD_POSITION);
    ActIO<T>::store(q, 0.0f);
    ActIO<T>::store(q + 1, 0.0f);
    return;
  }
  const int i = (r % kDRope) >> 1;
  const float c = f.cos_t[static_cast<int64_t>(pos) * (kDRope / 2) + i];
  const float s = f.sin_t[static_cast<int64_t>(pos) * (kDRope / 2) + i];
  ActIO<T>::store(q, __fsub_rn(__fmul_rn(v0, c), __fmul_rn(v1, s)));
  ActIO<T>::store(q + 1, __fadd_rn(__fmul_rn(v0, s), __fmul_rn(v1, c)));
}

template <typename T>
cudaError_t launch_front_t(const FrontArgs& f, cudaStream_t s) {
  const FrontLayout l = front_layout(f.n_tokens, f.d_model, f.d_cq, f.heads, f.act);
  uint8_t* ws = static_cast<uint8_t*>(f.workspace);
  float* part_a = reinterpret_cast<float*>(ws);
  T* c_q = reinterpret_cast<T*>(ws + l.off_cq);
  float* part_b = reinterpret_cast<float*>(ws + l.off_b);
  // the weights are the caller's, written by no kernel of this library
  LinearArgs a{f.h, f.w_dqkv, nullptr, part_a, f.n_tokens, l.ma, f.d_model, l.splits_a, f.act, 1};
  cudaError_t e = launch_linear(a, s, false);
  if (e != cudaSuccess) return e;
  e = launch_pdl(front_finish_a_kernel<T>, dim3(f.n_tokens), dim3(kFinishThreads), 0, s, f,
                 static_cast<const float*>(part_a),
                 l.splits_a, c_q);
  if (e != cudaSuccess) return e;
  LinearArgs b{c_q, f.w_uqr, nullptr, part_b, f.n_tokens, l.mb, f.d_cq, l.splits_b, f.act, 1};
  e = launch_linear(b, s, false);
  if (e != cudaSuccess) return e;
  const dim3 grid(f.n_tokens, (l.mb / 2 + 255) / 256);
  return launch_pdl(front_finish_b_kernel<T>, grid, dim3(256), 0, s, f, static_cast<const float*>(part_b),
                    l.splits_b);
}

}  // namespace

size_t front_workspace_bytes(int32_t n_tokens, int32_t d_model, int32_t d_cq, int32_t heads, mla_dtype_t act) {
  return front_layout(n_tokens, d_model, d_cq, heads, act).total;
}

cudaError_t launch_front(const FrontArgs& f, cudaStream_t s) {
  if (f.n_tokens == 0) return cudaSuccess;
  if (f.act == MLA_F32) return launch_front_t<float>(f, s);
  return launch_front_t<__nv_bfloat16>(f, s);
}

}  // namespace mla
