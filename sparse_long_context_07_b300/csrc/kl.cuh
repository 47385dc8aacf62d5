// The lightning indexer's dense warm-up loss and its gradient (CUDA cores,
// fp32 arithmetic).
//
// "DeepSeek V3.2: How Far Can Open Models Go If You Actually Try?", §3.3
// (Stage 1, dense warm-up): the indexer learns where dense attention goes,
//   L_I = sum_t KL( p_t || softmax(I_t) ),
// with p_t the dense attention scores of token t aggregated over the heads
// and L1-normalised ("DeepSeek-V3.2: Pushing the Frontier of Open Large
// Language Models", Modeling, Objective Functions).  Read here as:
//   p_t[s] = (1/H) sum_h softmax_s(scale * Q[t,h] . kv[s])   over s = 0..p,
//   softmax(I_t) over the same candidates, 0 log 0 = 0,
// and the gradient taken with respect to the real-valued indexer inputs
// (q_I = code * q_scale, k_I = code * k_scale, and w), ReLU'(0) = 0:
//   g[t,s]     = softmax(I_t)_s - p_t[s]               (dL/dI[t,s])
//   x[t,j,s]   = q_I[t,j] . k_I[s]
//   dw[t,j]    = sum_s ReLU(x[t,j,s]) g[t,s]
//   dq_I[t,j]  = sum_s c[t,j,s] k_I[s],   c[t,j,s] = w[t,j] 1[x[t,j,s] > 0] g[t,s]
//   dk_I[s]    = sum_t sum_j c[t,j,s] q_I[t,j]
// The index scores themselves come from the forward indexer kernels.
#pragma once

#include <cstdint>

#include "common.cuh"
#include "simt.cuh"

namespace dsa {
namespace kl {

constexpr int kThreads = 256;
constexpr int kBwdThreads = 128;

__device__ __forceinline__ float block_max(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  float m = red[0];
  for (int w = 1; w < static_cast<int>(blockDim.x >> 5); ++w) m = fmaxf(m, red[w]);
  return m;
}

__device__ __forceinline__ float block_sum(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  float s = 0.f;
  for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) s += red[w];
  return s;
}

// grid (rows of the chunk), block kThreads.  P[i][s] = p_t[s] for the row
// r = row0 + i; Z[i] is scratch for one head's scores.
__global__ void __launch_bounds__(kThreads) target_kernel(
    const void* __restrict__ Q, const void* __restrict__ KV, int dtype, int H, int dqk, float scale,
    const int32_t* __restrict__ cu_q, const int32_t* __restrict__ cu_kv, int num_seqs, int64_t row0,
    float* __restrict__ P, float* __restrict__ Z, int64_t ld) {
  __shared__ float qh[simt::kMaxMlaDim];
  __shared__ float red[32];
  const int64_t r = row0 + blockIdx.x;
  const RowGeom g = row_geom(cu_q, cu_kv, num_seqs, r);
  const int n = g.p + 1;
  float* prow = P + blockIdx.x * ld;
  float* zrow = Z + blockIdx.x * ld;
  for (int s = threadIdx.x; s < n; s += kThreads) prow[s] = 0.f;
  const float inv_h = 1.f / static_cast<float>(H);
  for (int h = 0; h < H; ++h) {
    __syncthreads();
    for (int d = threadIdx.x; d < dqk; d += kThreads) qh[d] = simt::load_elem(Q, (r * H + h) * dqk + d, dtype);
    __syncthreads();
    float m = -INFINITY;
    for (int s = threadIdx.x; s < n; s += kThreads) {
      const int64_t base = (g.kv0 + s) * dqk;
      float z = 0.f;
      for (int d = 0; d < dqk; ++d) z = fmaf(qh[d], simt::load_elem(KV, base + d, dtype), z);
      z *= scale;
      zrow[s] = z;
      m = fmaxf(m, z);
    }
    m = block_max(m, red);
    float e = 0.f;
    for (int s = threadIdx.x; s < n; s += kThreads) e += expf(zrow[s] - m);
    const float lse = m + logf(block_sum(e, red));
    for (int s = threadIdx.x; s < n; s += kThreads) prow[s] += expf(zrow[s] - lse) * inv_h;
  }
}

// grid (rows of the chunk), block kThreads.  IG[i] holds I[r, 0..n) on entry
// and g[r, 0..n) on exit; loss_rows[r] = KL(p_r || softmax(I_r)).
__global__ void __launch_bounds__(kThreads) loss_kernel(
    float* __restrict__ IG, const float* __restrict__ P, int64_t ld, const int32_t* __restrict__ cu_q,
    const int32_t* __restrict__ cu_kv, int num_seqs, int64_t row0, float* __restrict__ loss_rows) {
  __shared__ float red[32];
  const int64_t r = row0 + blockIdx.x;
  const RowGeom g = row_geom(cu_q, cu_kv, num_seqs, r);
  const int n = g.p + 1;
  float* irow = IG + blockIdx.x * ld;
  const float* prow = P + blockIdx.x * ld;
  float m = -INFINITY;
  for (int s = threadIdx.x; s < n; s += kThreads) m = fmaxf(m, irow[s]);
  m = block_max(m, red);
  float e = 0.f;
  for (int s = threadIdx.x; s < n; s += kThreads) e += expf(irow[s] - m);
  const float log_z = m + logf(block_sum(e, red));
  float kl = 0.f;
  for (int s = threadIdx.x; s < n; s += kThreads) {
    const float p = prow[s], log_q = irow[s] - log_z;
    if (p > 0.f) kl += p * (logf(p) - log_q);
    irow[s] = expf(log_q) - p;
  }
  kl = block_sum(kl, red);
  if (threadIdx.x == 0) loss_rows[r] = kl;
}

// grid (ceil(max_kv / 128), rows of the chunk), block 128: thread = key s of
// row r.  C[i][j][s] = c[r,j,s]; dw[r][j] += sum over the block's keys of
// ReLU(x) g (dw is zero before the first chunk).
__global__ void __launch_bounds__(kBwdThreads) bwd_x_kernel(
    const void* __restrict__ q, const float* __restrict__ q_scale, const void* __restrict__ k,
    const float* __restrict__ k_scale, const float* __restrict__ w, int HI, int D, int dtype,
    const float* __restrict__ G, int64_t ld, const int32_t* __restrict__ cu_q, const int32_t* __restrict__ cu_kv,
    int num_seqs, int64_t row0, float* __restrict__ C, float* __restrict__ dw) {
  __shared__ float qs[simt::kMaxIdxHeads * simt::kMaxIdxDim];
  __shared__ float ws[simt::kMaxIdxHeads];
  const int64_t r = row0 + blockIdx.y;
  const RowGeom geo = row_geom(cu_q, cu_kv, num_seqs, r);
  const int n = geo.p + 1;
  if (static_cast<int>(blockIdx.x) * kBwdThreads >= n) return;  // uniform per block
  const float qsc = q_scale ? q_scale[r] : 1.f;
  for (int i = threadIdx.x; i < HI * D; i += kBwdThreads) qs[i] = simt::load_elem(q, r * HI * D + i, dtype) * qsc;
  for (int j = threadIdx.x; j < HI; j += kBwdThreads) ws[j] = w[r * HI + j];
  __syncthreads();
  const int s = blockIdx.x * kBwdThreads + threadIdx.x;
  const bool valid = s < n;
  const int64_t krow = geo.kv0 + (valid ? s : 0);
  const float ksc = (valid && k_scale) ? k_scale[krow] : 1.f;
  float kv[simt::kMaxIdxDim];
#pragma unroll
  for (int d = 0; d < simt::kMaxIdxDim; ++d) kv[d] = (valid && d < D) ? simt::load_elem(k, krow * D + d, dtype) * ksc : 0.f;
  const float gs = valid ? G[blockIdx.y * ld + s] : 0.f;
  const int lane = threadIdx.x & 31;
  for (int j = 0; j < HI; ++j) {
    float x = 0.f;
#pragma unroll
    for (int d = 0; d < simt::kMaxIdxDim; ++d)
      if (d < D) x = fmaf(qs[j * D + d], kv[d], x);
    const bool on = valid && x > 0.f;
    if (valid) C[(blockIdx.y * static_cast<int64_t>(HI) + j) * ld + s] = on ? ws[j] * gs : 0.f;
    float contrib = on ? x * gs : 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) contrib += __shfl_xor_sync(0xffffffffu, contrib, o);
    if (lane == 0 && contrib != 0.f) atomicAdd(dw + r * HI + j, contrib);
  }
}

// grid (rows of the chunk), block D: dq[r][j][d] = sum_s C[i][j][s] k_I[s][d].
__global__ void __launch_bounds__(kBwdThreads) bwd_dq_kernel(
    const float* __restrict__ C, const void* __restrict__ k, const float* __restrict__ k_scale, int HI, int D,
    int dtype, int64_t ld, const int32_t* __restrict__ cu_q, const int32_t* __restrict__ cu_kv, int num_seqs,
    int64_t row0, float* __restrict__ dq) {
  const int64_t r = row0 + blockIdx.x;
  const RowGeom geo = row_geom(cu_q, cu_kv, num_seqs, r);
  const int n = geo.p + 1;
  const int d = threadIdx.x;
  if (d >= D) return;
  for (int j = 0; j < HI; ++j) {
    const float* crow = C + (blockIdx.x * static_cast<int64_t>(HI) + j) * ld;
    float acc = 0.f;
    for (int s = 0; s < n; ++s) {
      const float c = crow[s];
      if (c != 0.f) {
        const int64_t krow = geo.kv0 + s;
        acc = fmaf(c, simt::load_elem(k, krow * D + d, dtype) * (k_scale ? k_scale[krow] : 1.f), acc);
      }
    }
    dq[(r * HI + j) * D + d] = acc;
  }
}

// grid (total_kv), block D: for key row `key` of sequence b at position s,
// dk[key][d] += sum over the chunk's rows t of b with p_t >= s of
// sum_j C[t - row0][j][s] q_I[t][j][d].  One block per key, so no atomics;
// chunks run in stream order.
__global__ void __launch_bounds__(kBwdThreads) bwd_dk_kernel(
    const float* __restrict__ C, const void* __restrict__ q, const float* __restrict__ q_scale, int HI, int D,
    int dtype, int64_t ld, const int32_t* __restrict__ cu_q, const int32_t* __restrict__ cu_kv, int num_seqs,
    int64_t row0, int64_t row1, float* __restrict__ dk) {
  const int64_t key = blockIdx.x;
  const int d = threadIdx.x;
  if (d >= D) return;
  const int b = find_seq(cu_kv, num_seqs, key);
  const int k0 = cu_kv[b], k1 = cu_kv[b + 1];
  if (key >= k1) return;   // past the last sequence (cannot happen for key < total_kv)
  const int s = static_cast<int>(key - k0);
  const int q0 = cu_q[b], q1 = cu_q[b + 1];
  // rows of b whose position nkv - nq + i reaches s
  int64_t t_lo = q0 + static_cast<int64_t>(s) - ((k1 - k0) - (q1 - q0));
  if (t_lo < q0) t_lo = q0;
  if (t_lo < row0) t_lo = row0;
  const int64_t t_hi = q1 < row1 ? q1 : row1;
  float acc = 0.f;
  for (int64_t t = t_lo; t < t_hi; ++t) {
    const float qsc = q_scale ? q_scale[t] : 1.f;
    const float* cbase = C + (t - row0) * static_cast<int64_t>(HI) * ld + s;
    for (int j = 0; j < HI; ++j) {
      const float c = cbase[j * ld];
      if (c != 0.f) acc = fmaf(c, simt::load_elem(q, (t * HI + j) * D + d, dtype) * qsc, acc);
    }
  }
  if (t_hi > t_lo) dk[key * D + d] += acc;
}

}  // namespace kl
}  // namespace dsa
