// CUDA-core kernels for the shapes the tensor-core kernels do not cover
// (small head counts and widths, fp32 inputs).  Same definitions:
//   indexer  I[t,s] = k_scale[s] * sum_j (w[t,j] q_scale[t]) ReLU(q[t,j] . k[s])
//            ("DeepSeek V3.2: How Far Can Open Models Go If You Actually Try?",
//            §3.1, with real inputs = code * per-row scale, positive scales)
//   attention softmax over the selected latent rows, V = first d_v columns of
//            the same row (same §3.1, MLA in MQA mode).
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "common.cuh"
#include "ptx.cuh"

namespace dsa {
namespace simt {

__device__ __forceinline__ float load_elem(const void* p, int64_t i, int dtype) {
  switch (dtype) {
    case DSA_DTYPE_E4M3: {
      const __nv_fp8_storage_t b = static_cast<const __nv_fp8_storage_t*>(p)[i];
      return __half2float(__half(__nv_cvt_fp8_to_halfraw(b, __NV_E4M3)));
    }
    case DSA_DTYPE_BF16:
      return __bfloat162float(static_cast<const __nv_bfloat16*>(p)[i]);
    default:
      return static_cast<const float*>(p)[i];
  }
}

constexpr int kIdxThreads = 128;
constexpr int kMaxIdxHeads = 64;
constexpr int kMaxIdxDim = 128;

// grid (ceil(max_kv / 128), rows); one thread per key s of row r.
__global__ void __launch_bounds__(kIdxThreads) indexer_kernel(
    const void* __restrict__ q, const float* __restrict__ q_scale, const void* __restrict__ k,
    const float* __restrict__ k_scale, const float* __restrict__ w, int H, int D, int dtype,
    float* __restrict__ scores, int64_t ld, const int32_t* __restrict__ cu_q,
    const int32_t* __restrict__ cu_kv, int num_seqs, int64_t row0) {
  __shared__ float qs[kMaxIdxHeads * kMaxIdxDim];
  __shared__ float ws[kMaxIdxHeads];
  const int64_t r = row0 + blockIdx.y;
  const RowGeom g = row_geom(cu_q, cu_kv, num_seqs, r);
  const int n = g.p + 1;
  if (static_cast<int>(blockIdx.x) * kIdxThreads >= n) return;  // uniform per block
  const float qsc = q_scale ? q_scale[r] : 1.f;
  for (int i = threadIdx.x; i < H * D; i += kIdxThreads) qs[i] = load_elem(q, r * H * D + i, dtype);
  for (int j = threadIdx.x; j < H; j += kIdxThreads) ws[j] = w[r * H + j] * qsc;
  __syncthreads();
  const int s = blockIdx.x * kIdxThreads + threadIdx.x;
  if (s >= n) return;
  const int64_t krow = g.kv0 + s;
  float kv[kMaxIdxDim];
#pragma unroll
  for (int d = 0; d < kMaxIdxDim; ++d) kv[d] = d < D ? load_elem(k, krow * D + d, dtype) : 0.f;
  float acc = 0.f;
  for (int j = 0; j < H; ++j) {
    float x = 0.f;
#pragma unroll
    for (int d = 0; d < kMaxIdxDim; ++d)
      if (d < D) x = fmaf(qs[j * D + d], kv[d], x);
    acc = fmaf(ws[j], fmaxf(x, 0.f), acc);
  }
  scores[(r - row0) * ld + s] = acc * (k_scale ? k_scale[krow] : 1.f);  // rows relative to row0
}

constexpr int kMlaWarps = 4;
constexpr int kMaxMlaDim = 1024;
constexpr int kMaxPerLane = kMaxMlaDim / 32;

// grid (rows); each warp handles heads warp, warp + 4, ...  Online softmax over
// the selected rows in index order.
__global__ void __launch_bounds__(kMlaWarps * 32) mla_kernel(
    const void* __restrict__ Q, const void* __restrict__ KV, const int32_t* __restrict__ idx, int k,
    int H, int d_qk, int d_v, float scale, int dtype, void* __restrict__ out,
    float* __restrict__ lse, const int32_t* __restrict__ cu_q, const int32_t* __restrict__ cu_kv,
    int num_seqs, int64_t row0) {
  const int64_t r = row0 + blockIdx.x;
  const RowGeom g = row_geom(cu_q, cu_kv, num_seqs, r);
  const int n = g.p + 1;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  // idx, out and lse hold the rows of this launch, starting at row0
  const int64_t rr = r - row0;
  const int32_t* __restrict__ sel = idx + rr * static_cast<int64_t>(k);
  for (int h = warp; h < H; h += kMlaWarps) {
    float qv[kMaxPerLane], o[kMaxPerLane];
#pragma unroll
    for (int i = 0; i < kMaxPerLane; ++i) {
      const int d = lane + 32 * i;
      qv[i] = d < d_qk ? load_elem(Q, (r * H + h) * d_qk + d, dtype) : 0.f;
      o[i] = 0.f;
    }
    float m = -INFINITY, l = 0.f;
    for (int i = 0; i < k; ++i) {
      const int s = __ldg(sel + i);
      if (s == -1) continue;
      if (s < -1 || s >= n) {
        if (lane == 0 && h == warp) flag_error(DSA_DEVERR_BAD_INDEX);
        continue;
      }
      const int64_t row = g.kv0 + s;
      float z = 0.f;
#pragma unroll
      for (int j = 0; j < kMaxPerLane; ++j) {
        const int d = lane + 32 * j;
        if (d < d_qk) z = fmaf(qv[j], load_elem(KV, row * d_qk + d, dtype), z);
      }
#pragma unroll
      for (int o2 = 16; o2 > 0; o2 >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o2);
      z *= scale;
      const float m_new = fmaxf(m, z);
      const float corr = __expf(m - m_new);
      const float p = __expf(z - m_new);
      l = l * corr + p;
#pragma unroll
      for (int j = 0; j < kMaxPerLane; ++j) {
        const int d = lane + 32 * j;
        if (d < d_v) o[j] = o[j] * corr + p * load_elem(KV, row * d_qk + d, dtype);
      }
      m = m_new;
    }
    const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
    for (int j = 0; j < kMaxPerLane; ++j) {
      const int d = lane + 32 * j;
      if (d < d_v) {
        const int64_t oi = (rr * H + h) * d_v + d;
        if (dtype == DSA_DTYPE_BF16)
          static_cast<__nv_bfloat16*>(out)[oi] = __float2bfloat16_rn(o[j] * inv);
        else
          static_cast<float*>(out)[oi] = o[j] * inv;
      }
    }
    if (lse && lane == 0) lse[rr * H + h] = l > 0.f ? m + logf(l) : -INFINITY;
  }
}

}  // namespace simt
}  // namespace dsa
