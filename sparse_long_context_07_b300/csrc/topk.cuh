// Step 2: fine-grained top-k selection of each index-score row.
//
// "DeepSeek V3.2: How Far Can Open Models Go If You Actually Try?", §3.1: for
// each query t keep the k tokens with the highest I[t,:] ("Top-k operation" in
// the System Modules of "DeepSeek-V3.2: Pushing the Frontier of Open Large
// Language Models").  Ties go to the lower position; -0.0 == +0.0.
//
// One CTA per row.  Scores map to order-preserving 32-bit keys; three radix
// passes (11 + 11 + 10 bits, shared-memory histograms) find the exact k-th key
// T and how many keys equal to T are taken (the lowest positions).  A final
// ordered pass compacts the selection in ascending position with block scans.
// Rows with n <= k take every candidate.
#pragma once

#include <cstdint>

#include "common.cuh"

namespace dsa {
namespace topk {

constexpr int kThreads = 512;
constexpr int kBins = 2048;     // histogram bins (11-bit digits)
constexpr int kPerThread = 8;   // elements per thread per compaction chunk

// Monotone map float -> uint32 (larger float, larger key); -0 maps like +0.
__device__ __forceinline__ uint32_t order_key(float x) {
  uint32_t b = __float_as_uint(x);
  b = (b == 0x80000000u) ? 0u : b;
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__global__ void __launch_bounds__(kThreads) topk_kernel(
    const float* __restrict__ scores, int64_t ld, int k, int32_t* __restrict__ idx,
    float* __restrict__ vals, const int32_t* __restrict__ cu_q, const int32_t* __restrict__ cu_kv,
    int num_seqs, int64_t row0) {
  __shared__ uint32_t hist[kBins];
  __shared__ uint32_t warp_sums[32];
  __shared__ uint32_t s_digit, s_above;

  const int tid = threadIdx.x;
  const int64_t r = row0 + blockIdx.x;
  const RowGeom g = row_geom(cu_q, cu_kv, num_seqs, r);
  const int n = g.p + 1;
  // scores, idx and vals hold the rows of this launch, starting at row0
  const float* __restrict__ row = scores + (r - row0) * ld;
  int32_t* __restrict__ out_idx = idx + (r - row0) * static_cast<int64_t>(k);
  float* __restrict__ out_val = vals ? vals + (r - row0) * static_cast<int64_t>(k) : nullptr;

  if (n <= k) {  // every candidate is selected (uniform per block)
    for (int i = tid; i < k; i += kThreads) {
      out_idx[i] = i < n ? i : -1;
      if (out_val) out_val[i] = i < n ? row[i] : -__int_as_float(0x7f800000);
    }
    return;
  }

  // ---- radix select of the exact k-th largest key
  uint32_t prefix = 0, pmask = 0, kr = static_cast<uint32_t>(k);
  const int n4 = n >> 2;
  const float4* __restrict__ row4 = reinterpret_cast<const float4*>(row);
#pragma unroll 1
  for (int pass = 0; pass < 3; ++pass) {
    const int shift = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
    const uint32_t dmask = pass == 2 ? 0x3FFu : 0x7FFu;
    for (int i = tid; i < kBins; i += kThreads) hist[i] = 0;
    __syncthreads();
    auto add = [&](float x) {
      const uint32_t key = order_key(x);
      if ((key & pmask) == prefix) atomicAdd(&hist[(key >> shift) & dmask], 1u);
    };
    for (int i = tid; i < n4; i += kThreads) {
      const float4 v = __ldg(row4 + i);
      add(v.x); add(v.y); add(v.z); add(v.w);
    }
    for (int i = 4 * n4 + tid; i < n; i += kThreads) add(__ldg(row + i));
    __syncthreads();
    // thread t owns bins [4t, 4t+4); find the digit holding the kr-th largest
    uint32_t c[4], s = 0;
#pragma unroll
    for (int q = 0; q < 4; ++q) { c[q] = hist[4 * tid + q]; s += c[q]; }
    uint32_t total;
    const uint32_t incl = block_inclusive_scan<kThreads>(s, warp_sums, total);
    const uint32_t above = total - incl;  // keys in higher bins than mine
    if (above < kr && above + s >= kr) {
      uint32_t a = above;
#pragma unroll
      for (int q = 3; q >= 0; --q) {
        if (a + c[q] >= kr) { s_digit = 4 * tid + q; s_above = a; break; }
        a += c[q];
      }
    }
    __syncthreads();
    kr -= s_above;
    prefix |= s_digit << shift;
    pmask |= dmask << shift;
    __syncthreads();
  }
  const uint32_t T = prefix;  // exact k-th largest key; take kr of the keys == T

  // ---- ordered compaction: key > T, or key == T among the first kr such
  uint32_t base_sel = 0, base_eq = 0;
#pragma unroll 1
  for (int chunk = 0; chunk < n; chunk += kThreads * kPerThread) {
    const int i0 = chunk + kPerThread * tid;
    float v[kPerThread];
    if (i0 + kPerThread <= n) {
#pragma unroll
      for (int q = 0; q < kPerThread; q += 4) {
        const float4 t4 = __ldg(reinterpret_cast<const float4*>(row + i0 + q));
        v[q] = t4.x; v[q + 1] = t4.y; v[q + 2] = t4.z; v[q + 3] = t4.w;
      }
    } else {
#pragma unroll
      for (int q = 0; q < kPerThread; ++q) v[q] = (i0 + q < n) ? __ldg(row + i0 + q) : 0.f;
    }
    uint32_t gt_bits = 0, eq_bits = 0;
#pragma unroll
    for (int q = 0; q < kPerThread; ++q) {
      if (i0 + q < n) {
        const uint32_t key = order_key(v[q]);
        gt_bits |= (key > T ? 1u : 0u) << q;
        eq_bits |= (key == T ? 1u : 0u) << q;
      }
    }
    const uint32_t ne = __popc(eq_bits);
    uint32_t tot_eq;
    const uint32_t excl_eq = block_inclusive_scan<kThreads>(ne, warp_sums, tot_eq) - ne;
    uint32_t rank = base_eq + excl_eq, sel_bits = gt_bits;
#pragma unroll
    for (int q = 0; q < kPerThread; ++q) {
      if ((eq_bits >> q) & 1u) {
        if (rank < kr) sel_bits |= 1u << q;
        ++rank;
      }
    }
    const uint32_t ns = __popc(sel_bits);
    uint32_t tot_sel;
    uint32_t pos = base_sel + block_inclusive_scan<kThreads>(ns, warp_sums, tot_sel) - ns;
#pragma unroll
    for (int q = 0; q < kPerThread; ++q) {
      if (((sel_bits >> q) & 1u) && pos < static_cast<uint32_t>(k)) {
        out_idx[pos] = i0 + q;
        if (out_val) out_val[pos] = v[q];
        ++pos;
      }
    }
    base_sel += tot_sel;
    base_eq += tot_eq;
    if (base_sel >= static_cast<uint32_t>(k)) break;
  }
}

}  // namespace topk
}  // namespace dsa
