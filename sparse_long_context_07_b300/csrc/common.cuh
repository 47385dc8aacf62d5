// Batch geometry and small block-level helpers shared by the kernels.
#pragma once

#include <cstdint>

namespace dsa {

// Largest b in [0, num_seqs) with cu[b] <= r (the sequence holding query row
// r when r < cu[num_seqs]; empty sequences are skipped).
__device__ __forceinline__ int find_seq(const int32_t* __restrict__ cu, int num_seqs, int64_t r) {
  int lo = 0, hi = num_seqs - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (static_cast<int64_t>(__ldg(cu + mid)) <= r) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Geometry of query row r: sequence, position p (bottom-right aligned) and
// first global key row of the sequence.  Candidates are s = 0..p.
struct RowGeom {
  int b;
  int p;
  int64_t kv0;
};

__device__ __forceinline__ RowGeom row_geom(const int32_t* __restrict__ cu_q,
                                            const int32_t* __restrict__ cu_kv, int num_seqs,
                                            int64_t r) {
  RowGeom g;
  g.b = find_seq(cu_q, num_seqs, r);
  const int q0 = __ldg(cu_q + g.b), q1 = __ldg(cu_q + g.b + 1);
  const int k0 = __ldg(cu_kv + g.b), k1 = __ldg(cu_kv + g.b + 1);
  g.p = (k1 - k0) - (q1 - q0) + static_cast<int>(r - q0);
  g.kv0 = k0;
  return g;
}

// Monotone map of an fp32 score to a 32-bit key (larger score, larger key);
// -0 maps like +0.  Selection works on these keys; the top kRadixBits bits
// are the first radix digit (histogram bin) of a score.
__device__ __forceinline__ uint32_t order_key(float x) {
  uint32_t b = __float_as_uint(x);
  b = (b == 0x80000000u) ? 0u : b;
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
constexpr int kRadixBits = 11;
constexpr int kRadixBins = 1 << kRadixBits;          // 2048 bins of the first digit
constexpr int kRadixShift = 32 - kRadixBits;         // bin = order_key >> 21

// Block-wide inclusive scan (ascending thread order) of one value per thread.
// `warp_sums` is shared scratch of 32 words.  Every thread must call it.
template <int kThreads>
__device__ __forceinline__ uint32_t block_inclusive_scan(uint32_t v, uint32_t* warp_sums,
                                                         uint32_t& total) {
  constexpr int kWarps = kThreads / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t t = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += t;
  }
  if (lane == 31) warp_sums[warp] = v;
  __syncthreads();
  if (warp == 0) {
    uint32_t s = lane < kWarps ? warp_sums[lane] : 0u;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t t = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += t;
    }
    warp_sums[lane] = s;
  }
  __syncthreads();
  const uint32_t add = warp > 0 ? warp_sums[warp - 1] : 0u;
  total = warp_sums[kWarps - 1];
  __syncthreads();
  return v + add;
}

}  // namespace dsa
