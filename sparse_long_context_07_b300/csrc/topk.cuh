// Step 2: fine-grained top-k selection of each index-score row.
//
// "DeepSeek V3.2: How Far Can Open Models Go If You Actually Try?", §3.1: for
// each query t keep the k tokens with the highest I[t,:] ("Top-k operation" in
// the System Modules of "DeepSeek-V3.2: Pushing the Frontier of Open Large
// Language Models").  Ties go to the lower position; -0.0 == +0.0.
//
// topk_kernel: one CTA per row (topk_cluster_kernel below serves batches of
// few rows).  Scores map to order-preserving 32-bit keys.
//   pass 1 (row read once): histogram of the top 11 key bits; the bin b* that
//            holds the k-th largest key and the count above it follow from a
//            block scan.
//   pass 2 (row read again): keys in bins above b* are selected outright (one
//            bit each in a shared-memory bitmap of positions); keys in b* are
//            kept as candidates (low 21 bits, position) in shared memory.
//   The candidates are narrowed by two more radix passes in shared memory to
//   the exact k-th key; the larger ones join the bitmap, the equal ones go to
//   a tie bitmap of which the lowest positions are taken.  Scanning the
//   bitmaps in position order writes the selection in ascending order.
// Rows longer than the bitmaps or whose boundary bin overflows the candidate
// store (heavy ties) take the general path: three radix passes over the row
// for the exact k-th key, then an ordered compaction with block scans.
// Rows with n <= k take every candidate.
#pragma once

#include <cstdint>

#include "common.cuh"
#include "ptx.cuh"

namespace dsa {
namespace topk {

constexpr int kThreads = 512;
constexpr int kBins = kRadixBins;   // histogram bins (11-bit digits)
constexpr int kPerThread = 8;   // elements per thread per compaction chunk
constexpr int kMaxFastN = 131072;                 // positions covered by the bitmaps
constexpr int kBitmapWords = kMaxFastN / 32;
constexpr int kWordsPerThread = kBitmapWords / kThreads;
constexpr int kCandCap = 4096;                    // boundary-bin candidates held in smem

struct Smem {
  uint32_t hist[kBins];
  uint32_t sel[kBitmapWords];    // selected positions
  uint32_t tie[kBitmapWords];    // positions whose key equals the k-th key
  uint32_t cand_key[kCandCap];   // low 21 key bits of the boundary-bin keys
  int32_t cand_idx[kCandCap];
  uint32_t warp_sums[32];
  uint32_t s_digit, s_above, ncand;
};
constexpr int kSmemBytes = static_cast<int>(sizeof(Smem));


// The digit (bin index) holding the kr-th largest key of `hist` (nbins bins,
// thread t owns bins [4t, 4t+4)), and the number of keys in higher bins.
__device__ __forceinline__ void find_digit(const uint32_t* hist, int nbins, uint32_t kr, Smem& sm) {
  const int tid = threadIdx.x;
  uint32_t c[4], s = 0;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    c[q] = (4 * tid + q < nbins) ? hist[4 * tid + q] : 0u;
    s += c[q];
  }
  uint32_t total;
  const uint32_t incl = block_inclusive_scan<kThreads>(s, sm.warp_sums, total);
  const uint32_t above = total - incl;  // keys in higher bins than mine
  if (above < kr && above + s >= kr) {
    uint32_t a = above;
#pragma unroll
    for (int q = 3; q >= 0; --q) {
      if (a + c[q] >= kr) { sm.s_digit = 4 * tid + q; sm.s_above = a; break; }
      a += c[q];
    }
  }
  __syncthreads();
}

// General path: exact k-th key by three radix passes over the row, then an
// ordered compaction with block scans.
__device__ void select_general(const float* __restrict__ row, int n, int k, int32_t* __restrict__ out_idx,
                               float* __restrict__ out_val, Smem& sm) {
  const int tid = threadIdx.x;
  uint32_t prefix = 0, pmask = 0, kr = static_cast<uint32_t>(k);
  const int n4 = n >> 2;
  const float4* __restrict__ row4 = reinterpret_cast<const float4*>(row);
#pragma unroll 1
  for (int pass = 0; pass < 3; ++pass) {
    const int shift = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
    const uint32_t dmask = pass == 2 ? 0x3FFu : 0x7FFu;
    for (int i = tid; i < kBins; i += kThreads) sm.hist[i] = 0;
    __syncthreads();
    auto add = [&](float x) {
      const uint32_t key = order_key(x);
      if ((key & pmask) == prefix) atomicAdd(&sm.hist[(key >> shift) & dmask], 1u);
    };
    for (int i = tid; i < n4; i += kThreads) {
      const float4 v = __ldg(row4 + i);
      add(v.x); add(v.y); add(v.z); add(v.w);
    }
    for (int i = 4 * n4 + tid; i < n; i += kThreads) add(__ldg(row + i));
    __syncthreads();
    find_digit(sm.hist, kBins, kr, sm);
    kr -= sm.s_above;
    prefix |= sm.s_digit << shift;
    pmask |= dmask << shift;
    __syncthreads();
  }
  const uint32_t T = prefix;  // exact k-th largest key; take kr of the keys == T

  // ordered compaction: key > T, or key == T among the first kr such
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
    const uint32_t excl_eq = block_inclusive_scan<kThreads>(ne, sm.warp_sums, tot_eq) - ne;
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
    uint32_t pos = base_sel + block_inclusive_scan<kThreads>(ns, sm.warp_sums, tot_sel) - ns;
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

__global__ void __launch_bounds__(kThreads) topk_kernel(
    const float* __restrict__ scores, int64_t ld, int k, int32_t* __restrict__ idx,
    float* __restrict__ vals, const int32_t* __restrict__ cu_q, const int32_t* __restrict__ cu_kv,
    int num_seqs, int64_t row0, const uint32_t* __restrict__ hist_in) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>(smem_raw);
  griddep_launch_dependents();   // the attention kernel may set up while rows are selected

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

  const int n4 = n >> 2;
  const float4* __restrict__ row4 = reinterpret_cast<const float4*>(row);
  int i4 = tid;
  if (hist_in) {
    // the indexer built this row's histogram of the top 11 key bits
    const uint32_t* h = hist_in + (r - row0) * kBins;
    for (int i = tid; i < kBins; i += kThreads) sm.hist[i] = __ldg(h + i);
    __syncthreads();
  } else {
  // ---- pass 1: histogram of the top 11 key bits
  for (int i = tid; i < kBins; i += kThreads) sm.hist[i] = 0;
  __syncthreads();
  // four 16-byte loads in flight per thread
  for (; i4 + 3 * kThreads < n4; i4 += 4 * kThreads) {
    float4 v[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) v[q] = __ldg(row4 + i4 + q * kThreads);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      atomicAdd(&sm.hist[order_key(v[q].x) >> 21], 1u);
      atomicAdd(&sm.hist[order_key(v[q].y) >> 21], 1u);
      atomicAdd(&sm.hist[order_key(v[q].z) >> 21], 1u);
      atomicAdd(&sm.hist[order_key(v[q].w) >> 21], 1u);
    }
  }
  for (; i4 < n4; i4 += kThreads) {
    const float4 v = __ldg(row4 + i4);
    atomicAdd(&sm.hist[order_key(v.x) >> 21], 1u);
    atomicAdd(&sm.hist[order_key(v.y) >> 21], 1u);
    atomicAdd(&sm.hist[order_key(v.z) >> 21], 1u);
    atomicAdd(&sm.hist[order_key(v.w) >> 21], 1u);
  }
  for (int i = 4 * n4 + tid; i < n; i += kThreads) atomicAdd(&sm.hist[order_key(__ldg(row + i)) >> 21], 1u);
  __syncthreads();
  }
  find_digit(sm.hist, kBins, static_cast<uint32_t>(k), sm);
  const uint32_t bstar = sm.s_digit;
  const uint32_t kr = static_cast<uint32_t>(k) - sm.s_above;   // keys to take from bin b*
  const uint32_t cstar = sm.hist[bstar];
  if (n > kMaxFastN || cstar > static_cast<uint32_t>(kCandCap)) {   // uniform per block
    __syncthreads();
    select_general(row, n, k, out_idx, out_val, sm);
    return;
  }

  // ---- pass 2: bins above b* are selected, bin b* keeps candidates
  const int nwords = (n + 31) >> 5;
  for (int i = tid; i < nwords; i += kThreads) { sm.sel[i] = 0u; sm.tie[i] = 0u; }
  if (tid == 0) sm.ncand = 0u;
  __syncthreads();
  auto classify = [&](float x, int i) {
    const uint32_t key = order_key(x);
    const uint32_t d = key >> 21;
    if (d > bstar) {
      atomicOr(&sm.sel[i >> 5], 1u << (i & 31));
    } else if (d == bstar) {
      const uint32_t slot = atomicAdd(&sm.ncand, 1u);
      sm.cand_key[slot] = key & 0x1FFFFFu;
      sm.cand_idx[slot] = i;
    }
  };
  i4 = tid;
  for (; i4 + 3 * kThreads < n4; i4 += 4 * kThreads) {
    float4 v[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) v[q] = __ldg(row4 + i4 + q * kThreads);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int i = i4 + q * kThreads;
      classify(v[q].x, 4 * i); classify(v[q].y, 4 * i + 1); classify(v[q].z, 4 * i + 2); classify(v[q].w, 4 * i + 3);
    }
  }
  for (; i4 < n4; i4 += kThreads) {
    const float4 v = __ldg(row4 + i4);
    classify(v.x, 4 * i4); classify(v.y, 4 * i4 + 1); classify(v.z, 4 * i4 + 2); classify(v.w, 4 * i4 + 3);
  }
  for (int i = 4 * n4 + tid; i < n; i += kThreads) classify(__ldg(row + i), i);
  __syncthreads();

  // ---- the kr-th largest low-21-bit value among the candidates (two radix
  // passes in shared memory: bits 20..10, then 9..0)
  uint32_t prefix = 0, pmask = 0, krr = kr;
#pragma unroll 1
  for (int pass = 0; pass < 2; ++pass) {
    const int shift = pass == 0 ? 10 : 0;
    const uint32_t dmask = pass == 0 ? 0x7FFu : 0x3FFu;
    for (int i = tid; i < kBins; i += kThreads) sm.hist[i] = 0;
    __syncthreads();
    for (uint32_t c = tid; c < cstar; c += kThreads) {
      const uint32_t lk = sm.cand_key[c];
      if ((lk & pmask) == prefix) atomicAdd(&sm.hist[(lk >> shift) & dmask], 1u);
    }
    __syncthreads();
    find_digit(sm.hist, pass == 0 ? kBins : 1024, krr, sm);
    krr -= sm.s_above;
    prefix |= sm.s_digit << shift;
    pmask |= dmask << shift;
    __syncthreads();
  }
  const uint32_t T21 = prefix;   // candidates above it are selected; take krr of the equal ones
  for (uint32_t c = tid; c < cstar; c += kThreads) {
    const uint32_t lk = sm.cand_key[c];
    const int i = sm.cand_idx[c];
    if (lk > T21) atomicOr(&sm.sel[i >> 5], 1u << (i & 31));
    else if (lk == T21) atomicOr(&sm.tie[i >> 5], 1u << (i & 31));
  }
  __syncthreads();

  // ---- ordered emission: thread t scans bitmap words [wpt t, wpt t + wpt),
  // the row's words spread over all threads
  const int wpt = (nwords + kThreads - 1) / kThreads;   // at most kWordsPerThread
  const int w0 = tid * wpt;
  uint32_t sel_cnt = 0, tie_cnt = 0;
#pragma unroll 1
  for (int q = 0; q < wpt; ++q) {
    if (w0 + q < nwords) {
      sel_cnt += __popc(sm.sel[w0 + q]);
      tie_cnt += __popc(sm.tie[w0 + q]);
    }
  }
  uint32_t tot;
  const uint32_t tie_before = block_inclusive_scan<kThreads>(tie_cnt, sm.warp_sums, tot) - tie_cnt;
  uint32_t take = tie_before >= krr ? 0u : min(krr - tie_before, tie_cnt);
  const uint32_t out_cnt = sel_cnt + take;
  uint32_t pos = block_inclusive_scan<kThreads>(out_cnt, sm.warp_sums, tot) - out_cnt;
#pragma unroll 1
  for (int q = 0; q < wpt; ++q) {
    const int w = w0 + q;
    if (w >= nwords) break;
    uint32_t bits = sm.sel[w];
    uint32_t tb = sm.tie[w];
    while (take > 0u && tb != 0u) {   // the lowest positions of the ties
      bits |= tb & (0u - tb);
      tb &= tb - 1u;
      --take;
    }
    while (bits != 0u) {
      const int b = __ffs(bits) - 1;
      bits &= bits - 1u;
      const int i = 32 * w + b;
      if (pos < static_cast<uint32_t>(k)) {
        out_idx[pos] = i;
        if (out_val) out_val[pos] = __ldg(row + i);
      }
      ++pos;
    }
  }
}

// ----------------------------------------------------------------------------
// Few long rows (decode): a cluster of kCluster CTAs per row.
//
// CTA c of a row's cluster owns the contiguous slice [c S, c S + S) of the
// candidates (S a multiple of 32).
//   pass 0 (slice read from memory): histogram of the top 11 key bits.
//            Every CTA adds its non-empty bins into every CTA's copy of the
//            row histogram (remote reductions in distributed shared memory),
//            so after one cluster barrier each CTA finds the same bin b*
//            that holds the k-th largest key.
//   stage:   a second read of the slice writes the bitmap words of its keys
//            above b* and in b*, and keeps the low 21 bits of its keys in b*
//            per warp in shared memory.
//   refine:  two radix passes (bits 20..10, 9..0) over the kept keys, their
//            histograms reduced across the cluster, give every CTA the exact
//            k-th key T.
//   emit:    each CTA compares its keys in b* with T (reloading only those),
//            the CTAs swap their counts of keys above and equal to T, and
//            each writes its selection in ascending position order (ties go
//            to the lowest positions).
// When a warp meets more keys of b* than it keeps (heavy ties), or the slices
// exceed the bitmaps, the exact key follows instead from two more radix
// passes over the slices.  Same result as topk_kernel, bit for bit.
// ----------------------------------------------------------------------------
constexpr int kCluster = 8;
constexpr int kCThreads = 256;
constexpr int kSliceBits = 16384;    // slice positions covered by the bitmaps
constexpr int kStagePerWarp = 2 * kRadixBins / (kCThreads / 32);   // staged keys per warp (in hist, ghist)
static_assert(kBins == kCluster * kCThreads, "one histogram bin per thread in the cluster reduction");

struct CSmem {
  uint32_t hg[2 * kBins];          // this CTA's histogram of a pass, then the row's (the
                                   // stage pass later keeps the keys in b* in both)
  uint32_t sel[kSliceBits / 32];   // slice positions above T
  uint32_t tie[kSliceBits / 32];   // slice positions equal to T
  uint32_t scratch[4 * kBins];     // pass 0: four sub-histograms; later the histograms of
                                   // the refining passes
  uint32_t warp_sums[32];
  uint32_t cnt[2 * kCluster];      // (selected, tied) keys of every CTA
  uint32_t wcnt[kCThreads / 32];   // keys in b* staged per warp
  uint32_t wovf[kCThreads / 32];   // a warp met more keys in b* than it stages
  uint32_t ovf[kCluster];          // the same, per CTA of the cluster
  uint32_t s_digit, s_above;
};
constexpr int kCSmemBytes = static_cast<int>(sizeof(CSmem));

__device__ __forceinline__ uint32_t ld_cluster_u32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ void st_cluster_u32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ void red_cluster_add_u32(uint32_t addr, uint32_t v) {
  asm volatile("red.relaxed.cluster.shared::cluster.add.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ void cluster_arrive_release() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_acquire() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// The digit holding the kr-th largest key of hist (nbins <= 2048 bins;
// thread t owns bins [8t, 8t + 8)) and the number of keys in higher bins.
__device__ __forceinline__ void find_digit_c(const uint32_t* hist, int nbins, uint32_t kr, CSmem& sm) {
  const int tid = threadIdx.x;
  uint32_t c[8], s = 0;
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    c[q] = (8 * tid + q < nbins) ? hist[8 * tid + q] : 0u;
    s += c[q];
  }
  uint32_t total;
  const uint32_t incl = block_inclusive_scan<kCThreads>(s, sm.warp_sums, total);
  const uint32_t above = total - incl;
  if (above < kr && above + s >= kr) {
    uint32_t a = above;
#pragma unroll
    for (int q = 7; q >= 0; --q) {
      if (a + c[q] >= kr) { sm.s_digit = 8 * tid + q; sm.s_above = a; break; }
      a += c[q];
    }
  }
  __syncthreads();
}

// Calls f(i, key) for every position i < len of the slice, each warp taking
// 128 consecutive positions per step (one float4 per lane, eight steps'
// loads in flight); positions past len are passed with valid = false, so the
// calls of a warp stay uniform (f may use warp votes).
template <typename F>
__device__ __forceinline__ void for_slice(const float* __restrict__ slice, int len, F&& f) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  constexpr int kWarps = kCThreads / 32;
  constexpr int kDepth = 8;
  const float4* __restrict__ s4 = reinterpret_cast<const float4*>(slice);
  const int n4 = (len + 3) >> 2;   // float4 steps covering the slice
  for (int b = warp * 32; b < n4; b += kWarps * 32 * kDepth) {
    float4 v[kDepth];
#pragma unroll
    for (int q = 0; q < kDepth; ++q) {
      const int i4 = b + q * kWarps * 32 + lane;
      if (4 * i4 + 3 < len) {
        v[q] = __ldg(s4 + i4);
      } else {
        const int i = 4 * i4;
        v[q].x = i < len ? __ldg(slice + i) : 0.f;
        v[q].y = i + 1 < len ? __ldg(slice + i + 1) : 0.f;
        v[q].z = i + 2 < len ? __ldg(slice + i + 2) : 0.f;
        v[q].w = 0.f;   // i + 3 >= len here
      }
    }
#pragma unroll
    for (int q = 0; q < kDepth; ++q) {
      const int base = b + q * kWarps * 32;
      if (base < n4) {   // uniform per warp
        const int i = 4 * (base + lane);
        f(i, order_key(v[q].x), i < len);
        f(i + 1, order_key(v[q].y), i + 1 < len);
        f(i + 2, order_key(v[q].z), i + 2 < len);
        f(i + 3, order_key(v[q].w), i + 3 < len);
      }
    }
  }
}

__global__ void __cluster_dims__(kCluster, 1, 1) __launch_bounds__(kCThreads, 4) topk_cluster_kernel(
    const float* __restrict__ scores, int64_t ld, int k, int32_t* __restrict__ idx,
    float* __restrict__ vals, const int32_t* __restrict__ cu_q, const int32_t* __restrict__ cu_kv,
    int num_seqs, int64_t row0, const uint32_t* __restrict__ hist_in) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  CSmem& sm = *reinterpret_cast<CSmem*>(smem_raw);
  griddep_launch_dependents();   // the attention kernel may set up while rows are selected

  const int tid = threadIdx.x, lane = tid & 31;
  const int c = static_cast<int>(cluster_ctarank());
  const int64_t rl = blockIdx.x / kCluster;   // row within this launch
  const int64_t r = row0 + rl;
  const RowGeom g = row_geom(cu_q, cu_kv, num_seqs, r);
  const int n = g.p + 1;
  const float* __restrict__ row = scores + rl * ld;
  int32_t* __restrict__ out_idx = idx + rl * static_cast<int64_t>(k);
  float* __restrict__ out_val = vals ? vals + rl * static_cast<int64_t>(k) : nullptr;

  if (n <= k) {  // every candidate is selected (uniform per cluster: no barrier is reached)
    for (int i = c * kCThreads + tid; i < k; i += kCluster * kCThreads) {
      out_idx[i] = i < n ? i : -1;
      if (out_val) out_val[i] = i < n ? row[i] : -__int_as_float(0x7f800000);
    }
    return;
  }

  const int S = ((n + 32 * kCluster - 1) / (32 * kCluster)) * 32;
  const int lo = c * S;
  const int len = max(0, min(n, lo + S) - lo);
  const bool bitmapped = S <= kSliceBits;   // uniform per cluster
  const float* __restrict__ slice = row + lo;
  uint32_t* const hist = sm.hg;            // this CTA's histogram
  uint32_t* const ghist = sm.hg + kBins;   // the row's histogram
  const uint32_t hist_base = smem_u32(hist), ghist_base = smem_u32(ghist);

  // ---- pass 0: the row histogram of the top 11 key bits
  if (hist_in) {
    // the indexer built it (the choice is uniform per cluster, so no CTA
    // skips a cluster barrier that the others reach)
    const uint32_t* h = hist_in + rl * kBins;
    for (int i = tid; i < kBins; i += kCThreads) ghist[i] = __ldg(h + i);
  } else {
    for (int i = tid; i < kBins; i += kCThreads) ghist[i] = 0u;
    for (int i = tid; i < 4 * kBins; i += kCThreads) sm.scratch[i] = 0u;
  }
  for (int i = tid; i < kSliceBits / 32; i += kCThreads) { sm.sel[i] = 0u; sm.tie[i] = 0u; }
  __syncthreads();
  cluster_arrive_release();   // this CTA's row histogram copy is zeroed
  if (!hist_in) {
    // four sub-histograms (lane % 4): most keys fall into a few bins, and
    // fewer lanes then hit the same counter
    uint32_t* sub = sm.scratch + (lane & 3) * kBins;
    for_slice(slice, len, [&](int, uint32_t key, bool valid) {
      if (valid) atomicAdd(&sub[key >> 21], 1u);
    });
    __syncthreads();
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int b = 8 * tid + q;
      hist[b] = sm.scratch[b] + sm.scratch[kBins + b] + sm.scratch[2 * kBins + b] + sm.scratch[3 * kBins + b];
    }
    __syncthreads();
  }
  cluster_wait_acquire();     // every CTA's copy is zeroed
  if (!hist_in) {
    // add the non-empty bins of this slice into every CTA's row histogram
#pragma unroll 1
    for (int q = 0; q < 8; ++q) {
      const int b = 8 * tid + q;
      const uint32_t v = hist[b];
      if (v != 0u) {
#pragma unroll
        for (int d = 0; d < kCluster; ++d) red_cluster_add_u32(mapa_shared(ghist_base + 4u * b, d), v);
      }
    }
  }
  cluster_sync();   // every CTA holds the row histogram
  find_digit_c(ghist, kBins, static_cast<uint32_t>(k), sm);
  const uint32_t bstar = sm.s_digit;
  uint32_t kr = static_cast<uint32_t>(k) - sm.s_above;   // keys to take from bin b*
  // staging needs the slice bitmaps (uniform per cluster)
  const bool try_stage = bitmapped;
  bool fallback = !try_stage;
  uint32_t T = 0, kr_here = 0, out_base = 0;
  // ties go to the lowest positions: the CTAs before this one take theirs
  // first (counts swapped through distributed shared memory)
  auto exchange_counts = [&](uint32_t sel_cnt, uint32_t tie_cnt) {
    uint32_t tot_sel, tot_tie;
    block_inclusive_scan<kCThreads>(sel_cnt, sm.warp_sums, tot_sel);
    block_inclusive_scan<kCThreads>(tie_cnt, sm.warp_sums, tot_tie);
    if (tid < kCluster) {
      const uint32_t base = smem_u32(sm.cnt);
      st_cluster_u32(mapa_shared(base + 8u * c, tid), tot_sel);
      st_cluster_u32(mapa_shared(base + 8u * c + 4u, tid), tot_tie);
    }
    cluster_sync();   // every CTA holds all counts; no shared memory is read remotely after this
    uint32_t ties_before = 0;
    for (int q = 0; q < c; ++q) {
      const uint32_t tq = sm.cnt[2 * q + 1];
      const uint32_t take_q = ties_before >= kr ? 0u : min(kr - ties_before, tq);
      out_base += sm.cnt[2 * q] + take_q;
      ties_before += tq;
    }
    kr_here = ties_before >= kr ? 0u : kr - ties_before;   // ties this CTA may take
  };
  if (try_stage) {
    __syncthreads();   // every thread has read the row histogram (the staging overwrites it)
    // ---- stage pass (the slice read once more): the bitmap words of the
    // keys above b* (sel) and in b* (tie, for now), and the low 21 bits of
    // the keys in b*, staged per warp in the histogram arrays (free now)
    const int warp = tid >> 5;
    const uint32_t lt_mask = (1u << lane) - 1u;
    uint32_t wc = 0;
    {
      constexpr int kWarps = kCThreads / 32;
      constexpr int kDepth = 4;
      const float4* __restrict__ s4 = reinterpret_cast<const float4*>(slice);
      const int n4 = (len + 3) >> 2;
      const int nw = (len + 31) >> 5;
      uint32_t* wst = sm.hg + warp * kStagePerWarp;
      for (int b0 = warp * 32; b0 < n4; b0 += kWarps * 32 * kDepth) {
        float4 v[kDepth];
#pragma unroll
        for (int q = 0; q < kDepth; ++q) {
          const int i4 = b0 + q * kWarps * 32 + lane;
          if (4 * i4 + 3 < len) {
            v[q] = __ldg(s4 + i4);
          } else {
            const int i = 4 * i4;
            v[q].x = i < len ? __ldg(slice + i) : 0.f;
            v[q].y = i + 1 < len ? __ldg(slice + i + 1) : 0.f;
            v[q].z = i + 2 < len ? __ldg(slice + i + 2) : 0.f;
            v[q].w = 0.f;   // i + 3 >= len here
          }
        }
#pragma unroll
        for (int q = 0; q < kDepth; ++q) {
          const int b = b0 + q * kWarps * 32;
          if (b >= n4) break;   // uniform per warp
          const int i0 = 4 * (b + lane);
          const float xs[4] = {v[q].x, v[q].y, v[q].z, v[q].w};
          uint32_t ma = 0u, mc = 0u;
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const uint32_t key = order_key(xs[e]);
            const uint32_t d = key >> 21;
            const bool valid = i0 + e < len;
            const bool cand = valid && d == bstar;
            ma |= (valid && d > bstar ? 1u : 0u) << e;
            mc |= (cand ? 1u : 0u) << e;
            const uint32_t bal = __ballot_sync(0xffffffffu, cand);
            const uint32_t slot = wc + static_cast<uint32_t>(__popc(bal & lt_mask));
            if (cand && slot < static_cast<uint32_t>(kStagePerWarp))
              wst[slot] = (static_cast<uint32_t>(c) << 21) | (key & 0x1FFFFFu);
            wc += static_cast<uint32_t>(__popc(bal));
          }
          // lanes 8 g .. 8 g + 7 hold the 32 positions of bitmap word b / 8 + g
          uint32_t ws = ma << (4 * (lane & 7)), wt = mc << (4 * (lane & 7));
#pragma unroll
          for (int o = 1; o < 8; o <<= 1) {
            ws |= __shfl_xor_sync(0xffffffffu, ws, o);
            wt |= __shfl_xor_sync(0xffffffffu, wt, o);
          }
          const int w = (b >> 3) + (lane >> 3);
          if ((lane & 7) == 0 && w < nw) { sm.sel[w] = ws; sm.tie[w] = wt; }
        }
      }
    }
    // ---- the exact k-th key: two more radix passes over the keys staged
    // in every CTA, the histograms reduced through distributed shared memory
    uint32_t* const h2 = sm.scratch;           // this CTA's histogram
    uint32_t* const g2 = sm.scratch + kBins;   // the row's histogram
    const uint32_t h2_base = smem_u32(h2), g2_base = smem_u32(g2);
    if (lane == 0) {
      sm.wcnt[warp] = min(wc, static_cast<uint32_t>(kStagePerWarp));
      sm.wovf[warp] = wc > static_cast<uint32_t>(kStagePerWarp) ? 1u : 0u;
    }
    for (int i = tid; i < kBins; i += kCThreads) h2[i] = 0u;
    __syncthreads();
    uint32_t ovf_here = 0;
    for (int w = 0; w < kCThreads / 32; ++w) ovf_here |= sm.wovf[w];
    uint32_t prefix = 0, pmask = 0;   // over the low 21 bits
#pragma unroll 1
    for (int pass = 0; pass < 2; ++pass) {
      const int shift = pass == 0 ? 10 : 0;
      const uint32_t dmask = pass == 0 ? 0x7FFu : 0x3FFu;
      if (pass == 1) {
        // every CTA has read this CTA's histogram of the first pass
        for (int i = tid; i < kBins; i += kCThreads) h2[i] = 0u;
        __syncthreads();
      }
      for (int w = 0; w < kCThreads / 32; ++w) {
        const uint32_t nr = sm.wcnt[w];
        for (uint32_t j = tid; j < nr; j += kCThreads) {
          const uint32_t lk = sm.hg[w * kStagePerWarp + j] & 0x1FFFFFu;
          if ((lk & pmask) == prefix) atomicAdd(&h2[(lk >> shift) & dmask], 1u);
        }
      }
      __syncthreads();
      if (pass == 0 && tid < kCluster) st_cluster_u32(mapa_shared(smem_u32(&sm.ovf[c]), tid), ovf_here);
      cluster_sync();   // every CTA's histogram (and overflow flag) is complete
      if (pass == 0) {
        uint32_t any = 0;
#pragma unroll
        for (int q = 0; q < kCluster; ++q) any |= sm.ovf[q];
        fallback = any != 0u;   // uniform per cluster
        if (fallback) break;
      }
      {
        const int b = kCThreads * c + tid;   // this thread's bin of the row histogram
        uint32_t v = 0;
#pragma unroll
        for (int q = 0; q < kCluster; ++q) v += ld_cluster_u32(mapa_shared(h2_base + 4u * b, q));
#pragma unroll
        for (int q = 0; q < kCluster; ++q) st_cluster_u32(mapa_shared(g2_base + 4u * b, q), v);
      }
      cluster_sync();   // every CTA holds the row histogram
      find_digit_c(g2, pass == 0 ? kBins : 1024, kr, sm);
      kr -= sm.s_above;
      prefix |= sm.s_digit << shift;
      pmask |= dmask << shift;
      __syncthreads();
    }
    if (!fallback) {
      T = (bstar << 21) | prefix;
      // ---- the keys in b* (tie bits for now) above T join sel, those equal
      // to T stay in tie
      const int nw = (len + 31) >> 5;
      uint32_t sel_cnt = 0, tie_cnt = 0;
      for (int w = tid; w < nw; w += kCThreads) {
        uint32_t t = sm.tie[w], s = sm.sel[w], keep = 0u;
        while (t != 0u) {
          const int b = __ffs(t) - 1;
          t &= t - 1u;
          const uint32_t key = order_key(__ldg(slice + 32 * w + b));
          if (key > T) s |= 1u << b;
          else if (key == T) keep |= 1u << b;
        }
        sm.sel[w] = s;
        sm.tie[w] = keep;
        sel_cnt += static_cast<uint32_t>(__popc(s));
        tie_cnt += static_cast<uint32_t>(__popc(keep));
      }
      exchange_counts(sel_cnt, tie_cnt);   // (its barriers also complete the bitmaps)
    }
  }
  if (fallback) {
    // ---- many keys in b*: two more radix passes over the slices, the
    // histograms reduced through distributed shared memory
    for (int i = tid; i < kSliceBits / 32; i += kCThreads) { sm.sel[i] = 0u; sm.tie[i] = 0u; }
    uint32_t prefix = bstar << 21, pmask = 0x7FFu << 21;
#pragma unroll 1
    for (int pass = 1; pass < 3; ++pass) {
      const int shift = pass == 1 ? 10 : 0;
      const uint32_t dmask = pass == 2 ? 0x3FFu : 0x7FFu;
      for (int i = tid; i < kBins; i += kCThreads) hist[i] = 0u;
      __syncthreads();
      for_slice(slice, len, [&](int, uint32_t key, bool valid) {
        if (valid && (key & pmask) == prefix) atomicAdd(&hist[(key >> shift) & dmask], 1u);
      });
      __syncthreads();
      cluster_sync();   // every CTA's histogram is complete
      {
        const int b = kCThreads * c + tid;   // this thread's bin of the row histogram
        uint32_t v = 0;
#pragma unroll
        for (int q = 0; q < kCluster; ++q) v += ld_cluster_u32(mapa_shared(hist_base + 4u * b, q));
#pragma unroll
        for (int q = 0; q < kCluster; ++q) st_cluster_u32(mapa_shared(ghist_base + 4u * b, q), v);
      }
      cluster_sync();   // every CTA holds the row histogram; the local ones may be reused
      find_digit_c(ghist, pass == 2 ? 1024 : kBins, kr, sm);
      kr -= sm.s_above;
      prefix |= sm.s_digit << shift;
      pmask |= dmask << shift;
      __syncthreads();
    }
    T = prefix;   // the k-th largest key; kr keys equal to it are taken

    // ---- bitmaps of the slice: keys above T, keys equal to T
    uint32_t sel_cnt = 0, tie_cnt = 0;
    for_slice(slice, len, [&](int i, uint32_t key, bool valid) {
      if (valid && key >= T) {
        if (key > T) {
          ++sel_cnt;
          if (bitmapped) atomicOr(&sm.sel[i >> 5], 1u << (i & 31));
        } else {
          ++tie_cnt;
          if (bitmapped) atomicOr(&sm.tie[i >> 5], 1u << (i & 31));
        }
      }
    });
    exchange_counts(sel_cnt, tie_cnt);
  }

  // ---- ordered emission of the slice: thread t scans words [wpt t, wpt t + wpt)
  const int nwords = (len + 31) >> 5;
  const int wpt = (nwords + kCThreads - 1) / kCThreads;
  // slices longer than the bitmaps rebuild the words from the scores
  auto words = [&](int w, uint32_t& bs, uint32_t& bt) {
    if (bitmapped) {
      bs = sm.sel[w];
      bt = sm.tie[w];
    } else {
      bs = 0u; bt = 0u;
      for (int j = 0; j < 32; ++j) {
        const int i = 32 * w + j;
        if (i < len) {
          const uint32_t key = order_key(__ldg(slice + i));
          bs |= (key > T ? 1u : 0u) << j;
          bt |= (key == T ? 1u : 0u) << j;
        }
      }
    }
  };
  const int w0 = tid * wpt;
  uint32_t my_sel = 0, my_tie = 0;
  for (int q = 0; q < wpt; ++q) {
    if (w0 + q < nwords) {
      uint32_t bs, bt;
      words(w0 + q, bs, bt);
      my_sel += __popc(bs);
      my_tie += __popc(bt);
    }
  }
  uint32_t tot;
  const uint32_t tie_before = block_inclusive_scan<kCThreads>(my_tie, sm.warp_sums, tot) - my_tie;
  uint32_t take = tie_before >= kr_here ? 0u : min(kr_here - tie_before, my_tie);
  const uint32_t out_cnt = my_sel + take;
  uint32_t pos = out_base + block_inclusive_scan<kCThreads>(out_cnt, sm.warp_sums, tot) - out_cnt;
  for (int q = 0; q < wpt; ++q) {
    const int w = w0 + q;
    if (w >= nwords) break;
    uint32_t bits, tb;
    words(w, bits, tb);
    while (take > 0u && tb != 0u) {   // the lowest positions of the ties
      bits |= tb & (0u - tb);
      tb &= tb - 1u;
      --take;
    }
    while (bits != 0u) {
      const int b = __ffs(bits) - 1;
      bits &= bits - 1u;
      const int i = lo + 32 * w + b;
      if (pos < static_cast<uint32_t>(k)) {
        out_idx[pos] = i;
        if (out_val) out_val[pos] = __ldg(row + i);
      }
      ++pos;
    }
  }
}

}  // namespace topk
}  // namespace dsa
