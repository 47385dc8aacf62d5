// Step 1 on the tensor cores: the FP8 lightning indexer.
//
//   I[t,s] = sum_j w[t,j] * ReLU(q_I[t,j] . k_I[s])       for s <= p(t)
// ("DeepSeek V3.2: How Far Can Open Models Go If You Actually Try?", §3.1; the
// indexer runs in FP8 with a handful of heads; ReLU is chosen for throughput,
// DSA section of the DeepSeek-V3.2 launch article).  Real inputs are e4m3
// codes times one fp32 scale per query token and per key; for positive scales
//   I[t,s] = k_scale[s] * sum_j (w[t,j] q_scale[t]) ReLU(qc[t,j] . kc[s]).
//
// Layout of the contraction: keys on the MMA M dimension (A = 128 keys x 128
// e4m3, K-major), query heads on N (B = G tokens x 64 heads x 128 e4m3,
// K-major, N = 64 G <= 256), fp32 accumulator in TMEM (128 lanes x 64 G cols).
// Each epilogue thread then owns one key (one TMEM lane) and holds all 64
// heads of a token in its registers: ReLU, head weights, head sum, key scale
// and the causal mask need no cross-thread traffic, and the stores of
// I[t, s..s+127] are coalesced.
//
// Warp roles (persistent CTA, one per SM):
//   warp 0      TMA producer: q block of the item, then a ring of key tiles
//   warp 1      MMA issuer (one thread): 4 x tcgen05.mma kind::f8f6f4 per tile
//   warp 2      TMEM allocator
//   warps 4-19  four epilogue warpgroups; warpgroup e handles column group e
// Two TMEM accumulator slots (2 x 256 columns) let the epilogue of one slot
// overlap the MMAs of the next.  A slot holds four 64-column groups: for an
// item of g query rows, 4/g consecutive key tiles (one for g >= 3), so the
// four epilogue warpgroups share the work also in decode (g = 1).
//
// Work items: a group of up to G consecutive query rows of one sequence (from
// the last rows backwards, so long causal rows start first) and a chunk of at
// most `max_tiles` key tiles.  CTA c takes items c, c + gridDim.x, ...
#pragma once

#include <cstdint>

#include "common.cuh"
#include "ptx.cuh"

namespace dsa {
namespace idx_tc {

constexpr int kKeys = 128;          // keys per tile (MMA M)
constexpr int kDim = 128;           // d_I (MMA K), one e4m3 byte each
constexpr int kHeads = 64;          // H_I
constexpr int kMaxTokens = 4;       // tokens per item (N = 64 G <= 256)
constexpr int kStages = 6;          // key-tile ring depth
constexpr int kEpiGroups = 4;      // epilogue warpgroups, one token each
constexpr int kThreads = 128 + 128 * kEpiGroups;
constexpr int kTileBytes = kKeys * kDim;                 // 16 KiB
constexpr int kQTokenBytes = kHeads * kDim;              // 8 KiB
constexpr int kQBytes = kMaxTokens * kQTokenBytes;       // 32 KiB
constexpr int kAccCols = 256;
constexpr int kTmemCols = 512;

// shared-memory map (offsets from a 1024-byte aligned base)
constexpr int kOffK = 0;
constexpr int kOffQ = kOffK + kStages * kTileBytes;
constexpr int kOffW = kOffQ + 2 * kQBytes;
constexpr int kOffH = kOffW + 2 * kMaxTokens * kHeads * 4;    // first-digit histograms of an item's rows
constexpr int kOffBar = kOffH + kMaxTokens * kRadixBins * 4;
constexpr int kNumBars = 2 * kStages + 2 + 2 + 2 + 2 + 1 + 2 * kEpiGroups + 2;
constexpr int kOffMisc = kOffBar + kNumBars * 8;
constexpr int kSmemBytes = kOffMisc + 16 + 1024;  // + alignment slack

struct Params {
  const float* q_scale;
  const float* k_scale;
  const float* w;
  float* scores;
  int64_t ld;
  uint32_t* hist;              // optional [rows of the launch][2048]: adds the first radix digit
                               // histogram of every row's scores (zero on entry)
  const int32_t* cu_q;
  const int32_t* cu_kv;
  int num_seqs;
  int64_t row_begin, row_end;  // query rows handled by this launch
  int group;                   // tokens per item, 1..4
  int max_tiles;               // key tiles per item
  uint32_t fault;              // test hook: 1 = producer skips one tile's load
};

struct Item {
  int64_t t0;      // first query row
  int g;           // rows in the item
  int pos0;        // position of row t0
  int kt0, kt1;    // key tiles [kt0, kt1)
  int64_t kv0;     // first global key row of the sequence
};

// Walks the item list in increasing global item index; each role of the CTA
// runs its own walker over the same sequence.
struct Walker {
  int b = -1;
  int64_t base = 0;
  int64_t items_b = 0;
  int64_t r_lo = 0, r_hi = 0;
  int nchunks = 1, nkv = 0, nq = 0;
  int64_t q0 = 0, kv0 = 0;

  __device__ bool seek(int64_t it, const Params& P, Item& out) {
    while (it >= base + items_b) {
      base += items_b;
      ++b;
      if (b >= P.num_seqs) return false;
      q0 = __ldg(P.cu_q + b);
      const int64_t q1 = __ldg(P.cu_q + b + 1);
      kv0 = __ldg(P.cu_kv + b);
      nkv = __ldg(P.cu_kv + b + 1) - static_cast<int>(kv0);
      nq = static_cast<int>(q1 - q0);
      r_lo = q0 > P.row_begin ? q0 : P.row_begin;
      r_hi = q1 < P.row_end ? q1 : P.row_end;
      const int64_t rows = r_hi > r_lo ? r_hi - r_lo : 0;
      const int64_t groups = (rows + P.group - 1) / P.group;
      const int ntiles = (nkv + kKeys - 1) / kKeys;
      nchunks = (ntiles + P.max_tiles - 1) / P.max_tiles;
      if (nchunks < 1) nchunks = 1;
      items_b = groups * nchunks;
    }
    const int64_t local = it - base;
    const int64_t gi = local / nchunks;
    const int c = static_cast<int>(local % nchunks);
    const int64_t hi = r_hi - gi * P.group;
    const int64_t lo = (hi - P.group) > r_lo ? (hi - P.group) : r_lo;
    out.t0 = lo;
    out.g = static_cast<int>(hi - lo);
    out.pos0 = nkv - nq + static_cast<int>(lo - q0);
    const int p_last = out.pos0 + out.g - 1;
    const int ntiles = (p_last + 1 + kKeys - 1) / kKeys;
    out.kt0 = c * P.max_tiles;
    out.kt1 = (c + 1) * P.max_tiles < ntiles ? (c + 1) * P.max_tiles : ntiles;
    out.kv0 = kv0;
    return true;
  }
};

// Key tiles packed into one 256-column accumulator slot for an item of g
// query rows: a slot holds 4 column groups of 64 (token, key tile) pairs, so
// an item of one row (decode) fills a slot with 4 consecutive key tiles and
// all four epilogue warpgroups work on it.
__device__ __forceinline__ int tiles_per_slot(int g) { return g >= 3 ? 1 : 4 / g; }

// acc += sum_j w[j] ReLU(x[j]) over 32 heads.  Even heads take ReLU as
// max(x, 0) (ALU pipe), odd heads as x + |x| = 2 ReLU(x) (FMA pipe) against
// weights staged at half value; both products then share one packed fp32x2
// FMA.  Both forms are exact, so the sum equals the plain formula up to the
// order of the additions.  Four independent partial sums keep the FMA chains
// short.
__device__ __forceinline__ void reduce_chunk(const uint32_t (&x)[32], const float* w, float2 (&acc)[4]) {
  const float4* wv = reinterpret_cast<const float4*>(w);
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const float4 wj = wv[j];
    const float x0 = __uint_as_float(x[4 * j + 0]), x1 = __uint_as_float(x[4 * j + 1]);
    const float x2 = __uint_as_float(x[4 * j + 2]), x3 = __uint_as_float(x[4 * j + 3]);
    float2& a0 = acc[(2 * j) & 3];
    float2& a1 = acc[(2 * j + 1) & 3];
    a0 = __ffma2_rn(make_float2(wj.x, wj.y), make_float2(fmaxf(x0, 0.f), x1 + fabsf(x1)), a0);
    a1 = __ffma2_rn(make_float2(wj.z, wj.w), make_float2(fmaxf(x2, 0.f), x3 + fabsf(x3)), a1);
  }
}

// kHist: also build the first radix digit histograms of the rows' scores
// into P.hist (the forward runs without them; see dsa_index_scores_hist).
template <bool kHist>
__global__ void __launch_bounds__(kThreads, 1)
    indexer_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const Params P) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // 1024-byte aligned base, derived by pointer arithmetic on the shared array
  // so that accesses through it stay shared-memory instructions
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  float* wbuf = reinterpret_cast<float*>(smem + kOffW);
  const uint32_t bar0 = sbase + kOffBar;
  auto kv_full = [&](int s) { return bar0 + 8u * s; };
  auto kv_empty = [&](int s) { return bar0 + 8u * (kStages + s); };
  auto q_full = [&](int b) { return bar0 + 8u * (2 * kStages + b); };
  auto q_empty = [&](int b) { return bar0 + 8u * (2 * kStages + 2 + b); };
  auto acc_full = [&](int b) { return bar0 + 8u * (2 * kStages + 4 + b); };
  auto acc_empty = [&](int b) { return bar0 + 8u * (2 * kStages + 6 + b); };
  const uint32_t drain_bar = bar0 + 8u * (2 * kStages + 8);
  // w_full(e, b): warpgroup e has staged the head weights of its item with parity b
  auto w_full = [&](int e, int b) { return bar0 + 8u * (2 * kStages + 9 + 2 * e + b); };
  // the item's histograms are cleared (h_zeroed) / complete (h_done): all
  // epilogue threads arrive once per item
  const uint32_t h_zeroed = bar0 + 8u * (2 * kStages + 9 + 2 * kEpiGroups);
  const uint32_t h_done = h_zeroed + 8u;
  uint32_t* hist_s = reinterpret_cast<uint32_t*>(smem + kOffH);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) { mbar_init(kv_full(s), 1); mbar_init(kv_empty(s), 1); }
    for (int b = 0; b < 2; ++b) {
      mbar_init(q_full(b), 1);
      mbar_init(q_empty(b), 1);
      mbar_init(acc_full(b), 1);
      mbar_init(acc_empty(b), kEpiGroups * 128);
    }
    mbar_init(drain_bar, 1);
    for (int b = 0; b < 2 * kEpiGroups; ++b) mbar_init(w_full(b >> 1, b & 1), 128);
    mbar_init(h_zeroed, kEpiGroups * 128);
    mbar_init(h_done, kEpiGroups * 128);
    *abort_flag = 0;
    fence_mbar_init();
    fence_proxy_async_smem();
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
  }
  if (warp == 2) tmem_alloc(smem_u32(tmem_slot), kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      Walker wk;
      Item item;
      int qi = 0, ti = 0;
      bool ok = true;
      for (int64_t it = blockIdx.x; ok && wk.seek(it, P, item); it += gridDim.x) {
        if (item.kt0 >= item.kt1) continue;
        const int qb = qi & 1;
        if (qi >= 2 && !mbar_wait(q_empty(qb), ((qi >> 1) - 1) & 1, abort_flag)) break;
        mbar_arrive_expect_tx(q_full(qb), item.g * kQTokenBytes);
        for (int g = 0; g < item.g; ++g)
          tma_load_2d(sbase + kOffQ + qb * kQBytes + g * kQTokenBytes, &tm_q, 0,
                      static_cast<int32_t>((item.t0 + g) * kHeads), q_full(qb));
        ++qi;
        for (int kt = item.kt0; kt < item.kt1; ++kt, ++ti) {
          const int st = ti % kStages;
          if (ti >= kStages && !mbar_wait(kv_empty(st), ((ti / kStages) - 1) & 1, abort_flag)) {
            ok = false;
            break;
          }
          if (P.fault == 1u && ti == 2) continue;  // test hook: this tile never arrives
          mbar_arrive_expect_tx(kv_full(st), kTileBytes);
          tma_load_2d(sbase + kOffK + st * kTileBytes, &tm_k, 0,
                      static_cast<int32_t>(item.kv0 + static_cast<int64_t>(kt) * kKeys), kv_full(st));
        }
      }
      // drain: wait for every load still in flight before the CTA may exit
      for (int j = (ti > kStages ? ti - kStages : 0); j < ti; ++j)
        if (!(P.fault == 1u && j == 2)) drain_wait(kv_full(j % kStages), (j / kStages) & 1);
      for (int j = (qi > 2 ? qi - 2 : 0); j < qi; ++j) drain_wait(q_full(j & 1), (j >> 1) & 1);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      Walker wk;
      Item item;
      int qi = 0, ti = 0, si = 0;   // q blocks, key tiles, accumulator slots
      bool ok = true;
      for (int64_t it = blockIdx.x; ok && wk.seek(it, P, item); it += gridDim.x) {
        if (item.kt0 >= item.kt1) continue;
        const int qb = qi & 1;
        if (!mbar_wait(q_full(qb), (qi >> 1) & 1, abort_flag)) break;
        tc_fence_after();
        const uint32_t idesc = make_idesc(0, 0, kKeys, kHeads * item.g, 0, 0);
        const uint32_t qaddr = sbase + kOffQ + qb * kQBytes;
        const int per = tiles_per_slot(item.g);
        if (per == 1) {
          // one key tile per slot (items of 3 or 4 rows)
          for (int kt = item.kt0; kt < item.kt1; ++kt, ++ti, ++si) {
            const int st = ti % kStages, ab = si & 1;
            if (si >= 2 && !mbar_wait(acc_empty(ab), ((si >> 1) - 1) & 1, abort_flag)) { ok = false; break; }
            if (!mbar_wait(kv_full(st), (ti / kStages) & 1, abort_flag)) { ok = false; break; }
            tc_fence_after();
            const uint32_t kaddr = sbase + kOffK + st * kTileBytes;
#pragma unroll
            for (int ks = 0; ks < kDim / 32; ++ks)
              mma_fp8(tmem + ab * kAccCols, make_desc_sw128(kaddr + ks * 32, 16, 1024),
                      make_desc_sw128(qaddr + ks * 32, 16, 1024), idesc, ks > 0 ? 1u : 0u);
            mma_commit(kv_empty(st));
            mma_commit(acc_full(ab));
          }
        } else
        for (int kt = item.kt0; kt < item.kt1 && ok; kt += per, ++si) {
          const int ab = si & 1;
          if (si >= 2 && !mbar_wait(acc_empty(ab), ((si >> 1) - 1) & 1, abort_flag)) { ok = false; break; }
          for (int u = 0; u < per && kt + u < item.kt1; ++u, ++ti) {
            const int st = ti % kStages;
            if (!mbar_wait(kv_full(st), (ti / kStages) & 1, abort_flag)) { ok = false; break; }
            tc_fence_after();
            const uint32_t kaddr = sbase + kOffK + st * kTileBytes;
            const uint32_t dcol = ab * kAccCols + u * kHeads * item.g;
#pragma unroll
            for (int ks = 0; ks < kDim / 32; ++ks)
              mma_fp8(tmem + dcol, make_desc_sw128(kaddr + ks * 32, 16, 1024),
                      make_desc_sw128(qaddr + ks * 32, 16, 1024), idesc, ks > 0 ? 1u : 0u);
            mma_commit(kv_empty(st));
          }
          if (!ok) break;
          mma_commit(acc_full(ab));
        }
        if (!ok) break;
        mma_commit(q_empty(qb));
        ++qi;
      }
      mma_commit(drain_bar);
      drain_wait(drain_bar, 0);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ epilogue
    const int e = (warp - 4) >> 2;         // warpgroup: column group e of each slot
    const int wq = warp & 3;               // TMEM lane quarter of this warp
    const int et = threadIdx.x - 128 - e * 128;
    Walker wk;
    Item item{};
    int qi = 0, si = 0;
    bool ok = true;
    // after the item's last tile: wait until every epilogue thread has added
    // its scores, then add this thread's share of the histograms to the rows'
    // global histograms (other CTAs may hold other key ranges of the rows)
    auto flush_hist = [&](int hq) {
      mbar_arrive(h_done);
      if (!warp_wait(h_done, hq & 1, abort_flag)) { ok = false; return; }
      const int ht = threadIdx.x - 128;
      for (int i = ht; i < item.g * kRadixBins; i += kEpiGroups * 128) {
        const uint32_t c = hist_s[i];
        if (c) atomicAdd(P.hist + (item.t0 - P.row_begin + i / kRadixBins) * kRadixBins + (i % kRadixBins), c);
      }
    };
    for (int64_t it = blockIdx.x; ok && wk.seek(it, P, item); it += gridDim.x) {
      if (item.kt0 >= item.kt1) continue;
      // column group e of a slot: key tile u = e / g of the slot, token e % g
      const int per = tiles_per_slot(item.g);
      const int u = e / item.g, te = e % item.g;
      const bool used = u < per;
      float* wsm = wbuf + (qi & 1) * (kMaxTokens * kHeads) + e * kHeads;
      if (used && et < kHeads) {
        const int64_t t = item.t0 + te;
        // odd heads are pre-halved: their ReLU is taken as x + |x| = 2 ReLU(x)
        wsm[et] = __ldg(P.w + t * kHeads + et) * (P.q_scale ? __ldg(P.q_scale + t) : 1.f) *
                  ((et & 1) ? 0.5f : 1.f);
      }
      mbar_arrive(w_full(e, qi & 1));
      if (!warp_wait(w_full(e, qi & 1), (qi >> 1) & 1, abort_flag)) break;
      // this thread's share of the item's row histograms starts at zero (it
      // flushed the same share at the end of its previous item)
      const int ht = threadIdx.x - 128;                   // 0 .. 511
      if (kHist) {
        for (int i = ht; i < item.g * kRadixBins; i += kEpiGroups * 128) hist_s[i] = 0u;
        mbar_arrive(h_zeroed);
        if (!warp_wait(h_zeroed, qi & 1, abort_flag)) break;
      }
      const int hq = qi;
      ++qi;
      const int64_t srow = item.t0 + te - P.row_begin;   // score row of this token
      const int plim = item.pos0 + te;                    // its last candidate
      if (per == 1) {
        // one key tile per slot (items of 3 or 4 rows): token e at columns
        // [64e, 64e + 64)
        for (int kt = item.kt0; kt < item.kt1; ++kt, ++si) {
          const int ab = si & 1;
          if (!warp_wait(acc_full(ab), (si >> 1) & 1, abort_flag)) { ok = false; break; }
          tc_fence_after();
          if (!used) {
            tc_fence_before();
            mbar_arrive(acc_empty(ab));
            continue;
          }
          const uint32_t ta = tmem + (static_cast<uint32_t>(wq * 32) << 16) + ab * kAccCols + e * kHeads;
          const int s = kt * kKeys + wq * 32 + lane;   // sequence-local key of this thread
          const float ks = (s <= plim && P.k_scale) ? __ldg(P.k_scale + item.kv0 + s) : 1.f;
          float2 acc[4];
#pragma unroll
          for (int v = 0; v < 4; ++v) acc[v] = make_float2(0.f, 0.f);
          {
            // the 64 head columns in two halves (32 registers of data live)
            uint32_t x[32];
            tmem_ld32(ta, x);
            tmem_wait_ld();
            reduce_chunk(x, wsm, acc);
            tmem_ld32(ta + 32, x);
            tmem_wait_ld();
            tc_fence_before();
            mbar_arrive(acc_empty(ab));      // accumulator read: the MMA may reuse it
            reduce_chunk(x, wsm + 32, acc);
          }
          const float2 tt = __fadd2_rn(__fadd2_rn(acc[0], acc[1]), __fadd2_rn(acc[2], acc[3]));
          if (s <= plim) {
            const float v = (tt.x + tt.y) * ks;
            P.scores[srow * P.ld + s] = v;
            if (kHist) atomicAdd(hist_s + te * kRadixBins + (order_key(v) >> kRadixShift), 1u);
          }
        }
        if (ok && kHist) flush_hist(hq);
        continue;
      }
      for (int kt0 = item.kt0; kt0 < item.kt1; kt0 += per, ++si) {
        const int ab = si & 1;
        if (!warp_wait(acc_full(ab), (si >> 1) & 1, abort_flag)) { ok = false; break; }
        tc_fence_after();
        const int kt = kt0 + u;
        if (!used || kt >= item.kt1) {
          tc_fence_before();
          mbar_arrive(acc_empty(ab));
          continue;
        }
        const uint32_t ta = tmem + (static_cast<uint32_t>(wq * 32) << 16) + ab * kAccCols +
                            u * kHeads * item.g + te * kHeads;
        const int s = kt * kKeys + wq * 32 + lane;   // sequence-local key of this thread
        const float ks = (s <= plim && P.k_scale) ? __ldg(P.k_scale + item.kv0 + s) : 1.f;
        float2 acc[4];
#pragma unroll
        for (int v = 0; v < 4; ++v) acc[v] = make_float2(0.f, 0.f);
        {
          // the 64 head columns in two halves (32 registers of data live)
          uint32_t x[32];
          tmem_ld32(ta, x);
          tmem_wait_ld();
          reduce_chunk(x, wsm, acc);
          tmem_ld32(ta + 32, x);
          tmem_wait_ld();
          tc_fence_before();
          mbar_arrive(acc_empty(ab));      // accumulator read: the MMA may reuse it
          reduce_chunk(x, wsm + 32, acc);
        }
        const float2 tt = __fadd2_rn(__fadd2_rn(acc[0], acc[1]), __fadd2_rn(acc[2], acc[3]));
        if (s <= plim) {
          const float v = (tt.x + tt.y) * ks;
          P.scores[srow * P.ld + s] = v;
          if (kHist) atomicAdd(hist_s + te * kRadixBins + (order_key(v) >> kRadixShift), 1u);
        }
      }
      if (ok && kHist) flush_hist(hq);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace idx_tc
}  // namespace dsa
