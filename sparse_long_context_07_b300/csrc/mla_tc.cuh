// Step 3 on the tensor cores: sparse MLA in MQA mode over the selected rows.
//
//   u_t[h] = sum_i softmax_i(scale * Q[t,h] . c_{s_i}) * c_{s_i}[0:d_v]
// over the selected positions s_i ("DeepSeek V3.2: How Far Can Open Models Go
// If You Actually Try?", §3.1: attention only over the top-k latents; MLA in
// MQA mode, one shared latent row per token read by all heads, §3.1 and §2.2).
// Dimensions: 128 heads, d_qk = 576, d_v = 512, bf16 in, fp32 accumulate.
//
// The fp32 output accumulator of one query token (128 heads x 512) fills the
// whole TMEM of an SM (128 lanes x 512 columns), leaving no room for the score
// tile.  So a cluster of two CTAs (two SMs) serves one token:
//   CTA r holds Q[:, 288r : 288r+288] and gathers the same columns of each
//   selected latent row, computes the partial scores S_r = Q_r K_r^T
//   (M = 128 heads, N = 64 rows, K = 288), and the two CTAs swap S_r through
//   distributed shared memory.  Both then hold S = S_0 + S_1 bit-identically
//   (fp32 addition commutes), run the same online softmax, and CTA r
//   accumulates O[:, 256r : 256r+256] += P V_r (M = 128, N = 256, K = 64) in
//   its TMEM (256 columns + 2 x 64 for S).
// Each latent row is fetched once per cluster (640 B per CTA, the 64 columns
// 256..319 by both), so all 128 heads share one gather (the MQA saving).
//
// Warp roles per CTA (320 threads):
//   warps 0-3  softmax / epilogue, thread h = head h = TMEM lane h
//   warps 4-7  gather: cp.async 16 B chunks of the selected rows into a
//              128-byte-swizzled K-major tile (2 stages)
//   warp 8     Q load (TMA) and the MMA issuer (one thread)
//   warp 9     TMEM allocator
// The MMA thread issues QK(j) before PV(j-1) so the softmax of tile j
// overlaps PV(j-1) on the tensor pipe.  The running max is updated lazily
// (only when a tile's max exceeds it by more than 2^8 in the exp2 domain), so
// the O rescale in TMEM is rare.
//
// Split-KV (decode): a cluster may take a contiguous range of 64-row tiles of
// a token; it then writes fp32 (O / l, lse) partials merged by combine_kernel.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>

#include "common.cuh"
#include "ptx.cuh"

namespace dsa {
namespace mla_tc {

constexpr int kHeads = 128;
constexpr int kDqk = 576;
constexpr int kDv = 512;
constexpr int kRows = 64;               // selected rows per tile
constexpr int kLocalBlocks = 5;         // 64-column blocks held per CTA
constexpr int kKSteps = 18;             // 288 / 16 MMA k-steps per CTA for QK
constexpr int kQBlockBytes = kHeads * 128;         // 16 KiB
constexpr int kKVBlockBytes = kRows * 128;         // 8 KiB
constexpr int kStageBytes = kLocalBlocks * kKVBlockBytes;  // 40 KiB
constexpr int kStages = 2;
constexpr int kPBytes = kHeads * kRows * 2;        // 16 KiB
constexpr int kXBytes = kHeads * kRows * 4;        // 32 KiB
constexpr int kThreads = 320;
constexpr int kTmemCols = 512;
constexpr int kSCol = 256;              // TMEM column of S buffer 0
constexpr float kRescaleThreshold = 8.f;

constexpr int kOffQ = 0;
constexpr int kOffKV = kOffQ + kLocalBlocks * kQBlockBytes;
constexpr int kOffP = kOffKV + kStages * kStageBytes;
constexpr int kOffX = kOffP + 2 * kPBytes;
constexpr int kOffBar = kOffX + kXBytes;
constexpr int kNumBars = 20;
constexpr int kOffMisc = kOffBar + kNumBars * 8;
constexpr int kSmemBytes = kOffMisc + 16 + 1024;

struct Params {
  const __nv_bfloat16* kv;   // [total_kv, 576]
  const int32_t* idx;        // [rows of this launch, k], relative to row0
  int k;
  float c_log2;              // scale * log2(e)
  const int32_t* cu_q;
  const int32_t* cu_kv;
  int num_seqs;
  int64_t row0;
  int nsplit;                // clusters per query row
  int tiles_per_split;
  __nv_bfloat16* out;        // nsplit == 1: [rows, 128, 512], relative to row0
  float* lse;                // nsplit == 1: [rows, 128] or nullptr
  float* part_o;             // nsplit > 1: [rows * nsplit, 128, 512] fp32
  float* part_lse;           // nsplit > 1: [rows * nsplit, 128]
};

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&v);
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    mla_kernel(const __grid_constant__ CUtensorMap tm_q, const Params P) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // 1024-byte aligned base, derived by pointer arithmetic on the shared array
  // so that accesses through it stay shared-memory instructions
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + kOffBar;
  const uint32_t q_full = bar0;
  auto kv_full = [&](int s) { return bar0 + 8u * (1 + s); };
  auto kv_empty = [&](int s) { return bar0 + 8u * (3 + s); };
  auto s_full = [&](int s) { return bar0 + 8u * (5 + s); };
  auto s_empty = [&](int s) { return bar0 + 8u * (7 + s); };
  auto p_full = [&](int s) { return bar0 + 8u * (9 + s); };
  auto p_empty = [&](int s) { return bar0 + 8u * (11 + s); };
  const uint32_t o_ready = bar0 + 8u * 13;
  const uint32_t x_full = bar0 + 8u * 14;
  const uint32_t x_empty = bar0 + 8u * 15;
  const uint32_t drain_bar = bar0 + 8u * 16;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const uint32_t peer = rank ^ 1u;

  // the work unit of this cluster
  const int64_t unit = blockIdx.x >> 1;
  const int64_t rrel = unit / P.nsplit;
  const int split = static_cast<int>(unit % P.nsplit);
  const int64_t row = P.row0 + rrel;
  const RowGeom geo = row_geom(P.cu_q, P.cu_kv, P.num_seqs, row);
  const int n = geo.p + 1;
  const int tiles_total = (P.k + kRows - 1) / kRows;
  const int t_begin = split * P.tiles_per_split;
  int t_end = t_begin + P.tiles_per_split;
  if (t_end > tiles_total) t_end = tiles_total;
  const int nt = t_end > t_begin ? t_end - t_begin : 0;
  const int32_t* __restrict__ idx_row = P.idx + rrel * static_cast<int64_t>(P.k);

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(kv_full(s), 128);
      mbar_init(kv_empty(s), 1);
      mbar_init(s_full(s), 1);
      mbar_init(s_empty(s), 128);
      mbar_init(p_full(s), 128);
      mbar_init(p_empty(s), 1);
    }
    mbar_init(o_ready, 1);
    mbar_init(x_full, 128);
    mbar_init(x_empty, 128);
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
    fence_proxy_async_smem();
  }
  if (warp == 9) tmem_alloc(smem_u32(tmem_slot), kTmemCols);
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // the peer's barriers exist before any remote access
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp >= 4 && warp < 8) {
    // ------------------------------------------------------------ gather
    const int pt = threadIdx.x - 128;
    bool ok = true;
    for (int j = 0; j < nt && ok; ++j) {
      const int st = j & 1;
      if (j >= 2 && !mbar_wait(kv_empty(st), ((j >> 1) - 1) & 1, abort_flag)) { ok = false; break; }
      const uint32_t stage = sbase + kOffKV + st * kStageBytes;
      const int e_base = (t_begin + j) * kRows;
#pragma unroll 4
      for (int m = 0; m < (kRows * kLocalBlocks * 8) / 128; ++m) {
        const int c = pt + 128 * m;
        const int i = c / (kLocalBlocks * 8);
        const int cc = c - i * (kLocalBlocks * 8);
        const int blk = cc >> 3, q = cc & 7;
        const int e = e_base + i;
        const int s = e < P.k ? __ldg(idx_row + e) : -1;
        const bool valid = s >= 0 && s < n;
        if (cc == 0 && (s < -1 || s >= n)) flag_error(DSA_DEVERR_BAD_INDEX);
        const __nv_bfloat16* src =
            P.kv + (valid ? (geo.kv0 + s) * kDqk : 0) + (4 * rank + blk) * 64 + q * 8;
        const uint32_t dst = stage + blk * kKVBlockBytes + i * 128 + ((q ^ (i & 7)) << 4);
        cp_async_16(dst, src, valid ? 16u : 0u);
      }
      cp_async_commit();
      cp_async_wait<0>();
      fence_proxy_async_smem();
      mbar_arrive(kv_full(st));
    }
  } else if (warp == 8) {
    // ------------------------------------------------------------ Q load + MMA
    if (lane == 0 && nt > 0) {
      mbar_arrive_expect_tx(q_full, kLocalBlocks * kQBlockBytes);
      for (int b = 0; b < kLocalBlocks; ++b)
        tma_load_2d(sbase + kOffQ + b * kQBlockBytes, &tm_q, (4 * rank + b) * 64,
                    static_cast<int32_t>(row * kHeads), q_full);
      const uint32_t idesc_qk = make_idesc(1, 1, kHeads, kRows, 0, 0);
      const uint32_t idesc_pv = make_idesc(1, 1, kHeads, 256, 0, 1);
      bool ok = mbar_wait(q_full, 0, abort_flag);
      tc_fence_after();
      auto issue_pv = [&](int i) -> bool {
        const int sb = i & 1;
        if (!mbar_wait(p_full(sb), (i >> 1) & 1, abort_flag)) return false;
        tc_fence_after();
        const uint32_t pa = sbase + kOffP + sb * kPBytes;
        const uint32_t va = sbase + kOffKV + sb * kStageBytes;
#pragma unroll
        for (int ks = 0; ks < kRows / 16; ++ks)
          mma_bf16(tmem, make_desc_sw128(pa + ks * 32, 16, 1024),
                   make_desc_sw128(va + ks * 2048, kKVBlockBytes, 1024), idesc_pv,
                   (i > 0 || ks > 0) ? 1u : 0u);
        mma_commit(p_empty(sb));
        mma_commit(kv_empty(sb));
        mma_commit(o_ready);
        return true;
      };
      for (int j = 0; j < nt && ok; ++j) {
        const int st = j & 1;
        if (!mbar_wait(kv_full(st), (j >> 1) & 1, abort_flag)) { ok = false; break; }
        if (j >= 2 && !mbar_wait(s_empty(st), ((j >> 1) - 1) & 1, abort_flag)) { ok = false; break; }
        tc_fence_after();
        fence_proxy_async_smem();
        const uint32_t stage = sbase + kOffKV + st * kStageBytes;
#pragma unroll
        for (int g = 0; g < kKSteps; ++g) {
          const int gk = kKSteps * rank + g;          // global k-step (16 columns)
          const int lb = (gk >> 2) - 4 * rank;        // local 64-column block
          const int sub = gk & 3;
          mma_bf16(tmem + kSCol + st * kRows,
                   make_desc_sw128(sbase + kOffQ + lb * kQBlockBytes + sub * 32, 16, 1024),
                   make_desc_sw128(stage + lb * kKVBlockBytes + sub * 32, 16, 1024), idesc_qk,
                   g > 0 ? 1u : 0u);
        }
        mma_commit(s_full(st));
        if (j >= 1 && !issue_pv(j - 1)) { ok = false; break; }
      }
      if (ok && nt > 0) issue_pv(nt - 1);
      mma_commit(drain_bar);
      drain_wait(drain_bar, 0);
      drain_wait(q_full, 0);
    }
  } else if (warp < 4) {
    // ------------------------------------------------------------ softmax
    const int h = threadIdx.x;
    const uint32_t t_lane = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    const uint32_t x_local = sbase + kOffX;
    const uint32_t x_peer = mapa_shared(x_local, peer);
    const uint32_t x_full_peer = mapa_shared(x_full, peer);
    const uint32_t x_empty_peer = mapa_shared(x_empty, peer);
    float m_use = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < nt; ++j) {
      const int sb = j & 1;
      const int e0 = (t_begin + j) * kRows + lane;
      const int s0 = e0 < P.k ? __ldg(idx_row + e0) : -1;
      const int s1 = e0 + 32 < P.k ? __ldg(idx_row + e0 + 32) : -1;
      const uint32_t mlo = __ballot_sync(0xffffffffu, s0 >= 0 && s0 < n);
      const uint32_t mhi = __ballot_sync(0xffffffffu, s1 >= 0 && s1 < n);

      if (!warp_wait(s_full(sb), (j >> 1) & 1, abort_flag)) { ok = false; break; }
      tc_fence_after();
      uint32_t a[32], bq[32];
      tmem_ld32(t_lane + kSCol + sb * kRows, a);
      tmem_ld32(t_lane + kSCol + sb * kRows + 32, bq);
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(s_empty(sb));

      // swap partial scores with the peer CTA
      if (j >= 1 && !warp_wait<true>(x_empty, (j - 1) & 1, abort_flag)) { ok = false; break; }
#pragma unroll
      for (int c4 = 0; c4 < 16; ++c4) {
        const uint32_t* src = c4 < 8 ? &a[4 * c4] : &bq[4 * (c4 - 8)];
        st_cluster_v4(x_peer + h * 256 + ((c4 ^ (h & 15)) << 4), __uint_as_float(src[0]),
                      __uint_as_float(src[1]), __uint_as_float(src[2]), __uint_as_float(src[3]));
      }
      mbar_arrive_cluster(x_full_peer);
      if (!warp_wait<true>(x_full, j & 1, abort_flag)) { ok = false; break; }
      float z[64];
      float mt = -INFINITY;
#pragma unroll
      for (int c4 = 0; c4 < 16; ++c4) {
        const float4 pv = *reinterpret_cast<const float4*>(smem + kOffX + h * 256 + ((c4 ^ (h & 15)) << 4));
        const uint32_t* own = c4 < 8 ? &a[4 * c4] : &bq[4 * (c4 - 8)];
        const float pvv[4] = {pv.x, pv.y, pv.z, pv.w};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int i = 4 * c4 + u;
          const bool valid = ((i < 32 ? (mlo >> i) : (mhi >> (i - 32))) & 1u) != 0u;
          const float sval = __uint_as_float(own[u]) + pvv[u];
          z[i] = valid ? sval * P.c_log2 : -INFINITY;
          mt = fmaxf(mt, z[i]);
        }
      }
      mbar_arrive_cluster(x_empty_peer);

      float alpha = 1.f;
      bool resc = false;
      if (mt > m_use + kRescaleThreshold) {
        if (m_use != -INFINITY) { alpha = ex2(m_use - mt); resc = true; }
        m_use = mt;
      }
      l *= alpha;
      uint32_t pk[32];
      float lsum = 0.f;
#pragma unroll
      for (int i = 0; i < 64; i += 2) {
        const float p0 = m_use == -INFINITY ? 0.f : ex2(z[i] - m_use);
        const float p1 = m_use == -INFINITY ? 0.f : ex2(z[i + 1] - m_use);
        pk[i >> 1] = pack_bf16(p0, p1);
        const __nv_bfloat162 r2 = *reinterpret_cast<const __nv_bfloat162*>(&pk[i >> 1]);
        lsum += __bfloat162float(r2.x) + __bfloat162float(r2.y);
      }
      l += lsum;

      if (j >= 2 && !warp_wait(p_empty(sb), ((j >> 1) - 1) & 1, abort_flag)) { ok = false; break; }
      uint8_t* prow = smem + kOffP + sb * kPBytes + h * 128;
#pragma unroll
      for (int cc = 0; cc < 8; ++cc)
        *reinterpret_cast<uint4*>(prow + ((cc ^ (h & 7)) << 4)) =
            make_uint4(pk[4 * cc], pk[4 * cc + 1], pk[4 * cc + 2], pk[4 * cc + 3]);
      fence_proxy_async_smem();
      if (__any_sync(0xffffffffu, resc)) {
        // O must hold PV(j-1) before it is rescaled
        if (!warp_wait(o_ready, (j - 1) & 1, abort_flag)) { ok = false; break; }
        tc_fence_after();
#pragma unroll 1
        for (int c = 0; c < 8; ++c) {
          uint32_t o[32];
          tmem_ld32(t_lane + 32 * c, o);
          tmem_wait_ld();
#pragma unroll
          for (int u = 0; u < 32; ++u) o[u] = __float_as_uint(__uint_as_float(o[u]) * alpha);
          tmem_st32(t_lane + 32 * c, o);
        }
        tmem_wait_st();
        tc_fence_before();
      }
      mbar_arrive(p_full(sb));
    }

    // ---- epilogue: O / l (and lse)
    // PV(nt-2) may still be pending here (it is issued after QK(nt-1)), so wait
    // for its phase before the last one: a parity wait is exact only when the
    // barrier is at most one phase behind.
    bool have_o = ok && nt > 0;
    if (have_o && nt >= 2) have_o = warp_wait(o_ready, (nt - 2) & 1, abort_flag);
    if (have_o) have_o = warp_wait(o_ready, (nt - 1) & 1, abort_flag);
    tc_fence_after();
    const float inv = l > 0.f ? 1.f / l : 0.f;
    const float lse_v = l > 0.f ? (m_use + __log2f(l)) * 0.6931471805599453f : -INFINITY;
    if (P.nsplit == 1) {
      __nv_bfloat16* orow = P.out + (rrel * kHeads + h) * kDv + rank * 256;
#pragma unroll 1
      for (int c = 0; c < 8; ++c) {
        uint32_t o[32];
        if (have_o) { tmem_ld32(t_lane + 32 * c, o); tmem_wait_ld(); }
        else {
#pragma unroll
          for (int u = 0; u < 32; ++u) o[u] = 0u;
        }
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          uint4 pk4;
          pk4.x = pack_bf16(__uint_as_float(o[8 * v + 0]) * inv, __uint_as_float(o[8 * v + 1]) * inv);
          pk4.y = pack_bf16(__uint_as_float(o[8 * v + 2]) * inv, __uint_as_float(o[8 * v + 3]) * inv);
          pk4.z = pack_bf16(__uint_as_float(o[8 * v + 4]) * inv, __uint_as_float(o[8 * v + 5]) * inv);
          pk4.w = pack_bf16(__uint_as_float(o[8 * v + 6]) * inv, __uint_as_float(o[8 * v + 7]) * inv);
          *reinterpret_cast<uint4*>(orow + 32 * c + 8 * v) = pk4;
        }
      }
      if (rank == 0 && P.lse) P.lse[rrel * kHeads + h] = lse_v;
    } else {
      float* orow = P.part_o + (unit * kHeads + h) * kDv + rank * 256;
#pragma unroll 1
      for (int c = 0; c < 8; ++c) {
        uint32_t o[32];
        if (have_o) { tmem_ld32(t_lane + 32 * c, o); tmem_wait_ld(); }
        else {
#pragma unroll
          for (int u = 0; u < 32; ++u) o[u] = 0u;
        }
#pragma unroll
        for (int v = 0; v < 8; ++v)
          *reinterpret_cast<float4*>(orow + 32 * c + 4 * v) =
              make_float4(__uint_as_float(o[4 * v]) * inv, __uint_as_float(o[4 * v + 1]) * inv,
                          __uint_as_float(o[4 * v + 2]) * inv, __uint_as_float(o[4 * v + 3]) * inv);
      }
      if (rank == 0) P.part_lse[unit * kHeads + h] = lse_v;
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();  // no remote access may target an exited CTA
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// Merge of split-KV partials: lse = log sum_i exp(lse_i),
// out = sum_i exp(lse_i - lse) * O_i.  grid (rows, 128 heads), 128 threads x 4 d.
__global__ void __launch_bounds__(128) combine_kernel(const float* __restrict__ part_o,
                                                      const float* __restrict__ part_lse, int nsplit,
                                                      __nv_bfloat16* __restrict__ out,
                                                      float* __restrict__ lse) {
  const int64_t r = blockIdx.x;
  const int h = blockIdx.y;
  float m = -INFINITY;
  for (int s = 0; s < nsplit; ++s) m = fmaxf(m, __ldg(part_lse + ((r * nsplit + s) * kHeads + h)));
  float tot = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int s = 0; s < nsplit; ++s) {
    const float ls = __ldg(part_lse + ((r * nsplit + s) * kHeads + h));
    const float wgt = (m == -INFINITY) ? 0.f : __expf(ls - m);
    tot += wgt;
    const float4 v = __ldg(reinterpret_cast<const float4*>(part_o + ((r * nsplit + s) * kHeads + h) * kDv) +
                           threadIdx.x);
    acc.x = fmaf(wgt, v.x, acc.x);
    acc.y = fmaf(wgt, v.y, acc.y);
    acc.z = fmaf(wgt, v.z, acc.z);
    acc.w = fmaf(wgt, v.w, acc.w);
  }
  const float inv = tot > 0.f ? 1.f / tot : 0.f;
  uint2 pk;
  pk.x = pack_bf16(acc.x * inv, acc.y * inv);
  pk.y = pack_bf16(acc.z * inv, acc.w * inv);
  *reinterpret_cast<uint2*>(out + (r * kHeads + h) * kDv + 4 * threadIdx.x) = pk;
  if (lse && threadIdx.x == 0) lse[r * kHeads + h] = tot > 0.f ? m + __logf(tot) : -INFINITY;
}

}  // namespace mla_tc
}  // namespace dsa
