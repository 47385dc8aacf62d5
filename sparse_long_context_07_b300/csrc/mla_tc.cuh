// Step 3 on the tensor cores: sparse MLA in MQA mode over the selected rows.
//
//   u_t[h] = sum_i softmax_i(scale * Q[t,h] . c_{s_i}) * c_{s_i}[0:d_v]
// over the selected positions s_i ("DeepSeek V3.2: How Far Can Open Models Go
// If You Actually Try?", §3.1: attention only over the top-k latents; MLA in
// MQA mode, one shared latent row per token read by all heads, §3.1 and §2.2).
// Dimensions: 128 heads, d_qk = 576, d_v = 512, bf16 in, fp32 accumulate.
//
// The fp32 output of one query token (128 heads x 512) would fill the whole
// TMEM of an SM, so two CTAs serve each token: CTA `half` owns the output
// columns [256 half, 256 half + 256).  Both CTAs compute the full score tile
// S = Q K^T over all 576 columns themselves, so they never exchange data
// (shared memory of another SM is far too slow for a per-tile exchange on
// this part); the price is that the Q K^T products are done twice.
//
// TMEM (512 columns): O half [0, 256), two score buffers S [256, 320) for
// tiles of 32 selected rows, and Q[:, 0:384] as the A operand of Q K^T
// [320, 512) (two bf16 per column).  Q[:, 384:576] stays in shared memory, so
// Q K^T runs 24 k-steps with A in TMEM and 12 with A in shared memory.  P
// (bf16) goes to shared memory (64-byte swizzle, two buffers), so a score
// buffer is free again as soon as the softmax has read it; P V takes A = P and
// B = V straight from the gathered tile (MN-major).
//
// One thread issues at most about one tcgen05.mma per ~50 cycles, far less
// than the tensor core retires at N = 32, so three warps issue MMAs, each
// into its own accumulator: Q K^T of the even tiles, Q K^T of the odd tiles,
// and P V of every tile (O has a single issuer, so its updates stay ordered).
//
// Warp roles (480 threads):
//   warps 0-3   softmax and epilogue; thread h = head h = TMEM lane h.  They
//               also copy Q[:, 0:384] into TMEM at the start.
//   warps 4-11  gather: 16-byte cp.async of the selected rows (full 1152 B)
//               into a 128-byte-swizzled K-major tile, 4-stage ring
//   warp 12     TMEM allocation; lane 0 loads Q[:, 384:576] with TMA and
//               issues Q K^T of the even tiles
//   warp 13     lane 0 issues Q K^T of the odd tiles
//   warp 14     lane 0 issues P V
// The running max is updated lazily (only when a tile's max exceeds it by
// more than 2^8 in the exp2 domain), so the O rescale in TMEM is rare.
//
// Split-KV (decode): a CTA may take a contiguous range of tiles of a token; it
// then writes fp32 (O / l, lse) partials merged by combine_kernel.
//
// Dense mode (the baseline that sparse selection is measured against): no
// index list, every candidate 0..p of the row is attended, i.e. causal
// MLA-MQA attention over the whole context.
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
constexpr int kHalf = 256;              // output columns per CTA
constexpr int kRows = 32;               // selected rows per tile (N of Q K^T)
constexpr int kRowChunks = kDqk / 8;    // 72 chunks of 16 B per latent row
constexpr int kQTmemD = 384;            // Q columns held in TMEM
constexpr int kQSmemBlocks = (kDqk - kQTmemD) / 64;  // 3 blocks of 64 columns
constexpr int kKStepsT = kQTmemD / 16;  // 24 k-steps with A in TMEM
constexpr int kKSteps = kDqk / 16;      // 36
constexpr int kStages = 4;
constexpr int kBlk = kRows * 128;                  // one 64-column block of a tile: 4 KiB
constexpr int kPBytes = kHeads * kRows * 2;        // 8 KiB
constexpr int kStageBytes = (kDqk / 64) * kBlk;    // 36 KiB
constexpr int kQBlk = kHeads * 128;                // 16 KiB
constexpr int kGatherWarps = 8;
constexpr int kGatherThreads = 32 * kGatherWarps;
constexpr int kMmaWarp = 4 + kGatherWarps;   // first of the three issuing warps
constexpr int kThreads = 32 * (kMmaWarp + 3);
constexpr int kTmemCols = 512;
constexpr int kTmemS = 256;             // two score buffers of kRows columns
constexpr int kTmemQ = 320;
constexpr float kRescaleThreshold = 8.f;
static_assert(kTmemQ + kQTmemD / 2 == kTmemCols, "TMEM layout");
static_assert(kGatherThreads == 8 * kRows, "gather: 8 threads per selected row");

constexpr int kOffKV = 0;
constexpr int kOffQ = kOffKV + kStages * kStageBytes;
constexpr int kOffP = kOffQ + kQSmemBlocks * kQBlk;
constexpr int kOffBar = kOffP + 2 * kPBytes;
constexpr int kNumBars = 2 * kStages + 14;
constexpr int kOffMisc = kOffBar + kNumBars * 8;
constexpr int kSmemBytes = kOffMisc + 16 + 1024;

struct Params {
  const __nv_bfloat16* q;    // [total_q, 128, 576]
  const __nv_bfloat16* kv;   // [total_kv, 576]
  const int32_t* idx;        // [rows of this launch, k], relative to row0 (unused when dense)
  int k;                     // selected entries per row (dense: the longest row's candidates)
  int dense;                 // 1: attend over every candidate 0..p (no index list)
  float c_log2;              // scale * log2(e)
  const int32_t* cu_q;
  const int32_t* cu_kv;
  int num_seqs;
  int64_t row0;
  int nsplit;                // CTA pairs per query row
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

__device__ __forceinline__ uint4 ldg_nc_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__global__ void __launch_bounds__(kThreads, 1)
    mla_kernel(const __grid_constant__ CUtensorMap tm_q, const Params P) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // 1024-byte aligned base, derived by pointer arithmetic on the shared array
  // so that accesses through it stay shared-memory instructions
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + kOffBar;
  auto kv_full = [&](int s) { return bar0 + 8u * s; };
  auto kv_empty = [&](int s) { return bar0 + 8u * (kStages + s); };
  const uint32_t qt_full = bar0 + 8u * (2 * kStages);      // Q columns in TMEM (128 arrivals)
  const uint32_t qs_full = bar0 + 8u * (2 * kStages + 1);  // Q columns in smem (TMA)
  auto s_full = [&](int b) { return bar0 + 8u * (2 * kStages + 2 + b); };   // S of a tile ready
  auto s_empty = [&](int b) { return bar0 + 8u * (2 * kStages + 4 + b); };  // S read by the softmax
  auto p_full = [&](int b) { return bar0 + 8u * (2 * kStages + 6 + b); };   // P written
  auto p_empty = [&](int b) { return bar0 + 8u * (2 * kStages + 8 + b); };  // P V of that buffer done
  const uint32_t o_ready = bar0 + 8u * (2 * kStages + 10);
  auto drain_bar = [&](int r) { return bar0 + 8u * (2 * kStages + 11 + r); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // the work unit of this CTA: (query row, split, output half)
  const int half = static_cast<int>(blockIdx.x & 1u);
  const int64_t unit = blockIdx.x >> 1;
  const int64_t rrel = unit / P.nsplit;
  const int split = static_cast<int>(unit % P.nsplit);
  const int64_t row = P.row0 + rrel;
  const RowGeom geo = row_geom(P.cu_q, P.cu_kv, P.num_seqs, row);
  const int n = geo.p + 1;
  // dense: a row's own candidates bound its tiles
  const int tiles_total = (((P.dense && n < P.k) ? n : P.k) + kRows - 1) / kRows;
  const int t_begin = split * P.tiles_per_split;
  int t_end = t_begin + P.tiles_per_split;
  if (t_end > tiles_total) t_end = tiles_total;
  const int nt = t_end > t_begin ? t_end - t_begin : 0;
  const int32_t* __restrict__ idx_row = P.dense ? nullptr : P.idx + rrel * static_cast<int64_t>(P.k);
  // selected position of entry e of this row (-1: none)
  auto sel_at = [&](int e) -> int {
    if (P.dense) return e < n ? e : -1;
    return e < P.k ? __ldg(idx_row + e) : -1;
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(kv_full(s), kGatherThreads);
      mbar_init(kv_empty(s), 1);
    }
    mbar_init(qt_full, 128);
    mbar_init(qs_full, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(s_full(b), 1);
      mbar_init(s_empty(b), 128);
      mbar_init(p_full(b), 128);
      mbar_init(p_empty(b), 1);
    }
    mbar_init(o_ready, 1);
    for (int r = 0; r < 3; ++r) mbar_init(drain_bar(r), 1);
    *abort_flag = 0;
    fence_mbar_init();
    fence_proxy_async_smem();
    tma_prefetch_desc(&tm_q);
  }
  if (warp == kMmaWarp) tmem_alloc(smem_u32(tmem_slot), kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp >= 4 && warp < kMmaWarp) {
    // ------------------------------------------------------------ gather
    // Thread gt copies row i = gt / 8 of each tile, 16-byte chunks 8u + gt % 8
    // (u = 0..8), so each warp instruction covers four full 128-byte segments.
    // The selected position is loaded two tiles ahead; completion of a
    // thread's copies is tracked by the stage's mbarrier (no blocking wait).
    const int gt = threadIdx.x - 128;
    const int i = gt >> 3, t8 = gt & 7;
    auto load_idx = [&](int j) -> int {
      const int e = (t_begin + j) * kRows + i;
      return j < nt ? sel_at(e) : -1;
    };
    int s_cur = load_idx(0), s_next = load_idx(1);
    for (int j = 0; j < nt; ++j) {
      const int s = s_cur;
      s_cur = s_next;
      s_next = load_idx(j + 2);
      const int st = j % kStages;
      if (j >= kStages && !warp_wait(kv_empty(st), ((j / kStages) - 1) & 1, abort_flag)) break;
      const bool valid = s >= 0 && s < n;
      if (t8 == 0 && (s < -1 || s >= n)) flag_error(DSA_DEVERR_BAD_INDEX);
      const __nv_bfloat16* src = P.kv + (valid ? (geo.kv0 + s) * kDqk : 0) + t8 * 8;
      const uint32_t dst = sbase + kOffKV + st * kStageBytes + i * 128 + ((t8 ^ (i & 7)) << 4);
#pragma unroll
      for (int u = 0; u < kDqk / 64; ++u) cp_async_16(dst + u * kBlk, src + u * 64, valid ? 16u : 0u);
      cp_async_arrive_noinc(kv_full(st));
    }
    // no copy may still be in flight when the CTA exits
    cp_async_commit();
    cp_async_wait<0>();
  } else if (warp >= kMmaWarp) {
    // ------------------------------------------------------------ MMA issuers
    const int role = warp - kMmaWarp;   // 0: QK even tiles, 1: QK odd tiles, 2: PV
    if (lane == 0 && nt > 0) {
      if (role == 0) {
        mbar_arrive_expect_tx(qs_full, kQSmemBlocks * kQBlk);
        for (int b = 0; b < kQSmemBlocks; ++b)
          tma_load_2d(sbase + kOffQ + b * kQBlk, &tm_q, kQTmemD + b * 64, static_cast<int32_t>(row * kHeads),
                      qs_full);
      }
      bool ok = true;
      if (role < 2) {
        const uint32_t idesc_qk = make_idesc(1, 1, kHeads, kRows, 0, 0);
        ok = mbar_wait(qs_full, 0, abort_flag) && mbar_wait(qt_full, 0, abort_flag);
        const uint32_t sacc = tmem + kTmemS + role * kRows;
        // descriptors are formed once; a k-step adds its byte offset >> 4 to
        // the start-address field (all addresses stay below 2^18, so the
        // 14-bit field cannot overflow)
        const uint64_t kv_desc0 = make_desc(sbase + kOffKV, 16, 1024, kSwizzle128B);
        const uint64_t q_desc0 = make_desc(sbase + kOffQ, 16, 1024, kSwizzle128B);
        for (int j = role; j < nt && ok; j += 2) {
          const int st = j % kStages;
          if (!mbar_wait(kv_full(st), (j / kStages) & 1, abort_flag)) { ok = false; break; }
          if (j >= 2 && !mbar_wait(s_empty(role), ((j >> 1) - 1) & 1, abort_flag)) { ok = false; break; }
          tc_fence_after();
          // the tile was written by cp.async (generic proxy); the MMA reads it
          // through the async proxy
          fence_proxy_async_smem();
          const uint64_t bdesc0 = kv_desc0 + static_cast<uint64_t>((st * kStageBytes) >> 4);
#pragma unroll
          for (int g = 0; g < kKSteps; ++g) {
            const uint64_t bdesc = bdesc0 + static_cast<uint64_t>(((g >> 2) * kBlk + (g & 3) * 32) >> 4);
            if (g < kKStepsT) {
              mma_bf16_ta(sacc, tmem + kTmemQ + 8 * g, bdesc, idesc_qk, g > 0 ? 1u : 0u);
            } else {
              const int gs = g - kKStepsT;
              mma_bf16(sacc, q_desc0 + static_cast<uint64_t>(((gs >> 2) * kQBlk + (gs & 3) * 32) >> 4), bdesc,
                       idesc_qk, 1u);
            }
          }
          mma_commit(s_full(role));
        }
        drain_wait(qs_full, 0);
      } else {
        const uint32_t idesc_pv = make_idesc(1, 1, kHeads, kHalf, 0, 1);
        for (int j = 0; j < nt; ++j) {
          const int st = j % kStages, pb = j & 1;
          if (!mbar_wait(kv_full(st), (j / kStages) & 1, abort_flag)) break;
          if (!mbar_wait(p_full(pb), (j >> 1) & 1, abort_flag)) break;
          tc_fence_after();
          fence_proxy_async_smem();
          const uint32_t va = sbase + kOffKV + st * kStageBytes + (4 * half) * kBlk;
          const uint32_t pa = sbase + kOffP + pb * kPBytes;
#pragma unroll
          for (int ks = 0; ks < kRows / 16; ++ks)
            mma_bf16(tmem, make_desc(pa + ks * 32, 16, 512, kSwizzle64B),
                     make_desc(va + ks * 2048, kBlk, 1024, kSwizzle128B), idesc_pv, (j > 0 || ks > 0) ? 1u : 0u);
          mma_commit(p_empty(pb));
          mma_commit(kv_empty(st));
          mma_commit(o_ready);
        }
      }
      mma_commit(drain_bar(role));
      drain_wait(drain_bar(role), 0);
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int h = threadIdx.x;
    const uint32_t t_lane = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    bool ok = true;
    if (nt > 0) {
      // Q[:, 0:384] of head h into TMEM columns [320, 512), two bf16 per column
      const __nv_bfloat16* qh = P.q + (row * kHeads + h) * kDqk;
      // 128 columns of Q (256 bytes) per round: 16 loads in flight
#pragma unroll 1
      for (int c = 0; c < kQTmemD / 128; ++c) {
        uint32_t r0[32], r1[32];
#pragma unroll
        for (int v = 0; v < 8; ++v) {
          const uint4 x = ldg_nc_v4(qh + c * 128 + v * 8);
          const uint4 y = ldg_nc_v4(qh + c * 128 + 64 + v * 8);
          r0[4 * v] = x.x; r0[4 * v + 1] = x.y; r0[4 * v + 2] = x.z; r0[4 * v + 3] = x.w;
          r1[4 * v] = y.x; r1[4 * v + 1] = y.y; r1[4 * v + 2] = y.z; r1[4 * v + 3] = y.w;
        }
        tmem_st32(t_lane + kTmemQ + 64 * c, r0);
        tmem_st32(t_lane + kTmemQ + 64 * c + 32, r1);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(qt_full);
    }
    float m_use = -INFINITY, l = 0.f;
    auto load_sel = [&](int j) -> int {
      const int e = (t_begin + j) * kRows + lane;
      return j < nt ? sel_at(e) : -1;
    };
    int sel_next = load_sel(0);
    for (int j = 0; j < nt; ++j) {
      const int pb = j & 1;
      const int sel = sel_next;
      sel_next = load_sel(j + 1);
      const uint32_t mask = __ballot_sync(0xffffffffu, sel >= 0 && sel < n);
      if (!warp_wait(s_full(pb), (j >> 1) & 1, abort_flag)) { ok = false; break; }
      tc_fence_after();
      uint32_t a[32];
      tmem_ld32(t_lane + kTmemS + pb * kRows, a);
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(s_empty(pb));

      float z[kRows];
      float mt = -INFINITY;
#pragma unroll
      for (int i = 0; i < kRows; ++i) {
        z[i] = ((mask >> i) & 1u) ? __uint_as_float(a[i]) * P.c_log2 : -INFINITY;
        mt = fmaxf(mt, z[i]);
      }
      float alpha = 1.f;
      bool resc = false;
      if (mt > m_use + kRescaleThreshold) {
        if (m_use != -INFINITY) { alpha = ex2(m_use - mt); resc = true; }
        m_use = mt;
      }
      l *= alpha;
      uint32_t pk[kRows / 2];
      float lsum = 0.f;
#pragma unroll
      for (int i = 0; i < kRows; i += 2) {
        const float p0 = m_use == -INFINITY ? 0.f : ex2(z[i] - m_use);
        const float p1 = m_use == -INFINITY ? 0.f : ex2(z[i + 1] - m_use);
        pk[i >> 1] = pack_bf16(p0, p1);
        const __nv_bfloat162 r2 = *reinterpret_cast<const __nv_bfloat162*>(&pk[i >> 1]);
        lsum += __bfloat162float(r2.x) + __bfloat162float(r2.y);
      }
      l += lsum;

      if (j >= 2 && !warp_wait(p_empty(pb), ((j >> 1) - 1) & 1, abort_flag)) { ok = false; break; }
      // P row h: 64 bytes, 64-byte swizzle (16-byte chunk c at c ^ ((h >> 1) & 3))
      uint8_t* prow = smem + kOffP + pb * kPBytes + h * 64;
#pragma unroll
      for (int cc = 0; cc < 4; ++cc)
        *reinterpret_cast<uint4*>(prow + ((cc ^ ((h >> 1) & 3)) << 4)) =
            make_uint4(pk[4 * cc], pk[4 * cc + 1], pk[4 * cc + 2], pk[4 * cc + 3]);
      fence_proxy_async_smem();
      if (__any_sync(0xffffffffu, resc)) {
        // O must hold PV(j-1) before it is rescaled
        if (!warp_wait(o_ready, (j - 1) & 1, abort_flag)) { ok = false; break; }
        tc_fence_after();
#pragma unroll 1
        for (int c = 0; c < kHalf / 32; ++c) {
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
      tc_fence_before();
      mbar_arrive(p_full(pb));
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
      __nv_bfloat16* orow = P.out + (rrel * kHeads + h) * kDv + half * kHalf;
#pragma unroll 1
      for (int c = 0; c < kHalf / 32; ++c) {
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
      if (half == 0 && P.lse) P.lse[rrel * kHeads + h] = lse_v;
    } else {
      float* orow = P.part_o + (unit * kHeads + h) * kDv + half * kHalf;
#pragma unroll 1
      for (int c = 0; c < kHalf / 32; ++c) {
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
      if (half == 0) P.part_lse[unit * kHeads + h] = lse_v;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
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
