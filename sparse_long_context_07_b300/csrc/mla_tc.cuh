// Step 3 on the tensor cores: sparse MLA in MQA mode over the selected rows.
//
//   u_t[h] = sum_i softmax_i(scale * Q[t,h] . c_{s_i}) * c_{s_i}[0:d_v]
// over the selected positions s_i ("DeepSeek V3.2: How Far Can Open Models Go
// If You Actually Try?", §3.1: attention only over the top-k latents; MLA in
// MQA mode, one shared latent row per token read by all heads, §3.1 and §2.2).
// Dimensions: 128 heads, d_qk = 576, d_v = 512, bf16 in, fp32 accumulate.
//
// The fp32 output of one query token (128 heads x 512) would fill the whole
// TMEM of an SM, so a cluster of two CTAs serves each token, CTA r owning the
// output columns [256 r, 256 r + 256).  The 576-column scores of a tile of 64
// selected rows are split by rows: CTA r computes S for tile rows
// [32 r, 32 r + 32) over all 576 columns, and the two CTAs swap these halves
// through distributed shared memory, so no Q K^T product is computed twice.
// A half travels as its per-head maximum (fp32) and the differences to it
// (fp16, 64 bytes per head): with the maximum subtracted first, the fp16
// rounding of a difference d changes exp2(d) by at most about 3.4e-4
// relative for the scores near the maximum, well below the bf16 rounding of
// P, and the swap costs 8.5 KB per tile each way.  Both CTAs rebuild the 64
// scores of a head from the same maxima and differences, so they run the
// same softmax on identical values; each then accumulates its half of O with
// P V over all 64 rows.  The swap uses asynchronous stores whose completion
// is counted in bytes on the receiver's mbarrier, so no thread waits on the
// inter-SM path (tens of GB/s per SM on this part).
//
// TMEM (512 columns): O half [0, 256), the scores of the 32 own rows as two
// partial sums [256, 288) and [288, 320) (Q K^T is split over the k-steps
// between two issuing threads, which halves its latency), and Q[:, 0:384] as
// the A operand of Q K^T [320, 512) (two bf16 per column).  Q[:, 384:576]
// stays in shared memory, so Q K^T runs 24 k-steps with A in TMEM and 12 with
// A in shared memory.
//
// Shared memory holds the selected rows in two rings, filled together for a
// tile:
//   ring V (three stages of 32 KB): the value columns of this CTA's half,
//     [256 r, 256 r + 256), of all 64 rows -- the own rows first, then the
//     peer's rows.  B operand of P V (MN-major), and for the own rows also
//     part of the B operand of Q K^T.  Released by P V.
//   ring K (two stages of 20 KB): the other 320 columns of the own rows
//     (the peer's value half and the 64 rope columns), B operand of Q K^T
//     only.  Released by Q K^T.
// Every block is [32 rows x 64 columns] with the 128-byte swizzle.
// P (bf16, [128 heads x 64 rows], 128-byte swizzle) has a single buffer.
//
// Warp roles (608 threads):
//   warps 0-3    own-row softmax: thread h = head h = TMEM lane h.  Reads the
//                own scores, sends them to the peer, and computes P for the
//                own 32 rows of the tile
//   warps 15-18  peer-row softmax: the same heads (TMEM lane quarter =
//                warp % 4); computes P for the peer's 32 rows
//   warps 4-11   gather: 16-byte cp.async of the selected rows
//   warp 12      TMEM allocation; lane 0 loads Q[:, 384:576] with TMA and
//                issues one half of the k-steps of Q K^T
//   warp 13      lane 0 issues the other half of the k-steps of Q K^T
//   warp 14      lane 0 issues P V
// The two softmax roles hold identical running maxima (computed from the
// same values) and partial sums l that are added at the end.  The running
// max is updated lazily (only when a tile's max exceeds it by more than 2^8
// in the exp2 domain), so the O rescale in TMEM is rare; each role rescales
// half of the columns.
//
// Split-KV (decode): a cluster may take a contiguous range of tiles of a
// token; it then writes fp32 (O / l, lse) partials merged by combine_kernel.
//
// Dense mode (the baseline that sparse selection is measured against): no
// index list, every candidate 0..p of the row is attended, i.e. causal
// MLA-MQA attention over the whole context.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "common.cuh"
#include "ptx.cuh"

namespace dsa {
namespace mla_tc {

constexpr int kHeads = 128;
constexpr int kDqk = 576;
constexpr int kDv = 512;
constexpr int kHalf = 256;              // output columns per CTA
constexpr int kRows = 64;               // selected rows per tile
constexpr int kOwn = 32;                // rows of a tile whose scores a CTA computes (N of Q K^T)
constexpr int kQTmemD = 384;            // Q columns held in TMEM
constexpr int kQSmemBlocks = (kDqk - kQTmemD) / 64;  // 3 blocks of 64 columns
constexpr int kKStepsT = kQTmemD / 16;  // 24 k-steps with A in TMEM
constexpr int kKSteps = kDqk / 16;      // 36
constexpr int kBlk = kOwn * 128;                   // one [32 rows x 64 columns] block: 4 KiB
constexpr int kVStages = 3;
constexpr int kKStages = 2;
constexpr int kVStageBytes = 2 * (kHalf / 64) * kBlk;          // 32 KiB: own rows, then peer rows
constexpr int kKStageBytes = ((kDqk - kHalf) / 64) * kBlk;     // 20 KiB
constexpr int kQBlk = kHeads * 128;                // 16 KiB
constexpr int kPBytes = kHeads * kRows * 2;        // 16 KiB
constexpr int kXMaxOff = kHeads * kOwn * 2;        // fp16 differences, then the fp32 maxima
constexpr int kXBytes = kXMaxOff + kHeads * 4;     // 8.5 KiB per swapped half
constexpr int kGatherWarps = 8;
constexpr int kGatherThreads = 32 * kGatherWarps;
constexpr int kMmaWarp = 4 + kGatherWarps;   // first of the three issuing warps
constexpr int kPeerWarp = kMmaWarp + 3;      // first of the four peer-row softmax warps
constexpr int kThreads = 32 * (kPeerWarp + 4);
constexpr int kSoftmaxThreads = 256;
constexpr int kTmemCols = 512;
constexpr int kTmemS = 256;             // two partial score sums of kOwn columns
constexpr int kTmemQ = 320;
constexpr float kRescaleThreshold = 8.f;
static_assert(kTmemQ + kQTmemD / 2 == kTmemCols, "TMEM layout");
static_assert(kGatherThreads == 8 * kOwn, "gather: 8 threads per row");

constexpr int kOffV = 0;
constexpr int kOffK = kOffV + kVStages * kVStageBytes;
constexpr int kOffQ = kOffK + kKStages * kKStageBytes;
constexpr int kOffP = kOffQ + kQSmemBlocks * kQBlk;
constexpr int kOffX = kOffP + kPBytes;
constexpr int kOffMo = kOffX + 2 * kXBytes;        // own maxima of the last two tiles [2][128]
constexpr int kOffL = kOffMo + 2 * kHeads * 4;     // partial sums of the two roles [2][128]
constexpr int kOffBar = kOffL + 2 * kHeads * 4;
constexpr int kNumBars = kVStages + kKStages + kVStages + 17;
constexpr int kOutBox = kHeads * 128;   // one [128 heads x 64 columns] bf16 box of the output, 16 KiB
constexpr int kOffMisc = kOffBar + kNumBars * 8;
constexpr int kSmemBytes = kOffMisc + 16 + 1024;
static_assert(kOffQ % 1024 == 0 && kOffP % 1024 == 0 && kOffX % 16 == 0, "operand alignment");
static_assert(kSmemBytes <= 232448, "shared memory per CTA");
static_assert((kHalf / 64) * kOutBox <= kVStages * kVStageBytes, "output staging fits in ring V");

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
  int nsplit;                // clusters per query row
  int tiles_per_split;
  int64_t units;             // (row, split) units of this launch
  int64_t prefetch_ahead;    // >0: also prefetch the queries of unit + this into L2
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

__device__ __forceinline__ uint32_t pack_f16(float a, float b) {
  const __half2 v = __floats2half2_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&v);
}

__device__ __forceinline__ float2 unpack_f16(uint32_t u) {
  return __half22float2(*reinterpret_cast<const __half2*>(&u));
}

// Always 0 (x * 0 is +-0 or NaN, and both convert to integer 0), but computed
// from x, so an instruction that uses the result cannot issue before x is
// known; the compiler may not fold x * 0 for floats.
__device__ __forceinline__ uint32_t dep_zero(float x) {
  uint32_t r;
  asm volatile("{\n\t.reg .f32 t;\n\tmul.rn.f32 t, %1, 0f00000000;\n\tcvt.rzi.u32.f32 %0, t;\n\t}"
               : "=r"(r)
               : "f"(x));
  return r;
}

__device__ __forceinline__ uint4 ldg_nc_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    mla_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_out, const Params P) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // 1024-byte aligned base, derived by pointer arithmetic on the shared array
  // so that accesses through it stay shared-memory instructions
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + kOffBar;
  // full(s): both rings of a tile gathered (ring-V stage index s)
  auto full = [&](int s) { return bar0 + 8u * s; };
  auto k_empty = [&](int s) { return bar0 + 8u * (kVStages + s); };             // Q K^T done
  auto v_empty = [&](int s) { return bar0 + 8u * (kVStages + kKStages + s); };  // P V done
  constexpr int kB = 2 * kVStages + kKStages;
  const uint32_t qt_full = bar0 + 8u * kB;        // Q columns in TMEM (256 arrivals)
  const uint32_t qs_full = bar0 + 8u * (kB + 1);  // Q columns in smem (TMA)
  const uint32_t s_full = bar0 + 8u * (kB + 2);   // own scores ready (two issuers)
  const uint32_t s_empty = bar0 + 8u * (kB + 3);  // own scores read
  const uint32_t p_full = bar0 + 8u * (kB + 4);   // P written (both roles)
  const uint32_t p_empty = bar0 + 8u * (kB + 5);  // P V of the tile done (O current, P free)
  // x_full(b): the peer's score half of a tile of parity b is in X[b] (one
  // local arrival that arms the expected bytes, then the peer's asynchronous
  // stores); x_free(b): the peer has read the half we wrote into its X[b]
  // (256 remote arrivals); mo_full(b): the own maxima of that tile are in
  // shared memory for the peer-row role
  auto x_full = [&](int b) { return bar0 + 8u * (kB + 6 + b); };
  auto x_free = [&](int b) { return bar0 + 8u * (kB + 8 + b); };
  auto mo_full = [&](int b) { return bar0 + 8u * (kB + 10 + b); };
  auto drain_bar = [&](int r) { return bar0 + 8u * (kB + 12 + r); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();   // output half and own row half
  const uint32_t peer = rank ^ 1u;
  const int half = static_cast<int>(rank);

  // the work unit of this cluster: (query row, split)
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
  // selected position of tile row tr of tile j of this unit (-1: none)
  auto sel_at = [&](int j, int tr) -> int {
    if (j >= nt) return -1;
    const int e = (t_begin + j) * kRows + tr;
    if (P.dense) return e < n ? e : -1;
    return e < P.k ? __ldg(idx_row + e) : -1;
  };

  if (threadIdx.x == 0) {
    if (half == 0 && P.prefetch_ahead > 0) {
      // this token's queries into L2 ahead of their loads, and the queries
      // of the token that will likely run next on this SM pair (a wave of
      // the grid later)
      if (nt > 0) prefetch_l2_bulk(P.q + row * kHeads * kDqk, kHeads * kDqk * 2);
      const int64_t nu = unit + P.prefetch_ahead;
      if (nu < P.units) prefetch_l2_bulk(P.q + (P.row0 + nu / P.nsplit) * kHeads * kDqk, kHeads * kDqk * 2);
    }
    for (int s = 0; s < kVStages; ++s) {
      mbar_init(full(s), kGatherThreads);
      mbar_init(v_empty(s), 1);
    }
    for (int s = 0; s < kKStages; ++s) mbar_init(k_empty(s), 2);
    mbar_init(qt_full, kSoftmaxThreads);
    mbar_init(qs_full, 1);
    mbar_init(s_full, 2);
    mbar_init(s_empty, 128);
    mbar_init(p_full, kSoftmaxThreads);
    mbar_init(p_empty, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(x_full(b), 1);
      mbar_init(x_free(b), kSoftmaxThreads);
      mbar_init(mo_full(b), 128);
    }
    for (int r = 0; r < 3; ++r) mbar_init(drain_bar(r), 1);
    *abort_flag = 0;
    fence_mbar_init();
    // arm the swap buffers for tiles 0 and 1
    for (int b = 0; b < 2; ++b) mbar_arrive_expect_tx(x_full(b), kXBytes);
    fence_proxy_async_smem();
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_out);
  }
  if (warp == kMmaWarp) tmem_alloc(smem_u32(tmem_slot), kTmemCols);
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // the peer's barriers are initialised before any remote arrival
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp >= 4 && warp < kMmaWarp) {
    // ------------------------------------------------------------ gather
    // Thread gt copies 16-byte chunk t8 = gt % 8 of every 64-column block of
    // own row i = gt / 8 (tile row 32 rank + i) and of the value blocks of
    // peer row i (tile row 32 peer + i), so each warp instruction covers four
    // full 128-byte segments.  The selected positions are loaded two tiles
    // ahead; completion is tracked by the tile's mbarrier.
    const int gt = threadIdx.x - 128;
    const int i = gt >> 3, t8 = gt & 7;
    const int tr_own = kOwn * half + i, tr_peer = kOwn * static_cast<int>(peer) + i;
    griddep_wait();   // the index lists may come from the kernel before this one
    int so_cur = sel_at(0, tr_own), sp_cur = sel_at(0, tr_peer);
    int so_next = sel_at(1, tr_own), sp_next = sel_at(1, tr_peer);
    const uint32_t swz = i * 128 + ((t8 ^ (i & 7)) << 4);
    for (int j = 0; j < nt; ++j) {
      const int so = so_cur, sp = sp_cur;
      so_cur = so_next;
      sp_cur = sp_next;
      so_next = sel_at(j + 2, tr_own);
      sp_next = sel_at(j + 2, tr_peer);
      const int sv = j % kVStages, sk = j & 1;
      if (j >= kKStages && !warp_wait(k_empty(sk), ((j >> 1) - 1) & 1, abort_flag)) break;
      if (j >= kVStages && !warp_wait(v_empty(sv), ((j / kVStages) - 1) & 1, abort_flag)) break;
      const uint32_t vst = sbase + kOffV + sv * kVStageBytes + swz;
      const uint32_t kst = sbase + kOffK + sk * kKStageBytes + swz;
      {
        const bool valid = so >= 0 && so < n;
        if (t8 == 0 && (so < -1 || so >= n)) flag_error(DSA_DEVERR_BAD_INDEX);
        const __nv_bfloat16* src = P.kv + (valid ? (geo.kv0 + so) * kDqk : 0) + t8 * 8;
        const uint32_t bytes = valid ? 16u : 0u;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          // value blocks of this half go to ring V, the others to ring K
          const uint32_t dst = ((u >> 2) == half ? vst : kst) + (u & 3) * kBlk;
          cp_async_16(dst, src + u * 64, bytes);
        }
        cp_async_16(kst + 4 * kBlk, src + 8 * 64, bytes);
      }
      {
        const bool valid = sp >= 0 && sp < n;
        if (t8 == 0 && (sp < -1 || sp >= n)) flag_error(DSA_DEVERR_BAD_INDEX);
        const __nv_bfloat16* src = P.kv + (valid ? (geo.kv0 + sp) * kDqk : 0) + half * kHalf + t8 * 8;
        const uint32_t bytes = valid ? 16u : 0u;
#pragma unroll
        for (int u = 0; u < 4; ++u) cp_async_16(vst + (4 + u) * kBlk, src + u * 64, bytes);
      }
      cp_async_arrive_noinc(full(sv));
    }
    // no copy may still be in flight when the CTA exits
    cp_async_commit();
    cp_async_wait<0>();
  } else if (warp >= kMmaWarp && warp < kPeerWarp) {
    // ------------------------------------------------------------ MMA issuers
    const int role = warp - kMmaWarp;   // 0, 1: the two halves of Q K^T; 2: P V
    if (lane == 0 && nt > 0) {
      if (role == 0) {
        mbar_arrive_expect_tx(qs_full, kQSmemBlocks * kQBlk);
        for (int b = 0; b < kQSmemBlocks; ++b)
          tma_load_2d(sbase + kOffQ + b * kQBlk, &tm_q, kQTmemD + b * 64, static_cast<int32_t>(row * kHeads),
                      qs_full);
      }
      if (role < 2) {
        // issuer `role` takes k-steps [12 role, 12 role + 12) (A in TMEM) and
        // [24 + 6 role, 30 + 6 role) (A in shared memory) into its own
        // partial sum
        const uint32_t idesc_qk = make_idesc(1, 1, kHeads, kOwn, 0, 0);
        bool ok = mbar_wait(qs_full, 0, abort_flag) && mbar_wait(qt_full, 0, abort_flag);
        const uint32_t sacc = tmem + kTmemS + role * kOwn;
        const uint64_t q_desc0 = make_desc(sbase + kOffQ, 16, 1024, kSwizzle128B);
        for (int j = 0; j < nt && ok; ++j) {
          const int sv = j % kVStages;
          if (!mbar_wait(full(sv), (j / kVStages) & 1, abort_flag)) break;
          if (j >= 1 && !mbar_wait(s_empty, (j - 1) & 1, abort_flag)) break;
          tc_fence_after();
          // the rows were written by cp.async (generic proxy); the MMA reads
          // them through the async proxy
          fence_proxy_async_smem();
          const uint32_t vst = sbase + kOffV + sv * kVStageBytes;
          const uint32_t kst = sbase + kOffK + (j & 1) * kKStageBytes;
          // descriptor of 64-column block u of the own rows; a k-step adds
          // its byte offset >> 4 to the start-address field (addresses stay
          // below 2^18, so the 14-bit field cannot overflow)
          auto bdesc = [&](int g) -> uint64_t {
            const int u = g >> 2;
            const uint32_t a = u < 8 ? ((u >> 2) == half ? vst : kst) + (u & 3) * kBlk : kst + 4 * kBlk;
            return make_desc(a + (g & 3) * 32, 16, 1024, kSwizzle128B);
          };
#pragma unroll
          for (int t = 0; t < 12; ++t) {
            const int g = 12 * role + t;
            mma_bf16_ta(sacc, tmem + kTmemQ + 8 * g, bdesc(g), idesc_qk, t > 0 ? 1u : 0u);
          }
#pragma unroll
          for (int t = 0; t < 6; ++t) {
            const int gs = 6 * role + t;
            mma_bf16(sacc, q_desc0 + static_cast<uint64_t>(((gs >> 2) * kQBlk + (gs & 3) * 32) >> 4),
                     bdesc(kKStepsT + gs), idesc_qk, 1u);
          }
          mma_commit(s_full);
          mma_commit(k_empty(j & 1));
        }
        drain_wait(qs_full, 0);
      } else {
        const uint32_t idesc_pv = make_idesc(1, 1, kHeads, kHalf, 0, 1);
        const uint32_t pa = sbase + kOffP;
        for (int j = 0; j < nt; ++j) {
          const int sv = j % kVStages;
          if (!mbar_wait(full(sv), (j / kVStages) & 1, abort_flag)) break;
          if (!mbar_wait(p_full, j & 1, abort_flag)) break;
          tc_fence_after();
          fence_proxy_async_smem();
          // tile rows 32 r .. 32 r + 31 are CTA r's own rows: k-steps 0, 1
          // take tile rows 0..31, k-steps 2, 3 rows 32..63
          const uint32_t v_own = sbase + kOffV + sv * kVStageBytes;
          const uint32_t v_peer = v_own + (kHalf / 64) * kBlk;
#pragma unroll
          for (int ks = 0; ks < kRows / 16; ++ks) {
            const bool own = (ks >> 1) == half;
            mma_bf16(tmem, make_desc(pa + ks * 32, 16, 1024, kSwizzle128B),
                     make_desc((own ? v_own : v_peer) + (ks & 1) * 2048, kBlk, 1024, kSwizzle128B), idesc_pv,
                     (j > 0 || ks > 0) ? 1u : 0u);
          }
          mma_commit(p_empty);
          mma_commit(v_empty(sv));
        }
      }
      mma_commit(drain_bar(role));
      drain_wait(drain_bar(role), 0);
    }
  } else {
    // ------------------------------------------------------------ softmax
    // sr = 0: own rows (warps 0-3); sr = 1: peer rows (warps 15-18)
    const int sr = warp < 4 ? 0 : 1;
    const int quarter = warp & 3;
    const int h = 32 * quarter + lane;
    const uint32_t t_lane = tmem + (static_cast<uint32_t>(32 * quarter) << 16);
    const uint32_t x_full_peer0 = mapa_shared(x_full(0), peer);
    const uint32_t x_free_peer0 = mapa_shared(x_free(0), peer);
    // head h's 64 bytes of differences: 16-byte chunk c at c ^ ((h >> 1) & 3)
    const uint32_t x_row = h * 64;
    const int xsw = (h >> 1) & 3;
    float* mo_s = reinterpret_cast<float*>(smem + kOffMo);
    float* l_s = reinterpret_cast<float*>(smem + kOffL);
    // this role's tile rows: 32 rank + t (own) or 32 peer + t; their bytes in
    // a P row are [64 tr, 64 tr + 64), i.e. 16-byte chunks 4 tr .. 4 tr + 3
    const int ptr = sr == 0 ? half : static_cast<int>(peer);
    bool ok = true;
    if (nt > 0) {
      // Q[:, 192 sr : 192 sr + 192] of head h into TMEM, two bf16 per column
      const __nv_bfloat16* qh = P.q + (row * kHeads + h) * kDqk + 192 * sr;
#pragma unroll 1
      for (int c = 0; c < 3; ++c) {
        uint32_t r0[32];
#pragma unroll
        for (int v = 0; v < 8; ++v) {
          const uint4 x = ldg_nc_v4(qh + c * 64 + v * 8);
          r0[4 * v] = x.x; r0[4 * v + 1] = x.y; r0[4 * v + 2] = x.z; r0[4 * v + 3] = x.w;
        }
        tmem_st32(t_lane + kTmemQ + 96 * sr + 32 * c, r0);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(qt_full);
    }
    float m_use = -INFINITY, l = 0.f;
    griddep_wait();   // (the queries above are inputs of the call; the index lists are not)
    int sel_own = sr == 0 ? sel_at(0, kOwn * half + lane) : -1;
    for (int j = 0; j < nt; ++j) {
      const int xb = j & 1;
      uint32_t d[kOwn / 2];   // fp16 differences of this role's rows
      float mine, other;      // tile maxima: own rows, peer rows
      if (sr == 0) {
        // ---- own rows: read, encode, publish, send
        const uint32_t vmask = __ballot_sync(0xffffffffu, sel_own >= 0 && sel_own < n);
        sel_own = sel_at(j + 1, kOwn * half + lane);
        if (!warp_wait(s_full, j & 1, abort_flag)) { ok = false; break; }
        tc_fence_after();
        float z[kOwn];
        {
          uint32_t sa[kOwn], sb[kOwn];
          tmem_ld32(t_lane + kTmemS, sa);
          tmem_ld32(t_lane + kTmemS + kOwn, sb);
          tmem_wait_ld();
          tc_fence_before();
          mbar_arrive(s_empty);
#pragma unroll
          for (int t = 0; t < kOwn; ++t)
            z[t] = ((vmask >> t) & 1u) ? (__uint_as_float(sa[t]) + __uint_as_float(sb[t])) * P.c_log2 : -INFINITY;
        }
        float mo = -INFINITY;
#pragma unroll
        for (int t = 0; t < kOwn; ++t) mo = fmaxf(mo, z[t]);
        const float mref = mo == -INFINITY ? 0.f : mo;
#pragma unroll
        for (int t = 0; t < kOwn; t += 2) d[t >> 1] = pack_f16(z[t] - mref, z[t + 1] - mref);
        mo_s[xb * kHeads + h] = mo;
        mbar_arrive(mo_full(xb));
        // the peer must have read what we sent into its X[xb] two tiles ago
        if (j >= 2 && !warp_wait<true>(x_free(xb), ((j >> 1) - 1) & 1, abort_flag)) { ok = false; break; }
        const uint32_t dst = mapa_shared(sbase + kOffX + xb * kXBytes, peer);
        const uint32_t xbar = x_full_peer0 + 8u * xb;
#pragma unroll
        for (int c = 0; c < 4; ++c)
          st_async_v4(dst + x_row + ((c ^ xsw) << 4), d[4 * c], d[4 * c + 1], d[4 * c + 2], d[4 * c + 3], xbar);
        st_async_b32(dst + kXMaxOff + h * 4, __float_as_uint(mo), xbar);
        mine = mo;
        if (!warp_wait<true>(x_full(xb), (j >> 1) & 1, abort_flag)) { ok = false; break; }
        other = *reinterpret_cast<const float*>(smem + kOffX + xb * kXBytes + kXMaxOff + h * 4);
      } else {
        // ---- peer rows: wait for the swapped half and the own maxima
        if (!warp_wait<true>(x_full(xb), (j >> 1) & 1, abort_flag)) { ok = false; break; }
        const uint8_t* xs = smem + kOffX + xb * kXBytes;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const uint4 v = *reinterpret_cast<const uint4*>(xs + x_row + ((c ^ xsw) << 4));
          d[4 * c] = v.x; d[4 * c + 1] = v.y; d[4 * c + 2] = v.z; d[4 * c + 3] = v.w;
        }
        other = *reinterpret_cast<const float*>(xs + kXMaxOff + h * 4);
        // X[xb] is complete for tile j; arm it for tile j + 2 (the peer sends
        // that tile only after all 256 softmax threads here have read this one)
        if (h == 0) mbar_arrive_expect_tx(x_full(xb), kXBytes);
        if (!warp_wait(mo_full(xb), (j >> 1) & 1, abort_flag)) { ok = false; break; }
        mine = mo_s[xb * kHeads + h];
      }
      // ---- both roles: identical running max, P for this role's 32 rows
      const float mrow = sr == 0 ? mine : other;   // maximum the differences refer to
      const float mt = fmaxf(mine, other);
      float alpha = 1.f;
      bool resc = false;
      if (mt > m_use + kRescaleThreshold) {
        if (m_use != -INFINITY) { alpha = ex2(m_use - mt); resc = true; }
        m_use = mt;
      }
      l *= alpha;
      uint32_t pk[kOwn / 2];
      float lsum = 0.f;
#pragma unroll
      for (int t = 0; t < kOwn / 2; ++t) {
        const float2 dd = unpack_f16(d[t]);
        // the score is rebuilt as m + d in both CTAs before the exponent
        const float p0 = m_use == -INFINITY ? 0.f : ex2((mrow + dd.x) - m_use);
        const float p1 = m_use == -INFINITY ? 0.f : ex2((mrow + dd.y) - m_use);
        pk[t] = pack_bf16(p0, p1);
        const __nv_bfloat162 r2 = *reinterpret_cast<const __nv_bfloat162*>(&pk[t]);
        lsum += __bfloat162float(r2.x) + __bfloat162float(r2.y);
      }
      l += lsum;
      // X[xb] may be written again.  The arrive is relaxed; its address
      // carries a data dependency on lsum (and, for the own-row role, on the
      // peer maximum it read), so it cannot issue before the reads of X[xb]
      // have completed.
      mbar_arrive_cluster_relaxed(x_free_peer0 + 8u * xb + dep_zero(lsum + other));
      // P V of the previous tile must be done: it reads the P buffer, and O
      // must hold it before a rescale
      if (j >= 1 && !warp_wait(p_empty, (j - 1) & 1, abort_flag)) { ok = false; break; }
      tc_fence_after();
      // P row h: 128 bytes, 128-byte swizzle (16-byte chunk c at c ^ (h & 7))
      uint8_t* prow = smem + kOffP + h * 128;
#pragma unroll
      for (int cc = 0; cc < 4; ++cc)
        *reinterpret_cast<uint4*>(prow + (((4 * ptr + cc) ^ (h & 7)) << 4)) =
            make_uint4(pk[4 * cc], pk[4 * cc + 1], pk[4 * cc + 2], pk[4 * cc + 3]);
      fence_proxy_async_smem();
      if (__any_sync(0xffffffffu, resc)) {
        // each role rescales half of the O columns
#pragma unroll 1
        for (int c = 0; c < kHalf / 64; ++c) {
          uint32_t o[32];
          const uint32_t col = 128 * sr + 32 * c;
          tmem_ld32(t_lane + col, o);
          tmem_wait_ld();
#pragma unroll
          for (int u = 0; u < 32; ++u) o[u] = __float_as_uint(__uint_as_float(o[u]) * alpha);
          tmem_st32(t_lane + col, o);
        }
        tmem_wait_st();
      }
      tc_fence_before();
      mbar_arrive(p_full);
    }

    // ---- epilogue: O / l (and lse); each role writes half of the columns
    // the softmax of tile nt-1 waited for P V of tile nt-2, so the barrier is
    // at most one phase behind and the parity wait is exact
    l_s[sr * kHeads + h] = l;
    named_bar_sync(1, kSoftmaxThreads);
    const float lt = l + l_s[(sr ^ 1) * kHeads + h];
    bool have_o = ok && nt > 0;
    if (have_o) have_o = warp_wait(p_empty, (nt - 1) & 1, abort_flag);
    tc_fence_after();
    const float inv = lt > 0.f ? 1.f / lt : 0.f;
    const float lse_v = lt > 0.f ? (m_use + __log2f(lt)) * 0.6931471805599453f : -INFINITY;
    if (P.nsplit == 1) {
      // O / l in bf16 into the freed ring V as four [128 heads x 64 columns]
      // boxes with the 128-byte swizzle (every copy and MMA of the tile loop
      // has completed: P V of the last tile was waited for), then TMA stores
      // of the CTA's 256 output columns
      uint8_t* ob = smem + kOffV;
#pragma unroll 1
      for (int c = 0; c < kHalf / 64; ++c) {
        uint32_t o[32];
        if (have_o) { tmem_ld32(t_lane + 128 * sr + 32 * c, o); tmem_wait_ld(); }
        else {
#pragma unroll
          for (int u = 0; u < 32; ++u) o[u] = 0u;
        }
        const int col = 128 * sr + 32 * c;   // column within this CTA's half
        uint8_t* rowp = ob + (col >> 6) * kOutBox + h * 128;
        const int ch0 = (col & 63) >> 3;
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          uint4 pk4;
          pk4.x = pack_bf16(__uint_as_float(o[8 * v + 0]) * inv, __uint_as_float(o[8 * v + 1]) * inv);
          pk4.y = pack_bf16(__uint_as_float(o[8 * v + 2]) * inv, __uint_as_float(o[8 * v + 3]) * inv);
          pk4.z = pack_bf16(__uint_as_float(o[8 * v + 4]) * inv, __uint_as_float(o[8 * v + 5]) * inv);
          pk4.w = pack_bf16(__uint_as_float(o[8 * v + 6]) * inv, __uint_as_float(o[8 * v + 7]) * inv);
          *reinterpret_cast<uint4*>(rowp + (((ch0 + v) ^ (h & 7)) << 4)) = pk4;
        }
      }
      fence_proxy_async_smem();
      named_bar_sync(1, kSoftmaxThreads);
      if (threadIdx.x == 0) {
#pragma unroll
        for (int b = 0; b < kHalf / 64; ++b)
          tma_store_2d(&tm_out, half * kHalf + 64 * b, static_cast<int32_t>(rrel * kHeads), sbase + kOffV + b * kOutBox);
        bulk_commit();
        bulk_wait_read();   // the staging buffer is read before the CTA may exit
      }
      if (half == 0 && sr == 0 && P.lse) P.lse[rrel * kHeads + h] = lse_v;
    } else {
      float* orow = P.part_o + (unit * kHeads + h) * kDv + half * kHalf + 128 * sr;
#pragma unroll 1
      for (int c = 0; c < kHalf / 64; ++c) {
        uint32_t o[32];
        if (have_o) { tmem_ld32(t_lane + 128 * sr + 32 * c, o); tmem_wait_ld(); }
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
      if (half == 0 && sr == 0) P.part_lse[unit * kHeads + h] = lse_v;
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();  // no remote access may target an exited CTA
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
