// C ABI of the DSA forward library (declared in include/dsa.h): argument
// validation, tensor-map encoding, launch configuration and the chunked
// forward scheduler.  All kernels live in the headers included below; this is
// the only translation unit of libdsa.so.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>

#include "nvtx3/nvToolsExt.h"

#include "dsa.h"
#include "common.cuh"
#include "indexer_tc.cuh"
#include "kl.cuh"
#include "mla_tc.cuh"
#include "quant.cuh"
#include "ptx.cuh"
#include "simt.cuh"
#include "topk.cuh"

namespace {

thread_local std::string g_last_msg;

// NVTX ranges (for timeline tools) around the entry points, the query chunks
// of the forward and every kernel launch, when the environment sets
// DSA_NVTX=1 (read once per process).  Without a tool attached a range is a
// no-op call.
bool nvtx_on() {
  static const bool on = [] {
    const char* v = std::getenv("DSA_NVTX");
    return v != nullptr && v[0] == '1';
  }();
  return on;
}

struct NvtxRange {
  const bool on;
  explicit NvtxRange(const char* name) : on(nvtx_on()) {
    if (on) nvtxRangePushA(name);
  }
  ~NvtxRange() {
    if (on) nvtxRangePop();
  }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

dsa_status_t fail(dsa_status_t st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_msg = buf;
  return st;
}

#define DSA_TRY(expr)                          \
  do {                                         \
    const dsa_status_t st_ = (expr);           \
    if (st_ != DSA_SUCCESS) return st_;        \
  } while (0)

// ---------------------------------------------------------------------------
// Device facts, cached per device
// ---------------------------------------------------------------------------
constexpr int kMaxDevices = 64;
struct DeviceInfo {
  bool ready = false;
  bool ok = false;
  int sms = 0;
  int smem_optin = 0;
  bool attrs_set = false;
};
DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

std::atomic<uint32_t> g_fault_next{0};

dsa_status_t device_info(DeviceInfo** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return fail(DSA_ERROR_DEVICE, "no current CUDA device");
  if (dev < 0 || dev >= kMaxDevices) return fail(DSA_ERROR_DEVICE, "device index %d out of range", dev);
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DeviceInfo& d = g_dev[dev];
  if (!d.ready) {
    int major = 0, minor = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
    cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    d.ok = (major == 10 && minor == 3);
    d.ready = true;
    if (!g_encode) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                           &q) == cudaSuccess &&
          q == cudaDriverEntryPointSuccess)
        g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
  }
  if (!d.ok) return fail(DSA_ERROR_DEVICE, "device %d is not an sm_103 (B300) GPU", dev);
  if (!g_encode) return fail(DSA_ERROR_DEVICE, "cuTensorMapEncodeTiled unavailable");
  if (!d.attrs_set) {
    if (cudaFuncSetAttribute(dsa::idx_tc::indexer_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             dsa::idx_tc::kSmemBytes) != cudaSuccess ||
        cudaFuncSetAttribute(dsa::idx_tc::indexer_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             dsa::idx_tc::kSmemBytes) != cudaSuccess ||
        cudaFuncSetAttribute(dsa::mla_tc::mla_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             dsa::mla_tc::kSmemBytes) != cudaSuccess ||
        cudaFuncSetAttribute(dsa::topk::topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             dsa::topk::kSmemBytes) != cudaSuccess ||
        cudaFuncSetAttribute(dsa::topk::topk_cluster_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             dsa::topk::kCSmemBytes) != cudaSuccess)
      return fail(DSA_ERROR_LAUNCH, "cudaFuncSetAttribute failed: %s",
                  cudaGetErrorString(cudaGetLastError()));
    d.attrs_set = true;
  }
  *out = &d;
  return DSA_SUCCESS;
}

dsa_status_t encode_2d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner,
                       uint64_t outer, uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer) {
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = g_encode(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(DSA_ERROR_INVALID_VALUE, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return DSA_SUCCESS;
}

// ---------------------------------------------------------------------------
// Launch trace
// ---------------------------------------------------------------------------
struct Tracer {
  dsa_trace_t* t;
  cudaStream_t s;
  bool broken = false;  // an event could not be recorded: stop tracing
  void record() {
    if (cudaEventRecord(t->events[t->count], s) != cudaSuccess) {
      cudaGetLastError();  // do not leave a sticky error for the next launch check
      broken = true;
      return;
    }
    ++t->count;
  }
  dsa_status_t begin() {
    if (t && t->events && t->count == 0 && t->capacity > 0) {
      record();
      if (broken) return fail(DSA_ERROR_INVALID_VALUE, "trace: cudaEventRecord failed on events[0]");
    }
    return DSA_SUCCESS;
  }
  void after(int kernel_id) {
    if (broken || !t || !t->events || t->count <= 0 || t->count >= t->capacity) return;
    if (t->kernel_ids) t->kernel_ids[t->count - 1] = kernel_id;
    record();
  }
};

dsa_status_t check_launch(const char* what) {
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(DSA_ERROR_LAUNCH, "%s launch failed: %s", what, cudaGetErrorString(e));
  return DSA_SUCCESS;
}

// ---------------------------------------------------------------------------
// Validation
// ---------------------------------------------------------------------------
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

dsa_status_t check_batch(const dsa_batch_t* b) {
  if (!b) return fail(DSA_ERROR_INVALID_VALUE, "batch is NULL");
  if (b->num_seqs < 1) return fail(DSA_ERROR_INVALID_VALUE, "num_seqs must be >= 1 (got %d)", b->num_seqs);
  if (!b->cu_seqlens_q || !b->cu_seqlens_kv) return fail(DSA_ERROR_INVALID_VALUE, "cu_seqlens pointer is NULL");
  if (b->total_q < 0 || b->total_kv < 0 || b->total_kv < b->total_q)
    return fail(DSA_ERROR_INVALID_VALUE, "totals must satisfy 0 <= total_q <= total_kv");
  if (b->max_seqlen_q < 0 || b->max_seqlen_kv < b->max_seqlen_q)
    return fail(DSA_ERROR_INVALID_VALUE, "max_seqlen_kv must be >= max_seqlen_q >= 0");
  if (b->total_q > 0 && (b->max_seqlen_q < 1 || b->max_seqlen_kv < 1))
    return fail(DSA_ERROR_INVALID_VALUE, "max_seqlen hints must be >= 1 for a non-empty batch");
  if (b->total_kv >= (int64_t(1) << 31) || b->total_q >= (int64_t(1) << 24))
    return fail(DSA_ERROR_NOT_SUPPORTED, "total_kv must be < 2^31 and total_q < 2^24");
  return DSA_SUCCESS;
}

bool indexer_is_tc(const dsa_indexer_t* ix) {
  return ix->dtype == DSA_DTYPE_E4M3 && ix->n_heads == dsa::idx_tc::kHeads &&
         ix->head_dim == dsa::idx_tc::kDim;
}

// Tensor pointers may be NULL only when the batch has no rows to read.
dsa_status_t check_indexer(const dsa_indexer_t* ix, const dsa_batch_t* b) {
  if (!ix) return fail(DSA_ERROR_INVALID_VALUE, "indexer is NULL");
  if ((b->total_q > 0 && (!ix->q || !ix->w)) || (b->total_kv > 0 && !ix->k))
    return fail(DSA_ERROR_INVALID_VALUE, "indexer q, k and w are required");
  if (!aligned16(ix->q) || !aligned16(ix->k) || !aligned16(ix->w) ||
      (ix->q_scale && !aligned16(ix->q_scale)) || (ix->k_scale && !aligned16(ix->k_scale)))
    return fail(DSA_ERROR_INVALID_VALUE, "indexer tensors must be 16-byte aligned");
  if (ix->dtype != DSA_DTYPE_E4M3 && ix->dtype != DSA_DTYPE_F32)
    return fail(DSA_ERROR_NOT_SUPPORTED, "indexer dtype must be E4M3 or F32");
  if (ix->n_heads < 1 || ix->n_heads > dsa::simt::kMaxIdxHeads || ix->head_dim < 16 ||
      ix->head_dim > dsa::simt::kMaxIdxDim || ix->head_dim % 16 != 0)
    return fail(DSA_ERROR_NOT_SUPPORTED, "indexer needs 1 <= n_heads <= 64 and head_dim in {16, 32, ..., 128}");
  return DSA_SUCCESS;
}

bool mla_is_tc(const dsa_mla_t* m) {
  return m->dtype == DSA_DTYPE_BF16 && m->n_heads == dsa::mla_tc::kHeads && m->d_qk == dsa::mla_tc::kDqk &&
         m->d_v == dsa::mla_tc::kDv;
}

dsa_status_t check_mla(const dsa_mla_t* m, const dsa_batch_t* b) {
  if (!m) return fail(DSA_ERROR_INVALID_VALUE, "mla is NULL");
  if ((b->total_q > 0 && !m->q) || (b->total_kv > 0 && !m->kv))
    return fail(DSA_ERROR_INVALID_VALUE, "mla q and kv are required");
  if (!aligned16(m->q) || !aligned16(m->kv)) return fail(DSA_ERROR_INVALID_VALUE, "mla tensors must be 16-byte aligned");
  if (m->dtype != DSA_DTYPE_BF16 && m->dtype != DSA_DTYPE_F32)
    return fail(DSA_ERROR_NOT_SUPPORTED, "mla dtype must be BF16 or F32");
  if (m->n_heads < 1 || m->d_qk < 1 || m->d_v < 1 || m->d_v > m->d_qk || m->d_qk > dsa::simt::kMaxMlaDim)
    return fail(DSA_ERROR_NOT_SUPPORTED, "mla needs n_heads >= 1 and 1 <= d_v <= d_qk <= 1024");
  if (!std::isfinite(m->scale)) return fail(DSA_ERROR_INVALID_VALUE, "mla scale must be finite");
  return DSA_SUCCESS;
}

dsa_status_t check_k(int32_t k) {
  if (k < 1 || k > 16384) return fail(DSA_ERROR_INVALID_VALUE, "k must be in [1, 16384] (got %d)", k);
  return DSA_SUCCESS;
}

// ---------------------------------------------------------------------------
// Per-step launchers over query rows [r0, r1).  Output/intermediate pointers
// (scores, idx, vals, out, lse) already point at row r0.
// ---------------------------------------------------------------------------
// hist (optional, tensor-core indexer only): [r1 - r0][2048] zeroed first-digit
// histograms that the indexer fills for the top-k.
dsa_status_t launch_index_scores(const DeviceInfo& dev, const dsa_batch_t* b, const dsa_indexer_t* ix,
                                 float* scores, int64_t ld, int64_t r0, int64_t r1, cudaStream_t s,
                                 Tracer& tr, uint32_t* hist = nullptr) {
  const int64_t rows = r1 - r0;
  if (rows <= 0) return DSA_SUCCESS;
  NvtxRange nvtx("dsa: indexer");
  if (indexer_is_tc(ix)) {
    CUtensorMap tm_q, tm_k;
    DSA_TRY(encode_2d(&tm_q, CU_TENSOR_MAP_DATA_TYPE_UINT8, ix->q, dsa::idx_tc::kDim,
                      static_cast<uint64_t>(b->total_q) * dsa::idx_tc::kHeads, dsa::idx_tc::kDim,
                      dsa::idx_tc::kDim, dsa::idx_tc::kHeads));
    DSA_TRY(encode_2d(&tm_k, CU_TENSOR_MAP_DATA_TYPE_UINT8, ix->k, dsa::idx_tc::kDim,
                      static_cast<uint64_t>(b->total_kv), dsa::idx_tc::kDim, dsa::idx_tc::kDim,
                      dsa::idx_tc::kKeys));
    dsa::idx_tc::Params P{};
    P.q_scale = ix->q_scale;
    P.k_scale = ix->k_scale;
    P.w = ix->w;
    P.scores = scores;
    P.ld = ld;
    P.hist = hist;
    P.cu_q = b->cu_seqlens_q;
    P.cu_kv = b->cu_seqlens_kv;
    P.num_seqs = b->num_seqs;
    P.row_begin = r0;
    P.row_end = r1;
    P.group = dsa::idx_tc::kMaxTokens;
    P.fault = g_fault_next.exchange(0);
    if (b->max_seqlen_q == 1) {
      // decode: one token per sequence; split long key ranges so every SM
      // works.  CTAs take items round-robin, so items of about 16 tiles
      // (16 per SM) keep the last round short; smaller ones cost more in
      // per-item start-up than they save.
      const int64_t tiles = (b->total_kv + dsa::idx_tc::kKeys - 1) / dsa::idx_tc::kKeys + b->num_seqs;
      const int64_t target = 16ll * dev.sms;
      P.max_tiles = static_cast<int>(std::max<int64_t>(8, (tiles + target - 1) / target));
    } else {
      P.max_tiles = 1 << 24;
    }
    const int grid = dev.sms;
    if (hist)
      dsa::idx_tc::indexer_kernel<true><<<grid, dsa::idx_tc::kThreads, dsa::idx_tc::kSmemBytes, s>>>(tm_q, tm_k, P);
    else
      dsa::idx_tc::indexer_kernel<false><<<grid, dsa::idx_tc::kThreads, dsa::idx_tc::kSmemBytes, s>>>(tm_q, tm_k, P);
    DSA_TRY(check_launch("indexer_tc"));
    tr.after(DSA_KERNEL_INDEXER_TC);
  } else {
    if (rows > 65535) {
      for (int64_t c = r0; c < r1; c += 65535) {
        const int64_t e = std::min<int64_t>(r1, c + 65535);
        DSA_TRY(launch_index_scores(dev, b, ix, scores + (c - r0) * ld, ld, c, e, s, tr, nullptr));
      }
      return DSA_SUCCESS;
    }
    dim3 grid(static_cast<unsigned>((b->max_seqlen_kv + dsa::simt::kIdxThreads - 1) / dsa::simt::kIdxThreads),
              static_cast<unsigned>(rows));
    dsa::simt::indexer_kernel<<<grid, dsa::simt::kIdxThreads, 0, s>>>(
        ix->q, ix->q_scale, ix->k, ix->k_scale, ix->w, ix->n_heads, ix->head_dim, ix->dtype,
        scores, ld, b->cu_seqlens_q, b->cu_seqlens_kv, b->num_seqs, r0);
    DSA_TRY(check_launch("indexer_simt"));
    tr.after(DSA_KERNEL_INDEXER_SIMT);
  }
  return DSA_SUCCESS;
}

// A few rows (a decode batch) cannot fill the device one CTA per row: each
// row then gets a cluster of CTAs, each taking a slice of the row.
// hist (optional): the rows' first-digit histograms from the indexer.
dsa_status_t launch_topk(const DeviceInfo& dev, const dsa_batch_t* b, const float* scores, int64_t ld,
                         int32_t k, int32_t* idx, float* vals, int64_t r0, int64_t r1, cudaStream_t s,
                         Tracer& tr, const uint32_t* hist = nullptr) {
  NvtxRange nvtx("dsa: top-k");
  if (r1 > r0 && (r1 - r0) * dsa::topk::kCluster <= 4 * static_cast<int64_t>(dev.sms)) {
    dsa::topk::topk_cluster_kernel<<<static_cast<unsigned>((r1 - r0) * dsa::topk::kCluster),
                                     dsa::topk::kCThreads, dsa::topk::kCSmemBytes, s>>>(
        scores, ld, k, idx, vals, b->cu_seqlens_q, b->cu_seqlens_kv, b->num_seqs, r0, hist);
    DSA_TRY(check_launch("topk_cluster"));
    tr.after(DSA_KERNEL_TOPK);
    return DSA_SUCCESS;
  }
  for (int64_t c = r0; c < r1; c += 2147483647ll) {
    const int64_t e = std::min<int64_t>(r1, c + 2147483647ll);
    dsa::topk::topk_kernel<<<static_cast<unsigned>(e - c), dsa::topk::kThreads, dsa::topk::kSmemBytes, s>>>(
        scores + (c - r0) * ld, ld, k, idx + (c - r0) * k, vals ? vals + (c - r0) * k : nullptr,
        b->cu_seqlens_q, b->cu_seqlens_kv, b->num_seqs, c, hist ? hist + (c - r0) * dsa::kRadixBins : nullptr);
    DSA_TRY(check_launch("topk"));
    tr.after(DSA_KERNEL_TOPK);
  }
  return DSA_SUCCESS;
}

// Split-KV plan for the tensor-core MLA kernel over `rows` query rows.
struct MlaPlan {
  int nsplit = 1;
  int tiles_per_split = 1;
  size_t ws_bytes = 0;
};

// Each (row, split) unit runs on two CTAs (one per half of the output
// columns).  When the rows alone would leave more than half of the SMs idle,
// each row's selected tiles are split over several units (partials merged by
// the combine kernel); a split costs a second wave and a second per-CTA
// start-up, so it is not taken for a mostly full wave.
// The split count shrinks until its scratch fits `ws_cap` bytes.
MlaPlan plan_mla(int sms, int64_t rows, int32_t k, size_t ws_cap = SIZE_MAX) {
  const int tiles = (k + dsa::mla_tc::kRows - 1) / dsa::mla_tc::kRows;
  const int64_t units_wanted = std::max(1, sms / 2);
  int want = 1;
  if (2 * rows < units_wanted) want = static_cast<int>((units_wanted + rows - 1) / rows);
  want = std::min(want, tiles);
  for (;; --want) {
    MlaPlan p;
    p.tiles_per_split = (tiles + want - 1) / want;
    p.nsplit = (tiles + p.tiles_per_split - 1) / p.tiles_per_split;
    if (p.nsplit > 1)
      p.ws_bytes = static_cast<size_t>(rows) * p.nsplit * dsa::mla_tc::kHeads * (dsa::mla_tc::kDv + 1) * 4 + 256;
    if (p.ws_bytes <= ws_cap || want <= 1) return p;
  }
}

// Dense mode: the longest row sets the tile count.  With fewer rows than SMs
// the rows are also split so that no unit exceeds kDenseTilesPerUnit tiles,
// which keeps rows of very different lengths from serialising on a few SMs.
constexpr int kDenseTilesPerUnit = 128;
MlaPlan plan_dense_mla(int sms, int64_t rows, int32_t max_n, size_t ws_cap = SIZE_MAX) {
  const int tiles = (max_n + dsa::mla_tc::kRows - 1) / dsa::mla_tc::kRows;
  const int64_t units_wanted = std::max(1, sms / 2);
  int want = 1;
  if (2 * rows < units_wanted) want = static_cast<int>((units_wanted + rows - 1) / rows);
  if (rows < sms) want = std::max(want, (tiles + kDenseTilesPerUnit - 1) / kDenseTilesPerUnit);
  want = std::max(1, std::min(want, tiles));
  for (;; --want) {
    MlaPlan p;
    p.tiles_per_split = (tiles + want - 1) / want;
    p.nsplit = (tiles + p.tiles_per_split - 1) / p.tiles_per_split;
    if (p.nsplit > 1)
      p.ws_bytes = static_cast<size_t>(rows) * p.nsplit * dsa::mla_tc::kHeads * (dsa::mla_tc::kDv + 1) * 4 + 256;
    if (p.ws_bytes <= ws_cap || want <= 1) return p;
  }
}

dsa_status_t launch_sparse_mla(const DeviceInfo& dev, const dsa_batch_t* b, const dsa_mla_t* m,
                               const int32_t* idx, int32_t k, void* out, float* lse, void* ws,
                               size_t ws_bytes, int64_t r0, int64_t r1, cudaStream_t s, Tracer& tr,
                               bool dense = false, bool pdl = false) {
  const int64_t rows = r1 - r0;
  if (rows <= 0) return DSA_SUCCESS;
  NvtxRange nvtx(dense ? "dsa: dense attention" : "dsa: sparse attention");
  if (mla_is_tc(m)) {
    const MlaPlan plan = dense ? plan_dense_mla(dev.sms, rows, k, ws ? ws_bytes : 0)
                               : plan_mla(dev.sms, rows, k, ws ? ws_bytes : 0);
    if (plan.ws_bytes > ws_bytes || (plan.ws_bytes > 0 && !ws))
      return fail(DSA_ERROR_INSUFFICIENT_WORKSPACE, "sparse MLA needs %zu bytes of workspace, got %zu",
                  plan.ws_bytes, ws_bytes);
    if (ws && !aligned16(ws)) return fail(DSA_ERROR_INVALID_VALUE, "workspace must be 16-byte aligned");
    CUtensorMap tm_q, tm_out;
    DSA_TRY(encode_2d(&tm_q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, m->q, dsa::mla_tc::kDqk,
                      static_cast<uint64_t>(b->total_q) * dsa::mla_tc::kHeads, dsa::mla_tc::kDqk * 2, 64,
                      dsa::mla_tc::kHeads));
    // the output rows of this launch, [rows x 128 heads, 512] bf16, stored in
    // boxes of 64 columns x 128 heads
    DSA_TRY(encode_2d(&tm_out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, out, dsa::mla_tc::kDv,
                      static_cast<uint64_t>(rows) * dsa::mla_tc::kHeads, dsa::mla_tc::kDv * 2, 64,
                      dsa::mla_tc::kHeads));
    dsa::mla_tc::Params P{};
    P.q = static_cast<const __nv_bfloat16*>(m->q);
    P.kv = static_cast<const __nv_bfloat16*>(m->kv);
    P.idx = idx;
    P.k = k;
    P.dense = dense ? 1 : 0;
    P.c_log2 = m->scale * 1.4426950408889634f;
    P.cu_q = b->cu_seqlens_q;
    P.cu_kv = b->cu_seqlens_kv;
    P.num_seqs = b->num_seqs;
    P.row0 = r0;
    P.nsplit = plan.nsplit;
    P.tiles_per_split = plan.tiles_per_split;
    P.units = rows * plan.nsplit;
    // about one wave of clusters (two CTAs per SM pair) runs at a time
    P.prefetch_ahead = std::max(1, dev.sms / 2);
    P.out = static_cast<__nv_bfloat16*>(out);
    P.lse = lse;
    if (plan.nsplit > 1) {
      P.part_o = static_cast<float*>(ws);
      P.part_lse = reinterpret_cast<float*>(static_cast<char*>(ws) + static_cast<size_t>(rows) * plan.nsplit *
                                                                        dsa::mla_tc::kHeads * dsa::mla_tc::kDv * 4);
    }
    const int64_t ctas = 2 * rows * plan.nsplit;
    if (ctas > 2147483647ll) return fail(DSA_ERROR_NOT_SUPPORTED, "too many query rows in one call");
    {
      // pdl: launched as dependent on the kernel before it (the top-k), so its
      // CTAs set up and load their queries while that kernel finishes; they
      // wait for it before reading the index lists
      cudaLaunchConfig_t cfg{};
      cfg.gridDim = dim3(static_cast<unsigned>(ctas));
      cfg.blockDim = dim3(dsa::mla_tc::kThreads);
      cfg.dynamicSmemBytes = dsa::mla_tc::kSmemBytes;
      cfg.stream = s;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
      attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      const cudaError_t e = cudaLaunchKernelEx(&cfg, dsa::mla_tc::mla_kernel, tm_q, tm_out, P);
      if (e != cudaSuccess) return fail(DSA_ERROR_LAUNCH, "mla_tc launch failed: %s", cudaGetErrorString(e));
    }
    DSA_TRY(check_launch("mla_tc"));
    tr.after(DSA_KERNEL_MLA_TC);
    if (plan.nsplit > 1) {
      dim3 grid(static_cast<unsigned>(rows), dsa::mla_tc::kHeads);
      dsa::mla_tc::combine_kernel<<<grid, 128, 0, s>>>(P.part_o, P.part_lse, plan.nsplit, P.out, lse);
      DSA_TRY(check_launch("mla_combine"));
      tr.after(DSA_KERNEL_MLA_COMBINE);
    }
  } else {
    for (int64_t c = r0; c < r1; c += 2147483647ll) {
      const int64_t e = std::min<int64_t>(r1, c + 2147483647ll);
      const size_t esz = m->dtype == DSA_DTYPE_BF16 ? 2 : 4;
      dsa::simt::mla_kernel<<<static_cast<unsigned>(e - c), dsa::simt::kMlaWarps * 32, 0, s>>>(
          m->q, m->kv, idx + (c - r0) * k, k, m->n_heads, m->d_qk, m->d_v, m->scale, m->dtype,
          static_cast<char*>(out) + (c - r0) * m->n_heads * m->d_v * static_cast<int64_t>(esz),
          lse ? lse + (c - r0) * m->n_heads : nullptr, b->cu_seqlens_q, b->cu_seqlens_kv, b->num_seqs, c);
      DSA_TRY(check_launch("mla_simt"));
      tr.after(DSA_KERNEL_MLA_SIMT);
    }
  }
  return DSA_SUCCESS;
}

int64_t round_up(int64_t x, int64_t m) { return (x + m - 1) / m * m; }

// Zero the first-digit histograms of `rows` query rows before the indexer
// adds to them (nothing to do without a histogram buffer).
dsa_status_t clear_hist(uint32_t* hist, int64_t rows, cudaStream_t s, Tracer& tr) {
  if (!hist || rows <= 0) return DSA_SUCCESS;
  if (cudaMemsetAsync(hist, 0, static_cast<size_t>(rows) * dsa::kRadixBins * 4, s) != cudaSuccess)
    return fail(DSA_ERROR_LAUNCH, "clearing the top-k histograms failed: %s", cudaGetErrorString(cudaGetLastError()));
  tr.after(DSA_KERNEL_HIST_CLEAR);
  return DSA_SUCCESS;
}

// Forward workspace: [scores chunk | idx chunk | MLA split scratch]
struct FwdPlan {
  int64_t chunk;
  int64_t ld;
  size_t scores_bytes, idx_bytes, mla_bytes, total;
};

FwdPlan plan_forward(int sms, const dsa_batch_t* b, const dsa_mla_t* m, int32_t k, int64_t chunk) {
  FwdPlan p;
  p.chunk = std::max<int64_t>(1, std::min<int64_t>(chunk, b->total_q));
  p.ld = round_up(std::max(1, b->max_seqlen_kv), 4);
  p.scores_bytes = static_cast<size_t>(round_up(p.chunk * p.ld * 4, 256));
  p.idx_bytes = static_cast<size_t>(round_up(p.chunk * static_cast<int64_t>(k) * 4, 256));
  p.mla_bytes = 0;
  if (m && mla_is_tc(m)) {
    // sized for a full chunk; a smaller tail chunk reduces its split count
    // to fit (plan_mla with a cap)
    p.mla_bytes = static_cast<size_t>(round_up(static_cast<int64_t>(plan_mla(sms, p.chunk, k).ws_bytes), 256));
  }
  p.total = p.scores_bytes + p.idx_bytes + p.mla_bytes;
  return p;
}

constexpr int64_t kPreferredChunk = 16384;
constexpr int64_t kMinChunk = 64;
// Query chunk of dsa_forward_streamed: the first chunk's inputs and the last
// chunk's results are copied while no kernel runs, so smaller chunks than the
// forward's shorten that fill and drain (copies, not kernels, bound that path).
constexpr int64_t kStreamedChunk = 4096;

int sms_for_sizing() {
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  return sms > 0 ? sms : 148;
}

// ---------------------------------------------------------------------------
// Built-in scratch for dsa_sparse_mla_noalloc
// ---------------------------------------------------------------------------
constexpr size_t kStaticScratchBytes = size_t(24) << 20;  // 24 MiB

}  // namespace

// Split-KV partials of dsa_sparse_mla_noalloc.  Every GPU that loads the
// library holds this array until the process exits.  Host code must not pass
// the symbol itself to a kernel (on the host it is only a stand-in): the
// device address comes from cudaGetSymbolAddress, looked up once per device.
static __device__ __align__(256) uint8_t g_static_scratch[kStaticScratchBytes];

namespace {

void* g_static_scratch_addr[kMaxDevices] = {};
std::mutex g_static_scratch_mu;

// Device address of g_static_scratch on the current device (first call per
// device does the lookup).
dsa_status_t static_scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return fail(DSA_ERROR_DEVICE, "no usable current CUDA device");
  std::lock_guard<std::mutex> lk(g_static_scratch_mu);
  if (!g_static_scratch_addr[dev]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess || !p)
      return fail(DSA_ERROR_LAUNCH, "cudaGetSymbolAddress of the built-in scratch failed: %s",
                  cudaGetErrorString(e));
    g_static_scratch_addr[dev] = p;
  }
  *out = g_static_scratch_addr[dev];
  return DSA_SUCCESS;
}

// ---------------------------------------------------------------------------
// Indexer warm-up loss: workspace per query row of a chunk is the scores /
// gradient row, the target row and its per-head scratch row, and the
// H_I x ld matrix c[t, j, s] of the backward.
size_t kl_row_bytes(const dsa_batch_t* b, const dsa_indexer_t* ix) {
  const int64_t ld = round_up(std::max(1, b->max_seqlen_kv), 4);
  return static_cast<size_t>((3 + ix->n_heads) * ld) * 4;
}
constexpr int64_t kKlMaxChunk = 65535;   // grid.y of the backward kernel

dsa_status_t check_kl(const dsa_batch_t* batch, const dsa_indexer_t* ix, const dsa_mla_t* mla) {
  DSA_TRY(check_batch(batch));
  DSA_TRY(check_indexer(ix, batch));
  DSA_TRY(check_mla(mla, batch));
  return DSA_SUCCESS;
}

}  // namespace

extern "C" {

int32_t dsa_abi_version(void) { return DSA_ABI_VERSION; }

const char* dsa_status_string(dsa_status_t s) {
  switch (s) {
    case DSA_SUCCESS: return "success";
    case DSA_ERROR_INVALID_VALUE: return "invalid value";
    case DSA_ERROR_NOT_SUPPORTED: return "not supported";
    case DSA_ERROR_INSUFFICIENT_WORKSPACE: return "insufficient workspace";
    case DSA_ERROR_LAUNCH: return "launch failure";
    case DSA_ERROR_DEVICE: return "unsupported or missing device";
    case DSA_ERROR_TIMEOUT: return "device wait timed out";
    case DSA_ERROR_BAD_INDEX: return "selected index out of range";
  }
  return "unknown status";
}

const char* dsa_last_error_message(void) { return g_last_msg.c_str(); }

dsa_status_t dsa_workspace_size(const dsa_batch_t* batch, const dsa_indexer_t* indexer, const dsa_mla_t* mla,
                                int32_t k, size_t* min_bytes, size_t* preferred_bytes) {
  DSA_TRY(check_batch(batch));
  DSA_TRY(check_k(k));
  if (mla) DSA_TRY(check_mla(mla, batch));
  const int sms = sms_for_sizing();
  size_t mn = 0, pref = 0;
  if (!indexer) {
    if (mla && mla_is_tc(mla) && batch->total_q > 0) mn = pref = plan_mla(sms, batch->total_q, k).ws_bytes;
  } else {
    DSA_TRY(check_indexer(indexer, batch));
    if (batch->total_q > 0) {
      mn = plan_forward(sms, batch, mla, k, kMinChunk).total;
      pref = plan_forward(sms, batch, mla, k, kPreferredChunk).total;
    }
  }
  if (min_bytes) *min_bytes = mn;
  if (preferred_bytes) *preferred_bytes = std::max(mn, pref);
  return DSA_SUCCESS;
}

dsa_status_t dsa_index_scores(const dsa_batch_t* batch, const dsa_indexer_t* indexer, float* scores,
                              int64_t ld_scores, cudaStream_t stream) {
  DSA_TRY(check_batch(batch));
  DSA_TRY(check_indexer(indexer, batch));
  if (batch->total_q == 0) return DSA_SUCCESS;
  if (!scores || !aligned16(scores)) return fail(DSA_ERROR_INVALID_VALUE, "scores must be non-NULL and 16-byte aligned");
  if (ld_scores < batch->max_seqlen_kv || ld_scores % 4 != 0)
    return fail(DSA_ERROR_INVALID_VALUE, "ld_scores must be >= max_seqlen_kv and a multiple of 4");
  DeviceInfo* dev;
  DSA_TRY(device_info(&dev));
  Tracer tr{nullptr, stream};
  return launch_index_scores(*dev, batch, indexer, scores, ld_scores, 0, batch->total_q, stream, tr);
}

dsa_status_t dsa_topk(const dsa_batch_t* batch, const float* scores, int64_t ld_scores, int32_t k, int32_t* idx,
                      float* vals, cudaStream_t stream) {
  DSA_TRY(check_batch(batch));
  DSA_TRY(check_k(k));
  if (batch->total_q == 0) return DSA_SUCCESS;
  if (!scores || !aligned16(scores) || !idx || !aligned16(idx) || (vals && !aligned16(vals)))
    return fail(DSA_ERROR_INVALID_VALUE, "scores and idx must be non-NULL and 16-byte aligned");
  if (ld_scores < batch->max_seqlen_kv || ld_scores % 4 != 0)
    return fail(DSA_ERROR_INVALID_VALUE, "ld_scores must be >= max_seqlen_kv and a multiple of 4");
  DeviceInfo* dev;
  DSA_TRY(device_info(&dev));
  Tracer tr{nullptr, stream};
  return launch_topk(*dev, batch, scores, ld_scores, k, idx, vals, 0, batch->total_q, stream, tr);
}

dsa_status_t dsa_index_scores_hist(const dsa_batch_t* batch, const dsa_indexer_t* indexer, float* scores,
                                   int64_t ld_scores, uint32_t* hist, cudaStream_t stream) {
  DSA_TRY(check_batch(batch));
  DSA_TRY(check_indexer(indexer, batch));
  if (!indexer_is_tc(indexer))
    return fail(DSA_ERROR_NOT_SUPPORTED, "dsa_index_scores_hist needs the tensor-core indexer (E4M3, 64 heads x 128)");
  if (batch->total_q == 0) return DSA_SUCCESS;
  if (!scores || !aligned16(scores) || !hist || !aligned16(hist))
    return fail(DSA_ERROR_INVALID_VALUE, "scores and hist must be non-NULL and 16-byte aligned");
  if (ld_scores < batch->max_seqlen_kv || ld_scores % 4 != 0)
    return fail(DSA_ERROR_INVALID_VALUE, "ld_scores must be >= max_seqlen_kv and a multiple of 4");
  DeviceInfo* dev;
  DSA_TRY(device_info(&dev));
  Tracer tr{nullptr, stream};
  DSA_TRY(clear_hist(hist, batch->total_q, stream, tr));
  return launch_index_scores(*dev, batch, indexer, scores, ld_scores, 0, batch->total_q, stream, tr, hist);
}

dsa_status_t dsa_topk_hist(const dsa_batch_t* batch, const float* scores, int64_t ld_scores, const uint32_t* hist,
                           int32_t k, int32_t* idx, float* vals, cudaStream_t stream) {
  DSA_TRY(check_batch(batch));
  DSA_TRY(check_k(k));
  if (batch->total_q == 0) return DSA_SUCCESS;
  if (!scores || !aligned16(scores) || !idx || !aligned16(idx) || (vals && !aligned16(vals)) || !hist ||
      !aligned16(hist))
    return fail(DSA_ERROR_INVALID_VALUE, "scores, hist and idx must be non-NULL and 16-byte aligned");
  if (ld_scores < batch->max_seqlen_kv || ld_scores % 4 != 0)
    return fail(DSA_ERROR_INVALID_VALUE, "ld_scores must be >= max_seqlen_kv and a multiple of 4");
  DeviceInfo* dev;
  DSA_TRY(device_info(&dev));
  Tracer tr{nullptr, stream};
  return launch_topk(*dev, batch, scores, ld_scores, k, idx, vals, 0, batch->total_q, stream, tr, hist);
}

dsa_status_t dsa_sparse_mla(const dsa_batch_t* batch, const dsa_mla_t* mla, const int32_t* idx, int32_t k,
                            void* out, float* lse, void* ws, size_t ws_bytes, cudaStream_t stream) {
  DSA_TRY(check_batch(batch));
  DSA_TRY(check_mla(mla, batch));
  DSA_TRY(check_k(k));
  if (batch->total_q == 0) return DSA_SUCCESS;
  if (!idx || !aligned16(idx) || !out || !aligned16(out) || (lse && !aligned16(lse)))
    return fail(DSA_ERROR_INVALID_VALUE, "idx and out must be non-NULL and 16-byte aligned");
  DeviceInfo* dev;
  DSA_TRY(device_info(&dev));
  Tracer tr{nullptr, stream};
  return launch_sparse_mla(*dev, batch, mla, idx, k, out, lse, ws, ws_bytes, 0, batch->total_q, stream, tr);
}

dsa_status_t dsa_dense_mla_workspace_size(const dsa_batch_t* batch, const dsa_mla_t* mla, size_t* bytes) {
  DSA_TRY(check_batch(batch));
  DSA_TRY(check_mla(mla, batch));
  if (!mla_is_tc(mla)) return fail(DSA_ERROR_NOT_SUPPORTED, "dense MLA needs 128 heads, d_qk 576, d_v 512, BF16");
  size_t need = 0;
  if (batch->total_q > 0) need = plan_dense_mla(sms_for_sizing(), batch->total_q, std::max(1, batch->max_seqlen_kv)).ws_bytes;
  if (bytes) *bytes = need;
  return DSA_SUCCESS;
}

dsa_status_t dsa_dense_mla(const dsa_batch_t* batch, const dsa_mla_t* mla, void* out, float* lse, void* ws,
                           size_t ws_bytes, cudaStream_t stream) {
  DSA_TRY(check_batch(batch));
  DSA_TRY(check_mla(mla, batch));
  if (!mla_is_tc(mla)) return fail(DSA_ERROR_NOT_SUPPORTED, "dense MLA needs 128 heads, d_qk 576, d_v 512, BF16");
  if (batch->total_q == 0) return DSA_SUCCESS;
  if (!out || !aligned16(out) || (lse && !aligned16(lse)))
    return fail(DSA_ERROR_INVALID_VALUE, "out must be non-NULL; out and lse 16-byte aligned");
  DeviceInfo* dev;
  DSA_TRY(device_info(&dev));
  Tracer tr{nullptr, stream};
  return launch_sparse_mla(*dev, batch, mla, nullptr, std::max(1, batch->max_seqlen_kv), out, lse, ws, ws_bytes, 0,
                           batch->total_q, stream, tr, true);
}

dsa_status_t dsa_sparse_mla_noalloc(const dsa_batch_t* batch, const dsa_mla_t* mla, const int32_t* idx,
                                    int32_t k, void* out, float* lse, cudaStream_t stream) {
  DSA_TRY(check_batch(batch));
  DSA_TRY(check_mla(mla, batch));
  DSA_TRY(check_k(k));
  if (batch->total_q == 0) return DSA_SUCCESS;
  if (!idx || !aligned16(idx) || !out || !aligned16(out) || (lse && !aligned16(lse)))
    return fail(DSA_ERROR_INVALID_VALUE, "idx and out must be non-NULL and 16-byte aligned");
  DeviceInfo* dev;
  DSA_TRY(device_info(&dev));
  // the split plan dsa_sparse_mla uses with a workspace of the built-in
  // scratch's size: a batch whose preferred split would not fit takes fewer
  // splits, so only a plan that cannot shrink below the array is refused
  const size_t need = mla_is_tc(mla) ? plan_mla(dev->sms, batch->total_q, k, kStaticScratchBytes).ws_bytes : 0;
  if (need > kStaticScratchBytes)
    return fail(DSA_ERROR_NOT_SUPPORTED,
                "dsa_sparse_mla_noalloc: this batch needs %zu bytes of split-KV scratch but the built-in "
                "scratch holds %zu bytes; call dsa_sparse_mla with a workspace instead",
                need, kStaticScratchBytes);
  void* scratch = nullptr;
  DSA_TRY(static_scratch_address(&scratch));
  Tracer tr{nullptr, stream};
  return launch_sparse_mla(*dev, batch, mla, idx, k, out, lse, scratch, kStaticScratchBytes, 0,
                           batch->total_q, stream, tr);
}

dsa_status_t dsa_quantize_e4m3(const void* x, dsa_dtype_t x_dtype, int64_t groups, int32_t group_elems,
                               uint8_t* codes, float* scales, cudaStream_t stream) {
  NvtxRange nvtx("dsa: quantize e4m3");
  if (groups < 0) return fail(DSA_ERROR_INVALID_VALUE, "groups must be >= 0");
  if (group_elems < 4 || group_elems > dsa::quant::kMaxGroup || group_elems % 4 != 0)
    return fail(DSA_ERROR_INVALID_VALUE, "group_elems must be a multiple of 4 in [4, %d]", dsa::quant::kMaxGroup);
  if (x_dtype != DSA_DTYPE_F32 && x_dtype != DSA_DTYPE_BF16)
    return fail(DSA_ERROR_NOT_SUPPORTED, "quantize: x dtype must be F32 or BF16");
  if (groups == 0) return DSA_SUCCESS;
  if (!x || !codes || !scales) return fail(DSA_ERROR_INVALID_VALUE, "quantize: x, codes and scales are required");
  if (!aligned16(x) || (reinterpret_cast<uintptr_t>(codes) & 3u) || (reinterpret_cast<uintptr_t>(scales) & 3u))
    return fail(DSA_ERROR_INVALID_VALUE, "quantize: x must be 16-byte aligned, codes and scales 4-byte aligned");
  if (groups > (int64_t(1) << 31) - 1) return fail(DSA_ERROR_NOT_SUPPORTED, "quantize: too many groups");
  DeviceInfo* dev;
  DSA_TRY(device_info(&dev));
  const bool bf16 = x_dtype == DSA_DTYPE_BF16;
  namespace q = dsa::quant;
  if (group_elems <= q::kWarpGroupMax) {
    const int64_t per_cta = q::kThreads / 32;   // one warp per group
    const int64_t ctas = (groups + per_cta - 1) / per_cta;
    q::quantize_warp_kernel<<<static_cast<unsigned>(ctas), q::kThreads, 0, stream>>>(x, bf16, groups, group_elems,
                                                                                    codes, scales);
  } else {
    // one CTA per group (groups < 2^31 was checked above)
    const unsigned grid = static_cast<unsigned>(groups);
    if (!bf16)
      q::quantize_cta_kernel<q::kF32x4><<<grid, 256, 0, stream>>>(x, group_elems, codes, scales);
    else if (group_elems % 8 == 0)
      q::quantize_cta_kernel<q::kBf16x8><<<grid, 256, 0, stream>>>(x, group_elems, codes, scales);
    else
      q::quantize_cta_kernel<q::kBf16x4><<<grid, 256, 0, stream>>>(x, group_elems, codes, scales);
  }
  return check_launch("quantize_e4m3");
}

dsa_status_t dsa_indexer_loss_workspace_size(const dsa_batch_t* batch, const dsa_indexer_t* indexer,
                                             const dsa_mla_t* mla, size_t* min_bytes, size_t* preferred_bytes) {
  DSA_TRY(check_kl(batch, indexer, mla));
  const size_t per_row = kl_row_bytes(batch, indexer);
  const size_t mn = batch->total_q > 0 ? per_row + 256 : 0;
  const size_t pref = batch->total_q > 0 ? per_row * std::min<int64_t>(batch->total_q, kKlMaxChunk) + 256 : 0;
  if (min_bytes) *min_bytes = mn;
  if (preferred_bytes) *preferred_bytes = pref;
  return DSA_SUCCESS;
}

dsa_status_t dsa_indexer_warmup_loss(const dsa_batch_t* batch, const dsa_indexer_t* indexer, const dsa_mla_t* mla,
                                     float* loss_rows, float* dq, float* dk, float* dw, void* ws, size_t ws_bytes,
                                     cudaStream_t stream) {
  NvtxRange nvtx("dsa: indexer warm-up loss");
  DSA_TRY(check_kl(batch, indexer, mla));
  if (batch->total_q == 0) return DSA_SUCCESS;
  if (!loss_rows || !dq || !dk || !dw || !aligned16(loss_rows) || !aligned16(dq) || !aligned16(dk) || !aligned16(dw))
    return fail(DSA_ERROR_INVALID_VALUE, "loss_rows, dq, dk and dw must be non-NULL and 16-byte aligned");
  if (!ws || !aligned16(ws)) return fail(DSA_ERROR_INVALID_VALUE, "workspace must be non-NULL and 16-byte aligned");
  const size_t per_row = kl_row_bytes(batch, indexer);
  if (ws_bytes < per_row + 256)
    return fail(DSA_ERROR_INSUFFICIENT_WORKSPACE, "dsa_indexer_warmup_loss needs at least %zu bytes of workspace, got %zu",
                per_row + 256, ws_bytes);
  DeviceInfo* dev;
  DSA_TRY(device_info(&dev));
  const int64_t ld = round_up(std::max(1, batch->max_seqlen_kv), 4);
  const int64_t chunk = std::min<int64_t>({batch->total_q, kKlMaxChunk, static_cast<int64_t>((ws_bytes - 256) / per_row)});
  const int HI = indexer->n_heads, D = indexer->head_dim;
  float* IG = static_cast<float*>(ws);
  float* P = IG + chunk * ld;
  float* Z = P + chunk * ld;
  float* C = Z + chunk * ld;
  if (cudaMemsetAsync(dk, 0, static_cast<size_t>(batch->total_kv) * D * 4, stream) != cudaSuccess ||
      cudaMemsetAsync(dw, 0, static_cast<size_t>(batch->total_q) * HI * 4, stream) != cudaSuccess)
    return fail(DSA_ERROR_LAUNCH, "clearing dk / dw failed: %s", cudaGetErrorString(cudaGetLastError()));
  const int idtype = indexer->dtype, mdtype = mla->dtype;
  Tracer tr{nullptr, stream};
  for (int64_t r0 = 0; r0 < batch->total_q; r0 += chunk) {
    const int64_t r1 = std::min<int64_t>(batch->total_q, r0 + chunk);
    const unsigned rows = static_cast<unsigned>(r1 - r0);
    // I[t, s] for the chunk (the forward indexer kernels)
    DSA_TRY(launch_index_scores(*dev, batch, indexer, IG, ld, r0, r1, stream, tr));
    dsa::kl::target_kernel<<<rows, dsa::kl::kThreads, 0, stream>>>(
        mla->q, mla->kv, mdtype, mla->n_heads, mla->d_qk, mla->scale, batch->cu_seqlens_q, batch->cu_seqlens_kv,
        batch->num_seqs, r0, P, Z, ld);
    DSA_TRY(check_launch("kl_target"));
    dsa::kl::loss_kernel<<<rows, dsa::kl::kThreads, 0, stream>>>(IG, P, ld, batch->cu_seqlens_q,
                                                                 batch->cu_seqlens_kv, batch->num_seqs, r0, loss_rows);
    DSA_TRY(check_launch("kl_loss"));
    dim3 gx(static_cast<unsigned>((batch->max_seqlen_kv + dsa::kl::kBwdThreads - 1) / dsa::kl::kBwdThreads), rows);
    dsa::kl::bwd_x_kernel<<<gx, dsa::kl::kBwdThreads, 0, stream>>>(
        indexer->q, indexer->q_scale, indexer->k, indexer->k_scale, indexer->w, HI, D, idtype, IG, ld,
        batch->cu_seqlens_q, batch->cu_seqlens_kv, batch->num_seqs, r0, C, dw);
    DSA_TRY(check_launch("kl_bwd_x"));
    dsa::kl::bwd_dq_kernel<<<rows, dsa::kl::kBwdThreads, 0, stream>>>(
        C, indexer->k, indexer->k_scale, HI, D, idtype, ld, batch->cu_seqlens_q, batch->cu_seqlens_kv,
        batch->num_seqs, r0, dq);
    DSA_TRY(check_launch("kl_bwd_dq"));
    if (batch->total_kv > 0) {
      dsa::kl::bwd_dk_kernel<<<static_cast<unsigned>(batch->total_kv), dsa::kl::kBwdThreads, 0, stream>>>(
          C, indexer->q, indexer->q_scale, HI, D, idtype, ld, batch->cu_seqlens_q, batch->cu_seqlens_kv,
          batch->num_seqs, r0, r1, dk);
      DSA_TRY(check_launch("kl_bwd_dk"));
    }
  }
  return DSA_SUCCESS;
}

dsa_status_t dsa_forward_traced(const dsa_batch_t* batch, const dsa_indexer_t* indexer, const dsa_mla_t* mla,
                                int32_t k, void* out, float* lse, int32_t* idx_out, void* ws, size_t ws_bytes,
                                cudaStream_t stream, dsa_trace_t* trace) {
  NvtxRange nvtx("dsa: forward");
  DSA_TRY(check_batch(batch));
  DSA_TRY(check_indexer(indexer, batch));
  DSA_TRY(check_mla(mla, batch));
  DSA_TRY(check_k(k));
  if ((batch->total_q > 0 && !out) || !aligned16(out) || (lse && !aligned16(lse)) ||
      (idx_out && !aligned16(idx_out)))
    return fail(DSA_ERROR_INVALID_VALUE, "out must be non-NULL; out, lse and idx_out 16-byte aligned");
  if (ws && !aligned16(ws)) return fail(DSA_ERROR_INVALID_VALUE, "workspace must be 16-byte aligned");
  DeviceInfo* dev;
  DSA_TRY(device_info(&dev));
  if (batch->total_q == 0) return DSA_SUCCESS;
  // largest chunk that fits the workspace
  const FwdPlan mn = plan_forward(dev->sms, batch, mla, k, kMinChunk);
  if (!ws || ws_bytes < mn.total)
    return fail(DSA_ERROR_INSUFFICIENT_WORKSPACE, "dsa_forward needs at least %zu bytes of workspace, got %zu",
                mn.total, ws ? ws_bytes : 0);
  // the preferred chunk when it fits, else the largest chunk that fits
  int64_t lo = mn.chunk, hi = std::min<int64_t>(kPreferredChunk, batch->total_q);
  if (plan_forward(dev->sms, batch, mla, k, hi).total <= ws_bytes) lo = hi;
  while (lo < hi) {
    const int64_t mid = (lo + hi + 1) / 2;
    if (plan_forward(dev->sms, batch, mla, k, mid).total <= ws_bytes) lo = mid; else hi = mid - 1;
  }
  const FwdPlan plan = plan_forward(dev->sms, batch, mla, k, lo);
  char* wsb = static_cast<char*>(ws);
  float* scores = reinterpret_cast<float*>(wsb);
  int32_t* idx_ws = reinterpret_cast<int32_t*>(wsb + plan.scores_bytes);
  void* mla_ws = plan.mla_bytes ? wsb + plan.scores_bytes + plan.idx_bytes : nullptr;
  const size_t esz = mla->dtype == DSA_DTYPE_BF16 ? 2 : 4;
  Tracer tr{trace, stream};
  DSA_TRY(tr.begin());
  for (int64_t r0 = 0; r0 < batch->total_q; r0 += plan.chunk) {
    const int64_t r1 = std::min<int64_t>(batch->total_q, r0 + plan.chunk);
    NvtxRange chunk_range("dsa: query chunk");
    int32_t* idx = idx_out ? idx_out + r0 * k : idx_ws;
    DSA_TRY(launch_index_scores(*dev, batch, indexer, scores, plan.ld, r0, r1, stream, tr));
    DSA_TRY(launch_topk(*dev, batch, scores, plan.ld, k, idx, nullptr, r0, r1, stream, tr));
    // (without a trace: each kernel's own time is not measured, so the
    // attention kernel may overlap the end of the top-k)
    DSA_TRY(launch_sparse_mla(*dev, batch, mla, idx, k,
                              static_cast<char*>(out) + r0 * mla->n_heads * mla->d_v * static_cast<int64_t>(esz),
                              lse ? lse + r0 * mla->n_heads : nullptr, mla_ws, plan.mla_bytes, r0, r1, stream, tr,
                              false, trace == nullptr));
  }
  return DSA_SUCCESS;
}

dsa_status_t dsa_forward(const dsa_batch_t* batch, const dsa_indexer_t* indexer, const dsa_mla_t* mla, int32_t k,
                         void* out, float* lse, int32_t* idx_out, void* ws, size_t ws_bytes, cudaStream_t stream) {
  return dsa_forward_traced(batch, indexer, mla, k, out, lse, idx_out, ws, ws_bytes, stream, nullptr);
}

dsa_status_t dsa_forward_streamed(const dsa_batch_t* batch, const dsa_indexer_t* indexer, const dsa_mla_t* mla,
                                  int32_t k, const dsa_host_inputs_t* host, void* out, float* lse, void* host_out,
                                  float* host_lse, void* ws, size_t ws_bytes, cudaStream_t stream,
                                  cudaStream_t copy_in, cudaStream_t copy_out) {
  NvtxRange nvtx("dsa: forward (streamed)");
  DSA_TRY(check_batch(batch));
  DSA_TRY(check_indexer(indexer, batch));
  DSA_TRY(check_mla(mla, batch));
  DSA_TRY(check_k(k));
  if (!host) return fail(DSA_ERROR_INVALID_VALUE, "host inputs are NULL");
  const bool has_q = batch->total_q > 0, has_kv = batch->total_kv > 0;
  if ((has_q && (!host->idx_q || !host->idx_w || !host->mla_q || !host_out)) ||
      (has_kv && (!host->idx_k || !host->mla_kv)) || (!indexer->q_scale != !host->idx_q_scale) ||
      (!indexer->k_scale != !host->idx_k_scale) || (host_lse && !lse))
    return fail(DSA_ERROR_INVALID_VALUE,
                "every device input needs its host copy (scales: both or neither); host_lse needs lse");
  if ((has_q && !out) || !aligned16(out) || (lse && !aligned16(lse)))
    return fail(DSA_ERROR_INVALID_VALUE, "out must be non-NULL; out and lse 16-byte aligned");
  if (ws && !aligned16(ws)) return fail(DSA_ERROR_INVALID_VALUE, "workspace must be 16-byte aligned");
  DeviceInfo* dev;
  DSA_TRY(device_info(&dev));
  if (!has_q) return DSA_SUCCESS;
  const FwdPlan mn = plan_forward(dev->sms, batch, mla, k, kMinChunk);
  if (!ws || ws_bytes < mn.total)
    return fail(DSA_ERROR_INSUFFICIENT_WORKSPACE, "dsa_forward_streamed needs at least %zu bytes of workspace, got %zu",
                mn.total, ws ? ws_bytes : 0);
  int64_t lo = mn.chunk, hi = std::min<int64_t>(std::max(kStreamedChunk, mn.chunk), batch->total_q);
  if (plan_forward(dev->sms, batch, mla, k, hi).total <= ws_bytes) lo = hi;
  while (lo < hi) {
    const int64_t mid = (lo + hi + 1) / 2;
    if (plan_forward(dev->sms, batch, mla, k, mid).total <= ws_bytes) lo = mid; else hi = mid - 1;
  }
  const FwdPlan plan = plan_forward(dev->sms, batch, mla, k, lo);
  char* wsb = static_cast<char*>(ws);
  float* scores = reinterpret_cast<float*>(wsb);
  int32_t* idx_ws = reinterpret_cast<int32_t*>(wsb + plan.scores_bytes);
  void* mla_ws = plan.mla_bytes ? wsb + plan.scores_bytes + plan.idx_bytes : nullptr;

  // bytes per row of every tensor that moves
  const size_t ie = indexer->dtype == DSA_DTYPE_E4M3 ? 1 : 4;
  const size_t me = mla->dtype == DSA_DTYPE_BF16 ? 2 : 4;
  const size_t row_iq = static_cast<size_t>(indexer->n_heads) * indexer->head_dim * ie;
  const size_t row_ik = static_cast<size_t>(indexer->head_dim) * ie;
  const size_t row_w = static_cast<size_t>(indexer->n_heads) * 4;
  const size_t row_mq = static_cast<size_t>(mla->n_heads) * mla->d_qk * me;
  const size_t row_kv = static_cast<size_t>(mla->d_qk) * me;
  const size_t row_out = static_cast<size_t>(mla->n_heads) * mla->d_v * me;
  const size_t row_lse = static_cast<size_t>(mla->n_heads) * 4;

  // Events order the three streams; each is destroyed once enqueued (its
  // resources are released when it completes).
  dsa_status_t st = DSA_SUCCESS;
  auto event = [&](cudaEvent_t* e) -> bool {
    if (cudaEventCreateWithFlags(e, cudaEventDisableTiming) != cudaSuccess) {
      st = fail(DSA_ERROR_LAUNCH, "cudaEventCreate failed: %s", cudaGetErrorString(cudaGetLastError()));
      return false;
    }
    return true;
  };
  // one event recorded on `from`, waited for on `to`
  auto link = [&](cudaStream_t from, cudaStream_t to) -> bool {
    cudaEvent_t e;
    if (!event(&e)) return false;
    const bool ok = cudaEventRecord(e, from) == cudaSuccess && cudaStreamWaitEvent(to, e, 0) == cudaSuccess;
    cudaEventDestroy(e);
    if (!ok) st = fail(DSA_ERROR_LAUNCH, "stream ordering failed: %s", cudaGetErrorString(cudaGetLastError()));
    return ok;
  };
  auto h2d = [&](const void* dst, const void* src, size_t bytes, cudaStream_t s) -> bool {
    if (bytes == 0) return true;
    if (cudaMemcpyAsync(const_cast<void*>(dst), src, bytes, cudaMemcpyHostToDevice, s) != cudaSuccess) {
      st = fail(DSA_ERROR_LAUNCH, "host-to-device copy failed: %s", cudaGetErrorString(cudaGetLastError()));
      return false;
    }
    return true;
  };
  auto d2h = [&](void* dst, const void* src, size_t bytes, cudaStream_t s) -> bool {
    if (bytes == 0) return true;
    if (cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDeviceToHost, s) != cudaSuccess) {
      st = fail(DSA_ERROR_LAUNCH, "device-to-host copy failed: %s", cudaGetErrorString(cudaGetLastError()));
      return false;
    }
    return true;
  };
  auto at = [](const void* base, int64_t row, size_t row_bytes) -> const char* {
    return static_cast<const char*>(base) + static_cast<size_t>(row) * row_bytes;
  };

  // start after the work already on `stream`
  if (!link(stream, copy_in) || !link(stream, copy_out)) return st;
  // key side in full
  const int64_t S = batch->total_kv;
  if (!h2d(indexer->k, host->idx_k, S * row_ik, copy_in) ||
      (indexer->k_scale && !h2d(indexer->k_scale, host->idx_k_scale, S * 4, copy_in)) ||
      !h2d(mla->kv, host->mla_kv, S * row_kv, copy_in))
    return st;
  Tracer tr{nullptr, stream};
  for (int64_t r0 = 0; r0 < batch->total_q; r0 += plan.chunk) {
    const int64_t r1 = std::min<int64_t>(batch->total_q, r0 + plan.chunk);
    const int64_t nr = r1 - r0;
    // this chunk's query side
    if (!h2d(at(indexer->q, r0, row_iq), at(host->idx_q, r0, row_iq), nr * row_iq, copy_in) ||
        (indexer->q_scale && !h2d(at(indexer->q_scale, r0, 4), at(host->idx_q_scale, r0, 4), nr * 4, copy_in)) ||
        !h2d(at(indexer->w, r0, row_w), at(host->idx_w, r0, row_w), nr * row_w, copy_in) ||
        !h2d(at(mla->q, r0, row_mq), at(host->mla_q, r0, row_mq), nr * row_mq, copy_in))
      return st;
    if (!link(copy_in, stream)) return st;
    DSA_TRY(launch_index_scores(*dev, batch, indexer, scores, plan.ld, r0, r1, stream, tr));
    DSA_TRY(launch_topk(*dev, batch, scores, plan.ld, k, idx_ws, nullptr, r0, r1, stream, tr));
    char* out_c = static_cast<char*>(out) + static_cast<size_t>(r0) * row_out;
    float* lse_c = lse ? lse + r0 * mla->n_heads : nullptr;
    DSA_TRY(launch_sparse_mla(*dev, batch, mla, idx_ws, k, out_c, lse_c, mla_ws, plan.mla_bytes, r0, r1, stream, tr));
    // this chunk's results back to the host
    if (!link(stream, copy_out)) return st;
    if (!d2h(static_cast<char*>(host_out) + static_cast<size_t>(r0) * row_out, out_c, nr * row_out, copy_out) ||
        (host_lse && !d2h(host_lse + r0 * mla->n_heads, lse_c, nr * row_lse, copy_out)))
      return st;
  }
  // later work on `stream` sees the host copies
  if (!link(copy_out, stream)) return st;
  return DSA_SUCCESS;
}

dsa_status_t dsa_read_device_errors(cudaStream_t stream, uint32_t* flags) {
  DeviceInfo* dev;
  DSA_TRY(device_info(&dev));
  if (cudaStreamSynchronize(stream) != cudaSuccess)
    return fail(DSA_ERROR_LAUNCH, "stream synchronize failed: %s", cudaGetErrorString(cudaGetLastError()));
  uint32_t v = 0;
  const uint32_t zero = 0;
  if (cudaMemcpyFromSymbol(&v, dsa::g_dev_errors, sizeof(v)) != cudaSuccess ||
      cudaMemcpyToSymbol(dsa::g_dev_errors, &zero, sizeof(zero)) != cudaSuccess)
    return fail(DSA_ERROR_LAUNCH, "reading the device error word failed: %s", cudaGetErrorString(cudaGetLastError()));
  if (flags) *flags = v;
  if (v & DSA_DEVERR_TIMEOUT) return fail(DSA_ERROR_TIMEOUT, "a device wait timed out (flags 0x%x)", v);
  if (v & DSA_DEVERR_BAD_INDEX) return fail(DSA_ERROR_BAD_INDEX, "an index was out of range (flags 0x%x)", v);
  return DSA_SUCCESS;
}

// Test hook: the next tensor-core indexer launch of this process runs with the
// given fault mode (1 = its producer skips one key tile, so the MMA warp's
// bounded wait runs out and the kernel reports DSA_DEVERR_TIMEOUT).
void dsa_debug_inject_fault(uint32_t mode) { g_fault_next.store(mode); }

}  // extern "C"
