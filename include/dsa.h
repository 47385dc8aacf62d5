/*
 * dsa.h - C ABI of the B300 (sm_103a) DeepSeek Sparse Attention forward library.
 *
 * The forward pass has three steps, each a hand-written CUDA kernel:
 *   1. lightning indexer  I[t,s] = sum_j w[t,j] * ReLU(q_I[t,j] . k_I[s])
 *      ("DeepSeek V3.2: How Far Can Open Models Go If You Actually Try?",
 *      §3.1, indexer equation; FP8, few heads);
 *   2. fine-grained selection of the top-k positions of each row I[t,:]
 *      (same §3.1; "Top-k operation" in the System Modules of "DeepSeek-V3.2:
 *      Pushing the Frontier of Open Large Language Models"; k = 2048 in its Key
 *      Hyperparameters);
 *   3. MLA in MQA mode over the selected latent rows only:
 *      u_t = Attn(h_t, {c_s : I[t,s] in Top-k(I[t,:])})  (same §3.1; §2.2 for
 *      the shared latent K/V bank read by every head).
 *
 * Conventions shared by every entry point
 *  - Ownership: every pointer is owned by the caller.  Tensors and workspace
 *    are device memory of the current device; structs are host memory.  The
 *    library allocates nothing, frees nothing and keeps no pointer after a
 *    call returns.
 *  - Layout: row-major and contiguous unless an ld (leading dimension, in
 *    elements) is given.  Every tensor base pointer must be 16-byte aligned.
 *  - Asynchrony: calls only enqueue work on `stream`; they return after host
 *    validation and launch.  No call synchronises except
 *    dsa_read_device_errors.
 *  - Errors: host-side problems return a status before anything is enqueued;
 *    launch failures return DSA_ERROR_LAUNCH.  Problems found on the device
 *    (a bounded wait that ran out, an out-of-range selected index) set bits in
 *    a per-device error word read by dsa_read_device_errors.
 *    dsa_last_error_message() gives a one-line description of the last
 *    non-success status returned on the calling host thread.
 *  - Device: sm_103 (B300) only; other devices get DSA_ERROR_DEVICE.
 *
 * Batch geometry (ragged; prefill and decode use the same struct)
 *  Sequence b has nq_b = cu_seqlens_q[b+1]-cu_seqlens_q[b] query tokens and
 *  nkv_b = cu_seqlens_kv[b+1]-cu_seqlens_kv[b] cached tokens, nkv_b >= nq_b.
 *  Query i of sequence b sits at position p = nkv_b - nq_b + i (bottom-right
 *  aligned: prefill has nq = nkv, decode nq = 1) and its candidates are the
 *  n = p + 1 keys s = 0..p of its own sequence (causal, self included).
 *  Positions s are sequence-local; the global row of key s is
 *  cu_seqlens_kv[b] + s.
 */
#ifndef DSA_H_
#define DSA_H_

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DSA_ABI_VERSION 1

typedef enum {
  DSA_SUCCESS = 0,
  DSA_ERROR_INVALID_VALUE = 1,          /* bad pointer, size, alignment or struct field */
  DSA_ERROR_NOT_SUPPORTED = 2,          /* valid but not implemented (dims/dtype combination) */
  DSA_ERROR_INSUFFICIENT_WORKSPACE = 3, /* ws_bytes below the minimum of dsa_workspace_size */
  DSA_ERROR_LAUNCH = 4,                 /* a CUDA launch or runtime call failed */
  DSA_ERROR_DEVICE = 5,                 /* current device is not an sm_103 GPU */
  DSA_ERROR_TIMEOUT = 6,                /* device error word: a bounded wait ran out */
  DSA_ERROR_BAD_INDEX = 7               /* device error word: a selected index was out of range */
} dsa_status_t;

typedef enum {
  DSA_DTYPE_F32 = 0,
  DSA_DTYPE_BF16 = 1,
  DSA_DTYPE_E4M3 = 2 /* OCP FP8 E4M3 ("fn": no infinities, 0x7F/0xFF are NaN) */
} dsa_dtype_t;

/* Bits of the per-device error word (dsa_read_device_errors). */
#define DSA_DEVERR_TIMEOUT 0x1u   /* an mbarrier wait exceeded its time limit; the kernel gave up */
#define DSA_DEVERR_BAD_INDEX 0x2u /* dsa_sparse_mla met an index outside [-1, n); it was skipped */

/* Ragged batch.  cu_seqlens_* are device arrays of num_seqs+1 non-decreasing
 * int32 offsets starting at 0.  The host fields must agree with them:
 * max_seqlen_* >= every per-sequence length, total_* = last offset. */
typedef struct {
  int32_t num_seqs;
  const int32_t* cu_seqlens_q;
  const int32_t* cu_seqlens_kv;
  int32_t max_seqlen_q;
  int32_t max_seqlen_kv;
  int64_t total_q;
  int64_t total_kv;
} dsa_batch_t;

/* Lightning-indexer inputs.  The real-valued q_I / k_I are code * scale, one
 * fp32 scale per query token (shared by its heads) and one per key row; NULL
 * scale = 1.  Scales must be positive and finite.
 *   q       [total_q, n_heads, head_dim]  dtype
 *   q_scale [total_q] fp32 or NULL
 *   k       [total_kv, head_dim]          dtype (one key per token, no head index)
 *   k_scale [total_kv] fp32 or NULL
 *   w       [total_q, n_heads] fp32       per-query head weights (any sign)
 * E4M3 with (n_heads, head_dim) = (64, 128) runs on the tcgen05 tensor cores;
 * other E4M3 / F32 shapes with n_heads <= 64 and head_dim <= 128 (head_dim a
 * multiple of 16) run on a CUDA-core kernel. */
typedef struct {
  int32_t n_heads;
  int32_t head_dim;
  dsa_dtype_t dtype;
  const void* q;
  const float* q_scale;
  const void* k;
  const float* k_scale;
  const float* w;
} dsa_indexer_t;

/* Sparse MLA (MQA mode) inputs.
 *   q   [total_q, n_heads, d_qk]  dtype (queries absorbed into the latent space)
 *   kv  [total_kv, d_qk]          dtype (one shared latent row per token; the
 *                                 value is its first d_v columns)
 * Scores are scale * (q . kv); softmax over the selected rows.
 * BF16 with (n_heads, d_qk, d_v) = (128, 576, 512) runs on the tcgen05 tensor
 * cores; other BF16 / F32 shapes with d_qk, d_v <= 1024 run on a CUDA-core
 * kernel.  The output has the input dtype. */
typedef struct {
  int32_t n_heads;
  int32_t d_qk;
  int32_t d_v;
  float scale;
  dsa_dtype_t dtype;
  const void* q;
  const void* kv;
} dsa_mla_t;

/* Optional launch trace: the library records `events[count++]` (caller-created
 * cudaEvents) before the first and after every kernel launch of a call, and
 * stores in kernel_ids[i] the kernel launched between events[i] and
 * events[i+1] (DSA_KERNEL_*).  Recording stops when capacity is reached. */
enum {
  DSA_KERNEL_INDEXER_TC = 1,
  DSA_KERNEL_INDEXER_SIMT = 2,
  DSA_KERNEL_TOPK = 3,
  DSA_KERNEL_MLA_TC = 4,
  DSA_KERNEL_MLA_SIMT = 5,
  DSA_KERNEL_MLA_COMBINE = 6,
  DSA_KERNEL_HIST_CLEAR = 7  /* zeroing of the first-digit histograms (dsa_index_scores_hist) */
};
typedef struct {
  int32_t capacity; /* number of events[] (kernel_ids[] holds capacity-1) */
  int32_t count;    /* events recorded so far; set to 0 before the call */
  cudaEvent_t* events;
  int32_t* kernel_ids;
} dsa_trace_t;

/* Workspace sizes (host only, no device access) for dsa_forward with the given
 * batch, indexer and MLA description and top-k.  min_bytes: the least ws_bytes
 * accepted; preferred_bytes: the size at which queries are processed in the
 * largest chunks the library uses.  With indexer == NULL the sizes are those
 * of dsa_sparse_mla alone.  Either output pointer may be NULL. */
dsa_status_t dsa_workspace_size(const dsa_batch_t* batch, const dsa_indexer_t* indexer,
                                const dsa_mla_t* mla, int32_t k, size_t* min_bytes,
                                size_t* preferred_bytes);

/* Step 1 alone.  Writes, for every query row r with n_r candidates,
 * scores[r * ld_scores + s] = I[r, s] for s in [0, n_r) (fp32); columns >= n_r
 * are not touched.  ld_scores >= max_seqlen_kv and a multiple of 4. */
dsa_status_t dsa_index_scores(const dsa_batch_t* batch, const dsa_indexer_t* indexer,
                              float* scores, int64_t ld_scores, cudaStream_t stream);

/* Step 2 alone.  For every query row r, reads scores[r * ld_scores + s] for
 * s in [0, n_r) and writes idx[r * k + i], i < k: the min(k, n_r) positions
 * with the largest scores in ascending position order, then -1.  Ties go to
 * the lower position and -0.0 equals +0.0 (NaN scores are outside the
 * contract).  vals (nullable, [total_q, k] fp32) receives the selected scores
 * (-inf in the -1 slots).  1 <= k <= 16384. */
dsa_status_t dsa_topk(const dsa_batch_t* batch, const float* scores, int64_t ld_scores,
                      int32_t k, int32_t* idx, float* vals, cudaStream_t stream);

/* Steps 1 and 2 with the selection's first pass fused into the indexer (no
 * counterpart on the pages beyond their separate indexer and "Top-k
 * operation" modules): dsa_index_scores_hist writes the scores exactly as
 * dsa_index_scores does and also, for every query row, the histogram of the
 * first radix digit of its scores (hist [total_q, 2048] uint32: bin = top 11
 * bits of the order-preserving 32-bit key of the fp32 score, -0 counted as
 * +0; the call clears hist first).  dsa_topk_hist then selects exactly as
 * dsa_topk does (same result, bit for bit) without re-reading a row for that
 * histogram.  Tensor-core indexer instance only (E4M3, 64 heads x 128), else
 * DSA_ERROR_NOT_SUPPORTED.  On one B300 and the 131072-token prefill the
 * histograms cost the indexer more time (+6 ms) than they save in the
 * selection (-4 ms), so dsa_forward runs the unfused pair; the fused pair
 * reads each score row once instead of twice. */
dsa_status_t dsa_index_scores_hist(const dsa_batch_t* batch, const dsa_indexer_t* indexer,
                                   float* scores, int64_t ld_scores, uint32_t* hist, cudaStream_t stream);
dsa_status_t dsa_topk_hist(const dsa_batch_t* batch, const float* scores, int64_t ld_scores,
                           const uint32_t* hist, int32_t k, int32_t* idx, float* vals, cudaStream_t stream);

/* Step 3 alone.  For every query row r: softmax attention of its n_heads
 * queries over the latent rows idx[r * k + i] (sequence-local positions; -1
 * slots are skipped; entries outside [-1, n_r) are skipped and flag
 * DSA_DEVERR_BAD_INDEX).  out [total_q, n_heads, d_v] (mla dtype);
 * lse (nullable) [total_q, n_heads] fp32 natural-log sum of exp of the scaled
 * scores (-inf and out = 0 for a row with nothing selected).  ws/ws_bytes:
 * scratch for split-KV decode, sized by dsa_workspace_size(batch, NULL, mla,
 * k, ...); may be NULL when that minimum is 0. */
dsa_status_t dsa_sparse_mla(const dsa_batch_t* batch, const dsa_mla_t* mla, const int32_t* idx,
                            int32_t k, void* out, float* lse, void* ws, size_t ws_bytes,
                            cudaStream_t stream);

/* Scratch-free variant of dsa_sparse_mla.  The pages have no counterpart: this
 * is an integration aid.  It is for callers that cannot hand the library a
 * device workspace, for example a plugin whose host runtime owns every device
 * allocation and offers no scratch buffer, or a serving loop that reserved
 * all device memory up front and may not call cudaMalloc in the middle of a
 * step (the call can fail, or synchronise the device).  Same arguments,
 * results and errors as dsa_sparse_mla, minus ws/ws_bytes: the split-KV
 * partials of small decode batches live in a 24 MiB array compiled into the
 * library, which every GPU that loads the library holds until the process
 * exits.  A batch whose preferred split needs more than 24 MiB (on a 148-SM
 * B300 with k = 2048: decode batches of 24 or of 32 to 36 query rows) splits
 * each row over fewer CTA pairs so that its partials fit, down to no split at
 * all; its results then agree with dsa_sparse_mla's to float rounding, not
 * bit for bit.  A plan that still did not fit would be refused with
 * DSA_ERROR_NOT_SUPPORTED (call dsa_sparse_mla with a workspace then); with
 * the split count able to fall to one, no batch of the tensor-core instance
 * is refused for its size.  The first call on each
 * device looks up the array's device address (cudaGetSymbolAddress), so make
 * that first call before any stream capture.  Every call shares the one
 * array and it keeps the last call's contents; the kernels overwrite
 * everything they read from it, so nothing needs clearing, but calls that
 * overlap on the GPU (other streams, other host threads) race on it and must
 * be serialised by the caller. */
dsa_status_t dsa_sparse_mla_noalloc(const dsa_batch_t* batch, const dsa_mla_t* mla,
                                    const int32_t* idx, int32_t k, void* out, float* lse,
                                    cudaStream_t stream);

/* Dense causal MLA-MQA attention: every query attends to all of its
 * candidates 0..p (no selection).  This is the baseline sparse selection is
 * measured against ("DeepSeek V3.2: How Far Can Open Models Go If You
 * Actually Try?", §3.4: decode at 128K about 2x cheaper than dense MLA; short
 * prompts run as dense masked attention).  Same layouts and outputs as
 * dsa_sparse_mla; only the tensor-core instance (128 heads, d_qk 576, d_v 512,
 * BF16) is supported, else DSA_ERROR_NOT_SUPPORTED.  Batches with fewer rows
 * than SMs split each row over several CTA pairs; their fp32 partials need
 * dsa_dense_mla_workspace_size bytes of workspace (0 otherwise), else
 * DSA_ERROR_INSUFFICIENT_WORKSPACE. */
dsa_status_t dsa_dense_mla_workspace_size(const dsa_batch_t* batch, const dsa_mla_t* mla, size_t* bytes);
dsa_status_t dsa_dense_mla(const dsa_batch_t* batch, const dsa_mla_t* mla, void* out, float* lse, void* ws,
                           size_t ws_bytes, cudaStream_t stream);

/* Producer step of the indexer inputs: per-group absmax e4m3 quantisation
 * ("DeepSeek V3.2: How Far Can Open Models Go If You Actually Try?", §3.1:
 * the indexer runs in FP8; e4m3 codes with one fp32 scale per query token and
 * per key row).  x holds `groups` groups of `group_elems` consecutive values
 * (dtype F32 or BF16): a token's H_I x d_I indexer query (group_elems =
 * 64 * 128) or a key row (group_elems = 128).  For each group:
 *   scales[g] = amax / 448 in fp32 (1 when amax = 0),
 *   codes[g * group_elems + i] = e4m3(x / scales[g]), the division in IEEE
 *   fp32, rounded to nearest even and saturated at +-448.
 * codes and scales may point into a larger cache at a row offset (appending
 * new keys to a key cache).  group_elems must be a multiple of 4 in
 * [4, 16384]; x must be 16-byte aligned, codes and scales 4-byte aligned,
 * else DSA_ERROR_INVALID_VALUE.  groups = 0 is a no-op.  Caller-owned
 * device memory; enqueued on `stream`. */
dsa_status_t dsa_quantize_e4m3(const void* x, dsa_dtype_t x_dtype, int64_t groups, int32_t group_elems,
                               uint8_t* codes, float* scales, cudaStream_t stream);

/* The lightning indexer's dense warm-up loss and its gradient ("DeepSeek V3.2:
 * How Far Can Open Models Go If You Actually Try?", §3.3, Stage 1:
 * L_I = sum_t KL(p_t || softmax(I_t)); "DeepSeek-V3.2: Pushing the Frontier
 * of Open Large Language Models", Modeling, Objective Functions: p_t is the
 * main attention's dense scores aggregated over the heads, L1-normalised).
 * For every query row t with candidates s = 0..p (the causal domain of the
 * forward pass):
 *   p_t[s] = (1/H) sum_h softmax_s(mla.scale * mla.q[t,h] . mla.kv[s]),
 *   I_t    = the index scores of dsa_index_scores,
 *   loss_rows[t] = sum_s p_t[s] (log p_t[s] - log softmax(I_t)_s), 0 log 0 = 0,
 * and the gradients of sum_t loss_rows[t] with respect to the real-valued
 * indexer inputs (code * scale for E4M3) and the head weights, ReLU'(0) = 0:
 *   dq [total_q, n_heads, head_dim], dk [total_kv, head_dim], dw [total_q,
 *   n_heads], all fp32 and overwritten (keys of no query row get 0).
 * loss_rows [total_q] fp32.  The mla value columns are not read.  Arithmetic
 * is fp32 on CUDA cores (the indexer scores use the forward kernels); the
 * workspace holds (3 + n_heads) * round_up(max_seqlen_kv, 4) fp32 per query
 * row of a chunk (dsa_indexer_loss_workspace_size: min_bytes = one row,
 * preferred_bytes = every row at once, up to 65535 rows per chunk).  Same
 * shape support as the forward's CUDA-core kernels (n_heads <= 64,
 * head_dim <= 128; MLA d_qk <= 1024, BF16 or F32).  All pointers 16-byte
 * aligned device memory; errors as dsa_forward. */
dsa_status_t dsa_indexer_loss_workspace_size(const dsa_batch_t* batch, const dsa_indexer_t* indexer,
                                             const dsa_mla_t* mla, size_t* min_bytes, size_t* preferred_bytes);
dsa_status_t dsa_indexer_warmup_loss(const dsa_batch_t* batch, const dsa_indexer_t* indexer,
                                     const dsa_mla_t* mla, float* loss_rows, float* dq, float* dk, float* dw,
                                     void* ws, size_t ws_bytes, cudaStream_t stream);

/* The whole forward pass: steps 1-3 for every query row, processed in query
 * chunks sized to ws_bytes.  out/lse as dsa_sparse_mla; idx_out (nullable)
 * [total_q, k] receives the selected positions as dsa_topk writes them. */
dsa_status_t dsa_forward(const dsa_batch_t* batch, const dsa_indexer_t* indexer,
                         const dsa_mla_t* mla, int32_t k, void* out, float* lse,
                         int32_t* idx_out, void* ws, size_t ws_bytes, cudaStream_t stream);

/* dsa_forward with an optional launch trace (trace may be NULL). */
dsa_status_t dsa_forward_traced(const dsa_batch_t* batch, const dsa_indexer_t* indexer,
                                const dsa_mla_t* mla, int32_t k, void* out, float* lse,
                                int32_t* idx_out, void* ws, size_t ws_bytes,
                                cudaStream_t stream, dsa_trace_t* trace);

/* Host copies of the inputs of dsa_forward_streamed.  Each pointer is the
 * host-memory counterpart of the device tensor with the same role in
 * dsa_indexer_t / dsa_mla_t (same shape and dtype); q_scale / k_scale are
 * NULL exactly when the device ones are.  Page-locked (pinned) host memory
 * lets the copies overlap the kernels; pageable memory works but serialises
 * them. */
typedef struct {
  const void* idx_q;       /* indexer q        [total_q, n_heads, head_dim] */
  const float* idx_q_scale;/* indexer q_scale  [total_q] or NULL */
  const void* idx_k;       /* indexer k        [total_kv, head_dim] */
  const float* idx_k_scale;/* indexer k_scale  [total_kv] or NULL */
  const float* idx_w;      /* indexer w        [total_q, n_heads] */
  const void* mla_q;       /* mla q            [total_q, n_heads, d_qk] */
  const void* mla_kv;      /* mla kv           [total_kv, d_qk] */
} dsa_host_inputs_t;

/* dsa_forward for inputs that live in host memory, with the output returned
 * to host memory.  The pages have no counterpart: this is the serving-side
 * integration of the same three steps.
 *
 * Copies and kernels overlap:
 *   - the key-side inputs (indexer k, k_scale and the latent cache) are
 *     copied in full first;
 *   - the query-side inputs are copied chunk by chunk on copy_in, in query
 *     chunks of up to 4096 rows (fewer if the workspace holds fewer);
 *   - each chunk's kernels run on `stream` once its inputs have arrived;
 *   - its out / lse rows return on copy_out while later chunks compute.
 *
 * The device tensors named in indexer / mla, and out / lse, are caller-owned
 * device buffers of the full size: they receive the copies and the results.
 * host_out [total_q, mla n_heads, d_v] and host_lse [total_q, n_heads]
 * (nullable; needs lse) receive the results.
 *
 * Stream order: the call's work starts after the work already enqueued on
 * `stream`, and work enqueued on `stream` afterwards sees every result,
 * including the host copies.  copy_in and copy_out may equal `stream` (no
 * overlap).  Errors as dsa_forward, plus DSA_ERROR_INVALID_VALUE for a
 * missing host pointer. */
dsa_status_t dsa_forward_streamed(const dsa_batch_t* batch, const dsa_indexer_t* indexer,
                                  const dsa_mla_t* mla, int32_t k, const dsa_host_inputs_t* host,
                                  void* out, float* lse, void* host_out, float* host_lse,
                                  void* ws, size_t ws_bytes, cudaStream_t stream,
                                  cudaStream_t copy_in, cudaStream_t copy_out);

/* Synchronises `stream`, then reads and clears the current device's error word
 * (DSA_DEVERR_* bits) into *flags.  Returns DSA_ERROR_TIMEOUT or
 * DSA_ERROR_BAD_INDEX when the corresponding bit was set, else DSA_SUCCESS. */
dsa_status_t dsa_read_device_errors(cudaStream_t stream, uint32_t* flags);

/* Static description of a status code. */
const char* dsa_status_string(dsa_status_t status);

/* Detail of the last non-success status returned on this host thread. */
const char* dsa_last_error_message(void);

/* ABI version compiled into the library (DSA_ABI_VERSION). */
int32_t dsa_abi_version(void);

/* Test hook for the bounded-wait failure path.  The next tensor-core indexer
 * launch of this process runs with the given mode: 1 = its producer skips the
 * load of one key tile, so the MMA warp's wait runs out after its time limit
 * (about 2 s), the kernel gives up cleanly and DSA_DEVERR_TIMEOUT is set.
 * 0 = normal.  Not for production use. */
void dsa_debug_inject_fault(uint32_t mode);

#ifdef __cplusplus
}
#endif

#endif /* DSA_H_ */
