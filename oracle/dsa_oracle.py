"""fp64 CPU oracle of the DSA forward pass (indexer -> top-k -> sparse MLA-MQA).

TEST INFRASTRUCTURE ONLY (see the package docstring): the product path never
imports this module.

Sources ("the pages"):
  [P1] "DeepSeek V3.2: How Far Can Open Models Go If You Actually Try?"
       §2.2 (MLA: one shared latent K/V bank, all heads read it),
       §3.1 (lightning indexer equation, FP8, top-k selection, attention over
       the selected latents, MQA sharing), §3.4 (short prompts behave as dense
       masked attention).
  [P2] "DeepSeek-V3.2: Pushing the Frontier of Open Large Language Models",
       System Modules (indexer over preceding tokens; top-k operation; MLA in
       MQA mode), Key Hyperparameters (selected_tokens_k = 2048).
  [P4] "DeepSeek-V3.2" (Baseten blog), §(1) DSA + MLA (indexer scores all past
       tokens, token selector keeps 2,048 of 128k).
  [OCP] OCP 8-bit Floating Point Specification (OFP8), E4M3 encoding: the
       pages only say "FP8"; the e4m3 variant and the per-token fp32 scales are
       the workload's stated input format.

Readings taken where the pages are silent (each also listed in the design notes):
  * Causal domain: query at position p sees keys s in [0, p] (self included).
  * Ragged batches are bottom-right aligned: query i of a sequence with nq
    queries and nkv keys sits at p = nkv - nq + i.
  * Fewer candidates than k: all candidates are selected, the rest is -1.
  * Ties in the index score: the lower key position wins; -0.0 equals +0.0.
  * Returned index sets are in ascending key position.
  * Quantised inputs: the real q_I / k_I are code * per-row fp32 scale
    (one scale per query token shared by its heads, one per key row).
  * V is the first d_v columns of the same latent row that serves as K.
  * The softmax scale multiplies q.k before the softmax.
  * Selected entries equal to -1 are skipped; a row with nothing selected has
    output 0 and lse -inf.
"""

from __future__ import annotations

import numpy as np

# ----------------------------------------------------------------------------
# Input decoding
# ----------------------------------------------------------------------------


def decode_e4m3(codes: np.ndarray) -> np.ndarray:
    """Decode OCP E4M3 bytes to float64 from the bit fields [OCP, E4M3].

    Layout: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits.
      exponent 0          -> subnormal   (-1)^s * 2^-6 * m/8
      exponent 1..15      -> normal      (-1)^s * 2^(e-7) * (1 + m/8)
      exponent 15, m = 7  -> NaN (the format has no infinities)
    """
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where((c >> 7) & 1, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    normal = sign * np.power(2.0, (e - 7).astype(np.float64)) * (1.0 + m / 8.0)
    sub = sign * (2.0 ** -6) * (m / 8.0)
    out = np.where(e == 0, sub, normal)
    out = np.where((e == 15) & ((c & 0x7) == 7), np.nan, out)
    return out


def encode_e4m3(values: np.ndarray) -> np.ndarray:
    """Encode float values to OCP E4M3 bytes [OCP, E4M3], rounding to nearest
    with ties to even and saturating at the largest finite magnitude, 448.

    The values are taken exactly (float64 holds every float32).  Normal codes
    are 2^(e-7) * (1 + m/8) for e = 1..15 (e = 15 with m = 7 is NaN, so the
    top finite value is 2^8 * 1.75 = 448); subnormals are 2^-6 * m/8.  A value
    is rounded on the grid of its binade: step 2^(E-3) for |v| in [2^E, 2^(E+1))
    with E >= -6, step 2^-9 below 2^-6.  -0.0 encodes as 0x80.
    """
    v = np.asarray(values, dtype=np.float64)
    out = np.zeros(v.shape, dtype=np.uint8)
    flat_v = v.reshape(-1)
    flat_o = out.reshape(-1)
    for i, x in enumerate(flat_v):
        sign = 0x80 if np.signbit(x) else 0x00
        a = abs(float(x))
        if a >= 448.0:
            flat_o[i] = sign | 0x7E
            continue
        if a < 2.0 ** -6:
            step = 2.0 ** -9                    # subnormal grid (and the first normal)
        else:
            E = int(np.floor(np.log2(a)))
            # guard the floor of log2 at exact powers of two
            if 2.0 ** E > a:
                E -= 1
            elif 2.0 ** (E + 1) <= a:
                E += 1
            step = 2.0 ** (E - 3)
        q = a / step                            # exact: step is a power of two
        n = np.floor(q)
        r = q - n
        if r > 0.5 or (r == 0.5 and int(n) % 2 == 1):
            n += 1
        y = n * step                            # the rounded magnitude
        if y >= 448.0:
            flat_o[i] = sign | 0x7E
            continue
        if y < 2.0 ** -6:
            code = int(round(y / 2.0 ** -9))    # subnormal m (0..7)
        else:
            E = int(np.floor(np.log2(y)))
            if 2.0 ** E > y:
                E -= 1
            elif 2.0 ** (E + 1) <= y:
                E += 1
            m = int(round((y / 2.0 ** E - 1.0) * 8.0))
            code = ((E + 7) << 3) | m
        flat_o[i] = sign | code
    return out


def quantize_e4m3_groups(x32: np.ndarray, group_elems: int):
    """Per-group absmax quantisation to E4M3 (the format of the indexer
    inputs, "FP8" [P1 §3.1], one fp32 scale per group): for each group of
    `group_elems` consecutive values, scale = amax / 448 in fp32 (1 when
    amax = 0) and code = E4M3(x / scale), the division done in fp32 -- the
    precision in which the kernel takes the same decision -- then rounded to
    nearest even with saturation.  x32: float32 array whose size is a multiple
    of group_elems.  Returns (uint8 codes of x's shape, float32 scales)."""
    x = np.asarray(x32, dtype=np.float32)
    g = x.reshape(-1, group_elems)
    amax = np.abs(g).max(axis=1)
    scale = np.where(amax > 0, amax / np.float32(448.0), np.float32(1.0)).astype(np.float32)
    y = (g / scale[:, None]).astype(np.float32)     # IEEE fp32 division
    codes = encode_e4m3(y).reshape(x.shape)
    return codes, scale


def decode_bf16(bits: np.ndarray) -> np.ndarray:
    """Decode bfloat16 bit patterns (uint16) to float64: a bf16 value is the
    upper half of the float32 with the same bits."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


# ----------------------------------------------------------------------------
# Batch geometry
# ----------------------------------------------------------------------------


def query_positions(cu_q: np.ndarray, cu_kv: np.ndarray):
    """Per query row r: (sequence b, position p, first key row of b, n = p+1).

    Bottom-right alignment (prefill nq = nkv gives p = i; decode nq = 1 gives
    p = nkv - 1, the cached row of the query itself).  Causal domain from [P1
    §3.1] ("previous token at position s") read as s <= p.
    """
    cu_q = np.asarray(cu_q, dtype=np.int64)
    cu_kv = np.asarray(cu_kv, dtype=np.int64)
    T = int(cu_q[-1])
    seq = np.empty(T, np.int64)
    pos = np.empty(T, np.int64)
    kv0 = np.empty(T, np.int64)
    for b in range(len(cu_q) - 1):
        nq = cu_q[b + 1] - cu_q[b]
        nkv = cu_kv[b + 1] - cu_kv[b]
        if nq > nkv:
            raise ValueError("each sequence needs nkv >= nq")
        i = np.arange(nq)
        seq[cu_q[b]:cu_q[b + 1]] = b
        pos[cu_q[b]:cu_q[b + 1]] = nkv - nq + i
        kv0[cu_q[b]:cu_q[b + 1]] = cu_kv[b]
    return seq, pos, kv0, pos + 1


# ----------------------------------------------------------------------------
# Step 1: lightning indexer  [P1 §3.1 indexer equation; P2 System Modules]
# ----------------------------------------------------------------------------


def index_scores_row(q_t: np.ndarray, k_seq: np.ndarray, w_t: np.ndarray) -> np.ndarray:
    """I[t, s] = sum_j w[t, j] * ReLU(q_I[t, j] . k_I[s]) for s = 0..n-1.

    q_t   : [H_I, d]  real-valued indexer queries of token t (already scaled)
    k_seq : [n, d]    real-valued indexer keys s = 0..p of t's sequence
    w_t   : [H_I]     per-head weights of token t
    The key has no head index: one key per token serves every indexer head.
    """
    x = q_t @ k_seq.T                      # [H_I, n]   q_I[t,j] . k_I[s]
    relu = np.maximum(x, 0.0)              # ReLU
    return w_t @ relu                      # sum over heads j


def index_scores(q, k, w, cu_q, cu_kv, rows=None):
    """Index scores for each requested query row (default: all rows).

    q : [T, H_I, d] float64 (code * q_scale), k : [S, d] float64 (code *
    k_scale), w : [T, H_I].  Returns a list with one float64 vector of length
    n = p + 1 per requested row (the candidates s = 0..p).
    """
    _, pos, kv0, n = query_positions(cu_q, cu_kv)
    if rows is None:
        rows = range(len(pos))
    out = []
    for r in rows:
        ks = k[kv0[r]:kv0[r] + n[r]]
        out.append(index_scores_row(q[r], ks, w[r]))
    return out


# ----------------------------------------------------------------------------
# Step 2: fine-grained top-k selection  [P1 §3.1; P2 "Top-k operation"]
# ----------------------------------------------------------------------------


def topk_indices(scores: np.ndarray, k: int) -> np.ndarray:
    """Indices of the k largest scores, ascending, padded with -1 to length k.

    Full sort by (score descending, position ascending), keep the first
    min(k, n).  -0.0 and +0.0 are the same score (adding +0.0 maps -0.0 to
    +0.0).
    """
    v = np.asarray(scores, dtype=np.float64) + 0.0
    n = v.shape[0]
    order = np.lexsort((np.arange(n), -v))  # primary: -v ascending; then position
    keep = np.sort(order[:min(k, n)])
    out = np.full(k, -1, dtype=np.int32)
    out[:keep.shape[0]] = keep
    return out


# ----------------------------------------------------------------------------
# Step 3: sparse MLA in MQA mode  [P1 §2.2, §3.1 attention over selected
# latents; P2 "Modified MLA in MQA mode"]
# ----------------------------------------------------------------------------


def sparse_mla_row(Q_t: np.ndarray, kv_seq: np.ndarray, idx_row: np.ndarray,
                   scale: float, d_v: int):
    """u_t = Attn(h_t, {c_s : s in selected set}) for one query token.

    Q_t    : [H, d_qk]   query heads of token t, in the latent space
    kv_seq : [nkv, d_qk] shared latent rows c_s of t's sequence (one row per
                         token, read by every head: MQA)
    idx_row: [k]         selected positions, -1 = empty slot
    Softmax over the selected set of scale * (Q_t[h] . c_s); the value is the
    first d_v columns of the same latent row.  Returns (out [H, d_v],
    lse [H]) with lse = log sum_s exp(scale * Q_t[h] . c_s) (natural log).
    """
    sel = np.asarray(idx_row)
    sel = sel[sel >= 0]
    H = Q_t.shape[0]
    if sel.shape[0] == 0:
        return np.zeros((H, d_v)), np.full(H, -np.inf)
    c = kv_seq[sel]                        # [n, d_qk]
    z = scale * (Q_t @ c.T)                # [H, n]
    m = z.max(axis=1, keepdims=True)
    e = np.exp(z - m)
    l = e.sum(axis=1, keepdims=True)
    out = (e @ c[:, :d_v]) / l
    lse = (m + np.log(l))[:, 0]
    return out, lse


def sparse_mla(Q, kv, idx, cu_q, cu_kv, scale, d_v, rows=None):
    """sparse_mla_row over requested rows; Q [T, H, d_qk], kv [S, d_qk],
    idx [T, k] sequence-local positions.  Returns (out [R, H, d_v], lse [R, H])."""
    _, pos, kv0, n = query_positions(cu_q, cu_kv)
    if rows is None:
        rows = range(len(pos))
    outs, lses = [], []
    for r in rows:
        seq_kv = kv[kv0[r]:kv0[r] + n[r]]  # causal: only rows 0..p exist for t
        o, l = sparse_mla_row(Q[r], seq_kv, idx[r], scale, d_v)
        outs.append(o)
        lses.append(l)
    return np.stack(outs), np.stack(lses)


def lse_merge(outs, lses):
    """Merge attention results over disjoint key subsets:
    lse = log sum_i exp(lse_i),  out = sum_i exp(lse_i - lse) * out_i.
    (Follows from splitting the softmax normaliser; used for split-KV decode.)"""
    lses = np.stack(lses)                  # [n_split, H]
    outs = np.stack(outs)                  # [n_split, H, d_v]
    m = lses.max(axis=0)
    finite = np.isfinite(m)
    msafe = np.where(finite, m, 0.0)
    wts = np.exp(lses - msafe)             # [n_split, H]
    tot = wts.sum(axis=0)
    lse = np.where(finite, msafe + np.log(np.where(tot > 0, tot, 1.0)), -np.inf)
    out = np.einsum("sh,shd->hd", wts, outs) / np.where(tot > 0, tot, 1.0)[:, None]
    return out, lse


# ----------------------------------------------------------------------------
# The whole forward pass for selected rows
# ----------------------------------------------------------------------------


def forward_rows(q, k, w, Q, kv, cu_q, cu_kv, topk, scale, d_v, rows):
    """Indexer -> top-k -> sparse MLA for each requested query row
    [P1 §3.1: u_t = Attn(h_t, {c_s : I_{t,s} in Top-k(I_{t,:})})].

    Returns (scores list, idx [R, topk], out [R, H, d_v], lse [R, H]).
    """
    _, pos, kv0, n = query_positions(cu_q, cu_kv)
    scores, idxs, outs, lses = [], [], [], []
    for r in rows:
        I = index_scores_row(q[r], k[kv0[r]:kv0[r] + n[r]], w[r])
        sel = topk_indices(I, topk)
        o, l = sparse_mla_row(Q[r], kv[kv0[r]:kv0[r] + n[r]], sel, scale, d_v)
        scores.append(I)
        idxs.append(sel)
        outs.append(o)
        lses.append(l)
    return scores, np.stack(idxs), np.stack(outs), np.stack(lses)
