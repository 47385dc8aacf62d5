"""fp64 CPU oracle of the indexer's dense warm-up loss and its gradient.

TEST INFRASTRUCTURE ONLY (see the package docstring): the product path never
imports this module.

Sources:
  [P1] "DeepSeek V3.2: How Far Can Open Models Go If You Actually Try?", §3.3
       (Stage 1, dense warm-up with the model frozen): the indexer is trained
       to match where dense attention goes, with
           L_I = sum_t KL( p_t || softmax(I_t) ).
  [P2] "DeepSeek-V3.2: Pushing the Frontier of Open Large Language Models",
       Modeling, Objective Functions (the indexer's warm-up objective): the
       KL divergence between the aggregated dense attention scores,
       L1-normalised, and the indexer outputs.

Readings taken where the pages are silent (each also listed in the design notes):
  * "Aggregated dense attention scores": the per-head softmax distributions
    of the main (MLA-MQA) attention over the causal candidates s = 0..p,
    summed over the heads; L1 normalisation then divides by their sum, H.
  * softmax(I_t) runs over the same causal candidates s = 0..p.
  * KL(p || q) = sum_s p_s (log p_s - log q_s), with 0 log 0 = 0.
  * The gradient is taken with respect to the real-valued indexer inputs
    (q_I, k_I after their scales, and w); ReLU'(0) = 0.
"""

from __future__ import annotations

import numpy as np

from .dsa_oracle import index_scores_row, query_positions


def dense_attention_target_row(Q_t: np.ndarray, kv_seq: np.ndarray, scale: float) -> np.ndarray:
    """p_t[s] for s = 0..n-1: the H per-head softmax distributions of
    scale * (Q_t[h] . c_s) over the candidates, summed over h and
    L1-normalised (divided by their total, H)."""
    z = scale * (Q_t @ kv_seq.T)           # [H, n]
    z = z - z.max(axis=1, keepdims=True)
    a = np.exp(z)
    a = a / a.sum(axis=1, keepdims=True)   # per-head attention distribution
    agg = a.sum(axis=0)                    # aggregated over heads
    return agg / agg.sum()                 # L1-normalised


def kl_to_softmax_row(p_t: np.ndarray, I_t: np.ndarray):
    """KL(p_t || softmax(I_t)) and its gradient with respect to I_t.

    log softmax(I)_s = I_s - log sum_u exp(I_u).  Since sum_s p_s = 1, the
    gradient of the KL with respect to I_s is softmax(I)_s - p_s.
    """
    m = I_t.max()
    log_z = m + np.log(np.exp(I_t - m).sum())
    log_q = I_t - log_z
    pos = p_t > 0
    loss = float(np.sum(p_t[pos] * (np.log(p_t[pos]) - log_q[pos])))
    grad = np.exp(log_q) - p_t
    return loss, grad


def indexer_scores_backward_row(g_t: np.ndarray, q_t: np.ndarray, k_seq: np.ndarray,
                                w_t: np.ndarray):
    """Back-propagate dL/dI_t through I_t[s] = sum_j w_j ReLU(q_j . k_s).

    g_t : [n] gradient with respect to I_t;  q_t [H_I, d], k_seq [n, d],
    w_t [H_I] as in index_scores_row.  Returns (dq [H_I, d], dk [n, d],
    dw [H_I]).
    """
    x = q_t @ k_seq.T                      # [H_I, n]
    relu = np.maximum(x, 0.0)
    dw = relu @ g_t                        # dI_s/dw_j = ReLU(x_js)
    dx = (w_t[:, None] * (x > 0)) * g_t[None, :]   # dI_s/dx_js = w_j 1[x_js > 0]
    dq = dx @ k_seq                        # dx_js/dq_j = k_s
    dk = dx.T @ q_t                        # dx_js/dk_s = q_j
    return dq, dk, dw


def indexer_warmup_loss(q, k, w, Q, kv, cu_q, cu_kv, scale, rows=None):
    """L_I over the requested query rows (default: all) and its gradients.

    q [T, H_I, d_I], k [S, d_I] (real-valued indexer inputs), w [T, H_I];
    Q [T, H, d_qk], kv [S, d_qk] (the main attention's inputs; V is not
    needed).  Returns (loss, dq [T, H_I, d_I], dk [S, d_I], dw [T, H_I]); the
    gradients are zero outside the requested rows and their keys.
    """
    _, pos, kv0, n = query_positions(cu_q, cu_kv)
    if rows is None:
        rows = range(len(pos))
    dq = np.zeros_like(q, dtype=np.float64)
    dk = np.zeros_like(k, dtype=np.float64)
    dw = np.zeros_like(w, dtype=np.float64)
    total = 0.0
    for r in rows:
        a, b = kv0[r], kv0[r] + n[r]
        p_t = dense_attention_target_row(Q[r], kv[a:b], scale)
        I_t = index_scores_row(q[r], k[a:b], w[r])
        loss, g = kl_to_softmax_row(p_t, I_t)
        total += loss
        gq, gk, gw = indexer_scores_backward_row(g, q[r], k[a:b], w[r])
        dq[r] += gq
        dk[a:b] += gk
        dw[r] += gw
    return total, dq, dk, dw
