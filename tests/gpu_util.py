"""Helpers for the GPU parity tests: wrap a synthetic workload for the C ABI
and evaluate the oracle on chosen rows of it."""

from __future__ import annotations

import numpy as np
import torch

import oracle
import sparse_long_context_07_b300 as dsa
from tests.helpers import cu_np, idx_real, mla_real

# Attention tolerance for bf16 inputs with fp32 accumulation.
ATT_MAX_ABS = 2e-2
ATT_MEAN_ABS = 2e-3


def structs(wl):
    b = dsa.Batch(wl.cu_q, wl.cu_kv, wl.seqlens_q, wl.seqlens_kv)
    ix = dsa.Indexer(wl.q_idx, wl.k_idx, wl.w, wl.q_scale, wl.k_scale)
    m = dsa.Mla(wl.Q, wl.KV, wl.scale, wl.d_v)
    return b, ix, m


def row_meta(wl):
    cu_q, cu_kv = cu_np(wl)
    seq, pos, kv0, n = oracle.query_positions(cu_q, cu_kv)
    return seq, pos, kv0, n


def oracle_scores(wl, rows):
    """fp64 index scores of the requested rows (list of vectors of length n)."""
    seq, pos, kv0, n = row_meta(wl)
    q = idx_real(wl, "q", rows)
    w = wl.w.index_select(0, torch.as_tensor(np.asarray(rows), device=wl.w.device)).cpu().numpy().astype(np.float64)
    out = []
    for i, r in enumerate(rows):
        kr = np.arange(kv0[r], kv0[r] + n[r])
        k = idx_real(wl, "k", kr)
        out.append(oracle.index_scores_row(q[i], k, w[i]))
    return out


def oracle_attention(wl, rows, idx_rows):
    """fp64 attention of the requested rows over the given selected positions."""
    seq, pos, kv0, n = row_meta(wl)
    Q = mla_real(wl.Q, rows)
    outs, lses = [], []
    for i, r in enumerate(rows):
        sel = np.asarray(idx_rows[i])
        valid = sel[(sel >= 0) & (sel < n[r])]
        # only the selected latent rows are needed
        kv_rows = kv0[r] + valid
        kv = mla_real(wl.KV, kv_rows) if len(kv_rows) else np.zeros((0, wl.d_qk))
        o, l = oracle.sparse_mla_row(Q[i], kv, np.arange(len(valid)), wl.scale, wl.d_v)
        outs.append(o)
        lses.append(l)
    return np.stack(outs), np.stack(lses)


def to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def assert_attention_close(got, ref, what=""):
    d = np.abs(got - ref)
    assert d.max() <= ATT_MAX_ABS, f"{what}: max abs err {d.max():.3e}"
    assert d.mean() <= ATT_MEAN_ABS, f"{what}: mean abs err {d.mean():.3e}"


def assert_lse_close(got, ref, what=""):
    fin = np.isfinite(ref)
    assert np.array_equal(fin, np.isfinite(got)), f"{what}: lse finiteness differs"
    if fin.any():
        d = np.abs(got[fin] - ref[fin])
        assert d.max() <= 1e-2, f"{what}: lse max abs err {d.max():.3e}"


def oracle_scores_cached(wl, rows, cache):
    """Like oracle_scores, decoding every key row of the workload once."""
    seq, pos, kv0, n = row_meta(wl)
    if "k" not in cache:
        cache["k"] = idx_real(wl, "k")
    k = cache["k"]
    q = idx_real(wl, "q", rows)
    w = wl.w.index_select(0, torch.as_tensor(np.asarray(rows), device=wl.w.device)).cpu().numpy().astype(np.float64)
    return [oracle.index_scores_row(q[i], k[kv0[r]:kv0[r] + n[r]], w[i]) for i, r in enumerate(rows)]


def random_selection(wl, k, seed, rows=None):
    """Seeded synthetic index lists: for each row, min(k, n) distinct positions
    of [0, n) in ascending order, then -1 (an input generator, CPU)."""
    seq, pos, kv0, n = row_meta(wl)
    g = torch.Generator()
    g.manual_seed(seed)
    T = len(n)
    idx = torch.full((T, k), -1, dtype=torch.int32)
    for r in range(T) if rows is None else rows:
        m = min(k, int(n[r]))
        sel = torch.randperm(int(n[r]), generator=g)[:m].sort().values
        idx[r, :m] = sel.to(torch.int32)
    return idx


def sample_rows(T, count, seed, must=()):
    g = np.random.default_rng(seed)
    base = set(int(r) for r in must if 0 <= r < T)
    extra = g.choice(T, size=min(T, count), replace=False)
    return sorted(base | set(int(x) for x in extra))
