"""Test helpers: turn a synthetic workload into the oracle's fp64 inputs and
compare results.  The decoding of e4m3 / bf16 bytes is the oracle's own."""

from __future__ import annotations

import os

import numpy as np
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def read_golden(name):
    """Parse a golden fixture: 'key v1 v2 ...' lines; '#' starts a comment.
    Repeated keys are collected in order."""
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, *vals = line.split()
            out.setdefault(key, []).append([float(v) for v in vals])
    return out


def _np(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy()


def idx_real(wl, which, rows=None):
    """Real-valued indexer q (which='q') or k (which='k') as fp64 numpy arrays
    (code * scale), optionally only for the given row indices."""
    codes = wl.q_idx if which == "q" else wl.k_idx
    scale = wl.q_scale if which == "q" else wl.k_scale
    if rows is not None:
        sel = torch.as_tensor(np.asarray(rows), dtype=torch.long, device=codes.device)
        codes = codes.index_select(0, sel)
        scale = None if scale is None else scale.index_select(0, sel)
    if wl.idx_dtype == "e4m3":
        x = oracle.decode_e4m3(_np(codes))
    else:
        x = _np(codes).astype(np.float64)
    if scale is not None:
        s = _np(scale).astype(np.float64)
        x = x * s.reshape((-1,) + (1,) * (x.ndim - 1))
    return x


def mla_real(t: torch.Tensor, rows=None):
    if rows is not None:
        sel = torch.as_tensor(np.asarray(rows), dtype=torch.long, device=t.device)
        t = t.index_select(0, sel)
    if t.dtype == torch.bfloat16:
        return oracle.decode_bf16(_np(t.view(torch.int16)).view(np.uint16))
    return _np(t).astype(np.float64)


def cu_np(wl):
    return _np(wl.cu_q).astype(np.int64), _np(wl.cu_kv).astype(np.int64)


def set_rule_ok(idx_gpu, idx_ref, scores_ref, k, rel=1e-3):
    """The random-input selection rule: the two index sets have the same size
    and every position in their symmetric difference has an oracle score within
    rel * max(|tau|, rms) of tau, the oracle's k-th largest score.  Returns
    (ok, n_diff)."""
    a = set(int(i) for i in idx_gpu if i >= 0)
    b = set(int(i) for i in idx_ref if i >= 0)
    if len(a) != len(b):
        return False, -1
    diff = a ^ b
    if not diff:
        return True, 0
    s = np.asarray(scores_ref, dtype=np.float64)
    tau = np.sort(s)[::-1][min(k, s.shape[0]) - 1]
    tol = rel * max(abs(tau), float(np.sqrt(np.mean(s * s))))
    ok = all(abs(s[i] - tau) <= tol for i in diff)
    return ok, len(diff)
