"""dsa_indexer_warmup_loss (the indexer's dense warm-up KL loss, forward and
backward) against the fp64 oracle's indexer_warmup_loss.

Tolerances (fp32 arithmetic against fp64): the target p_t takes 576-term
fp32 dot products and softmaxes over at most a few hundred candidates, and
each gradient entry is an fp32 sum of at most a few hundred products, so the
relative error stays well below 1e-4 of the largest magnitude.  On
integer-grid indexer inputs with power-of-two scales every index score and
every q.k product is exact in fp32, so the ReLU decisions equal the
oracle's; there the bound is 1e-4 of the largest reference magnitude.  On
random e4m3 inputs a product within fp32 rounding of 0 may take the other
side of the ReLU, a discrete change of one term, so the gradient bound is
2e-3 of the largest reference magnitude; the losses keep 1e-4."""

import numpy as np
import pytest
import torch

import dsa_synth
import oracle
import sparse_long_context_07_b300 as dsa
from tests.gpu_util import row_meta, structs
from tests.helpers import cu_np, idx_real, mla_real

pytestmark = pytest.mark.gpu


def _run(wl, ws_bytes=None):
    b, ix, m = structs(wl)
    T, S = wl.total_q, wl.total_kv
    HI, D = wl.n_idx_heads, wl.idx_dim
    loss = torch.full((T,), float("nan"), device="cuda")
    dq = torch.full((T, HI, D), float("nan"), device="cuda")
    dk = torch.full((S, D), float("nan"), device="cuda")
    dw = torch.full((T, HI), float("nan"), device="cuda")
    mn, pref = dsa.indexer_loss_workspace_size(b, ix, m)
    ws = torch.empty(ws_bytes or pref, dtype=torch.uint8, device="cuda")
    dsa.indexer_warmup_loss(b, ix, m, loss, dq, dk, dw, ws)
    torch.cuda.synchronize()
    assert dsa.read_device_errors() == 0
    return [t.cpu().numpy().astype(np.float64) for t in (loss, dq, dk, dw)]


def _oracle(wl):
    cu_q, cu_kv = cu_np(wl)
    q = idx_real(wl, "q")
    k = idx_real(wl, "k")
    w = wl.w.cpu().numpy().astype(np.float64)
    Q = mla_real(wl.Q)
    kv = mla_real(wl.KV)
    total, dq, dk, dw = oracle.indexer_warmup_loss(q, k, w, Q, kv, cu_q, cu_kv, wl.scale)
    rows = [oracle.indexer_warmup_loss(q, k, w, Q, kv, cu_q, cu_kv, wl.scale, rows=[r])[0]
            for r in range(wl.total_q)]
    return np.asarray(rows), total, dq, dk, dw


def _close(got, ref, rel, what):
    tol = rel * max(np.abs(ref).max(), 1e-30) + 1e-7
    err = np.abs(got - ref).max()
    assert err <= tol, f"{what}: max abs err {err:.3e} > {tol:.3e}"


def _check(wl, got, ref, grad_rel):
    loss, dq, dk, dw = got
    ref_rows, ref_total, rdq, rdk, rdw = ref
    assert np.all(np.abs(loss - ref_rows) <= 1e-4 * np.abs(ref_rows) + 1e-5), np.abs(loss - ref_rows).max()
    assert abs(loss.sum() - ref_total) <= 1e-4 * abs(ref_total) + 1e-5
    _close(dq, rdq, grad_rel, "dq")
    _close(dk, rdk, grad_rel, "dk")
    _close(dw, rdw, grad_rel, "dw")


def _grid_workload(seed):
    # production dimensions; indexer codes on the integer grid with scales
    # 1/64 (powers of two), so every q.k product and index score is exact
    wl = dsa_synth.make_workload("kl-grid", [40, 1, 7], [40, 300, 90], grid=True, device="cuda", seed=seed)
    wl.q_scale.fill_(1.0 / 64)
    wl.k_scale.fill_(1.0 / 64)
    return wl


def test_warmup_loss_integer_grid_production_dims():
    wl = _grid_workload(61)
    _check(wl, _run(wl), _oracle(wl), 1e-4)


def test_warmup_loss_random_e4m3():
    wl = dsa_synth.make_workload("kl-rand", [30, 1, 1], [30, 257, 129], device="cuda", seed=62)
    _check(wl, _run(wl), _oracle(wl), 2e-3)


def test_warmup_loss_fp32_small_dims():
    # the tiny workload's shapes: fp32 indexer 4 x 32, 8 heads of width 64
    wl = dsa_synth.make_workload("kl-tiny", [64, 1], [64, 80], n_idx_heads=4, idx_dim=32, idx_dtype="f32",
                                 n_heads=8, d_qk=64, d_v=64, mla_dtype="f32", topk=32, scale=0.125,
                                 device="cuda", seed=63)
    _check(wl, _run(wl), _oracle(wl), 1e-4)


def test_warmup_loss_chunking_matches():
    # the minimum workspace processes one query row per chunk; the key
    # gradient accumulates over chunks to the same result
    wl = _grid_workload(64)
    b, ix, m = structs(wl)
    mn, pref = dsa.indexer_loss_workspace_size(b, ix, m)
    a = _run(wl, ws_bytes=mn)
    c = _run(wl)
    for x, y, name in zip(a, c, ("loss", "dq", "dk", "dw")):
        _close(x, y, 1e-5, f"chunked {name}")
    with pytest.raises(dsa.DSAError) as e:
        _run(wl, ws_bytes=mn - 256)
    assert e.value.status == dsa.ERROR_INSUFFICIENT_WORKSPACE


def test_warmup_loss_is_zero_when_the_indexer_matches_the_target():
    # a one-candidate row has p = softmax(I) = 1: zero loss and zero gradient
    wl = dsa_synth.make_workload("kl-one", [1], [1], device="cuda", seed=65)
    loss, dq, dk, dw = _run(wl)
    assert loss[0] == 0.0 and not dq.any() and not dk.any() and not dw.any()
