"""dsa_forward (indexer -> top-k -> sparse MLA) against the oracle's forward
pass on the same inputs.

Selection: bit-exact on integer-grid indexer inputs; on random inputs the
sets may differ only at positions whose oracle score lies within 1e-3 of the
oracle's k-th score.  Output: max-abs 2e-2, mean-abs 2e-3."""

import numpy as np
import pytest
import torch

import dsa_synth
import oracle
import sparse_long_context_07_b300 as dsa
from tests.gpu_util import (assert_attention_close, assert_lse_close, oracle_attention, oracle_scores_cached,
                            row_meta, sample_rows, structs, to_f64)
from tests.helpers import set_rule_ok

pytestmark = pytest.mark.gpu


def run_forward(wl, k, ws_bytes=None):
    b, ix, m = structs(wl)
    T = wl.total_q
    out = torch.full((T, wl.n_heads, wl.d_v), float("nan"), dtype=wl.Q.dtype, device="cuda")
    lse = torch.full((T, wl.n_heads), float("nan"), device="cuda")
    idx = torch.full((T, k), -7, dtype=torch.int32, device="cuda")
    mn, pref = dsa.workspace_size(b, ix, m, k)
    ws = torch.empty(ws_bytes or pref, dtype=torch.uint8, device="cuda")
    dsa.forward(b, ix, m, k, out, lse, idx, ws)
    torch.cuda.synchronize()
    assert dsa.read_device_errors() == 0
    return out, lse, idx


def check_rows(wl, k, out, lse, idx, rows, exact_sets, what, cache=None):
    """Selection of each row against the oracle's top-k (bit-exact, or the
    near-tie set rule), then the oracle's attention over the set the GPU
    returned (once that set has passed) against the GPU's output."""
    cache = {} if cache is None else cache
    scores = oracle_scores_cached(wl, rows, cache)
    gi = idx.cpu().numpy()
    gpu_sets = []
    for i, r in enumerate(rows):
        ref = oracle.topk_indices(scores[i], k)
        if exact_sets:
            assert np.array_equal(gi[r], ref), f"{what}: row {r} selection differs"
        else:
            ok, nd = set_rule_ok(gi[r], ref, scores[i], k)
            assert ok, f"{what}: row {r} selection differs beyond near-ties ({nd})"
            valid = gi[r][gi[r] >= 0]
            assert np.all(np.diff(valid) > 0), f"{what}: row {r} not ascending"
            assert np.all(gi[r][len(valid):] == -1), f"{what}: row {r} padding"
        gpu_sets.append(gi[r])
    # attention of the oracle over the GPU's selection
    ref_o, ref_l = oracle_attention(wl, rows, gpu_sets)
    assert_attention_close(to_f64(out[rows]), ref_o, what)
    assert_lse_close(to_f64(lse[rows]), ref_l, what)


def test_forward_tiny_fp32():
    for grid in (False, True):
        wl = dsa_synth.tiny(device="cuda", grid=grid)
        out, lse, idx = run_forward(wl, wl.topk)
        rows = list(range(wl.total_q))
        cache = {}
        scores = oracle_scores_cached(wl, rows, cache)
        gi = idx.cpu().numpy()
        sels = []
        for r in rows:
            ref = oracle.topk_indices(scores[r], wl.topk)
            if grid:
                assert np.array_equal(gi[r], ref)
            else:
                assert set_rule_ok(gi[r], ref, scores[r], wl.topk)[0]
            sels.append(gi[r] if not grid else ref)
        ref_o, ref_l = oracle_attention(wl, rows, sels)
        assert np.abs(to_f64(out) - ref_o).max() <= 1e-4
        assert np.abs(to_f64(lse) - ref_l).max() <= 1e-4


def test_forward_integer_grid_production_dims():
    # exact FP8 scores: the selected sets must equal the oracle's bit for bit
    k = 256
    wl = dsa_synth.make_workload("fwd-grid", [900, 1, 1, 40], [900, 3000, 257, 300], grid=True,
                                 device="cuda", seed=31)
    out, lse, idx = run_forward(wl, k)
    rows = sample_rows(wl.total_q, 48, seed=1, must=[0, 255, 256, 899, 900, 901, 902, 941])
    check_rows(wl, k, out, lse, idx, rows, True, "grid")


def test_forward_small_workspace_chunks():
    # the minimum workspace forces 64-row chunks; results are unchanged
    k = 128
    wl = dsa_synth.make_workload("fwd-chunk", [300], [300], grid=True, device="cuda", seed=32)
    b, ix, m = structs(wl)
    mn, pref = dsa.workspace_size(b, ix, m, k)
    out1, lse1, idx1 = run_forward(wl, k, ws_bytes=mn)
    out2, lse2, idx2 = run_forward(wl, k)
    assert torch.equal(idx1, idx2)
    assert torch.equal(out1, out2) and torch.equal(lse1, lse2)
    with pytest.raises(dsa.DSAError) as e:
        run_forward(wl, k, ws_bytes=mn - 256)
    assert e.value.status == dsa.ERROR_INSUFFICIENT_WORKSPACE


def test_forward_decode8k():
    wl = dsa_synth.decode8k(device="cuda")
    out, lse, idx = run_forward(wl, wl.topk)
    check_rows(wl, wl.topk, out, lse, idx, list(range(4)), False, "decode8k")


def test_forward_edge_cases():
    # k = 1; a 1-token sequence; candidates fewer than k; an empty query batch
    wl = dsa_synth.make_workload("fwd-edge", [1, 3, 1], [1, 3, 9], grid=True, device="cuda", seed=33)
    for k in (1, 2, 16):
        out, lse, idx = run_forward(wl, k)
        check_rows(wl, k, out, lse, idx, list(range(wl.total_q)), True, f"edge k={k}")
    empty = dsa_synth.make_workload("fwd-empty", [0], [5], grid=True, device="cuda", seed=34)
    b, ix, m = structs(empty)
    out = torch.empty((0, 128, 512), dtype=torch.bfloat16, device="cuda")
    dsa.forward(b, ix, m, 16, out, None, None, torch.empty(16, dtype=torch.uint8, device="cuda"))


def test_forward_misaligned_pointer_rejected():
    wl = dsa_synth.make_workload("fwd-mis", [8], [8], grid=True, device="cuda", seed=35)
    b, ix, m = structs(wl)
    raw = torch.empty(8 * 128 * 512 * 2 + 16, dtype=torch.uint8, device="cuda")
    out = raw[2:2 + 8 * 128 * 512 * 2].view(torch.bfloat16)
    with pytest.raises(dsa.DSAError) as e:
        dsa.forward(b, ix, m, 4, out, None, None, torch.empty(1 << 20, dtype=torch.uint8, device="cuda"))
    assert e.value.status == dsa.ERROR_INVALID_VALUE


def test_forward_decode8k_integer_grid_exact_sets():
    # production dims, k = 2048 over 8192 candidates: the cluster top-k path
    wl = dsa_synth.decode8k(device="cuda", grid=True)
    out, lse, idx = run_forward(wl, wl.topk)
    check_rows(wl, wl.topk, out, lse, idx, list(range(wl.total_q)), True, "decode8k grid")


def test_forward_prefill32k_integer_grid_exact_sets():
    # k = 2048 over up to 32768 candidates, two 16384-row chunks of the
    # forward's workspace: selections bit-exact on both sides of every boundary
    wl = dsa_synth.prefill32k(device="cuda", grid=True)
    out, lse, idx = run_forward(wl, wl.topk)
    T = wl.total_q
    must = [0, 1, 2046, 2047, 2048, 2049, 4095, 4096, 16383, 16384, 16385, 24576, T - 2, T - 1]
    rows = sample_rows(T, 56, seed=3, must=must)
    assert len(rows) >= 64
    check_rows(wl, wl.topk, out, lse, idx, rows, True, "prefill32k grid")
    del wl, out, lse, idx
    torch.cuda.empty_cache()


def test_forward_ragged128k_every_row():
    # all 64 decode rows (contexts of 16K to 128K, planted keys)
    wl = dsa_synth.WORKLOADS["ragged128k"](device="cuda")
    out, lse, idx = run_forward(wl, wl.topk)
    check_rows(wl, wl.topk, out, lse, idx, list(range(wl.total_q)), False, "ragged128k")
    del wl, out, lse, idx
    torch.cuda.empty_cache()


def stratified_rows(T, count, seed, must):
    """`must` plus one seeded row from each of `count` equal strata of [0, T)."""
    g = np.random.default_rng(seed)
    edges = np.linspace(0, T, count + 1).astype(np.int64)
    rows = {int(g.integers(edges[i], max(edges[i] + 1, edges[i + 1]))) for i in range(count)}
    rows |= {int(r) for r in must if 0 <= r < T}
    return sorted(rows)


def test_forward_prefill32k_sampled():
    wl = dsa_synth.prefill32k(device="cuda")
    out, lse, idx = run_forward(wl, wl.topk)
    T = wl.total_q
    rows = stratified_rows(T, 64, seed=7, must=[0, 1, 2047, 2048, 2049, 16383, 16384, T - 1])
    check_rows(wl, wl.topk, out, lse, idx, rows, False, "prefill32k")
    del wl, out, lse, idx
    torch.cuda.empty_cache()


def test_forward_prefill128k_sampled():
    # the bench workload in the bench's launch configuration (preferred
    # workspace: 16384-row chunks); >= 256 rows including both sides of every
    # chunk boundary
    wl = dsa_synth.WORKLOADS["prefill128k"](device="cuda")
    out, lse, idx = run_forward(wl, wl.topk)
    T = wl.total_q
    must = [0, 1, 2047, 2048, 2049, T - 1]
    for c in range(16384, T, 16384):
        must += [c - 1, c]
    rows = stratified_rows(T, 240, seed=5, must=must)
    assert len(rows) >= 256
    check_rows(wl, wl.topk, out, lse, idx, rows, False, "prefill128k")
    del wl, out, lse, idx
    torch.cuda.empty_cache()
