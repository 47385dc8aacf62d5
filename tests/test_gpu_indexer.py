"""dsa_index_scores against the oracle's index scores.

Integer-grid inputs make every score an exact small integer, so the FP8
tensor-core kernel must match the fp64 oracle bit for bit; random e4m3 inputs
are compared within fp32 accumulation error.  Columns beyond each row's
candidates must stay untouched."""

import numpy as np
import pytest
import torch

import dsa_synth
import sparse_long_context_07_b300 as dsa
from tests.gpu_util import oracle_scores, oracle_scores_cached, row_meta, sample_rows, structs

pytestmark = pytest.mark.gpu

SENTINEL = 12345.5


def _run(wl, ld=None):
    b, ix, _ = structs(wl)
    ld = ld or ((wl.max_kv + 3) // 4 * 4 + 4)
    scores = torch.full((wl.total_q, ld), SENTINEL, device="cuda")
    dsa.index_scores(b, ix, scores, ld)
    torch.cuda.synchronize()
    assert dsa.read_device_errors() == 0
    return scores.cpu().numpy()


# ragged mix: two prefills, a 5-token chunk appended to 695 cached tokens and a
# 1-token decode over 1000 cached tokens; several 128-key tiles and ragged tails
RAGGED_Q = [300, 1, 5, 130]
RAGGED_KV = [300, 1000, 700, 130]


def test_indexer_tc_integer_grid_bit_exact():
    wl = dsa_synth.make_workload("idx-grid", RAGGED_Q, RAGGED_KV, grid=True, device="cuda",
                                 n_heads=8, d_qk=64, d_v=64)
    S = _run(wl)
    _, pos, _, n = row_meta(wl)
    rows = list(range(wl.total_q))
    ref = oracle_scores(wl, rows)
    for r in rows:
        assert np.array_equal(S[r, :n[r]].astype(np.float64), ref[r]), f"row {r}"
        assert np.all(S[r, n[r]:] == SENTINEL), f"row {r} wrote past its candidates"


def test_indexer_tc_random_e4m3():
    wl = dsa_synth.make_workload("idx-rand", [1000, 1, 1, 1], [1000, 5000, 300, 129], device="cuda",
                                 seed=7, n_heads=8, d_qk=64, d_v=64)
    S = _run(wl)
    _, pos, _, n = row_meta(wl)
    rows = sample_rows(wl.total_q, 120, seed=1, must=[0, 1, 127, 128, 999, 1000, 1001, 1002])
    ref = oracle_scores(wl, rows)
    for i, r in enumerate(rows):
        scale = np.abs(ref[i]).max() + 1e-30
        err = np.abs(S[r, :n[r]] - ref[i]).max()
        assert err <= 1e-5 * scale, f"row {r}: rel err {err / scale:.2e}"
        assert np.all(S[r, n[r]:] == SENTINEL)


def test_indexer_simt_fp32_tiny():
    for grid in (False, True):
        wl = dsa_synth.tiny(device="cuda", grid=grid)
        S = _run(wl)
        _, pos, _, n = row_meta(wl)
        rows = list(range(wl.total_q))
        ref = oracle_scores(wl, rows)
        for r in rows:
            if grid:
                assert np.array_equal(S[r, :n[r]].astype(np.float64), ref[r])
            else:
                assert np.abs(S[r, :n[r]] - ref[r]).max() <= 1e-5 * (np.abs(ref[r]).max() + 1e-30)


def test_indexer_tc_prefill32k_sampled():
    wl = dsa_synth.prefill32k(device="cuda")
    S = _run(wl, ld=32768)
    _, pos, _, n = row_meta(wl)
    rows = sample_rows(wl.total_q, 12, seed=3, must=[0, 2047, 2048, 32767])
    ref = oracle_scores_cached(wl, rows, {})
    for i, r in enumerate(rows):
        scale = np.abs(ref[i]).max() + 1e-30
        assert np.abs(S[r, :n[r]] - ref[i]).max() <= 1e-5 * scale, f"row {r}"
