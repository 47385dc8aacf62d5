"""The fused indexer -> top-k pair (dsa_index_scores_hist, dsa_topk_hist)
against the unfused steps (dsa_index_scores, dsa_topk).

With dsa_index_scores_hist the tensor-core indexer also builds, for every
query row, the histogram of the first radix digit (top 11 bits of the order
key) of the row's scores, and dsa_topk_hist takes that histogram instead of
reading the row once more for it.  The scores must equal dsa_index_scores'
and the selection dsa_topk's bit for bit: both select exactly from the same
fp32 scores.  The histograms are checked against their definition applied to
the scores.  Covered: the one-CTA-per-row kernel (prefill), the cluster
kernel (few decode rows), the heavy-tie path (integer-grid scores) and
several items per row (decode rows split over CTAs)."""

import numpy as np
import pytest
import torch

import dsa_synth
import sparse_long_context_07_b300 as dsa
from tests.gpu_util import row_meta, structs

pytestmark = pytest.mark.gpu


def _ld(wl):
    return (wl.max_kv + 3) // 4 * 4


def _fused(wl, k):
    b, ix, _ = structs(wl)
    ld = _ld(wl)
    scores = torch.empty((wl.total_q, ld), device="cuda")
    hist = torch.full((wl.total_q, 2048), 12345, dtype=torch.int32, device="cuda")   # cleared by the call
    dsa.index_scores_hist(b, ix, scores, ld, hist)
    idx = torch.full((wl.total_q, k), -7, dtype=torch.int32, device="cuda")
    dsa.topk_hist(b, scores, ld, hist, k, idx)
    torch.cuda.synchronize()
    assert dsa.read_device_errors() == 0
    return idx.cpu().numpy(), scores.cpu().numpy(), hist.cpu().numpy()


def _unfused(wl, k):
    b, ix, _ = structs(wl)
    ld = _ld(wl)
    scores = torch.empty((wl.total_q, ld), device="cuda")
    dsa.index_scores(b, ix, scores, ld)
    idx = torch.full((wl.total_q, k), -7, dtype=torch.int32, device="cuda")
    dsa.topk(b, scores, ld, k, idx)
    torch.cuda.synchronize()
    return idx.cpu().numpy(), scores.cpu().numpy()


def _first_digit_hist(row):
    """Histogram of the top 11 bits of the order-preserving key of fp32
    scores (-0 counted as +0), from its definition."""
    b = (np.asarray(row, dtype=np.float32) + np.float32(0.0)).view(np.uint32)
    key = np.where(b & 0x80000000, ~b, b | 0x80000000).astype(np.uint32)
    return np.bincount(key >> 21, minlength=2048)


@pytest.mark.parametrize("case", ["prefill", "decode", "ragged", "grid"])
def test_fused_selection_equals_unfused(case):
    k = 2048
    if case == "prefill":
        wl = dsa_synth.make_workload("fused-prefill", [5000], [5000], device="cuda", seed=71)
    elif case == "decode":
        wl = dsa_synth.make_workload("fused-decode", [1] * 6, [70000, 3000, 2049, 40000, 131072, 9000],
                                     device="cuda", seed=72, planted=0.1)
    elif case == "ragged":
        wl = dsa_synth.make_workload("fused-ragged", [300, 1, 2500, 7], [300, 12000, 2500, 4100],
                                     device="cuda", seed=73)
    else:
        wl = dsa_synth.make_workload("fused-grid", [4000, 1], [4000, 20000], grid=True, device="cuda", seed=74)
    got, gs, hist = _fused(wl, k)
    ref, rs = _unfused(wl, k)
    _, _, _, n = row_meta(wl)
    for r in range(wl.total_q):
        assert np.array_equal(gs[r, :n[r]], rs[r, :n[r]]), f"{case}: row {r} scores differ"
        assert np.array_equal(hist[r], _first_digit_hist(gs[r, :n[r]])), f"{case}: row {r} histogram"
    bad = np.nonzero((got != ref).any(axis=1))[0]
    assert bad.size == 0, f"{case}: rows {bad[:8]} differ"


def test_fused_entry_points_reject_the_cuda_core_indexer():
    wl = dsa_synth.tiny(device="cuda")
    b, ix, _ = structs(wl)
    scores = torch.empty((wl.total_q, 256), device="cuda")
    hist = torch.empty((wl.total_q, 2048), dtype=torch.int32, device="cuda")
    with pytest.raises(dsa.DSAError) as e:
        dsa.index_scores_hist(b, ix, scores, 256, hist)
    assert e.value.status == dsa.ERROR_NOT_SUPPORTED
