"""dsa_dense_mla (causal MLA-MQA attention over every candidate, the baseline
the sparse path is measured against) against the oracle's softmax attention
over all candidates, and against dsa_sparse_mla given complete index lists:
max-abs 2e-2 / mean-abs 2e-3, lse within 1e-2."""

import numpy as np
import pytest
import torch

import dsa_synth
import sparse_long_context_07_b300 as dsa
from tests.gpu_util import assert_attention_close, assert_lse_close, oracle_attention, row_meta, sample_rows, structs, to_f64

pytestmark = pytest.mark.gpu


def _dense(wl, with_ws=True):
    b, _, m = structs(wl)
    T = wl.total_q
    out = torch.full((T, wl.n_heads, wl.d_v), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((T, wl.n_heads), float("nan"), device="cuda")
    need = dsa.dense_mla_workspace_size(b, m)
    ws = torch.empty(max(need, 16), dtype=torch.uint8, device="cuda") if with_ws else None
    dsa.dense_mla(b, m, out, lse, ws)
    torch.cuda.synchronize()
    assert dsa.read_device_errors() == 0
    return out, lse, need


def _all_candidates(wl, rows):
    _, _, _, n = row_meta(wl)
    return [np.arange(n[r]) for r in rows]


@pytest.mark.parametrize("with_ws", [True, False])
def test_dense_decode_rows(with_ws):
    wl = dsa_synth.make_workload("dense-dec", [1] * 4, [8192, 3000, 2048, 9000], n_idx_heads=16, idx_dim=32,
                                 idx_dtype="f32", device="cuda", seed=31)
    out, lse, need = _dense(wl, with_ws)
    assert need > 0      # four rows are split over several CTA pairs
    rows = list(range(4))
    ref_o, ref_l = oracle_attention(wl, rows, _all_candidates(wl, rows))
    assert_attention_close(to_f64(out[rows]), ref_o, "dense decode")
    assert_lse_close(to_f64(lse[rows]), ref_l, "dense decode")


def test_dense_prefill_rows():
    wl = dsa_synth.make_workload("dense-pf", [700], [700], n_idx_heads=16, idx_dim=32, idx_dtype="f32",
                                 device="cuda", seed=32)
    out, lse, need = _dense(wl)
    assert need == 0     # 700 rows fill the SMs without splitting
    rows = sample_rows(wl.total_q, 40, seed=3, must=[0, 1, 31, 32, 33, 699])
    ref_o, ref_l = oracle_attention(wl, rows, _all_candidates(wl, rows))
    assert_attention_close(to_f64(out[rows]), ref_o, "dense prefill")
    assert_lse_close(to_f64(lse[rows]), ref_l, "dense prefill")


def test_dense_equals_sparse_with_complete_index_lists():
    wl = dsa_synth.make_workload("dense-eq", [300, 1], [300, 777], n_idx_heads=16, idx_dim=32, idx_dtype="f32",
                                 device="cuda", seed=33)
    b, _, m = structs(wl)
    T = wl.total_q
    _, _, _, n = row_meta(wl)
    k = 800
    idx = torch.full((T, k), -1, dtype=torch.int32)
    for r in range(T):
        idx[r, :n[r]] = torch.arange(n[r], dtype=torch.int32)
    sp_o = torch.empty((T, wl.n_heads, wl.d_v), dtype=torch.bfloat16, device="cuda")
    sp_l = torch.empty((T, wl.n_heads), device="cuda")
    mn, _ = dsa.workspace_size(b, None, m, k)
    ws = torch.empty(max(mn, 16), dtype=torch.uint8, device="cuda")
    dsa.sparse_mla(b, m, idx.cuda(), k, sp_o, sp_l, ws)
    de_o, de_l, _ = _dense(wl)
    assert_attention_close(to_f64(de_o), to_f64(sp_o), "dense vs sparse")
    assert_lse_close(to_f64(de_l), to_f64(sp_l), "dense vs sparse")


def test_dense_rejects_the_small_instance():
    wl = dsa_synth.tiny(device="cuda")
    b, _, m = structs(wl)
    out = torch.empty((wl.total_q, wl.n_heads, wl.d_v), dtype=wl.Q.dtype, device="cuda")
    with pytest.raises(dsa.DSAError) as e:
        dsa.dense_mla(b, m, out)
    assert e.value.status == dsa.ERROR_NOT_SUPPORTED
