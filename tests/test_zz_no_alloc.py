"""The scratch-free sparse MLA entry point (dsa_sparse_mla_noalloc) against
the workspace-taking one (dsa_sparse_mla) and against the oracle.

Callers that cannot allocate device memory (a runtime that owns all device
allocations, a serving loop that reserved its memory up front) use the
scratch-free entry point; its split-KV partials live in a fixed array inside
the library.  Two calls in a row, each on new selections, must match the
regular entry point and the fp64 oracle within the attention tolerance used by
every test here.  A batch whose preferred split would overflow the fixed array
runs with fewer splits and still matches.  This file sorts last so that a run
stopping at its first failure has already run every other test."""

import numpy as np
import pytest
import torch

import dsa_synth
import sparse_long_context_07_b300 as dsa
from tests.gpu_util import (assert_attention_close, assert_lse_close, oracle_attention, random_selection, structs,
                            to_f64)

pytestmark = pytest.mark.gpu


def _decode_batch(lens, seed):
    return dsa_synth.make_workload("noalloc", [1] * len(lens), lens, n_idx_heads=16, idx_dim=32,
                                   idx_dtype="f32", device="cuda", seed=seed)


def _both(wl, idx, k, ws):
    b, _, m = structs(wl)
    T = wl.total_q
    ref_out = torch.full((T, wl.n_heads, wl.d_v), float("nan"), dtype=torch.bfloat16, device="cuda")
    ref_lse = torch.full((T, wl.n_heads), float("nan"), device="cuda")
    dsa.sparse_mla(b, m, idx, k, ref_out, ref_lse, ws)
    out = torch.full_like(ref_out, float("nan"))
    lse = torch.full_like(ref_lse, float("nan"))
    dsa.sparse_mla_noalloc(b, m, idx, k, out, lse)
    torch.cuda.synchronize()
    assert dsa.read_device_errors() == 0
    return out, lse, ref_out, ref_lse


def test_noalloc_matches_workspace_entry_point_on_two_calls():
    k = 2048
    wl = _decode_batch([8192, 3000, 2048, 9000], seed=41)   # 4 rows: split-KV path
    b, _, m = structs(wl)
    mn, _ = dsa.workspace_size(b, None, m, k)
    assert mn > 0   # this batch does use split scratch
    ws = torch.empty(mn, dtype=torch.uint8, device="cuda")
    for call, seed in enumerate((5, 6)):
        idx = random_selection(wl, k, seed=seed)
        out, lse, ref_out, ref_lse = _both(wl, idx.cuda(), k, ws)
        assert_attention_close(to_f64(out), to_f64(ref_out), f"call {call}")
        assert_lse_close(to_f64(lse), to_f64(ref_lse), f"call {call}")
        assert np.isfinite(to_f64(out)).all()
        # and against the fp64 oracle on the same selections
        rows = list(range(wl.total_q))
        o_ref, l_ref = oracle_attention(wl, rows, [idx[r].numpy() for r in rows])
        assert_attention_close(to_f64(out), o_ref, f"call {call} vs oracle")
        assert_lse_close(to_f64(lse), l_ref, f"call {call} vs oracle")


def test_noalloc_batch_beyond_preferred_split_takes_fewer_splits():
    # 34 rows x 3 splits of fp32 partials would exceed the 24 MiB array: the
    # entry point splits less and still gives the same attention
    k = 2048
    wl = _decode_batch([4096] * 34, seed=42)
    b, _, m = structs(wl)
    mn, _ = dsa.workspace_size(b, None, m, k)
    assert mn > 24 << 20
    ws = torch.empty(mn, dtype=torch.uint8, device="cuda")
    idx = random_selection(wl, k, seed=7)
    out, lse, ref_out, ref_lse = _both(wl, idx.cuda(), k, ws)
    assert_attention_close(to_f64(out), to_f64(ref_out), "34 rows")
    assert_lse_close(to_f64(lse), to_f64(ref_lse), "34 rows")
    rows = [0, 17, 33]
    o_ref, l_ref = oracle_attention(wl, rows, [idx[r].numpy() for r in rows])
    assert_attention_close(to_f64(out[rows]), o_ref, "34 rows vs oracle")
