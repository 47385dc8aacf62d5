"""The scratch-free sparse MLA entry point (dsa_sparse_mla_noalloc) against
the workspace-taking one (dsa_sparse_mla).

Callers that cannot allocate device memory (a runtime that owns all device
allocations, a serving loop that reserved its memory up front) use the
scratch-free entry point; its split-KV partials live in a fixed array inside
the library.  Two calls in a row, each on new selections, must match the
regular entry point within the attention tolerance used by every test here,
and a batch whose partials exceed the fixed array must be refused.  This file
sorts last so that a run stopping at its first failure has already run every
other test."""

import numpy as np
import pytest
import torch

import dsa_synth
import sparse_long_context_07_b300 as dsa
from tests.gpu_util import assert_attention_close, assert_lse_close, random_selection, structs, to_f64

pytestmark = pytest.mark.gpu


def _decode_batch(lens, seed):
    return dsa_synth.make_workload("noalloc", [1] * len(lens), lens, n_idx_heads=16, idx_dim=32,
                                   idx_dtype="f32", device="cuda", seed=seed)


def test_noalloc_matches_workspace_entry_point_on_two_calls():
    k = 2048
    wl = _decode_batch([8192, 3000, 2048, 9000], seed=41)   # 4 rows: split-KV path
    b, _, m = structs(wl)
    T = wl.total_q
    mn, _ = dsa.workspace_size(b, None, m, k)
    assert mn > 0   # this batch does use split scratch
    ws = torch.empty(mn, dtype=torch.uint8, device="cuda")
    for call, seed in enumerate((5, 6)):
        idx = random_selection(wl, k, seed=seed).cuda()
        ref_out = torch.full((T, wl.n_heads, wl.d_v), float("nan"), dtype=torch.bfloat16, device="cuda")
        ref_lse = torch.full((T, wl.n_heads), float("nan"), device="cuda")
        dsa.sparse_mla(b, m, idx, k, ref_out, ref_lse, ws)
        out = torch.full_like(ref_out, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        dsa.sparse_mla_noalloc(b, m, idx, k, out, lse)
        torch.cuda.synchronize()
        assert dsa.read_device_errors() == 0
        assert_attention_close(to_f64(out), to_f64(ref_out), f"call {call}")
        assert_lse_close(to_f64(lse), to_f64(ref_lse), f"call {call}")
        assert np.isfinite(to_f64(out)).all()


def test_noalloc_refuses_batches_beyond_its_scratch():
    k = 2048
    wl = _decode_batch([4096] * 34, seed=42)   # 34 rows x 3 splits of fp32 partials > 24 MiB
    b, _, m = structs(wl)
    idx = random_selection(wl, k, seed=7).cuda()
    out = torch.empty((wl.total_q, wl.n_heads, wl.d_v), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(dsa.DSAError) as e:
        dsa.sparse_mla_noalloc(b, m, idx, k, out, None)
    assert e.value.status == dsa.ERROR_NOT_SUPPORTED
    assert "scratch" in str(e.value)
