"""dsa_sparse_mla against the oracle's softmax attention over the same
selected rows: output within max-abs 2e-2 / mean-abs 2e-3 (bf16 inputs, fp32
accumulation), lse within 1e-2."""

import numpy as np
import pytest
import torch

import dsa_synth
import sparse_long_context_07_b300 as dsa
from tests.gpu_util import (assert_attention_close, assert_lse_close, oracle_attention, random_selection,
                            row_meta, sample_rows, structs, to_f64)

pytestmark = pytest.mark.gpu


def _run(wl, idx, k):
    b, _, m = structs(wl)
    T = wl.total_q
    out = torch.full((T, wl.n_heads, wl.d_v), float("nan"), dtype=wl.Q.dtype, device="cuda")
    lse = torch.full((T, wl.n_heads), float("nan"), device="cuda")
    mn, _ = dsa.workspace_size(b, None, m, k)
    ws = torch.empty(max(mn, 16), dtype=torch.uint8, device="cuda")
    dsa.sparse_mla(b, m, idx.cuda(), k, out, lse, ws)
    torch.cuda.synchronize()
    return out, lse


def _compare(wl, idx, out, lse, rows, what):
    ref_o, ref_l = oracle_attention(wl, rows, idx[rows].numpy())
    got_o = to_f64(out[rows])
    got_l = to_f64(lse[rows])
    assert_attention_close(got_o, ref_o, what)
    assert_lse_close(got_l, ref_l, what)


def test_mla_tc_prefill_partial_tiles():
    # rows with fewer candidates than k, a ragged last tile (k = 200), 700 tokens
    k = 200
    wl = dsa_synth.make_workload("mla-pf", [700], [700], n_idx_heads=16, idx_dim=32, idx_dtype="f32",
                                 device="cuda", seed=21)
    idx = random_selection(wl, k, seed=1)
    out, lse = _run(wl, idx, k)
    assert dsa.read_device_errors() == 0
    rows = sample_rows(wl.total_q, 60, seed=2, must=[0, 1, 63, 64, 199, 200, 699])
    _compare(wl, idx, out, lse, rows, "prefill")


def test_mla_tc_decode_split_kv():
    # 4 decode rows over 8192 cached tokens, k = 2048: split-KV + combine path
    k = 2048
    wl = dsa_synth.make_workload("mla-dec", [1] * 4, [8192, 3000, 2048, 9000], n_idx_heads=16, idx_dim=32,
                                 idx_dtype="f32", device="cuda", seed=22)
    idx = random_selection(wl, k, seed=3)
    out, lse = _run(wl, idx, k)
    assert dsa.read_device_errors() == 0
    _compare(wl, idx, out, lse, list(range(4)), "decode")


def test_mla_tc_rescale_path():
    # the rope columns (512..575, which take part in the scores but not in the
    # value) of later latent rows are scaled up, so the running max of the
    # scores keeps growing by more than the lazy-rescale threshold from tile to
    # tile while the values stay N(0, 1)
    k = 1024
    wl = dsa_synth.make_workload("mla-resc", [1] * 2 + [400], [4096, 2500] + [400], n_idx_heads=16,
                                 idx_dim=32, idx_dtype="f32", device="cuda", seed=23)
    S = wl.KV.shape[0]
    grow = torch.ones(S, device="cuda")
    for b in range(3):
        s0, s1 = int(wl.cu_kv[b]), int(wl.cu_kv[b + 1])
        grow[s0:s1] = 1.0 + 15.0 * torch.arange(s1 - s0, device="cuda") / (s1 - s0)
    kv = wl.KV.float()
    kv[:, wl.d_v:] *= grow[:, None]
    wl.KV = kv.to(torch.bfloat16)
    idx = random_selection(wl, k, seed=4)
    out, lse = _run(wl, idx, k)
    assert dsa.read_device_errors() == 0
    rows = [0, 1] + list(range(2, wl.total_q, 37)) + [wl.total_q - 1]
    _compare(wl, idx, out, lse, rows, "rescale")


def test_mla_tc_out_of_range_indices_are_skipped_and_flagged():
    k = 128
    wl = dsa_synth.make_workload("mla-bad", [1] * 2, [1000, 600], n_idx_heads=16, idx_dim=32, idx_dtype="f32",
                                 device="cuda", seed=24)
    idx = random_selection(wl, k, seed=5)
    bad = idx.clone()
    bad[0, 3] = 1000      # == n: out of range
    bad[1, 7] = -5
    bad[1, 100] = 123456
    out, lse = _run(wl, bad, k)
    assert dsa.read_device_errors() & dsa.DEVERR_BAD_INDEX
    ref_idx = bad.clone()
    ref_idx[(ref_idx < -1)] = -1
    ref_idx[0, 3] = -1
    ref_idx[1, 100] = -1
    _compare(wl, ref_idx, out, lse, [0, 1], "bad-index")


def test_mla_simt_fp32_tiny():
    wl = dsa_synth.tiny(device="cuda")
    idx = random_selection(wl, wl.topk, seed=6)
    out, lse = _run(wl, idx, wl.topk)
    assert dsa.read_device_errors() == 0
    ref_o, ref_l = oracle_attention(wl, list(range(wl.total_q)), idx.numpy())
    assert np.abs(to_f64(out) - ref_o).max() <= 1e-4
    assert np.abs(to_f64(lse) - ref_l).max() <= 1e-4
