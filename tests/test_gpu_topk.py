"""dsa_topk against the oracle's full-sort selection on identical fp32 score
rows: index sets, their order and the returned values must be bit-exact."""

import numpy as np
import pytest
import torch

import oracle
import sparse_long_context_07_b300 as dsa
from tests.gpu_util import sample_rows

pytestmark = pytest.mark.gpu


def _cu(lens):
    c = [0]
    for x in lens:
        c.append(c[-1] + x)
    return torch.tensor(c, dtype=torch.int32, device="cuda")


def _scores(T, ld, kind, seed):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    if kind == "normal":
        return torch.randn((T, ld), generator=g, device="cuda")
    if kind == "ties":   # small integers: heavy ties, both signed zeros
        s = torch.randint(-3, 4, (T, ld), generator=g, device="cuda").float()
        neg = torch.rand((T, ld), generator=g, device="cuda") < 0.5
        return torch.where((s == 0) & neg, torch.full_like(s, -0.0), s)
    if kind == "const":
        return torch.full((T, ld), 1.5, device="cuda")
    raise ValueError(kind)


def _check(batch, scores, ld, k, rows, n_of_row):
    T = batch.total_q
    idx = torch.full((T, k), -7, dtype=torch.int32, device="cuda")
    vals = torch.full((T, k), float("nan"), device="cuda")
    dsa.topk(batch, scores, ld, k, idx, vals)
    torch.cuda.synchronize()
    assert dsa.read_device_errors() == 0
    S = scores.cpu().numpy()
    I = idx.cpu().numpy()
    V = vals.cpu().numpy()
    for r in rows:
        n = n_of_row[r]
        ref = oracle.topk_indices(S[r, :n].astype(np.float64), k)
        assert np.array_equal(I[r], ref), f"row {r} (n={n}, k={k})"
        m = min(k, n)
        assert np.array_equal(V[r, :m].view(np.uint32), S[r, ref[:m]].view(np.uint32)), f"vals row {r}"
        assert np.all(np.isneginf(V[r, m:]))


@pytest.mark.parametrize("kind", ["normal", "ties"])
@pytest.mark.parametrize("k", [1, 64, 2048])
def test_topk_prefill_rows(kind, k):
    L = 5000
    ld = L + 4
    batch = dsa.Batch(_cu([L]), _cu([L]), [L], [L])
    scores = _scores(L, ld, kind, seed=11 + k)
    rows = sample_rows(L, 160, seed=k, must=[0, 1, k - 2, k - 1, k, k + 1, L - 1])
    _check(batch, scores, ld, k, rows, {r: r + 1 for r in range(L)})


def test_topk_long_decode_rows():
    lens = [131072, 70001, 2049, 2048, 2047, 1, 5000, 100003]
    k = 2048
    ld = 131072
    batch = dsa.Batch(_cu([1] * len(lens)), _cu(lens), [1] * len(lens), lens)
    for kind in ("normal", "ties"):
        scores = _scores(len(lens), ld, kind, seed=5)
        _check(batch, scores, ld, k, range(len(lens)), dict(enumerate(lens)))


def test_topk_all_equal_and_large_k():
    lens = [20000, 16384, 16385, 3]
    ld = 20000
    batch = dsa.Batch(_cu([1] * 4), _cu(lens), [1] * 4, lens)
    scores = _scores(4, ld, "const", seed=0)
    _check(batch, scores, ld, 16384, range(4), dict(enumerate(lens)))
    _check(batch, _scores(4, ld, "normal", seed=3), ld, 16384, range(4), dict(enumerate(lens)))


def test_topk_rows_beyond_the_bitmap_and_boundary_overflow():
    # rows longer than 131072 candidates take the general path; so does a row
    # whose boundary histogram bin holds more than 4096 keys (many equal keys
    # at the k-th value: normal scores with a block of 6000 copies of one value)
    lens = [140000, 131073, 131072, 9000]
    k = 2048
    ld = 140000
    batch = dsa.Batch(_cu([1] * len(lens)), _cu(lens), [1] * len(lens), lens)
    scores = _scores(len(lens), ld, "normal", seed=8)
    row = scores[3]
    kth = torch.sort(row[:9000], descending=True).values[k - 100]
    row[1000:7000] = kth
    _check(batch, scores, ld, k, range(len(lens)), dict(enumerate(lens)))


def test_topk_cluster_and_row_kernels_agree():
    # a batch of few rows takes a cluster of CTAs per row, a larger batch one
    # CTA per row; the same rows must come out identical either way
    props = torch.cuda.get_device_properties(0)
    few = (4 * props.multi_processor_count) // 8          # largest batch on the cluster path
    lens = [16384 + 997 * i for i in range(few + 1)]
    k = 2048
    ld = ((max(lens) + 3) // 4) * 4
    for kind in ("normal", "ties"):
        scores = _scores(len(lens), ld, kind, seed=21)
        outs = []
        for rows in (few, few + 1):
            sub = lens[:rows]
            batch = dsa.Batch(_cu([1] * rows), _cu(sub), [1] * rows, sub)
            idx = torch.full((rows, k), -7, dtype=torch.int32, device="cuda")
            dsa.topk(batch, scores, ld, k, idx)
            torch.cuda.synchronize()
            assert dsa.read_device_errors() == 0
            outs.append(idx[:few].cpu())
        assert torch.equal(outs[0], outs[1]), kind
        S = scores.cpu().numpy()
        for r in (0, few // 2, few - 1):
            ref = oracle.topk_indices(S[r, :lens[r]].astype(np.float64), k)
            assert np.array_equal(outs[0][r].numpy(), ref), f"{kind} row {r}"


@pytest.mark.parametrize("nbin", [8000, 8192, 8193, 12000])
def test_topk_cluster_boundary_bin_sizes(nbin):
    # decode rows whose k-th key sits in a top-11-bit bin of nbin keys
    # (distinct values in [2, 2.5), one bin; the rest below): the cluster
    # kernel keeps the bin's keys per warp and refines them across the CTAs
    L, k = 60000, 2048
    lens = [L, L - 5, 30001]
    ld = L
    batch = dsa.Batch(_cu([1] * len(lens)), _cu(lens), [1] * len(lens), lens)
    g = torch.Generator(device="cuda")
    g.manual_seed(nbin)
    scores = torch.randn((len(lens), ld), generator=g, device="cuda") * 0.3
    for r, n in enumerate(lens):
        m = min(nbin, n)
        pos = torch.randperm(n, generator=g, device="cuda")[:m]
        scores[r, pos] = 2.0 + 0.5 * torch.rand((m,), generator=g, device="cuda") * 0.999
    # a few exact copies of one in-bin value: ties inside the refined bin
    scores[0, 100:140] = scores[0, 99]
    _check(batch, scores, ld, k, range(len(lens)), dict(enumerate(lens)))


@pytest.mark.parametrize("nbin", [8000, 12000])
def test_topk_cluster_boundary_bin_concentrated(nbin):
    # nbin distinct keys of one top-11-bit bin in the first nbin positions of
    # a 131072-candidate decode row: the first CTA's warps each hold about
    # 1000 of them, more than a warp keeps, so the row takes the multi-pass
    # path over the slices; the same keys spread over the row are kept per
    # warp and refined across the cluster
    n, k = 131072, 2048
    batch = dsa.Batch(_cu([1, 1]), _cu([n, n]), [1, 1], [n, n])
    g = torch.Generator(device="cuda")
    g.manual_seed(77 + nbin)
    scores = torch.randn((2, n), generator=g, device="cuda") * 0.3
    vals = 2.0 + 0.5 * torch.rand((nbin,), generator=g, device="cuda") * 0.999
    scores[0, :nbin] = vals
    scores[1, torch.randperm(n, generator=g, device="cuda")[:nbin]] = vals
    _check(batch, scores, n, k, range(2), {0: n, 1: n})
