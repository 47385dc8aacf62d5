"""Pins of the fp64 oracle against values and results it does not produce
itself: hand-worked examples (tests/golden), closed forms, library routines on
special cases, brute force on tiny inputs, and invariants.  A mutation check
confirms that plausible mistakes fail at least one pin.  CPU only."""

import itertools
import math

import numpy as np
import pytest
import torch

import oracle
from tests.helpers import read_golden

# --------------------------------------------------------------------------
# Input decoding
# --------------------------------------------------------------------------


def test_e4m3_decode_matches_library_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.decode_e4m3(codes)
    lib = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(ours), np.isnan(lib))
    ok = ~np.isnan(lib)
    assert np.array_equal(ours[ok], lib[ok])
    # signed zero preserved
    assert np.signbit(ours[0x80]) and not np.signbit(ours[0x00])


def test_e4m3_decode_spec_values():
    d = lambda c: float(oracle.decode_e4m3(np.array([c], np.uint8))[0])
    assert d(0x7E) == 448.0            # largest finite
    assert d(0xFE) == -448.0
    assert d(0x01) == 2.0 ** -9        # smallest subnormal
    assert d(0x07) == 7 * 2.0 ** -9    # largest subnormal
    assert d(0x08) == 2.0 ** -6        # smallest normal
    assert d(0x38) == 1.0 and d(0xB8) == -1.0
    assert d(0x40) == 2.0 and d(0x3C) == 1.5
    assert math.isnan(d(0x7F)) and math.isnan(d(0xFF))


def test_bf16_decode_matches_library():
    rng = np.random.default_rng(0)
    bits = rng.integers(0, 1 << 16, size=4096, dtype=np.uint16)
    exp = (bits >> 7) & 0xFF
    bits = bits[exp != 0xFF]  # skip inf/nan patterns
    ours = oracle.decode_bf16(bits)
    lib = torch.from_numpy(bits.astype(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(ours, lib)
    assert oracle.decode_bf16(np.array([0x3F80], np.uint16))[0] == 1.0
    assert oracle.decode_bf16(np.array([0xC040], np.uint16))[0] == -3.0


def test_e4m3_encode_round_trips_every_finite_code():
    codes = np.arange(256, dtype=np.uint8)
    vals = oracle.decode_e4m3(codes)
    fin = ~np.isnan(vals)
    assert np.array_equal(oracle.encode_e4m3(vals[fin]), codes[fin])


def _e4m3_midpoint_cases():
    # each pair of adjacent finite codes of one sign, the value halfway between
    # them, and the code round-to-nearest-even picks (even mantissa field)
    vals = oracle.decode_e4m3(np.arange(0x7F, dtype=np.uint8))
    out = []
    for c in range(0x7E):
        lo, hi = vals[c], vals[c + 1]
        out.append(((lo + hi) / 2.0, c if (c & 1) == 0 else c + 1))
    return out


def test_e4m3_encode_ties_to_even_and_nearest():
    for mid, want in _e4m3_midpoint_cases():
        assert int(oracle.encode_e4m3(np.array([mid]))[0]) == want, mid
        assert int(oracle.encode_e4m3(np.array([-mid]))[0]) == want | 0x80, mid
    # just off the midpoint goes to the nearer neighbour
    v = oracle.decode_e4m3(np.array([0x38, 0x39], np.uint8))   # 1.0, 1.125
    assert oracle.encode_e4m3(np.array([1.0625 + 1e-9]))[0] == 0x39
    assert oracle.encode_e4m3(np.array([1.0625 - 1e-9]))[0] == 0x38
    assert v[0] == 1.0 and v[1] == 1.125


def test_e4m3_encode_saturates_and_keeps_signed_zero():
    enc = lambda x: int(oracle.encode_e4m3(np.array([x]))[0])
    assert enc(448.0) == 0x7E and enc(-448.0) == 0xFE
    assert enc(460.0) == 0x7E and enc(1e30) == 0x7E and enc(-1e30) == 0xFE
    assert enc(0.0) == 0x00 and enc(-0.0) == 0x80
    assert enc(2.0 ** -10) == 0x00          # half the smallest subnormal: tie to even (0)
    assert enc(3 * 2.0 ** -10) == 0x02      # 1.5 subnormal steps: tie to even (2)


def test_e4m3_encode_matches_library_cast():
    # torch's float8_e4m3fn cast (round to nearest even) on values inside the
    # finite range: an independent implementation of the same encoding
    rng = np.random.default_rng(1)
    x = rng.standard_normal(30000) * rng.choice([1e-5, 1e-3, 0.1, 1.0, 40.0, 300.0], 30000)
    x = np.clip(x, -448.0, 448.0).astype(np.float32)
    lib = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(oracle.encode_e4m3(x), lib)


def test_quantize_groups_scale_and_extremes():
    rng = np.random.default_rng(2)
    x = (rng.standard_normal((7, 96)) * rng.uniform(0.01, 50, (7, 1))).astype(np.float32)
    x[3] = 0.0                               # an all-zero group
    codes, scale = oracle.quantize_e4m3_groups(x, 96)
    assert codes.shape == x.shape and scale.dtype == np.float32
    amax = np.abs(x).max(axis=1)
    for g in range(7):
        if amax[g] == 0:
            assert scale[g] == 1.0 and not codes[g].any()
            continue
        assert scale[g] == np.float32(amax[g] / np.float32(448.0))
        j = int(np.argmax(np.abs(x[g])))
        assert codes[g, j] in (0x7E, 0xFE)   # the extreme value lands on +-448
        deq = oracle.decode_e4m3(codes[g]) * float(scale[g])
        # e4m3 keeps 3 mantissa bits: relative error <= 2^-4 above the subnormals
        big = np.abs(x[g]) >= 2.0 ** -6 * float(scale[g])
        assert np.all(np.abs(deq[big] - x[g][big]) <= 2.0 ** -4 * np.abs(x[g][big]) + 1e-30)


# --------------------------------------------------------------------------
# Batch geometry
# --------------------------------------------------------------------------


def test_query_positions_bottom_right_aligned():
    # seq 0: prefill of 3 tokens; seq 1: one decode query over 5 cached tokens
    seq, pos, kv0, n = oracle.query_positions([0, 3, 4], [0, 3, 8])
    assert list(seq) == [0, 0, 0, 1]
    assert list(pos) == [0, 1, 2, 4]
    assert list(kv0) == [0, 0, 0, 3]
    assert list(n) == [1, 2, 3, 5]
    with pytest.raises(ValueError):
        oracle.query_positions([0, 4], [0, 3])


# --------------------------------------------------------------------------
# Indexer
# --------------------------------------------------------------------------


def _hand():
    g = read_golden("indexer_hand_example.txt")
    q = np.array([g["q_head1"][0], g["q_head2"][0]])          # [H_I=2, d=2]
    w = np.array(g["w"][0])
    k = np.array(g["k"])                                       # [4, 2]
    return g, q, w, k


def check_indexer_hand(index_fn, topk_fn):
    g, q, w, k = _hand()
    # case A, query at position 3 sees k0..k3, at position 1 sees k0..k1
    I3 = index_fn(q, k, w)
    I1 = index_fn(q, k[:2], w)
    ok = np.array_equal(I3, g["I_A_t3"][0]) and np.array_equal(I1, g["I_A_t1"][0])
    for kk, key in ((1, "topk_A_t3_k1"), (2, "topk_A_t3_k2"), (3, "topk_A_t3_k3")):
        ok &= list(topk_fn(I3, kk)) == [int(v) for v in g[key][0]]
    ok &= list(topk_fn(I1, 2)) == [int(v) for v in g["topk_A_t1_k2"][0]]
    # case B, per-row scales on the codes
    qs = g["q_scale_B"][0][0]
    ks = np.array(g["k_scale_B"][0])
    IB = index_fn(q * qs, k * ks[:, None], w)
    ok &= np.allclose(IB, g["I_B_t3"][0], rtol=0, atol=1e-15)
    for kk, key in ((1, "topk_B_t3_k1"), (2, "topk_B_t3_k2"), (3, "topk_B_t3_k3")):
        ok &= list(topk_fn(IB, kk)) == [int(v) for v in g[key][0]]
    return bool(ok)


def test_indexer_hand_example():
    assert check_indexer_hand(oracle.index_scores_row, oracle.topk_indices)


def test_indexer_single_head_is_relu_matmul():
    # H_I = 1, w = 1: I = ReLU(q . k) -- a library matmul + relu
    rng = np.random.default_rng(1)
    q = rng.standard_normal((1, 16))
    k = rng.standard_normal((40, 16))
    ours = oracle.index_scores_row(q, k, np.ones(1))
    lib = torch.relu(torch.from_numpy(k) @ torch.from_numpy(q[0])).numpy()
    assert np.allclose(ours, lib, rtol=1e-14, atol=1e-14)


def test_indexer_invariants():
    rng = np.random.default_rng(2)
    q = rng.standard_normal((4, 8))
    k = rng.standard_normal((30, 8))
    w = rng.standard_normal(4)
    I = oracle.index_scores_row(q, k, w)
    # homogeneous of degree 1 in w; ReLU makes it sign-sensitive in q
    assert np.allclose(oracle.index_scores_row(q, k, 3.0 * w), 3.0 * I)
    Ineg = oracle.index_scores_row(-q, k, w)
    assert not np.allclose(Ineg, -I)
    # I(q) - I(-q) = sum_j w_j (q_j . k)   (ReLU(x) - ReLU(-x) = x)
    assert np.allclose(I - Ineg, (w[:, None] * (q @ k.T)).sum(0))
    # every key shared by all heads: permuting heads together with w is a no-op
    perm = rng.permutation(4)
    assert np.allclose(oracle.index_scores_row(q[perm], k, w[perm]), I)


def test_index_scores_causal_row_lengths():
    rng = np.random.default_rng(3)
    cu_q, cu_kv = np.array([0, 5, 6]), np.array([0, 5, 12])
    q = rng.standard_normal((6, 2, 4))
    k = rng.standard_normal((12, 4))
    w = rng.standard_normal((6, 2))
    rows = oracle.index_scores(q, k, w, cu_q, cu_kv)
    assert [r.shape[0] for r in rows] == [1, 2, 3, 4, 5, 7]
    # decode row of sequence 1 only sees sequence 1's keys
    assert np.allclose(rows[5], oracle.index_scores_row(q[5], k[5:12], w[5]))


# --------------------------------------------------------------------------
# Top-k
# --------------------------------------------------------------------------


def brute_force_topk(v, k):
    """The unique k-subset S with: every selected score >= every unselected
    score, and among equal scores the selected positions are all lower than the
    unselected ones.  Enumerates every subset."""
    n = len(v)
    kk = min(k, n)
    found = []
    for S in itertools.combinations(range(n), kk):
        Sset = set(S)
        good = True
        for i in S:
            for j in range(n):
                if j in Sset:
                    continue
                if v[i] < v[j] or (v[i] == v[j] and i > j):
                    good = False
                    break
            if not good:
                break
        if good:
            found.append(S)
    assert len(found) == 1
    out = np.full(k, -1, np.int32)
    out[:kk] = found[0]
    return out


def test_topk_brute_force_small():
    rng = np.random.default_rng(4)
    for trial in range(150):
        n = int(rng.integers(1, 10))
        k = int(rng.integers(1, 12))
        v = rng.integers(-3, 4, size=n).astype(np.float64)   # many ties
        v[v == 0] = np.where(rng.random((v == 0).sum()) < 0.5, -0.0, 0.0)
        assert np.array_equal(oracle.topk_indices(v, k), brute_force_topk(v, k)), (v, k)


def test_topk_signed_zero_is_one_value():
    v = np.array([-0.0, 0.0, -0.0, -1.0])
    assert list(oracle.topk_indices(v, 2)) == [0, 1]
    assert list(oracle.topk_indices(v, 3)) == [0, 1, 2]


def test_topk_invariant_random():
    rng = np.random.default_rng(5)
    for n, k in ((1000, 64), (513, 512), (100, 200), (4096, 2048)):
        v = rng.standard_normal(n).astype(np.float32).astype(np.float64)
        sel = oracle.topk_indices(v, k)
        kk = min(k, n)
        assert (sel[:kk] >= 0).all() and (sel[kk:] == -1).all()
        assert np.all(np.diff(sel[:kk]) > 0)
        mask = np.zeros(n, bool)
        mask[sel[:kk]] = True
        if kk < n:
            assert v[mask].min() >= v[~mask].max()


# --------------------------------------------------------------------------
# Attention
# --------------------------------------------------------------------------


def check_attention_closed_form(attn_fn):
    g = read_golden("attention_closed_form.txt")
    ok = True
    for c in ("case1", "case2", "case3"):
        d_qk, d_v = (int(x) for x in g[c + "_dims"][0])
        rows = np.array(g[c + "_rows"][0]).reshape(-1, d_qk)
        q = np.array(g[c + "_q"][0]).reshape(1, d_qk)
        out, lse = attn_fn(q, rows, np.arange(rows.shape[0]), 1.0, d_v)
        ok &= np.allclose(out[0], g[c + "_out"][0], rtol=1e-14, atol=1e-14)
        ok &= abs(lse[0] - g[c + "_lse"][0][0]) < 1e-14
    return bool(ok)


def test_attention_closed_form():
    assert check_attention_closed_form(oracle.sparse_mla_row)


def _sdpa_dense_causal(Q, KV, scale, d_v):
    """Dense causal MQA attention with torch's library SDPA in fp64."""
    T, H, d = Q.shape
    q = torch.from_numpy(Q).permute(1, 0, 2)[None]                 # [1, H, T, d]
    kk = torch.from_numpy(KV)[None, None].expand(1, H, T, d)
    vv = torch.from_numpy(KV[:, :d_v])[None, None].expand(1, H, T, d_v)
    o = torch.nn.functional.scaled_dot_product_attention(q, kk, vv, is_causal=True, scale=scale)
    return o[0].permute(1, 0, 2).numpy()


def test_dense_equivalence_when_k_covers_context():
    # k >= number of candidates: DSA == dense causal attention ("For short
    # prompts, V3.2 emulates dense attention", How Far Can Open Models Go §3.4)
    rng = np.random.default_rng(6)
    T, HI, dI, H, d, dv = 24, 3, 8, 4, 16, 12
    q = rng.standard_normal((T, HI, dI))
    k = rng.standard_normal((T, dI))
    w = rng.standard_normal((T, HI))
    Q = rng.standard_normal((T, H, d))
    KV = rng.standard_normal((T, d))
    cu = np.array([0, T])
    _, idx, out, lse = oracle.forward_rows(q, k, w, Q, KV, cu, cu, topk=T, scale=0.3,
                                           d_v=dv, rows=range(T))
    ref = _sdpa_dense_causal(Q, KV, 0.3, dv)
    assert np.allclose(out, ref, rtol=1e-12, atol=1e-12)
    # with k < n the result differs from dense attention for late rows
    _, _, out_s, _ = oracle.forward_rows(q, k, w, Q, KV, cu, cu, topk=4, scale=0.3,
                                         d_v=dv, rows=range(T))
    assert np.allclose(out_s[:4], ref[:4]) and not np.allclose(out_s[-1], ref[-1])


def _sdpa_bottom_right(Q, KV, scale, d_v):
    """Dense MQA attention of one sequence with torch's library SDPA in fp64:
    nq queries over nkv keys, query i seeing keys 0 .. nkv - nq + i (an
    explicit boolean mask, so no causal convention of the library is used)."""
    nq, H, d = Q.shape
    nkv = KV.shape[0]
    allowed = np.arange(nkv)[None, :] <= (nkv - nq + np.arange(nq))[:, None]
    q = torch.from_numpy(Q).permute(1, 0, 2)[None]
    kk = torch.from_numpy(KV)[None, None].expand(1, H, nkv, d)
    vv = torch.from_numpy(KV[:, :d_v])[None, None].expand(1, H, nkv, d_v)
    o = torch.nn.functional.scaled_dot_product_attention(q, kk, vv, attn_mask=torch.from_numpy(allowed),
                                                         scale=scale)
    return o[0].permute(1, 0, 2).numpy()


def test_two_sequence_batch_against_per_sequence_dense_attention():
    # a 10-token prefill and a 6-token chunk appended to 9 cached tokens: with
    # k covering every candidate, forward_rows and sparse_mla over the whole
    # ragged batch must equal dense attention computed on each sequence's own
    # slice, so a wrong key offset of the second sequence fails here
    rng = np.random.default_rng(12)
    nq, nkv = [10, 6], [10, 15]
    cu_q, cu_kv = np.array([0, 10, 16]), np.array([0, 10, 25])
    T, S, HI, dI, H, d, dv = 16, 25, 3, 8, 4, 16, 12
    q = rng.standard_normal((T, HI, dI))
    k = rng.standard_normal((S, dI))
    w = rng.standard_normal((T, HI))
    Q = rng.standard_normal((T, H, d))
    KV = rng.standard_normal((S, d))
    ref = np.concatenate([_sdpa_bottom_right(Q[0:10], KV[0:10], 0.4, dv),
                          _sdpa_bottom_right(Q[10:16], KV[10:25], 0.4, dv)])
    _, idx, out, lse = oracle.forward_rows(q, k, w, Q, KV, cu_q, cu_kv, topk=S, scale=0.4, d_v=dv,
                                           rows=range(T))
    assert np.allclose(out, ref, rtol=1e-12, atol=1e-12)
    # the selection of a second-sequence row is every candidate of its own sequence
    assert list(idx[10][idx[10] >= 0]) == list(range(10))
    full = np.full((T, S), -1, dtype=np.int64)
    for r in range(T):
        n = (r + 1) if r < 10 else (nkv[1] - nq[1] + (r - 10) + 1)
        full[r, :n] = np.arange(n)
    out2, lse2 = oracle.sparse_mla(Q, KV, full, cu_q, cu_kv, 0.4, dv)
    assert np.allclose(out2, ref, rtol=1e-12, atol=1e-12)
    assert np.allclose(lse2, lse, rtol=1e-13)
    # and sparse_mla's lse is the library logsumexp of the second sequence's scores
    z = 0.4 * torch.from_numpy(Q[15]) @ torch.from_numpy(KV[10:25]).T
    assert np.allclose(lse2[15], torch.logsumexp(z, dim=1).numpy(), rtol=1e-13)


def test_attention_lse_against_library_logsumexp():
    rng = np.random.default_rng(7)
    Q = rng.standard_normal((3, 10))
    kv = rng.standard_normal((20, 10))
    idx = np.array([3, 7, -1, 0, 19, -1])
    out, lse = oracle.sparse_mla_row(Q, kv, idx, 0.5, 6)
    z = 0.5 * torch.from_numpy(Q) @ torch.from_numpy(kv[[3, 7, 0, 19]]).T
    assert np.allclose(lse, torch.logsumexp(z, dim=1).numpy(), rtol=1e-14)
    p = torch.softmax(z, dim=1).numpy()
    assert np.allclose(out, p @ kv[[3, 7, 0, 19], :6], rtol=1e-13, atol=1e-14)


def test_attention_invariants():
    rng = np.random.default_rng(8)
    Q = rng.standard_normal((5, 12))
    kv = rng.standard_normal((30, 12))
    idx = rng.permutation(30)[:9].astype(np.int32)
    out, lse = oracle.sparse_mla_row(Q, kv, idx, 0.7, 8)
    # order of the selected set does not matter; -1 slots are skipped
    out2, lse2 = oracle.sparse_mla_row(Q, kv, np.concatenate([idx[::-1], [-1, -1]]), 0.7, 8)
    assert np.allclose(out, out2) and np.allclose(lse, lse2)
    # empty selection: zero output and lse = -inf
    o0, l0 = oracle.sparse_mla_row(Q, kv, np.full(4, -1), 0.7, 8)
    assert np.all(o0 == 0) and np.all(np.isneginf(l0))
    # merging the halves of a split selection gives the whole (split-KV decode)
    oa, la = oracle.sparse_mla_row(Q, kv, idx[:4], 0.7, 8)
    ob, lb = oracle.sparse_mla_row(Q, kv, idx[4:], 0.7, 8)
    om, lm = oracle.lse_merge([oa, ob], [la, lb])
    assert np.allclose(om, out, rtol=1e-13) and np.allclose(lm, lse, rtol=1e-13)
    # merging with an empty split is a no-op
    om, lm = oracle.lse_merge([out, o0], [lse, l0])
    assert np.allclose(om, out) and np.allclose(lm, lse)


# --------------------------------------------------------------------------
# Mutation check: each plausible mistake below fails at least one pin.
# --------------------------------------------------------------------------


def _idx_no_relu(q, k, w):
    return w @ (q @ k.T)


def _idx_relu_after_sum(q, k, w):
    return np.maximum(w @ (q @ k.T), 0.0)


def _idx_transposed_weights(q, k, w):
    return (np.maximum(q @ k.T, 0.0).T @ w[::-1])


def _topk_ties_high(v, k):
    v = np.asarray(v, dtype=np.float64)
    n = v.shape[0]
    order = np.lexsort((-np.arange(n), -v))
    keep = np.sort(order[:min(k, n)])
    out = np.full(k, -1, np.int32)
    out[:keep.shape[0]] = keep
    return out


def _topk_smallest(v, k):
    return oracle.topk_indices(-np.asarray(v), k)


def _attn_no_max_sub_wrong_value(Q, kv, idx, scale, d_v):
    sel = idx[idx >= 0]
    c = kv[sel]
    z = scale * (Q @ c.T)
    e = np.exp(z)
    return (e @ c[:, -d_v:]) / e.sum(1, keepdims=True), np.log(e.sum(1))


def _attn_no_scale(Q, kv, idx, scale, d_v):
    return oracle.sparse_mla_row(Q, kv, idx, 1.0 if scale != 1.0 else 2.0, d_v)


@pytest.mark.parametrize("bad", [_idx_no_relu, _idx_relu_after_sum, _idx_transposed_weights])
def test_mutant_indexer_fails_pin(bad):
    assert not check_indexer_hand(bad, oracle.topk_indices)


@pytest.mark.parametrize("bad", [_topk_ties_high, _topk_smallest])
def test_mutant_topk_fails_pin(bad):
    assert not check_indexer_hand(oracle.index_scores_row, bad)


@pytest.mark.parametrize("bad", [_attn_no_max_sub_wrong_value, _attn_no_scale])
def test_mutant_attention_fails_pin(bad):
    # value-column mistake fails the closed form; scale mistake fails it too
    assert not check_attention_closed_form(bad)


def check_e4m3_encoder(enc) -> bool:
    """The encoder pins (round trip, midpoints, saturation) as one predicate."""
    codes = np.arange(256, dtype=np.uint8)
    vals = oracle.decode_e4m3(codes)
    fin = ~np.isnan(vals)
    if not np.array_equal(enc(vals[fin]), codes[fin]):
        return False
    for mid, want in _e4m3_midpoint_cases():
        if int(enc(np.array([mid]))[0]) != want:
            return False
    return int(enc(np.array([460.0]))[0]) == 0x7E and int(enc(np.array([1e6]))[0]) == 0x7E


def _enc_ties_away(v):
    # rounds halfway cases away from zero: nudge every value up by a hair
    v = np.asarray(v, dtype=np.float64)
    return oracle.encode_e4m3(v * (1 + 1e-12))


def _enc_truncate(v):
    # rounds toward zero: the nearest code not above |v|
    v = np.asarray(v, dtype=np.float64)
    grid = oracle.decode_e4m3(np.arange(0x7F, dtype=np.uint8))
    out = np.searchsorted(grid, np.abs(v), side="right") - 1
    out = np.clip(out, 0, 0x7E).astype(np.uint8)
    return out | np.where(np.signbit(v), 0x80, 0x00).astype(np.uint8)


def _enc_no_saturation(v):
    # overflow lands on the NaN code instead of +-448
    out = oracle.encode_e4m3(v)
    big = np.abs(np.asarray(v, dtype=np.float64)) > 448.0
    out[big] = out[big] | 0x7F
    return out


def test_oracle_encoder_passes_its_pins():
    assert check_e4m3_encoder(oracle.encode_e4m3)


@pytest.mark.parametrize("bad", [_enc_ties_away, _enc_truncate, _enc_no_saturation])
def test_mutant_encoder_fails_pin(bad):
    assert not check_e4m3_encoder(bad)
