"""dsa_quantize_e4m3 (the producer step of the indexer's FP8 inputs) against
the oracle's per-group absmax quantisation: codes and scales bit-exact, for
fp32 and bf16 inputs, query-sized and key-sized groups, appends into a cache
at a row offset, zero groups and the argument checks."""

import numpy as np
import pytest
import torch

import oracle
import sparse_long_context_07_b300 as dsa

pytestmark = pytest.mark.gpu


def _oracle(x: torch.Tensor, group_elems: int):
    return oracle.quantize_e4m3_groups(x.float().cpu().numpy(), group_elems)


def _run(x, group_elems):
    codes = torch.full((x.numel(),), 0xAB, dtype=torch.uint8, device="cuda")
    scales = torch.full((x.numel() // group_elems,), -1.0, device="cuda")
    dsa.quantize_e4m3(x, codes, scales, group_elems)
    torch.cuda.synchronize()
    return codes.cpu().numpy(), scales.cpu().numpy()


def _values(shape, seed, dtype):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    x = torch.randn(shape, generator=g, device="cuda")
    # a spread of group magnitudes, so scales differ by orders of magnitude
    mag = torch.exp(torch.randn((shape[0],) + (1,) * (len(shape) - 1), generator=g, device="cuda") * 3.0)
    return (x * mag).to(dtype)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_quantize_query_groups(dtype):
    x = _values((37, 64, 128), seed=1, dtype=dtype)          # a token's 64 x 128 indexer query per group
    x[5] = 0.0                                              # an all-zero token
    codes, scales = _run(x, 64 * 128)
    ref_c, ref_s = _oracle(x, 64 * 128)
    assert np.array_equal(codes, ref_c.reshape(-1))
    assert np.array_equal(scales.view(np.uint32), ref_s.view(np.uint32))
    assert scales[5] == 1.0 and not codes.reshape(37, -1)[5].any()


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("group_elems", [4, 36, 128, 1024, 1028, 16384])
def test_quantize_group_sizes(dtype, group_elems):
    groups = max(3, 20000 // group_elems)
    x = _values((groups, group_elems), seed=group_elems, dtype=dtype)
    codes, scales = _run(x, group_elems)
    ref_c, ref_s = _oracle(x, group_elems)
    assert np.array_equal(codes, ref_c.reshape(-1))
    assert np.array_equal(scales.view(np.uint32), ref_s.view(np.uint32))


def test_quantize_appends_into_a_key_cache():
    S, d, s0, n = 2000, 128, 700, 300
    cache = torch.full((S, d), 0xAB, dtype=torch.uint8, device="cuda")
    cache_scale = torch.full((S,), -1.0, device="cuda")
    x = _values((n, d), seed=7, dtype=torch.bfloat16)
    dsa.quantize_e4m3(x, cache[s0:s0 + n], cache_scale[s0:s0 + n], d)
    torch.cuda.synchronize()
    ref_c, ref_s = _oracle(x, d)
    c = cache.cpu().numpy()
    sc = cache_scale.cpu().numpy()
    assert np.array_equal(c[s0:s0 + n], ref_c)
    assert np.array_equal(sc[s0:s0 + n].view(np.uint32), ref_s.view(np.uint32))
    assert (c[:s0] == 0xAB).all() and (c[s0 + n:] == 0xAB).all()
    assert (sc[:s0] == -1.0).all() and (sc[s0 + n:] == -1.0).all()


def test_quantize_matches_the_input_generator():
    # the seeded workloads quantise on the host side with the same definition
    import dsa_synth
    x = _values((50, 128), seed=9, dtype=torch.float32)
    codes, scales = _run(x, 128)
    gc, gs = dsa_synth.quantize_e4m3_rows(x)
    assert np.array_equal(codes, gc.cpu().numpy().reshape(-1))
    assert np.array_equal(scales.view(np.uint32), gs.cpu().numpy().view(np.uint32))


def test_quantize_argument_checks():
    x = torch.zeros(64, device="cuda")
    codes = torch.zeros(64, dtype=torch.uint8, device="cuda")
    scales = torch.zeros(16, device="cuda")
    with pytest.raises(dsa.DSAError) as e:
        dsa.quantize_e4m3(x[:60], codes, scales, 6)
    assert e.value.status == dsa.ERROR_INVALID_VALUE
    with pytest.raises(dsa.DSAError) as e:
        dsa.quantize_e4m3(x[1:61], codes, scales, 4)     # x not 16-byte aligned
    assert e.value.status == dsa.ERROR_INVALID_VALUE
    dsa.quantize_e4m3(x[:0], codes, scales, 4)            # no groups: nothing to do


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("group_elems", [128, 8192, 1028])
def test_quantize_rounding_midpoints_bit_exact(dtype, group_elems):
    # quotients x / scale on, and one fp32 ulp either side of, every e4m3
    # rounding midpoint (and on the codes themselves), for group scales of
    # awkward mantissas: the division and the round-to-nearest-even must
    # agree with the oracle's IEEE fp32 division and encoder bit for bit
    v = oracle.decode_e4m3(np.arange(0x7F, dtype=np.uint8))          # finite non-negative codes, ascending
    mid = ((v[1:] + v[:-1]) / 2).astype(np.float32)
    t = np.concatenate([mid, np.nextafter(mid, np.float32(np.inf)), np.nextafter(mid, np.float32(-np.inf)),
                        v.astype(np.float32)])
    rng = np.random.default_rng(group_elems)
    groups = []
    for amax in (448.0 * 1.3, 448.0 * 0.7371, 3.1e-3, 7.77e4, 1.0, 448.0):
        scale = np.float32(amax) / np.float32(448.0)
        for _ in range(2):
            tt = rng.permutation(np.resize(t, group_elems - 1))
            x = (tt * scale).astype(np.float32)
            x = np.minimum(np.abs(x), np.float32(amax)) * rng.choice([-1, 1], size=x.shape).astype(np.float32)
            groups.append(np.concatenate([[np.float32(amax)], x]).astype(np.float32))
    xg = torch.from_numpy(np.stack(groups)).to(dtype).cuda().contiguous()
    codes, scales = _run(xg, group_elems)
    ref_c, ref_s = _oracle(xg, group_elems)
    assert np.array_equal(scales.view(np.uint32), ref_s.view(np.uint32))
    bad = np.nonzero(codes != ref_c.reshape(-1))[0]
    assert bad.size == 0, f"{bad.size} codes differ, first at {bad[:5]}"
