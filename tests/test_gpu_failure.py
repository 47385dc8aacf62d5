"""The bounded-wait failure path of the tensor-core indexer, on the GPU.

Every mbarrier wait in the library's kernels gives up after a time limit
(about 2 s), sets DSA_DEVERR_TIMEOUT in the device error word and lets every
role of the CTA leave its loop, drain the copies and MMAs still in flight and
free its tensor memory.  The test hook dsa_debug_inject_fault(1) makes the
next indexer launch skip one key-tile load, so the MMA warp's wait on that
tile runs out: nothing faults, traps or spins without limit.  The test then
checks that the error word reports the timeout, and that the library and the
GPU context are healthy afterwards: the same call without the fault gives the
oracle's scores bit for bit on integer-grid inputs."""

import time

import numpy as np
import pytest
import torch

import dsa_synth
import sparse_long_context_07_b300 as dsa
from tests.gpu_util import oracle_scores, row_meta, structs

pytestmark = pytest.mark.gpu


def _scores(wl, ld):
    return torch.full((wl.total_q, ld), 7.25, device="cuda")


def test_indexer_wait_times_out_then_recovers():
    # one 600-token prefill: items of 4 rows with up to 5 key tiles each, so
    # every CTA whose items hold 3 or more tiles meets the skipped tile
    wl = dsa_synth.make_workload("fault", [600], [600], grid=True, device="cuda", seed=51,
                                 n_heads=8, d_qk=64, d_v=64)
    b, ix, _ = structs(wl)
    ld = 608
    assert dsa.read_device_errors() == 0   # start from a clean error word

    scores = _scores(wl, ld)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    dsa.debug_inject_fault(1)
    dsa.index_scores(b, ix, scores, ld)
    flags = dsa.read_device_errors()        # synchronises the stream
    elapsed = time.perf_counter() - t0
    assert flags & dsa.DEVERR_TIMEOUT, f"expected the timeout bit, got flags {flags:#x}"
    assert not flags & dsa.DEVERR_BAD_INDEX
    # the wait limit is 2 s; the drain waits are bounded by the same limit
    assert elapsed < 15.0, f"the timed-out launch took {elapsed:.1f} s"
    assert dsa.read_device_errors() == 0   # reading cleared the word

    # the hook applies to one launch only: the next call is clean and exact
    scores = _scores(wl, ld)
    dsa.index_scores(b, ix, scores, ld)
    assert dsa.read_device_errors() == 0
    S = scores.cpu().numpy()
    _, _, _, n = row_meta(wl)
    rows = [0, 1, 127, 128, 300, 511, 512, 599]
    ref = oracle_scores(wl, rows)
    for i, r in enumerate(rows):
        assert np.array_equal(S[r, :n[r]].astype(np.float64), ref[i]), f"row {r} after recovery"
        assert np.all(S[r, n[r]:] == 7.25)
