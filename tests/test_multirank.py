"""The bench's multi-rank logic on CPU (gloo, world size 2): each rank runs
its own replica, the step time is the slowest rank's, and the job's rate is
every rank's tokens over that time."""

import multiprocessing as mp
import os
import socket
import sys

import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world, init_method=f"tcp://127.0.0.1:{port}")
    ms = bench.max_over_ranks(10.0 + 7.5 * rank, world, "cpu")
    rate = bench.job_rate(1000 * world, ms)
    dist.barrier()
    out.put((rank, ms, rate))
    dist.destroy_process_group()


def test_two_ranks_time_by_the_slowest_and_add_tokens():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    try:
        res = sorted(out.get(timeout=120) for _ in procs)
    finally:
        for p in procs:
            p.join(timeout=60)
    assert [r for r, _, _ in res] == [0, 1]
    for _, ms, rate in res:
        assert ms == 17.5
        assert abs(rate - 2000 / 0.0175) < 1e-6


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.25, 1, "cpu") == 3.25
    assert bench.job_rate(131072, 216.0) == 131072 / 0.216


def test_replicas_draw_independent_inputs():
    sys.path.insert(0, ROOT)
    import bench
    import dsa_synth
    wl = dsa_synth.make_workload("replica", [6], [6], device="cpu", seed=5)
    a1 = bench.reseed(wl, 1, "cpu")
    a2 = bench.reseed(wl, 2, "cpu")
    b1 = bench.reseed(wl, 1, "cpu")
    assert torch.equal(a1.Q, b1.Q) and torch.equal(a1.k_idx, b1.k_idx)
    assert not torch.equal(a1.Q, a2.Q)
    assert a1.Q.shape == wl.Q.shape and a1.total_q == wl.total_q


def test_replicas_keep_the_workload_recipe():
    # planted keys, non-default dimensions and dtypes survive the reseed
    sys.path.insert(0, ROOT)
    import bench
    import dsa_synth
    wl = dsa_synth.make_workload("replica-planted", [1, 1], [300, 200], device="cpu", seed=8, planted=0.10,
                                 n_idx_heads=4, idx_dim=32, idx_dtype="f32", n_heads=8, d_qk=64, d_v=64,
                                 mla_dtype="f32", topk=32, scale=0.125)
    r = bench.reseed(wl, 1, "cpu")
    assert r.gen_kwargs == {**wl.gen_kwargs, "seed": 1001}
    assert r.gen_kwargs["planted"] == 0.10
    for name in ("q_idx", "k_idx", "w", "Q", "KV"):
        a, b = getattr(wl, name), getattr(r, name)
        assert a.shape == b.shape and a.dtype == b.dtype, name
        assert not torch.equal(a, b), name
    assert (r.topk, r.scale, r.d_v, r.idx_dtype, r.mla_dtype) == (wl.topk, wl.scale, wl.d_v, wl.idx_dtype, wl.mla_dtype)
    tiny = dsa_synth.tiny(device="cpu", grid=True)
    rt = bench.reseed(tiny, 1, "cpu")
    assert rt.n_idx_heads == 4 and rt.idx_dim == 32 and rt.n_heads == 8 and rt.topk == 32
    assert rt.gen_kwargs["grid"] is True
    # grid values stay on the integer grid
    assert torch.equal(rt.q_idx, rt.q_idx.round()) and rt.q_idx.abs().max() <= 2
