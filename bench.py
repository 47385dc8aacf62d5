#!/usr/bin/env python
"""Benchmark of the DSA forward pass (lightning indexer + top-k + sparse MLA).

One step = one dsa_forward call over the whole workload (every query row
through all three kernels).  Default workload: one 131072-token causal prefill
(the 128K-context case), production dimensions, synthetic seeded inputs
already resident in HBM.  Prints one JSON line.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl native|reference]

Multi-GPU (torchrun): every rank runs an independent replica of the workload
(independent sequences: no data-path collective); the step time is the max over
ranks and the value is all ranks' tokens over that time.

--impl reference times the fp64 CPU oracle (the reference implementation of
this method) on the host cores, on an evenly spaced sample of query rows of the
same workload per step, extrapolated to the workload's token rate.
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "DSA fwd tokens/s (indexer+top-k+sparse MLA) at 128K ctx; % of HBM/FP8 roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--workload", default="prefill128k")
    ap.add_argument("--e2e-steps", type=int, default=5)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true", help="skip the oracle cpu_baseline leg")
    ap.add_argument("--cpu-seconds", type=float, default=24.0,
                    help="oracle time of the cpu_baseline leg (split between all cores and one thread)")
    ap.add_argument("--decode-steps", type=int, default=10,
                    help="timed steps of the ragged 128K decode measurement (0 = skip)")
    ap.add_argument("--dense-steps", type=int, default=1,
                    help="timed calls of dense MLA over the same prefill, for the sparse/dense ratio (0 = skip)")
    return ap.parse_args()


# ----------------------------------------------------------------------------
# algorithmic work of the workload (per query row: n = p+1 candidates)
# ----------------------------------------------------------------------------
def row_candidates(seqlens_q, seqlens_kv):
    out = []
    for nq, nkv in zip(seqlens_q, seqlens_kv):
        out.append(np.arange(nkv - nq, nkv, dtype=np.int64) + 1)
    return np.concatenate(out) if out else np.zeros(0, np.int64)


def work_model(wl):
    n = row_candidates(wl.seqlens_q, wl.seqlens_kv)
    kk = np.minimum(n, wl.topk)
    HI, dI, H = wl.n_idx_heads, wl.idx_dim, wl.n_heads
    return {
        "n": n,
        # indexer: one H_I x d_I dot product per (query, candidate) pair
        "indexer_flops": lambda rows: 2.0 * HI * dI * float(n[rows].sum()),
        # sparse MLA: QK^T over d_qk and PV over d_v, per (query, head, selected row)
        "mla_flops": lambda rows: 2.0 * H * (wl.d_qk + wl.d_v) * float(kk[rows].sum()),
        # top-k: read each candidate score once, write k indices
        "topk_bytes": lambda rows: 4.0 * float(n[rows].sum()) + 4.0 * wl.topk * len(n[rows]),
        # sparse MLA bytes: gathered latent rows, Q, out, indices
        "mla_bytes": lambda rows: float((kk[rows] * wl.d_qk * 2).sum()
                                        + len(n[rows]) * (H * wl.d_qk * 2 + H * wl.d_v * 2 + wl.topk * 4)),
    }


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


KERNEL_SOURCES = {"mla_tc": "mla_tc.cuh", "indexer_tc": "indexer_tc.cuh", "topk": "topk.cuh"}


def kernel_source_sha(name):
    """sha256 of the kernel's source file plus the shared headers: traffic
    counters taken on another version of the kernel are not reused."""
    import hashlib
    csrc = os.path.join(ROOT, "sparse_long_context_07_b300", "csrc")
    h = hashlib.sha256()
    for f in (KERNEL_SOURCES.get(name, ""), "ptx.cuh", "common.cuh"):
        p = os.path.join(csrc, f)
        if f and os.path.exists(p):
            with open(p, "rb") as fh:
                h.update(fh.read())
    return h.hexdigest()[:16]


def load_traffic():
    """DRAM bytes per launch from the committed ncu summary, for kernels whose
    source still matches the one the counters were taken on."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            tab = json.load(f)
    except Exception:
        return {}
    out = {}
    for name, ent in tab.items():
        if isinstance(ent, dict) and ent.get("source_sha") == kernel_source_sha(name):
            out[name] = {k: v for k, v in ent.items() if k != "source_sha"}
    return out


# ----------------------------------------------------------------------------
# clocks during the timed region
# ----------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = tempfile.mktemp(suffix=".csv")

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    mx = max(mx, float(parts[2]))
                except ValueError:
                    continue
                for nm, v in zip(names, parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(nm)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------
# oracle timing (cpu_baseline and the reference arm)
# ----------------------------------------------------------------------------
def oracle_sample(wl, target_s, seed=0, threads=None):
    """Time the fp64 oracle on evenly spaced query rows of the workload (the
    grid of rows is shifted by a seeded offset, so different seeds time
    different rows).  `threads` limits the BLAS threads (None: all).
    Returns (tokens/s extrapolated to the whole workload, description, seconds
    measured, threads used)."""
    import oracle
    from tests.helpers import cu_np, idx_real, mla_real

    cu_q, cu_kv = cu_np(wl)
    _, pos, kv0, n = oracle.query_positions(cu_q, cu_kv)
    T = len(n)
    w_all = wl.w.float().cpu().numpy().astype(np.float64)
    with _blas().limit(threads):
        used = blas_threads()
        # decode of the key rows is per sequence, timed once and charged in full
        t0 = time.perf_counter()
        k_all = idx_real(wl, "k")
        t_decode = time.perf_counter() - t0

        def one(r):
            q = idx_real(wl, "q", [r])[0]
            I = oracle.index_scores_row(q, k_all[kv0[r]:kv0[r] + n[r]], w_all[r])
            sel = oracle.topk_indices(I, wl.topk)
            valid = sel[sel >= 0]
            Q = mla_real(wl.Q, [r])[0]
            kv = mla_real(wl.KV, kv0[r] + valid)
            oracle.sparse_mla_row(Q, kv, np.arange(len(valid)), wl.scale, wl.d_v)

        # probe the per-row cost on the middle row (second, warm call), then
        # size the sample
        one(T // 2)
        t0 = time.perf_counter()
        one(T // 2)
        probe = time.perf_counter() - t0
        R = int(max(4, min(T, target_s / max(probe, 1e-4))))
        off = np.random.default_rng(seed).random() if seed else 0.5
        rows = np.unique(np.minimum(T - 1, ((np.arange(R) + off) * T / R).astype(np.int64)))
        t0 = time.perf_counter()
        for r in rows:
            one(int(r))
        el = time.perf_counter() - t0
    per_row = el / len(rows)
    total_s = t_decode + per_row * T
    desc = (f"{len(rows)} evenly spaced query rows of {wl.name} (T={T}, offset {off:.3f}); per-row oracle "
            f"time x T + one decode of the key cache, {el + t_decode:.1f} s measured, {used} BLAS thread(s)")
    return T / total_s, desc, el + t_decode, used


def cpu_baseline(wl, seconds):
    """The oracle on all host cores and on one thread (each about half of
    `seconds`); `value` is the all-core figure."""
    tps, desc, _, used = oracle_sample(wl, seconds / 2)
    tps1, desc1, _, _ = oracle_sample(wl, seconds / 2, seed=1, threads=1)
    return {"value": tps, "unit": "tokens/s", "cores": used, "kind": "oracle", "sample": desc,
            "single_thread": {"value": tps1, "unit": "tokens/s", "cores": 1, "sample": desc1},
            "host_cpus": os.cpu_count()}


class _BlasThreads:
    """Get / set the thread count of numpy's OpenBLAS: threadpoolctl when it is
    installed, else the library's own entry points found through ctypes."""

    def __init__(self):
        self.get = self.set = None
        try:
            import threadpoolctl  # noqa: F401
            self.kind = "threadpoolctl"
            return
        except Exception:
            pass
        import ctypes
        import re
        import numpy  # noqa: F401  (loads its BLAS)
        try:
            with open("/proc/self/maps") as f:
                libs = sorted(set(re.findall(r"(/\S*openblas\S*\.so\S*)", f.read())))
        except OSError:
            libs = []
        for path in libs:
            h = ctypes.CDLL(path)
            for pre in ("scipy_openblas_", "openblas_"):
                for suf in ("64_", ""):
                    g, st = f"{pre}get_num_threads{suf}", f"{pre}set_num_threads{suf}"
                    if hasattr(h, g) and hasattr(h, st):
                        self.get, self.set = getattr(h, g), getattr(h, st)
                        self.get.restype = ctypes.c_int
                        self.set.argtypes = [ctypes.c_int]
                        self.kind = "openblas"
                        return
        self.kind = None

    def limit(self, n):
        """Context manager: at most n BLAS threads inside (None: unchanged)."""
        import contextlib
        if n is None or self.kind is None:
            return contextlib.nullcontext()
        if self.kind == "threadpoolctl":
            from threadpoolctl import threadpool_limits
            return threadpool_limits(limits=n, user_api="blas")
        outer = self

        class _Ctx:
            def __enter__(self):
                self.old = outer.get()
                outer.set(int(n))

            def __exit__(self, *exc):
                outer.set(self.old)
        return _Ctx()


_BLAS = None


def _blas():
    global _BLAS
    if _BLAS is None:
        _BLAS = _BlasThreads()
    return _BLAS


def blas_threads():
    """Threads numpy's BLAS uses now."""
    b = _blas()
    if b.kind == "openblas":
        return int(b.get())
    try:
        from threadpoolctl import threadpool_info
        th = [i.get("num_threads", 1) for i in threadpool_info() if i.get("user_api") == "blas"]
        if th:
            return int(max(th))
    except Exception:
        pass
    return os.cpu_count() or 1


# ----------------------------------------------------------------------------
def main():
    a = parse()
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl" if a.impl == "native" else "gloo")

    import dsa_synth

    if a.impl == "reference":
        if rank != 0:
            return
        run_reference(a, world)
        return

    import sparse_long_context_07_b300 as dsa

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    # each rank owns an independent replica (its own seeded sequence)
    wl = dsa_synth.WORKLOADS[a.workload](device=dev)
    if world > 1 and rank > 0:
        wl = reseed(wl, rank, dev)
    b = dsa.Batch(wl.cu_q, wl.cu_kv, wl.seqlens_q, wl.seqlens_kv)
    ix = dsa.Indexer(wl.q_idx, wl.k_idx, wl.w, wl.q_scale, wl.k_scale)
    m = dsa.Mla(wl.Q, wl.KV, wl.scale, wl.d_v)
    T = wl.total_q
    k = wl.topk
    out = torch.empty((T, wl.n_heads, wl.d_v), dtype=wl.Q.dtype, device=dev)
    lse = torch.empty((T, wl.n_heads), dtype=torch.float32, device=dev)
    _, pref = dsa.workspace_size(b, ix, m, k)
    ws = torch.empty(pref, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(trace=None):
        dsa.forward(b, ix, m, k, out, lse, None, ws, stream=stream, trace=trace)

    for _ in range(max(3, a.warmup)):
        step()
    torch.cuda.synchronize()
    if dsa.read_device_errors() != 0:
        raise RuntimeError("device error word set during warm-up")

    traces = [dsa.Trace(capacity=1024) for _ in range(a.steps)]
    clocks = ClockSampler(local)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(a.steps + 1)]
    evs[0].record(stream)
    for i in range(a.steps):
        step(traces[i])
        evs[i + 1].record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    if world > 1:
        dist.barrier()
    per_step = [evs[i].elapsed_time(evs[i + 1]) for i in range(a.steps)]
    # the median step of the slowest rank; the mean of all K steps beside it
    ms_per_step = max_over_ranks(statistics.median(per_step), world, dev)
    ms_mean = max_over_ranks(evs[0].elapsed_time(evs[-1]) / a.steps, world, dev)
    tokens_per_step = T * world
    value = job_rate(tokens_per_step, ms_per_step)

    # per-kernel durations from the launch trace
    per_kernel = {}
    launches = 0
    for tr in traces:
        for name, t in tr.launches():
            d = per_kernel.setdefault(name, [0.0, 0])
            d[0] += t
            d[1] += 1
            launches += 1
    roof = roofline(wl, per_kernel, a.steps)
    if roof is not None:
        roof["launch_ms_note"] = "per-kernel CUDA-event times summed over the K timed steps"

    e2e = None
    if not a.no_e2e:
        e2e = measure_e2e(a, wl, dsa, b, ix, m, out, lse, ws, stream, world, dev)

    dense = None
    if a.dense_steps > 0:
        dense = measure_dense(a, dsa, wl, b, m, out, lse, stream, ms_per_step)

    decode = None
    if a.decode_steps > 0 and a.workload != "ragged128k":
        del out, lse, ws
        torch.cuda.empty_cache()
        decode = measure_decode(a, dsa, dev, stream)
        decode["quantize"] = measure_quant(a, dsa, dev, stream)
        if roof is not None:
            roof["kernels"] += decode_rooflines(decode)

    if rank != 0:
        return
    cpu = None
    if world == 1 and not a.no_cpu:
        cpu = cpu_baseline(wl, a.cpu_seconds)
    line = {
        "metric": METRIC,
        "value": value,
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": a.steps,
        "warmup": max(3, a.warmup),
        "ms_per_step": ms_per_step,
        "ms_per_step_mean": ms_mean,
        "timing": "median of K per-step CUDA-event times (max over ranks); mean beside it",
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "e4m3+bf16",
        "data": "synthetic",
        "config": {"workload": wl.name, "seqlens_q": summarize(wl.seqlens_q),
                   "seqlens_kv": summarize(wl.seqlens_kv), "topk": k,
                   "indexer": f"{wl.n_idx_heads}x{wl.idx_dim} {wl.idx_dtype}",
                   "mla": f"{wl.n_heads} heads d_qk={wl.d_qk} d_v={wl.d_v} {wl.mla_dtype}",
                   "tokens_per_step": tokens_per_step,
                   "l2": "inputs larger than L2 (no flush needed)", "parallelism": f"replicas x{world}"},
        "roofline": roof,
        "kernels_ms_per_step": {kname: v[0] / a.steps for kname, v in per_kernel.items()},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": launches,
        "clocks": clk,
        "decode": decode,
        "dense_prefill": dense,
    }
    print(json.dumps(line))


def summarize(lens):
    if len(set(lens)) == 1:
        return f"{len(lens)}x{lens[0]}"
    return f"{len(lens)} seqs, {min(lens)}..{max(lens)}, total {sum(lens)}"


def max_over_ranks(value, world, device):
    """The largest of every rank's value: the job's step time is that of its
    slowest rank.  `device` holds the reduction tensor (the GPU under NCCL,
    the CPU under gloo)."""
    if world <= 1:
        return float(value)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(tokens_all_ranks, ms_per_step):
    """Whole-job throughput: every rank's tokens over the slowest rank's time."""
    return tokens_all_ranks / (ms_per_step / 1e3)


def reseed(wl, rank, dev):
    """Rank `rank`'s replica: the workload's own recipe with another seed."""
    import dsa_synth
    return dsa_synth.reseeded(wl, 1000 + rank, dev)


def _peaks():
    """(peaks dict with the e4m3 figures derived, source label).  e4m3 dense
    = 2 x the measured bf16 cuBLAS rate (the nominal fp8:bf16 ratio)."""
    peaks, src = load_peaks()
    burst = peaks.get("bf16_tflops")
    sus = peaks.get("bf16_tflops_sustained", burst)
    return {"bf16_burst": burst, "bf16_sustained": sus, "e4m3_burst": 2.0 * burst,
            "e4m3_sustained": 2.0 * sus, "hbm": peaks.get("hbm_gbs")}, src


def _entry(kernel, bound, unit, work, seconds, pk, peak_key, src, extra=None):
    """One roofline entry: algorithmic work over measured time against the
    sustained (timed inside a long step) and the burst peak."""
    achieved = work / seconds / (1e12 if unit == "TFLOP/s" else 1e9)
    if peak_key == "hbm":
        sus = burst = pk["hbm"]
        note = f"{src} copy bandwidth"
    else:
        sus, burst = pk[peak_key + "_sustained"], pk[peak_key + "_burst"]
        note = (f"{src} cuBLAS bf16" if peak_key == "bf16" else f"2 x {src} cuBLAS bf16 (e4m3 dense)") + \
            " rate; frac against the sustained figure, frac_burst against the burst one"
    e = {"kernel": kernel, "bound": bound, "unit": unit, "achieved": achieved, "peak": sus,
         "frac": achieved / sus, "peak_burst": burst, "frac_burst": achieved / burst, "peak_note": note}
    if extra:
        e.update(extra)
    return e


def roofline(wl, per_kernel, steps):
    """Roofline of every kernel of the step: algorithmic work of all its
    launches over their total CUDA-event time, against the measured peaks.
    The top-level fields are those of the dominant kernel (largest total
    time); `kernels` lists all of them."""
    if not per_kernel:
        return None
    pk, src = _peaks()
    wm = work_model(wl)
    allrows = np.arange(len(wm["n"]))
    traffic_tab = load_traffic()
    entries = []
    for name, (tot_ms, nl) in per_kernel.items():
        extra = {"ms_per_step": tot_ms / steps, "launches_per_step": nl / steps, "workload": wl.name}
        secs = tot_ms / 1e3
        if name.startswith("indexer"):
            e = _entry(name, "tensor", "TFLOP/s", wm["indexer_flops"](allrows) * steps, secs, pk, "e4m3", src, extra)
        elif name == "mla_tc" or name == "mla_simt":
            e = _entry(name, "tensor", "TFLOP/s", wm["mla_flops"](allrows) * steps, secs, pk, "bf16", src, extra)
        elif name == "topk":
            e = _entry(name, "hbm", "GB/s", wm["topk_bytes"](allrows) * steps, secs, pk, "hbm", src, extra)
        else:
            continue
        tr = traffic_tab.get(name, {}).get(wl.name)
        e["traffic"] = tr if tr else None
        entries.append(e)
    if not entries:
        return None
    dom = max(entries, key=lambda e: e["ms_per_step"])
    res = {k: dom[k] for k in ("bound", "achieved", "peak", "unit", "frac", "traffic", "kernel", "peak_burst",
                               "frac_burst", "peak_note", "ms_per_step", "launches_per_step")}
    res["kernels"] = entries
    return res


def decode_rooflines(decode):
    """The ragged 128K decode's HBM-bound kernels as roofline entries."""
    out = []
    pk, src = _peaks()
    traffic_tab = load_traffic()
    for key, kernel, tk in (("mla_hbm", "mla_tc+combine (decode)", "mla_tc"),
                            ("indexer_hbm", "indexer_tc (decode)", "indexer_tc")):
        d = decode.get(key)
        if not d:
            continue
        ms = d["ms"]
        out.append(_entry(kernel, "hbm", "GB/s", d["bytes"], ms / 1e3, pk, "hbm", src,
                          {"ms_per_step": ms, "workload": decode["workload"], "l2": "flushed before every step",
                           "traffic": traffic_tab.get(tk, {}).get(decode["workload"])}))
    q = decode.get("quantize")
    if q:
        out.append(_entry("quantize_e4m3", "hbm", "GB/s", q["bytes"], q["ms"] / 1e3, pk, "hbm", src,
                          {"ms_per_step": q["ms"], "workload": q["workload"]}))
    return out


def measure_decode(a, dsa, dev, stream):
    """Secondary measurement: one decode step of 64 sequences with 16K-128K
    cached tokens each (1 query token per sequence), L2 flushed before every
    timed step; reports tokens/s and the HBM fraction of the sparse attention
    and of the indexer (both bandwidth-bound in decode)."""
    import torch
    import dsa_synth
    wl = dsa_synth.WORKLOADS["ragged128k"](device=dev)
    b = dsa.Batch(wl.cu_q, wl.cu_kv, wl.seqlens_q, wl.seqlens_kv)
    ix = dsa.Indexer(wl.q_idx, wl.k_idx, wl.w, wl.q_scale, wl.k_scale)
    m = dsa.Mla(wl.Q, wl.KV, wl.scale, wl.d_v)
    T, k = wl.total_q, wl.topk
    out = torch.empty((T, wl.n_heads, wl.d_v), dtype=wl.Q.dtype, device=dev)
    lse = torch.empty((T, wl.n_heads), dtype=torch.float32, device=dev)
    _, pref = dsa.workspace_size(b, ix, m, k)
    ws = torch.empty(pref, dtype=torch.uint8, device=dev)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)   # 512 MiB > L2
    for _ in range(3):
        dsa.forward(b, ix, m, k, out, lse, None, ws, stream=stream)
    torch.cuda.synchronize()
    # the step as a caller runs it (no launch trace: the attention kernel may
    # overlap the end of the top-k), then the same number of traced steps for
    # each kernel's own time
    totals, traced_totals, per_kernel = [], [], {}
    for traced in (False, True):
        for _ in range(a.decode_steps):
            flush.fill_(1)
            tr = dsa.Trace(capacity=64) if traced else None
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            dsa.forward(b, ix, m, k, out, lse, None, ws, stream=stream, trace=tr)
            e1.record(stream)
            torch.cuda.synchronize()
            (traced_totals if traced else totals).append(e0.elapsed_time(e1))
            if traced:
                for name, t in tr.launches():
                    per_kernel.setdefault(name, []).append(t)
    if dsa.read_device_errors() != 0:
        raise RuntimeError("device error word set during the decode measurement")
    # dense baseline: MLA over every cached token of every sequence
    need = dsa.dense_mla_workspace_size(b, m)
    dws = torch.empty(max(need, 16), dtype=torch.uint8, device=dev) if need else None
    dsa.dense_mla(b, m, out, lse, dws, stream=stream)
    dense_t = []
    for _ in range(max(3, a.decode_steps // 2)):
        flush.fill_(1)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        dsa.dense_mla(b, m, out, lse, dws, stream=stream)
        e1.record(stream)
        torch.cuda.synchronize()
        dense_t.append(e0.elapsed_time(e1))
    peaks, src = load_peaks()
    ms = statistics.median(totals)
    kms = {kname: statistics.median(v) for kname, v in per_kernel.items()}
    nkv = np.asarray(wl.seqlens_kv, dtype=np.float64)
    kk = np.minimum(nkv, k)
    # algorithmic bytes: indexer reads every candidate key (128 B + 4 B scale) and
    # the query (8 KiB + 256 B weights + scale); sparse MLA gathers the selected
    # latent rows and reads Q, writes out, reads the indices
    idx_bytes = float((nkv * (wl.idx_dim + 4)).sum() + T * (wl.n_idx_heads * wl.idx_dim + 4 * wl.n_idx_heads + 4))
    mla_bytes = float((kk * wl.d_qk * 2).sum() + T * (wl.n_heads * wl.d_qk * 2 + wl.n_heads * wl.d_v * 2 + 4 * k))
    mla_ms = kms.get("mla_tc", 0.0) + kms.get("mla_combine", 0.0)
    res = {"workload": wl.name, "tokens_per_step": T, "ms_per_step": ms, "value": T / (ms / 1e3),
           "unit": "tokens/s", "steps": a.decode_steps, "l2": "flushed before every step (512 MiB write)",
           "ms_per_step_traced": statistics.median(traced_totals),
           "kernels_ms_per_step": kms, "kernels_note": "from as many steps again with a launch trace",
           "dense_mla_ms": statistics.median(dense_t),
           "dense_mla_over_dsa_step": statistics.median(dense_t) / ms}
    if mla_ms > 0:
        gbs = mla_bytes / (mla_ms / 1e3) / 1e9
        res["mla_hbm"] = {"achieved": gbs, "peak": peaks.get("hbm_gbs"), "unit": "GB/s",
                          "frac": gbs / peaks.get("hbm_gbs"), "bytes": mla_bytes, "ms": mla_ms,
                          "note": f"{src} copy bandwidth"}
    if kms.get("indexer_tc"):
        gbs = idx_bytes / (kms["indexer_tc"] / 1e3) / 1e9
        res["indexer_hbm"] = {"achieved": gbs, "peak": peaks.get("hbm_gbs"), "unit": "GB/s",
                              "frac": gbs / peaks.get("hbm_gbs"), "bytes": idx_bytes, "ms": kms["indexer_tc"]}
    return res


def measure_dense(a, dsa, wl, b, m, out, lse, stream, dsa_ms):
    """Dense causal MLA-MQA over every candidate of the same workload (the
    baseline of the pages' DSA-vs-dense cost claims), against the whole DSA
    forward step just measured."""
    import torch
    need = dsa.dense_mla_workspace_size(b, m)
    ws = torch.empty(max(need, 16), dtype=torch.uint8, device=out.device) if need else None
    dsa.dense_mla(b, m, out, lse, ws, stream=stream)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(a.dense_steps):
        dsa.dense_mla(b, m, out, lse, ws, stream=stream)
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / a.dense_steps
    n = row_candidates(wl.seqlens_q, wl.seqlens_kv).astype(np.float64)
    flops = 2.0 * wl.n_heads * (wl.d_qk + wl.d_v) * float(n.sum())
    return {"workload": wl.name, "dense_mla_ms": ms, "dsa_forward_ms": dsa_ms, "dense_over_dsa": ms / dsa_ms,
            "dense_tflops": flops / (ms / 1e3) / 1e12, "steps": a.dense_steps}


def measure_quant(a, dsa, dev, stream):
    """Producer step: e4m3 quantisation of the 131072-token prefill's indexer
    queries (bf16 [131072, 64, 128] in, codes + one scale per token out), an
    HBM-bound stream; reports GB/s against the measured copy bandwidth."""
    import torch
    T, G = 131072, 64 * 128
    g = torch.Generator(device=dev)
    g.manual_seed(11)
    x = torch.randn((T, G), generator=g, device=dev).to(torch.bfloat16)
    codes = torch.empty((T, G), dtype=torch.uint8, device=dev)
    scales = torch.empty((T,), dtype=torch.float32, device=dev)
    for _ in range(3):
        dsa.quantize_e4m3(x, codes, scales, G, stream=stream)
    torch.cuda.synchronize()
    n = max(3, a.decode_steps)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(n):
        dsa.quantize_e4m3(x, codes, scales, G, stream=stream)
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / n
    nbytes = float(T * G * 2 + T * G + 4 * T)   # bf16 read, codes written, scales written
    peaks, src = load_peaks()
    gbs = nbytes / (ms / 1e3) / 1e9
    return {"workload": "indexer queries of the 131072-token prefill, bf16 -> e4m3", "ms": ms, "bytes": nbytes,
            "achieved": gbs, "peak": peaks.get("hbm_gbs"), "unit": "GB/s", "frac": gbs / peaks.get("hbm_gbs"),
            "note": f"{src} copy bandwidth; inputs larger than L2"}


def measure_e2e(a, wl, dsa, b, ix, m, out, lse, ws, stream, world, dev):
    """Same metric end to end through dsa_forward_streamed: every step copies
    the inputs from pinned host memory into the device tensors the forward
    reads and returns out + lse to pinned host memory.  The library overlaps
    the copies (two copy streams) with the kernels, query chunk by chunk."""
    import torch
    pin = {name: (getattr(wl, name).cpu().pin_memory() if getattr(wl, name) is not None else None)
           for name in ("q_idx", "q_scale", "k_idx", "k_scale", "w", "Q", "KV")}
    host = dsa.HostInputs(pin["q_idx"], pin["k_idx"], pin["w"], pin["Q"], pin["KV"], pin["q_scale"],
                          pin["k_scale"])
    host_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    host_lse = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in pin.values() if t is not None)
    d2h = host_out.numel() * host_out.element_size() + host_lse.numel() * host_lse.element_size()
    copy_in, copy_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def step():
        dsa.forward_streamed(b, ix, m, wl.topk, host, out, lse, host_out, host_lse, ws, stream=stream,
                             copy_in=copy_in, copy_out=copy_out)

    step()
    torch.cuda.synchronize()
    n = max(1, a.e2e_steps)
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(n + 1)]
    evs[0].record(stream)
    for i in range(n):
        step()
        evs[i + 1].record(stream)
    torch.cuda.synchronize()
    per_step = [evs[i].elapsed_time(evs[i + 1]) for i in range(n)]
    ms = max_over_ranks(statistics.median(per_step), world, dev)
    ms_mean = max_over_ranks(evs[0].elapsed_time(evs[-1]) / n, world, dev)
    return {"value": job_rate(wl.total_q * world, ms), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": ms, "ms_per_step_mean": ms_mean, "steps": n,
            "api": "dsa_forward_streamed (copies overlap the kernels, query chunk by chunk)"}


def run_reference(a, world):
    """The fp64 oracle on the host cores, on the native arm's workload."""
    import torch
    import dsa_synth
    # inputs are drawn on the GPU when there is one (generation is not timed);
    # the oracle reads the rows it needs back to the host
    gen_dev = "cuda" if torch.cuda.is_available() else "cpu"
    wl = dsa_synth.WORKLOADS[a.workload](device=gen_dev)
    for _ in range(max(0, a.warmup)):
        pass  # the oracle has no state to warm up
    vals, descs, secs = [], [], []
    cores = blas_threads()
    for i in range(a.steps):
        # each step times a different seeded grid of rows
        tps, desc, s, cores = oracle_sample(wl, max(1.0, a.cpu_seconds / max(1, a.steps)), seed=i + 1)
        vals.append(tps)
        descs.append(desc)
        secs.append(s)
    value = statistics.median(vals)
    line = {
        "impl": "reference",
        "metric": METRIC,
        "value": value,
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": a.steps,
        "warmup": a.warmup,
        "ms_per_step": wl.total_q / value * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": wl.name, "seqlens_q": summarize(wl.seqlens_q),
                   "seqlens_kv": summarize(wl.seqlens_kv), "topk": wl.topk},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": descs[0]},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


if __name__ == "__main__":
    main()
