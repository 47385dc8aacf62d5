"""Seeded synthetic inputs for the DSA forward pass.

Shared by the tests, ``bench.py`` and ``__graft_entry__.smoke()``: it builds the
input tensors that both the CUDA library and the CPU oracle consume.  It holds
none of the method's arithmetic (no index score, no selection, no attention);
only random draws, the per-row e4m3 quantisation that produces the FP8 inputs,
and the batch geometry.

Workloads (sizes and value distributions of the 128K-context DSA workloads):
  tiny        L=256 prefill, indexer fp32 4 heads x 32, top-k 32,
              MLA 8 heads d_qk=d_v=64 fp32, scale 1/8, N(0,1)  (seed 1;
              integer-grid variant with values in {-2..2}: seed 101)
  decode8k    4 sequences x 8192 cached tokens, 1 query each            (seed 2)
  prefill32k  one 32768-token causal prefill                             (seed 3)
  prefill16k  one 16384-token causal prefill (profiling size)            (seed 6)
  ragged128k  64 decode sequences, context ~ U[16384, 131072], 10% of
              each sequence's keys planted toward its query             (seed 4)
  prefill128k one 131072-token causal prefill                            (seed 5)
  prefill128k_tail, prefill128k_mid, ragged128k_16: profiling-size cases
All but ``tiny`` use the production dimensions: indexer 64 heads x 128 in
e4m3 with per-token fp32 scales and w ~ N(0, 1/64); MLA-MQA 128 heads,
d_qk = 576 (512 latent + 64 rope), d_v = 512, bf16, scale 192^-0.5, top-k 2048.
"""

from __future__ import annotations

import dataclasses
import math
from typing import List, Optional

import torch

E4M3_MAX = 448.0


@dataclasses.dataclass
class Workload:
    name: str
    seqlens_q: List[int]
    seqlens_kv: List[int]
    cu_q: torch.Tensor            # int32 [B+1]
    cu_kv: torch.Tensor           # int32 [B+1]
    # indexer
    idx_dtype: str                # "e4m3" | "f32"
    q_idx: torch.Tensor           # uint8 codes or float32, [T, H_I, d_I]
    q_scale: Optional[torch.Tensor]   # float32 [T] or None
    k_idx: torch.Tensor           # [S, d_I]
    k_scale: Optional[torch.Tensor]   # float32 [S] or None
    w: torch.Tensor               # float32 [T, H_I]
    # sparse MLA
    mla_dtype: str                # "bf16" | "f32"
    Q: torch.Tensor               # [T, H, d_qk]
    KV: torch.Tensor              # [S, d_qk]
    scale: float
    d_v: int
    topk: int
    # every keyword argument of make_workload that drew this workload, so
    # that a replica with another seed (reseeded) has the same recipe
    gen_kwargs: dict = dataclasses.field(default_factory=dict)

    @property
    def total_q(self) -> int:
        return int(sum(self.seqlens_q))

    @property
    def total_kv(self) -> int:
        return int(sum(self.seqlens_kv))

    @property
    def max_q(self) -> int:
        return int(max(self.seqlens_q))

    @property
    def max_kv(self) -> int:
        return int(max(self.seqlens_kv))

    @property
    def n_idx_heads(self) -> int:
        return int(self.q_idx.shape[1])

    @property
    def idx_dim(self) -> int:
        return int(self.q_idx.shape[2])

    @property
    def n_heads(self) -> int:
        return int(self.Q.shape[1])

    @property
    def d_qk(self) -> int:
        return int(self.Q.shape[2])

    def nbytes_inputs(self) -> int:
        ts = [self.cu_q, self.cu_kv, self.q_idx, self.k_idx, self.w, self.Q, self.KV]
        ts += [t for t in (self.q_scale, self.k_scale) if t is not None]
        return int(sum(t.numel() * t.element_size() for t in ts))


def _cu(lens, device):
    cu = [0]
    for n in lens:
        cu.append(cu[-1] + int(n))
    return torch.tensor(cu, dtype=torch.int32, device=device)


def quantize_e4m3_rows(x: torch.Tensor):
    """Per-row absmax quantisation to e4m3: scale = amax / 448, code =
    round-to-nearest-even(x / scale) (saturating).  x: [rows, ...] float32.
    Returns (uint8 codes with x's shape, float32 scales [rows])."""
    rows = x.shape[0]
    flat = x.reshape(rows, -1)
    amax = flat.abs().amax(dim=1)
    # a tensor divisor: division by a Python scalar may run as a multiply by
    # its reciprocal, one ulp away from the IEEE quotient the definition uses
    scale = torch.where(amax > 0, amax / torch.full_like(amax, E4M3_MAX), torch.ones_like(amax))
    y = (flat / scale[:, None]).clamp_(-E4M3_MAX, E4M3_MAX)
    codes = y.to(torch.float8_e4m3fn).view(torch.uint8).reshape(x.shape)
    return codes, scale.to(torch.float32)


def _randn(shape, gen, device, dtype=torch.float32, std=1.0):
    t = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t.to(dtype)


def _grid(shape, gen, device):
    return torch.randint(-2, 3, shape, generator=gen, device=device).to(torch.float32)


def make_workload(name, seqlens_q, seqlens_kv, *, n_idx_heads=64, idx_dim=128,
                  idx_dtype="e4m3", n_heads=128, d_qk=576, d_v=512, mla_dtype="bf16",
                  topk=2048, scale=None, seed=0, grid=False, planted=0.0,
                  w_std=None, device="cpu", chunk_rows=4096):
    """Generic seeded workload.  ``grid`` puts the indexer inputs on the integer
    grid {-2..2} (exact in e4m3 and fp32; scales 1; integer w) so that every
    index score is an exactly representable integer.  ``planted`` > 0 shifts that
    fraction of each sequence's keys toward the sequence's last query (the
    direction sum_j w_j q_j, normalised to norm sqrt(d_I)) before quantisation.
    Large tensors are drawn in row chunks to bound temporary memory."""
    gen_kwargs = dict(n_idx_heads=n_idx_heads, idx_dim=idx_dim, idx_dtype=idx_dtype, n_heads=n_heads,
                      d_qk=d_qk, d_v=d_v, mla_dtype=mla_dtype, topk=topk, scale=scale, seed=seed,
                      grid=grid, planted=planted, w_std=w_std, chunk_rows=chunk_rows)
    device = torch.device(device)
    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed))
    B = len(seqlens_q)
    assert len(seqlens_kv) == B
    T, S = int(sum(seqlens_q)), int(sum(seqlens_kv))
    if scale is None:
        scale = 1.0 / math.sqrt(192.0)
    if w_std is None:
        w_std = 1.0 / 8.0 if idx_dtype == "e4m3" else 1.0
    HI, dI = n_idx_heads, idx_dim

    # ---- indexer queries and weights
    if grid:
        qf = _grid((T, HI, dI), gen, device)
        w = _grid((T, HI), gen, device)
    else:
        qf = _randn((T, HI, dI), gen, device)
        w = _randn((T, HI), gen, device, std=w_std)
    # ---- indexer keys (chunked), planted toward each sequence's last query
    kf = torch.empty((S, dI), dtype=torch.float32, device=device)
    for r0 in range(0, S, chunk_rows * 16):
        r1 = min(S, r0 + chunk_rows * 16)
        kf[r0:r1] = _grid((r1 - r0, dI), gen, device) if grid else _randn((r1 - r0, dI), gen, device)
    if planted > 0.0:
        cq = [0]
        ck = [0]
        for b in range(B):
            cq.append(cq[-1] + seqlens_q[b])
            ck.append(ck[-1] + seqlens_kv[b])
        for b in range(B):
            t_last = cq[b + 1] - 1
            u = (w[t_last][:, None] * qf[t_last]).sum(0)
            u = u * (math.sqrt(dI) / max(float(u.norm()), 1e-12))
            nkv = seqlens_kv[b]
            n_pl = int(round(planted * nkv))
            perm = torch.randperm(nkv, generator=gen, device=device)[:n_pl]
            kf[ck[b] + perm] += u[None, :]
    if idx_dtype == "e4m3":
        if grid:
            q_idx = qf.to(torch.float8_e4m3fn).view(torch.uint8)
            k_idx = kf.to(torch.float8_e4m3fn).view(torch.uint8)
            q_scale = torch.ones(T, dtype=torch.float32, device=device)
            k_scale = torch.ones(S, dtype=torch.float32, device=device)
        else:
            q_idx, q_scale = quantize_e4m3_rows(qf)
            k_idx = torch.empty((S, dI), dtype=torch.uint8, device=device)
            k_scale = torch.empty(S, dtype=torch.float32, device=device)
            for r0 in range(0, S, chunk_rows * 16):
                r1 = min(S, r0 + chunk_rows * 16)
                k_idx[r0:r1], k_scale[r0:r1] = quantize_e4m3_rows(kf[r0:r1])
    elif idx_dtype == "f32":
        q_idx, k_idx, q_scale, k_scale = qf, kf, None, None
    else:
        raise ValueError(idx_dtype)
    del kf

    # ---- MLA queries and latent cache (chunked)
    mdt = torch.bfloat16 if mla_dtype == "bf16" else torch.float32
    Q = torch.empty((T, n_heads, d_qk), dtype=mdt, device=device)
    for r0 in range(0, T, chunk_rows):
        r1 = min(T, r0 + chunk_rows)
        Q[r0:r1] = _randn((r1 - r0, n_heads, d_qk), gen, device, mdt)
    KV = torch.empty((S, d_qk), dtype=mdt, device=device)
    for r0 in range(0, S, chunk_rows * 16):
        r1 = min(S, r0 + chunk_rows * 16)
        KV[r0:r1] = _randn((r1 - r0, d_qk), gen, device, mdt)

    return Workload(name=name, seqlens_q=list(map(int, seqlens_q)),
                    seqlens_kv=list(map(int, seqlens_kv)),
                    cu_q=_cu(seqlens_q, device), cu_kv=_cu(seqlens_kv, device),
                    idx_dtype=idx_dtype, q_idx=q_idx, q_scale=q_scale, k_idx=k_idx,
                    k_scale=k_scale, w=w, mla_dtype=mla_dtype, Q=Q, KV=KV,
                    scale=float(scale), d_v=int(d_v), topk=int(topk), gen_kwargs=gen_kwargs)


def reseeded(wl: Workload, seed: int, device) -> Workload:
    """The same recipe as `wl` (lengths, dimensions, dtypes, grid, planted
    fraction, ...) drawn with another seed: an independent replica."""
    kw = dict(wl.gen_kwargs)
    kw["seed"] = int(seed)
    return make_workload(wl.name, wl.seqlens_q, wl.seqlens_kv, device=device, **kw)


def ragged_lengths(batch, lo, hi, seed):
    """Context lengths uniform in [lo, hi], drawn from a seeded CPU generator."""
    g = torch.Generator()
    g.manual_seed(int(seed))
    return [int(x) for x in torch.randint(lo, hi + 1, (batch,), generator=g)]


def tiny(device="cpu", grid=False):
    """L=256 causal prefill, fp32 indexer 4x32, top-k 32, MLA 8 heads d=64/64,
    scale 1/8 (seed 1; integer-grid variant seed 101)."""
    return make_workload("tiny-grid" if grid else "tiny", [256], [256], n_idx_heads=4,
                         idx_dim=32, idx_dtype="f32", n_heads=8, d_qk=64, d_v=64,
                         mla_dtype="f32", topk=32, scale=1.0 / 8.0,
                         seed=101 if grid else 1, grid=grid, device=device)


def decode8k(device="cpu", grid=False):
    """4 decode sequences x 8192 cached tokens, 1 query token each."""
    return make_workload("decode8k", [1] * 4, [8192] * 4, seed=2, grid=grid, device=device)


def prefill16k(device="cpu", grid=False):
    """One 16384-token causal prefill (a profiling-size case, inputs > L2)."""
    return make_workload("prefill16k", [16384], [16384], seed=6, grid=grid, device=device)


def prefill32k(device="cpu", grid=False):
    """One 32768-token causal prefill."""
    return make_workload("prefill32k", [32768], [32768], seed=3, grid=grid, device=device)


def ragged128k(device="cpu"):
    """64 decode sequences with context ~ U[16384, 131072], 10% planted keys."""
    lens = ragged_lengths(64, 16384, 131072, seed=4)
    return make_workload("ragged128k", [1] * 64, lens, seed=4, planted=0.10, device=device)


def prefill128k(device="cpu"):
    """One 131072-token causal prefill."""
    return make_workload("prefill128k", [131072], [131072], seed=5, device=device)


def prefill128k_tail(device="cpu"):
    """The last 2048 queries of a 131072-token causal prefill (the whole
    131072-key cache, larger than L2): a profiling case shaped like the late
    query chunks of prefill128k with a few GB on the device."""
    return make_workload("prefill128k_tail", [2048], [131072], seed=5, device=device)


def prefill128k_mid(device="cpu"):
    """The last 2048 queries of a 65536-token causal prefill: shaped like the
    middle query chunks of prefill128k (a 75 MB latent cache in play), with a
    few GB on the device; a profiling case."""
    return make_workload("prefill128k_mid", [2048], [65536], seed=5, device=device)


def ragged128k_16(device="cpu"):
    """The first 16 sequences of ragged128k (same lengths, planted keys): a
    profiling-size decode case."""
    lens = ragged_lengths(64, 16384, 131072, seed=4)[:16]
    return make_workload("ragged128k_16", [1] * 16, lens, seed=4, planted=0.10, device=device)


WORKLOADS = {
    "tiny": tiny,
    "decode8k": decode8k,
    "prefill16k": prefill16k,
    "prefill32k": prefill32k,
    "ragged128k": ragged128k,
    "prefill128k": prefill128k,
    "prefill128k_tail": prefill128k_tail,
    "prefill128k_mid": prefill128k_mid,
    "ragged128k_16": ragged128k_16,
}
