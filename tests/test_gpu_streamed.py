"""dsa_forward_streamed: inputs copied from pinned host memory chunk by chunk
while earlier chunks compute, results copied back.  The same kernels run on
the same values as dsa_forward, so outputs must match bit for bit; the device
buffers start empty, so every input has to arrive through the copies."""

import pytest
import torch

import dsa_synth
import sparse_long_context_07_b300 as dsa
from tests.gpu_util import structs

pytestmark = pytest.mark.gpu


def _streamed(wl, k, ws_bytes=None, split_streams=True):
    # fresh device buffers: the streamed call must fill them from the host
    dev = {name: torch.zeros_like(getattr(wl, name)) if getattr(wl, name) is not None else None
           for name in ("q_idx", "q_scale", "k_idx", "k_scale", "w", "Q", "KV")}
    ix = dsa.Indexer(dev["q_idx"], dev["k_idx"], dev["w"], dev["q_scale"], dev["k_scale"])
    m = dsa.Mla(dev["Q"], dev["KV"], wl.scale, wl.d_v)
    b = dsa.Batch(wl.cu_q, wl.cu_kv, wl.seqlens_q, wl.seqlens_kv)
    pin = {name: (getattr(wl, name).cpu().pin_memory() if getattr(wl, name) is not None else None)
           for name in dev}
    host = dsa.HostInputs(pin["q_idx"], pin["k_idx"], pin["w"], pin["Q"], pin["KV"], pin["q_scale"],
                          pin["k_scale"])
    T = wl.total_q
    out = torch.empty((T, wl.n_heads, wl.d_v), dtype=wl.Q.dtype, device="cuda")
    lse = torch.empty((T, wl.n_heads), device="cuda")
    host_out = torch.full(out.shape, float("nan"), dtype=out.dtype).pin_memory()
    host_lse = torch.full(lse.shape, float("nan")).pin_memory()
    mn, pref = dsa.workspace_size(b, ix, m, k)
    ws = torch.empty(ws_bytes or pref, dtype=torch.uint8, device="cuda")
    s = torch.cuda.current_stream()
    cin = torch.cuda.Stream() if split_streams else None
    cout = torch.cuda.Stream() if split_streams else None
    dsa.forward_streamed(b, ix, m, k, host, out, lse, host_out, host_lse, ws, stream=s, copy_in=cin,
                         copy_out=cout)
    s.synchronize()
    assert dsa.read_device_errors() == 0
    for name in dev:
        if dev[name] is not None:
            a, b_ = dev[name], getattr(wl, name)
            if a.element_size() == 1:      # compare e4m3 codes as bytes
                a, b_ = a.view(torch.uint8), b_.view(torch.uint8)
            assert torch.equal(a, b_), f"device copy of {name}"
    return host_out, host_lse


def _reference(wl, k, ws_bytes=None):
    b, ix, m = structs(wl)
    T = wl.total_q
    out = torch.empty((T, wl.n_heads, wl.d_v), dtype=wl.Q.dtype, device="cuda")
    lse = torch.empty((T, wl.n_heads), device="cuda")
    mn, pref = dsa.workspace_size(b, ix, m, k)
    ws = torch.empty(ws_bytes or pref, dtype=torch.uint8, device="cuda")
    dsa.forward(b, ix, m, k, out, lse, None, ws)
    torch.cuda.synchronize()
    assert dsa.read_device_errors() == 0
    return out.cpu(), lse.cpu()


def test_streamed_matches_forward_over_many_chunks():
    # the minimum workspace forces 64-row chunks: five chunks of copies in,
    # kernels and copies out
    k = 128
    wl = dsa_synth.make_workload("stream-chunks", [300], [300], grid=True, device="cuda", seed=41)
    b, ix, m = structs(wl)
    mn, _ = dsa.workspace_size(b, ix, m, k)
    ref_o, ref_l = _reference(wl, k, ws_bytes=mn)
    for split in (True, False):
        ho, hl = _streamed(wl, k, ws_bytes=mn, split_streams=split)
        assert torch.equal(ho, ref_o) and torch.equal(hl, ref_l)


def test_streamed_matches_forward_ragged_decode():
    wl = dsa_synth.decode8k(device="cuda")
    ref_o, ref_l = _reference(wl, wl.topk)
    ho, hl = _streamed(wl, wl.topk)
    assert torch.equal(ho, ref_o) and torch.equal(hl, ref_l)


def test_streamed_rejects_missing_host_copies():
    wl = dsa_synth.make_workload("stream-bad", [64], [64], grid=True, device="cuda", seed=42)
    b, ix, m = structs(wl)
    assert wl.q_scale is not None
    host = dsa.HostInputs(wl.q_idx.cpu(), wl.k_idx.cpu(), wl.w.cpu(), wl.Q.cpu(), wl.KV.cpu(),
                          None, None if wl.k_scale is None else wl.k_scale.cpu())
    out = torch.empty((64, wl.n_heads, wl.d_v), dtype=wl.Q.dtype, device="cuda")
    host_out = torch.empty(out.shape, dtype=out.dtype)
    mn, pref = dsa.workspace_size(b, ix, m, 64)
    ws = torch.empty(pref, dtype=torch.uint8, device="cuda")
    with pytest.raises(dsa.DSAError) as e:
        dsa.forward_streamed(b, ix, m, 64, host, out, None, host_out, None, ws)
    assert e.value.status == dsa.ERROR_INVALID_VALUE
