"""Python binding of libdsa.so, the B300 DeepSeek Sparse Attention forward
library (C ABI in include/dsa.h).

Argument marshalling only: every step of the forward pass runs in the
library's CUDA kernels.  Tensors are torch CUDA tensors (PyTorch provides the
device memory and streams); their data pointers go straight to the C entry
points.  The library is loaded on first use; every entry point raises
ImportError when libdsa.so has not been built (``python -m
sparse_long_context_07_b300.build``).  There is no fallback path.
"""

from __future__ import annotations

import ctypes
import os
import re
from typing import Optional, Sequence

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdsa.so")
HEADER_PATH = os.path.join(os.path.dirname(_HERE), "include", "dsa.h")

_lib = None

# ---- constants mirrored from dsa.h
SUCCESS = 0
ERROR_INVALID_VALUE = 1
ERROR_NOT_SUPPORTED = 2
ERROR_INSUFFICIENT_WORKSPACE = 3
ERROR_LAUNCH = 4
ERROR_DEVICE = 5
ERROR_TIMEOUT = 6
ERROR_BAD_INDEX = 7
DTYPE_F32, DTYPE_BF16, DTYPE_E4M3 = 0, 1, 2
DEVERR_TIMEOUT, DEVERR_BAD_INDEX = 0x1, 0x2
KERNEL_NAMES = {1: "indexer_tc", 2: "indexer_simt", 3: "topk", 4: "mla_tc", 5: "mla_simt",
                6: "mla_combine", 7: "hist_clear"}


class DSAError(RuntimeError):
    def __init__(self, status: int, where: str):
        msg = lib().dsa_last_error_message().decode()
        super().__init__(f"{where}: {status_string(status)} ({status}): {msg}")
        self.status = status


class _Batch(ctypes.Structure):
    _fields_ = [("num_seqs", ctypes.c_int32), ("cu_seqlens_q", ctypes.c_void_p),
                ("cu_seqlens_kv", ctypes.c_void_p), ("max_seqlen_q", ctypes.c_int32),
                ("max_seqlen_kv", ctypes.c_int32), ("total_q", ctypes.c_int64),
                ("total_kv", ctypes.c_int64)]


class _Indexer(ctypes.Structure):
    _fields_ = [("n_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("dtype", ctypes.c_int),
                ("q", ctypes.c_void_p), ("q_scale", ctypes.c_void_p), ("k", ctypes.c_void_p),
                ("k_scale", ctypes.c_void_p), ("w", ctypes.c_void_p)]


class _Mla(ctypes.Structure):
    _fields_ = [("n_heads", ctypes.c_int32), ("d_qk", ctypes.c_int32), ("d_v", ctypes.c_int32),
                ("scale", ctypes.c_float), ("dtype", ctypes.c_int), ("q", ctypes.c_void_p),
                ("kv", ctypes.c_void_p)]


class _HostInputs(ctypes.Structure):
    _fields_ = [("idx_q", ctypes.c_void_p), ("idx_q_scale", ctypes.c_void_p), ("idx_k", ctypes.c_void_p),
                ("idx_k_scale", ctypes.c_void_p), ("idx_w", ctypes.c_void_p), ("mla_q", ctypes.c_void_p),
                ("mla_kv", ctypes.c_void_p)]


class _Trace(ctypes.Structure):
    _fields_ = [("capacity", ctypes.c_int32), ("count", ctypes.c_int32),
                ("events", ctypes.POINTER(ctypes.c_void_p)),
                ("kernel_ids", ctypes.POINTER(ctypes.c_int32))]


_P = ctypes.c_void_p
_sig = {
    "dsa_abi_version": (ctypes.c_int32, []),
    "dsa_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "dsa_last_error_message": (ctypes.c_char_p, []),
    "dsa_workspace_size": (ctypes.c_int, [_P, _P, _P, ctypes.c_int32, ctypes.POINTER(ctypes.c_size_t),
                                          ctypes.POINTER(ctypes.c_size_t)]),
    "dsa_index_scores": (ctypes.c_int, [_P, _P, _P, ctypes.c_int64, _P]),
    "dsa_dense_mla_workspace_size": (ctypes.c_int, [_P, _P, ctypes.POINTER(ctypes.c_size_t)]),
    "dsa_dense_mla": (ctypes.c_int, [_P, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "dsa_quantize_e4m3": (ctypes.c_int, [_P, ctypes.c_int, ctypes.c_int64, ctypes.c_int32, _P, _P, _P]),
    "dsa_topk": (ctypes.c_int, [_P, _P, ctypes.c_int64, ctypes.c_int32, _P, _P, _P]),
    "dsa_index_scores_hist": (ctypes.c_int, [_P, _P, _P, ctypes.c_int64, _P, _P]),
    "dsa_topk_hist": (ctypes.c_int, [_P, _P, ctypes.c_int64, _P, ctypes.c_int32, _P, _P, _P]),
    "dsa_sparse_mla": (ctypes.c_int, [_P, _P, _P, ctypes.c_int32, _P, _P, _P, ctypes.c_size_t, _P]),
    "dsa_sparse_mla_noalloc": (ctypes.c_int, [_P, _P, _P, ctypes.c_int32, _P, _P, _P]),
    "dsa_forward": (ctypes.c_int, [_P, _P, _P, ctypes.c_int32, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "dsa_forward_traced": (ctypes.c_int, [_P, _P, _P, ctypes.c_int32, _P, _P, _P, _P, ctypes.c_size_t,
                                          _P, _P]),
    "dsa_forward_streamed": (ctypes.c_int, [_P, _P, _P, ctypes.c_int32, _P, _P, _P, _P, _P, _P,
                                            ctypes.c_size_t, _P, _P, _P]),
    "dsa_indexer_loss_workspace_size": (ctypes.c_int, [_P, _P, _P, ctypes.POINTER(ctypes.c_size_t),
                                                       ctypes.POINTER(ctypes.c_size_t)]),
    "dsa_indexer_warmup_loss": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "dsa_read_device_errors": (ctypes.c_int, [_P, ctypes.POINTER(ctypes.c_uint32)]),
    "dsa_debug_inject_fault": (None, [ctypes.c_uint32]),
}


def lib():
    """The loaded libdsa.so (loaded on first call)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(
                f"{LIB_PATH} is missing: build it with `python -m sparse_long_context_07_b300.build`")
        handle = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _sig.items():
            f = getattr(handle, name)
            f.restype = res
            f.argtypes = args
        _lib = handle
    return _lib


def header_functions() -> list:
    """Names of the functions declared in include/dsa.h."""
    with open(HEADER_PATH) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*(dsa_[a-z_0-9]+)\s*\(",
                                 text, flags=re.M)))


def status_string(status: int) -> str:
    return lib().dsa_status_string(int(status)).decode()


def abi_version() -> int:
    return int(lib().dsa_abi_version())


def _check(status: int, where: str):
    if status != SUCCESS:
        raise DSAError(status, where)


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensors passed to libdsa must live on a CUDA device")
    if not t.is_contiguous():
        raise ValueError("tensors passed to libdsa must be contiguous")
    return t.data_ptr()


def _stream(stream) -> int:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


class Batch:
    """Ragged batch: device cu_seqlens (int32, B+1) plus the host-side lengths."""

    def __init__(self, cu_q, cu_kv, seqlens_q: Sequence[int], seqlens_kv: Sequence[int]):
        self.cu_q, self.cu_kv = cu_q, cu_kv
        self.c = _Batch(len(seqlens_q), _ptr(cu_q), _ptr(cu_kv), max(seqlens_q) if seqlens_q else 0,
                        max(seqlens_kv) if seqlens_kv else 0, int(sum(seqlens_q)), int(sum(seqlens_kv)))

    @property
    def total_q(self):
        return int(self.c.total_q)

    @property
    def max_kv(self):
        return int(self.c.max_seqlen_kv)


def _idx_dtype(t):
    import torch
    if t.dtype in (torch.uint8, torch.float8_e4m3fn):
        return DTYPE_E4M3
    if t.dtype == torch.float32:
        return DTYPE_F32
    raise ValueError(f"unsupported indexer dtype {t.dtype}")


class Indexer:
    """Lightning-indexer inputs: q [T, H_I, d] and k [S, d] as e4m3 codes (uint8
    or float8_e4m3fn) or fp32; optional fp32 per-row scales; w [T, H_I] fp32."""

    def __init__(self, q, k, w, q_scale=None, k_scale=None):
        self.keep = (q, k, w, q_scale, k_scale)
        self.c = _Indexer(q.shape[1], q.shape[2], _idx_dtype(q), _ptr(q), _ptr(q_scale), _ptr(k),
                          _ptr(k_scale), _ptr(w))


class Mla:
    """Sparse MLA inputs: q [T, H, d_qk], kv [S, d_qk] (bf16 or fp32), value =
    first d_v columns of each kv row, scores scaled by `scale`."""

    def __init__(self, q, kv, scale: float, d_v: int):
        import torch
        dt = {torch.bfloat16: DTYPE_BF16, torch.float32: DTYPE_F32}.get(q.dtype)
        if dt is None:
            raise ValueError(f"unsupported MLA dtype {q.dtype}")
        self.keep = (q, kv)
        self.c = _Mla(q.shape[1], q.shape[2], d_v, float(scale), dt, _ptr(q), _ptr(kv))


def _ref(x):
    return None if x is None else ctypes.byref(x.c)


def workspace_size(batch: Batch, indexer: Optional[Indexer], mla: Optional[Mla], k: int):
    mn, pref = ctypes.c_size_t(0), ctypes.c_size_t(0)
    _check(lib().dsa_workspace_size(_ref(batch), _ref(indexer), _ref(mla), int(k), ctypes.byref(mn),
                                   ctypes.byref(pref)), "dsa_workspace_size")
    return int(mn.value), int(pref.value)


def index_scores(batch: Batch, indexer: Indexer, scores, ld: int, stream=None):
    _check(lib().dsa_index_scores(_ref(batch), _ref(indexer), _ptr(scores), int(ld), _stream(stream)),
           "dsa_index_scores")


def topk(batch: Batch, scores, ld: int, k: int, idx, vals=None, stream=None):
    _check(lib().dsa_topk(_ref(batch), _ptr(scores), int(ld), int(k), _ptr(idx), _ptr(vals),
                         _stream(stream)), "dsa_topk")


def index_scores_hist(batch: Batch, indexer: Indexer, scores, ld: int, hist, stream=None):
    """dsa_index_scores plus each row's first-digit histogram (hist: int32 or
    uint32 [total_q, 2048], cleared by the call)."""
    _check(lib().dsa_index_scores_hist(_ref(batch), _ref(indexer), _ptr(scores), int(ld), _ptr(hist),
                                       _stream(stream)), "dsa_index_scores_hist")


def topk_hist(batch: Batch, scores, ld: int, hist, k: int, idx, vals=None, stream=None):
    """dsa_topk taking the rows' first-digit histograms from index_scores_hist."""
    _check(lib().dsa_topk_hist(_ref(batch), _ptr(scores), int(ld), _ptr(hist), int(k), _ptr(idx), _ptr(vals),
                               _stream(stream)), "dsa_topk_hist")


def sparse_mla(batch: Batch, mla: Mla, idx, k: int, out, lse=None, ws=None, stream=None):
    nbytes = 0 if ws is None else ws.numel() * ws.element_size()
    _check(lib().dsa_sparse_mla(_ref(batch), _ref(mla), _ptr(idx), int(k), _ptr(out), _ptr(lse), _ptr(ws),
                               nbytes, _stream(stream)), "dsa_sparse_mla")


def sparse_mla_noalloc(batch: Batch, mla: Mla, idx, k: int, out, lse=None, stream=None):
    """dsa_sparse_mla without a workspace argument, for callers that cannot
    allocate device scratch: its split-KV partials live in a fixed 24 MiB array
    inside the library (shared by all calls; overlapping calls race).  Batches
    whose preferred split would need more take fewer splits."""
    _check(lib().dsa_sparse_mla_noalloc(_ref(batch), _ref(mla), _ptr(idx), int(k), _ptr(out), _ptr(lse),
                                        _stream(stream)), "dsa_sparse_mla_noalloc")


class Trace:
    """Launch trace: cudaEvents recorded around every kernel of a forward call."""

    def __init__(self, capacity: int = 512):
        import torch
        self.events = [torch.cuda.Event(enable_timing=True) for _ in range(capacity)]
        for e in self.events:   # torch creates the CUDA event on first record
            e.record()
        torch.cuda.current_stream().synchronize()
        self._ev = (ctypes.c_void_p * capacity)(*[e.cuda_event for e in self.events])
        self._ids = (ctypes.c_int32 * capacity)()
        self.c = _Trace(capacity, 0, ctypes.cast(self._ev, ctypes.POINTER(ctypes.c_void_p)),
                        ctypes.cast(self._ids, ctypes.POINTER(ctypes.c_int32)))

    def reset(self):
        self.c.count = 0

    def launches(self):
        """[(kernel name, milliseconds)] for the recorded launches (synchronises)."""
        n = int(self.c.count)
        if n:
            self.events[n - 1].synchronize()
        return [(KERNEL_NAMES.get(int(self._ids[i]), "?"), self.events[i].elapsed_time(self.events[i + 1]))
                for i in range(n - 1)]


def dense_mla_workspace_size(batch: Batch, mla: Mla) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().dsa_dense_mla_workspace_size(_ref(batch), _ref(mla), ctypes.byref(n)),
           "dsa_dense_mla_workspace_size")
    return int(n.value)


def dense_mla(batch: Batch, mla: Mla, out, lse=None, ws=None, stream=None):
    """Dense causal MLA-MQA attention over every candidate (dsa_dense_mla): the
    baseline for the sparse path."""
    nbytes = 0 if ws is None else ws.numel() * ws.element_size()
    _check(lib().dsa_dense_mla(_ref(batch), _ref(mla), _ptr(out), _ptr(lse), _ptr(ws), nbytes, _stream(stream)),
           "dsa_dense_mla")


def quantize_e4m3(x, codes, scales, group_elems: int, stream=None):
    """Per-group absmax e4m3 quantisation (dsa_quantize_e4m3): x (float32 or
    bfloat16 CUDA tensor) is read as groups of `group_elems` consecutive
    values; codes (uint8, x.numel() elements) and scales (float32, one per
    group) may be views into a larger cache."""
    import torch
    dt = {torch.float32: DTYPE_F32, torch.bfloat16: DTYPE_BF16}.get(x.dtype)
    if dt is None:
        raise ValueError("quantize_e4m3: x must be float32 or bfloat16")
    if x.numel() % group_elems:
        raise ValueError("quantize_e4m3: x.numel() must be a multiple of group_elems")
    _check(lib().dsa_quantize_e4m3(_ptr(x), dt, x.numel() // group_elems, int(group_elems), _ptr(codes),
                                   _ptr(scales), _stream(stream)), "dsa_quantize_e4m3")


def forward(batch: Batch, indexer: Indexer, mla: Mla, k: int, out, lse=None, idx_out=None, ws=None,
            stream=None, trace: Optional[Trace] = None):
    nbytes = 0 if ws is None else ws.numel() * ws.element_size()
    if trace is None:
        st = lib().dsa_forward(_ref(batch), _ref(indexer), _ref(mla), int(k), _ptr(out), _ptr(lse),
                              _ptr(idx_out), _ptr(ws), nbytes, _stream(stream))
    else:
        st = lib().dsa_forward_traced(_ref(batch), _ref(indexer), _ref(mla), int(k), _ptr(out), _ptr(lse),
                                     _ptr(idx_out), _ptr(ws), nbytes, _stream(stream), ctypes.byref(trace.c))
    _check(st, "dsa_forward")


def indexer_loss_workspace_size(batch: Batch, indexer: Indexer, mla: Mla):
    mn, pref = ctypes.c_size_t(0), ctypes.c_size_t(0)
    _check(lib().dsa_indexer_loss_workspace_size(_ref(batch), _ref(indexer), _ref(mla), ctypes.byref(mn),
                                                 ctypes.byref(pref)), "dsa_indexer_loss_workspace_size")
    return int(mn.value), int(pref.value)


def indexer_warmup_loss(batch: Batch, indexer: Indexer, mla: Mla, loss_rows, dq, dk, dw, ws, stream=None):
    """The indexer's dense warm-up loss per query row and its gradients with
    respect to the real-valued indexer q, k and the head weights w
    (dsa_indexer_warmup_loss); every output is fp32 and overwritten."""
    nbytes = 0 if ws is None else ws.numel() * ws.element_size()
    _check(lib().dsa_indexer_warmup_loss(_ref(batch), _ref(indexer), _ref(mla), _ptr(loss_rows), _ptr(dq), _ptr(dk),
                                         _ptr(dw), _ptr(ws), nbytes, _stream(stream)), "dsa_indexer_warmup_loss")


def _host_ptr(t) -> Optional[int]:
    if t is None:
        return None
    if t.is_cuda:
        raise ValueError("host inputs and outputs of forward_streamed must live in host memory")
    if not t.is_contiguous():
        raise ValueError("tensors passed to libdsa must be contiguous")
    return t.data_ptr()


class HostInputs:
    """Host copies (ideally pinned) of an Indexer's and an Mla's tensors, in
    the same shapes and dtypes, for forward_streamed."""

    def __init__(self, idx_q, idx_k, idx_w, mla_q, mla_kv, idx_q_scale=None, idx_k_scale=None):
        self.keep = (idx_q, idx_q_scale, idx_k, idx_k_scale, idx_w, mla_q, mla_kv)
        self.c = _HostInputs(_host_ptr(idx_q), _host_ptr(idx_q_scale), _host_ptr(idx_k), _host_ptr(idx_k_scale),
                             _host_ptr(idx_w), _host_ptr(mla_q), _host_ptr(mla_kv))


def forward_streamed(batch: Batch, indexer: Indexer, mla: Mla, k: int, host: HostInputs, out, lse,
                     host_out, host_lse=None, ws=None, stream=None, copy_in=None, copy_out=None):
    """dsa_forward_streamed: inputs copied from host memory chunk by chunk
    while earlier chunks compute, results copied back to host_out / host_lse.
    The device tensors of `indexer` / `mla`, `out` and `lse` receive the
    copies and results; copy_in / copy_out default to `stream`."""
    nbytes = 0 if ws is None else ws.numel() * ws.element_size()
    s = _stream(stream)
    st = lib().dsa_forward_streamed(_ref(batch), _ref(indexer), _ref(mla), int(k), _ref(host), _ptr(out),
                                    _ptr(lse), _host_ptr(host_out), _host_ptr(host_lse), _ptr(ws), nbytes, s,
                                    s if copy_in is None else _stream(copy_in),
                                    s if copy_out is None else _stream(copy_out))
    _check(st, "dsa_forward_streamed")


def read_device_errors(stream=None) -> int:
    """Synchronise the stream, read and clear the device error word.  Returns
    the DEVERR_* bits; raises DSAError when any is set."""
    flags = ctypes.c_uint32(0)
    st = lib().dsa_read_device_errors(_stream(stream), ctypes.byref(flags))
    if st not in (SUCCESS, ERROR_TIMEOUT, ERROR_BAD_INDEX):
        _check(st, "dsa_read_device_errors")
    return int(flags.value)


def debug_inject_fault(mode: int):
    """Test hook: the next tensor-core indexer launch runs in fault mode `mode`."""
    lib().dsa_debug_inject_fault(int(mode))
