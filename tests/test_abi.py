"""The C-ABI library loads, exports every function include/dsa.h declares, and
rejects bad arguments on the host before touching a device.  CPU only: no
compute call runs here."""

import ctypes
import subprocess

import pytest

import sparse_long_context_07_b300 as dsa


def test_library_exports_every_header_function():
    names = dsa.header_functions()
    assert "dsa_forward" in names and "dsa_index_scores" in names and "dsa_topk" in names
    assert "dsa_sparse_mla" in names and "dsa_workspace_size" in names
    out = subprocess.run(["nm", "-D", "--defined-only", dsa.LIB_PATH], capture_output=True, text=True,
                         check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    missing = [n for n in names if n not in exported]
    assert not missing, missing


def test_abi_version_and_status_strings():
    assert dsa.abi_version() == 1
    for code in range(8):
        assert dsa.status_string(code) and dsa.status_string(code) != "unknown status"
    assert dsa.status_string(99) == "unknown status"


FAKE = 0x10000  # an aligned fake device address: never dereferenced (validation fails first)


def _batch(num_seqs=1, tq=8, tkv=8, mq=8, mkv=8, cu=FAKE):
    return dsa._Batch(num_seqs, cu, cu, mq, mkv, tq, tkv)


def _indexer(dtype=dsa.DTYPE_E4M3, heads=64, dim=128, q=FAKE, k=FAKE, w=FAKE):
    return dsa._Indexer(heads, dim, dtype, q, None, k, None, w)


def _mla(dtype=dsa.DTYPE_BF16, heads=128, dqk=576, dv=512, q=FAKE, kv=FAKE, scale=0.07):
    return dsa._Mla(heads, dqk, dv, scale, dtype, q, kv)


def _index_scores(b, ix, scores=FAKE, ld=8):
    return dsa.lib().dsa_index_scores(ctypes.byref(b) if b is not None else None,
                                      ctypes.byref(ix) if ix is not None else None, scores, ld, None)


@pytest.mark.parametrize("case,expect", [
    (dict(b=None), dsa.ERROR_INVALID_VALUE),
    (dict(b=_batch(num_seqs=0)), dsa.ERROR_INVALID_VALUE),
    (dict(b=_batch(cu=0)), dsa.ERROR_INVALID_VALUE),
    (dict(b=_batch(tq=9, tkv=8)), dsa.ERROR_INVALID_VALUE),
    (dict(b=_batch(mq=9, mkv=8)), dsa.ERROR_INVALID_VALUE),
    (dict(ix=None), dsa.ERROR_INVALID_VALUE),
    (dict(ix=_indexer(q=FAKE + 4)), dsa.ERROR_INVALID_VALUE),        # misaligned
    (dict(ix=_indexer(dtype=dsa.DTYPE_BF16)), dsa.ERROR_NOT_SUPPORTED),
    (dict(ix=_indexer(heads=65)), dsa.ERROR_NOT_SUPPORTED),
    (dict(ix=_indexer(dim=136)), dsa.ERROR_NOT_SUPPORTED),
    (dict(scores=FAKE + 8), dsa.ERROR_INVALID_VALUE),
    (dict(ld=6), dsa.ERROR_INVALID_VALUE),                             # < max_seqlen_kv
    (dict(ld=10), dsa.ERROR_INVALID_VALUE),                            # not a multiple of 4
])
def test_index_scores_rejects_bad_arguments(case, expect):
    args = dict(b=_batch(), ix=_indexer(), scores=FAKE, ld=8)
    args.update(case)
    assert _index_scores(**args) == expect
    assert dsa.lib().dsa_last_error_message().decode()


def test_topk_rejects_bad_k():
    b = _batch()
    for k in (0, -1, 16385):
        assert dsa.lib().dsa_topk(ctypes.byref(b), FAKE, 8, k, FAKE, None, None) == dsa.ERROR_INVALID_VALUE


def test_sparse_mla_rejects_bad_arguments():
    b = _batch()
    lib = dsa.lib()
    assert lib.dsa_sparse_mla(ctypes.byref(b), ctypes.byref(_mla(dv=600)), FAKE, 16, FAKE, None, None, 0,
                              None) == dsa.ERROR_NOT_SUPPORTED
    assert lib.dsa_sparse_mla(ctypes.byref(b), ctypes.byref(_mla(dtype=dsa.DTYPE_E4M3)), FAKE, 16, FAKE, None,
                              None, 0, None) == dsa.ERROR_NOT_SUPPORTED
    assert lib.dsa_sparse_mla(ctypes.byref(b), ctypes.byref(_mla(kv=FAKE + 2)), FAKE, 16, FAKE, None, None, 0,
                              None) == dsa.ERROR_INVALID_VALUE
    assert lib.dsa_sparse_mla(ctypes.byref(b), ctypes.byref(_mla(scale=float("inf"))), FAKE, 16, FAKE, None,
                              None, 0, None) == dsa.ERROR_INVALID_VALUE


def test_workspace_size_is_host_only_and_monotone():
    lib = dsa.lib()
    mn, pref = ctypes.c_size_t(0), ctypes.c_size_t(0)
    # 128K-token prefill, production dims
    b = _batch(tq=131072, tkv=131072, mq=131072, mkv=131072)
    st = lib.dsa_workspace_size(ctypes.byref(b), ctypes.byref(_indexer()), ctypes.byref(_mla()), 2048,
                                ctypes.byref(mn), ctypes.byref(pref))
    assert st == dsa.SUCCESS
    # scores chunk of >= 64 rows of 131072 fp32 plus their indices
    assert mn.value >= 64 * 131072 * 4 + 64 * 2048 * 4
    assert pref.value >= mn.value
    assert pref.value >= 16384 * 131072 * 4
    # MLA alone for a small decode batch needs split scratch; a large batch none
    small = _batch(num_seqs=4, tq=4, tkv=4 * 8192, mq=1, mkv=8192)
    assert lib.dsa_workspace_size(ctypes.byref(small), None, ctypes.byref(_mla()), 2048, ctypes.byref(mn),
                                  ctypes.byref(pref)) == dsa.SUCCESS
    assert mn.value > 0
    big = _batch(num_seqs=1, tq=4096, tkv=4096, mq=4096, mkv=4096)
    assert lib.dsa_workspace_size(ctypes.byref(big), None, ctypes.byref(_mla()), 2048, ctypes.byref(mn),
                                  ctypes.byref(pref)) == dsa.SUCCESS
    assert mn.value == 0
