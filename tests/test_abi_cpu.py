"""The C-ABI library without a GPU: it loads, exports every entry point the
header declares, and rejects bad arguments on the host before touching CUDA."""
import ctypes
import os
import re

import pytest

from block_sparse_attention_nvfp4_gb300 import _lib
from block_sparse_attention_nvfp4_gb300 import build as msa_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    msa_build.build()
    return _lib.load()


def declared():
    text = open(os.path.join(ROOT, "include", "msa.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(msa_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = declared()
    assert len(names) >= 10
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(_lib.EXPORTS) == names


def test_status_strings(lib):
    for code in (0, -1, -2, -3, -4, -5, -6):
        assert lib.msa_status_string(code)
    assert lib.msa_status_string(12345) == b"unknown status"


def _args():
    a = _lib.Args()
    a.num_reqs, a.total_rows, a.max_rows_per_req, a.num_pages, a.max_pages_per_req = 1, 1, 1, 4, 4
    a.num_kv_heads, a.q_per_kv, a.head_dim, a.block_size, a.top_k = 4, 8, 128, 128, 16
    a.sm_scale = 0.0883883
    fake = 0x10000  # never dereferenced: every call below fails validation first
    for f in ("context_lens", "q_indptr", "block_table", "q", "q_idx", "k_data", "k_scale", "v_data", "v_scale",
              "ki_data", "ki_scale"):
        setattr(a, f, fake)
    return a


@pytest.mark.parametrize("field,value,code", [
    ("head_dim", 64, -2), ("num_kv_heads", 8, -2), ("block_size", 64, -2), ("top_k", 32, -2),
    ("max_rows_per_req", 9, -1), ("max_rows_per_req", 0, -1), ("num_reqs", -1, -1), ("total_rows", 5, -1),
    ("sm_scale", 0.0, -1), ("num_pages", 0, -1), ("q", 0x10001, -1),
])
def test_host_validation_rejects_before_any_cuda_call(lib, field, value, code):
    a = _args()
    setattr(a, field, value)
    n = ctypes.c_size_t(0)
    ws_rc = lib.msa_workspace_size(ctypes.byref(a), ctypes.byref(n))
    if field == "q":
        # the workspace size depends on the batch's sizes only, not on its data pointers
        assert ws_rc != -1
    else:
        assert ws_rc == code
    rc = lib.msa_decode(ctypes.byref(a), ctypes.c_void_p(0x20000), ctypes.c_void_p(0x30000), None,
                        ctypes.c_void_p(0x40000), 1 << 20, None)
    assert rc == code


def test_null_pointer_arguments(lib):
    assert lib.msa_workspace_size(None, None) == -1
    assert lib.msa_decode(None, None, None, None, None, 0, None) == -1
    assert lib.msa_dequant_rows(None, None, 1, None, 0, None) == -1
    assert lib.msa_workspace_init(None, 0, None) == -4
    a = _args()
    assert lib.msa_decode(ctypes.byref(a), None, None, None, None, 0, None) == -1


def test_kv_insert_host_validation(lib):
    """msa_kv_insert_nvfp4 rejects bad arguments before any CUDA call."""
    A = _lib.KvInsertArgs
    f = lib.msa_kv_insert_nvfp4
    ws = ctypes.c_void_p(1 << 20)                       # never dereferenced: checks fail first
    assert f(None, ws, 256, None) == -1
    a = A(num_tokens=-1, num_pages=1)
    assert f(ctypes.byref(a), ws, 256, None) == -1
    a = A(num_tokens=4, num_pages=1)                    # no slot mapping
    assert f(ctypes.byref(a), ws, 256, None) == -1
    a = A(num_tokens=4, num_pages=1, slot_mapping=1 << 20, k=(1 << 20) + 4, k_data=1 << 21, k_scale=1 << 22)
    assert f(ctypes.byref(a), ws, 256, None) == -1       # source not 16-byte aligned
    a = A(num_tokens=4, num_pages=1, slot_mapping=1 << 20, k=1 << 20)
    assert f(ctypes.byref(a), ws, 256, None) == -1       # source without its cache
    a = A(num_tokens=4, num_pages=1, slot_mapping=1 << 20, k=1 << 20, k_data=1 << 21, k_scale=1 << 22)
    assert f(ctypes.byref(a), None, 256, None) == -4     # no workspace
    assert f(ctypes.byref(a), ws, 16, None) == -4        # workspace too small


def test_dcp_host_validation(lib):
    """The DCP entry points reject bad ranks, worlds, group ranges and pointers before any
    CUDA call."""
    a = _args()
    keys = ctypes.c_void_p(0x50000)
    ws = ctypes.c_void_p(0x40000)
    loc = lib.msa_dcp_local_topk
    for rank, world in ((0, 0), (1, 1), (-1, 2), (2, 2), (0, 9)):
        assert loc(ctypes.byref(a), rank, world, keys, ws, 1 << 20, None) == -1, (rank, world)
    assert loc(ctypes.byref(a), 0, 2, None, ws, 1 << 20, None) == -1
    assert loc(ctypes.byref(a), 0, 2, ctypes.c_void_p(0x50004), ws, 1 << 20, None) == -1  # not 8-byte aligned
    assert loc(None, 0, 2, keys, ws, 1 << 20, None) == -1
    mrg = lib.msa_dcp_merge_topk
    ids = ctypes.c_void_p(0x60000)
    for world, g0, ng in ((0, 0, 4), (9, 0, 4), (2, -1, 1), (2, 0, 0), (2, 3, 2), (2, 4, 1)):
        assert mrg(ctypes.byref(a), world, g0, ng, keys, ids, ws, 1 << 20, None) == -1, (world, g0, ng)
    assert mrg(ctypes.byref(a), 2, 0, 4, None, ids, ws, 1 << 20, None) == -1
    assert mrg(ctypes.byref(a), 2, 0, 4, keys, None, ws, 1 << 20, None) == -1
    a.head_dim = 64
    assert mrg(ctypes.byref(a), 2, 0, 4, keys, ids, ws, 1 << 20, None) == -2


def test_selftest_host_validation(lib):
    assert lib.msa_selftest_wait_timeout(None, 256, None) == -4
    assert lib.msa_selftest_wait_timeout(ctypes.c_void_p(0x40010), 256, None) == -4  # misaligned
    assert lib.msa_selftest_wait_timeout(ctypes.c_void_p(0x40000), 16, None) == -4   # too small
