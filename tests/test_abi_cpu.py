"""Host-side checks of the C ABI that need no GPU: the library builds, loads,
exports every function include/mla_decode.h declares, and rejects bad
arguments before touching the device."""
import ctypes
import os
import re

import pytest

import paged_mla_decode_09_gb300 as mla
from paged_mla_decode_09_gb300.build import build_library

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build_library()
    return mla.load_library()


def declared_functions():
    names = set()
    for fname in os.listdir(os.path.join(ROOT, "include")):
        if not fname.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", fname)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names |= set(re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(mla_\w+)\s*\(", text, flags=re.M))
    return sorted(names)


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("mla_decode", "mla_decode_workspace_size", "mla_query_status", "mla_gather_rows"):
        assert n in names
    assert set(names) == set(mla.ENTRY_POINTS)


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_exported_symbols_with_nm(lib):
    import shutil
    import subprocess

    nm = shutil.which("nm")
    if nm is None:
        pytest.skip("nm not available")
    out = subprocess.run([nm, "-D", "--defined-only", mla.LIB_PATH], capture_output=True, text=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    for name in declared_functions():
        assert name in exported, name


def test_status_strings(lib):
    assert lib.mla_status_string(0) == b"ok"
    assert lib.mla_status_string(-4) == b"workspace too small"
    assert lib.mla_status_string(12345) == b"unknown status"


def _dims(**kw):
    d = dict(batch=2, num_heads=16, q_len=1, page_size=64, num_pages=16, max_pages_per_req=5,
             page_table_stride=5, kv_dtype=0)
    d.update(kw)
    return mla.MlaDims(**d)


P = ctypes.c_void_p(256)


@pytest.mark.parametrize("bad", [
    dict(batch=0), dict(num_heads=0), dict(q_len=0), dict(num_pages=0), dict(max_pages_per_req=0),
    dict(page_table_stride=4),
])
def test_invalid_dims_rejected_without_device(lib, bad):
    d = _dims(**bad)
    assert lib.mla_decode_workspace_size(ctypes.byref(d), 0) == 0
    rc = lib.mla_decode(ctypes.byref(d), P, P, P, P, P, d.q_len, 1.0, 1.0, P, P, P, 1 << 30, None)
    assert rc == -1


@pytest.mark.parametrize("bad", [dict(page_size=32), dict(kv_dtype=7), dict(num_heads=129, q_len=2)])
def test_unsupported_dims(lib, bad):
    d = _dims(**bad)
    rc = lib.mla_decode(ctypes.byref(d), P, P, P, P, P, d.q_len, 1.0, 1.0, P, P, P, 1 << 30, None)
    assert rc == -2


def test_null_and_misaligned_pointers(lib):
    d = _dims()
    assert lib.mla_decode(ctypes.byref(d), None, P, P, P, P, 1, 1.0, 1.0, P, P, P, 1 << 30, None) == -1
    assert lib.mla_decode(ctypes.byref(d), P, P, P, P, P, 2, 1.0, 1.0, P, P, P, 1 << 30, None) == -1  # q_len
    M = ctypes.c_void_p(264)  # 8-byte aligned only
    assert lib.mla_decode(ctypes.byref(d), M, P, P, P, P, 1, 1.0, 1.0, P, P, P, 1 << 30, None) == -3
    W = ctypes.c_void_p(256 + 128)  # workspace must be 256-aligned
    assert lib.mla_decode(ctypes.byref(d), P, P, P, P, P, 1, 1.0, 1.0, P, P, W, 1 << 30, None) == -3


@pytest.mark.parametrize("scale,kv_scale,dtype", [(0.0, 1.0, 0), (-1.0, 1.0, 0), (float("nan"), 1.0, 0),
                                                   (float("inf"), 1.0, 0), (0.1, 0.0, 1), (0.1, float("nan"), 1)])
def test_scales_must_be_positive_and_finite(lib, scale, kv_scale, dtype):
    d = _dims(kv_dtype=dtype)
    assert lib.mla_decode(ctypes.byref(d), P, P, P, P, P, 1, scale, kv_scale, P, P, P, 1 << 30, None) == -1
    assert lib.mla_decode_noalloc(ctypes.byref(d), P, P, P, P, P, 1, scale, kv_scale, P, P, None, None) == -1


def test_profiled_entry_needs_four_events(lib):
    d = _dims()
    ev = (ctypes.c_void_p * 4)(None, None, None, None)
    rc = lib.mla_decode_profiled(ctypes.byref(d), P, P, P, P, P, 1, 1.0, 1.0, P, P, P, 1 << 30, None, ev)
    assert rc == -1


def test_selftest_rejects_bad_limits(lib):
    assert lib.mla_selftest_wait_timeout(None, 10, None) == -1
    assert lib.mla_selftest_wait_timeout(P, 0, None) == -1
    assert lib.mla_selftest_wait_timeout(P, 10**8, None) == -1


def test_binding_refuses_cpu_tensors(lib):
    torch = pytest.importorskip("torch")
    t = torch.zeros(2, 1, 16, 512, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        mla.mla_decode(t, t, t, t, t, 1, 1.0, 1.0, t, t, t)


def _pack_dims(**kw):
    d = dict(batch=2, num_new=2, num_pages=16, max_pages_per_req=5, page_table_stride=5, kv_dtype=1)
    d.update(kw)
    return mla.MlaKvPackDims(**d)


@pytest.mark.parametrize("bad", [dict(batch=0), dict(num_new=0), dict(num_pages=0), dict(max_pages_per_req=0),
                                 dict(page_table_stride=4)])
def test_kv_pack_invalid_dims_rejected_without_device(lib, bad):
    d = _pack_dims(**bad)
    assert lib.mla_kv_pack(ctypes.byref(d), P, P, P, 1.0, P, P, None) == -1


def test_kv_pack_checks_type_scale_and_pointers(lib):
    assert lib.mla_kv_pack(ctypes.byref(_pack_dims(kv_dtype=5)), P, P, P, 1.0, P, P, None) == -2
    for s in (0.0, -1.0, float("nan"), float("inf")):
        assert lib.mla_kv_pack(ctypes.byref(_pack_dims()), P, P, P, s, P, P, None) == -1
    # a bf16 cache ignores kv_scale: only the pointer checks remain, and a
    # misaligned row buffer is refused before the device is touched
    M = ctypes.c_void_p(264)
    assert lib.mla_kv_pack(ctypes.byref(_pack_dims(kv_dtype=0)), M, P, P, 0.0, P, P, None) == -3
    assert lib.mla_kv_pack(ctypes.byref(_pack_dims()), P, P, P, 1.0, M, P, None) == -3
    assert lib.mla_kv_pack(ctypes.byref(_pack_dims()), P, P, P, 1.0, P, None, None) == -1
    assert lib.mla_kv_pack(None, P, P, P, 1.0, P, P, None) == -1


def test_kv_pack_binding_refuses_cpu_tensors(lib):
    torch = pytest.importorskip("torch")
    rows = torch.zeros(2, 1, 576, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        mla.mla_kv_pack(rows, rows, rows, 1.0, rows, rows)


def test_sparse_and_cascade_sizes_reject_bad_arguments(lib):
    d = _dims()
    assert lib.mla_decode_sparse_workspace_size(ctypes.byref(d), 0, 0) == 0      # top-k < 1
    assert lib.mla_decode_sparse_workspace_size(ctypes.byref(d), 70000, 0) == 0  # top-k too large
    assert lib.mla_decode_cascade_workspace_size(ctypes.byref(d), 0, 0) == 0     # no prefix
    assert lib.mla_decode_cascade_workspace_size(ctypes.byref(d), 5, 0) == 0     # prefix = whole table
    assert lib.mla_decode_cascade_workspace_size(ctypes.byref(_dims(num_heads=129, q_len=2)), 2, 0) == 0


def test_sparse_and_cascade_reject_before_the_device(lib):
    d = _dims()
    args = (P, P, P, P, P)
    assert lib.mla_decode_sparse(ctypes.byref(d), *args, None, 8, 1, 1.0, 1.0, P, P, P, 1 << 30, None) == -1
    assert lib.mla_decode_sparse(ctypes.byref(d), *args, P, 0, 1, 1.0, 1.0, P, P, P, 1 << 30, None) == -1
    assert lib.mla_decode_sparse(ctypes.byref(d), *args, P, 8, 2, 1.0, 1.0, P, P, P, 1 << 30, None) == -1  # q_len
    assert lib.mla_decode_sparse(ctypes.byref(_dims(page_size=32)), *args, P, 8, 1, 1.0, 1.0, P, P, P, 1 << 30,
                                 None) == -2
    M = ctypes.c_void_p(258)
    assert lib.mla_decode_sparse(ctypes.byref(d), *args, M, 8, 1, 1.0, 1.0, P, P, P, 1 << 30, None) == -3
    assert lib.mla_decode_cascade(ctypes.byref(d), *args, 2, 1, 1.0, 1.0, P, P, None, 1 << 30, None) == -1
    assert lib.mla_decode_cascade(ctypes.byref(d), *args, 2, 3, 1.0, 1.0, P, P, P, 1 << 30, None) == -1  # q_len
    W = ctypes.c_void_p(256 + 64)
    assert lib.mla_decode_cascade(ctypes.byref(d), *args, 2, 1, 1.0, 1.0, P, P, W, 1 << 30, None) == -3
