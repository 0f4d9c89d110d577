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
    big = _dims(batch=70000)  # more (request, draft) pairs than the gather grid holds
    assert lib.mla_decode_sparse(ctypes.byref(big), *args, P, 8, 1, 1.0, 1.0, P, P, P, 1 << 30, None) == -2
    assert lib.mla_decode_sparse_workspace_size(ctypes.byref(big), 8, 0) == 0
    assert lib.mla_decode_cascade(ctypes.byref(d), *args, 2, 1, 1.0, 1.0, P, P, None, 1 << 30, None) == -1
    assert lib.mla_decode_cascade(ctypes.byref(d), *args, 2, 3, 1.0, 1.0, P, P, P, 1 << 30, None) == -1  # q_len
    W = ctypes.c_void_p(256 + 64)
    assert lib.mla_decode_cascade(ctypes.byref(d), *args, 2, 1, 1.0, 1.0, P, P, W, 1 << 30, None) == -3


# ---- the binding's layout checks (run on CPU tensors: the checks look only
# at shapes, element types and strides; the CUDA check comes before them) ----

def _decode_tensors(kv_dtype="bf16", Q=2):
    torch = pytest.importorskip("torch")
    from paged_mla_decode_09_gb300 import workloads as W
    from paged_mla_decode_09_gb300.device_inputs import to_device

    wl = W.custom([100, 70], num_heads=16, q_len=Q, kv_dtype=kv_dtype, seed=3)
    db = to_device(wl, "cpu")
    B, H = wl.batch, wl.num_heads
    t = dict(q_nope=db.q_nope, q_pe=db.q_pe, kv_cache=db.kv_cache, page_table=db.page_table, seq_lens=db.seq_lens,
             out=torch.empty(B, Q, H, 512, dtype=torch.bfloat16), lse=torch.empty(B, Q, H, dtype=torch.float32),
             workspace=torch.empty(4096, dtype=torch.uint8))
    return torch, wl, t


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8_e4m3"])
def test_layout_checks_accept_what_the_tests_pass(kv_dtype):
    torch, wl, t = _decode_tensors(kv_dtype)
    mla._check_decode_tensors(**t)
    # a page table that is a column slice of a wider one keeps unit column stride
    wide = torch.full((wl.batch, wl.max_pages + 3), -1, dtype=torch.int32)
    wide[:, :wl.max_pages] = t["page_table"]
    mla._check_decode_tensors(**{**t, "page_table": wide[:, :wl.max_pages]})
    idx = torch.from_numpy(__import__("paged_mla_decode_09_gb300.workloads", fromlist=["x"]).topk_indices(wl, 8, 1))
    mla._check_indices(idx, t["q_nope"])


def _bad_variants(torch, t):
    B, Q, H, _ = t["q_nope"].shape
    yield "q_nope", t["q_nope"][:1].expand(B, Q, H, 512)          # broadcast view: smaller storage
    yield "q_nope", t["q_nope"].float()
    yield "q_pe", t["q_pe"][..., :32]
    yield "out", torch.empty(B, Q, 512, H, dtype=torch.bfloat16).transpose(2, 3)
    yield "lse", torch.empty(B, Q, H, dtype=torch.bfloat16)
    yield "seq_lens", t["seq_lens"].long()
    yield "page_table", t["page_table"].long()
    yield "page_table", t["page_table"].t().contiguous().t()       # column-major
    yield "page_table", t["page_table"][:1]
    yield "kv_cache", t["kv_cache"][..., :512]
    yield "kv_cache", t["kv_cache"].float() if t["kv_cache"].dtype == torch.bfloat16 else t["kv_cache"].short()
    yield "workspace", torch.empty(64, 2, dtype=torch.uint8).t()


@pytest.mark.parametrize("case", range(12))
def test_layout_checks_reject_mismatched_tensors(case):
    torch, wl, t = _decode_tensors()
    name, bad = list(_bad_variants(torch, t))[case]
    with pytest.raises((ValueError, TypeError)):
        mla._check_decode_tensors(**{**t, name: bad})


def test_index_and_cache_write_layout_checks():
    torch, wl, t = _decode_tensors()
    good = torch.zeros(wl.batch, wl.q_len, 8, dtype=torch.int32)
    mla._check_indices(good, t["q_nope"])
    for bad in (good.long(), good[:1], good.transpose(1, 2).contiguous().transpose(1, 2), good[..., None]):
        with pytest.raises(ValueError):
            mla._check_indices(bad, t["q_nope"])
    # the cache write, with the tensors its tests build
    rows = torch.zeros(wl.batch, 2, 576, dtype=torch.bfloat16)
    cache = torch.zeros(8, 64, 576, dtype=torch.uint8)
    status = torch.zeros(1, dtype=torch.int32)
    mla._check_kv_pack_tensors(rows, t["page_table"], t["seq_lens"], cache, status)
    for args in ((rows.view(torch.int16), t["page_table"], t["seq_lens"], cache, status),
                 (rows, t["page_table"], t["seq_lens"], cache, status.long()),
                 (rows, t["page_table"].long(), t["seq_lens"], cache, status),
                 (rows[:, :, :512], t["page_table"], t["seq_lens"], cache, status)):
        with pytest.raises(ValueError):
            mla._check_kv_pack_tensors(*args)


def test_binding_constants_match_the_headers():
    """Every MLA_* constant the binding defines has the value the C headers
    give it (status codes, device status bits, cache types)."""
    vals = {}
    for fname in os.listdir(os.path.join(ROOT, "include")):
        if fname.endswith(".h"):
            text = re.sub(r"/\*.*?\*/", "", open(os.path.join(ROOT, "include", fname)).read(), flags=re.S)
            for name, v in re.findall(r"\b(MLA_[A-Z0-9_]+)\s*=\s*(-?\d+)", text):
                vals[name] = int(v)
    mine = {k: getattr(mla, k) for k in dir(mla) if re.fullmatch(r"MLA_[A-Z0-9_]+", k) and isinstance(getattr(mla, k), int)}
    assert mine, "the binding defines no constants"
    for k, v in mine.items():
        assert k in vals, f"{k} is not declared in include/"
        assert vals[k] == v, f"{k}: binding {v}, header {vals[k]}"
    # the device status bits are distinct powers of two
    bits = [v for k, v in vals.items() if k.startswith("MLA_DEV_")]
    assert len(set(bits)) == len(bits) and all(b > 0 and b & (b - 1) == 0 for b in bits)


@pytest.mark.parametrize("bad", [
    dict(max_pages_per_req=1 << 25, page_table_stride=1 << 25),  # token positions of a request overflow int32
    dict(batch=1 << 12, max_pages_per_req=1 << 20, page_table_stride=1 << 20),  # the schedule's page sums
])
def test_int32_overflowing_dims_are_unsupported(lib, bad):
    d = _dims(**bad)
    assert lib.mla_decode_workspace_size(ctypes.byref(d), 0) == 0
    rc = lib.mla_decode(ctypes.byref(d), P, P, P, P, P, d.q_len, 1.0, 1.0, P, P, P, 1 << 30, None)
    assert rc == -2
    assert lib.mla_decode_noalloc(ctypes.byref(d), P, P, P, P, P, d.q_len, 1.0, 1.0, P, P, None, None) == -2


def test_gather_rows_refuses_batches_beyond_the_grid(lib):
    d = _dims(batch=65536, num_pages=1 << 20)
    R = ctypes.c_void_p(1 << 20)
    assert lib.mla_gather_rows(ctypes.byref(d), P, P, P, R, P, P, None) == -2
