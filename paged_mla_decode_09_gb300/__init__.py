"""Paged MLA decode for GB300: Python binding of the C ABI in include/mla_decode.h,
include/mla_kv_pack.h, include/mla_sparse.h and include/mla_cascade.h.

The functions here only marshal arguments (torch tensors -> device
pointers, shapes -> ``mla_dims``); every step of the decode runs in the
CUDA library.  There is no CPU fallback: if the library is missing or the
device is not sm_103a, calls raise.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

from .build import LIB_PATH, build_library

MLA_OK = 0
MLA_KV_BF16 = 0
MLA_KV_FP8_E4M3 = 1
MLA_DEV_BAD_PAGE_ID = 1
MLA_DEV_BAD_SEQ_LEN = 2
MLA_DEV_TIMEOUT = 4
MLA_DEV_INTERNAL = 8
MLA_DEV_BAD_INDEX = 16
MLA_DEV_BAD_PREFIX = 32

ENTRY_POINTS = (
    "mla_decode_workspace_size",
    "mla_decode",
    "mla_decode_profiled",
    "mla_query_status",
    "mla_gather_rows",
    "mla_selftest_wait_timeout",
    "mla_status_string",
    "mla_decode_launch_shape",
    "mla_decode_noalloc",
    "mla_kv_pack",
    "mla_decode_sparse_workspace_size",
    "mla_decode_sparse",
    "mla_decode_sparse_query_status",
    "mla_decode_cascade_workspace_size",
    "mla_decode_cascade",
    "mla_decode_cascade_query_status",
)


class MlaError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {status_string(code)} ({code})")


class MlaDims(ctypes.Structure):
    _fields_ = [
        ("batch", ctypes.c_int32),
        ("num_heads", ctypes.c_int32),
        ("q_len", ctypes.c_int32),
        ("page_size", ctypes.c_int32),
        ("num_pages", ctypes.c_int32),
        ("max_pages_per_req", ctypes.c_int32),
        ("page_table_stride", ctypes.c_int32),
        ("kv_dtype", ctypes.c_int32),
    ]


class MlaKvPackDims(ctypes.Structure):
    _fields_ = [
        ("batch", ctypes.c_int32),
        ("num_new", ctypes.c_int32),
        ("num_pages", ctypes.c_int32),
        ("max_pages_per_req", ctypes.c_int32),
        ("page_table_stride", ctypes.c_int32),
        ("kv_dtype", ctypes.c_int32),
    ]


_lib = None


def load_library(path: str | None = None, build: bool = False) -> ctypes.CDLL:
    """Load (optionally building first) the CUDA library; raises if absent."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if build:
        build_library()
    if not os.path.exists(p):
        raise RuntimeError(
            f"CUDA library {p} is missing: build it with __graft_entry__.build() or "
            "`python -m paged_mla_decode_09_gb300.build` (there is no CPU fallback)"
        )
    lib = ctypes.CDLL(p)
    P, I32, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
    D = ctypes.POINTER(MlaDims)
    lib.mla_decode_workspace_size.argtypes = [D, ctypes.c_int]
    lib.mla_decode_workspace_size.restype = SZ
    dec_args = [D, P, P, P, P, P, I32, ctypes.c_float, ctypes.c_float, P, P, P, SZ, P]
    lib.mla_decode.argtypes = dec_args
    lib.mla_decode.restype = ctypes.c_int
    lib.mla_decode_profiled.argtypes = dec_args + [ctypes.POINTER(P)]
    lib.mla_decode_profiled.restype = ctypes.c_int
    lib.mla_query_status.argtypes = [P, P, ctypes.POINTER(I32)]
    lib.mla_query_status.restype = ctypes.c_int
    lib.mla_gather_rows.argtypes = [D, P, P, P, P, P, P, P]
    lib.mla_gather_rows.restype = ctypes.c_int
    lib.mla_selftest_wait_timeout.argtypes = [P, ctypes.c_uint32, P]
    lib.mla_selftest_wait_timeout.restype = ctypes.c_int
    lib.mla_status_string.argtypes = [ctypes.c_int]
    lib.mla_status_string.restype = ctypes.c_char_p
    lib.mla_decode_launch_shape.argtypes = [D, ctypes.c_int, ctypes.POINTER(I32), ctypes.POINTER(I32)]
    lib.mla_decode_launch_shape.restype = ctypes.c_int
    lib.mla_decode_noalloc.argtypes = [D, P, P, P, P, P, I32, ctypes.c_float, ctypes.c_float, P, P, P, P]
    lib.mla_decode_noalloc.restype = ctypes.c_int
    lib.mla_kv_pack.argtypes = [ctypes.POINTER(MlaKvPackDims), P, P, P, ctypes.c_float, P, P, P]
    lib.mla_kv_pack.restype = ctypes.c_int
    lib.mla_decode_sparse_workspace_size.argtypes = [D, I32, ctypes.c_int]
    lib.mla_decode_sparse_workspace_size.restype = SZ
    lib.mla_decode_sparse.argtypes = [D, P, P, P, P, P, P, I32, I32, ctypes.c_float, ctypes.c_float, P, P, P, SZ, P]
    lib.mla_decode_sparse.restype = ctypes.c_int
    lib.mla_decode_sparse_query_status.argtypes = [D, I32, P, P, ctypes.POINTER(I32)]
    lib.mla_decode_sparse_query_status.restype = ctypes.c_int
    lib.mla_decode_cascade_workspace_size.argtypes = [D, I32, ctypes.c_int]
    lib.mla_decode_cascade_workspace_size.restype = SZ
    lib.mla_decode_cascade.argtypes = [D, P, P, P, P, P, I32, I32, ctypes.c_float, ctypes.c_float, P, P, P, SZ, P]
    lib.mla_decode_cascade.restype = ctypes.c_int
    lib.mla_decode_cascade_query_status.argtypes = [D, I32, P, P, ctypes.POINTER(I32)]
    lib.mla_decode_cascade_query_status.restype = ctypes.c_int
    if path is None:
        _lib = lib
    return lib


def status_string(code: int) -> str:
    try:
        return load_library().mla_status_string(int(code)).decode()
    except RuntimeError:
        return "library not loaded"


def _ptr(t) -> ctypes.c_void_p:
    return ctypes.c_void_p(t.data_ptr())


def _stream_handle(stream):
    import torch

    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def kv_dtype_code(kv_cache) -> int:
    import torch

    if kv_cache.dtype == torch.bfloat16:
        return MLA_KV_BF16
    if kv_cache.dtype in (torch.uint8, torch.float8_e4m3fn):
        return MLA_KV_FP8_E4M3
    raise TypeError(f"unsupported cache dtype {kv_cache.dtype}")


def make_dims(q_nope, kv_cache, page_table) -> MlaDims:
    B, Q, H, _ = q_nope.shape
    return MlaDims(
        batch=B,
        num_heads=H,
        q_len=Q,
        page_size=int(kv_cache.shape[1]),
        num_pages=int(kv_cache.shape[0]),
        max_pages_per_req=int(page_table.shape[1]),
        page_table_stride=int(page_table.stride(0)),
        kv_dtype=kv_dtype_code(kv_cache),
    )


def mla_decode_workspace_size(dims: MlaDims, device: int | None = None) -> int:
    import torch

    dev = torch.cuda.current_device() if device is None else device
    n = load_library().mla_decode_workspace_size(ctypes.byref(dims), dev)
    if n == 0:
        raise MlaError(-1, "mla_decode_workspace_size")
    return int(n)


def mla_decode_launch_shape(dims: MlaDims, device: int | None = None):
    import torch

    dev = torch.cuda.current_device() if device is None else device
    c, s = ctypes.c_int32(), ctypes.c_int32()
    rc = load_library().mla_decode_launch_shape(ctypes.byref(dims), dev, ctypes.byref(c), ctypes.byref(s))
    if rc != MLA_OK:
        raise MlaError(rc, "mla_decode_launch_shape")
    return c.value, s.value


def _check_cuda(*tensors):
    for t in tensors:
        if not t.is_cuda:
            raise ValueError("all tensors must be CUDA tensors (the decode runs only on the GPU)")


def _check_layout(name, t, shape, dtypes):
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {list(shape)}, got {list(t.shape)}")
    if t.dtype not in dtypes:
        raise TypeError(f"{name} must be {' or '.join(str(d) for d in dtypes)}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _check_cache_and_table(kv_cache, page_table, seq_lens, B):
    import torch

    if kv_cache.dim() != 3 or kv_cache.shape[2] != 576 or not kv_cache.is_contiguous():
        raise ValueError("kv_cache must be a contiguous [num_pages, page_size, 576] tensor")
    kv_dtype_code(kv_cache)  # raises for other element types
    if (page_table.dtype != torch.int32 or page_table.dim() != 2 or page_table.shape[0] != B
            or page_table.stride(1) != 1 or page_table.stride(0) < page_table.shape[1]):
        raise ValueError("page_table must be an int32 [B, max_pages] tensor with unit column stride")
    _check_layout("seq_lens", seq_lens, (B,), (torch.int32,))


def _check_decode_tensors(q_nope, q_pe, kv_cache, page_table, seq_lens, out, lse, workspace):
    """The shapes, element types and layouts the C ABI assumes.  It receives
    bare pointers, so a tensor that does not match (a broadcast view, another
    dtype, a transposed copy) would be read or written with the wrong extent.
    One combined test on the fast path (it runs on every call); the detailed
    checks below name what is wrong."""
    import torch

    bf16, i32 = torch.bfloat16, torch.int32
    s = q_nope.shape
    if len(s) == 4:
        B, Q, H = s[0], s[1], s[2]
        dev = q_nope.get_device()
        if (s[3] == 512 and q_nope.dtype is bf16 and q_nope.is_contiguous()
                and q_pe.dtype is bf16 and q_pe.shape == (B, Q, H, 64) and q_pe.is_contiguous()
                and out.dtype is bf16 and out.shape == s and out.is_contiguous()
                and lse.dtype is torch.float32 and lse.shape == (B, Q, H) and lse.is_contiguous()
                and seq_lens.dtype is i32 and seq_lens.shape == (B,) and seq_lens.is_contiguous()
                and page_table.dtype is i32 and page_table.dim() == 2 and page_table.shape[0] == B
                and page_table.stride(1) == 1 and page_table.stride(0) >= page_table.shape[1]
                and kv_cache.dim() == 3 and kv_cache.shape[2] == 576 and kv_cache.is_contiguous()
                and kv_cache.dtype in (bf16, torch.uint8, torch.float8_e4m3fn) and workspace.is_contiguous()
                and q_pe.get_device() == dev and out.get_device() == dev and lse.get_device() == dev
                and seq_lens.get_device() == dev and page_table.get_device() == dev
                and kv_cache.get_device() == dev and workspace.get_device() == dev):
            return
    _explain_decode_tensors(q_nope, q_pe, kv_cache, page_table, seq_lens, out, lse, workspace)
    raise ValueError("decode tensors do not have the shapes, types and layouts the library expects")


def _explain_decode_tensors(q_nope, q_pe, kv_cache, page_table, seq_lens, out, lse, workspace):
    import torch

    if q_nope.dim() != 4 or q_nope.shape[3] != 512:
        raise ValueError(f"q_nope must be [B, q_len, H, 512], got {list(q_nope.shape)}")
    B, Q, H, _ = q_nope.shape
    _check_layout("q_nope", q_nope, (B, Q, H, 512), (torch.bfloat16,))
    _check_layout("q_pe", q_pe, (B, Q, H, 64), (torch.bfloat16,))
    _check_layout("out", out, (B, Q, H, 512), (torch.bfloat16,))
    _check_layout("lse", lse, (B, Q, H), (torch.float32,))
    _check_cache_and_table(kv_cache, page_table, seq_lens, B)
    if not workspace.is_contiguous():
        raise ValueError("workspace must be contiguous")
    for t in (q_pe, kv_cache, page_table, seq_lens, out, lse, workspace):
        if t.device != q_nope.device:
            raise ValueError("all tensors must be on one device")


def mla_decode(q_nope, q_pe, kv_cache, page_table, seq_lens, q_len, scale, kv_scale, out, lse, workspace,
               stream=None, events=None) -> None:
    """Enqueue one decode step (see include/mla_decode.h).  Raises MlaError on a host-side error.

    ``events``: optional 4 torch.cuda.Event objects (already recorded once)
    to time the schedule / attention / combine launches.
    """
    _check_cuda(q_nope, q_pe, kv_cache, page_table, seq_lens, out, lse, workspace)
    _check_decode_tensors(q_nope, q_pe, kv_cache, page_table, seq_lens, out, lse, workspace)
    if int(q_len) != q_nope.shape[1]:
        raise ValueError(f"q_len {q_len} does not match q_nope's second dimension {q_nope.shape[1]}")
    dims = make_dims(q_nope, kv_cache, page_table)
    lib = load_library()
    args = [ctypes.byref(dims), _ptr(q_nope), _ptr(q_pe), _ptr(kv_cache), _ptr(page_table), _ptr(seq_lens),
            int(q_len), float(scale), float(kv_scale), _ptr(out), _ptr(lse), _ptr(workspace),
            ctypes.c_size_t(workspace.numel() * workspace.element_size()), _stream_handle(stream)]
    if events is None:
        rc = lib.mla_decode(*args)
    else:
        arr = (ctypes.c_void_p * 4)(*[ctypes.c_void_p(e.cuda_event) for e in events])
        rc = lib.mla_decode_profiled(*args, arr)
    if rc != MLA_OK:
        raise MlaError(rc, "mla_decode")


def mla_query_status(workspace, stream=None) -> int:
    st = ctypes.c_int32(0)
    rc = load_library().mla_query_status(_ptr(workspace), _stream_handle(stream), ctypes.byref(st))
    if rc != MLA_OK:
        raise MlaError(rc, "mla_query_status")
    return st.value


def timeout_diagnostics(workspace) -> dict:
    """Words 0..3 of the workspace: status bits and, after a device timeout,
    which wait gave up (tag, page counter, cluster, rank, warp)."""
    import torch

    w = workspace[:16].view(torch.int32).cpu().tolist()
    return {"status": w[0], "wait_tag": w[1], "page_counter": w[2], "cluster": w[3] >> 16,
            "rank": (w[3] >> 8) & 0xFF, "warp": w[3] & 0xFF}


def mla_gather_rows(kv_cache, page_table, seq_lens, row_offsets, rows_out, workspace, q_len: int = 1,
                    stream=None) -> None:
    _check_cuda(kv_cache, page_table, seq_lens, row_offsets, rows_out, workspace)
    dims = MlaDims(batch=int(seq_lens.shape[0]), num_heads=1, q_len=q_len, page_size=int(kv_cache.shape[1]),
                   num_pages=int(kv_cache.shape[0]), max_pages_per_req=int(page_table.shape[1]),
                   page_table_stride=int(page_table.stride(0)), kv_dtype=kv_dtype_code(kv_cache))
    rc = load_library().mla_gather_rows(ctypes.byref(dims), _ptr(kv_cache), _ptr(page_table), _ptr(seq_lens),
                                        _ptr(row_offsets), _ptr(rows_out), _ptr(workspace), _stream_handle(stream))
    if rc != MLA_OK:
        raise MlaError(rc, "mla_gather_rows")


def mla_selftest_wait_timeout(workspace, timeout_us: int, stream=None) -> None:
    rc = load_library().mla_selftest_wait_timeout(_ptr(workspace), int(timeout_us), _stream_handle(stream))
    if rc != MLA_OK:
        raise MlaError(rc, "mla_selftest_wait_timeout")


def _check_kv_pack_tensors(rows, page_table, seq_lens, kv_cache, status):
    import torch

    if rows.dim() != 3 or rows.shape[2] != 576 or not rows.is_contiguous() or rows.dtype != torch.bfloat16:
        raise ValueError("rows must be a contiguous bf16 [B, num_new, 576] tensor")
    _check_cache_and_table(kv_cache, page_table, seq_lens, rows.shape[0])
    if status.dtype != torch.int32 or status.numel() < 1:
        raise ValueError("status must be an int32 tensor of at least one element")
    for t in (page_table, seq_lens, kv_cache, status):
        if t.device != rows.device:
            raise ValueError("all tensors must be on one device")


def mla_kv_pack(rows, page_table, seq_lens, kv_scale, kv_cache, status, stream=None) -> None:
    """Enqueue the cache write of a step's new rows (see include/mla_kv_pack.h).

    rows: bf16 [B, num_new, 576]; kv_cache: bf16 or uint8 (e4m3 codes)
    [num_pages, 64, 576]; status: int32 [1] on the device (flags OR-ed in).
    Raises MlaError on a host-side error.
    """
    _check_cuda(rows, page_table, seq_lens, kv_cache, status)
    _check_kv_pack_tensors(rows, page_table, seq_lens, kv_cache, status)
    B, N, _ = rows.shape
    dims = MlaKvPackDims(batch=B, num_new=N, num_pages=int(kv_cache.shape[0]),
                         max_pages_per_req=int(page_table.shape[1]), page_table_stride=int(page_table.stride(0)),
                         kv_dtype=kv_dtype_code(kv_cache))
    rc = load_library().mla_kv_pack(ctypes.byref(dims), _ptr(rows), _ptr(page_table), _ptr(seq_lens),
                                    float(kv_scale), _ptr(kv_cache), _ptr(status), _stream_handle(stream))
    if rc != MLA_OK:
        raise MlaError(rc, "mla_kv_pack")


def mla_decode_sparse_workspace_size(dims: MlaDims, topk: int, device: int | None = None) -> int:
    import torch

    dev = torch.cuda.current_device() if device is None else device
    n = load_library().mla_decode_sparse_workspace_size(ctypes.byref(dims), int(topk), dev)
    if n == 0:
        raise MlaError(-1, "mla_decode_sparse_workspace_size")
    return int(n)


def _check_indices(indices, q_nope):
    import torch

    if (indices.dim() != 3 or tuple(indices.shape[:2]) != tuple(q_nope.shape[:2]) or not indices.is_contiguous()
            or indices.dtype != torch.int32 or indices.device != q_nope.device):
        raise ValueError("indices must be a contiguous int32 [B, q_len, topk] tensor")


def mla_decode_sparse(q_nope, q_pe, kv_cache, page_table, seq_lens, indices, scale, kv_scale, out, lse, workspace,
                      stream=None) -> None:
    """Enqueue a top-k decode (see include/mla_sparse.h); indices: int32
    [B, q_len, topk] token positions, -1 = unused."""
    _check_cuda(q_nope, q_pe, kv_cache, page_table, seq_lens, indices, out, lse, workspace)
    _check_decode_tensors(q_nope, q_pe, kv_cache, page_table, seq_lens, out, lse, workspace)
    _check_indices(indices, q_nope)
    B, Q, topk = indices.shape
    dims = make_dims(q_nope, kv_cache, page_table)
    rc = load_library().mla_decode_sparse(
        ctypes.byref(dims), _ptr(q_nope), _ptr(q_pe), _ptr(kv_cache), _ptr(page_table), _ptr(seq_lens),
        _ptr(indices), int(topk), int(Q), float(scale), float(kv_scale), _ptr(out), _ptr(lse), _ptr(workspace),
        ctypes.c_size_t(workspace.numel() * workspace.element_size()), _stream_handle(stream))
    if rc != MLA_OK:
        raise MlaError(rc, "mla_decode_sparse")


def mla_decode_sparse_query_status(q_nope, kv_cache, page_table, topk: int, workspace, stream=None) -> int:
    dims = make_dims(q_nope, kv_cache, page_table)
    st = ctypes.c_int32(0)
    rc = load_library().mla_decode_sparse_query_status(ctypes.byref(dims), int(topk), _ptr(workspace),
                                                        _stream_handle(stream), ctypes.byref(st))
    if rc != MLA_OK:
        raise MlaError(rc, "mla_decode_sparse_query_status")
    return st.value


def mla_decode_cascade_workspace_size(dims: MlaDims, prefix_pages: int, device: int | None = None) -> int:
    import torch

    dev = torch.cuda.current_device() if device is None else device
    n = load_library().mla_decode_cascade_workspace_size(ctypes.byref(dims), int(prefix_pages), dev)
    if n == 0:
        raise MlaError(-1, "mla_decode_cascade_workspace_size")
    return int(n)


def mla_decode_cascade(q_nope, q_pe, kv_cache, page_table, seq_lens, prefix_pages, scale, kv_scale, out, lse,
                       workspace, stream=None) -> None:
    """Enqueue a cascade decode over a shared prefix (see include/mla_cascade.h)."""
    _check_cuda(q_nope, q_pe, kv_cache, page_table, seq_lens, out, lse, workspace)
    _check_decode_tensors(q_nope, q_pe, kv_cache, page_table, seq_lens, out, lse, workspace)
    dims = make_dims(q_nope, kv_cache, page_table)
    rc = load_library().mla_decode_cascade(
        ctypes.byref(dims), _ptr(q_nope), _ptr(q_pe), _ptr(kv_cache), _ptr(page_table), _ptr(seq_lens),
        int(prefix_pages), int(q_nope.shape[1]), float(scale), float(kv_scale), _ptr(out), _ptr(lse), _ptr(workspace),
        ctypes.c_size_t(workspace.numel() * workspace.element_size()), _stream_handle(stream))
    if rc != MLA_OK:
        raise MlaError(rc, "mla_decode_cascade")


def mla_decode_cascade_query_status(q_nope, kv_cache, page_table, prefix_pages: int, workspace, stream=None) -> int:
    dims = make_dims(q_nope, kv_cache, page_table)
    st = ctypes.c_int32(0)
    rc = load_library().mla_decode_cascade_query_status(ctypes.byref(dims), int(prefix_pages), _ptr(workspace),
                                                         _stream_handle(stream), ctypes.byref(st))
    if rc != MLA_OK:
        raise MlaError(rc, "mla_decode_cascade_query_status")
    return st.value


@dataclass
class DecodeBuffers:
    out: object
    lse: object
    workspace: object


def alloc_buffers(q_nope, kv_cache, page_table) -> DecodeBuffers:
    """torch allocations sized for one decode step (caller-owned memory)."""
    import torch

    B, Q, H, _ = q_nope.shape
    dims = make_dims(q_nope, kv_cache, page_table)
    ws = torch.empty(mla_decode_workspace_size(dims, q_nope.device.index), dtype=torch.uint8, device=q_nope.device)
    out = torch.empty(B, Q, H, 512, dtype=torch.bfloat16, device=q_nope.device)
    lse = torch.empty(B, Q, H, dtype=torch.float32, device=q_nope.device)
    return DecodeBuffers(out, lse, ws)


def decode(q_nope, q_pe, kv_cache, page_table, seq_lens, scale, kv_scale=1.0, buffers: DecodeBuffers | None = None,
           stream=None):
    """Convenience wrapper: allocates outputs/workspace if not given; returns (out, lse)."""
    if buffers is None:
        buffers = alloc_buffers(q_nope, kv_cache, page_table)
    mla_decode(q_nope, q_pe, kv_cache, page_table, seq_lens, q_nope.shape[1], scale, kv_scale, buffers.out,
               buffers.lse, buffers.workspace, stream)
    return buffers.out, buffers.lse
