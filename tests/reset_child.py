"""Child process of test_gpu_context_reset: decodes one small seeded batch
through the C ABI with plain cudaMalloc'd buffers, resets the device
(cudaDeviceReset ends this process's context, and with it every allocation
and the library's loaded device code), then decodes it again in the new
context, with both mla_decode and mla_decode_noalloc each time.  No torch
CUDA state exists in this process, so nothing holds a pointer of the old
context.  Writes the return codes and the raw results to ARGV[1] (.npz).

Usage: python tests/reset_child.py OUT.npz
"""
import ctypes
import os
import sys

import numpy as np

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

import paged_mla_decode_09_gb300 as mla  # noqa: E402
from paged_mla_decode_09_gb300 import workloads as W  # noqa: E402


def cudart():
    """The CUDA runtime the library is linked against (the same loaded copy)."""
    with open("/proc/self/maps") as f:
        for line in f:
            path = line.split()[-1]
            if os.path.basename(path).startswith("libcudart.so"):
                return ctypes.CDLL(path)
    raise RuntimeError("libcudart is not loaded")


def main(out_path):
    lib = mla.load_library()
    rt = cudart()
    P = ctypes.c_void_p
    rt.cudaMalloc.argtypes = [ctypes.POINTER(P), ctypes.c_size_t]
    rt.cudaMemcpy.argtypes = [P, P, ctypes.c_size_t, ctypes.c_int]
    rt.cudaMemset.argtypes = [P, ctypes.c_int, ctypes.c_size_t]
    rt.cudaFree.argtypes = [P]
    H2D, D2H = 1, 2

    def check(rc, what):
        if rc != 0:
            raise RuntimeError(f"{what} returned {rc}")

    wl = W.custom([300, 2000, 70], num_heads=64, q_len=1, seed=71)
    dims = mla.MlaDims(batch=wl.batch, num_heads=wl.num_heads, q_len=wl.q_len, page_size=64,
                       num_pages=wl.num_pages, max_pages_per_req=wl.max_pages,
                       page_table_stride=wl.max_pages, kv_dtype=mla.MLA_KV_BF16)
    host = {
        "q_nope": np.ascontiguousarray(wl.q_nope),
        "q_pe": np.ascontiguousarray(wl.q_pe),
        "kv": np.ascontiguousarray(wl.kv_cache),
        "pt": np.ascontiguousarray(wl.page_table),
        "sl": np.ascontiguousarray(wl.seq_lens),
    }
    out_elems = wl.batch * wl.q_len * wl.num_heads * 512
    lse_elems = wl.batch * wl.q_len * wl.num_heads

    def decode(noalloc):
        check(rt.cudaSetDevice(0), "cudaSetDevice")
        ptrs = {}
        try:
            for k, a in host.items():
                ptrs[k] = P()
                check(rt.cudaMalloc(ctypes.byref(ptrs[k]), a.nbytes), "cudaMalloc")
                check(rt.cudaMemcpy(ptrs[k], a.ctypes.data, a.nbytes, H2D), "cudaMemcpy")
            ws_bytes = lib.mla_decode_workspace_size(ctypes.byref(dims), 0)
            if ws_bytes == 0:
                return -1, None, None
            for k, n in (("out", out_elems * 2), ("lse", lse_elems * 4), ("ws", ws_bytes)):
                ptrs[k] = P()
                check(rt.cudaMalloc(ctypes.byref(ptrs[k]), n), "cudaMalloc")
                check(rt.cudaMemset(ptrs[k], 0xFF, n), "cudaMemset")
            if noalloc:
                rc = lib.mla_decode_noalloc(ctypes.byref(dims), ptrs["q_nope"], ptrs["q_pe"], ptrs["kv"], ptrs["pt"],
                                            ptrs["sl"], wl.q_len, wl.scale, 1.0, ptrs["out"], ptrs["lse"], None,
                                            None)
            else:
                rc = lib.mla_decode(ctypes.byref(dims), ptrs["q_nope"], ptrs["q_pe"], ptrs["kv"], ptrs["pt"],
                                    ptrs["sl"], wl.q_len, wl.scale, 1.0, ptrs["out"], ptrs["lse"], ptrs["ws"],
                                    ws_bytes, None)
            check(rt.cudaDeviceSynchronize(), "cudaDeviceSynchronize")
            out = np.empty(out_elems, dtype=np.uint16)
            lse = np.empty(lse_elems, dtype=np.float32)
            if rc == 0:
                check(rt.cudaMemcpy(out.ctypes.data, ptrs["out"], out.nbytes, D2H), "cudaMemcpy")
                check(rt.cudaMemcpy(lse.ctypes.data, ptrs["lse"], lse.nbytes, D2H), "cudaMemcpy")
            return rc, out, lse
        finally:
            for p in ptrs.values():
                rt.cudaFree(p)

    res = {}
    for phase in ("before", "after"):
        if phase == "after":
            check(rt.cudaDeviceReset(), "cudaDeviceReset")
        for name, noalloc in (("decode", False), ("noalloc", True)):
            rc, out, lse = decode(noalloc)
            res[f"rc_{name}_{phase}"] = np.int32(rc)
            if rc == 0:
                res[f"out_{name}_{phase}"] = out
                res[f"lse_{name}_{phase}"] = lse
    np.savez(out_path, **res)


if __name__ == "__main__":
    main(sys.argv[1])
