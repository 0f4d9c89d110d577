"""The allocation-free entry point, checked against the workspace-based one.

mla_decode_noalloc exists for callers that cannot allocate device memory:
a serving loop that must never call cudaMalloc, a process that handed all
device memory to its own pool at start-up, or a plug-in that only receives
buffers from its host.  It keeps its scratch (status words, schedule, split
partials) in a fixed 40 MiB array inside the library instead of a caller
workspace.  Two calls in a row, made through the C ABI, must agree with
mla_decode and with the CPU oracle within the parity tolerance (they may
split the keys over fewer clusters, so only rounding may differ) and with
each other bit for bit, and the status word they copy out must be clear.

This file is collected last on purpose and also runs on its own.
"""
import ctypes

import numpy as np
import pytest

from paged_mla_decode_09_gb300 import workloads as W

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

TOL = {"bf16": (1e-2, 1e-2), "fp8_e4m3": (4e-2, 4e-2)}


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import paged_mla_decode_09_gb300 as mla
    from paged_mla_decode_09_gb300.build import build_library

    build_library()
    return mla.load_library()


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _noalloc(lib, db, dims, out, lse, status):
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.mla_decode_noalloc(ctypes.byref(dims), _p(db.q_nope), _p(db.q_pe), _p(db.kv_cache),
                                  _p(db.page_table), _p(db.seq_lens), db.q_len, db.scale, db.kv_scale, _p(out),
                                  _p(lse), _p(status), stream)


@pytest.mark.parametrize("lens,H,Q,dtype", [
    ([3000, 700, 129, 5000, 64], 64, 1, "bf16"),
    ([4100, 1500, 2], 128, 2, "fp8_e4m3"),
])
def test_noalloc_matches_mla_decode_twice(lib, lens, H, Q, dtype):
    import paged_mla_decode_09_gb300 as mla
    from paged_mla_decode_09_gb300.device_inputs import to_device

    wl = W.custom(lens, num_heads=H, q_len=Q, kv_dtype=dtype, seed=sum(lens) + 7)
    db = to_device(wl)
    ref = mla.alloc_buffers(db.q_nope, db.kv_cache, db.page_table)
    mla.mla_decode(db.q_nope, db.q_pe, db.kv_cache, db.page_table, db.seq_lens, db.q_len, db.scale, db.kv_scale,
                   ref.out, ref.lse, ref.workspace)
    torch.cuda.synchronize()
    assert mla.mla_query_status(ref.workspace) == 0
    ref_out = ref.out.float().cpu().numpy()
    ref_lse = ref.lse.cpu().numpy()

    import oracle

    ora_out, ora_lse = oracle.mla_decode_ref(wl.q_nope, wl.q_pe, wl.kv_cache, wl.page_table, wl.seq_lens, wl.q_len,
                                             wl.scale, wl.kv_scale, wl.kv_dtype)
    dims = mla.make_dims(db.q_nope, db.kv_cache, db.page_table)
    atol, rtol = TOL[dtype]
    results = []
    for _ in range(2):
        out = torch.full_like(ref.out, float("nan"))
        lse = torch.full_like(ref.lse, float("nan"))
        status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
        assert _noalloc(lib, db, dims, out, lse, status) == 0
        torch.cuda.synchronize()
        assert status.item() == 0
        o = out.float().cpu().numpy()
        l = lse.cpu().numpy()
        assert np.all(np.abs(o - ref_out) <= atol + rtol * np.abs(ref_out))
        assert np.all(np.abs(l - ref_lse) <= atol + rtol * np.abs(ref_lse))
        assert np.all(np.abs(o - ora_out) <= atol + rtol * np.abs(ora_out))
        assert np.all(np.abs(l - ora_lse) <= atol + rtol * np.abs(ora_lse))
        results.append((o, l))
    assert np.array_equal(results[0][0], results[1][0]) and np.array_equal(results[0][1], results[1][1])


def test_noalloc_rejects_batches_beyond_its_scratch(lib):
    import paged_mla_decode_09_gb300 as mla
    from paged_mla_decode_09_gb300.device_inputs import to_device

    wl = W.custom([100], num_heads=16, seed=3)
    db = to_device(wl)
    dims = mla.make_dims(db.q_nope, db.kv_cache, db.page_table)
    dims.batch = 5_000_000  # the schedule alone would need 60 MB: refused before any launch
    out = torch.empty(1, 1, 16, 512, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(1, 1, 16, dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert _noalloc(lib, db, dims, out, lse, status) == -7
    assert b"40 MiB" in lib.mla_status_string(-7)
