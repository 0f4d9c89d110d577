"""A device reset between calls (cudaDeviceReset, a primary-context reset)
loads the library's device code again: the allocation-free entry point's
static scratch may then sit at another address, which the next call must
look up again.  The cached launch shapes (this device's occupancy) and the
kernels' shared-memory attributes stay valid: the runtime keeps the
attributes across the reset.  Both entry points must give the same results
after the reset as before it.

Runs in a child process (tests/reset_child.py) that touches CUDA only
through the library and the runtime, so that the reset leaves no torch
tensor of the old context behind in the test process.
"""
import os
import subprocess
import sys

import numpy as np
import pytest

from paged_mla_decode_09_gb300 import workloads as W

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_mla_decode_09_gb300.build import build_library

    build_library()


def test_decode_after_device_reset(tmp_path):
    import oracle
    from gpu_helpers import compare

    out_path = tmp_path / "reset.npz"
    child = os.path.join(os.path.dirname(os.path.abspath(__file__)), "reset_child.py")
    r = subprocess.run([sys.executable, child, str(out_path)], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    res = np.load(out_path)
    for name in ("decode", "noalloc"):
        for phase in ("before", "after"):
            assert int(res[f"rc_{name}_{phase}"]) == 0, (name, phase, int(res[f"rc_{name}_{phase}"]))
    ref_out, ref_lse = res["out_decode_before"], res["lse_decode_before"]
    for key in ("decode_after", "noalloc_before", "noalloc_after"):
        assert np.array_equal(res[f"out_{key}"], ref_out), key
        assert np.array_equal(res[f"lse_{key}"], ref_lse), key
    # the same seeded batch the child decoded, against the oracle
    wl = W.custom([300, 2000, 70], num_heads=64, q_len=1, seed=71)
    shape = (wl.batch, wl.q_len, wl.num_heads)
    out = oracle.bf16_bits_to_f64(ref_out.reshape(shape + (512,)))
    compare(wl, out, ref_lse.reshape(shape).astype(np.float64), label="after device reset")
