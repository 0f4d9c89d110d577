"""The named decode batches at full size, in the launch configuration the
benchmark times, checked against the oracle element by element on every
request of the batch (out and lse), plus whole-batch properties (finite
outputs, status word clear).  The oracle runs request by request in chunks,
so that host memory stays bounded (the e4m3 batch holds 33.5 M outputs)."""
import numpy as np
import pytest

from paged_mla_decode_09_gb300 import workloads as W

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import paged_mla_decode_09_gb300 as mla
    from paged_mla_decode_09_gb300.build import build_library

    build_library()
    mla.load_library()


from gpu_helpers import compare_chunked, run_gpu  # noqa: E402


@pytest.mark.parametrize("name", ["kimi", "dsv3", "prefix", "fp8", "verify4"])
def test_full_size_config_every_request(name):
    wl = W.make_config(name)
    out, lse, status, *_ = run_gpu(wl)
    assert status == 0
    assert np.all(np.isfinite(out)) and np.all(np.isfinite(lse))
    stats = compare_chunked(wl, out, lse, label=name)
    print(name, stats)
