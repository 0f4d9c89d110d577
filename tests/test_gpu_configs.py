"""The named decode batches at full size, in the launch configuration the
benchmark times, checked against the oracle on sampled requests (the first,
the last and the longest) element by element, plus whole-batch properties
(finite outputs, status word clear)."""
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


from gpu_helpers import compare, run_gpu  # noqa: E402


@pytest.mark.parametrize("name", ["kimi", "dsv3", "prefix", "fp8", "verify4"])
def test_full_size_config_sampled(name):
    wl = W.make_config(name)
    out, lse, status, *_ = run_gpu(wl)
    assert status == 0
    assert np.all(np.isfinite(out)) and np.all(np.isfinite(lse))
    reqs = sorted({0, wl.batch - 1, int(np.argmax(wl.seq_lens))})
    stats = compare(wl, out, lse, requests=reqs, label=name)
    print(name, reqs, stats)
