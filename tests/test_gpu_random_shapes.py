"""Seeded random decode batches against the oracle, element by element: the
batch size, head count, draft count, lengths (including 1-token, page-edge
and multi-split ones) and cache type are drawn from one generator, so the
sweep covers combinations the hand-written cases do not.  Sizes stay small
enough for the oracle to finish in seconds."""
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


def draw_case(seed):
    rng = np.random.default_rng(seed)
    H = int(rng.choice([1, 8, 16, 24, 32, 48, 64, 96, 128]))
    q_max = max(1, min(4, 256 // H))
    Q = int(rng.integers(1, q_max + 1))
    B = int(rng.integers(1, 9))
    kind = rng.choice(["short", "edge", "mixed", "long"], p=[0.2, 0.3, 0.3, 0.2])
    if kind == "short":
        lens = rng.integers(Q, Q + 70, size=B)
    elif kind == "edge":
        lens = 64 * rng.integers(1, 12, size=B) + rng.choice([-1, 0, 1], size=B)
    elif kind == "mixed":
        lens = np.exp(rng.uniform(np.log(Q + 1), np.log(6000), size=B)).astype(int)
    else:
        lens = rng.integers(3000, 9000, size=B)
    lens = np.maximum(lens, Q)
    dtype = "fp8_e4m3" if rng.random() < 0.3 else "bf16"
    return [int(x) for x in lens], H, Q, dtype


@pytest.mark.parametrize("seed", list(range(16)))
def test_random_shape_parity(seed):
    lens, H, Q, dtype = draw_case(1000 + seed)
    wl = W.custom(lens, num_heads=H, q_len=Q, kv_dtype=dtype, seed=5000 + seed)
    out, lse, status, *_ = run_gpu(wl)
    assert status == 0
    stats = compare(wl, out, lse, label=f"seed {seed}: lens={lens} H={H} Q={Q} {dtype}")
    print(seed, lens, H, Q, dtype, stats)
