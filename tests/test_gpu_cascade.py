"""GPU parity of the cascade decode over a shared prefix against the CPU
oracle's plain decode (the cascade computes the same operation): several
requests per prefix-pass row block (g = 2, 4), one (g = 1), an odd batch
(the ungrouped tail), two draft positions, both cache types, the full-size
prefix batch on sampled requests, and a prefix that is not shared."""
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


from gpu_helpers import compare  # noqa: E402


def run_cascade(wl, prefix_pages):
    import paged_mla_decode_09_gb300 as mla
    from paged_mla_decode_09_gb300.device_inputs import out_to_f64, to_device

    db = to_device(wl, "cuda")
    dims = mla.make_dims(db.q_nope, db.kv_cache, db.page_table)
    ws = torch.full((mla.mla_decode_cascade_workspace_size(dims, prefix_pages),), 0xFF, dtype=torch.uint8,
                    device="cuda")
    B, Q, H, _ = db.q_nope.shape
    out = torch.full((B, Q, H, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((B, Q, H), float("nan"), dtype=torch.float32, device="cuda")
    mla.mla_decode_cascade(db.q_nope, db.q_pe, db.kv_cache, db.page_table, db.seq_lens, prefix_pages, db.scale,
                           db.kv_scale, out, lse, ws)
    torch.cuda.synchronize()
    st = mla.mla_decode_cascade_query_status(db.q_nope, db.kv_cache, db.page_table, prefix_pages, ws)
    return out_to_f64(out), lse.cpu().numpy().astype(np.float64), st


@pytest.mark.parametrize("batch,H,Q,prefix,dtype", [
    (6, 64, 1, 40, "bf16"),        # g = 2
    (5, 64, 1, 17, "bf16"),        # g = 2 and a tail of one request
    (7, 16, 2, 9, "bf16"),         # g = 4 (32 rows per request) and a tail of 3
    (3, 128, 1, 30, "bf16"),       # g = 1
    (4, 48, 1, 12, "bf16"),        # 48 rows do not divide 128: g = 1
    (6, 64, 2, 25, "fp8_e4m3"),    # g = 1 (128 rows), e4m3 cache
])
def test_cascade_parity(batch, H, Q, prefix, dtype):
    wl = W.prefix_shaped(batch=batch, num_heads=H, prefix_pages=prefix, suffix_range=(Q + 1, 700),
                         seed=batch * 100 + H + prefix, kv_dtype=dtype, q_len=Q)
    out, lse, st = run_cascade(wl, prefix)
    assert st == 0
    compare(wl, out, lse, label=f"cascade B={batch} H={H} Q={Q}")


def test_cascade_full_size_prefix_batch_sampled():
    wl = W.make_config("prefix")
    out, lse, st = run_cascade(wl, wl.meta["shared_prefix_pages"])
    assert st == 0
    assert np.all(np.isfinite(out)) and np.all(np.isfinite(lse))
    compare(wl, out, lse, requests=[0, wl.batch - 1, int(np.argmax(wl.seq_lens))], label="cascade prefix")


def test_cascade_flags_a_prefix_that_is_not_shared():
    wl = W.prefix_shaped(batch=4, num_heads=64, prefix_pages=10, suffix_range=(100, 300), seed=5)
    wl.page_table[2, 3] = wl.page_table[2, 11]  # request 2 names another page in the prefix columns
    _, _, st = run_cascade(wl, 10)
    import paged_mla_decode_09_gb300 as mla

    assert st & mla.MLA_DEV_BAD_PREFIX
