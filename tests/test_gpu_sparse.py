"""GPU parity of the top-k decode (gather of the picked rows + paged decode)
against the CPU oracle: small cases element by element (both cache types,
one and two draft positions, padding, repeated and invalid picks), and the
DeepSeek-V3.2-shaped batch in the benchmark's launch on sampled requests."""
import numpy as np
import pytest

import oracle
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


from gpu_helpers import TOL  # noqa: E402


def run_sparse(wl, idx):
    import paged_mla_decode_09_gb300 as mla
    from paged_mla_decode_09_gb300.device_inputs import out_to_f64, to_device

    db = to_device(wl, "cuda")
    ix = torch.from_numpy(np.ascontiguousarray(idx, dtype=np.int32)).cuda()
    dims = mla.make_dims(db.q_nope, db.kv_cache, db.page_table)
    ws = torch.full((mla.mla_decode_sparse_workspace_size(dims, idx.shape[2]),), 0xFF, dtype=torch.uint8,
                    device="cuda")
    B, Q, H, _ = db.q_nope.shape
    out = torch.full((B, Q, H, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((B, Q, H), float("nan"), dtype=torch.float32, device="cuda")
    mla.mla_decode_sparse(db.q_nope, db.q_pe, db.kv_cache, db.page_table, db.seq_lens, ix, db.scale, db.kv_scale,
                          out, lse, ws)
    torch.cuda.synchronize()
    st = mla.mla_decode_sparse_query_status(db.q_nope, db.kv_cache, db.page_table, idx.shape[2], ws)
    return out_to_f64(out), lse.cpu().numpy().astype(np.float64), st


def check(wl, idx, out, lse, requests=None):
    ro, rl, rst = oracle.mla_decode_sparse_ref(wl.q_nope, wl.q_pe, wl.kv_cache, wl.page_table, wl.seq_lens,
                                               wl.q_len, idx, wl.scale, wl.kv_scale, wl.kv_dtype, requests=requests)
    sel = np.arange(wl.batch) if requests is None else np.asarray(requests)
    atol, rtol = TOL["fp8_e4m3" if wl.kv_dtype == "fp8_e4m3" else "bf16"]
    eo = np.abs(out[sel] - ro[sel])
    el = np.abs(lse[sel] - rl[sel])
    assert np.all(eo <= atol + rtol * np.abs(ro[sel])), float(eo.max())
    assert np.all(el <= atol + rtol * np.abs(rl[sel])), float(el.max())
    return rst


@pytest.mark.parametrize("seq_lens,H,Q,topk,dtype", [
    ([70, 300, 1000], 16, 1, 100, "bf16"),
    ([130, 2000, 64], 128, 2, 300, "bf16"),
    ([4, 900, 5000], 64, 2, 256, "fp8_e4m3"),
    ([3000, 65], 64, 1, 2048, "bf16"),
    ([40, 41], 16, 2, 1, "bf16"),
])
def test_sparse_parity(seq_lens, H, Q, topk, dtype):
    wl = W.custom(seq_lens, num_heads=H, q_len=Q, kv_dtype=dtype, seed=sum(seq_lens) + topk)
    idx = W.topk_indices(wl, topk, seed=topk + 1)
    out, lse, st = run_sparse(wl, idx)
    assert st == 0
    assert check(wl, idx, out, lse) == 0


def test_sparse_repeated_and_invalid_picks():
    wl = W.custom([200, 500], num_heads=64, q_len=2, seed=77)
    idx = W.topk_indices(wl, 64, seed=5)
    idx[0, 0, :4] = [10, 10, 10, 3]       # repeated picks count each time
    idx[1, 1, 5] = 500                    # beyond the visible positions: flagged, skipped
    idx[1, 0, 7] = -9                     # negative but not -1: flagged, skipped
    idx[0, 1, 20:] = -1                   # padding in the middle of the list is skipped silently
    out, lse, st = run_sparse(wl, idx)
    assert st == oracle.sparse.BAD_INDEX
    assert check(wl, idx, out, lse) == oracle.sparse.BAD_INDEX


def test_sparse_empty_pick_list_gives_empty_result():
    wl = W.custom([100, 100, 300], num_heads=16, q_len=2, seed=78)
    idx = W.topk_indices(wl, 8, seed=6)
    idx[1, 0, :] = -1
    idx[2, 1, :] = -1
    out, lse, st = run_sparse(wl, idx)
    assert st == oracle.sparse.BAD_INDEX
    assert np.all(out[1, 0] == 0) and np.all(lse[1, 0] == -np.inf)
    assert np.all(out[2, 1] == 0) and np.all(lse[2, 1] == -np.inf)
    assert np.all(np.isfinite(lse[1, 1])) and np.all(np.isfinite(lse[2, 0]))
    check(wl, idx, out, lse, requests=[0])
    ro, rl, _ = oracle.mla_decode_sparse_ref(wl.q_nope, wl.q_pe, wl.kv_cache, wl.page_table, wl.seq_lens, 2, idx,
                                             wl.scale, requests=[1, 2])
    assert np.all(np.abs(out[1, 1] - ro[1, 1]) <= 1e-2 + 1e-2 * np.abs(ro[1, 1]))
    assert np.all(np.abs(lse[2, 0] - rl[2, 0]) <= 1e-2 + 1e-2 * np.abs(rl[2, 0]))


def test_sparse_full_size_sampled():
    wl = W.make_config("dsa")
    idx = W.topk_indices(wl, wl.meta["topk"], seed=2)
    out, lse, st = run_sparse(wl, idx)
    assert st == 0
    assert np.all(np.isfinite(out)) and np.all(np.isfinite(lse))
    check(wl, idx, out, lse, requests=[0, wl.batch - 1])
