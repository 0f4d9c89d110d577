"""GPU parity of the cache write (quantise-and-scatter of a step's new rows)
against the CPU oracle: bit-exact on every byte of the cache, for both cache
types, with the edge values of the e4m3 encoding, and on a full-size cache
in the launch the benchmark times (sampled rows)."""
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


def _tables(rng, seq_lens, pages, width):
    table = np.full((len(seq_lens), width), -1, dtype=np.int32)
    perm = rng.permutation(pages).astype(np.int32)
    pos = 0
    for b, L in enumerate(seq_lens):
        n = (int(L) + 63) // 64
        table[b, :n] = perm[pos:pos + n]
        pos += n
    return table


def _edge_rows(rng, B, n_new, kv_scale):
    """bf16 rows mixing ordinary values with the encoding's edge cases."""
    x = rng.standard_normal((B, n_new, 576)).astype(np.float32) * np.float32(40 * kv_scale)
    flat = x.reshape(-1)
    k = flat.size
    sel = rng.choice(k, size=k // 8, replace=False)
    kinds = rng.integers(0, 5, size=sel.size)
    flat[sel[kinds == 0]] = np.float32(1e4 * kv_scale)      # saturates to 448
    flat[sel[kinds == 1]] = np.float32(-1e4 * kv_scale)     # to -448
    flat[sel[kinds == 2]] = np.float32(2.0**-11 * kv_scale)  # rounds to zero
    flat[sel[kinds == 3]] = np.float32(-(2.0**-12) * kv_scale)  # to -0
    flat[sel[kinds == 4]] = 0.0
    return W.f32_to_bf16_bits(x)


def _run(rows_bits, table, seq_lens, kv_scale, cache_np, kv_dtype):
    import paged_mla_decode_09_gb300 as mla

    rows = torch.from_numpy(rows_bits.view(np.int16)).cuda().view(torch.bfloat16)
    if kv_dtype == "bf16":
        cache = torch.from_numpy(cache_np.view(np.int16)).cuda().view(torch.bfloat16)
    else:
        cache = torch.from_numpy(cache_np).cuda()
    pt = torch.from_numpy(table).cuda()
    sl = torch.from_numpy(np.asarray(seq_lens, dtype=np.int32)).cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    mla.mla_kv_pack(rows, pt, sl, kv_scale, cache, status)
    torch.cuda.synchronize()
    out = cache.view(torch.int16).cpu().numpy().view(np.uint16) if kv_dtype == "bf16" else cache.cpu().numpy()
    return out, int(status.item())


@pytest.mark.parametrize("kv_dtype,n_new", [("fp8_e4m3", 1), ("fp8_e4m3", 2), ("fp8_e4m3", 4), ("bf16", 2),
                                            ("fp8_e4m3", 130)])
def test_kv_pack_bit_exact(kv_dtype, n_new):
    rng = np.random.default_rng(100 + n_new)
    seq_lens = np.array([n_new, 64 + n_new, 63 + n_new, 700, 130 + n_new], dtype=np.int32)
    pages = 40
    table = _tables(rng, seq_lens, pages, 14)
    kv_scale = 0.0173 if kv_dtype == "fp8_e4m3" else 1.0
    rows = _edge_rows(rng, len(seq_lens), n_new, kv_scale)
    dt = np.uint8 if kv_dtype == "fp8_e4m3" else np.uint16
    cache = rng.integers(0, 250, size=(pages, 64, 576)).astype(dt)  # stale contents
    got, status = _run(rows, table, seq_lens, kv_scale, cache, kv_dtype)
    ref, ref_status = oracle.kv_pack_ref(rows, table, seq_lens, kv_scale, cache, kv_dtype)
    assert status == ref_status == 0
    assert np.array_equal(got, ref)


def test_kv_pack_nan_gives_nan_codes():
    rng = np.random.default_rng(7)
    seq_lens = np.array([5], dtype=np.int32)
    table = _tables(rng, seq_lens, 2, 1)
    rows = W.f32_to_bf16_bits(np.full((1, 2, 576), np.nan, dtype=np.float32))
    cache = np.zeros((2, 64, 576), dtype=np.uint8)
    got, status = _run(rows, table, seq_lens, 0.5, cache, "fp8_e4m3")
    assert status == 0
    page = table[0, 0]
    assert np.all((got[page, 3:5] & 0x7F) == 0x7F)


def test_kv_pack_bad_rows_flagged_and_skipped():
    rng = np.random.default_rng(8)
    table = np.array([[0, 99], [1, -1], [2, 3]], dtype=np.int32)
    seq_lens = np.array([66, 1, 300], dtype=np.int32)  # page 99 outside; 1 < 2 new; 300 > 2 pages
    rows = _edge_rows(rng, 3, 2, 0.1)
    cache = rng.integers(0, 250, size=(4, 64, 576)).astype(np.uint8)
    got, status = _run(rows, table, seq_lens, 0.1, cache, "fp8_e4m3")
    ref, ref_status = oracle.kv_pack_ref(rows, table, seq_lens, 0.1, cache, "fp8_e4m3")
    assert status == ref_status == 3
    assert np.array_equal(got, ref)


def test_kv_pack_full_size_sampled():
    """The benchmark's write (Kimi-shaped prefill into an e4m3 cache: B=64,
    4096 new tokens each) in its launch configuration: 512 sampled rows,
    each found at its page and slot, bit-exact against the oracle's encoding."""
    import paged_mla_decode_09_gb300 as mla

    wl = W.kv_pack_batch()
    rows = torch.from_numpy(wl.rows_bits.view(np.int16)).cuda().view(torch.bfloat16)
    cache = torch.zeros(wl.num_pages, 64, 576, dtype=torch.uint8, device="cuda")
    pt = torch.from_numpy(wl.page_table).cuda()
    sl = torch.from_numpy(wl.seq_lens).cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    mla.mla_kv_pack(rows, pt, sl, wl.kv_scale, cache, status)
    torch.cuda.synchronize()
    assert status.item() == 0
    rng = np.random.default_rng(3)
    B, n_new = wl.rows_bits.shape[:2]
    for _ in range(512):
        b, i = int(rng.integers(B)), int(rng.integers(n_new))
        t = int(wl.seq_lens[b]) - n_new + i
        page = int(wl.page_table[b, t // 64])
        got = cache[page, t % 64].cpu().numpy()
        assert np.array_equal(got, oracle.kv_pack.quantise_e4m3(wl.rows_bits[b, i], wl.kv_scale)), (b, i)


def test_kv_pack_rounds_the_exact_quotient_near_midpoints():
    """Values whose quotient x / kv_scale lies within a hair of a midpoint
    between two e4m3 codes, where multiplying by the fp32 reciprocal of the
    scale would pick the other code: bit-exact against the oracle (exact
    division), one call per scale."""
    from kvpack_cases import distinguishing_cases

    rng = np.random.default_rng(21)
    for x_bits, kv_scale in distinguishing_cases(6):
        seq_lens = np.array([3], dtype=np.int32)
        table = _tables(rng, seq_lens, 2, 1)
        rows = _edge_rows(rng, 1, 3, kv_scale)
        rows[0, :, :8] = x_bits
        rows[0, :, 8:16] = x_bits ^ np.uint16(0x8000)  # the same magnitude, negative
        cache = rng.integers(0, 250, size=(2, 64, 576)).astype(np.uint8)
        got, status = _run(rows, table, seq_lens, kv_scale, cache, "fp8_e4m3")
        ref, ref_status = oracle.kv_pack_ref(rows, table, seq_lens, kv_scale, cache, "fp8_e4m3")
        assert status == ref_status == 0
        assert np.array_equal(got, ref), (hex(int(x_bits)), kv_scale)
