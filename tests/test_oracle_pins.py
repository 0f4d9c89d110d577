"""Pins for the CPU oracle: each check is independent of the oracle's own code.

* non-absorbed multi-head attention with random up-projections (the form the
  absorbed decode is derived from) must equal the absorbed result;
* closed forms (one key; all keys scored equally; a hand-derived two-token
  golden case);
* the split-KV pieces merged by log-sum-exp equal the unsplit result;
* a pure-Python brute force with its own gather, math.fsum and a softmax
  without max subtraction;
* torch's float8_e4m3fn decoder for every E4M3 code, and its float8
  conversion (round to nearest-even) for the encoder on in-range values;
* the encoder's round trips, ties and saturation points derived by hand;
* the cache write's scatter against positions computed independently;
* causal masking of two draft positions against single-position calls;
* page relabelling, prefix copies and tail sentinels leave the result alone.
"""
import math
import os

import numpy as np
import pytest

import oracle
from oracle import attend, lse_merge, mla_decode_ref, mla_decode_ref_pieces
from paged_mla_decode_09_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ----------------------------------------------------------------- encodings
def test_e4m3_table_matches_torch():
    torch = pytest.importorskip("torch")
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    mine = oracle.e4m3_to_f64(codes)
    assert np.array_equal(np.isnan(ref), np.isnan(mine))
    ok = ~np.isnan(ref)
    assert np.array_equal(ref[ok], mine[ok])


def test_e4m3_extremes():
    t = oracle.e4m3_decode_table()
    assert t[0x7E] == 448.0 and t[0xFE] == -448.0
    assert t[0x01] == 2.0**-9  # smallest subnormal
    assert t[0x08] == 2.0**-6  # smallest normal
    assert t[0x38] == 1.0
    assert np.isnan(t[0x7F]) and np.isnan(t[0xFF])
    assert np.sum(np.isnan(t)) == 2
    assert t[0x80] == 0.0 and math.copysign(1.0, t[0x80]) == -1.0


def test_e4m3_encode_round_trips_every_finite_code():
    t = oracle.e4m3_decode_table()
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    assert np.array_equal(oracle.e4m3_encode(t[codes]), codes)


def test_e4m3_encode_ties_go_to_the_even_code():
    t = oracle.e4m3_decode_table()
    # between consecutive positive values c and c + 1 the midpoint goes to
    # whichever of the two has mantissa bit 0 clear; a hair off it goes to
    # the nearer one
    for c in range(0, 0x7E):
        mid = (t[c] + t[c + 1]) / 2
        even = c if c % 2 == 0 else c + 1
        assert oracle.e4m3_encode([mid])[0] == even, c
        assert oracle.e4m3_encode([mid - (t[c + 1] - t[c]) * 1e-3])[0] == c
        assert oracle.e4m3_encode([mid + (t[c + 1] - t[c]) * 1e-3])[0] == c + 1
        assert oracle.e4m3_encode([-mid])[0] == (even | 0x80)


def test_e4m3_encode_saturation_zero_and_nan():
    enc = oracle.e4m3_encode
    assert list(enc([448.0, 449.0, 464.0, 480.0, 1e30, np.inf])) == [0x7E] * 6
    assert list(enc([-448.0, -1e30, -np.inf])) == [0xFE] * 3
    assert list(enc([2.0**-10, 2.0**-10 * 1.01, 2.0**-9 * 1.5, 2.0**-9 * 1.49])) == [0x00, 0x01, 0x02, 0x01]
    assert list(enc([0.0, -0.0, -(2.0**-12)])) == [0x00, 0x80, 0x80]
    assert enc([np.nan])[0] & 0x7F == 0x7F


def test_e4m3_encode_matches_torch_rounding_in_range():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(5)
    x = np.concatenate([rng.standard_normal(20000) * 50, rng.standard_normal(5000) * 1e-2,
                        rng.uniform(-448, 448, 5000)]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(oracle.e4m3_encode(x), ref)


def test_kv_pack_writes_exactly_the_new_positions():
    rng = np.random.default_rng(9)
    B, n_new, pages = 3, 3, 12
    seq_lens = np.array([3, 66, 130], dtype=np.int32)
    table = np.full((B, 4), -1, dtype=np.int32)
    perm = rng.permutation(pages)
    table[0, :1], table[1, :2], table[2, :3] = perm[:1], perm[1:3], perm[3:6]
    rows = W.f32_to_bf16_bits(rng.standard_normal((B, n_new, 576)).astype(np.float32) * 30)
    for kv_dtype, scale in (("bf16", 1.0), ("fp8_e4m3", 0.05)):
        dt = np.uint16 if kv_dtype == "bf16" else np.uint8
        cache = rng.integers(0, 200, size=(pages, 64, 576)).astype(dt)
        out, status = oracle.kv_pack_ref(rows, table, seq_lens, scale, cache, kv_dtype)
        assert status == 0
        written = set()
        for b in range(B):
            for i in range(n_new):
                t = int(seq_lens[b]) - n_new + i  # positions L-3, L-2, L-1
                page, slot = int(table[b, t // 64]), t % 64
                written.add((page, slot))
                vals = (rows[b, i].astype(np.uint32) << 16).view(np.float32)
                if kv_dtype == "bf16":
                    assert np.array_equal(out[page, slot], rows[b, i])
                else:  # decodes to the nearest e4m3 value of x / scale
                    dec = oracle.e4m3_to_f64(out[page, slot])
                    grid = oracle.e4m3_decode_table()[:0x7F]
                    target = np.clip(np.abs(vals.astype(np.float64) / scale), 0, 448)
                    best = np.min(np.abs(grid[None, :] - target[:, None]), axis=1)
                    assert np.allclose(np.abs(np.abs(dec) - target), best, rtol=0, atol=1e-6 * (1 + target))
        mask = np.ones((pages, 64), dtype=bool)
        for page, slot in written:
            mask[page, slot] = False
        assert np.array_equal(out[mask], cache[mask])  # nothing else touched
        assert len(written) == B * n_new


def test_kv_pack_flags_bad_rows_and_skips_them():
    rng = np.random.default_rng(12)
    table = np.array([[0, 99], [1, -1]], dtype=np.int32)
    rows = W.f32_to_bf16_bits(rng.standard_normal((2, 2, 576)).astype(np.float32))
    cache = rng.integers(0, 120, size=(4, 64, 576)).astype(np.uint8)
    out, status = oracle.kv_pack_ref(rows, table, np.array([66, 1], dtype=np.int32), 1.0, cache, "fp8_e4m3")
    assert status == 3  # page 99 is outside the pool; length 1 < 2 new tokens
    assert np.array_equal(out, cache)  # neither bad row was written anywhere
    out, status = oracle.kv_pack_ref(rows, table, np.array([64, 200], dtype=np.int32), 1.0, cache, "fp8_e4m3")
    assert status == 2  # 200 > 2 pages * 64
    changed = np.argwhere(np.any(out != cache, axis=2))
    assert {tuple(x) for x in changed} <= {(0, 62), (0, 63)}  # only request 0's two rows


def test_bf16_decode_patterns():
    bits = np.array([0x3F80, 0xC000, 0x0000, 0x3E80, 0x4049], dtype=np.uint16)
    v = oracle.bf16_bits_to_f64(bits)
    assert list(v[:4]) == [1.0, -2.0, 0.0, 0.25]
    assert v[4] == 3.140625


def test_generator_bf16_rounding_is_nearest_even():
    x = np.array([1.0 + 2.0**-8, 1.0 + 3 * 2.0**-8, 1.0 + 2.0**-9], dtype=np.float32)
    bits = W.f32_to_bf16_bits(x)
    # 1+2^-8 is a tie between 1 and 1+2^-7 -> even (1); 1+3*2^-8 ties -> 1+2^-6
    assert list(oracle.bf16_bits_to_f64(bits)) == [1.0, 1.0 + 2.0**-6, 1.0]


# ----------------------------------------------- non-absorbed equivalence
def _mha_nonabsorbed(q_h, q_pe, c, k_pe, w_uk, w_uv, nvis, scale):
    """Standard attention with decompressed keys/values for one head."""
    K = np.concatenate([c @ w_uk.T, k_pe], axis=1)  # [L, 128 + 64]
    V = c @ w_uv.T  # [L, 128]
    q = np.concatenate([q_h, q_pe])
    s = (K[:nvis] @ q) * scale
    m = s.max()
    p = np.exp(s - m)
    z = p.sum()
    return (p / z) @ V[:nvis], m + np.log(z)


def test_non_absorbed_equivalence_dense_weights():
    rng = np.random.default_rng(11)
    H, L, dh = 4, 37, 128
    scale = 1 / math.sqrt(192)
    c = rng.standard_normal((L, 512))
    k_pe = rng.standard_normal((L, 64))
    rows = np.concatenate([c, k_pe], axis=1)
    qrows, expect = [], []
    for h in range(H):
        w_uk = rng.standard_normal((dh, 512)) / math.sqrt(512)
        w_uv = rng.standard_normal((dh, 512)) / math.sqrt(512)
        q_h = rng.standard_normal(dh)
        q_pe = rng.standard_normal(64)
        qrows.append((np.concatenate([w_uk.T @ q_h, q_pe]), w_uv))
        expect.append(_mha_nonabsorbed(q_h, q_pe, c, k_pe, w_uk, w_uv, L, scale))
    out, lse = attend(np.stack([q for q, _ in qrows]), rows, L, scale)
    for h in range(H):
        w_uv = qrows[h][1]
        np.testing.assert_allclose(w_uv @ out[h], expect[h][0], rtol=1e-10, atol=1e-12)
        assert abs(lse[h] - expect[h][1]) <= 1e-10 * max(1.0, abs(expect[h][1]))


def test_non_absorbed_equivalence_through_paged_bf16_entry():
    """End to end through the bf16 entry point: W_UK maps every latent
    coordinate to one signed coordinate of q_h, so the absorbed query is
    exactly representable in bf16; W_UV is dense."""
    rng = np.random.default_rng(5)
    H, dh = 3, 128
    wl = W.custom([150], num_heads=H, seed=77)
    L = int(wl.seq_lens[0])
    rows = oracle.decode_cache_rows(oracle.gather_rows(wl.kv_cache, wl.page_table[0], L), "bf16", 1.0)
    c, k_pe = rows[:, :512], rows[:, 512:]
    q_pe = oracle.bf16_bits_to_f64(wl.q_pe[0, 0])
    qn_bits = np.empty((1, 1, H, 512), dtype=np.uint16)
    expect = []
    for h in range(H):
        q_h_bits = W.f32_to_bf16_bits(rng.standard_normal(dh).astype(np.float32))
        q_h = oracle.bf16_bits_to_f64(q_h_bits)
        pi = rng.integers(0, dh, size=512)
        sg = rng.choice([-1.0, 1.0], size=512)
        w_uk = np.zeros((dh, 512))
        w_uk[pi, np.arange(512)] = sg
        qn = w_uk.T @ q_h  # each entry = +-q_h[pi[j]], exact in bf16
        qn_bits[0, 0, h] = W.f32_to_bf16_bits(qn.astype(np.float32))
        assert np.array_equal(oracle.bf16_bits_to_f64(qn_bits[0, 0, h]), qn)
        w_uv = rng.standard_normal((dh, 512)) / math.sqrt(512)
        expect.append((w_uv, _mha_nonabsorbed(q_h, q_pe[h], c, k_pe, w_uk, w_uv, L, wl.scale)))
    out, lse = mla_decode_ref(qn_bits, wl.q_pe, wl.kv_cache, wl.page_table, wl.seq_lens, 1, wl.scale)
    for h in range(H):
        w_uv, (o_ref, lse_ref) = expect[h]
        np.testing.assert_allclose(w_uv @ out[0, 0, h], o_ref, rtol=1e-10, atol=1e-12)
        assert abs(lse[0, 0, h] - lse_ref) <= 1e-10 * max(1.0, abs(lse_ref))


# ------------------------------------------------------------ closed forms
def test_single_key_returns_its_latent_row():
    wl = W.custom([1], num_heads=4, seed=3)
    out, lse = mla_decode_ref(wl.q_nope, wl.q_pe, wl.kv_cache, wl.page_table, wl.seq_lens, 1, wl.scale)
    row = oracle.bf16_bits_to_f64(wl.kv_cache[wl.page_table[0, 0], 0])
    for h in range(4):
        assert np.array_equal(out[0, 0, h], row[:512])
        q = np.concatenate([oracle.bf16_bits_to_f64(wl.q_nope[0, 0, h]), oracle.bf16_bits_to_f64(wl.q_pe[0, 0, h])])
        assert abs(lse[0, 0, h] - wl.scale * math.fsum(q * row)) < 1e-12


def test_zero_query_gives_mean_and_log_count():
    wl = W.custom([70, 129], num_heads=2, seed=4)
    zn = np.zeros_like(wl.q_nope)
    zp = np.zeros_like(wl.q_pe)
    out, lse = mla_decode_ref(zn, zp, wl.kv_cache, wl.page_table, wl.seq_lens, 1, wl.scale)
    for b in range(2):
        L = int(wl.seq_lens[b])
        rows = oracle.bf16_bits_to_f64(oracle.gather_rows(wl.kv_cache, wl.page_table[b], L))
        mean = np.array([math.fsum(rows[:, d]) / L for d in range(512)])
        np.testing.assert_allclose(out[b, 0, 0], mean, rtol=0, atol=1e-13)
        assert abs(lse[b, 0, 1] - math.log(L)) < 1e-13


def test_equal_scores_from_rope_only():
    """q_nope = 0 and every k_pe identical: all scores equal s, so the output
    is the mean latent row and lse = s + ln L."""
    wl = W.custom([91], num_heads=2, seed=6)
    cache = wl.kv_cache.copy()
    pe = W.f32_to_bf16_bits(np.linspace(-1, 1, 64).astype(np.float32))
    for p in range(cache.shape[0]):
        cache[p, :, 512:] = pe
    zn = np.zeros_like(wl.q_nope)
    out, lse = mla_decode_ref(zn, wl.q_pe, cache, wl.page_table, wl.seq_lens, 1, wl.scale)
    L = 91
    rows = oracle.bf16_bits_to_f64(oracle.gather_rows(cache, wl.page_table[0], L))
    mean = rows[:, :512].mean(axis=0)
    for h in range(2):
        s = wl.scale * math.fsum(oracle.bf16_bits_to_f64(wl.q_pe[0, 0, h]) * oracle.bf16_bits_to_f64(pe))
        np.testing.assert_allclose(out[0, 0, h], mean, rtol=0, atol=1e-13)
        assert abs(lse[0, 0, h] - (s + math.log(L))) < 1e-12


def _read_golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                k, v = line.split()
                vals[k] = float(v)
    return vals


def test_golden_two_token_logistic():
    g = _read_golden("two_token_logistic.txt")
    one, two = np.uint16(0x3F80), np.uint16(0x4000)
    qn = np.zeros((1, 1, 1, 512), dtype=np.uint16)
    qn[0, 0, 0, 0] = two
    qp = np.zeros((1, 1, 1, 64), dtype=np.uint16)
    cache = np.zeros((1, 64, 576), dtype=np.uint16)
    cache[0, 0, 1] = one  # token 0: c_kv = e_1
    cache[0, 1, 0] = one  # token 1: c_kv = e_0
    out, lse = mla_decode_ref(qn, qp, cache, np.zeros((1, 1), np.int32), np.array([2], np.int32), 1, 1.0)
    assert abs(out[0, 0, 0, 0] - g["out0"]) < 1e-15
    assert abs(out[0, 0, 0, 1] - g["out1"]) < 1e-15
    assert abs(lse[0, 0, 0] - g["lse"]) < 1e-15
    assert np.all(out[0, 0, 0, 2:] == 0)


# ------------------------------------------------------------ split / merge
@pytest.mark.parametrize("q_len", [1, 2])
def test_split_pieces_merge_to_unsplit(q_len):
    rng = np.random.default_rng(21)
    wl = W.custom([257, 64, 130, 1000], num_heads=4, q_len=q_len, seed=9)
    cuts = []
    for L in wl.seq_lens:
        L = int(L)
        k = int(rng.integers(0, min(6, L)))
        inner = sorted(set(rng.integers(1, L, size=k).tolist())) if L > 1 else []
        cuts.append([0] + inner + [L])
    cuts[0] = [0, 256, 257]  # a last piece holding one key only: row 0 of q_len=2 sees nothing there
    a = mla_decode_ref(wl.q_nope, wl.q_pe, wl.kv_cache, wl.page_table, wl.seq_lens, q_len, wl.scale)
    b = mla_decode_ref_pieces(wl.q_nope, wl.q_pe, wl.kv_cache, wl.page_table, wl.seq_lens, q_len, wl.scale, cuts)
    np.testing.assert_allclose(b[0], a[0], rtol=0, atol=1e-12)
    np.testing.assert_allclose(b[1], a[1], rtol=0, atol=1e-12)


def test_lse_merge_of_empty_piece_is_neutral():
    o = np.random.default_rng(1).standard_normal((2, 3, 512))
    l = np.array([[0.5, -1.0, 2.0], [-np.inf, -np.inf, -np.inf]])
    out, lse = lse_merge(o, l)
    np.testing.assert_array_equal(out, o[0])
    np.testing.assert_array_equal(lse, l[0])


# -------------------------------------------------------------- brute force
def _brute(qn, qp, cache, table, seq_lens, q_len, scale, kv_scale, kv_dtype):
    """Scalar loops, own gather, math.fsum, softmax without max subtraction."""
    dec = (lambda r: oracle.bf16_bits_to_f64(r)) if kv_dtype == "bf16" else \
        (lambda r: oracle.e4m3_to_f64(r) * kv_scale)
    B, Q, H, _ = qn.shape
    res = {}
    for b in range(B):
        L = int(seq_lens[b])
        keys = []
        for t in range(L):
            page = int(table[b][t // 64])
            keys.append(list(dec(cache[page, t % 64])))
        for i in range(Q):
            n = L - Q + i + 1
            for h in range(H):
                q = list(oracle.bf16_bits_to_f64(qn[b, i, h])) + list(oracle.bf16_bits_to_f64(qp[b, i, h]))
                s = [scale * math.fsum(q[d] * keys[t][d] for d in range(576)) for t in range(n)]
                e = [math.exp(x) for x in s]
                z = math.fsum(e)
                o = [math.fsum(e[t] * keys[t][d] for t in range(n)) / z for d in range(512)]
                res[(b, i, h)] = (o, math.log(z))
    return res


@pytest.mark.parametrize("q_len,kv_dtype", [(1, "bf16"), (2, "bf16"), (2, "fp8_e4m3")])
def test_brute_force_tiny(q_len, kv_dtype):
    wl = W.custom([5, 3], num_heads=2, q_len=q_len, seed=31, kv_dtype=kv_dtype)
    out, lse = mla_decode_ref(wl.q_nope, wl.q_pe, wl.kv_cache, wl.page_table, wl.seq_lens, q_len, wl.scale,
                              wl.kv_scale, kv_dtype)
    ref = _brute(wl.q_nope, wl.q_pe, wl.kv_cache, wl.page_table, wl.seq_lens, q_len, wl.scale, wl.kv_scale, kv_dtype)
    for (b, i, h), (o, l) in ref.items():
        np.testing.assert_allclose(out[b, i, h], o, rtol=1e-12, atol=1e-13)
        assert abs(lse[b, i, h] - l) < 1e-12


def test_fp8_path_equals_torch_decoded_values():
    torch = pytest.importorskip("torch")
    wl = W.custom([200, 77], num_heads=3, q_len=2, seed=41, kv_dtype="fp8_e4m3")
    out, lse = mla_decode_ref(wl.q_nope, wl.q_pe, wl.kv_cache, wl.page_table, wl.seq_lens, 2, wl.scale,
                              wl.kv_scale, "fp8_e4m3")
    for b in range(2):
        L = int(wl.seq_lens[b])
        raw = oracle.gather_rows(wl.kv_cache, wl.page_table[b], L)
        rows = torch.from_numpy(raw).view(torch.float8_e4m3fn).to(torch.float64).numpy() * wl.kv_scale
        q = np.concatenate([oracle.bf16_bits_to_f64(wl.q_nope[b]), oracle.bf16_bits_to_f64(wl.q_pe[b])], -1)
        o, l = attend(q.reshape(-1, 576), rows, np.repeat([L - 1, L], 3), wl.scale)
        np.testing.assert_array_equal(o.reshape(2, 3, 512), out[b])
        np.testing.assert_array_equal(l.reshape(2, 3), lse[b])


# ------------------------------------------------------------------ causal
def test_causal_rows_equal_single_position_calls():
    wl = W.custom([300, 65, 2], num_heads=3, q_len=2, seed=12)
    out2, lse2 = mla_decode_ref(wl.q_nope, wl.q_pe, wl.kv_cache, wl.page_table, wl.seq_lens, 2, wl.scale)
    for i, shift in ((1, 0), (0, 1)):
        qn = np.ascontiguousarray(wl.q_nope[:, i : i + 1])
        qp = np.ascontiguousarray(wl.q_pe[:, i : i + 1])
        o1, l1 = mla_decode_ref(qn, qp, wl.kv_cache, wl.page_table, wl.seq_lens - shift, 1, wl.scale)
        np.testing.assert_allclose(out2[:, i], o1[:, 0], rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse2[:, i], l1[:, 0], rtol=0, atol=1e-12)


# ------------------------------------------------------------ invariances
def test_page_relabelling_is_invisible():
    wl = W.custom([100, 257, 64], num_heads=2, seed=13)
    wl2 = W.relabel_pages(wl, seed=99)
    assert not np.array_equal(wl.page_table, wl2.page_table)
    a = mla_decode_ref(wl.q_nope, wl.q_pe, wl.kv_cache, wl.page_table, wl.seq_lens, 1, wl.scale)
    b = mla_decode_ref(wl2.q_nope, wl2.q_pe, wl2.kv_cache, wl2.page_table, wl2.seq_lens, 1, wl2.scale)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


def test_prefix_share_equals_prefix_copy():
    wl = W.prefix_shaped(batch=3, num_heads=2, prefix_pages=3, suffix_range=(10, 100), seed=14)
    wc = W.copy_shared_prefix(wl)
    assert wc.num_pages == wl.num_pages + 2 * 3
    a = mla_decode_ref(wl.q_nope, wl.q_pe, wl.kv_cache, wl.page_table, wl.seq_lens, 1, wl.scale)
    b = mla_decode_ref(wc.q_nope, wc.q_pe, wc.kv_cache, wc.page_table, wc.seq_lens, 1, wc.scale)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8_e4m3"])
def test_tail_sentinels_do_not_leak(kv_dtype):
    res = []
    for sentinel in ("nan", "big", "zero"):
        wl = W.custom([100, 1, 63], num_heads=2, q_len=1, seed=15, kv_dtype=kv_dtype, sentinel=sentinel)
        res.append(mla_decode_ref(wl.q_nope, wl.q_pe, wl.kv_cache, wl.page_table, wl.seq_lens, 1, wl.scale,
                                  wl.kv_scale, kv_dtype))
    for r in res[1:]:
        np.testing.assert_array_equal(r[0], res[0][0])
        np.testing.assert_array_equal(r[1], res[0][1])
    assert np.all(np.isfinite(res[0][0]))


# ----------------------------------------------------------------- errors
def test_bad_page_id_and_length_are_errors():
    wl = W.custom([100], num_heads=1, seed=16)
    bad = wl.page_table.copy()
    bad[0, 1] = wl.num_pages
    with pytest.raises(IndexError):
        mla_decode_ref(wl.q_nope, wl.q_pe, wl.kv_cache, bad, wl.seq_lens, 1, wl.scale)
    with pytest.raises(ValueError):
        mla_decode_ref(wl.q_nope, wl.q_pe, wl.kv_cache, wl.page_table, np.array([64 * wl.max_pages + 1]), 1,
                       wl.scale)
    with pytest.raises(ValueError):
        mla_decode_ref(wl.q_nope, wl.q_pe, wl.kv_cache, wl.page_table, np.array([0]), 1, wl.scale)


# ------------------------------------------------------------- workloads
def test_named_workload_shapes_small():
    wl = W.make_config("tiny")
    assert wl.batch == 2 and wl.num_heads == 16 and wl.num_pages == 16
    assert list(wl.seq_lens) == [100, 257]
    used = set(wl.page_table[0, :2]) | set(wl.page_table[1, :5])
    assert len(used) == 7 and all(0 <= p < 16 for p in used)
    assert abs(wl.scale - 1 / math.sqrt(192)) < 1e-15


# ------------------------------------------------------------ top-k decode
def _sparse_case(kv_dtype="bf16", q_len=2):
    wl = W.custom([130, 70, 300], num_heads=8, q_len=q_len, kv_dtype=kv_dtype, seed=61)
    return wl


def test_sparse_with_every_visible_position_is_the_dense_decode():
    wl = _sparse_case()
    idx = np.full((wl.batch, wl.q_len, 320), -1, dtype=np.int32)
    for b in range(wl.batch):
        for i in range(wl.q_len):
            n = int(wl.seq_lens[b]) - wl.q_len + i + 1
            idx[b, i, :n] = np.arange(n)
    o, l, st = oracle.mla_decode_sparse_ref(wl.q_nope, wl.q_pe, wl.kv_cache, wl.page_table, wl.seq_lens, wl.q_len,
                                            idx, wl.scale)
    ro, rl = mla_decode_ref(wl.q_nope, wl.q_pe, wl.kv_cache, wl.page_table, wl.seq_lens, wl.q_len, wl.scale)
    assert st == 0
    assert np.allclose(o, ro, rtol=0, atol=1e-12) and np.allclose(l, rl, rtol=0, atol=1e-12)


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8_e4m3"])
def test_sparse_equals_dense_over_a_cache_of_the_picked_rows(kv_dtype):
    """Copy the picked rows (in list order) into a fresh paged cache and run
    the dense decode over it: same result (position i sees all its picks)."""
    wl = _sparse_case(kv_dtype, q_len=1)
    idx = W.topk_indices(wl, 90, seed=4)
    o, l, st = oracle.mla_decode_sparse_ref(wl.q_nope, wl.q_pe, wl.kv_cache, wl.page_table, wl.seq_lens, 1, idx,
                                            wl.scale, wl.kv_scale, kv_dtype)
    assert st == 0
    for b in range(wl.batch):
        picks = [int(t) for t in idx[b, 0] if t >= 0]
        rows = np.stack([wl.kv_cache[wl.page_table[b, t // 64], t % 64] for t in picks])
        npg = (len(picks) + 63) // 64
        cache = np.zeros((npg, 64, 576), dtype=wl.kv_cache.dtype)
        cache.reshape(-1, 576)[:len(picks)] = rows
        table = np.arange(npg, dtype=np.int32)[None, :]
        ro, rl = mla_decode_ref(wl.q_nope[b:b + 1], wl.q_pe[b:b + 1], cache, table,
                                np.array([len(picks)], dtype=np.int32), 1, wl.scale, wl.kv_scale, kv_dtype)
        assert np.allclose(o[b], ro[0], rtol=0, atol=1e-12) and np.allclose(l[b], rl[0], rtol=0, atol=1e-12)


def test_sparse_closed_forms_single_and_repeated_pick():
    wl = _sparse_case(q_len=1)
    t = 45
    one = np.array([[[t, -1, -1]]] * wl.batch, dtype=np.int32)
    two = np.array([[[t, t, -1]]] * wl.batch, dtype=np.int32)
    o1, l1, s1 = oracle.mla_decode_sparse_ref(wl.q_nope, wl.q_pe, wl.kv_cache, wl.page_table, wl.seq_lens, 1, one,
                                              wl.scale)
    o2, l2, s2 = oracle.mla_decode_sparse_ref(wl.q_nope, wl.q_pe, wl.kv_cache, wl.page_table, wl.seq_lens, 1, two,
                                              wl.scale)
    assert s1 == s2 == 0
    for b in range(wl.batch):
        row = oracle.bf16_bits_to_f64(wl.kv_cache[wl.page_table[b, 0], t])[:512]
        assert np.array_equal(o1[b, 0], np.broadcast_to(row, o1[b, 0].shape))  # one key: its latent row
    assert np.allclose(o2, o1, rtol=0, atol=1e-15)
    assert np.allclose(l2, l1 + math.log(2.0), rtol=0, atol=1e-12)  # twice the same key: lse + ln 2


def test_sparse_pick_order_does_not_matter():
    wl = _sparse_case()
    idx = W.topk_indices(wl, 50, seed=8)
    rev = idx[:, :, ::-1].copy()
    a = oracle.mla_decode_sparse_ref(wl.q_nope, wl.q_pe, wl.kv_cache, wl.page_table, wl.seq_lens, 2, idx, wl.scale)
    b = oracle.mla_decode_sparse_ref(wl.q_nope, wl.q_pe, wl.kv_cache, wl.page_table, wl.seq_lens, 2, rev, wl.scale)
    assert np.allclose(a[0], b[0], rtol=0, atol=1e-12) and np.allclose(a[1], b[1], rtol=0, atol=1e-12)


def test_sparse_bad_entries_are_flagged_and_skipped():
    wl = _sparse_case(q_len=2)
    idx = np.array([[[0, 5, 129, 128, -1], [0, 5, 129, -7, -1]]] * wl.batch, dtype=np.int32)
    # request 0 has L=130: draft 0 sees 0..128, draft 1 sees 0..129
    ok = np.array([[[0, 5, 128, -1, -1], [0, 5, 129, -1, -1]]] * wl.batch, dtype=np.int32)
    a = oracle.mla_decode_sparse_ref(wl.q_nope, wl.q_pe, wl.kv_cache, wl.page_table, wl.seq_lens, 2, idx, wl.scale,
                                     requests=[0])
    b = oracle.mla_decode_sparse_ref(wl.q_nope, wl.q_pe, wl.kv_cache, wl.page_table, wl.seq_lens, 2, ok, wl.scale,
                                     requests=[0])
    assert a[2] == oracle.sparse.BAD_INDEX and b[2] == 0
    assert np.allclose(a[0][0], b[0][0], rtol=0, atol=1e-15)
    empty = np.full((wl.batch, 2, 3), -1, dtype=np.int32)
    o, l, st = oracle.mla_decode_sparse_ref(wl.q_nope, wl.q_pe, wl.kv_cache, wl.page_table, wl.seq_lens, 2, empty,
                                            wl.scale, requests=[1])
    assert st == oracle.sparse.BAD_INDEX and np.all(o[1] == 0) and np.all(l[1] == -np.inf)
    # merged with any piece by log-sum-exp, the empty list's result is neutral
    rng = np.random.default_rng(4)
    po, pl = rng.standard_normal(o[1].shape), rng.standard_normal(l[1].shape)
    mo, ml = oracle.lse_merge(np.stack([o[1], po]), np.stack([l[1], pl]))
    assert np.array_equal(mo, po) and np.array_equal(ml, pl)


# ------------------------------------------------- properties (hypothesis)
# Randomised statements of the same mathematics: any partition of the keys
# merges back to the unsplit result; the merge is order-free; a rope term
# that scores every key alike moves lse and leaves out alone.

def _hyp():
    return pytest.importorskip("hypothesis")


def test_property_any_partition_merges_to_unsplit():
    hyp = _hyp()
    st = hyp.strategies

    @hyp.settings(max_examples=25, deadline=None, derandomize=True)
    @hyp.given(L=st.integers(1, 200), Q=st.integers(1, 3), H=st.integers(1, 3), data=st.data())
    def check(L, Q, H, data):
        L = max(L, Q)
        wl = W.custom([L], num_heads=H, q_len=Q, seed=L * 7 + Q * 3 + H)
        inner = data.draw(st.lists(st.integers(1, L - 1), max_size=6, unique=True)) if L > 1 else []
        cuts = [[0] + sorted(inner) + [L]]
        a = mla_decode_ref(wl.q_nope, wl.q_pe, wl.kv_cache, wl.page_table, wl.seq_lens, Q, wl.scale)
        b = mla_decode_ref_pieces(wl.q_nope, wl.q_pe, wl.kv_cache, wl.page_table, wl.seq_lens, Q, wl.scale, cuts)
        np.testing.assert_allclose(b[0], a[0], rtol=0, atol=1e-12)
        np.testing.assert_allclose(b[1], a[1], rtol=0, atol=1e-12)

    check()


def test_property_lse_merge_is_order_free_and_associative():
    hyp = _hyp()
    st = hyp.strategies

    @hyp.settings(max_examples=50, deadline=None, derandomize=True)
    @hyp.given(seed=st.integers(0, 10**6), n=st.integers(2, 5), empty=st.integers(-1, 4))
    def check(seed, n, empty):
        rng = np.random.default_rng(seed)
        outs = rng.standard_normal((n, 3, 8))
        lses = rng.uniform(-30, 30, size=(n, 3))
        if 0 <= empty < n:
            lses[empty] = -np.inf
            outs[empty] = 0.0
        o, l = lse_merge(outs, lses)
        perm = rng.permutation(n)
        op, lp = lse_merge(outs[perm], lses[perm])
        np.testing.assert_allclose(op, o, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(lp, l, rtol=1e-12, atol=1e-12)
        k = n // 2  # merge the first k, then the rest
        with np.errstate(divide="ignore"):  # a half holding only the empty piece merges to lse = -inf
            o1, l1 = lse_merge(outs[:k], lses[:k])
            o2, l2 = lse_merge(outs[k:], lses[k:])
        oc, lc = lse_merge(np.stack([o1, o2]), np.stack([l1, l2]))
        np.testing.assert_allclose(oc, o, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(lc, l, rtol=1e-12, atol=1e-12)

    check()


def test_property_uniform_rope_term_shifts_lse_only():
    hyp = _hyp()
    st = hyp.strategies

    @hyp.settings(max_examples=15, deadline=None, derandomize=True)
    @hyp.given(L=st.integers(1, 150), H=st.integers(1, 4), seed=st.integers(0, 1000))
    def check(L, H, seed):
        wl = W.custom([L], num_heads=H, q_len=1, seed=seed)
        cache = wl.kv_cache.copy()
        k_pe = cache[wl.page_table[0, 0], 0, 512:].copy()
        for j in range((L + 63) // 64):  # every visible key gets the same k_pe
            cache[wl.page_table[0, j], :, 512:] = k_pe
        zero_pe = np.zeros_like(wl.q_pe)  # bf16 bits of +0.0
        a_out, a_lse = mla_decode_ref(wl.q_nope, wl.q_pe, cache, wl.page_table, wl.seq_lens, 1, wl.scale)
        b_out, b_lse = mla_decode_ref(wl.q_nope, zero_pe, cache, wl.page_table, wl.seq_lens, 1, wl.scale)
        shift = wl.scale * (oracle.bf16_bits_to_f64(wl.q_pe[0, 0]) @ oracle.bf16_bits_to_f64(k_pe))  # [H]
        np.testing.assert_allclose(a_out, b_out, rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(a_lse[0, 0], b_lse[0, 0] + shift, rtol=1e-12, atol=1e-10)

    check()


def test_property_e4m3_encoder_is_monotone():
    hyp = _hyp()
    st = hyp.strategies

    @hyp.settings(max_examples=40, deadline=None, derandomize=True)
    @hyp.given(xs=st.lists(st.floats(-600, 600, allow_nan=False, width=32), min_size=2, max_size=64))
    def check(xs):
        x = np.sort(np.asarray(xs, dtype=np.float32))
        v = oracle.e4m3_to_f64(oracle.e4m3_encode(x))
        assert np.all(np.diff(v) >= 0)
        assert np.all(np.abs(v) <= 448)

    check()


def test_kv_pack_quantises_the_exact_quotient():
    """The tag page's quantisation article quantises a value as round(value /
    scale).  On inputs where that exact quotient and the fp32 product with
    the scale's reciprocal round to different e4m3 codes, the oracle writes
    the code of the exact quotient (checked with rational arithmetic against
    torch's e4m3 values), and so tells the two readings apart."""
    from fractions import Fraction

    from kvpack_cases import bits_to_float, distinguishing_cases, e4m3_values, nearest_code

    pytest.importorskip("torch")
    mags = e4m3_values()
    cases = distinguishing_cases(8)
    for xb, s in cases:
        x = bits_to_float(xb)
        for sign_bits in (xb, xb ^ np.uint16(0x8000)):
            xv = bits_to_float(sign_bits)
            rows = np.full((1, 1, 576), sign_bits, dtype=np.uint16)
            table = np.array([[0]], dtype=np.int32)
            out, status = oracle.kv_pack_ref(rows, table, np.array([1], dtype=np.int32), s,
                                             np.zeros((1, 64, 576), dtype=np.uint8), "fp8_e4m3")
            assert status == 0
            exact = nearest_code(Fraction(xv) / Fraction(s), mags)
            prod = np.float32(np.float32(xv) * (np.float32(1.0) / np.float32(s)))
            assert out[0, 0, 0] == exact != nearest_code(Fraction(float(prod)), mags), (x, s)
    # an exact midpoint (power-of-two scale) goes to the even code both ways
    rows = np.full((1, 1, 576), np.uint16(0x4008), dtype=np.uint16)  # 2.125 = 2 * 1.0625
    out, _ = oracle.kv_pack_ref(rows, np.array([[0]], dtype=np.int32), np.array([1], dtype=np.int32), 2.0,
                                np.zeros((1, 64, 576), dtype=np.uint8), "fp8_e4m3")
    assert out[0, 0, 0] == 0x38  # 1.0625 lies between 1.0 (0x38, even) and 1.125 (0x39)
