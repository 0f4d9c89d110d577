"""Plain float64 MLA decode over a paged latent cache (test infrastructure).

This is the definition of the operation, written out with numpy and no
blocking, fusion or reordering beyond a matrix product per request.  It is
what the CUDA path must reproduce.

Sources (page title and section):

* TokenSpeed code audit (mlqm.cn/news/403565), section 完整技术清单 > MLA:
  every cached token is ONE latent row of 512 latent values followed by 64
  RoPE values; that single row serves both as the key (all 576 values) and
  as the value (the 512 latent values) through a transposed view.
* Same section: decode may be split over the keys; split results are merged
  by rescaling with their log-sum-exp (see :func:`lse_merge`).
* guijiagi.com "推理优化" tag page, FlashAttention article: tiled attention
  reaches exactly the result of plain attention, so the oracle is plain
  attention (a stable softmax over all visible keys).
* Same tag page, KV-cache article (PagedAttention): the cache is cut into
  fixed-size blocks addressed through a per-request page table.

Readings where the pages are silent:

* the log-sum-exp is the natural log of sum(exp(score)), score including the
  softmax scale;
* ``seq_lens[b]`` counts the ``q_len`` new tokens, already in the cache;
  query position i sees keys 0 .. L_b - q_len + i (causal between drafts);
* the FP8 cache value is e4m3(code) * kv_scale for both the latent and the
  RoPE part; queries are never scaled;
* row order inside a cached token: [c_kv (512) | k_pe (64)];
* cache slots past L_b and unreferenced pages may hold any bits; they must
  not influence the result;
* a page id outside [0, num_pages) or L_b outside [q_len, pages*page_size]
  is an error.

Parity: pinned by tests/test_oracle_pins.py (non-absorbed attention,
closed forms, split/merge identity, pure-Python brute force).
"""
from __future__ import annotations

import numpy as np

from .e4m3 import e4m3_to_f64

D_LATENT = 512
D_ROPE = 64
D_ROW = D_LATENT + D_ROPE


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """bfloat16 bit patterns (uint16) -> float64: bf16 is the top half of a float32."""
    bits = np.asarray(bits)
    if bits.dtype != np.uint16:
        raise TypeError("bf16 data must be given as uint16 bit patterns")
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def decode_cache_rows(raw_rows: np.ndarray, kv_dtype: str, kv_scale: float) -> np.ndarray:
    """Raw cache rows -> float64 values.

    bf16: the stored value itself.  fp8_e4m3: e4m3(code) * kv_scale.
    """
    if kv_dtype == "bf16":
        return bf16_bits_to_f64(raw_rows)
    if kv_dtype == "fp8_e4m3":
        return e4m3_to_f64(raw_rows) * np.float64(kv_scale)
    raise ValueError(f"unknown kv dtype {kv_dtype!r}")


def visible_keys(seq_len: int, q_len: int, i: int) -> int:
    """Number of keys that query position i of a request sees (causal drafts)."""
    return seq_len - q_len + i + 1


def gather_rows(kv_cache: np.ndarray, page_table_row: np.ndarray, n: int, page_size: int = 64) -> np.ndarray:
    """Raw cache rows of tokens 0..n-1 of one request, in token order.

    Token t lives in page page_table_row[t // page_size], slot t % page_size.
    Pages shared between requests are simply the same ids in several rows of
    the page table: they are read in place.
    """
    num_pages = kv_cache.shape[0]
    out = np.empty((n, kv_cache.shape[2]), dtype=kv_cache.dtype)
    for t in range(0, n, page_size):
        pid = int(page_table_row[t // page_size])
        if not 0 <= pid < num_pages:
            raise IndexError(f"page id {pid} outside the pool of {num_pages} pages")
        cnt = min(page_size, n - t)
        out[t : t + cnt] = kv_cache[pid, :cnt]
    return out


def _check(q_nope, q_pe, kv_cache, page_table, seq_lens, q_len, page_size):
    B, Q, H, dn = q_nope.shape
    if Q != q_len:
        raise ValueError("q_nope's second axis must equal q_len")
    if dn != D_LATENT or q_pe.shape != (B, Q, H, D_ROPE):
        raise ValueError("queries must be [B, q_len, H, 512] and [B, q_len, H, 64]")
    if kv_cache.ndim != 3 or kv_cache.shape[1] != page_size or kv_cache.shape[2] != D_ROW:
        raise ValueError("cache must be [num_pages, page_size, 576]")
    if len(seq_lens) != B or page_table.shape[0] != B:
        raise ValueError("seq_lens and page_table must have one entry/row per request")
    max_pages = page_table.shape[1]
    for b in range(B):
        L = int(seq_lens[b])
        if L < q_len or L > max_pages * page_size:
            raise ValueError(f"seq_lens[{b}]={L} outside [q_len, max_pages*page_size]")
    return B, Q, H


def attend(qrows: np.ndarray, rows: np.ndarray, nvis, scale: float):
    """Plain softmax attention of R absorbed query rows over latent rows.

    ``qrows`` float64 [R, 576] (q_nope | q_pe), ``rows`` float64 [n, 576]
    (c_kv | k_pe), ``nvis[r]`` = number of leading rows query r sees.
    Returns out [R, 512] and natural-log lse [R].  A query that sees no row
    gets out = 0 and lse = -inf.
    """
    R = qrows.shape[0]
    nvis = np.broadcast_to(np.asarray(nvis), (R,))
    scores = (qrows @ rows.T) * scale  # [R, n]
    out = np.zeros((R, D_LATENT))
    lse = np.full(R, -np.inf)
    for n in np.unique(nvis):
        n = int(n)
        if n <= 0:
            continue
        sel = np.nonzero(nvis == n)[0]
        s = scores[sel, :n]
        m = s.max(axis=1, keepdims=True)
        w = np.exp(s - m)
        z = w.sum(axis=1, keepdims=True)
        out[sel] = (w / z) @ rows[:n, :D_LATENT]
        lse[sel] = (m + np.log(z))[:, 0]
    return out, lse


def mla_decode_ref(
    q_nope: np.ndarray,
    q_pe: np.ndarray,
    kv_cache: np.ndarray,
    page_table: np.ndarray,
    seq_lens: np.ndarray,
    q_len: int,
    scale: float,
    kv_scale: float = 1.0,
    kv_dtype: str = "bf16",
    page_size: int = 64,
    requests=None,
):
    """Absorbed MLA decode, float64.

    Arguments follow the C entry point: ``q_nope`` uint16 bf16 bits
    [B, q_len, H, 512], ``q_pe`` [B, q_len, H, 64]; ``kv_cache`` uint16
    (bf16) or uint8 (e4m3) [num_pages, page_size, 576]; ``page_table``
    int [B, max_pages]; ``seq_lens`` int [B].

    For request b, query position i and head h, with n visible keys::

        s_t  = (q_nope . c_kv[t] + q_pe . k_pe[t]) * scale
        out  = sum_t softmax(s)_t * c_kv[t]        (512-d latent)
        lse  = log(sum_t exp(s_t))                 (natural log)

    ``requests`` optionally restricts the work to a subset of requests
    (used for sampled checks at full size); other rows are left NaN.
    Returns (out float64 [B, q_len, H, 512], lse float64 [B, q_len, H]).
    """
    B, Q, H = _check(q_nope, q_pe, kv_cache, page_table, seq_lens, q_len, page_size)
    out = np.full((B, Q, H, D_LATENT), np.nan)
    lse = np.full((B, Q, H), np.nan)
    todo = range(B) if requests is None else requests
    for b in todo:
        L = int(seq_lens[b])
        rows = decode_cache_rows(gather_rows(kv_cache, page_table[b], L, page_size), kv_dtype, kv_scale)
        qrows = np.concatenate([bf16_bits_to_f64(q_nope[b]), bf16_bits_to_f64(q_pe[b])], axis=-1)
        nvis = np.repeat([visible_keys(L, Q, i) for i in range(Q)], H)
        o, l = attend(qrows.reshape(Q * H, D_ROW), rows, nvis, scale)
        out[b] = o.reshape(Q, H, D_LATENT)
        lse[b] = l.reshape(Q, H)
    return out, lse


def lse_merge(outs: np.ndarray, lses: np.ndarray):
    """Merge partial attention results computed over disjoint key sets.

    ``outs`` [S, ..., D] are the softmax-normalised partial outputs and
    ``lses`` [S, ...] their log-sum-exps; an empty part has lse = -inf and
    contributes nothing.  The merged result is
    lse = log(sum_s exp(lse_s)), out = sum_s exp(lse_s - lse) * out_s.
    """
    outs = np.asarray(outs, dtype=np.float64)
    lses = np.asarray(lses, dtype=np.float64)
    m = np.max(lses, axis=0)
    safe_m = np.where(np.isfinite(m), m, 0.0)
    w = np.exp(lses - safe_m)  # exp(-inf) = 0 for empty parts
    z = w.sum(axis=0)
    lse = safe_m + np.log(z)
    wn = w / np.where(z > 0, z, 1.0)
    out = np.einsum("s...,s...d->...d", wn, outs)
    return out, lse


def mla_decode_ref_pieces(
    q_nope,
    q_pe,
    kv_cache,
    page_table,
    seq_lens,
    q_len,
    scale,
    cuts,
    kv_scale: float = 1.0,
    kv_dtype: str = "bf16",
    page_size: int = 64,
):
    """The same decode computed as independent pieces over key ranges.

    ``cuts[b]`` is a sorted list of token positions 0 = c_0 < ... < c_k = L_b
    that partitions request b's keys.  Each piece [c_j, c_{j+1}) is decoded
    on its own (rows that see no key of the piece get lse = -inf and a zero
    output) and the pieces are merged with :func:`lse_merge`.  This is the
    split-KV decomposition the pages describe; mathematically it equals
    :func:`mla_decode_ref`.
    """
    B, Q, H = _check(q_nope, q_pe, kv_cache, page_table, seq_lens, q_len, page_size)
    out = np.empty((B, Q, H, D_LATENT))
    lse = np.empty((B, Q, H))
    for b in range(B):
        L = int(seq_lens[b])
        c = list(cuts[b])
        if c[0] != 0 or c[-1] != L or any(x >= y for x, y in zip(c, c[1:])):
            raise ValueError("cuts must increase strictly from 0 to L_b")
        rows = decode_cache_rows(gather_rows(kv_cache, page_table[b], L, page_size), kv_dtype, kv_scale)
        qrows = np.concatenate([bf16_bits_to_f64(q_nope[b]), bf16_bits_to_f64(q_pe[b])], axis=-1)
        qrows = qrows.reshape(Q * H, D_ROW)
        nvis = np.repeat([visible_keys(L, Q, i) for i in range(Q)], H)
        p_out = np.zeros((len(c) - 1, Q * H, D_LATENT))
        p_lse = np.full((len(c) - 1, Q * H), -np.inf)
        for j, (lo, hi) in enumerate(zip(c, c[1:])):
            # keys lo..hi-1 only: a query sees min(hi, nvis) - lo of them
            p_out[j], p_lse[j] = attend(qrows, rows[lo:hi], np.minimum(hi, nvis) - lo, scale)
        o, l = lse_merge(p_out, p_lse)
        out[b] = o.reshape(Q, H, D_LATENT)
        lse[b] = l.reshape(Q, H)
    return out, lse
