"""Top-k sparse decode, float64 (test infrastructure).

Source: TokenSpeed code audit (mlqm.cn/news/403565), section 完整技术清单 >
Attention 接入 / KV: DeepSeek sparse attention, where an indexer picks the
top-k latent rows and the decode attends to those only.  The indexer is
not part of this operation; its output (token positions per request and
draft position) is an input.  The attention over the picked rows is the
plain decode of mla_oracle (softmax over the picked keys only).

Readings where the pages are silent:

* an entry t is used when 0 <= t < n, n = seq_len - q_len + i + 1 (the
  causal visibility of draft i); -1 means unused; any other entry is
  skipped and flagged (BAD_INDEX);
* a position listed twice counts twice (the list is a multiset);
* a (request, draft) with no used entry is flagged and gets lse = -inf
  (the natural log of an empty sum) and out = 0: the value of an empty key
  set under which it drops out of the log-sum-exp merge of split pieces
  (the same audit section's split-KV merge), as for a query that sees no
  key in mla_oracle.attend.
"""
from __future__ import annotations

import numpy as np

from .mla_oracle import D_LATENT, D_ROW, attend, bf16_bits_to_f64, decode_cache_rows, visible_keys

BAD_INDEX = 16


def mla_decode_sparse_ref(q_nope, q_pe, kv_cache, page_table, seq_lens, q_len, indices, scale, kv_scale=1.0,
                          kv_dtype="bf16", page_size=64, requests=None):
    """Returns (out float64 [B, q_len, H, 512], lse float64 [B, q_len, H],
    status).  ``indices`` int [B, q_len, topk]; other arguments as for
    mla_oracle.mla_decode_ref.  Requests not in ``requests`` stay NaN."""
    B, Q, H, _ = q_nope.shape
    out = np.full((B, Q, H, D_LATENT), np.nan)
    lse = np.full((B, Q, H), np.nan)
    status = 0
    todo = range(B) if requests is None else requests
    for b in todo:
        L = int(seq_lens[b])
        for i in range(Q):
            n = visible_keys(L, Q, i)
            used = []
            for t in indices[b, i]:
                t = int(t)
                if 0 <= t < n:
                    used.append(t)
                elif t != -1:
                    status |= BAD_INDEX
            if used:
                raw = np.stack([kv_cache[int(page_table[b, t // page_size]), t % page_size] for t in used])
                rows = decode_cache_rows(raw, kv_dtype, kv_scale)
            else:
                status |= BAD_INDEX
                rows = np.zeros((0, D_ROW))
            qrows = np.concatenate([bf16_bits_to_f64(q_nope[b, i]), bf16_bits_to_f64(q_pe[b, i])], axis=-1)
            o, l = attend(qrows, rows, rows.shape[0], scale)  # no rows: out = 0, lse = -inf
            out[b, i], lse[b, i] = o, l
    return out, lse, status
