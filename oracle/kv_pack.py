"""Quantise-and-scatter of a step's new cache rows (test infrastructure).

Source: TokenSpeed code audit (mlqm.cn/news/403565), section 完整技术清单 >
Attention 接入 / KV: a fused FP8 KV-pack kernel quantises the new tokens'
rows and writes them into the paged cache through the page table.  The
cache layout and the position of new tokens follow the decode: a sequence
of length L holds its tokens at positions 0 .. L - 1, position t in slot
t % 64 of page page_table[b][t // 64], and the step's num_new new tokens
are the last num_new positions (they are already counted in L).

The quantisation itself follows the guijiagi.com "推理优化" tag page,
quantisation article (三大量化方案原理 > INT8量化): a value is quantised as
round(value / scale) and dequantised as scale * code.  Here the grid is
e4m3's, so the code is the e4m3 value nearest to x / kv_scale (ties to the
even code, saturated to +-448; see e4m3.e4m3_encode), kv_scale taken as the
fp32 number the C entry point receives.  x / kv_scale is formed in float64:
x has 8 significant bits, kv_scale 24 and an e4m3 midpoint 5, so x / kv_scale
is either exactly a midpoint or at least 2**-38 of it away (relative), far
beyond float64's 2**-53 rounding; the float64 quotient therefore rounds to
the same code as the exact quotient.

Readings where the pages are silent:

* a bf16 cache receives the row unchanged;
* a row whose page id is outside the pool, or whose sequence length is
  outside [num_new, max_pages * 64], is not written and raises a flag
  (1 = bad page id, 2 = bad length), as the decode reports them.

Plain loops over rows; nothing here is shared with the CUDA library.
"""
from __future__ import annotations

import numpy as np

from .e4m3 import e4m3_encode

BAD_PAGE_ID = 1
BAD_SEQ_LEN = 2


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) to the float32 values they denote."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def quantise_e4m3(rows_bits: np.ndarray, kv_scale: float) -> np.ndarray:
    """e4m3 codes of bf16 values (uint16 bits, any shape): the code nearest to
    x / kv_scale, kv_scale taken as an fp32 number."""
    x = bf16_bits_to_f32(rows_bits).astype(np.float64)
    return e4m3_encode(x / np.float64(np.float32(kv_scale)))


def kv_pack_ref(rows_bits: np.ndarray, page_table: np.ndarray, seq_lens: np.ndarray, kv_scale: float,
                kv_cache: np.ndarray, kv_dtype: str, page_size: int = 64):
    """Returns (new cache, status flags).  rows_bits: uint16 [B, num_new, 576]
    (bf16 bits); kv_cache: uint8 [P, 64, 576] (e4m3) or uint16 (bf16 bits);
    the input cache is not modified."""
    rows_bits = np.asarray(rows_bits, dtype=np.uint16)
    B, n_new, width = rows_bits.shape
    if width != 576:
        raise ValueError("a cache row has 576 values")
    cache = np.array(kv_cache, copy=True)
    num_pages, max_pages = cache.shape[0], page_table.shape[1]
    status = 0
    for b in range(B):
        L = int(seq_lens[b])
        if L < n_new or L > max_pages * page_size:
            status |= BAD_SEQ_LEN
            continue
        for i in range(n_new):
            t = L - n_new + i
            page = int(page_table[b, t // page_size])
            if page < 0 or page >= num_pages:
                status |= BAD_PAGE_ID
                continue
            if kv_dtype == "bf16":
                cache[page, t % page_size] = rows_bits[b, i]
            elif kv_dtype == "fp8_e4m3":
                cache[page, t % page_size] = quantise_e4m3(rows_bits[b, i], kv_scale)
            else:
                raise ValueError(kv_dtype)
    return cache, status
