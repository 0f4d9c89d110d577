"""Seeded synthetic decode batches for paged MLA.

This module only builds INPUTS: shapes, seeded N(0,1) values rounded to the
storage type, page tables and sequence lengths.  It holds none of the
attention arithmetic, so both the CUDA path and the CPU oracle can be fed
from it without sharing any of the method.

The five named shapes follow the decode workloads of the TokenSpeed pages
(latent 512 + RoPE 64 per cached token, 64-token pages, long agentic
contexts, prefix reuse, speculative verification with two draft tokens):

=========  ====  ====  ==  =================================================
name       B     H     Q   sequence lengths / cache
=========  ====  ====  ==  =================================================
tiny       2     16    1   {100, 257}; 16-page pool
kimi       64    64    1   8192 each; pool sized to the batch
dsv3       128   128   1   floor(exp(U(ln 1024, ln 32768))); split-KV needed
prefix     32    64    1   768 shared prefix pages + U{1024..4096} private
fp8        256   128   2   U{4096..16384}; E4M3 cache, one fp32 scale
verify4    64    64    4   8192 each: kimi's shape verifying 3 draft tokens
dsa        64    128   1   16384 each; top-k decode over 2048 picked rows
=========  ====  ====  ==  =================================================

``dsa`` is a DeepSeek-V3.2-shaped batch for the top-k (sparse) decode: its
picked positions come from ``topk_indices``: for every (request, draft
position) a seeded random subset of the visible positions of size
min(topk, visible), in random order, padded with -1.

The cache write before a step (quantise-and-scatter of the new rows) is
measured on its own batch, ``kv_pack_batch()``: 64 requests whose 4096-token
prompts are all new (a Kimi-shaped prefill), N(0,1) bf16 rows written into
an e4m3 cache of 4096 pages through a seeded page permutation, kv_scale =
max|x| / 448 over the rows.

Recipe (all integers drawn from one ``numpy.random.Generator(PCG64(seed))``
in this order: sequence lengths, page permutation, q_nope, q_pe):

* page ids are a seeded permutation of the pool, handed out request by
  request in token order (the prefix pages first for ``prefix``);
* q and cache values are N(0,1) float32 rounded to nearest-even bf16;
  cache values come from per-chunk streams ``SeedSequence(seed).spawn``
  (chunks of 256 pages) so generation can run in parallel and still be
  reproducible;
* for the E4M3 cache, kv_scale = max|x| / 448 over the referenced values
  and the codes are torch's round-to-nearest float8_e4m3fn conversion of
  x / kv_scale (never above 448, so never NaN);
* cache slots past a request's length and pages no request references are
  filled with a sentinel (NaN by default) that must never reach a result;
* unused page-table entries hold -1.
"""
from __future__ import annotations

import math
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field, replace

import numpy as np

PAGE_SIZE = 64
D_LATENT = 512
D_ROPE = 64
D_ROW = D_LATENT + D_ROPE
SCALE_192 = 1.0 / math.sqrt(192.0)
_CHUNK_PAGES = 256

BF16_NAN = np.uint16(0x7FC0)
E4M3_NAN = np.uint8(0x7F)

CONFIG_NAMES = ("tiny", "kimi", "dsv3", "prefix", "fp8", "verify4", "dsa", "long")


@dataclass
class Workload:
    name: str
    batch: int
    num_heads: int
    q_len: int
    seq_lens: np.ndarray  # int32 [B]
    page_table: np.ndarray  # int32 [B, max_pages]
    kv_cache: np.ndarray  # uint16 (bf16 bits) or uint8 (e4m3) [num_pages, 64, 576]
    q_nope: np.ndarray  # uint16 bf16 bits [B, Q, H, 512]
    q_pe: np.ndarray  # uint16 bf16 bits [B, Q, H, 64]
    scale: float
    kv_dtype: str  # "bf16" or "fp8_e4m3"
    kv_scale: float = 1.0
    seed: int = 0
    meta: dict = field(default_factory=dict)

    @property
    def num_pages(self) -> int:
        return int(self.kv_cache.shape[0])

    @property
    def max_pages(self) -> int:
        return int(self.page_table.shape[1])

    @property
    def kv_tokens(self) -> int:
        return int(self.seq_lens.astype(np.int64).sum())

    def describe(self) -> dict:
        return {
            "workload": self.name,
            "batch": self.batch,
            "num_heads": self.num_heads,
            "q_len": self.q_len,
            "page_size": PAGE_SIZE,
            "kv_dtype": self.kv_dtype,
            "num_pages": self.num_pages,
            "kv_tokens": self.kv_tokens,
            "seq_len_min": int(self.seq_lens.min()),
            "seq_len_max": int(self.seq_lens.max()),
            "seed": self.seed,
        }


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to the nearest bf16 (ties to even); finite inputs only."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    b = b + (np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1)))
    return (b >> np.uint32(16)).astype(np.uint16)


def _normal_pages(seed: int, num_pages: int, threads: int = 8) -> np.ndarray:
    """N(0,1) float32 [num_pages, 64, 576], chunked seeded streams."""
    out = np.empty((num_pages, PAGE_SIZE, D_ROW), dtype=np.float32)
    nchunks = (num_pages + _CHUNK_PAGES - 1) // _CHUNK_PAGES
    seqs = np.random.SeedSequence(seed).spawn(nchunks)

    def work(k):
        lo = k * _CHUNK_PAGES
        hi = min(num_pages, lo + _CHUNK_PAGES)
        g = np.random.Generator(np.random.PCG64(seqs[k]))
        out[lo:hi] = g.standard_normal((hi - lo, PAGE_SIZE, D_ROW), dtype=np.float32)

    if nchunks <= 1:
        for k in range(nchunks):
            work(k)
    else:
        with ThreadPoolExecutor(max_workers=threads) as ex:
            list(ex.map(work, range(nchunks)))
    return out


def _used_mask(num_pages: int, page_table: np.ndarray, seq_lens: np.ndarray) -> np.ndarray:
    """bool [num_pages, 64]: slot holds a token some request can see."""
    used = np.zeros((num_pages, PAGE_SIZE), dtype=bool)
    for b in range(len(seq_lens)):
        L = int(seq_lens[b])
        npg = (L + PAGE_SIZE - 1) // PAGE_SIZE
        for j in range(npg):
            cnt = min(PAGE_SIZE, L - j * PAGE_SIZE)
            used[page_table[b, j], :cnt] = True
    return used


def build(
    name: str,
    num_heads: int,
    q_len: int,
    seq_lens,
    page_table: np.ndarray,
    num_pages: int,
    rng: np.random.Generator,
    seed: int,
    kv_dtype: str = "bf16",
    scale: float = SCALE_192,
    sentinel: str = "nan",
    q_scale: float = 1.0,
    meta=None,
) -> Workload:
    """Fill queries and cache for a given page-table structure."""
    seq_lens = np.asarray(seq_lens, dtype=np.int32)
    B = len(seq_lens)
    qn = rng.standard_normal((B, q_len, num_heads, D_LATENT), dtype=np.float32) * np.float32(q_scale)
    qp = rng.standard_normal((B, q_len, num_heads, D_ROPE), dtype=np.float32) * np.float32(q_scale)
    vals = _normal_pages(seed + 7919, num_pages)
    used = _used_mask(num_pages, page_table, seq_lens)
    if kv_dtype == "bf16":
        cache = f32_to_bf16_bits(vals)
        if sentinel == "nan":
            cache[~used] = BF16_NAN
        elif sentinel == "big":
            signs = np.where(np.arange(D_ROW) % 2 == 0, 1.0, -1.0).astype(np.float32)
            cache[~used] = f32_to_bf16_bits(np.float32(1e4) * signs)
        elif sentinel == "zero":
            cache[~used] = 0
        else:
            raise ValueError(sentinel)
        kv_scale = 1.0
    elif kv_dtype == "fp8_e4m3":
        import torch  # library float8 conversion; no attention arithmetic

        amax = float(np.abs(vals[used]).max()) if used.any() else 1.0
        kv_scale = amax / 448.0
        scaled = torch.from_numpy(vals / np.float32(kv_scale))
        scaled = torch.clamp(scaled, -448.0, 448.0)
        cache = scaled.to(torch.float8_e4m3fn).view(torch.uint8).numpy().copy()
        if sentinel == "nan":
            cache[~used] = E4M3_NAN
        elif sentinel == "zero":
            cache[~used] = 0
        elif sentinel == "big":
            cache[~used] = np.uint8(0x7E)  # 448
        else:
            raise ValueError(sentinel)
    else:
        raise ValueError(kv_dtype)
    del vals
    return Workload(
        name=name,
        batch=B,
        num_heads=num_heads,
        q_len=q_len,
        seq_lens=seq_lens,
        page_table=np.ascontiguousarray(page_table, dtype=np.int32),
        kv_cache=cache,
        q_nope=f32_to_bf16_bits(qn),
        q_pe=f32_to_bf16_bits(qp),
        scale=float(scale),
        kv_dtype=kv_dtype,
        kv_scale=float(kv_scale),
        seed=seed,
        meta=dict(meta or {}),
    )


def topk_indices(wl: "Workload", topk: int, seed: int) -> np.ndarray:
    """int32 [B, q_len, topk]: for each (request, draft position) a seeded
    random subset of its visible positions (min(topk, visible) of them, in
    random order), padded with -1."""
    rng = np.random.Generator(np.random.PCG64(seed))
    out = np.full((wl.batch, wl.q_len, topk), -1, dtype=np.int32)
    for b in range(wl.batch):
        for i in range(wl.q_len):
            n = int(wl.seq_lens[b]) - wl.q_len + i + 1
            k = min(topk, n)
            out[b, i, :k] = rng.choice(n, size=k, replace=False)
    return out


def _tables_private(seq_lens, perm, extra_cols: int = 0):
    """Hand out permuted page ids request by request."""
    npg = [(int(L) + PAGE_SIZE - 1) // PAGE_SIZE for L in seq_lens]
    width = max(npg) + extra_cols
    table = np.full((len(seq_lens), width), -1, dtype=np.int32)
    pos = 0
    for b, n in enumerate(npg):
        table[b, :n] = perm[pos : pos + n]
        pos += n
    return table, pos


def custom(
    seq_lens,
    num_heads: int,
    q_len: int = 1,
    kv_dtype: str = "bf16",
    seed: int = 1,
    extra_pages: int = 3,
    extra_cols: int = 1,
    scale: float = SCALE_192,
    sentinel: str = "nan",
    q_scale: float = 1.0,
    name: str = "custom",
) -> Workload:
    """Arbitrary lengths: private pages drawn from a permuted pool with a few
    unreferenced pages and one unused page-table column."""
    rng = np.random.Generator(np.random.PCG64(seed))
    seq_lens = np.asarray(seq_lens, dtype=np.int32)
    need = sum((int(L) + PAGE_SIZE - 1) // PAGE_SIZE for L in seq_lens)
    pool = need + extra_pages
    perm = rng.permutation(pool).astype(np.int32)
    table, _ = _tables_private(seq_lens, perm, extra_cols)
    return build(name, num_heads, q_len, seq_lens, table, pool, rng, seed, kv_dtype, scale, sentinel, q_scale)


def default_seed(name: str) -> int:
    """Seed of a named batch: 1000 + its index in CONFIG_NAMES."""
    return 1000 + CONFIG_NAMES.index(name)


@dataclass
class KvPackBatch:
    rows_bits: np.ndarray   # uint16 [B, num_new, 576]: bf16 bits of the new rows
    page_table: np.ndarray  # int32 [B, pages per request]
    seq_lens: np.ndarray    # int32 [B]; the new tokens are the last num_new positions
    num_pages: int
    kv_scale: float
    seed: int

    def describe(self) -> dict:
        B, n_new, _ = self.rows_bits.shape
        return {"batch": int(B), "num_new": int(n_new), "rows": int(B * n_new), "num_pages": int(self.num_pages),
                "kv_dtype": "fp8_e4m3", "seed": self.seed}


def kv_pack_batch(seed: int = 2000, batch: int = 64, num_new: int = 4096) -> KvPackBatch:
    """The cache-write batch (module docstring): all of each prompt is new."""
    rng = np.random.Generator(np.random.PCG64(seed))
    pages_per_req = (num_new + PAGE_SIZE - 1) // PAGE_SIZE
    pool = batch * pages_per_req
    seq_lens = np.full(batch, num_new, dtype=np.int32)
    perm = rng.permutation(pool).astype(np.int32)
    table, _ = _tables_private(seq_lens, perm)
    vals = _normal_pages(seed + 7919, batch * num_new // PAGE_SIZE).reshape(batch, num_new, D_ROW)
    kv_scale = float(np.abs(vals).max()) / 448.0
    return KvPackBatch(f32_to_bf16_bits(vals), table, seq_lens, pool, kv_scale, seed)


def make_config(name: str, seed: int | None = None, sentinel: str = "nan") -> Workload:
    """One of the named decode batches (default seed: default_seed(name))."""
    seed = default_seed(name) if seed is None else seed
    rng = np.random.Generator(np.random.PCG64(seed))
    if name == "tiny":
        seq_lens = np.array([100, 257], dtype=np.int32)
        perm = rng.permutation(16).astype(np.int32)
        table = np.full((2, 5), -1, dtype=np.int32)
        table[0, :2] = perm[0:2]
        table[1, :5] = perm[2:7]
        return build(name, 16, 1, seq_lens, table, 16, rng, seed, "bf16", sentinel=sentinel)
    if name == "kimi":
        B, H = 64, 64
        seq_lens = np.full(B, 8192, dtype=np.int32)
        pool = B * 128
        perm = rng.permutation(pool).astype(np.int32)
        table, _ = _tables_private(seq_lens, perm)
        return build(name, H, 1, seq_lens, table, pool, rng, seed, "bf16", sentinel=sentinel)
    if name == "dsv3":
        B, H = 128, 128
        u = rng.uniform(math.log(1024.0), math.log(32768.0), size=B)
        seq_lens = np.floor(np.exp(u)).astype(np.int32)
        pool = int(sum((int(L) + PAGE_SIZE - 1) // PAGE_SIZE for L in seq_lens))
        perm = rng.permutation(pool).astype(np.int32)
        table, _ = _tables_private(seq_lens, perm)
        return build(name, H, 1, seq_lens, table, pool, rng, seed, "bf16", sentinel=sentinel)
    if name == "prefix":
        B, H = 32, 64
        prefix_pages = 768
        suffix = rng.integers(1024, 4096, size=B, endpoint=True).astype(np.int32)
        seq_lens = (prefix_pages * PAGE_SIZE + suffix).astype(np.int32)
        spg = [(int(s) + PAGE_SIZE - 1) // PAGE_SIZE for s in suffix]
        pool = prefix_pages + sum(spg)
        perm = rng.permutation(pool).astype(np.int32)
        width = prefix_pages + max(spg)
        table = np.full((B, width), -1, dtype=np.int32)
        table[:, :prefix_pages] = perm[:prefix_pages]
        pos = prefix_pages
        for b in range(B):
            table[b, prefix_pages : prefix_pages + spg[b]] = perm[pos : pos + spg[b]]
            pos += spg[b]
        return build(
            name, H, 1, seq_lens, table, pool, rng, seed, "bf16", sentinel=sentinel,
            meta={"shared_prefix_pages": prefix_pages},
        )
    if name == "fp8":
        B, H = 256, 128
        seq_lens = rng.integers(4096, 16384, size=B, endpoint=True).astype(np.int32)
        pool = int(sum((int(L) + PAGE_SIZE - 1) // PAGE_SIZE for L in seq_lens))
        perm = rng.permutation(pool).astype(np.int32)
        table, _ = _tables_private(seq_lens, perm)
        return build(name, H, 2, seq_lens, table, pool, rng, seed, "fp8_e4m3", sentinel=sentinel)
    if name == "dsa":
        B, H, L = 64, 128, 16384
        seq_lens = np.full(B, L, dtype=np.int32)
        pool = B * (L // PAGE_SIZE)
        perm = rng.permutation(pool).astype(np.int32)
        table, _ = _tables_private(seq_lens, perm)
        return build(name, H, 1, seq_lens, table, pool, rng, seed, "bf16", sentinel=sentinel, meta={"topk": 2048})
    if name == "verify4":
        # speculative verification: the new token and 3 drafts per request,
        # causal among themselves; 4 * 64 = 256 query rows per request
        B, H = 64, 64
        seq_lens = np.full(B, 8192, dtype=np.int32)
        pool = B * 128
        perm = rng.permutation(pool).astype(np.int32)
        table, _ = _tables_private(seq_lens, perm)
        return build(name, H, 4, seq_lens, table, pool, rng, seed, "bf16", sentinel=sentinel)
    if name == "long":
        # one long-context request (not one of the benchmark's batches): every
        # slice of the work holds a piece of it, and the merge of 76 pieces
        # per query row dominates the step outside the attention kernel
        B, H, L = 1, 128, 131072
        seq_lens = np.full(B, L, dtype=np.int32)
        pool = B * (L // PAGE_SIZE)
        perm = rng.permutation(pool).astype(np.int32)
        table, _ = _tables_private(seq_lens, perm)
        return build(name, H, 1, seq_lens, table, pool, rng, seed, "bf16", sentinel=sentinel)
    raise ValueError(name)


def prefix_shaped(batch: int, num_heads: int, prefix_pages: int, suffix_range, seed: int,
                  kv_dtype: str = "bf16", q_len: int = 1) -> Workload:
    """A smaller prefix-shared batch: every table starts with the same pages."""
    rng = np.random.Generator(np.random.PCG64(seed))
    suffix = rng.integers(suffix_range[0], suffix_range[1], size=batch, endpoint=True).astype(np.int32)
    seq_lens = (prefix_pages * PAGE_SIZE + suffix).astype(np.int32)
    spg = [(int(s) + PAGE_SIZE - 1) // PAGE_SIZE for s in suffix]
    pool = prefix_pages + sum(spg)
    perm = rng.permutation(pool).astype(np.int32)
    table = np.full((batch, prefix_pages + max(spg)), -1, dtype=np.int32)
    table[:, :prefix_pages] = perm[:prefix_pages]
    pos = prefix_pages
    for b in range(batch):
        table[b, prefix_pages : prefix_pages + spg[b]] = perm[pos : pos + spg[b]]
        pos += spg[b]
    return build("prefix_small", num_heads, q_len, seq_lens, table, pool, rng, seed, kv_dtype,
                 meta={"shared_prefix_pages": prefix_pages})


def relabel_pages(wl: Workload, seed: int) -> Workload:
    """Same logical batch with the pool's page ids permuted (pages moved)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    sigma = rng.permutation(wl.num_pages).astype(np.int32)  # old id -> new id
    cache = np.empty_like(wl.kv_cache)
    cache[sigma] = wl.kv_cache
    table = np.where(wl.page_table >= 0, sigma[np.maximum(wl.page_table, 0)], -1).astype(np.int32)
    return replace(wl, kv_cache=cache, page_table=table, name=wl.name + "_relabelled")


def copy_shared_prefix(wl: Workload) -> Workload:
    """Same logical batch with every shared prefix page physically duplicated
    per request (the copy the prefix-shared layout avoids)."""
    npre = int(wl.meta["shared_prefix_pages"])
    B = wl.batch
    extra = (B - 1) * npre
    cache = np.concatenate([wl.kv_cache, np.repeat(wl.kv_cache[wl.page_table[0, :npre]][None], B - 1, 0).reshape(
        extra, PAGE_SIZE, D_ROW)], axis=0)
    table = wl.page_table.copy()
    base = wl.num_pages
    for b in range(1, B):
        table[b, :npre] = base + (b - 1) * npre + np.arange(npre, dtype=np.int32)
    return replace(wl, kv_cache=cache, page_table=table, name=wl.name + "_copied", meta=dict(wl.meta))
