"""CPU float64 oracle for paged MLA decode.

TEST INFRASTRUCTURE ONLY. Nothing on the product path may import this
package: only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline /
reference legs of ``bench.py`` use it. It shares no code with the CUDA
library (no kernels, headers, tables or helpers).

Parity status: every public function is pinned by ``tests/test_oracle_pins.py``
against an independent check (non-absorbed attention, closed forms, the
split/merge identity, brute force, and torch's own float8 decoder).
"""
from .e4m3 import e4m3_decode_table, e4m3_encode, e4m3_to_f64
from .kv_pack import kv_pack_ref
from .sparse import mla_decode_sparse_ref
from .mla_oracle import (
    attend,
    bf16_bits_to_f64,
    decode_cache_rows,
    gather_rows,
    lse_merge,
    mla_decode_ref,
    mla_decode_ref_pieces,
    visible_keys,
)

__all__ = [
    "attend",
    "e4m3_decode_table",
    "e4m3_encode",
    "e4m3_to_f64",
    "bf16_bits_to_f64",
    "decode_cache_rows",
    "gather_rows",
    "kv_pack_ref",
    "lse_merge",
    "mla_decode_ref",
    "mla_decode_ref_pieces",
    "mla_decode_sparse_ref",
    "visible_keys",
]
