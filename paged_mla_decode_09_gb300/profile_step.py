"""Decode steps of a named synthetic batch, for profilers.

    python -m paged_mla_decode_09_gb300.profile_step NAME [REPS]

runs mla_decode on the batch NAME (see workloads.CONFIG_NAMES) REPS times
(default 2), the L2 flushed before each (512 MiB written, then read back, as
in the benchmark), and exits 0 if the device status word is clear.  The ncu
summaries under profiles/ capture one attention-kernel launch of this
program (``-k regex:mla_decode_kernel -s 1 -c 1``: the second step).
"""
from __future__ import annotations

import sys


def main(argv) -> int:
    import torch

    import paged_mla_decode_09_gb300 as mla
    from paged_mla_decode_09_gb300 import workloads as W
    from paged_mla_decode_09_gb300.build import build_library
    from paged_mla_decode_09_gb300.device_inputs import to_device

    name = argv[1]
    reps = int(argv[2]) if len(argv) > 2 else 2
    build_library()
    mla.load_library()
    wl = W.make_config(name)
    db = to_device(wl, "cuda")
    bufs = mla.alloc_buffers(db.q_nope, db.kv_cache, db.page_table)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device="cuda")
    acc = torch.empty((), dtype=torch.int64, device="cuda")
    for _ in range(reps):
        flush.fill_(1)
        torch.sum(flush.view(torch.int64), dim=0, out=acc)
        mla.mla_decode(db.q_nope, db.q_pe, db.kv_cache, db.page_table, db.seq_lens, db.q_len, db.scale,
                       db.kv_scale, bufs.out, bufs.lse, bufs.workspace)
    torch.cuda.synchronize()
    status = mla.mla_query_status(bufs.workspace)
    print(f"{name}: {reps} step(s), device status {status}")
    return 0 if status == 0 else 1


if __name__ == "__main__":
    sys.exit(main(sys.argv))
