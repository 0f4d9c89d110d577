"""The N > 1 benchmark path on CPU: two gloo ranks run the same cross-rank
reduction the benchmark uses (slowest rank's time, total tokens), the ranks
get distinct batches of one shape, and the oracle arm prints from rank 0 only."""
import io
import json
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as tmp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from paged_mla_decode_09_gb300 import workloads as W  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, outdir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # each rank decodes its own replica; rank r pretends its step took 1 + r ms
        wl = W.make_config("dsv3", seed=bench.rank_seed(None, "dsv3", rank))
        ms, tokens = bench.reduce_over_ranks(1.0 + rank, wl.kv_tokens, torch.device("cpu"))
        dist.barrier()
        with open(os.path.join(outdir, f"r{rank}.json"), "w") as f:
            json.dump({"ms": ms, "tokens": tokens, "mine": wl.kv_tokens,
                       "lens": [int(x) for x in wl.seq_lens[:8]]}, f)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_reduce_like_the_benchmark(tmp_path):
    world = 2
    tmp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True,
                        start_method="spawn")
    r = [json.load(open(tmp_path / f"r{k}.json")) for k in range(world)]
    total = r[0]["mine"] + r[1]["mine"]
    for k in range(world):
        assert r[k]["ms"] == 2.0  # max over ranks
        assert r[k]["tokens"] == total  # whole-job tokens
    assert r[0]["lens"] != r[1]["lens"]  # independent replicas, not the same batch twice


def test_single_process_reduction_is_identity():
    assert bench.reduce_over_ranks(3.5, 1234, torch.device("cpu")) == (3.5, 1234)


def test_rank_zero_uses_the_standard_batch():
    for name in W.CONFIG_NAMES:
        assert bench.rank_seed(None, name, 0) == W.default_seed(name)
        assert bench.rank_seed(None, name, 1) != W.default_seed(name)
    assert bench.rank_seed(5, "kimi", 0) == 5


def test_reference_arm_prints_on_rank_zero_only(monkeypatch):
    args = bench.argparse.Namespace(config="tiny", seed=None, steps=1, warmup=3, gpus=2, ref_step_budget=0.2)
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    buf = io.StringIO()
    with redirect_stdout(buf):
        assert bench.run_reference(args) == 0
    assert buf.getvalue() == ""
    monkeypatch.setenv("RANK", "0")
    buf = io.StringIO()
    with redirect_stdout(buf):
        assert bench.run_reference(args) == 0
    line = json.loads(buf.getvalue())
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
