#!/usr/bin/env python3
"""Decode-step benchmark for the paged MLA decode library.

One step = one decode of a whole synthetic batch (schedule + split-KV
attention + log-sum-exp combine) through the C ABI.  Default workload: the
largest batch, FP8 speculative verification (B=256 requests, H=128 heads,
q_len=2 with a causal mask between the drafts, 4096-16384 cached tokens each,
64-token pages, e4m3 latent cache with one fp32 scale).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME]
    python bench.py --impl reference ...   # the CPU float64 oracle instead
    python bench.py --op kv_pack ...       # the cache write before a step
    python bench.py --op sparse ...        # top-k decode on the dsa batch
    python bench.py --op cascade ...       # shared-prefix cascade on the prefix batch

``--op kv_pack``: one step = one quantise-and-scatter of a Kimi-shaped
prefill (64 requests x 4096 new tokens) into an e4m3 cache; metric rows/s.

Prints one JSON line (rank 0).  With N > 1 (torchrun, one rank per GPU)
every rank decodes its own replica of the batch (requests are independent,
so the path shards by request with no collective: weak scaling).

Timing: W untimed warm-up steps, then K steps, each between two CUDA events
on the launching stream; between steps the L2 is flushed (512 MiB written,
then read back).  Without --steps, K is sized so the timed steps take about
a second.  After everything timed, a soak of back-to-back steps (about 1.5 s,
untimed) records the SM clock under sustained load (``clocks_soak``).  ``value`` is whole-job throughput with inputs resident in
HBM; ``e2e`` is the same metric through the public call with host buffers
(inputs up, out and lse down, pipelined on two copy streams);
``roofline`` compares the dominant kernel's algorithmic bytes or FLOPs per
launch, over its event-timed duration, with the measured peaks;
``cpu_baseline`` times the float64 oracle on a bounded sample on the host.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from paged_mla_decode_09_gb300 import workloads as W  # noqa: E402

METRIC = "MLA decode KV-tokens/s"
UNIT = "KV-tokens/s"
FLOP_PER_ROW_TOKEN = 2 * 576 + 2 * 512  # QK + PV per (query row, visible key)
L2_FLUSH_BYTES = 512 << 20


class L2Flush:
    """Evicts the L2 (129 MB) between timed steps: a 512 MiB buffer is
    written, then read back, so that when the step starts the L2 holds only
    clean lines of this buffer.  After the write alone the L2 is full of
    dirty lines, and the step would pay for writing the flush buffer back to
    HBM (measured on GB300: Kimi step 138.9 us after the write, 129-131 us
    after write + read)."""

    DESC = "flushed between steps (512 MiB written, then read back: L2 left holding clean lines)"

    def __init__(self, dev):
        import torch

        self.buf = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
        self.acc = torch.empty((), dtype=torch.int64, device=dev)

    def __call__(self, k=1):
        import torch

        self.buf.fill_(k & 0xFF)
        torch.sum(self.buf.view(torch.int64), dim=0, out=self.acc)


def algorithmic_work(wl):
    """Bytes (unique cache rows once + queries + outputs + tables) and FLOPs."""
    esz = 1 if wl.kv_dtype == "fp8_e4m3" else 2
    rows_per_page = {}
    for b in range(wl.batch):
        L = int(wl.seq_lens[b])
        for j in range((L + 63) // 64):
            pid = int(wl.page_table[b, j])
            rows_per_page[pid] = max(rows_per_page.get(pid, 0), min(64, L - 64 * j))
    unique_rows = sum(rows_per_page.values())
    B, Q, H = wl.batch, wl.q_len, wl.num_heads
    pages_read = sum((int(L) + 63) // 64 for L in wl.seq_lens)
    nbytes = (unique_rows * 576 * esz + B * Q * H * 576 * 2 + B * Q * H * 512 * 2 + B * Q * H * 4
              + pages_read * 4 + B * 4)
    flops = 0
    for b in range(B):
        L = int(wl.seq_lens[b])
        for i in range(Q):
            flops += (L - Q + i + 1) * H * FLOP_PER_ROW_TOKEN
    return nbytes, flops, unique_rows


def profiled_traffic(config: str):
    """DRAM bytes (read + write) of one attention-kernel launch on this batch,
    from the ncu capture summarised in profiles/, or None when the kernel
    sources changed since that capture (or the batch was not captured)."""
    import hashlib

    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    rec = json.load(open(path))
    h = hashlib.sha256()
    for f in rec["sources"]:
        fp = os.path.join(ROOT, f)
        if not os.path.exists(fp):
            return None
        h.update(open(fp, "rb").read())
    if h.hexdigest() != rec["sha256"]:
        return None
    return rec["dram_bytes_per_launch"].get(config)


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            m = json.load(f)
        return float(m["hbm_gbs"]), float(m["bf16_tflops"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, 1900.0, "fallback"


class ClockSampler:
    """nvidia-smi sampling during the timed region."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=self.fh, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.fh.close()

    def summary(self):
        if self.proc is None or not self.path:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        loaded = [s for s in sm if s > 0.5 * max(sm)] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


def cpu_oracle_rate(wl, budget_s: float, max_requests: int | None = None):
    """KV-tokens/s of the float64 oracle on a bounded sample of requests."""
    import oracle

    done_tokens, t_total, reqs = 0, 0.0, []
    for b in range(wl.batch):
        t0 = time.perf_counter()
        oracle.mla_decode_ref(wl.q_nope, wl.q_pe, wl.kv_cache, wl.page_table, wl.seq_lens, wl.q_len, wl.scale,
                              wl.kv_scale, wl.kv_dtype, requests=[b])
        t_total += time.perf_counter() - t0
        done_tokens += int(wl.seq_lens[b])
        reqs.append(b)
        if t_total >= budget_s or (max_requests and len(reqs) >= max_requests):
            break
    cores = len(os.sched_getaffinity(0))
    return done_tokens / t_total, {"requests": len(reqs), "kv_tokens": done_tokens, "seconds": t_total,
                                   "cores": cores}


def host_info():
    """CPU model and the BLAS thread count the oracle's matrix products use."""
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.split(":")[0].strip() == "Model name":
                model = line.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    if model is None:
        try:
            for line in open("/proc/cpuinfo"):
                if line.lower().startswith("model name"):
                    model = line.split(":", 1)[1].strip()
                    break
        except OSError:
            pass
    threads = None
    try:
        from threadpoolctl import threadpool_info

        blas = [i for i in threadpool_info() if i.get("user_api") == "blas"]
        if blas:
            threads = int(blas[0]["num_threads"])
    except Exception:  # threadpoolctl absent (the Arm machine) or a library it cannot query
        pass
    if threads is None:
        for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
            if os.environ.get(var, "").isdigit():
                threads = int(os.environ[var])
                break
    if threads is None:
        threads = len(os.sched_getaffinity(0))  # OpenBLAS' default: one thread per usable core
    return {"cpu_model": model or "unknown", "blas_threads": threads}


def whole_batch_parity(wl, go, gl, tol, chunk=32):
    """out and lse of every request against the oracle, element by element,
    |gpu - ref| <= tol + tol * |ref|; the oracle runs `chunk` requests at a
    time so that host memory stays bounded."""
    import oracle

    t0 = time.perf_counter()
    max_o = max_l = 0.0
    bad = 0
    for b0 in range(0, wl.batch, chunk):
        reqs = list(range(b0, min(wl.batch, b0 + chunk)))
        ro, rl = oracle.mla_decode_ref(wl.q_nope, wl.q_pe, wl.kv_cache, wl.page_table, wl.seq_lens, wl.q_len,
                                       wl.scale, wl.kv_scale, wl.kv_dtype, requests=reqs)
        eo = np.abs(go[reqs] - ro[reqs])
        el = np.abs(gl[reqs] - rl[reqs])
        max_o, max_l = max(max_o, float(eo.max())), max(max_l, float(el.max()))
        bad += int(np.sum(eo > tol + tol * np.abs(ro[reqs]))) + int(np.sum(el > tol + tol * np.abs(rl[reqs])))
    return {"requests": f"all {wl.batch}", "elements": int(go.size + gl.size), "max_abs_out": max_o,
            "max_abs_lse": max_l, "tolerance": f"{tol} + {tol} * |ref|", "outside_tol": bad,
            "within_tol": bad == 0, "oracle_seconds": time.perf_counter() - t0}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def rank_seed(base_seed, config: str, rank: int):
    """Seed of rank `rank`'s replica: rank 0 decodes the standard batch, the
    others independent batches of the same shape."""
    if base_seed is None:
        base_seed = W.default_seed(config)
    return base_seed + 7919 * rank


def reduce_over_ranks(ms: float, kv_tokens: int, device):
    """Whole-job figures of a replicated step: the slowest rank's time and
    the KV tokens all ranks decoded.  Every rank must call it (a collective
    when the process group is up); with one process it is the identity."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return ms, kv_tokens
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    n = torch.tensor([kv_tokens], dtype=torch.int64, device=device)
    dist.all_reduce(n, op=dist.ReduceOp.SUM)
    return float(t.item()), int(n.item())


def run_reference(args):
    world, rank, _ = dist_setup()
    if rank != 0:
        return 0
    wl = W.make_config(args.config, seed=args.seed)
    budget = args.ref_step_budget
    for _ in range(args.warmup):  # untimed warm-up steps
        cpu_oracle_rate(wl, budget, max_requests=1)
    rates, secs, samples = [], [], []
    for _ in range(args.steps):
        r, info = cpu_oracle_rate(wl, budget)
        rates.append(r)
        secs.append(info["seconds"])
        samples.append(info)
    value = float(np.mean(rates))
    hi = host_info()
    sample_desc = (f"{samples[0]['requests']} request(s) of the {args.config} batch per step "
                   f"({samples[0]['kv_tokens']} KV tokens), float64 numpy oracle")
    line = {
        "impl": "reference",
        "metric": METRIC,
        "value": value,
        "unit": UNIT,
        "n_gpus": args.gpus,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": 1e3 * float(np.mean(secs)),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": args.config, **wl.describe()},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": hi["blas_threads"], "kind": "oracle",
                         "sample": sample_desc, "cpu_model": hi["cpu_model"], "blas_threads": hi["blas_threads"],
                         "usable_cores": samples[0]["cores"]},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


def run_ours(args):
    import torch

    world, rank, local = dist_setup()
    if world > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())

    import paged_mla_decode_09_gb300 as mla
    from paged_mla_decode_09_gb300.build import build_library
    from paged_mla_decode_09_gb300.device_inputs import out_to_f64, to_device

    build_library()
    mla.load_library()
    wl = W.make_config(args.config, seed=rank_seed(args.seed, args.config, rank))
    db = to_device(wl, dev)
    bufs = mla.alloc_buffers(db.q_nope, db.kv_cache, db.page_table)
    nbytes, flops, unique_rows = algorithmic_work(wl)
    kv_tokens = wl.kv_tokens
    hbm_peak, bf16_peak, peak_src = measured_peaks()
    f8 = wl.kv_dtype == "fp8_e4m3"
    flop_peak = bf16_peak * (2.0 if f8 else 1.0)  # e4m3 tensor rate = 2x bf16 (nominal ratio)
    stream = torch.cuda.current_stream()
    flush = L2Flush(dev)

    def step(events=None):
        mla.mla_decode(db.q_nope, db.q_pe, db.kv_cache, db.page_table, db.seq_lens, db.q_len, db.scale,
                       db.kv_scale, bufs.out, bufs.lse, bufs.workspace, stream, events=events)

    for _ in range(args.warmup):
        flush(1)
        step()
        torch.cuda.synchronize()
        status = mla.mla_query_status(bufs.workspace)
        if status != 0:
            print(json.dumps({"error": "device status during warm-up", **mla.timeout_diagnostics(bufs.workspace)}),
                  file=sys.stderr)
            return 3
    if args.steps is None:  # about one second of timed steps (flush included)
        t0 = time.perf_counter()
        for _ in range(3):
            flush(1)
            step()
        torch.cuda.synchronize()
        per = (time.perf_counter() - t0) / 3
        steps = max(20, int(np.ceil(1.0 / per)))
        if world > 1:  # every rank times the same number of steps
            import torch.distributed as dist

            t = torch.tensor([steps], dtype=torch.int64, device=dev)
            dist.all_reduce(t, op=dist.ReduceOp.MAX)
            steps = int(t.item())
        args.steps = steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    for evs in ev:  # materialise the event handles
        for e in evs:
            e.record(stream)
    torch.cuda.synchronize()

    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    # the timed steps: one event before and one after each step (events
    # between the launches would keep them from overlapping)
    se = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    with ClockSampler(dev.index) as clk:
        t0 = time.perf_counter()
        for k in range(args.steps):
            flush(k & 0xFF)  # L2 flush between steps (outside the step events)
            se[k][0].record(stream)
            step()
            se[k][1].record(stream)
        torch.cuda.synchronize()
        wall = time.perf_counter() - t0
    if world > 1:
        torch.distributed.barrier()
    status = mla.mla_query_status(bufs.workspace)
    clocks = clk.summary()
    step_ms = [a.elapsed_time(b) for a, b in se]
    # the per-kernel breakdown (and the attention kernel's time for the
    # roofline) from as many steps with events between the launches
    for k in range(args.steps):
        flush(k & 0xFF)
        step(ev[k])
    torch.cuda.synchronize()
    k1_ms = [ev[k][1].elapsed_time(ev[k][2]) for k in range(args.steps)]
    k0_ms = [ev[k][0].elapsed_time(ev[k][1]) for k in range(args.steps)]
    k2_ms = [ev[k][2].elapsed_time(ev[k][3]) for k in range(args.steps)]
    ms, job_tokens = reduce_over_ranks(float(np.mean(step_ms)), kv_tokens, dev)
    ms_median, _ = reduce_over_ranks(float(np.median(step_ms)), kv_tokens, dev)
    value = job_tokens / (ms * 1e-3)

    # end to end through the public API with host buffers: every step copies
    # its inputs (queries, page table, lengths) up from pinned memory and its
    # out and lse back; the cache is resident decode state.  Serial: one step
    # at a time.  Pipelined (the e2e figure): two buffer sets, step k + 1's
    # inputs go up and step k - 1's results come back on a copy stream while
    # step k decodes on the compute stream (the cache, larger than L2, is
    # not flushed between these steps); uploads and downloads use two streams.
    h_qn = db.q_nope.cpu().pin_memory()
    h_qp = db.q_pe.cpu().pin_memory()
    h_pt = db.page_table.cpu().pin_memory()
    h_sl = db.seq_lens.cpu().pin_memory()
    h_out = [torch.empty(bufs.out.shape, dtype=bufs.out.dtype).pin_memory() for _ in range(2)]
    h_lse = [torch.empty(bufs.lse.shape, dtype=bufs.lse.dtype).pin_memory() for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in (h_qn, h_qp, h_pt, h_sl))
    d2h = h_out[0].numel() * h_out[0].element_size() + h_lse[0].numel() * h_lse[0].element_size()
    e2e_ms = []
    for k in range(args.warmup + args.steps):
        flush(1)
        torch.cuda.synchronize()
        e_start = torch.cuda.Event(enable_timing=True)
        e_end = torch.cuda.Event(enable_timing=True)
        e_start.record(stream)
        db.q_nope.copy_(h_qn, non_blocking=True)
        db.q_pe.copy_(h_qp, non_blocking=True)
        db.page_table.copy_(h_pt, non_blocking=True)
        db.seq_lens.copy_(h_sl, non_blocking=True)
        step()
        h_out[0].copy_(bufs.out, non_blocking=True)
        h_lse[0].copy_(bufs.lse, non_blocking=True)
        e_end.record(stream)
        torch.cuda.synchronize()
        if k >= args.warmup:
            e2e_ms.append(e_start.elapsed_time(e_end))
    e2e_serial_ms, _ = reduce_over_ranks(float(np.mean(e2e_ms)), kv_tokens, dev)

    dsets = [db, to_device(wl, dev)]
    osets = [bufs, mla.alloc_buffers(db.q_nope, db.kv_cache, db.page_table)]
    s_comp, s_copy, s_down = stream, torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_comp = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def pipelined(n):
        for k in range(n):
            i = k % 2
            d, o = dsets[i], osets[i]
            with torch.cuda.stream(s_copy):
                if k >= 2:
                    s_copy.wait_event(ev_comp[i])  # step k - 2 is done with these inputs
                d.q_nope.copy_(h_qn, non_blocking=True)
                d.q_pe.copy_(h_qp, non_blocking=True)
                d.page_table.copy_(h_pt, non_blocking=True)
                d.seq_lens.copy_(h_sl, non_blocking=True)
                ev_in[i].record(s_copy)
            s_comp.wait_event(ev_in[i])
            if k >= 2:
                s_comp.wait_event(ev_out[i])  # step k - 2's results are back
            mla.mla_decode(d.q_nope, d.q_pe, d.kv_cache, d.page_table, d.seq_lens, d.q_len, d.scale, d.kv_scale,
                           o.out, o.lse, o.workspace, s_comp)
            ev_comp[i].record(s_comp)
            with torch.cuda.stream(s_down):  # results down on their own stream (the other copy engine)
                s_down.wait_event(ev_comp[i])
                h_out[i].copy_(o.out, non_blocking=True)
                h_lse[i].copy_(o.lse, non_blocking=True)
                ev_out[i].record(s_down)

    pipelined(args.warmup)
    torch.cuda.synchronize()
    p_start, p_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    p_start.record(s_comp)
    s_copy.wait_event(p_start)
    s_down.wait_event(p_start)
    pipelined(args.steps)
    s_comp.wait_stream(s_copy)
    s_comp.wait_stream(s_down)
    p_end.record(s_comp)
    torch.cuda.synchronize()
    e2e_max_ms, _ = reduce_over_ranks(p_start.elapsed_time(p_end) / args.steps, kv_tokens, dev)
    e2e_value = job_tokens / (e2e_max_ms * 1e-3)
    # the parity sample below checks the last pipelined step's results
    h_out = h_out[(args.steps - 1) % 2]
    h_lse = h_lse[(args.steps - 1) % 2]

    # clocks under sustained load: back-to-back steps (with the L2 flush) for
    # about 1.5 s, untimed, after everything timed above
    with ClockSampler(dev.index) as clk_soak:
        t_end = time.perf_counter() + 1.5
        while time.perf_counter() < t_end:
            for _ in range(8):
                flush(1)
                step()
            torch.cuda.synchronize()
    clocks_soak = clk_soak.summary()

    parity = None  # parity against the oracle on this very batch: every request
    if rank == 0 and not args.no_parity:
        parity = whole_batch_parity(wl, out_to_f64(h_out), h_lse.numpy().astype(np.float64), 4e-2 if f8 else 1e-2)

    k1 = float(np.mean(k1_ms))
    t_bytes = nbytes / (hbm_peak * 1e9)
    t_flops = flops / (flop_peak * 1e12)
    bound = "hbm" if t_bytes >= t_flops else "tensor"
    if bound == "hbm":
        achieved, peak, unit_r = nbytes / (k1 * 1e-3) / 1e9, hbm_peak, "GB/s"
    else:
        achieved, peak, unit_r = flops / (k1 * 1e-3) / 1e12, flop_peak, "TFLOP/s"
    roofline = {"bound": bound, "achieved": achieved, "peak": peak, "unit": unit_r, "frac": achieved / peak,
                "achieved_gbs": nbytes / (k1 * 1e-3) / 1e9, "achieved_tflops": flops / (k1 * 1e-3) / 1e12,
                "step_gbs": nbytes / (ms * 1e-3) / 1e9, "step_tflops": flops / (ms * 1e-3) / 1e12,
                "traffic": profiled_traffic(args.config), "traffic_unit": "bytes per launch (ncu dram read + write)",
                "peak_source": peak_src + (" (e4m3 = 2x bf16, nominal ratio)" if f8 and bound == "tensor" else ""),
                "kernel": "mla_decode_kernel", "alg_bytes": nbytes, "alg_flops": flops,
                "step_frac": max(t_bytes, t_flops) / (ms * 1e-3)}

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        rate, info = cpu_oracle_rate(wl, args.cpu_budget)
        hi = host_info()
        cpu = {"value": rate, "unit": UNIT, "cores": hi["blas_threads"], "kind": "oracle",
               "sample": f"{info['requests']} request(s), {info['kv_tokens']} KV tokens of the {args.config} "
                         f"batch, float64 numpy oracle, {info['seconds']:.1f} s",
               "cpu_model": hi["cpu_model"], "blas_threads": hi["blas_threads"], "usable_cores": info["cores"]}
    nclusters, csize = mla.mla_decode_launch_shape(mla.make_dims(db.q_nope, db.kv_cache, db.page_table),
                                                   dev.index)
    if rank == 0:
        line = {
            "metric": METRIC,
            "value": value,
            "unit": UNIT,
            "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": ms,
            "us_per_step": ms * 1e3,
            "us_per_step_median": ms_median * 1e3,
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "f8e4m3" if f8 else "bf16",
            "data": "synthetic",
            "config": {"workload": args.config, **wl.describe(), "l2": L2Flush.DESC,
                       "parallelism": f"replicas x{world}", "clusters": nclusters, "cluster_size": csize},
            "roofline": roofline,
            "kernel_ms": {"schedule": float(np.mean(k0_ms)), "attention": k1, "combine": float(np.mean(k2_ms))},
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "pipelined": "2 buffer sets; step k+1's inputs up and k-1's results down on two copy "
                                 "streams while step k decodes",
                    "serial_value": job_tokens / (e2e_serial_ms * 1e-3)},
            # schedule, (e4m3: query scales,) attention, combine
            "gpu_launches": (4 if f8 else 3) * args.steps,
            "clocks": clocks,
            "clocks_soak": clocks_soak,
            "device_status": status,
            "parity": parity,
            "wall_s_timed_region": wall,
        }
        print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


KV_PACK_METRIC = "KV-pack rows/s"
KV_PACK_UNIT = "rows/s"


def kv_pack_oracle_rate(wl, budget_s: float):
    """rows/s of the oracle's quantise-and-scatter on a bounded sample of
    rows (one request's rows at a time, until the budget is spent)."""
    import oracle

    B, n_new, _ = wl.rows_bits.shape
    rows, t_total = 0, 0.0
    cache = np.zeros((wl.num_pages, 64, 576), dtype=np.uint8)
    per = 64  # rows of one request per call
    for b in range(B):
        t0 = time.perf_counter()
        sub_table = wl.page_table[b:b + 1]
        oracle.kv_pack_ref(wl.rows_bits[b:b + 1, :per], sub_table, np.array([per], dtype=np.int32), wl.kv_scale,
                           cache, "fp8_e4m3")
        t_total += time.perf_counter() - t0
        rows += per
        if t_total >= budget_s:
            break
    return rows / t_total, {"rows": rows, "seconds": t_total, "cores": len(os.sched_getaffinity(0))}


def run_kv_pack(args):
    """The cache write, timed like the decode: device events around the one
    launch per step, inputs (302 MB of rows) larger than L2 and L2 flushed
    between steps; e2e adds the H2D copy of the rows from pinned memory and
    the D2H read of the status word."""
    import torch

    world, rank, local = dist_setup()
    if world > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())
    import paged_mla_decode_09_gb300 as mla
    from paged_mla_decode_09_gb300.build import build_library

    build_library()
    mla.load_library()
    wl = W.kv_pack_batch(seed=2000 + 7919 * rank if args.seed is None else args.seed + 7919 * rank)
    B, n_new, _ = wl.rows_bits.shape
    n_rows = B * n_new
    rows = torch.from_numpy(wl.rows_bits.view(np.int16)).to(dev).view(torch.bfloat16)
    cache = torch.zeros(wl.num_pages, 64, 576, dtype=torch.uint8, device=dev)
    pt = torch.from_numpy(wl.page_table).to(dev)
    sl = torch.from_numpy(wl.seq_lens).to(dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream()
    flush = L2Flush(dev)

    def step():
        mla.mla_kv_pack(rows, pt, sl, wl.kv_scale, cache, status, stream)

    for _ in range(args.warmup):
        flush(1)
        step()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(dev.index) as clk:
        for k in range(args.steps):
            flush(k & 0xFF)
            ev[k][0].record(stream)
            step()
            ev[k][1].record(stream)
        torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    ms_k = [a.elapsed_time(b) for a, b in ev]
    ms, job_rows = reduce_over_ranks(float(np.mean(ms_k)), n_rows, dev)
    value = job_rows / (ms * 1e-3)
    st = int(status.item())

    # end to end: the rows arrive from pinned host memory every step
    h_rows = rows.cpu().pin_memory()
    h_status = torch.empty(1, dtype=torch.int32).pin_memory()
    h2d, d2h = h_rows.numel() * h_rows.element_size(), 4
    e2e = []
    for k in range(args.warmup + args.steps):
        flush(1)
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        rows.copy_(h_rows, non_blocking=True)
        step()
        h_status.copy_(status, non_blocking=True)
        b.record(stream)
        torch.cuda.synchronize()
        if k >= args.warmup:
            e2e.append(a.elapsed_time(b))
    e2e_ms, _ = reduce_over_ranks(float(np.mean(e2e)), n_rows, dev)

    parity = None
    if rank == 0 and not args.no_parity:  # sampled rows, bit-exact against the oracle
        import oracle

        rng = np.random.default_rng(1)
        ok = True
        for _ in range(64):
            b, i = int(rng.integers(B)), int(rng.integers(n_new))
            t = int(wl.seq_lens[b]) - n_new + i
            got = cache[int(wl.page_table[b, t // 64]), t % 64].cpu().numpy()
            ref = oracle.e4m3_encode(oracle.kv_pack.bf16_bits_to_f32(wl.rows_bits[b, i]) * (np.float32(1.0) / np.float32(wl.kv_scale)))
            ok &= bool(np.array_equal(got, ref))
        parity = {"rows_checked": 64, "bit_exact": ok}

    hbm_peak, _, peak_src = measured_peaks()
    nbytes = n_rows * (576 * 2 + 576)  # read a bf16 row, write its e4m3 codes
    achieved = nbytes / (ms * 1e-3) / 1e9
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        rate, info = kv_pack_oracle_rate(wl, min(args.cpu_budget, 10.0))
        cpu = {"value": rate, "unit": KV_PACK_UNIT, "cores": info["cores"], "kind": "oracle",
               "sample": f"{info['rows']} rows of the kv_pack batch, numpy oracle, {info['seconds']:.1f} s"}
    if rank == 0:
        print(json.dumps({
            "metric": KV_PACK_METRIC, "value": value, "unit": KV_PACK_UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "us_per_step": ms * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16->e4m3", "data": "synthetic",
            "config": {"workload": "kv_pack", **wl.describe(), "l2": L2Flush.DESC,
                       "parallelism": f"replicas x{world}"},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                         "frac": achieved / hbm_peak, "traffic": None, "peak_source": peak_src,
                         "kernel": "mla_kv_pack_kernel", "alg_bytes": nbytes},
            "cpu_baseline": cpu,
            "e2e": {"value": job_rows / (e2e_ms * 1e-3), "unit": KV_PACK_UNIT, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h},
            "gpu_launches": args.steps, "clocks": clk.summary(), "device_status": st, "parity_sample": parity,
        }))
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


SPARSE_METRIC = "MLA top-k decode picked-KV-tokens/s"


def sparse_oracle_rate(wl, idx, budget_s: float):
    """picked-KV-tokens/s of the float64 oracle on a bounded sample of requests."""
    import oracle

    done, t_total, reqs = 0, 0.0, 0
    for b in range(wl.batch):
        t0 = time.perf_counter()
        oracle.mla_decode_sparse_ref(wl.q_nope, wl.q_pe, wl.kv_cache, wl.page_table, wl.seq_lens, wl.q_len, idx,
                                     wl.scale, wl.kv_scale, wl.kv_dtype, requests=[b])
        t_total += time.perf_counter() - t0
        done += int((idx[b] >= 0).sum())
        reqs += 1
        if t_total >= budget_s:
            break
    return done / t_total, {"requests": reqs, "picked": done, "seconds": t_total,
                            "cores": len(os.sched_getaffinity(0))}


def run_sparse(args):
    """Top-k decode of the dsa batch: one step = gather of the picked rows +
    the paged decode over them, timed with device events around the call."""
    import torch

    world, rank, local = dist_setup()
    if world > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())
    import paged_mla_decode_09_gb300 as mla
    from paged_mla_decode_09_gb300.build import build_library
    from paged_mla_decode_09_gb300.device_inputs import to_device

    build_library()
    mla.load_library()
    wl = W.make_config("dsa", seed=rank_seed(args.seed, "dsa", rank))
    topk = int(wl.meta["topk"])
    idx = W.topk_indices(wl, topk, seed=rank_seed(args.seed, "dsa", rank) + 1)
    db = to_device(wl, dev)
    ix = torch.from_numpy(idx).to(dev)
    dims = mla.make_dims(db.q_nope, db.kv_cache, db.page_table)
    ws = torch.zeros(mla.mla_decode_sparse_workspace_size(dims, topk, dev.index), dtype=torch.uint8, device=dev)
    B, Q, H, _ = db.q_nope.shape
    out = torch.empty(B, Q, H, 512, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(B, Q, H, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    flush = L2Flush(dev)

    def step():
        mla.mla_decode_sparse(db.q_nope, db.q_pe, db.kv_cache, db.page_table, db.seq_lens, ix, db.scale,
                              db.kv_scale, out, lse, ws, stream)

    for _ in range(args.warmup):
        flush(1)
        step()
    torch.cuda.synchronize()
    st = mla.mla_decode_sparse_query_status(db.q_nope, db.kv_cache, db.page_table, topk, ws)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(dev.index) as clk:
        for k in range(args.steps):
            flush(k & 0xFF)
            ev[k][0].record(stream)
            step()
            ev[k][1].record(stream)
        torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    picked = int((idx >= 0).sum())
    ms, job_picked = reduce_over_ranks(float(np.mean([a.elapsed_time(b) for a, b in ev])), picked, dev)
    value = job_picked / (ms * 1e-3)

    # end to end: queries and picks arrive from pinned memory, out and lse go back
    h_in = [t.cpu().pin_memory() for t in (db.q_nope, db.q_pe, ix)]
    h_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h_lse = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in h_in)
    d2h = h_out.numel() * h_out.element_size() + h_lse.numel() * h_lse.element_size()
    e2e = []
    for k in range(args.warmup + args.steps):
        flush(1)
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for d_t, h_t in zip((db.q_nope, db.q_pe, ix), h_in):
            d_t.copy_(h_t, non_blocking=True)
        step()
        h_out.copy_(out, non_blocking=True)
        h_lse.copy_(lse, non_blocking=True)
        b.record(stream)
        torch.cuda.synchronize()
        if k >= args.warmup:
            e2e.append(a.elapsed_time(b))
    e2e_ms, _ = reduce_over_ranks(float(np.mean(e2e)), picked, dev)

    parity = None
    if rank == 0 and not args.no_parity:
        import oracle

        reqs = [0, B - 1]
        ro, rl, _ = oracle.mla_decode_sparse_ref(wl.q_nope, wl.q_pe, wl.kv_cache, wl.page_table, wl.seq_lens,
                                                 wl.q_len, idx, wl.scale, requests=reqs)
        go = h_out.float().numpy().astype(np.float64)
        gl = h_lse.numpy().astype(np.float64)
        eo, el = np.abs(go[reqs] - ro[reqs]), np.abs(gl[reqs] - rl[reqs])
        parity = {"requests": reqs, "max_abs_out": float(eo.max()), "max_abs_lse": float(el.max()),
                  "within_tol": bool(np.all(eo <= 1e-2 + 1e-2 * np.abs(ro[reqs])) and
                                     np.all(el <= 1e-2 + 1e-2 * np.abs(rl[reqs])))}
    hbm_peak, bf16_peak, peak_src = measured_peaks()
    nbytes = picked * 1152 + sum(t.numel() * t.element_size() for t in (db.q_nope, db.q_pe, ix, out, lse))
    flops = picked * H * FLOP_PER_ROW_TOKEN
    t_b, t_f = nbytes / (hbm_peak * 1e9), flops / (bf16_peak * 1e12)
    if t_b >= t_f:
        roof = {"bound": "hbm", "achieved": nbytes / (ms * 1e-3) / 1e9, "peak": hbm_peak, "unit": "GB/s"}
    else:
        roof = {"bound": "tensor", "achieved": flops / (ms * 1e-3) / 1e12, "peak": bf16_peak, "unit": "TFLOP/s"}
    roof.update({"frac": roof["achieved"] / roof["peak"], "traffic": None, "peak_source": peak_src,
                 "kernel": "mla_topk_gather_kernel + decode (whole step)", "alg_bytes": nbytes, "alg_flops": flops})
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        rate, info = sparse_oracle_rate(wl, idx, min(args.cpu_budget, 10.0))
        cpu = {"value": rate, "unit": "picked-KV-tokens/s", "cores": info["cores"], "kind": "oracle",
               "sample": f"{info['requests']} request(s) of the dsa batch, float64 oracle, {info['seconds']:.1f} s"}
    if rank == 0:
        print(json.dumps({
            "metric": SPARSE_METRIC, "value": value, "unit": "picked-KV-tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "us_per_step": ms * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": "dsa", **wl.describe(), "topk": topk,
                       "l2": L2Flush.DESC, "parallelism": f"replicas x{world}"},
            "roofline": roof, "cpu_baseline": cpu,
            "e2e": {"value": job_picked / (e2e_ms * 1e-3), "unit": "picked-KV-tokens/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h},
            # gather, schedule, attention, combine
            "gpu_launches": 4 * args.steps, "clocks": clk.summary(), "device_status": st, "parity_sample": parity,
        }))
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def run_cascade(args):
    """The prefix batch through the cascade entry point (prefix pass, suffix
    pass, merge), timed with device events around the call; same metric and
    algorithmic work as the plain decode of that batch."""
    import torch

    world, rank, local = dist_setup()
    if world > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())
    import paged_mla_decode_09_gb300 as mla
    from paged_mla_decode_09_gb300.build import build_library
    from paged_mla_decode_09_gb300.device_inputs import out_to_f64, to_device

    build_library()
    mla.load_library()
    wl = W.make_config("prefix", seed=rank_seed(args.seed, "prefix", rank))
    npre = int(wl.meta["shared_prefix_pages"])
    db = to_device(wl, dev)
    dims = mla.make_dims(db.q_nope, db.kv_cache, db.page_table)
    ws = torch.zeros(mla.mla_decode_cascade_workspace_size(dims, npre, dev.index), dtype=torch.uint8, device=dev)
    B, Q, H, _ = db.q_nope.shape
    out = torch.empty(B, Q, H, 512, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(B, Q, H, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    flush = L2Flush(dev)

    def step():
        mla.mla_decode_cascade(db.q_nope, db.q_pe, db.kv_cache, db.page_table, db.seq_lens, npre, db.scale,
                               db.kv_scale, out, lse, ws, stream)

    for _ in range(args.warmup):
        flush(1)
        step()
    torch.cuda.synchronize()
    st = mla.mla_decode_cascade_query_status(db.q_nope, db.kv_cache, db.page_table, npre, ws)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(dev.index) as clk:
        for k in range(args.steps):
            flush(k & 0xFF)
            ev[k][0].record(stream)
            step()
            ev[k][1].record(stream)
        torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    ms, job_tokens = reduce_over_ranks(float(np.mean([a.elapsed_time(b) for a, b in ev])), wl.kv_tokens, dev)
    value = job_tokens / (ms * 1e-3)

    h_in = [t.cpu().pin_memory() for t in (db.q_nope, db.q_pe, db.page_table, db.seq_lens)]
    h_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h_lse = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in h_in)
    d2h = h_out.numel() * h_out.element_size() + h_lse.numel() * h_lse.element_size()
    e2e = []
    for k in range(args.warmup + args.steps):
        flush(1)
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for d_t, h_t in zip((db.q_nope, db.q_pe, db.page_table, db.seq_lens), h_in):
            d_t.copy_(h_t, non_blocking=True)
        step()
        h_out.copy_(out, non_blocking=True)
        h_lse.copy_(lse, non_blocking=True)
        b.record(stream)
        torch.cuda.synchronize()
        if k >= args.warmup:
            e2e.append(a.elapsed_time(b))
    e2e_ms, _ = reduce_over_ranks(float(np.mean(e2e)), wl.kv_tokens, dev)

    parity = None
    if rank == 0 and not args.no_parity:
        import oracle

        reqs = [0, B - 1]
        ro, rl = oracle.mla_decode_ref(wl.q_nope, wl.q_pe, wl.kv_cache, wl.page_table, wl.seq_lens, wl.q_len,
                                       wl.scale, wl.kv_scale, wl.kv_dtype, requests=reqs)
        go, gl = out_to_f64(h_out), h_lse.numpy().astype(np.float64)
        eo, el = np.abs(go[reqs] - ro[reqs]), np.abs(gl[reqs] - rl[reqs])
        parity = {"requests": reqs, "max_abs_out": float(eo.max()), "max_abs_lse": float(el.max()),
                  "within_tol": bool(np.all(eo <= 1e-2 + 1e-2 * np.abs(ro[reqs])) and
                                     np.all(el <= 1e-2 + 1e-2 * np.abs(rl[reqs])))}
    nbytes, flops, _ = algorithmic_work(wl)
    hbm_peak, bf16_peak, peak_src = measured_peaks()
    t_b, t_f = nbytes / (hbm_peak * 1e9), flops / (bf16_peak * 1e12)
    if t_b >= t_f:
        roof = {"bound": "hbm", "achieved": nbytes / (ms * 1e-3) / 1e9, "peak": hbm_peak, "unit": "GB/s"}
    else:
        roof = {"bound": "tensor", "achieved": flops / (ms * 1e-3) / 1e12, "peak": bf16_peak, "unit": "TFLOP/s"}
    roof.update({"frac": roof["achieved"] / roof["peak"], "traffic": None, "peak_source": peak_src,
                 "kernel": "cascade step (prefix decode, suffix decode, merge)", "alg_bytes": nbytes,
                 "alg_flops": flops})
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        rate, info = cpu_oracle_rate(wl, min(args.cpu_budget, 10.0))
        cpu = {"value": rate, "unit": UNIT, "cores": info["cores"], "kind": "oracle",
               "sample": f"{info['requests']} request(s) of the prefix batch, float64 oracle, {info['seconds']:.1f} s"}
    if rank == 0:
        print(json.dumps({
            "metric": METRIC + " (cascade)", "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "us_per_step": ms * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": "prefix", **wl.describe(), "shared_prefix_pages": npre,
                       "l2": L2Flush.DESC, "parallelism": f"replicas x{world}"},
            "roofline": roof, "cpu_baseline": cpu,
            "e2e": {"value": job_tokens / (e2e_ms * 1e-3), "unit": UNIT, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h},
            # prefix pass (schedule, attention, combine), suffix pass (the same three), merge
            "gpu_launches": 7 * args.steps, "clocks": clk.summary(), "device_status": st, "parity_sample": parity,
        }))
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def run_reference_sparse(args):
    world, rank, _ = dist_setup()
    if rank != 0:
        return 0
    wl = W.make_config("dsa", seed=args.seed)
    idx = W.topk_indices(wl, int(wl.meta["topk"]), seed=(W.default_seed("dsa") if args.seed is None else args.seed) + 1)
    for _ in range(args.warmup):
        sparse_oracle_rate(wl, idx, 0.05)
    rates, secs, info = [], [], None
    for _ in range(args.steps):
        r, info = sparse_oracle_rate(wl, idx, args.ref_step_budget)
        rates.append(r)
        secs.append(info["seconds"])
    value = float(np.mean(rates))
    print(json.dumps({
        "impl": "reference", "metric": SPARSE_METRIC, "value": value, "unit": "picked-KV-tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * float(np.mean(secs)),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "dsa", **wl.describe(), "topk": int(wl.meta["topk"])},
        "cpu_baseline": {"value": value, "unit": "picked-KV-tokens/s", "cores": info["cores"], "kind": "oracle",
                         "sample": f"{info['requests']} request(s) per step, float64 oracle"},
        "e2e": {"value": value, "unit": "picked-KV-tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }))
    return 0


def run_reference_kv_pack(args):
    world, rank, _ = dist_setup()
    if rank != 0:
        return 0
    wl = W.kv_pack_batch(seed=2000 if args.seed is None else args.seed)
    for _ in range(args.warmup):
        kv_pack_oracle_rate(wl, 0.05)
    rates, secs, info = [], [], None
    for _ in range(args.steps):
        r, info = kv_pack_oracle_rate(wl, args.ref_step_budget)
        rates.append(r)
        secs.append(info["seconds"])
    value = float(np.mean(rates))
    print(json.dumps({
        "impl": "reference", "metric": KV_PACK_METRIC, "value": value, "unit": KV_PACK_UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * float(np.mean(secs)),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "kv_pack", **wl.describe()},
        "cpu_baseline": {"value": value, "unit": KV_PACK_UNIT, "cores": info["cores"], "kind": "oracle",
                         "sample": f"{info['rows']} rows per step, numpy oracle"},
        "e2e": {"value": value, "unit": KV_PACK_UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }))
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps (default: about one second of decode steps; 20 for the other ops)")
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", choices=list(W.CONFIG_NAMES), default="fp8")
    ap.add_argument("--seed", type=int, default=None)
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--ref-step-budget", type=float, default=2.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-parity", action="store_true")
    ap.add_argument("--op", choices=["decode", "kv_pack", "sparse", "cascade"], default="decode")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.steps is None and (args.op != "decode" or args.impl == "reference"):
        args.steps = 20
    if args.op == "kv_pack":
        return run_reference_kv_pack(args) if args.impl == "reference" else run_kv_pack(args)
    if args.op == "cascade":
        if args.impl == "reference":  # the cascade computes the plain decode: same oracle arm
            args.config = "prefix"
            return run_reference(args)
        return run_cascade(args)
    if args.op == "sparse":
        return run_reference_sparse(args) if args.impl == "reference" else run_sparse(args)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
