"""Shared helpers of the GPU tests: run the CUDA path on a seeded workload and
compare it with the CPU oracle element by element."""
import numpy as np

import oracle
import paged_mla_decode_09_gb300 as mla
from paged_mla_decode_09_gb300.device_inputs import out_to_f64, to_device

# |gpu - ref| <= ATOL + RTOL * |ref| on out and lse
TOL = {"bf16": (1e-2, 1e-2), "fp8_e4m3": (4e-2, 4e-2)}


def run_gpu(wl, device="cuda"):
    import torch

    db = to_device(wl, device)
    bufs = mla.alloc_buffers(db.q_nope, db.kv_cache, db.page_table)
    bufs.out.fill_(float("nan"))
    bufs.lse.fill_(float("nan"))
    bufs.workspace.fill_(0xFF)  # stale partials must never leak into a result
    mla.mla_decode(db.q_nope, db.q_pe, db.kv_cache, db.page_table, db.seq_lens, db.q_len, db.scale, db.kv_scale,
                   bufs.out, bufs.lse, bufs.workspace)
    torch.cuda.synchronize()
    status = mla.mla_query_status(bufs.workspace)
    if status & mla.MLA_DEV_TIMEOUT:
        raise AssertionError(f"device timeout: {mla.timeout_diagnostics(bufs.workspace)}")
    return out_to_f64(bufs.out), bufs.lse.cpu().numpy().astype(np.float64), status, db, bufs


def reference(wl, requests=None):
    return oracle.mla_decode_ref(wl.q_nope, wl.q_pe, wl.kv_cache, wl.page_table, wl.seq_lens, wl.q_len, wl.scale,
                                 wl.kv_scale, wl.kv_dtype, requests=requests)


def compare(wl, out, lse, requests=None, label="", tol=None):
    """Asserts the tolerance on every compared element; returns error stats."""
    ref_out, ref_lse = reference(wl, requests)
    sel = np.arange(wl.batch) if requests is None else np.asarray(requests)
    atol, rtol = tol or TOL[wl.kv_dtype]
    o, ro = out[sel], ref_out[sel]
    l, rl = lse[sel], ref_lse[sel]
    assert np.all(np.isfinite(o)), f"{label}: non-finite output"
    eo = np.abs(o - ro)
    el = np.abs(l - rl)
    bad_o = eo > atol + rtol * np.abs(ro)
    bad_l = el > atol + rtol * np.abs(rl)
    rms_ref = float(np.sqrt(np.mean(ro ** 2)))
    stats = {
        "max_abs_out": float(eo.max()),
        "max_abs_lse": float(el.max()),
        "max_err_over_rms_ref": float(eo.max() / rms_ref),
        "rms_err_over_rms_ref": float(np.sqrt(np.mean(eo ** 2)) / rms_ref),
    }
    if bad_o.any() or bad_l.any():
        idx = np.argwhere(bad_o)[:5].tolist()
        raise AssertionError(f"{label}: {int(bad_o.sum())} out / {int(bad_l.sum())} lse elements outside "
                             f"tolerance; first out idx {idx}; stats {stats}")
    return stats


def compare_chunked(wl, out, lse, label="", tol=None, chunk=32):
    """compare() over every request of the batch, `chunk` requests at a time;
    returns the worst error statistics."""
    worst = {}
    for b0 in range(0, wl.batch, chunk):
        reqs = list(range(b0, min(wl.batch, b0 + chunk)))
        st = compare(wl, out, lse, requests=reqs, label=f"{label} requests {reqs[0]}..{reqs[-1]}", tol=tol)
        for k, v in st.items():
            worst[k] = max(worst.get(k, 0.0), v)
    worst["requests"] = wl.batch
    return worst
