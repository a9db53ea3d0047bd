"""Benchmark of the hot path on GB300, printing one JSON line.

Headline step: diagonal scan forward + backward on the 8 x 4096 x 1024 fp32
workload (scan_diag_fwd then scan_diag_bwd through the C ABI), inputs resident
in HBM, L2 flushed (256 MB write, untimed) before every timed step, each step
timed with CUDA events on the launching stream.  value = algorithmic bytes of
the step (fwd: read a, b, write h = 12 B per element; bwd: read a, h, dh,
write da, db = 20 B per element) / mean step time.

The same line carries, under "workloads", the other workloads of the hot path
(small diagonal scan, selective scan, chunkwise linear attention with constant
and with data-dependent decay) with tokens/s, TFLOP/s and roofline fractions
(each forward and backward: 5 warm-up calls, then the median of 20 calls
timed with CUDA events, L2 flushed before each), and:
  roofline      the dominant kernel of the headline step against the measured
                HBM copy bandwidth (MEASURED_PEAKS.json)
  cpu_baseline  the float64 C oracle on this host's cores, on a bounded sample
  e2e           the headline metric through the C ABI from pinned host
                buffers, host<->device copies of every step inside the timed
                region; steps pipelined over three streams (inputs of the
                next step, compute, outputs of the previous step overlap on
                the full-duplex host link), device buffers in two sets
  clocks        nvidia-smi samples taken during the timed region

--impl reference times the oracle (the reference arm of this build) instead.
Multi-GPU (torchrun): every rank runs an independent replica (weak scaling);
value = bytes of all ranks / the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "scan fwd+bwd HBM GB/s; chunk lin-attn tokens/s & TFLOP/s vs roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


SM_MAX_HZ = 2.07e9  # GB300 maximum SM clock (nvidia-smi clocks.max.sm, 2070 MHz)


def kernel_traffic(kernel: str):
    """dram bytes per launch from the committed ncu summary, if it was taken on
    the current source of the kernel (else None)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    e = d.get(kernel)
    if not e:
        return None
    src = os.path.join(ROOT, e["source"])
    try:
        h = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    except OSError:
        return None
    if h != e.get("source_sha256_16"):
        return None
    return e


# ------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index=0, period_ms=100):
        self.proc = None
        self.lines = []
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", str(period_ms)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (OSError, ValueError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for l in self.lines:
            parts = [x.strip() for x in l.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append(dict(sm=float(parts[1]), smax=float(parts[2]), reasons=parts[4:]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        active = set()
        for r in rows:
            for n, v in zip(names, r["reasons"][1:]):
                if v.lower().startswith("active"):
                    active.add(n)
        return {"sm_mhz": statistics.median(r["sm"] for r in rows), "sm_max_mhz": max(r["smax"] for r in rows),
                "reasons": sorted(active), "samples": len(rows)}


# ------------------------------------------------------------------ helpers
def _events(torch):
    return torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)


class Flusher:
    def __init__(self, torch, dev, nbytes=256 * 1024 * 1024):
        self.buf = torch.empty(nbytes // 4, dtype=torch.float32, device=dev)

    def __call__(self):
        self.buf.fill_(1.0)


def _sync_all(torch, dist_on):
    if dist_on:
        import torch.distributed as dist

        dist.barrier()
    if torch.cuda.is_available():
        torch.cuda.synchronize()


def _max_over_ranks(torch, x, dist_on):
    if not dist_on:
        return x
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(world, bytes_per_step, slowest_step_ms):
    """Whole-job GB/s of `world` independent replicas, each moving
    `bytes_per_step` per step, timed by the slowest rank (weak scaling)."""
    return world * bytes_per_step / (slowest_step_ms / 1e3) / 1e9


# ------------------------------------------------------------------ end to end
def e2e_pipelined(torch, dev, host_in, host_out, compute, n, dist_on=False):
    """Mean ms per step of `n` end-to-end steps: each step copies every pinned host input to
    the device, runs compute(device_inputs, device_outputs, stream) and copies every output
    back to its pinned host buffer.  Steps are pipelined over three streams (inputs of step
    i + 1, compute of step i and outputs of step i - 1 overlap: the host link is full duplex)
    with device buffers in two sets; the timed region ends when the last outputs are on the
    host."""
    for v in host_out.values():
        v.zero_()  # touch the pages before timing
    sets = [({k: torch.empty_like(v, device=dev) for k, v in host_in.items()},
             {k: torch.empty_like(v, device=dev) for k, v in host_out.items()}) for _ in range(2)]
    s_in, s_cp, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)

    def ev():
        return torch.cuda.Event()

    def run(n):
        done_cp = [None, None]   # compute of the step that last used each set
        done_out = [None, None]  # output copies of the step that last used each set
        last_out = None
        for i in range(n):
            di, do = sets[i % 2]
            if done_cp[i % 2] is not None:
                s_in.wait_event(done_cp[i % 2])  # the set's inputs were consumed
            with torch.cuda.stream(s_in):
                for k in host_in:
                    di[k].copy_(host_in[k], non_blocking=True)
            e_in = ev()
            e_in.record(s_in)
            s_cp.wait_event(e_in)
            if done_out[i % 2] is not None:
                s_cp.wait_event(done_out[i % 2])  # the set's outputs were copied out
            compute(di, do, s_cp)
            e_cp = ev()
            e_cp.record(s_cp)
            done_cp[i % 2] = e_cp
            s_out.wait_event(e_cp)
            with torch.cuda.stream(s_out):
                for k in host_out:
                    host_out[k].copy_(do[k], non_blocking=True)
            last_out = ev()
            last_out.record(s_out)
            done_out[i % 2] = last_out
        return last_out

    run(2)
    torch.cuda.synchronize()
    s, e = _events(torch)
    _sync_all(torch, dist_on)
    s.record(s_in)
    last = run(n)
    s_in.wait_event(last)  # the last outputs are on the host (they follow every earlier copy and kernel)
    e.record(s_in)
    _sync_all(torch, dist_on)
    ms = s.elapsed_time(e) / n
    del sets
    return ms


# ------------------------------------------------------------------ headline: diagonal scan
def bench_scan(torch, cla, workloads, dev, steps, warmup, dist_on):
    inp = workloads.make("scan")
    a, b, h0, dh = (inp[k].to(dev) for k in ("a", "b", "h0", "dh"))
    B, T, D = a.shape
    n = B * T * D
    ws = torch.empty(cla.scan_diag_workspace_size(B, T, D), dtype=torch.uint8, device=dev)
    h = torch.empty_like(a)
    hT = torch.empty(B, D, device=dev)
    da, db = torch.empty_like(a), torch.empty_like(a)
    dh0 = torch.empty(B, D, device=dev)
    flush = Flusher(torch, dev)
    stream = torch.cuda.current_stream()

    def step(ev):
        ev[0].record(stream)
        cla.scan_diag_fwd(a, b, h0, h=h, hT=hT, workspace=ws, stream=stream)
        ev[1].record(stream)
        cla.scan_diag_bwd(a, None, h0, h, dh, da=da, db=db, dh0=dh0, workspace=ws, stream=stream)
        ev[2].record(stream)

    for _ in range(warmup):
        flush()
        step([torch.cuda.Event(enable_timing=True) for _ in range(3)])
    cla.check_status(ws)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    _sync_all(torch, dist_on)
    t_wall = time.perf_counter()
    for i in range(steps):
        flush()
        step(evs[i])
    _sync_all(torch, dist_on)
    t_wall = time.perf_counter() - t_wall
    cla.check_status(ws)
    fwd = [e[0].elapsed_time(e[1]) for e in evs]
    bwd = [e[1].elapsed_time(e[2]) for e in evs]
    step_ms = statistics.mean(f + b_ for f, b_ in zip(fwd, bwd))
    res = dict(n=n, B=B, T=T, D=D, step_ms=step_ms, fwd_ms=statistics.mean(fwd), bwd_ms=statistics.mean(bwd),
               bytes_fwd=12 * n, bytes_bwd=20 * n, wall_s=t_wall, launches=2 * steps)
    # e2e: pinned host inputs -> device, fwd + bwd, outputs -> host, every step
    host_in = {k: inp[k].pin_memory() for k in ("a", "b", "h0", "dh")}
    host_out = {"h": torch.empty(B, T, D).pin_memory(), "hT": torch.empty(B, D).pin_memory(),
                "da": torch.empty(B, T, D).pin_memory(), "db": torch.empty(B, T, D).pin_memory(),
                "dh0": torch.empty(B, D).pin_memory()}

    def compute(di, do, s):
        cla.scan_diag_fwd(di["a"], di["b"], di["h0"], h=do["h"], hT=do["hT"], workspace=ws, stream=s)
        cla.scan_diag_bwd(di["a"], None, di["h0"], do["h"], di["dh"], da=do["da"], db=do["db"], dh0=do["dh0"],
                          workspace=ws, stream=s)

    res["e2e_ms"] = e2e_pipelined(torch, dev, host_in, host_out, compute, max(3, min(steps, 20)), dist_on)
    cla.check_status(ws)
    res["h2d_bytes"] = sum(v.numel() * v.element_size() for v in host_in.values())
    res["d2h_bytes"] = sum(v.numel() * v.element_size() for v in host_out.values())
    del a, b, h0, dh, h, da, db, host_in, host_out
    return res


# ------------------------------------------------------------------ other workloads
def _time_calls(torch, fn, flush, iters, warmup=5):
    """Median device time of `iters` calls, L2 flushed before each, after `warmup` calls.
    A short device-side sleep after the flush keeps the GPU busy while the host enqueues
    the call, so that the events bracket the call's device time and not the host's launch
    path (which matters for the microsecond-scale calls)."""
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    ts = []
    for _ in range(iters):
        flush()
        torch.cuda._sleep(100_000)  # about 50 us at the SM clock
        s, e = _events(torch)
        s.record(stream)
        fn()
        e.record(stream)
        torch.cuda.synchronize()
        ts.append(s.elapsed_time(e))
    return statistics.median(ts)


def bench_scan_small(torch, cla, workloads, dev, flush, peaks, iters=20, shape=None):
    inp = workloads.make("scan_small", **(shape or {}))
    a, b = inp["a"].to(dev), inp["b"].to(dev)
    B, T, D = a.shape
    ws = torch.empty(cla.scan_diag_workspace_size(B, T, D), dtype=torch.uint8, device=dev)
    h = torch.empty_like(a)
    ms = _time_calls(torch, lambda: cla.scan_diag_fwd(a, b, h=h, workspace=ws), flush, iters)
    # the same bracket around a one-element fill kernel: what the events and a launch cost alone
    one = torch.empty(1, device=dev)
    floor_ms = _time_calls(torch, lambda: one.fill_(1.0), flush, iters)
    by = 12 * B * T * D
    return {"workload": f"diagonal scan fwd fp32 B={B} T={T} D={D}", "fwd_us": round(ms * 1e3, 2),
            "timing_floor_us": round(floor_ms * 1e3, 2),
            "GBps": round(by / ms / 1e6, 1), "frac_hbm": round(by / ms / 1e6 / peaks["hbm_gbs"], 4)}


def bench_scan_blelloch(torch, cla, workloads, dev, flush, peaks, iters=20, shape=None):
    """Forward diagonal scan on the headline workload with the runs of a chunk
    composed by Hillis-Steele (the library's path) and by a Blelloch tree (the
    measured alternative), timed alternately in one process."""
    inp = workloads.make("scan", **(shape or {}))
    a, b, h0 = inp["a"].to(dev), inp["b"].to(dev), inp["h0"].to(dev)
    B, T, D = a.shape
    ws = torch.empty(cla.scan_diag_workspace_size(B, T, D), dtype=torch.uint8, device=dev)
    h = torch.empty_like(a)
    by = 12 * B * T * D
    hs, bl = [], []
    f_hs = lambda: cla.scan_diag_fwd(a, b, h0, h=h, workspace=ws)
    f_bl = lambda: cla.scan_diag_fwd_blelloch(a, b, h0, h=h, workspace=ws)
    for _ in range(5):
        f_hs()
        f_bl()
    for _ in range(iters):  # alternately, one timed call each
        hs.append(_time_calls(torch, f_hs, flush, 1, warmup=0))
        bl.append(_time_calls(torch, f_bl, flush, 1, warmup=0))
    cla.check_status(ws)
    ms_hs, ms_bl = statistics.median(hs), statistics.median(bl)
    return {"workload": f"diagonal scan fwd fp32 B={B} T={T} D={D}: Hillis-Steele vs Blelloch across a chunk's runs",
            "hillis_steele_us": round(ms_hs * 1e3, 2), "blelloch_us": round(ms_bl * 1e3, 2),
            "hillis_steele_GBps": round(by / ms_hs / 1e6, 1), "blelloch_GBps": round(by / ms_bl / 1e6, 1)}


def bench_scan_bwd_recompute(torch, cla, workloads, dev, flush, peaks, iters=20, shape=None):
    """Backward diagonal scan on the headline workload given the forward's states h (read:
    a, h, dh; written: da, db) and without them (read: a, b, dh; states rebuilt from the state
    entering each chunk, which a forward pass without h output writes first)."""
    inp = workloads.make("scan", **(shape or {}))
    a, b, h0, dh = (inp[k].to(dev) for k in ("a", "b", "h0", "dh"))
    B, T, D = a.shape
    ws = torch.empty(cla.scan_diag_workspace_size(B, T, D), dtype=torch.uint8, device=dev)
    h, _ = cla.scan_diag_fwd(a, b, h0, workspace=ws)
    da, db = torch.empty_like(a), torch.empty_like(a)
    dh0 = torch.empty(B, D, device=dev)
    f_h = lambda: cla.scan_diag_bwd(a, None, h0, h, dh, da=da, db=db, dh0=dh0, workspace=ws)
    f_r = lambda: cla.scan_diag_bwd(a, b, h0, None, dh, da=da, db=db, dh0=dh0, workspace=ws)
    ms_h = _time_calls(torch, f_h, flush, iters)
    ms_r = _time_calls(torch, f_r, flush, iters)
    cla.check_status(ws)
    by = 20 * B * T * D
    return {"workload": f"diagonal scan bwd fp32 B={B} T={T} D={D}: saved states vs recomputed",
            "with_h_us": round(ms_h * 1e3, 2), "recompute_us": round(ms_r * 1e3, 2),
            "with_h_GBps": round(by / ms_h / 1e6, 1), "recompute_GBps_of_20B": round(by / ms_r / 1e6, 1),
            "recompute_hbm_bytes_per_element": 28,
            "note": "recompute = forward scan writing only chunk states (8 B/elem read) + backward reading b "
                    "in place of h (20 B/elem)"}


def bench_la(torch, cla, workloads, dev, flush, peaks, name, chunk, iters=20, shape=None, e2e_steps=0):
    inp = workloads.make(name, **(shape or {}))
    t = {k: (v.to(dev) if v is not None else None) for k, v in inp.items()}
    B, H, T, d = t["q"].shape
    ws = torch.empty(cla.chunk_la_workspace_size(B, H, T, d, d, chunk), dtype=torch.uint8, device=dev)
    o = torch.empty(B, H, T, d, device=dev)
    ST = torch.empty(B, H, d, d, device=dev)
    g = [torch.empty(B, H, T, d, device=dev) for _ in range(3)]
    dl = torch.empty(B, H, T, device=dev)
    dS0 = torch.empty(B, H, d, d, device=dev)
    # training step: the forward saves the state entering each segment, the backward starts
    # its forward-order traversal from them
    ck = cla.chunk_la_ckpt(t["q"], t["v"], chunk=chunk)
    fwd = lambda: cla.chunk_la_fwd(t["q"], t["k"], t["v"], t["log_a"], t["S0"], chunk=chunk, o=o, ST=ST, ckpt=ck,
                                   workspace=ws)
    bwd = lambda: cla.chunk_la_bwd(t["q"], t["k"], t["v"], t["log_a"], t["S0"], t["dO"], chunk=chunk, dq=g[0],
                                   dk=g[1], dv=g[2], dlog_decay=dl, dS0=dS0, ckpt=ck, workspace=ws)
    tf = _time_calls(torch, fwd, flush, iters)
    tb = _time_calls(torch, bwd, flush, iters)
    cla.check_status(ws)
    ntok = B * H * T
    fl_f = ntok * (2 * chunk * 2 * d + 4 * d * d)
    fl_b = ntok * (5 * 2 * chunk * d + 5 * 2 * d * d)
    # bytes as this library moves them (bf16 inputs, fp32 outputs o, dq, dk, dv) ...
    by_f = ntok * (3 * 2 * d + 4 + 4 * d)
    by_b = ntok * (4 * 2 * d + 4 + 3 * 4 * d + 4)
    # ... and the method's minimum with bf16 outputs (516 and 904 B per token and head at d = 64)
    by_f_min = ntok * (3 * 2 * d + 4 + 2 * d)
    by_b_min = ntok * (4 * 2 * d + 4 + 3 * 2 * d + 4)
    hbm = peaks["hbm_gbs"] * 1e9
    bf = peaks["bf16_tflops"] * 1e12
    roof = max(by_f + by_b, 0) / hbm, (fl_f + fl_b) / bf
    roof_min = (by_f_min + by_b_min) / hbm, (fl_f + fl_b) / bf
    tot = (tf + tb) / 1e3
    res = {"workload": f"chunkwise linear attention {name} B={B} H={H} T={T} d={d} chunk={chunk}",
           "fwd_us": round(tf * 1e3, 1), "bwd_us": round(tb * 1e3, 1),
           "tokens_per_s": round(B * T / tot, 1),
           "fwd_TFLOPs": round(fl_f / (tf / 1e3) / 1e12, 2), "bwd_TFLOPs": round(fl_b / (tb / 1e3) / 1e12, 2),
           "fwd_GBps": round(by_f / (tf / 1e3) / 1e9, 1), "bwd_GBps": round(by_b / (tb / 1e3) / 1e9, 1),
           "frac_bf16_peak": round((fl_f + fl_b) / tot / bf, 4),
           "frac_binding_roofline": round(max(roof) / tot, 4),
           "frac_binding_roofline_note": "HBM bytes as moved: bf16 inputs, fp32 outputs o, dq, dk, dv",
           "frac_binding_roofline_min_bytes": round(max(roof_min) / tot, 4),
           "frac_binding_roofline_min_bytes_note": "HBM bytes of the method with bf16 outputs "
                                                   f"({(by_f_min + by_b_min) // ntok} B per token and head fwd+bwd)",
           "binding": "hbm" if roof[0] >= roof[1] else "tensor",
           "ckpt_bytes": cla.chunk_la_ckpt_size(B, H, T, d, d, chunk)}
    if e2e_steps > 0:
        # end to end through the C ABI: inputs from pinned host buffers, outputs back, every step
        keys_in = [k for k in ("q", "k", "v", "log_a", "S0", "dO") if inp.get(k) is not None]
        host_in = {k: inp[k].pin_memory() for k in keys_in}
        host_out = {"o": torch.empty(B, H, T, d).pin_memory(), "ST": torch.empty(B, H, d, d).pin_memory(),
                    "dq": torch.empty(B, H, T, d).pin_memory(), "dk": torch.empty(B, H, T, d).pin_memory(),
                    "dv": torch.empty(B, H, T, d).pin_memory(), "dlog_decay": torch.empty(B, H, T).pin_memory(),
                    "dS0": torch.empty(B, H, d, d).pin_memory()}
        del t, o, g, dl, dS0
        torch.cuda.empty_cache()

        def compute(di, do, s):
            cla.chunk_la_fwd(di["q"], di["k"], di["v"], di["log_a"], di.get("S0"), chunk=chunk, o=do["o"],
                             ST=do["ST"], ckpt=ck, workspace=ws, stream=s)
            cla.chunk_la_bwd(di["q"], di["k"], di["v"], di["log_a"], di.get("S0"), di["dO"], chunk=chunk,
                             dq=do["dq"], dk=do["dk"], dv=do["dv"], dlog_decay=do["dlog_decay"], dS0=do["dS0"],
                             ckpt=ck, workspace=ws, stream=s)

        ms = e2e_pipelined(torch, dev, host_in, host_out, compute, e2e_steps)
        cla.check_status(ws)
        h2d = sum(v.numel() * v.element_size() for v in host_in.values())
        d2h = sum(v.numel() * v.element_size() for v in host_out.values())
        res["e2e"] = {"value": round(B * T / (ms / 1e3), 1), "unit": "tokens/s", "ms_per_step": round(ms, 3),
                      "steps": e2e_steps, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                      "note": "fwd + bwd through the C ABI from pinned host buffers, copies inside the timed "
                              "region, pipelined over three streams (the compute stream shares one workspace and "
                              "checkpoint, so the kernels of consecutive steps do not overlap)"}
        del host_in, host_out
    else:
        del t, o, g
    del ws, ck
    torch.cuda.empty_cache()
    return res


def bench_gla(torch, cla, workloads, dev, flush, peaks, iters=20, shape=None):
    """Gated linear attention forward and backward (one decay per key dimension), chunk 64."""
    inp = workloads.make("gla", **(shape or {}))
    t = {k: (v.to(dev) if v is not None else None) for k, v in inp.items()}
    B, H, T, dk = t["q"].shape
    dv = t["v"].shape[-1]
    ws = torch.empty(cla.gla_workspace_size(B, H, T, dk, dv, 64), dtype=torch.uint8, device=dev)
    o = torch.empty(B, H, T, dv, device=dev)
    ST = torch.empty(B, H, dk, dv, device=dev)
    wb = torch.empty(cla.gla_bwd_workspace_size(B, H, T, dk, dv, 64), dtype=torch.uint8, device=dev)
    grads = dict(dq=torch.empty(B, H, T, dk, device=dev), dk=torch.empty(B, H, T, dk, device=dev),
                 dv=torch.empty(B, H, T, dv, device=dev), dlog_decay=torch.empty(B, H, T, dk, device=dev),
                 dS0=torch.empty(B, H, dk, dv, device=dev))
    # the training step's path: the forward saves the state entering every segment, the
    # backward's dq traversal starts from it
    ck = cla.gla_ckpt(t["q"], t["v"])
    fwd = lambda: cla.gla_fwd(t["q"], t["k"], t["v"], t["log_a"], t["S0"], o=o, ST=ST, ckpt=ck, workspace=ws)
    bwd = lambda ckpt: cla.gla_bwd(t["q"], t["k"], t["v"], t["log_a"], t["S0"], t["dO"], ckpt=ckpt, workspace=wb,
                                   **grads)
    tf = _time_calls(torch, fwd, flush, iters)
    tb = _time_calls(torch, lambda: bwd(ck), flush, iters)
    tb_plain = _time_calls(torch, lambda: bwd(None), flush, iters)
    cla.check_status(ws)
    cla.check_status(wb)
    ntok = B * H * T
    fl = ntok * (2 * 64 * (dk + dv) + 4 * dk * dv)
    # backward: dQ and dK traversals (scores, two products each) and the adjoint traversal
    # giving dV, at the same count per product as the forward's
    fl_b = ntok * (5 * 2 * 64 * max(dk, dv) + 5 * 2 * dk * dv)
    by = ntok * (2 * (2 * dk + dv) + 4 * dk + 4 * dv)  # q, k, v bf16, log decays fp32 per key dim, o fp32
    by_min = ntok * (2 * (2 * dk + dv) + 4 * dk + 2 * dv)
    by_b_min = ntok * (2 * (2 * dk + 2 * dv) + 4 * dk + 2 * (2 * dk + dv) + 4 * dk)
    hbm = peaks["hbm_gbs"] * 1e9
    bf = peaks["bf16_tflops"] * 1e12
    sec, secb = tf / 1e3, tb / 1e3
    res = {"workload": f"gated linear attention fwd+bwd B={B} H={H} T={T} dk={dk} dv={dv} chunk=64",
           "fwd_us": round(tf * 1e3, 1), "bwd_us": round(tb * 1e3, 1),
           "bwd_us_without_checkpoint": round(tb_plain * 1e3, 1),
           "checkpoint": "the forward saves the state entering every segment; the backward's dq traversal starts from it",
           "tokens_per_s": round(B * T / (sec + secb), 1),
           "fwd_TFLOPs": round(fl / sec / 1e12, 2), "bwd_TFLOPs": round(fl_b / secb / 1e12, 2),
           "fwd_GBps": round(by / sec / 1e9, 1),
           "frac_bf16_peak": round((fl + fl_b) / (sec + secb) / bf, 4),
           "frac_binding_roofline_min_bytes": round(max((by_min + by_b_min) / hbm, (fl + fl_b) / bf) / (sec + secb), 4),
           "kernels": "gla_tc_kernel (the forward and the backward's reversed dV traversal), gla_tc_qk_kernel "
                      "(dQ, dK): tcgen05.mma kind::f16, fp32 accumulators in tensor memory, bf16 hi/lo operand "
                      "parts; gla_dlog_tile_sums/tile_suffix/finalize"}
    del t, ws, wb, o, ST, grads
    torch.cuda.empty_cache()
    return res


def bench_delta(torch, cla, workloads, dev, flush, peaks, iters=20, shape=None):
    """Delta rule with a decay per head (Gated DeltaNet) forward and backward, chunk 64."""
    inp = workloads.make("delta", **(shape or {}))
    t = {k: (v.to(dev) if v is not None else None) for k, v in inp.items()}
    B, H, T, dk = t["q"].shape
    dv = t["v"].shape[-1]
    ws = torch.empty(max(cla.delta_workspace_size(B, H, T, dk, dv, 64), 256), dtype=torch.uint8, device=dev)
    o = torch.empty(B, H, T, dv, device=dev)
    ST = torch.empty(B, H, dk, dv, device=dev)
    # the training step's path: the forward saves the state entering every chunk, the backward starts from it
    ck = cla.delta_ckpt(t["q"], t["v"])
    fwd = lambda: cla.delta_fwd(t["q"], t["k"], t["v"], t["log_a"], t["beta"], t["S0"], o=o, ST=ST, ckpt=ck,
                                workspace=ws)
    tf = _time_calls(torch, fwd, flush, iters)
    cla.check_status(ws)
    wb = torch.empty(max(cla.delta_bwd_workspace_size(B, H, T, dk, dv, 64), 256), dtype=torch.uint8, device=dev)
    g = [torch.empty(B, H, T, dk, device=dev), torch.empty(B, H, T, dk, device=dev), torch.empty(B, H, T, dv, device=dev),
         torch.empty(B, H, T, device=dev), torch.empty(B, H, T, device=dev), torch.empty(B, H, dk, dv, device=dev)]
    bwd = lambda ckpt: cla.delta_bwd(t["q"], t["k"], t["v"], t["log_a"], t["beta"], t["S0"], t["dO"], None, dq=g[0],
                                     dk=g[1], dv=g[2], dlog_decay=g[3], dbeta=g[4], dS0=g[5], ckpt=ckpt, workspace=wb)
    tb = _time_calls(torch, lambda: bwd(ck), flush, iters)
    tb_plain = _time_calls(torch, lambda: bwd(None), flush, iters)
    cla.check_status(wb)
    ntok = B * H * T
    # the decayed-linear-attention part (scores, P Veff, Q S, state update) plus the chunk's own
    # extra products (K K^T, K S, (I + A)^-1 X): 2 C (2 dk + 2 dv) + 6 dk dv per token
    fl = ntok * (2 * 64 * (2 * dk + 2 * dv) + 6 * dk * dv)
    # backward from the checkpoint: the chunk adjoint (recomputed K K^T, K S, U; P^T, P^T dO, K dS', dX,
    # dP, P, dA, dQ's two products, dK's five, dS's two): 2 C (7 dk + 5 dv) + 16 dk dv per token
    flb = ntok * (2 * 64 * (7 * dk + 5 * dv) + 16 * dk * dv)
    by_min = ntok * (2 * (2 * dk + dv) + 8 + 2 * dv)
    sec, secb = tf / 1e3, tb / 1e3
    return {"workload": f"delta rule (Gated DeltaNet) fwd+bwd B={B} H={H} T={T} dk={dk} dv={dv} chunk=64",
            "fwd_us": round(tf * 1e3, 1), "bwd_us": round(tb * 1e3, 1),
            "bwd_us_without_checkpoint": round(tb_plain * 1e3, 1),
            "checkpoint": "the forward saves the state entering every chunk; the backward starts from it",
            "tokens_per_s": round(B * T / (sec + secb), 1),
            "fwd_TFLOPs": round(fl / sec / 1e12, 2), "bwd_TFLOPs": round(flb / secb / 1e12, 2),
            "frac_bf16_peak": round((fl + flb) / (sec + secb) / (peaks["bf16_tflops"] * 1e12), 4),
            "frac_hbm_min_bytes": round(by_min / sec / (peaks["hbm_gbs"] * 1e9), 4),
            "kernels": "delta_wy_kernel (every chunk's (I + A)^-1, all chunks in parallel, into the checkpoint), "
                       "delta_fwd_kernel (mma.sync m16n8k16; chunks of a head in order, no look-back; saves the "
                       "checkpoint); backward: delta_bwd_kernel (chunks in reverse, from the checkpoint's states "
                       "and inverses; without one delta_wy_kernel and a states pass of delta_fwd_kernel run "
                       "first), delta_bwd_reduce_kernel"}


def bench_selective(torch, cla, workloads, dev, flush, peaks, iters=20, shape=None):
    inp = workloads.make("selective", **(shape or {}))
    t = {k: (v.to(dev) if v is not None else None) for k, v in inp.items()}
    B, T, D = t["x"].shape
    N = t["A"].shape[1]
    ws = torch.empty(cla.selective_scan_workspace_size(B, T, D, N), dtype=torch.uint8, device=dev)
    y = torch.empty(B, T, D, device=dev)
    hT = torch.empty(B, D, N, device=dev)
    ck = torch.empty(cla.selective_scan_ckpt_elems(B, T, D, N), device=dev)
    outs = dict(dx=torch.empty(B, T, D, device=dev), ddelta=torch.empty(B, T, D, device=dev),
                dA=torch.empty(D, N, device=dev), dB=torch.empty(B, T, N, device=dev),
                dC=torch.empty(B, T, N, device=dev), dh0=torch.empty(B, D, N, device=dev))
    fwd = lambda: cla.selective_scan_fwd(t["x"], t["delta"], t["A"], t["Bm"], t["Cm"], None, y=y, hT=hT, ckpt=ck,
                                         workspace=ws)
    bwd = lambda: cla.selective_scan_bwd(t["x"], t["delta"], t["A"], t["Bm"], t["Cm"], None, ck, t["dy"],
                                         workspace=ws, **outs)
    tf = _time_calls(torch, fwd, flush, iters)
    tb = _time_calls(torch, bwd, flush, iters)
    cla.check_status(ws)
    nt = B * T * D
    by_f = nt * (2 + 4 + 4) + B * T * N * 4 + ck.numel() * 4
    by_b = nt * (2 + 4 + 4 + 4 + 4) + B * T * N * 4 * 2 + ck.numel() * 4
    upd = nt * N
    tot = (tf + tb) / 1e3
    # Arithmetic floor of the method per state update (t, d, n): one exp2 and three FP32
    # operations forward, three times that backward.  Unit rates at the maximum clock:
    # 16 MUFU results and 128 FP32 FMAs per SM per clock, 152 SMs.  (This build evaluates
    # 2^x with FMAs instead of the MUFU unit, for accuracy: more work than the floor counts.)
    sfu = 152 * 16 * SM_MAX_HZ
    fp32 = 152 * 128 * SM_MAX_HZ
    floor_alu = max(4 * upd / sfu, 4 * 3 * upd / fp32)  # s, fwd + 3x fwd; the two pipes run side by side
    floor_hbm = (by_f + by_b) / (peaks["hbm_gbs"] * 1e9)
    return {"workload": f"selective scan B={B} T={T} D={D} N={N}", "fwd_us": round(tf * 1e3, 1),
            "bwd_us": round(tb * 1e3, 1), "fwd_GBps": round(by_f / (tf / 1e3) / 1e9, 1),
            "bwd_GBps": round(by_b / (tb / 1e3) / 1e9, 1),
            "frac_hbm": round((by_f + by_b) / tot / (peaks["hbm_gbs"] * 1e9), 4),
            "frac_binding_roofline": round(max(floor_alu, floor_hbm) / tot, 4),
            "binding": "alu (exp2 on the special-function unit)" if floor_alu >= floor_hbm else "hbm",
            "state_updates_per_s": round(2 * upd / tot, 1),
            "kernels": "sel_fwd_seq_kernel, sel_bwd_seq_kernel (one walk per channel, each decay evaluated once; "
                       "taken when B*D >= 16 x SMs) + sel_reduce_bc_kernel, sel_reduce_a_kernel; "
                       "sel_fwd_kernel / sel_bwd_kernel (chunk look-back) for fewer channels"}


# ------------------------------------------------------------------ CPU oracle
def oracle_scan_sample(workloads, seconds_hint=10.0):
    """The oracle's scan fwd+bwd on a bounded sample of the headline workload;
    returns (GB/s, sample description, threads)."""
    import oracle

    inp = workloads.make("scan")
    a, b, h0, dh = (inp[k].double().numpy() for k in ("a", "b", "h0", "dh"))
    B = a.shape[0]
    # grow the sample (batch rows) until it takes about seconds_hint
    rows, elapsed, done = 1, 0.0, 0
    while True:
        t0 = time.perf_counter()
        oracle.scan_diag_fwd(a[:rows], b[:rows], h0[:rows])
        oracle.scan_diag_bwd(a[:rows], b[:rows], h0[:rows], dh[:rows])
        dt = time.perf_counter() - t0
        elapsed += dt
        done = rows
        if elapsed >= seconds_hint or rows >= B:
            break
        rows = min(B, rows * 2)
    n = done * a.shape[1] * a.shape[2]
    return 32 * n / dt / 1e9, f"scan fwd+bwd on batch rows 0..{done - 1} of 8 ({n} elements), {dt:.2f} s", \
        oracle.num_threads()


HEAD_WORKLOAD = "diagonal scan fwd+bwd fp32, B=8 T=4096 D=1024, h0 ~ N(0,1), dL/dh ~ N(0,1)"


def run_reference(args, rank, world):
    """--impl reference: the float64 oracle on this host's cores, on the whole headline
    workload every step (the oracle does the 8 x 4096 x 1024 step in about a tenth of a
    second on the GPU host's cores)."""
    import workloads
    import oracle

    if rank != 0:
        return 0
    oracle.build()
    inp = workloads.make("scan")
    a, b, h0, dh = (inp[k].double().numpy() for k in ("a", "b", "h0", "dh"))
    Bn, T, D = a.shape
    n = a.size
    for _ in range(args.warmup):
        oracle.scan_diag_fwd(a, b, h0)
        oracle.scan_diag_bwd(a, b, h0, dh)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.scan_diag_fwd(a, b, h0)
        oracle.scan_diag_bwd(a, b, h0, dh)
    dt = (time.perf_counter() - t0) / args.steps
    value = 32 * n / dt / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": HEAD_WORKLOAD, "B": Bn, "T": T, "D": D, "parallelism": "host cores"},
            "cpu_baseline": {"value": round(value, 3), "unit": "GB/s", "cores": oracle.num_threads(),
                             "kind": "oracle", "sample": f"the whole {Bn} x {T} x {D} workload per step"},
            "e2e": {"value": round(value, 3), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ main
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--headline-only", action="store_true")
    ap.add_argument("--only", default=None,
                    choices=["scan_small", "scan_fwd_blelloch", "scan_bwd_recompute", "selective", "la_const", "la_long",
                             "la_long_chunk64", "gla", "delta"],
                    help="time one workload only (forward and backward), e.g. for profiling")
    ap.add_argument("--shape", default="", help="shape overrides for --only, e.g. H=32,T=4096")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        return run_reference(args, rank, world)

    import torch

    dist_on = world > 1
    if dist_on:
        import torch.distributed as dist

        dist.init_process_group("nccl")
    dev = torch.device(f"cuda:{local_rank}")
    torch.cuda.set_device(dev)

    import chunkwise_linear_attention_gb300 as cla
    import workloads

    cla.lib()
    peaks, peak_kind = load_peaks()
    if args.only:
        shape = {kv.split("=")[0]: int(kv.split("=")[1]) for kv in args.shape.split(",") if kv}
        flush = Flusher(torch, dev)
        it = max(1, args.steps)
        fns = {"scan_small": lambda: bench_scan_small(torch, cla, workloads, dev, flush, peaks, it, shape),
               "scan_fwd_blelloch": lambda: bench_scan_blelloch(torch, cla, workloads, dev, flush, peaks, it, shape),
               "scan_bwd_recompute": lambda: bench_scan_bwd_recompute(torch, cla, workloads, dev, flush, peaks, it,
                                                                      shape),
               "selective": lambda: bench_selective(torch, cla, workloads, dev, flush, peaks, it, shape),
               "la_const": lambda: bench_la(torch, cla, workloads, dev, flush, peaks, "la_const", 64, it, shape),
               "la_long": lambda: bench_la(torch, cla, workloads, dev, flush, peaks, "la_long", 128, it, shape),
               "la_long_chunk64": lambda: bench_la(torch, cla, workloads, dev, flush, peaks, "la_long", 64, it, shape),
               "gla": lambda: bench_gla(torch, cla, workloads, dev, flush, peaks, it, shape),
               "delta": lambda: bench_delta(torch, cla, workloads, dev, flush, peaks, it, shape)}
        print(json.dumps({"only": args.only, "shape": shape, "result": fns[args.only]()}), flush=True)
        return 0

    sampler = ClockSampler(local_rank) if rank == 0 else None
    head = bench_scan(torch, cla, workloads, dev, args.steps, args.warmup, dist_on)
    clocks = sampler.stop() if sampler else None

    step_ms = _max_over_ranks(torch, head["step_ms"], dist_on)
    bwd_ms = _max_over_ranks(torch, head["bwd_ms"], dist_on)
    fwd_ms = _max_over_ranks(torch, head["fwd_ms"], dist_on)
    e2e_ms = _max_over_ranks(torch, head["e2e_ms"], dist_on)
    bytes_step = head["bytes_fwd"] + head["bytes_bwd"]
    value = replica_throughput(world, bytes_step, step_ms)

    extra = {}
    if not args.headline_only and rank == 0:
        flush = Flusher(torch, dev)
        for key, fn in (
                ("scan_small", lambda: bench_scan_small(torch, cla, workloads, dev, flush, peaks)),
                ("scan_fwd_blelloch", lambda: bench_scan_blelloch(torch, cla, workloads, dev, flush, peaks)),
                ("scan_bwd_recompute", lambda: bench_scan_bwd_recompute(torch, cla, workloads, dev, flush, peaks)),
                ("selective", lambda: bench_selective(torch, cla, workloads, dev, flush, peaks)),
                ("la_const", lambda: bench_la(torch, cla, workloads, dev, flush, peaks, "la_const", 64)),
                ("la_long", lambda: bench_la(torch, cla, workloads, dev, flush, peaks, "la_long", 128, e2e_steps=3)),
                ("la_long_chunk64", lambda: bench_la(torch, cla, workloads, dev, flush, peaks, "la_long", 64)),
                ("gla", lambda: bench_gla(torch, cla, workloads, dev, flush, peaks)),
                ("delta", lambda: bench_delta(torch, cla, workloads, dev, flush, peaks))):
            try:
                extra[key] = fn()
            except Exception as e:  # an entry point without a kernel yet reports itself
                extra[key] = {"status": f"not measured: {type(e).__name__}: {str(e)[:160]}"}
            torch.cuda.empty_cache()

    if dist_on:
        import torch.distributed as dist

        dist.barrier()
    if rank != 0:
        return 0

    # roofline of the dominant kernel of the headline step
    dom = "scan_diag_bwd_kernel" if head["bwd_ms"] >= head["fwd_ms"] else "scan_diag_fwd_kernel"
    dom_ms = head["bwd_ms"] if dom == "scan_diag_bwd_kernel" else head["fwd_ms"]
    dom_bytes = head["bytes_bwd"] if dom == "scan_diag_bwd_kernel" else head["bytes_fwd"]
    achieved = dom_bytes / (dom_ms / 1e3) / 1e9
    tr = kernel_traffic(dom)
    roofline = {"bound": "hbm", "kernel": dom, "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4), "peak_source": peak_kind,
                "algorithmic_bytes_per_launch": dom_bytes,
                "traffic": (tr["dram_bytes_per_launch"] if tr else None),
                "other_kernel": {"kernel": "scan_diag_fwd_kernel" if dom != "scan_diag_fwd_kernel" else
                                 "scan_diag_bwd_kernel",
                                 "GBps": round((head["bytes_fwd"] if dom != "scan_diag_fwd_kernel" else head["bytes_bwd"])
                                               / ((fwd_ms if dom != "scan_diag_fwd_kernel" else bwd_ms) / 1e3) / 1e9, 1)}}

    cpu = None
    if not args.no_cpu_baseline:
        try:
            v, sample, cores = oracle_scan_sample(workloads)
            cpu = {"value": round(v, 3), "unit": "GB/s", "cores": cores, "kind": "oracle", "sample": sample}
        except Exception as e:
            cpu = {"value": None, "unit": "GB/s", "cores": os.cpu_count(), "kind": "oracle",
                   "sample": f"failed: {type(e).__name__}: {str(e)[:120]}"}

    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(step_ms, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": HEAD_WORKLOAD,
                   "B": head["B"], "T": head["T"], "D": head["D"], "l2": "flushed (256 MB write) before each timed step",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": {"value": round(replica_throughput(world, bytes_step, e2e_ms), 1), "unit": "GB/s",
                "h2d_bytes_per_step": head["h2d_bytes"], "d2h_bytes_per_step": head["d2h_bytes"]},
        "gpu_launches": head["launches"],
        "clocks": clocks,
        "fwd_ms": round(fwd_ms, 4), "bwd_ms": round(bwd_ms, 4),
        "workloads": extra,
    }
    print(json.dumps(line), flush=True)
    if dist_on:
        import torch.distributed as dist

        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
