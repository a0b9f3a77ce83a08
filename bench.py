"""Benchmark of the selective-scan hot path on GB300.

Headline: the Mamba-1 selective scan on a Mamba-130m-shaped layer (batch 8, d_inner
1536, d_state 16, L 2048, bf16 x/delta/z/B/C, fp32 state, SiLU gate), reported as
state updates per second (batch * L * d_inner * d_state / time) and as achieved HBM
GB/s against the measured copy bandwidth.  One step = one ssm_scan_fwd call over one
batch; several input sets (together larger than L2) rotate between steps.

The end-to-end figure ("e2e") runs the same scan through the public API with pinned host
buffers: every step copies its inputs in and y back inside the timed region, and the
host link's own rate for those bytes is measured beside it ("e2e.link_peak").

Also reported (in "paths"): the Mamba-2 chunked SSD (130m-shaped, chunk 64 and 256),
the decode update (780m-shaped, 1024 steps), multi-token decode, a decode serving loop
over a hybrid Mamba-1/Mamba-2 stack, the Mamba-1 backward (130m layer), the SSD backward
(130m SSD shape), the Mamba-3 scan (130m layer shape), S4D (recurrent form, FFT
convolution form and kernel) and the long-context Mamba-1 sweep.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line.  Under torchrun (N > 1) each rank runs its own batch (weak
scaling, no collective on the data path) and rank 0 prints the line.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from selective_scan_mamba_gb300 import synth  # noqa: E402

WORKLOAD = "m1_130m_layer"
METRIC = "scan state-updates/s (B*L*D*N) and achieved HBM GB/s as % of GB300 peak"
UNIT = "state-updates/s"


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            d = json.load(fh)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "source": "fallback"}


# ---------------------------------------------------------------------------------------
# algorithmic bytes and work
# ---------------------------------------------------------------------------------------
def m1_bytes(batch, dim, N, L, es_in=2, es_out=2, with_z=True, h_final=False):
    """Each input element read once, each output written once."""
    per_row = (2 + (1 if with_z else 0)) * es_in + es_out  # x, delta, (z) in; y out
    b = batch * dim * L * per_row + 2 * batch * N * L * es_in  # + B, C
    b += dim * N * 4 + dim * 8  # A, D, bias
    if h_final:
        b += batch * dim * N * 4
    return b


def ssd_bytes(batch, L, H, P, N, G, es=2, with_z=False):
    b = batch * L * H * P * es * (2 + (1 if with_z else 0))  # x, (z) in, y out
    b += batch * L * H * es  # dt
    b += 2 * batch * L * G * N * es  # B, C
    b += batch * H * P * N * 4  # h_final
    return b


def ssd_flops(batch, L, H, P, N, G, Q):
    """Dense per-chunk tile products: C.B^T (per group), (CB^T o L).X, chunk states, C.h."""
    nch = -(-L // Q)
    per_bhc = 2 * Q * Q * P + 2 * P * Q * N + 2 * Q * N * P
    per_bgc = 2 * Q * Q * N
    return batch * nch * (H * per_bhc + G * per_bgc)


# The roofline of the scan is HBM bandwidth: algorithmic bytes (each input read once, each
# output written once) over the measured copy rate.  Its arithmetic ceiling is reported
# beside it: the update h = exp(Delta A) h + (Delta x) B, y += C h needs at least one
# exponential (MUFU.EX2) and four FP32 FMA-pipe operations (Delta A, (Delta x) B, the state
# FMA, the C h FMA).  A GB300 SM retires 32 EX2 and 128 FP32 FMA lanes per clock (measured
# with a microbenchmark of independent ex2 / FFMA chains; the f32x2 forms save issue slots,
# not FP32 lanes), so both units cap the scan at 32 updates per SM clock.  At 1.99 updates
# per algorithmic byte (130m layer) that is ~75% of the HBM copy rate.
EX2_PER_CLK_SM = 32
FP32_LANES_PER_CLK_SM = 128
FP32_OPS_PER_UPDATE = 4


def alu_peak_updates(sms, sm_max_mhz):
    per_clk = min(EX2_PER_CLK_SM / 1.0, FP32_LANES_PER_CLK_SM / FP32_OPS_PER_UPDATE)
    return sms * sm_max_mhz * 1e6 * per_clk


def ssd_bwd_macs(batch, L, H, P, N, Q=64):
    """Multiply-adds of the chunked SSD backward: per (batch, head) and Q-step chunk,
    C B^T twice (Q^2 N each), the decayed-weight products of dB and dC (Q^2 N each),
    do x^T and the outputs' and dx's intra-chunk products (Q^2 P each), and six products
    with a chunk state or adjoint (Q N P each: the chunk state, the outputs' state term,
    the adjoint sum, and the state terms of dx, dB and dC)."""
    nch = -(-L // Q)
    return batch * H * nch * (4 * Q * Q * N + 3 * Q * Q * P + 6 * Q * N * P)


def fp32_fma_peak(sms, sm_max_mhz):
    """FP32 multiply-adds per second: 128 FMA lanes per SM clock."""
    return sms * sm_max_mhz * 1e6 * FP32_LANES_PER_CLK_SM


def bwd_bytes(batch, dim, N, L, G=1):
    """Backward of the Mamba-1 scan: x, delta, z, dy (bf16) and B, C read once; dx,
    ddelta, dz (float32) and dB, dC (float32) written once; A, D, bias and their
    gradients."""
    b = batch * dim * L * (4 * 2 + 3 * 4)
    b += batch * G * N * L * (2 * 2 + 2 * 4)
    b += dim * N * 8 + dim * 16
    return b


def step_bytes(batch, H, P, N, G, es=2, with_z=True):
    b = 2 * batch * H * P * N * 4  # state read + write
    b += batch * H * P * es * (2 + (1 if with_z else 0))  # x, z, y
    b += batch * H * es + 2 * batch * G * N * es
    return b


# ---------------------------------------------------------------------------------------
# clocks under load
# ---------------------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = None

    def __enter__(self):
        import tempfile
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        return False

    def summary(self):
        rows = []
        try:
            with open(self.path) as fh:
                for line in fh:
                    parts = [p.strip() for p in line.split(",")]
                    if len(parts) >= 8:
                        rows.append(parts)
        except Exception:
            pass
        finally:
            if self.path and os.path.exists(self.path):
                os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[0]) for r in rows if num(r[0]) is not None]
        mx = [num(r[1]) for r in rows if num(r[1]) is not None]
        pw = [num(r[2]) for r in rows if num(r[2]) is not None]
        loaded = [s for s, p in zip(sm, pw) if p is not None and p > 250.0] or sm
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = []
        for i, n in enumerate(names):
            if any(r[4 + i].lower() == "active" for r in rows):
                reasons.append(n)
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(rows),
                "power_w_max": max(pw) if pw else None}


# ---------------------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------------------
def _dev(inp, torch):
    out = {}
    for k, v in inp.arrays.items():
        if inp.dtypes[k] == synth.BF16:
            out[k] = torch.from_numpy(synth.bf16_bits(v).view(np.int16).copy()).cuda().view(
                torch.bfloat16)
        else:
            out[k] = torch.from_numpy(np.ascontiguousarray(v)).cuda()
    return out


def time_launches(torch, fn, n, warmup, stream):
    """Average device time of fn() over n calls, CUDA events on the launching stream."""
    for i in range(warmup):
        fn(i)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(n):
        fn(i)
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / 1e3 / n


def host_link_peak(torch, h_in, d_in, d_out, h_out, in_streams, out_stream, stream, reps):
    """Rate of the host link for one end-to-end step's transfers, the e2e leg's roofline.

    Copies the given pinned host tensors to device buffers, each on its own stream, while
    a device buffer of the output's size goes back to pinned host memory on another, and
    times `reps` repetitions with CUDA events.  `floor_ms` is the time one step's bytes
    need on this link with both directions busy at once; `h2d_gbs` and `d2h_gbs` are the
    one-direction rates."""
    def run(h2d, d2h):
        start = torch.cuda.Event()
        start.record(stream)
        evs = []
        if h2d:
            for cs, src, dst in zip(in_streams, h_in, d_in.values()):
                cs.wait_event(start)
                with torch.cuda.stream(cs):
                    dst.copy_(src, non_blocking=True)
                    ev = torch.cuda.Event()
                    ev.record(cs)
                evs.append(ev)
        if d2h:
            out_stream.wait_event(start)
            with torch.cuda.stream(out_stream):
                h_out.copy_(d_out, non_blocking=True)
                ev = torch.cuda.Event()
                ev.record(out_stream)
            evs.append(ev)
        for ev in evs:
            stream.wait_event(ev)

    def timed(h2d, d2h):
        run(h2d, d2h)
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            run(h2d, d2h)
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / 1e3 / reps

    bi = sum(t.numel() * t.element_size() for t in h_in)
    bo = h_out.numel() * h_out.element_size()
    t_both, t_in, t_out = timed(True, True), timed(True, False), timed(False, True)
    return {"floor_ms": t_both * 1e3, "both_gbs": (bi + bo) / t_both / 1e9,
            "h2d_gbs": bi / t_in / 1e9, "d2h_gbs": bo / t_out / 1e9,
            "source": "pinned host <-> device copies of one step's bytes, timed in this run"}


def max_over_ranks(dist, value, device):
    """The largest of the ranks' values (the job's time is its slowest rank's); the value
    itself when there is no process group."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank, world, t_max):
    """Weak scaling: every rank processes `units_per_rank` (its own batch); the job's rate
    is all ranks' units over the slowest rank's time."""
    return units_per_rank * world / t_max


def bench_ours(args, rank, world):
    import torch
    import selective_scan_mamba_gb300 as ssm

    dev = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(dev)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", dev))
    stream = torch.cuda.current_stream()
    peaks = measured_peaks()
    cfg = synth.WORKLOADS[WORKLOAD]
    Bt, D, N, L = cfg["batch"], cfg["dim"], cfg["dstate"], cfg["seqlen"]
    inp = synth.mamba1(Bt, D, N, L, dtype=cfg["dtype"], delta_scale=cfg["delta_scale"],
                       with_z=cfg["with_z"], seed=rank)
    base = _dev(inp, torch)
    # rotating input sets: together larger than L2 (129 MB), so no step reads another's
    # inputs from cache
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    set_bytes = m1_bytes(Bt, D, N, L)
    nsets = max(2, -(-3 * l2 // set_bytes))
    sets = []
    for k in range(nsets):
        s = {n: (torch.roll(t, shifts=17 * k, dims=-1).contiguous()
                 if n in ("x", "delta", "z", "B", "C") else t) for n, t in base.items()}
        s["y"] = torch.empty_like(s["x"])
        sets.append(s)
    torch.cuda.synchronize()

    def step(i):
        s = sets[i % nsets]
        ssm.ssm_scan_fwd(s["x"], s["delta"], s["A"], s["B"], s["C"], D=s["D"], z=s["z"],
                         delta_bias=s["delta_bias"], y=s["y"])

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    with ClockSampler(dev) as clk:
        torch.cuda.synchronize()
        if dist:
            dist.barrier()
        # one event between consecutive steps: the region from the first to the last is
        # exactly the K steps, and the gaps give the per-step times
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
        evs[0].record(stream)
        for i in range(args.steps):
            step(i)
            evs[i + 1].record(stream)
        torch.cuda.synchronize()
        if dist:
            dist.barrier()
        t_step = evs[0].elapsed_time(evs[-1]) / 1e3 / args.steps
        per_step = [evs[i].elapsed_time(evs[i + 1]) for i in range(args.steps)]
    clocks = clk.summary()
    t_step = max_over_ranks(dist, t_step, "cuda")
    updates = Bt * L * D * N
    value = whole_job_rate(updates, world, t_step)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    sm_max = clocks.get("sm_max_mhz") or 2070.0
    alu_peak = alu_peak_updates(sms, sm_max)
    gbs = set_bytes / t_step / 1e9
    launches_per_step = 2 if ssm.ssm_scan_workspace_size(sets[0]["x"], sets[0]["B"]) else 1

    # end to end through the public API with host buffers: every step copies its inputs
    # in from pinned host memory and its y back, inside the timed region.  Each input has
    # its own copy stream (concurrent host-to-device copies), y goes back on a stream of
    # its own (so the next scan does not queue behind the read-back), and the device
    # buffers rotate through --e2e-sets sets, so the copies of step i+1 overlap the scan and
    # read-back of step i; a copy into a set waits for the read-back that last used it.
    host = {n: t.cpu().pin_memory() for n, t in sets[0].items() if n in ("x", "delta", "z", "B", "C")}
    nbuf = max(2, args.e2e_sets)
    dbufs = [{n: torch.empty_like(sets[0][n]) for n in host} for _ in range(nbuf)]
    ybufs = [torch.empty_like(sets[0]["y"]) for _ in range(nbuf)]
    y_hosts = [torch.empty(sets[0]["y"].shape, dtype=sets[0]["y"].dtype).pin_memory() for _ in range(nbuf)]
    copy_streams = [torch.cuda.Stream() for _ in host]
    d2h_stream = torch.cuda.Stream()
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = y_hosts[0].numel() * y_hosts[0].element_size()
    last_use = [None] * nbuf

    def h2d_copies(k, start):
        buf, evs = dbufs[k], []
        for cs, (n, t) in zip(copy_streams, host.items()):
            if start is not None:
                cs.wait_event(start)
            if last_use[k] is not None:
                cs.wait_event(last_use[k])
            with torch.cuda.stream(cs):
                buf[n].copy_(t, non_blocking=True)
                ev = torch.cuda.Event()
                ev.record(cs)
            evs.append(ev)
        return buf, evs

    def e2e_step(i, start=None):
        k = i % nbuf
        buf, evs = h2d_copies(k, start)
        for ev in evs:
            stream.wait_event(ev)
        if last_use[k] is not None:
            stream.wait_event(last_use[k])  # ybufs[k] is free once its read-back is done
        s = sets[0]
        y = ssm.ssm_scan_fwd(buf["x"], buf["delta"], s["A"], buf["B"], buf["C"], D=s["D"],
                             z=buf["z"], delta_bias=s["delta_bias"], y=ybufs[k])
        scanned = torch.cuda.Event()
        scanned.record(stream)
        d2h_stream.wait_event(scanned)
        with torch.cuda.stream(d2h_stream):
            y_hosts[k].copy_(y, non_blocking=True)
            done = torch.cuda.Event()
            done.record(d2h_stream)
        last_use[k] = done

    e2e_steps = max(3, min(args.steps, 20))
    for i in range(nbuf):
        e2e_step(i)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(e2e_steps):
        e2e_step(i, start=e0 if i < nbuf else None)
    for ev in last_use:
        stream.wait_event(ev)  # the timed region ends after the last read-back
    e1.record(stream)
    torch.cuda.synchronize()
    t_e2e = max_over_ranks(dist, e0.elapsed_time(e1) / 1e3 / e2e_steps, "cuda")
    link = host_link_peak(torch, list(host.values()), dbufs[0], ybufs[0], y_hosts[0],
                          copy_streams, d2h_stream, stream, e2e_steps)

    paths = {}
    if rank == 0 and not args.headline_only:
        try:
            paths = other_paths(args, torch, ssm, peaks, stream, l2)
        except Exception as exc:  # a failing secondary path is reported, not fatal to the line
            paths = {"error": f"{type(exc).__name__}: {exc}"}

    result = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": t_step * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "Mamba-1 selective scan, Mamba-130m-shaped layer",
                   "batch": Bt, "d_inner": D, "d_state": N, "seq_len": L,
                   "inputs": "bf16 x, delta, z, B, C; fp32 A, D, bias; fp32 state; bf16 y",
                   "l2": f"{nsets} rotating input sets, {nsets * set_bytes / 1e6:.0f} MB > "
                         f"L2 {l2 / 1e6:.0f} MB",
                   "parallelism": f"replicas x{world} (independent batches per GPU)"},
        "ms_median": statistics.median(per_step),
        "ms_p95": percentile(per_step, 95),
        "hbm_gbs": gbs,
        "hbm_frac": gbs / peaks["hbm_gbs"],
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": gbs / peaks["hbm_gbs"],
                     "traffic": recorded_traffic("m1_scan_tmem"),
                     "kernel": "m1_scan_tmem", "bytes_per_launch": set_bytes,
                     "updates_per_launch": updates,
                     "peak_source": f"{peaks['source']} copy bandwidth (MEASURED_PEAKS.json hbm_gbs)",
                     "alu": {"achieved": updates / t_step / 1e9, "peak": alu_peak / 1e9,
                             "unit": "Gupd/s", "frac": updates / t_step / alu_peak,
                             "peak_source": f"derived: {sms} SMs x {sm_max:.0f} MHz x 32 updates/clk/SM "
                                            "(1 MUFU.EX2 + 4 FP32 FMA-pipe ops per update; 32 EX2 "
                                            "and 128 FP32 lanes per clk per SM, measured)"},
                     "paths": {}},
        "e2e": {"value": whole_job_rate(updates, world, t_e2e), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": t_e2e * 1e3,
                "link_gbs": (h2d + d2h) / t_e2e / 1e9,
                "link_peak": link, "link_frac": link["floor_ms"] / (t_e2e * 1e3), "buffer_sets": nbuf},
        "gpu_launches": args.steps * launches_per_step,
        "clocks": clocks,
        "meta": run_metadata(torch, dev, seed=rank),
        "paths": paths,
    }
    result["roofline"]["paths"] = path_rooflines(paths)
    if rank == 0 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(inp, budget_s=args.cpu_seconds)
    if dist:
        dist.destroy_process_group()
    return result


def percentile(xs, q):
    """The q-th percentile of xs by linear interpolation between order statistics."""
    v = sorted(xs)
    if not v:
        return None
    pos = (len(v) - 1) * q / 100.0
    lo = int(pos)
    hi = min(lo + 1, len(v) - 1)
    return v[lo] + (v[hi] - v[lo]) * (pos - lo)


def _run(cmd):
    try:
        return subprocess.run(cmd, capture_output=True, text=True, timeout=20,
                              cwd=ROOT).stdout.strip() or None
    except Exception:
        return None


def sources_digest():
    """sha256 (16 hex digits) of the library, oracle and bench sources: identifies the code
    a result was measured on where no git history is available (the GPU machine gets a copy of
    the tree without .git)."""
    import glob
    import hashlib
    h = hashlib.sha256()
    files = sorted(glob.glob(os.path.join(ROOT, "selective_scan_mamba_gb300", "csrc", "*")) +
                   glob.glob(os.path.join(ROOT, "include", "*.h")) +
                   glob.glob(os.path.join(ROOT, "oracle", "*.[ch]")) +
                   glob.glob(os.path.join(ROOT, "selective_scan_mamba_gb300", "*.py")) +
                   [os.path.abspath(__file__)])
    for f in files:
        with open(f, "rb") as fh:
            h.update(os.path.relpath(f, ROOT).encode() + fh.read())
    return h.hexdigest()[:16]


def run_metadata(torch, dev, seed):
    """The environment block that goes with every result: GPU, driver, CUDA, torch, seed,
    command, time, host and the code it ran."""
    import datetime
    import platform
    props = torch.cuda.get_device_properties(dev)
    drv = _run(["nvidia-smi", "-i", str(dev), "--query-gpu=driver_version", "--format=csv,noheader"])
    cpu = None
    try:
        with open("/proc/cpuinfo") as fh:
            for line in fh:
                if line.lower().startswith(("model name", "cpu part")):
                    cpu = line.split(":", 1)[1].strip()
                    break
    except OSError:
        pass
    return {"gpu": props.name, "sms": props.multi_processor_count, "driver": drv,
            "cuda_runtime": torch.version.cuda, "torch": torch.__version__,
            "seed": seed, "command": " ".join([os.path.basename(sys.executable)] + sys.argv),
            "utc": datetime.datetime.now(datetime.timezone.utc).strftime("%Y-%m-%dT%H:%M:%SZ"),
            "host": {"machine": platform.machine(), "cpu": cpu, "cores": os.cpu_count()},
            "git": _run(["git", "rev-parse", "--short=12", "HEAD"]),
            "sources_sha256": sources_digest()}


def path_rooflines(paths):
    """One roofline fraction per measured path (the SSD against max(HBM, bf16 tensor) time,
    the SSD backward against the FP32 FMA rate, the others against HBM), compact, so that
    the line's head carries them."""
    out = {}
    for q in ("64", "256"):
        r = paths.get(f"ssd_130m_chunk{q}")
        if r:
            out[f"ssd_130m_chunk{q}"] = {"bound": r["roofline_bound"], "frac": r["roofline_frac"],
                                         "ms": r["ms"]}
    r = paths.get("decode_780m")
    if r:
        out["decode_780m"] = {"bound": "hbm", "frac": r["hbm_frac"], "us": r["us_per_step"]}
    r = paths.get("ssd_130m_bwd")
    if r and "fma_frac" in r:
        out["ssd_130m_bwd"] = {"bound": "alu", "frac": r["fma_frac"], "ms": r["ms"]}
    r = paths.get("s4d_256")
    if r and "conv_hbm_frac" in r:
        out["s4d_256_conv"] = {"bound": "hbm", "frac": r["conv_hbm_frac"], "ms": r["conv_ms"]}
    for L, r in paths.get("m1_790m_long", {}).items():
        out[f"m1_790m_L{L}"] = {"bound": "hbm", "frac": r["hbm_frac"], "ms": r["ms"],
                                "alu_frac": r.get("alu_frac")}
    return out


def recorded_traffic(kernel):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on the
    current kernel source; otherwise None."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    src = _source_digest(kernel)
    try:
        with open(path) as fh:
            for line in fh:
                parts = line.split()
                if len(parts) >= 3 and parts[0] == kernel and parts[2] == src:
                    return float(parts[1])
    except OSError:
        pass
    return None


# the sources each recorded kernel is built from (its unit and the headers it includes)
KERNEL_SOURCES = {
    "m1_scan_tmem": ("scan_m1_tmem.cu", "common.cuh", "launch.h", "tcgen05.cuh", "tma.cuh",
                     "ssmscan.h"),
}


def _source_digest(kernel="m1_scan_tmem"):
    import hashlib
    h = hashlib.sha256()
    pkg = os.path.join(ROOT, "selective_scan_mamba_gb300", "csrc")
    for name in KERNEL_SOURCES[kernel]:
        path = os.path.join(pkg, name)
        if not os.path.exists(path):
            path = os.path.join(ROOT, "include", name)
        with open(path, "rb") as fh:
            h.update(name.encode() + fh.read())
    return h.hexdigest()[:16]


def other_paths(args, torch, ssm, peaks, stream, l2):
    out = {}
    hbm = peaks["hbm_gbs"]
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    # Mamba-2 chunked SSD, 130m-shaped
    c4 = synth.WORKLOADS["ssd_130m"]
    s_inp = synth.ssd(c4["batch"], c4["seqlen"], c4["nheads"], c4["headdim"], c4["dstate"],
                      c4["ngroups"], dtype=c4["dtype"], delta_scale=c4["delta_scale"], seed=0)
    t = _dev(s_inp, torch)
    nb = ssd_bytes(c4["batch"], c4["seqlen"], c4["nheads"], c4["headdim"], c4["dstate"],
                   c4["ngroups"])
    nsets = max(2, -(-3 * l2 // nb))
    sets = []
    for k in range(nsets):
        s = {n: (torch.roll(v, shifts=k, dims=1).contiguous() if n in ("x", "dt", "B", "C") else v)
             for n, v in t.items()}
        s["y"] = torch.empty_like(s["x"])
        s["hf"] = torch.empty((c4["batch"], c4["nheads"], c4["headdim"], c4["dstate"]),
                              dtype=torch.float32, device="cuda")
        sets.append(s)
    for Q in c4["chunks"]:
        ws = torch.empty(ssm.ssd_chunk_scan_workspace_size(sets[0]["x"], sets[0]["B"], Q),
                         dtype=torch.uint8, device="cuda")

        def f(i, Q=Q, ws=ws):
            s = sets[i % nsets]
            ssm.ssd_chunk_scan_fwd(s["x"], s["dt"], s["A"], s["B"], s["C"], Q, D=s["D"],
                                   dt_bias=s["dt_bias"], y=s["y"], h_final=s["hf"], workspace=ws)
        n = max(5, min(args.steps, 20))
        tsec = time_launches(torch, f, n, 3, stream)
        # dense per-chunk products at chunk Q (the roofline's count) and the products the
        # tensor-core kernels execute (64-step tiles for every Q)
        fl = ssd_flops(c4["batch"], c4["seqlen"], c4["nheads"], c4["headdim"], c4["dstate"],
                       c4["ngroups"], Q)
        fl_exec = ssd_flops(c4["batch"], c4["seqlen"], c4["nheads"], c4["headdim"],
                            c4["dstate"], c4["ngroups"], 64)
        t_hbm, t_tc = nb / (hbm * 1e9), fl / (peaks["bf16_tflops"] * 1e12)
        t_roof = max(t_hbm, t_tc)
        upd = c4["batch"] * c4["seqlen"] * c4["nheads"] * c4["headdim"] * c4["dstate"]
        out[f"ssd_130m_chunk{Q}"] = {
            "ms": tsec * 1e3, "state_updates_per_s": upd / tsec, "hbm_gbs": nb / tsec / 1e9,
            "tflops_executed": fl_exec / tsec / 1e12, "roofline_s": t_roof,
            "roofline_frac": t_roof / tsec, "roofline_bound": "hbm" if t_hbm >= t_tc else "tensor",
            "bytes": nb, "flops_dense_chunk": fl,
            "flops_executed": fl_exec}
    del sets
    # decode step, 780m-shaped: 4 layers' states rotate (each 100.7 MB; together > L2)
    c5 = synth.WORKLOADS["step_780m"]
    Bt, H, P, N, G = c5["batch"], c5["nheads"], c5["headdim"], c5["dstate"], c5["ngroups"]
    par = _dev(synth.step_params(H, N, seed=0), torch)
    states = [torch.from_numpy(synth.step_state(Bt, H, P, N, seed=k)).cuda() for k in range(4)]
    toks = [_dev(synth.step_tokens(Bt, H, P, N, G, step=k, seed=0), torch) for k in range(8)]
    y = torch.empty((Bt, H, P), dtype=torch.bfloat16, device="cuda")

    def g(i):
        tk = toks[i % 8]
        ssm.ssm_state_update(states[i % 4], tk["x"], tk["dt"], par["A"], tk["B"], tk["C"],
                             D=par["D"], z=tk["z"], dt_bias=par["dt_bias"], y=y)
    steps = c5["steps"]
    # the 1024-step decode is captured once in a CUDA graph and replayed
    gs = torch.cuda.Stream()
    gs.wait_stream(stream)
    with torch.cuda.stream(gs):
        for i in range(4):
            g(i)
    stream.wait_stream(gs)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for i in range(steps):
            g(i)
    graph.replay()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    graph.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    tstep = e0.elapsed_time(e1) / 1e3 / steps
    sb = step_bytes(Bt, H, P, N, G)
    out["decode_780m"] = {"us_per_step": tstep * 1e6, "steps": steps,
                          "state_updates_per_s": Bt * H * P * N / tstep,
                          "hbm_gbs": sb / tstep / 1e9, "hbm_frac": sb / tstep / 1e9 / hbm,
                          "bytes_per_step": sb, "note": "4 layer states rotate (403 MB > L2)"}
    del graph
    # multi-token decode: T tokens per call, the state read and written once per call
    tok_runs = {}
    for T in (4, 16):
        stk = {n: torch.stack([toks[k % 8][n] for k in range(T)]) for n in ("x", "dt", "B", "C", "z")}
        yT = torch.empty((T, Bt, H, P), dtype=torch.bfloat16, device="cuda")

        def gt(i, stk=stk, yT=yT):
            ssm.ssm_state_update_tokens(states[i % 4], stk["x"], stk["dt"], par["A"], stk["B"],
                                        stk["C"], D=par["D"], z=stk["z"], dt_bias=par["dt_bias"],
                                        y=yT)
        tcall = time_launches(torch, gt, 32, 4, stream)
        tb = 2 * Bt * H * P * N * 4 + T * (step_bytes(Bt, H, P, N, G) - 2 * Bt * H * P * N * 4)
        tok_runs[str(T)] = {"us_per_call": tcall * 1e6, "us_per_token": tcall * 1e6 / T,
                            "state_updates_per_s": T * Bt * H * P * N / tcall,
                            "hbm_gbs": tb / tcall / 1e9, "hbm_frac": tb / tcall / 1e9 / hbm,
                            "bytes_per_call": tb}
    out["decode_780m_tokens"] = dict(tok_runs, note="T consecutive tokens per call; 4 layer "
                                     "states rotate (403 MB > L2)")
    del states
    # serving loop over a hybrid stack: Mamba-1-form layers (790m-shaped: 3072 channels,
    # 16 states, A per state) alternate with Mamba-2-form layers (780m-shaped); one CUDA
    # graph of 256 tokens through all four layers, 8 token sets rotating
    c3 = synth.WORKLOADS["m1_790m_long"]
    stack = [(c3["dim"], 1, c3["dstate"], 1, True), (H, P, N, G, False)] * 2
    lays = []
    for li, (Hl, Pl, Nl, Gl, m1) in enumerate(stack):
        lays.append(dict(
            par=_dev(synth.step_params(Hl, Nl, a_per_state=m1, seed=li), torch),
            state=torch.from_numpy(synth.step_state(Bt, Hl, Pl, Nl, seed=li)).cuda(),
            toks=[_dev(synth.step_tokens(Bt, Hl, Pl, Nl, Gl, step=k, seed=li), torch)
                  for k in range(8)],
            y=torch.empty((Bt, Hl, Pl), dtype=torch.bfloat16, device="cuda")))

    def mixed_token(i):
        for lay in lays:
            tk, pr = lay["toks"][i % 8], lay["par"]
            ssm.ssm_state_update(lay["state"], tk["x"], tk["dt"], pr["A"], tk["B"], tk["C"],
                                 D=pr["D"], z=tk["z"], dt_bias=pr["dt_bias"], y=lay["y"])
    ntok = 256
    gs.wait_stream(stream)
    with torch.cuda.stream(gs):
        for i in range(2):
            mixed_token(i)
    stream.wait_stream(gs)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for i in range(ntok):
            mixed_token(i)
    graph.replay()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    graph.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    ttok = e0.elapsed_time(e1) / 1e3 / ntok
    mb = sum(step_bytes(Bt, Hl, Pl, Nl, Gl) for Hl, Pl, Nl, Gl, _ in stack)
    mupd = sum(Bt * Hl * Pl * Nl for Hl, Pl, Nl, Gl, _ in stack)
    out["decode_mixed_stack"] = {
        "us_per_token": ttok * 1e6, "tokens": ntok, "layers": len(stack),
        "state_updates_per_s": mupd / ttok, "hbm_gbs": mb / ttok / 1e9,
        "hbm_frac": mb / ttok / 1e9 / hbm, "bytes_per_token": mb,
        "note": f"batch {Bt}; Mamba-1 form {c3['dim']} channels x {c3['dstate']} states and "
                f"Mamba-2 form {H} x {P} x {N}, alternating; one CUDA graph of {ntok} tokens"}
    del graph, lays
    # Mamba-1 backward on the 130m layer: dy in, every gradient out (float32)
    c1 = synth.WORKLOADS["m1_130m_layer"]
    Bt1, D1, N1, L1 = c1["batch"], c1["dim"], c1["dstate"], c1["seqlen"]
    bsets = []
    for k in range(2):
        inp = synth.mamba1(Bt1, D1, N1, L1, dtype=c1["dtype"], delta_scale=c1["delta_scale"],
                           with_z=c1["with_z"], seed=20 + k)
        s = _dev(inp, torch)
        s["dy"] = torch.randn((Bt1, D1, L1), device="cuda").to(torch.bfloat16)
        bsets.append(s)
    bws = torch.empty(ssm.ssm_scan_bwd_workspace_size(bsets[0]["x"], bsets[0]["B"]),
                      dtype=torch.uint8, device="cuda")

    def fb(i):
        s = bsets[i % 2]
        ssm.ssm_scan_bwd(s["x"], s["delta"], s["A"], s["B"], s["C"], s["dy"], D=s["D"], z=s["z"],
                         delta_bias=s["delta_bias"], workspace=bws)
    tb = time_launches(torch, fb, max(3, min(args.steps, 10)), 2, stream)
    nbwd = bwd_bytes(Bt1, D1, N1, L1)
    out["m1_130m_bwd"] = {"ms": tb * 1e3, "state_updates_per_s": Bt1 * D1 * N1 * L1 / tb,
                          "hbm_gbs": nbwd / tb / 1e9, "bytes": nbwd,
                          "workspace_bytes": bws.numel(),
                          "note": "x, delta, z, dy bf16 in; dx, ddelta, dz, dA, dB, dC, dD, "
                                  "dbias float32 out; 2 input sets rotate"}
    del bsets, bws
    # SSD backward on the 130m SSD shape (batch 4, L 4096, 24 heads x 64, dstate 128)
    c4 = synth.WORKLOADS["ssd_130m"]
    sb_inp = synth.ssd(c4["batch"], c4["seqlen"], c4["nheads"], c4["headdim"], c4["dstate"],
                       c4["ngroups"], dtype=c4["dtype"], delta_scale=c4["delta_scale"], seed=60)
    sb = _dev(sb_inp, torch)
    sb_dy = torch.randn(sb["x"].shape, device="cuda").to(torch.bfloat16)
    sbws = torch.empty(max(1, ssm.ssd_scan_bwd_workspace_size(sb["x"], sb["B"])), dtype=torch.uint8,
                       device="cuda")

    def fsb(i):
        ssm.ssd_scan_bwd(sb["x"], sb["dt"], sb["A"], sb["B"], sb["C"], sb_dy, D=sb["D"],
                         dt_bias=sb["dt_bias"], workspace=sbws)
    tsb = time_launches(torch, fsb, 3, 1, stream)
    upd_sb = c4["batch"] * c4["seqlen"] * c4["nheads"] * c4["headdim"] * c4["dstate"]
    macs_sb = ssd_bwd_macs(c4["batch"], c4["seqlen"], c4["nheads"], c4["headdim"], c4["dstate"])
    out["ssd_130m_bwd"] = {"ms": tsb * 1e3, "state_updates_per_s": upd_sb / tsb,
                           "multiply_adds": macs_sb,
                           "fma_frac": macs_sb / tsb / fp32_fma_peak(sms, 2070.0),
                           "fma_peak_source": f"derived: {sms} SMs x 2070 MHz x 128 FP32 FMA lanes/clk/SM",
                           "workspace_bytes": sbws.numel(),
                           "note": "x, dt, B, C, dy bf16 in; every gradient float32 out; "
                                   "chunked form (64-step chunks, float32 products)"}
    del sb, sb_dy, sbws
    # Mamba-3 scan on the 130m layer shape (complex states, trapezoid weight lam)
    m3sets = []
    for k in range(2):
        inp = synth.mamba1(Bt1, D1, N1, L1, dtype=c1["dtype"], delta_scale=c1["delta_scale"],
                           with_z=c1["with_z"], seed=30 + k)
        s = _dev(inp, torch)
        s["A_im"] = 3.0 * torch.randn((D1, N1), device="cuda")
        s["lam"] = torch.rand((Bt1, D1, L1), device="cuda").to(torch.bfloat16)
        s["y"] = torch.empty_like(s["x"])
        m3sets.append(s)

    def fm3(i):
        s = m3sets[i % 2]
        ssm.ssm_mamba3_scan_fwd(s["x"], s["delta"], s["A"], s["A_im"], s["lam"], s["B"], s["C"],
                                D=s["D"], z=s["z"], delta_bias=s["delta_bias"], y=s["y"])
    tm3 = time_launches(torch, fm3, max(3, min(args.steps, 10)), 2, stream)
    nm3 = m1_bytes(Bt1, D1, N1, L1) + Bt1 * D1 * L1 * 2 + D1 * N1 * 4  # + lam, A_im
    out["m3_130m"] = {"ms": tm3 * 1e3, "state_updates_per_s": Bt1 * D1 * N1 * L1 / tm3,
                      "hbm_gbs": nm3 / tm3 / 1e9, "bytes": nm3,
                      "note": "complex states; x, delta, lam, z, B, C bf16; 2 input sets rotate"}
    del m3sets
    # S4D recurrent form and convolution kernel, the pages' efficiency-sweep shape
    # (batch 8, d_model 256), 32 complex states, L 4096
    Bs, Ds, Ns, Ls = 8, 256, 32, 4096
    g = torch.Generator(device="cuda").manual_seed(40)
    s4 = {"log_dt": torch.empty(Ds, device="cuda").uniform_(float(np.log(1e-3)), float(np.log(1e-1)),
                                                              generator=g),
          "A": torch.stack([torch.full((Ds, Ns), -0.5, device="cuda"),
                            (np.pi * torch.arange(Ns, device="cuda", dtype=torch.float32)).expand(Ds, Ns)],
                           dim=-1).contiguous(),
          "B": torch.stack([torch.ones(Ds, Ns, device="cuda"), torch.zeros(Ds, Ns, device="cuda")],
                           dim=-1).contiguous(),
          "C": torch.randn(Ds, Ns, 2, device="cuda", generator=g),
          "D": torch.randn(Ds, device="cuda", generator=g)}
    us = [torch.randn(Bs, Ds, Ls, device="cuda", generator=g).to(torch.bfloat16) for _ in range(2)]
    ys = torch.empty_like(us[0])

    def fs(i):
        ssm.ssm_s4d_scan_fwd(us[i % 2], s4["log_dt"], s4["A"], s4["B"], s4["C"], D=s4["D"], y=ys)
    ts = time_launches(torch, fs, max(3, min(args.steps, 10)), 2, stream)
    Kbuf = torch.empty((Ds, Ls), dtype=torch.float32, device="cuda")
    tk = time_launches(torch, lambda i: ssm.ssm_s4d_kernel(s4["log_dt"], s4["A"], s4["B"], s4["C"],
                                                           Ls, out=Kbuf), 3, 1, stream)
    # the convolution form: K, its spectrum and the FFT convolution (three launches)
    cws = torch.empty(ssm.ssm_s4d_conv_workspace_size(us[0], s4["log_dt"], s4["A"], s4["B"], s4["C"]),
                      dtype=torch.uint8, device="cuda")
    tc_ = time_launches(torch, lambda i: ssm.ssm_s4d_conv_fwd(us[i % 2], s4["log_dt"], s4["A"], s4["B"],
                                                              s4["C"], D=s4["D"], y=ys, workspace=cws),
                        max(3, min(args.steps, 10)), 2, stream)
    # algorithmic bytes of the convolution call: u in, y out (bf16), K and its spectrum
    # written and read once (float32, complex64 of the padded length)
    nfft = 1 << (2 * Ls - 1).bit_length()
    cbytes = 2 * Bs * Ds * Ls * 2 + Ds * Ls * 4 * 2 + Ds * nfft * 8 * 2
    out["s4d_256"] = {"scan_ms": ts * 1e3, "state_updates_per_s": Bs * Ds * Ns * Ls / ts,
                      "scan_hbm_gbs": Bs * Ds * Ls * 4 / ts / 1e9, "kernel_ms": tk * 1e3,
                      "conv_ms": tc_ * 1e3, "conv_hbm_gbs": cbytes / tc_ / 1e9,
                      "conv_hbm_frac": cbytes / tc_ / 1e9 / hbm,
                      "shape": f"batch {Bs}, dim {Ds}, N {Ns} complex, L {Ls}; bf16 u, y"}
    del us, ys, Kbuf
    # long-context Mamba-1 sweep, 790m-shaped (batch 1, d_inner 3072, no z, h_final out)
    c3 = synth.WORKLOADS["m1_790m_long"]
    sweep = {}
    for L in c3["seqlens"]:
        inp = synth.mamba1(1, c3["dim"], c3["dstate"], L, dtype=c3["dtype"],
                           delta_scale=c3["delta_scale"], with_z=False, seed=0)
        t0 = _dev(inp, torch)
        nbytes = m1_bytes(1, c3["dim"], c3["dstate"], L, with_z=False, h_final=True)
        # rotate input copies (shifted in time) until the working set exceeds L2 three times
        nsets = max(2, -(-3 * l2 // nbytes))
        sets = [{n: (torch.roll(v, shifts=k, dims=-1).contiguous() if n in ("x", "delta", "B", "C")
                     else v) for n, v in t0.items()} for k in range(nsets)]
        yb = torch.empty_like(t0["x"])
        hf = torch.empty((1, c3["dim"], c3["dstate"]), dtype=torch.float32, device="cuda")
        wsb = ssm.ssm_scan_workspace_size(t0["x"], t0["B"])
        ws = torch.empty(max(wsb, 1), dtype=torch.uint8, device="cuda")

        def m(i, yb=yb, hf=hf, ws=ws, sets=sets, nsets=nsets):
            tt = sets[i % nsets]
            ssm.ssm_scan_fwd(tt["x"], tt["delta"], tt["A"], tt["B"], tt["C"], D=tt["D"],
                             delta_bias=tt["delta_bias"], y=yb, h_final=hf, workspace=ws)
        tsec = time_launches(torch, m, max(5, nsets), 2, stream)
        upd3 = c3["dim"] * c3["dstate"] * L
        sweep[str(L)] = {"ms": tsec * 1e3, "state_updates_per_s": upd3 / tsec,
                         "hbm_gbs": nbytes / tsec / 1e9, "hbm_frac": nbytes / tsec / 1e9 / hbm,
                         "alu_frac": upd3 / tsec / alu_peak_updates(sms, 2070.0),
                         "input_sets": nsets, "workspace_bytes": wsb}
        del t0, sets, yb, hf, ws
    out["m1_790m_long"] = sweep
    return out


# ---------------------------------------------------------------------------------------
# CPU baseline: the float64 oracle, as it stands, on a bounded sample of the workload
# ---------------------------------------------------------------------------------------
def cpu_baseline(inp, budget_s=10.0):
    import oracle
    oracle.build()
    f = inp.f64
    dims = inp.dims
    D, N, L = dims["dim"], dims["dstate"], dims["seqlen"]
    x, dl, z = f("x"), f("delta"), f("z")
    B, C, A, Dv, bias = f("B"), f("C"), f("A"), f("D"), f("delta_bias")

    batch = dims["batch"]

    def run(nb):
        t0 = time.perf_counter()
        oracle.mamba1_scan(x[:nb], dl[:nb], A, B[:nb], C[:nb], D=Dv,
                           z=None if z is None else z[:nb], delta_bias=bias)
        return time.perf_counter() - t0

    # whole batch rows of the workload, repeated until about budget_s of CPU time
    nb, reps, total = 1, 0, 0.0
    first = run(1)
    nb = max(1, min(batch, int(budget_s / max(first, 1e-3) / 4)))
    while total < budget_s and reps < 64:
        total += run(nb)
        reps += 1
    upd = reps * nb * D * L * N
    # the same oracle on one thread, on a sample of channels of one batch row (about a
    # third of the budget)
    oracle.set_num_threads(1)
    try:
        def run1(nch):
            t0 = time.perf_counter()
            oracle.mamba1_scan(x[:1, :nch], dl[:1, :nch], A[:nch], B[:1], C[:1], D=Dv[:nch],
                               z=None if z is None else z[:1, :nch], delta_bias=bias[:nch])
            return time.perf_counter() - t0
        t8 = run1(8)
        nch = max(8, min(D, int(budget_s / 3 / max(t8, 1e-4) * 8)))
        t1 = run1(nch)
    finally:
        oracle.set_num_threads(0)
    return {"value": upd / total, "unit": UNIT, "cores": oracle.num_threads(),
            "kind": "oracle",
            "sample": f"{reps} x {nb} batch rows ({nb * D} channels x {L} steps x {N} states), "
                      f"float64 sequential oracle, {total:.1f} s",
            "single_thread": {"value": nch * L * N / t1, "unit": UNIT, "cores": 1,
                              "sample": f"{nch} channels of one batch row x {L} steps x {N} "
                                        f"states, {t1:.1f} s"}}


def bench_reference(args, rank, world):
    """The reference arm is the float64 CPU oracle on this workload (each step a bounded
    sample), timed on the host cores; rank 0 only."""
    if rank != 0:
        return None
    cfg = synth.WORKLOADS[WORKLOAD]
    inp = synth.mamba1(1, cfg["dim"], cfg["dstate"], cfg["seqlen"], dtype=cfg["dtype"],
                       delta_scale=cfg["delta_scale"], with_z=cfg["with_z"], seed=0)
    import oracle
    oracle.build()
    f = inp.f64
    nch = 96
    args_ = (f("x")[:, :nch], f("delta")[:, :nch], f("A")[:nch], f("B"), f("C"))
    kw = dict(D=f("D")[:nch], z=f("z")[:, :nch], delta_bias=f("delta_bias")[:nch])
    for _ in range(args.warmup):
        oracle.mamba1_scan(*args_, **kw)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.mamba1_scan(*args_, **kw)
    dt = (time.perf_counter() - t0) / args.steps
    L, N = cfg["seqlen"], cfg["dstate"]
    value = nch * L * N / dt
    sample = f"{nch} channels of one batch row per step ({L} steps x {N} states), float64 oracle"
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": "Mamba-1 selective scan, Mamba-130m-shaped layer",
                       "batch": cfg["batch"], "d_inner": cfg["dim"], "d_state": N, "seq_len": L},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.num_threads(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def run_case(args):
    """Runs one kernel workload --warmup + --steps times with no timing (for profiler
    captures): m1 (130m layer), m1_long (790m, L 32768), ssd64 / ssd256 (130m SSD),
    step (780m decode), bwd / ssd_bwd (the backwards on the 130m shapes) and the others
    named in --case."""
    import torch
    import selective_scan_mamba_gb300 as ssm
    torch.cuda.set_device(0)
    n = args.warmup + args.steps
    if args.case in ("m1", "m1_long"):
        cfg = synth.WORKLOADS["m1_130m_layer" if args.case == "m1" else "m1_790m_long"]
        L = cfg["seqlen"] if args.case == "m1" else 32768
        inp = synth.mamba1(cfg["batch"], cfg["dim"], cfg["dstate"], L, dtype=cfg["dtype"],
                           delta_scale=cfg["delta_scale"], with_z=cfg["with_z"], seed=0)
        t = _dev(inp, torch)
        y = torch.empty_like(t["x"])
        for _ in range(n):
            ssm.ssm_scan_fwd(t["x"], t["delta"], t["A"], t["B"], t["C"], D=t["D"], z=t.get("z"),
                             delta_bias=t["delta_bias"], y=y)
    elif args.case in ("ssd64", "ssd256"):
        c4 = synth.WORKLOADS["ssd_130m"]
        Q = 64 if args.case == "ssd64" else 256
        inp = synth.ssd(c4["batch"], c4["seqlen"], c4["nheads"], c4["headdim"], c4["dstate"],
                        c4["ngroups"], dtype=c4["dtype"], delta_scale=c4["delta_scale"], seed=0)
        t = _dev(inp, torch)
        y = torch.empty_like(t["x"])
        for _ in range(n):
            ssm.ssd_chunk_scan_fwd(t["x"], t["dt"], t["A"], t["B"], t["C"], Q, D=t["D"],
                                   dt_bias=t["dt_bias"], y=y)
    elif args.case == "step":
        c5 = synth.WORKLOADS["step_780m"]
        Bt, H, P, N, G = c5["batch"], c5["nheads"], c5["headdim"], c5["dstate"], c5["ngroups"]
        par = _dev(synth.step_params(H, N, seed=0), torch)
        states = [torch.from_numpy(synth.step_state(Bt, H, P, N, seed=k)).cuda() for k in range(4)]
        tok = _dev(synth.step_tokens(Bt, H, P, N, G, step=0, seed=0), torch)
        y = torch.empty((Bt, H, P), dtype=torch.bfloat16, device="cuda")
        for i in range(n):
            ssm.ssm_state_update(states[i % 4], tok["x"], tok["dt"], par["A"], tok["B"], tok["C"],
                                 D=par["D"], z=tok["z"], dt_bias=par["dt_bias"], y=y)
    elif args.case == "step_m1":  # Mamba-1-form decode: batch 64, 3072 channels x 16 states
        c5 = synth.WORKLOADS["step_780m"]
        c3 = synth.WORKLOADS["m1_790m_long"]
        Bt, H, N = c5["batch"], c3["dim"], c3["dstate"]
        par = _dev(synth.step_params(H, N, a_per_state=True, seed=0), torch)
        states = [torch.from_numpy(synth.step_state(Bt, H, 1, N, seed=k)).cuda() for k in range(4)]
        tok = _dev(synth.step_tokens(Bt, H, 1, N, 1, step=0, seed=0), torch)
        y = torch.empty((Bt, H, 1), dtype=torch.bfloat16, device="cuda")
        for i in range(n):
            ssm.ssm_state_update(states[i % 4], tok["x"], tok["dt"], par["A"], tok["B"], tok["C"],
                                 D=par["D"], z=tok["z"], dt_bias=par["dt_bias"], y=y)
    elif args.case == "bwd":  # Mamba-1 backward, 130m layer
        cfg = synth.WORKLOADS["m1_130m_layer"]
        inp = synth.mamba1(cfg["batch"], cfg["dim"], cfg["dstate"], cfg["seqlen"], dtype=cfg["dtype"],
                           delta_scale=cfg["delta_scale"], with_z=cfg["with_z"], seed=0)
        t = _dev(inp, torch)
        dy = torch.randn(t["x"].shape, device="cuda").to(torch.bfloat16)
        for _ in range(n):
            ssm.ssm_scan_bwd(t["x"], t["delta"], t["A"], t["B"], t["C"], dy, D=t["D"], z=t["z"],
                             delta_bias=t["delta_bias"])
    elif args.case == "ssd_bwd":  # SSD backward, 130m SSD shape
        cfg = synth.WORKLOADS["ssd_130m"]
        inp = synth.ssd(cfg["batch"], cfg["seqlen"], cfg["nheads"], cfg["headdim"], cfg["dstate"],
                        cfg["ngroups"], dtype=cfg["dtype"], delta_scale=cfg["delta_scale"], seed=60)
        t = _dev(inp, torch)
        dy = torch.randn(t["x"].shape, device="cuda").to(torch.bfloat16)
        for _ in range(n):
            ssm.ssd_scan_bwd(t["x"], t["dt"], t["A"], t["B"], t["C"], dy, D=t["D"], dt_bias=t["dt_bias"])
    elif args.case == "m3":  # Mamba-3 scan, 130m layer shape
        cfg = synth.WORKLOADS["m1_130m_layer"]
        inp = synth.mamba1(cfg["batch"], cfg["dim"], cfg["dstate"], cfg["seqlen"], dtype=cfg["dtype"],
                           delta_scale=cfg["delta_scale"], with_z=cfg["with_z"], seed=0)
        t = _dev(inp, torch)
        A_im = 3.0 * torch.randn(t["A"].shape, device="cuda")
        lam = torch.rand(t["x"].shape, device="cuda").to(torch.bfloat16)
        for _ in range(n):
            ssm.ssm_mamba3_scan_fwd(t["x"], t["delta"], t["A"], A_im, lam, t["B"], t["C"], D=t["D"],
                                    z=t["z"], delta_bias=t["delta_bias"])
    elif args.case in ("s4d", "s4d_conv"):  # S4D, batch 8, d_model 256, 32 states, L 4096
        Ds, Ns = 256, 32
        log_dt = torch.empty(Ds, device="cuda").uniform_(float(np.log(1e-3)), float(np.log(1e-1)))
        A = torch.stack([torch.full((Ds, Ns), -0.5, device="cuda"),
                         (np.pi * torch.arange(Ns, device="cuda", dtype=torch.float32)).expand(Ds, Ns)],
                        dim=-1).contiguous()
        Bm = torch.stack([torch.ones(Ds, Ns, device="cuda"), torch.zeros(Ds, Ns, device="cuda")],
                         dim=-1).contiguous()
        Cm = torch.randn(Ds, Ns, 2, device="cuda")
        u = torch.randn(8, Ds, 4096, device="cuda").to(torch.bfloat16)
        for _ in range(n):
            if args.case == "s4d":  # recurrent form
                ssm.ssm_s4d_scan_fwd(u, log_dt, A, Bm, Cm)
            else:  # FFT convolution form
                ssm.ssm_s4d_conv_fwd(u, log_dt, A, Bm, Cm)
    elif args.case == "tokens":  # 16 decode tokens per call, one state buffer
        c5 = synth.WORKLOADS["step_780m"]
        Bt, H, P, N, G = c5["batch"], c5["nheads"], c5["headdim"], c5["dstate"], c5["ngroups"]
        T = 16
        par = _dev(synth.step_params(H, N, seed=0), torch)
        state = torch.from_numpy(synth.step_state(Bt, H, P, N, seed=0)).cuda()
        toks = [_dev(synth.step_tokens(Bt, H, P, N, G, step=k, seed=0), torch) for k in range(T)]
        stk = {n: torch.stack([tk[n] for tk in toks]) for n in ("x", "dt", "B", "C", "z")}
        y = torch.empty((T, Bt, H, P), dtype=torch.bfloat16, device="cuda")
        for _ in range(n):
            ssm.ssm_state_update_tokens(state, stk["x"], stk["dt"], par["A"], stk["B"], stk["C"],
                                        D=par["D"], z=stk["z"], dt_bias=par["dt_bias"], y=y)
    else:
        raise SystemExit(f"unknown case {args.case}")
    torch.cuda.synchronize()
    print("done")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--headline-only", action="store_true",
                    help="skip the SSD, decode and long-context measurements")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--e2e-sets", type=int, default=3,
                    help="device buffer sets the end-to-end leg rotates through (>= 2)")
    ap.add_argument("--case", choices=["m1", "m1_long", "ssd64", "ssd256", "step", "step_m1", "tokens",
                                       "bwd", "ssd_bwd", "m3", "s4d", "s4d_conv"],
                    help="run one kernel workload untimed (for profiler captures) and exit")
    args = ap.parse_args()
    if args.case:
        run_case(args)
        return
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if args.impl == "reference":
        res = bench_reference(args, rank, world)
    else:
        res = bench_ours(args, rank, world)
    if rank == 0 and res is not None:
        print(json.dumps(res))


if __name__ == "__main__":
    main()
