#!/usr/bin/env python3
"""Benchmark of the gated temporal scan layer: forward + backward on GB300.

One step = m2scan_fwd + m2scan_bwd over one batch of the 8192-sample workload
(K=8, SH2=256, D=16, fp32), inputs resident in HBM. L2 is flushed (a 512 MiB
write, then a 512 MiB read of another buffer, so that the write's dirty lines
are back in HBM too) before every timed forward and every timed backward,
outside the timed intervals, so both read their inputs from HBM. Each rank times K steps
with CUDA events on its stream; the line reports the maximum over ranks.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl native|reference]
                  [--workload pages|long_history|wide_state|stress|tiny|bias_fc|...]

Prints one JSON line (rank 0). ``--impl reference`` times the fp64 CPU oracle
(the only reference the layer has) on the host cores instead. The ``bias_*``
workloads time the bias-gradient column sum (m2scan_bias_grad) instead of the
layer: one step = one call over dy [N, C], L2 flushed before each.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

UNIT = "samples/s"
FLUSH_BYTES = 512 << 20
L2_NOTE = ("flushed before every timed call: a 512 MiB write, then a 512 MiB read of another "
           "buffer (no dirty flush lines left for the timed call to write back)")


class L2Flush:
    """Evicts L2 (129 MB): writes a 512 MiB buffer, then reads another of the
    same size, so that the timed call finds neither its inputs nor dirty
    lines of the flush in L2."""

    def __init__(self, torch, dev):
        self.torch = torch
        self.w = torch.empty(FLUSH_BYTES // 4, device=dev, dtype=torch.float32)
        self.r = torch.ones(FLUSH_BYTES // 4, device=dev, dtype=torch.float32)
        self.sink = torch.empty((), device=dev, dtype=torch.float32)

    def __call__(self):
        self.w.zero_()
        self.torch.sum(self.r, dim=(0,), out=self.sink)
CLOCK_QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,utilization.gpu,"
               "clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
               "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
               "clocks_event_reasons.sw_power_cap")


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--workload", default="pages")
    ap.add_argument("--e2e-steps", type=int, default=100)
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--dtype", choices=["f32", "bf16"], default="f32",
                    help="activations (h_history, h_s2, d_h_enriched and the layer's outputs) "
                         "in fp32 or bfloat16; arithmetic is fp32 either way")
    return ap.parse_args(argv)


# ------------------------------------------------------------ multi-rank plumbing

def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


def init_dist(world: int, backend: str):
    if world <= 1:
        return None
    import torch.distributed as dist
    if not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend)
    return dist


def barrier(dist, device=None):
    if dist is not None:
        if device is not None and dist.get_backend() == "nccl":
            dist.barrier(device_ids=[device])
        else:
            dist.barrier()


def max_over_ranks(dist, values, device="cpu"):
    """Elementwise maximum of a list of floats over all ranks."""
    if dist is None:
        return list(values)
    import torch
    t = torch.tensor(list(values), dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.cpu()]


def whole_job_throughput(units_per_rank: int, world: int, seconds_max: float) -> float:
    """Units processed by all ranks divided by the slowest rank's time."""
    return units_per_rank * world / seconds_max if seconds_max > 0 else 0.0


# ------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi clock/throttle samples every 200 ms while the timed region runs."""

    def __init__(self):
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "--query-gpu=" + CLOCK_QUERY,
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
            return
        # nvidia-smi's start-up (driver and NVML initialisation) can hold up
        # the GPU for seconds: let it finish, i.e. wait for its first sample,
        # before the timed region begins
        t0 = time.time()
        while time.time() - t0 < 15.0 and self.proc.poll() is None:
            try:
                if os.path.getsize(self.path) > 0:
                    break
            except OSError:
                pass
            time.sleep(0.05)

    def stop(self, gpus):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                p = [s.strip() for s in line.split(",")]
                if len(p) < 10:
                    continue
                try:
                    rows.append(dict(idx=int(p[0]), sm=float(p[1]), smax=float(p[2]),
                                     util=float(p[4]) if p[4] not in ("[N/A]", "") else 0.0,
                                     hw=p[6], hwt=p[7], swt=p[8], swp=p[9]))
                except ValueError:
                    continue
        os.unlink(self.path)
        rows = [r for r in rows if r["idx"] in gpus] or rows
        load = [r for r in rows if r["util"] >= 50.0] or rows
        reasons = set()
        for r in load:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                              ("swt", "sw_thermal_slowdown"), ("swp", "sw_power_cap")):
                if r[key].lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median([r["sm"] for r in load]) if load else None,
                "sm_max_mhz": max((r["smax"] for r in load), default=None),
                "reasons": sorted(reasons), "samples": len(load)}


# ------------------------------------------------------------------ helpers

def metric_for(w) -> str:
    """The headline metric's name, with the workload's own dimensions."""
    return "fwd+bwd samples/s (B=%d, K=%d, SH2=%d, D=%d)" % (w.B, w.K, w.SH2, w.D)


def layer_config(w, world: int, activations: str) -> dict:
    """The workload's config, the same dict on both arms (the native line and
    the oracle's reference line); ``l2`` states how the native arm's timed
    calls treat L2."""
    return {"workload": "%s: B=%d K=%d SH2=%d D=%d tw=%g" % (w.name, w.B, w.K, w.SH2, w.D, w.tw),
            "B": w.B, "K": w.K, "SH2": w.SH2, "D": w.D, "parallelism": "replicas x%d" % world,
            "activations": activations, "l2": L2_NOTE}


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


# nominal dense tensor rates (PFLOP/s): tf32 1.1, bf16 2.25
TF32_PER_BF16 = 1.1 / 2.25


def fp32_product_peak():
    """TFLOP/s of fp32-accurate products on the tensor cores: the bf16 burst
    peak (measured, else the fallback 1.9 PFLOP/s) times the nominal
    tf32:bf16 ratio, divided by 3 for the three tf32 products of a 3 x TF32
    split. Returns (peak, source)."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            bf16, src = float(json.load(f)["bf16_tflops"]), "measured"
    except (OSError, KeyError, ValueError):
        bf16, src = 1900.0, "fallback"
    return bf16 * TF32_PER_BF16 / 3.0, src


def kernel_sources_sha() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "gated_ssm_temporal_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + b"\0" + f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str):
    """DRAM bytes per launch from the committed ncu summary, if it matches this
    source: (reads + writes, the record) or (None, None)."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            t = json.load(f)[kernel]
        if t.get("kernel_sha") == kernel_sources_sha():
            return float(t["dram_bytes_per_launch"]), t
    except (OSError, KeyError, ValueError):
        pass
    return None, None


def traffic_fields(kernel: str, alg_read: float, alg_write: float) -> dict:
    """roofline.traffic and the fields that say what it counts. DRAM writes are
    counted when L2 evicts them: output lines still dirty in L2 when the kernel
    ends are written back during the next kernel, so a one-launch capture can
    show fewer write bytes than the kernel stored. Reads are complete."""
    total, rec = recorded_traffic(kernel)
    out = {"traffic": total, "traffic_algorithmic_read": alg_read,
           "traffic_algorithmic_write": alg_write}
    if rec is None:
        out["traffic_note"] = "no capture of the current kernel sources"
        return out
    rd, wr = float(rec["dram_bytes_read"]), float(rec["dram_bytes_write"])
    out.update({"traffic_read": rd, "traffic_write_evicted": wr,
                "traffic_read_over_algorithmic": rd / alg_read if alg_read else None,
                "traffic_write_left_in_l2": max(0.0, alg_write - wr),
                "traffic_note": "traffic = DRAM reads + DRAM writes seen during the launch; "
                                "writes still dirty in L2 at its end reach DRAM later and are "
                                "not counted (traffic_write_left_in_l2 = algorithmic writes - "
                                "evicted writes)"})
    if "l2_write_bytes_from_sm" in rec:
        out["traffic_l2_write_from_sm"] = float(rec["l2_write_bytes_from_sm"])
    return out


def cpu_baseline(x, seconds: float, gpu_out=None, act_bound=None):
    """The fp64 oracle on this host's cores, repeated on the workload batch for
    ~seconds. ``gpu_out``: the outputs of the last timed GPU step, which are
    then checked against the oracle's result of the same inputs (``x`` holds
    the values the GPU read); ``act_bound``: relative bound of the activation
    outputs (None: the layer's fp32 criterion)."""
    import oracle
    threads = oracle.default_threads()
    B = x["h_history"].shape[0]
    done, t0 = 0, time.perf_counter()
    while True:
        oracle.forward(x["h_history"], x["h_s2"], x["W_A"], x["W_B"], x["W_C"], x["W_O"],
                       x["tw"], n_threads=threads)
        oracle.backward(x["h_history"], x["h_s2"], x["W_A"], x["W_B"], x["W_C"], x["W_O"],
                        x["tw"], x["d_h_enriched"], n_threads=threads)
        done += B
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    res = {"value": done / el, "unit": UNIT, "cores": threads, "kind": "oracle",
           "sample": "%d passes of fwd+bwd over the full %d-sample batch (%.1f s)"
                     % (done // B, B, el)}
    if gpu_out is not None:
        res["output_check"] = check_outputs(x, gpu_out, act_bound)
    return res


def check_outputs(x, gpu_out, act_bound=None):
    """Every output of the last timed step against the oracle, with the parity
    criteria of the tests (tests/tolerance.py): activation outputs element by
    element, weight gradients on the bound from their sums of |terms|."""
    import numpy as np
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import tolerance
    import oracle
    y, ya = oracle.forward(x["h_history"], x["h_s2"], x["W_A"], x["W_B"], x["W_C"], x["W_O"],
                           x["tw"], abs_terms=True)
    ref = {"h_enriched": y}
    ref.update(oracle.backward(x["h_history"], x["h_s2"], x["W_A"], x["W_B"], x["W_C"],
                               x["W_O"], x["tw"], x["d_h_enriched"], abs_terms=True))
    B, K, SH2 = x["h_history"].shape
    D = x["W_A"].shape[1]
    out = {}
    ok = True
    for n, got in gpu_out.items():
        got = np.asarray(got, dtype=np.float64)
        if n in ("dW_A", "dW_B", "dW_C", "dW_O"):
            r = tolerance.compare(n, got, ref[n], ref[n + "_abs"],
                                  tolerance.coefficient(n, B, K, SH2, D))
        elif act_bound is not None:
            err = np.abs(got - ref[n])
            bound = act_bound * np.abs(ref[n]) + tolerance.ATOL
            r = {"n_fail": int((err > bound).sum()),
                 "max_err_over_bound": float((err / bound).max()) if err.size else 0.0}
        else:
            r = tolerance.compare(n, got, ref[n])
        ok = ok and r["n_fail"] == 0
        out[n] = {"n_fail": r["n_fail"], "max_err_over_bound": r["max_err_over_bound"]}
    out["pass"] = ok
    return out


# -------------------------------------------------------------- native arm

def run_native(args, rank, world, local):
    import numpy as np
    import torch

    import gated_ssm_temporal_gb300 as g
    from gated_ssm_temporal_gb300 import build as gbuild
    from gated_ssm_temporal_gb300.workloads import (WORKLOADS, algorithmic_bytes, algorithmic_flops,
                                                    make_inputs)

    torch.cuda.set_device(local)
    dist = init_dist(world, "nccl")
    gbuild.build()
    g.load_library()
    base = WORKLOADS[args.workload]
    w = base.with_batch(base.B, seed=base.seed + rank)
    B, K, SH2, D = w.B, w.K, w.SH2, w.D
    x = make_inputs(w)
    dev = torch.device("cuda", local)
    bf16 = args.dtype == "bf16"
    act_dtype = torch.bfloat16 if bf16 else torch.float32
    acts = ("h_history", "h_s2", "d_h_enriched")
    d = {k: (torch.from_numpy(v).to(dev) if isinstance(v, np.ndarray) else v) for k, v in x.items()}
    for k in acts:
        d[k] = d[k].to(act_dtype)

    def alloc_outs():
        o = g.alloc_bwd_outputs(B, K, SH2, D, dev)
        for k in ("d_h_history", "d_h_s2"):
            o[k] = o[k].to(act_dtype)
        return o

    y = torch.empty((B, SH2), device=dev, dtype=act_dtype)
    outs = alloc_outs()
    ws = g.alloc_workspace(B, K, SH2, D, dev)
    flush = L2Flush(torch, dev)
    stream = torch.cuda.current_stream()
    fwd_call = g.fwd_bf16 if bf16 else g.fwd
    bwd_call = g.bwd_bf16 if bf16 else g.bwd

    def fwd():
        fwd_call(d["h_history"], d["h_s2"], d["W_A"], d["W_B"], d["W_C"], d["W_O"], d["tw"], out=y,
                 stream=stream)

    def bwd():
        bwd_call(d["h_history"], d["h_s2"], d["W_A"], d["W_B"], d["W_C"], d["W_O"], d["tw"],
                 d["d_h_enriched"], outs=outs, workspace=ws, stream=stream)

    for _ in range(max(3, args.warmup)):
        flush()
        fwd()
        flush()
        bwd()
    torch.cuda.synchronize()

    n = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(n)]
    sampler = ClockSampler()
    if rank == 0:
        sampler.start()
        time.sleep(0.3)
    barrier(dist, local)
    torch.cuda.synchronize()
    launches_before = 0
    wall0 = time.perf_counter()
    for i in range(n):
        flush()
        ev[i][0].record(stream)
        fwd()
        launches_before += g.m2scan_last_launch_count()
        ev[i][1].record(stream)
        flush()
        ev[i][2].record(stream)
        bwd()
        launches_before += g.m2scan_last_launch_count()
        ev[i][3].record(stream)
    torch.cuda.synchronize()
    barrier(dist, local)
    wall = time.perf_counter() - wall0
    clocks = sampler.stop(gpus=list(range(max(world, 1)))) if rank == 0 else None
    fwd_t = [e[0].elapsed_time(e[1]) for e in ev]
    bwd_t = [e[2].elapsed_time(e[3]) for e in ev]
    step_t = [a + b for a, b in zip(fwd_t, bwd_t)]
    # medians of the per-step event times (the means are reported beside them)
    fwd_ms, bwd_ms, step_ms, fwd_mean, bwd_mean = max_over_ranks(
        dist, [statistics.median(fwd_t), statistics.median(bwd_t), statistics.median(step_t),
               sum(fwd_t) / n, sum(bwd_t) / n], device=dev)
    # the last timed step's outputs, for the check against the oracle
    last_out = None
    if rank == 0 and not args.no_cpu_baseline:
        last_out = {"h_enriched": y.float().cpu().numpy()}
        last_out.update({k: v.float().cpu().numpy() for k, v in outs.items()})
    flags_timed = g.m2scan_read_device_flags()
    value = whole_job_throughput(B, world, step_ms / 1e3)

    # end to end: every step copies its inputs in from pinned host memory and
    # all of its outputs back to pinned host memory. Three streams and two
    # sets of device buffers let step i+1's copy-in and step i-1's copy-out
    # run during step i's kernels (the host link is full duplex); the time
    # runs from the first copy-in to the last copy-out.
    host_in = {k: torch.from_numpy(x[k]).to(act_dtype).pin_memory() for k in acts}
    host_out = {"h_enriched": torch.empty((B, SH2), dtype=act_dtype).pin_memory()}
    host_out.update({k: torch.empty(tuple(v.shape), dtype=v.dtype).pin_memory()
                     for k, v in outs.items()})
    h2d = sum(t.numel() * t.element_size() for t in host_in.values())
    d2h = sum(t.numel() * t.element_size() for t in host_out.values())
    dev_in = [d, dict(d, **{k: torch.empty_like(d[k]) for k in host_in})]
    dev_y = [y, torch.empty_like(y)]
    dev_outs = [outs, alloc_outs()]
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_comp = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    n_e2e = [0]

    def e2e_step():
        i = n_e2e[0]
        n_e2e[0] += 1
        b = i & 1
        di, do = dev_in[b], dev_outs[b]
        with torch.cuda.stream(s_in):
            if i >= 2:
                s_in.wait_event(ev_comp[b])  # step i-2's kernels are done with these inputs
            for k, t in host_in.items():
                di[k].copy_(t, non_blocking=True)
            ev_in[b].record(s_in)
        stream.wait_event(ev_in[b])
        if i >= 2:
            stream.wait_event(ev_out[b])  # step i-2's outputs have been copied out
        fwd_call(di["h_history"], di["h_s2"], di["W_A"], di["W_B"], di["W_C"], di["W_O"], di["tw"],
                 out=dev_y[b], stream=stream)
        bwd_call(di["h_history"], di["h_s2"], di["W_A"], di["W_B"], di["W_C"], di["W_O"], di["tw"],
                 di["d_h_enriched"], outs=do, workspace=ws, stream=stream)
        ev_comp[b].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_comp[b])
            host_out["h_enriched"].copy_(dev_y[b], non_blocking=True)
            for k, t in do.items():
                host_out[k].copy_(t, non_blocking=True)
            ev_out[b].record(s_out)

    for _ in range(4):
        e2e_step()
    torch.cuda.synchronize()
    barrier(dist, local)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    for _ in range(args.e2e_steps):
        e2e_step()
    e1.record(s_out)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / args.e2e_steps
    (e2e_ms,) = max_over_ranks(dist, [e2e_ms], device=dev)
    flags_e2e = g.m2scan_read_device_flags()
    (flags_any,) = max_over_ranks(dist, [float(flags_timed | flags_e2e)], device=dev)

    if rank != 0:
        return
    elem = 2 if bf16 else 4
    ab = algorithmic_bytes(B, K, SH2, elem=elem)
    af = algorithmic_flops(B, K, SH2, D)
    peak, peak_src = measured_peaks()
    wide = g.m2scan_path_for(K, SH2, D) == 3
    bwd_kernel = ("m2scan_bwd_bf16" if bf16 else
                  "m2scan_bwd (wide-state weight split, tile kernel, d_h_s2, dW products, slot "
                  "reduction)" if wide else "m2scan_bwd (fused backward + slot reduction)")
    bwd_write = elem * SH2 * (K + 1) * B  # d_h_history and d_h_s2
    # the bound of the backward call: its bytes at the HBM peak against its
    # method FLOPs as 3 x TF32 tensor-core products (fp32 arithmetic only)
    tpeak, tpeak_src = fp32_product_peak()
    tensor_bound = not bf16 and af["bwd"] / (tpeak * 1e12) > ab["bwd"] / (peak * 1e9)
    if tensor_bound:
        achieved = af["bwd"] / (bwd_ms / 1e3) / 1e12
        roof = {"kernel": bwd_kernel, "bound": "tensor", "achieved": achieved, "peak": tpeak,
                "peak_source": tpeak_src + " bf16_tflops burst x nominal tf32:bf16 (1.1/2.25) / 3 "
                               "(3 x TF32: three tf32 products per fp32 product)",
                "unit": "TFLOP/s", "frac": achieved / tpeak, "algorithmic_flops": af["bwd"],
                "algorithmic_bytes": ab["bwd"],
                "hbm_frac_of_measured": ab["bwd"] / (bwd_ms / 1e3) / 1e9 / peak,
                "traffic": None, "traffic_note": "no DRAM-counter record for this call"}
    else:
        achieved = ab["bwd"] / (bwd_ms / 1e3) / 1e9
        traffic = traffic_fields("m2scan_bwd_bf16" if bf16 else "m2scan_bwd", ab["bwd"] - bwd_write,
                                 bwd_write)
        roof = dict({"kernel": bwd_kernel, "bound": "hbm", "achieved": achieved, "peak": peak,
                     "peak_source": peak_src + " hbm_gbs burst", "unit": "GB/s",
                     "frac": achieved / peak, "algorithmic_bytes": ab["bwd"]}, **traffic)
    line = {
        "metric": metric_for(w) + (" with bf16 activations" if bf16 else ""), "value": value, "unit": UNIT, "n_gpus": world, "steps": n,
        "warmup": max(3, args.warmup), "ms_per_step": step_ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if bf16 else "f32",
        "data": "synthetic",
        "config": layer_config(w, world, args.dtype),
        "arithmetic": ("bf16 tensor-core operands (exact products), fp32 sums"
                       if bf16 else "fp32 (3 x TF32 tensor-core products)"),
        "timing": "median of the per-step CUDA-event times (fwd, bwd and their sum)",
        "fwd_ms": fwd_ms, "bwd_ms": bwd_ms, "fwd_ms_mean": fwd_mean, "bwd_ms_mean": bwd_mean,
        "hbm_gbs": ab["total"] / (step_ms / 1e3) / 1e9,
        "hbm_frac_of_measured": ab["total"] / (step_ms / 1e3) / 1e9 / peak,
        "roofline": roof,
        "device_flags": int(flags_any),
        "e2e": {"value": whole_job_throughput(B, world, e2e_ms / 1e3), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
        "gpu_launches": launches_before,
        "clocks": clocks,
        "wall_s_timed_region": wall,
        "pages_h100_context_ms": {"fwd": 22.0, "bwd": 1567.0},
    }
    if not args.no_cpu_baseline:
        xo = dict(x)
        if bf16:  # the oracle sees the values the GPU read
            for k in acts:
                xo[k] = d[k].float().cpu().numpy()
        line["cpu_baseline"] = cpu_baseline(xo, args.cpu_seconds, last_out,
                                            act_bound=2.0 ** -8 if bf16 else None)
    if flags_any:
        # a kernel gave up on a barrier wait: its results and times are garbage
        line["invalid"] = "device error flags %d: a kernel gave up waiting" % int(flags_any)
    print(json.dumps(line), flush=True)
    if flags_any or not line.get("cpu_baseline", {}).get("output_check", {"pass": True})["pass"]:
        sys.exit(3)


# ------------------------------------------------------------ reference arm

def run_reference(args, rank, world):
    """The fp64 CPU oracle timed on the host cores (rank 0 only)."""
    if rank != 0:
        return
    import oracle
    from gated_ssm_temporal_gb300.workloads import WORKLOADS, make_inputs
    base = WORKLOADS[args.workload]
    threads = oracle.default_threads()
    x = make_inputs(base)
    # size each step so the whole run stays within about two minutes
    cal = {k: (v[:64] if hasattr(v, "shape") and v.shape[0] == base.B else v) for k, v in x.items()}
    t0 = time.perf_counter()
    oracle.forward(cal["h_history"], cal["h_s2"], cal["W_A"], cal["W_B"], cal["W_C"], cal["W_O"],
                   cal["tw"], n_threads=threads)
    oracle.backward(cal["h_history"], cal["h_s2"], cal["W_A"], cal["W_B"], cal["W_C"],
                    cal["W_O"], cal["tw"], cal["d_h_enriched"], n_threads=threads)
    per_sample = max((time.perf_counter() - t0) / 64, 1e-7)
    budget = min(5.0, 120.0 / max(1, args.steps + args.warmup))
    ns = int(max(16, min(base.B, budget / per_sample)))
    xs = {k: (v[:ns] if hasattr(v, "shape") and v.shape[0] == base.B else v) for k, v in x.items()}

    def step():
        oracle.forward(xs["h_history"], xs["h_s2"], xs["W_A"], xs["W_B"], xs["W_C"], xs["W_O"],
                       xs["tw"], n_threads=threads)
        oracle.backward(xs["h_history"], xs["h_s2"], xs["W_A"], xs["W_B"], xs["W_C"], xs["W_O"],
                        xs["tw"], xs["d_h_enriched"], n_threads=threads)

    for _ in range(max(0, args.warmup)):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    el = time.perf_counter() - t0
    value = ns * args.steps / el
    line = {
        "impl": "reference", "metric": metric_for(base), "value": value, "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": el / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": layer_config(base, world, "f32"),
        "arithmetic": "fp64 loops on the host cores (the oracle); each step a bounded sample of "
                      "the batch; the config's l2 entry describes the native arm's timed calls",
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": "first %d of the %d samples per step" % (ns, base.B)},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------ bias-gradient column sum

def bias_metric(w) -> str:
    return "bias-gradient column sum GB/s of dy (N=%d, C=%d)" % (w.N, w.C)


def run_bias_native(args, rank, world, local):
    import numpy as np
    import torch

    import gated_ssm_temporal_gb300 as g
    from gated_ssm_temporal_gb300 import build as gbuild
    from gated_ssm_temporal_gb300.workloads import BIAS_WORKLOADS, make_bias_input

    torch.cuda.set_device(local)
    dist = init_dist(world, "nccl")
    gbuild.build()
    g.load_library()
    w = BIAS_WORKLOADS[args.workload]
    N, C = w.N, w.C
    dy_h = make_bias_input(N, C, w.seed + rank)
    dev = torch.device("cuda", local)
    dy = torch.from_numpy(dy_h).to(dev)
    db = torch.empty((C,), device=dev)
    ws = torch.empty((max(1, g.m2scan_bias_grad_workspace_bytes(N, C) // 4),), device=dev)
    flush = L2Flush(torch, dev)
    stream = torch.cuda.current_stream()

    def call(src, dst):
        g.bias_grad(src, dst, workspace=ws, stream=stream)

    for _ in range(max(3, args.warmup)):
        flush()
        call(dy, db)
    torch.cuda.synchronize()
    n = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n)]
    sampler = ClockSampler()
    if rank == 0:
        sampler.start()
        time.sleep(0.3)
    barrier(dist, local)
    torch.cuda.synchronize()
    launches = 0
    wall0 = time.perf_counter()
    for i in range(n):
        flush()
        ev[i][0].record(stream)
        call(dy, db)
        launches += g.m2scan_last_launch_count()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    barrier(dist, local)
    wall = time.perf_counter() - wall0
    clocks = sampler.stop(gpus=list(range(max(world, 1)))) if rank == 0 else None
    t_ms = sum(e[0].elapsed_time(e[1]) for e in ev) / n
    (t_ms,) = max_over_ranks(dist, [t_ms], device=dev)
    nbytes = N * C * 4
    value = nbytes * world / (t_ms / 1e3) / 1e9

    # end to end through the same call: dy copied in from pinned host memory,
    # db copied back, every step (copy-in of step i+1 overlaps step i)
    host_dy = torch.from_numpy(dy_h).pin_memory()
    host_db = torch.empty((C,)).pin_memory()
    dev_dy = [dy, torch.empty_like(dy)]
    s_in = torch.cuda.Stream(device=dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    cnt = [0]

    def e2e_step():
        b = cnt[0] & 1
        cnt[0] += 1
        with torch.cuda.stream(s_in):
            s_in.wait_event(ev_done[b])
            dev_dy[b].copy_(host_dy, non_blocking=True)
            ev_in[b].record(s_in)
        stream.wait_event(ev_in[b])
        call(dev_dy[b], db)
        host_db.copy_(db, non_blocking=True)
        ev_done[b].record(stream)

    for _ in range(4):
        e2e_step()
    torch.cuda.synchronize()
    barrier(dist, local)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    for _ in range(args.e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / args.e2e_steps
    (e2e_ms,) = max_over_ranks(dist, [e2e_ms], device=dev)
    if rank != 0:
        return
    peak, peak_src = measured_peaks()
    achieved = nbytes / (t_ms / 1e3) / 1e9
    line = {
        "metric": bias_metric(w), "value": value, "unit": "GB/s", "n_gpus": world, "steps": n,
        "warmup": max(3, args.warmup), "ms_per_step": t_ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": "%s: N=%d C=%d" % (w.name, N, C), "N": N, "C": C,
                   "parallelism": "replicas x%d" % world,
                   "l2": L2_NOTE},
        "roofline": {"kernel": "m2scan_bias_grad (partial sums + ordered final sum)",
                     "bound": "hbm", "achieved": achieved, "peak": peak,
                     "peak_source": peak_src + " hbm_gbs burst", "unit": "GB/s",
                     "frac": achieved / peak, "traffic": recorded_traffic(w.name)[0],
                     "algorithmic_bytes": nbytes},
        "e2e": {"value": nbytes * world / (e2e_ms / 1e3) / 1e9, "unit": "GB/s",
                "h2d_bytes_per_step": nbytes, "d2h_bytes_per_step": C * 4, "ms_per_step": e2e_ms},
        "gpu_launches": launches,
        "clocks": clocks,
        "wall_s_timed_region": wall,
    }
    if not args.no_cpu_baseline:
        import oracle
        done, t0 = 0, time.perf_counter()
        while True:
            oracle.bias_grad(dy_h)
            done += 1
            el = time.perf_counter() - t0
            if el >= min(args.cpu_seconds, 5.0):
                break
        line["cpu_baseline"] = {"value": nbytes * done / el / 1e9, "unit": "GB/s", "cores": 1,
                                "kind": "oracle",
                                "sample": "%d passes over the full [%d, %d] matrix (%.1f s)"
                                          % (done, N, C, el)}
    print(json.dumps(line), flush=True)


def run_bias_reference(args, rank, world):
    """The fp64 oracle column sum on the host (one core: a plain loop), rank 0 only."""
    if rank != 0:
        return
    import oracle
    from gated_ssm_temporal_gb300.workloads import BIAS_WORKLOADS, make_bias_input
    w = BIAS_WORKLOADS[args.workload]
    dy = make_bias_input(w.N, w.C, w.seed)
    for _ in range(max(0, args.warmup)):
        oracle.bias_grad(dy)
    done, t0 = 0, time.perf_counter()
    while done < max(1, args.steps):
        oracle.bias_grad(dy)
        done += 1
        if time.perf_counter() - t0 > 60.0:  # keep the run within about a minute
            break
    el = time.perf_counter() - t0
    value = w.N * w.C * 4 * done / el / 1e9
    line = {
        "impl": "reference", "metric": bias_metric(w), "value": value, "unit": "GB/s",
        "n_gpus": world, "steps": done, "warmup": args.warmup, "ms_per_step": el / done * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": "%s: N=%d C=%d" % (w.name, w.N, w.C), "N": w.N, "C": w.C},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": "the full matrix per step"},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    args = parse_args(argv)
    rank, world, local = dist_env()
    bias = args.workload.startswith("bias_")
    if args.impl == "reference":
        (run_bias_reference if bias else run_reference)(args, rank, world)
    else:
        (run_bias_native if bias else run_native)(args, rank, world, local)


if __name__ == "__main__":
    main()
