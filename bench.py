#!/usr/bin/env python
"""Benchmark of the GB300 attention sublayer.

One step is one pass of the path over one batch of synthetic inputs resident
in HBM: the fused Q/K/V projection plus attention of the sublayer workload
(fp32 storage, TF32 tensor-core products, x [8,512,512], Wqkv [512,1536],
H=8, D=64, non-causal), through the C ABI (la_layer_attn).  The line also
reports, each timed the same way, the other workloads of the path: fp32
causal attention B=8 H=8 S=2048 D=64 (with and without key padding), bf16
causal attention B=4 H=16 S=4096 D=128, the chunked 100k-token mode (bf16
causal B=2 H=16 S=100000 D=64, windows of 4096 against a growing cache), the
small fp32 case B=1 H=2 S=128 D=64 (also per-call latency, direct against
CUDA-graph replay), and the sublayer with and without its output
projection and with a LayerNorm in front (fp32, bf16 and fp16, B=8 S=512
d_model=512).

FLOPs are algorithmic (useful work only): 2*rows*d*3d for the projection,
2*rows*d*d for the output projection and 4*D per (query, visible key) pair
per head for attention.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Multi-GPU: one process per GPU under torchrun; every rank runs the same
workload on its own GPU (independent replicas: the path has no exchange
step), the time is the max over ranks and the value counts all ranks' work.
--impl reference times the fp64 CPU oracle on the host cores on a bounded
sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

METRIC = "attention fwd TFLOP/s and ms per layer at 1 GB300; % of tensor-pipe peak"
NOMINAL_TF32_OVER_BF16 = 1.1 / 2.25   # nominal dense TF32 / BF16 tensor rates
L2_FLUSH_BYTES = 256 << 20           # larger than the 129 MB L2

HEADLINE = dict(B=8, S=512, d_model=512, H=8)
HEADLINE_NAME = "attention sublayer fp32 (TF32 MMA) B=8 S=512 d_model=512 H=8 D=64 non-causal: qkv_proj + attention"


# ---------------------------------------------------------------------------
# helpers
# ---------------------------------------------------------------------------
def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        out = {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
               "bf16_tflops_sustained": p.get("bf16_tflops_sustained", p["bf16_tflops"]), "source": "measured"}
    except Exception:
        out = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}
    # the nominal figures, for context beside the measured denominators
    out["nominal"] = {"bf16_tflops": 2250.0, "tf32_tflops": 1100.0, "hbm_gbs": 7900.0}
    return out


def _tensor_peak(dtype, peaks, sustained=False):
    bf16 = peaks["bf16_tflops_sustained" if sustained else "bf16_tflops"]
    return bf16 * NOMINAL_TF32_OVER_BF16 if dtype == torch.float32 else bf16


def _source_sha(files):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "layer_attn_fwd_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def _traffic(kernel, workload, files):
    """DRAM bytes per launch from the committed ncu summary, or None when the
    kernel source changed since the counters were taken."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            t = json.load(f)
        e = t[f"{kernel} | {workload}"]
        return e["bytes_per_launch"] if e["source_sha"] == _source_sha(files) else None
    except Exception:
        return None


class Clocks:
    """Sample SM clocks and throttle reasons with nvidia-smi while running."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = None

    def __enter__(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None or self.path is None:
            return None
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = max((float(r[2]) for r in rows if r[2].replace(".", "").isdigit()), default=None)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        load = [s for s in sm if mx and s > 0.5 * mx] or sm
        med = statistics.median(load) if load else None
        # a run counts only if no slowdown reason was active and the clock held
        # at least 85% of its maximum (sw_power_cap is normal under load)
        bad = [r for r in reasons if r != "sw_power_cap"]
        ok = not bad and med is not None and mx is not None and med >= 0.85 * mx
        return {"sm_mhz": med, "sm_max_mhz": mx, "reasons": reasons, "samples": len(rows), "ok": ok}


def skip_reason(nbytes, free):
    """Why a workload needing `nbytes` of device memory is not run with
    `free` bytes free (10% and 256 MB of headroom), or None when it fits."""
    if nbytes * 1.1 + (256 << 20) > free:
        return f"needs about {nbytes / 1e9:.2f} GB on the device, {free / 1e9:.2f} GB free"
    return None


def require_clean(commit):
    """The --require-clean refusal for a work tree state (`_commit()`'s
    string, or None outside a git work tree), or None when it may run."""
    if commit is None:
        return "--require-clean: not a git work tree"
    if commit.endswith("+dirty"):
        return f"--require-clean: tracked files differ from {commit[:-6]}"
    return None


def _commit():
    try:
        r = subprocess.run(["git", "-C", ROOT, "rev-parse", "--short", "HEAD"], capture_output=True, text=True,
                           timeout=10)
        if r.returncode != 0:
            return None
        dirty = subprocess.run(["git", "-C", ROOT, "status", "--porcelain", "--untracked-files=no"],
                               capture_output=True, text=True, timeout=10).stdout.strip()
        return r.stdout.strip() + ("+dirty" if dirty else "")
    except Exception:
        return None


def emit(line, log_path=None):
    """Print the bench line; with a log path also append it, with the commit
    it ran from, to that append-only JSON-lines file."""
    text = json.dumps(line)
    print(text, flush=True)
    if log_path:
        rec = dict(line)
        rec["commit"] = _commit()
        rec["logged_at"] = time.strftime("%Y-%m-%dT%H:%M:%SZ", time.gmtime())
        with open(log_path, "a") as f:
            f.write(json.dumps(rec) + "\n")


def max_over_ranks(x, dist=None, device="cpu"):
    """Max of a per-rank float over all ranks (identity without a process group)."""
    if dist is None or not dist.is_initialized():
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# Before each timed step the stream spins this many SM cycles (after the L2
# flush, outside the events), so that the host has enqueued the whole step
# before its first kernel starts: the events then see device time only, not
# the host's argument checks and launch calls.
SPIN_CYCLES = 200_000


def _pre_step(flush, stream):
    with torch.cuda.stream(stream):
        flush.zero_()
        torch.cuda._sleep(SPIN_CYCLES)


def _time_steps(step, K, W, flush, stream, barrier):
    """W untimed steps, then K steps each bracketed by CUDA events on `stream`
    with an L2 flush (not timed) between them.  Returns total device ms."""
    for _ in range(W):
        step()
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    evs = []
    with torch.cuda.stream(stream):
        for _ in range(K):
            _pre_step(flush, stream)
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s.record(stream)
            step()
            e.record(stream)
            evs.append((s, e))
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    return sum(s.elapsed_time(e) for s, e in evs)


def kernel_times(api, step, K, flush, stream):
    """Device time of each kernel of a step, each launch bracketed by CUDA
    events on its own stream by the library (la_profile_start): K steps with
    an L2 flush before each; per kernel name the median over steps of its
    summed launch times, and its launches per step."""
    torch.cuda.synchronize()
    with api.Profile(max_launches=256 * K) as prof:
        for _ in range(K):
            _pre_step(flush, stream)
            step()
    torch.cuda.synchronize()
    recs = prof.records
    if not recs or len(recs) % K or len(recs) >= 256 * K:  # (a full record buffer would drop launches)
        return {}
    per = len(recs) // K
    out = {}
    for i in range(K):
        step_sum = {}
        for name, ms in recs[i * per:(i + 1) * per]:
            step_sum[name] = step_sum.get(name, 0.0) + ms
        for name, ms in step_sum.items():
            out.setdefault(name, []).append(ms)
    launches = {}
    for name, _ in recs[:per]:
        launches[name] = launches.get(name, 0) + 1
    return {name: {"ms": statistics.median(v), "launches_per_step": launches[name]} for name, v in out.items()}


# ---------------------------------------------------------------------------
# our implementation
# ---------------------------------------------------------------------------
def run_ours(args):
    from layer_attn_fwd_gb300 import api, build, flops, inputs

    ws_n, rank, local = _dist()
    torch.cuda.set_device(local)
    dist = None
    if ws_n > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    def barrier():
        if dist is not None:
            dist.barrier()

    build.build()
    api.load()
    peaks = _peaks()
    dev = torch.device("cuda", local)
    stream = torch.cuda.Stream(device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    K, W = args.steps, args.warmup

    if args.only:
        # one named workload alone (for profiler captures of one kernel)
        res = other_workloads(args, dev, stream, flush, barrier, peaks,
                              cpu_ok=rank == 0 and ws_n == 1 and not args.no_cpu)
        if rank == 0:
            print(json.dumps({"only": args.only, "workloads": res}), flush=True)
        if dist is not None:
            dist.destroy_process_group()
        return

    # ---- headline: the sublayer -------------------------------------------
    B, S, dm, H = HEADLINE["B"], HEADLINE["S"], HEADLINE["d_model"], HEADLINE["H"]
    D = dm // H
    x_h, W_h, b_h = inputs.layer_inputs(B, S, dm, torch.float32, seed=0)
    x, Wq, bq = x_h.to(dev), W_h.to(dev), b_h.to(dev)
    o = torch.empty_like(x)
    ws_layer = api.workspace_size(api.LA_OP_LAYER_ATTN, B, H, S, S, D, torch.float32)
    ws = torch.empty(ws_layer, dtype=torch.uint8, device=dev)
    fl_proj = flops.proj_flops(B, S, dm)
    fl_attn = flops.attn_flops(B, H, S, S, D, False)
    fl_step = fl_proj + fl_attn

    # Wqkv in the projection's layout (fp32: Wqkv^T, the K-major operand the
    # TF32 products read), prepared once before timing as at model load; the
    # form that converts the weight inside every step is timed beside it.
    Wqp = api.prepare_weight(Wq, stream=stream)
    torch.cuda.synchronize()

    def layer_step():
        api.layer_attn_prepared(x, Wqp, bq, H, out=o, workspace=ws, stream=stream)

    def layer_step_per_call():
        api.layer_attn(x, Wq, bq, H, out=o, workspace=ws, stream=stream)

    # (the per-call form first: the first timed steps of a process measured
    # a few per cent slow whichever form they ran)
    with Clocks(local) as clk:
        ms_per_call = _time_steps(layer_step_per_call, K, W, flush, stream, barrier)
        ms_total = _time_steps(layer_step, K, W, flush, stream, barrier)
    clocks = clk.summary()
    ms_per_call = max_over_ranks(ms_per_call, dist, dev)
    st = api.get_last_error(stream)
    if st != api.LA_OK:
        raise RuntimeError(f"device status after the timed steps: {api.status_string(st)}")
    ms_max = max_over_ranks(ms_total, dist, dev)
    ms_step = ms_max / K
    value = fl_step * K * ws_n / (ms_max * 1e-3) / 1e12

    # ---- each kernel of the step alone (events around every launch) -----------
    kt = kernel_times(api, layer_step, K, flush, stream)
    kernel_flops = {"qkv_proj_kernel": fl_proj, "attn_fwd_kernel": fl_attn}
    # algorithmic bytes of each stage (fp32): the projection reads x and
    # Wqkv^T and writes q, k, V^T; the attention reads those and writes o
    act = B * S * dm * 4
    kernel_bytes = {"qkv_proj_kernel": act + 3 * dm * dm * 4 + 3 * act, "attn_fwd_kernel": 3 * act + act}
    per_kernel = {}
    for name, t in kt.items():
        e = {"ms": round(t["ms"], 5), "launches_per_step": t["launches_per_step"]}
        if name in kernel_flops:
            e["tflops"] = round(kernel_flops[name] / (t["ms"] * 1e-3) / 1e12, 2)
            e["gbs"] = round(kernel_bytes[name] / (t["ms"] * 1e-3) / 1e9, 1)
        elif name == "transpose32_kernel":  # Wqkv^T, 3 d^2 fp32 read and written
            e["gbs"] = round(2 * 3 * dm * dm * 4 / (t["ms"] * 1e-3) / 1e9, 1)
        per_kernel[name] = e
    dom = max((n for n in per_kernel if n in kernel_flops), key=lambda n: per_kernel[n]["ms"])
    peak_tf32 = _tensor_peak(torch.float32, peaks)
    src = ["la_attn.cu", "la_device.cuh"] if dom == "attn_fwd_kernel" else ["la_proj.cu", "la_device.cuh"]
    roofline = {"bound": "tensor", "kernel": dom, "achieved": per_kernel[dom]["tflops"],
                "peak": round(peak_tf32, 1), "unit": "TFLOP/s",
                "frac": round(per_kernel[dom]["tflops"] / peak_tf32, 4),
                "traffic": _traffic(dom, "sublayer fp32 B8 S512 d512", src),
                "algorithmic": f"{kernel_flops[dom] / 1e9:.3f} GFLOP per launch",
                "timing": "CUDA events around each launch on its stream (la_profile_start), median of the steps",
                "peak_note": f"TF32 = {peaks['source']} bf16 burst x nominal 1.1/2.25 (of measured)"}

    # ---- end to end through the public API, host buffers -------------------------
    # Serial: each step copies its input in, runs the sublayer and reads the
    # result back on one stream (L2 flushed before each step, outside the
    # events).
    x_pin = x_h.pin_memory()
    o_pin = torch.empty_like(x_h).pin_memory()

    def e2e_step():
        with torch.cuda.stream(stream):
            x.copy_(x_pin, non_blocking=True)
            api.layer_attn_prepared(x, Wqp, bq, H, out=o, workspace=ws, stream=stream)
            o_pin.copy_(o, non_blocking=True)

    ms_serial = max_over_ranks(_time_steps(e2e_step, K, W, flush, stream, barrier), dist, dev)
    del x_pin, o_pin
    # Pipelined, as a serving loop runs: step i's input copy and step i-1's
    # result read run on their own streams beside step i's compute.  Inputs
    # and outputs rotate through 16 slots (134 MB each way, more than L2),
    # so no flush is needed.
    ms_pipe = max_over_ranks(e2e_pipelined(api, x_h, Wqp, bq, H, ws, stream, dev, K, W, barrier), dist, dev)
    link = link_peak(dev)
    step_link_gbs = 2 * x_h.numel() * 4 / (ms_pipe / K * 1e-3) / 1e9
    e2e = {"value": round(fl_step * K * ws_n / (ms_pipe * 1e-3) / 1e12, 3), "unit": "TFLOP/s",
           "link": {"achieved_gbs": round(step_link_gbs, 1), "peak_gbs": link["both_gbs"],
                    "frac": round(step_link_gbs / link["both_gbs"], 4), "measured": link,
                    "note": "the pipelined step's copies in and out (both directions at once) against the measured "
                            "pinned copy bandwidth with both directions busy"},
           "ms_per_step": round(ms_pipe / K, 4), "h2d_bytes_per_step": x_h.numel() * 4,
           "d2h_bytes_per_step": x_h.numel() * 4,
           "pipeline": "input copy, sublayer and result read on three streams, step i's compute overlapping "
                       "step i+1's copy in and step i-1's copy out; 16 rotating input/output slots (134 MB "
                       "each way > L2), no flush; timed from the first copy in to the last copy out",
           "serial": {"value": round(fl_step * K * ws_n / (ms_serial * 1e-3) / 1e12, 3),
                      "ms_per_step": round(ms_serial / K, 4),
                      "note": "copy in, sublayer, copy out on one stream; L2 flushed before each step"}}

    # ---- the other workloads of the path --------------------------------------------
    workloads = {}
    if not args.headline_only:
        workloads = other_workloads(args, dev, stream, flush, barrier, peaks,
                                    cpu_ok=rank == 0 and ws_n == 1 and not args.no_cpu)

    # ---- CPU baseline: the oracle on the host cores (rank 0, N=1 only) ------------------
    cpu = None
    if rank == 0 and ws_n == 1 and not args.no_cpu:
        cpu = cpu_baseline_sample(x_h, W_h, b_h, H, seconds=args.cpu_seconds)

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 3), "unit": "TFLOP/s", "n_gpus": ws_n, "steps": K, "warmup": W,
            "ms_per_step": round(ms_step, 5), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f32", "data": "synthetic",
            "config": {"workload": HEADLINE_NAME, "math": "TF32 tensor-core products, fp32 accumulate and softmax",
                       "weights": "Wqkv prepared once before timing (la_prepare_weight: fp32 Wqkv^T, the K-major "
                                  "operand of the TF32 products), as at model load; per_call_weights times the "
                                  "call that transposes Wqkv inside every step",
                       "l2": "flushed between timed steps (256 MB write)", "parallelism": f"replicas x{ws_n}",
                       "batch": B, "seq_len": S, "d_model": dm, "heads": H},
            "frac_of_tensor_peak": round(value / ws_n / peak_tf32, 4),
            "roofline": roofline, "per_kernel": per_kernel, "e2e": e2e,
            "per_call_weights": {"ms_per_step": round(ms_per_call / K, 5),
                                 "value": round(fl_step * K * ws_n / (ms_per_call * 1e-3) / 1e12, 3),
                                 "note": "la_layer_attn: Wqkv transposed by a pre-pass inside every step"},
            "gpu_launches": sum(t["launches_per_step"] for t in kt.values()) * K, "clocks": clocks,
            "cpu_baseline": cpu,
            "workloads": workloads, "peaks": peaks,
        }
        emit(line, args.log)
    if dist is not None:
        dist.destroy_process_group()


def link_peak(dev, nbytes=256 << 20, reps=5):
    """Measured pinned host <-> device copy bandwidth (GB/s): host to device
    alone, device to host alone, and both at once on two streams (best of
    `reps`, CUDA events, 256 MB each way)."""
    h_in = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    h_out = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    d_in = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    d_out = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    s1, s2 = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)

    def best(fn):
        t = []
        for _ in range(reps):
            torch.cuda.synchronize()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(s1)
            s2.wait_event(a)
            fn()
            s1.wait_stream(s2)
            b.record(s1)
            torch.cuda.synchronize()
            t.append(a.elapsed_time(b))
        return min(t)

    def h2d():
        with torch.cuda.stream(s1):
            d_in.copy_(h_in, non_blocking=True)

    def d2h():
        with torch.cuda.stream(s2):
            h_out.copy_(d_out, non_blocking=True)

    def both():
        h2d()
        d2h()

    t_in, t_out, t_both = best(h2d), best(d2h), best(both)
    res = {"h2d_gbs": round(nbytes / (t_in * 1e-3) / 1e9, 1), "d2h_gbs": round(nbytes / (t_out * 1e-3) / 1e9, 1),
           "both_gbs": round(2 * nbytes / (t_both * 1e-3) / 1e9, 1),
           "how": "256 MB pinned buffers, best of 5, CUDA events; both = the two directions at once on two streams"}
    del h_in, h_out, d_in, d_out
    return res


def e2e_pipelined(api, x_h, Wq, bq, H, ws, stream, dev, K, W, barrier, slots=16, copy_streams=1):
    """K steps of host input -> sublayer (on the prepared weight Wq) -> host
    output, pipelined: the copies
    in and out run on their own streams (copy_streams of each, taken by
    consecutive steps in turn) beside the compute stream; returns device ms
    from the first input copy to the last output copy (CUDA events)."""
    x_pins = [x_h.pin_memory() for _ in range(slots)]
    o_pins = [torch.empty_like(x_h).pin_memory() for _ in range(slots)]
    xs = [torch.empty(x_h.shape, dtype=x_h.dtype, device=dev) for _ in range(slots)]
    outs = [torch.empty_like(t) for t in xs]
    s_ins = [torch.cuda.Stream(device=dev) for _ in range(copy_streams)]
    s_outs = [torch.cuda.Stream(device=dev) for _ in range(copy_streams)]
    ev_in = [torch.cuda.Event() for _ in range(slots)]
    ev_done = [torch.cuda.Event() for _ in range(slots)]
    ev_out = [torch.cuda.Event() for _ in range(slots)]

    def run(first, n):
        for i in range(first, first + n):
            k = i % slots
            s_in, s_out = s_ins[i % copy_streams], s_outs[i % copy_streams]
            if i >= slots:
                s_in.wait_event(ev_done[k])       # the slot's previous input has been consumed
            with torch.cuda.stream(s_in):
                xs[k].copy_(x_pins[k], non_blocking=True)
            ev_in[k].record(s_in)
            stream.wait_event(ev_in[k])
            if i >= slots:
                stream.wait_event(ev_out[k])      # the slot's previous output has been read out
            api.layer_attn_prepared(xs[k], Wq, bq, H, out=outs[k], workspace=ws, stream=stream)
            ev_done[k].record(stream)
            s_out.wait_event(ev_done[k])
            with torch.cuda.stream(s_out):
                o_pins[k].copy_(outs[k], non_blocking=True)
            ev_out[k].record(s_out)

    run(0, W)
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for s in s_ins:
        s.wait_event(start)
    run(W, K)
    for s in s_ins + s_outs:
        stream.wait_stream(s)
    end.record(stream)
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    return start.elapsed_time(end)


def other_workloads(args, dev, stream, flush, barrier, peaks, cpu_ok=False):
    from layer_attn_fwd_gb300 import api, flops, inputs

    res = {}
    Kx = max(3, min(args.steps, 20))

    def wanted(key):
        return not args.only or args.only == key

    def fits(name, nbytes):
        """Memory pre-check: a workload whose device tensors would not fit in
        the free device memory is recorded as skipped, with the reason,
        instead of being run."""
        why = skip_reason(nbytes, torch.cuda.mem_get_info(dev)[0])
        if why is not None:
            res[name] = {"skipped": why}
            return False
        return True

    def attn_case(key, name, B, H, S, D, dt, causal, padded=False, small=False):
        if not wanted(key):
            return
        esz = torch.tensor([], dtype=dt).element_size()
        if not fits(name, 4 * B * H * S * D * esz + api.workspace_size(api.LA_OP_ATTN_FWD, B, H, S, S, D, dt)):
            return
        qh, kh, vh = inputs.attn_inputs(B, H, S, S, D, dt, seed=0)
        q, k, v = (t.to(dev) for t in (qh, kh, vh))
        kv = inputs.padding_kv_len(B, S) if padded else None
        kl = kv.to(dev) if kv is not None else None
        o = torch.empty_like(q)
        n = api.workspace_size(api.LA_OP_ATTN_FWD, B, H, S, S, D, dt)
        ws = torch.empty(max(n, 16), dtype=torch.uint8, device=dev)

        def step():
            api.attn_fwd(q, k, v, causal=causal, kv_len=kl, out=o, workspace=ws, stream=stream)

        ms = _time_steps(step, Kx, 3, flush, stream, barrier) / Kx
        kt = kernel_times(api, step, Kx, flush, stream)
        fl = flops.attn_flops(B, H, S, S, D, causal, kv)
        tf = fl / (ms * 1e-3) / 1e12
        pk = _tensor_peak(dt, peaks)
        ka = kt.get("attn_fwd_kernel", {}).get("ms")
        r = {"ms": round(ms, 4), "tflops": round(tf, 2), "frac_of_tensor_peak": round(tf / pk, 4),
             "gflop": round(fl / 1e9, 3),
             "per_kernel_ms": {n_: round(t["ms"], 5) for n_, t in kt.items()}}
        if ka:
            r["attn_kernel"] = {"ms": round(ka, 5), "tflops": round(fl / (ka * 1e-3) / 1e12, 2),
                                "frac_of_tensor_peak": round(fl / (ka * 1e-3) / 1e12 / pk, 4)}
        if small:  # latency bound: also bytes moved (q, k, v read, o written once) against the copy bandwidth
            nbytes = 4 * B * H * S * D * q.element_size()
            r["gbs"] = round(nbytes / (ms * 1e-3) / 1e9, 2)
            r["frac_of_hbm"] = round(nbytes / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 5)
        if cpu_ok:
            r["cpu_baseline"] = cpu_attn_baseline(qh, kh, vh, causal, kv, fl, full=small)
        res[name] = r
        del q, k, v, o, ws

    attn_case("fp32-causal-2048", "fp32 causal B8 H8 S2048 D64", 8, 8, 2048, 64, torch.float32, True)
    attn_case("fp32-causal-2048-padded", "fp32 causal B8 H8 S2048 D64, last 25% keys padded for half the batch",
              8, 8, 2048, 64, torch.float32, True, padded=True)
    attn_case("bf16-causal-4096", "bf16 causal B4 H16 S4096 D128", 4, 16, 4096, 128, torch.bfloat16, True)
    attn_case("fp32-small", "fp32 B1 H2 S128 D64 non-causal", 1, 2, 128, 64, torch.float32, False, small=True)
    if args.only == "attn-window-bf16":
        # one window of the chunked mode on its own (profiling: 0.4 GB on the
        # device instead of the whole 100k-token run): 4096 queries against
        # 40960 keys, causal rows aligned to the end
        B, H, S_q, S_kv, D = 2, 16, 4096, 40960, 64
        q, k, v = (t.to(dev) for t in inputs.attn_inputs(B, H, S_q, S_kv, D, torch.bfloat16, seed=0))
        o = torch.empty_like(q)
        n = api.workspace_size(api.LA_OP_ATTN_FWD, B, H, S_q, S_kv, D, torch.bfloat16)
        ws = torch.empty(max(n, 16), dtype=torch.uint8, device=dev)
        ms = _time_steps(lambda: api.attn_fwd(q, k, v, causal=True, out=o, workspace=ws, stream=stream),
                         Kx, 3, flush, stream, barrier) / Kx
        fl = flops.attn_flops(B, H, S_q, S_kv, D, True)
        res["bf16 causal window B2 H16 S_q4096 S_kv40960 D64"] = {
            "ms": round(ms, 4), "tflops": round(fl / (ms * 1e-3) / 1e12, 2), "gflop": round(fl / 1e9, 1)}
        return res
    if args.only == "sublayer-fp32":
        # the headline step alone (profiling)
        B, S, dm, H = HEADLINE["B"], HEADLINE["S"], HEADLINE["d_model"], HEADLINE["H"]
        x, Wq, bq = (t.to(dev) for t in inputs.layer_inputs(B, S, dm, torch.float32, seed=0))
        y = torch.empty_like(x)
        ws = torch.empty(api.workspace_size(api.LA_OP_LAYER_ATTN, B, H, S, S, dm // H, torch.float32),
                         dtype=torch.uint8, device=dev)
        ms = _time_steps(lambda: api.layer_attn(x, Wq, bq, H, out=y, workspace=ws, stream=stream),
                         Kx, 3, flush, stream, barrier) / Kx
        fl = flops.proj_flops(B, S, dm) + flops.attn_flops(B, H, S, S, dm // H, False)
        res[HEADLINE_NAME] = {"ms": round(ms, 4), "tflops": round(fl / (ms * 1e-3) / 1e12, 2)}
        return res

    def layer_out_case(key, name, dt):
        """The sublayer (la_layer_attn), the sublayer with its output projection
        (la_layer_attn_out), the pre-norm block (la_layer_attn_ln: LayerNorm,
        sublayer, output projection), and the output projection alone."""
        if not wanted(key):
            return
        B, S, dm, H = 8, 512, 512, 8
        esz = torch.tensor([], dtype=dt).element_size()
        if not fits(name, (4 * B * S * dm + 6 * dm * dm) * esz
                    + api.workspace_size(api.LA_OP_LAYER_ATTN_LN, B, H, S, S, dm // H, dt)):
            return
        x, Wq, bq = (t.to(dev) for t in inputs.layer_inputs(B, S, dm, dt, seed=0))
        Wo, bo = (t.to(dev) for t in inputs.out_proj_inputs(dm, dt, seed=1))
        y = torch.empty_like(x)
        gam, bet = (t.to(dev) for t in inputs.ln_inputs(dm, dt, seed=2))
        n = api.workspace_size(api.LA_OP_LAYER_ATTN_LN, B, H, S, S, dm // H, dt)
        ws = torch.empty(n, dtype=torch.uint8, device=dev)
        ms_l = _time_steps(lambda: api.layer_attn(x, Wq, bq, H, out=y, workspace=ws, stream=stream),
                           Kx, 3, flush, stream, barrier) / Kx
        ms = _time_steps(lambda: api.layer_attn_out(x, Wq, bq, Wo, bo, H, out=y, workspace=ws, stream=stream),
                         Kx, 3, flush, stream, barrier) / Kx
        ms_ln = _time_steps(lambda: api.layer_attn_ln(x, gam, bet, Wq, bq, Wo, bo, H, out=y, workspace=ws,
                                                      stream=stream), Kx, 3, flush, stream, barrier) / Kx
        # the same three forms on weights prepared once (la_prepare_weight), as a
        # server runs them: no per-call conversion of the constant weights
        Wqp, Wop = api.prepare_weight(Wq), api.prepare_weight(Wo)
        ms_lp = _time_steps(lambda: api.layer_attn_prepared(x, Wqp, bq, H, out=y, workspace=ws, stream=stream),
                            Kx, 3, flush, stream, barrier) / Kx
        ms_op = _time_steps(lambda: api.layer_attn_prepared(x, Wqp, bq, H, Wo_p=Wop, bo=bo, out=y, workspace=ws,
                                                            stream=stream), Kx, 3, flush, stream, barrier) / Kx
        ms_lnp = _time_steps(lambda: api.layer_attn_prepared(x, Wqp, bq, H, gamma=gam, beta=bet, Wo_p=Wop, bo=bo,
                                                             out=y, workspace=ws, stream=stream),
                             Kx, 3, flush, stream, barrier) / Kx
        fl_l = flops.proj_flops(B, S, dm) + flops.attn_flops(B, H, S, S, dm // H, False)
        fl = fl_l + flops.out_proj_flops(B, S, dm)
        o = api.layer_attn(x, Wq, bq, H, stream=stream)
        wo_ws = torch.empty(max(api.workspace_size(api.LA_OP_OUT_PROJ, 1, H, B * S, B * S, dm // H, dt), 16),
                            dtype=torch.uint8, device=dev)
        ms_o = _time_steps(lambda: api.out_proj(o, Wo, bo, out=y, workspace=wo_ws, stream=stream),
                           Kx, 3, flush, stream, barrier) / Kx
        fl_o = flops.out_proj_flops(B, S, dm)
        pk = _tensor_peak(dt, peaks)
        tf, tf_o = fl / (ms * 1e-3) / 1e12, fl_o / (ms_o * 1e-3) / 1e12
        tf_l = fl_l / (ms_l * 1e-3) / 1e12
        res[name] = {"ms": round(ms, 4), "tflops": round(tf, 2), "frac_of_tensor_peak": round(tf / pk, 4),
                     "gflop": round(fl / 1e9, 3),
                     "sublayer_without_out_proj": {"ms": round(ms_l, 4), "tflops": round(tf_l, 2),
                                                   "frac_of_tensor_peak": round(tf_l / pk, 4)},
                     "prenorm_block": {"ms": round(ms_ln, 4), "layernorm_cost_ms": round(ms_ln - ms, 4),
                                       "note": "LayerNorm + sublayer + output projection"},
                     "out_proj": {"ms": round(ms_o, 4), "tflops": round(tf_o, 2),
                                  "frac_of_tensor_peak": round(tf_o / pk, 4),
                                  "note": "fp32 includes the Wo^T pre-pass" if dt == torch.float32 else ""},
                     "prepared_weights": {
                         "sublayer_ms": round(ms_lp, 4), "sublayer_tflops": round(fl_l / (ms_lp * 1e-3) / 1e12, 2),
                         "with_out_proj_ms": round(ms_op, 4),
                         "with_out_proj_tflops": round(fl / (ms_op * 1e-3) / 1e12, 2),
                         "prenorm_block_ms": round(ms_lnp, 4),
                         "note": "la_layer_attn_prepared on weights prepared once (fp32: transposed) by "
                                 "la_prepare_weight"}}
        del x, Wq, bq, Wo, bo, y, ws, o, wo_ws, gam, bet, Wqp, Wop

    def small_latency(key, name):
        """Small-shape latency: back-to-back calls, host wall clock per call
        (argument checks, tensor-map encoding and launches included), direct
        calls against replays of the same call captured in a CUDA graph."""
        if not wanted(key):
            return
        B, H, S, D = 1, 2, 128, 64
        q, k, v = (t.to(dev) for t in inputs.attn_inputs(B, H, S, S, D, torch.float32, seed=0))
        o = torch.empty_like(q)
        ws = torch.empty(api.workspace_size(api.LA_OP_ATTN_FWD, B, H, S, S, D, torch.float32), dtype=torch.uint8,
                         device=dev)

        def direct():
            api.attn_fwd(q, k, v, out=o, workspace=ws, stream=stream)

        g = api.Graph(lambda: api.attn_fwd(q, k, v, out=o, workspace=ws), stream=stream)

        def replay():
            with torch.cuda.stream(stream):
                g.replay()

        def per_call_us(fn, n=500):
            for _ in range(50):
                fn()
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            for _ in range(n):
                fn()
            torch.cuda.synchronize()
            return (time.perf_counter() - t0) / n * 1e6

        us_direct, us_graph = per_call_us(direct), per_call_us(replay)
        with api.Profile() as prof:
            direct()
        torch.cuda.synchronize()
        n_launch = len(prof.records)
        fl = flops.attn_flops(B, H, S, S, D, False)
        res[name] = {"direct_us_per_call": round(us_direct, 2), "graph_us_per_call": round(us_graph, 2),
                     "graph_speedup": round(us_direct / us_graph, 3),
                     "graph_tflops": round(fl / (us_graph * 1e-6) / 1e12, 3), "gflop": round(fl / 1e9, 5),
                     "launches_per_call": n_launch,
                     "note": "500 back-to-back calls, inputs L2-resident (0.26 MB), no flush"}

    small_latency("small-graph", "fp32 B1 H2 S128 D64 non-causal, per-call latency: direct vs CUDA-graph replay")
    layer_out_case("layer-out-fp32", "sublayer + output projection fp32 B8 S512 d512 H8 non-causal", torch.float32)
    layer_out_case("layer-out-bf16", "sublayer + output projection bf16 B8 S512 d512 H8 non-causal", torch.bfloat16)
    layer_out_case("layer-out-f16", "sublayer + output projection fp16 B8 S512 d512 H8 non-causal", torch.float16)
    if not wanted("chunked-100k"):
        return res

    # chunked 100k-token mode: 25 windows of 4096 (the last 1696) per step
    B, H, S, D, C = 2, 16, 100000, 64, 4096
    name_c = f"chunked bf16 causal B{B} H{H} S{S} D{D}, windows of {C}"
    # windowed q, k, v and outputs, the cache's K and V
    if not fits(name_c, 6 * B * H * S * D * 2 + api.workspace_size(api.LA_OP_ATTN_CHUNKED, B, H, C, S, D,
                                                                   torch.bfloat16)):
        return res
    q, k, v = inputs.attn_inputs(B, H, S, S, D, torch.bfloat16, seed=0)
    wins = inputs.chunk_bounds(S, C)
    qs = [q[:, :, s:s + L].contiguous().to(dev) for s, L in wins]
    ks = [k[:, :, s:s + L].contiguous().to(dev) for s, L in wins]
    vs = [v[:, :, s:s + L].contiguous().to(dev) for s, L in wins]
    if not cpu_ok:
        del q, k, v
    cache = api.KVCache(B, H, S, D, torch.bfloat16, device=dev)
    outs = [torch.empty_like(t) for t in qs]
    n = api.workspace_size(api.LA_OP_ATTN_CHUNKED, B, H, C, S, D, torch.bfloat16)
    ws = torch.empty(max(n, 16), dtype=torch.uint8, device=dev)

    def chunked_step():
        cache.reset()
        for i in range(len(wins)):
            api.attn_chunked(qs[i], ks[i], vs[i], cache, out=outs[i], workspace=ws, stream=stream)

    torch.cuda.reset_peak_memory_stats(dev)
    kc = 3 if not args.only else max(1, min(args.steps, 3))
    ms = _time_steps(chunked_step, kc, 1, flush, stream, barrier) / kc
    fl = flops.attn_flops(B, H, S, S, D, True)
    tf = fl / (ms * 1e-3) / 1e12
    peak_mem = torch.cuda.max_memory_allocated(dev)
    kt = kernel_times(api, chunked_step, 1, flush, stream)
    r = {"ms": round(ms, 3), "tflops": round(tf, 2), "frac_of_tensor_peak": round(tf / _tensor_peak(torch.bfloat16, peaks), 4),
         "gflop": round(fl / 1e9, 1), "windows": len(wins), "workspace_bytes": n, "peak_device_bytes": peak_mem,
         "per_kernel_ms": {n_: round(t["ms"], 4) for n_, t in kt.items()}}
    ka = kt.get("attn_fwd_kernel", {}).get("ms")
    if ka:
        r["attn_kernel"] = {"ms": round(ka, 4), "tflops": round(fl / (ka * 1e-3) / 1e12, 2),
                            "frac_of_tensor_peak": round(fl / (ka * 1e-3) / 1e12 / _tensor_peak(torch.bfloat16, peaks), 4)}
    if cpu_ok:
        # the window-by-window result is attention over the whole sequence:
        # the oracle on 256 sampled rows (window boundaries and the last row
        # included), extrapolated per (query, key) pair
        rows = inputs.sample_rows(B, H, S, n=256, seed=1234, forced=(0, 4095, 4096, 98303, 98304, 99999))
        t0 = time.perf_counter()
        import oracle
        oracle.attn_rows(q, k, v, rows, causal=True)
        t = time.perf_counter() - t0
        pairs = _visible_keys(rows, S, S, True, None)
        t_full = t / pairs * (fl / (4 * D))
        r["cpu_baseline"] = {"value": round(fl / t_full / 1e12, 6), "unit": "TFLOP/s", "cores": oracle.num_threads(),
                             "kind": "oracle", "extrapolated": True,
                             "sample": f"256 seeded sampled rows incl. window boundaries ({t:.2f} s, {pairs} query-key "
                                       f"pairs, fp64, OpenMP); extrapolated per pair to the whole workload "
                                       f"({t_full / 3600:.1f} h)"}
        del q, k, v
    res[name_c] = r
    st = api.get_last_error(stream)
    if st != api.LA_OK:
        raise RuntimeError(f"device status after the extra workloads: {api.status_string(st)}")
    return res


# ---------------------------------------------------------------------------
# the CPU oracle
# ---------------------------------------------------------------------------
def cpu_baseline_sample(x_h, W_h, b_h, H, seconds=20.0):
    """Time the fp64 oracle on a bounded sample of the sublayer workload: the
    first batch entries, as many as fit in about `seconds` of CPU work."""
    import oracle
    from layer_attn_fwd_gb300 import flops

    S, dm = x_h.shape[1], x_h.shape[2]
    D = dm // H
    done_b, t_total = 0, 0.0
    while done_b < x_h.shape[0] and t_total < seconds:
        t0 = time.perf_counter()
        oracle.layer_attn(x_h[done_b:done_b + 1].contiguous(), W_h, b_h, H)
        t_total += time.perf_counter() - t0
        done_b += 1
    fl = done_b * (flops.proj_flops(1, S, dm) + flops.attn_flops(1, H, S, S, D, False))
    # the same on one core: the first batch entry with the oracle on one thread
    oracle.set_num_threads(1)
    try:
        t0 = time.perf_counter()
        oracle.layer_attn(x_h[:1].contiguous(), W_h, b_h, H)
        t1 = time.perf_counter() - t0
    finally:
        oracle.set_num_threads(0)
    fl1 = flops.proj_flops(1, S, dm) + flops.attn_flops(1, H, S, S, D, False)
    return {"value": round(fl / t_total / 1e12, 6), "unit": "TFLOP/s", "cores": oracle.num_threads(),
            "kind": "oracle",
            "sample": f"{done_b} of {x_h.shape[0]} batch entries of the sublayer workload ({t_total:.1f} s, fp64, OpenMP)",
            "single_core": {"value": round(fl1 / t1 / 1e12, 6), "unit": "TFLOP/s", "cores": 1,
                            "sample": f"1 batch entry of the sublayer workload ({t1:.1f} s, fp64, one thread)"}}


def _visible_keys(rows, S_q, S_kv, causal, kv_len):
    """Keys each sampled row (b, h, i) sees (the mask's definition, counted)."""
    r = rows.numpy()
    n = 0
    for b, _, i in r:
        lim = S_kv if kv_len is None else min(int(kv_len[b]), S_kv)
        if causal:
            lim = min(lim, int(i) + S_kv - S_q + 1)
        n += max(lim, 0)
    return n


def cpu_attn_baseline(q, k, v, causal, kv_len, flops_total, full=False, seconds=2.0, seed=777):
    """The fp64 oracle timed on the host cores on a bounded sample of an
    attention workload.  full: the whole workload, repeated for about
    `seconds`.  Otherwise seeded sampled rows (doubling their number until
    the sample takes about `seconds`), timed, and extrapolated to the whole
    workload per (query, visible key) pair."""
    import oracle
    from layer_attn_fwd_gb300 import inputs

    B, H, S_q, D = q.shape
    S_kv = k.shape[2]
    cores = oracle.num_threads()
    if full:
        n, t = 0, 0.0
        while n < 3 or t < seconds:
            t0 = time.perf_counter()
            oracle.attn(q, k, v, causal=causal, kv_len=kv_len)
            t += time.perf_counter() - t0
            n += 1
        return {"value": round(flops_total * n / t / 1e12, 6), "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                "sample": f"the whole workload, {n} runs ({t:.1f} s, fp64, OpenMP)", "extrapolated": False}
    n_rows, t, pairs = 64, 0.0, 0
    while True:
        rows = inputs.sample_rows(B, H, S_q, n=n_rows, seed=seed)
        t0 = time.perf_counter()
        oracle.attn_rows(q, k, v, rows, causal=causal, kv_len=kv_len)
        t = time.perf_counter() - t0
        pairs = _visible_keys(rows, S_q, S_kv, causal, kv_len)
        if t >= seconds / 2 or n_rows >= 1 << 16:
            break
        n_rows *= 2
    total_pairs = flops_total / (4 * D)
    t_full = t / max(pairs, 1) * total_pairs
    return {"value": round(flops_total / t_full / 1e12, 6), "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "sample": f"{n_rows} seeded sampled rows ({t:.2f} s, {pairs} query-key pairs, fp64, OpenMP); "
                      f"extrapolated per pair to the whole workload ({t_full:.1f} s)",
            "extrapolated": True}


def run_reference(args):
    ws_n, rank, _ = _dist()
    if rank != 0:
        return
    import oracle
    from layer_attn_fwd_gb300 import flops, inputs

    B, S, dm, H = HEADLINE["B"], HEADLINE["S"], HEADLINE["d_model"], HEADLINE["H"]
    D = dm // H
    x, W, b = inputs.layer_inputs(B, S, dm, torch.float32, seed=0)
    oracle.build()
    # one step = the oracle on one batch entry of the workload (a bounded sample)
    xs = [x[i:i + 1].contiguous() for i in range(B)]
    fl = flops.proj_flops(1, S, dm) + flops.attn_flops(1, H, S, S, D, False)
    for i in range(args.warmup):
        oracle.layer_attn(xs[i % B], W, b, H)
    t0 = time.perf_counter()
    for i in range(args.steps):
        oracle.layer_attn(xs[i % B], W, b, H)
    t = time.perf_counter() - t0
    value = fl * args.steps / t / 1e12
    cores = oracle.num_threads()
    sample = f"one of the {B} batch entries per step (x [1,{S},{dm}]), fp64, OpenMP"
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": ws_n,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(t / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": HEADLINE_NAME, "sample": sample},
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    emit(line, args.log)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--headline-only", action="store_true", help="skip the other workloads")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--cpu-seconds", type=float, default=20.0)
    ap.add_argument("--log", metavar="PATH", help="also append the line, with the commit it ran from, to PATH "
                                                  "(JSON lines)")
    ap.add_argument("--only", choices=["fp32-causal-2048", "fp32-causal-2048-padded", "bf16-causal-4096",
                                       "fp32-small", "small-graph", "layer-out-fp32", "layer-out-bf16", "layer-out-f16",
                                       "chunked-100k", "attn-window-bf16", "sublayer-fp32"],
                    help="time one named attention workload alone and print its figures (no contract line)")
    ap.add_argument("--require-clean", action="store_true",
                    help="refuse to run unless the git work tree matches its commit (tracked files unmodified), "
                         "so that a logged number names the code it measured")
    args = ap.parse_args()
    if args.require_clean:
        why = require_clean(_commit())
        if why is not None:
            print(json.dumps({"error": why}))
            sys.exit(2)
    if args.warmup < 3 and args.impl == "ours":
        ap.error("--warmup must be at least 3")
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        # no launcher set up the ranks: start one process per GPU the same way
        # torchrun would (independent replicas; rank 0 prints the line)
        if args.impl == "ours" and torch.cuda.device_count() < args.gpus:
            ap.error(f"--gpus {args.gpus}: only {torch.cuda.device_count()} GPU(s) visible")
        import socket
        with socket.socket() as sk:
            sk.bind(("127.0.0.1", 0))
            port = sk.getsockname()[1]
        cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={args.gpus}",
               "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.abspath(__file__)] + sys.argv[1:]
        sys.exit(subprocess.run(cmd).returncode)
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
