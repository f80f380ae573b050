#!/usr/bin/env python
"""Throughput of the channelwise gated delta rule forward on GB300.

One JSON line on stdout (rank 0).  The headline is prefill tokens/s on the
long-prefill workload (B=4, T=16384, HK=16, HV=32, dk=dv=128, chunk 64, bf16
q/k/v, float32 g/beta/state, beta near 1 and slow decay, nonzero h0): a step
is one gdr_forward over that batch, inputs resident in HBM (2.7 GB, larger
than L2, so no flush is needed).  The same line carries the decode half of
the metric under "decode": one T=1 step for B=64 sequences with the float32
state updated in place, reported as state GB/s (read + write); four input
sets (4 x 134 MB of state) are rotated so each step streams its state from
HBM rather than L2.

    python bench.py [--steps K] [--warmup W] [--impl gdr|reference]

--impl reference times the fp64 CPU oracle (the reference arm of this
build) on a bounded sample of the same workload, in the same unit.
Under torchrun each rank runs the same per-GPU workload (weak scaling, no
collective on the data path); timing is the max over ranks.
"""
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

import torch  # noqa: E402

METRIC = "GDR prefill tokens/s (HV=32,d=128) and decode state HBM GB/s, 1×GB300"
PREFILL = "prefill_t16k"
DECODE = "decode_b64"

# DRAM bytes (read + write) per launch from an ncu capture, keyed by kernel,
# with the sha256 of the source file the capture was taken from: a kernel
# whose source has changed since reports traffic null.
NCU_TRAFFIC = {
    # decode B64: one launch of the persistent bulk-copy kernel, --set full
    # capture (136.4 MB read + 74.2 MB written)
    "gdr_decode_kernel": {"bytes": 210_509_000, "sha": "5f7ea947d98305b5"},
    # prefill_t16k: one launch of the warp-specialised kernel, DRAM counters
    # (2.1658 GB read + 0.5204 GB written)
    "gdr_prefill_fused": {"bytes": 2_686_235_392, "sha": "98697b02e7caf9d6"},
}


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["gdr", "reference"], default="gdr")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workload", choices=["all", "prefill", "decode", "prefill_t4k", "tree",
                                           "ragged_f32", "prefill_f32_t16k",
                                           "prefill_f32_t4k"],
                    default="all",
                    help="prefill: the headline only; decode: only the decode measurement "
                         "(printed as its own line, for profiling the decode kernel); "
                         "prefill_t4k: the B=1 T=4096 prefill alone (its own line), the "
                         "small-batch case the segmented state scan serves; tree: tree "
                         "verification of 8 beam trees of 512 draft tokens (its own line); "
                         "ragged_f32: the ragged float32 batch through the packed entry "
                         "(its own line); prefill_f32_t16k / prefill_f32_t4k: the long-"
                         "prefill and the 4k-prefill shapes with float32 q/k/v (own lines)")
    ap.add_argument("--no-segments", action="store_true",
                    help="prefill workloads: one walk per head (GDR_FLAG_NO_SEGMENTS)")
    return ap.parse_args()


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


# ----------------------------------------------------------------- clocks
class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi every 200 ms."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.device = str(device_index)
        self.rows = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.device, "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) == 7:
                self.rows.append(parts)

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=5)
        sm = [float(r[0]) for r in self.rows if r[0].replace(".", "", 1).isdigit()]
        mx = [float(r[1]) for r in self.rows if r[1].replace(".", "", 1).isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in self.rows for i in range(4)
                          if r[3 + i].lower().startswith("active")})
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": reasons, "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(sm)}


# ----------------------------------------------------------------- helpers
def src_sha(name):
    with open(os.path.join(ROOT, "channelwise_gated_delta_gb300", "csrc", name), "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


KERNEL_SOURCE = {"gdr_decode_kernel": "decode.cu", "gdr_chunk_prep": "prefill_generic.cu",
                 "gdr_chunk_scan": "prefill_generic.cu", "gdr_prefill_fused": "prefill_tc.cu",
                 "gdr_chunk_prep_tc": "prep_tc.cu", "gdr_chunk_scan_tc": "scan_tc.cu"}


def traffic_for(kernel):
    rec = NCU_TRAFFIC.get(kernel)
    src = KERNEL_SOURCE.get(kernel)
    if not rec or not src or rec["sha"] != src_sha(src):
        return None
    return rec["bytes"]


def prefill_bytes_per_launch(w):
    """Algorithmic HBM bytes of one prefill call: every input read once, every
    output written once (q, k per key head; v, g, beta, o per value head;
    h0 read and ht written once per head)."""
    es = torch.tensor([], dtype=w.dtype).element_size()
    per_token = (2 * w.HK * w.dk * es + w.HV * w.dv * es + w.HV * w.dk * 4 + w.HV * 4 +
                 w.HV * w.dv * es)
    state = w.B * w.HV * w.dk * w.dv * 4 * (2 if w.h0 else 1)
    return w.B * w.T * per_token + state, per_token


def decode_bytes_per_launch(w):
    es = torch.tensor([], dtype=w.dtype).element_size()
    state = 2 * w.B * w.HV * w.dk * w.dv * 4
    small = w.B * (2 * w.HK * w.dk * es + w.HV * w.dv * es + w.HV * w.dk * 4 + w.HV * 4 +
                   w.HV * w.dv * es)
    return state + small, state


# GB300 HBM3e nominal bandwidth, reported beside the measured-peak fraction
NOMINAL_HBM_GBS = 8000.0


def roofline(kernel, launches, total_ms, bytes_per_launch, peak, peak_kind):
    avg_s = total_ms / 1e3 / max(launches, 1)
    achieved = bytes_per_launch / avg_s / 1e9
    return {"bound": "hbm", "kernel": kernel, "achieved": round(achieved, 1),
            "peak": peak, "peak_source": peak_kind, "unit": "GB/s",
            "frac": round(achieved / peak, 4), "traffic": traffic_for(kernel),
            "frac_nominal": round(achieved / NOMINAL_HBM_GBS, 4),
            "avg_launch_us": round(avg_s * 1e6, 2), "launches": launches}


def max_over_ranks(x, ws):
    """Largest value of x over all ranks (timing: the slowest rank counts)."""
    if ws == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


# ----------------------------------------------------------------- GPU arm
def timed_pass(steps, step, stream, dev, ws, traced):
    """K steps between CUDA events on `stream`, a barrier and a device
    synchronize on both sides; the library's launch trace on or off."""
    from channelwise_gated_delta_gb300 import gdr_trace_enable
    barrier(ws)
    torch.cuda.synchronize(dev)
    gdr_trace_enable(traced)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(steps):
        step()
    t1.record(stream)
    torch.cuda.synchronize(dev)
    gdr_trace_enable(False)
    barrier(ws)
    return t0.elapsed_time(t1)


def bench_prefill(args, ws, rank, dev, name=PREFILL):
    from channelwise_gated_delta_gb300 import (GDR_FLAG_NO_SEGMENTS, gdr_forward, gdr_trace_enable,
                                               gdr_trace_read)
    from channelwise_gated_delta_gb300.inputs import WORKLOADS, draw_workload

    w = WORKLOADS[name]
    flags = GDR_FLAG_NO_SEGMENTS if args.no_segments else 0
    d = draw_workload(w, seed=1000 + rank, device=dev)
    out = torch.empty(w.B, w.T, w.HV, w.dv, dtype=w.dtype, device=dev)
    ht = torch.empty(w.B, w.HV, w.dk, w.dv, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        gdr_forward(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], out=out, ht=ht,
                    chunk=w.chunk, stream=stream, flags=flags)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    gdr_trace_read()
    clocks = ClockSampler(dev.index if ws == 1 else int(os.environ.get("LOCAL_RANK", "0")))
    clocks.start()
    # the K steps as a caller runs them, then the same K steps again with the
    # library's launch trace (two events around each launch) for the
    # kernels' own times and the launch count
    ms = timed_pass(args.steps, step, stream, dev, ws, traced=False)
    ms_traced = timed_pass(args.steps, step, stream, dev, ws, traced=True)
    clk = clocks.stop()
    trace = gdr_trace_read()
    ms = max_over_ranks(ms, ws)
    tokens = w.B * w.T * args.steps * ws
    res = dict(w=w, ms=ms, ms_traced=ms_traced, tokens_per_s=tokens / (ms / 1e3), trace=trace,
               clocks=clk)

    if not args.no_e2e:
        res["e2e"] = bench_prefill_e2e(args, w, d, out, ht, stream, dev, ws)
    del d
    return res


def bench_prefill_e2e(args, w, d, out, ht, stream, dev, ws):
    """Same metric through the public C ABI with HOST buffers
    (gdr_forward_host): per step every input is copied in from pinned host
    memory and the output and final state are copied back to pinned host
    memory, the batch elements pipelined through two device slots."""
    from channelwise_gated_delta_gb300 import gdr_forward_host, gdr_host_staging_bytes
    names = ("q", "k", "v", "g", "beta", "h0")
    host = {n: d[n].to("cpu").pin_memory() for n in names}
    out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    ht_h = torch.empty(ht.shape, dtype=ht.dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = out_h.numel() * out_h.element_size() + ht_h.numel() * ht_h.element_size()
    steps = max(1, min(args.steps, 5))
    staging = torch.empty(gdr_host_staging_bytes(w.B, w.T, w.HK, w.HV, w.dk, w.dv, w.chunk,
                                                 w.dtype), dtype=torch.uint8, device=dev)

    def step():
        gdr_forward_host(host["q"], host["k"], host["v"], host["g"], host["beta"], host["h0"],
                         out_h, ht_h, chunk=w.chunk, stream=stream, staging=staging)

    for _ in range(2):  # warm-up: first touches of the pinned buffers and the staging
        step()
    torch.cuda.synchronize(dev)
    barrier(ws)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(steps):
        step()
    t1.record(stream)
    torch.cuda.synchronize(dev)
    ms = max_over_ranks(t0.elapsed_time(t1), ws)
    del staging
    return {"value": round(w.B * w.T * steps * ws / (ms / 1e3), 1), "unit": "tokens/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": steps,
            "ms_per_step": round(ms / steps, 3),
            "path": "gdr_forward_host: pinned host buffers streamed in 2048-token segments "
                    "through two device slots, copies in and out overlapped with compute"}


def bench_decode(args, ws, rank, dev, peak, peak_kind):
    from channelwise_gated_delta_gb300 import gdr_forward, gdr_trace_enable, gdr_trace_read
    from channelwise_gated_delta_gb300.inputs import WORKLOADS, draw_workload

    w = WORKLOADS[DECODE]
    nbuf = 4
    sets = [draw_workload(w, seed=2000 + 10 * rank + i, device=dev) for i in range(nbuf)]
    outs = [torch.empty(w.B, 1, w.HV, w.dv, dtype=w.dtype, device=dev) for _ in range(nbuf)]
    stream = torch.cuda.current_stream(dev)
    steps = max(args.steps, 20)

    def step(i):
        s = sets[i % nbuf]
        gdr_forward(s["q"], s["k"], s["v"], s["g"], s["beta"], s["h0"], out=outs[i % nbuf],
                    ht=s["h0"], chunk=w.chunk, stream=stream)

    for i in range(max(args.warmup, 3)):
        step(i)
    torch.cuda.synchronize(dev)
    gdr_trace_read()

    def timed(traced):
        barrier(ws)
        gdr_trace_enable(traced)
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for i in range(steps):
            step(i)
        t1.record(stream)
        torch.cuda.synchronize(dev)
        gdr_trace_enable(False)
        return t0.elapsed_time(t1)

    # the steps as a caller runs them (no launch trace: its two events per
    # launch are a few microseconds of a 46-microsecond step), then the same
    # steps again with the trace for the kernel's own time and launch count
    ms = max_over_ranks(timed(False), ws)
    ms_traced = timed(True)
    trace = gdr_trace_read()
    total_bytes, state_bytes = decode_bytes_per_launch(w)
    n, kms = trace.get("gdr_decode_kernel", (0, 0.0))
    state_gbs = state_bytes * steps * ws / (ms / 1e3) / 1e9
    res = {"workload": "decode B64 T1 HK16 HV32 dk=dv=128 bf16 q/k/v, f32 g/beta, f32 state in "
                       "place; 4 rotating input sets (537 MB of state > L2)",
           "value": round(state_gbs, 1), "unit": "GB/s (state read+write)",
           "tokens_per_s": round(w.B * steps * ws / (ms / 1e3), 1),
           "ms_per_step": round(ms / steps, 4), "steps": steps,
           "ms_per_step_traced": round(ms_traced / steps, 4),
           "roofline": roofline("gdr_decode_kernel", n, kms, total_bytes, peak, peak_kind),
           "gpu_launches": sum(v[0] for v in trace.values())}
    res["roofline"]["state_gbs_kernel"] = round(state_bytes / (kms / 1e3 / max(n, 1)) / 1e9, 1)
    del sets
    return res


# ----------------------------------------------------------------- CPU oracle
def oracle_batch_element(w, seed, threads=None, T=None):
    """Times the fp64 oracle on one batch element of workload w (all HV value
    heads, T tokens, w's distributions).  Returns (seconds, head_tokens, cores)."""
    import oracle
    from channelwise_gated_delta_gb300.inputs import draw, to_f64
    T = T or w.T
    d = draw(1, T, w.HK, w.HV, w.dk, w.dv, dtype=w.dtype, h0=w.h0, seed=seed, g_mu=w.g_mu,
             g_sigma=w.g_sigma, beta_mu=w.beta_mu, beta_sigma=w.beta_sigma)
    arrs = [to_f64(d[n]) for n in ("q", "k", "v", "g", "beta")]
    h0 = to_f64(d["h0"])
    del d
    cores = threads or oracle.default_threads()
    t = time.perf_counter()
    oracle.recurrence(*arrs, h0, threads=cores)
    dt = time.perf_counter() - t
    return dt, w.HV * T, min(cores, w.HV)


def cpu_baseline(w):
    """The oracle over the whole workload, one batch element at a time."""
    import oracle
    cores = oracle.default_threads()
    total_s, head_tokens, used = 0.0, 0, 1
    for bi in range(w.B):
        dt, ht_, used = oracle_batch_element(w, seed=7 + bi, threads=cores)
        total_s += dt
        head_tokens += ht_
    tok_s = head_tokens / total_s / w.HV
    return {"value": round(tok_s, 2), "unit": "tokens/s", "cores": used, "kind": "oracle",
            "sample": "the full workload: %d batch elements x %d value heads x %d tokens, fp64 "
                      "recurrence, %.1f s of oracle time" % (w.B, w.HV, w.T, total_s)}


def prefill_config(w, ws):
    """The workload the headline metric is quoted on (both arms report it)."""
    return {"workload": "prefill B4 T16384 HK16 HV32 dk=dv=128 chunk64, bf16 q/k/v, f32 "
                        "g/beta/state, beta=sigmoid(N(2,0.5)), g=-softplus(N(-3,1)), "
                        "h0=0.3N(0,1)",
            "B": w.B, "T": w.T, "HK": w.HK, "HV": w.HV, "dk": w.dk, "dv": w.dv,
            "chunk": w.chunk, "l2": "inputs 2.7 GB > L2 (no flush); decode rotates 4 "
                                    "state sets (537 MB)",
            "parallelism": "replicas" if ws > 1 else "single"}


def run_reference(args):
    """Reference arm: the fp64 oracle on the host cores, same metric and unit.
    Each step is one batch element of the workload (all value heads, all tokens)."""
    from channelwise_gated_delta_gb300.inputs import WORKLOADS
    import oracle
    w = WORKLOADS[PREFILL]
    cores = oracle.default_threads()
    for i in range(args.warmup):
        oracle_batch_element(w, seed=50 + i, threads=cores, T=64)
    total_s, total_ht, used = 0.0, 0, 1
    for i in range(args.steps):
        dt, ht_, used = oracle_batch_element(w, seed=100 + i, threads=cores)
        total_s += dt
        total_ht += ht_
    tok_s = total_ht / total_s / w.HV
    sample = "one batch element per step (%d value heads x %d tokens) of the %s workload" % (
        w.HV, w.T, w.name)
    line = {"impl": "reference", "metric": METRIC, "value": round(tok_s, 3), "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(1e3 * total_s / args.steps, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": prefill_config(w, args.gpus),
            "cpu_baseline": {"value": round(tok_s, 3), "unit": "tokens/s", "cores": used,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(tok_s, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)


def bench_small_prefill(args, ws, rank, dev, hbm_peak, peak_kind):
    """prefill_t4k (B=1, 32 value heads): one line of its own.  The automatic
    route cuts the state scan into segments here, so a step is several
    launches (the segment waves, their state set-up and the map combine);
    its roofline is the step's algorithmic bytes over the device time of
    all of them."""
    args.no_e2e = True
    pre = bench_prefill(args, ws, rank, dev, name="prefill_t4k")
    w = pre["w"]
    bytes_step, per_token = prefill_bytes_per_launch(w)
    trace = pre["trace"]
    dev_ms = sum(v[1] for v in trace.values())
    roof = roofline("step: " + " + ".join(sorted(trace)), args.steps, dev_ms, bytes_step,
                    hbm_peak, peak_kind)
    roof["algorithmic_bytes_per_token"] = per_token
    line = {
        "metric": "GDR prefill tokens/s [prefill_t4k]", "value": round(pre["tokens_per_s"], 1),
        "unit": "tokens/s", "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(pre["ms"] / args.steps, 4),
        "ms_per_step_traced": round(pre["ms_traced"] / args.steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "prefill B1 T4096 HK16 HV32 dk=dv=128 chunk64, bf16 q/k/v, "
                               "f32 g/beta, no h0, final state stored",
                   "l2": "inputs 168 MB > 129 MB L2, streamed once per step"},
        "roofline": roof,
        "kernels": {k: {"launches": v[0], "ms_total": round(v[1], 3)} for k, v in trace.items()},
        "gpu_launches": sum(v[0] for v in trace.values()),
        "clocks": pre["clocks"],
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


def timed_steps(args, dev, step):
    """W untimed steps, then K steps between CUDA events on the current
    stream (untraced: the value), the same K steps again with the library's
    launch trace (the kernels' times), and the SM clocks over both."""
    from channelwise_gated_delta_gb300 import gdr_trace_read
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    gdr_trace_read()
    clocks = ClockSampler(dev.index)
    clocks.start()
    stream = torch.cuda.current_stream(dev)
    ms = timed_pass(args.steps, step, stream, dev, 1, traced=False)
    timed_pass(args.steps, step, stream, dev, 1, traced=True)
    clk = clocks.stop()
    return ms, gdr_trace_read(), clk


def side_line(args, metric, workload, tokens, bytes_step, dtype, ms, trace, clk, hbm_peak,
              peak_kind):
    """One JSON line for a side workload: tokens/s over the timed steps, and
    the step's algorithmic bytes over the device time of all its launches."""
    dev_ms = sum(v[1] for v in trace.values())
    roof = roofline("step: " + " + ".join(sorted(trace)), args.steps, dev_ms, bytes_step,
                    hbm_peak, peak_kind)
    return {
        "metric": metric, "value": round(tokens * args.steps / (ms / 1e3), 1), "unit": "tokens/s",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms / args.steps, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": dtype, "data": "synthetic",
        "config": {"workload": workload}, "roofline": roof,
        "kernels": {k: {"launches": v[0], "ms_total": round(v[1], 3)} for k, v in trace.items()},
        "gpu_launches": sum(v[0] for v in trace.values()), "clocks": clk,
    }


def bench_tree(args, dev, hbm_peak, peak_kind):
    """Tree verification: 8 beam-shaped draft trees of 512 tokens (up to 4
    children a node), HK=16, HV=32, dk=dv=128, bf16 q/k/v, with h0.  Bytes per
    step: q, k per key head, v, g, beta and o per value head, h0 read once."""
    from channelwise_gated_delta_gb300 import gdr_forward_tree
    from channelwise_gated_delta_gb300.inputs import draw, draw_parents
    B, T, HK, HV, d = 8, 512, 16, 32, 128
    x = {k: (None if v is None else v.to(dev))
         for k, v in draw(B, T, HK, HV, d, d, dtype=torch.bfloat16, seed=1).items()}
    parent = draw_parents(B, T, "beam", seed=1, branching=4)
    out = torch.empty(B, T, HV, d, dtype=torch.bfloat16, device=dev)
    ws = torch.empty(1 << 30, dtype=torch.uint8, device=dev)

    def step():
        gdr_forward_tree(x["q"], x["k"], x["v"], x["g"], x["beta"], parent, h0=x["h0"], out=out,
                         workspace=ws)

    ms, trace, clk = timed_steps(args, dev, step)
    per_token = 2 * HK * d * 2 + HV * d * 2 + HV * d * 4 + HV * 4 + HV * d * 2
    bytes_step = B * T * per_token + B * HV * d * d * 4
    return side_line(args, "GDR tree verification tokens/s [tree B8 T512 beam]",
                     "tree verification B8 T512 (beam trees, up to 4 children) HK16 HV32 "
                     "dk=dv=128, bf16 q/k/v, f32 g/beta/h0, blocked solve",
                     B * T, bytes_step, "bf16", ms, trace, clk, hbm_peak, peak_kind)


def bench_ragged_f32(args, dev, hbm_peak, peak_kind):
    """The ragged float32 batch (lengths 1 .. 512, h0 given) through the
    packed entry: the single token on the decode kernel, the rest on the
    chunk prep and the tensor-core state scan."""
    from channelwise_gated_delta_gb300 import gdr_forward_varlen
    from channelwise_gated_delta_gb300.inputs import WORKLOADS, draw_workload, pack
    w = WORKLOADS["ragged_b8"]
    packed, cu = pack(draw_workload(w, seed=1))
    x = {k: (None if v is None else v.to(dev)) for k, v in packed.items()}
    ws = torch.empty(1 << 28, dtype=torch.uint8, device=dev)
    tokens = cu[-1]

    def step():
        gdr_forward_varlen(x["q"], x["k"], x["v"], x["g"], x["beta"], cu, h0=x["h0"],
                           chunk=w.chunk, workspace=ws)

    ms, trace, clk = timed_steps(args, dev, step)
    per_token = 2 * w.HK * w.dk * 4 + w.HV * w.dv * 4 + w.HV * w.dk * 4 + w.HV * 4 + w.HV * w.dv * 4
    bytes_step = tokens * per_token + 2 * (len(cu) - 1) * w.HV * w.dk * w.dv * 4
    return side_line(args, "GDR prefill tokens/s [ragged_b8 f32]",
                     "ragged batch, lengths 1 33 49 64 97 128 256 512, HK16 HV32 dk=dv=128 "
                     "chunk64, f32 q/k/v/g/beta/state, h0 given, packed entry",
                     tokens, bytes_step, "f32", ms, trace, clk, hbm_peak, peak_kind)


def bench_f32_prefill(args, dev, hbm_peak, peak_kind, long):
    """A prefill shape with float32 q/k/v through gdr_forward: the chunk prep
    and the state scan on the tensor cores (BF16x3).  long: the long-prefill
    stress shape (B4 T16384 HK16 HV32, slow decay, beta near 1, h0 given);
    else the 4k prefill (B1 T4096, the configs' default decay and beta, h0 =
    0), whose scan the automatic choice cuts into segments."""
    from channelwise_gated_delta_gb300 import gdr_forward
    from channelwise_gated_delta_gb300.inputs import draw
    HK, HV, d = 16, 32, 128
    if long:
        B, T = 4, 16384
        x = draw(B, T, HK, HV, d, d, dtype=torch.float32, seed=1, g_mu=-3.0, g_sigma=1.0,
                 beta_mu=2.0, beta_sigma=0.5, h0=True, device=dev)
    else:
        B, T = 1, 4096
        x = draw(B, T, HK, HV, d, d, dtype=torch.float32, seed=1, h0=False, device=dev)
    out = torch.empty(B, T, HV, d, dtype=torch.float32, device=dev)
    ht = torch.empty(B, HV, d, d, dtype=torch.float32, device=dev)

    def step():
        gdr_forward(x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"], out=out, ht=ht, chunk=64)

    ms, trace, clk = timed_steps(args, dev, step)
    per_token = 2 * HK * d * 4 + HV * d * 4 + HV * d * 4 + HV * 4 + HV * d * 4
    bytes_step = B * T * per_token + (2 if long else 1) * B * HV * d * d * 4
    if long:
        return side_line(args, "GDR prefill tokens/s [prefill_t16k shape, f32 q/k/v]",
                         "B4 T16384 HK16 HV32 dk=dv=128 chunk64, f32 q/k/v/g/beta/state, beta "
                         "near 1, slow decay, h0 given; chunk prep and state scan on tcgen05",
                         B * T, bytes_step, "f32", ms, trace, clk, hbm_peak, peak_kind)
    return side_line(args, "GDR prefill tokens/s [prefill_t4k shape, f32 q/k/v]",
                     "B1 T4096 HK16 HV32 dk=dv=128 chunk64, f32 q/k/v/g/beta/state, h0 = 0; "
                     "chunk prep and state scan on tcgen05, scan segmented automatically",
                     B * T, bytes_step, "f32", ms, trace, clk, hbm_peak, peak_kind)


# ----------------------------------------------------------------- main
def main():
    args = parse_args()
    ws, rank, local = dist_env()
    if args.impl == "reference":
        if rank == 0:
            run_reference(args)
        return
    if args.warmup < 3:
        args.warmup = 3
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if ws > 1 else torch.cuda.current_device())
    hbm_peak, _, peak_kind = load_peaks()

    if args.workload in ("tree", "ragged_f32", "prefill_f32_t16k", "prefill_f32_t4k"):
        if rank == 0:
            fn = {"tree": bench_tree, "ragged_f32": bench_ragged_f32,
                  "prefill_f32_t16k": lambda *a: bench_f32_prefill(*a, long=True),
                  "prefill_f32_t4k": lambda *a: bench_f32_prefill(*a, long=False)}[args.workload]
            print(json.dumps(fn(args, dev, hbm_peak, peak_kind)), flush=True)
        if ws > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return
    if args.workload == "prefill_t4k":
        bench_small_prefill(args, ws, rank, dev, hbm_peak, peak_kind)
        if ws > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return
    if args.workload == "decode":
        dec = bench_decode(args, ws, rank, dev, hbm_peak, peak_kind)
        if rank == 0:
            print(json.dumps({"metric": METRIC + " [decode only]", "decode": dec}), flush=True)
        if ws > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return
    pre = bench_prefill(args, ws, rank, dev)
    w = pre["w"]
    dec = None if args.workload == "prefill" else bench_decode(args, ws, rank, dev, hbm_peak,
                                                               peak_kind)

    bytes_launch, per_token = prefill_bytes_per_launch(w)
    trace = pre["trace"]
    dom = max(trace.items(), key=lambda kv: kv[1][1]) if trace else ("none", (0, 0.0))
    line = {
        "metric": METRIC, "value": round(pre["tokens_per_s"], 1), "unit": "tokens/s",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(pre["ms"] / args.steps, 4),
        "ms_per_step_traced": round(pre["ms_traced"] / args.steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": prefill_config(w, ws),
        "roofline": roofline(dom[0], dom[1][0], dom[1][1], bytes_launch, hbm_peak, peak_kind),
        "kernels": {k: {"launches": v[0], "ms_total": round(v[1], 3)} for k, v in trace.items()},
        "gpu_launches": sum(v[0] for v in trace.values()),
        "clocks": pre["clocks"],
    }
    line["roofline"]["algorithmic_bytes_per_token"] = per_token
    if "e2e" in pre:
        line["e2e"] = pre["e2e"]
    if dec is not None:
        line["decode"] = dec
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
