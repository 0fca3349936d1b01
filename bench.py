"""Benchmark of the MLA decode post-attention stage on GB300.

One step = one call of the whole stage (LSE combine -> MXFP4 latents -> W_UV
-> gate) over the large multi-token-prediction batch: 1024 requests x q=4
(S=4096 tokens), 96 heads, 4 splits per request (compact [4, 4096, 96, 512]
bf16 partials, lse with 2% -inf), MXFP4 W_V.  It is the largest single-GPU
workload of the recipe and the one that runs every step of the path.

Prints one JSON line.  ``value`` is tokens/s over all ranks with the inputs
resident in HBM (device-timed with CUDA events on the launching stream);
``e2e`` is the same metric through the Python binding with the step's inputs
copied from pinned host memory and the output copied back inside the timed
region.  ``--impl reference`` times the CPU oracle instead (bounded samples
of the same workload).

Multi-GPU: the stage has no exchange step on one GPU's data, so N > 1 runs N
independent replicas (one per rank, launched by torch.distributed.run) and
``value`` sums their tokens over the slowest rank's time.
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
sys.path.insert(0, ROOT)

METRIC = "combine+W_UV tokens/s and achieved HBM GB/s (% of GB300 roofline)"
DEFAULT_WORKLOAD = "mtp_mxfp4"
L2_DEFEAT_BYTES = 256 << 20  # working set per rotation, about twice the 129 MB L2


# nominal figures, for the labelled second fraction only (the measured peaks
# are the denominators of `frac`)
NOMINAL_HBM_GBS = 7900.0            # HBM3e, nominal
NOMINAL_FP4_OVER_BF16 = 13.5 / 2.25  # dense tensor-core rates, nominal
OPROJ_N_OUT = 7168  # o_proj outputs of the decode step (the hidden size; K = 12 heads x 128)


def nominal_hbm(achieved_gbs: float) -> dict:
    """The labelled second fraction of an HBM-bound line: achieved GB/s over
    the nominal HBM3e rate (the first, `frac`, is over the measured copy peak)."""
    return {"peak": NOMINAL_HBM_GBS, "unit": "GB/s", "frac": achieved_gbs / NOMINAL_HBM_GBS,
            "peak_source": "nominal HBM3e 7.9 TB/s"}
DECODE_WORKLOADS = ("tiny_split", "nosplit", "splitkv", "splitkv_rm", "stacked_mxfp4")


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d.get("hbm_gbs", 6800.0), "measured"
    return 6800.0, "fallback"


def tensor_peak(w_fmt: int):
    """(TFLOP/s, description) of the tensor-core peak for the W_UV contraction
    of a W_V format: the measured bf16 burst rate, times the nominal FP4:bf16
    ratio for MXFP4."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    bf16, src = 1900.0, "fallback bf16 1900 TFLOP/s"
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        if "bf16_tflops" in d:
            bf16, src = d["bf16_tflops"], f"measured bf16 {d['bf16_tflops']} TFLOP/s (burst)"
    if w_fmt == 1:
        return bf16 * NOMINAL_FP4_OVER_BF16, f"{src} x {NOMINAL_FP4_OVER_BF16:g} (nominal FP4:bf16 ratio)"
    return bf16, src


# the source file of each kernel named in a bench line; the shared headers
# (device helpers, parameter structs, launch declarations) count for every one
KERNEL_FILES = {"tc": "kernel_tc.cu", "tc_ksplit_cluster4": "kernel_ks.cu", "simt": "kernel_simt.cu",
                "dcp_pack": "kernel_pack.cu", "attn_split_kv": "kernel_attn.cu",
                "attn_combine_uv_fused": "kernel_attn.cu", "attn_combine_uv_oproj_fused": "kernel_attn.cu",
                "o_proj": ("kernel_oproj.cu", "kernel_oproj.h")}
SHARED_SOURCES = ("device_common.cuh", "kernels.h", "kparams.h")


def kernel_source_hash(kernel: str | None = None) -> str:
    """Hash of the sources a kernel is built from (all of csrc/ when no kernel
    is named)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "mla_decode_attention_lse_gb300", "csrc")
    if kernel is None:
        files = sorted(os.listdir(csrc))
    else:
        own = KERNEL_FILES[kernel]
        files = sorted(SHARED_SOURCES + (own if isinstance(own, tuple) else (own,)))
    for f in files:
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(f.encode())
            h.update(fh.read())
    return h.hexdigest()[:16]


def traffic_from_profile(workload: str, kernel: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel sources (else None)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(f"{workload}/{kernel}")
    if not e or kernel not in KERNEL_FILES or e.get("source_hash") != kernel_source_hash(kernel):
        return None
    return e.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during a region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100", "-f", self.path],
                stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except FileNotFoundError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t_start: float | None = None):
        rows = []
        if self.path and os.path.exists(self.path):
            with open(self.path) as f:
                for line in f:
                    parts = [x.strip() for x in line.split(",")]
                    if len(parts) >= 9:
                        rows.append(parts)
            os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(rows)}


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def init_dist(ws, backend):
    import torch.distributed as dist

    if ws > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend)
    return dist


def reduce_max(x: float, dist, device=None) -> float:
    """Maximum of a per-rank value over all ranks (the value itself at N=1)."""
    import torch

    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_rate(tokens_per_step: int, steps: int, world: int, max_ms: float) -> float:
    """Whole-job tokens/s of `world` independent replicas: every rank's tokens
    over the slowest rank's time."""
    return tokens_per_step * steps * world / (max_ms / 1e3)


def host_cpu() -> dict:
    """The host the CPU baseline ran on: core count and model name."""
    model = ""
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                k = line.split(":")[0].strip().lower()
                if k in ("model name", "cpu part", "hardware") and not model:
                    model = line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform

    parts = {"0xd4f": "Arm Neoverse V2 (CPU part 0xd4f)", "0xd40": "Arm Neoverse V1 (CPU part 0xd40)"}
    model = parts.get(model, model)
    return {"nproc": os.cpu_count(), "cpu": model or platform.processor() or platform.machine()}


def cold_launch_us(fn, stream, dev) -> float:
    """One launch after the L2 is flushed (a 256 MB write), timed with events."""
    import torch

    flush = torch.empty(L2_DEFEAT_BYTES, dtype=torch.uint8, device=dev)
    times = []
    for _ in range(3):
        flush.fill_(1)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        fn()
        e1.record(stream)
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1) * 1e3)
    del flush
    return statistics.median(times)


def host_copy_inputs(inp):
    import torch

    pin = {}
    for k in ("o", "lse", "gate"):
        if inp[k] is not None:
            t = torch.empty(inp[k].shape, dtype=inp[k].dtype, pin_memory=True)
            t.copy_(inp[k])
            pin[k] = t
    return pin


def oracle_sample_rate(inp, budget_s: float, rows_hint: int | None = None):
    """Time the oracle (as it stands, one thread) on a bounded sample of the
    workload's (t, h) rows; returns (tokens/s, rows timed, seconds)."""
    import numpy as np

    import oracle

    pr = oracle.problem_from_tensors(inp)
    rng = np.random.default_rng(0)
    S, H = inp["S"], inp["H"]
    # calibrate on a few rows, then size the sample to the budget
    cal = 8
    t0 = time.perf_counter()
    pr.rows(rng.integers(0, S, cal), rng.integers(0, H, cal))
    per_row = (time.perf_counter() - t0) / cal
    n = rows_hint or max(H, int(budget_s / max(per_row, 1e-6)))
    ts = np.repeat(rng.integers(0, S, (n + H - 1) // H), H)[:n]
    hs = np.tile(np.arange(H), (n + H - 1) // H)[:n]
    t0 = time.perf_counter()
    pr.rows(ts, hs)
    dt = time.perf_counter() - t0
    return (n / H) / dt, n, dt, pr, per_row


def run_reference(args):
    """The oracle on the host cores, on bounded samples of the workload."""
    import torch

    ws, rank, _ = dist_env()
    if ws > 1:
        dist = init_dist(ws, "gloo")
        if rank != 0:
            dist.barrier()
            return
    import dataclasses

    from mla_decode_attention_lse_gb300 import synth

    # Every (t, h) row costs the oracle the same, so the sample is drawn from a
    # copy of the workload with 64 tokens (same heads, partials, splits, W_V
    # and value distributions) instead of generating all of it on the host.
    wl = synth.WORKLOADS[args.workload]
    s_small = max(wl.q, (min(wl.S, 64) // wl.q) * wl.q)
    small = dataclasses.replace(wl, S=s_small, S_out=None,
                                P=wl.P if wl.P in (1, wl.spr) else (s_small // wl.q) * wl.spr)
    inp = synth.make(small, device="cpu")
    S, H = inp["S"], inp["H"]
    # per-step sample sized so the whole run stays within ~2 minutes
    _, _, _, pr, per_row = oracle_sample_rate(inp, 0.0, rows_hint=H)
    budget = args.ref_budget / max(1, args.steps + args.warmup)
    rows = max(1, int(budget / max(per_row, 1e-6)))
    import numpy as np

    rng = np.random.default_rng(1)
    for _ in range(args.warmup):
        pr.rows(rng.integers(0, S, rows), rng.integers(0, H, rows))
    t0 = time.perf_counter()
    for _ in range(args.steps):
        pr.rows(rng.integers(0, S, rows), rng.integers(0, H, rows))
    dt = time.perf_counter() - t0
    value = rows * args.steps / H / dt
    sample = (f"{rows} random (t, h) rows per step from a {S}-token copy of {args.workload} "
              f"(H={H}, P={inp['P']}, same W_V and distributions)")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": args.workload, "S": wl.S, "H": H, "P": wl.P,
                   "w_fmt": ["bf16", "mxfp4"][inp["w_fmt"]]},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                         "sample": sample, "host": host_cpu()},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.barrier()


def run_gpu(args):
    import torch

    import mla_decode_attention_lse_gb300 as m
    from mla_decode_attention_lse_gb300 import synth

    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    dist = init_dist(ws, "nccl") if ws > 1 else None
    dev = torch.device("cuda", local)
    m.load_library()

    seed0 = synth.WORKLOADS[args.workload].seed + rank
    inp = synth.make(args.workload, device=dev, seed=seed0)
    S, H, S_out = inp["S"], inp["H"], inp["S_out"]
    nbytes = synth.algorithmic_bytes(inp)
    # Workloads smaller than L2 cycle through independent copies of every
    # input (W_V too: another layer's weights) so each step reads HBM.
    rotate = args.rotate
    if rotate == 0:
        rotate = 1 if nbytes >= L2_DEFEAT_BYTES else -(-L2_DEFEAT_BYTES // nbytes)
    copies = [inp] + [synth.make(args.workload, device=dev, seed=seed0 + 1000 * k) for k in range(1, rotate)]
    outs = [torch.empty(S_out, H * 128, dtype=torch.bfloat16, device=dev) for _ in range(rotate)]
    out = outs[0]
    stream = torch.cuda.current_stream(dev)

    def call(k=0):  # on the current stream (the capture stream inside a graph capture)
        c = copies[k % rotate]
        m.mla_combine_uv(c["o"], c["lse"], c["q"], c["spr"], c["w_v"], c["w_fmt"], c["gate"],
                         outs[k % rotate], w_scale=c["w_scale"], kernel=args.kernel,
                         tile_tokens=args.tile)

    a = m.make_args(inp["o"], inp["lse"], inp["q"], inp["spr"], inp["w_v"], inp["w_fmt"],
                    inp["gate"], out, inp["w_scale"], kernel=args.kernel, tile_tokens=args.tile)
    plan = m.mla_combine_uv_plan(a)
    kname = {m.MLA_KERNEL_TC: "tc", m.MLA_KERNEL_KSPLIT: "tc_ksplit_cluster4"}.get(plan["kernel"], "simt")
    use_graph = args.graph or (args.graph is None and nbytes < L2_DEFEAT_BYTES)

    for k in range(max(3, args.warmup)):
        call(k)
    torch.cuda.synchronize()
    assert m.mla_combine_uv_status(stream) == m.MLA_OK

    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    if use_graph:
        # the K launches back to back in one CUDA graph (no host launch gaps);
        # per-launch time = the replay's time / K
        graph = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream(dev)
        with torch.cuda.graph(graph, stream=cap):
            for k in range(args.steps):
                call(k)
        graph.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with ClockSampler(local) as clk:
            graph.replay()  # untimed: the GPU is busy right up to the timed replay
            t_wall0 = time.perf_counter()
            e0.record(stream)
            graph.replay()
            e1.record(stream)
            torch.cuda.synchronize()
            t_wall = time.perf_counter() - t_wall0
        total_ms = e0.elapsed_time(e1)
        kern_ms = [total_ms / args.steps]
    else:
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        with ClockSampler(local) as clk:
            # untimed warm-up steps again, enqueued right before the timed ones,
            # so the GPU does not idle (and drop its clocks) while the clock
            # sampler starts
            for k in range(args.warmup):
                call(k)
            t_wall0 = time.perf_counter()
            for i in range(args.steps):
                starts[i].record(stream)
                call(i)
                ends[i].record(stream)
            torch.cuda.synchronize()
            t_wall = time.perf_counter() - t_wall0
        kern_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
        total_ms = starts[0].elapsed_time(ends[-1])
    if dist:
        dist.barrier()
    clocks = clk.summary()
    assert m.mla_combine_uv_status(stream) == m.MLA_OK
    cold_us = cold_launch_us(lambda: call(0), stream, dev)

    # max over ranks of the timed region
    total_ms = reduce_max(total_ms, dist, dev)
    value = replica_rate(S, args.steps, ws, total_ms)
    avg_kern_s = statistics.mean(kern_ms) / 1e3
    peak, peak_kind = load_peaks()
    achieved = nbytes / avg_kern_s / 1e9
    nbytes_all = synth.algorithmic_bytes_all_rows(inp)
    tflops = synth.flops(inp) / avg_kern_s / 1e12
    tpeak, tpeak_src = tensor_peak(inp["w_fmt"])

    # end to end: pinned host inputs -> device, the call, output -> host, with
    # the copies of step i+1 overlapping the call and read-back of step i
    e2e_steps = max(3, min(args.steps, 20))
    e2e_ms, h2d, d2h = e2e_overlapped(m, inp, out.shape, args, stream, dev, e2e_steps, dist)
    e2e_value = replica_rate(S, e2e_steps, ws, e2e_ms)
    decode = None
    if args.workload == DEFAULT_WORKLOAD and ws == 1 and not args.no_decode:
        decode = decode_leg(m, synth, dev, stream, args.decode_launches)

    line = None
    if rank == 0:
        cpu = None
        if not args.no_cpu_baseline and ws == 1:
            host_inp = {k: (v.cpu() if hasattr(v, "cpu") else v) for k, v in inp.items()}
            rate, n, dt, _, _ = oracle_sample_rate(host_inp, args.cpu_budget)
            cpu = {"value": rate, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                   "sample": f"{n} (t, h) rows ({n // H} tokens x {H} heads) of the same "
                             f"workload, single-threaded oracle, {dt:.1f} s", "host": host_cpu()}
        wl = synth.WORKLOADS[args.workload]
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": total_ms / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "mxfp4" if inp["w_fmt"] else "bf16",
            "data": "synthetic",
            "config": {"workload": f"{args.workload}: {wl.S // wl.q} requests x q={wl.q} "
                                   f"(S={S}), H={H}, {inp['spr']} splits per request, "
                                   f"P={inp['P']} "
                                   + ("passthrough" if inp["P"] == 1 else
                                      "compact" if inp["P"] == inp["spr"] else "request-major")
                                   + f", {'MXFP4' if inp['w_fmt'] else 'bf16'} W_V",
                       "S": S, "H": H, "P": inp["P"], "w_fmt": ["bf16", "mxfp4"][inp["w_fmt"]],
                       "parallelism": f"replicas x{ws}", "kernel": kname,
                       "tile_tokens": plan["tile_tokens"], "grid": plan["grid"],
                       "l2": (f"inputs {nbytes / 1e9:.2f} GB per step, larger than L2: no flush"
                              if rotate == 1 else
                              f"{rotate} independent input copies ({rotate * nbytes / 1e6:.0f} MB) "
                              "cycled, one per step: every step reads HBM"),
                       "timing": ("CUDA graph of the timed steps, per-step time = replay / steps"
                                  if use_graph else "CUDA events around each launch")},
            "achieved_gbs": achieved,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "peak_source": peak_kind,
                         "traffic": traffic_from_profile(args.workload, kname),
                         "algorithmic_bytes": nbytes,
                         "algorithmic_bytes_note": "partial rows with a finite LSE (the rows that can "
                                                   "carry weight) + LSE + W_V + gate + out",
                         "algorithmic_bytes_all_rows": nbytes_all,
                         "frac_all_rows": nbytes_all / avg_kern_s / 1e9 / peak,
                         "nominal": nominal_hbm(achieved)},
            "tensor": {"tflops": tflops, "peak": tpeak, "frac": tflops / tpeak, "peak_source": tpeak_src},
            "kernel_ms": {"mean": statistics.mean(kern_ms), "min": min(kern_ms),
                          "max": max(kern_ms)},
            "cold_launch_us": cold_us,
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "steps": e2e_steps, "ms_per_step": e2e_ms / e2e_steps,
                    "link_h2d_gbs": h2d * e2e_steps / (e2e_ms / 1e3) / 1e9,
                    "copies": "double-buffered: step i+1's host->device copy (its own stream) overlaps "
                              "step i's call and its device->host read-back (a third stream)"},
            "gpu_launches": args.steps,
            "clocks": clocks,
            "wall_s": t_wall,
        }
        if decode is not None:
            line["decode"] = decode
        print(json.dumps(line), flush=True)
    if dist:
        dist.barrier()
        dist.destroy_process_group()
    return line


def e2e_overlapped(m, inp, out_shape, args, stream, dev, steps, dist):
    """Time `steps` end-to-end calls: each step copies its inputs from pinned
    host memory, calls the stage and reads the output back.  Two device input
    / output sets alternate, so the host->device copy of step i+1 (on its own
    stream) overlaps the call of step i and its read-back (a third stream).
    Returns (ms for all steps, max over ranks; h2d bytes per step; d2h bytes
    per step)."""
    import torch

    pin = host_copy_inputs(inp)
    outs_host = [torch.empty(tuple(out_shape), dtype=torch.bfloat16, pin_memory=True) for _ in range(2)]
    bufs = [{k: torch.empty_like(inp[k]) for k in pin} for _ in range(2)]
    outs = [torch.empty(tuple(out_shape), dtype=torch.bfloat16, device=dev) for _ in range(2)]
    cs_in, cs_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    comp_done, d2h_done = [None, None], [None, None]

    def step(i):
        b = i % 2
        if comp_done[b] is not None:  # the call of step i-2 has read set b
            cs_in.wait_event(comp_done[b])
        with torch.cuda.stream(cs_in):
            for k in pin:
                bufs[b][k].copy_(pin[k], non_blocking=True)
        h = torch.cuda.Event()
        h.record(cs_in)
        stream.wait_event(h)
        if d2h_done[b] is not None:  # out[b] of step i-2 has been read back
            stream.wait_event(d2h_done[b])
        m.mla_combine_uv(bufs[b]["o"], bufs[b].get("lse"), inp["q"], inp["spr"], inp["w_v"], inp["w_fmt"],
                         bufs[b]["gate"], outs[b], w_scale=inp["w_scale"], stream=stream, kernel=args.kernel,
                         tile_tokens=args.tile)
        c = torch.cuda.Event()
        c.record(stream)
        comp_done[b] = c
        cs_out.wait_event(c)
        with torch.cuda.stream(cs_out):
            outs_host[b].copy_(outs[b], non_blocking=True)
        d = torch.cuda.Event()
        d.record(cs_out)
        d2h_done[b] = d

    for i in range(2):
        step(i)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    cs_in.wait_event(e0)
    for i in range(steps):
        step(i)
    for d in d2h_done:
        stream.wait_event(d)
    e1.record(stream)
    torch.cuda.synchronize()
    assert m.mla_combine_uv_status(stream) == m.MLA_OK
    h2d = sum(t.numel() * t.element_size() for t in pin.values())
    d2h = outs_host[0].numel() * outs_host[0].element_size()
    return reduce_max(e0.elapsed_time(e1), dist, dev), h2d, d2h


def decode_leg(m, synth, dev, stream, launches):
    """The decode-shaped workloads, each timed like the headline's small
    cases: `launches` back-to-back calls captured in one CUDA graph over enough
    independent input copies (W_V included) that every launch reads HBM; and,
    in the same harness, the read-only streaming kernel reading the same byte
    count from a rotation of the same size (0 and 1 dependent round trips
    first) -- the fastest any single launch of that size can be -- plus the
    floor of a chain of launches that read almost nothing."""
    import torch

    peak, peak_kind = load_peaks()
    sink = torch.zeros(1, dtype=torch.int32, device=dev)

    def graph_time(fn):
        fn(0)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream(dev)
        with torch.cuda.graph(g, stream=cap):
            for k in range(launches):
                fn(k)
        g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        g.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        del g
        return e0.elapsed_time(e1) * 1e3 / launches  # us per launch

    def calib_us(nbytes, rot, trips):
        n16 = -(-nbytes // 16) * 16
        buf = torch.randn(rot * n16 // 4, device=dev)  # finite data
        us = graph_time(lambda k: m.mla_calib_stream_read(buf[(k % rot) * n16 // 4:], n16, trips, sink))
        del buf
        return us

    out = {"launches_per_graph": launches, "peak": peak, "peak_source": peak_kind,
           "nominal_peak": NOMINAL_HBM_GBS, "workloads": {}}
    with ClockSampler(torch.cuda.current_device()) as clk:
        tiny = torch.zeros(1 << 10, dtype=torch.float32, device=dev)
        out["launch_floor_us"] = graph_time(lambda k: m.mla_calib_stream_read(tiny, 64, 0, sink))
        for name in DECODE_WORKLOADS:
            wl = synth.WORKLOADS[name]
            inp = synth.make(name, device=dev, seed=wl.seed)
            nb = synth.algorithmic_bytes(inp)
            nb_all = synth.algorithmic_bytes_all_rows(inp)
            rot = -(-L2_DEFEAT_BYTES // nb)
            copies = [inp] + [synth.make(name, device=dev, seed=wl.seed + 1000 * k) for k in range(1, rot)]
            outs = [torch.empty(inp["S_out"], inp["H"] * 128, dtype=torch.bfloat16, device=dev) for _ in range(rot)]

            def call(k):
                c = copies[k % rot]
                m.mla_combine_uv(c["o"], c["lse"], c["q"], c["spr"], c["w_v"], c["w_fmt"], c["gate"],
                                 outs[k % rot], w_scale=c["w_scale"])

            a = m.make_args(inp["o"], inp["lse"], inp["q"], inp["spr"], inp["w_v"], inp["w_fmt"], inp["gate"],
                            outs[0], inp["w_scale"])
            plan = m.mla_combine_uv_plan(a)
            us = graph_time(call)
            assert m.mla_combine_uv_status(stream) == m.MLA_OK
            del copies, outs
            torch.cuda.empty_cache()
            c0 = calib_us(nb, rot, 0)
            c1 = calib_us(nb, rot, 1)
            gbs = nb / (us / 1e6) / 1e9
            out["workloads"][name] = {
                "us_per_launch": us, "algorithmic_bytes": nb, "algorithmic_bytes_all_rows": nb_all,
                "gbs": gbs, "frac": gbs / peak, "frac_all_rows": nb_all / (us / 1e6) / 1e9 / peak,
                "frac_nominal": gbs / NOMINAL_HBM_GBS,
                "ceiling_us": c0, "ceiling_dep1_us": c1, "ceiling_frac": nb / (c0 / 1e6) / 1e9 / peak,
                "of_ceiling": c0 / us, "rotation": rot,
                "kernel": {m.MLA_KERNEL_TC: "tc", m.MLA_KERNEL_KSPLIT: "tc_ksplit_cluster4"}.get(
                    plan["kernel"], "simt"), "tile_tokens": plan["tile_tokens"], "grid": plan["grid"]}
    out["clocks"] = clk.summary()
    return out


def dcp_oracle_rate(host, budget_s: float):
    """The oracle's DCP step on the host: the full pack for the destination
    rank, then the combine on a bounded sample of (t, h) rows.  Returns
    (tokens/s, description)."""
    import numpy as np

    import oracle

    import torch

    def u16(t):  # bf16 bits as uint16
        return t.contiguous().view(torch.int16).numpy().view(np.uint16)

    t0 = time.perf_counter()
    cmb_o, cmb_lse = oracle.dcp_pack(u16(host["o_all"]), host["lse_all"].numpy(), host["seq_lens"].numpy(),
                                     host["qsl"].numpy(), host["q"], host["dst"])
    t_pack = time.perf_counter() - t0
    ws = None if host["w_scale"] is None else host["w_scale"].numpy()
    w = u16(host["w_v"]) if host["w_fmt"] == 0 else host["w_v"].numpy()
    pr = oracle.Problem(cmb_o, cmb_lse, host["q"], host["R"], w, ws, host["w_fmt"], u16(host["gate"]))
    S, H = host["S"], host["H"]
    rng = np.random.default_rng(0)
    t0 = time.perf_counter()
    pr.rows(rng.integers(0, S, 8), rng.integers(0, H, 8))
    per_row = (time.perf_counter() - t0) / 8
    n = max(H, int(budget_s / max(per_row, 1e-6)))
    t0 = time.perf_counter()
    pr.rows(rng.integers(0, S, n), rng.integers(0, H, n))
    per_row = (time.perf_counter() - t0) / n
    step_s = t_pack + per_row * S * H
    desc = (f"full pack for rank {host['dst']} ({t_pack:.3f} s) + combine timed on {n} random (t, h) "
            f"rows and scaled to the step's {S * H}, single-threaded oracle")
    return host["live"] / step_s, desc


def run_reference_dcp(args):
    """The oracle's DCP step (full pack + sampled combine) on the host cores."""
    import torch

    ws, rank, _ = dist_env()
    if ws > 1:
        dist = init_dist(ws, "gloo")
        if rank != 0:
            dist.barrier()
            return
    from mla_decode_attention_lse_gb300 import synth

    wl = synth.DCP_WORKLOADS[args.workload]
    inp = synth.make_dcp(wl, device="cpu")
    budget = args.ref_budget / max(1, args.steps + args.warmup) / 2
    for _ in range(args.warmup):
        dcp_oracle_rate(inp, budget)
    secs, desc = 0.0, ""
    for _ in range(args.steps):
        rate, desc = dcp_oracle_rate(inp, budget)
        secs += inp["live"] / rate
    value = inp["live"] * args.steps / secs
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": secs / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": args.workload, "R": wl.R, "S": wl.S, "live": wl.live, "H": wl.H,
                   "w_fmt": ["bf16", "mxfp4"][inp["w_fmt"]]},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": 1, "kind": "oracle", "sample": desc,
                         "host": host_cpu()},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.barrier()


def run_gpu_dcp(args):
    """One step = the DCP pack for one destination rank + the combine on it."""
    import torch

    import mla_decode_attention_lse_gb300 as m
    from mla_decode_attention_lse_gb300 import synth

    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    dist = init_dist(ws, "nccl") if ws > 1 else None
    dev = torch.device("cuda", local)
    m.load_library()
    wl = synth.DCP_WORKLOADS[args.workload]
    seed0 = wl.seed + rank
    inp = synth.make_dcp(wl, device=dev, seed=seed0)
    R, S, H, q, dst, live = inp["R"], inp["S"], inp["H"], inp["q"], inp["dst"], inp["live"]

    def with_bufs(c):
        c["cmb_o"] = torch.empty(R, S, H, 512, dtype=torch.bfloat16, device=dev)
        c["cmb_lse"] = torch.empty(R, S, H, dtype=torch.float32, device=dev)
        c["out"] = torch.empty(S, H * 128, dtype=torch.bfloat16, device=dev)
        return c

    def pack(c, stream=None):
        m.mla_dcp_pack(c["o_all"], c["lse_all"], c["seq_lens"], c["qsl"], q, dst, c["cmb_o"], c["cmb_lse"],
                       stream=stream)

    def combine(c, stream=None):
        m.mla_combine_uv(c["cmb_o"], c["cmb_lse"], q, R, c["w_v"], c["w_fmt"], c["gate"], c["out"],
                         w_scale=c["w_scale"], stream=stream, kernel=args.kernel, tile_tokens=args.tile)

    inp = with_bufs(inp)
    pack(inp)
    torch.cuda.synchronize()
    cinp = dict(o=inp["cmb_o"], lse=inp["cmb_lse"], q=q, spr=R, w_v=inp["w_v"], w_scale=inp["w_scale"],
                w_fmt=inp["w_fmt"], gate=inp["gate"], S=S, S_out=S, H=H, P=R)
    comb_bytes = synth.algorithmic_bytes(cinp)
    pack_bytes = synth.dcp_pack_bytes(inp)
    nbytes = pack_bytes + comb_bytes
    rotate = args.rotate or max(1, -(-L2_DEFEAT_BYTES // nbytes))
    copies = [inp] + [with_bufs(synth.make_dcp(wl, device=dev, seed=seed0 + 1000 * k)) for k in range(1, rotate)]
    a = m.make_args(inp["cmb_o"], inp["cmb_lse"], q, R, inp["w_v"], inp["w_fmt"], inp["gate"], inp["out"],
                    inp["w_scale"], kernel=args.kernel, tile_tokens=args.tile)
    plan = m.mla_combine_uv_plan(a)
    kname = {m.MLA_KERNEL_TC: "tc", m.MLA_KERNEL_KSPLIT: "tc_ksplit_cluster4"}.get(plan["kernel"], "simt")
    stream = torch.cuda.current_stream(dev)
    for k in range(max(3, args.warmup)):
        c = copies[k % rotate]
        pack(c)
        combine(c)
    torch.cuda.synchronize()
    assert m.mla_combine_uv_status(stream) == m.MLA_OK

    def graph_of(fn):
        g = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream(dev)
        with torch.cuda.graph(g, stream=cap):
            for k in range(args.steps):
                fn(copies[k % rotate])
        g.replay()
        torch.cuda.synchronize()
        return g

    def timed(g, clk=None):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        g.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1)

    g_step = graph_of(lambda c: (pack(c), combine(c)))
    g_pack = graph_of(pack)
    g_comb = graph_of(combine)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        t_wall0 = time.perf_counter()
        total_ms = timed(g_step)
        t_wall = time.perf_counter() - t_wall0
    clocks = clk.summary()
    pack_ms = timed(g_pack) / args.steps
    comb_ms = timed(g_comb) / args.steps
    cold_us = cold_launch_us(lambda: (pack(copies[0]), combine(copies[0])), stream, dev)
    assert m.mla_combine_uv_status(stream) == m.MLA_OK
    total_ms = reduce_max(total_ms, dist, dev)
    value = replica_rate(live, args.steps, ws, total_ms)
    peak, peak_kind = load_peaks()
    kern = {"dcp_pack": (pack_ms, pack_bytes), kname: (comb_ms, comb_bytes)}
    dom = max(kern, key=lambda k: kern[k][0])
    achieved = kern[dom][1] / (kern[dom][0] / 1e3) / 1e9

    # end to end: every input the step's calls take, pinned on the host -> device
    pin = {}
    for k in ("o_all", "lse_all", "seq_lens", "qsl", "gate"):
        t = torch.empty(inp[k].shape, dtype=inp[k].dtype, pin_memory=True)
        t.copy_(inp[k])
        pin[k] = t
    out_host = torch.empty(inp["out"].shape, dtype=torch.bfloat16, pin_memory=True)
    dbuf = with_bufs({k: torch.empty_like(inp[k]) for k in pin})
    dbuf.update(w_v=inp["w_v"], w_scale=inp["w_scale"], w_fmt=inp["w_fmt"])
    e2e_steps = max(3, min(args.steps, 20))

    def e2e_step():
        for k in pin:
            dbuf[k].copy_(pin[k], non_blocking=True)
        pack(dbuf, stream=stream)
        combine(dbuf, stream=stream)
        out_host.copy_(dbuf["out"], non_blocking=True)

    e2e_step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_value = replica_rate(live, e2e_steps, ws, reduce_max(e0.elapsed_time(e1), dist, dev))
    h2d = sum(t.numel() * t.element_size() for t in pin.values())
    d2h = out_host.numel() * out_host.element_size()

    line = None
    if rank == 0:
        cpu = None
        if not args.no_cpu_baseline and ws == 1:
            host = {k: (v.cpu() if hasattr(v, "cpu") else v) for k, v in inp.items()}
            rate, desc = dcp_oracle_rate(host, args.cpu_budget)
            cpu = {"value": rate, "unit": "tokens/s", "cores": 1, "kind": "oracle", "sample": desc,
                   "host": host_cpu()}
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": total_ms / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "mxfp4" if inp["w_fmt"] else "bf16",
            "data": "synthetic",
            "config": {"workload": f"{args.workload}: decode context parallelism over {R} ranks x {H} heads "
                                   f"({R * H} global), S={S} rows ({live} live by qsl), q={q}; one step = "
                                   f"the pack for rank {dst} + the combine on it, "
                                   f"{'MXFP4' if inp['w_fmt'] else 'bf16'} W_V",
                       "R": R, "S": S, "live": live, "H": H, "w_fmt": ["bf16", "mxfp4"][inp["w_fmt"]],
                       "parallelism": f"replicas x{ws}", "kernel": f"dcp_pack + {kname}",
                       "grid_combine": plan["grid"],
                       "l2": f"{rotate} independent input copies cycled, one per step: every step reads HBM",
                       "timing": "CUDA graphs of the timed steps (step, pack alone, combine alone), "
                                 "per-step time = replay / steps"},
            "achieved_gbs": achieved,
            "roofline": {"bound": "hbm", "kernel": dom, "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "peak_source": peak_kind,
                         "traffic": traffic_from_profile(args.workload, dom),
                         "algorithmic_bytes": kern[dom][1], "nominal": nominal_hbm(achieved)},
            "kernels": {k: {"us_per_launch": v[0] * 1e3, "algorithmic_bytes": v[1],
                            "gbs": v[1] / (v[0] / 1e3) / 1e9} for k, v in kern.items()},
            "tensor": {"tflops": 2 * S * H * 128 * 512 / (comb_ms / 1e3) / 1e12},
            "kernel_ms": {"mean": total_ms / args.steps},
            "cold_step_us": cold_us,
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "steps": e2e_steps},
            "gpu_launches": 2 * args.steps,
            "clocks": clocks,
            "wall_s": t_wall,
        }
        print(json.dumps(line), flush=True)
    if dist:
        dist.barrier()
        dist.destroy_process_group()
    return line


def attn_oracle_rate(host, budget_s: float):
    """The oracle's attention step on the host: the attention of whole
    requests (random order) until the budget is spent, scaled to the step's
    cached rows, plus the combine on a bounded sample of (t, h) rows.
    Returns (tokens/s, description)."""
    import numpy as np

    import oracle

    import torch

    def u16(t):
        return t.contiguous().view(torch.int16).numpy().view(np.uint16)

    B, q, H, spr = host["B"], host["q"], host["H"], host["spr"]
    lens = host["kv_len"].numpy().astype(np.int64)
    rng = np.random.default_rng(0)
    order = rng.permutation(B)
    done_rows, spent, reqs = 0, 0.0, 0
    for b in order:
        qv = u16(host["qv"][b * q:(b + 1) * q])
        kv = u16(host["kv"][b:b + 1, :max(int(lens[b]), 1)])
        t0 = time.perf_counter()
        o_r, l_r = oracle.mla_attn_split(qv, kv, lens[b:b + 1].astype(np.int32), q, spr, host["scale"])
        spent += time.perf_counter() - t0
        done_rows += max(int(lens[b]), 1)
        reqs += 1
        if spent > budget_s / 2:
            break
    attn_s = spent * lens.clip(min=1).sum() / done_rows
    # the combine of the partials, on sampled rows (the last request's partials stand in)
    pr = oracle.Problem(o_r, l_r, q, spr, u16(host["w_v"]), None, 0, u16(host["gate"][:q]))
    n = 8
    t0 = time.perf_counter()
    pr.rows(rng.integers(0, q, n), rng.integers(0, H, n))
    per_row = (time.perf_counter() - t0) / n
    step_s = attn_s + per_row * B * q * H
    desc = (f"attention of {reqs} whole requests ({done_rows} cached rows, {spent:.2f} s) scaled to the step's "
            f"{int(lens.clip(min=1).sum())} rows, + combine timed on {n} (t, h) rows and scaled to {B * q * H}; "
            "single-threaded oracle")
    return B * q / step_s, desc


def run_reference_attn(args):
    """The oracle's attention -> combine step on the host cores (bounded samples)."""
    import torch

    ws, rank, _ = dist_env()
    if ws > 1:
        dist = init_dist(ws, "gloo")
        if rank != 0:
            dist.barrier()
            return
    from mla_decode_attention_lse_gb300 import synth

    wl = synth.ATTN_WORKLOADS[args.workload]
    inp = synth.make_attn(wl, device="cpu")
    budget = args.ref_budget / max(1, args.steps + args.warmup)
    for _ in range(args.warmup):
        attn_oracle_rate(inp, budget)
    secs, desc = 0.0, ""
    S = wl.B * wl.q
    for _ in range(args.steps):
        rate, desc = attn_oracle_rate(inp, budget)
        secs += S / rate
    value = S * args.steps / secs
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": secs / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": args.workload, "B": wl.B, "q": wl.q, "H": wl.H, "spr": wl.spr, "Lmax": wl.Lmax},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": 1, "kind": "oracle", "sample": desc,
                         "host": host_cpu()},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.barrier()


def run_gpu_attn(args):
    """One step = the split-KV attention (partial producer) + the combine of
    its partials (P = splits, compact)."""
    import torch

    import mla_decode_attention_lse_gb300 as m
    from mla_decode_attention_lse_gb300 import synth

    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    dist = init_dist(ws, "nccl") if ws > 1 else None
    dev = torch.device("cuda", local)
    m.load_library()
    wl = synth.ATTN_WORKLOADS[args.workload]
    seed0 = wl.seed + rank
    B, q, H, spr = wl.B, wl.q, wl.H, wl.spr
    S = B * q

    n_out = OPROJ_N_OUT

    def with_bufs(c, seed=0):
        c["o"] = torch.empty(spr, S, H, 512, dtype=torch.bfloat16, device=dev)
        c["lse"] = torch.empty(spr, S, H, dtype=torch.float32, device=dev)
        c["out"] = torch.empty(S, H * 128, dtype=torch.bfloat16, device=dev)
        c["ws"] = torch.zeros(m.mla_attn_combine_uv_workspace_words(B, q), dtype=torch.int32, device=dev)
        # the o_proj shard's weight (another layer's weight per copy) and output
        g = torch.Generator(device=dev)
        g.manual_seed(7919 + seed)
        c["w_o"] = (torch.randn((n_out, H * 128), generator=g, device=dev) / (H * 128) ** 0.5).to(torch.bfloat16)
        c["y"] = torch.empty(S, n_out, dtype=torch.bfloat16, device=dev)
        return c

    def fused(c, stream=None):  # the same step in one launch
        m.mla_attn_combine_uv(c["qv"], c["kv"], c["kv_len"], q, spr, c["scale"], c["o"], c["lse"], c["w_v"],
                              c["gate"], c["out"], c["ws"], stream=stream)

    def fused_op(c, stream=None):  # the same step and the o_proj shard, in one launch
        m.mla_attn_combine_uv(c["qv"], c["kv"], c["kv_len"], q, spr, c["scale"], c["o"], c["lse"], c["w_v"],
                              c["gate"], c["out"], c["ws"], stream=stream, w_o=c["w_o"], y=c["y"])

    def oproj(c, stream=None):
        m.mla_o_proj(c["out"], c["w_o"], c["y"], stream=stream)

    def attn(c, stream=None):
        m.mla_attn_split_kv(c["qv"], c["kv"], c["kv_len"], q, spr, c["scale"], c["o"], c["lse"], stream=stream)

    def combine(c, stream=None):
        m.mla_combine_uv(c["o"], c["lse"], q, spr, c["w_v"], c["w_fmt"], c["gate"], c["out"],
                         w_scale=c["w_scale"], stream=stream, kernel=args.kernel, tile_tokens=args.tile)

    inp = with_bufs(synth.make_attn(wl, device=dev, seed=seed0))
    attn(inp)
    torch.cuda.synchronize()
    attn_b = synth.attn_bytes(inp)
    cinp = dict(o=inp["o"], lse=inp["lse"], q=q, spr=spr, w_v=inp["w_v"], w_scale=None, w_fmt=0,
                gate=inp["gate"], S=S, S_out=S, H=H, P=spr)
    comb_b = synth.algorithmic_bytes(cinp)
    rotate = args.rotate or max(1, -(-L2_DEFEAT_BYTES // (attn_b + comb_b)))
    copies = [inp] + [with_bufs(synth.make_attn(wl, device=dev, seed=seed0 + 1000 * k), k) for k in range(1, rotate)]
    a = m.make_args(inp["o"], inp["lse"], q, spr, inp["w_v"], 0, inp["gate"], inp["out"], None,
                    kernel=args.kernel, tile_tokens=args.tile)
    plan = m.mla_combine_uv_plan(a)
    kname = {m.MLA_KERNEL_TC: "tc", m.MLA_KERNEL_KSPLIT: "tc_ksplit_cluster4"}.get(plan["kernel"], "simt")
    stream = torch.cuda.current_stream(dev)
    for k in range(max(3, args.warmup)):
        c = copies[k % rotate]
        attn(c)
        combine(c)
    torch.cuda.synchronize()
    assert m.mla_combine_uv_status(stream) == m.MLA_OK

    def graph_of(fn):
        g = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream(dev)
        with torch.cuda.graph(g, stream=cap):
            for k in range(args.steps):
                fn(copies[k % rotate])
        g.replay()
        torch.cuda.synchronize()
        return g

    def timed(g):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        g.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1)

    for k in range(max(3, args.warmup)):
        fused(copies[k % rotate])
        fused_op(copies[k % rotate])
        oproj(copies[k % rotate])
    torch.cuda.synchronize()
    assert m.mla_combine_uv_status(stream) == m.MLA_OK
    g_step = graph_of(fused)
    g_step_op = graph_of(fused_op)
    g_step_then_op = graph_of(lambda c: (fused(c), oproj(c)))
    g_two = graph_of(lambda c: (attn(c), combine(c)))
    g_attn = graph_of(attn)
    g_comb = graph_of(combine)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        t_wall0 = time.perf_counter()
        total_ms = timed(g_step)
        t_wall = time.perf_counter() - t_wall0
    clocks = clk.summary()
    two_ms = timed(g_two) / args.steps
    attn_ms = timed(g_attn) / args.steps
    comb_ms = timed(g_comb) / args.steps
    step_op_ms = timed(g_step_op) / args.steps
    step_then_op_ms = timed(g_step_then_op) / args.steps
    cold_us = cold_launch_us(lambda: fused(copies[0]), stream, dev)
    assert m.mla_combine_uv_status(stream) == m.MLA_OK
    total_ms = reduce_max(total_ms, dist, dev)
    value = replica_rate(S, args.steps, ws, total_ms)
    peak, peak_kind = load_peaks()
    # the fused step moves the attention's bytes (its partials written once)
    # and the combine's W_V, gate and output; its partials are read back
    # within the launch
    fused_b = attn_b + inp["w_v"].numel() * 2 + 2 * S * H * 128 * 2
    kern = {"attn_combine_uv_fused": (total_ms / args.steps, fused_b), "attn_split_kv": (attn_ms, attn_b),
            kname: (comb_ms, comb_b)}
    dom = "attn_combine_uv_fused"
    achieved = kern[dom][1] / (kern[dom][0] / 1e3) / 1e9
    rows = int(inp["kv_len"].long().sum())
    attn_flops = 2.0 * 2 * rows * q * H * 576  # QK^T (576) and PV (512 of it), per visible row and query row

    # end to end: the step's inputs pinned on the host -> device, the core back
    pin = {}
    for k in ("qv", "kv", "kv_len", "gate"):
        t = torch.empty(inp[k].shape, dtype=inp[k].dtype, pin_memory=True)
        t.copy_(inp[k])
        pin[k] = t
    out_host = torch.empty(inp["out"].shape, dtype=torch.bfloat16, pin_memory=True)
    dbuf = with_bufs({k: torch.empty_like(inp[k]) for k in pin})
    dbuf.update(w_v=inp["w_v"], w_scale=None, w_fmt=0, scale=inp["scale"])
    e2e_steps = max(3, min(args.steps, 20))

    def e2e_step():
        for k in pin:
            dbuf[k].copy_(pin[k], non_blocking=True)
        fused(dbuf, stream=stream)
        out_host.copy_(dbuf["out"], non_blocking=True)

    e2e_step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_value = replica_rate(S, e2e_steps, ws, reduce_max(e0.elapsed_time(e1), dist, dev))
    h2d = sum(t.numel() * t.element_size() for t in pin.values())
    d2h = out_host.numel() * out_host.element_size()

    line = None
    if rank == 0:
        cpu = None
        if not args.no_cpu_baseline and ws == 1:
            host = {k: (v.cpu() if hasattr(v, "cpu") else v) for k, v in inp.items()}
            rate, desc = attn_oracle_rate(host, args.cpu_budget)
            cpu = {"value": rate, "unit": "tokens/s", "cores": 1, "kind": "oracle", "sample": desc,
                   "host": host_cpu()}
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": total_ms / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": f"{args.workload}: split-KV MLA decode attention of {B} requests x q={q}, "
                                   f"H={H}, {spr} splits per request, up to {wl.Lmax} cached positions "
                                   f"({rows} in all), then the combine of its partials (bf16 W_V), "
                                   "in one launch (mla_attn_combine_uv)",
                       "B": B, "q": q, "H": H, "spr": spr, "Lmax": wl.Lmax, "cached_rows": rows,
                       "parallelism": f"replicas x{ws}", "kernel": "attn_combine_uv_fused",
                       "l2": f"{rotate} independent input copies cycled, one per step: every step reads HBM",
                       "timing": "CUDA graphs of the timed steps (the fused step; for comparison the two-launch "
                                 "step, the attention alone, the combine alone), per-step time = replay / steps"},
            "two_launch_step_us": two_ms * 1e3,
            "with_oproj": {"n_out": n_out, "one_launch_us": step_op_ms * 1e3,
                           "step_then_oproj_us": step_then_op_ms * 1e3,
                           "note": "the decode step followed by this rank's o_proj shard (W_o [n_out, H*128]): "
                                   "in the same launch (mla_attn_combine_uv with w_o), and as the fused step "
                                   "followed by mla_o_proj on the stream"},
            "achieved_gbs": achieved,
            "roofline": {"bound": "hbm", "kernel": dom, "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "peak_source": peak_kind,
                         "traffic": traffic_from_profile(args.workload, dom),
                         "algorithmic_bytes": kern[dom][1], "nominal": nominal_hbm(achieved)},
            "kernels": {k: {"us_per_launch": v[0] * 1e3, "algorithmic_bytes": v[1],
                            "gbs": v[1] / (v[0] / 1e3) / 1e9} for k, v in kern.items()},
            "tensor": {"attn_tflops": attn_flops / (attn_ms / 1e3) / 1e12},
            "kernel_ms": {"mean": total_ms / args.steps},
            "cold_step_us": cold_us,
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "steps": e2e_steps},
            "gpu_launches": args.steps,
            "clocks": clocks,
            "wall_s": t_wall,
        }
        print(json.dumps(line), flush=True)
    if dist:
        dist.barrier()
        dist.destroy_process_group()
    return line


def oproj_oracle_rate(host, budget_s: float):
    """The oracle's o_proj on a bounded sample of token rows (all outputs of
    each), scaled to the call.  Returns (tokens/s, description)."""
    import numpy as np

    import oracle

    import torch

    def u16(t):
        return t.contiguous().view(torch.int16).numpy().view(np.uint16)

    x, w = u16(host["x"]), u16(host["w"])
    n, spent = 0, 0.0
    while spent < budget_s and n < host["S"]:
        t0 = time.perf_counter()
        oracle.o_proj(x[n:n + 1].copy(), w)
        spent += time.perf_counter() - t0
        n += 1
    return n / spent, f"{n} token rows x {host['Nout']} outputs x K={host['K']}, single-threaded oracle"


def run_reference_oproj(args):
    """The oracle's o_proj shard on the host cores (bounded sample)."""
    import torch

    ws, rank, _ = dist_env()
    if ws > 1:
        dist = init_dist(ws, "gloo")
        if rank != 0:
            dist.barrier()
            return
    from mla_decode_attention_lse_gb300 import synth

    wl = synth.OPROJ_WORKLOADS[args.workload]
    inp = synth.make_oproj(wl, device="cpu")
    budget = args.ref_budget / max(1, args.steps + args.warmup)
    for _ in range(args.warmup):
        oproj_oracle_rate(inp, budget)
    secs, desc = 0.0, ""
    for _ in range(args.steps):
        rate, desc = oproj_oracle_rate(inp, budget)
        secs += wl.S / rate
    value = wl.S * args.steps / secs
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": secs / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": args.workload, "S": wl.S, "K": wl.K, "Nout": wl.Nout},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": 1, "kind": "oracle", "sample": desc,
                         "host": host_cpu()},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.barrier()


def run_gpu_oproj(args):
    """One step = this rank's o_proj shard on the decode step's core rows."""
    import torch

    import mla_decode_attention_lse_gb300 as m
    from mla_decode_attention_lse_gb300 import synth

    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    dist = init_dist(ws, "nccl") if ws > 1 else None
    dev = torch.device("cuda", local)
    m.load_library()
    wl = synth.OPROJ_WORKLOADS[args.workload]
    seed0 = wl.seed + rank

    def with_out(c):
        c["out"] = torch.empty(wl.S, wl.Nout, dtype=torch.bfloat16, device=dev)
        return c

    def call(c, stream=None):
        m.mla_o_proj(c["x"], c["w"], c["out"], stream=stream)

    inp = with_out(synth.make_oproj(wl, device=dev, seed=seed0))
    nbytes = synth.oproj_bytes(inp)
    rotate = args.rotate or max(1, -(-L2_DEFEAT_BYTES // nbytes))
    copies = [inp] + [with_out(synth.make_oproj(wl, device=dev, seed=seed0 + 1000 * k)) for k in range(1, rotate)]
    stream = torch.cuda.current_stream(dev)
    for k in range(max(3, args.warmup)):
        call(copies[k % rotate])
    torch.cuda.synchronize()
    assert m.mla_combine_uv_status(stream) == m.MLA_OK
    g = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream(dev)
    with torch.cuda.graph(g, stream=cap):
        for k in range(args.steps):
            call(copies[k % rotate])
    g.replay()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        t_wall0 = time.perf_counter()
        e0.record(stream)
        g.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        t_wall = time.perf_counter() - t_wall0
    clocks = clk.summary()
    total_ms = reduce_max(e0.elapsed_time(e1), dist, dev)
    cold_us = cold_launch_us(lambda: call(copies[0]), stream, dev)
    assert m.mla_combine_uv_status(stream) == m.MLA_OK
    ms = total_ms / args.steps
    value = replica_rate(wl.S, args.steps, ws, total_ms)
    peak, peak_kind = load_peaks()
    achieved = nbytes / (ms / 1e3) / 1e9
    # end to end: the core rows from pinned host memory, the output back (the
    # weight stays resident, as a model's would)
    x_host = torch.empty(inp["x"].shape, dtype=torch.bfloat16, pin_memory=True)
    x_host.copy_(inp["x"])
    out_host = torch.empty(inp["out"].shape, dtype=torch.bfloat16, pin_memory=True)
    dbuf = with_out({"x": torch.empty_like(inp["x"]), "w": inp["w"]})
    e2e_steps = max(3, min(args.steps, 50))

    def e2e_step():
        dbuf["x"].copy_(x_host, non_blocking=True)
        call(dbuf, stream=stream)
        out_host.copy_(dbuf["out"], non_blocking=True)

    e2e_step()
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_value = replica_rate(wl.S, e2e_steps, ws, reduce_max(e0.elapsed_time(e1), dist, dev))
    line = None
    if rank == 0:
        cpu = None
        if not args.no_cpu_baseline and ws == 1:
            host = {k: (v.cpu() if hasattr(v, "cpu") else v) for k, v in inp.items()}
            rate, desc = oproj_oracle_rate(host, args.cpu_budget)
            cpu = {"value": rate, "unit": "tokens/s", "cores": 1, "kind": "oracle", "sample": desc,
                   "host": host_cpu()}
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": f"{args.workload}: this rank's o_proj shard, {wl.S} tokens x K={wl.K} "
                                   f"(core rows) times the weight slice [{wl.Nout}, {wl.K}]",
                       "S": wl.S, "K": wl.K, "Nout": wl.Nout, "parallelism": f"replicas x{ws}",
                       "kernel": "o_proj",
                       "l2": f"{rotate} independent input copies cycled, one per launch: every launch reads HBM",
                       "timing": "CUDA graph of the timed launches, per-launch time = replay / steps"},
            "achieved_gbs": achieved,
            "roofline": {"bound": "hbm", "kernel": "o_proj", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "peak_source": peak_kind,
                         "traffic": traffic_from_profile(args.workload, "o_proj"), "algorithmic_bytes": nbytes,
                         "nominal": nominal_hbm(achieved)},
            "tensor": {"tflops": 2.0 * wl.S * wl.K * wl.Nout / (ms / 1e3) / 1e12},
            "kernel_ms": {"mean": ms},
            "cold_launch_us": cold_us,
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_value, "unit": "tokens/s",
                    "h2d_bytes_per_step": x_host.numel() * 2, "d2h_bytes_per_step": out_host.numel() * 2,
                    "steps": e2e_steps},
            "gpu_launches": args.steps,
            "clocks": clocks,
            "wall_s": t_wall,
        }
        print(json.dumps(line), flush=True)
    if dist:
        dist.barrier()
        dist.destroy_process_group()
    return line


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of oracle work")
    ap.add_argument("--ref-budget", type=float, default=120.0,
                    help="seconds of oracle work for the whole --impl reference run")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--kernel", type=int, default=0, help="0 auto, 1 CUDA cores, 2 tensor cores (persistent), "
                    "3 tensor cores with the latents split over a 4-CTA cluster")
    ap.add_argument("--tile", type=int, default=0, help="tensor-core token tile (8/16/32; 0 auto)")
    ap.add_argument("--rotate", type=int, default=0,
                    help="independent input copies cycled per step (0: enough to exceed L2)")
    ap.add_argument("--graph", action=argparse.BooleanOptionalAction, default=None,
                    help="capture the timed steps in a CUDA graph (default: for workloads under L2 size)")
    ap.add_argument("--no-decode", action="store_true",
                    help="skip the decode-size leg of the default line")
    ap.add_argument("--decode-launches", type=int, default=1000,
                    help="launches per CUDA graph in the decode-size leg")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    from mla_decode_attention_lse_gb300 import synth

    if args.workload in synth.OPROJ_WORKLOADS:
        run_reference_oproj(args) if args.impl == "reference" else run_gpu_oproj(args)
        return
    if args.workload in synth.ATTN_WORKLOADS:
        run_reference_attn(args) if args.impl == "reference" else run_gpu_attn(args)
        return
    dcp = args.workload in synth.DCP_WORKLOADS
    if args.impl == "reference":
        run_reference_dcp(args) if dcp else run_reference(args)
    else:
        run_gpu_dcp(args) if dcp else run_gpu(args)


if __name__ == "__main__":
    main()
