"""Write the profile summaries in this folder from ncu reports.

Usage: python profiles/make_summaries.py <dir with prof_tc_<workload>.ncu-rep and launches_mtp_mxfp4.csv>
Reads ncu reports with `ncu -i ... --page raw --csv` (counters only).
"""
import csv
import json
import os
import subprocess
import sys
from collections import defaultdict

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(HERE))
import bench  # noqa: E402  (kernel source hash)


def raw(path):
    out = subprocess.run(["ncu", "-i", path, "--page", "raw", "--csv"], capture_output=True, text=True).stdout
    rows = list(csv.reader(out.splitlines()))
    return dict(zip(rows[0], rows[2])), dict(zip(rows[0], rows[1]))


def to_bytes(v, u):
    return float(v) * {"Gbyte": 1e9, "Mbyte": 1e6, "Kbyte": 1e3, "byte": 1.0}[u]


def main(src):
    h = bench.kernel_source_hash()
    traffic = {}
    for w, fmt in (("mtp_mxfp4", "MXFP4"), ("mtp", "bf16")):
        d, u = raw(os.path.join(src, f"prof_tc_{w}.ncu-rep"))
        rd = to_bytes(d["dram__bytes_read.sum"], u["dram__bytes_read.sum"])
        wr = to_bytes(d["dram__bytes_write.sum"], u["dram__bytes_write.sum"])
        traffic[f"{w}/tc"] = {"source_hash": h, "dram_bytes_per_launch": rd + wr, "dram_read": rd,
                              "dram_write": wr, "capture_duration_us": float(d["gpu__time_duration.sum"])}
        stalls = sorted(((float(v), k) for k, v in d.items()
                         if k.startswith("smsp__average_warps_issue_stalled_") and k.endswith("per_issue_active.ratio")),
                        reverse=True)[:6]
        pipes = sorted(((float(v), k) for k, v in d.items()
                        if k.startswith("sm__inst_executed_pipe_") and k.endswith(".avg.pct_of_peak_sustained_active")),
                       reverse=True)[:4]
        txt = f"""# Fused tensor-core kernel on the large MTP batch, {fmt} W_V

Workload: 1024 requests x q=4 (S=4096), H=96, 4 splits per request (compact `o` [4,4096,96,512] bf16,
lse with 2% -inf), {fmt} W_V, the launch configuration `bench.py` times (automatic plan).
Kernel sources: hash `{h}` (what `bench.py` hashes over `mla_decode_attention_lse_gb300/csrc/`).

Commands (one launch captured, after the same command exited 0 without ncu):

```
python bench.py --steps 3 --warmup 3 --no-cpu-baseline --workload {w}
ncu --set full --clock-control none -k regex:tc_kernel -s 3 -c 1 -o prof_tc_{w} \\
    python bench.py --steps 3 --warmup 3 --no-cpu-baseline --workload {w}
python profiles/make_summaries.py <folder with the reports>
```

| metric | value |
|---|---|
| gpu__time_duration.sum (one launch, under ncu) | {float(d['gpu__time_duration.sum']):.1f} us |
| dram__bytes_read.sum | {rd / 1e9:.4f} GB |
| dram__bytes_write.sum | {wr / 1e6:.1f} MB |
| DRAM throughput (% of ncu's peak) | {float(d['gpu__dram_throughput.avg.pct_of_peak_sustained_elapsed']):.1f} % |
| smsp__inst_executed.sum | {float(d['smsp__inst_executed.sum']) / 1e6:.1f} M |
| issue active (% of active cycles) | {float(d['smsp__issue_active.avg.pct_of_peak_sustained_active']):.1f} % |
| tensor pipe active (% of elapsed) | {float(d['sm__pipe_tensor_cycles_active.avg.pct_of_peak_sustained_elapsed']):.2f} % |
| warps active (% of peak) | {float(d['sm__warps_active.avg.pct_of_peak_sustained_active']):.1f} % |
| registers / thread | {d['launch__registers_per_thread']} |
| local-memory (spill) load sectors | {d['l1tex__t_sectors_pipe_lsu_mem_local_op_ld.sum']} |

Busiest pipes (% of active cycles): {', '.join(f"{k.replace('sm__inst_executed_pipe_', '').replace('.avg.pct_of_peak_sustained_active', '')} {v:.1f}" for v, k in pipes)}.
Top warp stall reasons (cycles per issued instruction): {', '.join(f"{k.replace('smsp__average_warps_issue_stalled_', '').replace('_per_issue_active.ratio', '')} {v:.2f}" for v, k in stalls)}.

Reading: DRAM bytes match the algorithmic bytes (partial rows with a live LSE, lse, W_V, gate, core;
the core writes still in L2 at the end of the launch are not counted): no re-reads. The kernel is
bounded by latency and instruction issue (16 warps per SM at 125-128 registers), not by the tensor
pipe, as expected for a 28 flop/byte contraction.
"""
        with open(os.path.join(HERE, f"tc_kernel_{w}.md"), "w") as f:
            f.write(txt)
    with open(os.path.join(HERE, "traffic.json"), "w") as f:
        json.dump(traffic, f, indent=1)

    rows = list(csv.reader(open(os.path.join(src, "launches_mtp_mxfp4.csv"))))
    hi = [i for i, r in enumerate(rows) if "Kernel Name" in r][0]
    hdr, data = rows[hi], rows[hi + 1:]
    ki, mi, vi, ui = (hdr.index(x) for x in ("Kernel Name", "Metric Name", "Metric Value", "Metric Unit"))
    agg = defaultdict(lambda: [0, 0.0])
    for r in data:
        if len(r) <= vi or r[mi] != "gpu__time_duration.sum":
            continue
        v = float(r[vi].replace(",", "")) * {"ns": 1.0, "us": 1e3, "ms": 1e6, "usecond": 1e3, "nsecond": 1.0}[r[ui]]
        agg[r[ki]][0] += 1
        agg[r[ki]][1] += v
    tot = sum(v[1] for v in agg.values())
    ours = [(k, v) for k, v in agg.items() if "tc_kernel" in k]
    out = """# Launch list of `python bench.py --steps 3 --warmup 3 --no-cpu-baseline` (large MTP batch, MXFP4 W_V)

```
ncu --metrics gpu__time_duration.sum --clock-control none --csv --log-file launches_mtp_mxfp4.csv \\
    python bench.py --steps 3 --warmup 3 --no-cpu-baseline
```

Per-launch times under ncu are cold-cache and serialised: compare shares, not absolutes. The run also
generates the inputs (PyTorch RNG and conversion kernels) and runs 3 warm-up, 3 timed and the e2e
launches of our kernel; inside the timed region our kernel is the only kernel (one launch per step).

| kernel | launches | total (us) | share |
|---|---|---|---|
"""
    for k, (n, t) in sorted(agg.items(), key=lambda x: -x[1][1])[:10]:
        out += f"| `{k[:90]}` | {n} | {t / 1e3:.1f} | {100 * t / tot:.1f} % |\n"
    for k, (n, t) in ours:
        out += f"\nOur kernel `{k}`: {n} launches, {t / n / 1e3:.1f} us per launch under ncu.\n"
    with open(os.path.join(HERE, "launches_mtp_mxfp4.md"), "w") as f:
        f.write(out)


if __name__ == "__main__":
    main(sys.argv[1] if len(sys.argv) > 1 else "gpurun_out")
