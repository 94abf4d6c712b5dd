"""Throughput of the fused residual-add + RMSNorm forward (bf16) at
n_rows = 4096, hidden = 4096 on GB300, through the C ABI of libdradd.

One step = one add_rmsnorm_fwd call over one 4096 x 4096 batch (x and
residual read, residual_out and out written: 8 bytes per element plus the
weight once).  Inputs follow the chained-depth workload's distributions
(x ~ N(0, 0.05), residual ~ N(0, 1), weight ~ N(1, 0.1)).  Timed steps run
back to back over 4 rotating buffer sets (512 MiB, four times the L2), so
every step streams from HBM.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line.  Under torchrun (N > 1) each rank runs the same
per-GPU workload on its own GPU (rows are independent: no collective on the
data path), and rank 0 reports the whole-job rate over the slowest rank.
`--impl reference` times the CPU oracle instead (rank 0 only).
"""
from __future__ import annotations

import argparse
import json
import os
import re
import statistics
import subprocess
import sys
import time
from pathlib import Path

import torch

ROOT = Path(__file__).resolve().parent
sys.path.insert(0, str(ROOT))

import deterministic_residual_add_gb300 as dr  # noqa: E402
from deterministic_residual_add_gb300 import inputs  # noqa: E402

METRIC = "add+RMSNorm GB/s and % of HBM peak at 4096×4096 bf16; bit-exact vs oracle"
N_ROWS, HIDDEN = 4096, 4096
N_SETS = 4
KERNEL_SOURCES = ["csrc/dradd_kernels.cu", "csrc/dradd_device.cuh"]
TRAFFIC_FILE = ROOT / "profiles" / "add_rmsnorm_fwd_4096x4096_ncu.md"


def algorithmic_bytes(n_rows: int, hidden: int) -> int:
    """x, residual read + residual_out, out written (2 bytes each) + weight."""
    return 8 * n_rows * hidden + 2 * hidden


def measured_peaks() -> dict:
    p = ROOT / "MEASURED_PEAKS.json"
    if p.exists():
        return json.loads(p.read_text())
    return {}


def kernel_source_hash() -> str:
    import hashlib
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        h.update((ROOT / "deterministic_residual_add_gb300" / rel).read_bytes())
    return h.hexdigest()[:16]


def recorded_traffic():
    """dram bytes per launch from the committed ncu summary, if it was taken
    on the current kernel source."""
    if not TRAFFIC_FILE.exists():
        return None
    text = TRAFFIC_FILE.read_text()
    m_src = re.search(r"kernel_source_sha256_16:\s*([0-9a-f]{16})", text)
    m_b = re.search(r"dram_bytes_per_launch:\s*([0-9]+)", text)
    if not m_src or not m_b or m_src.group(1) != kernel_source_hash():
        return None
    return int(m_b.group(1))


# ------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.lines = []
        try:
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            gid = uuid if uuid.startswith("GPU-") else f"GPU-{uuid}"
        except Exception:  # noqa: BLE001
            gid = str(device_index)
        self.cmd = ["nvidia-smi", "-i", gid, f"--query-gpu={self.FIELDS}",
                    "--format=csv,noheader,nounits", "-lms", "200"]

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(self.cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except (OSError, ValueError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self) -> dict:
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for name, val in zip(names, parts[4:8]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------- distributed
def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as tdist
        torch.cuda.set_device(local)
        tdist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(local)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as tdist
        tdist.barrier()


def max_over_ranks(v: float, world: int) -> float:
    if world == 1:
        return v
    import torch.distributed as tdist
    t = torch.tensor([v], dtype=torch.float64, device="cuda")
    tdist.all_reduce(t, op=tdist.ReduceOp.MAX)
    return float(t.item())


# -------------------------------------------------------------- our kernel
class RawCall:
    """Precomputed C-ABI call: add_rmsnorm_fwd(out, ro, x, r, w, eps, n, h, stream)."""

    def __init__(self, sets, w, stream):
        import ctypes
        self.fn = dr.lib().add_rmsnorm_fwd
        self.args = [(s["out"].data_ptr(), s["ro"].data_ptr(), s["x"].data_ptr(), s["r"].data_ptr(),
                      w.data_ptr(), ctypes.c_float(inputs.EPS), N_ROWS, HIDDEN, stream.cuda_stream)
                     for s in sets]

    def __call__(self, i: int):
        st = self.fn(*self.args[i % len(self.args)])
        if st != 0:
            raise dr.DraddError(st, "add_rmsnorm_fwd")


def make_sets(device):
    """N_SETS independent (x, residual, out, residual_out) buffers: x_k from
    the chained workload's generator k, residual_0 in every set."""
    ch = inputs.CHAIN4096
    r0, w = ch.initial()
    sets = []
    for k in range(N_SETS):
        x = ch.delta(k).to(device)
        sets.append({"x": x, "r": r0.to(device), "out": torch.empty_like(x),
                     "ro": torch.empty_like(x)})
    return sets, w.to(device), r0


GRAPH_CHUNK = 256  # launches per captured graph (a multiple of N_SETS)


def time_device(call, steps, warmup, stream, world, use_graph):
    """Exactly `steps` launches back to back on `stream`, timed with CUDA
    events; with use_graph the launches are replayed from CUDA graphs of
    GRAPH_CHUNK launches (plus one graph for the remainder)."""
    for i in range(warmup):
        call(i)
    torch.cuda.synchronize()
    plan = []
    if use_graph:
        full, rest = divmod(steps, GRAPH_CHUNK)
        graphs = {}
        for n in {GRAPH_CHUNK if full else 0, rest} - {0}:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for i in range(n):
                    call(i)
            g.replay()  # untimed
            graphs[n] = g
        plan = [graphs[GRAPH_CHUNK]] * full + ([graphs[rest]] if rest else [])
        torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    start.record(stream)
    if use_graph:
        for g in plan:
            g.replay()
    else:
        for i in range(steps):
            call(i)
    end.record(stream)
    end.synchronize()
    torch.cuda.synchronize()
    barrier(world)
    return start.elapsed_time(end)  # ms


def time_e2e(steps, device, stream, w_dev):
    """Public API with host data: per step, copy x and residual (and weight)
    from pinned host memory, run the op, read out and residual_out back."""
    ch = inputs.CHAIN4096
    r0, w = ch.initial()
    x_h = ch.delta(0).pin_memory()
    r_h = r0.pin_memory()
    w_h = w.pin_memory()
    out_h = torch.empty_like(x_h).pin_memory()
    ro_h = torch.empty_like(x_h).pin_memory()
    x_d, r_d, wd = torch.empty_like(x_h, device=device), torch.empty_like(r_h, device=device), \
        torch.empty_like(w_h, device=device)
    out_d, ro_d = torch.empty_like(x_d), torch.empty_like(x_d)

    def step():
        x_d.copy_(x_h, non_blocking=True)
        r_d.copy_(r_h, non_blocking=True)
        wd.copy_(w_h, non_blocking=True)
        dr.add_rmsnorm_fwd(x_d, r_d, wd, inputs.EPS, out=out_d, residual_out=ro_d, stream=stream)
        out_h.copy_(out_d, non_blocking=True)
        ro_h.copy_(ro_d, non_blocking=True)

    with torch.cuda.stream(stream):
        for _ in range(2):
            step()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(steps):
            step()
        stream.synchronize()
        dt = time.perf_counter() - t0
    bi = (x_h.numel() + r_h.numel() + w_h.numel()) * 2
    bo = (out_h.numel() + ro_h.numel()) * 2
    return dt, bi, bo


def cpu_baseline(seconds: float, gpu_sets=None):
    """The CPU oracle (single thread) on leading rows of the same workload,
    for about `seconds`; also checks those rows against the GPU's output."""
    import numpy as np
    import oracle
    o = oracle.lib()
    ch = inputs.CHAIN4096
    r0, w = ch.initial()
    x0 = ch.delta(0)
    chunk = 64
    rows = 0
    t0 = time.perf_counter()
    first = None
    while True:
        lo = rows % N_ROWS
        hi = min(N_ROWS, lo + chunk)
        res = o.add_rmsnorm_fwd(x0[lo:hi], r0[lo:hi], w, inputs.EPS)
        if first is None:
            first = res
        rows += hi - lo
        if time.perf_counter() - t0 >= seconds:
            break
    dt = time.perf_counter() - t0
    out = {"value": algorithmic_bytes(rows, HIDDEN) / dt / 1e9, "unit": "GB/s", "cores": 1,
           "kind": "oracle",
           "sample": f"{rows} rows of the 4096x4096 workload ({rows * HIDDEN} elements) in "
                     f"{dt:.1f} s, single thread",
           "seconds": round(dt, 3)}
    if gpu_sets is not None:
        s = gpu_sets[0]
        got_out = s["out"][:chunk].view(torch.int16).cpu().numpy().view(np.uint16)
        got_ro = s["ro"][:chunk].view(torch.int16).cpu().numpy().view(np.uint16)
        out["parity_rows_checked"] = chunk
        out["parity_bit_exact"] = bool(np.array_equal(got_out, first[0]) and np.array_equal(got_ro, first[1]))
    return out


def run_ours(args):
    world, rank, local = dist_setup()
    device = torch.device("cuda", local)
    dr.lib()
    stream = torch.cuda.Stream(device)
    sets, w_dev, _ = make_sets(device)
    torch.cuda.synchronize()
    call = RawCall(sets, w_dev, stream)
    with torch.cuda.stream(stream):
        sampler = ClockSampler(local)
        with sampler:
            ms = time_device(call, args.steps, args.warmup, stream, world, args.graph)
    ms = max_over_ranks(ms, world)
    bytes_step = algorithmic_bytes(N_ROWS, HIDDEN)
    ms_per_step = ms / args.steps
    value = world * bytes_step * args.steps / (ms / 1e3) / 1e9
    per_launch_gbs = bytes_step / (ms_per_step / 1e3) / 1e9
    peaks = measured_peaks()
    peak = peaks.get("hbm_gbs")
    peak_src = "measured" if peak else "fallback"
    if not peak:
        peak = 6800.0

    e2e_steps = max(3, min(args.steps, args.e2e_steps))
    e2e = None
    if not args.no_e2e:
        dt, bi, bo = time_e2e(e2e_steps, device, stream, w_dev)
        dt = max_over_ranks(dt, world)
        e2e = {"value": world * bytes_step * e2e_steps / dt / 1e9, "unit": "GB/s",
               "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo, "steps": e2e_steps,
               "ms_per_step": dt / e2e_steps * 1e3}

    cfg = dr.resolve_config(N_ROWS, HIDDEN, sm_count=torch.cuda.get_device_properties(device).multi_processor_count)
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 6),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": "add_rmsnorm_fwd 4096x4096 bf16 in/out (chained-depth inputs)",
                   "n_rows": N_ROWS, "hidden": HIDDEN, "io_dtype": "bf16",
                   "l2": f"{N_SETS} rotating buffer sets ({N_SETS * 128} MiB) > L2",
                   "launch": {"variant": "rows" if cfg.variant == 1 else "staged",
                              "threads_per_row": cfg.threads_per_row, "rows_per_cta": cfg.rows_per_cta,
                              "grid_ctas": cfg.grid_ctas},
                   "cuda_graph": bool(args.graph), "parallelism": f"replicas x{world}"},
        "rows_per_s": round(world * N_ROWS * args.steps / (ms / 1e3), 1),
        "roofline": {"bound": "hbm", "achieved": round(per_launch_gbs, 2), "peak": peak,
                     "unit": "GB/s", "frac": round(per_launch_gbs / peak, 4),
                     "peak_source": f"{peak_src} hbm_gbs",
                     "traffic": recorded_traffic(),
                     "algorithmic_bytes_per_launch": bytes_step},
        "gpu_launches": args.steps,
        "e2e": e2e,
    }
    if rank == 0:
        line["clocks"] = sampler.summary()
        if not args.no_cpu:
            line["cpu_baseline"] = cpu_baseline(args.cpu_seconds, sets)
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as tdist
        tdist.destroy_process_group()


def run_reference(args):
    """The oracle on the host, on the same metric, unit and workload: each
    step runs a bounded sample of rows of the 4096 x 4096 batch."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    o = oracle.lib()
    ch = inputs.CHAIN4096
    r0, w = ch.initial()
    x0 = ch.delta(0)
    t0 = time.perf_counter()
    o.add_rmsnorm_fwd(x0[:16], r0[:16], w, inputs.EPS)
    t_row = max(1e-6, (time.perf_counter() - t0) / 16)
    total = args.warmup + args.steps
    rows = int(max(1, min(N_ROWS, args.reference_seconds / total / t_row)))
    for i in range(args.warmup):
        o.add_rmsnorm_fwd(x0[:rows], r0[:rows], w, inputs.EPS)
    t0 = time.perf_counter()
    for i in range(args.steps):
        lo = (i * rows) % (N_ROWS - rows + 1)
        o.add_rmsnorm_fwd(x0[lo:lo + rows], r0[lo:lo + rows], w, inputs.EPS)
    dt = time.perf_counter() - t0
    value = algorithmic_bytes(rows, HIDDEN) * args.steps / dt / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": "add_rmsnorm_fwd 4096x4096 bf16 in/out (chained-depth inputs)",
                   "n_rows": N_ROWS, "hidden": HIDDEN, "io_dtype": "bf16",
                   "rows_per_step": rows},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": f"{rows} rows of 4096 per step, single thread"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--graph", type=int, default=1, help="replay the timed steps as a CUDA graph")
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--reference-seconds", type=float, default=60.0)
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
