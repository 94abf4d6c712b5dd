"""Throughput of the fused residual-add + RMSNorm forward on GB300, through
the C ABI of libdradd.

Default workload: add_rmsnorm_fwd at n_rows = 4096, hidden = 4096, bf16 in
and out.  One step = one call over one 4096 x 4096 batch (x and residual
read, residual_out and out written: 8 bytes per element, plus the weight
once).  Inputs follow the chained-depth workload's distributions (x ~
N(0, 0.05), residual ~ N(0, 1), weight ~ N(1, 0.1)).  Timed steps run back
to back over 8 rotating buffer sets (1 GiB, about eight times the L2), so
every step streams from HBM.  Other workloads (--workload) exist for profiling.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line.  Under torchrun (N > 1) each rank runs the same
per-GPU workload on its own GPU (rows are independent: no collective on the
data path), and rank 0 reports the whole-job rate over the slowest rank.
`--impl reference` times the CPU oracle instead (rank 0 only).
"""
from __future__ import annotations

import argparse
import ctypes
import dataclasses
import hashlib
import json
import os
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
QK_METRIC = "fused q/k RMSNorm GB/s and % of HBM peak; bit-exact vs oracle"
N_SETS = 4
# Bytes the rotating buffer sets of a timed loop hold together: 1 GiB,
# about eight times the 129 MB L2, so a set has left L2 before it comes round.
ROTATION_BYTES = 2**30
PROFILES = ROOT / "profiles"

# name -> (n_rows, hidden, op, input recipe).  The first is the headline
# workload; the others are for profiling and context.  op is one of
# add_rmsnorm, add_rmsnorm_quant, add_rmsnorm_fp8, add_rmsnorm_fp4, rmsnorm,
# rmsnorm_quant, rmsnorm_fp8, residual_add.
WORKLOADS = {
    "4096x4096": (4096, 4096, "add_rmsnorm", "chain4096"),
    "tiny": (64, 1024, "add_rmsnorm", "tiny"),
    "2048x4096": (2048, 4096, "add_rmsnorm", "2048x4096"),
    "4096x8192": (4096, 8192, "add_rmsnorm", "4096x8192"),
    "8192x4096": (8192, 4096, "add_rmsnorm", "8192x4096"),
    "16384x4096": (16384, 4096, "add_rmsnorm", "16384x4096"),
    "2048x16384": (2048, 16384, "add_rmsnorm", "quant2048x16384"),
    "quant2048x16384": (2048, 16384, "add_rmsnorm_quant", "quant2048x16384"),
    "quant4096x4096": (4096, 4096, "add_rmsnorm_quant", "chain4096"),
    "quant4096x8192": (4096, 8192, "add_rmsnorm_quant", "4096x8192"),
    "rmsnorm4096x4096": (4096, 4096, "rmsnorm", "chain4096"),
    "rmsnorm_quant4096x4096": (4096, 4096, "rmsnorm_quant", "chain4096"),
    "rmsnorm_quant2048x8192": (2048, 8192, "rmsnorm_quant", "4096x8192"),
    "rmsnorm_quant16384x1024": (16384, 1024, "rmsnorm_quant", "tiny"),
    "residual_add4096x4096": (4096, 4096, "residual_add", "chain4096"),
    "fp8_2048x16384": (2048, 16384, "add_rmsnorm_fp8", "quant2048x16384"),
    "fp8_4096x4096": (4096, 4096, "add_rmsnorm_fp8", "chain4096"),
    "rmsnorm_fp8_4096x4096": (4096, 4096, "rmsnorm_fp8", "chain4096"),
    "rmsnorm_fp8_2048x8192": (2048, 8192, "rmsnorm_fp8", "4096x8192"),
    "fp4_2048x16384": (2048, 16384, "add_rmsnorm_fp4", "quant2048x16384"),
    "fp4_4096x4096": (4096, 4096, "add_rmsnorm_fp4", "chain4096"),
    # the shapes of the aiter page's "Cost of fixing" table, bf16 and int8 out
    "8192x2048": (8192, 2048, "add_rmsnorm", "8192x2048"),
    "quant2048x4096": (2048, 4096, "add_rmsnorm_quant", "2048x4096"),
    "quant8192x2048": (8192, 2048, "add_rmsnorm_quant", "8192x2048"),
    "quant8192x4096": (8192, 4096, "add_rmsnorm_quant", "8192x4096"),
}


# Launch variants of the main op as config.launch names them (the resolved
# plan; "staged" with rows_per_cta 2 is the two-rows-per-thread kernel).
VARIANT_NAMES = {dr.VARIANT_ROWS: "rows", dr.VARIANT_STAGED: "staged", dr.VARIANT_SPLIT: "split",
                 dr.VARIANT_WARP: "warp"}


def algorithmic_bytes(n_rows: int, hidden: int, op: str = "add_rmsnorm") -> int:
    """Bytes the op must move: bf16 reads of x (and residual), bf16 writes of
    residual_out (add forms) and out (2 bytes) or int8 out (1 byte) plus a
    4-byte scale per row, and the weight once (norm forms)."""
    e = n_rows * hidden
    return int({"add_rmsnorm": 8 * e + 2 * hidden,
            "add_rmsnorm_quant": 7 * e + 4 * n_rows + 2 * hidden,
            "add_rmsnorm_fp8": 7 * e + 4 * n_rows + 2 * hidden,
            "add_rmsnorm_fp4": 6.5 * e + 4 * n_rows + 2 * hidden,
            "rmsnorm": 4 * e + 2 * hidden,
            "rmsnorm_quant": 3 * e + 4 * n_rows + 2 * hidden,
            "rmsnorm_fp8": 3 * e + 4 * n_rows + 2 * hidden,
            "residual_add": 6 * e}[op])


# GB300 HBM3e nominal bandwidth (about 8 TB/s), reported beside the measured
# copy bandwidth that the roofline fraction uses.
NOMINAL_HBM_GBS = 8000.0


def measured_peaks() -> dict:
    p = ROOT / "MEASURED_PEAKS.json"
    return json.loads(p.read_text()) if p.exists() else {}


# ------------------------------------------------------------ ncu records
# DRAM traffic per launch comes from one ncu capture of the workload's own
# bench command (one pass: gpu__time_duration and the two dram byte
# counters), stored as profiles/ncu_<workload>.json by `--ncu-record`.  A
# record is used only while the sources its kernels are built from hash to
# the value it was taken on; otherwise the line's traffic is null.
SOURCE_FAMILIES = {
    "main": ["dradd_device.cuh", "dradd_kernels.cuh", "dradd_internal.h", "dradd_kernels.cu",
             "dradd_staged_*.cu", "dradd_warp.cuh", "dradd_warp_*.cu", "dradd_split.cuh", "dradd_split_*.cu",
             "dradd_abi.cu"],
    "qk": ["dradd_device.cuh", "dradd_kernels.cuh", "dradd_internal.h", "dradd_warp.cuh", "dradd_qk.cuh",
           "dradd_qk_*.cu", "dradd_abi.cu"],
    "elem": ["dradd_device.cuh", "dradd_internal.h", "dradd_lse.cu", "dradd_abi.cu"],
}
NCU_METRICS = "dram__bytes_read.sum,dram__bytes_write.sum,gpu__time_duration.sum"
NCU_KERNELS = ("regex:staged_kernel|staged_pair_kernel|rows_kernel|split_kernel|warp_kernel|qk_kernel|qk_chunk_kernel|"
               "lse_merge_kernel|unary_kernel|residual_add_kernel")
NCU_WARMUP = 5


def workload_family(name: str) -> str:
    if name in inputs.QK_WORKLOADS:
        return "qk"
    if name in inputs.ELEM_WORKLOADS:
        return "elem"
    return "main"


def source_files(family: str):
    csrc = ROOT / "deterministic_residual_add_gb300" / "csrc"
    files = []
    for pat in SOURCE_FAMILIES[family]:
        files += sorted(csrc.glob(pat))
    return files + [ROOT / "include" / "dradd.h"]


def source_hash(family: str) -> str:
    """First 16 hex digits of the SHA-256 over the family's kernel sources
    (names and contents, in a fixed order)."""
    h = hashlib.sha256()
    for f in source_files(family):
        h.update(f.name.encode() + b"\0" + f.read_bytes())
    return h.hexdigest()[:16]


def workload_n_sets(name: str) -> int:
    """Buffer sets the timed loop rotates through for any workload."""
    if name in inputs.QK_WORKLOADS:
        w = inputs.QK_WORKLOADS[name]
        return max(N_SETS, -(-ROTATION_BYTES // qk_algorithmic_bytes(w, w.n_tokens)))
    if name in inputs.ELEM_WORKLOADS:
        return max(N_SETS, -(-ROTATION_BYTES // elem_bytes(inputs.ELEM_WORKLOADS[name])))
    return n_sets_for(name)


def workload_bytes(name: str) -> int:
    if name in inputs.QK_WORKLOADS:
        w = inputs.QK_WORKLOADS[name]
        return qk_algorithmic_bytes(w, w.n_tokens)
    if name in inputs.ELEM_WORKLOADS:
        return elem_bytes(inputs.ELEM_WORKLOADS[name])
    n, h, op, _ = WORKLOADS[name]
    return algorithmic_bytes(n, h, op)


def ncu_plan(name: str):
    """(skip, count, steps): the capture skips the warm-up launches and one
    full rotation of the buffer sets, then takes one full rotation (at least
    4 launches), so each set's outputs are written back once in the window."""
    k = workload_n_sets(name)
    count = max(4, k)
    skip = NCU_WARMUP + k
    return skip, count, k + count + 2


def ncu_capture_command(name: str) -> str:
    """The capture behind profiles/ncu_<name>.json, run from the repository
    root after the same bench command has exited 0 without ncu."""
    skip, count, steps = ncu_plan(name)
    return (f"ncu --metrics {NCU_METRICS} --print-units base --cache-control none --clock-control none "
            f"-k '{NCU_KERNELS}' -s {skip} -c {count} --csv --log-file gpurun_out/ncu_{name}.csv "
            f"python bench.py --workload {name} {ncu_bench_args(name)}")


def ncu_bench_args(name: str) -> str:
    _, _, steps = ncu_plan(name)
    return f"--steps {steps} --warmup {NCU_WARMUP} --graph 0 --no-e2e --no-cpu"


_UNIT = {"byte": 1.0, "kbyte": 1e3, "mbyte": 1e6, "gbyte": 1e9,
         "nsecond": 1.0, "usecond": 1e3, "msecond": 1e6, "second": 1e9}


def parse_ncu_csv(text: str):
    """Launches of an ncu --csv metric log: [{kernel, grid, block, device,
    metrics: {name: value in bytes or ns}}] in capture order."""
    import csv
    import io
    lines = text.splitlines()
    start = next((i for i, ln in enumerate(lines) if ln.startswith('"ID"')), None)
    if start is None:
        raise ValueError("no ncu CSV header in the log")
    launches = {}
    for row in csv.DictReader(io.StringIO("\n".join(lines[start:]))):
        if not row.get("ID") or not row.get("Metric Name"):
            continue
        lid = int(row["ID"])
        rec = launches.setdefault(lid, {"kernel": row.get("Kernel Name", ""), "grid": row.get("Grid Size", ""),
                                        "block": row.get("Block Size", ""), "device": row.get("Device", ""),
                                        "metrics": {}})
        unit = (row.get("Metric Unit") or "").strip().lower()
        val = float(row["Metric Value"].replace(",", ""))
        rec["metrics"][row["Metric Name"]] = val * _UNIT.get(unit, 1.0)
    return [launches[k] for k in sorted(launches)]


def make_ncu_record(name: str, csv_text: str) -> dict:
    launches = parse_ncu_csv(csv_text)
    if not launches:
        raise ValueError("the ncu log holds no launch")
    kernels = sorted({ln["kernel"] for ln in launches})
    if len(kernels) != 1:
        raise ValueError(f"expected one kernel in the capture, found {kernels}")

    def mean(metric):
        return statistics.fmean(ln["metrics"][metric] for ln in launches)
    rd, wr = mean("dram__bytes_read.sum"), mean("dram__bytes_write.sum")
    alg = workload_bytes(name)
    fam = workload_family(name)
    return {
        "workload": name, "kernel": kernels[0], "grid": launches[0]["grid"], "block": launches[0]["block"],
        "launches_captured": len(launches), "rotating_sets": workload_n_sets(name),
        "dram_bytes_read_per_launch": round(rd), "dram_bytes_write_per_launch": round(wr),
        "dram_bytes_per_launch": round(rd) + round(wr),
        "gpu_time_duration_ns_mean": round(mean("gpu__time_duration.sum"), 1),
        "algorithmic_bytes_per_launch": alg, "traffic_over_algorithmic": round((rd + wr) / alg, 4),
        "note": "means over consecutive launches of the back-to-back bench loop, caches not flushed: "
                "outputs left dirty in L2 are written back during later launches; under ncu each launch "
                "is serialised, so the duration is not the bench's",
        "source_family": fam, "source_sha256_16": source_hash(fam),
        "sources": [str(f.relative_to(ROOT)) for f in source_files(fam)],
        "command": ncu_capture_command(name),
    }


def ncu_record_path(name: str) -> Path:
    return PROFILES / f"ncu_{name}.json"


def recorded_traffic(name: str):
    """(DRAM bytes per launch, record file) from profiles/ncu_<name>.json if
    the record was taken on the current sources, else (None, reason)."""
    p = ncu_record_path(name)
    if not p.exists():
        return None, "no ncu record"
    rec = json.loads(p.read_text())
    if rec.get("source_sha256_16") != source_hash(workload_family(name)):
        return None, f"{p.name} was taken on other sources"
    return int(rec["dram_bytes_per_launch"]), p.name


L2_BYTES = 129 * 10**6


def l2_desc(n_sets: int, bytes_step: int) -> str:
    """config.l2: how the timed loop keeps its inputs out of L2."""
    total = n_sets * bytes_step
    where = ("more than L2 (129 MB): every step streams from HBM; roofline.traffic_over_algorithmic "
             "gives the share of DRAM bytes measured" if total > L2_BYTES
             else "fits in L2 (129 MB): a latency-bound size, not an HBM figure")
    return f"{n_sets} rotating buffer sets ({total // 2**20} MiB), {where}"


def traffic_fields(name: str, ms_per_step: float, peak: float) -> dict:
    """roofline.traffic and what it says: the measured DRAM bytes over the
    algorithmic bytes, and the DRAM-only fraction (traffic / time / peak)."""
    traffic, src = recorded_traffic(name)
    out = {"traffic": traffic, "traffic_source": src}
    if traffic is not None:
        out["traffic_over_algorithmic"] = round(traffic / workload_bytes(name), 4)
        out["frac_dram"] = round(traffic / (ms_per_step / 1e3) / 1e9 / peak, 4)
    return out


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi clock and throttle-reason samples every 200 ms."""
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
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as tdist
        tdist.init_process_group("nccl", device_id=torch.device("cuda", local))
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as tdist
        tdist.barrier()


def max_over_ranks(v: float, world: int) -> float:
    """The largest of every rank's value (the slowest rank's time)."""
    if world == 1:
        return v
    import torch.distributed as tdist
    device = "cuda" if tdist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=device)
    tdist.all_reduce(t, op=tdist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------- workload
IO_DESC = {"add_rmsnorm": "bf16 in/out", "add_rmsnorm_quant": "bf16 in, int8 + fp32 scale + bf16 residual_out out",
           "rmsnorm": "bf16 in/out", "rmsnorm_quant": "bf16 in, int8 + fp32 scale out",
           "residual_add": "bf16 in/out",
           "add_rmsnorm_fp8": "bf16 in, e4m3 + fp32 scale + bf16 residual_out out",
           "rmsnorm_fp8": "bf16 in, e4m3 + fp32 scale out",
           "add_rmsnorm_fp4": "bf16 in, packed e2m1 + fp32 scale + bf16 residual_out out"}


def workload_desc(name: str) -> str:
    """config.workload of a main-op workload (the same on both arms)."""
    n, h, op, _ = WORKLOADS[name]
    return f"{op}_fwd {n}x{h} {IO_DESC[op]}"


def qk_workload_desc(w) -> str:
    qdesc = (f"q {w.q_heads}x{w.q_head}" + (" + residual" if w.residual else "") +
             (f" -> e4m3 groups of {w.group_size}" if w.group_size else " -> bf16"))
    return f"fused_qk_rmsnorm_group_quant_fwd {w.n_tokens} tokens: {qdesc}; k {w.k_heads}x{w.k_head} -> bf16"


def elem_workload_desc(w) -> str:
    if w.kind == "merge":
        return (f"lse_merge_2d_fwd: [{w.rows} x {w.cols}] running fp32 lse, last {w.step_cols} columns of each "
                f"row merged in place with a [{w.rows} x {w.step_cols}] step lse")
    return f"invariant_unary_fwd log1p of {w.rows * w.cols} fp32 values"


def host_cpu() -> str:
    """The host CPU the oracle runs on: architecture, model and logical CPUs
    (from lscpu where it is present)."""
    import platform
    model = ""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name:"):
                model = line.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    return f"{platform.machine()}, {model or 'model not reported'}, {os.cpu_count()} logical CPUs"


def n_sets_for(name: str) -> int:
    """Buffer sets the timed loop rotates through: the smallest power of two
    >= N_SETS whose sets together hold at least ROTATION_BYTES of the op's
    algorithmic bytes, at most 64."""
    n, h, op, _ = WORKLOADS[name]
    b = algorithmic_bytes(n, h, op)
    k = N_SETS
    while k * b < ROTATION_BYTES and k < 64:
        k *= 2
    return k


def workload_inputs(name: str, n_sets: int = N_SETS):
    """(one x per buffer set, residual, weight) as CPU bf16 tensors."""
    n, h, _, recipe = WORKLOADS[name]
    if recipe == "chain4096":
        ch = inputs.CHAIN4096
        r0, w = ch.initial()
        return [ch.delta(k) for k in range(n_sets)], r0, w
    c = inputs.WORKLOADS[recipe].make(n_rows=n)
    xs = [c["x"]] + [inputs.normal_bf16(inputs.generator(1000 + k), (n, h), 0.0, 1.0)
                     for k in range(1, n_sets)]
    assert all(tuple(x.shape) == (n, h) for x in xs) and tuple(c["residual"].shape) == (n, h), name
    return xs, c["residual"], c["weight"]


def make_sets(device, name: str):
    """n_sets_for(name) independent buffer sets; set 0 holds the workload's
    own first draw (used by the parity spot check)."""
    n, h, op, _ = WORKLOADS[name]
    xs, r0, w = workload_inputs(name, n_sets_for(name))
    sets = []
    for x_cpu in xs:
        x = x_cpu.to(device)
        s = {"x": x, "r": r0.to(device), "out": torch.empty_like(x), "ro": torch.empty_like(x)}
        if op.endswith("quant") or op.endswith("fp8") or op.endswith("fp4"):
            s["q"] = torch.empty(n, h // 2 if op.endswith("fp4") else h, dtype=torch.int8, device=device)
            s["scale"] = torch.empty(n, dtype=torch.float32, device=device)
        sets.append(s)
    return sets, w.to(device), (xs[0], r0, w)


class RawCall:
    """Precomputed C-ABI calls, one per buffer set, of the workload's op:
    add_rmsnorm_fwd(out, residual_out, x, residual, weight, eps, n, h, stream),
    add_rmsnorm_quant_fwd(out_q, scale, residual_out, x, residual, ...),
    rmsnorm_fwd(out, x, weight, ...), rmsnorm_quant_fwd(out_q, scale, x, ...)
    or residual_add_fwd(residual_out, x, residual, n, h, stream)."""

    def __init__(self, sets, w, stream, n_rows, hidden, op):
        L = dr.lib()
        self.name = op + "_fwd"
        self.fn = getattr(L, self.name)
        eps = ctypes.c_float(inputs.EPS)
        st = stream.cuda_stream
        wp = w.data_ptr()

        def args(s):
            x, r, ro = s["x"].data_ptr(), s["r"].data_ptr(), s["ro"].data_ptr()
            if op == "add_rmsnorm":
                return (s["out"].data_ptr(), ro, x, r, wp, eps, n_rows, hidden, st)
            if op in ("add_rmsnorm_quant", "add_rmsnorm_fp8", "add_rmsnorm_fp4"):
                return (s["q"].data_ptr(), s["scale"].data_ptr(), ro, x, r, wp, eps, n_rows, hidden, st)
            if op == "rmsnorm":
                return (s["out"].data_ptr(), x, wp, eps, n_rows, hidden, st)
            if op in ("rmsnorm_quant", "rmsnorm_fp8"):
                return (s["q"].data_ptr(), s["scale"].data_ptr(), x, wp, eps, n_rows, hidden, st)
            return (ro, x, r, n_rows, hidden, st)

        self.args = [args(s) for s in sets]

    def __call__(self, i: int):
        st = self.fn(*self.args[i % len(self.args)])
        if st != 0:
            raise dr.DraddError(st, self.name)


GRAPH_CHUNK = 256  # most launches captured in one CUDA graph
PREROLL_CYCLES = 1_000_000


def graph_plan(steps: int, n_sets: int, chunk: int = GRAPH_CHUNK):
    """The CUDA graphs that replay `steps` launches, in order: a list of
    (launches, first buffer set).  Launch k of the timed run (k = 0 ..
    steps - 1) uses buffer set k mod n_sets whatever the split, so a graph
    starts its rotation where the previous one stopped; graphs with the same
    (launches, first set) are one captured graph replayed again."""
    if steps < 0 or n_sets < 1 or chunk < 1:
        raise ValueError("graph_plan: steps >= 0, n_sets >= 1, chunk >= 1")
    plan, k = [], 0
    while k < steps:
        n = min(chunk, steps - k)
        plan.append((n, k % n_sets))
        k += n
    return plan


def time_device(call, steps, warmup, stream, world, use_graph, n_sets):
    """Exactly `steps` launches back to back on `stream`, timed with CUDA
    events; launch k uses buffer set k mod n_sets (call(k)).  With use_graph
    the launches are replayed from CUDA graphs of at most GRAPH_CHUNK
    launches (graph_plan)."""
    for i in range(warmup):
        call(i)
    torch.cuda.synchronize()
    plan, graphs = graph_plan(steps, n_sets), {}
    if use_graph:
        for key in dict.fromkeys(plan):
            n, first = key
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for i in range(n):
                    call(first + i)
            g.replay()  # untimed
            graphs[key] = g
        torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    # Keep the stream busy (about half a millisecond, untimed) while the
    # host enqueues the start event and the first launches, so the timed
    # region holds the launches themselves and no host submission gap.
    with torch.cuda.stream(stream):
        torch.cuda._sleep(PREROLL_CYCLES)
    start.record(stream)
    if use_graph:
        for key in plan:
            graphs[key].replay()
    else:
        for i in range(steps):
            call(i)
    end.record(stream)
    end.synchronize()
    torch.cuda.synchronize()
    barrier(world)
    return start.elapsed_time(end)  # ms


def time_e2e(steps, device, stream, name):
    """Public API with host data: per step, the kernel reads that step's
    inputs (x, residual, weight) from pinned host memory over the host link
    and writes out and residual_out back to pinned host memory
    (host.add_rmsnorm_fwd_host, zero copy); the step ends when the stream
    has finished, i.e. when the results are in host memory."""
    from deterministic_residual_add_gb300.host import add_rmsnorm_fwd_host
    n, h, op, _ = WORKLOADS[name]
    quant = op == "add_rmsnorm_quant"
    xs, r0, w = workload_inputs(name)
    x_h, r_h, w_h = xs[0].pin_memory(), r0.pin_memory(), w.pin_memory()
    ro_h = torch.empty_like(x_h).pin_memory()
    if quant:
        outs = (torch.empty(n, h, dtype=torch.int8).pin_memory(),
                torch.empty(n, dtype=torch.float32).pin_memory(), ro_h)
    else:
        outs = (torch.empty_like(x_h).pin_memory(), ro_h)
    with torch.cuda.stream(stream):
        for _ in range(3):
            add_rmsnorm_fwd_host(x_h, r_h, w_h, inputs.EPS, outs, stream=stream, quant=quant)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(steps):
            add_rmsnorm_fwd_host(x_h, r_h, w_h, inputs.EPS, outs, stream=stream, quant=quant)
        torch.cuda.synchronize()
        dt = time.perf_counter() - t0
    bi = (x_h.numel() + r_h.numel() + w_h.numel()) * 2
    bo = sum(t.numel() * t.element_size() for t in outs)
    return dt, bi, bo


def cpu_baseline(seconds: float, name: str, first_inputs, gpu_set0=None):
    """The CPU oracle (single thread) on leading rows of the same workload,
    for about `seconds`; also checks those rows against the GPU's output."""
    import numpy as np
    import oracle
    o = oracle.lib()
    n, h, op, _ = WORKLOADS[name]
    x0, r0, w = first_inputs
    fns = {"add_rmsnorm": lambda x, r: o.add_rmsnorm_fwd(x, r, w, inputs.EPS),
           "add_rmsnorm_quant": lambda x, r: o.add_rmsnorm_quant_fwd(x, r, w, inputs.EPS),
           "rmsnorm": lambda x, r: (o.rmsnorm_fwd(x, w, inputs.EPS),),
           "rmsnorm_quant": lambda x, r: o.rmsnorm_quant_fwd(x, w, inputs.EPS),
           "residual_add": lambda x, r: (o.residual_add_fwd(x, r),),
           "add_rmsnorm_fp8": lambda x, r: o.rmsnorm_fp8_fwd(x, w, inputs.EPS, residual=r),
           "rmsnorm_fp8": lambda x, r: o.rmsnorm_fp8_fwd(x, w, inputs.EPS),
           "add_rmsnorm_fp4": lambda x, r: o.rmsnorm_fp4_fwd(x, w, inputs.EPS, residual=r)}
    fn = fns[op]
    chunk = 64
    rows = 0
    first = None
    t0 = time.perf_counter()
    while True:
        lo = rows % n
        hi = min(n, lo + chunk)
        res = fn(x0[lo:hi], r0[lo:hi])
        if first is None:
            first = res
        rows += hi - lo
        if time.perf_counter() - t0 >= seconds:
            break
    dt = time.perf_counter() - t0
    out = {"value": algorithmic_bytes(rows, h, op) / dt / 1e9, "unit": "GB/s", "cores": 1,
           "host": host_cpu(), "kind": "oracle",
           "sample": f"{rows} rows of the {n}x{h} workload ({rows * h} elements) in "
                     f"{dt:.1f} s, single thread",
           "seconds": round(dt, 3)}
    # The same per-row code with the rows split over every host core (rows
    # are independent, so the bits are the single-threaded run's).
    threaded = {"add_rmsnorm": o.add_rmsnorm_fwd, "add_rmsnorm_quant": o.add_rmsnorm_quant_fwd}.get(op)
    if threaded is not None:
        cores = oracle.default_threads()
        tchunk = min(n, chunk * cores)
        trows = 0
        t0 = time.perf_counter()
        while True:
            lo = trows % n
            hi = min(n, lo + tchunk)
            threaded(x0[lo:hi], r0[lo:hi], w, inputs.EPS, threads=cores)
            trows += hi - lo
            if time.perf_counter() - t0 >= max(1.0, seconds / 3):
                break
        tdt = time.perf_counter() - t0
        out["all_cores"] = {"value": round(algorithmic_bytes(trows, h, op) / tdt / 1e9, 4), "cores": cores,
                            "sample": f"{trows} rows in {tdt:.1f} s, rows split over {cores} threads"}
    if gpu_set0 is not None:
        def host(t):
            t = t[:chunk].cpu()
            if t.dtype == torch.bfloat16:
                t = t.view(torch.int16)
            return t.numpy()
        keys = {"add_rmsnorm": ["out", "ro"], "add_rmsnorm_quant": ["q", "scale", "ro"],
                "rmsnorm": ["out"], "rmsnorm_quant": ["q", "scale"], "residual_add": ["ro"],
                "add_rmsnorm_fp8": ["q", "scale", "ro"], "rmsnorm_fp8": ["q", "scale"],
                "add_rmsnorm_fp4": ["q", "scale", "ro"]}[op]
        got = [host(gpu_set0[k]) for k in keys]
        out["parity_rows_checked"] = chunk
        out["parity_bit_exact"] = bool(all(
            np.array_equal(np.ascontiguousarray(g).view(np.uint8), np.ascontiguousarray(e).view(np.uint8))
            for g, e in zip(got, first)))
        if op == "add_rmsnorm":
            out["numerics"] = spot_numerics(x0[:chunk], r0[:chunk], w, got[0], got[1])
    return out


def spot_numerics(x, r, w, out_bits, ro_bits) -> dict:
    """On the spot-checked rows: the largest error of out against the fp64
    evaluation of the page's formula, in bf16 ulps of the exact value, and
    the mean signed magnitude error of residual_out against the exact fp32
    sum (the page's bias metric; truncation gives about -1.5e-3 here)."""
    import numpy as np

    def val(bits):
        return (np.ascontiguousarray(bits).view(np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    xf = x.float().numpy().astype(np.float64)
    rf = r.float().numpy().astype(np.float64)
    wf = w.float().numpy().astype(np.float64)
    acc = xf + rf
    y = acc / np.sqrt((acc * acc).mean(axis=1, keepdims=True) + np.float64(np.float32(inputs.EPS))) * wf
    ulp = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(y), 2.0 ** -133))) - 7)
    acc32 = (x.float() + r.float()).numpy().astype(np.float64)
    nz = acc32 != 0
    bias = float(((np.abs(val(ro_bits)) - np.abs(acc32))[nz] / np.abs(acc32)[nz]).mean())
    return {"rows": int(x.shape[0]), "out_max_ulp_vs_f64": round(float((np.abs(val(out_bits) - y) / ulp).max()), 4),
            "residual_out_magnitude_bias": float(f"{bias:.3e}")}


def run_ours(args):
    world, rank, local = dist_setup()
    device = torch.device("cuda", local)
    n_rows, hidden, op, _ = WORKLOADS[args.workload]
    quant = op.endswith("quant") or op.endswith("fp8") or op.endswith("fp4")
    dr.lib()
    stream = torch.cuda.Stream(device)
    sets, w_dev, first_inputs = make_sets(device, args.workload)
    torch.cuda.synchronize()
    call = RawCall(sets, w_dev, stream, n_rows, hidden, op)
    with torch.cuda.stream(stream):
        sampler = ClockSampler(local)
        with sampler:
            ms = time_device(call, args.steps, args.warmup, stream, world, args.graph, len(sets))
    ms = max_over_ranks(ms, world)
    bytes_step = algorithmic_bytes(n_rows, hidden, op)
    ms_per_step = ms / args.steps
    value = world * bytes_step * args.steps / (ms / 1e3) / 1e9
    per_launch_gbs = bytes_step / (ms_per_step / 1e3) / 1e9
    peak = measured_peaks().get("hbm_gbs")
    peak_src = "measured" if peak else "fallback"
    if not peak:
        peak = 6800.0

    e2e = None
    if not args.no_e2e and op in ("add_rmsnorm", "add_rmsnorm_quant"):
        e2e_steps = max(3, min(args.steps, args.e2e_steps))
        dt, bi, bo = time_e2e(e2e_steps, device, stream, args.workload)
        dt = max_over_ranks(dt, world)
        e2e = {"value": round(world * bytes_step * e2e_steps / dt / 1e9, 2), "unit": "GB/s",
               "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo, "steps": e2e_steps,
               "ms_per_step": round(dt / e2e_steps * 1e3, 4),
               "pipeline": "zero copy: the kernel reads and writes pinned host memory over the host link"}

    sm_count = torch.cuda.get_device_properties(device).multi_processor_count
    if op == "residual_add":
        launch = {"variant": "elementwise"}
    else:
        cfg = dr.resolve_config(n_rows, hidden, quant=quant, sm_count=sm_count, add=op.startswith("add"),
                                fp8=op.endswith("fp8"), fp4=op.endswith("fp4"))
        launch = {"variant": VARIANT_NAMES[cfg.variant],
                  "threads_per_row": cfg.threads_per_row, "rows_per_cta": cfg.rows_per_cta,
                  "stages": cfg.stages}
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 6),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": workload_desc(args.workload), "n_rows": n_rows, "hidden": hidden,
                   "io_dtype": "bf16",
                   "l2": l2_desc(len(sets), bytes_step),
                   "launch": launch,
                   "cuda_graph": bool(args.graph), "parallelism": f"replicas x{world}"},
        "rows_per_s": round(world * n_rows * args.steps / (ms / 1e3), 1),
        "roofline": {"bound": "hbm", "achieved": round(per_launch_gbs, 2), "peak": peak,
                     "unit": "GB/s", "frac": round(per_launch_gbs / peak, 4),
                     "peak_source": f"{peak_src} hbm_gbs",
                     "frac_of_nominal": round(per_launch_gbs / NOMINAL_HBM_GBS, 4),
                     **traffic_fields(args.workload, ms_per_step, peak),
                     "algorithmic_bytes_per_launch": bytes_step},
        "gpu_launches": args.steps,
        "e2e": e2e,
    }
    if rank == 0:
        line["clocks"] = sampler.summary()
        if not args.no_cpu:
            line["cpu_baseline"] = cpu_baseline(args.cpu_seconds, args.workload, first_inputs, sets[0])
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as tdist
        tdist.destroy_process_group()


# ------------------------------------------------------- fused q/k RMSNorm
def qk_algorithmic_bytes(w, n_tokens: int) -> int:
    """q: bf16 read, residual read + residual_out write (with a residual),
    e4m3 codes (1 byte) + a 4-byte scale per group, or a bf16 store; k: bf16
    read and store; both weights once."""
    eq = n_tokens * w.q_heads * w.q_head
    ek = n_tokens * w.k_heads * w.k_head
    q_bytes = 2 * eq + (4 * eq if w.residual else 0)
    q_bytes += (eq + 4 * eq // w.group_size) if w.group_size else 2 * eq
    return q_bytes + 4 * ek + 2 * (w.q_head + w.k_head)


def qk_oracle_fn(o, w):
    def fn(d):
        return o.qk_rmsnorm_fwd(d["q"], d["q_weight"], d["k"], d["k_weight"], inputs.EPS, inputs.EPS,
                                group_size=w.group_size, q_residual=d["residual"])
    return fn


def qk_slice(d, w, lo, hi):
    """Tokens [lo, hi) of a q/k input dict."""
    out = dict(d)
    out["q"] = d["q"][lo * w.q_heads:hi * w.q_heads]
    out["k"] = d["k"][lo * w.k_heads:hi * w.k_heads]
    if d["residual"] is not None:
        out["residual"] = d["residual"][lo * w.q_heads:hi * w.q_heads]
    return out


def run_qk(args):
    """The fused q/k RMSNorm workloads: same timing rules as the main op,
    with enough rotating buffer sets to exceed L2 four times over."""
    import numpy as np
    world, rank, local = dist_setup()
    device = torch.device("cuda", local)
    w = inputs.QK_WORKLOADS[args.workload]
    L = dr.lib()
    stream = torch.cuda.Stream(device)
    d0 = w.make()
    bytes_step = qk_algorithmic_bytes(w, w.n_tokens)
    n_sets = workload_n_sets(args.workload)
    nq, nk = d0["q"].shape[0], d0["k"].shape[0]
    qw, kw = d0["q_weight"].to(device), d0["k_weight"].to(device)
    sets = []
    for i in range(n_sets):
        g = inputs.generator(2000 + i)
        q = d0["q"] if i == 0 else inputs.normal_bf16(g, tuple(d0["q"].shape), 0.0, 1.0)
        k = d0["k"] if i == 0 else inputs.normal_bf16(g, tuple(d0["k"].shape), 0.0, 1.0)
        s = {"q": q.to(device), "k": k.to(device), "k_out": torch.empty(tuple(k.shape), dtype=torch.bfloat16,
                                                                          device=device)}
        s["r"] = d0["residual"].to(device) if w.residual else None
        s["ro"] = torch.empty_like(s["q"]) if w.residual else None
        if w.group_size:
            s["q_out"] = torch.empty(tuple(q.shape), dtype=torch.uint8, device=device)
            s["q_scale"] = torch.empty(nq, w.q_head // w.group_size, dtype=torch.float32, device=device)
        else:
            s["q_out"] = torch.empty_like(s["q"])
            s["q_scale"] = None
        sets.append(s)
    torch.cuda.synchronize()
    eps = ctypes.c_float(inputs.EPS)
    st = stream.cuda_stream
    argv = []
    for s in sets:
        argv.append((s["q_out"].data_ptr(), s["q_scale"].data_ptr() if s["q_scale"] is not None else None,
                     s["ro"].data_ptr() if s["ro"] is not None else None, s["k_out"].data_ptr(),
                     s["q"].data_ptr(), s["r"].data_ptr() if s["r"] is not None else None, qw.data_ptr(),
                     s["k"].data_ptr(), kw.data_ptr(), eps, eps, nq, w.q_head, nk, w.k_head, w.group_size, st))
    fn = L.fused_qk_rmsnorm_group_quant_fwd

    def call(i):
        rc = fn(*argv[i % n_sets])
        if rc != 0:
            raise dr.DraddError(rc, "fused_qk_rmsnorm_group_quant_fwd")

    with torch.cuda.stream(stream):
        sampler = ClockSampler(local)
        with sampler:
            ms = time_device(call, args.steps, args.warmup, stream, world, args.graph, n_sets)
    ms = max_over_ranks(ms, world)
    ms_per_step = ms / args.steps
    per_launch_gbs = bytes_step / (ms_per_step / 1e3) / 1e9
    peak = measured_peaks().get("hbm_gbs")
    peak_src = "measured" if peak else "fallback"
    if not peak:
        peak = 6800.0
    # sm_count 0: the device's plan, with the grid the call launches
    plan = dr.qk_resolve_config(nq, w.q_head, nk, w.k_head, w.group_size, q_residual=w.residual, sm_count=0)
    line = {
        "metric": QK_METRIC, "value": round(world * bytes_step * args.steps / (ms / 1e3) / 1e9, 2), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 6),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": qk_workload_desc(w),
                   "n_q_rows": nq, "q_hidden": w.q_head, "n_k_rows": nk, "k_hidden": w.k_head,
                   "group_size": w.group_size, "io_dtype": "bf16",
                   "l2": l2_desc(n_sets, bytes_step),
                   "launch": dataclasses.asdict(plan), "cuda_graph": bool(args.graph),
                   "parallelism": f"replicas x{world}"},
        "tokens_per_s": round(world * w.n_tokens * args.steps / (ms / 1e3), 1),
        "roofline": {"bound": "hbm", "achieved": round(per_launch_gbs, 2), "peak": peak, "unit": "GB/s",
                     "frac": round(per_launch_gbs / peak, 4), "peak_source": f"{peak_src} hbm_gbs",
                     "frac_of_nominal": round(per_launch_gbs / NOMINAL_HBM_GBS, 4),
                     **traffic_fields(args.workload, ms_per_step, peak),
                     "algorithmic_bytes_per_launch": bytes_step},
        "gpu_launches": args.steps,
        "e2e": None,
    }
    if rank == 0:
        line["clocks"] = sampler.summary()
        if not args.no_cpu:
            import oracle
            fn_o = qk_oracle_fn(oracle.lib(), w)
            chunk = 16
            tokens, first = 0, None
            t0 = time.perf_counter()
            while True:
                lo = tokens % w.n_tokens
                hi = min(w.n_tokens, lo + chunk)
                res = fn_o(qk_slice(d0, w, lo, hi))
                first = first or res
                tokens += hi - lo
                if time.perf_counter() - t0 >= args.cpu_seconds:
                    break
            dt = time.perf_counter() - t0
            s0 = sets[0]
            got = {"q_out": s0["q_out"][:chunk * w.q_heads], "k_out": s0["k_out"][:chunk * w.k_heads]}
            if w.group_size:
                got["q_scale"] = s0["q_scale"][:chunk * w.q_heads]
            if w.residual:
                got["q_residual_out"] = s0["ro"][:chunk * w.q_heads]

            def raw(t):
                t = t.detach().cpu().contiguous()
                return t.view(torch.uint8).numpy() if t.dtype != torch.uint8 else t.numpy()
            exact = all(np.array_equal(raw(got[k]), np.ascontiguousarray(first[k]).view(np.uint8))
                        for k in got)
            line["cpu_baseline"] = {
                "value": round(qk_algorithmic_bytes(w, tokens) / dt / 1e9, 4), "unit": "GB/s", "cores": 1,
                "host": host_cpu(),
                "kind": "oracle", "sample": f"{tokens} tokens of the {w.n_tokens}-token workload in {dt:.1f} s, "
                                            "single thread", "seconds": round(dt, 3),
                "parity_rows_checked": chunk, "parity_bit_exact": bool(exact)}
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as tdist
        tdist.destroy_process_group()


# ------------------------------------------- log-sum-exp merge and log1p
ELEM_METRIC = "launch-invariant LSE merge / log1p GB/s and % of HBM peak; within the stated bound of the oracle"


def elem_bytes(w) -> int:
    """merge: read the running lse and the step lse, write the merged lse
    (12 B per merged element); log1p: 8 B per element."""
    return 12 * w.rows * w.step_cols if w.kind == "merge" else 8 * w.rows * w.cols


def run_elem(args):
    import numpy as np
    world, rank, local = dist_setup()
    device = torch.device("cuda", local)
    w = inputs.ELEM_WORKLOADS[args.workload]
    L = dr.lib()
    stream = torch.cuda.Stream(device)
    d0 = w.make()
    bytes_step = elem_bytes(w)
    n_sets = workload_n_sets(args.workload)
    st = stream.cuda_stream
    sets, argv = [], []
    for i in range(n_sets):
        if w.kind == "merge":
            run = (d0["lse"] if i == 0 else d0["lse"].roll(i, 0)).to(device).contiguous()
            step = d0["step"].to(device)
            off = w.cols - w.step_cols
            half = run[:, off:]
            sets.append((run, step))
            argv.append((half.data_ptr(), w.cols, half.data_ptr(), w.cols, step.data_ptr(), w.step_cols,
                         w.rows, w.step_cols, st))
        else:
            x = d0["x"].to(device)
            y = torch.empty_like(x)
            sets.append((x, y))
            argv.append((y.data_ptr(), x.data_ptr(), x.numel(), 0, st))
    fn = L.lse_merge_2d_fwd if w.kind == "merge" else L.invariant_unary_fwd
    torch.cuda.synchronize()

    def call(i):
        rc = fn(*argv[i % n_sets])
        if rc != 0:
            raise dr.DraddError(rc, fn.__name__)

    with torch.cuda.stream(stream):
        sampler = ClockSampler(local)
        with sampler:
            ms = time_device(call, args.steps, args.warmup, stream, world, args.graph, n_sets)
    ms = max_over_ranks(ms, world)
    ms_per_step = ms / args.steps
    per_launch = bytes_step / (ms_per_step / 1e3) / 1e9
    peak = measured_peaks().get("hbm_gbs")
    peak_src = "measured" if peak else "fallback"
    if not peak:
        peak = 6800.0
    desc = elem_workload_desc(w)
    line = {
        "metric": ELEM_METRIC, "value": round(world * bytes_step * args.steps / (ms / 1e3) / 1e9, 2), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 6),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": desc, "io_dtype": "f32",
                   "l2": l2_desc(n_sets, bytes_step),
                   "launch": {"threads_per_cta": 128, "elements_per_thread": 8}, "cuda_graph": bool(args.graph),
                   "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "hbm", "achieved": round(per_launch, 2), "peak": peak, "unit": "GB/s",
                     "frac": round(per_launch / peak, 4), "peak_source": f"{peak_src} hbm_gbs",
                     **traffic_fields(args.workload, ms_per_step, peak),
                     "frac_of_nominal": round(per_launch / NOMINAL_HBM_GBS, 4),
                     "algorithmic_bytes_per_launch": bytes_step},
        "gpu_launches": args.steps,
        "e2e": None,
    }
    if rank == 0:
        line["clocks"] = sampler.summary()
        if not args.no_cpu:
            import oracle.lse as lse_oracle
            o = lse_oracle.lib()
            t0 = time.perf_counter()
            done = 0
            if w.kind == "merge":
                run_np, step_np = d0["lse"].numpy(), d0["step"].numpy()
                off = w.cols - w.step_cols
                while time.perf_counter() - t0 < args.cpu_seconds:
                    r = done % w.rows
                    o.merge(run_np[r, off:], step_np[r])
                    done += 1
                units, elems = "rows", done * w.step_cols
                cpu_bytes = 12 * elems
                # the timed steps merged in place repeatedly: check a fresh call
                fresh = d0["lse"].to(device)
                half = fresh[:, off:]
                dr.lse_merge_fwd(half, d0["step"].to(device), out=half)
                torch.cuda.synchronize()
                got = fresh[0, off:].cpu().numpy()
                ref = o.merge(run_np[0, off:], step_np[0])
            else:
                x_np = d0["x"].numpy()
                chunk = 1 << 16
                while time.perf_counter() - t0 < args.cpu_seconds:
                    lo = (done * chunk) % (x_np.size - chunk + 1) if x_np.size > chunk else 0
                    o.unary(x_np[lo:lo + chunk], "log1p")
                    done += 1
                units, elems = "chunks", done * min(chunk, x_np.size)
                cpu_bytes = 8 * elems
                got = sets[0][1][:4096].cpu().numpy()
                ref = o.unary(x_np[:4096], "log1p")
            dt = time.perf_counter() - t0
            a = np.abs(ref)
            ulp = 2.0 ** (np.floor(np.log2(np.maximum(a, 2.0 ** -126))) - 23)
            bound = ulp + (2.0 ** -22 if w.kind == "merge" else 0.0)
            line["cpu_baseline"] = {
                "value": round(cpu_bytes / dt / 1e9, 4), "unit": "GB/s", "cores": 1,
                "host": host_cpu(), "kind": "oracle",
                "sample": f"{done} {units} ({elems} elements) of the workload in {dt:.1f} s, single thread, double",
                "seconds": round(dt, 3), "parity_elements_checked": int(ref.size),
                "parity_within_bound": bool(np.all(np.abs(got.astype(np.float64) - ref) <= bound))}
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as tdist
        tdist.destroy_process_group()


def run_elem_reference(args):
    if int(os.environ.get("RANK", "0")) != 0:
        return
    import oracle.lse as lse_oracle
    o = lse_oracle.lib()
    w = inputs.ELEM_WORKLOADS[args.workload]
    d0 = w.make()
    if w.kind == "merge":
        run_np, step_np = d0["lse"].numpy(), d0["step"].numpy()
        off = w.cols - w.step_cols
        t0 = time.perf_counter()
        o.merge(run_np[0, off:], step_np[0])
        t_row = max(1e-6, time.perf_counter() - t0)
        rows = int(max(1, min(w.rows, args.reference_seconds / (args.warmup + args.steps) / t_row)))
        def fn(i):
            lo = (i * rows) % (w.rows - rows + 1)
            o.merge(run_np[lo:lo + rows, off:], step_np[lo:lo + rows])
        per_step = 12 * rows * w.step_cols
        sample = f"{rows} of {w.rows} rows per step"
    else:
        x_np = d0["x"].numpy()
        t0 = time.perf_counter()
        o.unary(x_np[:4096], "log1p")
        t_el = max(1e-9, (time.perf_counter() - t0) / 4096)
        n = int(max(1, min(x_np.size, args.reference_seconds / (args.warmup + args.steps) / t_el)))
        fn = lambda i: o.unary(x_np[:n], "log1p")
        per_step = 8 * n
        sample = f"{n} of {x_np.size} values per step"
    for i in range(args.warmup):
        fn(i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        fn(i)
    dt = time.perf_counter() - t0
    value = per_step * args.steps / dt / 1e9
    print(json.dumps({
        "impl": "reference", "metric": ELEM_METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": elem_workload_desc(w), "engine": "CPU oracle", "sample": sample},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1,
                         "host": host_cpu(), "kind": "oracle",
                         "sample": f"{sample}, single thread"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0}), flush=True)


def run_qk_reference(args):
    """The oracle on the host cores for a fused q/k workload."""
    if int(os.environ.get("RANK", "0")) != 0:
        return
    import oracle
    w = inputs.QK_WORKLOADS[args.workload]
    fn = qk_oracle_fn(oracle.lib(), w)
    d0 = w.make()
    t0 = time.perf_counter()
    fn(qk_slice(d0, w, 0, 4))
    t_tok = max(1e-6, (time.perf_counter() - t0) / 4)
    total = args.warmup + args.steps
    tokens = int(max(1, min(w.n_tokens, args.reference_seconds / total / t_tok)))
    for _ in range(args.warmup):
        fn(qk_slice(d0, w, 0, tokens))
    t0 = time.perf_counter()
    for i in range(args.steps):
        lo = (i * tokens) % (w.n_tokens - tokens + 1)
        fn(qk_slice(d0, w, lo, lo + tokens))
    dt = time.perf_counter() - t0
    value = qk_algorithmic_bytes(w, tokens) * args.steps / dt / 1e9
    print(json.dumps({
        "impl": "reference", "metric": QK_METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": qk_workload_desc(w), "engine": "CPU oracle", "tokens_per_step": tokens},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1,
                         "host": host_cpu(), "kind": "oracle",
                         "sample": f"{tokens} of {w.n_tokens} tokens per step, single thread"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0}), flush=True)


def run_reference(args):
    """The oracle on the host cores, on the same metric, unit and workload:
    each step runs a bounded sample of rows of the batch."""
    if int(os.environ.get("RANK", "0")) != 0:
        return
    import oracle
    o = oracle.lib()
    n, h, op, _ = WORKLOADS[args.workload]
    xs, r0, w = workload_inputs(args.workload)
    x0 = xs[0]
    fns = {"add_rmsnorm": lambda x, r: o.add_rmsnorm_fwd(x, r, w, inputs.EPS),
           "add_rmsnorm_quant": lambda x, r: o.add_rmsnorm_quant_fwd(x, r, w, inputs.EPS),
           "rmsnorm": lambda x, r: o.rmsnorm_fwd(x, w, inputs.EPS),
           "rmsnorm_quant": lambda x, r: o.rmsnorm_quant_fwd(x, w, inputs.EPS),
           "residual_add": lambda x, r: o.residual_add_fwd(x, r),
           "add_rmsnorm_fp8": lambda x, r: o.rmsnorm_fp8_fwd(x, w, inputs.EPS, residual=r),
           "rmsnorm_fp8": lambda x, r: o.rmsnorm_fp8_fwd(x, w, inputs.EPS),
           "add_rmsnorm_fp4": lambda x, r: o.rmsnorm_fp4_fwd(x, w, inputs.EPS, residual=r)}
    fn = fns[op]
    t0 = time.perf_counter()
    fn(x0[:16], r0[:16])
    t_row = max(1e-6, (time.perf_counter() - t0) / 16)
    total = args.warmup + args.steps
    rows = int(max(1, min(n, args.reference_seconds / total / t_row)))
    for _ in range(args.warmup):
        fn(x0[:rows], r0[:rows])
    t0 = time.perf_counter()
    for i in range(args.steps):
        lo = (i * rows) % (n - rows + 1)
        fn(x0[lo:lo + rows], r0[lo:lo + rows])
    dt = time.perf_counter() - t0
    value = algorithmic_bytes(rows, h, op) * args.steps / dt / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": workload_desc(args.workload), "engine": "CPU oracle", "n_rows": n, "hidden": h,
                   "io_dtype": "bf16", "rows_per_step": rows},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1,
                         "host": host_cpu(), "kind": "oracle",
                         "sample": f"{rows} of {n} rows per step, single thread"},
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
    ap.add_argument("--workload", choices=list(WORKLOADS) + list(inputs.QK_WORKLOADS) + list(inputs.ELEM_WORKLOADS),
                    default="4096x4096")
    ap.add_argument("--graph", type=int, default=1, help="replay the timed steps from CUDA graphs")
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--reference-seconds", type=float, default=60.0)
    ap.add_argument("--ncu-command", action="store_true",
                    help="print the ncu capture command behind the workload's traffic record and exit")
    ap.add_argument("--ncu-record", metavar="CSV",
                    help="write profiles/ncu_<workload>.json from the log of that capture and exit")
    args = ap.parse_args()
    if args.ncu_command:
        print(f"python bench.py --workload {args.workload} {ncu_bench_args(args.workload)}")
        print(ncu_capture_command(args.workload))
        return
    if args.ncu_record:
        rec = make_ncu_record(args.workload, Path(args.ncu_record).read_text())
        ncu_record_path(args.workload).write_text(json.dumps(rec, indent=1) + "\n")
        print(json.dumps(rec))
        return
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.workload in inputs.QK_WORKLOADS:
        (run_qk_reference if args.impl == "reference" else run_qk)(args)
    elif args.workload in inputs.ELEM_WORKLOADS:
        (run_elem_reference if args.impl == "reference" else run_elem)(args)
    else:
        (run_reference if args.impl == "reference" else run_ours)(args)


if __name__ == "__main__":
    main()
