"""bench.py's host-side rules, without a GPU: the algorithmic byte counts,
the rotating buffer sets (together at least 1 GiB, about eight times the L2, so
no step reads its inputs from L2), and the workload descriptions that both
arms print."""
import torch

import bench
from deterministic_residual_add_gb300 import inputs


def test_algorithmic_bytes():
    e = 4096 * 4096
    assert bench.algorithmic_bytes(4096, 4096) == 8 * e + 2 * 4096
    assert bench.algorithmic_bytes(2048, 16384, "add_rmsnorm_quant") == 7 * 2048 * 16384 + 4 * 2048 + 2 * 16384
    assert bench.algorithmic_bytes(4096, 4096, "rmsnorm_quant") == 3 * e + 4 * 4096 + 2 * 4096
    assert bench.algorithmic_bytes(4096, 4096, "residual_add") == 6 * e


def test_rotating_sets_exceed_l2():
    for name, (n, h, op, _) in bench.WORKLOADS.items():
        k = bench.n_sets_for(name)
        assert k >= bench.N_SETS and k & (k - 1) == 0 and bench.GRAPH_CHUNK % k == 0, name
        assert k * bench.algorithmic_bytes(n, h, op) >= bench.ROTATION_BYTES or k == 64, name
        assert k == bench.N_SETS or (k // 2) * bench.algorithmic_bytes(n, h, op) < bench.ROTATION_BYTES, name
    assert bench.n_sets_for("4096x4096") == 8
    assert bench.n_sets_for("rmsnorm_quant4096x4096") == 32


def test_workload_descriptions():
    assert bench.workload_desc("4096x4096") == "add_rmsnorm_fwd 4096x4096 bf16 in/out"
    assert "int8 + fp32 scale" in bench.workload_desc("quant2048x16384")
    w = inputs.QK_WORKLOADS["qk_lowrank4096"]
    assert bench.qk_workload_desc(w).startswith("fused_qk_rmsnorm_group_quant_fwd 4096 tokens")
    assert bench.elem_workload_desc(inputs.ELEM_WORKLOADS["log1p16M"]).startswith("invariant_unary_fwd log1p")


def test_input_recipes_draw_the_stated_distributions():
    """x ~ N(0, x_std), residual ~ N(0, residual_std), weight ~ N(1, 0.1),
    bf16, at the stated shapes; the first rows of a full draw equal a draw
    of those rows alone."""
    for name, (mx, sx, sr) in {"tiny": (0.0, 1.0, 1.0), "2048x4096": (0.0, 1.0, 4.0),
                               "8192x2048": (0.0, 1.0, 4.0)}.items():
        w = inputs.WORKLOADS[name]
        c = w.make()
        assert tuple(c["x"].shape) == (w.n_rows, w.hidden) and c["x"].dtype == torch.bfloat16
        assert tuple(c["residual"].shape) == (w.n_rows, w.hidden) and tuple(c["weight"].shape) == (w.hidden,)
        x, r, wt = (c[k].float() for k in ("x", "residual", "weight"))
        tol = 6.0 / (w.n_rows * w.hidden) ** 0.5
        assert abs(x.mean().item() - mx) < tol * sx and abs(x.std().item() / sx - 1) < 0.01, name
        assert abs(r.mean().item()) < tol * sr and abs(r.std().item() / sr - 1) < 0.01, name
        assert abs(wt.mean().item() - 1.0) < 0.02 and abs(wt.std().item() / 0.1 - 1) < 0.1, name
        head = w.make(n_rows=5)
        assert torch.equal(head["x"], c["x"][:5]) and torch.equal(head["residual"], c["residual"][:5])


def test_reference_arm_line():
    """`bench.py --impl reference` runs the CPU oracle on the headline
    workload (no GPU needed) and prints one JSON line with the keys the
    measurement contract names, on the same metric, unit and workload as
    the library's arm."""
    import json
    import subprocess
    import sys
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "3"],
                         cwd=bench.ROOT, capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == "GB/s"
    assert d["higher_is_better"] is True and d["steps"] == 1 and d["warmup"] == 3 and d["value"] > 0
    assert d["config"]["workload"] == bench.workload_desc("4096x4096")
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_launch_variant_names():
    """config.launch names the variant the automatic plan resolves to, for
    every main-op workload (152 SMs)."""
    import deterministic_residual_add_gb300 as dr
    names = {}
    for name, (n, h, op, _) in bench.WORKLOADS.items():
        if op == "residual_add":
            continue
        cfg = dr.resolve_config(n, h, quant=op not in ("add_rmsnorm", "rmsnorm"), sm_count=152,
                                add=op.startswith("add"), fp8=op.endswith("fp8"), fp4=op.endswith("fp4"))
        names[name] = bench.VARIANT_NAMES[cfg.variant]
    assert names["4096x4096"] == "staged"
    assert names["8192x2048"] == "warp"


def test_graph_plan_covers_every_launch_once():
    for steps in (0, 1, 3, 20, 255, 256, 257, 600, 50000):
        for n_sets in (1, 3, 4, 7, 16, 64):
            plan = bench.graph_plan(steps, n_sets)
            assert sum(n for n, _ in plan) == steps
            assert all(0 < n <= bench.GRAPH_CHUNK for n, _ in plan)
            seq = [(first + i) % n_sets for n, first in plan for i in range(n)]
            assert seq == [k % n_sets for k in range(steps)], (steps, n_sets)
    assert bench.graph_plan(20, 4) == [(20, 0)]
    assert bench.graph_plan(257, 4) == [(256, 0), (1, 0)]
    assert len(set(bench.graph_plan(50000, 4))) == 2


class _FakeCuda:
    """Stands in for torch.cuda in time_device: graphs record the call
    indices made while they are captured and replay them into `ran`."""

    def __init__(self):
        self.ran, self.capturing, self.captured = [], None, 0
        fake = self

        class Graph:
            def __init__(self):
                self.calls = []
                fake.captured += 1

            def replay(self):
                fake.ran.extend(self.calls)

        class Capture:
            def __init__(self, g, stream=None):
                self.g = g

            def __enter__(self):
                fake.capturing = self.g

            def __exit__(self, *exc):
                fake.capturing = None

        class Event:
            def __init__(self, enable_timing=False):
                pass

            def record(self, stream=None):
                pass

            def synchronize(self):
                pass

            def elapsed_time(self, other):
                return 1.0

        self.CUDAGraph, self.graph, self.Event = Graph, Capture, Event

    def synchronize(self):
        pass

    def _sleep(self, cycles):
        pass

    def call(self, i):
        (self.capturing.calls if self.capturing is not None else self.ran).append(i)


def test_time_device_runs_exactly_the_timed_launches(monkeypatch):
    """The timed region replays exactly `steps` launches in rotation order,
    for step counts below, at and above one graph (the driver's default
    run is 20 steps)."""
    for steps in (1, 20, 255, 256, 257, 600):
        for n_sets in (4, 16, 6):
            fake = _FakeCuda()
            for name in ("CUDAGraph", "graph", "Event", "synchronize", "_sleep"):
                monkeypatch.setattr(bench.torch.cuda, name, getattr(fake, name))
            warmup = 5
            bench.time_device(lambda i: fake.call(i % n_sets), steps, warmup, None, 1, True, n_sets)
            plan = bench.graph_plan(steps, n_sets)
            # warm-up launches, one untimed replay of each distinct graph, then the timed steps
            untimed = warmup + sum(n for n, _ in dict.fromkeys(plan))
            assert fake.captured == len(set(plan))
            assert fake.ran[untimed:] == [k % n_sets for k in range(steps)], (steps, n_sets)
            fake = _FakeCuda()
            for name in ("CUDAGraph", "graph", "Event", "synchronize", "_sleep"):
                monkeypatch.setattr(bench.torch.cuda, name, getattr(fake, name))
            bench.time_device(lambda i: fake.call(i % n_sets), steps, warmup, None, 1, False, n_sets)
            assert fake.ran[warmup:] == [k % n_sets for k in range(steps)]


_NCU_CSV = '''==PROF== Connected to process 1234 (/usr/bin/python3.12)
==PROF== Disconnected from process 1234
"ID","Process ID","Process Name","Host Name","Kernel Name","Context","Stream","Block Size","Grid Size","Device","CC","Section Name","Metric Name","Metric Unit","Metric Value"
"0","1234","python3.12","127.0.0.1","void dradd::staged_kernel<128, 4, 0, 1>(dradd::Params)","1","13","(128, 1, 1)","(608, 1, 1)","0","10.3","Command line profiler metrics","dram__bytes_read.sum","byte","65,000,000"
"0","1234","python3.12","127.0.0.1","void dradd::staged_kernel<128, 4, 0, 1>(dradd::Params)","1","13","(128, 1, 1)","(608, 1, 1)","0","10.3","Command line profiler metrics","dram__bytes_write.sum","byte","66,000,000"
"0","1234","python3.12","127.0.0.1","void dradd::staged_kernel<128, 4, 0, 1>(dradd::Params)","1","13","(128, 1, 1)","(608, 1, 1)","0","10.3","Command line profiler metrics","gpu__time_duration.sum","nsecond","18,000"
"1","1234","python3.12","127.0.0.1","void dradd::staged_kernel<128, 4, 0, 1>(dradd::Params)","1","13","(128, 1, 1)","(608, 1, 1)","0","10.3","Command line profiler metrics","dram__bytes_read.sum","Mbyte","67"
"1","1234","python3.12","127.0.0.1","void dradd::staged_kernel<128, 4, 0, 1>(dradd::Params)","1","13","(128, 1, 1)","(608, 1, 1)","0","10.3","Command line profiler metrics","dram__bytes_write.sum","byte","64000000"
"1","1234","python3.12","127.0.0.1","void dradd::staged_kernel<128, 4, 0, 1>(dradd::Params)","1","13","(128, 1, 1)","(608, 1, 1)","0","10.3","Command line profiler metrics","gpu__time_duration.sum","usecond","20"
'''


def test_ncu_record_from_csv(tmp_path, monkeypatch):
    """The traffic record is the mean of the captured launches, in bytes and
    ns whatever units ncu printed, keyed by the hash of the current sources;
    bench lines use it only while that hash still matches."""
    rec = bench.make_ncu_record("4096x4096", _NCU_CSV)
    assert rec["launches_captured"] == 2
    assert rec["dram_bytes_read_per_launch"] == 66_000_000
    assert rec["dram_bytes_write_per_launch"] == 65_000_000
    assert rec["dram_bytes_per_launch"] == 131_000_000
    assert rec["gpu_time_duration_ns_mean"] == 19_000.0
    assert rec["algorithmic_bytes_per_launch"] == bench.algorithmic_bytes(4096, 4096)
    assert rec["source_sha256_16"] == bench.source_hash("main")
    assert rec["command"].startswith("ncu --metrics ") and "--clock-control none" in rec["command"]
    monkeypatch.setattr(bench, "PROFILES", tmp_path)
    bench.ncu_record_path("4096x4096").write_text(bench.json.dumps(rec))
    assert bench.recorded_traffic("4096x4096")[0] == 131_000_000
    f = bench.traffic_fields("4096x4096", 0.021, 6800.0)
    assert f["traffic"] == 131_000_000 and abs(f["traffic_over_algorithmic"] - 131e6 / rec["algorithmic_bytes_per_launch"]) < 1e-4
    rec["source_sha256_16"] = "0" * 16
    bench.ncu_record_path("4096x4096").write_text(bench.json.dumps(rec))
    assert bench.recorded_traffic("4096x4096")[0] is None
    assert bench.traffic_fields("4096x4096", 0.021, 6800.0)["traffic"] is None


def test_committed_ncu_records_are_well_formed():
    for p in sorted(bench.PROFILES.glob("ncu_*.json")):
        rec = bench.json.loads(p.read_text())
        name = p.stem[len("ncu_"):]
        assert rec["workload"] == name
        assert rec["algorithmic_bytes_per_launch"] == bench.workload_bytes(name)
        assert rec["dram_bytes_per_launch"] == rec["dram_bytes_read_per_launch"] + rec["dram_bytes_write_per_launch"]
        assert rec["command"] == bench.ncu_capture_command(name)
