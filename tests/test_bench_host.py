"""bench.py's host-side rules, without a GPU: the algorithmic byte counts,
the rotating buffer sets (together at least 512 MiB, four times the L2, so
no step reads its inputs from L2), and the workload descriptions that both
arms print."""
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
        assert k * bench.algorithmic_bytes(n, h, op) >= 512 * 2**20 or k == 64, name
        assert k == bench.N_SETS or (k // 2) * bench.algorithmic_bytes(n, h, op) < 512 * 2**20, name
    assert bench.n_sets_for("4096x4096") == 4
    assert bench.n_sets_for("rmsnorm_quant4096x4096") == 16


def test_workload_descriptions():
    assert bench.workload_desc("4096x4096") == "add_rmsnorm_fwd 4096x4096 bf16 in/out"
    assert "int8 + fp32 scale" in bench.workload_desc("quant2048x16384")
    w = inputs.QK_WORKLOADS["qk_lowrank4096"]
    assert bench.qk_workload_desc(w).startswith("fused_qk_rmsnorm_group_quant_fwd 4096 tokens")
    assert bench.elem_workload_desc(inputs.ELEM_WORKLOADS["log1p16M"]).startswith("invariant_unary_fwd log1p")
