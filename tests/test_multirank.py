"""The N > 1 path on the CPU: two gloo ranks each take their contiguous row
block, run the forward on it (the oracle stands in for the GPU here), and
the gathered blocks equal the single-rank result bit for bit.  The ranks
exchange nothing but the final gather the test does to check them."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as tdist
import torch.multiprocessing as mp

from deterministic_residual_add_gb300.shard import row_range, shard_rows


def test_row_range_partitions():
    for n in (0, 1, 5, 4096, 4097):
        for world in (1, 2, 3, 8):
            spans = [row_range(n, r, world) for r in range(world)]
            assert spans[0][0] == 0 and spans[-1][1] == n
            assert all(a[1] == b[0] for a, b in zip(spans, spans[1:]))
            sizes = [hi - lo for lo, hi in spans]
            assert max(sizes) - min(sizes) <= 1
    with pytest.raises(ValueError):
        row_range(4, 2, 2)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, result_dir):
    import sys
    from pathlib import Path
    root = Path(__file__).resolve().parents[1]
    sys.path.insert(0, str(root))
    import oracle
    from deterministic_residual_add_gb300 import inputs
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    tdist.init_process_group("gloo", rank=rank, world_size=world)
    c = inputs.WORKLOADS["tiny"].make()
    x, r = shard_rows(c["x"], rank, world), shard_rows(c["residual"], rank, world)
    out, ro = oracle.lib().add_rmsnorm_fwd(x, r, c["weight"], c["eps"])
    parts = [None] * world
    tdist.all_gather_object(parts, (out, ro))
    if rank == 0:
        np.save(os.path.join(result_dir, "out.npy"), np.concatenate([p[0] for p in parts]))
        np.save(os.path.join(result_dir, "ro.npy"), np.concatenate([p[1] for p in parts]))
    tdist.barrier()
    tdist.destroy_process_group()


def test_two_ranks_match_one(tmp_path, orc):
    from deterministic_residual_add_gb300 import inputs
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       join=True, start_method="spawn")
    c = inputs.WORKLOADS["tiny"].make()
    out, ro = orc.add_rmsnorm_fwd(c["x"], c["residual"], c["weight"], c["eps"])
    assert np.array_equal(np.load(tmp_path / "out.npy"), out)
    assert np.array_equal(np.load(tmp_path / "ro.npy"), ro)


def _bench_rank_main(rank, world, port, result_dir):
    import sys
    from pathlib import Path
    root = Path(__file__).resolve().parents[1]
    sys.path.insert(0, str(root))
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    tdist.init_process_group("gloo", rank=rank, world_size=world)
    bench.barrier(world)
    # each rank reports its own elapsed time; every rank must get the slowest
    got = bench.max_over_ranks(1.5 + rank * 2.25, world)
    np.save(os.path.join(result_dir, f"max{rank}.npy"), np.array([got]))
    bench.barrier(world)
    tdist.destroy_process_group()


def test_bench_reduces_to_the_slowest_rank(tmp_path):
    """The bench's timing reduction over ranks (gloo stands in for nccl)."""
    world = 2
    mp.start_processes(_bench_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       join=True, start_method="spawn")
    for r in range(world):
        assert float(np.load(tmp_path / f"max{r}.npy")[0]) == 1.5 + (world - 1) * 2.25
