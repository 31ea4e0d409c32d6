"""The N > 1 path on CPU, with world_size-2 gloo process groups.

The engine runs replicas only (rows are independent and no data-path
collective exists): every rank times its own copy of the workload, and the
bench reports the maximum device time over the ranks. These tests cover that
reduction, the launch of the bench under torch.distributed.run, through
the reference arm (the CPU oracle), which needs no GPU, and the row
partitioner that splits one matrix's rows across workers.
"""
import json
import os
import socket
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, values, out_dir):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    sys.path.insert(0, ROOT)
    import bench
    got = bench.max_over_ranks(values[rank], dist)
    with open(os.path.join(out_dir, f"rank{rank}.txt"), "w") as f:
        f.write(repr(got))
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_with_gloo(tmp_path):
    values = [3.25, 7.5]
    mp.start_processes(_rank_main, args=(2, _free_port(), values, str(tmp_path)), nprocs=2,
                       start_method="spawn")
    for r in range(2):
        assert float((tmp_path / f"rank{r}.txt").read_text()) == max(values)


def _shard_main(rank, world, port, out_dir):
    """One worker: its rows from spmm_partition_rows, its share of the product
    from the oracle (test infrastructure), gathered on every rank."""
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    sys.path.insert(0, ROOT)
    import numpy as np
    import gen
    import oracle
    import sparse_dense_matrix_gb300 as sdm
    g = gen.rmat(scale=10, edge_factor=8, seed=3)
    B = gen.features(g.K, 8, seed=3)
    bounds = sdm.spmm_partition_rows(g.rowptr, world)
    b, e = bounds[rank], bounds[rank + 1]
    C, A, _ = oracle.spmm(g.rowptr, g.col, g.val, B, "max", rows=np.arange(b, e))
    parts = [None] * world
    dist.all_gather_object(parts, (bounds, b, e, C, A))
    if rank == 0:
        np.savez(os.path.join(out_dir, "shards.npz"),
                 bounds=np.array(bounds), C=np.concatenate([p[3] for p in parts]),
                 A=np.concatenate([p[4] for p in parts]),
                 same_bounds=np.array(all(p[0] == bounds for p in parts)))
    dist.barrier()
    dist.destroy_process_group()


def test_row_shards_cover_every_row_once_with_gloo(tmp_path):
    """Two workers split the rows of a skewed graph with the library's
    partitioner; their results, concatenated in rank order, are the whole
    product bit for bit (rows are independent, so no exchange is needed)."""
    import numpy as np
    sys.path.insert(0, ROOT)
    import __graft_entry__
    __graft_entry__.build()
    import gen
    import oracle
    mp.start_processes(_shard_main, args=(2, _free_port(), str(tmp_path)), nprocs=2,
                       start_method="spawn")
    r = np.load(tmp_path / "shards.npz")
    g = gen.rmat(scale=10, edge_factor=8, seed=3)
    B = gen.features(g.K, 8, seed=3)
    C, A, _ = oracle.spmm(g.rowptr, g.col, g.val, B, "max")
    assert bool(r["same_bounds"]) and r["bounds"][0] == 0 and r["bounds"][-1] == g.M
    assert 0 < r["bounds"][1] < g.M
    assert np.array_equal(r["C"].view(np.int32), C.view(np.int32))
    assert np.array_equal(r["A"], A)


def test_max_over_ranks_without_a_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(2.5, None) == 2.5


def test_reference_arm_under_torchrun_two_ranks():
    """Rank 0 prints one JSON line for the whole job; rank 1 exits 0 silently."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2", "--steps", "2",
           "--warmup", "1", "--config", "1", "--ref-budget", "2"]
    env = dict(os.environ, OMP_NUM_THREADS="2")
    p = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600, env=env)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [ln for ln in p.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, p.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["steps"] == 2
    assert d["value"] > 0 and d["unit"] == "GFLOP/s" and d["higher_is_better"] is True
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"
