"""Host-side pieces of bench.py that need no GPU: run selection and the
roofline numerator (compulsory bytes) on the 2k-row Erdos-Renyi workload."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def test_run_selection():
    import bench
    spec, g, runs = bench.workload(1)
    assert runs == [(32, "sum"), (32, "mean"), (32, "max")] and g.M == g.K == 2048
    spec, g, runs = bench.workload(1, "32", "max")
    assert runs == [(32, "max")] and list(spec["N"]) == [32] and list(spec["reduce"]) == ["max"]
    with pytest.raises(SystemExit):
        bench.workload(1, "7", None)           # not one of the workload's widths
    with pytest.raises(SystemExit):
        bench.workload(1, None, "min")


def test_compulsory_bytes_by_hand():
    import bench
    _, g, _ = bench.workload(1)
    assert g.nnz == 16384 and g.val is not None
    # rowptr 4 * 2049, col + val 8 * 16384, B 4 * 2048 * 32, C 4 * 2048 * 32
    assert bench.compulsory_bytes(g, 32, "sum") == 8196 + 131072 + 262144 + 262144
    assert bench.compulsory_bytes(g, 32, "max") == 8196 + 131072 + 3 * 262144   # + argmax


def test_default_workload_is_the_largest(monkeypatch):
    """With no flags the bench times the 4M-row Chung-Lu workload at N = 16,
    64 and 256 with sum, mean and max (no graph is generated here)."""
    import bench
    import gen
    monkeypatch.setattr(sys, "argv", ["bench.py"])
    args = bench.parse()
    assert args.config == 5 and args.gpus == 1 and args.warmup >= 3
    assert gen.CONFIGS[5]["name"] == "chung_lu_4M"
    assert bench.DEFAULT_N[5] == (16, 64, 256)
    assert set(gen.CONFIGS[5]["reduce"]) == {"sum", "mean", "max"}


def test_traffic_key_ignores_comments_only():
    """The DRAM traffic recorded for a kernel build stays valid across comment
    and layout edits, and no longer applies once the code changes."""
    import bench
    a = 'int a; // one\n/* two */ asm("x // y");\nchar c = \'"\';'
    b = 'int   a;\n\n asm("x // y"); // other\nchar c = \'"\'; /* */'
    assert bench._code_only(a) == bench._code_only(b) == 'int a; asm("x // y"); char c = \'"\';'
    assert bench._code_only(a) != bench._code_only(a.replace("int a", "int b"))
    for key, ent in bench.NCU_TRAFFIC.items():
        assert len(ent["sources_sha256"]) == 64 and ent["bytes"] > 0
