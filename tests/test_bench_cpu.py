"""The benchmark's JSON line, checked through its reference arm (the CPU oracle).

The reference arm needs no GPU, so its output contract can be checked here:
one JSON line with the keys the benchmark promises, and, under a multi-process
launch, nothing at all from ranks other than 0.
"""
import json
import os
import subprocess
import sys

REPO = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
KEYS = {"impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
        "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
        "cpu_baseline", "e2e"}


def run_bench(*args, env=None):
    e = dict(os.environ)
    e.update(env or {})
    return subprocess.run([sys.executable, "bench.py", *args], cwd=REPO, env=e,
                          capture_output=True, text=True, timeout=300)


def test_reference_arm_prints_one_complete_json_line():
    r = run_bench("--impl", "reference", "--workload", "tiny_mha", "--steps", "3", "--warmup", "3",
                  env={"RANK": "0", "WORLD_SIZE": "1"})
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert KEYS <= set(d), KEYS - set(d)
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["value"] > 0
    assert d["steps"] == 3 and d["warmup"] == 3 and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["config"]["workload"].startswith("tiny")


def test_reference_arm_other_ranks_print_nothing():
    r = run_bench("--impl", "reference", "--workload", "tiny_mha", "--steps", "3", "--warmup", "3",
                  env={"RANK": "1", "WORLD_SIZE": "2"})
    assert r.returncode == 0, r.stderr[-2000:]
    assert not [ln for ln in r.stdout.splitlines() if ln.startswith("{")]


def test_traffic_record_matches_the_kernel_source():
    """bench.py reports DRAM traffic from a committed ncu record only while the
    record's hash matches the kernel source; a kernel edit must re-take it."""
    sys.path.insert(0, REPO)
    import bench

    for workload, whiches in (("mla78_dsa", ("backup_all_layers", "load_burst_signalling")),
                              ("llama3_8b_mha", ("backup_all_layers", "load_one_layer",
                                                 "load_burst_signalling"))):
        for which in whiches:
            t = bench.traffic_per_launch(workload, which, 1 << 30)
            assert t is not None, \
                f"{workload} {which}: the record does not match csrc/row_copy_kernel.cuh"
            assert (1 << 30) * 0.95 < t < (1 << 30) * 1.05 or which != "backup_all_layers"
    # a launch or workload the record does not hold has no traffic figure
    assert bench.traffic_per_launch("mla78_dsa", "load_one_layer", 1 << 30) is None
    assert bench.traffic_per_launch("mla78_dsa:page_first", "backup_all_layers", 1 << 30) is None
