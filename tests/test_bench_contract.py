"""bench.py's reference arm (the oracle, as it stands, on the host cores)
prints one JSON line with the benchmark contract's keys; under N > 1 only
rank 0 runs and prints, the other ranks exit 0 without work."""

import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(**env_extra):
    env = dict(os.environ, **env_extra)
    return subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "0"],
                          cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)


def test_reference_arm_prints_the_contract_line():
    r = _run()
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    line = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference"
    assert line["n_gpus"] == 1 and line["steps"] == 1 and line["warmup"] == 0
    assert line["value"] > 0 and line["ms_per_step"] > 0
    assert line["higher_is_better"] is True
    assert isinstance(line["config"], dict) and "workload" in line["config"]
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["sample"]
    assert cb["value"] == line["value"] and cb["unit"] == line["unit"]
    e2e = line["e2e"]
    assert e2e["value"] == line["value"] and e2e["unit"] == line["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_reference_arm_other_ranks_exit_without_output():
    r = _run(RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""


def test_multi_query_kernel_names_follow_the_dispatch():
    sys.path.insert(0, ROOT)
    import bench
    # verify (6 queries x G 4 = 24 rows): the balanced split with 3 row tiles
    assert bench.mq_kernel_name(True, 128, 4, 6).startswith("multi_query_balanced_kernel<bf16, 128, 3>")
    # a 512-token slice at head dim 128: the tcgen05 kernel
    assert bench.mq_kernel_name(False, 128, 4, 512).startswith("prefill_tc_kernel")
    # 64 rows or fewer, head dim 64 or G outside {1, 2, 4, 8}: the one-pass tiles
    assert bench.mq_kernel_name(False, 128, 4, 16) == "multi_query_kernel<bf16, 128, 2> (mma.sync)"
    assert bench.mq_kernel_name(False, 64, 4, 512) == "multi_query_kernel<bf16, 64, 2> (mma.sync)"
    assert bench.mq_kernel_name(False, 128, 2, 4) == "multi_query_kernel<bf16, 128, 1> (mma.sync)"
    assert bench.mq_kernel_name(False, 128, 3, 512).startswith("multi_query_kernel")
