"""The benchmark's reference arm on CPU: `bench.py --impl reference` times the
fp64 oracle on the host cores and prints one JSON line of the benchmark's
contract; under a multi-rank launch only rank 0 works and prints.  No GPU."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(env_extra):
    env = dict(os.environ, **env_extra)
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1",
                        "--warmup", "0"], cwd=ROOT, env=env, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-2000:]
    return [json.loads(l) for l in r.stdout.splitlines() if l.startswith("{")]


def test_reference_arm_prints_one_contract_line():
    lines = _run({"RANK": "0", "WORLD_SIZE": "1", "LOCAL_RANK": "0"})
    assert len(lines) == 1
    d = lines[0]
    assert d["impl"] == "reference"
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["metric"] == "csa_decode_queries_per_s" and d["unit"] == "queries/s"
    assert d["value"] > 0 and d["steps"] == 1 and d["warmup"] == 0 and d["n_gpus"] == 1
    assert d["higher_is_better"] is True
    assert d["config"]["workload"] == "long_ragged_b64"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1 and cb["sample"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_reference_arm_other_ranks_exit_quietly():
    assert _run({"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"}) == []
    lines = _run({"RANK": "0", "WORLD_SIZE": "2", "LOCAL_RANK": "0"})
    assert len(lines) == 1 and lines[0]["n_gpus"] == 2


def test_e2e_groups_cover_every_step_once():
    # the end-to-end loop's group plan: exactly n steps, no group empty or
    # above G, one step first and last (so one upload precedes the first
    # kernels and one read-back follows the last)
    sys.path.insert(0, ROOT)
    import bench
    for G in (1, 4, 8):
        for n in range(0, 41):
            g = bench.e2e_group_sizes(n, G)
            assert sum(g) == n and all(1 <= x <= G for x in g), (n, G, g)
            if n >= 2:
                assert g[0] == 1 and g[-1] == 1
