"""The reference arm of bench.py (the CPU oracle on the headline workload) runs on the host
alone: one short run prints one JSON line with the keys the benchmark contract asks for."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_contract_line():
    env = dict(os.environ)
    env.pop("WORLD_SIZE", None)
    p = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "0"],
                       cwd=ROOT, capture_output=True, text=True, timeout=600, env=env)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [l for l in p.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    j = json.loads(lines[0])
    assert j["impl"] == "reference" and j["value"] > 0 and j["higher_is_better"] is True
    assert j["metric"].startswith("hybrid attn decode req-tokens/s per layer")
    assert j["unit"] == "req-tokens/s per layer" and j["config"]["workload"].startswith("hybrid_32layer")
    assert j["cpu_baseline"]["kind"] == "oracle" and j["cpu_baseline"]["cores"] >= 1
    assert j["e2e"]["value"] == j["value"] and j["e2e"]["h2d_bytes_per_step"] == 0


def test_every_row_can_be_timed_alone():
    """`--workload` accepts the headline and every row (the default rows and the extra ones),
    so each can be run on its own, e.g. under a profiler."""
    sys.path.insert(0, ROOT)
    import bench
    argv = sys.argv
    try:
        for name in ["hybrid_32layer", *bench.ROWS, *bench.EXTRA_ROWS]:
            sys.argv = ["bench.py", "--workload", name]
            assert bench.parse().workload == name
    finally:
        sys.argv = argv
    assert set(bench.CPU_ROWS) <= set(bench.ROWS)
