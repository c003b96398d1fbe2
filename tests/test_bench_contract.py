"""bench.py's JSON line keeps the contract the benchmark driver reads (CPU: the reference arm, which
times the fp64 oracle on the host cores)."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_contract_line():
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--config", "1", "--steps", "1",
                          "--warmup", "0"], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
              "vs_baseline", "dtype", "data", "config", "impl", "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference" and d["value"] > 0 and d["higher_is_better"] is True
    assert d["scaling"] == "weak" and d["vs_baseline"] is None
    assert d["config"]["workload"] and d["config"]["T"] == 4096
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0


def test_score_accounting_helpers():
    sys.path.insert(0, ROOT)
    import bench
    from synth import recipe
    w = recipe.workload(2)
    # S computed once: 2 d_k (n N - n(n-1)/2) per query head, one 32K request, n = 128
    n, N = 128, 32768
    assert bench.score_flops(w) == 2 * 128 * (n * N - n * (n - 1) // 2) * 32
    # K once plus the window rows of Q
    assert bench.score_input_bytes(w) == N * 8 * 128 * 2 + n * 32 * 128 * 2
