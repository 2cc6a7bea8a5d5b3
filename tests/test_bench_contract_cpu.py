"""bench.py's reference arm (the CPU oracle on the host cores) runs without a
GPU: run it from the command line, with a tiny step count, and check that its one
JSON line carries every key of the bench contract with the reference arm's
additions (impl, cpu_baseline describing the run, an e2e with no transfers)."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_json_line_has_the_contract_keys():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "0"],
                       cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "impl", "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference" and d["value"] > 0 and d["steps"] == 1 and d["warmup"] == 0
    assert d["higher_is_better"] is True and d["config"]["workload"] == "lm_head_q4_0_248320x2048"
    # the GPU arm prints the same config dict for its headline
    sys.path.insert(0, ROOT)
    import bench
    from gguf_block_quant_gb300 import synth
    assert d["config"] == bench.headline_config(synth.LM_HEAD_Q4_0, bench.LM_HEAD_COPIES)
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0
