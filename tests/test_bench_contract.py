"""CPU check of bench.py's output contract on its reference arm (the oracle timed on the
host cores), run as the driver runs it, on the tiny workload: one JSON line with the
keys and types the contract names."""

import json
import pathlib
import subprocess
import sys

ROOT = pathlib.Path(__file__).resolve().parent.parent


def _line(*args):
    out = subprocess.run([sys.executable, str(ROOT / "bench.py"), *args], cwd=ROOT, capture_output=True, text=True,
                         timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, out.stdout
    return json.loads(lines[0])


def test_reference_arm_prints_one_contract_line():
    d = _line("--impl", "reference", "--config", "tiny", "--steps", "2", "--warmup", "3")
    assert d["impl"] == "reference"
    for k in ("metric", "unit", "data", "scaling", "dtype"):
        assert isinstance(d[k], str) and d[k], k
    assert d["value"] > 0 and d["ms_per_step"] > 0
    assert d["n_gpus"] == 1 and d["steps"] == 2 and d["warmup"] == 3
    assert d["higher_is_better"] is True and d["vs_baseline"] is None
    assert d["config"]["workload"] == "tiny"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["sample"] and cb["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_warmup_is_at_least_three():
    d = _line("--impl", "reference", "--config", "tiny", "--steps", "1", "--warmup", "1")
    assert d["warmup"] == 3


def test_reference_arm_config_is_the_gpu_arms_config():
    """Both arms print the same `config` object for a workload (the GPU arm builds it with
    the same function and adds nothing to it), so the driver can pair the two lines."""
    sys.path.insert(0, str(ROOT))
    import bench
    import synthetic
    d = _line("--impl", "reference", "--config", "tiny", "--steps", "1", "--warmup", "3")
    assert d["config"] == bench.workload_config(synthetic.WORKLOADS["tiny"], 1)
    assert bench.DEFAULT_CONFIG == "qwen3-8b-b1"
