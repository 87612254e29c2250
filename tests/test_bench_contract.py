"""CPU checks of bench.py's output contract on its reference arm (the oracle
timed on the host cores, no GPU): one JSON line with the keys the contract
names, the reference arm's own cpu_baseline and e2e objects, and no output
from ranks other than 0."""
import json
import os
import subprocess
import sys

from helpers import ROOT

CMD = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "tiny", "--steps", "1",
       "--warmup", "0"]


def _run(extra_env=None):
    env = dict(os.environ)
    env.update(extra_env or {})
    return subprocess.run(CMD, cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)


def test_reference_arm_prints_one_contract_line():
    r = _run()
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference"
    assert d["n_gpus"] == 1 and d["steps"] == 1 and d["warmup"] == 0
    assert d["value"] > 0 and d["ms_per_step"] > 0 and d["higher_is_better"] is True
    assert "workload" in d["config"]
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["sample"] and cb["value"] == d["value"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_reference_arm_is_silent_on_other_ranks():
    r = _run({"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"})
    assert r.returncode == 0, r.stderr[-2000:]
    assert not [l for l in r.stdout.splitlines() if l.startswith("{")]


def _bench_module():
    import importlib.util
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_gemm_traffic_is_dropped_once_the_kernels_change(tmp_path):
    """The roofline's `traffic` comes from recorded ncu counters only while
    the GEMM sources still hash to the value recorded with them."""
    import hashlib
    import shutil
    bench = _bench_module()
    root = tmp_path / "repo"
    csrc = root / "grouped_gemm_top_gb300" / "csrc"
    shutil.copytree(os.path.join(ROOT, "grouped_gemm_top_gb300", "csrc"), csrc)
    h = hashlib.sha256()
    for fn in ["common.cuh", "gemm_common.cuh", "gemm.cu", "gemm2sm.cu"]:
        h.update((csrc / fn).read_bytes())
    (root / "profiles").mkdir()
    rec = {"kernel_source_hash": h.hexdigest()[:16], "gemm_launches": [{"dram_read": 1.0, "dram_write": 2.0}] * 6}
    (root / "profiles" / "gemm_traffic.json").write_text(json.dumps(rec))
    bench.ROOT = str(root)
    assert bench._gemm_traffic() == rec["gemm_launches"]
    with open(csrc / "gemm.cu", "a") as f:
        f.write("\n// edited\n")
    assert bench._gemm_traffic() is None


def test_peaks_fall_back_when_the_measured_file_is_absent(tmp_path):
    bench = _bench_module()
    bench.ROOT = str(tmp_path)
    peaks, src = bench._peaks()
    assert src == "fallback" and peaks["hbm_gbs"] == 6800.0 and peaks["bf16_tflops"] == 1900.0
