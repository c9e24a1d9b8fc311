"""The reference arm of bench.py (CPU only): `--impl reference` times the fp64
oracle on the host cores and prints one JSON line of the bench contract."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_contract_line():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "3"],
                       cwd=ROOT, capture_output=True, text=True, timeout=300, check=True)
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "tokens/s" and d["value"] > 0
    assert d["higher_is_better"] is True and d["n_gpus"] == 1 and d["warmup"] >= 3
    assert d["config"]["workload"] == "glm_decode_t4096" and d["dtype"] == "f64"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_ncu_traffic_goes_stale_with_its_kernel_sources(monkeypatch):
    """A stored ncu traffic figure is reported only while the sources of its
    kernel are the ones it was captured on."""
    sys.path.insert(0, ROOT)
    import bench
    key = ("glm_decode_t4096", "attention")
    monkeypatch.setattr(bench, "NCU_TRAFFIC", {key: (4887552, bench.kernel_digest("attention"))})
    assert bench.ncu_traffic(*key) == 4887552
    monkeypatch.setattr(bench, "NCU_TRAFFIC", {key: (4887552, "0" * 16)})
    assert bench.ncu_traffic(*key) is None
    assert bench.ncu_traffic("glm_decode_t4096", "no_such_kernel") is None
    # every kernel the bench times has its sources listed, and they exist
    for k, files in bench.KERNEL_SOURCES.items():
        for f in files + bench.SHARED_SOURCES:
            assert os.path.exists(os.path.join(ROOT, "mla_latent_kv_06_gb300", "csrc", f)), (k, f)
