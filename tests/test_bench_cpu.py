"""Host-side logic of bench.py (CPU only): the DRAM-traffic record is used
only for the kernel source it was captured from, and the oracle reference
arm prints the JSON line the measurement contract asks for."""

import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bench():
    sys.path.insert(0, ROOT)
    import bench as b
    return b


def test_blob_hash_matches_git(bench, tmp_path):
    p = tmp_path / "f.bin"
    p.write_bytes(b"nvfp4\x00\xff" * 100)
    try:
        want = subprocess.run(["git", "hash-object", str(p)], capture_output=True, text=True, check=True).stdout.strip()
    except (OSError, subprocess.CalledProcessError):
        pytest.skip("git not available")
    assert bench.git_blob_hash(str(p)) == want


def test_traffic_record_follows_the_kernel_source(bench, monkeypatch):
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        rec = json.load(f)[bench.GEMM_KERNEL][bench.WORKLOAD]
    src = os.path.join(ROOT, "nvfp4_w4a4_gemm_gb300", "csrc", "gemm.cu")
    if bench.git_blob_hash(src) == rec["gemm_cu_blob"]:
        assert bench.gemm_traffic() == rec["bytes"] == rec["dram_read"] + rec["dram_write"]
    else:
        assert bench.gemm_traffic() is None
    monkeypatch.setattr(bench, "git_blob_hash", lambda path: "0" * 40)
    assert bench.gemm_traffic() is None  # a changed kernel invalidates the counters


def test_reference_arm_json_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "1", "--cpu-rows", "128"], capture_output=True, text=True, cwd=ROOT,
                       timeout=600, env=dict(os.environ, WORLD_SIZE="1"))
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference"
    assert line["warmup"] >= 3 and line["steps"] == 1 and line["n_gpus"] == 1
    assert line["value"] > 0 and line["unit"] == "TFLOP/s" and line["higher_is_better"] is True
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and "sample" in cb and cb["value"] == line["value"]
    e2e = line["e2e"]
    assert e2e["value"] == line["value"] and e2e["unit"] == line["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0
    assert "workload" in line["config"]
