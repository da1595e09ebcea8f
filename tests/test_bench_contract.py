"""The benchmark's JSON line (CPU only): the reference arm, which times the
oracle on the host cores, runs here without a GPU and prints the one line
the measurement contract defines."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_contract_line():
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "tiny", "--steps", "1",
                          "--warmup", "0"], cwd=ROOT, capture_output=True, text=True, timeout=600, check=True)
    lines = [ln for ln in out.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    sys.path.insert(0, ROOT)
    import bench

    assert d["impl"] == "reference" and d["metric"] == bench.METRIC
    assert d["value"] > 0 and d["unit"] == "GB/s" and d["higher_is_better"] is True
    assert d["n_gpus"] == 1 and d["steps"] == 1 and d["warmup"] == 0 and d["ms_per_step"] > 0
    assert d["scaling"] == "weak" and d["vs_baseline"] is None and d["data"].startswith("synthetic")
    assert d["config"]["workload"] == "tiny_256x256_T4"
    cpu = d["cpu_baseline"]
    assert cpu["kind"] == "oracle" and cpu["cores"] >= 1 and cpu["sample"] and cpu["value"] == d["value"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_two_ranks_through_the_spawn_path():
    """--gpus 2 without a launcher relaunches the script under
    torch.distributed.run with two ranks; rank 0 alone prints the line."""
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "tiny", "--steps", "1",
                          "--warmup", "0", "--gpus", "2"], cwd=ROOT, capture_output=True, text=True, timeout=600,
                         check=True)
    lines = [ln for ln in out.stdout.splitlines() if ln.strip().startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["n_gpus"] == 2 and d["scaling"] == "strong" and d["impl"] == "reference"
    assert d["config"]["parallelism"].startswith("rows2")


def test_gpus_must_match_the_launcher(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench

    monkeypatch.setenv("WORLD_SIZE", "2")
    try:
        bench.main(["--gpus", "1", "--impl", "reference"])
    except SystemExit as e:
        assert "WORLD_SIZE" in str(e)
    else:
        raise AssertionError("a launcher/--gpus mismatch must fail")
