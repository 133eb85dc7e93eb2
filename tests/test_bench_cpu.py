"""bench.py's output contract on the host (no GPU): the reference arm (the fp64 oracle
timed on the host cores) prints one JSON line with the GPU arm's metric, unit and config
and the keys the contract names; the GPU arm, with no device, fails instead of falling
back to the CPU."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(*args, timeout=300):
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT,
                          capture_output=True, text=True, timeout=timeout)


def test_reference_arm_json_line():
    r = _run("--impl", "reference", "--steps", "2", "--warmup", "3")
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    assert d["metric"] == "KDA decode state-bytes GB/s" and d["unit"] == "GB/s"
    assert d["higher_is_better"] is True and d["n_gpus"] == 1
    assert d["steps"] == 2 and d["warmup"] == 3
    assert d["value"] > 0 and d["ms_per_step"] > 0
    assert d["data"] == "synthetic" and d["dtype"] == "f64"
    assert "serving decode" in d["config"]["workload"]
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    e = d["e2e"]
    assert e["value"] == d["value"] and e["unit"] == d["unit"]
    assert e["h2d_bytes_per_step"] == 0 and e["d2h_bytes_per_step"] == 0


def test_gpu_arm_fails_without_a_device():
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    r = _run("--steps", "2", "--warmup", "3", "--no-cpu-baseline", "--no-secondary")
    assert r.returncode != 0
    assert not [ln for ln in r.stdout.splitlines() if ln.startswith("{") and '"value"' in ln]


def test_traffic_records_match_the_keys_and_sources_the_bench_reads():
    """profiles/traffic.json holds one record per DRAM-traffic figure bench.py reports, keyed
    as bench.py looks it up, with the per-launch bytes equal to read + write. A record whose
    source hash no longer matches is reported as null by the bench; here each is checked to
    carry a hash of the right form and the capture command that produced it."""
    sys.path.insert(0, ROOT)
    import bench
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        d = json.load(f)
    src = open(os.path.join(ROOT, "bench.py")).read()
    for key in ("decode_kernel<128,128> serving_decode",
                "prefill (prep_kernel + chain_kernel) chunked_prefill"):
        assert f'ncu_traffic("{key}"' in src, key
        e = d[key]
        assert len(e["source_sha"]) == 16 and "ncu" in e["capture"] and "--clock-control none" in e["capture"]
        assert e["dram_bytes_per_launch"] > 0
    dec = d["decode_kernel<128,128> serving_decode"]
    assert dec["dram_bytes_per_launch"] == dec["dram_read_bytes"] + dec["dram_write_bytes"]
    pf = d["prefill (prep_kernel + chain_kernel) chunked_prefill"]
    parts = [pf[k] for k in ("prep_kernel", "prep_kernel_marked_pass", "chain_kernel")]
    assert pf["dram_bytes_per_launch"] == sum(p["dram_read_bytes"] + p["dram_write_bytes"] for p in parts)
    # a record is reported only for the source it was taken on
    assert bench.ncu_traffic("decode_kernel<128,128> serving_decode", "0" * 16) is None
