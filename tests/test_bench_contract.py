"""The benchmark's own checks: the algorithmic byte counts against the
formulas written out independently here, and (on a GPU) the JSON line's
schema for both arms."""

import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


@pytest.mark.parametrize("N,H,e,ew", [(8192, 1024, 2, 2), (8192, 5120, 2, 4), (64, 256, 4, 4), (3, 7, 2, 2)])
def test_algorithmic_bytes(N, H, e, ew):
    row = N * H * e   # one pass over a row tensor
    want = {
        "ln_fwd": 2 * row + 2 * H * ew + 8 * N,          # x in, y out, gamma+beta, mean+rstd
        "rms_fwd": 2 * row + H * ew + 4 * N,             # x in, y out, gamma, rstd
        "fused_fwd": 4 * row + H * ew + 4 * N,           # x, res in; h, y out; gamma; rstd
        "ln_bwd": 3 * row + 3 * H * ew + 8 * N,          # x, dy in; dx out; gamma in; dgamma, dbeta out
        "rms_bwd": 3 * row + 2 * H * ew + 4 * N,
        "fused_bwd": 5 * row + 2 * H * ew + 4 * N,       # dy, h, stream grad in; dx, dres out
        "ln_bwd_y": 3 * row + 4 * H * ew + 4 * N,        # y instead of x, beta read, no mean
        "rms_bwd_y": 3 * row + 2 * H * ew + 4 * N,
        "fused_fwd_ip": 4 * row + H * ew + 4 * N,
    }
    for op, v in want.items():
        assert bench.alg_bytes(op, N, H, e, ew) == v, op
    assert set(bench.LAUNCHES) >= set(bench.OPS) | set(bench.EXTRA_OPS)


REQUIRED = {"metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
            "vs_baseline", "dtype", "data", "config", "roofline", "cpu_baseline", "e2e", "gpu_launches", "clocks"}


def _json_line(out):
    lines = [ln for ln in out.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, out[-2000:]
    return json.loads(lines[0])


@pytest.mark.gpu
@pytest.mark.slow
def test_bench_json_line():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    p = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--steps", "3", "--warmup", "3",
                        "--e2e-steps", "1", "--cpu-seconds", "0.5", "--cpu-rows", "16"],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert p.returncode == 0, p.stderr[-3000:]
    j = _json_line(p.stdout)
    assert REQUIRED <= set(j), REQUIRED - set(j)
    assert j["value"] > 0 and j["ms_per_step"] > 0 and j["n_gpus"] == 1 and j["steps"] == 3 and j["warmup"] == 3
    assert j["higher_is_better"] is True and j["vs_baseline"] is None and j["config"]["workload"]
    r = j["roofline"]
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["achieved"] > 0 and r["peak"] > 0
    assert abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-2
    c = j["cpu_baseline"]
    assert c["kind"] == "oracle" and c["value"] > 0 and c["cores"] >= 1 and c["sample"]
    e = j["e2e"]
    assert e["value"] > 0 and e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] > 0
    assert j["gpu_launches"] > 0
    assert "sm_mhz" in j["clocks"] and "reasons" in j["clocks"]


def test_reference_arm_json_line():
    # the reference arm times the oracle on the host cores: no GPU involved
    p = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "2",
                        "--warmup", "3", "--ref-rows", "8"], capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert p.returncode == 0, p.stderr[-3000:]
    j = _json_line(p.stdout)
    assert j["impl"] == "reference" and j["value"] > 0 and j["ms_per_step"] > 0
    assert j["n_gpus"] == 1 and j["steps"] == 2 and j["warmup"] == 3
    assert j["higher_is_better"] is True and j["vs_baseline"] is None and j["config"]["workload"]
    assert j["unit"] == "GB/s" and j["metric"]
    assert j["e2e"]["value"] == j["value"] and j["e2e"]["unit"] == j["unit"]
    assert j["e2e"]["h2d_bytes_per_step"] == 0 and j["e2e"]["d2h_bytes_per_step"] == 0
    c = j["cpu_baseline"]
    assert c["kind"] == "oracle" and c["value"] == j["value"] and c["cores"] >= 1 and c["sample"]


def test_cpu_baseline_on_host_cores(monkeypatch):
    # the CUDA arm's cpu_baseline leg: the oracle on one core, then one spawned
    # process per core (two here, to keep the test short)
    from types import SimpleNamespace
    monkeypatch.setattr(os, "cpu_count", lambda: 2)
    c = bench.cpu_baseline(SimpleNamespace(cpu_seconds=0.2, cpu_rows=8))
    assert c["kind"] == "oracle" and c["unit"] == "GB/s" and c["cores"] == 2 and c["sample"]
    assert c["value"] > 0 and c["single_core"]["value"] > 0 and c["single_core"]["cores"] == 1
    assert c["value"] > 0.5 * c["single_core"]["value"]


def test_record_traffic_sums_launches_in_base_units(tmp_path):
    """The traffic table is computed from ncu's raw CSV (units row honoured,
    every captured launch of the call summed) and stamped with the digest of
    the kernel sources, which is what makes bench.py report it."""
    csv = tmp_path / "traffic_ln_bwd_8192x5120.csv"
    csv.write_text('"ID","Kernel Name","dram__bytes_read.sum","dram__bytes_write.sum"\n'
                   '"","","Mbyte","Kbyte"\n'
                   '"0","main","167.90","36700.5"\n'
                   '"1","reduce","12.5","0"\n')
    csv2 = tmp_path / "traffic_ln_fwd_8192x1024.csv"
    csv2.write_text('"ID","Kernel Name","dram__bytes_read.sum","dram__bytes_write.sum"\n'
                    '"","","byte","byte"\n'
                    '"0","fwd","16777216","1000"\n')
    out = tmp_path / "roofline_traffic.txt"
    rows = bench.record_traffic([str(csv), str(csv2)], str(out))
    assert rows["ln_bwd_8192x5120"] == (int(167.9e6 + 36700.5e3 + 12.5e6), 2)
    assert rows["ln_fwd_8192x1024"] == (16777216 + 1000, 1)
    kv = dict(line.strip().split("=", 1) for line in out.read_text().splitlines() if "=" in line and
              not line.startswith("#"))
    assert kv["src_digest"] == bench.src_digest()
    assert int(kv["ln_bwd_8192x5120"]) == rows["ln_bwd_8192x5120"][0]
    with pytest.raises(ValueError):
        bench.record_traffic([str(tmp_path / "other.csv")], str(out))
