"""bench.py's JSON line: the keys and the consistency the benchmark contract asks
for, on the reference arm (the CPU oracle, no GPU) and on a small batch of the
library's arm (GPU)."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
BASE_KEYS = {"metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
             "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config"}


def run_bench(*args, timeout=900):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT,
                       capture_output=True, text=True, timeout=timeout)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    return json.loads(lines[0])


def test_reference_arm_line():
    d = run_bench("--impl", "reference", "--steps", "1", "--warmup", "3", "--ref-block", "256")
    assert BASE_KEYS <= set(d) and d["impl"] == "reference"
    assert d["unit"] == "GB/s" and d["higher_is_better"] is True and d["value"] > 0
    assert d["steps"] == 1 and d["warmup"] == 3 and d["n_gpus"] == 1
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] == 1 and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
    assert d["config"]["workload"] and d["config"]["tokens"] == 32768


def test_warmup_below_three_is_refused():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--warmup", "2"],
                       cwd=ROOT, capture_output=True, text=True, timeout=120)
    assert r.returncode != 0 and "warmup" in r.stderr


@pytest.mark.gpu
def test_library_arm_line():
    import __graft_entry__
    __graft_entry__.build()
    d = run_bench("--tokens", "2048", "--steps", "20", "--warmup", "3", "--cpu-seconds", "0.5")
    assert BASE_KEYS <= set(d) and "impl" not in d
    assert d["unit"] == "GB/s" and d["scaling"] == "weak" and d["vs_baseline"] is None
    assert d["steps"] == 20 and d["ms_per_step"] > 0 and d["value"] > 0
    roof = d["roofline"]
    assert roof["bound"] == "hbm" and roof["unit"] == "GB/s"
    assert abs(roof["frac"] - roof["achieved"] / roof["peak"]) < 1e-3
    assert "traffic" in roof
    assert roof["kernel"] in d["kernels"] and d["kernels"][roof["kernel"]]["gbs"] == roof["achieved"]
    e = d["e2e"]
    assert e["unit"] == "GB/s" and e["value"] > 0
    assert e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] > 0
    assert e["host_link"]["floor_ms_per_step"] > 0
    assert e["ms_per_step"] >= 0.5 * e["host_link"]["floor_ms_per_step"]
    clk = d["clocks"]
    assert {"sm_mhz", "sm_max_mhz", "reasons", "samples", "source"} <= set(clk)
    # clocks are read in-process through NVML every millisecond during the timed region
    assert clk["source"].startswith("NVML") and clk["samples"] >= 1
    assert abs(d["ms_per_step_x_sm_mhz"] - d["ms_per_step"] * clk["sm_mhz"]) < 1
    # 2048 tokens: one layout launch (the cluster kernel, or the cooperative one
    # when the cluster kernel is switched off) or three, then three data kernels
    single = os.environ.get("EP_GB300_LAYOUT_CLUSTER", "1") != "0" or \
        os.environ.get("EP_GB300_LAYOUT_FUSED", "1") != "0"
    assert d["gpu_launches"] == (4 if single else 6) * d["steps"]
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] == 1 and cb["value"] > 0 and cb["sample"]
    assert d["config"]["tokens"] == 2048
    # the decode workload measured beside the step (context for the small-batch shape)
    dw = d["decode_workload"]
    assert dw["workload"] == "decode" and dw["tokens"] == 1024
    for k in ("layout", "dispatch", "combine", "layout_dispatch", "step"):
        assert dw[k]["us_median"] > 0 and dw[k]["gbs"] > 0
    assert dw["layout"]["variant"].startswith("ep_layout_")
    ow = d["other_workloads"]
    assert set(ow) == {"tiny", "skewed"}
    for name, w in ow.items():
        assert w["workload"] == name and w["step"]["us_median"] > 0 and w["combine"]["gbs"] > 0


def test_mix_probe_kernels_compile(tmp_path):
    """The --mix-ceilings probe kernels build for sm_103a (nvcc cross-compiles
    without a GPU) and export the launchers bench.py calls."""
    import shutil
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("no nvcc")
    sys.path.insert(0, ROOT)
    import bench
    src, so = tmp_path / "mix_probe.cu", tmp_path / "mix_probe.so"
    src.write_text(bench.MIX_PROBE_CU)
    subprocess.check_call([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-shared",
                           "-Xcompiler", "-fPIC", "-o", str(so), str(src)], timeout=300)
    import ctypes
    lib = ctypes.CDLL(str(so))
    for name in ("mix_write", "mix_read", "mix_copy", "mix_bcast8", "mix_reduce8"):
        assert hasattr(lib, name)


@pytest.mark.gpu
def test_mix_ceilings_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--mix-ceilings",
                        "--steps", "2", "--warmup", "3"], cwd=ROOT, capture_output=True, text=True,
                       timeout=900)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-2000:]
    d = json.loads([l for l in r.stdout.splitlines() if l.startswith("{")][-1])
    assert set(d["cases"]) == {"write_only", "read_only", "copy_1to1", "bcast_1to8", "reduce_8to1"}
    for c in d["cases"].values():
        assert c["us_best"] > 0 and c["gbs_best"] >= c["gbs_median"] > 0


def test_traffic_record_is_scaled_and_tied_to_the_sources(tmp_path, monkeypatch):
    """The roofline's DRAM traffic comes from the committed ncu record only while
    the kernel's sources are the captured ones, and is scaled to the batch that
    ran (traffic grows with the tokens processed)."""
    sys.path.insert(0, ROOT)
    import bench
    rec = json.load(open(os.path.join(ROOT, "profiles", "ncu_traffic.json")))
    for name, k in rec["kernels"].items():
        full = bench.ncu_traffic(name)
        if full is None:      # sources changed since the capture: nothing to check
            continue
        assert full == k["dram_bytes_per_launch"]
        assert bench.ncu_traffic(name, bench.TRAFFIC_TOKENS // 2) == round(full / 2)
    # a record taken on other sources gives no traffic
    fake = dict(rec, kernels={n: dict(k, source_digest="0" * 16) for n, k in rec["kernels"].items()})
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "ncu_traffic.json").write_text(json.dumps(fake))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_source_digest", lambda kernel: "f" * 16)
    assert all(bench.ncu_traffic(n) is None for n in rec["kernels"])
