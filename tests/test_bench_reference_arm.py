"""The benchmark's reference arm (the CPU oracle on the host cores) prints one
JSON line with the same metric, unit and workload as the GPU arm, and the keys
the benchmark's consumers read.  Runs on the CPU: one bounded sample."""
import json
import subprocess
import sys

from tests.conftest import ROOT

sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_reference_arm_line():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "1"],
                       cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    d = json.loads(r.stdout.strip().splitlines()[-1])
    assert d["impl"] == "reference"
    assert d["metric"] == bench.METRIC and d["unit"] == "us/layer-token"
    assert d["higher_is_better"] is False and d["n_gpus"] == 1
    assert d["steps"] == 1 and d["warmup"] == 1
    assert d["config"] == bench.workload_config(32768, 1)
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["sample"]
    assert cb["value"] == d["value"] > 0
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    # one step is one timed layer-token: no extrapolation between the two
    assert d["step"] == "one layer-token"
    assert abs(d["ms_per_step"] - d["value"] / 1e3) < 1e-6 * d["ms_per_step"]


def test_traffic_is_reported_only_for_the_captured_sources(monkeypatch):
    """The ncu traffic figure belongs to the kernel sources it was captured on:
    once their hash differs, the bench reports none."""
    cap = dict(bench.TRAFFIC_CAPTURE)
    monkeypatch.setattr(bench, "TRAFFIC_CAPTURE", dict(cap, sources_sha16=bench.sources_sha16()))
    assert bench.traffic_bytes(32768) == cap["bytes"][32768]
    monkeypatch.setattr(bench, "TRAFFIC_CAPTURE", dict(cap, sources_sha16="0" * 16))
    assert bench.traffic_bytes(32768) is None


def test_rows_summary_keeps_the_floats():
    rows = {"store": {"workload": "text", "us": 12.345678, "rows_per_s": 2.5e9, "cache_bytes": 123}}
    assert bench.rows_summary(rows) == {"store": {"us": 12.35, "rows_per_s": 2.5e9}}


class _Props:
    multi_processor_count = 152


class _Cuda:
    @staticmethod
    def get_device_properties(_):
        return _Props()


class _Torch:
    cuda = _Cuda()


def test_step_form_follows_the_decode_grid():
    """--step auto takes the single decode-step launch while the decode grid
    (512-key partitions x 4 KV heads) fits one wave of two CTAs per SM, as the
    library's choice of the warp-specialised kernel does, and the three
    launches beyond; the explicit forms are kept as given."""
    t = _Torch()
    assert bench.resolve_step(t, "auto", 32769) == "fused"  # 65 x 4 = 260 CTAs <= 304
    assert bench.resolve_step(t, "auto", 262145) == "separate"  # 513 x 4 = 2052
    assert bench.resolve_step(t, "auto", 76 * 512) == "fused"  # 304: one wave
    assert bench.resolve_step(t, "auto", 76 * 512 + 1) == "separate"
    assert bench.resolve_step(t, "separate", 32769) == "separate"
    assert bench.resolve_step(t, "fused", 262145) == "fused"
    assert bench.KERNELS_PER_LAYER == {"fused": 2, "separate": 3}
    assert "kvq_decode_step" in bench.workload_config(32768, 1, "fused")["step"]
    assert "kvq_store_rotate" in bench.workload_config(32768, 1, "separate")["step"]
