"""Host-side arithmetic and output of bench.py (CPU only): the decode
launch's algorithmic bytes, the traffic taken from a committed profile only
while its kernel source is unchanged, the clock summary's throttle reasons,
and the reference arm's JSON line."""
import hashlib
import io
import json
import types
from contextlib import redirect_stdout

import numpy as np

import bench
from gated_delta_rule_gateddeltanet_gb300 import workloads as wl


def test_decode_bytes_equal_the_arrays_one_step_moves():
    """The decode roofline's bytes: the FP32 state read and written once, the
    q, k, v inputs and the output (v-shaped) in FP16, raw a and b in FP32,
    counted here from the decode workload's own arrays."""
    inp = wl.decode_step()
    Hk, Hv, dk, dv = inp.dims
    assert inp.q.dtype == np.float16 and inp.initial_state.dtype == np.float32
    state = 2 * inp.initial_state.nbytes
    io_bytes = inp.q.nbytes + inp.k.nbytes + 2 * inp.v.nbytes + inp.a.nbytes + inp.b.nbytes
    assert bench.decode_bytes_per_launch(inp.B, Hk, Hv, dk, dv) == state + io_bytes
    assert state + io_bytes == 404_774_912


def _profile(root, name, sha, traffic):
    (root / "profiles").mkdir(exist_ok=True)
    (root / "profiles" / name).write_text(f"# k\nsource_sha256: {sha}\n\ntraffic_bytes_per_launch: {traffic}\n")


def test_traffic_only_while_the_kernel_source_is_unchanged(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    src = tmp_path / "k.cu"
    src.write_text("__global__ void k() {}\n")
    sha = hashlib.sha256(src.read_bytes()).hexdigest()
    _profile(tmp_path, "k.md", sha, 123456)
    assert bench.recorded_traffic(str(src), "k.md") == 123456.0
    src.write_text("__global__ void k() { }\n")      # the kernel changed since the capture
    assert bench.recorded_traffic(str(src), "k.md") is None
    assert bench.recorded_traffic(str(src), "absent.md") is None


def test_committed_profiles_name_a_source_and_traffic():
    """Every committed summary that feeds a roofline carries both fields the
    bench reads (whether the hashes are current is the bench's concern)."""
    import re
    for name in ("decode_step.recurrent_kernel.ncu.md", "varlen_prefill.wy_kernels.ncu.md"):
        text = open(f"{bench.ROOT}/profiles/{name}").read()
        assert re.search(r"source_sha256:\s*[0-9a-f]{64}", text), name
        assert re.search(r"traffic_bytes_per_launch:\s*[0-9]+", text), name


def test_clock_summary_reports_throttle_reasons():
    lines = [
        "0, 2070, 2070, 900.1, 0x0, Not Active, Not Active, Not Active, Not Active\n",
        "0, 2055, 2070, 1100.0, 0x4, Not Active, Not Active, Not Active, Active\n",
        "0, 1800, 2070, 1300.0, 0x8, Active, Not Active, Not Active, Not Active\n",
        "garbage line\n",
        "0, [N/A], 2070, 1.0, 0x0, Not Active, Not Active, Not Active, Not Active\n",
    ]
    c = bench.ClockSampler.summarise(lines)
    assert c["samples"] == 3
    assert c["sm_mhz"] == 2055 and c["sm_max_mhz"] == 2070
    assert c["reasons"] == ["hw_slowdown", "sw_power_cap"]
    assert bench.ClockSampler.summarise([])["sm_mhz"] is None


def test_reference_arm_prints_one_contract_line(monkeypatch):
    monkeypatch.setattr(bench, "REFERENCE_BUDGET_S", 2.0)
    args = types.SimpleNamespace(gpus=1, steps=1, warmup=1)
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.run_reference(args, types.SimpleNamespace(rank=0))
    lines = [ln for ln in buf.getvalue().splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == "tokens/s"
    assert d["value"] > 0 and d["higher_is_better"] is True and d["steps"] == 1 and d["warmup"] == 1
    # the same config object as the GPU arm's line
    assert d["config"] == bench.workload_config(64, 16, 48, 128, 128, 1)
    assert d["config"]["workload"] == bench.WORKLOAD
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1 and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    # other ranks print nothing
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.run_reference(args, types.SimpleNamespace(rank=1))
    assert buf.getvalue() == ""


def test_clock_sampler_reads_its_process_output(tmp_path, monkeypatch):
    """The sampler's own start / stop path, with a stand-in for nvidia-smi
    that prints two samples and then waits to be stopped."""
    fake = tmp_path / "nvidia-smi"
    fake.write_text("#!/bin/sh\n"
                    "echo '0, 2070, 2070, 800.0, 0x0, Not Active, Not Active, Not Active, Not Active'\n"
                    "echo '0, 2040, 2070, 900.0, 0x4, Not Active, Not Active, Not Active, Active'\n"
                    "exec sleep 30\n")
    fake.chmod(0o755)
    monkeypatch.setattr(bench.shutil, "which", lambda name: str(fake))
    s = bench.ClockSampler()
    import time
    time.sleep(0.5)
    c = s.stop()
    assert c["samples"] == 2 and c["sm_mhz"] == 2055 and c["reasons"] == ["sw_power_cap"]
    monkeypatch.setattr(bench.shutil, "which", lambda name: None)
    assert bench.ClockSampler().stop() is None


def test_only_names_every_sub_measurement():
    """--only accepts exactly the sub-measurements the full run reports."""
    import inspect
    import re
    src = inspect.getsource(bench.run_gdn)
    reported = set(re.findall(r'extra\["(\w+)"\]', src))
    assert reported == set(bench.SUB_MEASUREMENTS)
    for name, fn in bench.SUB_MEASUREMENTS.items():
        assert (len(inspect.signature(fn).parameters) == 4) == (name in bench.NEEDS_LIB), name
