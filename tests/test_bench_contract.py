"""bench.py's host side on the CPU: the reference arm's JSON line and the
clock-sample summary (no GPU; the GPU arm is exercised by the GPU runs)."""
import datetime
import importlib.util
import json
import os
import subprocess
import sys
import time

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def load_bench():
    spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_reference_arm_prints_one_contract_line():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "tiny_4k",
                        "--steps", "3", "--warmup", "3"], cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference"
    assert d["steps"] == 3 and d["warmup"] == 3 and d["n_gpus"] == 1
    assert d["higher_is_better"] is False and d["value"] > 0
    assert d["config"]["workload"] == "tiny_4k"
    bench = load_bench()
    from speculative_decoding_attention_gb300 import workloads
    # the same config keys and values as the GPU arm reports for this workload
    assert d["config"] == bench.workload_config(workloads.get("tiny_4k"), 1, None, 1)
    cb = d["cpu_baseline"]
    assert cb["sample"].startswith("3 whole steps")
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1 and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def write_samples(path, t0, rows):
    with open(path, "w") as f:
        for k, (mhz, reasons) in enumerate(rows):
            ts = datetime.datetime.fromtimestamp(t0 + 0.02 * k).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
            flags = ["Active" if r else "Not Active" for r in reasons]
            f.write(f"{ts}, {mhz}, 2070, 900.0, 0x0, " + ", ".join(flags) + "\n")


def test_clock_summary_counts_samples_in_the_timed_region(tmp_path):
    bench = load_bench()
    clk = bench.ClockSampler(torch.device("cpu"))
    clk.path = str(tmp_path / "clocks.csv")
    clk.interval_ms = 20
    t0, m0 = time.time(), time.monotonic()
    quiet = (False, False, False, False)
    write_samples(clk.path, t0, [(2070, quiet)] * 3 + [(2055, quiet)] * 4 + [(2070, quiet)] * 2)
    clk.mark(m0 + 0.05, m0 + 0.13)  # samples 3..6 (the summary maps the wall-clock stamps to monotonic time)
    s = clk.summary()
    assert s["samples"] == 9 and s["samples_in_timed_region"] == 4
    assert s["sm_mhz"] == 2070 and s["sm_max_mhz"] == 2070 and s["reasons"] == []
    assert not os.path.exists(clk.path)  # the summary removes its scratch file


@pytest.mark.parametrize("which,name", [(0, "hw_slowdown"), (1, "hw_thermal_slowdown"),
                                        (2, "sw_thermal_slowdown"), (3, "sw_power_cap")])
def test_clock_summary_names_each_throttle_reason(tmp_path, which, name):
    bench = load_bench()
    clk = bench.ClockSampler(torch.device("cpu"))
    clk.path = str(tmp_path / "clocks.csv")
    clk.interval_ms = 20
    flags = tuple(i == which for i in range(4))
    write_samples(clk.path, time.time(), [(2070, (False,) * 4), (1800, flags)])
    assert clk.summary()["reasons"] == [name]


def test_clock_summary_without_samples(tmp_path):
    bench = load_bench()
    clk = bench.ClockSampler(torch.device("cpu"))
    clk.path = str(tmp_path / "missing.csv")
    assert clk.summary() == {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}


def test_reference_arm_under_two_ranks():
    """Under torchrun with two ranks only rank 0 prints (one line), and it runs
    the oracle on every host core even though the launcher caps OpenMP
    threads per rank."""
    import socket

    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    r = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
                        "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl", "reference",
                        "--workload", "tiny_4k", "--gpus", "2", "--steps", "3", "--warmup", "3"],
                       cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip().startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2
    assert d["cpu_baseline"]["cores"] == len(os.sched_getaffinity(0))


def test_packed_buffers_are_aligned_views():
    bench = load_bench()
    buf, views = bench._packed([("a", (3, 1, 16, 256), torch.bfloat16), ("l", (3, 1, 16), torch.float32),
                                ("c", (1, 4, 16, 256), torch.bfloat16)], torch.device("cpu"), pinned=False)
    base = buf.data_ptr()
    for name, t in views.items():
        assert t.is_contiguous() and (t.data_ptr() - base) % 256 == 0
    # the views do not overlap and stay inside the buffer
    ends = sorted((t.data_ptr() - base, t.data_ptr() - base + t.numel() * t.element_size()) for t in views.values())
    assert all(a[1] <= b[0] for a, b in zip(ends, ends[1:])) and ends[-1][1] <= buf.numel()


def test_nvml_samples_and_reason_bits(tmp_path):
    """The NVML sampler's rows: monotonic time, SM MHz, max MHz, reason bits."""
    bench = load_bench()
    clk = bench.ClockSampler(torch.device("cpu"))
    clk.path = str(tmp_path / "nvml.csv")
    clk.source, clk.interval_ms = "nvml", 0.5
    m0 = time.monotonic()
    rows = [(m0 + 0.0005 * k, 2070, 2070, 0) for k in range(20)]
    rows[7] = (rows[7][0], 1950, 2070, 0x4)      # sw_power_cap
    rows[15] = (rows[15][0], 1500, 2070, 0x8 | 0x40)  # hw_slowdown, hw_thermal_slowdown
    with open(clk.path, "w") as f:
        for r in rows:
            f.write(f"{r[0]:.6f},{r[1]},{r[2]},{r[3]}\n")
    clk.mark(m0 + 0.0026, m0 + 0.0061)  # samples 6..12
    s = clk.summary()
    assert s["samples"] == 20 and s["samples_in_timed_region"] == 7 and s["source"] == "nvml"
    assert s["reasons"] == ["hw_slowdown", "hw_thermal_slowdown", "sw_power_cap"]
    assert s["sm_mhz"] == 2070 and s["sm_mhz_timed_region"] == 2070
