"""Host-side bookkeeping of bench.py on CPU: launch counts, lane-operation counts, and how the
bench reads DRAM traffic from the committed ncu summaries (only while their recorded kernel
source hash matches the sources being built)."""
import os

import numpy as np
import pytest

import bench
from selective_state_space_diagonal_b300 import workloads as wl

PROFILES = [
    # summary, kernel prefix, workload, the kernel sources its hash covers
    ("nscan_kernel_trap_bf16_batch.md", "nscan_kernel", wl.WORKLOADS["trap_bf16_batch"], bench.KERNEL_SOURCES),
    ("scan_kernel_zoh_bf16_batch.md", "scan_kernel", wl.WORKLOADS["zoh_bf16_batch"], bench.ZOH_KERNEL_SOURCES),
    ("mscan_kernel_mimo_trap_bf16_batch.md", "mscan_kernel", wl.MIMO_WORKLOADS["mimo_trap_bf16_batch"],
     bench.MIMO_KERNEL_SOURCES),
]


def machine_values(path):
    vals = {}
    with open(path) as f:
        for line in f:
            if ":" in line and line.split(":", 1)[0].strip() in ("kernel_source_sha256_16", "dram_bytes_per_launch"):
                k, v = line.split(":", 1)
                vals[k.strip()] = v.strip()
    return vals


@pytest.mark.parametrize("name,kernel,w,sources", PROFILES, ids=[p[0] for p in PROFILES])
def test_profile_traffic_is_near_the_algorithmic_bytes(name, kernel, w, sources):
    """Each summary records DRAM bytes per launch within a few percent above the workload's
    algorithmic bytes (more would be re-reads; less is impossible for a kernel that reads its
    inputs and writes its output once)."""
    vals = machine_values(os.path.join(bench.ROOT, "profiles", name))
    assert len(vals["kernel_source_sha256_16"]) == 16
    traffic = int(vals["dram_bytes_per_launch"])
    assert 1.0 <= traffic / w.min_bytes() <= 1.05


def test_traffic_read_only_for_matching_sources(tmp_path, monkeypatch):
    src = tmp_path / "k.cuh"
    src.write_text("// kernel v1\n")
    (tmp_path / "profiles").mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h = bench.kernel_source_hash(("k.cuh",))
    (tmp_path / "profiles" / "scan_kernel_demo.md").write_text(
        f"# demo\n\nkernel_source_sha256_16: {h}\ndram_bytes_per_launch: 1234\n")
    assert bench.traffic_from_profiles("demo", "scan_kernel", ("k.cuh",)) == 1234
    src.write_text("// kernel v2\n")   # the sources changed since the capture: the figure is stale
    assert bench.traffic_from_profiles("demo", "scan_kernel", ("k.cuh",)) is None
    assert bench.traffic_from_profiles("absent", "scan_kernel", ("k.cuh",)) is None


def test_launch_and_operation_counts():
    for w in wl.WORKLOADS.values():
        assert bench.launches_per_step(w) == 2        # table kernel + scan kernel in every mode
    assert bench.mimo_alu_ops_per_elem(4, 1) == bench.mimo_alu_ops_per_elem(4, 0) == pytest.approx(4.75)
    assert bench.mimo_alu_ops_per_elem(1, 1) == pytest.approx(7.0)
    w = wl.MIMO_WORKLOADS["mimo_trap_bf16_batch"]
    assert bench.mimo_staged(w) and bench.mimo_launches(w, 148) == 2
    assert not bench.mimo_staged(w.with_shape(H=5)) and not bench.mimo_staged(w.with_shape(N=4))
    assert bench.ALU_OPS_PER_ELEM[0] == bench.ALU_OPS_PER_ELEM[1] == 6
    assert bench.ZOH_ALU_OPS_PER_ELEM == bench.ALU_OPS_PER_ELEM[2] > bench.ALU_OPS_PER_ELEM[1]
    assert bench.scan_kernel_name(wl.WORKLOADS["trap_bf16_batch"]) == "nscan_kernel"
    assert bench.scan_kernel_name(wl.WORKLOADS["zoh_bf16_batch"]) == "scan_kernel"


def test_workload_config_names_the_mode():
    names = {w.mode: bench.workload_config(w)["mode"] for w in wl.WORKLOADS.values()}
    assert names == {0: "exp-Euler", 1: "exp-trapezoidal", 2: "zero-order hold"}


def test_clock_summary_and_alu_roofline():
    s = bench.clock_summary([(2032.0, 2032.0, 700.0, []), (1990.0, 2032.0, 900.0, ["sw_power_cap"]),
                             (2010.0, 2032.0, 800.0, [])])
    assert s["sm_mhz"] == 2010.0 and s["sm_max_mhz"] == 2032.0 and s["samples"] == 3
    assert s["reasons"] == ["sw_power_cap"] and s["power_w_max"] == 900.0
    empty = bench.clock_summary([])
    assert empty["sm_mhz"] is None and empty["reasons"] == ["unsampled"]
    # the FP32 peak follows the sampled clock; without a sample the fraction is unknown
    r = bench.alu_roofline(6, 10 ** 9, 1e-3, s)
    assert r["peak"] == pytest.approx(128 * 148 * 2010e6 / 1e12)
    assert r["achieved"] == pytest.approx(6.0) and r["frac"] == pytest.approx(6.0 / r["peak"])
    assert bench.alu_roofline(6, 10 ** 9, 1e-3, empty)["frac"] is None


def test_parity_errors():
    x = np.ones((1, 4, 2))
    d = np.array([2.0, 0.0])
    y_ref = np.array([[[3.0, 1.0], [2.5, 0.5], [2.0, 0.0], [4.0, 2.0]]])
    y = y_ref.copy()
    y[0, 3, 1] += 0.01
    e, e_ssm = bench.parity_errors(y, y_ref, x, d)
    assert e == pytest.approx(0.01 / 4.0)
    assert e_ssm == pytest.approx(0.01 / 2.0)   # the state-space part y - Dskip x peaks at 2


def test_shape_overrides():
    """--batch, --length and --states change only the named dimensions of the workload."""
    a = bench.parse_args(["--workload", "zoh_bf16_batch", "--states", "64", "--length", "512"])
    w = bench.selected_workload(a)
    base = wl.WORKLOADS["zoh_bf16_batch"]
    assert (w.B, w.L, w.D, w.N, w.mode, w.dtype) == (base.B, 512, base.D, 64, base.mode, base.dtype)
    assert bench.selected_workload(bench.parse_args([])) == wl.WORKLOADS[bench.DEFAULT_WORKLOAD]
