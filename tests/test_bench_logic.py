"""Host logic of bench.py that the bench line's fields come from (CPU only):
algorithmic bytes per launch, the roofline's choice of kernel, and the DRAM
traffic taken from the committed profile only while it matches the sources."""
import json
import re
import os

import numpy as np

import bench


def test_algorithmic_bytes_count_each_routed_expert_once():
    H, I, E, K = 2048, 768, 128, 8
    ids = np.array([[3, 3, 7, 7, 9, 1, 2, 4], [3, 5, 6, 8, 10, 11, 12, 13]], np.int32)
    uniq = np.unique(ids).size
    per_gu = 2 * I * H + 2 * I * H // 32
    per_dn = H * I + H * I // 32
    B = ids.shape[0]
    assert bench.gate_up_bytes(ids, B, H, I, E, K) == uniq * per_gu + 2 * B * H + 2 * B * K * I + 4 * B * K
    assert bench.down_bytes(ids, B, H, I, E, K) == uniq * per_dn + 2 * B * K * I + 2 * B * H + 8 * B * K
    bad = ids.copy()
    bad[0, 0] = -1   # ids outside [0, E) move no weight bytes
    bad[1, 0] = E
    # both replaced ids were a duplicate of expert 3, still routed elsewhere: the
    # routed set is unchanged; replacing expert 5, routed once, removes its bytes
    assert bench.gate_up_bytes(bad, B, H, I, E, K) == uniq * per_gu + 2 * B * H + 2 * B * K * I + 4 * B * K
    bad[1, 1] = -7
    assert bench.gate_up_bytes(bad, B, H, I, E, K) == (uniq - 1) * per_gu + 2 * B * H + 2 * B * K * I + 4 * B * K


def test_roofline_names_the_kernel_with_the_longest_launch():
    k = {"a<1>": {"ms": 0.070, "bytes": 364e6, "launches": 96},
         "b<2>": {"ms": 0.049, "bytes": 182e6, "launches": 96}}
    r = bench.roofline_of(k, 6783.8, "measured")
    assert r["kernel"] == "a<1>" and r["chosen_by"] == "longest mean launch of the plan"
    assert abs(r["achieved"] - 364e6 / 0.070 / 1e6) < 0.1
    assert abs(r["frac"] - r["achieved"] / 6783.8) < 1e-4
    k["b<2>"]["ms"] = 0.080
    assert bench.roofline_of(k, 6783.8, "measured")["kernel"] == "b<2>"


def test_traffic_comes_from_the_same_profiled_launch_and_only_for_current_sources(tmp_path, monkeypatch):
    prof = tmp_path / "profiles"
    prof.mkdir()
    data = {"kernels": {"moe_k": {"dram_bytes_profiled_launch": 1010, "algorithmic_bytes_profiled_launch": 1000,
                                  "profiled": "x", "kernel_sources_sha": "1111222233334444"}}}
    (prof / "dram_traffic.json").write_text(json.dumps(data))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_file_sha", lambda k: "1111222233334444")
    t = bench.profile_traffic("moe_k", 2000)
    assert t["bytes_per_launch"] == 2020 and t["dram_over_algorithmic"] == 1.01
    assert bench.profile_traffic("other", 2000) is None
    data["kernels"]["moe_k"]["kernel_sources_sha"] = "0000000000000000"  # kernel changed since the capture
    (prof / "dram_traffic.json").write_text(json.dumps(data))
    assert bench.profile_traffic("moe_k", 2000) is None


def test_kernel_file_hash_follows_the_kernels_own_file_and_its_headers(tmp_path, monkeypatch):
    csrc = tmp_path / "moe_decode_gate_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "a.cuh").write_text("// shared\n")
    (csrc / "b.cuh").write_text('#include "a.cuh"\n')
    (csrc / "k1.cu").write_text('#include "b.cuh"\n__global__ void k1() {}\n')
    (csrc / "k2.cu").write_text('#include "a.cuh"\n__global__ void k2() {}\n')
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "KERNEL_SOURCE", {"k1": "k1.cu", "k2": "k2.cu"})
    h1, h2 = bench.kernel_file_sha("k1"), bench.kernel_file_sha("k2")
    (csrc / "k2.cu").write_text('#include "a.cuh"\n__global__ void k2() { }\n')
    assert bench.kernel_file_sha("k1") == h1 and bench.kernel_file_sha("k2") != h2
    (csrc / "a.cuh").write_text("// shared, edited\n")  # reached from k1 through b.cuh
    assert bench.kernel_file_sha("k1") != h1
    assert bench.kernel_file_sha("unknown") is None


def test_committed_traffic_profile_has_both_figures_for_every_plan_kernel():
    p = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "profiles",
                     "dram_traffic.json")
    d = json.load(open(p))
    for name in ("moe_gate_up_mma", "moe_down_dimblock", "moe_gate_up_3d_batched", "moe_down_3d_batched"):
        k = d["kernels"][name]
        ratio = k["dram_bytes_profiled_launch"] / k["algorithmic_bytes_profiled_launch"]
        assert 0.95 < ratio < 1.1, (name, ratio)  # each routed row read from HBM once


def test_kernel_source_map_names_the_file_that_defines_each_kernel():
    csrc = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                        "moe_decode_gate_gb300", "csrc")
    for kernel, f in bench.KERNEL_SOURCE.items():
        text = open(os.path.join(csrc, f)).read()
        assert re.search(r"__global__[^;{]*\b" + kernel + r"\s*\(", text), (kernel, f)
