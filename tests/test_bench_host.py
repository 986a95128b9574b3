"""Host-side logic of bench.py that needs no GPU: reading an ncu CSV capture into the
per-launch DRAM traffic record, and the roofline arithmetic of the per-kernel figures."""
import json
import os

import pytest

import bench

CSV = '''==PROF== Connected to process 11 (/usr/bin/python3.12)
==PROF== Disconnected from process 11
"ID","Process ID","Process Name","Host Name","Kernel Name","Context","Stream","Block Size","Grid Size","Device","CC","Section Name","Metric Name","Metric Unit","Metric Value"
"0","11","python3.12","127.0.0.1","void rlk::gemm_kernel<(int)0>(rlk::TileMaps, rlk::GemmArgs)","1","7","(192, 1, 1)","(152, 1, 1)","0","10.3","Command line profiler metrics","dram__bytes_read.sum","byte","3000000000"
"0","11","python3.12","127.0.0.1","void rlk::gemm_kernel<(int)0>(rlk::TileMaps, rlk::GemmArgs)","1","7","(192, 1, 1)","(152, 1, 1)","0","10.3","Command line profiler metrics","dram__bytes_write.sum","byte","12000000"
"1","11","python3.12","127.0.0.1","void rlk::leaf_tree_kernel(rlk::TreeArgs)","1","7","(256, 1, 1)","(1024, 1, 1)","0","10.3","Command line profiler metrics","dram__bytes_read.sum","byte","15000000"
"2","11","python3.12","127.0.0.1","void gemm_kernel<2>(TileMaps, GemmArgs)","1","7","(192, 1, 1)","(152, 1, 1)","0","10.3","Command line profiler metrics","dram__bytes_read.sum","Gbyte","8.5"
"2","11","python3.12","127.0.0.1","void gemm_kernel<2>(TileMaps, GemmArgs)","1","7","(192, 1, 1)","(152, 1, 1)","0","10.3","Command line profiler metrics","dram__bytes_write.sum","Mbyte","64"
"3","11","python3.12","127.0.0.1","void gemm_kernel<2>(TileMaps, GemmArgs)","1","7","(192, 1, 1)","(152, 1, 1)","0","10.3","Command line profiler metrics","dram__bytes_read.sum","Gbyte","9.5"
"3","11","python3.12","127.0.0.1","void gemm_kernel<2>(TileMaps, GemmArgs)","1","7","(192, 1, 1)","(152, 1, 1)","0","10.3","Command line profiler metrics","dram__bytes_write.sum","Mbyte","64"
'''


def test_record_traffic_averages_per_launch(tmp_path, monkeypatch):
    src = tmp_path / "cap.csv"
    src.write_text(CSV)
    out = tmp_path / "traffic.json"
    rec = bench.record_traffic(str(src), "ncu ... python bench.py", out_path=str(out))
    k = rec["kernels"]
    assert set(k) == {"fwd", "dH"}                       # the leaf-tree kernel is not a tile kernel
    assert k["fwd"]["launches"] == 1
    assert k["fwd"]["traffic_bytes_per_launch"] == pytest.approx(3.012e9)
    assert k["dH"]["launches"] == 2
    assert k["dH"]["dram_bytes_read_per_launch"] == pytest.approx(9.0e9)
    assert k["dH"]["traffic_bytes_per_launch"] == pytest.approx(9.064e9)
    assert json.loads(out.read_text())["kernels"] == k
    # read back only while the sources still hash to the recorded value
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(out))
    b, _ = bench.traffic_per_launch("dH")
    assert b == pytest.approx(9.064e9)
    rec["library_sources_sha256"] = "0" * 64
    out.write_text(json.dumps(rec))
    b, why = bench.traffic_per_launch("dH")
    assert b is None and "predates" in why
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(tmp_path / "missing.json"))
    assert bench.traffic_per_launch("dH")[0] is None


def test_per_kernel_roofline_arithmetic():
    f = 2.0 * 8192 * 4096 * 151669
    r = bench.per_kernel_roofline({"fwd": 5.5, "dH": 6.0, "merge": 0.01}, f, 1952.5, 1749.2)
    assert set(r) == {"fwd", "dH"}
    assert r["dH"]["tflops"] == pytest.approx(f / 6.0e-3 / 1e12)
    assert r["dH"]["frac_of_sustained"] == pytest.approx(r["dH"]["tflops"] / 1749.2)
    assert r["dH"]["frac_of_burst"] == pytest.approx(r["dH"]["tflops"] / 1952.5)


def test_committed_traffic_record_is_well_formed():
    if not os.path.exists(bench.TRAFFIC_FILE):
        pytest.skip("no traffic record committed")
    rec = json.load(open(bench.TRAFFIC_FILE))
    assert len(rec["library_sources_sha256"]) == 64 and rec["command"]
    for stage, k in rec["kernels"].items():
        assert stage in ("fwd", "dz", "dH", "dW") and k["launches"] >= 1
        assert k["traffic_bytes_per_launch"] > 0
