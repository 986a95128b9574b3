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


class _FakeRlk:
    """Records the binding calls bench.Path makes (no GPU, no library)."""
    RLK_BWD_DZ, RLK_BWD_DH, RLK_BWD_DW = 1, 2, 4

    def __init__(self):
        self.calls = []

    def fwd_workspace_bytes(self, T, H, n):
        return 16

    bwd_workspace_bytes = fwd_workspace_bytes

    def linear_logp_fwd(self, h, W, y, V_true, vocab_start=0, partial=False, **kw):
        self.calls.append(("fwd", vocab_start, W.shape[0], partial))

    def linear_logp_bwd(self, h, W, y, lse, g, V_true, vocab_start=0, dH_fp32_partial=False,
                        stages=None, **kw):
        self.calls.append(("bwd", vocab_start, W.shape[0], dH_fp32_partial, stages))

    def lse_merge(self, parts, **kw):
        self.calls.append(("merge", parts.shape[0]))

    def shard_sum_bf16(self, parts, **kw):
        self.calls.append(("sum", parts.shape[0]))


def _path(w):
    import numpy as np
    import torch
    d = {"h": np.zeros((w.T, w.H), np.uint16), "W": np.zeros((w.V, w.H), np.uint16),
         "y": np.zeros(w.T, np.int64), "g": np.zeros(w.T, np.float32)}
    fake = _FakeRlk()
    return bench.Path(fake, torch, w, d, torch.device("cpu")), fake


def test_staged_step_calls_every_stage_once_in_order():
    import workloads
    w = workloads.Workload("s", T=8, H=16, V=64, V_true=60)
    path, fake = _path(w)
    calls = path.staged_calls()
    assert [n for n, _ in calls] == ["fwd", "dz", "dH", "dW"]
    for _, fn in calls:
        fn()
    assert fake.calls == [("fwd", 0, 64, False), ("bwd", 0, 64, False, 1), ("bwd", 0, 64, False, 2),
                          ("bwd", 0, 64, False, 4)]
    assert path.launches_per_step() == 5


def test_staged_sharded_step_attributes_each_shard_launch_to_its_stage():
    import workloads
    w = workloads.Workload("s2", T=8, H=16, V=20480, V_true=20000, shards=((0, 12288), (12288, 8192)))
    path, fake = _path(w)
    calls = path.staged_calls()
    assert [n for n, _ in calls] == ["fwd", "fwd", "merge", "dz", "dH", "dW", "dz", "dH", "dW", "sum"]
    for _, fn in calls:
        fn()
    assert fake.calls == [("fwd", 0, 12288, True), ("fwd", 12288, 8192, True), ("merge", 2),
                          ("bwd", 0, 12288, True, 1), ("bwd", 0, 12288, True, 2),
                          ("bwd", 0, 12288, True, 4), ("bwd", 12288, 8192, True, 1),
                          ("bwd", 12288, 8192, True, 2), ("bwd", 12288, 8192, True, 4), ("sum", 2)]
    # one step launches: per shard 2 forward kernels and 3 backward kernels, the merge, the sum
    assert path.launches_per_step() == 2 * 2 + 1 + 3 * 2 + 1
