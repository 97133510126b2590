"""Host-side logic of bench.py (CPU only): the roofline, the recorded DRAM traffic and its
staleness rule, and the clock-sample summary."""
import os

import pytest

import bench

PEAKS = {"hbm_gbs": 6000.0, "bf16_tflops": 2000.0, "source": "test"}


def test_roofline_picks_the_binding_resource():
    # 1 GB and 1 TFLOP: HBM takes 1/6000 s, the tensor pipe 1/2000 s -> tensor-bound
    r = bench.roofline(1e9, 1e12, 1e-3, PEAKS)
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    assert r["achieved"] == pytest.approx(1e12 / 1e-3 / 1e12)
    assert r["frac"] == pytest.approx(r["achieved"] / PEAKS["bf16_tflops"])
    # 1 GB and 0.1 TFLOP: HBM takes longer -> HBM-bound, achieved in GB/s
    r = bench.roofline(1e9, 1e11, 1e-3, PEAKS)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert r["achieved"] == pytest.approx(1e9 / 1e-3 / 1e9)
    assert r["frac"] == pytest.approx(1000.0 / 6000.0)
    assert r["traffic"] is None  # filled in from the recorded captures, never from here


def test_recorded_traffic_names_current_kernels_only():
    for (workload, kernel), (nbytes, sha) in bench.TRAFFIC.items():
        assert kernel in bench.KERNEL_SOURCES
        for name in bench.KERNEL_SOURCES[kernel]:
            assert os.path.exists(os.path.join(bench.ROOT, "sparse_mla_decode_smla_gb300", "csrc", name))
        assert nbytes > 0 and len(sha) == 16


def test_recorded_traffic_is_null_once_the_kernel_changes(monkeypatch):
    kernel = "decode_hg_kernel"
    current = bench.kernel_sources_sha(kernel)
    monkeypatch.setattr(bench, "TRAFFIC", {("w", kernel): (123, current), ("x", kernel): (456, "0" * 16)})
    assert bench.recorded_traffic("w", kernel) == 123
    assert bench.recorded_traffic("x", kernel) is None   # captured on other sources
    assert bench.recorded_traffic("y", kernel) is None   # never captured


def test_clock_summary_flags_throttle_reasons(tmp_path):
    path = tmp_path / "clocks.csv"
    path.write_text("2070, 2070, 900.1, 0x0, Not Active, Not Active, Not Active, Not Active\n"
                    "1980, 2070, 1390.0, 0x4, Not Active, Not Active, Not Active, Active\n"
                    "2070, 2070, 1000.0, 0x0, Not Active, Not Active, Not Active, Not Active\n")
    cs = bench.ClockSampler(0)
    cs.proc, cs.path = object(), str(path)
    s = cs.summary()
    assert s["sm_mhz"] == 2070.0 and s["sm_max_mhz"] == 2070.0 and s["samples"] == 3
    assert s["reasons"] == ["sw_power_cap"]


def test_both_arms_share_one_config():
    # the reference arm's line carries the same `config` object as the GPU arm's line for the
    # same workload and world size, so the two lines describe one workload
    import json
    import subprocess
    import sys

    import workloads as W
    w = W.BY_NAME["tiny_bf16_T2_H16_K128"]
    problem = W.make_problem(w, device="cpu")
    valid = bench.algorithmic_work(problem)[0]
    cfg = bench.workload_config(problem, valid, 0, 1)
    assert cfg["workload"] == w.name and cfg["valid_indices"] == valid == w.num_tokens * w.topk
    assert cfg["num_splits"] == "auto" and cfg["parallelism"] == "replicas x1"
    out = subprocess.run([sys.executable, os.path.join(bench.ROOT, "bench.py"), "--impl", "reference",
                          "--workload", w.name, "--steps", "2", "--warmup", "1"],
                         capture_output=True, text=True, timeout=300, check=True).stdout
    line = json.loads(out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["config"] == cfg
    assert line["metric"] == bench.METRIC and line["unit"] == "query-tokens/s" and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"


def test_launch_count_comes_from_the_library_plan():
    # gpu_launches counts the decode launches of the library's own plan, plus its merge kernel
    smla = pytest.importorskip("sparse_mla_decode_smla_gb300")
    if not os.path.exists(smla.LIB_PATH):
        pytest.skip("libsmla.so is not built")

    def desc(tokens, heads, next_n=1):
        return smla.make_desc(tokens, heads, 2048, tokens // next_n, 64, 4096, 2048, smla.SMLA_KV_FP8_DS,
                              1 / 24, next_n=next_n)

    assert bench.decode_launches(smla, desc(256, 128, next_n=4), 152) == 2  # whole waves + the tail
    assert bench.decode_launches(smla, desc(32, 64), 152) == 1   # splits merged in the cluster
    assert bench.decode_launches(smla, desc(128, 128), 152) == 1
    assert bench.decode_launches(smla, desc(4, 16), 152) == 2    # mma.sync splits + the merge kernel
