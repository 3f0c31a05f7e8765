"""The benchmark's host logic on CPU: clock parsing, traffic staleness, max-over-ranks with two
gloo ranks, and the reference (oracle) arm end to end on the small workload."""
import json
import os
import subprocess
import sys

import pytest

import bench
from conftest import ROOT


def test_parse_clocks_selects_the_timed_window_and_flags_reasons():
    lines = [
        "100.0, 0, 1900 MHz, 2070 MHz, 900 W, 0x0, Not Active, Not Active, Not Active, Not Active",
        "101.0, 0, 2000 MHz, 2070 MHz, 1300 W, 0x4, Not Active, Not Active, Not Active, Active",
        "102.0, 0, 1950 MHz, 2070 MHz, 1300 W, 0x0, Not Active, Not Active, Not Active, Not Active",
        "109.0, 0, 300 MHz, 2070 MHz, 100 W, 0x0, Not Active, Not Active, Not Active, Not Active",
    ]
    c = bench.parse_clocks("\n".join(lines), 100.5, 102.5)
    assert c["samples"] == 2 and c["window"] == "timed"
    assert c["sm_mhz"] == 1975.0 and c["sm_max_mhz"] == 2070.0
    assert c["reasons"] == ["sw_power_cap"]
    c2 = bench.parse_clocks("\n".join(lines), 200.0, 201.0)
    assert c2["window"] == "whole run" and c2["samples"] == 4
    assert bench.parse_clocks("", 0, 1)["samples"] == 0


def test_traffic_record_is_dropped_when_the_kernel_source_changes(tmp_path, monkeypatch):
    rec = {"w": {"kernel": "k", "source_sha": bench.source_hash(), "dram_bytes_per_launch": 123}}
    f = tmp_path / "traffic.json"
    f.write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(f))
    assert bench.recorded_traffic("w", "k") == 123
    assert bench.recorded_traffic("w", "other_kernel") is None
    rec["w"]["source_sha"] = "0" * 16
    f.write_text(json.dumps(rec))
    assert bench.recorded_traffic("w", "k") is None


def test_kernel_hash_follows_only_that_kernels_sources(tmp_path, monkeypatch):
    # a kernel's hash covers its launcher units, the headers they include and the planner's own
    # text: a change to another kernel's source leaves it unchanged
    d = tmp_path / "csrc"
    d.mkdir()
    (d / "launch_splitk.cu").write_text('#include "gemm16_splitk.cuh"\nint a;\n')
    (d / "gemm16_splitk.cuh").write_text('#include "common.cuh"\nint b;\n')
    (d / "common.cuh").write_text("int c;\n")
    (d / "dtc_gemm.cu").write_text('#include "gemm16_splitk.cuh"\nint d;\n')
    (d / "other.cuh").write_text("int e;\n")
    monkeypatch.setattr(bench, "CSRC", str(d))
    h0, all0 = bench.source_hash("gemm16_splitk_kernel"), bench.source_hash()
    (d / "other.cuh").write_text("int e2;\n")
    assert bench.source_hash("gemm16_splitk_kernel") == h0 and bench.source_hash() != all0
    (d / "common.cuh").write_text("int c2;\n")
    assert bench.source_hash("gemm16_splitk_kernel") != h0


def test_code_hash_ignores_comments_but_not_code():
    a = 'int f(int x) {  // add one\n    return x + 1; /* done */ }\nconst char* s = "a // b";\n'
    b = 'int f(int x) {\n  return x + 1;   }\n// a note\nconst char* s = "a // b";\n'
    c = 'int f(int x) {\n  return x + 2; }\nconst char* s = "a // b";\n'
    d = 'int f(int x) {\n  return x + 1; }\nconst char* s = "a // c";\n'
    assert bench.code_text(a) == bench.code_text(b)
    assert bench.code_text(a) != bench.code_text(c)
    assert bench.code_text(a) != bench.code_text(d)  # text inside a literal is code
    assert "note" not in bench.code_text(b) and '"a // b"' in bench.code_text(b)


_WORKER = r"""
import os, sys
sys.path.insert(0, {root!r})
import torch.distributed as dist
import bench
dist.init_process_group("gloo")
rank = dist.get_rank()
v = bench.max_over_ranks(10.0 + 5.0 * rank, dist.get_world_size())
bench.barrier(dist.get_world_size())
print("RESULT", rank, v, flush=True)
dist.destroy_process_group()
"""


def test_max_over_ranks_with_two_gloo_ranks(tmp_path):
    script = tmp_path / "w.py"
    script.write_text(_WORKER.format(root=ROOT))
    env = dict(os.environ, MASTER_ADDR="127.0.0.1", MASTER_PORT="29531", WORLD_SIZE="2")
    procs = []
    for r in range(2):
        e = dict(env, RANK=str(r), LOCAL_RANK=str(r))
        procs.append(subprocess.Popen([sys.executable, str(script)], env=e, stdout=subprocess.PIPE,
                                      stderr=subprocess.PIPE, text=True))
    outs = [p.communicate(timeout=120) for p in procs]
    for p, (o, e) in zip(procs, outs):
        assert p.returncode == 0, e
    vals = sorted(line.split()[1:] for o, _ in outs for line in o.splitlines()
                  if line.startswith("RESULT"))
    assert vals == [["0", "15.0"], ["1", "15.0"]]


def test_reference_arm_prints_one_json_line():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload",
                        "bf16_nt_256x256x512", "--steps", "3", "--warmup", "3"], cwd=ROOT,
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "TFLOP/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["steps"] == 3


def test_reference_arm_non_zero_ranks_exit_quietly():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload",
                        "bf16_nt_256x256x512", "--steps", "3", "--warmup", "3"], cwd=ROOT,
                       capture_output=True, text=True, timeout=300, env=env)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_warmup_below_three_is_refused():
    with pytest.raises(SystemExit):
        bench.main(["--warmup", "2"])


def test_nvml_samples_summarised_over_the_timed_window():
    import bench

    samples = [{"t": 1.0, "sm": 1000.0, "max": 2070.0, "power": 100.0, "reasons": 0x1},
               {"t": 2.0, "sm": 2070.0, "max": 2070.0, "power": 900.0, "reasons": 0x0},
               {"t": 2.5, "sm": 2055.0, "max": 2070.0, "power": 1300.0, "reasons": 0x4},
               {"t": 3.0, "sm": 2070.0, "max": 2070.0, "power": 950.0, "reasons": 0x0},
               {"t": 9.0, "sm": 900.0, "max": 2070.0, "power": 90.0, "reasons": 0x48}]
    r = bench.summarise_samples(samples, 1.5, 3.5)
    assert r["window"] == "timed" and r["samples"] == 3
    assert r["sm_mhz"] == 2070.0 and r["sm_max_mhz"] == 2070.0
    assert r["reasons"] == ["sw_power_cap"]  # idle (0x1) outside the window is not reported
    r = bench.summarise_samples(samples, 8.0, 10.0)
    assert r["reasons"] == ["hw_slowdown", "hw_thermal_slowdown"]
    assert bench.summarise_samples(samples, 20.0, 21.0)["window"] == "whole run"


def test_bench_configs_name_known_workloads():
    import bench
    from dense_tensor_core_gb300 import workloads

    ids = [c[0] for c in bench.BENCH_CONFIGS]
    assert ids == ["1", "2", "3", "4a", "4b", "5"]
    for _, name, bound in bench.BENCH_CONFIGS:
        assert name in workloads.WORKLOADS and bound in ("latency", "tensor", "hbm")


def test_launches_per_step_counts_the_extra_kernels():
    import bench
    from dense_tensor_core_gb300 import workloads

    W = workloads.WORKLOADS
    assert bench.launches_per_step(W["bf16_nt_4096x4096x8192"], {"sf_packed": 0}) == 1
    assert bench.launches_per_step(W["bf16_sp24_nt_4096x4096x8192"], {"sf_packed": 0}) == 2
    assert bench.launches_per_step(W["mxfp8_b32_nt_4096x4096x8192"], {"sf_packed": 1}) == 2
    assert bench.launches_per_step(W["mxfp8_nt_4096x4096x8192"], {"sf_packed": 0}) == 1
    assert bench.launches_per_step(W["nvfp4_nt_4096x4096x8192"], {"sf_packed": 0}) == 2


def test_nvfp4_workload_bytes_and_inputs():
    # the NVFP4 workload's compulsory bytes (packed e2m1 rows, a UE4M3 byte per 16 elements, bf16
    # C) and the shapes and code ranges its generator produces
    import numpy as np

    from dense_tensor_core_gb300 import workloads

    w = workloads.WORKLOADS["nvfp4_nt_4096x4096x8192"]
    assert w.min_bytes == 2 * 4096 * (4096 + 512) + 2 * 4096 * 4096
    A, B, sfA, sfB = workloads.make_nvfp4(64, 48, 96, seed=3)
    assert A.shape == (64, 48) and B.shape == (48, 48) and sfA.shape == (64, 6) and sfB.shape == (48, 6)
    e = sfA >> 3
    assert ((e >= 4) & (e <= 10)).all() and not (sfA & 0x80).any()
    nib = np.concatenate([A & 15, A >> 4]).ravel()
    assert set(np.unique(nib)) <= set(range(16)) and len(np.unique(nib)) > 8
