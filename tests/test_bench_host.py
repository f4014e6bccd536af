"""bench.py host logic on CPU: which runs time the oracle on one core, and how the committed ncu
traffic figures are matched to a kernel, a workload and that kernel's sources."""
import json
import os
import subprocess
import sys

import bench
import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_oracle_arms_are_recognised_from_the_command_line():
    assert bench._times_the_oracle(["--impl", "reference", "--steps", "3"])
    assert bench._times_the_oracle(["--impl=reference"])
    assert bench._times_the_oracle(["--cpu-worker", "--workload", "tiny"])
    assert not bench._times_the_oracle(["--impl", "ours"])
    assert not bench._times_the_oracle(["--workload", "reference"])
    assert not bench._times_the_oracle([])


def test_reference_arm_pins_blas_before_numpy_loads():
    # a fresh interpreter that imports bench as `bench.py --impl reference` would
    code = ("import sys, os; sys.argv = ['bench.py', '--impl', 'reference']; sys.path.insert(0, %r); "
            "import bench; print(os.environ.get('OPENBLAS_NUM_THREADS'), os.environ.get('OMP_NUM_THREADS'))" % ROOT)
    env = {k: v for k, v in os.environ.items() if k not in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS")}
    out = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, check=True)
    assert out.stdout.split() == ["1", "1"]


def test_traffic_is_keyed_by_kernel_and_workload():
    mixed = synth.workload("mixed", quantum=2048)
    decode = synth.workload("decode")
    assert bench.traffic_key("tc_gateup", mixed) != bench.traffic_key("tc_gateup", decode)
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as fh:
        committed = json.load(fh)
    for key, ent in committed.items():
        if key.startswith("_"):
            continue
        kernel = key.split("@")[0]
        assert kernel in bench.KERNEL_SOURCES, key
        assert abs(ent["bytes_per_launch"] - (ent["read"] + ent["write"])) <= 1  # each rounded on its own
    # a workload with no capture gets no traffic figure, whatever the other workloads hold
    tiny = synth.workload("tiny")
    assert bench.committed_traffic("tc_gateup", tiny) is None


def test_kernel_source_hash_covers_only_that_kernels_sources(tmp_path, monkeypatch):
    csrc = tmp_path / "decode_batches_gb300" / "csrc"
    csrc.mkdir(parents=True)
    names = set(bench._COMMON_SOURCES) | {f for srcs in bench.KERNEL_SOURCES.values() for f in srcs} | {"route.cu"}
    for n in names:
        (csrc / n).write_text(n)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    gemm = bench.kernel_source_hash("tc_gateup")
    comb = bench.kernel_source_hash("combine")
    (csrc / "route.cu").write_text("changed")            # not a source of either kernel
    assert bench.kernel_source_hash("tc_gateup") == gemm
    (csrc / "combine.cu").write_text("changed")          # the combine's own file
    assert bench.kernel_source_hash("combine") != comb
    assert bench.kernel_source_hash("tc_gateup") == gemm
    (csrc / "common.cuh").write_text("changed")          # shared by every kernel
    assert bench.kernel_source_hash("tc_gateup") != gemm
