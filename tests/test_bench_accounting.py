"""The bench's accounting, on the CPU: the algorithmic bytes of one step of
each workload (logits read once, 18 bytes of outputs and masks per row, six
more per row for the large workload's second rule), and the rule that a
recorded ncu traffic figure is reported only while the kernel code it was
measured on is unchanged (comments aside)."""
import os
import shutil

import numpy as np
import pytest

import bench
import dllm_workloads as W

# bytes per step: V * e per row of logits + 12 (x0, prob, entropy) + 1
# (candidate) + 1 (commit) + 4 (canvas) per row, + 6 per row for large
EXPECTED = {
    "tiny": 64 * (4096 * 4 + 18),
    "llada": 32 * (126464 * 2 + 18),
    "dream": 2048 * (152064 * 2 + 18),
    "large": 16384 * (126464 * 4 + 18 + 6),
}


@pytest.mark.parametrize("name", sorted(EXPECTED))
def test_algorithmic_bytes_per_step(name):
    w = W.build(name, rows=np.arange(0))      # shapes and parameters only
    assert bench.algorithmic_bytes(w) == EXPECTED[name]


def test_documented_figures():
    # the per-step figures quoted with the measurements
    assert EXPECTED == {"tiny": 1_049_728, "llada": 8_094_272, "dream": 622_891_008, "large": 8_288_337_920}


def test_whole_job_rate_counts_every_rank():
    # 2 ranks x 10 steps of 1 GB in 1 s (the slowest rank's time) = 20 GB/s
    assert bench.whole_job_gbs(10**9, 10, 2, 1000.0) == pytest.approx(20.0)


def _copy_sources(dst):
    src = os.path.join(bench.ROOT, "commit_step_gb300", "csrc")
    os.makedirs(os.path.join(dst, "commit_step_gb300", "csrc"))
    for name in bench.KERNEL_SOURCES:
        shutil.copy(os.path.join(src, name), os.path.join(dst, "commit_step_gb300", "csrc", name))
    return os.path.join(dst, "commit_step_gb300", "csrc")


def test_kernel_hash_follows_code_not_comments(tmp_path, monkeypatch):
    base = bench.kernel_source_hash()
    csrc = _copy_sources(str(tmp_path))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.kernel_source_hash() == base
    path = os.path.join(csrc, bench.KERNEL_SOURCES[0])
    text = open(path).read()
    open(path, "w").write("// a new comment line\n/* and a block\n   comment */\n" + text.replace("\n", "\n\n", 3))
    assert bench.kernel_source_hash() == base          # comments and blank space do not count
    open(path, "w").write(text + "\nstatic const int kExtra = 1;\n")
    assert bench.kernel_source_hash() != base          # code does


def test_recorded_traffic_only_for_the_current_code(monkeypatch):
    got = bench.recorded_traffic("llada")
    assert got is None or got > 8_093_696              # at least the logits, when recorded
    monkeypatch.setattr(bench, "kernel_source_hash", lambda *a: "0" * 16)
    assert bench.recorded_traffic("llada") is None


def test_issue_roofline_arithmetic(monkeypatch):
    # 152 SMs x 4 schedulers x 2000 MHz = 1216 G warp instructions/s; 608 M
    # instructions in 1 ms is 608 G/s, half of it; at full issue the launch
    # would take 0.5 ms, so 1 GB of logits would stream at 2000 GB/s
    r = bench.issue_roofline(608e6, 1.0, 152, 2000.0, 10**9, 4000.0)
    assert r["bound"] == "issue"
    assert r["peak"] == pytest.approx(1216.0)
    assert r["achieved"] == pytest.approx(608.0)
    assert r["frac"] == pytest.approx(0.5)
    assert r["hbm_frac_at_full_issue"] == pytest.approx(0.5)
    assert bench.issue_roofline(None, 1.0, 152, 2000.0, 10**9, 4000.0) is None
    got = bench.recorded_inst("dream")
    assert got is None or got > 622_891_008 / 16      # at least one warp instruction per 16-byte vector
    monkeypatch.setattr(bench, "kernel_source_hash", lambda *a: "0" * 16)
    assert bench.recorded_inst("dream") is None


def test_recorded_traffic_follows_its_own_sources(tmp_path, monkeypatch):
    # the mask's record is hashed over the mask's own sources, not the statistics kernels'
    got = bench.recorded_traffic("mask")
    assert got is None or got > 0
    monkeypatch.setattr(bench, "KERNEL_SOURCES", ("dllm_rules.cuh",))
    assert bench.recorded_traffic("mask") == got
    assert bench.recorded_traffic("llada") is None
