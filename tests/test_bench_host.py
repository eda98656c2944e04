"""Host logic of bench.py (CPU only): the kernel fingerprint that decides
whether the committed DRAM-traffic capture still describes the timed launch,
and the whole-job rate."""
import json
import os
import shutil

import pytest

import bench

PARAMS = {"stride": 256, "rho0": 2.0, "rho1": 2.25, "sample_min_len": 12288, "long_len": 786432,
          "long_stride": 512, "long_rho0": 2.75, "long_rho1": 3.0, "direct_max": 16384,
          "force_kind": 0, "kv_segments": 0}
PLAN = {"kind": "persistent", "grid": 304}


def test_fingerprint_is_stable_and_sees_every_input():
    base = bench.kernel_fingerprint(PARAMS, "persistent", 304, 4)
    assert base == bench.kernel_fingerprint(dict(PARAMS), "persistent", 304, 4)
    seen = {base}
    for knob in bench.SAMPLING_KNOBS:
        p = dict(PARAMS)
        p[knob] = p[knob] * 2 + 1
        seen.add(bench.kernel_fingerprint(p, "persistent", 304, 4))
    seen.add(bench.kernel_fingerprint(PARAMS, "kvsplit", 304, 4))
    seen.add(bench.kernel_fingerprint(PARAMS, "persistent", 152, 4))
    seen.add(bench.kernel_fingerprint(PARAMS, "persistent", 304, 1))
    assert len(seen) == len(bench.SAMPLING_KNOBS) + 4
    # knobs that do not change a persistent launch's traffic are left out
    p = dict(PARAMS, force_kind=2, direct_max=1)
    assert bench.kernel_fingerprint(p, "persistent", 304, 4) == base


SRC = os.path.join(bench.ROOT, "exact_top_sparse_gb300", "csrc")


def _tree(tmp_path, fingerprint_of):
    """A copy of the kernel sources under tmp_path and a capture record."""
    src = SRC
    dst = tmp_path / "exact_top_sparse_gb300" / "csrc"
    dst.mkdir(parents=True)
    for name in bench.FINGERPRINT_SOURCES:
        shutil.copy(os.path.join(src, name), dst / name)
    (tmp_path / "profiles").mkdir()
    rec = {"kernel_fingerprint": fingerprint_of, "dram_bytes_per_valid_byte": 1.25}
    (tmp_path / "profiles" / "k_persistent_traffic.json").write_text(json.dumps(rec))
    return dst


def test_traffic_only_while_the_capture_matches(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    _tree(tmp_path, "0" * 16)
    fp = bench.kernel_fingerprint(PARAMS, "persistent", 304, 4)
    (tmp_path / "profiles" / "k_persistent_traffic.json").write_text(
        json.dumps({"kernel_fingerprint": fp, "dram_bytes_per_valid_byte": 1.25}))
    assert bench.profiled_traffic(PARAMS, PLAN, 8e9, 4) == pytest.approx(1e10)
    # another element size, launch kind or sampling tier: no figure
    assert bench.profiled_traffic(PARAMS, PLAN, 8e9, 1) is None
    assert bench.profiled_traffic(PARAMS, {"kind": "kvsplit", "grid": 304}, 8e9, 4) is None
    assert bench.profiled_traffic(dict(PARAMS, long_rho1=3.5), PLAN, 8e9, 4) is None
    # a kernel source edited after the capture: no figure
    src = tmp_path / "exact_top_sparse_gb300" / "csrc" / "topk_kernels.cu"
    src.write_text(src.read_text() + "\n// edited\n")
    assert bench.profiled_traffic(PARAMS, PLAN, 8e9, 4) is None


def test_whole_job_rate():
    # rows of every rank over the slowest rank's time
    assert bench.job_rows_per_s(4, 8192, 10, 50.0) == pytest.approx(4 * 8192 * 10 / 0.05)


def test_step_rates():
    # one figure per step: 2 GB in 0.01 s is 200 GB/s, in 0.02 s 100 GB/s
    assert bench.step_gbs(2e9, [0.01, 0.02]) == [200.0, 100.0]
    assert bench.step_gbs(1e9, []) == []
