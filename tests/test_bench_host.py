"""CPU tests of bench.py's host-side pieces: the workload description, the L2 note, the
DRAM-traffic record's source-hash check, and the parsing of nvidia-smi clock samples."""

import hashlib
import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from quantization_aware_attention_gb300.inputs import WORKLOADS, Workload  # noqa: E402


def test_workload_text_follows_the_shape():
    assert bench.workload_config(WORKLOADS["c4"])["workload"].startswith(
        "c4: video-DiT self-attention B=1 H=40 Nq=Nkv=32768 D=128 non-causal")
    w = Workload("custom", 9, 4, 32, 8192, 8192, 128, causal=True)
    assert "Nq=8192 Nkv=8192 D=128 causal" in bench.workload_config(w)["workload"]
    w = Workload("custom", 9, 1, 40, 16384, 512, 128)
    assert "Nq=16384 Nkv=512 D=128 non-causal" in bench.workload_config(w)["workload"]


def test_l2_note_says_when_inputs_fit_in_l2():
    assert bench.l2_note(WORKLOADS["c4"]).startswith("inputs larger than L2 (335.5 MB")
    assert "not a measurement under the timing rules" in bench.l2_note(WORKLOADS["c1"])


def test_kernel_traffic_is_null_once_a_source_changes(tmp_path, monkeypatch):
    src = tmp_path / "k.cu"
    src.write_bytes(b"kernel v1\n")
    (tmp_path / "profiles").mkdir()
    rec = {"kern": {"dram_bytes_per_launch": 1234, "source": "k.cu",
                    "sha256": hashlib.sha256(b"kernel v1\n").hexdigest()},
           "other": {"dram_bytes_per_launch": 10, "source": "k.cu",
                     "sha256": hashlib.sha256(b"kernel v1\n").hexdigest()}}
    (tmp_path / "profiles" / "roofline_traffic.json").write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.kernel_traffic("kern") == 1234
    assert bench.kernel_traffic("kern", "other") == 1244
    assert bench.kernel_traffic("missing") is None
    src.write_bytes(b"kernel v2\n")
    assert bench.kernel_traffic("kern") is None


class _FakeProc:
    def terminate(self):
        pass

    def wait(self, timeout=None):
        return 0


def test_clock_sampler_median_and_reasons():
    cs = bench.ClockSampler(0)
    cs.proc = _FakeProc()
    cs.lines = [
        "0, 1950, 2070, 1100.5, 0x4, Not Active, Not Active, Not Active, Active",
        "0, 1980, 2070, 1200.0, 0x4, Not Active, Not Active, Not Active, Active",
        "0, 1900, 2070, 1150.0, 0x0, Not Active, Not Active, Not Active, Not Active",
        "garbled line",
    ]
    r = cs.stop()
    assert r["sm_mhz"] == pytest.approx(1950.0)
    assert r["sm_max_mhz"] == pytest.approx(2070.0)
    assert r["reasons"] == ["sw_power_cap"]
    assert r["samples"] == 3


def test_clock_sampler_without_nvidia_smi():
    assert bench.ClockSampler(0).stop()["reasons"] == ["nvidia-smi unavailable"]
