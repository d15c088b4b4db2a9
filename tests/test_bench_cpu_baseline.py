"""The benchmark's CPU-baseline suite runs the oracle on every workload kind
(here on tiny stand-ins of the five workloads) and labels what it
extrapolates. CPU only."""
import sys
import os

import pytest
import torch

import workloads

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_cpu_baseline_suite_tiny(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setattr(workloads, "TINY_FLAT", workloads.PrefillSpec("tiny", [300], 4, 1, 4))
    monkeypatch.setattr(workloads, "PAGED_DECODE",
                        workloads.DecodeSpec("dec", 6, (200, 3000), 16, 2, 8))
    monkeypatch.setattr(workloads, "MIXED_E4M3",
                        workloads.PrefillSpec("mixed", None, 8, 2, 8, kv_dtype="e4m3",
                                              draw_lengths=(3, 300, 1500)))
    monkeypatch.setattr(workloads, "TWO_STAGE", workloads.TwoStageSpec("ts", [1500], 8, 8, 2, 8))
    inp2 = workloads.make_prefill(
        workloads.PrefillSpec("fv", [1200, 900], 16, 2, 8, first_prev=True), 0, device="cpu")
    res = bench.cpu_baseline_suite("cpu", 4, inp2)
    assert set(res) == {"one_thread", "tiny_flat", "paged_decode_sq1", "paged_decode_sq4",
                        "mixed_e4m3", "two_stage"}
    assert res["one_thread"]["threads"] == 1
    for key in ("tiny_flat", "paged_decode_sq1", "paged_decode_sq4"):
        assert res[key]["sample"] == "full" and res[key]["tflops"] > 0
    for key in ("mixed_e4m3", "two_stage"):
        assert res[key]["extrapolated"] is True
        assert res[key]["full_seconds_extrapolated"] >= res[key]["seconds"]
