"""Host logic of bench.py that needs no GPU: the roofline's DRAM traffic is taken
from the committed ncu summary only while that summary was captured on the
current kernel source, and the workload shapes follow their definitions."""

import os
import shutil

import numpy as np

import bench

SRC = ("decode.cu", "kitty_common.cuh", "quant_tile.cuh")


def _tree(tmp_path):
    """A copy of the files the traffic lookup reads, under tmp_path."""
    csrc = tmp_path / "mixed_precision_bit_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for f in SRC:
        shutil.copy(os.path.join(bench.ROOT, "mixed_precision_bit_gb300", "csrc", f), csrc / f)
    (tmp_path / "profiles").mkdir()
    shutil.copy(os.path.join(bench.ROOT, "profiles", "decode_kernel_budget_layer.md"),
                tmp_path / "profiles" / "decode_kernel_budget_layer.md")
    return csrc


def test_traffic_ratio_is_plausible_or_absent():
    r = bench.profiled_traffic_ratio()
    # DRAM traffic can sit a little above the algorithmic bytes (split partials,
    # re-read query rows), never below
    assert r is None or 1.0 <= r < 1.1


def test_traffic_ratio_dropped_when_a_kernel_source_changes(tmp_path, monkeypatch):
    expected = bench.profiled_traffic_ratio()
    csrc = _tree(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.profiled_traffic_ratio() == expected
    for f in SRC:
        p = csrc / f
        original = p.read_bytes()
        p.write_bytes(original + b"\n// a comment changes no code\n\n")
        assert bench.profiled_traffic_ratio() == expected, f
        p.write_bytes(original + b"\nnamespace { constexpr int kUnusedChange = 1; }\n")
        assert bench.profiled_traffic_ratio() is None, f
        p.write_bytes(original)
    assert bench.profiled_traffic_ratio() == expected
    (tmp_path / "profiles" / "decode_kernel_budget_layer.md").unlink()
    assert bench.profiled_traffic_ratio() is None


def test_budget_workload_shape():
    spec = bench.workload_spec("budget", 60)
    assert (spec["B"], spec["Hq"], spec["Hkv"], spec["layers"], spec["n_hi"]) == (177, 32, 8, 32, 32)
    assert spec["running"] and (spec["pages"] == 256).all()
    assert spec["tails"].min() >= 0 and spec["tails"].max() <= 31
    uni = bench.workload_spec("budget_uniform", 60)
    assert uni["n_hi"] == 0 and not uni["running"] and uni["B"] > spec["B"]


def test_headroom_covers_every_step():
    tails = np.array([0, 31, 17])
    for steps in (1, 31, 32, 33, 100):
        h = bench.headroom_pages(tails, steps)
        # the fullest tail gains `steps` tokens: every page it completes needs a slot
        assert h * 32 >= int(tails.max()) + steps
