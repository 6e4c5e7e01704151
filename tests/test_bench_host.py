"""Host-side logic of bench.py (no GPU): which sources key a profiled kernel's DRAM
traffic, when a committed figure is reported and when it goes stale, and the
roofline fraction's arithmetic."""
from __future__ import annotations

import os
import shutil

import pytest

import bench

CSRC = os.path.join("tiled_exact_attention_gb300", "csrc")

# every kernel key the bench asks profiles/traffic.md for
BENCH_KEYS = [
    "fa_prefill_kernel", "fa_prefill_kernel_gqa", "fa_prefill_kernel_d64", "fa_prefill_kernel_d256",
    "fa_prefill_kernel_e4m3", "fa_prefill_kernel_e4m3_d64", "fa_prefill_kernel_e4m3_d256",
    "fa_decode_kernel", "fa_decode_kernel_b1", "fa_decode_kernel_d64", "fa_decode_kernel_e4m3",
    "fa_bwd_dkdv_kernel",
]


@pytest.fixture
def tree(tmp_path, monkeypatch):
    """A copy of the kernel sources and of the traffic table, with bench.py pointed at it."""
    shutil.copytree(os.path.join(bench.ROOT, CSRC), tmp_path / CSRC)
    (tmp_path / "profiles").mkdir()
    shutil.copy(os.path.join(bench.ROOT, "profiles", "traffic.md"), tmp_path / "profiles" / "traffic.md")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    return tmp_path


def _touch(tree, name):
    with open(tree / CSRC / name, "a") as f:
        f.write("\n// edited\n")


def test_every_bench_key_has_a_source_family():
    for key in BENCH_KEYS:
        fam = next((k for k in bench.KERNEL_SOURCES if key.startswith(k)), None)
        assert fam is not None, key
        for f in bench.KERNEL_SOURCES[fam]:
            assert os.path.exists(os.path.join(bench.ROOT, CSRC, f)), f
    assert bench._kernel_source_hash("some_other_kernel") is None


def test_every_bench_key_has_a_row_in_the_traffic_table():
    rows = {}
    with open(os.path.join(bench.ROOT, "profiles", "traffic.md")) as f:
        for line in f:
            parts = [x.strip() for x in line.strip().strip("|").split("|")]
            if len(parts) == 4 and parts[0].startswith("fa_"):
                rows[parts[0]] = parts
    for key in BENCH_KEYS:
        assert key in rows, key
        h, nbytes, capture = rows[key][1:]
        assert len(h) == 16 and int(h, 16) >= 0
        assert int(nbytes) > 0
        assert os.path.exists(os.path.join(bench.ROOT, "profiles", capture)), capture


def test_a_family_edit_stales_only_that_family(tree):
    before = {k: bench._profiled_traffic(k) for k in BENCH_KEYS}
    hashes = {k: bench._kernel_source_hash(k) for k in BENCH_KEYS}
    _touch(tree, "fa_backward.cu")
    after = {k: bench._profiled_traffic(k) for k in BENCH_KEYS}
    for k in BENCH_KEYS:
        if k.startswith("fa_bwd_"):
            assert bench._kernel_source_hash(k) != hashes[k]
            assert after[k] is None
        else:
            assert bench._kernel_source_hash(k) == hashes[k]
            assert after[k] == before[k]


def test_a_shared_header_edit_stales_every_family(tree):
    _touch(tree, "fa_internal.h")
    assert all(bench._profiled_traffic(k) is None for k in BENCH_KEYS)


def test_traffic_is_read_when_the_hash_matches(tree):
    key = "fa_prefill_kernel"
    h = bench._kernel_source_hash(key)
    with open(tree / "profiles" / "traffic.md", "w") as f:
        f.write("| kernel | source hash | bytes per launch | capture |\n|---|---|---|---|\n")
        f.write(f"| {key} | {h} | 12345 | x.md |\n")
        f.write(f"| fa_decode_kernel | {'0' * 16} | 999 | y.md |\n")
    assert bench._profiled_traffic(key) == 12345
    assert bench._profiled_traffic("fa_decode_kernel") is None  # captured on other sources
    assert bench._profiled_traffic("fa_bwd_dkdv_kernel") is None  # no row


def test_tensor_roofline_fraction_is_value_over_the_burst_peak():
    burst = bench._peak_tflops()[0]
    r = bench._tensor_roofline(burst / 2)
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    assert r["frac"] == pytest.approx(0.5, abs=1e-4)
    r8 = bench._tensor_roofline(burst / 2, ratio=2.0)
    assert r8["peak"] == pytest.approx(2 * burst, abs=0.1)
    assert r8["frac"] == pytest.approx(0.25, abs=1e-4)
