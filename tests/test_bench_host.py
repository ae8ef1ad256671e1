"""Host-side logic of bench.py: the algorithmic byte counts behind the
roofline, the profile lookup that supplies the DRAM traffic, and the labels
of the JSON line (no GPU)."""
import argparse
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from combine_ep_layout_05_gb300 import inputs  # noqa: E402


def test_algorithmic_bytes_prefill():
    # 8 ranks x 4096 tokens, H 7168, top-8: read x once, write D rows, read
    # them back, write out (plus routing and slots)
    T, H, k, R, E, N, D = 32768, 7168, 8, 8, 256, 1, 173443
    b = bench.algorithmic_bytes(T, H, k, R, E, N, D)
    assert b["dispatch"] == T * H * 2 + T * R * 4 + D * H * 2
    assert b["combine"] == D * H * 2 + T * k * 12 + T * R * 4 + T * H * 2
    assert b["layout"] == T * k * 8 + T * R + 2 * T * R * 4 + T * k * 4
    total = b["dispatch"] + b["combine"]
    assert abs(total - 5.914e9) < 0.01e9     # the prefill figure of the scope table


def test_algorithmic_bytes_variants():
    T, H, k, R, E, N, D, A = 65536, 7168, 8, 16, 256, 2, 151045, 67486
    b = bench.algorithmic_bytes(T, H, k, R, E, N, D, A=A)
    # two-level: the staged rows are written and read once each way
    assert b["dispatch"] == T * H * 2 + T * R * 4 + 2 * A * H * 2 + D * H * 2
    assert b["combine"] == D * H * 2 + T * k * 12 + T * R * 4 + 2 * A * H * 2 + T * H * 2
    f = bench.algorithmic_bytes(1024, H, k, 8, 256, 1, 8192, dtype="fp8_e4m3")
    assert f["expert"] == 8192 * ((H + H // 128 * 4) + H * 2)
    for fmt, row in (("mxfp8", H + H // 32), ("nvfp4", H // 2 + H // 8)):
        assert bench.wire_row_bytes(H, fmt) == row
        w = bench.algorithmic_bytes(T, H, k, R, E, N, D, combine_fmt=fmt)
        assert w["combine"] == D * row + T * k * 12 + T * R * 4 + T * H * 2
        assert w["wire"] == D * (H * 2 + row)


def test_traffic_keys_and_sources():
    a = argparse.Namespace(two_level=False, combine_fmt="bf16")
    assert bench.traffic_key("dispatch", a) == "dispatch"
    assert bench.traffic_key("combine", a) == "combine"
    a2 = argparse.Namespace(two_level=True, combine_fmt="bf16")
    assert bench.traffic_key("combine", a2) == "combine_two_level"
    assert bench.traffic_key("dispatch", a2) == "dispatch_two_level"
    aw = argparse.Namespace(two_level=False, combine_fmt="nvfp4")
    assert bench.traffic_key("combine", aw) == "combine_nvfp4"
    assert bench.traffic_key("wire", aw) == "wire_nvfp4"
    # every key names existing source files
    for key, files in bench.KERNEL_SOURCES.items():
        for f in files:
            assert os.path.exists(os.path.join(ROOT, f)), (key, f)


def test_profile_traffic_needs_matching_sources(tmp_path, monkeypatch):
    assert bench.profile_traffic("no_such_kernel", bench.KERNEL_SOURCES["dispatch"]) is None
    # a summary is used only while its hash matches the sources
    prof = tmp_path / "profiles"
    prof.mkdir()
    h = bench.source_hash(bench.KERNEL_SOURCES["combine"])
    (prof / "combine_w.md").write_text(f"traffic_bytes_per_launch: 1.5e9\nsource_sha256: {h}\n")
    (prof / "dispatch_w.md").write_text("traffic_bytes_per_launch: 1.5e9\nsource_sha256: 0000000000000000\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "source_hash", lambda files, _h=h: _h if files is bench.KERNEL_SOURCES["combine"]
                        else "ffffffffffffffff")
    assert bench.profile_traffic("combine", bench.KERNEL_SOURCES["combine"], "w") == 1.5e9
    assert bench.profile_traffic("dispatch", bench.KERNEL_SOURCES["dispatch"], "w") is None


@pytest.mark.parametrize("name", list(inputs.WORKLOADS))
def test_config_labels(name):
    wl = inputs.WORKLOADS[name]
    c = bench._config(wl)
    assert c["workload"] == name and c["tokens"] == wl.tokens
    assert "model" not in c
    label = c["routing"]
    if wl.routing == "group_limited":
        assert "group-limited" in label
    elif wl.zipf_s:
        assert "Zipf" in label
    else:
        assert "uniform" in label


def test_same_mix_peak_reads_the_probe_summary(tmp_path, monkeypatch):
    prof = tmp_path / "profiles"
    prof.mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.same_mix_peak("w") is None
    (prof / "hbm_mix_w.md").write_text("# probe\n\nsame_mix_bound_gbs: 6123.4\n")
    peak, src = bench.same_mix_peak("w")
    assert peak == 6123.4 and src == os.path.join("profiles", "hbm_mix_w.md")


def test_hold_gpu_is_a_no_op_without_time():
    bench.hold_gpu(0.0)   # no launch, no GPU needed


def test_one_launch_layout_dispatch_policy():
    # the pipeline's default: one ep_layout_dispatch launch for small
    # problems the library's single small-problem kernel covers, up to 32
    # tokens per rank; two calls otherwise
    from combine_ep_layout_05_gb300.pipeline import one_launch_layout_dispatch as one
    assert one(32, 4, "bf16")                  # decode workload
    assert one(8 * 32, 8, "fp8_e4m3")          # 32 tokens/rank
    assert not one(1024, 8, "fp8_e4m3")        # low-latency workload: 128 tokens/rank, two calls
    assert not one(32768, 8, "bf16")           # prefill
    assert not one(8 * 256, 8, "bf16")         # 256 tokens/rank
    assert not one(64 * 32, 64, "bf16")        # bf16 from 2048 tokens: bulk copies, two calls
    assert one(64 * 32, 64, "fp8_e4m3")
    assert not one(64 * 128, 64, "fp8_e4m3")   # 63 x 128 tokens before the last source rank
    assert not one(256 * 32, 256, "fp8_e4m3")  # 255 x 32 tokens before the last source rank
