"""The bench's reporting helpers, on the CPU: roofline arithmetic, and DRAM
traffic records that apply only while the kernel's sources are unchanged."""
import os
import types

import pytest

import bench


def _case(kind="affine_sample", dtype="float32", nbytes=268436992, flops=0.0,
          tag="band_kernel<f32,linear>", name="stn2d"):
    return types.SimpleNamespace(w=types.SimpleNamespace(kind=kind), dtype=dtype, bytes=nbytes,
                                 flops=flops, kernel_tag=tag, name=name)


PEAKS = {"hbm_gbs": 8000.0, "bf16_tflops": 2000.0, "bf16_tflops_sustained": 1800.0,
         "source": "measured"}


def test_hbm_roofline_is_algorithmic_bytes_over_time(monkeypatch):
    monkeypatch.setattr(bench, "recorded_traffic", lambda *a: None)
    r = bench.roofline_for(_case(nbytes=400_000_000), 0.1, PEAKS)   # 400 MB in 0.1 ms
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert r["achieved"] == pytest.approx(4000.0)
    assert r["frac"] == pytest.approx(0.5)
    assert r["algorithmic_bytes"] == 400_000_000 and r["traffic"] is None


def test_deform_conv_in_16_bit_is_tensor_bound(monkeypatch):
    monkeypatch.setattr(bench, "recorded_traffic", lambda *a: 123.0)
    r = bench.roofline_for(_case(kind="deform_conv", dtype="bfloat16", flops=2.0e12), 10.0, PEAKS)
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    assert r["achieved"] == pytest.approx(200.0)    # 2 TFLOP in 10 ms
    assert r["frac"] == pytest.approx(0.1)
    assert r["traffic"] == 123.0
    # fp32 DeformConv contracts on FFMA: reported against the fp32 FMA peak
    # derived from the SM count and clock (152 x 128 x 2 x 2.07 GHz)
    r32 = bench.roofline_for(_case(kind="deform_conv", dtype="float32", flops=8.0e9), 1.0, PEAKS)
    assert r32["bound"] == "alu" and r32["unit"] == "TFLOP/s"
    assert r32["achieved"] == pytest.approx(8.0)    # 8 GFLOP in 1 ms
    assert r32["peak"] == pytest.approx(80.5, abs=0.1)
    assert r32["frac"] == pytest.approx(8.0 / (152 * 128 * 2 * 2.07e9 / 1e12), rel=1e-3)


def _tree(tmp_path, source="int a;"):
    csrc = tmp_path / "spatial_transformer_sampling_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for name in bench.KERNEL_SOURCES["band_kernel"]:
        (csrc / name).write_text(source if name == "gs_band.cuh" else name)
    (tmp_path / "profiles").mkdir()
    return csrc


def test_traffic_record_applies_only_to_the_sources_it_was_taken_on(tmp_path, monkeypatch):
    csrc = _tree(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    tag = "band_kernel<f32,linear>"
    sha = bench.kernel_source_sha(tag)
    (tmp_path / "profiles" / "dram_traffic.txt").write_text(
        "# comment\n\n"
        f"kernel={tag} workload=stn2d dtype=float32 src_sha={sha} dram_bytes_per_launch=221243136\n"
        f"kernel={tag} workload=stn2d dtype=bfloat16 src_sha=0000 dram_bytes_per_launch=5\n")
    assert bench.recorded_traffic(tag, "stn2d", "float32") == 221243136.0
    assert bench.recorded_traffic(tag, "stn2d", "bfloat16") is None     # other sources
    assert bench.recorded_traffic(tag, "stn3d", "float32") is None      # no record
    # any change to one of the kernel's files retires the record
    (csrc / "gs_band.cuh").write_text("int b;")
    assert bench.kernel_source_sha(tag) != sha
    assert bench.recorded_traffic(tag, "stn2d", "float32") is None


def test_source_hash_covers_only_the_kernel_files(tmp_path, monkeypatch):
    csrc = _tree(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    sha = bench.kernel_source_sha("band_kernel<bf16,linear>")
    (csrc / "gs_unrelated.cu").write_text("int c;")
    assert bench.kernel_source_sha("band_kernel<bf16,linear>") == sha
    assert bench.kernel_source_sha() != sha     # no tag: every file


def test_missing_peaks_file_falls_back(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    pk = bench.peaks()
    assert pk["source"] == "fallback" and pk["hbm_gbs"] == 6800.0
    (tmp_path / "MEASURED_PEAKS.json").write_text('{"hbm_gbs": 7000, "bf16_tflops": 1950}')
    pk = bench.peaks()
    assert pk["source"] == "measured" and pk["hbm_gbs"] == 7000.0
    assert pk["bf16_tflops_sustained"] == 1950.0   # absent: the burst figure


def test_every_kernel_tag_has_its_sources_in_the_tree():
    csrc = os.path.join(bench.ROOT, "spatial_transformer_sampling_gb300", "csrc")
    for tag, files in bench.KERNEL_SOURCES.items():
        for f in files:
            assert os.path.exists(os.path.join(csrc, f)), (tag, f)
