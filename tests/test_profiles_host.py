"""The committed traffic record that the benchmark's roofline object reads:
internally consistent, and reported only while the kernel sources are the ones
it was captured from.  No GPU is needed."""
import json
import os

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PATH = os.path.join(ROOT, "profiles", "traffic.json")


def load():
    with open(PATH) as f:
        return json.load(f)


def test_per_kernel_bytes_sum_to_the_forward():
    for workload, e in load().items():
        per = e["per_kernel"]
        total = sum(v["read"] + v["write"] for v in per.values())
        assert total == e["dram_bytes_per_launch"], workload
        assert len(e["source_digest"]) == 16 and "ncu" in e["command"]
        # the --clock-control flag is part of every recorded capture
        assert "--clock-control none" in e["command"]


def test_recorded_traffic_is_plausible_for_the_bench_layer():
    # 2-D fp32 bench layer: x, w, y once = 37 748 736 bytes; a capture far
    # above that would mean re-reads, far below a capture of the wrong work
    e = load()["2d_f32"]
    assert 0.5 * 37748736 < e["dram_bytes_per_launch"] < 2.0 * 37748736


def test_recorded_traffic_is_plausible_for_the_headline_layer():
    # 2-D fp16 layer: x, w, y once = 570 425 344 bytes
    e = load()["2d_f16"]
    assert 0.9 * 570425344 < e["dram_bytes_per_launch"] < 1.3 * 570425344
    assert set(e["per_kernel"]) == {"k_phase_a_tc", "k_mix_tc", "k_inv16"}


def test_stale_record_is_not_reported(tmp_path, monkeypatch):
    d = load()
    d["2d_f32"]["source_digest"] = "0" * 16
    fake_root = tmp_path
    (fake_root / "profiles").mkdir()
    (fake_root / "profiles" / "traffic.json").write_text(json.dumps(d))
    csrc = fake_root / "fft_gemm_ifft_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "k.cu").write_text("// kernel")
    monkeypatch.setattr(bench, "ROOT", str(fake_root))
    assert bench.recorded_traffic("2d_f32") is None
    d["2d_f32"]["source_digest"] = bench.kernel_source_digest(d["2d_f32"].get("sources"))
    (fake_root / "profiles" / "traffic.json").write_text(json.dumps(d))
    assert bench.recorded_traffic("2d_f32") == d["2d_f32"]["dram_bytes_per_launch"]
    assert bench.recorded_traffic("no_such_workload") is None


def test_record_follows_only_its_own_sources(tmp_path, monkeypatch):
    # a record names the translation units of its kernels: editing another
    # unit keeps it, editing one of its own (or any header) retires it
    csrc = tmp_path / "fft_gemm_ifft_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (tmp_path / "profiles").mkdir()
    (csrc / "mine.cu").write_text("// a")
    (csrc / "other.cu").write_text("// b")
    (csrc / "shared.cuh").write_text("// c")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    rec = {"w": {"dram_bytes_per_launch": 5, "sources": ["mine.cu"],
                 "source_digest": bench.kernel_source_digest(["mine.cu"])}}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(rec))
    assert bench.recorded_traffic("w") == 5
    (csrc / "other.cu").write_text("// b changed")
    assert bench.recorded_traffic("w") == 5
    (csrc / "shared.cuh").write_text("// c changed")
    assert bench.recorded_traffic("w") is None
    rec["w"]["source_digest"] = bench.kernel_source_digest(["mine.cu"])
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(rec))
    (csrc / "mine.cu").write_text("// a changed")
    assert bench.recorded_traffic("w") is None
