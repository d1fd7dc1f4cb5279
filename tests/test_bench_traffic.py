"""bench.py host logic: a recorded DRAM traffic figure is reported only while the source files of
its kernel family are unchanged, and a change elsewhere in the CUDA sources does not void it."""
import json
import os
import shutil
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _tree(tmp_path):
    csrc = tmp_path / "quantized_moe_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for names in bench.KERNEL_SOURCES.values():
        for n in names:
            (csrc / n).write_text(f"// {n}\n")
    (csrc / "router.cu").write_text("// router\n")
    (tmp_path / "profiles").mkdir()
    return csrc


def test_traffic_follows_its_family_hash(tmp_path, monkeypatch):
    csrc = _tree(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    rec = {"prefill-4096:routed_gateup": {"dram_bytes_per_launch": 123.0, "source_hash": bench.kernel_source_hash("gemm")},
           "decode-1:gateup": {"dram_bytes_per_launch": 45.0, "source_hash": bench.kernel_source_hash("decode")}}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(rec))
    assert bench.recorded_traffic("routed_gateup", "prefill-4096") == 123.0
    assert bench.recorded_traffic("gateup", "decode-1") == 45.0
    # a kernel of another family changes: both records stay valid
    (csrc / "router.cu").write_text("// router, changed\n")
    assert bench.recorded_traffic("routed_gateup", "prefill-4096") == 123.0
    # the GEMM changes: its record is void, the decode record is not
    (csrc / "gemm_tc.cu").write_text("// gemm, changed\n")
    assert bench.recorded_traffic("routed_gateup", "prefill-4096") is None
    assert bench.recorded_traffic("gateup", "decode-1") == 45.0
    # a header both families include voids both
    (csrc / "common.cuh").write_text("// common, changed\n")
    assert bench.recorded_traffic("gateup", "decode-1") is None


def test_unknown_kernel_or_workload_has_no_traffic(tmp_path, monkeypatch):
    _tree(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.recorded_traffic("routed_gateup", "prefill-4096") is None  # no file
    (tmp_path / "profiles" / "traffic.json").write_text("{}")
    assert bench.recorded_traffic("combine", "prefill-4096") is None
    assert bench.recorded_traffic("routed_gateup", "prefill-512") is None


def test_every_family_file_exists():
    csrc = os.path.join(ROOT, "quantized_moe_gb300", "csrc")
    for fam, names in bench.KERNEL_SOURCES.items():
        for n in names:
            assert os.path.exists(os.path.join(csrc, n)), (fam, n)
    assert set(bench.TRAFFIC_FAMILY.values()) <= set(bench.KERNEL_SOURCES)
