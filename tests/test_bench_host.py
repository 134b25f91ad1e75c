"""Host logic of bench.py that needs no GPU: the include closure a kernel's
recorded ncu traffic is tied to, and the validity check of that record."""
import json
import os

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _names(paths):
    return {os.path.relpath(p, ROOT) for p in paths}


def test_closure_follows_quoted_includes_transitively():
    got = _names(bench.source_closure("small_fast_c128.cu"))
    csrc = "triangular_solve_gb300/csrc/"
    # the unit, its headers, their headers, and the public header through
    # a relative path and through the include directory
    for f in ("small_fast_c128.cu", "small_fast.cuh", "small_kernels.cuh", "small_launch.cuh", "mbarrier.cuh",
              "common.cuh", "internal.h"):
        assert csrc + f in got, f
    assert "include/trsm.h" in got
    # nothing it does not include
    assert csrc + "tc_gemm.cu" not in got and csrc + "tc_gemm.cuh" not in got
    assert len(got) == len(set(got))


def test_closure_hash_moves_with_its_files_only(tmp_path, monkeypatch):
    csrc = tmp_path / "triangular_solve_gb300" / "csrc"
    inc = tmp_path / "include"
    csrc.mkdir(parents=True)
    inc.mkdir()
    (inc / "api.h").write_text("int f();\n")
    (csrc / "a.cuh").write_text('#include "../../include/api.h"\n')
    (csrc / "k.cu").write_text('#include "a.cuh"\n#include <stdio.h>\n')
    (csrc / "other.cu").write_text("int g;\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert _names_rel(bench.source_closure("k.cu"), tmp_path) == {
        "triangular_solve_gb300/csrc/k.cu", "triangular_solve_gb300/csrc/a.cuh", "include/api.h"}
    h0 = bench.kernel_source_hash("k.cu")
    (csrc / "other.cu").write_text("int g = 1;\n")  # outside the closure
    assert bench.kernel_source_hash("k.cu") == h0
    (inc / "api.h").write_text("int f(int);\n")    # inside, two levels down
    assert bench.kernel_source_hash("k.cu") != h0


def _names_rel(paths, root):
    return {os.path.relpath(p, root) for p in paths}


def test_recorded_traffic_needs_a_matching_hash(tmp_path, monkeypatch):
    csrc = tmp_path / "triangular_solve_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (tmp_path / "profiles").mkdir()
    (csrc / "k.cu").write_text("int x;\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    rec = {"k/w": {"translation_unit": "k.cu", "source_hash": bench.kernel_source_hash("k.cu"),
                   "dram_bytes_per_launch": 123}}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(rec))
    assert bench.recorded_traffic("k/w") == 123
    assert bench.recorded_traffic("missing/w") is None
    (csrc / "k.cu").write_text("int x = 2;\n")
    assert bench.recorded_traffic("k/w") is None


def test_committed_records_name_their_units():
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        d = json.load(f)
    for key, e in d.items():
        if isinstance(e, dict):
            assert os.path.exists(os.path.join(ROOT, "triangular_solve_gb300", "csrc", e["translation_unit"])), key
            assert len(e["source_hash"]) == 16
