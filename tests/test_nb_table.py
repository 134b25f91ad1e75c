"""The compile-time NB table: generated from a sweep's JSON lines (best NB
per size and type), consistent with the committed sweep, and looked up by
nearest size at run time."""
import json
import os

import pytest

from triangular_solve_gb300 import nb_table_gen

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SWEEP = os.path.join(ROOT, "triangular_solve_gb300", "nb_sweep_gb300.jsonl")
HEADER = os.path.join(ROOT, "triangular_solve_gb300", "csrc", "nb_table.h")


def test_best_nb_keeps_fastest_block_size():
    lines = [json.dumps(r) for r in [
        {"dtype": "f64", "m": 1024, "nb": 128, "gflops": 900.0},
        {"dtype": "f64", "m": 1024, "nb": 256, "gflops": 1100.0},
        {"dtype": "f64", "m": 1024, "nb": 512, "gflops": 1000.0},
        {"dtype": "f64", "m": 1024, "best_nb": 256},
        {"dtype": "c64", "m": 4096, "nb": 512, "gflops": 5.0},
    ]] + ["not json", ""]
    best = nb_table_gen.best_nb(lines)
    assert best == {("f64", 1024): (256, 1100.0), ("c64", 4096): (512, 5.0)}
    text = nb_table_gen.render(best, "test", "x.jsonl")
    assert "{1, 1024, 256}" in text and "{2, 4096, 512}" in text


def test_committed_table_matches_committed_sweep():
    if not os.path.exists(SWEEP):
        pytest.skip("no sweep recorded yet")
    with open(SWEEP) as f:
        best = nb_table_gen.best_nb(f.readlines())
    header = open(HEADER).read()
    for (d, m), (nb, _) in best.items():
        assert f"{{{nb_table_gen.CODES[d]}, {m}, {nb}}}" in header, (d, m, nb)
