"""Writes the stored expected values under tests/golden/.  Calls only the
oracle and the seeded input generators.

Usage:  python tests/golden/make_golden.py
"""
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402
import trsm_inputs as ti  # noqa: E402


def solve_tri_8x64x6():
    """The batched f32 shape of llama.cpp PR 17457 ("SOLVE_TRI CUDA kernel for
    small matrices", the test-backend-ops benchmark line ne_lhs=[64,64,4,2],
    ne_rhs=[6,64,4,2]): 8 row-major systems, 64 x 64, 6 right-hand sides."""
    w = ti.WORKLOADS["solve_tri_8x64x6"]
    m, n, batch = w["m"], w["n"], w["batch"]
    L, B = ti.generate("f32", m, n, batch, kind=w["kind"])
    a = ti.to_storage(L, "row")
    b = ti.to_storage(B, "row")
    oracle.trsm_llnn("f32", m, n, 1.0, a, m, b, n, layout="row", stride_a=m * m,
                     stride_b=m * n, batch=batch)
    path = os.path.join(HERE, "solve_tri_8x64x6_f32.txt")
    with open(path, "w") as f:
        f.write("# X = L^-1 B for the 8 x (64 x 64, 6 RHS) f32 row-major batch, seed 0,\n")
        f.write("# L strictly lower U(-0.1,0.1), diagonal U(1,2); B U(-1,1); alpha = 1.\n")
        f.write("# Shape from llama.cpp PR 17457 (test-backend-ops SOLVE_TRI line).\n")
        f.write("# Written by tests/golden/make_golden.py from the oracle.\n")
        f.write("# One line per row of the row-major (8*64) x 6 result, float32 as hex.\n")
        for r in b.reshape(batch * m, n):
            f.write(" ".join(float(v).hex() for v in r) + "\n")
    return path


if __name__ == "__main__":
    print(solve_tri_8x64x6())
