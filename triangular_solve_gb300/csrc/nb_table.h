// Compile-time "problem size x element type -> block size NB" table of the
// blocked path ("Hierarchical Shared Memory-Aware Optimization for TRSM on
// GPU Platforms", adaptive blocking: an offline sweep keeps the best NB per
// (size, type); at run time the nearest tabulated size is looked up).
//
// Entries: {dtype, m, NB}.  The sweep behind them is reproduced by
// bench.py --nb-sweep; each row holds the NB with the highest measured
// GFLOPS for square m = n on one GB300.
#pragma once

namespace trsm {

struct NbEntry {
    int dtype;  // trsm_dtype_t
    int m;
    int nb;
};

// Provisional values until the GB300 sweep is recorded: the pages' reported
// trend (NB 256 at m = 1024 growing to 512 at m = 8192).
constexpr NbEntry kNbTable[] = {
    {0, 1024, 256}, {0, 2048, 256}, {0, 4096, 512}, {0, 8192, 512}, {0, 16384, 512},
    {1, 1024, 256}, {1, 2048, 256}, {1, 4096, 512}, {1, 8192, 512}, {1, 16384, 512},
    {2, 1024, 256}, {2, 2048, 256}, {2, 4096, 512}, {2, 8192, 512}, {2, 16384, 512},
    {3, 1024, 256}, {3, 2048, 256}, {3, 4096, 512}, {3, 8192, 512}, {3, 16384, 512},
};

}  // namespace trsm
