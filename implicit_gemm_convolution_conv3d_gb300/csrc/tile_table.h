// tile_table.h -- per-shape tile choices for conv_fwd, filled from a measured
// sweep on GB300 (sweep_tiles.py beside the package re-measures and prints
// the rows).  A row matches on (dtype, dispatch class, C, K, T*R*S) and an
// inclusive range of GEMM rows M; 0 in a tile field keeps the default rule.
#pragma once

namespace c3d {

struct TileEntry {
    int fp8;            // 0 bf16, 1 e4m3
    int cls;            // conv_class
    long long C, K, TRS;
    long long m_lo, m_hi;
    int BN, BK, stages, group_m, splits;
    int pair;           // CTA-pair kernel: -1 default rule, 0 off, 1 on
    int msub;           // row sub-tiles sharing each B stage: 0 default rule, 1 or 2
};

static const TileEntry kTileTable[] = {
    // fp8 cls C     K     TRS  m_lo     m_hi       BN   BK  st  grp split pair msub
    {0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, -1, 0},   // sentinel (never matches: C = 0)
    // measured on GB300 (sweep_tiles.py --quick, then an interleaved A/B of
    // the leaders under the power cap, and of the leaders against these
    // rows; medians of 18-60 L2-flushed runs):
    {0, 0, 2048, 2048, 27, 100000, 1LL << 40, 256, 128, 0, 1, 0, 1, 0},   // video 3x3x3: 24.98 ms
    {1, 0, 1024, 1024, 9, 100000, 1LL << 40, 256, 256, 0, 8, 0, 1, 1},    // fp8 1x3x3: 9.38 ms
    {0, 1, 640, 640, 3, 100000, 1LL << 40, 224, 256, 0, 4, 0, 1, 1},      // temporal 3x1x1: 5.43 ms
    {0, 2, 3, 1280, 196, 4096, 1LL << 40, 224, 128, 0, 4, 0, 0, 1},      // patch 14x14: 0.031 ms
    // backward data of the 14x14x3 patch embedding: dy [M, 1280] x w^T [588, 1280]
    {0, 2, 1280, 588, 1, 4096, 1LL << 40, 160, 256, 0, 1, 0, 1, 1},      // 28.3 us (33.5 default)
};

}  // namespace c3d
