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
};

static const TileEntry kTileTable[] = {
    // fp8 cls C     K     TRS  m_lo     m_hi       BN   BK  st  grp split
    {0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0},   // sentinel (never matches: C = 0)
};

}  // namespace c3d
