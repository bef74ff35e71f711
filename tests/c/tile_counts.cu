// Host-side check of the phase-3 launch sizes: prints p3_tiles (the grid of
// every phase-3 launch) for each tile set, symmetry, block-row count and
// block round, for tests/test_tile_counts.py to compare with the sets'
// definitions.  Runs on the host only; no device code is called.
#include <cstdio>

#include "../../blocked_floyd_warshall_gb300/csrc/p3_tile.cuh"

int main() {
    using namespace bs;
    const int parts[] = {P3_ALL,    P3_NEXT,  P3_REST,  P3_PANELS, P3_ALL_OFF,
                         P3_REST2,  P3_NEAR2, P3_PREV2, P3_CORNER2};
    for (int part : parts)
        for (int sym = 0; sym < 2; ++sym)
            for (int nb = 1; nb <= 24; ++nb)
                for (int K = 0; K < nb; ++K)
                    std::printf("%d %d %d %d %d\n", part, sym, nb, K, p3_tiles(sym != 0, part, nb, K));
    return 0;
}
