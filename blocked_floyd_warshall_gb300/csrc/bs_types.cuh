// Types and constants the kernels are built from: the tile sizes, the view of
// a batch of matrices a launch receives, the profile categories and the tile
// sets of a phase-3 launch.  (Host-side declarations live in bs_internal.cuh.)
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace bs {

// Floyd-Warshall block (tile) sizes of the three-phase schedule: 128 for large
// matrices, 64 for small ones (an eighth of the serial phase-1 work per block
// round, and four times the tiles to spread over the SMs).
constexpr int FB_LARGE = 128;
constexpr int FB_SMALL = 64;

// One batch of matrices as the kernels see it.
struct Mats {
    void* U;
    void* L;              // nullptr: upper bounds only
    int n;
    int ld;
    long long bstride;    // elements between molecules
    int batch;
    bool vec;             // 16-byte vector IO allowed (ld % 4 == 0, bases 16B-aligned)
    int fb;               // blocked mode: tile size FB_LARGE or FB_SMALL
    bool sym;             // blocked mode: inputs symmetric, compute half and mirror
    int sms;              // multiprocessors of the device
};

// profile categories (the index of bs_profile's arrays)
enum Phase { PH_ROUND = 0, PH_ONE = 1, PH_TWO = 2, PH_THREE = 3, PH_NEXT = 4, PH_FUSED = 5 };

// Which tiles a phase-3 launch covers (see p3_tile in p3_tile.cuh).  The
// last four belong to the schedule that takes block rounds in pairs.
enum {
    P3_ALL = 0, P3_NEXT = 1, P3_REST = 2, P3_PANELS = 3, P3_ALL_OFF = 4,
    P3_REST2 = 5, P3_NEAR2 = 6, P3_PREV2 = 7, P3_CORNER2 = 8
};

}  // namespace bs
