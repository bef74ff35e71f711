// Internal declarations shared by the CUDA translation units of libbsmooth.
#pragma once

#include "bs_types.cuh"

namespace bs {

// Launch bookkeeping (api.cu): counts launches and, when profiling, records an
// event pair around each launch on `s`.
void before_launch(cudaStream_t s, int phase);
void after_launch(cudaStream_t s, int phase);
// Counts a launch without recording profile events.
void note_launch();

// Per-round (reference) mode, round k.
cudaError_t launch_round(bool is_int, const Mats& m, int k, bool literal, cudaStream_t s);
cudaError_t launch_cross(bool is_int, const Mats& m, int k, cudaStream_t s);
// Rounds k and k+1 in one pass, then their rows and columns (two launches).
cudaError_t launch_round2(bool is_int, const Mats& m, int k, bool literal, cudaStream_t s);

// Blocked mode, block round K.
cudaError_t blocked_setup(bool is_int);   // once per device: shared-memory limits
cudaError_t phase3_setup(bool is_int);
// pre: first apply block round K-1's update to tile (K,K) (its product with
// the panels of round K-1), which the look-ahead schedule then leaves out of
// phase 3 of round K-1; 64-wide tiles only.
cudaError_t launch_phase1(bool is_int, const Mats& m, int K, bool pre, cudaStream_t s);
cudaError_t launch_phase2(bool is_int, const Mats& m, int K, cudaStream_t s);
// Phase 3 of block round K over the tiles `part` selects (P3_* in bs_types.cuh).
cudaError_t launch_phase3(bool is_int, const Mats& m, int K, int part, cudaStream_t s);
// Symmetric mode, after the last block round: the lower triangle written as
// the transpose of the upper one.
cudaError_t launch_mirror(bool is_int, const Mats& m, cudaStream_t s);

// The whole blocked smoothing in one launch, one cluster per molecule
// (fused.cu); fused_setup once per device and dtype.
cudaError_t fused_setup(bool is_int);
cudaError_t launch_fused(bool is_int, const Mats& m, cudaStream_t s);
int fused_cluster_size();   // CTAs per cluster on the current device (0: not set up)

// Feasibility count and precondition checks.  `count` and `flags` are device
// words the caller has zeroed on `s`.
cudaError_t launch_feasible(bool is_int, const Mats& m, unsigned char* mask,
                            unsigned long long* count, cudaStream_t s);
cudaError_t launch_validate(bool is_int, const Mats& m, unsigned int* flags, cudaStream_t s);

// flag bits written by the validation kernel
enum : unsigned int {
    VF_DIAG = 1u,       // nonzero diagonal
    VF_NEG = 2u,        // negative value
    VF_NAN = 4u,        // NaN
    VF_LINF = 8u,       // infinite lower bound
    VF_RANGE = 16u,     // int32 value >= 2^30
    VF_ASYM = 32u       // Mats::sym set but U or L not symmetric
};

}  // namespace bs
