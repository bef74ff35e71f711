/*
 * bsmooth.h -- distance-bound smoothing on one GPU (sm_103a), C ABI.
 *
 * The operation (GPU Gems 2, ch. 43, "GPU Computing for Protein Structure
 * Prediction"):
 *   section 1 -- a molecule of n atoms is the complete graph K_n; pair (i, j)
 *     carries an upper bound U[i,j] and a lower bound L[i,j], stored as two
 *     dense n x n matrices with a zero diagonal;
 *   section 2 -- through every middle atom k the triangle inequality tightens
 *       U[i,j] <- min(U[i,j], U[i,k] + U[k,j])
 *       L[i,j] <- max(L[i,j], L[i,k] - U[k,j], L[k,j] - U[i,k])
 *     with the upper bound tightened before the lower bound uses it;
 *   section 3 -- Floyd-Warshall: k = 0..n-1 in order, all pairs updated in
 *     each round, each round seeing the matrix the previous round produced.
 *
 * Results.  Every smoothing call leaves U and L at the fixed point of those
 * inequalities: U[i,j] is the shortest path i..j over upper-bound edges, and
 *   L[i,j] = max(L0[i,j], max_{a,b} L0[a,b] - U[i,a] - U[b,j]).
 * Where L[k,k] > 0 (only for contradictory bounds) the lower-bound column
 * value of round k is first raised to max(L[i,k], L[k,k] - U[i,k]) (the
 * "closure" rule); with consistent bounds L[k,k] stays 0 and this is the
 * printed rule exactly.  BS_RULE_LITERAL keeps the printed formula as is, and
 * is accepted by the per-round mode only.
 *
 * Data layout.  U and L are row-major n x n matrices with leading dimension
 * ld >= n (in elements), device memory, updated in place.  Element (i, j) is
 * at ptr[i*ld + j].  Each matrix must span (n-1)*ld + n elements; columns
 * n..ld-1 are never read or written.  Element type: fp32 in Angstrom
 * (BS_FP32) or int32 in units of 1/1024 Angstrom (BS_INT32_Q10).  Inputs need
 * not be symmetric; symmetric inputs give symmetric outputs.
 *
 * Preconditions (not checked unless BS_VALIDATE is set):
 *   diagonal of U and L is 0; U >= 0 and L >= 0; no NaN; fp32 U may be +inf,
 *   fp32 L is finite; int32 values lie in [0, 2^30) so U+U cannot overflow.
 *
 * Streams and devices.  Work is enqueued on `stream` (NULL = the legacy
 * default stream) of the calling thread's current device, which must hold
 * the matrices.  Smoothing calls return before the GPU finishes.
 * bs_check_feasible synchronises `stream` before it returns.  In blocked mode
 * with three or more block rows (unless BS_NO_LOOKAHEAD) the tiles of block
 * row and column K+1 and phases 1 and 2 of block round K+1 run on an internal
 * high-priority stream of the library, forked from and joined back into
 * `stream` with events inside the call, while the rest of round K's phase 3
 * runs on `stream` (for small matrices all of it but tile (K+1,K+1), whose
 * update phase 1 of round K+1 applies); all work still completes in
 * `stream` order.  The
 * smoothing calls can be captured into a CUDA graph (stream capture on
 * `stream`) once the library has run one smoothing of the same kind on the
 * device, which sets up its per-device state; the look-ahead fork and join
 * are captured with it, and the internal stream's priority is kept on its
 * kernels as a launch attribute.  Replaying a captured call saves the
 * per-launch host overhead, which matters for small n (n = 256: about a
 * quarter of the call).
 *
 * Memory.  The caller owns U, L and the mask.  Smoothing allocates nothing.
 * bs_check_feasible and BS_VALIDATE use one small internal device buffer per
 * device, allocated on first use and kept until exit.
 *
 * Errors.  Argument errors return before anything is enqueued.  BS_ERR_CUDA
 * reports a failed launch or CUDA call (cudaGetLastError after the launches).
 * No call aborts the process.
 */
#ifndef BSMOOTH_H
#define BSMOOTH_H

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; C callers need no CUDA header. */
typedef struct CUstream_st *bs_stream_t;

typedef enum {
    BS_OK = 0,
    BS_ERR_ARG = 1,      /* bad n, ld, batch, stride, null pointer, mode bits */
    BS_ERR_ALIGN = 2,    /* a matrix pointer is not aligned to its element size */
    BS_ERR_RANGE = 3,    /* BS_VALIDATE: an int32 value outside [0, 2^30) */
    BS_ERR_CUDA = 4,     /* a CUDA launch or call failed */
    BS_ERR_TIMEOUT = 5,  /* reserved: a bounded device wait ran out */
    BS_ERR_INPUT = 6     /* BS_VALIDATE: nonzero diagonal, negative value, NaN,
                            or an infinite lower bound */
} bs_status;

/* mode bits */
enum {
    BS_FP32 = 0,              /* element type: float, Angstrom */
    BS_INT32_Q10 = 1,         /* element type: int32, 1/1024 Angstrom */
    BS_DTYPE_MASK = 3,
    BS_BLOCKED = 0,           /* three-phase blocked Floyd-Warshall (default) */
    BS_PERK = 1 << 2,         /* round by round over the middle atoms k,
                                 round-synchronous: one pass over the matrix
                                 per round (the plain reference mode) */
    BS_RULE_CLOSURE = 0,      /* default lower-bound rule (see above) */
    BS_RULE_LITERAL = 1 << 3, /* printed rule; BS_PERK only, else BS_ERR_ARG */
    BS_VALIDATE = 1 << 4,     /* check the preconditions first (synchronises) */
    /* Blocked-mode schedule knobs; every setting gives identical results. */
    BS_TILE_64 = 1 << 5,      /* force 64 x 64 tiles (default: 128 from 48
                                 block rows of 128 with general inputs
                                 (block rounds in pairs), or once a block
                                 round's phase 3 holds at least 9000 tiles of
                                 128 over the batch, 768 for the upper bound
                                 alone, else 64) */
    BS_TILE_128 = 1 << 6,     /* force 128 x 128 tiles; both tile bits: BS_ERR_ARG */
    BS_NO_LOOKAHEAD = 1 << 7, /* run the three phases of each block round in
                                 sequence on `stream` only (see below) */
    /* 1 << 9 is not used (any unknown bit: BS_ERR_ARG) */
    BS_PERK_PAIRED = 1 << 10, /* with BS_PERK: two rounds per pass over the
                                 matrix (half the memory traffic), each round
                                 exactly as alone; without BS_PERK: BS_ERR_ARG */
    BS_ONE_LAUNCH = 1 << 11,  /* blocked mode in a single kernel launch: one
                                 thread-block cluster per molecule (16 CTAs
                                 where the device allows, else 8, while every
                                 molecule's cluster fits at once; 4 or 8 for
                                 larger batches), 64 x 64 tiles, the phases of
                                 each block round separated by cluster
                                 barriers only; same results.  Meant for
                                 batches of small molecules.  With BS_PERK,
                                 BS_TILE_128 or BS_NO_LOOKAHEAD: BS_ERR_ARG */
    BS_PAIRED_ROUNDS = 1 << 12, /* blocked mode: block rounds taken in pairs
                                 whatever the size (the bulk tiles update
                                 both rounds of a pair in one pass), on
                                 128 x 128 tiles unless BS_TILE_64 is given;
                                 by default pairs run from 48 block rows of
                                 128, and on 64-wide tiles once a pair's bulk
                                 holds 2500 tiles over the batch; same
                                 results.  With BS_PERK, BS_ONE_LAUNCH or
                                 BS_NO_LOOKAHEAD: BS_ERR_ARG */
    BS_SYMMETRIC = 1 << 8     /* blocked mode, symmetric U and L (both triangles
                                 stored, section 6): only tiles on and above the
                                 diagonal are computed (the panels of each block
                                 round stored on both sides), and the lower
                                 triangle is written as the transpose of the
                                 upper one at the end -- about half the work,
                                 same output on the 1/1024 grid (off it, within
                                 the fp32 rounding of the general schedule).
                                 With BS_PERK: BS_ERR_ARG.  With BS_VALIDATE,
                                 asymmetric input returns BS_ERR_INPUT. */
};

/* Upper bounds only (min-plus all-pairs shortest paths, section 3's loop).
 * U: device, n x n, leading dimension ld.  Rule bits are ignored. */
bs_status bs_smooth_upper(void *U, int n, int ld, bs_stream_t stream, int mode);

/* Upper and lower bounds together (sections 2 and 3).
 * U, L: device, n x n each, same leading dimension ld, distinct buffers. */
bs_status bs_smooth_bounds(void *U, void *L, int n, int ld, bs_stream_t stream,
                           int mode);

/* `batch` independent molecules of n atoms each; molecule b starts at
 * U + b*batch_stride and L + b*batch_stride (elements).  batch_stride >=
 * (n-1)*ld + n.  The number of kernel launches does not depend on batch. */
bs_status bs_smooth_bounds_batched(void *U, void *L, int n, int ld,
                                   long long batch_stride, int batch,
                                   bs_stream_t stream, int mode);

/* Infeasibility flags: counts the cells (i, j) of the n x n block, diagonal
 * included, with L[i,j] > U[i,j] strictly, and stores the count in
 * *out_count (host memory).  If mask != NULL (device, same layout and ld as
 * U, one byte per cell), mask[i*ld+j] is set to 1 for a flagged cell and 0
 * otherwise; its columns n..ld-1 are untouched.  Only the dtype bits of
 * `mode` are used.  Synchronises `stream`. */
bs_status bs_check_feasible(const void *U, const void *L, int n, int ld,
                            bs_stream_t stream, int mode, long long *out_count,
                            unsigned char *mask);

/* Static text for a status code. */
const char *bs_strerror(bs_status status);

/* Infeasibility counts for callers that cannot allocate device memory.
 * The method has no counterpart of this call; it exists for callers whose
 * device memory belongs entirely to their own allocator (a framework's caching
 * allocator that accounts for every byte, or a budget reserved up front) and
 * for paths where the implicit synchronisation and latency of cudaMalloc are
 * not allowed.  bs_check_feasible allocates a small buffer on its first call on
 * a device; this call allocates nothing (no cudaMalloc, cudaFree or other
 * allocating routine): its counters live in a fixed array of
 * BS_NOALLOC_MAX_BATCH 8-byte counters in the library's own static device
 * memory, which every device that loads the library holds until the process
 * exits.
 *
 * Counts, for each of `batch` molecules (molecule b at U + b*batch_stride and
 * L + b*batch_stride elements, as in bs_smooth_bounds_batched), the cells of
 * its n x n block with L > U strictly, diagonal included, into out_counts[b]
 * (host array of `batch` entries).  batch > BS_NOALLOC_MAX_BATCH returns
 * BS_ERR_ARG without touching the GPU.  Only the dtype bits of `mode` are
 * accepted.  Synchronises `stream`.
 *
 * The first call on each device looks up the device address of the array
 * (cudaGetSymbolAddress, with that device current) and keeps it for the life
 * of the process; make that first call before any stream capture on the
 * device.  cudaDeviceReset unloads the array with the device's context, so do
 * not call this entry point on a device after resetting it.  Every call clears the counters it
 * uses, but all calls share one array: calls whose GPU work can overlap
 * (different streams or host threads) race and must be serialised by the
 * caller. */
#define BS_NOALLOC_MAX_BATCH 4096
bs_status bs_check_feasible_noalloc(const void *U, const void *L, int n, int ld,
                                    long long batch_stride, int batch,
                                    bs_stream_t stream, int mode,
                                    long long *out_counts);

/* ---- instrumentation (not part of the method) ---------------------------- */

/* Number of kernels this library has launched since it was loaded. */
long long bs_launch_count(void);

/* CTAs per thread-block cluster of BS_ONE_LAUNCH for a single molecule on the
 * current device (16 or 8), or 0 before the library's first smoothing call on
 * it.  Batches larger than the number of such clusters resident at once use
 * clusters of 4 or 8. */
int bs_one_launch_cluster(void);

/* The schedule a blocked smoothing call would take, without running it (host
 * logic only: no GPU, stream or memory involved).  bounds: nonzero for
 * bs_smooth_bounds(_batched), zero for bs_smooth_upper; n, batch and mode as
 * in those calls (a contiguous layout is assumed).  *tile: 64 or 128, the tile
 * width (0 with BS_PERK); *pairs: 1 if the bulk tiles take block rounds in
 * pairs, else 0.  Mode bits the smoothing calls would reject give
 * BS_ERR_ARG, as do null outputs. */
bs_status bs_schedule_info(int n, int batch, int mode, int bounds, int *tile, int *pairs);

/* Per-phase device time.  After bs_profile_begin(), every smoothing call
 * records a CUDA event pair around each of its kernel launches, on the stream
 * the kernel runs on (the caller's, or the library's look-ahead stream).
 * bs_profile_end() waits for those events, writes the summed milliseconds and
 * launch counts per phase and stops recording.  Index: 0 per-round kernels,
 * 1 phase 1, 2 phase 2, 3 phase 3 on the caller's stream, 4 phase 3 of the
 * next block row and column on the look-ahead stream (these overlap index 3
 * in time), 5 the single kernel of BS_ONE_LAUNCH.  At most 1<<16 launches
 * are recorded per session; more set *overflow to 1. */
#define BS_PROFILE_PHASES 6
typedef struct {
    double ms[BS_PROFILE_PHASES];
    long long launches[BS_PROFILE_PHASES];
    int overflow;
} bs_profile;

bs_status bs_profile_begin(void);
bs_status bs_profile_end(bs_profile *out);

/* ALU issue-rate probe.  Runs one 1024-thread CTA per SM, each thread
 * iterating `iters` x 128 instructions of one form in 8 independent chains,
 * and stores the measured thread-instructions retired per SM clock (SM cycle
 * counter around the loop, mean over SMs) in *instr_per_clk_per_sm.
 * Allocates and frees a small device buffer; synchronises the device. */
enum {
    BS_PROBE_FADD = 0,         /* add.rn.f32 */
    BS_PROBE_FMNMX = 1,        /* min.f32, two inputs */
    BS_PROBE_FMNMX3 = 2,       /* min.f32, three inputs */
    BS_PROBE_FADD2 = 3,        /* add.rn.f32x2 (two lanes per instruction) */
    BS_PROBE_FADD2_FMNMX3 = 4, /* the two above interleaved 1:1 */
    BS_PROBE_IADD = 5,         /* add.s32 */
    BS_PROBE_IMNMX = 6,        /* min.s32 */
    BS_PROBE_VIADDMIN = 7,     /* __viaddmin_s32: min(a + b, c) */
    BS_PROBE_VIMNMX3 = 8       /* __vimin3_s32: min(a, b, c) */
};
bs_status bs_probe_alu(int which, int iters, double *instr_per_clk_per_sm);

#ifdef __cplusplus
}
#endif

#endif /* BSMOOTH_H */
