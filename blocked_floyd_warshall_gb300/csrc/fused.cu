// The whole blocked smoothing of a molecule in one launch: one thread-block
// cluster per molecule, the phases of every block round separated by cluster
// barriers only (GPU Gems 2 ch. 43, section 3: the rounds over the middle
// atoms are sequential, only the pairs of one round run in parallel; here a
// "round" is a block round of 64 middle atoms).
//
// Each CTA of a cluster of C runs every block round K (C = 16 where the
// device allows clusters that large, else 8, for a single molecule and small
// batches; 4 or 8 for larger batches, see pick_cluster):
//   phase 2: the panel tiles of round K, t = rank, rank + C, ...;
//   cluster barrier;
//   phase 3: rank 0 updates tile (K+1,K+1) and at once closes it (phase 1 of
//            round K+1); ranks 1..C-1 share every other tile of round K;
//   cluster barrier.
// With symmetric inputs the CTAs then share the 64-wide blocks above the
// diagonal, each written transposed over its mirror block.
// Phase 1 of round K+1 needs only tile (K+1,K+1) after round K, and tiles
// (K+1,K) and (K,K+1), which phase 2 of round K finished; phase 2 of round
// K+1 waits for all of round K at the barrier.  Phase 1 of round 0 runs
// before the loop.  Every CTA passes the same 2 nb + 1 barriers; there is no
// other wait, so no CTA ever spins on another.
//
// Tiles are 64 wide.  The closure is the one-CTA form (p1_tile.cuh), the
// tile update the 256-thread form of phases 2 and 3 (p3_tile.cuh).  Global
// memory written by one CTA before a barrier is read by the others after it:
// barrier.cluster.arrive has release and barrier.cluster.wait acquire
// semantics at cluster scope.
#include "../../include/bsmooth.h"
#include "p1_tile.cuh"
#include "p3_tile.cuh"

namespace bs {

namespace {

constexpr int FZ_FB = FB_SMALL;
constexpr int FZ_NT = 256;
static_assert(P1S<FZ_FB>::NT == FZ_NT && P3S<FZ_FB, true>::NT == FZ_NT,
              "the closure and the tile update run on the same threads");

template <class T, bool HAS_L>
constexpr size_t fz_smem() {
    return P1Smem<T, HAS_L, FZ_FB>::BYTES > P3Smem<T, HAS_L, FZ_FB>::BYTES
               ? P1Smem<T, HAS_L, FZ_FB>::BYTES
               : P3Smem<T, HAS_L, FZ_FB>::BYTES;
}

static_assert(2 * FZ_FB * (FZ_FB + 4) * 4 <= fz_smem<float, true>() &&
                  FZ_FB * (FZ_FB + 4) * 4 <= fz_smem<float, false>(),
              "the mirrored blocks fit the shared memory");

__device__ __forceinline__ int fz_rank() {
    unsigned r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return (int)r;
}
__device__ __forceinline__ int fz_size() {
    unsigned r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return (int)r;
}
// Every thread of every CTA of the cluster arrives (release) and waits
// (acquire): the tiles stored before it are visible to all CTAs after it.
__device__ __forceinline__ void fz_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

template <class T, bool HAS_L>
__global__ void __launch_bounds__(FZ_NT, 2)
k_fused(T* __restrict__ U, T* __restrict__ L, int n, int ld, long long bstride, bool vec,
        bool sym) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    T* sm = reinterpret_cast<T*>(smem_raw);
    const size_t off = (size_t)blockIdx.z * (size_t)bstride;
    U += off;
    if (HAS_L) L += off;
    const int rank = fz_rank(), C = fz_size();
    const int nb = (n + FZ_FB - 1) / FZ_FB;
    int I, J;

    if (rank == 0) p1_close_tile<T, HAS_L, FZ_FB>(U, L, n, ld, 0, vec, smem_raw);
    fz_sync();
    for (int K = 0; K < nb; ++K) {
        const int np = p3_tiles(sym, P3_PANELS, nb, K);
        for (int t = rank; t < np; t += C) {
            p3_tile(P3_PANELS, sym, t, nb, K, I, J);
            p3_update_tile<T, HAS_L, FZ_FB, true>(U, L, n, ld, I, J, K, vec, sym, sm);
        }
        fz_sync();
        if (K + 1 < nb) {
            if (rank == 0) {
                p3_update_tile<T, HAS_L, FZ_FB, true>(U, L, n, ld, K + 1, K + 1, K, vec, false, sm);
                __syncthreads();   // the tile's stores, before the closure loads it
                p1_close_tile<T, HAS_L, FZ_FB>(U, L, n, ld, K + 1, vec, smem_raw);
            } else {
                const int nt = p3_tiles(sym, P3_ALL_OFF, nb, K);
                for (int t = rank - 1; t < nt; t += C - 1) {
                    p3_tile(P3_ALL_OFF, sym, t, nb, K, I, J);
                    p3_update_tile<T, HAS_L, FZ_FB, true>(U, L, n, ld, I, J, K, vec, false, sm);
                }
            }
        } else {
            const int nt = p3_tiles(sym, P3_ALL, nb, K);
            for (int t = rank; t < nt; t += C) {
                p3_tile(P3_ALL, sym, t, nb, K, I, J);
                p3_update_tile<T, HAS_L, FZ_FB, true>(U, L, n, ld, I, J, K, vec, false, sm);
            }
        }
        fz_sync();
    }
    if (sym) {
        // every tile's last store came before the last barrier
        const int np = (nb - 1) * nb / 2;
        for (int t = rank; t < np; t += C) {
            int a, c;
            p3_tri(t, a, c);
            p3_mirror_block<T, HAS_L>(U, L, n, ld, a, c + 1, vec, sm);
        }
    }
}

// Per device: the largest cluster size that can be placed (16 where the
// device allows clusters that large, else 8) and how many clusters of it, and
// of 4 CTAs, are resident at once (0: not set up).
struct FzDevice {
    int big = 0;
    int active_big = 0;
    int active4 = 0;
};
FzDevice g_fz[64];

template <class T, bool HAS_L>
int active_clusters(int c) {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = c;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(c, 1, 1);
    cfg.blockDim = dim3(FZ_NT);
    cfg.dynamicSmemBytes = fz_smem<T, HAS_L>();
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int active = 0;
    if (cudaOccupancyMaxActiveClusters(&active, k_fused<T, HAS_L>, &cfg) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    return active;
}

template <class T, bool HAS_L>
cudaError_t setup_t(FzDevice* d) {
    auto kernel = k_fused<T, HAS_L>;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)fz_smem<T, HAS_L>());
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess || d->big) return e;
    const int a16 = active_clusters<T, HAS_L>(16);
    d->big = a16 > 0 ? 16 : 8;
    d->active_big = a16 > 0 ? a16 : active_clusters<T, HAS_L>(8);
    d->active4 = active_clusters<T, HAS_L>(4);
    return cudaSuccess;
}

// CTAs per cluster for a launch of `batch` molecules.  While every molecule's
// cluster of the largest size is resident at once, the largest (more CTAs
// per molecule); then 4 while every molecule's cluster of 4 is (more
// clusters fit: measured, 32 molecules of n = 256: 0.58 ms with 16, 0.28
// with 8, 0.24 with 4); beyond, 8 (256 molecules of n = 512: 11.6 ms with 16,
// 8.8 with 8, 8.9 with 4).
int pick_cluster(const FzDevice& d, int batch) {
    if (batch <= d.active_big) return d.big;
    if (batch <= d.active4) return 4;
    return 8;
}

template <class T, bool HAS_L>
cudaError_t fused_t(const Mats& m, int cluster, cudaStream_t s) {
    return for_batch_chunks(m, [&](int b0, int nbz) {
        T* U = static_cast<T*>(m.U) + (size_t)b0 * m.bstride;
        T* L = HAS_L ? static_cast<T*>(m.L) + (size_t)b0 * m.bstride : nullptr;
        int prio = 0;
        cudaError_t e = cudaStreamGetPriority(s, &prio);
        if (e != cudaSuccess) return e;
        cudaLaunchAttribute attr[2];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = cluster;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        attr[1].id = cudaLaunchAttributePriority;
        attr[1].val.priority = prio;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(cluster, 1, nbz);
        cfg.blockDim = dim3(FZ_NT);
        cfg.dynamicSmemBytes = fz_smem<T, HAS_L>();
        cfg.stream = s;
        cfg.attrs = attr;
        cfg.numAttrs = prio != 0 ? 2 : 1;
        before_launch(s, PH_FUSED);
        e = cudaLaunchKernelEx(&cfg, k_fused<T, HAS_L>, U, L, m.n, m.ld, m.bstride, m.vec,
                               m.sym);
        after_launch(s, PH_FUSED);
        return e;
    });
}

}  // namespace

cudaError_t fused_setup(bool is_int) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    FzDevice* c = &g_fz[dev];
    if (is_int) {
        e = setup_t<int, true>(c);
        if (e == cudaSuccess) e = setup_t<int, false>(c);
    } else {
        e = setup_t<float, true>(c);
        if (e == cudaSuccess) e = setup_t<float, false>(c);
    }
    return e;
}

cudaError_t launch_fused(bool is_int, const Mats& m, cudaStream_t s) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64 || g_fz[dev].big == 0) return cudaErrorInitializationError;
    const int c = pick_cluster(g_fz[dev], m.batch);
    if (is_int) return m.L ? fused_t<int, true>(m, c, s) : fused_t<int, false>(m, c, s);
    return m.L ? fused_t<float, true>(m, c, s) : fused_t<float, false>(m, c, s);
}

int fused_cluster_size() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    return g_fz[dev].big;
}

}  // namespace bs
