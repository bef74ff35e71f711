// Three-phase blocked Floyd-Warshall over the bound pair (U, L).
//
// The matrix is cut into FB x FB tiles; block round K processes the middle
// atoms k of tile-row K in order, in three launches:
//   phase 1: tile (K,K), its closure over block K, one CTA (this file);
//   phase 2: row panel (K,J) and column panel (I,K) against the finished
//            diagonal tile (phase3.cu);
//   phase 3: every other tile (I,J), against the finished panels (phase3.cu).
//
// Rules (GPU Gems 2 ch. 43, section 2): U[i,j] = min(U[i,j], U[i,k] + U[k,j]);
// L[i,j] = max(L[i,j], L[k,j] - U[i,k], Lcol[i] - U[k,j]), with the upper
// bound tightened first.  Lcol[i] is L[i,k] raised to max(L[i,k], L[k,k] -
// U[i,k]) while column k is still being formed (phase 1); phases 2 and 3 read
// finished tiles, which already contain that raise.
//
// Why phases 2 and 3 need no serial k.  Read the pair as shortest paths on a
// doubled graph (each atom a has copies aL and aR; aL->bL and aR->bR weigh
// U[a,b], aL->bR weighs -L[a,b]; U[i,j] is the iL->jL distance and -L[i,j] the
// iL->jR distance).  Once tile (K,K) holds the closure D over the middle atoms
// of block K, a path from a row-panel atom i (in K) to j (outside K) through
// block K splits at its last visit of block K: D[i,k] (or -D_L[i,k]) followed
// by one edge of the panel itself.  So the panel is a single min/max-plus
// product of D with the panel's values from before the round,
//   U[i,j] = min(U[i,j], min_k D_U[i,k] + U[k,j])
//   L[i,j] = max(L[i,j], max_k L[k,j] - D_U[i,k], max_k D_L[i,k] - U[k,j]),
// and the column panel the mirror product (split at the first visit).  These
// are the phase-3 rules with D as one operand, so one kernel serves both, and
// the k order is free in both.  The result is the fixed point of the triangle
// inequalities, the same as the round-by-round schedule (exactly in int32; in
// fp32 exactly for values on the 1/1024 grid below 2^14).
//
// Phase 1 itself applies the same blocked scheme one level down (p1_tile.cuh);
// only its 16-wide sub-blocks are closed step by step, each step
// round-synchronous.
#include "p1_tile.cuh"

namespace bs {

template <class T, bool HAS_L, int FB>
__global__ void __launch_bounds__(P1S<FB>::NT)
k_phase1(T* __restrict__ U, T* __restrict__ L, int n, int ld, long long bstride, int K, bool vec) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    const size_t off = (size_t)blockIdx.z * (size_t)bstride;
    U += off;
    if (HAS_L) L += off;
    p1_close_tile<T, HAS_L, FB>(U, L, n, ld, K, vec, smem_raw);
}

// ---------------------------------------------------------------- phase 1 on a cluster

// Phase 1 of a 64-wide tile on a cluster of four CTAs.  CTA c holds stripe c
// (tile rows 16c .. 16c+15) in registers: its four 64-thread groups hold one
// 16 x 16 block each, group g the block in sub-block column g, thread t of a
// group row t/4 and columns 4(t%4) .. +3 of it (the layout of step (a) in
// p1_tile.cuh).  Sub-block s (middle atoms 16s .. 16s+15):
//   CTA s closes block (s,s) (group s, step (a)) and stores the closed
//   block, and its row sub-panel as it stood before the sub-block, R0, into
//   the shared memory of every CTA of the cluster (distributed shared
//   memory); one cluster barrier;
//   every other CTA takes the product of its cells in sub-block column s
//   with the closed block (its column sub-panel C, as in phase 2), then the
//   product of C with R0 for the rest of its stripe;
//   CTA s, meanwhile, updates its own row sub-panel against the closed block.
// R0 in place of the updated row sub-panel R = R0 + D R0 (min-plus sums and
// products of the doubled bound graph, D the closed block) gives the same
// cells: D is closed with a zero diagonal, so D D = D and C = C0 + C0 D
// already contains C0 D, hence C R = C R0 + C0 D R0 = C R0.  R0 is ready
// before the closure, so only the 2 KB closed block is sent after it.  The
// critical path per sub-block: closure of block (s,s), its store to the
// other CTAs, barrier, the column sub-panel product, block (s+1, s+1)'s
// product (both over all 256 threads, one cell each), closure of block
// (s+1, s+1).
// Remote stores: sub-block s's data lands in buffer s % 2 of every CTA.  A
// CTA stores it only after passing barrier s-1, when every CTA has finished
// sub-block s-2, the last reader of that buffer, and barrier s makes it
// visible.  A first barrier at entry makes sure every CTA of the cluster is
// running before any remote store; no CTA touches another's shared memory
// after barrier 3, so none has to wait for the others before it exits.
// With `pre` (the merged look-ahead of small matrices) each CTA first applies
// the previous block round's product to its own stripe, before the closures.

constexpr int CL = FB_SMALL / SB;   // CTAs per cluster: one per 16-row stripe
constexpr int CNT = CL * AT;        // threads per CTA: one group per sub-block column
constexpr int CS = SB + 2;          // row stride of the row-major 16 x 16 buffers (pairs aligned)
static_assert(CNT == SB * SB, "one thread per cell of a 16 x 16 block");
constexpr int PTS = FB_SMALL + 4;   // row stride of the staged column panel stripe (16-byte rows)

// Dynamic shared memory of a launch that first applies the previous block
// round's update (pre): the row panel tile k-interleaved and this stripe's
// rows of the column panel tile, U and L.
template <bool HAS_L>
constexpr size_t p1c_pre_bytes() {
    return (HAS_L ? 2 : 1) * (size_t)(FB_SMALL * FB_SMALL + SB * PTS) * 4;
}

template <class T>
struct P1CSmem {
    // written by the CTA that closes sub-block s, into buffer s % 2
    __align__(16) T dx[2][2][SB * SB];       // closed block (s,s), k-interleaved [k/2][j][k%2]; U, L
    __align__(16) T rx[2][2][SB * FB_SMALL]; // row sub-panel of stripe s before sub-block s, k-interleaved
    // private
    __align__(16) T dR[2][SB * CS];          // own closed block, row-major
    __align__(16) T cP[2][SB * CS];          // column sub-panel block before the sub-block
    __align__(16) T cQ[2][SB * CS];          // after
    __align__(16) T bD[2][SB * CS];          // own diagonal block through its last product
    __align__(16) T xr[2 * 2 * SB];          // closure exchange
    __align__(16) T xc[2 * 2 * SB];
};

__device__ __forceinline__ void cluster_arrive() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ unsigned cluster_addr(const void* p, unsigned rank) {
    unsigned a;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;"
                 : "=r"(a)
                 : "r"((unsigned)__cvta_generic_to_shared(p)), "r"(rank));
    return a;
}
template <class T>
__device__ __forceinline__ void st_cluster4(unsigned a, T x, T y, T z, T w) {
    static_assert(sizeof(T) == 4, "32-bit elements");
    asm volatile("st.shared::cluster.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a),
                 "r"(__builtin_bit_cast(unsigned, x)), "r"(__builtin_bit_cast(unsigned, y)),
                 "r"(__builtin_bit_cast(unsigned, z)), "r"(__builtin_bit_cast(unsigned, w))
                 : "memory");
}

// Store the thread's cells (i, j .. j+3) k-interleaved (middle atom i, BW
// columns) into the arrays dU, dL of every CTA of the cluster.  Rows i and
// i^1 meet in one 16-byte piece per column pair: the thread holding the even
// row stores columns j, j+1 of both rows, its partner (thread t^4, same
// warp) columns j+2, j+3.  Whole warps only.
template <class T, bool HAS_L, int BW>
__device__ __forceinline__ void p1c_push_k(T* dU, T* dL, int i, int j, const T (&u)[4],
                                           const T (&l)[4]) {
    const bool odd = i & 1;
    const int e = (i >> 1) * (2 * BW) + 2 * j + (odd ? 4 : 0);
    T pu[4], pl[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        pu[q] = __shfl_xor_sync(0xffffffffu, u[q], 4);
        pl[q] = HAS_L ? __shfl_xor_sync(0xffffffffu, l[q], 4) : T(0);
    }
    const T a0 = odd ? pu[2] : u[0], a1 = odd ? u[2] : pu[0];
    const T a2 = odd ? pu[3] : u[1], a3 = odd ? u[3] : pu[1];
    const T b0 = odd ? pl[2] : l[0], b1 = odd ? l[2] : pl[0];
    const T b2 = odd ? pl[3] : l[1], b3 = odd ? l[3] : pl[1];
#pragma unroll
    for (int r = 0; r < CL; ++r) {
        st_cluster4(cluster_addr(dU + e, r), a0, a1, a2, a3);
        if (HAS_L) st_cluster4(cluster_addr(dL + e, r), b0, b1, b2, b3);
    }
}

// Product step for the thread's cells (i, j0 .. j0+3): X[i,j] against
// A[i,k] (row i of a row-major array: aU, aL at row i) and B[k,j]
// (k-interleaved, BW columns; the thread's columns at jb) over KN middle
// atoms, in pairs as in phase 3.
template <class T, bool HAS_L, int BW, int KN = SB>
__device__ __forceinline__ void p1c_product(T (&u)[4], T (&l)[4], const T* aU, const T* aL,
                                            const T* bU, const T* bL, int jb) {
    using LD = PairLoad<T>;
    using P = typename LD::P;
    constexpr bool NEG = std::is_same<T, int>::value;
#pragma unroll 8
    for (int kk = 0; kk < KN; kk += 2) {
        P a = LD::ld2(aU + kk);
        P al = a;
        if (HAS_L) al = LD::ld2(aL + kk);
        P b[4], bl[4];
        const int o = (kk >> 1) * (2 * BW) + 2 * jb;
        LD::ld4(bU + o, b[0], b[1]);
        LD::ld4(bU + o + 4, b[2], b[3]);
        if (HAS_L) {
            LD::ld4(bL + o, bl[0], bl[1]);
            LD::ld4(bL + o + 4, bl[2], bl[3]);
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) PairOps<T>::upper(u[q], a, b[q]);
        if (HAS_L) {
            if (NEG) {
                a = LD::neg(a);
#pragma unroll
                for (int q = 0; q < 4; ++q) b[q] = LD::neg(b[q]);
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) PairOps<T>::lower(l[q], a, al, b[q], bl[q]);
        }
    }
}

// The same for one cell (i, j) of a 16 x 16 block: its value is read from
// the row-major buffer x (16 x CS), updated and written to y (may be x).
template <class T, bool HAS_L, int BW>
__device__ __forceinline__ void p1c_cell(const T (*x)[SB * CS], T (*y)[SB * CS], int i, int j,
                                         const T* aU, const T* aL, const T* bU, const T* bL,
                                         int jb) {
    using LD = PairLoad<T>;
    using P = typename LD::P;
    constexpr bool NEG = std::is_same<T, int>::value;
    T u = x[0][i * CS + j];
    T l = HAS_L ? x[1][i * CS + j] : T(0);
#pragma unroll
    for (int kk = 0; kk < SB; kk += 2) {
        P a = LD::ld2(aU + kk);
        P al = a;
        if (HAS_L) al = LD::ld2(aL + kk);
        const int o = (kk >> 1) * (2 * BW) + 2 * jb;
        P b = LD::ld2(bU + o);
        P bl = b;
        if (HAS_L) bl = LD::ld2(bL + o);
        PairOps<T>::upper(u, a, b);
        if (HAS_L) {
            if (NEG) {
                a = LD::neg(a);
                b = LD::neg(b);
            }
            PairOps<T>::lower(l, a, al, b, bl);
        }
    }
    y[0][i * CS + j] = u;
    if (HAS_L) y[1][i * CS + j] = l;
}

// The thread's cells to or from a row-major 16-wide buffer (row i, columns
// c0 ..).
template <class T, bool HAS_L>
__device__ __forceinline__ void p1c_put_rows(T (*buf)[SB * CS], int i, int c0, const T (&u)[4],
                                             const T (&l)[4]) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        buf[0][i * CS + c0 + q] = u[q];
        if (HAS_L) buf[1][i * CS + c0 + q] = l[q];
    }
}
template <class T, bool HAS_L>
__device__ __forceinline__ void p1c_get_rows(const T (*buf)[SB * CS], int i, int c0, T (&u)[4],
                                             T (&l)[4]) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        u[q] = buf[0][i * CS + c0 + q];
        if (HAS_L) l[q] = buf[1][i * CS + c0 + q];
    }
}

template <class T, bool HAS_L>
__global__ void __cluster_dims__(CL, 1, 1) __launch_bounds__(CNT)
k_phase1c(T* __restrict__ U, T* __restrict__ L, int n, int ld, long long bstride, int K, bool vec,
          bool pre) {
    using E = El<T>;
    constexpr int FB = FB_SMALL;
    __shared__ P1CSmem<T> sm;
    extern __shared__ __align__(16) unsigned char p1c_dyn[];

    const int c = blockIdx.x;                 // cluster rank = stripe
    const int g = threadIdx.x / AT;           // column block held
    const int t = threadIdx.x % AT;
    const int i = t >> 2;                     // row within the stripe
    const int jc = (t & 3) * 4;               // first column within the block
    const int j0 = g * SB + jc;               // first column within the tile
    const int ci = threadIdx.x / SB;          // one-cell steps: cell (ci, cj) of a block
    const int cj = threadIdx.x % SB;

    cluster_arrive();   // every CTA is running: waited for below, before any remote store

    const size_t off = (size_t)blockIdx.z * (size_t)bstride;
    const int o = K * FB;
    const int m = min(FB, n - o);
    const int row = c * SB + i;
    T* Ur = U + off + (size_t)(o + row) * ld + o;
    T* Lr = HAS_L ? L + off + (size_t)(o + row) * ld + o : nullptr;
    const bool live = c * SB < m;             // the stripe holds real rows

    T u[4], l[4];
    if (vec && row < m && j0 + 4 <= m) {
        using V4 = typename E::V4;
        const V4 v = *reinterpret_cast<const V4*>(Ur + j0);
        u[0] = v.x; u[1] = v.y; u[2] = v.z; u[3] = v.w;
        if (HAS_L) {
            const V4 w = *reinterpret_cast<const V4*>(Lr + j0);
            l[0] = w.x; l[1] = w.y; l[2] = w.z; l[3] = w.w;
        }
    } else {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const bool in = row < m && j0 + q < m;
            u[q] = in ? Ur[j0 + q] : E::upad();
            l[q] = HAS_L ? (in ? Lr[j0 + q] : E::lpad()) : T(0);
        }
    }

    // Block round K-1's update of this tile, which the look-ahead schedule
    // leaves to this launch: X = X + C R over the middle atoms of block K-1
    // (min-plus, the phase-3 rules), C = tile (K, K-1) (this stripe's rows),
    // R = tile (K-1, K), both staged here, R k-interleaved.  Block K-1 is
    // full, so only the columns of R and the rows of C beyond m get pads.
    if (pre) {
        T* RU = reinterpret_cast<T*>(p1c_dyn);
        T* RL = RU + FB * FB;
        T* CU = RU + (HAS_L ? 2 : 1) * FB * FB;
        T* CL = CU + SB * PTS;
        const int op = o - FB;
        const size_t rg = off + (size_t)op * ld + o;             // tile (K-1, K)
        const size_t cg = off + (size_t)(o + c * SB) * ld + op;  // tile (K, K-1), stripe c
        // every copy in flight at once: R element by element into its
        // k-interleaved place, C in 16-byte pieces where rows allow
        for (int e = threadIdx.x; e < FB * FB; e += CNT) {
            const int k = e / FB, j = e % FB;
            const int d = (k >> 1) * (2 * FB) + 2 * j + (k & 1);
            if (j < m) {
                cp_async4(RU + d, U + rg + (size_t)k * ld + j);
                if (HAS_L) cp_async4(RL + d, L + rg + (size_t)k * ld + j);
            } else {
                RU[d] = E::upad();
                if (HAS_L) RL[d] = E::lpad();
            }
        }
        for (int e = threadIdx.x; e < SB * FB / 4; e += CNT) {
            const int r = e / (FB / 4), k = (e % (FB / 4)) * 4;
            T* cu = CU + r * PTS + k;
            T* cl = CL + r * PTS + k;
            if (c * SB + r < m) {
                const size_t g = cg + (size_t)r * ld + k;
                if (vec) {
                    cp_async16(cu, U + g);
                    if (HAS_L) cp_async16(cl, L + g);
                } else {
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        cp_async4(cu + q, U + g + q);
                        if (HAS_L) cp_async4(cl + q, L + g + q);
                    }
                }
            } else {
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    cu[q] = E::upad();
                    if (HAS_L) cl[q] = E::lpad();
                }
            }
        }
        cp_async_commit();
        cp_async_wait<0>();
        __syncthreads();
        p1c_product<T, HAS_L, FB, FB>(u, l, CU + i * PTS, CL + i * PTS, RU, RL, j0);
    }
    cluster_wait();

    // What CTA c sends for sub-block c: the closed block (group c) and the
    // row sub-panel before the sub-block (the other groups).
    auto close_own = [&]() {
        p1_block_close<T, HAS_L>(u, l, t, sm.xr, sm.xc);
        p1c_put_rows<T, HAS_L>(sm.dR, i, jc, u, l);
        p1c_push_k<T, HAS_L, SB>(sm.dx[c & 1][0], sm.dx[c & 1][1], i, jc, u, l);
    };
    auto push_r0 = [&]() {
        p1c_push_k<T, HAS_L, FB>(sm.rx[c & 1][0], sm.rx[c & 1][1], i, j0, u, l);
    };
    if (c == 0 && live) {
        if (g == 0) close_own();
        else push_r0();
    }

    for (int s = 0; s < CL; ++s) {
        cluster_arrive();
        cluster_wait();
        if (!live || s * SB >= m) continue;
        const int b = s & 1;
        if (s == c) {
            // own row sub-panel against the closed block
            if (g != c)
                p1c_product<T, HAS_L, FB>(u, l, sm.dR[0] + i * CS, sm.dR[1] + i * CS, sm.rx[b][0],
                                          sm.rx[b][1], j0);
            continue;
        }
        const bool next = s + 1 == c;   // this CTA closes the next sub-block
        if (g == s) p1c_put_rows<T, HAS_L>(sm.cP, i, jc, u, l);
        if (next && g == c) p1c_put_rows<T, HAS_L>(sm.bD, i, jc, u, l);
        __syncthreads();
        // column sub-panel: cell (ci, cj) of block (c, s) against the closed block
        p1c_cell<T, HAS_L, SB>(sm.cP, sm.cQ, ci, cj, sm.cP[0] + ci * CS, sm.cP[1] + ci * CS,
                               sm.dx[b][0], sm.dx[b][1], cj);
        __syncthreads();
        if (g == s) p1c_get_rows<T, HAS_L>(sm.cQ, i, jc, u, l);
        if (next) {
            // block (c, c) first, over all threads, then its closure
            p1c_cell<T, HAS_L, FB>(sm.bD, sm.bD, ci, cj, sm.cQ[0] + ci * CS, sm.cQ[1] + ci * CS,
                                   sm.rx[b][0], sm.rx[b][1], c * SB + cj);
            __syncthreads();
            if (g == c) {
                p1c_get_rows<T, HAS_L>(sm.bD, i, jc, u, l);
                close_own();
            }
        }
        if (g != s && !(next && g == c))
            p1c_product<T, HAS_L, FB>(u, l, sm.cQ[0] + i * CS, sm.cQ[1] + i * CS, sm.rx[b][0],
                                      sm.rx[b][1], j0);
        if (next && g != c) push_r0();
    }

    if (row < m) {
        if (vec && j0 + 4 <= m) {
            using V4 = typename E::V4;
            *reinterpret_cast<V4*>(Ur + j0) = V4{u[0], u[1], u[2], u[3]};
            if (HAS_L) *reinterpret_cast<V4*>(Lr + j0) = V4{l[0], l[1], l[2], l[3]};
        } else {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                if (j0 + q >= m) continue;
                Ur[j0 + q] = u[q];
                if (HAS_L) Lr[j0 + q] = l[q];
            }
        }
    }
}

// ---------------------------------------------------------------- launchers

template <class T>
static cudaError_t setup1() {
    cudaError_t e = cudaSuccess;
    auto set = [&](auto kernel, size_t bytes) {
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    };
    set(k_phase1<T, true, FB_LARGE>, P1Smem<T, true, FB_LARGE>::BYTES);
    set(k_phase1<T, false, FB_LARGE>, P1Smem<T, false, FB_LARGE>::BYTES);
    set(k_phase1c<T, true>, p1c_pre_bytes<true>());
    set(k_phase1c<T, false>, p1c_pre_bytes<false>());
    return e;
}

cudaError_t blocked_setup(bool is_int) {
    cudaError_t e = is_int ? setup1<int>() : setup1<float>();
    return e == cudaSuccess ? phase3_setup(is_int) : e;
}

template <class T, bool HAS_L, int FB>
static cudaError_t phase1_t(const Mats& m, int K, cudaStream_t s) {
    return for_batch_chunks(m, [&](int b0, int nbz) {
        T* U = static_cast<T*>(m.U) + (size_t)b0 * m.bstride;
        T* L = HAS_L ? static_cast<T*>(m.L) + (size_t)b0 * m.bstride : nullptr;
        before_launch(s, PH_ONE);
        const cudaError_t e = launch_prio(k_phase1<T, HAS_L, FB>, dim3(1, 1, nbz), dim3(P1S<FB>::NT),
                                          P1Smem<T, HAS_L, FB>::BYTES, s, U, L, m.n, m.ld,
                                          m.bstride, K, m.vec);
        after_launch(s, PH_ONE);
        return e;
    });
}

template <class T, bool HAS_L>
static cudaError_t phase1c_t(const Mats& m, int K, bool pre, cudaStream_t s) {
    return for_batch_chunks(m, [&](int b0, int nbz) {
        T* U = static_cast<T*>(m.U) + (size_t)b0 * m.bstride;
        T* L = HAS_L ? static_cast<T*>(m.L) + (size_t)b0 * m.bstride : nullptr;
        before_launch(s, PH_ONE);
        const size_t dyn = pre ? p1c_pre_bytes<HAS_L>() : 0;
        const cudaError_t e = launch_prio(k_phase1c<T, HAS_L>, dim3(CL, 1, nbz), dim3(CNT), dyn,
                                          s, U, L, m.n, m.ld, m.bstride, K, m.vec, pre);
        after_launch(s, PH_ONE);
        return e;
    });
}

template <class T, bool HAS_L>
static cudaError_t phase1_fb(const Mats& m, int K, bool pre, cudaStream_t s) {
    if (m.fb == FB_SMALL) return phase1c_t<T, HAS_L>(m, K, pre && K > 0, s);
    if (pre) return cudaErrorInvalidValue;   // 128-wide tiles: NEXT keeps the diagonal tile
    return phase1_t<T, HAS_L, FB_LARGE>(m, K, s);
}

cudaError_t launch_phase1(bool is_int, const Mats& m, int K, bool pre, cudaStream_t s) {
    if (is_int)
        return m.L ? phase1_fb<int, true>(m, K, pre, s) : phase1_fb<int, false>(m, K, pre, s);
    return m.L ? phase1_fb<float, true>(m, K, pre, s) : phase1_fb<float, false>(m, K, pre, s);
}

}  // namespace bs
