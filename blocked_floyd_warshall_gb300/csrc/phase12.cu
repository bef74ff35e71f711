// Three-phase blocked Floyd-Warshall over the bound pair (U, L).
//
// The matrix is cut into FB x FB tiles; block round K processes the middle
// atoms k of tile-row K in order, in three launches:
//   phase 1: tile (K,K), k serially, one CTA;
//   phase 2: row panel (K,J) and column panel (I,K), k serially, against the
//            finished diagonal tile;
//   phase 3: every other tile (I,J), against the finished panels.  Its
//            operands are final, so the k order inside the block is free and U
//            and L are updated together in one pass.
//
// Rules (GPU Gems 2 ch. 43, section 2): U[i,j] = min(U[i,j], U[i,k] + U[k,j]);
// L[i,j] = max(L[i,j], L[k,j] - U[i,k], Lcol[i] - U[k,j]), with the upper
// bound tightened first.  Lcol[i] is L[i,k] raised to max(L[i,k], L[k,k] -
// U[i,k]) wherever column k is still being formed (phase 1, column panel);
// phase-2 row panels and phase 3 read finished column values where that raise
// is already contained.  The result is the fixed point of the triangle
// inequalities, the same as the round-by-round schedule (exactly in int32; in
// fp32 exactly for values on the 1/1024 grid below 2^14).
//
// Inside phases 1 and 2 each step k is round-synchronous: every thread keeps
// its cells in registers and the lines a step reads are published to shared
// memory, double-buffered, one barrier per publication (phase 1: one middle
// atom per barrier; phase 2: two).
//
// This file: phases 1 and 2 and the shared-memory set-up of all three phases.
#include "pairops.cuh"

namespace bs {

// Micro-tile shapes.  Phases 1 and 2 advance one (phase 2: two) middle atoms
// per barrier, so their per-step latency, not their throughput, sets their
// time: 4 x 4 cells per thread on 64-wide tiles (256 threads); on 128-wide
// tiles phase 1 runs 8 x 8 (256 threads) and phase 2 8 x 4 (512 threads), the
// faster shape for each measured on the GB300.
template <int FB> using P1S = Shape<FB, (FB == FB_SMALL ? 4 : 8), (FB == FB_SMALL ? 4 : 8)>;
template <int FB> using P2S = Shape<FB, (FB == FB_SMALL ? 4 : 8), 4>;

// ---------------------------------------------------------------- phase 1

template <class T, bool HAS_L, int FB>
__global__ void __launch_bounds__(P1S<FB>::NT)
k_phase1(T* __restrict__ U, T* __restrict__ L, int n, int ld, long long bstride, int K, bool vec) {
    using S = P1S<FB>;
    using E = El<T>;
    __shared__ T sRU[2][FB], sRL[2][FB], sCU[2][FB], sCL[2][FB];
    const size_t off = (size_t)blockIdx.z * (size_t)bstride;
    U += off;
    if (HAS_L) L += off;
    const int o = K * FB;
    const int m = min(FB, n - o);
    T* Ut = U + (size_t)o * ld + o;
    T* Lt = HAS_L ? L + (size_t)o * ld + o : nullptr;

    T u[S::TM][S::TN], l[S::TM][S::TN];
    load_tile<S>(u, Ut, ld, m, m, vec, E::upad());
    if (HAS_L) load_tile<S>(l, Lt, ld, m, m, vec, E::lpad());
    publish_row<S, T, HAS_L>(u, l, 0, sRU[0], sRL[0]);
    publish_col<S, T, HAS_L>(u, l, 0, sCU[0], sCL[0]);
    __syncthreads();

    const int r0 = S::row0();
    for (int k = 0; k < m; ++k) {
        const int b = k & 1;
        T a[S::TM], al[S::TM], bb[S::TN], bl[S::TN];
#pragma unroll
        for (int r = 0; r < S::TM; ++r) {
            a[r] = sCU[b][r0 + r];
            al[r] = HAS_L ? sCL[b][r0 + r] : T(0);
        }
#pragma unroll
        for (int c = 0; c < S::TN; ++c) {
            bb[c] = sRU[b][S::col(c)];
            bl[c] = HAS_L ? sRL[b][S::col(c)] : T(0);
        }
        if (HAS_L) {
            const T lkk = sRL[b][k];
#pragma unroll
            for (int r = 0; r < S::TM; ++r) al[r] = E::mx(al[r], E::sub(lkk, a[r]));
        }
        fw_update<S, T, HAS_L>(u, l, a, al, bb, bl);
        if (k + 1 < m) {
            publish_row<S, T, HAS_L>(u, l, k + 1, sRU[b ^ 1], sRL[b ^ 1]);
            publish_col<S, T, HAS_L>(u, l, k + 1, sCU[b ^ 1], sCL[b ^ 1]);
        }
        __syncthreads();
    }
    store_tile<S>(u, Ut, ld, m, m, vec);
    if (HAS_L) store_tile<S>(l, Lt, ld, m, m, vec);
}

// ---------------------------------------------------------------- phase 2
//
// Panels of block round K against the finished diagonal tile D = (K,K), two
// middle atoms (k, k+1) per barrier.  Row k and row k+1 of a row-panel tile
// (columns k and k+1 of a column-panel tile) belong to one thread: it applies
// step k to line k+1 from its own registers and publishes the pair (line k,
// line k+1 after step k).  Every cell then takes both steps with the paired
// instructions of phase 3 -- the same sums and the same exact min/max as two
// sequential steps.
//   row panel (K,P):   b = (U[k,j], U'[k+1,j]),      a = (D_U[i,k], D_U[i,k+1])
//   column panel (P,K): a = (U[i,k], U'[i,k+1]),      b = (D_U[k,j], D_U[k+1,j])
//                       al = the column values raised by the closure rule.
// D is staged as [i][k] (row panel) or k-interleaved [k/2][j][k%2] (column
// panel), so each operand pair is one 8-byte load.  An odd last step pairs
// with a padding line, which changes nothing.

constexpr int DPAD = 2;   // diagonal tile row stride FB + DPAD: even, so pairs stay aligned

// Row panel: the owner of rows k, k+1 publishes (row k, row k+1 after step k).
template <class T, bool HAS_L, int FB>
__device__ __forceinline__ void p2_publish_rows(const T (&u)[P2S<FB>::TM][P2S<FB>::TN],
                                                const T (&l)[P2S<FB>::TM][P2S<FB>::TN], int k,
                                                const T* dU, const T* dL, T* sU, T* sL) {
    using S = P2S<FB>;
    using E = El<T>;
    constexpr int DS = FB + DPAD;
    const int r0 = S::row0();
#pragma unroll
    for (int rr = 0; rr < S::TM; rr += 2) {
        if (r0 + rr != k) continue;
        const T a1 = dU[(k + 1) * DS + k];
        const T al1 = HAS_L ? dL[(k + 1) * DS + k] : T(0);
#pragma unroll
        for (int c = 0; c < S::TN; ++c) {
            const int j = S::col(c);
            sU[2 * j] = u[rr][c];
            sU[2 * j + 1] = E::mn(u[rr + 1][c], E::add(a1, u[rr][c]));
            if (HAS_L) {
                sL[2 * j] = l[rr][c];
                sL[2 * j + 1] = E::mx(l[rr + 1][c], E::mx(E::sub(l[rr][c], a1), E::sub(al1, u[rr][c])));
            }
        }
    }
}

// Column panel: the owner of columns k, k+1 publishes, per row, (U[i,k],
// U'[i,k+1]) and the closure-raised column values (Lc_k[i], Lc_k+1[i]).
// dU, dL: the diagonal tile, k-interleaved.
template <class T, bool HAS_L, int FB>
__device__ __forceinline__ void p2_publish_cols(const T (&u)[P2S<FB>::TM][P2S<FB>::TN],
                                                const T (&l)[P2S<FB>::TM][P2S<FB>::TN], int k,
                                                const T* dU, const T* dL, T* sU, T* sL) {
    using S = P2S<FB>;
    using E = El<T>;
    const int r0 = S::row0();
#pragma unroll
    for (int c = 0; c < S::TN; c += 2) {
        if (S::col(c) != k) continue;
        const int kb = (k >> 1) * (2 * FB);
        const T ukk1 = dU[kb + 2 * (k + 1)];                        // D[k][k+1]
        const T lkk = HAS_L ? dL[kb + 2 * k] : T(0);                // D[k][k]
        const T lkk1 = HAS_L ? dL[kb + 2 * (k + 1)] : T(0);         // D[k][k+1]
        const T lk1k1 = HAS_L ? dL[kb + 2 * (k + 1) + 1] : T(0);    // D[k+1][k+1]
#pragma unroll
        for (int r = 0; r < S::TM; ++r) {
            const T uk = u[r][c];
            const T u1 = E::mn(u[r][c + 1], E::add(uk, ukk1));
            sU[2 * (r0 + r)] = uk;
            sU[2 * (r0 + r) + 1] = u1;
            if (HAS_L) {
                const T lc0 = E::mx(l[r][c], E::sub(lkk, uk));
                const T l1 = E::mx(l[r][c + 1], E::mx(E::sub(lkk1, uk), E::sub(lc0, ukk1)));
                sL[2 * (r0 + r)] = lc0;
                sL[2 * (r0 + r) + 1] = E::mx(l1, E::sub(lk1k1, u1));
            }
        }
    }
}

template <class T, bool HAS_L, int FB>
__device__ __forceinline__ void p2_row_panel(T* U, T* L, size_t ld, int o, int op, int mk,
                                             int mp, bool vec, bool sym, T* dU, T* dL,
                                             T (*sU)[2 * FB], T (*sL)[2 * FB]) {
    using S = P2S<FB>;
    using E = El<T>;
    using LD = PairLoad<T>;
    using P = typename LD::P;
    constexpr bool NEG = std::is_same<T, int>::value;
    constexpr int DS = FB + DPAD;
    const int r0 = S::row0(), cq = S::cq();
    T* Ut = U + (size_t)o * ld + op;
    T* Lt = HAS_L ? L + (size_t)o * ld + op : nullptr;
    T u[S::TM][S::TN], l[S::TM][S::TN];
    load_tile<S>(u, Ut, ld, mk, mp, vec, E::upad());
    if (HAS_L) load_tile<S>(l, Lt, ld, mk, mp, vec, E::lpad());

    p2_publish_rows<T, HAS_L, FB>(u, l, 0, dU, dL, sU[0], sL[0]);
    __syncthreads();
#pragma unroll 1
    for (int k = 0; k < mk; k += 2) {
        const int b = (k >> 1) & 1;
        P a[S::TM], al[S::TM], bb[S::TN], bl[S::TN];
#pragma unroll
        for (int r = 0; r < S::TM; ++r) {
            a[r] = LD::ld2(dU + (r0 + r) * DS + k);
            if (HAS_L) al[r] = LD::ld2(dL + (r0 + r) * DS + k);
        }
#pragma unroll
        for (int h = 0; h < S::QUADS; ++h) {
            const int jb = (h * S::QSTRIDE + cq) * 2;
            LD::ld4(&sU[b][jb], bb[h * 4 + 0], bb[h * 4 + 1]);
            LD::ld4(&sU[b][jb + 4], bb[h * 4 + 2], bb[h * 4 + 3]);
            if (HAS_L) {
                LD::ld4(&sL[b][jb], bl[h * 4 + 0], bl[h * 4 + 1]);
                LD::ld4(&sL[b][jb + 4], bl[h * 4 + 2], bl[h * 4 + 3]);
            }
        }
#pragma unroll
        for (int r = 0; r < S::TM; ++r)
#pragma unroll
            for (int q = 0; q < S::TN; ++q) PairOps<T>::upper(u[r][q], a[r], bb[q]);
        if (HAS_L) {
            if (NEG) {
#pragma unroll
                for (int r = 0; r < S::TM; ++r) a[r] = LD::neg(a[r]);
#pragma unroll
                for (int q = 0; q < S::TN; ++q) bb[q] = LD::neg(bb[q]);
            }
#pragma unroll
            for (int r = 0; r < S::TM; ++r)
#pragma unroll
                for (int q = 0; q < S::TN; ++q) PairOps<T>::lower(l[r][q], a[r], al[r], bb[q], bl[q]);
        }
        if (k + 2 < mk) p2_publish_rows<T, HAS_L, FB>(u, l, k + 2, dU, dL, sU[b ^ 1], sL[b ^ 1]);
        __syncthreads();
    }
    store_tile<S>(u, Ut, ld, mk, mp, vec);
    if (HAS_L) store_tile<S>(l, Lt, ld, mk, mp, vec);
    if (sym) {
        // symmetric inputs: the column panel tile (P, K) is the transpose
        store_tile_t<S>(u, U + (size_t)op * ld + o, ld, mk, mp, vec);
        if (HAS_L) store_tile_t<S>(l, L + (size_t)op * ld + o, ld, mk, mp, vec);
    }
}

template <class T, bool HAS_L, int FB>
__device__ __forceinline__ void p2_col_panel(T* U, T* L, size_t ld, int o, int op, int mk,
                                             int mp, bool vec, T* dU, T* dL,
                                             T (*sU)[2 * FB], T (*sL)[2 * FB]) {
    using S = P2S<FB>;
    using E = El<T>;
    using LD = PairLoad<T>;
    using P = typename LD::P;
    constexpr bool NEG = std::is_same<T, int>::value;
    const int r0 = S::row0(), cq = S::cq();
    T* Ut = U + (size_t)op * ld + o;
    T* Lt = HAS_L ? L + (size_t)op * ld + o : nullptr;
    T u[S::TM][S::TN], l[S::TM][S::TN];
    load_tile<S>(u, Ut, ld, mp, mk, vec, E::upad());
    if (HAS_L) load_tile<S>(l, Lt, ld, mp, mk, vec, E::lpad());

    p2_publish_cols<T, HAS_L, FB>(u, l, 0, dU, dL, sU[0], sL[0]);
    __syncthreads();
#pragma unroll 1
    for (int k = 0; k < mk; k += 2) {
        const int b = (k >> 1) & 1;
        P a[S::TM], al[S::TM], bb[S::TN], bl[S::TN];
#pragma unroll
        for (int r = 0; r < S::TM; ++r) {
            a[r] = LD::ld2(&sU[b][2 * (r0 + r)]);
            if (HAS_L) al[r] = LD::ld2(&sL[b][2 * (r0 + r)]);
        }
        const int bo = (k >> 1) * (2 * FB);
#pragma unroll
        for (int h = 0; h < S::QUADS; ++h) {
            const int jb = bo + (h * S::QSTRIDE + cq) * 2;
            LD::ld4(dU + jb, bb[h * 4 + 0], bb[h * 4 + 1]);
            LD::ld4(dU + jb + 4, bb[h * 4 + 2], bb[h * 4 + 3]);
            if (HAS_L) {
                LD::ld4(dL + jb, bl[h * 4 + 0], bl[h * 4 + 1]);
                LD::ld4(dL + jb + 4, bl[h * 4 + 2], bl[h * 4 + 3]);
            }
        }
#pragma unroll
        for (int r = 0; r < S::TM; ++r)
#pragma unroll
            for (int q = 0; q < S::TN; ++q) PairOps<T>::upper(u[r][q], a[r], bb[q]);
        if (HAS_L) {
            if (NEG) {
#pragma unroll
                for (int r = 0; r < S::TM; ++r) a[r] = LD::neg(a[r]);
#pragma unroll
                for (int q = 0; q < S::TN; ++q) bb[q] = LD::neg(bb[q]);
            }
#pragma unroll
            for (int r = 0; r < S::TM; ++r)
#pragma unroll
                for (int q = 0; q < S::TN; ++q) PairOps<T>::lower(l[r][q], a[r], al[r], bb[q], bl[q]);
        }
        if (k + 2 < mk) p2_publish_cols<T, HAS_L, FB>(u, l, k + 2, dU, dL, sU[b ^ 1], sL[b ^ 1]);
        __syncthreads();
    }
    store_tile<S>(u, Ut, ld, mp, mk, vec);
    if (HAS_L) store_tile<S>(l, Lt, ld, mp, mk, vec);
}

template <class T, bool HAS_L, int FB>
__global__ void __launch_bounds__(P2S<FB>::NT)
k_phase2(T* __restrict__ U, T* __restrict__ L, int n, int ld, long long bstride, int K, bool vec,
         bool sym) {
    using S = P2S<FB>;
    using E = El<T>;
    constexpr int NT = P2S<FB>::NT;
    constexpr int DS = FB + DPAD;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    T* dU = reinterpret_cast<T*>(smem_raw);
    T* dL = dU + FB * DS;
    __shared__ __align__(16) T sU[2][2 * FB];
    __shared__ __align__(16) T sL[2][2 * FB];

    const size_t off = (size_t)blockIdx.z * (size_t)bstride;
    U += off;
    if (HAS_L) L += off;
    const int o = K * FB;
    const int mk = min(FB, n - o);
    const int P = (int)blockIdx.x + ((int)blockIdx.x >= K);
    const int op = P * FB;
    const int mp = min(FB, n - op);
    const bool row_panel = blockIdx.y == 0;

    // the finished diagonal tile, padded: [i][k] for the row panel,
    // k-interleaved [k/2][j][k%2] for the column panel
    for (int e = threadIdx.x; e < FB * FB; e += NT) {
        const int i = e / FB, j = e % FB;
        const bool in = i < mk && j < mk;
        const int d = row_panel ? i * DS + j : (i >> 1) * (2 * FB) + 2 * j + (i & 1);
        dU[d] = in ? U[(size_t)(o + i) * ld + o + j] : E::upad();
        if (HAS_L) dL[d] = in ? L[(size_t)(o + i) * ld + o + j] : E::lpad();
    }
    __syncthreads();
    if (row_panel)
        p2_row_panel<T, HAS_L, FB>(U, L, ld, o, op, mk, mp, vec, sym, dU, dL, sU, sL);
    else
        p2_col_panel<T, HAS_L, FB>(U, L, ld, o, op, mk, mp, vec, dU, dL, sU, sL);
}

// ---------------------------------------------------------------- launchers

template <class T, bool HAS_L, int FB>
static size_t p2_smem() {
    return (size_t)(HAS_L ? 2 : 1) * FB * (FB + DPAD) * sizeof(T);
}

template <class T>
static cudaError_t setup12() {
    cudaError_t e = cudaSuccess;
    auto set = [&](auto kernel, size_t bytes) {
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    };
    set(k_phase2<T, true, FB_LARGE>, p2_smem<T, true, FB_LARGE>());
    set(k_phase2<T, false, FB_LARGE>, p2_smem<T, false, FB_LARGE>());
    set(k_phase2<T, true, FB_SMALL>, p2_smem<T, true, FB_SMALL>());
    set(k_phase2<T, false, FB_SMALL>, p2_smem<T, false, FB_SMALL>());
    return e;
}

cudaError_t blocked_setup(bool is_int) {
    cudaError_t e = is_int ? setup12<int>() : setup12<float>();
    return e == cudaSuccess ? phase3_setup(is_int) : e;
}

template <class T, bool HAS_L, int FB>
static cudaError_t phase1_t(const Mats& m, int K, cudaStream_t s) {
    return for_batch_chunks(m, [&](int b0, int nbz) {
        T* U = static_cast<T*>(m.U) + (size_t)b0 * m.bstride;
        T* L = HAS_L ? static_cast<T*>(m.L) + (size_t)b0 * m.bstride : nullptr;
        before_launch(s, PH_ONE);
        k_phase1<T, HAS_L, FB><<<dim3(1, 1, nbz), P1S<FB>::NT, 0, s>>>(U, L, m.n, m.ld,
                                                                       m.bstride, K, m.vec);
        after_launch(s, PH_ONE);
    });
}

template <class T, bool HAS_L, int FB>
static cudaError_t phase2_t(const Mats& m, int K, cudaStream_t s) {
    const int nb = (m.n + FB - 1) / FB;
    if (nb < 2) return cudaSuccess;
    return for_batch_chunks(m, [&](int b0, int nbz) {
        T* U = static_cast<T*>(m.U) + (size_t)b0 * m.bstride;
        T* L = HAS_L ? static_cast<T*>(m.L) + (size_t)b0 * m.bstride : nullptr;
        before_launch(s, PH_TWO);
        k_phase2<T, HAS_L, FB><<<dim3(nb - 1, m.sym ? 1 : 2, nbz), P2S<FB>::NT,
                                 p2_smem<T, HAS_L, FB>(), s>>>(U, L, m.n, m.ld, m.bstride, K,
                                                              m.vec, m.sym);
        after_launch(s, PH_TWO);
    });
}

template <class T, bool HAS_L>
static cudaError_t phase12_fb(int which, const Mats& m, int K, cudaStream_t s) {
    if (which == 1)
        return m.fb == FB_SMALL ? phase1_t<T, HAS_L, FB_SMALL>(m, K, s)
                                : phase1_t<T, HAS_L, FB_LARGE>(m, K, s);
    return m.fb == FB_SMALL ? phase2_t<T, HAS_L, FB_SMALL>(m, K, s)
                            : phase2_t<T, HAS_L, FB_LARGE>(m, K, s);
}

static cudaError_t phase12(int which, bool is_int, const Mats& m, int K, cudaStream_t s) {
    if (is_int) return m.L ? phase12_fb<int, true>(which, m, K, s) : phase12_fb<int, false>(which, m, K, s);
    return m.L ? phase12_fb<float, true>(which, m, K, s) : phase12_fb<float, false>(which, m, K, s);
}

cudaError_t launch_phase1(bool is_int, const Mats& m, int K, cudaStream_t s) {
    return phase12(1, is_int, m, K, s);
}
cudaError_t launch_phase2(bool is_int, const Mats& m, int K, cudaStream_t s) {
    return phase12(2, is_int, m, K, s);
}

}  // namespace bs
