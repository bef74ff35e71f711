// Three-phase blocked Floyd-Warshall over the bound pair (U, L).
//
// The matrix is cut into FB x FB tiles; block round K processes the middle
// atoms k of tile-row K in order, in three launches:
//   phase 1: tile (K,K), k serially, one CTA (this file);
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
// Inside phase 1 each step k is round-synchronous: every thread keeps its
// cells in registers and row and column k are published to shared memory,
// double-buffered, one barrier per middle atom.
#include "pairops.cuh"

namespace bs {

// Phase 1 computes the closure of tile (K,K) by the same blocked scheme one
// level down, on the tile held in shared memory: for each SB-wide sub-block s
// of its middle atoms,
//   (a) one warp closes sub-block (s,s), k serially, exchanging row and column
//       k by warp shuffles (no barrier per middle atom);
//   (b) the sub-panels in sub-block row s and sub-block column s take the
//       product with the closed sub-block (each cell computed into registers,
//       written after a barrier, so every operand is the value from before);
//   (c) every other cell takes the product of its sub-panels, paired middle
//       atoms as in phase 3.
// (b) and (c) are the update of the other phases, X[i,j] against T[i,k] and
// T[k,j] over the sub-block's middle atoms k.  Four barriers per sub-block
// instead of one per middle atom.

constexpr int SB = 16;          // sub-block width
constexpr int CPL = SB * SB / 32;  // (a): cells per lane
constexpr int LPR = SB / CPL;      // (a): lanes per sub-block row
constexpr int HALVES = SB / 8;     // (b): 8-cell units per sub-panel line

// (c) micro-tile: 4 x 4 cells on 64-wide tiles (256 threads), 8 x 4 on 128-wide
// tiles (512 threads).  In both, warp w covers tile rows 8w .. 8w+7 and thread
// tx columns 4tx .. 4tx+3, so a sub-block row is whole warps and a sub-block
// column whole quads.
template <int FB> using P1S = Shape<FB, (FB == FB_SMALL ? 4 : 8), 4>;

template <class T, bool HAS_L, int FB>
struct P1Smem {
    static constexpr int TS = FB + 2;            // tile row stride: even, so pairs stay 8-byte aligned
    static constexpr int TILE = FB * TS;         // T[i][j] at i * TS + j
    static constexpr int RP = SB * FB;           // sub-block row panel, k-interleaved [k/2][j][k%2]
    static constexpr int DI = SB * SB;           // closed sub-block, k-interleaved [k/2][j][k%2]
    static constexpr int MATS = HAS_L ? 2 : 1;
    static constexpr size_t BYTES = MATS * (TILE + RP + DI) * sizeof(T);   // tU tL | rU rL | dU dL
};

// (a): closure of the SB x SB sub-block at (sb, sb), one warp.  Lane
// LPR*i + h holds row i, columns CPL*h .. CPL*h + CPL-1.  Step k: row k comes
// from lanes LPR*k + h, column k of row i from lane LPR*i + k/CPL; all
// shuffles precede the updates, so each step reads the values from before it
// (round-synchronous), and the lower-bound column is raised by the closure
// rule, Lc = max(L[i,k], L[k,k] - U[i,k]).  The closed sub-block is written
// back row-major and k-interleaved (dU, dL) for the column sub-panel.
template <class T, bool HAS_L, int TS>
__device__ __forceinline__ void p1_sub_closure(T* tU, T* tL, T* dU, T* dL, int sb) {
    using E = El<T>;
    constexpr unsigned FULL = 0xffffffffu;
    const int lane = threadIdx.x & 31;
    const int i = lane / LPR, h = lane % LPR;
    T* pu = tU + (sb + i) * TS + sb + CPL * h;
    T* pl = HAS_L ? tL + (sb + i) * TS + sb + CPL * h : nullptr;
    T u[CPL], l[CPL];
#pragma unroll
    for (int c = 0; c < CPL; ++c) {
        u[c] = pu[c];
        l[c] = HAS_L ? pl[c] : T(0);
    }
#pragma unroll
    for (int k = 0; k < SB; ++k) {
        const int own = LPR * i + k / CPL;   // holder of (i, k)
        const int row = LPR * k + h;         // holder of (k, my columns)
        const T uik = __shfl_sync(FULL, u[k % CPL], own);
        T ukj[CPL], lkj[CPL];
#pragma unroll
        for (int c = 0; c < CPL; ++c) ukj[c] = __shfl_sync(FULL, u[c], row);
        T lc = T(0);
        if (HAS_L) {
            const T lik = __shfl_sync(FULL, l[k % CPL], own);
            const T lkk = __shfl_sync(FULL, l[k % CPL], LPR * k + k / CPL);
#pragma unroll
            for (int c = 0; c < CPL; ++c) lkj[c] = __shfl_sync(FULL, l[c], row);
            lc = E::mx(lik, E::sub(lkk, uik));
        }
#pragma unroll
        for (int c = 0; c < CPL; ++c) u[c] = E::mn(u[c], E::add(uik, ukj[c]));
        if (HAS_L) {
#pragma unroll
            for (int c = 0; c < CPL; ++c)
                l[c] = E::mx(l[c], E::mx(E::sub(lkj[c], uik), E::sub(lc, ukj[c])));
        }
    }
#pragma unroll
    for (int c = 0; c < CPL; ++c) {
        pu[c] = u[c];
        const int d = (i >> 1) * (2 * SB) + 2 * (CPL * h + c) + (i & 1);
        dU[d] = u[c];
        if (HAS_L) {
            pl[c] = l[c];
            dL[d] = l[c];
        }
    }
}

// ---------------------------------------------------------------- phase 1

template <class T, bool HAS_L, int FB>
__global__ void __launch_bounds__(P1S<FB>::NT)
k_phase1(T* __restrict__ U, T* __restrict__ L, int n, int ld, long long bstride, int K, bool vec) {
    using S = P1S<FB>;
    using E = El<T>;
    using SM = P1Smem<T, HAS_L, FB>;
    using LD = PairLoad<T>;
    using P = typename LD::P;
    constexpr int NT = S::NT, TS = SM::TS;
    constexpr int W = FB - SB;                          // sub-panel length outside the sub-block
    static_assert(2 * HALVES * W <= NT, "one (b) unit per thread");
    constexpr bool NEG = std::is_same<T, int>::value;   // int lower bound adds negated values
    extern __shared__ __align__(16) unsigned char smem_raw[];
    T* tU = reinterpret_cast<T*>(smem_raw);
    T* tL = tU + SM::TILE;
    T* rU = tU + SM::MATS * SM::TILE;
    T* rL = rU + SM::RP;
    T* dU = rU + SM::MATS * SM::RP;
    T* dL = dU + SM::DI;

    const size_t off = (size_t)blockIdx.z * (size_t)bstride;
    U += off;
    if (HAS_L) L += off;
    const int o = K * FB;
    const int m = min(FB, n - o);
    T* Ut = U + (size_t)o * ld + o;
    T* Lt = HAS_L ? L + (size_t)o * ld + o : nullptr;

    // the tile into shared memory; cells outside the m x m block get pads
    for (int e = threadIdx.x; e < FB * FB / 4; e += NT) {
        const int i = e / (FB / 4), j = (e % (FB / 4)) * 4;
        T xu[4], xl[4];
        if (vec && i < m && j + 4 <= m) {
            using V4 = typename E::V4;
            const V4 v = *reinterpret_cast<const V4*>(Ut + (size_t)i * ld + j);
            xu[0] = v.x; xu[1] = v.y; xu[2] = v.z; xu[3] = v.w;
            if (HAS_L) {
                const V4 w = *reinterpret_cast<const V4*>(Lt + (size_t)i * ld + j);
                xl[0] = w.x; xl[1] = w.y; xl[2] = w.z; xl[3] = w.w;
            }
        } else {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const bool in = i < m && j + q < m;
                xu[q] = in ? Ut[(size_t)i * ld + j + q] : E::upad();
                if (HAS_L) xl[q] = in ? Lt[(size_t)i * ld + j + q] : E::lpad();
            }
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            tU[i * TS + j + q] = xu[q];
            if (HAS_L) tL[i * TS + j + q] = xl[q];
        }
    }
    __syncthreads();

    const int r0 = S::row0(), cq = S::cq();
    const int warp = threadIdx.x >> 5;
    for (int sb = 0; sb < m; sb += SB) {
        // (a)
        if (warp == 0) p1_sub_closure<T, HAS_L, TS>(tU, tL, dU, dL, sb);
        __syncthreads();

        // (b): thread t < HALVES*W: row-panel cells (sb + 8hh + q, p), q < 8;
        //      t < 2*HALVES*W: column-panel cells (p, sb + 8hh + q), q < 8.
        // Both are whole warps.  Operand pairs (k, k+1): the row panel reads
        // the closed sub-block's rows as pairs and packs its own column; the
        // column panel reads its row as pairs and the k-interleaved copy of
        // the closed sub-block.
        const int t = threadIdx.x;
        const bool rowp = t < HALVES * W;
        const bool unit = t < 2 * HALVES * W;
        const int v = rowp ? t : t - HALVES * W;
        const int hh = v / W, p = v % W + (v % W >= sb ? SB : 0);
        T xu[8], xl[8];
        if (rowp) {
            const int i0 = sb + 8 * hh;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                xu[q] = tU[(i0 + q) * TS + p];
                xl[q] = HAS_L ? tL[(i0 + q) * TS + p] : T(0);
            }
#pragma unroll 2
            for (int kk = 0; kk < SB; kk += 2) {
                P a[8], al[8];
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    a[q] = LD::ld2(tU + (i0 + q) * TS + sb + kk);
                    if (HAS_L) al[q] = LD::ld2(tL + (i0 + q) * TS + sb + kk);
                }
                P b = LD::mk(tU[(sb + kk) * TS + p], tU[(sb + kk + 1) * TS + p]);
                P bl = b;
                if (HAS_L) bl = LD::mk(tL[(sb + kk) * TS + p], tL[(sb + kk + 1) * TS + p]);
#pragma unroll
                for (int q = 0; q < 8; ++q) PairOps<T>::upper(xu[q], a[q], b);
                if (HAS_L) {
                    if (NEG) {
#pragma unroll
                        for (int q = 0; q < 8; ++q) a[q] = LD::neg(a[q]);
                        b = LD::neg(b);
                    }
#pragma unroll
                    for (int q = 0; q < 8; ++q) PairOps<T>::lower(xl[q], a[q], al[q], b, bl);
                }
            }
        } else if (unit) {
            const int j0 = 8 * hh;   // within the sub-block
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                xu[q] = tU[p * TS + sb + j0 + q];
                xl[q] = HAS_L ? tL[p * TS + sb + j0 + q] : T(0);
            }
#pragma unroll 2
            for (int kk = 0; kk < SB; kk += 2) {
                P a = LD::ld2(tU + p * TS + sb + kk);
                P al = a;
                if (HAS_L) al = LD::ld2(tL + p * TS + sb + kk);
                P b[8], bl[8];
                const int db = (kk >> 1) * (2 * SB) + 2 * j0;
#pragma unroll
                for (int q = 0; q < 8; q += 2) {
                    LD::ld4(dU + db + 2 * q, b[q], b[q + 1]);
                    if (HAS_L) LD::ld4(dL + db + 2 * q, bl[q], bl[q + 1]);
                }
#pragma unroll
                for (int q = 0; q < 8; ++q) PairOps<T>::upper(xu[q], a, b[q]);
                if (HAS_L) {
                    if (NEG) {
                        a = LD::neg(a);
#pragma unroll
                        for (int q = 0; q < 8; ++q) b[q] = LD::neg(b[q]);
                    }
#pragma unroll
                    for (int q = 0; q < 8; ++q) PairOps<T>::lower(xl[q], a, al, b[q], bl[q]);
                }
            }
        }
        __syncthreads();
        if (unit) {
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const int ci = rowp ? (sb + 8 * hh + q) * TS + p : p * TS + sb + 8 * hh + q;
                tU[ci] = xu[q];
                if (HAS_L) tL[ci] = xl[q];
                if (rowp) {
                    // row-panel copy for (c): middle atom k = 8hh + q, column p
                    const int d = ((8 * hh + q) >> 1) * (2 * FB) + 2 * p + (q & 1);
                    rU[d] = xu[q];
                    if (HAS_L) rL[d] = xl[q];
                }
            }
        }
        __syncthreads();

        // (c): threads whose rows lie in sub-block row s skip (whole warps);
        // those whose columns lie in sub-block column s compute but do not store.
        if ((r0 / SB) != (sb / SB)) {
            const bool keep = (cq / SB) != (sb / SB);
            T u[S::TM][S::TN], l[S::TM][S::TN];
#pragma unroll
            for (int r = 0; r < S::TM; ++r)
#pragma unroll
                for (int q = 0; q < S::TN; ++q) {
                    u[r][q] = tU[(r0 + r) * TS + cq + q];
                    l[r][q] = HAS_L ? tL[(r0 + r) * TS + cq + q] : T(0);
                }
#pragma unroll 2
            for (int kk = 0; kk < SB; kk += 2) {
                P a[S::TM], al[S::TM], b[S::TN], bl[S::TN];
#pragma unroll
                for (int r = 0; r < S::TM; ++r) {
                    a[r] = LD::ld2(tU + (r0 + r) * TS + sb + kk);
                    if (HAS_L) al[r] = LD::ld2(tL + (r0 + r) * TS + sb + kk);
                }
                const int jb = (kk >> 1) * (2 * FB) + cq * 2;
                LD::ld4(rU + jb, b[0], b[1]);
                LD::ld4(rU + jb + 4, b[2], b[3]);
                if (HAS_L) {
                    LD::ld4(rL + jb, bl[0], bl[1]);
                    LD::ld4(rL + jb + 4, bl[2], bl[3]);
                }
#pragma unroll
                for (int r = 0; r < S::TM; ++r)
#pragma unroll
                    for (int q = 0; q < S::TN; ++q) PairOps<T>::upper(u[r][q], a[r], b[q]);
                if (HAS_L) {
                    if (NEG) {
#pragma unroll
                        for (int r = 0; r < S::TM; ++r) a[r] = LD::neg(a[r]);
#pragma unroll
                        for (int q = 0; q < S::TN; ++q) b[q] = LD::neg(b[q]);
                    }
#pragma unroll
                    for (int r = 0; r < S::TM; ++r)
#pragma unroll
                        for (int q = 0; q < S::TN; ++q)
                            PairOps<T>::lower(l[r][q], a[r], al[r], b[q], bl[q]);
                }
            }
            if (keep) {
#pragma unroll
                for (int r = 0; r < S::TM; ++r)
#pragma unroll
                    for (int q = 0; q < S::TN; ++q) {
                        tU[(r0 + r) * TS + cq + q] = u[r][q];
                        if (HAS_L) tL[(r0 + r) * TS + cq + q] = l[r][q];
                    }
            }
        }
        __syncthreads();
    }

    for (int e = threadIdx.x; e < FB * FB / 4; e += NT) {
        const int i = e / (FB / 4), j = (e % (FB / 4)) * 4;
        if (i >= m) continue;
        if (vec && j + 4 <= m) {
            using V4 = typename E::V4;
            const T* su = tU + i * TS + j;
            *reinterpret_cast<V4*>(Ut + (size_t)i * ld + j) = V4{su[0], su[1], su[2], su[3]};
            if (HAS_L) {
                const T* sl = tL + i * TS + j;
                *reinterpret_cast<V4*>(Lt + (size_t)i * ld + j) = V4{sl[0], sl[1], sl[2], sl[3]};
            }
        } else {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                if (j + q >= m) continue;
                Ut[(size_t)i * ld + j + q] = tU[i * TS + j + q];
                if (HAS_L) Lt[(size_t)i * ld + j + q] = tL[i * TS + j + q];
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
    set(k_phase1<T, true, FB_SMALL>, P1Smem<T, true, FB_SMALL>::BYTES);
    set(k_phase1<T, false, FB_SMALL>, P1Smem<T, false, FB_SMALL>::BYTES);
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
        k_phase1<T, HAS_L, FB><<<dim3(1, 1, nbz), P1S<FB>::NT, P1Smem<T, HAS_L, FB>::BYTES, s>>>(
            U, L, m.n, m.ld, m.bstride, K, m.vec);
        after_launch(s, PH_ONE);
    });
}

template <class T, bool HAS_L>
static cudaError_t phase1_fb(const Mats& m, int K, cudaStream_t s) {
    return m.fb == FB_SMALL ? phase1_t<T, HAS_L, FB_SMALL>(m, K, s)
                            : phase1_t<T, HAS_L, FB_LARGE>(m, K, s);
}

cudaError_t launch_phase1(bool is_int, const Mats& m, int K, cudaStream_t s) {
    if (is_int) return m.L ? phase1_fb<int, true>(m, K, s) : phase1_fb<int, false>(m, K, s);
    return m.L ? phase1_fb<float, true>(m, K, s) : phase1_fb<float, false>(m, K, s);
}

}  // namespace bs
