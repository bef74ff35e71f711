// Phase 1 of the three-phase blocked Floyd-Warshall as device code: the
// closure of the diagonal tile by one CTA, and the 16-wide sub-block steps it
// is built from (also used by the cluster form in phase1.cu).
#pragma once

#include "pairops.cuh"

namespace bs {

// Phase 1 computes the closure of tile (K,K) by the same blocked scheme one
// level down.  On one CTA (p1_close_tile below: 128-wide tiles, and the
// one-launch form; 64-wide tiles otherwise take the cluster form of
// phase1.cu), on the tile held in shared memory: for each
// SB-wide sub-block s of its middle atoms,
//   (a) two warps close sub-block (s,s), k serially, exchanging row and
//       column k through shared memory with a two-warp barrier per middle
//       atom; for s > 0 this runs during (c) of s-1, on the two warps (c)
//       leaves idle;
//   (b) the sub-panels in sub-block row s and sub-block column s take the
//       product with the closed sub-block (each cell computed into registers,
//       written after a barrier, so every operand is the value from before);
//   (c) every other cell takes the product of its sub-panels, paired middle
//       atoms as in phase 3.
// (b) and (c) are the update of the other phases, X[i,j] against T[i,k] and
// T[k,j] over the sub-block's middle atoms k.  Three barriers per sub-block
// instead of one per middle atom.

constexpr int SB = 16;          // sub-block width
constexpr int HALVES = SB / 8;     // (b): 8-cell units per sub-panel line

// (c) micro-tile: 8 x 4 cells on 128-wide tiles (512 threads; the shape
// gives 4 x 4 and 256 threads for a 64-wide tile).  Warp w covers tile rows
// 8w .. 8w+7 and thread tx columns 4tx .. 4tx+3, so a sub-block row is whole
// warps and a sub-block column whole quads.
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

// (a): closure of the SB x SB sub-block at (sb, sb) by two warps (AT
// threads), in registers: thread t holds row t/4, columns 4(t%4) .. +3 of the
// block.  Step k reads row k and column k from a double-buffered exchange in
// shared memory that the holders of row and column k filled after step k-1,
// so each step uses the values from before it (round-synchronous); one
// two-warp barrier per step.  The lower-bound column is raised by the closure
// rule, Lc = max(L[i,k], L[k,k] - U[i,k]).  xr, xc: [2 buffers][U, L][SB].
constexpr int AT = 64;
static_assert(SB * SB == AT * 4, "(a): four cells per thread");

__device__ __forceinline__ void p1_pair_sync() { asm volatile("bar.sync 1, 64;" ::: "memory"); }

template <class T, bool HAS_L>
__device__ __forceinline__ void p1_publish(const T (&u)[4], const T (&l)[4], int t, int k, T* xr,
                                           T* xc) {
    const int i = t >> 2, c0 = (t & 3) * 4;
    T* r = xr + (k & 1) * 2 * SB;
    T* c = xc + (k & 1) * 2 * SB;
    if (i == k) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            r[c0 + q] = u[q];
            if (HAS_L) r[SB + c0 + q] = l[q];
        }
    }
    if (c0 == (k & ~3)) {
        const int q = k & 3;
        c[i] = q == 0 ? u[0] : q == 1 ? u[1] : q == 2 ? u[2] : u[3];
        if (HAS_L) c[SB + i] = q == 0 ? l[0] : q == 1 ? l[1] : q == 2 ? l[2] : l[3];
    }
}

template <class T, bool HAS_L>
__device__ __forceinline__ void p1_block_close(T (&u)[4], T (&l)[4], int t, T* xr, T* xc) {
    using E = El<T>;
    const int i = t >> 2, c0 = (t & 3) * 4;
    p1_publish<T, HAS_L>(u, l, t, 0, xr, xc);
    p1_pair_sync();
#pragma unroll
    for (int k = 0; k < SB; ++k) {
        const T* r = xr + (k & 1) * 2 * SB;
        const T* c = xc + (k & 1) * 2 * SB;
        const T uik = c[i];
        T ukj[4], lkj[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            ukj[q] = r[c0 + q];
            lkj[q] = HAS_L ? r[SB + c0 + q] : T(0);
        }
        T lc = T(0);
        if (HAS_L) lc = E::mx(c[SB + i], E::sub(r[SB + k], uik));
#pragma unroll
        for (int q = 0; q < 4; ++q) u[q] = E::mn(u[q], E::add(uik, ukj[q]));
        if (HAS_L) {
#pragma unroll
            for (int q = 0; q < 4; ++q)
                l[q] = E::mx(l[q], E::mx(E::sub(lkj[q], uik), E::sub(lc, ukj[q])));
        }
        if (k + 1 < SB) {
            p1_publish<T, HAS_L>(u, l, t, k + 1, xr, xc);
            p1_pair_sync();
        }
    }
}

// The block (sb, sb) to or from the (a) threads' registers.  The store also
// writes the closed block k-interleaved (dU, dL) for the column sub-panel.
template <class T, bool HAS_L, int TS>
__device__ __forceinline__ void p1_block_load(const T* tU, const T* tL, int sb, int t, T (&u)[4],
                                              T (&l)[4]) {
    const int o = (sb + (t >> 2)) * TS + sb + (t & 3) * 4;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        u[q] = tU[o + q];
        l[q] = HAS_L ? tL[o + q] : T(0);
    }
}

template <class T, bool HAS_L, int TS>
__device__ __forceinline__ void p1_block_store(T* tU, T* tL, T* dU, T* dL, int sb, int t,
                                               const T (&u)[4], const T (&l)[4]) {
    const int i = t >> 2, c0 = (t & 3) * 4;
    const int o = (sb + i) * TS + sb + c0;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        tU[o + q] = u[q];
        const int d = (i >> 1) * (2 * SB) + 2 * (c0 + q) + (i & 1);
        dU[d] = u[q];
        if (HAS_L) {
            tL[o + q] = l[q];
            dL[d] = l[q];
        }
    }
}

// Step (c) of sub-block sp for the cells of block (sb, sb), in the (a)
// layout: the product of the column sub-panel T[i][sp + k] (row-major tile)
// with the row sub-panel T[sp + k][j] (its k-interleaved copy rU, rL), middle
// atoms in pairs as in phase 3.
template <class T, bool HAS_L, int FB, int TS>
__device__ __forceinline__ void p1_block_product(T (&u)[4], T (&l)[4], const T* tU, const T* tL,
                                                 const T* rU, const T* rL, int sb, int sp,
                                                 int t) {
    using LD = PairLoad<T>;
    using P = typename LD::P;
    constexpr bool NEG = std::is_same<T, int>::value;
    const int row = (sb + (t >> 2)) * TS + sp;
    const int j0 = sb + (t & 3) * 4;
#pragma unroll 2
    for (int kk = 0; kk < SB; kk += 2) {
        P a = LD::ld2(tU + row + kk);
        P al = a;
        if (HAS_L) al = LD::ld2(tL + row + kk);
        P b[4], bl[4];
        const int jb = (kk >> 1) * (2 * FB) + 2 * j0;
        LD::ld4(rU + jb, b[0], b[1]);
        LD::ld4(rU + jb + 4, b[2], b[3]);
        if (HAS_L) {
            LD::ld4(rL + jb, bl[0], bl[1]);
            LD::ld4(rL + jb + 4, bl[2], bl[3]);
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

// ---------------------------------------------------------------- the closure

// The closure of tile (K,K) over its own middle atoms, by one CTA of
// P1S<FB>::NT threads, on the tile held in shared memory (`smem_raw`:
// P1Smem<T, HAS_L, FB>::BYTES); U and L point at the molecule.  Ends with the
// closed tile stored.  Used by the phase-1 launch of 128-wide tiles
// (phase1.cu) and by the one-launch form (fused.cu).
template <class T, bool HAS_L, int FB>
__device__ __forceinline__ void p1_close_tile(T* __restrict__ U, T* __restrict__ L, int n, int ld,
                                              int K, bool vec, unsigned char* smem_raw) {
    using S = P1S<FB>;
    using E = El<T>;
    using SM = P1Smem<T, HAS_L, FB>;
    using LD = PairLoad<T>;
    using P = typename LD::P;
    constexpr int NT = S::NT, TS = SM::TS;
    constexpr int W = FB - SB;                          // sub-panel length outside the sub-block
    static_assert(2 * HALVES * W <= NT, "one (b) unit per thread");
    constexpr bool NEG = std::is_same<T, int>::value;   // int lower bound adds negated values
    T* tU = reinterpret_cast<T*>(smem_raw);
    T* tL = tU + SM::TILE;
    T* rU = tU + SM::MATS * SM::TILE;
    T* rL = rU + SM::RP;
    T* dU = rU + SM::MATS * SM::RP;
    T* dL = dU + SM::DI;

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
    // (a) of the first sub-block; each later one runs inside (c) of the
    // previous sub-block, on a warp that (c) leaves idle
    __shared__ __align__(16) T xr[2 * 2 * SB], xc[2 * 2 * SB];   // (a) exchange
    if (threadIdx.x < AT) {
        T u[4], l[4];
        p1_block_load<T, HAS_L, TS>(tU, tL, 0, threadIdx.x, u, l);
        p1_block_close<T, HAS_L>(u, l, threadIdx.x, xr, xc);
        p1_block_store<T, HAS_L, TS>(tU, tL, dU, dL, 0, threadIdx.x, u, l);
    }
    __syncthreads();
    for (int sb = 0; sb < m; sb += SB) {

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
        // those whose columns lie in sub-block column s compute but do not
        // store.  The skipping warps take block (s+1, s+1) instead: its (c)
        // step, then its closure (a), so that the next sub-block's (a)
        // overlaps this (c); the others leave that block alone.
        const int nsb = sb + SB;
        if (warp >> 1 == sb / SB) {
            if (nsb < m) {
                const int t = threadIdx.x - AT * (sb / SB);
                T u[4], l[4];
                p1_block_load<T, HAS_L, TS>(tU, tL, nsb, t, u, l);
                p1_block_product<T, HAS_L, FB, TS>(u, l, tU, tL, rU, rL, nsb, sb, t);
                p1_block_close<T, HAS_L>(u, l, t, xr, xc);
                p1_block_store<T, HAS_L, TS>(tU, tL, dU, dL, nsb, t, u, l);
            }
        } else if ((r0 / SB) != (sb / SB)) {
            const bool keep = (cq / SB) != (sb / SB) &&
                              !(nsb < m && r0 / SB == nsb / SB && cq / SB == nsb / SB);
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

}  // namespace bs
