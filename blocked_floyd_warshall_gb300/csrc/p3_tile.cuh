// Phases 2 and 3 of the three-phase blocked Floyd-Warshall as device code:
// the update of one tile against its column and row operands, the staging of
// those operands, and the map from a launch's tile index to the tile.  Used
// by the per-phase launches (phase3.cu) and by the one-launch form
// (fused.cu).
#pragma once

#include "pairops.cuh"

namespace bs {

// Micro-tile shape: no barrier per step, so many cells per thread (few
// shared-memory loads per cell update).  128-wide tiles: 8 x 8 cells, 256
// threads, one CTA per SM.  64-wide tiles: 8 x 4 cells, 128 threads: half the
// registers of 8 x 8, so four CTAs per SM hold twice the warps (measured
// against 8 x 8 with 64 threads: n = 3000 16 % faster, n = 4096 on 64-wide
// tiles 11 %).  When a launch has too few tiles to fill the GPU, each CTA is
// latency-bound; the wide form of the 64-wide tile then spreads it over 256
// threads (4 x 4 cells each).
template <int FB, bool WIDE>
using P3S = Shape<FB, (WIDE ? 4 : 8), (WIDE || FB == FB_SMALL ? 4 : 8)>;

// ---------------------------------------------------------------- phase 3
//
// The kernel updates tile (I,J) from the column operand (I,K) and the row
// operand (K,J): in phase 3 the finished panels; in phase 2 the finished
// diagonal tile (K,K) and the panel tile itself, read before the CTA writes it
// (no other CTA touches it).  Both are streamed through shared memory in chunks of BK
// middle atoms (two stages, cp.async).  The inner loop takes the middle atoms
// two at a time: a thread holds, per row r, the pair (U[i,k], U[i,k+1]) in one
// 64-bit register (the column panel is stored [i][k], so the pair is one
// 8-byte load), and per column c the pair (U[k,j], U[k+1,j]) (the row panel is
// stored k-interleaved, [k/2][j][k%2]).  For fp32 one add.rn.f32x2 then forms
// both candidate sums of a cell and one three-input min.f32 folds them into
// the accumulator; the lower bound takes two sub.rn.f32x2 and two three-input
// max.f32.  3 instructions per cell update instead of 6.  min and max are
// exact, so the grouping of k changes no result; every sum is the same
// round-to-nearest fp32 add.  int32 uses the add-then-min/max forms
// (__viaddmin_s32 / __viaddmax_s32).

// Middle atoms staged per pipeline stage: 32 on 128-wide tiles (half the
// barriers of 16; measured 5 % faster), 16 on 64-wide tiles (keeps four CTAs
// per SM within shared memory).  The column panel's row stride BK + 4 keeps its
// rows 16-byte aligned.
template <int FB> struct P3K {
    static constexpr int BK = FB == FB_LARGE ? 32 : 16;
    static constexpr int AST = BK + 4;
};

template <class T, bool HAS_L, int FB>
struct P3Smem {
    static constexpr int BK = P3K<FB>::BK;
    static constexpr int AST = P3K<FB>::AST;
    // one stage: column panel A[i][k] (FB x AST) and row panel B[k/2][j][k%2]
    static constexpr int A_ELEMS = FB * AST;
    static constexpr int B_ELEMS = BK * FB;
    static constexpr int MATS = HAS_L ? 2 : 1;
    static constexpr int STAGE = MATS * (A_ELEMS + B_ELEMS);   // layout AU | BU | AL | BL
    static constexpr size_t BYTES = 2 * STAGE * sizeof(T);
};

// Stage k-chunk `c` of both panels into shared memory stage `stage`.
template <class T, bool HAS_L, int FB, int NT>
__device__ __forceinline__ void p3_stage(T* stage, const T* U, const T* L, size_t ld, int oi,
                                         int oj, int ok, int mi, int mj, int mk, int c,
                                         bool vec) {
    using E = El<T>;
    using SM = P3Smem<T, HAS_L, FB>;
    constexpr int BK = P3K<FB>::BK, AST = P3K<FB>::AST;
    T* AU = stage;
    T* BU = stage + SM::A_ELEMS;
    T* AL = HAS_L ? BU + SM::B_ELEMS : nullptr;
    T* BL = HAS_L ? AL + SM::A_ELEMS : nullptr;
    const int kc = c * BK;
    if (vec && mi == FB && mj == FB && kc + BK <= mk) {
        // Whole chunk inside the matrix: fixed per-thread bases, constant
        // strides, no bounds tests.  Column panel: thread t copies 16-byte
        // piece t % QP of rows t / QP + RSTEP i; row panel: column t % FB of
        // middle atoms t / FB + KSTEP i (KSTEP even keeps its pair slot).
        constexpr int QP = BK / 4, RSTEP = NT / QP, KSTEP = NT / FB;
        static_assert(NT % QP == 0 && FB % RSTEP == 0, "column-panel passes");
        static_assert(NT % FB == 0 && KSTEP % 2 == 0 && BK % KSTEP == 0, "row-panel passes");
        const int r = threadIdx.x / QP, kq = (threadIdx.x % QP) * 4;
        const T* gu = U + (size_t)(oi + r) * ld + ok + kc + kq;
        const T* gl = HAS_L ? L + (size_t)(oi + r) * ld + ok + kc + kq : nullptr;
        const size_t rstride = (size_t)RSTEP * ld;
#pragma unroll
        for (int i = 0; i < FB / RSTEP; ++i) {
            cp_async16(AU + (r + i * RSTEP) * AST + kq, gu + i * rstride);
            if (HAS_L) cp_async16(AL + (r + i * RSTEP) * AST + kq, gl + i * rstride);
        }
        const int j = threadIdx.x % FB, k0 = threadIdx.x / FB;
        const int d0 = (k0 >> 1) * (2 * FB) + j * 2 + (k0 & 1);
        const T* hu = U + (size_t)(ok + kc + k0) * ld + oj + j;
        const T* hl = HAS_L ? L + (size_t)(ok + kc + k0) * ld + oj + j : nullptr;
        const size_t kstride = (size_t)KSTEP * ld;
#pragma unroll
        for (int i = 0; i < BK / KSTEP; ++i) {
            cp_async4(BU + d0 + i * KSTEP * FB, hu + i * kstride);
            if (HAS_L) cp_async4(BL + d0 + i * KSTEP * FB, hl + i * kstride);
        }
        return;
    }
    // column panel: FB rows x BK middle atoms, [i][k]
    if (vec) {
        for (int p = threadIdx.x; p < FB * (BK / 4); p += NT) {
            const int i = p / (BK / 4);
            const int kq = (p % (BK / 4)) * 4;
            const size_t g = (size_t)(oi + i) * ld + ok + kc + kq;
            if (i < mi && kc + kq + 4 <= mk) {
                cp_async16(AU + i * AST + kq, U + g);
                if (HAS_L) cp_async16(AL + i * AST + kq, L + g);
            } else {
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const bool in = i < mi && kc + kq + q < mk;
                    AU[i * AST + kq + q] = in ? U[g + q] : E::upad();
                    if (HAS_L) AL[i * AST + kq + q] = in ? L[g + q] : E::lpad();
                }
            }
        }
    } else {
        for (int p = threadIdx.x; p < FB * BK; p += NT) {
            const int i = p / BK, k = p % BK;
            const size_t g = (size_t)(oi + i) * ld + ok + kc + k;
            if (i < mi && kc + k < mk) {
                cp_async4(AU + i * AST + k, U + g);
                if (HAS_L) cp_async4(AL + i * AST + k, L + g);
            } else {
                AU[i * AST + k] = E::upad();
                if (HAS_L) AL[i * AST + k] = E::lpad();
            }
        }
    }
    // row panel: BK middle atoms x FB columns, k-interleaved
    for (int p = threadIdx.x; p < BK * FB; p += NT) {
        const int k = p / FB, j = p % FB;
        const int d = (k >> 1) * (2 * FB) + j * 2 + (k & 1);
        const size_t g = (size_t)(ok + kc + k) * ld + oj + j;
        if (kc + k < mk && j < mj) {
            cp_async4(BU + d, U + g);
            if (HAS_L) cp_async4(BL + d, L + g);
        } else {
            BU[d] = E::upad();
            if (HAS_L) BL[d] = E::lpad();
        }
    }
}

// Which tiles a launch covers (block round K, nb tile rows):
//   P3_ALL    : every tile outside block-row K and block-column K;
//   P3_NEXT   : those in block-row K+1 or block-column K+1 (the tiles the next
//               block round's phases 1 and 2 read and write);
//   P3_REST   : the others;
//   P3_ALL_OFF: P3_ALL without tile (K+1,K+1), whose update phase 1 of round
//               K+1 takes over;
//   P3_PANELS : phase 2, the row panel (K,J) then the column panel (I,K).
// Block rounds in pairs (K, K+1) (see run_pairs; symmetric forms below):
//   P3_REST2  : tiles outside block-rows and -columns K .. K+3, rounds K and
//               K+1 in one pass;
//   P3_NEAR2  : tiles in block-rows or -columns K+2, K+3, outside K and K+1,
//               rounds K and K+1 in one pass;
//   P3_PREV2  : (launched with K = the pair's second round) tiles in block-row
//               or -column K-1 outside K .. K+2, round K;
//   P3_CORNER2: (the same) tiles (K+1,K-1), (K+2,K-1), (K-1,K+1), (K-1,K+2),
//               round K.
// With symmetric inputs only tiles with I <= J are computed (the first four
// sets: (nb-1)nb/2, nb-1, (nb-2)(nb-1)/2 and (nb-1)nb/2 - 1 tiles).  Phase 2
// computes, for each block column j != K, the panel tile on the upper side -- (K,j) for j > K,
// the column panel tile (j,K) for j < K -- and stores it also transposed, so
// that both panels are whole for phase 3.  Phase-3 tiles are stored once:
// no later step reads a tile below the diagonal but a panel, and the lower
// triangle is written as the transpose of the upper one at the end
// (p3_mirror_block).  With symmetric U and L the column panel tile (j,K) is
// the transpose of the row panel tile (K,j), to the bit (the same sums, min
// and max), so either side can be computed.

// t -> (a, b), a <= b, enumerating the upper triangle column by column.
__device__ __forceinline__ void p3_tri(int t, int& a, int& b) {
    int c = (int)((sqrtf(8.0f * (float)t + 1.0f) - 1.0f) * 0.5f);
    while (c * (c + 1) / 2 > t) --c;
    while ((c + 1) * (c + 2) / 2 <= t) ++c;
    b = c;
    a = t - c * (c + 1) / 2;
}

// The tile sets of the pair schedule (see the list above); with symmetric
// inputs the tiles on and above the diagonal of each set (CORNER2: (K-1,K+1)
// and (K-1,K+2); PREV2: block row K-1 from the diagonal on, without
// K .. K+2, and block column K-1 above the diagonal).
__host__ __device__ inline int p3_pair_w(int nb, int K) { return min(4, nb - K); }
__host__ __device__ inline int p3_pair_h(int nb, int K) { return max(0, min(2, nb - K - 2)); }
__host__ __device__ inline int p3_pair_e(int nb, int Kb) { return min(3, nb - 1 - Kb); }
// symmetric NEAR2: the near block rows' tiles from the diagonal on
__host__ __device__ inline int p3_pair_near_rows(int nb, int K) {
    const int h = p3_pair_h(nb, K), a = nb - K - 2;
    return h == 2 ? 2 * a - 1 : h == 1 ? a : 0;
}

__device__ __forceinline__ void p3_tile_pair(int part, bool sym, int t, int nb, int K, int& I,
                                             int& J) {
    if (part == P3_REST2) {
        const int w = p3_pair_w(nb, K), m = nb - w;
        int a, b;
        if (sym) {
            p3_tri(t, a, b);
        } else {
            a = t / m;
            b = t % m;
        }
        I = a + (a >= K ? w : 0);
        J = b + (b >= K ? w : 0);
    } else if (part == P3_NEAR2) {
        const int h = p3_pair_h(nb, K);
        if (sym) {
            const int a = nb - K - 2, rows = p3_pair_near_rows(nb, K);
            if (t < a) {
                I = K + 2;
                J = K + 2 + t;
            } else if (t < rows) {
                I = K + 3;
                J = K + 3 + (t - a);
            } else {
                const int u = t - rows;
                I = u % K;
                J = K + 2 + u / K;
            }
        } else if (t < h * (nb - 2)) {
            const int j = t % (nb - 2);
            I = K + 2 + t / (nb - 2);
            J = j + (j >= K ? 2 : 0);
        } else {
            const int u = t - h * (nb - 2), m = nb - 2 - h;
            const int i = u % m;
            J = K + 2 + u / m;
            I = i + (i >= K ? 2 + h : 0);
        }
    } else if (part == P3_PREV2) {
        const int Kb = K - 1, e = p3_pair_e(nb, Kb);
        if (sym) {
            const int r = nb - Kb - e;
            I = t < r ? Kb : t - r;
            J = t < r ? (t == 0 ? Kb : Kb + e + t) : Kb;
        } else if (t < nb - e) {
            I = Kb;
            J = t + (t >= Kb + 1 ? e : 0);
        } else {
            const int u = t - (nb - e);
            I = u + (u >= Kb ? 1 + e : 0);
            J = Kb;
        }
    } else {   // P3_CORNER2
        const int Kb = K - 1, h = p3_pair_h(nb, Kb);
        I = t < h && !sym ? Kb + 2 + t : Kb;
        J = t < h && !sym ? Kb : Kb + 2 + (sym ? t : t - h);
    }
}

__device__ __forceinline__ void p3_tile(int part, bool sym, int t, int nb, int K, int& I,
                                        int& J) {
    if (part == P3_PANELS) {
        if (t < nb - 1) {
            const int j = t + (t >= K);
            I = sym && j < K ? j : K;
            J = sym && j < K ? K : j;
        } else {
            const int u = t - (nb - 1);
            I = u + (u >= K);
            J = K;
        }
        return;
    }
    if (!sym) {
        if (part == P3_ALL || part == P3_ALL_OFF) {
            if (part == P3_ALL_OFF) t += t >= K * nb;   // skip (K+1,K+1): ti = tj = K
            const int ti = t / (nb - 1), tj = t % (nb - 1);
            I = ti + (ti >= K);
            J = tj + (tj >= K);
        } else if (part == P3_NEXT) {
            if (t < nb - 1) {
                I = K + 1;
                J = t + (t >= K);
            } else {
                const int u = t - (nb - 1);
                I = u + 2 * (u >= K);
                J = K + 1;
            }
        } else {
            const int ti = t / (nb - 2), tj = t % (nb - 2);
            I = ti + 2 * (ti >= K);
            J = tj + 2 * (tj >= K);
        }
        return;
    }
    int a, b;
    if (part == P3_ALL || part == P3_ALL_OFF) {
        if (part == P3_ALL_OFF) t += t >= K * (K + 1) / 2 + K;   // skip (K+1,K+1): a = b = K
        p3_tri(t, a, b);
        I = a + (a >= K);
        J = b + (b >= K);
    } else if (part == P3_NEXT) {
        if (t < nb - K - 1) {
            I = K + 1;
            J = K + 1 + t;
        } else {
            I = t - (nb - K - 1);
            J = K + 1;
        }
    } else {
        p3_tri(t, a, b);
        I = a + 2 * (a >= K);
        J = b + 2 * (b >= K);
    }
}

// Tiles a phase-3 launch covers (see p3_tile).
__host__ __device__ inline int p3_tiles(bool sym, int part, int nb, int K) {
    if (nb < 2) return 0;
    if (part == P3_REST2) {
        const int m = nb - p3_pair_w(nb, K);
        return K + 1 < nb ? (sym ? m * (m + 1) / 2 : m * m) : 0;
    }
    if (part == P3_NEAR2) {
        const int h = p3_pair_h(nb, K);
        if (K + 1 >= nb) return 0;
        return sym ? p3_pair_near_rows(nb, K) + h * K : h * (2 * nb - 4 - h);
    }
    if (part == P3_PREV2) {
        if (K < 1) return 0;
        const int e = p3_pair_e(nb, K - 1);
        return sym ? nb - e : 2 * nb - 1 - 2 * e;
    }
    if (part == P3_CORNER2) return K >= 1 ? (sym ? 1 : 2) * p3_pair_h(nb, K - 1) : 0;
    if (part == P3_PANELS) return sym ? nb - 1 : 2 * (nb - 1);
    if (sym)
        return part == P3_ALL ? (nb - 1) * nb / 2
               : part == P3_NEXT ? (K + 1 < nb ? nb - 1 : 0)
               : part == P3_ALL_OFF ? (K + 1 < nb ? (nb - 1) * nb / 2 - 1 : 0)
                                     : (K + 1 < nb ? (nb - 2) * (nb - 1) / 2 : 0);
    return part == P3_ALL ? (nb - 1) * (nb - 1)
           : part == P3_NEXT ? (K + 1 < nb ? 2 * nb - 3 : 0)
           : part == P3_ALL_OFF ? (K + 1 < nb ? (nb - 1) * (nb - 1) - 1 : 0)
                                 : (K + 1 < nb ? (nb - 2) * (nb - 2) : 0);
}

// Tile (I,J) of block round K: the product of the column operand (I,K) with
// the row operand (K,J) applied to the tile, U and L fused (see above).  `sm`:
// P3Smem<T, HAS_L, FB>::BYTES of shared memory.  Every thread of the CTA
// (P3S<FB, WIDE>::NT) calls it; it ends with the tile stored (and, with
// `mirror` off the diagonal -- the panels of symmetric inputs -- stored
// transposed too), after a block barrier that ends every read of `sm`.
template <class T, bool HAS_L, int FB, bool WIDE>
__device__ __forceinline__ void p3_update_tile(T* __restrict__ U, T* __restrict__ L, int n, int ld,
                                               int I, int J, int K, bool vec, bool mirror, T* sm,
                                               int K2 = -1) {
    using S = P3S<FB, WIDE>;
    using E = El<T>;
    using SM = P3Smem<T, HAS_L, FB>;
    using LD = PairLoad<T>;
    constexpr int BK = P3K<FB>::BK, AST = P3K<FB>::AST;
    using P = typename LD::P;
    constexpr bool NEG = std::is_same<T, int>::value;   // int lower bound adds negated values
    const int oi = I * FB, oj = J * FB, ok = K * FB;
    const int mi = min(FB, n - oi), mj = min(FB, n - oj), mk = min(FB, n - ok);

    T u[S::TM][S::TN], l[S::TM][S::TN];
    load_tile<S>(u, U + (size_t)oi * ld + oj, ld, mi, mj, vec, E::upad());
    if (HAS_L) load_tile<S>(l, L + (size_t)oi * ld + oj, ld, mi, mj, vec, E::lpad());

    // K2 >= 0: block round K2 too, in the same pass (its panels final, the
    // tile's own values after round K are never needed: min and max are
    // exact, so folding both rounds' products in changes no bit)
    // (the pair schedule runs the 8 x 8 and 8 x 4 forms, not the wide one)
    constexpr bool PAIRS = !WIDE;
    const int ok2 = PAIRS ? K2 * FB : 0, mk2 = PAIRS && K2 >= 0 ? min(FB, n - ok2) : 0;
    const int n1 = (mk + BK - 1) / BK;
    const int nchunks = n1 + (PAIRS ? (mk2 + BK - 1) / BK : 0);
    auto stage = [&](T* dst, int c) {
        if constexpr (PAIRS) {
            if (c >= n1) {
                p3_stage<T, HAS_L, FB, S::NT>(dst, U, L, ld, oi, oj, ok2, mi, mj, mk2, c - n1, vec);
                return;
            }
        }
        p3_stage<T, HAS_L, FB, S::NT>(dst, U, L, ld, oi, oj, ok, mi, mj, mk, c, vec);
    };
    stage(sm, 0);
    cp_async_commit();
    const int r0 = S::row0(), cq = S::cq();
    for (int c = 0; c < nchunks; ++c) {
        if (c + 1 < nchunks) stage(sm + ((c + 1) & 1) * SM::STAGE, c + 1);
        cp_async_commit();
        cp_async_wait<1>();
        __syncthreads();
        const T* AU = sm + (c & 1) * SM::STAGE;
        const T* BU = AU + SM::A_ELEMS;
        const T* AL = BU + SM::B_ELEMS;
        const T* BL = AL + SM::A_ELEMS;
        auto step = [&](int kk) {
            P a[S::TM], al[S::TM], b[S::TN], bl[S::TN];
#pragma unroll
            for (int r = 0; r < S::TM; ++r) {
                a[r] = LD::ld2(AU + (r0 + r) * AST + kk);
                if (HAS_L) al[r] = LD::ld2(AL + (r0 + r) * AST + kk);
            }
            const int bo = (kk >> 1) * (2 * FB);
#pragma unroll
            for (int h = 0; h < S::QUADS; ++h) {
                const int jb = bo + (h * S::QSTRIDE + cq) * 2;
                LD::ld4(BU + jb, b[h * 4 + 0], b[h * 4 + 1]);
                LD::ld4(BU + jb + 4, b[h * 4 + 2], b[h * 4 + 3]);
                if (HAS_L) {
                    LD::ld4(BL + jb, bl[h * 4 + 0], bl[h * 4 + 1]);
                    LD::ld4(BL + jb + 4, bl[h * 4 + 2], bl[h * 4 + 3]);
                }
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
        };
        // 128-wide tiles with L: the chunk's upper-bound updates first, then its
        // lower-bound updates, each pass loading only the operands it uses.
        // The upper pass needs half the registers of the fused step, so it is
        // unrolled over the whole chunk (every shared-memory address an
        // immediate), and the lower pass is unrolled four times (int32: two).
        // Measured on the GB300 against the fused step: n = 16384 fp32
        // 816.8 -> 778.5 ms, n = 4096 int32 14.09 -> 13.79 ms.  The operands
        // a and b are loaded twice per chunk; shared memory is not the limit.
        auto stepU = [&](int kk) {
            P a[S::TM], b[S::TN];
#pragma unroll
            for (int r = 0; r < S::TM; ++r) a[r] = LD::ld2(AU + (r0 + r) * AST + kk);
            const int bo = (kk >> 1) * (2 * FB);
#pragma unroll
            for (int h = 0; h < S::QUADS; ++h) {
                const int jb = bo + (h * S::QSTRIDE + cq) * 2;
                LD::ld4(BU + jb, b[h * 4 + 0], b[h * 4 + 1]);
                LD::ld4(BU + jb + 4, b[h * 4 + 2], b[h * 4 + 3]);
            }
#pragma unroll
            for (int r = 0; r < S::TM; ++r)
#pragma unroll
                for (int q = 0; q < S::TN; ++q) PairOps<T>::upper(u[r][q], a[r], b[q]);
        };
        auto stepL = [&](int kk) {
            P a[S::TM], al[S::TM], b[S::TN], bl[S::TN];
#pragma unroll
            for (int r = 0; r < S::TM; ++r) {
                a[r] = LD::ld2(AU + (r0 + r) * AST + kk);
                al[r] = LD::ld2(AL + (r0 + r) * AST + kk);
            }
            const int bo = (kk >> 1) * (2 * FB);
#pragma unroll
            for (int h = 0; h < S::QUADS; ++h) {
                const int jb = bo + (h * S::QSTRIDE + cq) * 2;
                LD::ld4(BU + jb, b[h * 4 + 0], b[h * 4 + 1]);
                LD::ld4(BU + jb + 4, b[h * 4 + 2], b[h * 4 + 3]);
                LD::ld4(BL + jb, bl[h * 4 + 0], bl[h * 4 + 1]);
                LD::ld4(BL + jb + 4, bl[h * 4 + 2], bl[h * 4 + 3]);
            }
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
        };
        if constexpr (HAS_L && FB == FB_LARGE) {
#pragma unroll
            for (int kk = 0; kk < BK; kk += 2) stepU(kk);
            if constexpr (NEG) {
#pragma unroll 2
                for (int kk = 0; kk < BK; kk += 2) stepL(kk);
            } else {
#pragma unroll 4
                for (int kk = 0; kk < BK; kk += 2) stepL(kk);
            }
        } else if constexpr (HAS_L || FB == FB_SMALL) {
            // 64-wide tiles: the fused step, unrolled twice within the 128
            // registers that keep four CTAs per SM (n = 4096: 13.40 -> 12.91
            // ms; 256 molecules of n = 512: 6.33 -> 6.23 ms)
#pragma unroll 2
            for (int kk = 0; kk < BK; kk += 2) step(kk);
        } else {
            // Upper bounds alone on 128-wide tiles: the whole chunk unrolled
            // (addresses become immediates; 128 registers, two CTAs per SM),
            // 5 % faster at n = 16384.
#pragma unroll
            for (int kk = 0; kk < BK; kk += 2) step(kk);
        }
        __syncthreads();
    }
    store_tile<S>(u, U + (size_t)oi * ld + oj, ld, mi, mj, vec);
    if (HAS_L) store_tile<S>(l, L + (size_t)oi * ld + oj, ld, mi, mj, vec);
    if (mirror && I != J) {
        // the k loop ended with a barrier: the stages are free
        static_assert((HAS_L ? 2 : 1) * S::FB * (S::FB + 4) <= 2 * SM::STAGE,
                      "the mirrored tiles fit the stages");
        store_tile_t<S, HAS_L>(u, l, U + (size_t)oj * ld + oi,
                               HAS_L ? L + (size_t)oj * ld + oi : nullptr, ld, mi, mj, vec, sm);
    }
}

// Symmetric inputs, at the end of the smoothing: the 64-wide block (a,b),
// a < b, written transposed over block (b,a), U and L.  Every thread of a CTA
// of P3S<FB_SMALL, true>::NT threads calls it; `sm`: (1 + HAS_L) x 64 x 68
// elements of shared memory, free again on return.
template <class T, bool HAS_L>
__device__ __forceinline__ void p3_mirror_block(T* __restrict__ U, T* __restrict__ L, int n, int ld,
                                                int a, int b, bool vec, T* sm) {
    using S = P3S<FB_SMALL, true>;
    using E = El<T>;
    const int oi = a * FB_SMALL, oj = b * FB_SMALL;
    const int mi = min(FB_SMALL, n - oi), mj = min(FB_SMALL, n - oj);
    T u[S::TM][S::TN], l[S::TM][S::TN];
    load_tile<S>(u, U + (size_t)oi * ld + oj, ld, mi, mj, vec, E::upad());
    if (HAS_L) load_tile<S>(l, L + (size_t)oi * ld + oj, ld, mi, mj, vec, E::lpad());
    store_tile_t<S, HAS_L>(u, HAS_L ? l : u, U + (size_t)oj * ld + oi,
                           HAS_L ? L + (size_t)oj * ld + oi : nullptr, ld, mi, mj, vec, sm);
}

}  // namespace bs
