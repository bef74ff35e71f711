// Device helpers: element traits, the per-thread 8 x 8 micro-tile, and the
// cell update of one Floyd-Warshall round.
#pragma once

#include "bs_internal.cuh"

namespace bs {

// Element traits.  Pads fill cells outside the n x n block; they never change
// a real cell: an upper pad plus anything stays >= every real upper bound, and
// a lower pad minus anything stays <= every real lower bound (>= 0).
template <class T> struct El;

template <> struct El<float> {
    using V2 = float2;
    using V4 = float4;
    static __device__ __forceinline__ float upad() { return __int_as_float(0x7f800000); }   // +inf
    static __device__ __forceinline__ float lpad() { return __int_as_float(0xff800000); }   // -inf
    static __device__ __forceinline__ float add(float a, float b) { return __fadd_rn(a, b); }
    static __device__ __forceinline__ float sub(float a, float b) { return __fsub_rn(a, b); }
    static __device__ __forceinline__ float mn(float a, float b) { return fminf(a, b); }
    static __device__ __forceinline__ float mx(float a, float b) { return fmaxf(a, b); }
};

// int32 in 1/1024 A.  Real values lie in [0, 2^30): pad + real < 2^31 and
// lower pad - real >= -2^31, so no expression below overflows.
template <> struct El<int> {
    using V2 = int2;
    using V4 = int4;
    static __device__ __forceinline__ int upad() { return (1 << 30) - 1; }
    static __device__ __forceinline__ int lpad() { return -(1 << 30); }
    static __device__ __forceinline__ int add(int a, int b) { return a + b; }
    static __device__ __forceinline__ int sub(int a, int b) { return a - b; }
    static __device__ __forceinline__ int mn(int a, int b) { return min(a, b); }
    static __device__ __forceinline__ int mx(int a, int b) { return max(a, b); }
};

// Micro-tile geometry: an FB x FB tile covered by (FB/TM) x (FB/TN) threads,
// each owning TM x TN cells: rows TM*ty .. TM*ty+TM-1 and TN/4 column quads,
// quad h covering columns h*FB/(TN/4) + 4*tx .. +3 (ty = tid / (FB/TN),
// tx = tid % (FB/TN)).  Rows 2m, 2m+1 always share a thread (TM even), and so
// do columns 2m, 2m+1 (same quad).
template <int FB_, int TM_, int TN_>
struct Shape {
    static constexpr int FB = FB_;
    static constexpr int COLS = FB_;                // columns of the block a CTA covers
    static constexpr int TM = TM_;
    static constexpr int TN = TN_;
    static constexpr int QUADS = TN / 4;
    static constexpr int TX = FB / TN;              // threads per row group
    static constexpr int NT = (FB / TM) * TX;       // threads per CTA
    static constexpr int QSTRIDE = FB / QUADS;      // column distance between quads
    static __device__ __forceinline__ int row0() { return (int)(threadIdx.x / TX) * TM; }
    static __device__ __forceinline__ int cq() { return (int)(threadIdx.x % TX) * 4; }
    static __device__ __forceinline__ int col(int c) { return (c >> 2) * QSTRIDE + cq() + (c & 3); }
};

// Load the thread's cells of the tile at `M` (tile origin; mr x mc cells
// valid).  Cells outside get `pad`.
template <class S, class T>
__device__ __forceinline__ void load_tile(T (&x)[S::TM][S::TN], const T* M, size_t ld, int mr,
                                          int mc, bool vec, T pad) {
    using V4 = typename El<T>::V4;
    const int r0 = S::row0(), cq = S::cq();
#pragma unroll
    for (int r = 0; r < S::TM; ++r) {
        const int i = r0 + r;
#pragma unroll
        for (int h = 0; h < S::QUADS; ++h) {
            const int j = h * S::QSTRIDE + cq;
            if (vec && i < mr && j + 4 <= mc) {
                const V4 v = *reinterpret_cast<const V4*>(M + (size_t)i * ld + j);
                x[r][h * 4 + 0] = v.x;
                x[r][h * 4 + 1] = v.y;
                x[r][h * 4 + 2] = v.z;
                x[r][h * 4 + 3] = v.w;
            } else {
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    x[r][h * 4 + q] = (i < mr && j + q < mc) ? M[(size_t)i * ld + j + q] : pad;
            }
        }
    }
}

// Store the thread's cells that lie inside the mr x mc block.
template <class S, class T>
__device__ __forceinline__ void store_tile(const T (&x)[S::TM][S::TN], T* M, size_t ld, int mr,
                                           int mc, bool vec) {
    using V4 = typename El<T>::V4;
    const int r0 = S::row0(), cq = S::cq();
#pragma unroll
    for (int r = 0; r < S::TM; ++r) {
        const int i = r0 + r;
        if (i >= mr) continue;
#pragma unroll
        for (int h = 0; h < S::QUADS; ++h) {
            const int j = h * S::QSTRIDE + cq;
            if (vec && j + 4 <= mc) {
                V4 v;
                v.x = x[r][h * 4 + 0];
                v.y = x[r][h * 4 + 1];
                v.z = x[r][h * 4 + 2];
                v.w = x[r][h * 4 + 3];
                *reinterpret_cast<V4*>(M + (size_t)i * ld + j) = v;
            } else {
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    if (j + q < mc) M[(size_t)i * ld + j + q] = x[r][h * 4 + q];
            }
        }
    }
}

// Store the transpose of the thread's cells of U (and of L if HAS_L): cell
// (i, j) of an mr x mc tile goes to MU[j*ld + i] (and ML[j*ld + i]), MU and
// ML being the origins of the mirrored tiles.  The cells pass through shared
// memory (`buf`: (1 + HAS_L) x S::FB x (S::FB + 4) elements, free when called;
// every thread of the CTA calls it): each thread writes its cells
// transposed, 4 rows of a column per 16-byte store, and then each warp copies
// whole rows of the mirrored tiles out, so that the global stores are
// coalesced (written from registers directly, every 16-byte store of a warp
// went to a different row).  Both matrices are staged before the one
// barrier, so no cell stays in a register across it.  Ends with a barrier,
// so `buf` is free again.
template <class S, bool HAS_L, class T>
__device__ __forceinline__ void store_tile_t(const T (&u)[S::TM][S::TN], const T (&l)[S::TM][S::TN],
                                             T* MU, T* ML, size_t ld, int mr, int mc, bool vec,
                                             T* buf) {
    using V4 = typename El<T>::V4;
    constexpr int FB = S::FB, TS = FB + 4;   // TS: 16-byte rows
    constexpr int MAT = FB * TS;
    static_assert(S::COLS == FB && S::TM % 4 == 0, "square tiles, whole 16-byte columns");
    const int r0 = S::row0();
#pragma unroll
    for (int c = 0; c < S::TN; ++c) {
        T* col = buf + S::col(c) * TS + r0;
#pragma unroll
        for (int r = 0; r < S::TM; r += 4) {
            *reinterpret_cast<V4*>(col + r) = V4{u[r][c], u[r + 1][c], u[r + 2][c], u[r + 3][c]};
            if (HAS_L)
                *reinterpret_cast<V4*>(col + MAT + r) =
                    V4{l[r][c], l[r + 1][c], l[r + 2][c], l[r + 3][c]};
        }
    }
    __syncthreads();
    // the mirrored tiles: mc rows (the tile's columns) of mr cells each
    for (int p = threadIdx.x; p < (HAS_L ? 2 : 1) * FB * (FB / 4); p += S::NT) {
        const int m = p / (FB * (FB / 4)), pp = p % (FB * (FB / 4));
        const int j = pp / (FB / 4), i = (pp % (FB / 4)) * 4;
        if (j >= mc) continue;
        const T* src = buf + m * MAT + j * TS + i;
        T* dst = (m ? ML : MU) + (size_t)j * ld + i;
        if (vec && i + 4 <= mr) {
            *reinterpret_cast<V4*>(dst) = *reinterpret_cast<const V4*>(src);
        } else {
#pragma unroll
            for (int q = 0; q < 4; ++q)
                if (i + q < mr) dst[q] = src[q];
        }
    }
    __syncthreads();
}

// One middle atom k applied to the thread's cells.  a/al: U[i,k] and the
// lower-bound column value for the thread's rows; b/bl: U[k,j] and L[k,j] for
// its columns.  Upper bound first, then the lower bound from the same
// (round-invariant) upper values:
//   U[i,j] = min(U[i,j], U[i,k] + U[k,j])
//   L[i,j] = max(L[i,j], L[k,j] - U[i,k], Lcol[i] - U[k,j])
template <class S, class T, bool HAS_L>
__device__ __forceinline__ void fw_update(T (&u)[S::TM][S::TN], T (&l)[S::TM][S::TN],
                                          const T (&a)[S::TM], const T (&al)[S::TM],
                                          const T (&b)[S::TN], const T (&bl)[S::TN]) {
#pragma unroll
    for (int r = 0; r < S::TM; ++r)
#pragma unroll
        for (int c = 0; c < S::TN; ++c) u[r][c] = El<T>::mn(u[r][c], El<T>::add(a[r], b[c]));
    if (HAS_L) {
#pragma unroll
        for (int r = 0; r < S::TM; ++r)
#pragma unroll
            for (int c = 0; c < S::TN; ++c)
                l[r][c] = El<T>::mx(l[r][c], El<T>::mx(El<T>::sub(bl[c], a[r]),
                                                       El<T>::sub(al[r], b[c])));
    }
}

// Row k of the tile (U and L) into shared vectors, by the threads that own it.
template <class S, class T, bool HAS_L>
__device__ __forceinline__ void publish_row(const T (&u)[S::TM][S::TN], const T (&l)[S::TM][S::TN],
                                            int k, T* dU, T* dL) {
    const int r0 = S::row0();
#pragma unroll
    for (int r = 0; r < S::TM; ++r) {
        if (r0 + r == k) {
#pragma unroll
            for (int c = 0; c < S::TN; ++c) {
                dU[S::col(c)] = u[r][c];
                if (HAS_L) dL[S::col(c)] = l[r][c];
            }
        }
    }
}

// Column k of the tile (U and L) into shared vectors, by the threads that own it.
template <class S, class T, bool HAS_L>
__device__ __forceinline__ void publish_col(const T (&u)[S::TM][S::TN], const T (&l)[S::TM][S::TN],
                                            int k, T* dU, T* dL) {
    const int r0 = S::row0();
#pragma unroll
    for (int c = 0; c < S::TN; ++c) {
        if (S::col(c) == k) {
#pragma unroll
            for (int r = 0; r < S::TM; ++r) {
                dU[r0 + r] = u[r][c];
                if (HAS_L) dL[r0 + r] = l[r][c];
            }
        }
    }
}

}  // namespace bs
