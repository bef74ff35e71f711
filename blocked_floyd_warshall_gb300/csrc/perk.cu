// Per-round mode (GPU Gems 2 ch. 43, section 3, "Floyd-Warshall rounds";
// section 5 computes each round from a copy of the matrix taken at its
// start).  Two forms:
//   BS_PERK              one round per pass: k_round, then k_cross, for every
//                        round k -- the plain round-synchronous reference;
//   BS_PERK | PAIRED     two rounds per pass (k_round2 + k_cross2 below), with
//                        n odd the last round in the plain form.
//
// Round k reads only row k and column k.  Round-synchronous semantics without
// a second matrix: k_round updates every cell OUTSIDE row k and column k, so
// nothing it reads changes during the launch (the 16-byte store that covers
// column k writes that lane back unchanged).  k_cross then gives row k and
// column k round k's update, whose new values depend only on themselves,
// L[k,k] and U (all unchanged by round k: U[i,k] + U[k,k] = U[i,k] because
// U[k,k] = 0 and U >= 0):
//   cell (i,k): L[i,k] <- max(L[i,k], L[k,k] - U[i,k])
//   cell (k,j): L[k,j] <- max(L[k,j], L[k,k] - U[k,j])
// Both rules give these same row/column updates.  The upper bound of row and
// column k never changes in round k, so the upper-only mode needs no k_cross.
//
// HBM-bound: each cell is read and written once per pass (U and L: 16 bytes
// per fp32 cell update for k_round, 8 for k_round2).
#include "bs_tile.cuh"

namespace bs {

template <class T, bool HAS_L, bool LITERAL>
__global__ void __launch_bounds__(256)
k_round(T* __restrict__ U, T* __restrict__ L, int n, int ld, long long bstride, int k,
        bool vec) {
    using E = El<T>;
    using V4 = typename E::V4;
    const size_t off = (size_t)blockIdx.z * (size_t)bstride;
    U += off;
    if (HAS_L) L += off;
    const int jq = blockIdx.x * blockDim.x + threadIdx.x;
    const int j = jq * 4;
    if (j >= n) return;
    const T* Uk = U + (size_t)k * ld;
    const T* Lk = HAS_L ? L + (size_t)k * ld : nullptr;

    // row k: the same four values serve every row i
    T ukj[4], lkj[4];
    const bool full = vec && j + 4 <= n;
    if (full) {
        const V4 v = *reinterpret_cast<const V4*>(Uk + j);
        ukj[0] = v.x; ukj[1] = v.y; ukj[2] = v.z; ukj[3] = v.w;
        if (HAS_L) {
            const V4 w = *reinterpret_cast<const V4*>(Lk + j);
            lkj[0] = w.x; lkj[1] = w.y; lkj[2] = w.z; lkj[3] = w.w;
        }
    } else {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            ukj[q] = j + q < n ? Uk[j + q] : E::upad();
            if (HAS_L) lkj[q] = j + q < n ? Lk[j + q] : E::lpad();
        }
    }
    const T lkk = HAS_L ? Lk[k] : T(0);

    for (int i = blockIdx.y; i < n; i += gridDim.y) {
        if (i == k) continue;
        T* Ui = U + (size_t)i * ld;
        T* Li = HAS_L ? L + (size_t)i * ld : nullptr;
        const T uik = Ui[k];
        T lc = T(0);
        if (HAS_L) {
            lc = Li[k];
            if (!LITERAL) lc = E::mx(lc, E::sub(lkk, uik));
        }
        T u[4], l[4];
        if (full) {
            const V4 v = *reinterpret_cast<const V4*>(Ui + j);
            u[0] = v.x; u[1] = v.y; u[2] = v.z; u[3] = v.w;
            if (HAS_L) {
                const V4 w = *reinterpret_cast<const V4*>(Li + j);
                l[0] = w.x; l[1] = w.y; l[2] = w.z; l[3] = w.w;
            }
        } else {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                u[q] = j + q < n ? Ui[j + q] : E::upad();
                if (HAS_L) l[q] = j + q < n ? Li[j + q] : E::lpad();
            }
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            if (j + q == k) continue;   // column k: k_cross
            u[q] = E::mn(u[q], E::add(uik, ukj[q]));
            if (HAS_L) l[q] = E::mx(l[q], E::mx(E::sub(lkj[q], uik), E::sub(lc, ukj[q])));
        }
        if (full) {
            // the column-k lane, if any, writes back the value it read
            *reinterpret_cast<V4*>(Ui + j) = V4{u[0], u[1], u[2], u[3]};
            if (HAS_L) *reinterpret_cast<V4*>(Li + j) = V4{l[0], l[1], l[2], l[3]};
        } else {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                if (j + q >= n || j + q == k) continue;
                Ui[j + q] = u[q];
                if (HAS_L) Li[j + q] = l[q];
            }
        }
    }
}

template <class T>
__global__ void __launch_bounds__(256)
k_cross(const T* __restrict__ U, T* __restrict__ L, int n, int ld, long long bstride, int k) {
    using E = El<T>;
    const size_t off = (size_t)blockIdx.z * (size_t)bstride;
    U += off;
    L += off;
    const int t = blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= 2 * n) return;
    const T lkk = L[(size_t)k * ld + k];
    size_t p;
    if (t < n) {
        if (t == k) return;
        p = (size_t)t * ld + k;            // column k
    } else {
        if (t - n == k) return;
        p = (size_t)k * ld + (t - n);      // row k
    }
    L[p] = E::mx(L[p], E::sub(lkk, U[p]));
}

// ---------------------------------------------------------------- two rounds per pass
//
// Rounds k and k+1 in one pass over the matrix: each cell is read and written
// once for both rounds (8 bytes per fp32 cell update instead of 16).  Round
// k+1's operands -- row k+1 and column k+1 after round k, and cell
// (k+1,k+1) -- are the expressions round k evaluates for those cells, on the
// same operands, so every thread forms the ones it needs itself, bit for bit
// the values round k would store.  As above, the pass (k_round2) leaves rows
// and columns k and k+1 alone, so nothing it reads changes; a second launch
// (k_cross2) then takes those 4n cells through both rounds, one thread per
// line m: cells (m,k), (m,k+1), (k,m), (k+1,m).  Besides its own line a
// thread needs only the four corner cells (k..k+1, k..k+1) as they were
// before; k_cross2 runs as one cluster per molecule, every thread reads the
// corners first, and a cluster barrier separates those reads from the two
// threads that rewrite the corners.

// One round on a cell: operands U[i,k], L[i,k], U[k,j], L[k,j], L[k,k] (the
// expressions of k_round above).
template <class T, bool HAS_L, bool LITERAL>
__device__ __forceinline__ void one_round(T& u, T& l, T uik, T lik, T ukj, T lkj, T lkk) {
    using E = El<T>;
    u = E::mn(u, E::add(uik, ukj));
    if (HAS_L) {
        const T lc = LITERAL ? lik : E::mx(lik, E::sub(lkk, uik));
        l = E::mx(l, E::mx(E::sub(lkj, uik), E::sub(lc, ukj)));
    }
}

// The corner cells before the pass: c[0..3] = U at (k,k), (k,k+1), (k+1,k),
// (k+1,k+1); c[4..7] = L at the same cells.
template <class T, bool HAS_L, bool LITERAL>
struct Corners {
    T v[8];
    // cell (k+1,k+1)'s lower bound after round k: round k+1's L[k,k]
    __device__ __forceinline__ T lk1k1() const {
        T u = v[3], l = v[7];
        one_round<T, HAS_L, LITERAL>(u, l, v[2], v[6], v[1], v[5], v[4]);
        return l;
    }
};

// Both rounds on cell (i,j) from values before the pass: the cell (u, l);
// row i at columns k and k+1 (ui0, li0, ui1, li1); column j at rows k and
// k+1 (u0j, l0j, u1j, l1j); the corners; l11 = cs.lk1k1().
template <class T, bool HAS_L, bool LITERAL>
__device__ __forceinline__ void two_rounds(T& u, T& l, T ui0, T li0, T ui1, T li1, T u0j, T l0j,
                                           T u1j, T l1j, const Corners<T, HAS_L, LITERAL>& cs,
                                           T l11) {
    one_round<T, HAS_L, LITERAL>(u, l, ui0, li0, u0j, l0j, cs.v[4]);
    one_round<T, HAS_L, LITERAL>(ui1, li1, ui0, li0, cs.v[1], cs.v[5], cs.v[4]);   // (i,k+1)
    one_round<T, HAS_L, LITERAL>(u1j, l1j, cs.v[2], cs.v[6], u0j, l0j, cs.v[4]);   // (k+1,j)
    one_round<T, HAS_L, LITERAL>(u, l, ui1, li1, u1j, l1j, l11);
}

template <class T, bool HAS_L, bool LITERAL>
__global__ void __launch_bounds__(256)
k_round2(T* __restrict__ U, T* __restrict__ L, int n, int ld, long long bstride, int k,
         bool vec) {
    using E = El<T>;
    using V4 = typename E::V4;
    const size_t off = (size_t)blockIdx.z * (size_t)bstride;
    U += off;
    if (HAS_L) L += off;
    const int jq = blockIdx.x * blockDim.x + threadIdx.x;
    const int j = jq * 4;
    if (j >= n) return;
    const int k1 = k + 1;
    Corners<T, HAS_L, LITERAL> cs;
    {
        const size_t p[4] = {(size_t)k * ld + k, (size_t)k * ld + k1, (size_t)k1 * ld + k,
                             (size_t)k1 * ld + k1};
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            cs.v[c] = U[p[c]];
            cs.v[4 + c] = HAS_L ? L[p[c]] : T(0);
        }
    }
    const T l11 = cs.lk1k1();

    // rows k and k+1 at the thread's four columns
    T u0j[4], l0j[4], u1j[4], l1j[4];
    const bool full = vec && j + 4 <= n;
    const T* U0 = U + (size_t)k * ld;
    const T* U1 = U + (size_t)k1 * ld;
    const T* L0 = HAS_L ? L + (size_t)k * ld : nullptr;
    const T* L1 = HAS_L ? L + (size_t)k1 * ld : nullptr;
    if (full) {
        const V4 a = *reinterpret_cast<const V4*>(U0 + j);
        const V4 b = *reinterpret_cast<const V4*>(U1 + j);
        u0j[0] = a.x; u0j[1] = a.y; u0j[2] = a.z; u0j[3] = a.w;
        u1j[0] = b.x; u1j[1] = b.y; u1j[2] = b.z; u1j[3] = b.w;
        if (HAS_L) {
            const V4 c = *reinterpret_cast<const V4*>(L0 + j);
            const V4 d = *reinterpret_cast<const V4*>(L1 + j);
            l0j[0] = c.x; l0j[1] = c.y; l0j[2] = c.z; l0j[3] = c.w;
            l1j[0] = d.x; l1j[1] = d.y; l1j[2] = d.z; l1j[3] = d.w;
        } else {
#pragma unroll
            for (int q = 0; q < 4; ++q) l0j[q] = l1j[q] = T(0);
        }
    } else {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const bool in = j + q < n;
            u0j[q] = in ? U0[j + q] : E::upad();
            u1j[q] = in ? U1[j + q] : E::upad();
            l0j[q] = HAS_L ? (in ? L0[j + q] : E::lpad()) : T(0);
            l1j[q] = HAS_L ? (in ? L1[j + q] : E::lpad()) : T(0);
        }
    }

    for (int i = blockIdx.y; i < n; i += gridDim.y) {
        if (i == k || i == k1) continue;
        T* Ui = U + (size_t)i * ld;
        T* Li = HAS_L ? L + (size_t)i * ld : nullptr;
        const T ui0 = Ui[k], ui1 = Ui[k1];
        const T li0 = HAS_L ? Li[k] : T(0), li1 = HAS_L ? Li[k1] : T(0);
        T u[4], l[4];
        if (full) {
            const V4 v = *reinterpret_cast<const V4*>(Ui + j);
            u[0] = v.x; u[1] = v.y; u[2] = v.z; u[3] = v.w;
            if (HAS_L) {
                const V4 w = *reinterpret_cast<const V4*>(Li + j);
                l[0] = w.x; l[1] = w.y; l[2] = w.z; l[3] = w.w;
            }
        } else {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                u[q] = j + q < n ? Ui[j + q] : E::upad();
                l[q] = HAS_L ? (j + q < n ? Li[j + q] : E::lpad()) : T(0);
            }
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            if (j + q == k || j + q == k1) continue;   // columns k, k+1: k_cross2
            two_rounds<T, HAS_L, LITERAL>(u[q], l[q], ui0, li0, ui1, li1, u0j[q], l0j[q], u1j[q],
                                          l1j[q], cs, l11);
        }
        if (full) {
            // lanes in columns k, k+1 write back the values they read
            *reinterpret_cast<V4*>(Ui + j) = V4{u[0], u[1], u[2], u[3]};
            if (HAS_L) *reinterpret_cast<V4*>(Li + j) = V4{l[0], l[1], l[2], l[3]};
        } else {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                if (j + q >= n || j + q == k || j + q == k1) continue;
                Ui[j + q] = u[q];
                if (HAS_L) Li[j + q] = l[q];
            }
        }
    }
}

// Rows and columns k, k+1 through both rounds: line m's thread takes cells
// (m,k) and (m,k+1), and for m outside {k, k+1} also (k,m) and (k+1,m).  One
// cluster of X2C CTAs per molecule; each thread first reads the corners, and
// only after the cluster barrier do the lines run (lines k and k+1 rewrite
// the corners).  The barrier is the only wait and every thread passes it.
constexpr int X2C = 8, X2T = 512;

template <class T, bool HAS_L, bool LITERAL>
__global__ void __cluster_dims__(X2C, 1, 1) __launch_bounds__(X2T)
k_cross2(T* __restrict__ U, T* __restrict__ L, int n, int ld, long long bstride, int k) {
    const size_t off = (size_t)blockIdx.z * (size_t)bstride;
    U += off;
    if (HAS_L) L += off;
    const int k1 = k + 1;
    Corners<T, HAS_L, LITERAL> cs;
    {
        const size_t p[4] = {(size_t)k * ld + k, (size_t)k * ld + k1, (size_t)k1 * ld + k,
                             (size_t)k1 * ld + k1};
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            cs.v[c] = U[p[c]];
            cs.v[4 + c] = HAS_L ? L[p[c]] : T(0);
        }
    }
    const T l11 = cs.lk1k1();
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");

    for (int mm = blockIdx.x * X2T + threadIdx.x; mm < n; mm += X2C * X2T) {
        const size_t pm0 = (size_t)mm * ld + k, pm1 = (size_t)mm * ld + k1;   // (m,k), (m,k+1)
        const T um0 = U[pm0], um1 = U[pm1];
        const T lm0 = HAS_L ? L[pm0] : T(0), lm1 = HAS_L ? L[pm1] : T(0);
        const bool rows = mm != k && mm != k1;
        const size_t p0m = (size_t)k * ld + mm, p1m = (size_t)k1 * ld + mm;   // (k,m), (k+1,m)
        const T u0m = rows ? U[p0m] : T(0), u1m = rows ? U[p1m] : T(0);
        const T l0m = HAS_L && rows ? L[p0m] : T(0), l1m = HAS_L && rows ? L[p1m] : T(0);

        // column cells: row m at columns k, k+1; column k (or k+1) at rows k, k+1
        T u = um0, l = lm0;
        two_rounds<T, HAS_L, LITERAL>(u, l, um0, lm0, um1, lm1, cs.v[0], cs.v[4], cs.v[2],
                                      cs.v[6], cs, l11);
        T v = um1, w = lm1;
        two_rounds<T, HAS_L, LITERAL>(v, w, um0, lm0, um1, lm1, cs.v[1], cs.v[5], cs.v[3],
                                      cs.v[7], cs, l11);
        U[pm0] = u;
        U[pm1] = v;
        if (HAS_L) {
            L[pm0] = l;
            L[pm1] = w;
        }
        if (!rows) continue;
        // row cells: row k (or k+1) at columns k, k+1 (corners); column m at rows k, k+1
        T a = u0m, b = l0m;
        two_rounds<T, HAS_L, LITERAL>(a, b, cs.v[0], cs.v[4], cs.v[1], cs.v[5], u0m, l0m, u1m,
                                      l1m, cs, l11);
        T c = u1m, d = l1m;
        two_rounds<T, HAS_L, LITERAL>(c, d, cs.v[2], cs.v[6], cs.v[3], cs.v[7], u0m, l0m, u1m,
                                      l1m, cs, l11);
        U[p0m] = a;
        U[p1m] = c;
        if (HAS_L) {
            L[p0m] = b;
            L[p1m] = d;
        }
    }
}

template <class T>
static cudaError_t round_t(const Mats& m, int k, bool literal, cudaStream_t s) {
    const int nq = (m.n + 3) / 4;
    for (int b0 = 0; b0 < m.batch; b0 += 65535) {
        const int nbz = m.batch - b0 < 65535 ? m.batch - b0 : 65535;
        dim3 grid((nq + 255) / 256, m.n < 65535 ? m.n : 65535, nbz);
        T* U = static_cast<T*>(m.U) + (size_t)b0 * m.bstride;
        T* L = m.L ? static_cast<T*>(m.L) + (size_t)b0 * m.bstride : nullptr;
        before_launch(s, PH_ROUND);
        if (!m.L)
            k_round<T, false, false><<<grid, 256, 0, s>>>(U, L, m.n, m.ld, m.bstride, k, m.vec);
        else if (literal)
            k_round<T, true, true><<<grid, 256, 0, s>>>(U, L, m.n, m.ld, m.bstride, k, m.vec);
        else
            k_round<T, true, false><<<grid, 256, 0, s>>>(U, L, m.n, m.ld, m.bstride, k, m.vec);
        after_launch(s, PH_ROUND);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

template <class T>
static cudaError_t cross_t(const Mats& m, int k, cudaStream_t s) {
    for (int b0 = 0; b0 < m.batch; b0 += 65535) {
        const int nbz = m.batch - b0 < 65535 ? m.batch - b0 : 65535;
        dim3 grid((2 * m.n + 255) / 256, 1, nbz);
        before_launch(s, PH_ROUND);
        k_cross<T><<<grid, 256, 0, s>>>(static_cast<const T*>(m.U) + (size_t)b0 * m.bstride,
                                        static_cast<T*>(m.L) + (size_t)b0 * m.bstride, m.n,
                                        m.ld, m.bstride, k);
        after_launch(s, PH_ROUND);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

template <class T, bool HAS_L, bool LITERAL>
static cudaError_t round2_tl(const Mats& m, int k, cudaStream_t s) {
    const int nq = (m.n + 3) / 4;
    for (int b0 = 0; b0 < m.batch; b0 += 65535) {
        const int nbz = m.batch - b0 < 65535 ? m.batch - b0 : 65535;
        T* U = static_cast<T*>(m.U) + (size_t)b0 * m.bstride;
        T* L = HAS_L ? static_cast<T*>(m.L) + (size_t)b0 * m.bstride : nullptr;
        before_launch(s, PH_ROUND);
        // eight rows per thread: the corners and the rows-k, k+1 operands are
        // loaded once for them
        const int rows = (m.n + 7) / 8;
        k_round2<T, HAS_L, LITERAL>
            <<<dim3((nq + 255) / 256, rows < 65535 ? rows : 65535, nbz), 256, 0, s>>>(
                U, L, m.n, m.ld, m.bstride, k, m.vec);
        after_launch(s, PH_ROUND);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        before_launch(s, PH_ROUND);
        k_cross2<T, HAS_L, LITERAL><<<dim3(X2C, 1, nbz), X2T, 0, s>>>(U, L, m.n, m.ld,
                                                                     m.bstride, k);
        after_launch(s, PH_ROUND);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

template <class T>
static cudaError_t round2_t(const Mats& m, int k, bool literal, cudaStream_t s) {
    if (!m.L) return round2_tl<T, false, false>(m, k, s);
    return literal ? round2_tl<T, true, true>(m, k, s) : round2_tl<T, true, false>(m, k, s);
}

cudaError_t launch_round2(bool is_int, const Mats& m, int k, bool literal, cudaStream_t s) {
    return is_int ? round2_t<int>(m, k, literal, s) : round2_t<float>(m, k, literal, s);
}

cudaError_t launch_round(bool is_int, const Mats& m, int k, bool literal, cudaStream_t s) {
    return is_int ? round_t<int>(m, k, literal, s) : round_t<float>(m, k, literal, s);
}

cudaError_t launch_cross(bool is_int, const Mats& m, int k, cudaStream_t s) {
    return is_int ? cross_t<int>(m, k, s) : cross_t<float>(m, k, s);
}

}  // namespace bs
