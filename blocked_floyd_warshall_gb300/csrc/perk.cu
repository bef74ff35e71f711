// Per-round mode: one launch per middle atom k (GPU Gems 2 ch. 43,
// section 3, "Floyd-Warshall rounds"; section 5 computes each round from a copy
// of the matrix taken at its start).
//
// Round k reads only row k and column k.  Round-synchronous semantics without
// a second matrix: k_round updates every cell OUTSIDE row k and column k, so
// nothing it reads changes during the launch (the 16-byte store that covers
// column k writes that lane back unchanged).  Row k and column k then take
// round k's update, whose new values depend only on themselves, L[k,k] and U
// (all unchanged by round k: U[i,k] + U[k,k] = U[i,k] because U[k,k] = 0):
//   cell (i,k): L[i,k] <- max(L[i,k], L[k,k] - U[i,k])
//   cell (k,j): L[k,j] <- max(L[k,j], L[k,k] - U[k,j])
// Both rules give these same row/column updates.  The upper bound of row and
// column k never changes in round k, so the upper-only mode needs none.
//
// That row/column update of round k is applied by the next launch, k_round
// of round k+1, as it loads those cells (the cell's own U, still the value
// round k left, and L[k,k], which round k+1 does not change); where round k+1
// reads one of them as an operand -- cell (k+1,k) of its row, cell (k,k+1) of
// its column -- it applies the update to the value it reads and one thread
// stores it.  Only the last round's needs its own launch (k_cross).  A
// second application changes nothing (max is idempotent), so concurrent
// readers of a cell being stored see an equivalent value.
//
// HBM-bound: each cell is read and written once per round (U and L: 16 bytes
// per fp32 cell update).
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
    T* Lk = HAS_L ? L + (size_t)k * ld : nullptr;
    // the row/column update of round kp = k-1, still to apply (see above)
    const int kp = k - 1;
    const bool cross = HAS_L && kp >= 0;
    const T lpp = cross ? L[(size_t)kp * ld + kp] : T(0);

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
    if (cross) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            if (j + q != kp) continue;
            // cell (k, kp): column kp's pending update
            lkj[q] = E::mx(lkj[q], E::sub(lpp, ukj[q]));
            if (blockIdx.y == 0) Lk[kp] = lkj[q];
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
            if (cross && i == kp) {
                // cell (kp, k): row kp's pending update; stored before the
                // loads below, so the thread whose quad holds column k writes
                // the new value back with its quad
                lc = E::mx(lc, E::sub(lpp, uik));
                if (j <= k && k < j + 4) Li[k] = lc;
            }
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
            if (j + q == k) continue;   // column k: next launch
            // row kp / column kp: round kp's pending update, from the U that
            // round kp left, before this round changes it
            if (cross && (i == kp || j + q == kp)) l[q] = E::mx(l[q], E::sub(lpp, u[q]));
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

cudaError_t launch_round(bool is_int, const Mats& m, int k, bool literal, cudaStream_t s) {
    return is_int ? round_t<int>(m, k, literal, s) : round_t<float>(m, k, literal, s);
}

cudaError_t launch_cross(bool is_int, const Mats& m, int k, cudaStream_t s) {
    return is_int ? cross_t<int>(m, k, s) : cross_t<float>(m, k, s);
}

}  // namespace bs
