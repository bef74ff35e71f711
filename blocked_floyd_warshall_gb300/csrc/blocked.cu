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
// its cells in registers, row k / column k are published to a shared vector
// double-buffered by k parity, one barrier per step.
#include <type_traits>

#include "bs_tile.cuh"

namespace bs {

namespace {

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
    const unsigned s = (unsigned)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;\n" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

}  // namespace

// Micro-tile shapes.  Phases 1 and 2 advance one (or two) middle atoms per
// barrier, so they want many threads with few cells each: 4 x 4 cells on 64-wide
// tiles (256 threads), 8 x 4 on 128-wide tiles (512 threads).  Phase 3 has no
// barrier per step and wants many cells per thread: 8 x 8 (64 or 256 threads).
template <int FB> using P12 = Shape<FB, (FB == FB_SMALL ? 4 : 8), 4>;
template <int FB> using P3S = Shape<FB, 8, 8>;

// ---------------------------------------------------------------- paired middle atoms

// Cell updates for a pair of middle atoms (k, k+1).
//   a, al : (U[i,k], U[i,k+1]), (L[i,k], L[i,k+1])   -- row i of the thread
//   b, bl : (U[k,j], U[k+1,j]), (L[k,j], L[k+1,j])   -- column j of the thread
template <class T> struct PairOps;

template <> struct PairOps<float> {
    using P = unsigned long long;   // two fp32 lanes: low = k, high = k+1
    static __device__ __forceinline__ void upper(float& u, P a, P b) {
        asm("{\n\t.reg .b64 s;\n\t.reg .f32 s0, s1;\n\t"
            "add.rn.f32x2 s, %1, %2;\n\t"
            "mov.b64 {s0, s1}, s;\n\t"
            "min.f32 %0, %0, s0, s1;\n\t}"
            : "+f"(u) : "l"(a), "l"(b));
    }
    // L = max(L, L[k,j] - U[i,k], L[i,k] - U[k,j]) over both k
    static __device__ __forceinline__ void lower(float& l, P a, P al, P b, P bl) {
        asm("{\n\t.reg .b64 d1, d2;\n\t.reg .f32 x0, x1, y0, y1;\n\t"
            "sub.rn.f32x2 d1, %1, %3;\n\t"
            "sub.rn.f32x2 d2, %2, %4;\n\t"
            "mov.b64 {x0, x1}, d1;\n\t"
            "mov.b64 {y0, y1}, d2;\n\t"
            "max.f32 %0, %0, x0, x1;\n\t"
            "max.f32 %0, %0, y0, y1;\n\t}"
            : "+f"(l) : "l"(bl), "l"(al), "l"(a), "l"(b));
    }
};

template <> struct PairOps<int> {
    using P = int2;
    static __device__ __forceinline__ void upper(int& u, P a, P b) {
        u = __viaddmin_s32(a.x, b.x, u);
        u = __viaddmin_s32(a.y, b.y, u);
    }
    // na, nb: negated a, b
    static __device__ __forceinline__ void lower(int& l, P na, P al, P nb, P bl) {
        l = __viaddmax_s32(bl.x, na.x, l);
        l = __viaddmax_s32(bl.y, na.y, l);
        l = __viaddmax_s32(al.x, nb.x, l);
        l = __viaddmax_s32(al.y, nb.y, l);
    }
};

template <class T> struct PairLoad;
template <> struct PairLoad<float> {
    using P = unsigned long long;
    static __device__ __forceinline__ P ld2(const float* p) {
        return *reinterpret_cast<const unsigned long long*>(p);
    }
    static __device__ __forceinline__ void ld4(const float* p, P& x, P& y) {
        const ulonglong2 v = *reinterpret_cast<const ulonglong2*>(p);
        x = v.x;
        y = v.y;
    }
    static __device__ __forceinline__ P neg(P x) { return x; }
};
template <> struct PairLoad<int> {
    using P = int2;
    static __device__ __forceinline__ P ld2(const int* p) { return *reinterpret_cast<const int2*>(p); }
    static __device__ __forceinline__ void ld4(const int* p, P& x, P& y) {
        const int4 v = *reinterpret_cast<const int4*>(p);
        x = make_int2(v.x, v.y);
        y = make_int2(v.z, v.w);
    }
    static __device__ __forceinline__ P neg(P x) { return make_int2(-x.x, -x.y); }
};

// ---------------------------------------------------------------- phase 1

template <class T, bool HAS_L, int FB>
__global__ void __launch_bounds__(P12<FB>::NT)
k_phase1(T* __restrict__ U, T* __restrict__ L, int n, int ld, long long bstride, int K, bool vec) {
    using S = P12<FB>;
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
__device__ __forceinline__ void p2_publish_rows(const T (&u)[P12<FB>::TM][P12<FB>::TN],
                                                const T (&l)[P12<FB>::TM][P12<FB>::TN], int k,
                                                const T* dU, const T* dL, T* sU, T* sL) {
    using S = P12<FB>;
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
__device__ __forceinline__ void p2_publish_cols(const T (&u)[P12<FB>::TM][P12<FB>::TN],
                                                const T (&l)[P12<FB>::TM][P12<FB>::TN], int k,
                                                const T* dU, const T* dL, T* sU, T* sL) {
    using S = P12<FB>;
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
    using S = P12<FB>;
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
    using S = P12<FB>;
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
__global__ void __launch_bounds__(P12<FB>::NT)
k_phase2(T* __restrict__ U, T* __restrict__ L, int n, int ld, long long bstride, int K, bool vec,
         bool sym) {
    using S = P12<FB>;
    using E = El<T>;
    constexpr int NT = P12<FB>::NT;
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

// ---------------------------------------------------------------- phase 3
//
// Phase 3 updates tile (I,J) from the finished column panel (I,K) and row
// panel (K,J).  Both are streamed through shared memory in chunks of BK
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

constexpr int BK = 16;        // middle atoms staged per pipeline stage
constexpr int AST = BK + 4;   // column-panel row stride (elements); rows stay 16-byte aligned

template <class T, bool HAS_L, int FB>
struct P3Smem {
    // one stage: column panel A[i][k] (FB x AST) and row panel B[k/2][j][k%2]
    static constexpr int A_ELEMS = FB * AST;
    static constexpr int B_ELEMS = BK * FB;
    static constexpr int MATS = HAS_L ? 2 : 1;
    static constexpr int STAGE = MATS * (A_ELEMS + B_ELEMS);   // layout AU | BU | AL | BL
    static constexpr size_t BYTES = 2 * STAGE * sizeof(T);
};

__device__ __forceinline__ void cp_async4(void* smem, const void* gmem) {
    const unsigned s = (unsigned)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(s), "l"(gmem) : "memory");
}

// Stage k-chunk `c` of both panels into shared memory stage `stage`.
template <class T, bool HAS_L, int FB>
__device__ __forceinline__ void p3_stage(T* stage, const T* U, const T* L, size_t ld, int oi,
                                         int oj, int ok, int mi, int mj, int mk, int c,
                                         bool vec) {
    using S = P3S<FB>;
    using E = El<T>;
    using SM = P3Smem<T, HAS_L, FB>;
    constexpr int NT = P3S<FB>::NT;
    T* AU = stage;
    T* BU = stage + SM::A_ELEMS;
    T* AL = HAS_L ? BU + SM::B_ELEMS : nullptr;
    T* BL = HAS_L ? AL + SM::A_ELEMS : nullptr;
    const int kc = c * BK;
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

// Which tiles a phase-3 launch covers (block round K, nb tile rows):
//   P3_ALL  : every tile outside block-row K and block-column K;
//   P3_NEXT : those in block-row K+1 or block-column K+1 (the tiles the next
//             block round's phases 1 and 2 read and write);
//   P3_REST : the others.
// With symmetric inputs only tiles with I <= J are computed (each off-diagonal
// one is also stored transposed): (nb-1)nb/2, nb-1 and (nb-2)(nb-1)/2 tiles.

// t -> (a, b), a <= b, enumerating the upper triangle column by column.
__device__ __forceinline__ void p3_tri(int t, int& a, int& b) {
    int c = (int)((sqrtf(8.0f * (float)t + 1.0f) - 1.0f) * 0.5f);
    while (c * (c + 1) / 2 > t) --c;
    while ((c + 1) * (c + 2) / 2 <= t) ++c;
    b = c;
    a = t - c * (c + 1) / 2;
}

__device__ __forceinline__ void p3_tile(int part, bool sym, int t, int nb, int K, int& I,
                                        int& J) {
    if (!sym) {
        if (part == P3_ALL) {
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
    if (part == P3_ALL) {
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

template <class T, bool HAS_L, int FB>
__global__ void __launch_bounds__(P3S<FB>::NT)
k_phase3(T* __restrict__ U, T* __restrict__ L, int n, int ld, long long bstride, int K,
         int part, bool vec, bool sym) {
    using S = P3S<FB>;
    using E = El<T>;
    using SM = P3Smem<T, HAS_L, FB>;
    using LD = PairLoad<T>;
    using P = typename LD::P;
    constexpr bool NEG = std::is_same<T, int>::value;   // int lower bound adds negated values
    extern __shared__ __align__(16) unsigned char smem_raw[];
    T* sm = reinterpret_cast<T*>(smem_raw);

    const size_t off = (size_t)blockIdx.z * (size_t)bstride;
    U += off;
    if (HAS_L) L += off;
    const int nb = (n + FB - 1) / FB;
    int I, J;
    p3_tile(part, sym, blockIdx.x, nb, K, I, J);
    const int oi = I * FB, oj = J * FB, ok = K * FB;
    const int mi = min(FB, n - oi), mj = min(FB, n - oj), mk = min(FB, n - ok);

    T u[S::TM][S::TN], l[S::TM][S::TN];
    load_tile<S>(u, U + (size_t)oi * ld + oj, ld, mi, mj, vec, E::upad());
    if (HAS_L) load_tile<S>(l, L + (size_t)oi * ld + oj, ld, mi, mj, vec, E::lpad());

    const int nchunks = (mk + BK - 1) / BK;
    p3_stage<T, HAS_L, FB>(sm, U, L, ld, oi, oj, ok, mi, mj, mk, 0, vec);
    cp_async_commit();
    const int r0 = S::row0(), cq = S::cq();
    for (int c = 0; c < nchunks; ++c) {
        if (c + 1 < nchunks)
            p3_stage<T, HAS_L, FB>(sm + ((c + 1) & 1) * SM::STAGE, U, L, ld, oi, oj, ok, mi, mj,
                                   mk, c + 1, vec);
        cp_async_commit();
        cp_async_wait<1>();
        __syncthreads();
        const T* AU = sm + (c & 1) * SM::STAGE;
        const T* BU = AU + SM::A_ELEMS;
        const T* AL = BU + SM::B_ELEMS;
        const T* BL = AL + SM::A_ELEMS;
#pragma unroll 1
        for (int kk = 0; kk < BK; kk += 2) {
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
        }
        __syncthreads();
    }
    store_tile<S>(u, U + (size_t)oi * ld + oj, ld, mi, mj, vec);
    if (HAS_L) store_tile<S>(l, L + (size_t)oi * ld + oj, ld, mi, mj, vec);
    if (sym && I != J) {
        store_tile_t<S>(u, U + (size_t)oj * ld + oi, ld, mi, mj, vec);
        if (HAS_L) store_tile_t<S>(l, L + (size_t)oj * ld + oi, ld, mi, mj, vec);
    }
}

// ---------------------------------------------------------------- launchers

template <class T, bool HAS_L, int FB>
static size_t p2_smem() {
    return (size_t)(HAS_L ? 2 : 1) * FB * (FB + DPAD) * sizeof(T);
}

template <class T, bool HAS_L, int FB>
static cudaError_t setup_t() {
    cudaError_t e = cudaFuncSetAttribute(k_phase2<T, HAS_L, FB>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)p2_smem<T, HAS_L, FB>());
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(k_phase3<T, HAS_L, FB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)P3Smem<T, HAS_L, FB>::BYTES);
}

template <class T>
static cudaError_t setup_all() {
    cudaError_t e = setup_t<T, true, FB_LARGE>();
    if (e == cudaSuccess) e = setup_t<T, false, FB_LARGE>();
    if (e == cudaSuccess) e = setup_t<T, true, FB_SMALL>();
    if (e == cudaSuccess) e = setup_t<T, false, FB_SMALL>();
    return e;
}

cudaError_t blocked_setup(bool is_int) { return is_int ? setup_all<int>() : setup_all<float>(); }

enum class Which { One, Two, Three };

template <class T, bool HAS_L, int FB>
static cudaError_t phase_t(Which w, const Mats& m, int K, int part, cudaStream_t s) {
    constexpr int NT12 = P12<FB>::NT;   // phases 1 and 2
    constexpr int NT3 = P3S<FB>::NT;    // phase 3
    const int nb = (m.n + FB - 1) / FB;
    int tiles = 0;
    if (w == Which::Three) {
        if (m.sym)
            tiles = part == P3_ALL ? (nb - 1) * nb / 2
                    : part == P3_NEXT ? (K + 1 < nb ? nb - 1 : 0)
                                      : (K + 1 < nb ? (nb - 2) * (nb - 1) / 2 : 0);
        else
            tiles = part == P3_ALL ? (nb - 1) * (nb - 1)
                    : part == P3_NEXT ? (K + 1 < nb ? 2 * nb - 3 : 0)
                                      : (K + 1 < nb ? (nb - 2) * (nb - 2) : 0);
        if (nb < 2 || tiles <= 0) return cudaSuccess;
    }
    if (w == Which::Two && nb < 2) return cudaSuccess;
    for (int b0 = 0; b0 < m.batch; b0 += 65535) {
        const int nbz = m.batch - b0 < 65535 ? m.batch - b0 : 65535;
        T* U = static_cast<T*>(m.U) + (size_t)b0 * m.bstride;
        T* L = HAS_L ? static_cast<T*>(m.L) + (size_t)b0 * m.bstride : nullptr;
        if (w == Which::One) {
            before_launch(s, PH_ONE);
            k_phase1<T, HAS_L, FB><<<dim3(1, 1, nbz), NT12, 0, s>>>(U, L, m.n, m.ld, m.bstride, K,
                                                                  m.vec);
            after_launch(s, PH_ONE);
        } else if (w == Which::Two) {
            before_launch(s, PH_TWO);
            k_phase2<T, HAS_L, FB><<<dim3(nb - 1, m.sym ? 1 : 2, nbz), NT12, p2_smem<T, HAS_L, FB>(),
                                     s>>>(U, L, m.n, m.ld, m.bstride, K, m.vec, m.sym);
            after_launch(s, PH_TWO);
        } else {
            before_launch(s, PH_THREE);
            k_phase3<T, HAS_L, FB><<<dim3(tiles, 1, nbz), NT3, P3Smem<T, HAS_L, FB>::BYTES, s>>>(
                U, L, m.n, m.ld, m.bstride, K, part, m.vec, m.sym);
            after_launch(s, PH_THREE);
        }
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

template <class T, bool HAS_L>
static cudaError_t phase_fb(Which w, const Mats& m, int K, int part, cudaStream_t s) {
    return m.fb == FB_SMALL ? phase_t<T, HAS_L, FB_SMALL>(w, m, K, part, s)
                            : phase_t<T, HAS_L, FB_LARGE>(w, m, K, part, s);
}

static cudaError_t phase(Which w, bool is_int, const Mats& m, int K, int part, cudaStream_t s) {
    if (is_int) return m.L ? phase_fb<int, true>(w, m, K, part, s) : phase_fb<int, false>(w, m, K, part, s);
    return m.L ? phase_fb<float, true>(w, m, K, part, s) : phase_fb<float, false>(w, m, K, part, s);
}

cudaError_t launch_phase1(bool is_int, const Mats& m, int K, cudaStream_t s) {
    return phase(Which::One, is_int, m, K, P3_ALL, s);
}
cudaError_t launch_phase2(bool is_int, const Mats& m, int K, cudaStream_t s) {
    return phase(Which::Two, is_int, m, K, P3_ALL, s);
}
cudaError_t launch_phase3(bool is_int, const Mats& m, int K, int part, cudaStream_t s) {
    return phase(Which::Three, is_int, m, K, part, s);
}

}  // namespace bs
