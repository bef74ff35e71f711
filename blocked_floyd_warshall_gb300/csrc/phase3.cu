// Phases 2 and 3 of the three-phase blocked Floyd-Warshall: the panel and
// bulk tile updates, one kernel.  (The schedule as a whole, and why the panels
// are the same product as the bulk tiles, is described at the top of
// phase1.cu.)
#include "p3_tile.cuh"

namespace bs {

// Occupancy floors: two CTAs per SM for the upper bound alone on 128-wide
// tiles, four for the 8 x 4 form of 64-wide tiles (128 registers each).
template <class T, bool HAS_L, int FB, bool WIDE>
__global__ void __launch_bounds__(P3S<FB, WIDE>::NT,
                                  (!HAS_L && FB == FB_LARGE) ? 2 : (FB == FB_SMALL && !WIDE ? 4 : 0))
k_phase3(T* __restrict__ U, T* __restrict__ L, int n, int ld, long long bstride, int K,
         int part, bool vec, bool sym) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    const size_t off = (size_t)blockIdx.z * (size_t)bstride;
    U += off;
    if (HAS_L) L += off;
    const int nb = (n + FB - 1) / FB;
    int I, J;
    if (!WIDE && part >= P3_REST2) p3_tile_pair(part, sym, blockIdx.x, nb, K, I, J);
    else p3_tile(part, sym, blockIdx.x, nb, K, I, J);
    const bool two = part == P3_REST2 || part == P3_NEAR2;   // rounds K and K+1
    p3_update_tile<T, HAS_L, FB, WIDE>(U, L, n, ld, I, J, K, vec, sym && part == P3_PANELS,
                                       reinterpret_cast<T*>(smem_raw), two ? K + 1 : -1);
}

// ---------------------------------------------------------------- strips
//
// When a launch has fewer 64-wide tiles than half the SMs (small n: a block
// round of n = 256 has 9 bulk tiles and 6 panel tiles), each tile is split
// among SPLIT = 4 CTAs (the template also takes 2), each computing one strip
// of it, so that more SMs
// share the round's critical path.  A strip is the 64 rows x 64/SPLIT columns
// of the tile, or for a column panel 64/SPLIT rows x 64 columns: a CTA then
// reads of its own tile (the panel operand of phase 2) only the lines it
// writes itself, and no two CTAs touch the same cell.  Same update as
// k_phase3: middle atoms in pairs, operands staged per 16 middle atoms with
// cp.async.  256 threads, each 64/(16 SPLIT) rows x 4 columns.

constexpr int SFB = FB_SMALL;      // strips only split 64-wide tiles
constexpr int SBK = P3K<SFB>::BK;  // 16
constexpr int SAST = SBK + 4;
constexpr int SNT = 256;

// One buffer per 16-middle-atom chunk (four): a strip's CTA is latency-bound,
// so every chunk is put in flight at once instead of two at a time.
template <class T, bool HAS_L>
struct StripSmem {
    static constexpr int A_ELEMS = SFB * SAST;   // A[i][k], up to 64 rows
    static constexpr int B_ELEMS = SBK * SFB;    // B[k/2][j][k%2], up to 64 columns
    static constexpr int STAGE = (HAS_L ? 2 : 1) * (A_ELEMS + B_ELEMS);
    static constexpr int STAGES = SFB / SBK;
    static constexpr size_t BYTES = STAGES * STAGE * sizeof(T);
};

// Stage chunk c of the column operand (rows gi .. gi+ri-1 of the global
// matrix, middle atoms ok + c*SBK ..) and of the row operand (columns
// gj .. gj+cj-1); rs x cs is the strip's full extent, cells beyond the valid
// ri x cj (and middle atoms beyond mk) get pads.
template <class T, bool HAS_L>
__device__ __forceinline__ void strip_stage(T* stage, const T* U, const T* L, size_t ld, int gi,
                                            int gj, int ok, int rs, int cs, int ri, int cj,
                                            int mk, int c, bool vec) {
    using E = El<T>;
    using SM = StripSmem<T, HAS_L>;
    T* AU = stage;
    T* BU = stage + SM::A_ELEMS;
    T* AL = HAS_L ? BU + SM::B_ELEMS : nullptr;
    T* BL = HAS_L ? AL + SM::A_ELEMS : nullptr;
    const int kc = c * SBK;
    for (int p = threadIdx.x; p < rs * (SBK / 4); p += SNT) {
        const int i = p / (SBK / 4), kq = (p % (SBK / 4)) * 4;
        const size_t g = (size_t)(gi + i) * ld + ok + kc + kq;
        if (vec && i < ri && kc + kq + 4 <= mk) {
            cp_async16(AU + i * SAST + kq, U + g);
            if (HAS_L) cp_async16(AL + i * SAST + kq, L + g);
        } else {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const bool in = i < ri && kc + kq + q < mk;
                AU[i * SAST + kq + q] = in ? U[g + q] : E::upad();
                if (HAS_L) AL[i * SAST + kq + q] = in ? L[g + q] : E::lpad();
            }
        }
    }
    for (int p = threadIdx.x; p < SBK * cs; p += SNT) {
        const int k = p / cs, j = p % cs;
        const int d = (k >> 1) * (2 * SFB) + j * 2 + (k & 1);
        const size_t g = (size_t)(ok + kc + k) * ld + gj + j;
        if (kc + k < mk && j < cj) {
            cp_async4(BU + d, U + g);
            if (HAS_L) cp_async4(BL + d, L + g);
        } else {
            BU[d] = E::upad();
            if (HAS_L) BL[d] = E::lpad();
        }
    }
}

template <class T, bool HAS_L, int SPLIT>
__global__ void __launch_bounds__(SNT)
k_strip(T* __restrict__ U, T* __restrict__ L, int n, int ld, long long bstride, int K, int part,
        bool vec, bool sym) {
    using E = El<T>;
    using SM = StripSmem<T, HAS_L>;
    using LD = PairLoad<T>;
    using P = typename LD::P;
    constexpr int W = SFB / SPLIT;    // strip width
    constexpr int TMS = W / 16;       // rows per thread: 64 * W cells over 256 threads, 4 columns each
    constexpr bool NEG = std::is_same<T, int>::value;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    T* sm = reinterpret_cast<T*>(smem_raw);

    const size_t off = (size_t)blockIdx.z * (size_t)bstride;
    U += off;
    if (HAS_L) L += off;
    const int nb = (n + SFB - 1) / SFB;
    int I, J;
    p3_tile(part, sym, blockIdx.x, nb, K, I, J);
    const int oi = I * SFB, oj = J * SFB, ok = K * SFB;
    const int mi = min(SFB, n - oi), mj = min(SFB, n - oj), mk = min(SFB, n - ok);
    // the strip: rows r0 .. r0+rs-1, columns c0 .. c0+cs-1 of the tile
    const bool rows_split = part == P3_PANELS && J == K && I != K;   // column panel
    const int s = blockIdx.y;
    const int r0 = rows_split ? s * W : 0, c0 = rows_split ? 0 : s * W;
    const int rs = rows_split ? W : SFB, cs = rows_split ? SFB : W;
    const int ri = max(0, min(rs, mi - r0)), cj = max(0, min(cs, mj - c0));
    const int qx = cs / 4;                       // column quads
    const int tx = threadIdx.x % qx, ty = threadIdx.x / qx;
    const int lr = ty * TMS, lc = tx * 4;        // the thread's cells, strip-relative
    T* Us = U + (size_t)(oi + r0) * ld + oj + c0;
    T* Ls = HAS_L ? L + (size_t)(oi + r0) * ld + oj + c0 : nullptr;

    T u[TMS][4], l[TMS][4];
#pragma unroll
    for (int r = 0; r < TMS; ++r) {
        const int i = lr + r;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const bool in = i < ri && lc + q < cj;
            u[r][q] = in ? Us[(size_t)i * ld + lc + q] : E::upad();
            l[r][q] = HAS_L && in ? Ls[(size_t)i * ld + lc + q] : E::lpad();
        }
    }

    const int nchunks = (mk + SBK - 1) / SBK;   // 1 .. SM::STAGES
    for (int c = 0; c < SM::STAGES; ++c) {
        if (c < nchunks)
            strip_stage<T, HAS_L>(sm + c * SM::STAGE, U, L, ld, oi + r0, oj + c0, ok, rs, cs, ri,
                                  cj, mk, c, vec);
        cp_async_commit();   // one group per buffer, empty past the last chunk
    }
    static_assert(SM::STAGES == 4, "the waits below count four groups");
    for (int c = 0; c < nchunks; ++c) {
        // chunk c landed once at most 3 - c younger groups are still pending
        if (c == 0) cp_async_wait<3>();
        else if (c == 1) cp_async_wait<2>();
        else if (c == 2) cp_async_wait<1>();
        else cp_async_wait<0>();
        __syncthreads();
        const T* AU = sm + c * SM::STAGE;
        const T* BU = AU + SM::A_ELEMS;
        const T* AL = BU + SM::B_ELEMS;
        const T* BL = AL + SM::A_ELEMS;
#pragma unroll 2
        for (int kk = 0; kk < SBK; kk += 2) {
            P a[TMS], al[TMS], b[4], bl[4];
#pragma unroll
            for (int r = 0; r < TMS; ++r) {
                a[r] = LD::ld2(AU + (lr + r) * SAST + kk);
                if (HAS_L) al[r] = LD::ld2(AL + (lr + r) * SAST + kk);
            }
            const int jb = (kk >> 1) * (2 * SFB) + lc * 2;
            LD::ld4(BU + jb, b[0], b[1]);
            LD::ld4(BU + jb + 4, b[2], b[3]);
            if (HAS_L) {
                LD::ld4(BL + jb, bl[0], bl[1]);
                LD::ld4(BL + jb + 4, bl[2], bl[3]);
            }
#pragma unroll
            for (int r = 0; r < TMS; ++r)
#pragma unroll
                for (int q = 0; q < 4; ++q) PairOps<T>::upper(u[r][q], a[r], b[q]);
            if (HAS_L) {
                if (NEG) {
#pragma unroll
                    for (int r = 0; r < TMS; ++r) a[r] = LD::neg(a[r]);
#pragma unroll
                    for (int q = 0; q < 4; ++q) b[q] = LD::neg(b[q]);
                }
#pragma unroll
                for (int r = 0; r < TMS; ++r)
#pragma unroll
                    for (int q = 0; q < 4; ++q) PairOps<T>::lower(l[r][q], a[r], al[r], b[q], bl[q]);
            }
        }
    }

#pragma unroll
    for (int r = 0; r < TMS; ++r) {
        const int i = lr + r;
        if (i >= ri) continue;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            if (lc + q >= cj) continue;
            Us[(size_t)i * ld + lc + q] = u[r][q];
            if (HAS_L) Ls[(size_t)i * ld + lc + q] = l[r][q];
            if (sym && part == P3_PANELS && I != J) {
                // the mirrored cell of tile (J, I)
                const size_t t = (size_t)(oj + c0 + lc + q) * ld + oi + r0 + i;
                U[t] = u[r][q];
                if (HAS_L) L[t] = l[r][q];
            }
        }
    }
}

// ---------------------------------------------------------------- mirror

// Symmetric mode, after the last block round: each CTA writes one 64-wide
// block (a,b), a < b, transposed over (b,a).  Blocks inside a diagonal tile
// of the schedule (a and b in the same block of fb) were computed whole and
// are left alone.
using MS = P3S<FB_SMALL, true>;

template <class T, bool HAS_L>
constexpr size_t mirror_bytes() {
    return (HAS_L ? 2 : 1) * (size_t)FB_SMALL * (FB_SMALL + 4) * sizeof(T);
}

template <class T, bool HAS_L>
__global__ void __launch_bounds__(MS::NT)
k_mirror(T* __restrict__ U, T* __restrict__ L, int n, int ld, long long bstride, int fb, bool vec) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    int a, c;
    p3_tri(blockIdx.x, a, c);
    const int b = c + 1, r = fb / FB_SMALL;
    if (a / r == b / r) return;   // the whole CTA
    const size_t off = (size_t)blockIdx.z * (size_t)bstride;
    p3_mirror_block<T, HAS_L>(U + off, HAS_L ? L + off : nullptr, n, ld, a, b, vec,
                              reinterpret_cast<T*>(smem_raw));
}

template <class T, bool HAS_L>
static cudaError_t mirror_t(const Mats& m, cudaStream_t s) {
    const int nb = (m.n + FB_SMALL - 1) / FB_SMALL;
    const long long pairs = (long long)(nb - 1) * nb / 2;
    if (pairs <= 0) return cudaSuccess;
    return for_batch_chunks(m, [&](int b0, int nbz) {
        T* U = static_cast<T*>(m.U) + (size_t)b0 * m.bstride;
        T* L = HAS_L ? static_cast<T*>(m.L) + (size_t)b0 * m.bstride : nullptr;
        before_launch(s, PH_THREE);
        const cudaError_t e = launch_prio(k_mirror<T, HAS_L>, dim3((unsigned)pairs, 1, nbz),
                                          dim3(MS::NT), mirror_bytes<T, HAS_L>(), s, U, L, m.n,
                                          m.ld, m.bstride, m.fb, m.vec);
        after_launch(s, PH_THREE);
        return e;
    });
}

cudaError_t launch_mirror(bool is_int, const Mats& m, cudaStream_t s) {
    if (is_int) return m.L ? mirror_t<int, true>(m, s) : mirror_t<int, false>(m, s);
    return m.L ? mirror_t<float, true>(m, s) : mirror_t<float, false>(m, s);
}

// ---------------------------------------------------------------- launchers

template <class T>
static cudaError_t setup3() {
    cudaError_t e = cudaSuccess;
    auto set = [&](auto kernel, size_t bytes) {
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    };
    set(k_phase3<T, true, FB_LARGE, false>, P3Smem<T, true, FB_LARGE>::BYTES);
    set(k_phase3<T, false, FB_LARGE, false>, P3Smem<T, false, FB_LARGE>::BYTES);
    set(k_phase3<T, true, FB_SMALL, false>, P3Smem<T, true, FB_SMALL>::BYTES);
    set(k_phase3<T, false, FB_SMALL, false>, P3Smem<T, false, FB_SMALL>::BYTES);
    set(k_phase3<T, true, FB_SMALL, true>, P3Smem<T, true, FB_SMALL>::BYTES);
    set(k_phase3<T, false, FB_SMALL, true>, P3Smem<T, false, FB_SMALL>::BYTES);
    set(k_strip<T, true, 4>, StripSmem<T, true>::BYTES);
    set(k_strip<T, false, 4>, StripSmem<T, false>::BYTES);
    return e;
}

cudaError_t phase3_setup(bool is_int) { return is_int ? setup3<int>() : setup3<float>(); }

template <class T, bool HAS_L, int FB, bool WIDE>
static cudaError_t phase3_t(const Mats& m, int K, int part, cudaStream_t s) {
    const int nb = (m.n + FB - 1) / FB;
    const int tiles = p3_tiles(m.sym, part, nb, K);
    if (tiles <= 0) return cudaSuccess;
    return for_batch_chunks(m, [&](int b0, int nbz) {
        T* U = static_cast<T*>(m.U) + (size_t)b0 * m.bstride;
        T* L = HAS_L ? static_cast<T*>(m.L) + (size_t)b0 * m.bstride : nullptr;
        const Phase ph = part == P3_PANELS ? PH_TWO
                         : part == P3_NEXT || part == P3_NEAR2 || part == P3_CORNER2 ? PH_NEXT
                                                                                   : PH_THREE;
        before_launch(s, ph);
        const cudaError_t e = launch_prio(k_phase3<T, HAS_L, FB, WIDE>, dim3(tiles, 1, nbz),
                                          dim3(P3S<FB, WIDE>::NT), P3Smem<T, HAS_L, FB>::BYTES, s,
                                          U, L, m.n, m.ld, m.bstride, K, part, m.vec, m.sym);
        after_launch(s, ph);
        return e;
    });
}

template <class T, bool HAS_L, int SPLIT>
static cudaError_t strip_t(const Mats& m, int K, int part, cudaStream_t s) {
    const int nb = (m.n + SFB - 1) / SFB;
    const int tiles = p3_tiles(m.sym, part, nb, K);
    if (tiles <= 0) return cudaSuccess;
    return for_batch_chunks(m, [&](int b0, int nbz) {
        T* U = static_cast<T*>(m.U) + (size_t)b0 * m.bstride;
        T* L = HAS_L ? static_cast<T*>(m.L) + (size_t)b0 * m.bstride : nullptr;
        const Phase ph = part == P3_PANELS ? PH_TWO : part == P3_NEXT ? PH_NEXT : PH_THREE;
        before_launch(s, ph);
        const cudaError_t e = launch_prio(k_strip<T, HAS_L, SPLIT>, dim3(tiles, SPLIT, nbz),
                                          dim3(SNT), StripSmem<T, HAS_L>::BYTES, s, U, L, m.n,
                                          m.ld, m.bstride, K, part, m.vec, m.sym);
        after_launch(s, ph);
        return e;
    });
}

// 64-wide tiles, by tiles per SM in the launch: up to half, four strips per
// tile; up to one, the wide form (a tile per SM, latency-bound); more, the
// 8 x 4 form, four CTAs per SM.  (Measured on the GB300: n = 2048, where the
// next block row and column and the panels, 61 and 62 tiles, run on the
// look-ahead critical path, is 12 % faster with four strips than with two;
// n = 1000's 196 and 225 bulk tiles are 6 % faster in the 8 x 4 form than in
// the wide form and 8 % slower as strips.)
template <class T, bool HAS_L>
static cudaError_t phase3_fb(const Mats& m, int K, int part, cudaStream_t s) {
    if (m.fb == FB_LARGE) return phase3_t<T, HAS_L, FB_LARGE, false>(m, K, part, s);
    // the pair schedule's sets: always the 8 x 4 form (the only 64-wide form with their maps)
    if (part >= P3_REST2) return phase3_t<T, HAS_L, FB_SMALL, false>(m, K, part, s);
    const int nb = (m.n + FB_SMALL - 1) / FB_SMALL;
    const double ctas = (double)p3_tiles(m.sym, part, nb, K) * m.batch;
    if (2.0 * ctas <= m.sms) return strip_t<T, HAS_L, 4>(m, K, part, s);
    return ctas <= 1.0 * m.sms ? phase3_t<T, HAS_L, FB_SMALL, true>(m, K, part, s)
                               : phase3_t<T, HAS_L, FB_SMALL, false>(m, K, part, s);
}

cudaError_t launch_phase3(bool is_int, const Mats& m, int K, int part, cudaStream_t s) {
    if (is_int) return m.L ? phase3_fb<int, true>(m, K, part, s) : phase3_fb<int, false>(m, K, part, s);
    return m.L ? phase3_fb<float, true>(m, K, part, s) : phase3_fb<float, false>(m, K, part, s);
}

cudaError_t launch_phase2(bool is_int, const Mats& m, int K, cudaStream_t s) {
    return launch_phase3(is_int, m, K, P3_PANELS, s);
}

}  // namespace bs
