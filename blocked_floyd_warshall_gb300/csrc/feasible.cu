// Infeasibility count (cells with L > U) and the optional precondition check.
// One pass over both matrices: HBM-bound, 8 bytes read per fp32 cell.
#include "bs_tile.cuh"

namespace bs {

// One pass over both matrices.  With 16-byte rows (vec) each thread compares
// four cells per step through 16-byte loads (and writes the mask as 4 bytes);
// otherwise one cell.  The count is reduced per warp, then per CTA, then one
// atomic per CTA.
template <class T>
__global__ void __launch_bounds__(256)
k_feasible(const T* __restrict__ U, const T* __restrict__ L, int n, int ld, long long bstride,
           bool vec, unsigned char* __restrict__ mask, unsigned long long* __restrict__ count) {
    using V4 = typename El<T>::V4;
    const size_t off = (size_t)blockIdx.z * (size_t)bstride;
    U += off;
    L += off;
    if (mask) mask += off;
    unsigned int c = 0;
    const int stride = gridDim.x * blockDim.x;
    const int j0 = blockIdx.x * blockDim.x + threadIdx.x;
    for (int i = blockIdx.y; i < n; i += gridDim.y) {
        const T* Ui = U + (size_t)i * ld;
        const T* Li = L + (size_t)i * ld;
        if (vec) {
            const int nq = n / 4;
            for (int q = j0; q < nq; q += stride) {
                const V4 u = reinterpret_cast<const V4*>(Ui)[q];
                const V4 l = reinterpret_cast<const V4*>(Li)[q];
                const unsigned b0 = l.x > u.x, b1 = l.y > u.y, b2 = l.z > u.z, b3 = l.w > u.w;
                c += b0 + b1 + b2 + b3;
                if (mask)
                    reinterpret_cast<uchar4*>(mask + (size_t)i * ld)[q] =
                        make_uchar4((unsigned char)b0, (unsigned char)b1, (unsigned char)b2,
                                    (unsigned char)b3);
            }
            for (int j = 4 * nq + j0; j < n; j += stride) {   // the last n % 4 cells
                const bool bad = Li[j] > Ui[j];
                c += bad;
                if (mask) mask[(size_t)i * ld + j] = bad ? 1 : 0;
            }
        } else {
            for (int j = j0; j < n; j += stride) {
                const bool bad = Li[j] > Ui[j];
                c += bad;
                if (mask) mask[(size_t)i * ld + j] = bad ? 1 : 0;
            }
        }
    }
    c = __reduce_add_sync(0xffffffffu, c);
    __shared__ unsigned int part[8];
    if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = c;
    __syncthreads();
    if (threadIdx.x == 0) {
        unsigned long long s = 0;
        for (int w = 0; w < (int)(blockDim.x >> 5); ++w) s += part[w];
        if (s) atomicAdd(count, s);
    }
}

__device__ __forceinline__ unsigned int check_value(float v, bool lower, bool diag) {
    unsigned int f = 0;
    if (v != v) f |= VF_NAN;
    if (v < 0.0f) f |= VF_NEG;
    if (lower && (v == __int_as_float(0x7f800000) || v == __int_as_float(0xff800000))) f |= VF_LINF;
    if (diag && v != 0.0f) f |= VF_DIAG;
    return f;
}

__device__ __forceinline__ unsigned int check_value(int v, bool, bool diag) {
    unsigned int f = 0;
    if (v < 0) f |= VF_NEG;
    if (v >= (1 << 30)) f |= VF_RANGE;
    if (diag && v != 0) f |= VF_DIAG;
    return f;
}

template <class T>
__global__ void __launch_bounds__(256)
k_validate(const T* __restrict__ U, const T* __restrict__ L, int n, int ld, long long bstride,
           bool sym, unsigned int* __restrict__ flags) {
    const size_t off = (size_t)blockIdx.z * (size_t)bstride;
    U += off;
    if (L) L += off;
    unsigned int f = 0;
    for (int i = blockIdx.y; i < n; i += gridDim.y) {
        for (int j = blockIdx.x * blockDim.x + threadIdx.x; j < n; j += gridDim.x * blockDim.x) {
            f |= check_value(U[(size_t)i * ld + j], false, i == j);
            if (L) f |= check_value(L[(size_t)i * ld + j], true, i == j);
            if (sym && j > i) {
                if (!(U[(size_t)i * ld + j] == U[(size_t)j * ld + i])) f |= VF_ASYM;
                if (L && !(L[(size_t)i * ld + j] == L[(size_t)j * ld + i])) f |= VF_ASYM;
            }
        }
    }
    f = __reduce_or_sync(0xffffffffu, f);
    if ((threadIdx.x & 31) == 0 && f) atomicOr(flags, f);
}

static dim3 pass_grid(int n, int nbz) {
    const int gx = (n + 255) / 256 < 8 ? (n + 255) / 256 : 8;
    const int gy = n < 4096 ? n : 4096;
    return dim3(gx > 0 ? gx : 1, gy > 0 ? gy : 1, nbz);
}

template <class T>
static cudaError_t feasible_t(const Mats& m, unsigned char* mask, unsigned long long* count,
                              cudaStream_t s) {
    for (int b0 = 0; b0 < m.batch; b0 += 65535) {
        const int nbz = m.batch - b0 < 65535 ? m.batch - b0 : 65535;
        const size_t o = (size_t)b0 * m.bstride;
        before_launch(s, PH_ROUND);
        // 16-byte loads need 16-byte rows (m.vec) and, for the mask, 4-byte rows
        const bool vec = m.vec && (!mask || reinterpret_cast<uintptr_t>(mask) % 4 == 0);
        k_feasible<T><<<pass_grid(m.n, nbz), 256, 0, s>>>(
            static_cast<const T*>(m.U) + o, static_cast<const T*>(m.L) + o, m.n, m.ld,
            m.bstride, vec, mask ? mask + o : nullptr, count);
        after_launch(s, PH_ROUND);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

template <class T>
static cudaError_t validate_t(const Mats& m, unsigned int* flags, cudaStream_t s) {
    for (int b0 = 0; b0 < m.batch; b0 += 65535) {
        const int nbz = m.batch - b0 < 65535 ? m.batch - b0 : 65535;
        const size_t o = (size_t)b0 * m.bstride;
        before_launch(s, PH_ROUND);
        k_validate<T><<<pass_grid(m.n, nbz), 256, 0, s>>>(
            static_cast<const T*>(m.U) + o, m.L ? static_cast<const T*>(m.L) + o : nullptr,
            m.n, m.ld, m.bstride, m.sym, flags);
        after_launch(s, PH_ROUND);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t launch_feasible(bool is_int, const Mats& m, unsigned char* mask,
                            unsigned long long* count, cudaStream_t s) {
    return is_int ? feasible_t<int>(m, mask, count, s) : feasible_t<float>(m, mask, count, s);
}

cudaError_t launch_validate(bool is_int, const Mats& m, unsigned int* flags, cudaStream_t s) {
    return is_int ? validate_t<int>(m, flags, s) : validate_t<float>(m, flags, s);
}

}  // namespace bs
