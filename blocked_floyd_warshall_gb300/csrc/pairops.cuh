// Helpers shared by the blocked kernels: cp.async staging, the paired
// middle-atom instructions, and the loop over batch chunks of a launch.
#pragma once

#include <type_traits>

#include "bs_tile.cuh"

namespace bs {

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
    const unsigned s = (unsigned)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async4(void* smem, const void* gmem) {
    const unsigned s = (unsigned)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;\n" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

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
    static __device__ __forceinline__ P mk(float lo, float hi) {
        return (unsigned long long)__float_as_uint(lo) |
               ((unsigned long long)__float_as_uint(hi) << 32);
    }
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
    static __device__ __forceinline__ P mk(int lo, int hi) { return make_int2(lo, hi); }
};

// Launch `launch(first, count)` over the batch in chunks the grid's z dimension
// can hold; returns the first launch error.
template <class F>
cudaError_t for_batch_chunks(const Mats& m, F launch) {
    for (int b0 = 0; b0 < m.batch; b0 += 65535) {
        const int nbz = m.batch - b0 < 65535 ? m.batch - b0 : 65535;
        cudaError_t e = launch(b0, nbz);
        if (e == cudaSuccess) e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

// Launch on `s` carrying the stream's priority as a launch attribute, so that
// a launch captured into a CUDA graph keeps it (a graph's kernel nodes do not
// inherit the priority of the stream they were captured from).  The
// look-ahead stream's kernels depend on it.
template <class... KArgs, class... Args>
cudaError_t launch_prio(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                        cudaStream_t s, Args... args) {
    int prio = 0;
    cudaError_t e = cudaStreamGetPriority(s, &prio);
    if (e != cudaSuccess) return e;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributePriority;
    attr[0].val.priority = prio;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = prio != 0 ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

}  // namespace bs
