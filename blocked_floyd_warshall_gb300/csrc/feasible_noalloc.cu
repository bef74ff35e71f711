// Infeasibility counts without any device allocation.
//
// Some callers cannot call cudaMalloc: code whose device memory is owned in
// full by its own allocator (a framework's caching allocator that accounts
// for every byte, or a fixed budget reserved up front), and code on paths
// where the implicit synchronisation and latency of cudaMalloc are not
// allowed.  bs_check_feasible allocates a small buffer on its first call on a
// device; this entry point instead keeps its counters in a fixed array in the
// library's own device memory (static storage, present on every device that
// loads the library, until the process exits).
//
// Scratch: kNoallocMaxBatch counters of 8 bytes (32 KiB).  One counter per
// molecule, cleared at the start of every call.  All calls share the array:
// calls whose GPU work overlaps (on different streams, or from different
// threads) race on it.
#include <mutex>

#include "../../include/bsmooth.h"
#include "bs_tile.cuh"

namespace bs {

namespace {

constexpr int kNoallocMaxBatch = BS_NOALLOC_MAX_BATCH;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned long long g_noalloc_counts[kNoallocMaxBatch];

std::mutex g_noalloc_mu;
unsigned long long* g_noalloc_ptr[kMaxDevices];   // device address of the array, per device

// Per-molecule count: as k_feasible, with counter blockIdx.z of `counts`.
template <class T>
__global__ void __launch_bounds__(256)
k_feasible_each(const T* __restrict__ U, const T* __restrict__ L, int n, int ld,
                long long bstride, unsigned long long* __restrict__ counts) {
    const size_t off = (size_t)blockIdx.z * (size_t)bstride;
    U += off;
    L += off;
    unsigned int c = 0;
    for (int i = blockIdx.y; i < n; i += gridDim.y) {
        const T* Ui = U + (size_t)i * ld;
        const T* Li = L + (size_t)i * ld;
        for (int j = blockIdx.x * blockDim.x + threadIdx.x; j < n; j += gridDim.x * blockDim.x)
            c += Li[j] > Ui[j];
    }
    c = __reduce_add_sync(0xffffffffu, c);
    __shared__ unsigned int part[8];
    if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = c;
    __syncthreads();
    if (threadIdx.x == 0) {
        unsigned long long s = 0;
        for (int w = 0; w < (int)(blockDim.x >> 5); ++w) s += part[w];
        if (s) atomicAdd(counts + blockIdx.z, s);
    }
}

// Device address of the static array on the current device.  Looked up once
// per device, with that device current, on the first call, and kept for the
// life of the process.  cudaDeviceReset destroys the device's context and
// with it the module holding the array, so the kept address is stale after
// one: this entry point must not be used on a device after a reset of it.
cudaError_t noalloc_counts(unsigned long long** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_counts);
        if (e != cudaSuccess) return e;
        g_noalloc_ptr[dev] = static_cast<unsigned long long*>(p);
    }
    *out = g_noalloc_ptr[dev];
    return cudaSuccess;
}

template <class T>
cudaError_t launch_each(const void* U, const void* L, int n, int ld, long long bstride, int batch,
                        unsigned long long* counts, cudaStream_t s) {
    const int gx = (n + 255) / 256 < 8 ? (n + 255) / 256 : 8;
    const int gy = n < 4096 ? n : 4096;
    note_launch();
    k_feasible_each<T><<<dim3(gx, gy, batch), 256, 0, s>>>(
        static_cast<const T*>(U), static_cast<const T*>(L), n, ld, bstride, counts);
    return cudaGetLastError();
}

}  // namespace

}  // namespace bs

extern "C" bs_status bs_check_feasible_noalloc(const void* U, const void* L, int n, int ld,
                                               long long batch_stride, int batch,
                                               bs_stream_t stream, int mode,
                                               long long* out_counts) {
    if (!out_counts || n < 0 || batch < 0) return BS_ERR_ARG;
    if (batch > BS_NOALLOC_MAX_BATCH) return BS_ERR_ARG;
    if ((mode & ~BS_DTYPE_MASK) != 0 || (mode & BS_DTYPE_MASK) > BS_INT32_Q10) return BS_ERR_ARG;
    if (n > 0 && ld < n) return BS_ERR_ARG;
    if (n == 0 || batch == 0) {
        for (int b = 0; b < batch; ++b) out_counts[b] = 0;
        return BS_OK;
    }
    if (!U || !L || U == L) return BS_ERR_ARG;
    if (batch > 1 && batch_stride < (long long)(n - 1) * ld + n) return BS_ERR_ARG;
    if (reinterpret_cast<uintptr_t>(U) % 4 || reinterpret_cast<uintptr_t>(L) % 4)
        return BS_ERR_ALIGN;
    const long long stride = batch > 1 ? batch_stride : 0;
    unsigned long long* counts = nullptr;
    cudaError_t e = bs::noalloc_counts(&counts);
    if (e == cudaSuccess)
        e = cudaMemsetAsync(counts, 0, sizeof(unsigned long long) * (size_t)batch, stream);
    if (e == cudaSuccess)
        e = (mode & BS_DTYPE_MASK) == BS_INT32_Q10
                ? bs::launch_each<int>(U, L, n, ld, stride, batch, counts, stream)
                : bs::launch_each<float>(U, L, n, ld, stride, batch, counts, stream);
    // The device counters are unsigned 64-bit; they are copied bit for bit
    // into the caller's long long array, as bs_check_feasible returns its
    // count.  A count is at most n^2 < 2^62, so it reads the same either way.
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(out_counts, counts, sizeof(unsigned long long) * (size_t)batch,
                            cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    return e == cudaSuccess ? BS_OK : BS_ERR_CUDA;
}
