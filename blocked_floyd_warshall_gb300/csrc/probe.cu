// ALU issue-rate probes: how many thread-instructions per clock one SM retires
// for each instruction form the min-plus / max-minus inner loops can use.
// These rates set the denominator of the ALU roofline; they are measured, not
// assumed.  Each probe runs one CTA of 1024 threads per SM, 8 independent
// dependency chains per thread, and reads the SM cycle counter around the loop.
#include <cuda_runtime.h>

#include "../../include/bsmooth.h"
#include "bs_internal.cuh"

namespace bs {

namespace {

constexpr int kChains = 8;
constexpr int kUnroll = 16;

template <int OP>
__device__ __forceinline__ void op_f(float& x, float y, float z) {
    if (OP == BS_PROBE_FADD) {
        asm volatile("add.rn.f32 %0, %0, %1;" : "+f"(x) : "f"(y));
    } else if (OP == BS_PROBE_FMNMX) {
        asm volatile("min.f32 %0, %0, %1;" : "+f"(x) : "f"(y));
    } else if (OP == BS_PROBE_FMNMX3) {
        asm volatile("min.f32 %0, %0, %1, %2;" : "+f"(x) : "f"(y), "f"(z));
    }
}

template <int OP>
__device__ __forceinline__ void op_i(int& x, int y, int z) {
    if (OP == BS_PROBE_IADD) {
        asm volatile("add.s32 %0, %0, %1;" : "+r"(x) : "r"(y));
    } else if (OP == BS_PROBE_IMNMX) {
        asm volatile("min.s32 %0, %0, %1;" : "+r"(x) : "r"(y));
    } else if (OP == BS_PROBE_VIADDMIN) {
        x = __viaddmin_s32(y, x, z);
    } else if (OP == BS_PROBE_VIMNMX3) {
        x = __vimin3_s32(x, y, z);
    }
}

template <int OP>
__global__ void __launch_bounds__(1024, 1) k_probe(float* sink, int iters, long long* cycles) {
    const float y = 1e-30f * (threadIdx.x + 1), z = 3e-30f;
    const int yi = (int)(threadIdx.x & 7) - 3, zi = 1 << 29;
    float xf[kChains];
    int xi[kChains];
    unsigned long long xp[kChains];
    const unsigned long long yp = 0x0080000000800000ull;   // two smallest normal floats
#pragma unroll
    for (int c = 0; c < kChains; ++c) {
        xf[c] = 1.0f + c;
        xi[c] = c;
        xp[c] = 0x3f8000003f800000ull + c;
    }
    __syncthreads();
    const long long t0 = clock64();
    for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
#pragma unroll
            for (int c = 0; c < kChains; ++c) {
                if (OP == BS_PROBE_FADD2) {
                    asm volatile("add.rn.f32x2 %0, %0, %1;" : "+l"(xp[c]) : "l"(yp));
                } else if (OP == BS_PROBE_FADD2_FMNMX3) {
                    if (c & 1)
                        asm volatile("add.rn.f32x2 %0, %0, %1;" : "+l"(xp[c]) : "l"(yp));
                    else
                        op_f<BS_PROBE_FMNMX3>(xf[c], y, z);
                } else if (OP >= BS_PROBE_IADD) {
                    op_i<OP>(xi[c], yi, zi);
                } else {
                    op_f<OP>(xf[c], y, z);
                }
            }
        }
    }
    __syncthreads();
    const long long t1 = clock64();
    if (threadIdx.x == 0) cycles[blockIdx.x] = t1 - t0;
    float s = 0.f;
#pragma unroll
    for (int c = 0; c < kChains; ++c) s += xf[c] + (float)xi[c] + __int_as_float((int)(xp[c] & 0xff));
    if (s == 12345.678f) sink[threadIdx.x] = s;
}

template <int OP>
cudaError_t run(int sms, int iters, float* sink, long long* cyc, cudaStream_t s) {
    k_probe<OP><<<sms, 1024, 0, s>>>(sink, iters, cyc);
    return cudaGetLastError();
}

}  // namespace

}  // namespace bs

extern "C" bs_status bs_probe_alu(int which, int iters, double* instr_per_clk_per_sm) {
    using namespace bs;
    if (!instr_per_clk_per_sm || iters <= 0 || which < BS_PROBE_FADD || which > BS_PROBE_VIMNMX3)
        return BS_ERR_ARG;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return BS_ERR_CUDA;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return BS_ERR_CUDA;
    float* sink = nullptr;
    long long* cyc = nullptr;
    if (cudaMalloc(&sink, 1024 * sizeof(float)) != cudaSuccess) return BS_ERR_CUDA;
    if (cudaMalloc(&cyc, sms * sizeof(long long)) != cudaSuccess) {
        cudaFree(sink);
        return BS_ERR_CUDA;
    }
    cudaStream_t s = nullptr;
    cudaError_t e = cudaSuccess;
    for (int rep = 0; rep < 2 && e == cudaSuccess; ++rep) {   // first pass warms up
        switch (which) {
            case BS_PROBE_FADD: e = run<BS_PROBE_FADD>(sms, iters, sink, cyc, s); break;
            case BS_PROBE_FMNMX: e = run<BS_PROBE_FMNMX>(sms, iters, sink, cyc, s); break;
            case BS_PROBE_FMNMX3: e = run<BS_PROBE_FMNMX3>(sms, iters, sink, cyc, s); break;
            case BS_PROBE_FADD2: e = run<BS_PROBE_FADD2>(sms, iters, sink, cyc, s); break;
            case BS_PROBE_FADD2_FMNMX3: e = run<BS_PROBE_FADD2_FMNMX3>(sms, iters, sink, cyc, s); break;
            case BS_PROBE_IADD: e = run<BS_PROBE_IADD>(sms, iters, sink, cyc, s); break;
            case BS_PROBE_IMNMX: e = run<BS_PROBE_IMNMX>(sms, iters, sink, cyc, s); break;
            case BS_PROBE_VIADDMIN: e = run<BS_PROBE_VIADDMIN>(sms, iters, sink, cyc, s); break;
            case BS_PROBE_VIMNMX3: e = run<BS_PROBE_VIMNMX3>(sms, iters, sink, cyc, s); break;
        }
        if (e == cudaSuccess) e = cudaDeviceSynchronize();
    }
    long long* h = new long long[sms];
    if (e == cudaSuccess) e = cudaMemcpy(h, cyc, sms * sizeof(long long), cudaMemcpyDeviceToHost);
    if (e == cudaSuccess) {
        double mean = 0;
        for (int i = 0; i < sms; ++i) mean += (double)h[i];
        mean /= sms;
        const double instr = 1024.0 * iters * kUnroll * kChains;   // thread-instructions per CTA
        *instr_per_clk_per_sm = instr / mean;
    }
    delete[] h;
    cudaFree(sink);
    cudaFree(cyc);
    return e == cudaSuccess ? BS_OK : BS_ERR_CUDA;
}
