// Test-only check of the library's bounded mbarrier wait (kda_ptx.cuh), the
// building block of every kernel's timeout path: one CTA initialises an
// mbarrier with one expected arrival and
//   mode 0: nobody arrives; the wait must give up after `budget` clock
//           cycles and report failure (the kernel then returns normally);
//   mode 1: thread 0 arrives first; the wait must succeed at once.
// Every wait is bounded, so the probe cannot hang. Built by
// tests/test_wait_timeout.py with nvcc into a temporary library.
#include <cuda_runtime.h>

#include <cstdint>

#include "kda_ptx.cuh"

__global__ void wait_probe_kernel(int mode, long long budget, unsigned *ok, long long *cycles) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        kda::ptx::mbar_init(&bar, 1);
        kda::ptx::fence_mbar_init();
    }
    __syncthreads();
    if (mode == 1 && threadIdx.x == 0) kda::ptx::mbar_arrive(&bar);
    __syncthreads();
    const long long t0 = clock64();
    const bool done = kda::ptx::mbar_wait(&bar, 0, budget);
    const long long t1 = clock64();
    if (threadIdx.x == 0) {
        *ok = done ? 1u : 0u;
        *cycles = t1 - t0;
    }
}

// Returns a cudaError_t; ok / cycles are host pointers.
extern "C" int wait_probe_run(int mode, long long budget, unsigned *ok, long long *cycles) {
    unsigned *d_ok = nullptr;
    long long *d_cy = nullptr;
    cudaError_t e = cudaMalloc(&d_ok, sizeof(unsigned));
    if (e == cudaSuccess) e = cudaMalloc(&d_cy, sizeof(long long));
    if (e == cudaSuccess) {
        wait_probe_kernel<<<1, 32>>>(mode, budget, d_ok, d_cy);
        e = cudaGetLastError();
    }
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e == cudaSuccess) e = cudaMemcpy(ok, d_ok, sizeof(unsigned), cudaMemcpyDeviceToHost);
    if (e == cudaSuccess) e = cudaMemcpy(cycles, d_cy, sizeof(long long), cudaMemcpyDeviceToHost);
    cudaFree(d_ok);
    cudaFree(d_cy);
    return (int)e;
}
