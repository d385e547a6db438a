// Test-only check of the library's tcgen05 wrappers (kda_umma.cuh): one CTA
// multiplies A [M x K] by B [N x K]^T on the tensor cores (kind::tf32, A from
// shared memory or from tensor memory) and dumps all 128 TMEM lanes of D.
// Built by tests/test_umma.py with nvcc into a temporary library.
#include <cuda_runtime.h>

#include <cstdint>

#include "kda_ptx.cuh"
#include "kda_umma.cuh"

using namespace kda;

constexpr int KMAX = 64, NMAX = 128;
constexpr uint32_t A_BYTES = 128 * KMAX * 4;   // 32 KB
constexpr uint32_t B_BYTES = NMAX * KMAX * 4;  // 32 KB
constexpr uint32_t SMEM = 232448;              // whole opt-in carve-out: every address in range

__global__ void __launch_bounds__(128, 1)
umma_probe_kernel(const float *A, const float *B, float *D, int M, int N, int K, int mode,
                  unsigned *status) {
    extern __shared__ __align__(1024) unsigned char sm[];
    unsigned char *sA = sm;
    unsigned char *sB = sm + A_BYTES;
    uint64_t *mbar = reinterpret_cast<uint64_t *>(sm + A_BYTES + B_BYTES);
    uint32_t *slot = reinterpret_cast<uint32_t *>(sm + A_BYTES + B_BYTES + 16);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool a_tmem = mode & 1, swap = mode & 2;
    const uint32_t kbytes = K * 4;

    for (int e = tid; e < 128 * K; e += 128) {
        const int r = e / K, k = e % K;
        *reinterpret_cast<float *>(sA + umma::kmajor_offset(r, k, 4, kbytes)) =
            r < M ? A[r * K + k] : 0.f;
    }
    for (int e = tid; e < N * K; e += 128) {
        const int r = e / K, k = e % K;
        *reinterpret_cast<float *>(sB + umma::kmajor_offset(r, k, 4, kbytes)) = B[r * K + k];
    }
    if (tid == 0) {
        ptx::mbar_init(mbar, 1);
        ptx::fence_mbar_init();
    }
    if (warp == 0) {
        umma::tmem_alloc(slot, 256);
        umma::tmem_relinquish();
    }
    umma::fence_smem_to_async();
    umma::fence_before_sync();
    __syncthreads();
    umma::fence_after_sync();
    const uint32_t tbase = *slot;
    const uint32_t acol = 128;  // A (when in TMEM) at columns [128, 128 + K)

    if (a_tmem) {  // lane = row of A
        const int row = warp * 32 + lane;
        for (int k = 0; k < K; k += 8) {
            float v[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] = row < M ? A[row * K + k + i] : 0.f;
            umma::st_x8(umma::taddr(tbase, warp * 32, acol + k), v);
        }
        umma::wait_st();
    }
    umma::fence_before_sync();
    __syncthreads();
    umma::fence_after_sync();

    if (tid == 0) {
        const uint32_t idesc = umma::instr_desc(M, N, umma::kFmtTF32);
        const uint32_t lbo = swap ? 8 * kbytes : 128, sbo = swap ? 128 : 8 * kbytes;
        const uint32_t a0 = ptx::smem_u32(sA), b0 = ptx::smem_u32(sB);
        for (int ks = 0; ks < K / 8; ++ks) {
            const uint64_t bd = umma::smem_desc(b0 + ks * 256, lbo, sbo);
            if (a_tmem)
                umma::mma_ts(tbase, umma::taddr(tbase, 0, acol + ks * 8), bd, idesc, ks > 0);
            else
                umma::mma_ss(tbase, umma::smem_desc(a0 + ks * 256, lbo, sbo), bd, idesc, ks > 0, 1);
        }
        umma::commit(mbar);
    }
    if (!ptx::mbar_wait(mbar, 0, 2000000000LL)) {
        if (lane == 0) atomicOr(status, 1u);
    }
    umma::fence_after_sync();
    const int row = warp * 32 + lane;
    for (int c = 0; c < N; c += 8) {
        float v[8];
        umma::ld_x8(umma::taddr(tbase, warp * 32, c), v);
        umma::wait_ld();
#pragma unroll
        for (int i = 0; i < 8; ++i) D[row * N + c + i] = v[i];
    }
    umma::fence_before_sync();
    __syncthreads();
    if (warp == 0) umma::tmem_dealloc(tbase, 256);
}

extern "C" int umma_probe_run(const float *hA, const float *hB, float *hD, int M, int N, int K,
                              int mode) {
    if (K % 8 || K > KMAX || N % 16 || N > NMAX || (M != 64 && M != 128)) return -1;
    float *A, *B, *D;
    unsigned *st;
    if (cudaMalloc(&A, 128 * K * 4) || cudaMalloc(&B, N * K * 4) || cudaMalloc(&D, 128 * N * 4) ||
        cudaMalloc(&st, 4))
        return -2;
    cudaMemcpy(A, hA, M * K * 4, cudaMemcpyHostToDevice);
    cudaMemcpy(B, hB, N * K * 4, cudaMemcpyHostToDevice);
    cudaMemset(D, 0, 128 * N * 4);
    cudaMemset(st, 0, 4);
    cudaFuncSetAttribute(umma_probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
    umma_probe_kernel<<<1, 128, SMEM>>>(A, B, D, M, N, K, mode, st);
    cudaError_t e = cudaDeviceSynchronize();
    unsigned status = 0;
    cudaMemcpy(&status, st, 4, cudaMemcpyDeviceToHost);
    cudaMemcpy(hD, D, 128 * N * 4, cudaMemcpyDeviceToHost);
    cudaFree(A);
    cudaFree(B);
    cudaFree(D);
    cudaFree(st);
    if (e != cudaSuccess) return 100 + (int)e;
    return (int)status;
}
