// Chunked KDA prefill on CUDA cores (SIMT): the straightforward GPU form of
// the chunkwise WY / UT recurrence of "GLM-5.3 deep dive", section 8.2.5
// (Eq. 6-9). It is the test double for the tensor-core prefill and the
// reference point for its performance.
//
// One CTA owns one (stream m, head h, half of the value columns) and walks the
// sequence chunk by chunk (C = 64 tokens), keeping its 128 x 64 slice of the
// state in shared memory (FP32). Per chunk, with per-channel cumulative
// log-decay G_r = sum_{t <= r} log alpha_t (inclusive, from the chunk start):
//
//   A  = StrictTril(Diag(beta) (e^G * K)(e^-G * K)^T)      64 x 64
//   P  = Tril((e^G * Q)(e^-G * K)^T)                        64 x 64
//   M  = (I + A)^-1 Diag(beta)                              forward substitution
//   Delta = M (V - (e^G * K) S)                             = U - W S of Eq. 7-8
//   O  = scale ((e^G * Q) S + P Delta)                      Eq. 9
//   S  = Diag(e^{G_C}) S + (e^{G_C - G} * K)^T Delta        Eq. 8
//
// Numerics. e^{-G} overflows FP32 once a channel's log-decay summed over the
// chunk passes about -88. The factors are therefore taken relative to the
// end of each 16-token block (g_R = G at the last token of block R):
//   e^{G_r - G_i} = e^{G_r - g_R} . e^{g_R - g_I} . e^{g_I - G_i}
// for token r in block R and i in block I <= R. The middle factor and the
// last one are <= 1; the first is >= 1 but bounded by e^{-(sum of 16
// log-decays)}, which stays inside FP32 whenever every per-token log-decay is
// above -5.4 (the model's gate keeps it above -5; section 8.2.3 ties the -5
// floor to 16-token blocks in exactly this way).
//
// Delta is formed as M (V - (e^G K) S): the same value as U - W S with
// U = M V and W = M (e^G K) (associativity), with one 64 x 128 product less.
// A ragged last chunk is padded with alpha = 1, beta = 0 and zero q, k, v,
// which leaves the state and the real outputs unchanged.

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/kda.h"
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int DK = kHeadDim;
constexpr int C = 64;        // tokens per chunk
constexpr int NB = C / 16;   // 16-token blocks per chunk
constexpr int DVS = 64;      // value columns per CTA
constexpr int NT = 256;
constexpr float kL2Eps = 1e-6f;

// shared-memory layout (floats)
constexpr int OFF_S = 0;                     // [DK][DVS]  state slice
constexpr int OFF_K = OFF_S + DK * DVS;      // [C][DK]    K -> KL -> Kd
constexpr int OFF_Q = OFF_K + C * DK;        // [C][DK]    Q -> QL -> Qd
constexpr int OFF_G = OFF_Q + C * DK;        // [C][DK]    log a -> G -> Kc -> Kdec
constexpr int OFF_V = OFF_G + C * DK;        // [C][DVS]   V -> Y = V - Kd S
constexpr int OFF_A = OFF_V + C * DVS;       // [C][C]     A -> M
constexpr int OFF_P = OFF_A + C * C;         // [C][C]     P
constexpr int OFF_D = OFF_P + C * C;         // [C][DVS]   Delta
constexpr int OFF_GE = OFF_D + C * DVS;      // [NB][DK]   g_R
constexpr int OFF_F = OFF_GE + NB * DK;      // [NB][NB][DK] e^{g_R - g_I}
constexpr int OFF_EG = OFF_F + NB * NB * DK; // [NB][DK]   e^{g_R}
constexpr int OFF_ED = OFF_EG + NB * DK;     // [NB][DK]   e^{g_last - g_R}
constexpr int OFF_B = OFF_ED + NB * DK;      // [C]        beta
constexpr int OFF_ROW = OFF_B + C;           // [C]        forward-substitution row
constexpr int SMEM_FLOATS = OFF_ROW + C;
constexpr int SMEM_BYTES = SMEM_FLOATS * 4;

__device__ __forceinline__ float load_in(const float *p) { return __ldg(p); }
__device__ __forceinline__ float load_in(const __nv_bfloat16 *p) {
    return __bfloat162float(*p);
}

// out[r][j] (rows r0..r0+3, cols j0..j0+3) = sum_k a[r][k] b[k][j]
template <int K>
__device__ __forceinline__ void mm4x4(const float *a, int lda, const float *b, int ldb, int r0,
                                      int j0, float (&acc)[4][4]) {
#pragma unroll 4
    for (int k = 0; k < K; ++k) {
        const float4 bv = *reinterpret_cast<const float4 *>(b + k * ldb + j0);
#pragma unroll
        for (int rr = 0; rr < 4; ++rr) {
            const float av = a[(r0 + rr) * lda + k];
            acc[rr][0] = fmaf(av, bv.x, acc[rr][0]);
            acc[rr][1] = fmaf(av, bv.y, acc[rr][1]);
            acc[rr][2] = fmaf(av, bv.z, acc[rr][2]);
            acc[rr][3] = fmaf(av, bv.w, acc[rr][3]);
        }
    }
}

template <typename TQ>
__global__ void __launch_bounds__(NT, 1) kda_prefill_simt_kernel(const PrefillArgs a) {
    extern __shared__ __align__(16) float sm[];
    float *sS = sm + OFF_S, *sK = sm + OFF_K, *sQ = sm + OFF_Q, *sG = sm + OFF_G;
    float *sV = sm + OFF_V, *sA = sm + OFF_A, *sP = sm + OFF_P, *sD = sm + OFF_D;
    float *sGe = sm + OFF_GE, *sF = sm + OFF_F, *sEg = sm + OFF_EG, *sEd = sm + OFF_ED;
    float *sB = sm + OFF_B, *sRow = sm + OFF_ROW;

    const int half = blockIdx.x, h = blockIdx.y, m = blockIdx.z;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int H = a.H, T = a.T;
    const TQ *q = static_cast<const TQ *>(a.q);
    const TQ *k = static_cast<const TQ *>(a.k);
    const TQ *v = static_cast<const TQ *>(a.v);
    float *state = a.state + ((size_t)m * H + h) * DK * DK + half * DVS;

    // state slice in
    for (int e = tid; e < DK * DVS; e += NT) sS[e] = state[(e / DVS) * DK + e % DVS];

    // thread tiles for the 64 x 64 products: rows tr..tr+3, cols tc..tc+3
    const int tr = (tid / 16) * 4, tc = (tid % 16) * 4;

    for (int c0 = 0; c0 < T; c0 += C) {
        const int L = min(C, T - c0);
        __syncthreads();

        // 1. load and L2-normalise q, k rows; log alpha, v slice, beta
        for (int rr = 0; rr < C / 8; ++rr) {
            const int r = warp * (C / 8) + rr;
            float qv[4], kv[4];
            float sq = 0.f, sk = 0.f;
            if (r < L) {
                const size_t base = (((size_t)m * T + c0 + r) * H + h) * DK + lane * 4;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    qv[e] = load_in(q + base + e);
                    kv[e] = load_in(k + base + e);
                    sq += qv[e] * qv[e];
                    sk += kv[e] * kv[e];
                }
            } else {
#pragma unroll
                for (int e = 0; e < 4; ++e) qv[e] = kv[e] = 0.f;
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                sq += __shfl_xor_sync(0xffffffffu, sq, off);
                sk += __shfl_xor_sync(0xffffffffu, sk, off);
            }
            const float rq = 1.0f / sqrtf(sq + kL2Eps), rk = 1.0f / sqrtf(sk + kL2Eps);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                sQ[r * DK + lane * 4 + e] = qv[e] * rq;
                sK[r * DK + lane * 4 + e] = kv[e] * rk;
            }
        }
        for (int e = tid; e < C * DK; e += NT) {
            const int r = e / DK;
            sG[e] = r < L ? logf(__ldg(a.alpha + (((size_t)m * T + c0 + r) * H + h) * DK + e % DK))
                          : 0.f;
        }
        for (int e = tid; e < C * DVS; e += NT) {
            const int r = e / DVS;
            sV[e] = r < L ? load_in(v + (((size_t)m * T + c0 + r) * H + h) * DK + half * DVS + e % DVS)
                          : 0.f;
        }
        if (tid < C) sB[tid] = tid < L ? __ldg(a.beta + ((size_t)m * T + c0 + tid) * H + h) : 0.f;
        __syncthreads();

        // 2. cumulative log-decay per channel, and the block ends g_R
        if (tid < DK) {
            float g = 0.f;
            for (int r = 0; r < C; ++r) {
                g += sG[r * DK + tid];
                sG[r * DK + tid] = g;
                if ((r & 15) == 15) sGe[(r >> 4) * DK + tid] = g;
            }
        }
        __syncthreads();

        // 3. per-channel factors: e^{g_R - g_I} (I <= R), e^{g_R}, e^{g_last - g_R}
        for (int e = tid; e < NB * DK; e += NT) {
            const int R = e / DK, c = e % DK;
            const float gR = sGe[e];
            for (int I = 0; I < NB; ++I)
                sF[(R * NB + I) * DK + c] = I <= R ? expf(gR - sGe[I * DK + c]) : 0.f;
            sEg[e] = expf(gR);
            sEd[e] = expf(sGe[(NB - 1) * DK + c] - gR);
        }
        // 4. local factors: KL = K e^{G - g_R} (>= 1), QL likewise, Kc = K e^{g_R - G} (<= 1)
        for (int e = tid; e < C * DK; e += NT) {
            const int R = (e / DK) >> 4;
            const float x = sG[e] - sGe[R * DK + e % DK];  // >= 0
            const float up = expf(x), down = expf(-x);
            const float kk = sK[e];
            sK[e] = kk * up;
            sQ[e] *= up;
            sG[e] = kk * down;
        }
        __syncthreads();

        // 5. A (strict lower, times beta_r) and P (lower with diagonal);
        //    thread: row r = tid / 4, column block I = tid % 4
        {
            const int r = tid >> 2, I = tid & 3, R = r >> 4;
            float acc_a[16], acc_p[16];
#pragma unroll
            for (int ii = 0; ii < 16; ++ii) acc_a[ii] = acc_p[ii] = 0.f;
            if (I <= R) {
                const float *F = sF + (R * NB + I) * DK;
                for (int c = 0; c < DK; ++c) {
                    const float f = F[c];
                    const float kl = sK[r * DK + c] * f, ql = sQ[r * DK + c] * f;
#pragma unroll
                    for (int ii = 0; ii < 16; ++ii) {
                        const float kc = sG[(I * 16 + ii) * DK + c];
                        acc_a[ii] = fmaf(kl, kc, acc_a[ii]);
                        acc_p[ii] = fmaf(ql, kc, acc_p[ii]);
                    }
                }
            }
            const float br = sB[r];
#pragma unroll
            for (int ii = 0; ii < 16; ++ii) {
                const int i = I * 16 + ii;
                sA[r * C + i] = i < r ? br * acc_a[ii] : 0.f;
                sP[r * C + i] = i <= r ? acc_p[ii] : 0.f;
            }
        }
        __syncthreads();

        // 6. M = (I + A)^-1 Diag(beta) by forward substitution, row by row
        //    (warps 0-1; row r overwrites A's row r once it is no longer read)
        if (tid < C) {
            for (int r = 0; r < C; ++r) {
                const int j = tid;
                float x = j == r ? sB[r] : 0.f;
                for (int i = j; i < r; ++i) x = fmaf(-sA[r * C + i], sA[i * C + j], x);
                sRow[j] = j <= r ? x : 0.f;
                asm volatile("bar.sync 1, 64;" ::: "memory");
                sA[r * C + j] = sRow[j];
                asm volatile("bar.sync 1, 64;" ::: "memory");
            }
        }
        // 7. Kd = KL e^{g_R} (= K e^G), Qd = QL e^{g_R}, Kdec = Kc e^{g_last - g_R}
        //    (warps 2-7, while warps 0-1 run the substitution)
        if (tid >= C) {
            for (int e = tid - C; e < C * DK; e += NT - C) {
                const int R = (e / DK) >> 4, c = e % DK;
                sK[e] *= sEg[R * DK + c];
                sQ[e] *= sEg[R * DK + c];
                sG[e] *= sEd[R * DK + c];
            }
        }
        __syncthreads();

        // 8. Y = V - Kd S (in place over V) and O1 = Qd S (kept in registers)
        float o1[4][4] = {}, y[4][4] = {};
        mm4x4<DK>(sK, DK, sS, DVS, tr, tc, y);
        mm4x4<DK>(sQ, DK, sS, DVS, tr, tc, o1);
        __syncthreads();
#pragma unroll
        for (int rr = 0; rr < 4; ++rr)
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) sV[(tr + rr) * DVS + tc + jj] -= y[rr][jj];
        __syncthreads();

        // 9. Delta = M Y
        {
            float d[4][4] = {};
            mm4x4<C>(sA, C, sV, DVS, tr, tc, d);
#pragma unroll
            for (int rr = 0; rr < 4; ++rr)
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) sD[(tr + rr) * DVS + tc + jj] = d[rr][jj];
        }
        __syncthreads();

        // 10. O = scale (Qd S + P Delta), rows of real tokens only
        mm4x4<C>(sP, C, sD, DVS, tr, tc, o1);
#pragma unroll
        for (int rr = 0; rr < 4; ++rr) {
            const int r = tr + rr;
            if (r < L) {
                float4 *op = reinterpret_cast<float4 *>(
                    a.o + (((size_t)m * T + c0 + r) * H + h) * DK + half * DVS + tc);
                *op = make_float4(a.scale * o1[rr][0], a.scale * o1[rr][1], a.scale * o1[rr][2],
                                  a.scale * o1[rr][3]);
            }
        }

        // 11. S = Diag(e^{g_last}) S + Kdec^T Delta   (thread: 8 rows x 4 cols)
        {
            const int sr = (tid / 16) * 8;
            float acc[8][4];
#pragma unroll
            for (int rr = 0; rr < 8; ++rr) {
                const float gam = sEg[(NB - 1) * DK + sr + rr];
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) acc[rr][jj] = gam * sS[(sr + rr) * DVS + tc + jj];
            }
#pragma unroll 4
            for (int i = 0; i < C; ++i) {
                const float4 dv = *reinterpret_cast<const float4 *>(sD + i * DVS + tc);
#pragma unroll
                for (int rr = 0; rr < 8; ++rr) {
                    const float kd = sG[i * DK + sr + rr];
                    acc[rr][0] = fmaf(kd, dv.x, acc[rr][0]);
                    acc[rr][1] = fmaf(kd, dv.y, acc[rr][1]);
                    acc[rr][2] = fmaf(kd, dv.z, acc[rr][2]);
                    acc[rr][3] = fmaf(kd, dv.w, acc[rr][3]);
                }
            }
            __syncthreads();  // every read of the old S is done
#pragma unroll
            for (int rr = 0; rr < 8; ++rr)
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) sS[(sr + rr) * DVS + tc + jj] = acc[rr][jj];
        }
    }
    __syncthreads();
    for (int e = tid; e < DK * DVS; e += NT) state[(e / DVS) * DK + e % DVS] = sS[e];
}

}  // namespace

cudaError_t launch_prefill_simt(const PrefillArgs &a, int qkv_dtype, cudaStream_t stream) {
    const dim3 grid(DK / DVS, a.H, a.M);
    if (qkv_dtype == KDA_BF16) {
        cudaError_t e = cudaFuncSetAttribute(kda_prefill_simt_kernel<__nv_bfloat16>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
        if (e != cudaSuccess) return e;
        kda_prefill_simt_kernel<__nv_bfloat16><<<grid, NT, SMEM_BYTES, stream>>>(a);
    } else {
        cudaError_t e = cudaFuncSetAttribute(kda_prefill_simt_kernel<float>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
        if (e != cudaSuccess) return e;
        kda_prefill_simt_kernel<float><<<grid, NT, SMEM_BYTES, stream>>>(a);
    }
    return cudaGetLastError();
}

}  // namespace kda
