// Chunked KDA prefill on the 5th-generation tensor cores (tcgen05, TF32
// operands, FP32 accumulators in tensor memory).
//
// What it computes: the chunkwise WY / UT form of the KDA recurrence
// ("GLM-5.3 deep dive", section 8.2.5, Eq. 6-9), the same result as the CUDA
// core kernel in kda_prefill_simt.cu. Per chunk of C = 64 tokens, with the
// per-channel cumulative log-decay G (inclusive, from the chunk start):
//   A  = StrictTril(Diag(beta) (e^G K)(e^-G K)^T),  P = Tril((e^G Q)(e^-G K)^T)
//   M  = (I + A)^-1 Diag(beta)
//   Delta = M (V - (e^G K) S)                          (= U - W S)
//   O  = scale ((e^G Q) S + P Delta)
//   S  = Diag(e^{G_63}) S + (e^{G_63 - G} K)^T Delta
//
// Organisation. One CTA (256 threads) owns one (stream, head) and walks its
// chunks in order. The state lives in tensor memory for the whole sequence,
// transposed (lane = value channel j, column = key channel i) and in FP32:
// it is the accumulator of the state update and, read as TF32, the A operand
// (from tensor memory) of the products with S. Every MMA has M = 128 rows:
//   MMA1  D1 = [L0; Lq0; L1; Lq1] [R0 | R1]^T     A and P, diagonal halves
//   MMA2  D2 = [Lo; Lqo] R0^T                      A and P, rows 32-63 x cols 0-31
//   MMA3  D3 = S^T [Kd; Qd]^T                       Y^T = (Kd S)^T and (Qd S)^T
//   MMA4  D4 = Z^T M^T,  Z = V - Y                  Delta^T
//   MMA5  D3[:, 64:] += Delta^T P^T                 O^T
//   MMA6  S^T += Delta^T Kdec,  after S^T *= e^{G_63} per column
// Operand tiles are written by the threads in the K-major core-matrix layout
// (kda_umma.cuh) and read through shared-memory descriptors.
//
// Numerics. Decay factors are taken relative to the middle token of each
// 32-token half (m_b = G_15, G_47): inside a half |G_r - m_b| spans at most 16
// per-token log-decays, which stays inside FP32 for log(alpha) above about
// -5.4 (the model's gate keeps it above -5; section 8.2.3 ties the -5 floor to
// 16-token spans). Rows of the second half against columns of the first use
// e^{G_r - m_0} <= 1 on the left and the first half's own right factor.
// Every factor of Kd, Qd, Kdec and the state decay is <= 1.
//
// The unit lower-triangular inverse is taken on CUDA cores in 16 x 16 blocks:
// diagonal blocks by forward substitution (one lane per column), off-diagonal
// blocks level by level from the block recurrence T_RI = -T_RR sum_Q A_RQ T_QI.
//
// Inputs of the next chunk are loaded into registers while the current one is
// processed. Every mbarrier wait is bounded; on timeout the kernel sets the
// device error word (kda_device_error) and stops.

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/kda.h"
#include "kda_internal.cuh"
#include "kda_ptx.cuh"
#include "kda_umma.cuh"

namespace kda {

__device__ unsigned int g_prefill_error;

namespace {

constexpr int DK = kHeadDim;
constexpr int C = 64;
constexpr int NT = 256;
constexpr float kL2Eps = 1e-6f;
constexpr long long kWaitBudget = 4000000000LL;

// operand tiles (bytes), K-major core-matrix layout
constexpr uint32_t KB128 = DK * 4;  // one row of a K = 128 tile
constexpr uint32_t KB64 = C * 4;    // one row of a K = 64 tile
// phase-1 tiles
constexpr uint32_t T_LO = 0;                       // [Lo; Lqo]      64 x 128 (+64 rows overlap LA)
constexpr uint32_t T_LA = T_LO + 64 * KB128;       // [L0;Lq0;L1;Lq1] 128 x 128
constexpr uint32_t T_RB = T_LA + 128 * KB128;      // [R0; R1]        64 x 128
constexpr uint32_t PH1_END = T_RB + 64 * KB128;    // 131072
// phase-2 tiles (overlay phase-1 after MMA1/2 complete)
constexpr uint32_t T_KQ = 0;                       // [Kd; Qd]       128 x 128
constexpr uint32_t T_KDEC = T_KQ + 128 * KB128;    // Kdec^T          128 x 64
constexpr uint32_t T_M = T_KDEC + 128 * KB64;      // M               64 x 64
constexpr uint32_t T_P = T_M + 64 * KB64;          // P               64 x 64
constexpr uint32_t T_A = T_P + 64 * KB64;          // A (plain [64][68] FP32)
constexpr int LDA = 68;
constexpr uint32_t T_T = T_A + 64 * LDA * 4;       // T = (I + A)^-1 (plain [64][68] FP32)
constexpr uint32_t T_X = T_T + 64 * LDA * 4;       // scratch: up to 3 blocks of 16 x 16
constexpr int LDK = 144;                           // Kdec staging row: 128 + 16 (bank shift)
constexpr uint32_t T_KST = T_X + 3 * 256 * 4;      // Kdec, token-major staging [64][LDK]
constexpr uint32_t PH2_END = T_KST + 64 * LDK * 4;
constexpr uint32_t TILES = PH2_END > PH1_END ? PH2_END : PH1_END;
// small buffers (bytes)
constexpr uint32_t S_NORM = TILES;                 // [2][8][64] partial sums of q^2, k^2
constexpr uint32_t S_BETA = S_NORM + 2 * 8 * 64 * 4;
constexpr uint32_t S_GAM = S_BETA + 64 * 4;        // [128] e^{G_63}
constexpr uint32_t S_BAR = S_GAM + 128 * 4;        // 4 mbarriers
constexpr uint32_t S_SLOT = S_BAR + 4 * 8;
constexpr uint32_t SMEM_BYTES = S_SLOT + 16;

// TMEM columns
constexpr uint32_t TM_S = 0, TM_D3 = 128, TM_Z = 256, TM_D4 = 320, TM_D1 = 384, TM_D2 = 448;
constexpr uint32_t TM_COLS = 512;

__device__ __forceinline__ void raise_error(unsigned int code) { atomicOr(&g_prefill_error, code); }

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float lg2(float x) {
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// 4 consecutive input elements -> floats
__device__ __forceinline__ void load4(const __nv_bfloat16 *p, float (&f)[4]) {
    const uint2 u = __ldg(reinterpret_cast<const uint2 *>(p));
    f[0] = __uint_as_float(u.x << 16);
    f[1] = __uint_as_float(u.x & 0xffff0000u);
    f[2] = __uint_as_float(u.y << 16);
    f[3] = __uint_as_float(u.y & 0xffff0000u);
}
__device__ __forceinline__ void load4(const float *p, float (&f)[4]) {
    const float4 u = __ldg(reinterpret_cast<const float4 *>(p));
    f[0] = u.x;
    f[1] = u.y;
    f[2] = u.z;
    f[3] = u.w;
}
__device__ __forceinline__ float load1(const __nv_bfloat16 *p) { return __bfloat162float(*p); }
__device__ __forceinline__ float load1(const float *p) { return __ldg(p); }

// FP32 -> TF32, round to nearest (ties away from zero), by adding half a
// TF32 ulp to the magnitude bits and clearing the 13 bits TF32 drops. The
// tensor cores read an FP32 operand as TF32 by ignoring those bits, a biased
// truncation; operands written here are rounded first so their errors stay
// unbiased. (Inputs are finite; nothing here rounds into inf or NaN.)
__device__ __forceinline__ float tf32r(float x) {
    return __uint_as_float((__float_as_uint(x) + 0x1000u) & 0xFFFFE000u);
}

__device__ __forceinline__ void st_tile4(unsigned char *tile, uint32_t row, uint32_t c4,
                                         uint32_t kbytes, float a, float b, float c, float d) {
    *reinterpret_cast<float4 *>(tile + (row >> 3) * (8u * kbytes) + c4 * 128u + (row & 7u) * 16u) =
        make_float4(tf32r(a), tf32r(b), tf32r(c), tf32r(d));
}
__device__ __forceinline__ void st_tile1(unsigned char *tile, uint32_t row, uint32_t k,
                                         uint32_t kbytes, float v) {
    *reinterpret_cast<float *>(tile + umma::kmajor_offset(row, k, 4, kbytes)) = tf32r(v);
}

// Per-thread inputs of one chunk, kept exactly as loaded (no arithmetic on
// them until the chunk is processed, so the loads overlap the previous
// chunk's work): rows r = 8 rg + rr, channels 4 c4 + e.
template <typename TQ> struct Raw;
template <> struct Raw<__nv_bfloat16> {
    typedef uint2 Q4;              // 4 BF16
    typedef unsigned short V1;     // 1 BF16
    __device__ __forceinline__ static Q4 load4(const __nv_bfloat16 *p) {
        return __ldg(reinterpret_cast<const uint2 *>(p));
    }
    __device__ __forceinline__ static void widen4(const Q4 &u, float (&f)[4]) {
        f[0] = __uint_as_float(u.x << 16);
        f[1] = __uint_as_float(u.x & 0xffff0000u);
        f[2] = __uint_as_float(u.y << 16);
        f[3] = __uint_as_float(u.y & 0xffff0000u);
    }
    __device__ __forceinline__ static V1 load1(const __nv_bfloat16 *p) {
        return __ldg(reinterpret_cast<const unsigned short *>(p));
    }
    __device__ __forceinline__ static float widen1(V1 v) { return __uint_as_float((uint32_t)v << 16); }
    __device__ __forceinline__ static V1 zero1() { return 0; }
};
template <> struct Raw<float> {
    typedef float4 Q4;
    typedef float V1;
    __device__ __forceinline__ static Q4 load4(const float *p) {
        return __ldg(reinterpret_cast<const float4 *>(p));
    }
    __device__ __forceinline__ static void widen4(const Q4 &u, float (&f)[4]) {
        f[0] = u.x;
        f[1] = u.y;
        f[2] = u.z;
        f[3] = u.w;
    }
    __device__ __forceinline__ static V1 load1(const float *p) { return __ldg(p); }
    __device__ __forceinline__ static float widen1(V1 v) { return v; }
    __device__ __forceinline__ static V1 zero1() { return 0.f; }
};

template <typename TQ>
struct ChunkRegs {
    typename Raw<TQ>::Q4 q[8], k[8];
    float4 al[8];                      // alpha (linear); 1 on padding rows
    typename Raw<TQ>::V1 v[32];        // v[r][j], r = 32 hw + i, j = 32 q4 + lane
    float beta;                        // beta of token tid (tid < 64)
};

template <typename TQ>
__device__ __forceinline__ void load_chunk(ChunkRegs<TQ> &R, const PrefillArgs &a, int m, int h,
                                           int c0, int rr, int c4, int q4, int hw, int lane, int tid) {
    using RW = Raw<TQ>;
    const TQ *q = static_cast<const TQ *>(a.q);
    const TQ *k = static_cast<const TQ *>(a.k);
    const TQ *v = static_cast<const TQ *>(a.v);
    const int T = a.T, H = a.H;
#pragma unroll
    for (int rg = 0; rg < 8; ++rg) {
        const int t = c0 + 8 * rg + rr;
        if (t < T) {
            const size_t base = (((size_t)m * T + t) * H + h) * DK + 4 * c4;
            R.q[rg] = RW::load4(q + base);
            R.k[rg] = RW::load4(k + base);
            R.al[rg] = __ldg(reinterpret_cast<const float4 *>(a.alpha + base));
        } else {
            R.q[rg] = R.k[rg] = typename RW::Q4{};
            R.al[rg] = make_float4(1.f, 1.f, 1.f, 1.f);
        }
    }
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        const int t = c0 + 32 * hw + i;
        R.v[i] = t < T ? RW::load1(v + (((size_t)m * T + t) * H + h) * DK + 32 * q4 + lane)
                       : RW::zero1();
    }
    if (tid < C) {
        const int t = c0 + tid;
        R.beta = t < T ? __ldg(a.beta + ((size_t)m * T + t) * H + h) : 0.f;
    }
}

template <typename TQ>
__global__ void __launch_bounds__(NT, 1) kda_prefill_tc_kernel(const PrefillArgs a) {
    extern __shared__ __align__(1024) unsigned char sm[];
    float *sNorm = reinterpret_cast<float *>(sm + S_NORM);
    float *sBeta = reinterpret_cast<float *>(sm + S_BETA);
    float *sGam = reinterpret_cast<float *>(sm + S_GAM);
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm + S_BAR);  // 0: MMA1/2, 1: MMA3, 2: MMA4, 3: MMA5/6
    uint32_t *slot = reinterpret_cast<uint32_t *>(sm + S_SLOT);
    float *sA = reinterpret_cast<float *>(sm + T_A);
    float *sT = reinterpret_cast<float *>(sm + T_T);
    float *sX = reinterpret_cast<float *>(sm + T_X);
    float *sKst = reinterpret_cast<float *>(sm + T_KST);

    const int h = blockIdx.x % a.H, m = blockIdx.x / a.H;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int rr = lane >> 2, qq = lane & 3, c4 = 4 * warp + qq;  // token-channel mapping
    const int q4 = warp & 3, hw = warp >> 2;                        // TMEM lane quarter, half
    const int j = 32 * q4 + lane;                                   // value channel (TMEM lane)
    const int T = a.T;
    const uint32_t sbase = ptx::smem_u32(sm);

    if (tid == 0) {
        for (int b = 0; b < 4; ++b) ptx::mbar_init(&bar[b], 1);
        ptx::fence_mbar_init();
    }
    if (warp == 0) {
        umma::tmem_alloc(slot, TM_COLS);
        umma::tmem_relinquish();
    }
    umma::fence_before_sync();
    __syncthreads();
    umma::fence_after_sync();
    const uint32_t tb = *slot;
    const uint32_t tq = tb + ((uint32_t)(32 * q4) << 16);  // this warp's TMEM lane quarter

    // state in: S^T[j][i] = S[i][j]; this thread: lane j, key channels [64 hw, 64 hw + 64)
    float *state = a.state + ((size_t)m * a.H + h) * DK * DK;
    for (int c = 64 * hw; c < 64 * hw + 64; c += 8) {
        float v8[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) v8[e] = state[(size_t)(c + e) * DK + j];
        umma::st_x8(tq + TM_S + c, v8);
    }
    umma::wait_st();

    using RW = Raw<TQ>;
    ChunkRegs<TQ> R;
    load_chunk<TQ>(R, a, m, h, 0, rr, c4, q4, hw, lane, tid);

    const uint32_t id128 = umma::instr_desc(128, 128, umma::kFmtTF32);
    const uint32_t id64 = umma::instr_desc(128, 64, umma::kFmtTF32);
    const uint32_t id32 = umma::instr_desc(128, 32, umma::kFmtTF32);
    bool ok = true;
    int phase = 0;

    for (int c0 = 0; c0 < T && ok; c0 += C, phase ^= 1) {
        // ---------------------------------------------------------- 1. decay, norms
        // cumulative log2-decay over the chunk's rows (rows across lanes rr, then rg)
        float G[8][4], qf[8][4], kf[8][4];
#pragma unroll
        for (int rg = 0; rg < 8; ++rg) {
            RW::widen4(R.q[rg], qf[rg]);
            RW::widen4(R.k[rg], kf[rg]);
            G[rg][0] = lg2(R.al[rg].x);
            G[rg][1] = lg2(R.al[rg].y);
            G[rg][2] = lg2(R.al[rg].z);
            G[rg][3] = lg2(R.al[rg].w);
        }
        float carry[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int rg = 0; rg < 8; ++rg) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                float x = G[rg][e];
#pragma unroll
                for (int d = 4; d < 32; d <<= 1) {
                    const float y = __shfl_up_sync(0xffffffffu, x, d);
                    if (lane >= d) x += y;
                }
                x += carry[e];
                G[rg][e] = x;
                carry[e] = __shfl_sync(0xffffffffu, x, 28 + qq);
            }
        }
        // references: m0 = G_15, m1 = G_47, e63 = G_63 (log2 units), from lanes rr = 7
        float m0[4], m1[4], e63[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            m0[e] = __shfl_sync(0xffffffffu, G[1][e], 28 + qq);
            m1[e] = __shfl_sync(0xffffffffu, G[5][e], 28 + qq);
            e63[e] = carry[e];
        }
        // L2-norm partial sums: 4 channels here, 16 per warp
#pragma unroll
        for (int rg = 0; rg < 8; ++rg) {
            float sq = 0.f, sk = 0.f;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                sq = fmaf(qf[rg][e], qf[rg][e], sq);
                sk = fmaf(kf[rg][e], kf[rg][e], sk);
            }
            sq += __shfl_xor_sync(0xffffffffu, sq, 1);
            sq += __shfl_xor_sync(0xffffffffu, sq, 2);
            sk += __shfl_xor_sync(0xffffffffu, sk, 1);
            sk += __shfl_xor_sync(0xffffffffu, sk, 2);
            if (qq == 0) {
                sNorm[(0 * 8 + warp) * 64 + 8 * rg + rr] = sq;
                sNorm[(1 * 8 + warp) * 64 + 8 * rg + rr] = sk;
            }
        }
        if (tid < C) sBeta[tid] = R.beta;
        if (rr == 0 && warp < 8) {
#pragma unroll
            for (int e = 0; e < 4; ++e) sGam[4 * c4 + e] = ex2(e63[e]);
        }
        __syncthreads();
        float rq[8], rk[8];
#pragma unroll
        for (int rg = 0; rg < 8; ++rg) {
            float sq = 0.f, sk = 0.f;
#pragma unroll
            for (int w = 0; w < 8; ++w) {
                sq += sNorm[(0 * 8 + w) * 64 + 8 * rg + rr];
                sk += sNorm[(1 * 8 + w) * 64 + 8 * rg + rr];
            }
            rq[rg] = 1.0f / sqrtf(sq + kL2Eps);
            rk[rg] = 1.0f / sqrtf(sk + kL2Eps);
        }

        // ---------------------------------------------------------- 2. A / P operands
        // u = e^{G - m_b} (>= 1 in the first quarter of a half, <= 1 after),
        // L = K u, Lq = Q u, R = K / u; rows of the second half also get
        // Lo = L e^{m1 - m0}, Lqo = Lq e^{m1 - m0} (= K e^{G - m0} <= 1).
        float f10[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) f10[e] = ex2(m1[e] - m0[e]);
#pragma unroll
        for (int rg = 0; rg < 8; ++rg) {
            const int r = 8 * rg + rr;
            const bool second = rg >= 4;
            float L[4], Lq[4], Rr[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float x = G[rg][e] - (second ? m1[e] : m0[e]);
                const float u = ex2(x), ui = ex2(-x);
                const float kh = kf[rg][e] * rk[rg], qh = qf[rg][e] * rq[rg];
                L[e] = kh * u;
                Lq[e] = qh * u;
                Rr[e] = kh * ui;
            }
            const int rowL = second ? r + 32 : r, rowLq = second ? r + 64 : r + 32;
            st_tile4(sm + T_LA, rowL, c4, KB128, L[0], L[1], L[2], L[3]);
            st_tile4(sm + T_LA, rowLq, c4, KB128, Lq[0], Lq[1], Lq[2], Lq[3]);
            st_tile4(sm + T_RB, r, c4, KB128, Rr[0], Rr[1], Rr[2], Rr[3]);
            if (second) {
                st_tile4(sm + T_LO, r - 32, c4, KB128, L[0] * f10[0], L[1] * f10[1], L[2] * f10[2],
                         L[3] * f10[3]);
                st_tile4(sm + T_LO, r, c4, KB128, Lq[0] * f10[0], Lq[1] * f10[1], Lq[2] * f10[2],
                         Lq[3] * f10[3]);
            }
        }
        umma::fence_smem_to_async();
        umma::fence_before_sync();
        __syncthreads();
        umma::fence_after_sync();
        if (tid == 0) {
#pragma unroll 1
            for (int ks = 0; ks < DK / 8; ++ks) {
                const uint64_t bd = umma::smem_desc(sbase + T_RB + ks * 256, 128, 8 * KB128);
                umma::mma_ss(tb + TM_D1, umma::smem_desc(sbase + T_LA + ks * 256, 128, 8 * KB128), bd,
                             id64, ks > 0, 1);
                umma::mma_ss(tb + TM_D2, umma::smem_desc(sbase + T_LO + ks * 256, 128, 8 * KB128), bd,
                             id32, ks > 0, 1);
            }
            umma::commit(&bar[0]);
        }
        if (!ptx::mbar_wait(&bar[0], phase, kWaitBudget)) {
            raise_error(1u);
            ok = false;
            break;
        }
        umma::fence_after_sync();

        // ---------------------------------------------------------- 3. A, P from TMEM
        // warp (q4, hw): q4 = 0 A-rows, 1 P-rows of the first half (D1) or, with
        // hw = 1, of rows 32-63 x columns 0-31 (D2); q4 = 2, 3: second half (D1).
        {
            const bool isP = q4 & 1;
            int r, i0;
            uint32_t col;
            bool active = true;
            if (hw == 0) {
                r = (q4 < 2 ? 0 : 32) + lane;
                i0 = q4 < 2 ? 0 : 32;
                col = TM_D1 + i0;
            } else {
                r = 32 + lane;
                i0 = 0;
                col = TM_D2;
                active = q4 < 2;
            }
            if (active) {
                const float br = sBeta[r];
                float d[32];
                umma::ld_x32(tq + col, d);
                umma::wait_ld();
#pragma unroll
                for (int cb = 0; cb < 32; cb += 4) {
                    float v4[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int i = i0 + cb + e;
                        v4[e] = isP ? (i <= r ? d[cb + e] : 0.f) : (i < r ? br * d[cb + e] : 0.f);
                    }
                    if (isP)
                        st_tile4(sm + T_P, r, (i0 + cb) >> 2, KB64, v4[0], v4[1], v4[2], v4[3]);
                    else
                        *reinterpret_cast<float4 *>(sA + r * LDA + i0 + cb) =
                            make_float4(v4[0], v4[1], v4[2], v4[3]);
                }
            } else if (q4 == 3) {  // P rows 0-31, columns 32-63 are zero
#pragma unroll
                for (int cb = 32; cb < 64; cb += 4) st_tile4(sm + T_P, lane, cb >> 2, KB64, 0.f, 0.f, 0.f, 0.f);
            }
        }
        umma::fence_before_sync();
        __syncthreads();  // A, P visible; MMA1/2 operands may now be overwritten

        // ---------------------------------------------------------- 4. state-pass operands
        //   Kd = K e^G = (K u) e^{m_b},   Qd = Q e^G,   Kdec = K e^{G63 - G} = (K / u) e^{G63 - m_b}
        {
            float em0[4], em1[4], ed0[4], ed1[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                em0[e] = ex2(m0[e]);
                em1[e] = ex2(m1[e]);
                ed0[e] = ex2(e63[e] - m0[e]);
                ed1[e] = ex2(e63[e] - m1[e]);
            }
#pragma unroll
            for (int rg = 0; rg < 8; ++rg) {
                const int r = 8 * rg + rr;
                const bool second = rg >= 4;
                float Kd[4], Qd[4], Kc[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float x = G[rg][e] - (second ? m1[e] : m0[e]);
                    const float u = ex2(x), ui = ex2(-x);
                    const float kh = kf[rg][e] * rk[rg], qh = qf[rg][e] * rq[rg];
                    const float em = second ? em1[e] : em0[e];
                    Kd[e] = kh * u * em;
                    Qd[e] = qh * u * em;
                    Kc[e] = kh * ui * (second ? ed1[e] : ed0[e]);
                }
                st_tile4(sm + T_KQ, r, c4, KB128, Kd[0], Kd[1], Kd[2], Kd[3]);
                st_tile4(sm + T_KQ, 64 + r, c4, KB128, Qd[0], Qd[1], Qd[2], Qd[3]);
                *reinterpret_cast<float4 *>(sKst + r * LDK + 4 * c4) =
                    make_float4(Kc[0], Kc[1], Kc[2], Kc[3]);
            }
        }
        __syncthreads();
        // Kdec^T tile (row = key channel c, K = token): 16-byte row segments,
        // 8 consecutive channels per quarter-warp (one core matrix)
#pragma unroll
        for (int it = 0; it < 8; ++it) {
            const int u = it * NT + tid;
            const int c8 = u & 7, kq = (u >> 3) & 15, cg = u >> 7;
            const int c = 8 * cg + c8;
            st_tile4(sm + T_KDEC, c, kq, KB64, sKst[(4 * kq + 0) * LDK + c], sKst[(4 * kq + 1) * LDK + c],
                     sKst[(4 * kq + 2) * LDK + c], sKst[(4 * kq + 3) * LDK + c]);
        }
        umma::fence_smem_to_async();
        umma::fence_before_sync();
        __syncthreads();
        umma::fence_after_sync();
        if (tid == 0) {
#pragma unroll 1
            for (int ks = 0; ks < DK / 8; ++ks)
                umma::mma_ts(tb + TM_D3, tb + TM_S + ks * 8,
                             umma::smem_desc(sbase + T_KQ + ks * 256, 128, 8 * KB128), id128, ks > 0);
            umma::commit(&bar[1]);
        }

        // ---------------------------------------------------------- 5. M = (I + A)^-1 Diag(beta)
        // (runs on CUDA cores while MMA3 is on the tensor cores)
        // 5a. diagonal 16 x 16 blocks, one lane per column: T_bb = (I + A_bb)^-1
        if (warp < 2) {
            const int b = 2 * warp + (lane >> 4), jj = lane & 15, j0 = 16 * b;
            float tcol[16];
#pragma unroll
            for (int r = 0; r < 16; ++r) {
                float x = r == jj ? 1.f : 0.f;
#pragma unroll
                for (int i = 0; i < r; ++i) x = fmaf(-sA[(j0 + r) * LDA + j0 + i], tcol[i], x);
                tcol[r] = r >= jj ? x : 0.f;
            }
#pragma unroll
            for (int r = 0; r < 16; ++r) sT[(j0 + r) * LDA + j0 + jj] = tcol[r];
        }
        __syncthreads();
        // 5b. off-diagonal blocks, level d = R - I at a time:
        //     T_RI = -T_RR X_RI,  X_RI = sum_{Q=I}^{R-1} A_RQ T_QI
        for (int d = 1; d < 4; ++d) {
            const int nblk = 4 - d;
            // unit: block I (R = I + d), row r16, four columns 4 q16 .. + 3
            const int I = tid >> 6, r16 = (tid >> 2) & 15, q16 = tid & 3, Rb = I + d;
            if (I < nblk) {
                float x4[4] = {0.f, 0.f, 0.f, 0.f};
                for (int Q = I; Q < Rb; ++Q) {
#pragma unroll
                    for (int t = 0; t < 16; ++t) {
                        const float av = sA[(16 * Rb + r16) * LDA + 16 * Q + t];
                        const float4 tv =
                            *reinterpret_cast<const float4 *>(sT + (16 * Q + t) * LDA + 16 * I + 4 * q16);
                        x4[0] = fmaf(av, tv.x, x4[0]);
                        x4[1] = fmaf(av, tv.y, x4[1]);
                        x4[2] = fmaf(av, tv.z, x4[2]);
                        x4[3] = fmaf(av, tv.w, x4[3]);
                    }
                }
                *reinterpret_cast<float4 *>(sX + (I * 16 + r16) * 16 + 4 * q16) =
                    make_float4(x4[0], x4[1], x4[2], x4[3]);
            }
            __syncthreads();
            if (I < nblk) {
                float t4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int t = 0; t < 16; ++t) {
                    const float tv = sT[(16 * Rb + r16) * LDA + 16 * Rb + t];
                    const float4 xv = *reinterpret_cast<const float4 *>(sX + (I * 16 + t) * 16 + 4 * q16);
                    t4[0] = fmaf(tv, xv.x, t4[0]);
                    t4[1] = fmaf(tv, xv.y, t4[1]);
                    t4[2] = fmaf(tv, xv.z, t4[2]);
                    t4[3] = fmaf(tv, xv.w, t4[3]);
                }
                *reinterpret_cast<float4 *>(sT + (16 * Rb + r16) * LDA + 16 * I + 4 * q16) =
                    make_float4(-t4[0], -t4[1], -t4[2], -t4[3]);
            }
            __syncthreads();
        }
        // 5c. M[r][i] = T[r][i] beta_i (lower with diagonal) into the operand tile
#pragma unroll
        for (int it = 0; it < 4; ++it) {
            const int u = it * NT + tid;
            const int r = 8 * (u >> 7) + (u & 7), iq = (u >> 3) & 15, i = 4 * iq;
            const float4 tv = *reinterpret_cast<const float4 *>(sT + r * LDA + i);
            const float4 bv = *reinterpret_cast<const float4 *>(sBeta + i);
            st_tile4(sm + T_M, r, iq, KB64, i <= r ? tv.x * bv.x : 0.f, i + 1 <= r ? tv.y * bv.y : 0.f,
                     i + 2 <= r ? tv.z * bv.z : 0.f, i + 3 <= r ? tv.w * bv.w : 0.f);
        }
        umma::fence_smem_to_async();

        // ---------------------------------------------------------- 6. Z = V - Y, decay S
        if (!ptx::mbar_wait(&bar[1], phase, kWaitBudget)) {
            raise_error(2u);
            ok = false;
            break;
        }
        umma::fence_after_sync();
        {
            float y[32];  // rows r = 32 hw .. 32 hw + 31
            umma::ld_x32(tq + TM_D3 + 32 * hw, y);
            umma::wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) y[e] = tf32r(RW::widen1(R.v[e]) - y[e]);
            umma::st_x32(tq + TM_Z + 32 * hw, y);
        }
#pragma unroll
        for (int c = 64 * hw; c < 64 * hw + 64; c += 32) {  // S^T[j][c] *= e^{G63_c}
            float s32[32];
            umma::ld_x32(tq + TM_S + c, s32);
            umma::wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) s32[e] *= sGam[c + e];
            umma::st_x32(tq + TM_S + c, s32);
        }
        umma::wait_st();

        // prefetch the next chunk's inputs (registers are free now)
        if (c0 + C < T) load_chunk<TQ>(R, a, m, h, c0 + C, rr, c4, q4, hw, lane, tid);

        umma::fence_before_sync();
        __syncthreads();
        umma::fence_after_sync();
        if (tid == 0) {
#pragma unroll 1
            for (int ks = 0; ks < C / 8; ++ks)
                umma::mma_ts(tb + TM_D4, tb + TM_Z + ks * 8,
                             umma::smem_desc(sbase + T_M + ks * 256, 128, 8 * KB64), id64, ks > 0);
            umma::commit(&bar[2]);
            if (!ptx::mbar_wait(&bar[2], phase, kWaitBudget)) {
                raise_error(4u);
            } else {
                umma::fence_after_sync();
#pragma unroll 1
                for (int ks = 0; ks < C / 8; ++ks) {
                    umma::mma_ts(tb + TM_D3 + 64, tb + TM_D4 + ks * 8,
                                 umma::smem_desc(sbase + T_P + ks * 256, 128, 8 * KB64), id64, 1);
                    umma::mma_ts(tb + TM_S, tb + TM_D4 + ks * 8,
                                 umma::smem_desc(sbase + T_KDEC + ks * 256, 128, 8 * KB64), id128, 1);
                }
            }
            umma::commit(&bar[3]);
        }
        if (!ptx::mbar_wait(&bar[3], phase, kWaitBudget)) {
            raise_error(8u);
            ok = false;
            break;
        }
        umma::fence_after_sync();

        // ---------------------------------------------------------- 7. O out
        {
            float o32[32];
            umma::ld_x32(tq + TM_D3 + 64 + 32 * hw, o32);
            umma::wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) {
                const int t = c0 + 32 * hw + e;
                if (t < T) a.o[(((size_t)m * T + t) * a.H + h) * DK + j] = a.scale * o32[e];
            }
        }
        umma::fence_before_sync();
        __syncthreads();
        umma::fence_after_sync();
    }

    // state out
    if (ok) {
        for (int c = 64 * hw; c < 64 * hw + 64; c += 8) {
            float v8[8];
            umma::ld_x8(tq + TM_S + c, v8);
            umma::wait_ld();
#pragma unroll
            for (int e = 0; e < 8; ++e) state[(size_t)(c + e) * DK + j] = v8[e];
        }
    }
    umma::fence_before_sync();
    __syncthreads();
    if (warp == 0) umma::tmem_dealloc(tb, TM_COLS);
}

}  // namespace

cudaError_t launch_prefill_tc(const PrefillArgs &a, int qkv_dtype, cudaStream_t stream) {
    const dim3 grid(a.M * a.H);
    if (qkv_dtype == KDA_BF16) {
        cudaError_t e = cudaFuncSetAttribute(kda_prefill_tc_kernel<__nv_bfloat16>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
        if (e != cudaSuccess) return e;
        kda_prefill_tc_kernel<__nv_bfloat16><<<grid, NT, SMEM_BYTES, stream>>>(a);
    } else {
        cudaError_t e = cudaFuncSetAttribute(kda_prefill_tc_kernel<float>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
        if (e != cudaSuccess) return e;
        kda_prefill_tc_kernel<float><<<grid, NT, SMEM_BYTES, stream>>>(a);
    }
    return cudaGetLastError();
}

cudaError_t take_prefill_error(unsigned int *code) {
    unsigned int zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(code, g_prefill_error, sizeof(unsigned int));
    if (e != cudaSuccess) return e;
    if (*code) e = cudaMemcpyToSymbol(g_prefill_error, &zero, sizeof(unsigned int));
    return e;
}

}  // namespace kda
