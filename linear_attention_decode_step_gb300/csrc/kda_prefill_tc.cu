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
// Organisation. One CTA (512 threads, 16 warps) owns one (stream, head) and
// walks its chunks in order. The state lives in tensor memory for the whole
// sequence, transposed (lane = value channel j, column = key channel i) and
// in FP32: it is the accumulator of the state update and, read as TF32, the
// A operand (from tensor memory) of the products with S. Every MMA has
// M = 128 rows:
//   MMA1  D1 = [L0; Lq0; L1; Lq1] [R0; R1; R0o]^T     A and P (N = 96)
//   MMA3  D3 = S^T [Kd; Qd]^T                           Y^T = (Kd S)^T and (Qd S)^T
//   MMA4  D4 = Z^T M^T,  Z = V - Y                      Delta^T
//   MMA5  D3[:, 64:] += Delta^T P^T                     O^T
//   MMA6  S^T += Delta^T Kdec,  after S^T *= e^{G_63} per column
// Operand tiles are written by the threads in the K-major core-matrix layout
// (kda_umma.cuh) and read through shared-memory descriptors.
//
// Numerics. Decay factors are taken relative to the middle token of each
// 32-token half (m_b = G_15, G_47): inside a half |G_r - m_b| spans at most 16
// per-token log-decays, which stays inside FP32 for log(alpha) above about
// -5.4 (the model's gate keeps it above -5; section 8.2.3 ties the -5 floor to
// 16-token spans). The block of second-half rows against first-half columns
// uses the second half's left factor and R0o = K e^{m_1 - G} <= 1 on the right,
// with its own exponent (a product of separately rounded factors would
// underflow where the decay is strong).
// Every factor of Kd, Qd, Kdec and the state decay is <= 1.
//
// Thread roles. "Token-channel" work (decay scan, norms, operand tiles): warp
// w covers channels 16 (w % 8) .. + 15 and the 32-token half w / 8; lane
// (qq, rr) = (lane / 8, lane % 8) holds tokens 8 g + rr (g = 0..3) of the half
// and channels 4 qq .. + 3 of the warp's group. A quarter-warp (8 lanes, the
// unit in which 16-byte shared-memory stores are served) thus writes the 8
// rows of one core matrix: the tile stores are free of bank conflicts.
// "Tensor-memory" work: warp w reads lanes 32 (w % 4) .. + 31 (value channel
// j) and column quarter w / 4.
//
// The unit lower-triangular inverse is taken on CUDA cores in 16 x 16 blocks:
// diagonal blocks by forward substitution (one lane per column), off-diagonal
// blocks level by level from the block recurrence T_RI = -T_RR sum_Q A_RQ T_QI.
// Warps 0-7 take it while warps 8-15 wait for MMA3 and do phase 6 (Z = V - Y,
// the state decay); the Kdec^T tile is built while MMA1 runs.
//
// Inputs arrive ahead of use through tensor maps (cp.async.bulk.tensor): with
// BF16 q, k the next chunk's q, k, alpha land as 128-byte-swizzled boxes in
// the [Kd; Qd] region once MMA3 has read it (FP32 q, k are loaded into
// registers a chunk ahead instead); v of the next chunk arrives in one tensor
// copy; O leaves through shared memory in one tensor store. Every mbarrier
// wait is bounded. A thread whose wait gives up sets the device error word
// (kda_device_error) and carries on to the next CTA-wide barrier, which ANDs
// every thread's outcome (__syncthreads_and), so the CTA leaves the chunk
// loop together; on the way out the thread that issued the tensor-core
// products and the thread that issued the tensor copies wait (bounded) for
// their last ones, and only then is the tensor memory freed.

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>

#include "../../include/kda.h"
#include "kda_internal.cuh"
#include "kda_ptx.cuh"
#include "kda_umma.cuh"

namespace kda {

__device__ unsigned int g_prefill_error;

namespace {

constexpr int DK = kHeadDim;
constexpr int C = 64;
constexpr int NT = 512;
constexpr float kL2Eps = 1e-6f;

// operand tiles (bytes), K-major core-matrix layout
constexpr uint32_t KB128 = DK * 4;  // one row of a K = 128 tile
constexpr uint32_t KB64 = C * 4;    // one row of a K = 64 tile
// phase-1 tiles
constexpr uint32_t T_LA = 0;                       // [L0; Lq0; L1; Lq1]  128 x 128
constexpr uint32_t T_RB = T_LA + 128 * KB128;      // [R0; R1; R0o]        96 x 128
constexpr uint32_t PH1_END = T_RB + 96 * KB128;    // 114688
// phase-2 tiles: [Kd; Qd], P, M, A, T and the inverse's scratch overlay the
// phase-1 tiles once MMA1 has completed; Kdec^T lies past them and is written
// while MMA1 runs
constexpr uint32_t T_KQ = 0;                       // [Kd; Qd]       128 x 128
constexpr uint32_t T_P = T_KQ + 128 * KB128;       // P               64 x 64
constexpr uint32_t T_M = T_P + 64 * KB64;          // M               64 x 64
constexpr uint32_t T_A = T_M + 64 * KB64;          // A (plain [64][68] FP32)
constexpr int LDA = 68;
constexpr uint32_t T_T = T_A + 64 * LDA * 4;       // T = (I + A)^-1 (plain [64][68] FP32)
constexpr uint32_t T_X = T_T + 64 * LDA * 4;       // scratch: up to 3 blocks of 16 x 16
constexpr uint32_t T_KDEC = (T_X + 3 * 256 * 4 + 1023) / 1024 * 1024;  // Kdec^T  128 x 64
constexpr uint32_t T_V = T_KDEC + 128 * KB64;      // v of the chunk, token-major [64][128] (tensor copies)
constexpr uint32_t PH2_END = T_V + 64 * DK * 4;
constexpr uint32_t T_O = T_KDEC;                   // O staging [64][128]: phase 7 to the next chunk's MMA1, over Kdec^T
static_assert(64 * DK * 4 <= T_V - T_O, "O staging fits the Kdec^T region");
static_assert(T_KDEC >= PH1_END, "Kdec^T is written while MMA1 reads the phase-1 tiles");
constexpr uint32_t TILES = PH2_END > PH1_END ? PH2_END : PH1_END;
// small buffers (bytes)
constexpr int LDN = 12;                            // norm partials row: 8 groups + 4 (bank shift)
constexpr uint32_t S_NORM = TILES;                 // [2][64 rows][LDN] partial sums of q^2, k^2
constexpr uint32_t S_XCH = S_NORM + 2 * 64 * LDN * 4;  // [3][128]: G_31, L_47, L_63 per channel
constexpr uint32_t S_BETA = S_XCH + 3 * 128 * 4;
constexpr uint32_t S_GAM = S_BETA + 64 * 4;        // [128] e^{G_63}
// the layer form: raw q, k of the three tokens before each half
// ([tensor][tap][channel]: xa = tokens 29-31 of this chunk, xb[2] = tokens
// 61-63 of the previous chunk by chunk parity) and the q, k conv weights
constexpr uint32_t S_XA = S_GAM + 128 * 4;
constexpr uint32_t XB_F = 2 * 3 * 128;
constexpr uint32_t S_XB = S_XA + XB_F * 4;
constexpr uint32_t S_WQK = S_XB + 2 * XB_F * 4;    // [3][128] float4: q, k, v conv weights
constexpr uint32_t S_BIAS = S_WQK + 3 * 128 * 16;  // [128] gate bias of the head
constexpr uint32_t S_VC = S_BIAS + 128 * 4;        // [2][3][128] raw v of the 3 tokens before a chunk
constexpr uint32_t S_BAR = S_VC + 2 * 3 * 128 * 4; // 5 mbarriers
constexpr uint32_t S_SLOT = S_BAR + 6 * 8;
constexpr uint32_t SMEM_BYTES = S_SLOT + 16;
static_assert(SMEM_BYTES <= 232448, "fits the 227 KiB opt-in shared memory");
// BF16 q, k: q, k and alpha of the next chunk are staged in the [Kd; Qd]
// region (free from the completion of MMA3 to the next chunk's operand
// stores) as tensor-copy boxes of 64 tokens x 128 bytes, 128-byte swizzled
constexpr uint32_t BOX = 64 * 128;
constexpr uint32_t ST_Q = T_KQ;                    // 2 boxes of 64 channels (BF16)
constexpr uint32_t ST_K = ST_Q + 2 * BOX;          // 2 boxes
constexpr uint32_t ST_AL = ST_K + 2 * BOX;         // 4 boxes of 32 channels (FP32)
constexpr uint32_t ST_END = ST_AL + 4 * BOX;
static_assert(ST_END <= T_KDEC, "the staging fits the [Kd; Qd] region");
static_assert(T_V % 1024 == 0 && T_O % 1024 == 0, "tensor-copy boxes start 1024-byte aligned");

// the thread that issues every MMA: lane 0 of the last warp (free of the
// phase-specific work that warps 0-1 carry in the inverse)
constexpr int kIssuer = NT - 32;
// lane 0 of this warp issues the tensor copies of q, k, alpha and v
constexpr int kVWarp = NT / 32 - 2;
constexpr int kLoader = 32 * kVWarp;
// named barriers (0 is __syncthreads): the issuer waits for all threads,
// the others only signal and move on
constexpr uint32_t kBarMma1 = 1, kBarMma3 = 2, kBarOut = 3;
// phase 5 splits the CTA: warps 0-7 take the inverse (their own barrier),
// warps 8-15 meanwhile the state-pass work of phase 6
constexpr uint32_t kBarInv = 4;
constexpr int kInvThreads = 256;

// TMEM columns
constexpr uint32_t TM_S = 0, TM_D3 = 128, TM_Z = 256, TM_D4 = 320, TM_D1 = 384;
constexpr uint32_t TM_COLS = 512;

__device__ __forceinline__ void raise_error(unsigned int code) { atomicOr(&g_prefill_error, code); }

// Tensor maps of one call (made on the host, kernel parameter). Every map
// views its tensor with the channel innermost, then head, [tensor,] token,
// stream, so that a box is 64 tokens of one head and tokens past T read as 0.
struct PrefillMaps {
    CUtensorMap q;      // q [M][T][H][128]; the layer form: x [M][T][3][H*128] (q and k); 128-byte swizzle
    CUtensorMap k;      // k (plain form); 128-byte swizzle
    CUtensorMap alpha;  // alpha, or the raw gate input of the layer form; 128-byte swizzle
    CUtensorMap v;      // v, or x of the layer form (tensor 2); boxes of 64 x 128 channels
    CUtensorMap o;      // o [M][T][H][128]; boxes of 64 x 128 channels (stores)
};

// Byte offset of (row, byte) in a box of 128-byte rows written with the
// 128-byte swizzle: the 16-byte chunk index is XORed with the row index
// modulo 8 (the box starts 1024-byte aligned).
__device__ __forceinline__ uint32_t swz(uint32_t row, uint32_t byte) {
    return row * 128u + ((((byte >> 4) ^ row) & 7u) << 4) + (byte & 15u);
}

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
// SiLU(x) = x sigmoid(x) with sigmoid(x) = (1 + tanh(x / 2)) / 2, i.e.
// h + h tanh(h) for h = x / 2: one hardware tanh (tanh.approx.f32, relative
// error about 2^-11) in place of an exponential and a reciprocal, the
// special-function pipe being what bounds the conv of the layer form
__device__ __forceinline__ float silu(float x) {
    const float h = 0.5f * x;
    float t;
    asm("tanh.approx.f32 %0, %1;" : "=f"(t) : "f"(h));
    return fmaf(h, t, h);
}
// sigmoid(x) = (1 + tanh(x / 2)) / 2 the same way, for the norm's output gate
// (a factor on an already normalised output: its error does not accumulate)
__device__ __forceinline__ float sigm(float x) {
    float t;
    asm("tanh.approx.f32 %0, %1;" : "=f"(t) : "f"(0.5f * x));
    return fmaf(0.5f, t, 0.5f);
}
__device__ __forceinline__ float lg2(float x) {
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// An FP32 operand prepared for a TF32 product: the tensor cores read it by
// dropping its 13 low mantissa bits (a biased truncation, pinned by the tensor
// core tests), so adding half a TF32 ulp to the magnitude bits first makes
// that a round to nearest (ties away from zero) and the errors unbiased. The
// low bits are left for the hardware to drop. (Inputs are finite; nothing
// here rounds into inf or NaN.)
__device__ __forceinline__ float tf32r(float x) { return __uint_as_float(__float_as_uint(x) + 0x1000u); }

__device__ __forceinline__ void st_tile4(unsigned char *tile, uint32_t row, uint32_t c4,
                                         uint32_t kbytes, float a, float b, float c, float d) {
    *reinterpret_cast<float4 *>(tile + (row >> 3) * (8u * kbytes) + c4 * 128u + (row & 7u) * 16u) =
        make_float4(tf32r(a), tf32r(b), tf32r(c), tf32r(d));
}

// Per-thread inputs of one chunk, kept exactly as loaded (no arithmetic on
// them until the chunk is processed, so the loads overlap the previous
// chunk's work).
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

// q, k, alpha of this thread's 4 tokens x 4 channels (token-channel mapping);
// tokens past T read as q = k = 0, alpha = 1
template <typename TQ>
struct QKA {
    typename Raw<TQ>::Q4 q[4], k[4];
    float4 al[4];
};
template <typename TQ, bool LAYER>
__device__ __forceinline__ void load_qka(QKA<TQ> &R, const PrefillArgs &a, int m, int h, int t0,
                                         int c4) {
    using RW = Raw<TQ>;
    const TQ *q = static_cast<const TQ *>(a.q);
    const TQ *k = static_cast<const TQ *>(a.k);
    const size_t D = (size_t)a.H * DK;
#pragma unroll
    for (int g = 0; g < 4; ++g) {
        const int t = t0 + 8 * g;
        if (t < a.T) {
            const size_t base = (((size_t)m * a.T + t) * a.H + h) * DK + 4 * c4;
            if (LAYER) {  // pre-conv x [M][T][3][D]: q is tensor 0, k tensor 1
                const size_t xb = (((size_t)m * a.T + t) * 3) * D + (size_t)h * DK + 4 * c4;
                R.q[g] = RW::load4(q + xb);
                R.k[g] = RW::load4(q + xb + D);
            } else {
                R.q[g] = RW::load4(q + base);
                R.k[g] = RW::load4(k + base);
            }
            R.al[g] = __ldg(reinterpret_cast<const float4 *>(a.alpha + base));
        } else {
            R.q[g] = R.k[g] = typename RW::Q4{};
            R.al[g] = make_float4(1.f, 1.f, 1.f, 1.f);
        }
    }
}
// The same values from the staged boxes (BF16 q, k): channels 4 c4 .. + 3
// sit in q / k box c4 / 16 at byte 8 (c4 % 16) and in alpha box c4 / 8 at
// byte 16 (c4 % 8). Lanes rr = 0..7 read rows of distinct residues mod 8, so
// the swizzle spreads a quarter-warp over all 32 banks.
__device__ __forceinline__ void fetch_qka(QKA<__nv_bfloat16> &R, const unsigned char *sm, int r0, int c4) {
#pragma unroll
    for (int g = 0; g < 4; ++g) {
        const uint32_t r = r0 + 8 * g;
        R.q[g] = *reinterpret_cast<const uint2 *>(sm + ST_Q + (c4 >> 4) * BOX + swz(r, (c4 & 15) * 8));
        R.k[g] = *reinterpret_cast<const uint2 *>(sm + ST_K + (c4 >> 4) * BOX + swz(r, (c4 & 15) * 8));
        R.al[g] = *reinterpret_cast<const float4 *>(sm + ST_AL + (c4 >> 3) * BOX + swz(r, (c4 & 7) * 16));
    }
}
template <typename TQ, bool LAYER, bool NORM>
__global__ void __launch_bounds__(NT, 1) kda_prefill_tc_kernel(const PrefillArgs a, const __grid_constant__ PrefillMaps mp,
                                                                const int item_base, const int piece_chunks) {
    // BF16 q, k arrive by tensor copies into shared memory; FP32 ones (twice
    // the bytes: no room to stage) by register loads a chunk ahead
    constexpr bool kTma = sizeof(TQ) == 2;
    extern __shared__ __align__(1024) unsigned char sm[];
    float *sNorm = reinterpret_cast<float *>(sm + S_NORM);
    float *sXch = reinterpret_cast<float *>(sm + S_XCH);
    float *sBeta = reinterpret_cast<float *>(sm + S_BETA);
    float *sGam = reinterpret_cast<float *>(sm + S_GAM);
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm + S_BAR);  // 0: MMA1, 1: MMA3, 2: MMA4, 3: MMA5/6, 4: v, 5: q, k, alpha
    uint32_t *slot = reinterpret_cast<uint32_t *>(sm + S_SLOT);
    float *sA = reinterpret_cast<float *>(sm + T_A);
    float *sT = reinterpret_cast<float *>(sm + T_T);
    float *sX = reinterpret_cast<float *>(sm + T_X);
    const TQ *sV = reinterpret_cast<const TQ *>(sm + T_V);
    float *sVc = reinterpret_cast<float *>(sm + S_VC);
    float *sO = reinterpret_cast<float *>(sm + T_O);
    float *sXa = reinterpret_cast<float *>(sm + S_XA);
    float *sXb = reinterpret_cast<float *>(sm + S_XB);
    float4 *sWqk = reinterpret_cast<float4 *>(sm + S_WQK);
    float *sBias = reinterpret_cast<float *>(sm + S_BIAS);

    // work item: piece `piece` (chunks piece * piece_chunks .. + piece_chunks - 1)
    // of sequence (m, h); a launch holds pieces whose predecessors an earlier
    // launch on the stream has finished (the state passes between them in place)
    const int item = item_base + (int)blockIdx.x;
    const int seq = item % (a.M * a.H), piece = item / (a.M * a.H);
    const int h = seq % a.H, m = seq / a.H;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // token-channel mapping
    const int cg = warp & 7, rh = warp >> 3, rr = lane & 7, qq = lane >> 3;
    const int c4 = 4 * cg + qq;                    // channels 4 c4 .. 4 c4 + 3
    const int r0 = 32 * rh + rr;                   // tokens r0 + 8 g, g = 0..3
    // tensor-memory mapping
    const int q4 = warp & 3, hq = warp >> 2;
    const int j = 32 * q4 + lane;                  // value channel (TMEM lane)
    const int T = a.T;
    const int t_begin = piece * piece_chunks * C;
    const int t_end = min(T, t_begin + piece_chunks * C);
    const uint32_t sbase = ptx::smem_u32(sm);
    if (sbase & 1023u) {  // the swizzled boxes need a 1024-byte aligned base
        if (tid == 0) raise_error(kPrefillErrMisaligned);
        return;
    }

    if (tid == 0) {
        for (int b = 0; b < 6; ++b) ptx::mbar_init(&bar[b], 1);
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
    // Launched with programmatic stream serialisation: the set-up above overlaps
    // the previous grid's tail (the previous round's pieces, or whatever ran
    // before); every global read comes after this wait, and the next grid may
    // start placing its CTAs as SMs free up.
    ptx::grid_dependency_wait();
    ptx::launch_dependents();

    // v of the chunk starting at token t0 -> sV (token-major [64][128], rows
    // past T zero), one tensor copy completing on bar[4]; thread kLoader
    auto issue_v = [&](int t0) {
        ptx::mbar_arrive_expect_tx(&bar[4], C * DK * (uint32_t)sizeof(TQ));
        if (LAYER) ptx::tma_load_5d(sm + T_V, &mp.v, &bar[4], 0, h, 2, t0, m);
        else ptx::tma_load_4d(sm + T_V, &mp.v, &bar[4], 0, h, t0, m);
    };
    // BF16 q, k: q, k, alpha of the chunk at t0 -> the staging boxes, completing on bar[5]
    auto issue_qka = [&](int t0) {
        ptx::mbar_arrive_expect_tx(&bar[5], ST_END - ST_Q);
#pragma unroll
        for (int b = 0; b < 2; ++b) {
            if (LAYER) {
                ptx::tma_load_5d(sm + ST_Q + b * BOX, &mp.q, &bar[5], 64 * b, h, 0, t0, m);
                ptx::tma_load_5d(sm + ST_K + b * BOX, &mp.q, &bar[5], 64 * b, h, 1, t0, m);
            } else {
                ptx::tma_load_4d(sm + ST_Q + b * BOX, &mp.q, &bar[5], 64 * b, h, t0, m);
                ptx::tma_load_4d(sm + ST_K + b * BOX, &mp.k, &bar[5], 64 * b, h, t0, m);
            }
        }
#pragma unroll
        for (int b = 0; b < 4; ++b) ptx::tma_load_4d(sm + ST_AL + b * BOX, &mp.alpha, &bar[5], 32 * b, h, t0, m);
    };
    if (tid == kLoader) {  // the first chunk's inputs, under the state copy below
        if (kTma) issue_qka(t_begin);
        issue_v(t_begin);
    }


    // state in: S^T[j][i] = S[i][j]; this thread: lane j, key channels [32 hq, 32 hq + 32)
    float *state = a.state + ((size_t)m * a.H + h) * DK * DK;
    for (int c = 32 * hq; c < 32 * hq + 32; c += 8) {
        float v8[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) v8[e] = state[(size_t)(c + e) * DK + j];
        umma::st_x8(tq + TM_S + c, v8);
    }
    umma::wait_st();

    using RW = Raw<TQ>;
    QKA<TQ> R;
    float beta_n = 0.f;
    if (!kTma) load_qka<TQ, LAYER>(R, a, m, h, t_begin + r0, c4);
    if (tid < C) beta_n = t_begin + tid < T ? __ldg(a.beta + ((size_t)m * T + t_begin + tid) * a.H + h) : 0.f;

    // the layer form: gate constants, conv weights, the cache as the tokens
    // before the first chunk, and the raw q, k before the second half
    const size_t D = (size_t)a.H * DK;
    if (LAYER) {
        const float4 *w4 = reinterpret_cast<const float4 *>(a.conv_w);
        if (tid < 3 * DK) sWqk[tid] = __ldg(w4 + (size_t)(tid >> 7) * D + (size_t)h * DK + (tid & 127));
        if (tid < DK) sBias[tid] = __ldg(a.dt_bias + (size_t)h * DK + tid);
        const TQ *cache = static_cast<const TQ *>(a.cache);
        const TQ *xg = static_cast<const TQ *>(a.q);
        // the three inputs before the piece's first chunk (the conv cache before
        // token 0, else x) -> the buffers that chunk reads: xb[p][X][tap][c] (q, k)
        // and vc[p][tap][c] (v), p = parity of the chunk before it
        const int pb = ((t_begin / C) + 1) & 1;
        for (int i = tid; i < 3 * 3 * DK; i += NT) {
            const int X = i / (3 * DK), tap = (i / DK) % 3, c = i % DK;
            const int t = t_begin - 3 + tap;
            const float v = RW::widen1(t < 0 ? RW::load1(cache + ((size_t)m * 9 + 3 * X + tap) * D + (size_t)h * DK + c)
                                             : RW::load1(xg + (((size_t)m * T + t) * 3 + X) * D + (size_t)h * DK + c));
            if (X < 2) sXb[pb * XB_F + i] = v;
            else sVc[pb * 3 * DK + tap * DK + c] = v;
        }
        if (!kTma && rh == 0 && rr >= 5) {  // tokens 29-31 of chunk 0 (lanes rr = 5, 6, 7 of g = 3)
            float xq[4], xk[4];
            RW::widen4(R.q[3], xq);
            RW::widen4(R.k[3], xk);
            *reinterpret_cast<float4 *>(sXa + (0 * 3 + rr - 5) * DK + 4 * c4) = make_float4(xq[0], xq[1], xq[2], xq[3]);
            *reinterpret_cast<float4 *>(sXa + (1 * 3 + rr - 5) * DK + 4 * c4) = make_float4(xk[0], xk[1], xk[2], xk[3]);
        }
        __syncthreads();
    }

    const uint32_t id128 = umma::instr_desc(128, 128, umma::kFmtTF32);
    const uint32_t id96 = umma::instr_desc(128, 96, umma::kFmtTF32);
    const uint32_t id64 = umma::instr_desc(128, 64, umma::kFmtTF32);
    // false once a wait of this thread gave up; folded into the next
    // CTA-wide barrier, where the whole CTA leaves the loop together
    bool ok = true;
    // the loader's tensor copies issued so far (bar[4]: v, bar[5]: q, k,
    // alpha) and the issuer's last commit (bar index, phase parity), for the
    // exit path
    int v_issued = tid == kLoader ? 1 : 0;
    int qka_issued = tid == kLoader && kTma ? 1 : 0;
    int last_bar = -1, last_par = 0;
    int phase = 0;

    for (int c0 = t_begin; c0 < t_end; c0 += C, phase ^= 1) {
        // ---------------------------------------------------------- 1. decay, norms
        if constexpr (kTma) {
            if (!ptx::mbar_wait(&bar[5], phase, ptx::kWaitBudget)) {
                raise_error(32u);
                ok = false;
            }
            fetch_qka(R, sm, r0, c4);
        }
        // cumulative log2-decay over the half's 32 tokens (lanes rr, then g)
        float G[4][4], qf[4][4], kf[4][4];
#pragma unroll
        for (int g = 0; g < 4; ++g) {
            RW::widen4(R.q[g], qf[g]);
            RW::widen4(R.k[g], kf[g]);
        }
        if (LAYER) {
            const int cidx = c0 / C;
            // tokens 61-63 of this chunk, for the next chunk's first half
            if (rh == 1 && rr >= 5) {
                float *xb = sXb + (cidx & 1) * XB_F;
                *reinterpret_cast<float4 *>(xb + (0 * 3 + rr - 5) * DK + 4 * c4) =
                    make_float4(qf[3][0], qf[3][1], qf[3][2], qf[3][3]);
                *reinterpret_cast<float4 *>(xb + (1 * 3 + rr - 5) * DK + 4 * c4) =
                    make_float4(kf[3][0], kf[3][1], kf[3][2], kf[3][3]);
            }
            // forget gate in log2 units: lb sigmoid(e^A (f + b)) / ln 2
            const float eA = __expf(__ldg(a.A_log + h));
            const float lbl2 = a.gate_lb * 1.4426950408889634f;
            const float4 b4 = *reinterpret_cast<const float4 *>(sBias + 4 * c4);
            const float bias[4] = {b4.x, b4.y, b4.z, b4.w};
#pragma unroll
            for (int g = 0; g < 4; ++g) {
                const int t = c0 + 32 * rh + 8 * g + rr;
                const float f4[4] = {R.al[g].x, R.al[g].y, R.al[g].z, R.al[g].w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float z = eA * (f4[e] + bias[e]);
                    G[g][e] = t < T ? __fdividef(lbl2, 1.0f + __expf(-z)) : 0.f;
                }
            }
            if constexpr (kTma) {
                // conv + SiLU with the raw taps (tokens t - 1, t - 2, t - 3) read from the
                // staged boxes; rows before the chunk from the previous chunk's last three
                const float *xp = sXb + ((cidx + 1) & 1) * XB_F;
#pragma unroll
                for (int g = 0; g < 4; ++g) {
                    const int t = c0 + 32 * rh + 8 * g + rr;
                    float tq3[3][4], tk3[3][4];
#pragma unroll
                    for (int kk = 1; kk <= 3; ++kk) {
                        const int row = 32 * rh + 8 * g + rr - kk;
                        const uint32_t off = (c4 >> 4) * BOX + swz(row < 0 ? 0 : row, (c4 & 15) * 8);
                        RW::widen4(*reinterpret_cast<const uint2 *>(sm + ST_Q + off), tq3[kk - 1]);
                        RW::widen4(*reinterpret_cast<const uint2 *>(sm + ST_K + off), tk3[kk - 1]);
                        if (row < 0) {  // tap row + 3 of the previous chunk's tokens 61-63
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                tq3[kk - 1][e] = xp[(0 * 3 + row + 3) * DK + 4 * c4 + e];
                                tk3[kk - 1][e] = xp[(1 * 3 + row + 3) * DK + 4 * c4 + e];
                            }
                        }
                    }
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float4 wq = sWqk[4 * c4 + e], wk = sWqk[DK + 4 * c4 + e];
                        const float pre_q = wq.x * tq3[2][e] + wq.y * tq3[1][e] + wq.z * tq3[0][e] + wq.w * qf[g][e];
                        const float pre_k = wk.x * tk3[2][e] + wk.y * tk3[1][e] + wk.z * tk3[0][e] + wk.w * kf[g][e];
                        const bool live = t < T;  // tokens past T stay out of the chunk
                        qf[g][e] = live ? silu(pre_q) : 0.f;
                        kf[g][e] = live ? silu(pre_k) : 0.f;
                    }
                }
            } else {
                // conv + SiLU, token groups from last to first (each reads the raw
                // values of the group before it): token 8 g + rr - kk sits in lane
                // rr - kk of group g, or in lane rr - kk + 8 of group g - 1, or (first
                // group) in the buffer of the three tokens before the half, at tap
                // rr - kk + 3
                const float *xp = rh ? sXa : sXb + ((cidx + 1) & 1) * XB_F;
#pragma unroll
                for (int g = 3; g >= 0; --g) {
                    const int t = c0 + 32 * rh + 8 * g + rr;
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        float wq3[3], wk3[3];  // tokens t - 1, t - 2, t - 3
#pragma unroll
                        for (int kk = 1; kk <= 3; ++kk) {
                            const int src = 8 * qq + ((rr - kk) & 7);
                            const float aq = __shfl_sync(0xffffffffu, qf[g][e], src);
                            const float ak = __shfl_sync(0xffffffffu, kf[g][e], src);
                            float bq, bk;
                            if (g > 0) {
                                bq = __shfl_sync(0xffffffffu, qf[g > 0 ? g - 1 : 0][e], src);
                                bk = __shfl_sync(0xffffffffu, kf[g > 0 ? g - 1 : 0][e], src);
                            } else {
                                const int tap = rr - kk + 3 < 2 ? rr - kk + 3 : 2;  // used only when rr < kk
                                bq = xp[(0 * 3 + tap) * DK + 4 * c4 + e];
                                bk = xp[(1 * 3 + tap) * DK + 4 * c4 + e];
                            }
                            wq3[kk - 1] = rr >= kk ? aq : bq;
                            wk3[kk - 1] = rr >= kk ? ak : bk;
                        }
                        const float4 wq = sWqk[4 * c4 + e], wk = sWqk[DK + 4 * c4 + e];
                        const float pre_q = wq.x * wq3[2] + wq.y * wq3[1] + wq.z * wq3[0] + wq.w * qf[g][e];
                        const float pre_k = wk.x * wk3[2] + wk.y * wk3[1] + wk.z * wk3[0] + wk.w * kf[g][e];
                        const bool live = t < T;  // tokens past T stay out of the chunk
                        qf[g][e] = live ? silu(pre_q) : 0.f;
                        kf[g][e] = live ? silu(pre_k) : 0.f;
                    }
                }
            }
        } else {
#pragma unroll
            for (int g = 0; g < 4; ++g) {  // tokens past T: no decay (staged alpha reads 0 there)
                const bool live = c0 + 32 * rh + 8 * g + rr < T;
                G[g][0] = live ? lg2(R.al[g].x) : 0.f;
                G[g][1] = live ? lg2(R.al[g].y) : 0.f;
                G[g][2] = live ? lg2(R.al[g].z) : 0.f;
                G[g][3] = live ? lg2(R.al[g].w) : 0.f;
            }
        }
        float carry[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int g = 0; g < 4; ++g) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                float x = G[g][e];
#pragma unroll
                for (int d = 1; d < 8; d <<= 1) {
                    const float y = __shfl_up_sync(0xffffffffu, x, d, 8);
                    if (rr >= d) x += y;
                }
                x += carry[e];
                G[g][e] = x;
                carry[e] = __shfl_sync(0xffffffffu, x, 8 * qq + 7);
            }
        }
        // mid (token 15 of the half) and total (token 31), from lanes rr = 7
        float mid[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) mid[e] = __shfl_sync(0xffffffffu, G[1][e], 8 * qq + 7);
        if (rr == 0) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                if (rh == 0) {
                    sXch[4 * c4 + e] = carry[e];              // G_31
                } else {
                    sXch[128 + 4 * c4 + e] = mid[e];          // L_47 = G_47 - G_31
                    sXch[256 + 4 * c4 + e] = carry[e];        // L_63 = G_63 - G_31
                }
            }
        }
        // L2-norm partial sums: 4 channels here, 16 per warp
#pragma unroll
        for (int g = 0; g < 4; ++g) {
            float sq = 0.f, sk = 0.f;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                sq = fmaf(qf[g][e], qf[g][e], sq);
                sk = fmaf(kf[g][e], kf[g][e], sk);
            }
            sq += __shfl_xor_sync(0xffffffffu, sq, 8);
            sq += __shfl_xor_sync(0xffffffffu, sq, 16);
            sk += __shfl_xor_sync(0xffffffffu, sk, 8);
            sk += __shfl_xor_sync(0xffffffffu, sk, 16);
            if (qq == 0) {
                const int r = r0 + 8 * g;
                sNorm[(0 * 64 + r) * LDN + cg] = sq;
                sNorm[(1 * 64 + r) * LDN + cg] = sk;
            }
        }
        if (tid < C) sBeta[tid] = beta_n;
        if (!__syncthreads_and(ok)) {
            ok = false;
            break;
        }
        float rq[4], rk[4];
#pragma unroll
        for (int g = 0; g < 4; ++g) {
            const int r = r0 + 8 * g;
            const float4 qa = *reinterpret_cast<const float4 *>(sNorm + r * LDN);
            const float4 qb = *reinterpret_cast<const float4 *>(sNorm + r * LDN + 4);
            const float4 ka = *reinterpret_cast<const float4 *>(sNorm + (64 + r) * LDN);
            const float4 kb = *reinterpret_cast<const float4 *>(sNorm + (64 + r) * LDN + 4);
            const float sq = qa.x + qa.y + qa.z + qa.w + qb.x + qb.y + qb.z + qb.w + kL2Eps;
            const float sk = ka.x + ka.y + ka.z + ka.w + kb.x + kb.y + kb.z + kb.w + kL2Eps;
            // the hardware reciprocal square root: a few ulp, far inside the
            // TF32 operand error
            rq[g] = rsqrtf(sq);
            rk[g] = rsqrtf(sk);
        }
        // per-channel factors (log2 units):
        //   half 0: u = e^{G - G_15};  R0o = K e^{m_1 - G} with m_1 = G_31 + L_47
        //           (its own exponent: R e^{m_1 - m_0} would lose it to underflow
        //           of e^{m_1 - m_0} when the decay is strong);
        //           Kd = L e^{G_15};   Kdec = R e^{G_31 + L_63 - G_15}
        //   half 1: u = e^{L - L_47};  Kd = L e^{G_31 + L_47};  Kdec = R e^{L_63 - L_47}
        float m1a[4], em[4], ed[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float g31 = sXch[4 * c4 + e], l47 = sXch[128 + 4 * c4 + e];
            const float l63 = sXch[256 + 4 * c4 + e];
            m1a[e] = g31 + l47;
            if (rh == 0) {
                em[e] = ex2(mid[e]);
                ed[e] = ex2(g31 + l63 - mid[e]);
            } else {
                em[e] = ex2(g31 + l47);
                ed[e] = ex2(l63 - l47);
            }
        }
        if (rh == 0 && rr == 0) {
#pragma unroll
            for (int e = 0; e < 4; ++e)
                sGam[4 * c4 + e] = ex2(sXch[4 * c4 + e] + sXch[256 + 4 * c4 + e]);
        }

        // ---------------------------------------------------------- 2. A / P operands
        // L = K u, Lq = Q u, R = K / u (normalised q, k); kept for the state-pass operands
        float Lk[4][4], Lq[4][4], Rk[4][4];
#pragma unroll
        for (int g = 0; g < 4; ++g) {
            const int r = r0 + 8 * g;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float x = G[g][e] - mid[e];
                const float u = ex2(x), ui = ex2(-x);
                const float kh = kf[g][e] * rk[g];
                Lk[g][e] = kh * u;
                Lq[g][e] = qf[g][e] * rq[g] * u;
                Rk[g][e] = kh * ui;
            }
            const int rowL = rh ? r + 32 : r, rowLq = rh ? r + 64 : r + 32;
            st_tile4(sm + T_LA, rowL, c4, KB128, Lk[g][0], Lk[g][1], Lk[g][2], Lk[g][3]);
            st_tile4(sm + T_LA, rowLq, c4, KB128, Lq[g][0], Lq[g][1], Lq[g][2], Lq[g][3]);
            st_tile4(sm + T_RB, r, c4, KB128, Rk[g][0], Rk[g][1], Rk[g][2], Rk[g][3]);
            if (rh == 0) {
                float Ro[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) Ro[e] = kf[g][e] * rk[g] * ex2(m1a[e] - G[g][e]);
                st_tile4(sm + T_RB, 64 + r, c4, KB128, Ro[0], Ro[1], Ro[2], Ro[3]);
            }
        }
        umma::fence_smem_to_async();
        umma::fence_before_sync();
        // the previous chunk's O staging (over Kdec^T, rewritten while MMA1 runs)
        // has been read by its tensor store before anyone passes this barrier
        if (tid == 0 && c0 > t_begin) ptx::bulk_wait_read_all();
        ptx::named_bar_sync(kBarMma1, NT);
        if (tid == kIssuer) {
            umma::fence_after_sync();
#pragma unroll 1
            for (int ks = 0; ks < DK / 8; ++ks)
                umma::mma_ss(tb + TM_D1, umma::smem_desc(sbase + T_LA + ks * 256, 128, 8 * KB128),
                             umma::smem_desc(sbase + T_RB + ks * 256, 128, 8 * KB128), id96, ks > 0,
                             1);
            umma::commit(&bar[0]);
            last_bar = 0;
            last_par = phase;
        }
        // under MMA1: Kdec = K e^{G63 - G} = R ed, as the Kdec^T tile
#pragma unroll
        for (int g = 0; g < 4; ++g) {
            // Kdec^T tile (row = key channel, K = token): a 4 x 4 transpose among
            // lanes rr = 4 hh .. 4 hh + 3, after which lane (hh, ce) holds channel
            // 4 c4 + ce of tokens 8 g + 4 hh .. + 3. Two butterfly stages: the
            // off-diagonal 2 x 2 blocks swap between lanes ce and ce ^ 2, then
            // each 2 x 2 block transposes between lanes ce and ce ^ 1.
            const int ce = rr & 3, hh = rr >> 2;
            const bool b1 = ce & 2, b0 = ce & 1;
            const float kc[4] = {Rk[g][0] * ed[0], Rk[g][1] * ed[1], Rk[g][2] * ed[2], Rk[g][3] * ed[3]};
            float x0 = __shfl_xor_sync(0xffffffffu, b1 ? kc[0] : kc[2], 2);
            float x1 = __shfl_xor_sync(0xffffffffu, b1 ? kc[1] : kc[3], 2);
            const float v4[4] = {b1 ? x0 : kc[0], b1 ? x1 : kc[1], b1 ? kc[2] : x0, b1 ? kc[3] : x1};
            x0 = __shfl_xor_sync(0xffffffffu, b0 ? v4[0] : v4[1], 1);
            x1 = __shfl_xor_sync(0xffffffffu, b0 ? v4[2] : v4[3], 1);
            const float ko[4] = {b0 ? x0 : v4[0], b0 ? v4[1] : x0, b0 ? x1 : v4[2], b0 ? v4[3] : x1};
            st_tile4(sm + T_KDEC, 4 * c4 + ce, 8 * rh + 2 * g + hh, KB64, ko[0], ko[1], ko[2], ko[3]);
        }
        if (!ptx::mbar_wait(&bar[0], phase, ptx::kWaitBudget)) {
            raise_error(1u);
            ok = false;
        }
        umma::fence_after_sync();

        // ---------------------------------------------------------- 3. A, P from TMEM
        // lane quarter q4: 0 A rows 0-31, 1 P rows 0-31, 2 A rows 32-63, 3 P rows 32-63.
        // D1 columns: 0-31 first-half columns (relative to m_0), 32-63 second-half
        // columns, 64-95 first-half columns relative to m_1 (for second-half rows).
        {
            const bool isP = q4 & 1;
            const int r = (q4 < 2 ? 0 : 32) + lane;
            const float br = sBeta[r];
            auto put4 = [&](int s, const float *d) {  // columns s .. s + 3 of row r
                float v4[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int i = s + e;
                    v4[e] = isP ? (i <= r ? d[e] : 0.f) : (i < r ? br * d[e] : 0.f);
                }
                if (isP)
                    st_tile4(sm + T_P, r, s >> 2, KB64, v4[0], v4[1], v4[2], v4[3]);
                else
                    *reinterpret_cast<float4 *>(sA + r * LDA + s) = make_float4(v4[0], v4[1], v4[2], v4[3]);
            };
            if (q4 < 2) {
                float d[8];
                umma::ld_x8(tq + TM_D1 + 8 * hq, d);
                umma::wait_ld();
                put4(8 * hq, d);
                put4(8 * hq + 4, d + 4);
                if (isP) {  // P rows 0-31, columns 32-63 are zero
                    st_tile4(sm + T_P, r, (32 + 8 * hq) >> 2, KB64, 0.f, 0.f, 0.f, 0.f);
                    st_tile4(sm + T_P, r, (36 + 8 * hq) >> 2, KB64, 0.f, 0.f, 0.f, 0.f);
                }
            } else {
                float d[16];
                umma::ld_x16(tq + TM_D1 + 32 + 16 * hq, d);
                umma::wait_ld();
                const int s0 = hq < 2 ? 32 + 16 * hq : 16 * (hq - 2);
#pragma unroll
                for (int b = 0; b < 4; ++b) put4(s0 + 4 * b, d + 4 * b);
            }
        }
        umma::fence_before_sync();
        // A, P visible; MMA1 operands may now be overwritten
        if (!__syncthreads_and(ok)) {
            ok = false;
            break;
        }

        // ---------------------------------------------------------- 4. state-pass operands
        //   Kd = K e^G = L em,   Qd = Lq em   (Kdec^T was written under MMA1)
#pragma unroll
        for (int g = 0; g < 4; ++g) {
            const int r = r0 + 8 * g;
            st_tile4(sm + T_KQ, r, c4, KB128, Lk[g][0] * em[0], Lk[g][1] * em[1], Lk[g][2] * em[2],
                     Lk[g][3] * em[3]);
            st_tile4(sm + T_KQ, 64 + r, c4, KB128, Lq[g][0] * em[0], Lq[g][1] * em[1],
                     Lq[g][2] * em[2], Lq[g][3] * em[3]);
        }
        umma::fence_smem_to_async();
        umma::fence_before_sync();
        if (warp == kIssuer / 32) ptx::named_bar_sync(kBarMma3, NT);
        else ptx::named_bar_arrive(kBarMma3, NT);
        if (tid == kIssuer) {
            umma::fence_after_sync();
#pragma unroll 1
            for (int ks = 0; ks < DK / 8; ++ks)
                umma::mma_ts(tb + TM_D3, tb + TM_S + ks * 8,
                             umma::smem_desc(sbase + T_KQ + ks * 256, 128, 8 * KB128), id128, ks > 0);
            umma::commit(&bar[1]);
            last_bar = 1;
            last_par = phase;
        }
        // the next chunk's q, k, alpha (the registers of this one are consumed);
        // issued after the proxy fence above, which would otherwise wait for them
        if (!kTma && c0 + C < t_end) load_qka<TQ, LAYER>(R, a, m, h, c0 + C + r0, c4);

        // ---------------------------------------------------------- 5. M = (I + A)^-1 Diag(beta)
        // (warps 0-7, on CUDA cores, while MMA3 runs on the tensor cores and
        // warps 8-15 take phase 6 as soon as MMA3 is done)
        auto inv_sync = [&]() { ptx::named_bar_sync(kBarInv, kInvThreads); };
        if (warp < kInvThreads / 32) {
            // 5a. diagonal 16 x 16 blocks, one lane per column: T_bb = (I + A_bb)^-1
            if (warp < 2) {
                const int b = 2 * warp + (lane >> 4), jj = lane & 15, j0 = 16 * b;
                float tcol[16];
#pragma unroll
                for (int r = 0; r < 16; ++r) {
                    float x0 = r == jj ? 1.f : 0.f, x1 = 0.f;
#pragma unroll
                    for (int i = 0; i < r; i += 2) {
                        x0 = fmaf(-sA[(j0 + r) * LDA + j0 + i], tcol[i], x0);
                        if (i + 1 < r) x1 = fmaf(-sA[(j0 + r) * LDA + j0 + i + 1], tcol[i + 1], x1);
                    }
                    tcol[r] = r >= jj ? x0 + x1 : 0.f;
                }
#pragma unroll
                for (int r = 0; r < 16; ++r) sT[(j0 + r) * LDA + j0 + jj] = tcol[r];
            }
            inv_sync();
            // 5b. off-diagonal blocks. The plain form, where the inverse is on the
            //     critical path, takes the right-looking order (fewer dependent block
            //     products); the layer form, where phase 6 is, the level order (fewer
            //     registers).
            if constexpr (!LAYER) {
                // 5b. off-diagonal blocks, right-looking: X_RI = sum_{Q=I}^{R-1} A_RQ T_QI
                //     collects each term as soon as T_QI exists (kept in the unused
                //     upper block (I, R) of A), so every step on the critical path is one
                //     16 x 16 block product: step 0 takes the six first terms A_RI T_II,
                //     level L solves T_RI = -T_RR X_RI for R = I + L, step k adds
                //     A_{R, I+k} T_{I+k, I} for R > I + k. Unit: row r16, columns 4 q16 .. + 3.
                {
                    const int r16 = (tid >> 2) & 15, q16 = tid & 3;
                    // X_RI += A_{R,Q} T_{Q,I} (or =, when first)
                    auto add_term = [&](int R, int I, int Q, int rr16, int qq16, bool first) {
                        float x4[4] = {0.f, 0.f, 0.f, 0.f};
                        float *xp = sA + (16 * I + rr16) * LDA + 16 * R + 4 * qq16;
                        if (!first) {
                            const float4 x0 = *reinterpret_cast<const float4 *>(xp);
                            x4[0] = x0.x;
                            x4[1] = x0.y;
                            x4[2] = x0.z;
                            x4[3] = x0.w;
                        }
#pragma unroll
                        for (int t = 0; t < 16; ++t) {
                            const float av = sA[(16 * R + rr16) * LDA + 16 * Q + t];
                            const float4 tv = *reinterpret_cast<const float4 *>(sT + (16 * Q + t) * LDA + 16 * I + 4 * qq16);
                            x4[0] = fmaf(av, tv.x, x4[0]);
                            x4[1] = fmaf(av, tv.y, x4[1]);
                            x4[2] = fmaf(av, tv.z, x4[2]);
                            x4[3] = fmaf(av, tv.w, x4[3]);
                        }
                        *reinterpret_cast<float4 *>(xp) = make_float4(x4[0], x4[1], x4[2], x4[3]);
                    };
                    // T_RI = -T_RR X_RI
                    auto solve = [&](int R, int I) {
                        float t4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                        for (int t = 0; t < 16; ++t) {
                            const float tv = sT[(16 * R + r16) * LDA + 16 * R + t];
                            const float4 xv = *reinterpret_cast<const float4 *>(sA + (16 * I + t) * LDA + 16 * R + 4 * q16);
                            t4[0] = fmaf(tv, xv.x, t4[0]);
                            t4[1] = fmaf(tv, xv.y, t4[1]);
                            t4[2] = fmaf(tv, xv.z, t4[2]);
                            t4[3] = fmaf(tv, xv.w, t4[3]);
                        }
                        *reinterpret_cast<float4 *>(sT + (16 * R + r16) * LDA + 16 * I + 4 * q16) =
                            make_float4(-t4[0], -t4[1], -t4[2], -t4[3]);
                    };
                    // step 0: the six blocks (R, I) = (1,0) (2,0) (3,0) (2,1) (3,1) (3,2), 384 units
                    for (int u = tid; u < 384; u += kInvThreads) {
                        const int p = u >> 6;
                        const int I = p < 3 ? 0 : (p < 5 ? 1 : 2), R = p < 3 ? p + 1 : (p < 5 ? p - 1 : 3);
                        add_term(R, I, I, (u >> 2) & 15, u & 3, true);
                    }
                    inv_sync();
                    if (tid < 192) solve((tid >> 6) + 1, tid >> 6);                       // T_10, T_21, T_32
                    inv_sync();
                    if (tid < 192) {                                                      // (2,0) (3,0) (3,1) += A T_{I+1,I}
                        const int p = tid >> 6, I = p < 2 ? 0 : 1, R = p == 0 ? 2 : 3;
                        add_term(R, I, I + 1, r16, q16, false);
                    }
                    inv_sync();
                    if (tid < 128) solve((tid >> 6) + 2, tid >> 6);                       // T_20, T_31
                    inv_sync();
                    if (tid < 64) add_term(3, 0, 2, r16, q16, false);                     // (3,0) += A_32 T_20
                    inv_sync();
                    if (tid < 64) solve(3, 0);                                            // T_30
                    inv_sync();
                }
            } else {
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
                    inv_sync();
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
                    inv_sync();
                }
            }
            // 5c. M[r][i] = T[r][i] beta_i (lower with diagonal) into the operand tile
#pragma unroll
            for (int it = 0; it < 1024 / kInvThreads; ++it) {
                const int u = it * kInvThreads + tid;
                const int r = 8 * (u >> 7) + (u & 7), iq = (u >> 3) & 15, i = 4 * iq;
                const float4 tv = *reinterpret_cast<const float4 *>(sT + r * LDA + i);
                const float4 bv = *reinterpret_cast<const float4 *>(sBeta + i);
                st_tile4(sm + T_M, r, iq, KB64, i <= r ? tv.x * bv.x : 0.f, i + 1 <= r ? tv.y * bv.y : 0.f,
                         i + 2 <= r ? tv.z * bv.z : 0.f, i + 3 <= r ? tv.w * bv.w : 0.f);
            }
            umma::fence_smem_to_async();
            // the next chunk's beta (sBeta of this chunk has been read)
            if (tid < C) {
                const int t = c0 + C + tid;
                beta_n = t < T ? __ldg(a.beta + ((size_t)m * T + t) * a.H + h) : 0.f;
            }
        } else {
            // ------------------------------------------------------ 6. Z = V - Y, decay S
            // (warps 8-15, while warps 0-7 invert): warp w does the units hq6 =
            // 2 ((w - 8) / 4) and + 1 of its lane quarter
            if (!ptx::mbar_wait(&bar[1], phase, ptx::kWaitBudget)) {
                raise_error(2u);
                ok = false;
            }
            umma::fence_after_sync();
            // MMA3 has read [Kd; Qd]: the region takes the next chunk's q, k, alpha
            if (kTma && tid == kLoader && c0 + C < t_end && ok) {
                issue_qka(c0 + C);
                ++qka_issued;
            }
            if (!ptx::mbar_wait(&bar[4], phase, ptx::kWaitBudget)) {
                raise_error(16u);
                ok = false;
            }
#pragma unroll 1
            for (int u6 = 0; u6 < 2; ++u6) {
                const int hq6 = 2 * ((warp - 8) >> 2) + u6;
                {
                    // v of tokens 16 hq6 .. + 15 at channel j from the staged chunk (0 past T)
                    float vf[16];
                    if constexpr (LAYER) {  // conv over tokens 16 hq6 - 3 .. 16 hq6 + 15 (the 3 before the chunk kept aside)
                        const float *vc = sVc + ((c0 / C + 1) & 1) * 3 * DK;
                        float raw[19];
#pragma unroll
                        for (int i = 0; i < 19; ++i) {
                            const int tl = 16 * hq6 - 3 + i;  // token within the chunk
                            raw[i] = tl < 0 ? vc[(tl + 3) * DK + j]
                                            : (c0 + tl < T ? RW::widen1(reinterpret_cast<const typename RW::V1 *>(sV)[tl * DK + j]) : 0.f);
                        }
                        if (hq6 == 3) {  // raw v of tokens 61-63, for the next chunk
                            float *vn = sVc + ((c0 / C) & 1) * 3 * DK;
#pragma unroll
                            for (int tap = 0; tap < 3; ++tap) vn[tap * DK + j] = raw[16 + tap];
                        }
                        const float4 wv = sWqk[2 * DK + j];
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            const float pre = wv.x * raw[i] + wv.y * raw[i + 1] + wv.z * raw[i + 2] + wv.w * raw[i + 3];
                            vf[i] = c0 + 16 * hq6 + i < T ? silu(pre) : 0.f;
                        }
                    } else {
#pragma unroll
                        for (int e = 0; e < 16; ++e) {
                            const int tl = 16 * hq6 + e;
                            vf[e] = c0 + tl < T ? RW::widen1(reinterpret_cast<const typename RW::V1 *>(sV)[tl * DK + j]) : 0.f;
                        }
                    }
                    float y[16];  // tokens 16 hq6 .. 16 hq6 + 15
                    umma::ld_x16(tq + TM_D3 + 16 * hq6, y);
                    umma::wait_ld();
#pragma unroll
                    for (int e = 0; e < 16; ++e) y[e] = tf32r(vf[e] - y[e]);
                    umma::st_x16(tq + TM_Z + 16 * hq6, y);
                }
                {  // S^T[j][c] *= e^{G63_c}
                    float s32[32];
                    umma::ld_x32(tq + TM_S + 32 * hq6, s32);
                    const float4 *gam4 = reinterpret_cast<const float4 *>(sGam + 32 * hq6);
                    umma::wait_ld();
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const float4 g4 = gam4[e];
                        const float2 a = __fmul2_rn(make_float2(s32[4 * e], s32[4 * e + 1]), make_float2(g4.x, g4.y));
                        const float2 b = __fmul2_rn(make_float2(s32[4 * e + 2], s32[4 * e + 3]), make_float2(g4.z, g4.w));
                        s32[4 * e] = a.x;
                        s32[4 * e + 1] = a.y;
                        s32[4 * e + 2] = b.x;
                        s32[4 * e + 3] = b.y;
                    }
                    umma::st_x32(tq + TM_S + 32 * hq6, s32);
                }
            }
            umma::wait_st();
        }
        // the layer form: raw q, k of tokens 29-31 of the next chunk (loaded in phase 4)
        if (!kTma && LAYER && rh == 0 && rr >= 5 && c0 + C < t_end) {
            float xq[4], xk[4];
            RW::widen4(R.q[3], xq);
            RW::widen4(R.k[3], xk);
            *reinterpret_cast<float4 *>(sXa + (0 * 3 + rr - 5) * DK + 4 * c4) = make_float4(xq[0], xq[1], xq[2], xq[3]);
            *reinterpret_cast<float4 *>(sXa + (1 * 3 + rr - 5) * DK + 4 * c4) = make_float4(xk[0], xk[1], xk[2], xk[3]);
        }

        umma::fence_before_sync();
        if (!__syncthreads_and(ok)) {
            ok = false;
            break;
        }
        umma::fence_after_sync();
        if (tid == kLoader && c0 + C < t_end) {
            issue_v(c0 + C);
            ++v_issued;
        }
        if (tid == kIssuer) {
#pragma unroll 1
            for (int ks = 0; ks < C / 8; ++ks)
                umma::mma_ts(tb + TM_D4, tb + TM_Z + ks * 8,
                             umma::smem_desc(sbase + T_M + ks * 256, 128, 8 * KB64), id64, ks > 0);
            umma::commit(&bar[2]);
            if (!ptx::mbar_wait(&bar[2], phase, ptx::kWaitBudget)) {
                raise_error(4u);
                ok = false;
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
            last_bar = 3;
            last_par = phase;
        }
        // the norm's output gate rows of this warp (4 w .. 4 w + 3) and weights, loaded
        // under the state-pass products
        float4 og[4], nw;
        if (NORM) {
            nw = __ldg(reinterpret_cast<const float4 *>(a.norm_w) + lane);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int t = 4 * warp + i;
                og[i] = c0 + t < T ? __ldg(reinterpret_cast<const float4 *>(a.out_gate + (((size_t)m * T + c0 + t) * a.H + h) * DK) + lane)
                                   : make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
        if (!ptx::mbar_wait(&bar[3], phase, ptx::kWaitBudget)) {
            raise_error(8u);
            ok = false;
        }
        umma::fence_after_sync();

        // ---------------------------------------------------------- 7. O out
        // O^T (tokens 16 hq .. + 15 at value channel j) -> staging rows -> one tensor store
        {
            float o16[16];
            umma::ld_x16(tq + TM_D3 + 64 + 16 * hq, o16);
            umma::wait_ld();
#pragma unroll
            for (int e = 0; e < 16; ++e) sO[(16 * hq + e) * DK + j] = a.scale * o16[e];
        }
        if (NORM) {  // y = o / sqrt(mean o^2 + eps) * w * sigmoid(gate), warp w: rows 4 w .. 4 w + 3
            if (!__syncthreads_and(ok)) {
                ok = false;
                break;
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int t = 4 * warp + i;
                float4 *row = reinterpret_cast<float4 *>(sO + t * DK) + lane;
                float4 o4 = *row;
                float ss = o4.x * o4.x + o4.y * o4.y + o4.z * o4.z + o4.w * o4.w;
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
                const float rn = rsqrtf(ss * (1.0f / DK) + a.norm_eps);
                const float4 g4 = og[i];
                o4.x = o4.x * rn * nw.x * sigm(g4.x);
                o4.y = o4.y * rn * nw.y * sigm(g4.y);
                o4.z = o4.z * rn * nw.z * sigm(g4.z);
                o4.w = o4.w * rn * nw.w * sigm(g4.w);
                *row = o4;
            }
        }
        umma::fence_smem_to_async();
        umma::fence_before_sync();
        if (warp == 0) ptx::named_bar_sync(kBarOut, NT);
        else ptx::named_bar_arrive(kBarOut, NT);
        if (tid == 0) {  // rows past T fall outside the tensor and are not written
            ptx::tma_store_4d(&mp.o, sO, 0, h, c0, m);
            ptx::bulk_commit();
        }
    }

    // Every thread arrives here (the loop ends, or breaks, for the whole CTA
    // at once); a wait that gave up after the last CTA-wide barrier of the
    // loop counts as well.
    const bool all_ok = __syncthreads_and(ok);
    // Before the shared and tensor memory go: the last tensor copies into
    // shared memory and the last tensor-core products have landed (at once
    // in a run without errors, where each was waited for already).
    if (tid == kLoader) {
        if (v_issued > 0) ptx::mbar_wait(&bar[4], (v_issued - 1) & 1, ptx::kDrainBudget);
        if (qka_issued > 0) ptx::mbar_wait(&bar[5], (qka_issued - 1) & 1, ptx::kDrainBudget);
    }
    if (tid == kIssuer && last_bar >= 0) ptx::mbar_wait(&bar[last_bar], last_par, ptx::kDrainBudget);

    // state out
    if (all_ok) {
        for (int c = 32 * hq; c < 32 * hq + 32; c += 8) {
            float v8[8];
            umma::ld_x8(tq + TM_S + c, v8);
            umma::wait_ld();
#pragma unroll
            for (int e = 0; e < 8; ++e) state[(size_t)(c + e) * DK + j] = v8[e];
        }
    }
    if (LAYER && all_ok && t_end == T && tid < 3 * DK) {  // conv cache <- the last three inputs of (cache, x)
        TQ *cache = static_cast<TQ *>(a.cache);
        const TQ *x = static_cast<const TQ *>(a.q);
        const int X = tid / DK, c = tid % DK;
        typename RW::V1 nv[3];
#pragma unroll
        for (int tap = 0; tap < 3; ++tap) {
            const int t = T - 3 + tap;
            nv[tap] = t >= 0 ? RW::load1(x + (((size_t)m * T + t) * 3 + X) * D + (size_t)h * DK + c)
                             : RW::load1(cache + ((size_t)m * 9 + 3 * X + t + 3) * D + (size_t)h * DK + c);
        }
#pragma unroll
        for (int tap = 0; tap < 3; ++tap)
            reinterpret_cast<typename RW::V1 *>(cache)[((size_t)m * 9 + 3 * X + tap) * D + (size_t)h * DK + c] = nv[tap];
    }
    if (tid == 0) ptx::bulk_wait_all();  // O stores complete before the CTA's shared memory goes
    umma::fence_before_sync();
    __syncthreads();
    if (warp == 0) umma::tmem_dealloc(tb, TM_COLS);
}

template <typename TQ, bool LAYER>
cudaError_t make_maps(const PrefillArgs &a, PrefillMaps *mp) {
    const bool bf16 = sizeof(TQ) == 2;
    const uint64_t H = a.H, T = a.T, M = a.M;
    const uint64_t d4[4] = {DK, H, T, M};   // [M][T][H][128]
    const uint64_t d5[5] = {DK, H, 3, T, M};  // [M][T][3][H*128]
    const uint32_t box_half[5] = {64, 1, 1, C, 1};  // 128 bytes of BF16 channels (swizzled)
    const uint32_t box_al[4] = {32, 1, C, 1};      // 128 bytes of FP32 channels (swizzled)
    const uint32_t box_row4[4] = {DK, 1, C, 1};
    const uint32_t box_row5[5] = {DK, 1, 1, C, 1};
    const uint32_t box_half4[4] = {64, 1, C, 1};
    cudaError_t e = cudaSuccess;
    memset(mp, 0, sizeof(PrefillMaps));
    if (LAYER) {
        e = make_tensor_map(&mp->v, a.q, bf16, 5, d5, box_row5, false);
        if (e == cudaSuccess && bf16) e = make_tensor_map(&mp->q, a.q, true, 5, d5, box_half, true);
    } else {
        e = make_tensor_map(&mp->v, a.v, bf16, 4, d4, box_row4, false);
        if (e == cudaSuccess && bf16) e = make_tensor_map(&mp->q, a.q, true, 4, d4, box_half4, true);
        if (e == cudaSuccess && bf16) e = make_tensor_map(&mp->k, a.k, true, 4, d4, box_half4, true);
    }
    if (e == cudaSuccess && bf16) e = make_tensor_map(&mp->alpha, a.alpha, false, 4, d4, box_al, true);
    if (e == cudaSuccess) e = make_tensor_map(&mp->o, a.o, false, 4, d4, box_row4, false);
    return e;
}

// Pieces per sequence. One CTA per SM walks one sequence's chunks one after
// another, so with more sequences than SMs the launch runs in waves and the
// last wave can leave SMs idle (256 sequences on 152 SMs: two waves, the
// second on 104 SMs). Cutting each sequence into P pieces of consecutive
// chunks and running the pieces in rounds of at most one per SM (piece p of
// every sequence before piece p + 1; the state passes from piece to piece in
// place, through the state buffer) balances the rounds. The cost model
// counts chunk steps on the busiest SM plus about 0.8 of a chunk per round
// (measured: the round boundary, state out and in, the first chunk's copies
// not yet overlapped). P = 1 whenever
// sequences do not outnumber SMs, so that every round holds at most one
// piece of a sequence.
int prefill_pieces(int sequences, int chunks, int sms) {
    if (sequences < sms || chunks < 2) return 1;
    int best = 1;
    double best_cost = 1e30;
    for (int p = 1; p <= 8 && p <= chunks; ++p) {
        const int per = (chunks + p - 1) / p;          // chunks per piece
        const int pieces = (chunks + per - 1) / per;   // pieces per sequence
        const int rounds = (sequences * pieces + sms - 1) / sms;
        const double cost = (double)rounds * per + 0.8 * rounds;
        if (cost < best_cost - 1e-9) {
            best_cost = cost;
            best = pieces;
        }
    }
    return best;
}

template <typename TQ, bool LAYER, bool NORM>
cudaError_t launch_tc_typed(const PrefillArgs &a, cudaStream_t stream) {
    PrefillMaps mp;
    cudaError_t e = make_maps<TQ, LAYER>(a, &mp);
    if (e != cudaSuccess) return e;
    auto kernel = kda_prefill_tc_kernel<TQ, LAYER, NORM>;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 0;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const int seqs = a.M * a.H, chunks = (a.T + C - 1) / C;
    const int pieces = prefill_pieces(seqs, chunks, sms);
    const int per = (chunks + pieces - 1) / pieces;
    const int items = seqs * ((chunks + per - 1) / per);
    // one launch per round of at most `sms` pieces when cut, else one launch
    // of one CTA per sequence
    const int round = pieces > 1 ? sms : items;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    for (int base = 0; base < items; base += round) {
        const int n = items - base < round ? items - base : round;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(n, 1, 1);
        cfg.blockDim = dim3(NT, 1, 1);
        cfg.dynamicSmemBytes = SMEM_BYTES;
        cfg.stream = stream;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, kernel, a, mp, base, per);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace

cudaError_t launch_prefill_tc(const PrefillArgs &a, int qkv_dtype, cudaStream_t stream) {
    if (qkv_dtype == KDA_BF16) return launch_tc_typed<__nv_bfloat16, false, false>(a, stream);
    return launch_tc_typed<float, false, false>(a, stream);
}

cudaError_t launch_prefill_layer(const PrefillArgs &a, int x_dtype, cudaStream_t stream) {
    if (x_dtype == KDA_BF16) {
        if (a.out_gate) return launch_tc_typed<__nv_bfloat16, true, true>(a, stream);
        return launch_tc_typed<__nv_bfloat16, true, false>(a, stream);
    }
    if (a.out_gate) return launch_tc_typed<float, true, true>(a, stream);
    return launch_tc_typed<float, true, false>(a, stream);
}

cudaError_t read_prefill_error(unsigned int *code) {
    return cudaMemcpyFromSymbol(code, g_prefill_error, sizeof(unsigned int));
}

cudaError_t clear_prefill_error() {
    const unsigned int zero = 0;
    return cudaMemcpyToSymbol(g_prefill_error, &zero, sizeof(unsigned int));
}

}  // namespace kda
