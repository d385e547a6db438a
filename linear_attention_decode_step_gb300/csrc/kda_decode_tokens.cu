// Multi-token KDA decode for sm_103a: T consecutive decode steps of one layer
// in one launch (conv + SiLU, L2 norm of q and k, the gated delta rule of
// "GLM-5.3 deep dive" section 8.2.3 Eq. 1 in the fade / predict / correct /
// read order of section 8.2.6, readout o = w + d (k.q)). Two kernels: short
// calls go token after token, as fla's fused-recurrent mode does for short
// inputs (section 8.2.5); calls of KDA_TOKENS_WY_MIN tokens or more take the
// same recurrence regrouped into chunks of up to 8 tokens (the WY
// representation and UT transform of section 8.2.4, exact in FP32 on CUDA
// cores), which passes over the state twice per chunk instead of four times
// per token.
//
// Every mbarrier wait is bounded (about two seconds of clock cycles). A
// thread whose wait gives up sets this file's device error word; the group's
// next barrier ANDs every thread's outcome, so the whole group leaves the
// loop together, before anything of that head is written. At exit the CTA
// meets once more and one thread waits (bounded) for the latest bulk copy
// into every stage. kda_device_error() reports the error word on the host.

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>

#include "../../include/kda.h"
#include "kda_internal.cuh"
#include "kda_ptx.cuh"

// Calls of at least this many tokens take the chunked kernel, shorter ones
// the token-by-token kernel.
#ifndef KDA_TOKENS_WY_MIN
#define KDA_TOKENS_WY_MIN 3
#endif

namespace kda {

__device__ unsigned int g_tokens_error;

namespace {

constexpr int DK = kHeadDim;
constexpr float kL2Eps = 1e-6f;
constexpr int kSmemLimit = 232448;               // 227 KiB opt-in per CTA
constexpr int kWarps = 16;

__device__ __forceinline__ uint32_t bf16x2_rn(float lo, float hi) {
    __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&p);
}
__device__ __forceinline__ float widen(float v) { return v; }
__device__ __forceinline__ float widen(__nv_bfloat16 v) { return __bfloat162float(v); }
__device__ __forceinline__ void raise_error(unsigned int code) { atomicOr(&g_tokens_error, code); }

// ---------------------------------------------------------------------------
// Organisation: persistent CTAs (one per SM) of 16 warps in two groups that
// take whole heads in turn; each head's state and conv cache arrive through a
// ring of shared-memory stages filled by cp.async.bulk (mbarrier-completed,
// the same ring protocol as the single-step streaming kernel). Layout chosen
// for many steps per head:
//  * A head's state is read once into registers, updated T times and written
//    once; the conv window of each channel also stays in registers.
//  * Warp cw of a group owns value columns 16 cw .. 16 cw + 15 for all 128
//    key rows: lane (rl, cc) = (lane / 4, lane % 4) holds columns 16 cw +
//    4 cc .. + 3 of rows rl + 8 r (r = 0 .. 15). The column sums u = k.s and
//    w = q.s then reduce inside the warp (three shuffle levels that halve the
//    values each time, so lane rl ends up with u (rl < 4) or w (rl >= 4) of
//    column 4 cc + rl % 4), and each warp runs its columns on its own.
//  * While a group's warps update the state with token t, its threads
//    convolve token t + 1 into the other half of a double buffer (q, k and
//    alpha stored row-permuted so a lane's 16 rows are contiguous); one group
//    barrier per token hands the buffer over.
//  * x, alpha and beta of later tokens are loaded into registers two tokens
//    ahead of their convolution (one token ahead left the load latency
//    exposed: about a sixth of the time at T = 8).
// ---------------------------------------------------------------------------
template <typename TS, typename TX, int G_>
struct TokCfg {
    static constexpr int G = G_;
    static constexpr int CWARPS = kWarps / G;          // warps per group (16 columns each)
    static constexpr int GT = CWARPS * 32;
    static constexpr int THREADS = kWarps * 32;
    static_assert(CWARPS * 16 == DK, "a group's warps cover the 128 value columns");
    static constexpr int S_BYTES = DK * DK * (int)sizeof(TS);
    static constexpr int C_OFF = S_BYTES;
    static constexpr int STAGE = C_OFF + 9 * DK * (int)sizeof(TX);
    // per group, two token buffers of: q, k (row-permuted) | alpha (row-permuted) | v;
    // then the head's conv weights [384] (float4, one per channel of q, k, v)
    // and the conv windows [3][384] (three most recent inputs per channel)
    static constexpr int BUF_F = 4 * DK;
    static constexpr int W_OFF = 2 * BUF_F * 4;
    static constexpr int WIN_OFF = W_OFF + 3 * DK * 16;
    static constexpr int WORK_BYTES = WIN_OFF + ((9 * DK * (int)sizeof(TX) + 15) / 16) * 16;
    static constexpr int BAR_BYTES = 2 * 8 * 8 + 8 * 4;  // full[8], issued[8], fills[8]
    static constexpr int NST_FIT = (kSmemLimit - BAR_BYTES - G * WORK_BYTES) / STAGE;
    static constexpr int NST = NST_FIT > 6 ? 6 : NST_FIT;
    static constexpr int SMEM = NST * STAGE + G * WORK_BYTES + BAR_BYTES;
    static_assert(NST >= 2, "at least two stages must fit");
    static_assert(STAGE % 16 == 0 && WORK_BYTES % 16 == 0, "16-byte alignment");
};

// Position of key row i in a row-permuted buffer: rows rl + 8 r (r = 0..15)
// of lane group rl are contiguous at 16 rl.
__device__ __forceinline__ int perm_row(int i) { return (i & 7) * 16 + (i >> 3); }

// Four consecutive state columns of one row: 16 bytes (FP32) or 8 bytes (BF16).
template <typename TS> struct Quad;
template <> struct Quad<float> {
    __device__ __forceinline__ static void load(const float *p, float (&f)[4]) {
        const float4 v = *reinterpret_cast<const float4 *>(p);
        f[0] = v.x; f[1] = v.y; f[2] = v.z; f[3] = v.w;
    }
    __device__ __forceinline__ static void store(float *p, const float (&f)[4]) {
        __stcs(reinterpret_cast<float4 *>(p), make_float4(f[0], f[1], f[2], f[3]));
    }
};
template <> struct Quad<__nv_bfloat16> {
    __device__ __forceinline__ static void load(const __nv_bfloat16 *p, float (&f)[4]) {
        const uint2 v = *reinterpret_cast<const uint2 *>(p);
        f[0] = __uint_as_float(v.x << 16); f[1] = __uint_as_float(v.x & 0xffff0000u);
        f[2] = __uint_as_float(v.y << 16); f[3] = __uint_as_float(v.y & 0xffff0000u);
    }
    __device__ __forceinline__ static void store(__nv_bfloat16 *p, const float (&f)[4]) {
        __stcs(reinterpret_cast<uint2 *>(p), make_uint2(bf16x2_rn(f[0], f[1]), bf16x2_rn(f[2], f[3])));
    }
};

// Copies of head u's state (one bulk copy) and conv cache into stage `st`:
// the cache by one tensor copy through `cmap` ([M][9][H*128] in boxes of 128
// channels x 9 taps) or, without a map, by nine bulk copies of a row each.
// The conv cache's tensor map for the token-by-token kernel, used when `on`.
struct TokCacheMap {
    CUtensorMap map;
    int on;
};

template <typename TS, typename TX, int G>
__device__ __forceinline__ void load_head_tokens(unsigned char *st, uint64_t *bar,
                                                 const DecodeArgs &a, int u, uint64_t pol,
                                                 const CUtensorMap *cmap) {
    using C = TokCfg<TS, TX, G>;
    const int H = a.H;
    const size_t D = (size_t)H * DK;
    const int m = u / H, h = u - m * H;
    const TX *cache = static_cast<const TX *>(a.cache);
    ptx::mbar_arrive_expect_tx(bar, C::STAGE);
    ptx::bulk_g2s_hint(st, static_cast<const TS *>(a.state) + (size_t)u * DK * DK, C::S_BYTES, bar,
                       pol);
    if (cmap) {
        ptx::tma_load_4d(st + C::C_OFF, cmap, bar, h * DK, 0, m, 0);
        return;
    }
#pragma unroll
    for (int j = 0; j < 9; ++j)
        ptx::bulk_g2s(st + C::C_OFF + j * DK * sizeof(TX),
                      cache + ((size_t)m * 9 + j) * D + (size_t)h * DK, DK * sizeof(TX), bar);
}

template <typename TX> __device__ __forceinline__ TX zero_tx();
template <> __device__ __forceinline__ float zero_tx<float>() { return 0.f; }
template <> __device__ __forceinline__ __nv_bfloat16 zero_tx<__nv_bfloat16>() {
    return __float2bfloat16_rn(0.f);
}

template <typename TX>
__device__ __forceinline__ float conv_silu(const float4 w, const TX (&win)[3], TX xt) {
    const float pre = w.x * widen(win[0]) + w.y * widen(win[1]) + w.z * widen(win[2]) + w.w * widen(xt);
    return __fdividef(pre, 1.0f + __expf(-pre));
}

// The exit wait: for the latest bulk copy into every stage to have landed
// (one thread; in a run without errors they all have, and it returns at
// once). Kept out of line so the kernel's loop keeps its registers.
template <typename C>
__device__ __noinline__ void drain_fills(unsigned char *smem) {
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::NST * C::STAGE + C::G * C::WORK_BYTES);
    const volatile uint32_t *fills = reinterpret_cast<const volatile uint32_t *>(full + 16);
    for (int s = 0; s < C::NST; ++s) {
        const uint32_t f = fills[s];
        if (f > 0) ptx::mbar_wait(&full[s], (f - 1) & 1, ptx::kDrainBudget);
    }
}

template <typename TS, typename TX, int G>
__global__ void __launch_bounds__(TokCfg<TS, TX, G>::THREADS, 1)
kda_decode_tokens_kernel(const DecodeArgs a, const int T, const __grid_constant__ TokCacheMap cm) {
    using C = TokCfg<TS, TX, G>;
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::NST * C::STAGE + G * C::WORK_BYTES);
    uint64_t *issued = full + 8;
    // bulk copies issued into each stage so far (written by the issuing
    // thread before it arrives on `issued`; read after the exit barrier)
    volatile uint32_t *fills = reinterpret_cast<volatile uint32_t *>(issued + 8);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int H = a.H;
    const int n_units = a.M * H;
    const size_t D = (size_t)H * DK;
    const uint64_t pol = ptx::policy_evict_first();

    if (tid == 0) {
        for (int s = 0; s < C::NST; ++s) {
            ptx::mbar_init(&full[s], 1);
            ptx::mbar_init(&issued[s], 1);
            fills[s] = blockIdx.x + s * gridDim.x < n_units ? 1u : 0u;  // the first fills, below
        }
        ptx::fence_mbar_init();
    }
    // warm L2 with the first heads' state while the previous grid drains (a
    // hint only: L2 also receives whatever the previous grid writes)
    if (tid == 0) {
        for (int s = 0; s < C::NST; ++s) {
            const int u = blockIdx.x + s * gridDim.x;
            if (u < n_units)
                ptx::bulk_prefetch_l2(static_cast<const TS *>(a.state) + (size_t)u * DK * DK, C::S_BYTES);
        }
    }
    __syncthreads();
    ptx::grid_dependency_wait();
    ptx::launch_dependents();
    if (tid == 0) {
        for (int s = 0; s < C::NST; ++s) {
            const int u = blockIdx.x + s * gridDim.x;
            if (u < n_units) load_head_tokens<TS, TX, G>(smem + s * C::STAGE, &full[s], a, u, pol, cm.on ? &cm.map : nullptr);
        }
    }

    const int g = warp / C::CWARPS;
    const int ct = tid - g * C::GT;
    const int cw = ct >> 5;
    const int rl = lane >> 2, cc = lane & 3;
    const int col0 = 16 * cw + 4 * cc;          // this lane's four value columns
    const int ocol = 16 * cw + 4 * cc + (rl & 3);  // the column whose total this lane ends with
    const uint32_t bar_id = 1 + g;
    float *buf = reinterpret_cast<float *>(smem + C::NST * C::STAGE + g * C::WORK_BYTES);
    float4 *wsm = reinterpret_cast<float4 *>(smem + C::NST * C::STAGE + g * C::WORK_BYTES + C::W_OFF);
    TX *win = reinterpret_cast<TX *>(smem + C::NST * C::STAGE + g * C::WORK_BYTES + C::WIN_OFF);
    const TX *x = static_cast<const TX *>(a.x);
    TX *cache = static_cast<TX *>(a.cache);
    const float4 *w4 = reinterpret_cast<const float4 *>(a.conv_w);

    // conv channels of this thread (c < 384: tensor c / 128, channel c % 128)
    const int c0 = ct, c1 = ct + C::GT;
    const bool has0 = c0 < 3 * DK, has1 = c1 < 3 * DK;
    const int X0 = c0 / DK, ch0 = c0 % DK, X1 = c1 / DK, ch1 = c1 % DK;
    // where this thread's conv outputs go in a token buffer
    const int dst0 = X0 < 2 ? X0 * DK + perm_row(ch0) : 3 * DK + ch0;
    const int dst1 = X1 < 2 ? X1 * DK + perm_row(ch1) : 3 * DK + ch1;

    for (int i = g, u = blockIdx.x + g * gridDim.x; u < n_units; i += G, u += G * gridDim.x) {
        const int s = i % C::NST, n = i / C::NST;
        const int m = u / H, h = u - m * H;
        const size_t hb = (size_t)h * DK;
        // per-token input pointers of this head (token stride: 3 D, H DK, H)
        // (channel c1 is v channel ct, 2 D - X0 D + ct - ch0 elements after c0's)
        const TX *xp0 = x + ((size_t)m * T * 3 + X0) * D + hb + ch0;
        const int off1 = (2 - X0) * (int)D + ct - ch0;
        const float *ap = a.alpha + ((size_t)m * T * H + h) * DK + (ct & (DK - 1));
        const float *bp = a.beta + (size_t)m * T * H + h;
        const size_t xs = 3 * D, as = (size_t)H * DK;
        // conv weights of this head, parked in shared memory (each thread reads
        // back only what it wrote)
        if (has0) wsm[c0] = __ldg(w4 + (size_t)X0 * D + hb + ch0);
        if (has1) wsm[c1] = __ldg(w4 + (size_t)X1 * D + hb + ch1);
        // inputs of tokens 0 and 1, loaded while the stage lands
        const TX x00 = has0 ? xp0[0] : zero_tx<TX>();
        const TX x10 = has1 ? xp0[off1] : zero_tx<TX>();
        const float a0 = ct < DK ? __ldg(ap) : 0.f;
        float beta_c = __ldg(bp), beta_n = 0.f, beta_m = 0.f;
        TX xn0 = zero_tx<TX>(), xn1 = zero_tx<TX>(), xm0 = zero_tx<TX>(), xm1 = zero_tx<TX>();
        float an = 0.f, am = 0.f;
        if (T > 1) {
            if (has0) xn0 = xp0[xs];
            if (has1) xn1 = xp0[xs + off1];
            if (ct < DK) an = __ldg(ap + as);
            beta_n = __ldg(bp + H);
        }
        if (T > 2) {
            if (has0) xm0 = xp0[2 * xs];
            if (has1) xm1 = xp0[2 * xs + off1];
            if (ct < DK) am = __ldg(ap + 2 * as);
            beta_m = __ldg(bp + 2 * H);
        }

        // the stage's refill was issued, then its bytes landed (a thread whose
        // wait gives up goes on to the group barrier below, where the group
        // leaves together; nothing reaches global memory before it)
        const bool landed = (n == 0 || ptx::mbar_wait(&issued[s], (n - 1) & 1, ptx::kWaitBudget)) &&
                            ptx::mbar_wait(&full[s], n & 1, ptx::kWaitBudget);
        if (!landed) raise_error(8u);
        const unsigned char *st = smem + s * C::STAGE;
        const TS *Ss = reinterpret_cast<const TS *>(st);
        const TX *cs = reinterpret_cast<const TX *>(st + C::C_OFF);

        float *op = a.o + ((size_t)m * T * H + h) * DK + ocol;
        // the state as column pairs: the FP32 arithmetic below runs on packed
        // pairs (fma.rn.f32x2 / mul.rn.f32x2: two exactly rounded FP32
        // operations per instruction)
        float2 sv[16][2];
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            float f4[4];
            Quad<TS>::load(Ss + (rl + 8 * r) * DK + col0, f4);
            sv[r][0] = make_float2(f4[0], f4[1]);
            sv[r][1] = make_float2(f4[2], f4[3]);
        }
        // conv windows (oldest first, exactly as stored); each thread owns its channels' slots
#pragma unroll
        for (int j = 0; j < 3; ++j) {
            if (has0) win[j * 3 * DK + c0] = cs[(X0 * 3 + j) * DK + ch0];
            if (has1) win[j * 3 * DK + c1] = cs[(X1 * 3 + j) * DK + ch1];
        }
        // convolve the buffered inputs of one token into a token buffer
        auto convolve = [&](float *b, float al, TX xa, TX xb) {
            if (has0) {
                const TX w0 = win[c0], w1 = win[3 * DK + c0], w2 = win[6 * DK + c0];
                const TX wv[3] = {w0, w1, w2};
                b[dst0] = conv_silu(wsm[c0], wv, xa);
                win[c0] = w1;
                win[3 * DK + c0] = w2;
                win[6 * DK + c0] = xa;
            }
            if (has1) {
                const TX w0 = win[c1], w1 = win[3 * DK + c1], w2 = win[6 * DK + c1];
                const TX wv[3] = {w0, w1, w2};
                b[dst1] = conv_silu(wsm[c1], wv, xb);
                win[c1] = w1;
                win[3 * DK + c1] = w2;
                win[6 * DK + c1] = xb;
            }
            if (ct < DK) b[2 * DK + perm_row(ct)] = al;
        };
        convolve(buf, a0, x00, x10);
        // stage read; token 0 in buffer 0; every thread's wait succeeded
        // (after a wait gave up anywhere in the group: the group finishes this
        // head without writing anything and without a refill, and the loop's
        // condition then ends it)
        const bool go = ptx::named_bar_and(bar_id, C::GT, landed);
        if (!go) u = n_units;
        if (ct == 0 && go) {
            const int ur = blockIdx.x + (i + C::NST) * gridDim.x;
            if (ur < n_units) {
                load_head_tokens<TS, TX, G>(smem + s * C::STAGE, &full[s], a, ur, pol, cm.on ? &cm.map : nullptr);
                fills[s] = fills[s] + 1u;
                ptx::mbar_arrive(&issued[s]);
            }
        }

        for (int t = 0; t < T; ++t) {
            const float *bc = buf + (t & 1) * C::BUF_F;
            const float beta = beta_c;
            if (t + 1 < T) {  // convolve token t + 1 into the other buffer, load token t + 3
                convolve(buf + ((t + 1) & 1) * C::BUF_F, an, xn0, xn1);
                beta_c = beta_n;
                xn0 = xm0;
                xn1 = xm1;
                an = am;
                beta_n = beta_m;
                if (t + 3 < T) {
                    if (has0) xm0 = xp0[(size_t)(t + 3) * xs];
                    if (has1) xm1 = xp0[(size_t)(t + 3) * xs + off1];
                    if (ct < DK) am = __ldg(ap + (size_t)(t + 3) * as);
                    beta_m = __ldg(bp + (size_t)(t + 3) * H);
                }
            }
            const float *qb = bc + 16 * rl, *kb = bc + DK + 16 * rl, *ab = bc + 2 * DK + 16 * rl;

            // norms: lane covers rows of quarter cc, then a full-warp sum
            float sq, sk, sqk;
            {
                const float4 q4 = *reinterpret_cast<const float4 *>(qb + 4 * cc);
                const float4 k4 = *reinterpret_cast<const float4 *>(kb + 4 * cc);
                sq = q4.x * q4.x + q4.y * q4.y + q4.z * q4.z + q4.w * q4.w;
                sk = k4.x * k4.x + k4.y * k4.y + k4.z * k4.z + k4.w * k4.w;
                sqk = q4.x * k4.x + q4.y * k4.y + q4.z * k4.z + q4.w * k4.w;
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                sq += __shfl_xor_sync(0xffffffffu, sq, off);
                sk += __shfl_xor_sync(0xffffffffu, sk, off);
                sqk += __shfl_xor_sync(0xffffffffu, sqk, off);
            }
            const float rq = rsqrtf(sq + kL2Eps);
            const float rk = rsqrtf(sk + kL2Eps);

            // fade, then raw column sums over this lane's 16 rows
            float2 uu2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
            float2 ww2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
            for (int r4 = 0; r4 < 4; ++r4) {
                const float4 q4 = *reinterpret_cast<const float4 *>(qb + 4 * r4);
                const float4 k4 = *reinterpret_cast<const float4 *>(kb + 4 * r4);
                const float4 a4 = *reinterpret_cast<const float4 *>(ab + 4 * r4);
                const float qv[4] = {q4.x, q4.y, q4.z, q4.w}, kv[4] = {k4.x, k4.y, k4.z, k4.w};
                const float av[4] = {a4.x, a4.y, a4.z, a4.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int r = 4 * r4 + e;
                    const float2 a2 = make_float2(av[e], av[e]);
                    const float2 k2 = make_float2(kv[e], kv[e]);
                    const float2 q2 = make_float2(qv[e], qv[e]);
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
                        sv[r][c] = __fmul2_rn(sv[r][c], a2);
                        uu2[c] = __ffma2_rn(k2, sv[r][c], uu2[c]);
                        ww2[c] = __ffma2_rn(q2, sv[r][c], ww2[c]);
                    }
                }
            }
            const float uu[4] = {uu2[0].x, uu2[0].y, uu2[1].x, uu2[1].y};
            const float ww[4] = {ww2[0].x, ww2[0].y, ww2[1].x, ww2[1].y};
            // reduce over the 8 lane groups rl, halving the values at each level
            const bool b2 = lane & 16, b1 = lane & 8, b0 = lane & 4;
            float x4[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float send = b2 ? uu[e] : ww[e];
                x4[e] = (b2 ? ww[e] : uu[e]) + __shfl_xor_sync(0xffffffffu, send, 16);
            }
            float y2[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const float send = b1 ? x4[e] : x4[e + 2];
                y2[e] = (b1 ? x4[e + 2] : x4[e]) + __shfl_xor_sync(0xffffffffu, send, 8);
            }
            const float z = (b0 ? y2[1] : y2[0]) + __shfl_xor_sync(0xffffffffu, b0 ? y2[0] : y2[1], 4);
            // lanes rl < 4: u of column ocol -> d; lanes rl >= 4: w of column ocol -> o
            float d = 0.f;
            if (!b2) d = beta * (bc[3 * DK + ocol] - rk * z);
            const float d_o = __shfl_xor_sync(0xffffffffu, d, 16);
            if (b2 && go) op[(size_t)t * as] = a.scale * (rq * z + d_o * (sqk * rq * rk));
            // S' = s + k_hat d: k_hat = rk k, so scale d by rk once
            const float dk = d * rk;
            float dd[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) dd[e] = __shfl_sync(0xffffffffu, dk, 4 * e + cc);
            const float2 dd2[2] = {make_float2(dd[0], dd[1]), make_float2(dd[2], dd[3])};
#pragma unroll
            for (int r4 = 0; r4 < 4; ++r4) {
                const float4 k4 = *reinterpret_cast<const float4 *>(kb + 4 * r4);
                const float kv[4] = {k4.x, k4.y, k4.z, k4.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 k2 = make_float2(kv[e], kv[e]);
#pragma unroll
                    for (int c = 0; c < 2; ++c) sv[4 * r4 + e][c] = __ffma2_rn(k2, dd2[c], sv[4 * r4 + e][c]);
                }
            }
            ptx::named_bar_sync(bar_id, C::GT);  // token t + 1 convolved; buffer t free
        }

        // state out (rounded once, here, for BF16 storage) and the final conv windows
        if (!go) continue;
        TS *Sg = static_cast<TS *>(a.state) + (size_t)u * DK * DK + col0;
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            const float f4[4] = {sv[r][0].x, sv[r][0].y, sv[r][1].x, sv[r][1].y};
            Quad<TS>::store(Sg + (size_t)(rl + 8 * r) * DK, f4);
        }
        const size_t cbase = (size_t)m * 9 * D + hb;
#pragma unroll
        for (int j = 0; j < 3; ++j) {
            if (has0) cache[cbase + (size_t)(3 * X0 + j) * D + ch0] = win[j * 3 * DK + c0];
            if (has1) cache[cbase + (size_t)(3 * X1 + j) * D + ch1] = win[j * 3 * DK + c1];
        }
    }

    // Exit: once both groups are here no thread issues another bulk copy, so
    // waiting for the latest fill of every stage covers any still in flight
    // after a wait gave up (without errors they have all landed already).
    __syncthreads();
    if (threadIdx.x == 0) drain_fills<C>(smem);
}

// ---------------------------------------------------------------------------
// Chunked form for several tokens per head: the WY representation with the
// UT transform of "GLM-5.3 deep dive" section 8.2.4, on CUDA cores in exact
// FP32, for chunks of up to CT = 8 tokens. Within a chunk with state S0 at
// its start, write R(t, j) = prod_{s = j+1 .. t} alpha_s (per key row; empty
// product 1) and Gamma_t = R(t, -1). Then, with k and q L2-normalised,
//   u_j   = (Gamma_j k_j) . S0 + sum_{i<j} A_ji d_i,  A_ji = sum_c k_jc k_ic R_c(j, i)
//   d_j   = beta_j (v_j - u_j)                      (forward substitution)
//   o_t   = scale ((Gamma_t q_t) . S0 + sum_{j<=t} P_tj d_j),  P_tj = sum_c q_tc k_jc R_c(t, j)
//   S_end = Gamma_last S0 + sum_j (k_j R(last, j)) d_j^T
// which is the token-by-token recurrence regrouped (no approximation). The
// decay ratios are formed as products of alphas, never as quotients, so no
// factor exceeds 1.
//
// Per chunk a group runs three phases:
//  P1 (thread per channel): conv + SiLU of the chunk's q, k (one channel
//     each) and v (one channel, half the tokens), alpha and beta into shared
//     memory (with BF16 inputs, x and alpha of the chunk were copied into
//     shared memory by two tensor copies one thread issued one chunk earlier,
//     on a per-group mbarrier; with FP32 state the head's conv cache comes
//     with its first chunk's inputs in a third one);            group barrier
//  P2 (warp t per token t): the norms of q_t, k_t, the rows A_t. and P_t. (raw,
//     unnormalised), and Gamma_t q_t, Gamma_t k_t, k_t R(last, t), Gamma_last
//     into row-permuted buffers; at a head's first chunk the state from its
//     stage into registers;                                     group barrier
//  P3 (the state in registers, warp cw owning value columns 16 cw .. + 15 of
//     all 128 key rows as in the token-by-token kernel): one pass forms the
//     2 x CT column sums (Gamma k) . S0 and (Gamma q) . S0 and reduces them
//     inside the warp; lanes holding u-side sums solve for d of their column,
//     lanes holding q-side sums form o; a second pass applies the fade and
//     the rank-CT update. No barrier: each warp owns its columns.
// The norms are applied by the consumers: with rq, rk the inverse norms,
// X_raw = (Gamma k_raw) . S0 and d'_j = rk_j d_j,
//   d_j = beta_j (v_j - rk_j (X_raw_j + sum_{i<j} A_raw_ji d'_i)),
//   o_t = scale rq_t (Y_raw_t + sum_{j<=t} P_raw_tj d'_j),
//   S_end = Gamma_last S0 + sum_j (k_raw_j R(last, j)) d'_j^T.
// ---------------------------------------------------------------------------
// Tensor maps of the staged inputs (encoded on the host per call): x as
// [M][T][3][H*128] in boxes of 128 channels x 3 tensors x (CT + 3) tokens,
// alpha as [M][T][H][128] in boxes of 128 channels x CT tokens, and the conv
// cache as [M][9][H*128] in boxes of 128 channels x 9 taps (FP32 state: with
// a head's first chunk of inputs; BF16 state: into the head's stage).
struct TokMaps {
    CUtensorMap x;
    CUtensorMap alpha;
    CUtensorMap cache;
};

template <typename TS, typename TX>
struct WyCfg {
    static constexpr int G = 2;
    static constexpr int CWARPS = kWarps / G;          // 8 warps, 16 value columns each
    static constexpr int GT = CWARPS * 32;
    static constexpr int THREADS = kWarps * 32;
    static constexpr int CT = 8;                       // tokens per chunk: one per warp in P2
    static_assert(CT == CWARPS && CWARPS * 16 == DK, "one warp per token, 16 columns per warp");
    // With BF16 inputs the next chunk's inputs are staged in shared memory by
    // tensor copies issued a chunk ahead (FP32 inputs would need twice the room);
    static constexpr bool kStageX = sizeof(TX) == 2;
    // With FP32 state (one stage per group) the conv cache arrives with them
    // too, so a stage holds only the state and is waited for where it is read
    // (BF16 state: two stages per group arrive early enough; measured slower)
    static constexpr bool kCacheX = kStageX && sizeof(TS) == 4;
    static constexpr int S_BYTES = DK * DK * (int)sizeof(TS);
    static constexpr int C_OFF = S_BYTES;
    static constexpr int STAGE = kCacheX ? S_BYTES : C_OFF + 9 * DK * (int)sizeof(TX);
    // row-permuted vectors: lane group rl's 16 rows at 16 rl + 4 (rl / 2), so
    // the 8 groups' 16-byte reads fall into 8 different bank quads
    static constexpr int VP = 144;
    // per group (floats): q | k conv outputs [CT][256] (channel order; during
    // P3 a warp keeps d' of its 16 columns in its own 32-float slots of each
    // row, which only its own threads write in P1), alpha [CT][128], v
    // [2][CT][128] and beta [2][CT] (by chunk parity: P3 of one chunk may still
    // read them while P1 of the next writes), Gamma q, Gamma k, k R(last, .)
    // [CT][VP], Gamma_last [VP], per token the P row, A row, rq, rk [CT][32],
    // and with staged inputs x of tokens t0 - 3 .. t0 + CT - 1 [CT + 3][3][128]
    // (the tensor copy's box order; XS and alpha start at 128-byte offsets)
    static constexpr int QK_F = 0;
    static constexpr int DXS = 2 * DK;             // row stride of the d' slots
    static constexpr int AL_F = QK_F + CT * 2 * DK;
    static constexpr int V_F = AL_F + CT * DK;
    static constexpr int BT_F = V_F + 2 * CT * DK;
    static constexpr int QD_F = BT_F + 2 * CT;
    static constexpr int KD_F = QD_F + CT * VP;
    static constexpr int KE_F = KD_F + CT * VP;
    static constexpr int GL_F = KE_F + CT * VP;
    static constexpr int RED_F = GL_F + VP;
    static constexpr int XS_F = RED_F + CT * 32;
    static constexpr int XS_BYTES = kStageX ? 3 * (CT + 3) * DK * (int)sizeof(TX) : 0;
    static constexpr int CS_F = XS_F + XS_BYTES / 4;
    static constexpr int CS_BYTES = kCacheX ? 9 * DK * (int)sizeof(TX) : 0;
    static constexpr int WORK_F = CS_F + CS_BYTES / 4;
    static constexpr int WORK_BYTES = WORK_F * 4;
    // full[8], issued[8], fills[8], then the input barriers xin[2] and their
    // fill counts [2]
    static constexpr int BAR_BYTES = 2 * 8 * 8 + 8 * 4 + 2 * 8 + 2 * 4 + 8;
    static constexpr int NST_FIT = (kSmemLimit - BAR_BYTES - G * WORK_BYTES) / STAGE;
    static constexpr int NST = NST_FIT > 6 ? 6 : NST_FIT;
    static constexpr int SMEM = NST * STAGE + G * WORK_BYTES + BAR_BYTES;
    static_assert(NST >= 2, "at least two stages must fit");
    static_assert(QD_F % 4 == 0 && STAGE % 16 == 0 && WORK_BYTES % 128 == 0 && XS_F % 32 == 0 &&
                      AL_F % 32 == 0 && (NST * STAGE) % 128 == 0,
                  "16-byte alignment; 128-byte tensor-copy destinations");
    static_assert(kCacheX || STAGE == TokCfg<TS, TX, G>::STAGE, "the stage layout of load_head_tokens");
    static_assert(CS_F % 32 == 0, "128-byte tensor-copy destination");
};

// A stage of the chunked kernel: the head's state (and, unless the conv cache
// arrives with the staged inputs, the cache as in load_head_tokens).
template <typename TS, typename TX, typename C>
__device__ __forceinline__ void load_stage_wy(unsigned char *st, uint64_t *bar, const DecodeArgs &a,
                                              const TokMaps &mp, int u, uint64_t pol) {
    if constexpr (C::kCacheX) {
        ptx::mbar_arrive_expect_tx(bar, C::S_BYTES);
        ptx::bulk_g2s_hint(st, static_cast<const TS *>(a.state) + (size_t)u * DK * DK, C::S_BYTES, bar, pol);
    } else {
        load_head_tokens<TS, TX, C::G>(st, bar, a, u, pol, C::kStageX ? &mp.cache : nullptr);
    }
}

__device__ __forceinline__ int wy_base(int rl) { return 16 * rl + 4 * (rl >> 1); }
__device__ __forceinline__ int wy_pos(int i) { return wy_base(i & 7) + (i >> 3); }

template <typename TX>
__device__ __forceinline__ float conv4(const float4 w, TX a0, TX a1, TX a2, TX a3) {
    const float pre = w.x * widen(a0) + w.y * widen(a1) + w.z * widen(a2) + w.w * widen(a3);
    return __fdividef(pre, 1.0f + __expf(-pre));
}

__device__ __forceinline__ float dot4(const float4 a, const float4 b) {
    return a.x * b.x + a.y * b.y + a.z * b.z + a.w * b.w;
}
__device__ __forceinline__ float4 mul4(const float4 a, const float4 b) {
    return make_float4(a.x * b.x, a.y * b.y, a.z * b.z, a.w * b.w);
}

// Sums v[0..15] over the 32 lanes of a warp; lane L returns the total of
// v[(L >> 1) & 15] (halving exchanges, then one full one).
__device__ __forceinline__ float warp_sum16(const float (&v)[16], int lane) {
    constexpr unsigned F = 0xffffffffu;
    float v8[8], v4[4], v2[2];
    const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4, b1 = lane & 2;
#pragma unroll
    for (int i = 0; i < 8; ++i)
        v8[i] = (b4 ? v[i + 8] : v[i]) + __shfl_xor_sync(F, b4 ? v[i] : v[i + 8], 16);
#pragma unroll
    for (int i = 0; i < 4; ++i)
        v4[i] = (b3 ? v8[i + 4] : v8[i]) + __shfl_xor_sync(F, b3 ? v8[i] : v8[i + 4], 8);
#pragma unroll
    for (int i = 0; i < 2; ++i)
        v2[i] = (b2 ? v4[i + 2] : v4[i]) + __shfl_xor_sync(F, b2 ? v4[i] : v4[i + 2], 4);
    const float v1 = (b1 ? v2[1] : v2[0]) + __shfl_xor_sync(F, b1 ? v2[0] : v2[1], 2);
    return v1 + __shfl_xor_sync(F, v1, 1);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    return v;
}

template <typename TS, typename TX, bool MULTI>
__global__ void __launch_bounds__(WyCfg<TS, TX>::THREADS, 1)
kda_decode_tokens_wy_kernel(const DecodeArgs a, const int T, const __grid_constant__ TokMaps mp) {
    using C = WyCfg<TS, TX>;
    constexpr int G = C::G, CT = C::CT, VP = C::VP;
    constexpr bool kRowPairs = sizeof(TS) == 2;
    constexpr unsigned FULL = 0xffffffffu;
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::NST * C::STAGE + G * C::WORK_BYTES);
    uint64_t *issued = full + 8;
    volatile uint32_t *fills = reinterpret_cast<volatile uint32_t *>(issued + 8);
    // staged inputs: per group an mbarrier and the number of fills issued into it
    uint64_t *xin = full + 20;
    volatile uint32_t *xfills = reinterpret_cast<volatile uint32_t *>(full + 22);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int H = a.H;
    const int n_units = a.M * H;
    const size_t D = (size_t)H * DK;
    const uint64_t pol = ptx::policy_evict_first();

    if (tid == 0) {
        for (int s = 0; s < C::NST; ++s) {
            ptx::mbar_init(&full[s], 1);
            ptx::mbar_init(&issued[s], 1);
            fills[s] = blockIdx.x + s * gridDim.x < n_units ? 1u : 0u;
        }
        for (int gg = 0; gg < G; ++gg) {
            ptx::mbar_init(&xin[gg], 1);
            xfills[gg] = 0u;
        }
        ptx::fence_mbar_init();
        for (int s = 0; s < C::NST; ++s) {
            const int u = blockIdx.x + s * gridDim.x;
            if (u < n_units)
                ptx::bulk_prefetch_l2(static_cast<const TS *>(a.state) + (size_t)u * DK * DK, C::S_BYTES);
        }
    }
    __syncthreads();
    ptx::grid_dependency_wait();
    ptx::launch_dependents();
    if (tid == 0) {
        for (int s = 0; s < C::NST; ++s) {
            const int u = blockIdx.x + s * gridDim.x;
            if (u < n_units) load_stage_wy<TS, TX, C>(smem + s * C::STAGE, &full[s], a, mp, u, pol);
        }
    }

    const int g = warp / C::CWARPS;
    const int ct = tid - g * C::GT;
    const int cw = ct >> 5;
    const int rl = lane >> 2, cc = lane & 3;
    const int col0 = 16 * cw + 4 * cc;           // this lane's four value columns
    const int lcol = 4 * cc + (rl & 3);           // the column (within the warp's 16) it ends with
    const bool yside = lane & 16;                 // ends with q-side sums (else u-side)
    const int rb = wy_base(rl);
    const uint32_t bar_id = 1 + g;
    float *buf = reinterpret_cast<float *>(smem + C::NST * C::STAGE + g * C::WORK_BYTES);
    float *dxw = buf + C::QK_F + 32 * cw;       // d' of this warp's columns, row stride DXS
    const TX *x = static_cast<const TX *>(a.x);
    TX *cache = static_cast<TX *>(a.cache);
    const float4 *w4 = reinterpret_cast<const float4 *>(a.conv_w);

    // P1 channels: q (X = 0) or k (X = 1) channel ch for every token of a
    // chunk, and v channel ch for half vh of the chunk's tokens
    const int X = ct >> 7, ch = ct & (DK - 1), vh = ct >> 7;
    // (T <= CT: one chunk, and the state is not live through P1 and P2)
    const int nchunks = MULTI ? (T + CT - 1) / CT : 1;
    const size_t xs = 3 * D;                      // token stride of x
    int par = 0;
    bool ok = true;

    // Staged inputs of unit (uu, cn) (head uu, chunk cn): two tensor copies
    // issued by one thread, x of tokens t0 - 3 .. t0 + CT - 1 into [slot =
    // token - t0 + 3][X][128] and alpha of tokens t0 .. t0 + CT - 1; tokens
    // outside 0 .. T - 1 arrive as zeros (before token 0 the window comes from
    // the conv cache instead). Completes on this group's input barrier.
    const TX *xsm = reinterpret_cast<const TX *>(buf + C::XS_F);
    uint32_t xk = 0;  // inputs consumed by this group
    auto stage_inputs = [&](int uu, int cn) {
        const int mm = uu / H, hh = uu - mm * H;
        ptx::mbar_arrive_expect_tx(&xin[g], (uint32_t)C::XS_BYTES + CT * DK * 4u +
                                                (cn == 0 ? (uint32_t)C::CS_BYTES : 0u));
        ptx::tma_load_4d(buf + C::XS_F, &mp.x, &xin[g], hh * DK, 0, cn * CT - 3, mm);
        ptx::tma_load_4d(buf + C::AL_F, &mp.alpha, &xin[g], 0, hh, cn * CT, mm);
        if (C::kCacheX && cn == 0) ptx::tma_load_4d(buf + C::CS_F, &mp.cache, &xin[g], hh * DK, 0, mm, 0);
        xfills[g] = xfills[g] + 1u;
    };
    if (C::kStageX && ct == 0 && blockIdx.x + g * gridDim.x < n_units)
        stage_inputs(blockIdx.x + g * gridDim.x, 0);

    for (int i = g, u = blockIdx.x + g * gridDim.x; u < n_units; i += G, u += G * gridDim.x) {
        const int s = i % C::NST, n = i / C::NST;
        const int m = u / H, h = u - m * H;
        const size_t hb = (size_t)h * DK;
        const TS *Ss = reinterpret_cast<const TS *>(smem + s * C::STAGE);
        const TX *cs = C::kCacheX ? reinterpret_cast<const TX *>(buf + C::CS_F)
                                  : reinterpret_cast<const TX *>(smem + s * C::STAGE + C::C_OFF);
        const TX *xqk = x + ((size_t)m * T * 3 + X) * D + hb + ch;
        const TX *xvv = x + ((size_t)m * T * 3 + 2) * D + hb + ch;
        // The lane's 64 state values as FP32 pairs. BF16 storage: sv[4 p + e] =
        // rows rl + 16 p and rl + 16 p + 8 of column col0 + e (a natural pair of
        // the row-permuted vectors, slots 2 p and 2 p + 1, so the column sums
        // and the update need no broadcasts; unpacking places the values
        // freely). FP32 storage: sv[2 r + k] = columns col0 + 2 k, + 1 of row
        // rl + 8 r (whole row quads move between memory and registers).
        float2 sv[32];

        for (int c = 0; c < nchunks; ++c, par ^= 1) {
            const int t0 = c * CT;
            const int nc = min(CT, T - t0);
            const bool last = c == nchunks - 1;
            const int h0 = (nc + 1) >> 1;
            const int vb = vh ? h0 : 0, vn = vh ? nc - h0 : h0;  // v tokens vb .. vb + vn - 1

            // ---- P1: inputs (x of tokens t0 - 3 .. t0 + nc - 1 for the windows) ----
            const float4 wq = __ldg(w4 + (size_t)X * D + hb + ch);
            const float4 wv = __ldg(w4 + 2 * D + hb + ch);
            TX xq[CT + 3], xv[CT / 2 + 3];
            float av[CT / 2];
            TX cq[3], cv[3];  // the conv cache after the call: inputs T - 3 .. T - 1
            bool landed = true;
            const float bt = ct < nc ? __ldg(a.beta + (size_t)(m * T + t0 + ct) * H + h) : 0.f;
            if constexpr (C::kStageX) {
                // this chunk's inputs landed (issued a chunk ahead)
                landed = ptx::mbar_wait(&xin[g], xk & 1, ptx::kWaitBudget);
                ++xk;
                if (!C::kCacheX && c == 0)  // the stage's refill was issued, then its bytes landed
                    landed = landed &&
                             (n == 0 || ptx::mbar_wait(&issued[s], (n - 1) & 1, ptx::kWaitBudget)) &&
                             ptx::mbar_wait(&full[s], n & 1, ptx::kWaitBudget);
                if (!landed) raise_error(8u);
#pragma unroll
                for (int j = 0; j < CT + 3; ++j)
                    xq[j] = j < nc + 3 ? xsm[(j * 3 + X) * DK + ch] : zero_tx<TX>();
#pragma unroll
                for (int j = 0; j < CT / 2 + 3; ++j)
                    xv[j] = j < vn + 3 ? xsm[((vb + j) * 3 + 2) * DK + ch] : zero_tx<TX>();
#pragma unroll
                for (int e = 0; e < 3; ++e) {
                    cq[e] = last ? xsm[((nc + e) * 3 + X) * DK + ch] : zero_tx<TX>();
                    cv[e] = last ? xsm[((nc + e) * 3 + 2) * DK + ch] : zero_tx<TX>();
                }
            } else {
#pragma unroll
                for (int j = 0; j < CT + 3; ++j) {
                    const int tau = t0 - 3 + j;
                    xq[j] = (j < nc + 3 && tau >= 0) ? xqk[(size_t)tau * xs] : zero_tx<TX>();
                }
#pragma unroll
                for (int j = 0; j < CT / 2 + 3; ++j) {
                    const int tau = t0 + vb - 3 + j;
                    xv[j] = (j < vn + 3 && tau >= 0) ? xvv[(size_t)tau * xs] : zero_tx<TX>();
                }
#pragma unroll
                for (int j = 0; j < CT / 2; ++j)
                    av[j] = j < vn ? __ldg(a.alpha + ((size_t)(m * T + t0 + vb + j) * H + h) * DK + ch) : 0.f;
#pragma unroll
                for (int e = 0; e < 3; ++e) {
                    const int tau = T - 3 + e;
                    cq[e] = (last && tau >= 0) ? xqk[(size_t)tau * xs] : zero_tx<TX>();
                    cv[e] = (last && vh && tau >= 0) ? xvv[(size_t)tau * xs] : zero_tx<TX>();
                }
                if (c == 0) {
                    // the stage's refill was issued, then its bytes landed
                    landed = (n == 0 || ptx::mbar_wait(&issued[s], (n - 1) & 1, ptx::kWaitBudget)) &&
                             ptx::mbar_wait(&full[s], n & 1, ptx::kWaitBudget);
                    if (!landed) raise_error(8u);
                }
            }
            if (c == 0) {  // the window slots before token 0 come from the stage's conv cache
#pragma unroll
                for (int j = 0; j < 3; ++j) xq[j] = cs[(3 * X + j) * DK + ch];
#pragma unroll
                for (int j = 0; j < 3; ++j)
                    if (vb - 3 + j < 0) xv[j] = cs[(6 + vb + j) * DK + ch];
#pragma unroll
                for (int e = 0; e < 3; ++e) {  // slots of the cache still in the window (T < 3)
                    const int tau = T - 3 + e;
                    if (last && tau < 0) {
                        cq[e] = cs[(3 * X + 3 + tau) * DK + ch];
                        cv[e] = cs[(9 + tau) * DK + ch];
                    }
                }
            }
            float *qk = buf + C::QK_F, *al = buf + C::AL_F;
            float *vbuf = buf + C::V_F + par * CT * DK, *bbuf = buf + C::BT_F + par * CT;
#pragma unroll
            for (int t = 0; t < CT; ++t)
                if (t < nc) qk[t * 2 * DK + ct] = conv4(wq, xq[t], xq[t + 1], xq[t + 2], xq[t + 3]);
#pragma unroll
            for (int j = 0; j < CT / 2; ++j)
                if (j < vn) {
                    vbuf[(vb + j) * DK + ch] = conv4(wv, xv[j], xv[j + 1], xv[j + 2], xv[j + 3]);
                    if (!C::kStageX) al[(vb + j) * DK + ch] = av[j];
                }
            if (ct < nc) bbuf[ct] = bt;

            // every thread's wait succeeded (else the group leaves together, before
            // anything of this chunk reaches global memory)
            if (c == 0 || C::kStageX) {
                if (!ptx::named_bar_and(bar_id, C::GT, landed)) {
                    ok = false;
                    break;
                }
            } else {
                ptx::named_bar_sync(bar_id, C::GT);
            }
            if (!C::kCacheX && last) {
                const size_t cbase = (size_t)m * 9 * D + hb;
#pragma unroll
                for (int e = 0; e < 3; ++e) {
                    cache[cbase + (size_t)(3 * X + e) * D + ch] = cq[e];
                    if (vh) cache[cbase + (size_t)(6 + e) * D + ch] = cv[e];
                }
            }

            // ---- P2: warp t = cw takes token t ----
            if (cw < nc) {
                const int t = cw;
                const float4 *qk4 = reinterpret_cast<const float4 *>(qk);
                const float4 *al4 = reinterpret_cast<const float4 *>(al);
                const float4 q4 = qk4[t * 64 + lane], k4 = qk4[t * 64 + 32 + lane];
                float red[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) red[j] = 0.f;
                const float qkd = dot4(q4, k4);
#pragma unroll
                for (int j = 0; j < CT; ++j)
                    if (j == t) red[j] = qkd;
                float4 R = make_float4(1.f, 1.f, 1.f, 1.f);
#pragma unroll
                for (int j = CT - 2; j >= 0; --j)
                    if (j < t) {
                        R = mul4(R, al4[(j + 1) * 32 + lane]);
                        const float4 kw = mul4(qk4[j * 64 + 32 + lane], R);
                        red[j] = dot4(q4, kw);      // P_tj
                        red[8 + j] = dot4(k4, kw);  // A_tj
                    }
                const float4 Gm = mul4(R, al4[lane]);  // Gamma_t
                float4 E = make_float4(1.f, 1.f, 1.f, 1.f);
#pragma unroll
                for (int j = 1; j < CT; ++j)
                    if (j > t && j < nc) E = mul4(E, al4[j * 32 + lane]);
                float *qd = buf + C::QD_F + t * VP, *kd = buf + C::KD_F + t * VP;
                float *ke = buf + C::KE_F + t * VP, *gl = buf + C::GL_F;
                const float qv[4] = {q4.x, q4.y, q4.z, q4.w}, kv[4] = {k4.x, k4.y, k4.z, k4.w};
                const float gv[4] = {Gm.x, Gm.y, Gm.z, Gm.w}, ev[4] = {E.x, E.y, E.z, E.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int p = wy_pos(4 * lane + e);
                    qd[p] = gv[e] * qv[e];
                    kd[p] = gv[e] * kv[e];
                    ke[p] = ev[e] * kv[e];
                    if (t == nc - 1) gl[p] = gv[e];
                }
                const float tot = warp_sum16(red, lane);
                const float qq = warp_sum(dot4(q4, q4)), kk = warp_sum(dot4(k4, k4));
                float *rr = buf + C::RED_F + t * 32;
                if ((lane & 1) == 0) rr[lane >> 1] = tot;
                if (lane == 1) {
                    rr[16] = rsqrtf(qq + kL2Eps);
                    rr[17] = rsqrtf(kk + kL2Eps);
                }
            }
            // with the cache staged with the inputs the state is waited for only
            // here, where it is read
            bool slanded = true;
            if (C::kCacheX && c == 0) {
                slanded = (n == 0 || ptx::mbar_wait(&issued[s], (n - 1) & 1, ptx::kWaitBudget)) &&
                          ptx::mbar_wait(&full[s], n & 1, ptx::kWaitBudget);
                if (!slanded) raise_error(8u);
            }
            if (c == 0) {
#pragma unroll
                for (int p = 0; p < 8; ++p) {
                    if constexpr (kRowPairs) {
                        float lo[4], hi[4];
                        Quad<TS>::load(Ss + (rl + 16 * p) * DK + col0, lo);
                        Quad<TS>::load(Ss + (rl + 16 * p + 8) * DK + col0, hi);
#pragma unroll
                        for (int e = 0; e < 4; ++e) sv[4 * p + e] = make_float2(lo[e], hi[e]);
                    } else {
#pragma unroll
                        for (int h2 = 0; h2 < 2; ++h2) {
                            float f4[4];
                            Quad<TS>::load(Ss + (rl + 16 * p + 8 * h2) * DK + col0, f4);
                            sv[2 * (2 * p + h2)] = make_float2(f4[0], f4[1]);
                            sv[2 * (2 * p + h2) + 1] = make_float2(f4[2], f4[3]);
                        }
                    }
                }
            }
            // the chunk's vectors and rows are ready (and every thread's wait for the
            // state succeeded)
            if (C::kCacheX && c == 0) {
                if (!ptx::named_bar_and(bar_id, C::GT, slanded)) {
                    ok = false;
                    break;
                }
            } else {
                ptx::named_bar_sync(bar_id, C::GT);
            }
            if (C::kCacheX && last) {  // after every wait of the chunk succeeded
                const size_t cbase = (size_t)m * 9 * D + hb;
#pragma unroll
                for (int e = 0; e < 3; ++e) {
                    cache[cbase + (size_t)(3 * X + e) * D + ch] = cq[e];
                    if (vh) cache[cbase + (size_t)(6 + e) * D + ch] = cv[e];
                }
            }
            if (C::kStageX && ct == 0) {  // the staged inputs are read: stage the next chunk's
                const bool more = c + 1 < nchunks;
                const int un = more ? u : u + G * gridDim.x;
                if (un < n_units) stage_inputs(un, more ? c + 1 : 0);
            }
            if (c == 0 && ct == 0) {             // the stage is read: refill it
                const int ur = blockIdx.x + (i + C::NST) * gridDim.x;
                if (ur < n_units) {
                    load_stage_wy<TS, TX, C>(smem + s * C::STAGE, &full[s], a, mp, ur, pol);
                    fills[s] = fills[s] + 1u;
                    ptx::mbar_arrive(&issued[s]);
                }
            }

            // ---- P3, first pass: column sums of Gamma k and Gamma q over this lane's rows ----
            // Per token, the lane's 2 x 4 sums reduce over the 8 lane groups rl in
            // three halving exchanges: u / q side (lane bit 4), then column pairs
            // (bit 3), then columns (bit 2). Lanes of the q side take the vectors in
            // the other order, so the first exchange needs no select.
            float xy[CT];
            {
                const float *own = buf + (yside ? C::QD_F : C::KD_F) + rb;
                const float *oth = buf + (yside ? C::KD_F : C::QD_F) + rb;
                const bool b3 = lane & 8, b2 = lane & 4;
#pragma unroll
                for (int t = 0; t < CT; ++t) {
                    xy[t] = 0.f;
                    if (t < nc) {
                        float so[4], sx[4];  // own / other kind, per column
                        if constexpr (kRowPairs) {
                            float2 ao[4], ax[4];
#pragma unroll
                            for (int e = 0; e < 4; ++e) ao[e] = ax[e] = make_float2(0.f, 0.f);
#pragma unroll
                            for (int r4 = 0; r4 < 4; ++r4) {
                                const float4 fo = *reinterpret_cast<const float4 *>(own + t * VP + 4 * r4);
                                const float4 fx = *reinterpret_cast<const float4 *>(oth + t * VP + 4 * r4);
                                const float2 o0 = make_float2(fo.x, fo.y), o1 = make_float2(fo.z, fo.w);
                                const float2 x0 = make_float2(fx.x, fx.y), x1 = make_float2(fx.z, fx.w);
#pragma unroll
                                for (int e = 0; e < 4; ++e) {
                                    ao[e] = __ffma2_rn(o0, sv[8 * r4 + e], ao[e]);
                                    ax[e] = __ffma2_rn(x0, sv[8 * r4 + e], ax[e]);
                                    ao[e] = __ffma2_rn(o1, sv[8 * r4 + 4 + e], ao[e]);
                                    ax[e] = __ffma2_rn(x1, sv[8 * r4 + 4 + e], ax[e]);
                                }
                            }
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                so[e] = ao[e].x + ao[e].y;
                                sx[e] = ax[e].x + ax[e].y;
                            }
                        } else {
                            float2 ao[2], ax[2];
#pragma unroll
                            for (int k = 0; k < 2; ++k) ao[k] = ax[k] = make_float2(0.f, 0.f);
#pragma unroll
                            for (int r4 = 0; r4 < 4; ++r4) {
                                const float4 fo = *reinterpret_cast<const float4 *>(own + t * VP + 4 * r4);
                                const float4 fx = *reinterpret_cast<const float4 *>(oth + t * VP + 4 * r4);
                                const float vo[4] = {fo.x, fo.y, fo.z, fo.w}, vx[4] = {fx.x, fx.y, fx.z, fx.w};
#pragma unroll
                                for (int e = 0; e < 4; ++e) {
                                    const float2 wo = make_float2(vo[e], vo[e]), wx = make_float2(vx[e], vx[e]);
#pragma unroll
                                    for (int k = 0; k < 2; ++k) {
                                        ao[k] = __ffma2_rn(wo, sv[2 * (4 * r4 + e) + k], ao[k]);
                                        ax[k] = __ffma2_rn(wx, sv[2 * (4 * r4 + e) + k], ax[k]);
                                    }
                                }
                            }
                            so[0] = ao[0].x; so[1] = ao[0].y; so[2] = ao[1].x; so[3] = ao[1].y;
                            sx[0] = ax[0].x; sx[1] = ax[0].y; sx[2] = ax[1].x; sx[3] = ax[1].y;
                        }
                        float l1[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) l1[e] = so[e] + __shfl_xor_sync(FULL, sx[e], 16);
                        float l2[2];
#pragma unroll
                        for (int e = 0; e < 2; ++e)
                            l2[e] = (b3 ? l1[2 + e] : l1[e]) + __shfl_xor_sync(FULL, b3 ? l1[e] : l1[2 + e], 8);
                        xy[t] = (b2 ? l2[1] : l2[0]) + __shfl_xor_sync(FULL, b2 ? l2[0] : l2[1], 4);
                    }
                }
            }
            const float *rrow = buf + C::RED_F;
            if (!yside) {  // forward substitution for d' of column lcol
                const float *vv = buf + C::V_F + par * CT * DK + 16 * cw + lcol;
                const float4 *bb4 = reinterpret_cast<const float4 *>(buf + C::BT_F + par * CT);
                const float4 ba = bb4[0], bz = bb4[1];
                const float bv[8] = {ba.x, ba.y, ba.z, ba.w, bz.x, bz.y, bz.z, bz.w};
                float dp[CT];
#pragma unroll
                for (int j = 0; j < CT; ++j) {
                    dp[j] = 0.f;
                    if (j < nc) {
                        const float4 *arow = reinterpret_cast<const float4 *>(rrow + j * 32 + 8);
                        const float4 a0 = arow[0], a1 = arow[1];
                        const float av8[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
                        const float2 nrm = *reinterpret_cast<const float2 *>(rrow + j * 32 + 16);
                        float acc = xy[j];
#pragma unroll
                        for (int i2 = 0; i2 < j; ++i2) acc += av8[i2] * dp[i2];
                        dp[j] = nrm.y * (bv[j] * (vv[j * DK] - nrm.y * acc));
                        dxw[j * C::DXS + lcol] = dp[j];
                    }
                }
            }
            __syncwarp();
            if (yside) {  // outputs of column lcol
                float dp[CT];
#pragma unroll
                for (int j = 0; j < CT; ++j) dp[j] = j < nc ? dxw[j * C::DXS + lcol] : 0.f;
                float *op = a.o + ((size_t)(m * T + t0) * H + h) * DK + 16 * cw + lcol;
#pragma unroll
                for (int t = 0; t < CT; ++t)
                    if (t < nc) {
                        const float4 *prow = reinterpret_cast<const float4 *>(rrow + t * 32);
                        const float4 p0 = prow[0], p1 = prow[1];
                        const float pv[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
                        float acc = xy[t];
#pragma unroll
                        for (int j = 0; j <= t; ++j) acc += pv[j] * dp[j];
                        op[(size_t)t * H * DK] = a.scale * rrow[t * 32 + 16] * acc;
                    }
            }

            // ---- P3, second pass: fade by Gamma_last, then the rank-nc update ----
            {
                const float *glv = buf + C::GL_F + rb, *kev = buf + C::KE_F + rb;
#pragma unroll
                for (int r4 = 0; r4 < 4; ++r4) {
                    const float4 g4 = *reinterpret_cast<const float4 *>(glv + 4 * r4);
                    if constexpr (kRowPairs) {
                        const float2 g0 = make_float2(g4.x, g4.y), g1 = make_float2(g4.z, g4.w);
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            sv[8 * r4 + e] = __fmul2_rn(sv[8 * r4 + e], g0);
                            sv[8 * r4 + 4 + e] = __fmul2_rn(sv[8 * r4 + 4 + e], g1);
                        }
                    } else {
                        const float gv[4] = {g4.x, g4.y, g4.z, g4.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float2 g2 = make_float2(gv[e], gv[e]);
                            sv[2 * (4 * r4 + e)] = __fmul2_rn(sv[2 * (4 * r4 + e)], g2);
                            sv[2 * (4 * r4 + e) + 1] = __fmul2_rn(sv[2 * (4 * r4 + e) + 1], g2);
                        }
                    }
                }
#pragma unroll 1
                for (int j = 0; j < nc; ++j) {
                    const float4 d4 = *reinterpret_cast<const float4 *>(dxw + j * C::DXS + 4 * cc);
                    if constexpr (kRowPairs) {
                        const float2 dd[4] = {make_float2(d4.x, d4.x), make_float2(d4.y, d4.y),
                                              make_float2(d4.z, d4.z), make_float2(d4.w, d4.w)};
#pragma unroll
                        for (int r4 = 0; r4 < 4; ++r4) {
                            const float4 e4 = *reinterpret_cast<const float4 *>(kev + j * VP + 4 * r4);
                            const float2 e0 = make_float2(e4.x, e4.y), e1 = make_float2(e4.z, e4.w);
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                sv[8 * r4 + e] = __ffma2_rn(e0, dd[e], sv[8 * r4 + e]);
                                sv[8 * r4 + 4 + e] = __ffma2_rn(e1, dd[e], sv[8 * r4 + 4 + e]);
                            }
                        }
                    } else {
                        const float2 dd[2] = {make_float2(d4.x, d4.y), make_float2(d4.z, d4.w)};
#pragma unroll
                        for (int r4 = 0; r4 < 4; ++r4) {
                            const float4 e4 = *reinterpret_cast<const float4 *>(kev + j * VP + 4 * r4);
                            const float ev[4] = {e4.x, e4.y, e4.z, e4.w};
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const float2 e2 = make_float2(ev[e], ev[e]);
                                sv[2 * (4 * r4 + e)] = __ffma2_rn(e2, dd[0], sv[2 * (4 * r4 + e)]);
                                sv[2 * (4 * r4 + e) + 1] = __ffma2_rn(e2, dd[1], sv[2 * (4 * r4 + e) + 1]);
                            }
                        }
                    }
                }
            }
        }
        if (!ok) break;

        // state out (rounded once, here, for BF16 storage)
        TS *Sg = static_cast<TS *>(a.state) + (size_t)u * DK * DK + col0;
#pragma unroll
        for (int p = 0; p < 8; ++p) {
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
                float f4[4];
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    f4[e] = kRowPairs ? (h2 ? sv[4 * p + e].y : sv[4 * p + e].x)
                                      : (e & 1 ? sv[2 * (2 * p + h2) + (e >> 1)].y
                                               : sv[2 * (2 * p + h2) + (e >> 1)].x);
                Quad<TS>::store(Sg + (size_t)(rl + 16 * p + 8 * h2) * DK, f4);
            }
        }
    }

    // Exit: as in the token-by-token kernel, and the latest staged inputs of
    // each group (in flight only if the group left early)
    __syncthreads();
    if (threadIdx.x == 0) {
        drain_fills<C>(smem);
        for (int gg = 0; gg < G; ++gg) {
            const uint32_t f = xfills[gg];
            if (f > 0) ptx::mbar_wait(&xin[gg], (f - 1) & 1, ptx::kDrainBudget);
        }
    }
}

template <typename KERNEL, typename... EXTRA>
cudaError_t launch_persistent(KERNEL kernel, int threads, int smem, const DecodeArgs &a, int T,
                              cudaStream_t stream, const EXTRA &...extra) {
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    const int units = a.M * a.H;
    const int grid = units < sms ? units : sms;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(threads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, a, T, extra...);
}

template <typename TS, typename TX>
cudaError_t launch_tokens_typed(const DecodeArgs &a, int T, cudaStream_t stream) {
    if (T >= KDA_TOKENS_WY_MIN) {
        using C = WyCfg<TS, TX>;
        TokMaps mp;
        memset(&mp, 0, sizeof(mp));
        if (C::kStageX) {
            const uint64_t D = (uint64_t)a.H * DK;
            const uint64_t dx[4] = {D, 3, (uint64_t)T, (uint64_t)a.M};
            const uint32_t bx[4] = {DK, 3, C::CT + 3, 1};
            const uint64_t da[4] = {DK, (uint64_t)a.H, (uint64_t)T, (uint64_t)a.M};
            const uint32_t ba[4] = {DK, 1, C::CT, 1};
            cudaError_t e = make_tensor_map(&mp.x, a.x, sizeof(TX) == 2, 4, dx, bx, false);
            if (e == cudaSuccess) e = make_tensor_map(&mp.alpha, a.alpha, false, 4, da, ba, false);
            const uint64_t dc[4] = {D, 9, (uint64_t)a.M, 1};
            const uint32_t bc[4] = {DK, 9, 1, 1};
            if (e == cudaSuccess) e = make_tensor_map(&mp.cache, a.cache, true, 4, dc, bc, false);
            if (e != cudaSuccess) return e;
        }
        if (T > C::CT)
            return launch_persistent(kda_decode_tokens_wy_kernel<TS, TX, true>, C::THREADS, C::SMEM, a, T,
                                     stream, mp);
        return launch_persistent(kda_decode_tokens_wy_kernel<TS, TX, false>, C::THREADS, C::SMEM, a, T,
                                 stream, mp);
    }
    using C = TokCfg<TS, TX, 2>;
    // the cache by one tensor copy per head: faster with BF16 state (M = 32,
    // T = 2: 44.0 -> 43.1 us) and with FP32 state from 1024 heads on (49.6 ->
    // 49.0), slower with FP32 state at M = 8 (15.2 -> 15.5)
    TokCacheMap cm;
    memset(&cm, 0, sizeof(cm));
    if (sizeof(TS) == 2 || a.M * a.H >= 1024) {
        const uint64_t dc[4] = {(uint64_t)a.H * DK, 9, (uint64_t)a.M, 1};
        const uint32_t bc[4] = {DK, 9, 1, 1};
        const cudaError_t e = make_tensor_map(&cm.map, a.cache, sizeof(TX) == 2, 4, dc, bc, false);
        if (e != cudaSuccess) return e;
        cm.on = 1;
    }
    return launch_persistent(kda_decode_tokens_kernel<TS, TX, 2>, C::THREADS, C::SMEM, a, T, stream, cm);
}

}  // namespace

cudaError_t launch_decode_tokens(const DecodeArgs &a, int T, int x_dtype, int state_dtype,
                                 cudaStream_t stream) {
    const bool xb = x_dtype == KDA_BF16, sb = state_dtype == KDA_BF16;
    if (sb && xb) return launch_tokens_typed<__nv_bfloat16, __nv_bfloat16>(a, T, stream);
    if (sb) return launch_tokens_typed<__nv_bfloat16, float>(a, T, stream);
    if (xb) return launch_tokens_typed<float, __nv_bfloat16>(a, T, stream);
    return launch_tokens_typed<float, float>(a, T, stream);
}

cudaError_t read_tokens_error(unsigned int *code) {
    return cudaMemcpyFromSymbol(code, g_tokens_error, sizeof(unsigned int));
}

cudaError_t clear_tokens_error() {
    const unsigned int zero = 0;
    return cudaMemcpyToSymbol(g_tokens_error, &zero, sizeof(unsigned int));
}

}  // namespace kda
