// Multi-token KDA decode for sm_103a: T consecutive decode steps of one layer
// in one launch (conv + SiLU, L2 norm of q and k, the gated delta rule of
// "GLM-5.3 deep dive" section 8.2.3 Eq. 1 in the fade / predict / correct /
// read order of section 8.2.6, readout o = w + d (k.q)), token after token,
// as fla's fused-recurrent mode does for short inputs (section 8.2.5).
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

#include "../../include/kda.h"
#include "kda_internal.cuh"
#include "kda_ptx.cuh"

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

// Bulk copies of head u's state and conv cache into stage `st`.
template <typename TS, typename TX, int G>
__device__ __forceinline__ void load_head_tokens(unsigned char *st, uint64_t *bar,
                                                 const DecodeArgs &a, int u, uint64_t pol) {
    using C = TokCfg<TS, TX, G>;
    const int H = a.H;
    const size_t D = (size_t)H * DK;
    const int m = u / H, h = u - m * H;
    const TX *cache = static_cast<const TX *>(a.cache);
    ptx::mbar_arrive_expect_tx(bar, C::STAGE);
    ptx::bulk_g2s_hint(st, static_cast<const TS *>(a.state) + (size_t)u * DK * DK, C::S_BYTES, bar,
                       pol);
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
kda_decode_tokens_kernel(const DecodeArgs a, const int T) {
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
            if (u < n_units) load_head_tokens<TS, TX, G>(smem + s * C::STAGE, &full[s], a, u, pol);
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
                load_head_tokens<TS, TX, G>(smem + s * C::STAGE, &full[s], a, ur, pol);
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

template <typename TS, typename TX>
cudaError_t launch_tokens_typed(const DecodeArgs &a, int T, cudaStream_t stream) {
    constexpr int G = 2;
    using C = TokCfg<TS, TX, G>;
    auto kernel = kda_decode_tokens_kernel<TS, TX, G>;
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    const int units = a.M * a.H;
    const int grid = units < sms ? units : sms;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(C::THREADS, 1, 1);
    cfg.dynamicSmemBytes = C::SMEM;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, a, T);
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
