// Persistent, bulk-copy-fed KDA decode step for sm_103a.
//
// Same arithmetic as kda_decode.cu (conv + SiLU, L2 norm of q and k, the
// gated delta rule of "GLM-5.3 deep dive" section 8.2.3 Eq. 1 in the fade /
// predict / correct / read order of section 8.2.6, readout via
// o = w + d (k.q)), organised for HBM streaming at large M:
//
//  * One CTA per SM loops over whole heads (stream m, head h); a head's state
//    is one contiguous block (64 KiB FP32, 32 KiB BF16).
//  * Each head's state, alpha, pre-conv x and conv-cache taps are copied into
//    a ring of NST shared-memory stages (state and alpha by cp.async.bulk, x
//    and the cache by one tensor copy each, or with FP32 state beyond 1024
//    heads by a bulk copy per row); the copies complete on the stage's
//    "full" mbarrier (transaction bytes).
//  * The CTA's 16 warps form G consumer groups (G = 1 or 2) that take heads
//    in turn (group g: heads g, g + G, ...). A group pulls its stage into
//    registers and convolves the head's 3 x 128 channels from the same stage;
//    after one group barrier the stage has been read, and the group's first
//    thread refills it with the head NST places further on and arrives on the
//    stage's "issued" mbarrier. With two groups, one group's barriers and
//    reductions overlap the other's loads and arithmetic.
//  * Ring protocol. The consumer of head j (stage s = j % NST, use n = j / NST)
//    waits for the n-th refill of s to have been issued, then for its bytes.
//    That refill was issued by the consumer of head j - NST, after reading
//    it; the refill before it was issued by this very group when it consumed
//    head j - 2 NST. So each wait is for the phase right after one already
//    observed, and mbarrier phase parities cannot alias.
//  * There is no separate producer warp (16 warps keep 128 registers per
//    thread available) and no "stage empty" barrier: the thread that refills
//    a stage is the one that knows it is free.
//  * The column sums u = k.s and w = q.s are reduced in registers, across the
//    lanes sharing a strip (BF16), then across the group's warps: each warp
//    writes its partial sums as contiguous [warp][column] rows (16-byte
//    stores, no bank conflicts); 128 threads add the partials of u and
//    publish d while 128 others add those of w and, after one more barrier,
//    write o. Every thread reads the d of its strip with one 16-byte load and
//    writes S' with 128-bit streaming stores straight from registers.
//  * Optionally the state of the head P places beyond the one being loaded is
//    prefetched into L2 (cp.async.bulk.prefetch.L2).
//  * Conv weights and beta of a group's next head are prefetched into
//    registers one head ahead.
//  * Optional fusions (template flags): the KDA forget gate in front
//    ("GLM-5.3 deep dive" 8.2.3: alpha = exp(lb sigmoid(e^{A_h} (f + b)))),
//    computed by 128 threads of a group one head ahead (while the group
//    reduces the current head) into a double-buffered shared array, so the
//    fade stays on the load path; and the gated RMSNorm behind (8.2.4 step 7:
//    y = o / sqrt(mean o^2 + eps) w sigmoid(gate)), applied by the 128 threads
//    that form o, with one 128-thread barrier for the sum of squares.
//  * Launched with programmatic stream serialisation: the kernel waits for
//    the preceding grid (griddepcontrol.wait) before its first global read,
//    and lets the next launch in the stream start placing CTAs early, which
//    hides launch latency between back-to-back layers. Before the wait it
//    only prefetches its first heads' state into L2 (a hint; L2 also holds
//    whatever the previous grid writes).
//
// Each conv-cache channel belongs to exactly one head, so the cache is read
// (by the bulk copy) and rewritten (by the consumer) by one CTA only.
//
// Every mbarrier wait is bounded (about two seconds of clock cycles). A
// thread whose wait gives up sets the device error word and skips its writes
// to global memory; the group's next barrier ANDs every thread's outcome, so
// the whole group leaves the loop together. At exit the CTA meets once more
// and one thread waits (bounded) for the latest bulk copy into every stage,
// so nothing lands in shared memory after the CTA is gone.
// kda_device_error() reports the error word on the host.

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>

#include "../../include/kda.h"
#include "kda_internal.cuh"
#include "kda_ptx.cuh"

namespace kda {

__device__ unsigned int g_stream_error;

namespace {

constexpr int DK = kHeadDim;
constexpr float kL2Eps = 1e-6f;
constexpr int kSmemLimit = 232448;               // 227 KiB opt-in per CTA
constexpr int kWarps = 16;

template <typename TS, typename TX, int G>
struct Cfg {
    static constexpr int VEC = 16 / (int)sizeof(TS);   // columns per 16-byte strip
    static constexpr int STRIPS = DK / VEC;            // strips per row (32 or 16)
    static constexpr int SUBS = 32 / STRIPS;           // rows per warp instruction
    static constexpr int CWARPS = kWarps / G;          // warps per consumer group
    static constexpr int GT = CWARPS * 32;             // threads per group
    static constexpr int THREADS = kWarps * 32;
    static constexpr int RGROUPS = CWARPS * SUBS;
    static constexpr int RPT = DK / RGROUPS;           // rows per thread
    static_assert(GT >= 2 * DK, "a group needs 256 threads for the column sums");
    // stage: state | alpha | x (q,k,v) | cache (q,k,v) x (3 taps)
    static constexpr int S_BYTES = DK * DK * (int)sizeof(TS);
    static constexpr int A_OFF = S_BYTES;
    static constexpr int X_OFF = A_OFF + DK * 4;
    static constexpr int C_OFF = X_OFF + 3 * DK * (int)sizeof(TX);
    static constexpr int STAGE = C_OFF + 9 * DK * (int)sizeof(TX);
    // per group: red_u, red_w [CWARPS][DK] | d [DK] | qk [2][DK] | v [DK] |
    //            alpha from the fused gate [DK] | norm partials [4] (+ pad)
    static constexpr int REDW_F = CWARPS * DK;
    static constexpr int DB_F = 2 * CWARPS * DK;
    static constexpr int QK_F = DB_F + DK;
    static constexpr int V_F = QK_F + 2 * DK;
    static constexpr int AB_F = V_F + DK;      // [2][DK]: alpha of this head and the next
    static constexpr int NRM_F = AB_F + 2 * DK;  // [4] norm partials | q.q | q.k | pad
    static constexpr int WORK_F = NRM_F + 8;
    static constexpr int WORK_BYTES = WORK_F * 4;
    static constexpr int BAR_BYTES = 2 * 8 * 8 + 8 * 4;  // full[8], issued[8], fills[8]
    static constexpr int NST_FIT = (kSmemLimit - BAR_BYTES - G * WORK_BYTES) / STAGE;
    static constexpr int NST = NST_FIT > 6 ? 6 : NST_FIT;
    static constexpr int SMEM = NST * STAGE + G * WORK_BYTES + BAR_BYTES;
    static_assert(NST >= 2, "at least two stages must fit");
    static_assert(STAGE % 16 == 0 && WORK_BYTES % 16 == 0, "16-byte alignment");
};

template <typename TS> struct Strip;
template <> struct Strip<float> {
    __device__ __forceinline__ static void unpack(const uint4 &r, float (&f)[4]) {
        f[0] = __uint_as_float(r.x); f[1] = __uint_as_float(r.y);
        f[2] = __uint_as_float(r.z); f[3] = __uint_as_float(r.w);
    }
    __device__ __forceinline__ static uint4 pack(const float (&f)[4]) {
        return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]),
                          __float_as_uint(f[2]), __float_as_uint(f[3]));
    }
};
__device__ __forceinline__ uint32_t bf16x2_rn(float lo, float hi) {
    __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&p);
}
template <> struct Strip<__nv_bfloat16> {
    __device__ __forceinline__ static void unpack(const uint4 &r, float (&f)[8]) {
        const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            f[2 * e] = __uint_as_float(w[e] << 16);
            f[2 * e + 1] = __uint_as_float(w[e] & 0xffff0000u);
        }
    }
    __device__ __forceinline__ static uint4 pack(const float (&f)[8]) {
        return make_uint4(bf16x2_rn(f[0], f[1]), bf16x2_rn(f[2], f[3]),
                          bf16x2_rn(f[4], f[5]), bf16x2_rn(f[6], f[7]));
    }
};

__device__ __forceinline__ float widen(float v) { return v; }
__device__ __forceinline__ float widen(__nv_bfloat16 v) { return __bfloat162float(v); }

__device__ __forceinline__ void raise_error(unsigned int code) { atomicOr(&g_stream_error, code); }

// conv (kernel 4) + SiLU of one channel from the staged taps; writes the
// shifted taps (c1, c2, x) back to the global cache.
template <typename TX>
__device__ __forceinline__ float conv_stage(const float4 w, const TX *cs, const TX *xs, int X,
                                            int ch, TX *cg, size_t D) {
    const TX c0 = cs[(X * 3 + 0) * DK + ch], c1 = cs[(X * 3 + 1) * DK + ch];
    const TX c2 = cs[(X * 3 + 2) * DK + ch], xt = xs[X * DK + ch];
    cg[0] = c1;
    cg[D] = c2;
    cg[2 * D] = xt;
    const float pre = w.x * widen(c0) + w.y * widen(c1) + w.z * widen(c2) + w.w * widen(xt);
    return pre / (1.0f + expf(-pre));
}

// Prefetches the state of head u into L2.
template <typename TS>
__device__ __forceinline__ void prefetch_head(const DecodeArgs &a, int u) {
    ptx::bulk_prefetch_l2(static_cast<const TS *>(a.state) + (size_t)u * DK * DK,
                          DK * DK * sizeof(TS));
}

// Tensor maps of one call's pre-conv inputs and conv cache (encoded on the
// host per call when `on`): x as [M][3][H*128] and the cache as [M][9][H*128],
// in boxes of 128 channels x 3 or 9 rows, so a head's q, k, v inputs and its
// nine cached taps arrive in one tensor copy each instead of twelve bulk
// copies issued one after another.
struct DecMaps {
    CUtensorMap x;
    CUtensorMap cache;
    int on;
};

// Issues the copies of head u into stage `st`, completing on `bar`: the state
// and alpha (not with the fused gate, which computes it) by bulk copies, x and
// the conv cache by tensor copies or, without maps, by a bulk copy per row.
template <typename TS, typename TX, int G, bool GATE>
__device__ __forceinline__ void load_head(unsigned char *st, uint64_t *bar, const DecodeArgs &a,
                                          const DecMaps &mp, int u, uint64_t pol) {
    using C = Cfg<TS, TX, G>;
    const int H = a.H;
    const size_t D = (size_t)H * DK;
    const int m = u / H, h = u - m * H;
    ptx::mbar_arrive_expect_tx(bar, GATE ? C::STAGE - DK * 4 : C::STAGE);
    ptx::bulk_g2s_hint(st, static_cast<const TS *>(a.state) + (size_t)u * DK * DK, C::S_BYTES, bar,
                       pol);
    if (!GATE) ptx::bulk_g2s(st + C::A_OFF, a.alpha + (size_t)u * DK, DK * 4, bar);
    if (mp.on) {
        ptx::tma_load_4d(st + C::X_OFF, &mp.x, bar, h * DK, 0, m, 0);
        ptx::tma_load_4d(st + C::C_OFF, &mp.cache, bar, h * DK, 0, m, 0);
        return;
    }
    const TX *x = static_cast<const TX *>(a.x);
    const TX *cache = static_cast<const TX *>(a.cache);
#pragma unroll
    for (int X = 0; X < 3; ++X)
        ptx::bulk_g2s(st + C::X_OFF + X * DK * sizeof(TX), x + ((size_t)m * 3 + X) * D + (size_t)h * DK,
                      DK * sizeof(TX), bar);
#pragma unroll
    for (int j = 0; j < 9; ++j)
        ptx::bulk_g2s(st + C::C_OFF + j * DK * sizeof(TX), cache + ((size_t)m * 9 + j) * D + (size_t)h * DK,
                      DK * sizeof(TX), bar);
}

// Up to this many heads, FP32-state calls take x and the cache by tensor
// copies (measured on the 34-layer stack: 5 % faster at M = 1, 2 % at M = 8,
// 1.6 % slower at M = 32, where the layer is bound by HBM); BF16-state calls
// always do (1-4 % faster at every M).
constexpr int kTensorInputsMaxHeadsF32 = 1024;

// The tensor maps of a decode call, encoded only if the call uses them.
template <typename TX>
cudaError_t make_decode_maps(DecMaps *mp, const DecodeArgs &a, bool on) {
    memset(mp, 0, sizeof(*mp));
    if (!on) return cudaSuccess;
    const uint64_t D = (uint64_t)a.H * DK;
    const uint64_t dx[4] = {D, 3, (uint64_t)a.M, 1}, dc[4] = {D, 9, (uint64_t)a.M, 1};
    const uint32_t bx[4] = {DK, 3, 1, 1}, bc[4] = {DK, 9, 1, 1};
    cudaError_t e = make_tensor_map(&mp->x, a.x, sizeof(TX) == 2, 4, dx, bx, false);
    if (e == cudaSuccess) e = make_tensor_map(&mp->cache, a.cache, sizeof(TX) == 2, 4, dc, bc, false);
    mp->on = 1;
    return e;
}

template <typename TS, typename TX, int G, bool GATE, bool NORM>
__global__ void __launch_bounds__(Cfg<TS, TX, G>::THREADS, 1)
kda_decode_stream_kernel(const DecodeArgs a, const __grid_constant__ DecMaps mp) {
    using C = Cfg<TS, TX, G>;
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
    const int P = a.l2_prefetch;

    if (tid == 0) {
        for (int s = 0; s < C::NST; ++s) {
            ptx::mbar_init(&full[s], 1);
            ptx::mbar_init(&issued[s], 1);
            fills[s] = blockIdx.x + s * gridDim.x < n_units ? 1u : 0u;  // the first fills, below
        }
        ptx::fence_mbar_init();
    }
    // While the previous grid drains, warm L2 with the state of this CTA's
    // first heads. A prefetch only fills L2, where the previous grid's writes
    // land as well, so it cannot expose stale data; the copies below (after
    // the dependency wait) then hit L2 instead of paying DRAM latency.
    if (tid == 0) {
        for (int s = 0; s < C::NST; ++s) {
            const int u = blockIdx.x + s * gridDim.x;
            if (u < n_units) prefetch_head<TS>(a, u);
        }
    }
    __syncthreads();
    ptx::grid_dependency_wait();  // the previous grid's writes are visible from here on
    ptx::launch_dependents();
    if (tid == 0) {
        for (int s = 0; s < C::NST; ++s) {
            const int u = blockIdx.x + s * gridDim.x;
            if (u < n_units) load_head<TS, TX, G, GATE>(smem + s * C::STAGE, &full[s], a, mp, u, pol);
        }
        for (int j = 0; j < P; ++j) {
            const int u = blockIdx.x + (C::NST + j) * gridDim.x;
            if (u < n_units) prefetch_head<TS>(a, u);
        }
    }

    const int g = warp / C::CWARPS;            // consumer group
    const int ct = tid - g * C::GT;            // thread index within the group
    const int cwarp = ct >> 5;
    const int strip = lane % C::STRIPS, sub = lane / C::STRIPS;
    const int rg = cwarp * C::SUBS + sub;
    const uint32_t bar_id = 1 + g;
    float *red = reinterpret_cast<float *>(smem + C::NST * C::STAGE + g * C::WORK_BYTES);
    float *redw = red + C::REDW_F;
    float *db = red + C::DB_F;
    float *qkb = red + C::QK_F;
    float *vb = red + C::V_F;
    float *ab = red + C::AB_F;
    float *nrm = red + C::NRM_F;
    TX *cache = static_cast<TX *>(a.cache);
    const float4 *w4 = reinterpret_cast<const float4 *>(a.conv_w);

    // conv channels of this thread: c0 = ct and, with 256-thread groups,
    // c1 = ct + 256 (c < 384 encodes tensor c / 128, channel c % 128)
    const int c0 = ct, c1 = ct + C::GT;
    float4 wA = make_float4(0.f, 0.f, 0.f, 0.f), wB = wA;
    float beta_n = 0.f;
    // fused gate: threads GT-128 .. GT-1 own key channel gi; fused norm:
    // threads 128 .. 255 (the o writers) own value channel ct - 128
    const int gi = ct - (C::GT - DK);
    float bias_n = 0.f, eA_n = 0.f, f_n = 0.f, og_n = 0.f;
    const float nw = (NORM && ct >= DK && ct < 2 * DK) ? __ldg(a.norm_w + ct - DK) : 0.f;
    auto prefetch = [&](int un) {
        const size_t hb = (size_t)(un % H) * DK;
        if (c0 < 3 * DK) wA = __ldg(w4 + (size_t)(c0 / DK) * D + hb + c0 % DK);
        if (c1 < 3 * DK) wB = __ldg(w4 + (size_t)(c1 / DK) * D + hb + c1 % DK);
        beta_n = __ldg(a.beta + un);
        if (GATE && gi >= 0) {
            bias_n = __ldg(a.dt_bias + hb + gi);
            eA_n = __ldg(a.A_log + un % H);
            f_n = __ldg(a.alpha + (size_t)un * DK + gi);
        }
        if (NORM && ct >= DK && ct < 2 * DK) og_n = __ldg(a.out_gate + (size_t)un * DK + ct - DK);
    };

    // alpha = exp(lb sigmoid(e^A (f + b))) of the prefetched head, into ab[buf]
    auto gate = [&](int buf) {
        const float z = __expf(eA_n) * (f_n + bias_n);
        ab[buf * DK + gi] = __expf(a.gate_lb / (1.0f + __expf(-z)));
    };

    int i = g;
    int u = blockIdx.x + i * gridDim.x;
    if (u < n_units) prefetch(u);
    if (GATE) {  // the group's first head; later heads are gated one iteration ahead
        if (u < n_units && gi >= 0) gate(0);
        __syncthreads();
    }
    for (; u < n_units; i += G, u += G * gridDim.x) {
        const int s = i % C::NST, n = i / C::NST;
        const int m = u / H, h = u - m * H;
        const float4 w0 = wA, w1 = wB;
        const float beta = beta_n;
        const float og = og_n;
        const int ib = (i / G) & 1;  // this head's alpha buffer (fused gate)
        const int un = u + G * gridDim.x;
        if (un < n_units) prefetch(un);

        // the stage's refill was issued, then its bytes landed; a thread whose
        // wait gives up reads no further data of this head and writes nothing
        // (the group leaves together at barrier 1)
        const bool landed = (n == 0 || ptx::mbar_wait(&issued[s], (n - 1) & 1, ptx::kWaitBudget)) &&
                            ptx::mbar_wait(&full[s], n & 1, ptx::kWaitBudget);
        if (!landed) raise_error(4u);
        const unsigned char *st = smem + s * C::STAGE;
        const TS *Ss = reinterpret_cast<const TS *>(st);
        const float *al = reinterpret_cast<const float *>(st + C::A_OFF);
        const TX *xs = reinterpret_cast<const TX *>(st + C::X_OFF);
        const TX *cs = reinterpret_cast<const TX *>(st + C::C_OFF);

        // (a) state strips into registers, faded by alpha of their row
        float sv[C::RPT][C::VEC];
#pragma unroll
        for (int p = 0; p < C::RPT; ++p) {
            const int row = p * C::RGROUPS + rg;
            const uint4 r = *reinterpret_cast<const uint4 *>(Ss + row * DK + strip * C::VEC);
            Strip<TS>::unpack(r, sv[p]);
            const float ar = GATE ? ab[ib * DK + row] : al[row];
            const float2 a2 = make_float2(ar, ar);
#pragma unroll
            for (int c = 0; c < C::VEC; c += 2) {  // packed FP32 pairs (mul.rn.f32x2)
                const float2 f = __fmul2_rn(make_float2(sv[p][c], sv[p][c + 1]), a2);
                sv[p][c] = f.x;
                sv[p][c + 1] = f.y;
            }
        }

        // (b) conv + SiLU of the head's 384 channels (q, k, v)
        const size_t cbase = (size_t)m * 9 * D + (size_t)h * DK;
        if (landed && c0 < 3 * DK) {
            const int X = c0 / DK, ch = c0 % DK;
            const float y = conv_stage(w0, cs, xs, X, ch, cache + cbase + 3 * X * D + ch, D);
            if (X < 2) qkb[X * DK + ch] = y;
            else vb[ch] = y;
        }
        if (landed && c1 < 3 * DK) {
            const int X = c1 / DK, ch = c1 % DK;
            const float y = conv_stage(w1, cs, xs, X, ch, cache + cbase + 3 * X * D + ch, D);
            if (X < 2) qkb[X * DK + ch] = y;
            else vb[ch] = y;
        }
        // barrier 1: stage read; q, k, v visible; every thread's wait succeeded
        if (!ptx::named_bar_and(bar_id, C::GT, landed)) break;
        if (ct == 0) {
            const int ur = blockIdx.x + (i + C::NST) * gridDim.x;  // refill with head i + NST
            if (ur < n_units) {
                load_head<TS, TX, G, GATE>(smem + s * C::STAGE, &full[s], a, mp, ur, pol);
                fills[s] = fills[s] + 1u;
                ptx::mbar_arrive(&issued[s]);
                const int up = ur + P * gridDim.x;
                if (P > 0 && up < n_units) prefetch_head<TS>(a, up);
            }
        }

        // fused gate: alpha of the group's next head (its inputs were
        // prefetched at the top of this iteration), visible after barrier 2
        if (GATE && gi >= 0 && un < n_units) gate(ib ^ 1);

        // (c) L2 norms. Plain step: they enter only through d and o below, since
        // u = k_hat.s = rk (k.s), w = rq (q.s) and S' = s + k_hat d = s + k (rk d);
        // the warps forming d (threads 0-127) take k.k, q.q and q.k and publish
        // the last two for the warps forming o. With the fused gate and norm
        // (more live registers in the o warps) every warp forms rq, rk and
        // k_hat.q_hat itself and the sums below use the normalised q and k.
        constexpr bool FOLD = !GATE && !NORM;
        float nA = 0.f;  // k.k in the d warps
        float rqw = 1.f, rkw = 1.f, kqw = 0.f;
        if (!FOLD) {
            const float4 q4 = reinterpret_cast<const float4 *>(qkb)[lane];
            const float4 k4 = reinterpret_cast<const float4 *>(qkb + DK)[lane];
            float sq = q4.x * q4.x + q4.y * q4.y + q4.z * q4.z + q4.w * q4.w;
            float sk = k4.x * k4.x + k4.y * k4.y + k4.z * k4.z + k4.w * k4.w;
            float sqk = q4.x * k4.x + q4.y * k4.y + q4.z * k4.z + q4.w * k4.w;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                sq += __shfl_xor_sync(0xffffffffu, sq, off);
                sk += __shfl_xor_sync(0xffffffffu, sk, off);
                sqk += __shfl_xor_sync(0xffffffffu, sqk, off);
            }
            rqw = 1.0f / sqrtf(sq + kL2Eps);
            rkw = 1.0f / sqrtf(sk + kL2Eps);
            kqw = sqk * rqw * rkw;
        } else if (ct < DK) {
            const float4 q4 = reinterpret_cast<const float4 *>(qkb)[lane];
            const float4 k4 = reinterpret_cast<const float4 *>(qkb + DK)[lane];
            nA = k4.x * k4.x + k4.y * k4.y + k4.z * k4.z + k4.w * k4.w;
            float nQ = q4.x * q4.x + q4.y * q4.y + q4.z * q4.z + q4.w * q4.w;
            float nB = q4.x * k4.x + q4.y * k4.y + q4.z * k4.z + q4.w * k4.w;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                nA += __shfl_xor_sync(0xffffffffu, nA, off);
                nQ += __shfl_xor_sync(0xffffffffu, nQ, off);
                nB += __shfl_xor_sync(0xffffffffu, nB, off);
            }
            if (ct == 0) {  // read by the o warps after barrier 3
                nrm[4] = nQ;
                nrm[5] = nB;
            }
        }

        // (d) column sums k.s and q.s over this thread's rows (raw q, k when folded)
        float uu[C::VEC], ww[C::VEC], kr[C::RPT];
#pragma unroll
        for (int c = 0; c < C::VEC; ++c) uu[c] = ww[c] = 0.f;
#pragma unroll
        for (int p = 0; p < C::RPT; ++p) {
            const int row = p * C::RGROUPS + rg;
            kr[p] = FOLD ? qkb[DK + row] : qkb[DK + row] * rkw;
            const float qr = FOLD ? qkb[row] : qkb[row] * rqw;
            const float2 k2 = make_float2(kr[p], kr[p]), q2 = make_float2(qr, qr);
#pragma unroll
            for (int c = 0; c < C::VEC; c += 2) {  // packed FP32 pairs (fma.rn.f32x2)
                const float2 s2 = make_float2(sv[p][c], sv[p][c + 1]);
                const float2 u2 = __ffma2_rn(k2, s2, make_float2(uu[c], uu[c + 1]));
                const float2 w2 = __ffma2_rn(q2, s2, make_float2(ww[c], ww[c + 1]));
                uu[c] = u2.x;
                uu[c + 1] = u2.y;
                ww[c] = w2.x;
                ww[c + 1] = w2.y;
            }
        }
        if (C::SUBS == 2) {
#pragma unroll
            for (int c = 0; c < C::VEC; ++c) {
                uu[c] += __shfl_xor_sync(0xffffffffu, uu[c], 16);
                ww[c] += __shfl_xor_sync(0xffffffffu, ww[c], 16);
            }
        }
        if (sub == 0) {
            float4 *ru = reinterpret_cast<float4 *>(red + cwarp * DK + strip * C::VEC);
            float4 *rw = reinterpret_cast<float4 *>(redw + cwarp * DK + strip * C::VEC);
#pragma unroll
            for (int e = 0; e < C::VEC / 4; ++e) {
                ru[e] = make_float4(uu[4 * e], uu[4 * e + 1], uu[4 * e + 2], uu[4 * e + 3]);
                rw[e] = make_float4(ww[4 * e], ww[4 * e + 1], ww[4 * e + 2], ww[4 * e + 3]);
            }
        }
        ptx::named_bar_sync(bar_id, C::GT);  // barrier 2: partial column sums

        // (e) threads 0-127 form d_j = beta (v_j - u_j) and publish rk d_j;
        // 128-255 sum w_j (raw)
        float wt = 0.f;
        if (ct < DK) {
            float ut = 0.f;
#pragma unroll
            for (int q = 0; q < C::CWARPS; ++q) ut += red[q * DK + ct];
            if (FOLD) {
                const float rk = 1.0f / sqrtf(nA + kL2Eps);
                db[ct] = rk * (beta * (vb[ct] - rk * ut));
            } else {
                db[ct] = beta * (vb[ct] - ut);
            }
        } else if (ct < 2 * DK) {
#pragma unroll
            for (int q = 0; q < C::CWARPS; ++q) wt += redw[q * DK + ct - DK];
        }
        ptx::named_bar_sync(bar_id, C::GT);  // barrier 3: d published
        if (ct >= DK && ct < 2 * DK) {  // o_j = scale (rq w_j + d_j (k_hat.q_hat)) = scale rq (w_j + (rk d_j) (k.q))
            float oj;
            if (FOLD) oj = a.scale * (1.0f / sqrtf(nrm[4] + kL2Eps)) * fmaf(db[ct - DK], nrm[5], wt);
            else oj = a.scale * fmaf(db[ct - DK], kqw, wt);
            if (NORM) {  // y_j = o_j / sqrt(mean o^2 + eps) * w_j * sigmoid(gate_j)
                float ss = oj * oj;
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
                if (lane == 0) nrm[(ct - DK) >> 5] = ss;
                ptx::named_bar_sync(3 + g, DK);
                ss = nrm[0] + nrm[1] + nrm[2] + nrm[3];
                oj = oj * rsqrtf(ss * (1.0f / DK) + a.norm_eps) * nw / (1.0f + __expf(-og));
            }
            a.o[(size_t)u * DK + ct - DK] = oj;
        }

        // (f) S' = s + k d, streamed out with 128-bit stores
        float dd[C::VEC];
#pragma unroll
        for (int e = 0; e < C::VEC / 4; ++e) {
            const float4 d4 = reinterpret_cast<const float4 *>(db + strip * C::VEC)[e];
            dd[4 * e] = d4.x;
            dd[4 * e + 1] = d4.y;
            dd[4 * e + 2] = d4.z;
            dd[4 * e + 3] = d4.w;
        }
        TS *Sg = static_cast<TS *>(a.state) + (size_t)u * DK * DK + strip * C::VEC;
#pragma unroll
        for (int p = 0; p < C::RPT; ++p) {
            const int row = p * C::RGROUPS + rg;
            float nv[C::VEC];
            const float2 k2 = make_float2(kr[p], kr[p]);
#pragma unroll
            for (int c = 0; c < C::VEC; c += 2) {  // packed FP32 pairs (fma.rn.f32x2)
                const float2 n2 = __ffma2_rn(k2, make_float2(dd[c], dd[c + 1]),
                                             make_float2(sv[p][c], sv[p][c + 1]));
                nv[c] = n2.x;
                nv[c + 1] = n2.y;
            }
            __stcs(reinterpret_cast<uint4 *>(Sg + (size_t)row * DK), Strip<TS>::pack(nv));
        }
    }

    // Exit. After a wait gave up, bulk copies into some stages may still be
    // in flight; once both groups are here no thread issues another one, so
    // waiting for the latest fill of every stage covers them all (in a run
    // without errors each of those has landed and was consumed: the waits
    // return at once).
    __syncthreads();
    if (tid == 0) {
        for (int s = 0; s < C::NST; ++s) {
            const uint32_t f = fills[s];
            if (f > 0) ptx::mbar_wait(&full[s], (f - 1) & 1, ptx::kDrainBudget);
        }
    }
}

// ---------------------------------------------------------------------------
// BF16 state, four consumer groups of four warps (launch_decode_stream with
// groups = 4). Same ring protocol, stage layout and arithmetic as the kernel
// above; what differs is the work split, for more heads in flight per SM:
//  * A group is 128 threads, one per channel: thread ct convolves q, k and v
//    channel ct and later forms d and o of value column ct, so a column's d
//    and o come from one thread.
//  * A thread holds 16 rows x 8 columns of the head's state packed as BF16
//    (64 registers) and widens them twice, once for the column sums and once
//    for the update (the state is rounded to BF16 exactly once, at the store,
//    as above).
//  * The fade is folded into the column sums (u = (alpha k).s, w = (alpha q).s)
//    and into the update (S' = alpha s + k (rk d)), so no faded copy is kept.
//  * Per row the conv thread publishes (alpha k, alpha q) for the column sums
//    and (alpha, k) for the update, 8 bytes each.
// ---------------------------------------------------------------------------
template <typename TX>
struct PCfg {
    using TS = __nv_bfloat16;
    using SC = Cfg<TS, TX, 2>;                   // the stage layout of load_head
    static constexpr int G = 4;
    static constexpr int CWARPS = kWarps / G;    // 4
    static constexpr int GT = CWARPS * 32;       // 128: one thread per channel
    static constexpr int THREADS = kWarps * 32;
    static constexpr int VEC = 8;                // BF16 columns per 16-byte strip
    static constexpr int STRIPS = DK / VEC;      // 16
    static constexpr int SUBS = 32 / STRIPS;     // 2 rows per warp instruction
    static constexpr int RGROUPS = CWARPS * SUBS;
    static constexpr int RPT = DK / RGROUPS;     // 16 rows per thread
    static_assert(GT == DK, "one thread per channel");
    static constexpr int STAGE = SC::STAGE;
    static constexpr int A_OFF = SC::A_OFF, X_OFF = SC::X_OFF, C_OFF = SC::C_OFF;
    // per group (floats): red_u, red_w [CWARPS][DK] | d [DK] | v [2][DK] |
    // per row (alpha k, alpha q) [DK][2] and (alpha, k) [DK][2], twice | norm
    // partials [CWARPS][4]. v and the row entries alternate by the group's head
    // parity: the update of one head still reads them after the last barrier
    // while faster threads write the next head's.
    static constexpr int REDW_F = CWARPS * DK;
    static constexpr int DB_F = 2 * CWARPS * DK;
    static constexpr int V_F = DB_F + DK;
    static constexpr int ROW_F = V_F + 2 * DK;
    static constexpr int NRM_F = ROW_F + 8 * DK;
    static constexpr int WORK_F = NRM_F + 4 * CWARPS;
    static constexpr int WORK_BYTES = WORK_F * 4;
    static constexpr int BAR_BYTES = 2 * 8 * 8 + 8 * 4;  // full[8], issued[8], fills[8]
    static constexpr int NST_FIT = (kSmemLimit - BAR_BYTES - G * WORK_BYTES) / STAGE;
    // a multiple of G, so every stage serves one group only: with four groups
    // and a stage shared between groups, a group running far enough ahead
    // could see a parity two phases old (tests/test_ring_protocol.py models it)
    static constexpr int NST = (NST_FIT > 8 ? 8 : NST_FIT) / G * G;
    static constexpr int SMEM = NST * STAGE + G * WORK_BYTES + BAR_BYTES;
    static_assert(NST >= G, "a stage per group at least");
    static_assert(STAGE % 16 == 0 && WORK_BYTES % 16 == 0, "16-byte alignment");
};

template <typename TX>
__global__ void __launch_bounds__(PCfg<TX>::THREADS, 1)
kda_decode_packed_kernel(const DecodeArgs a, const __grid_constant__ DecMaps mp) {
    using C = PCfg<TX>;
    using TS = __nv_bfloat16;
    constexpr int G = C::G;
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::NST * C::STAGE + G * C::WORK_BYTES);
    uint64_t *issued = full + 8;
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
            fills[s] = blockIdx.x + s * gridDim.x < n_units ? 1u : 0u;
        }
        ptx::fence_mbar_init();
        for (int s = 0; s < C::NST; ++s) {
            const int u = blockIdx.x + s * gridDim.x;
            if (u < n_units) prefetch_head<TS>(a, u);
        }
    }
    __syncthreads();
    ptx::grid_dependency_wait();
    ptx::launch_dependents();
    if (tid == 0) {
        for (int s = 0; s < C::NST; ++s) {
            const int u = blockIdx.x + s * gridDim.x;
            if (u < n_units) load_head<TS, TX, 2, false>(smem + s * C::STAGE, &full[s], a, mp, u, pol);
        }
    }

    const int g = warp / C::CWARPS;
    const int ct = tid - g * C::GT;              // channel / value column of this thread
    const int cwarp = ct >> 5;
    const int strip = lane % C::STRIPS, sub = lane / C::STRIPS;
    const int rg = cwarp * C::SUBS + sub;        // rows rg + RGROUPS p
    const uint32_t bar_id = 1 + g;
    float *red = reinterpret_cast<float *>(smem + C::NST * C::STAGE + g * C::WORK_BYTES);
    float *redw = red + C::REDW_F;
    float *db = red + C::DB_F;
    float *vb = red + C::V_F;
    float *rowd = red + C::ROW_F;
    float *nrm = red + C::NRM_F;
    TX *cache = static_cast<TX *>(a.cache);
    const float4 *w4 = reinterpret_cast<const float4 *>(a.conv_w);

    for (int i = g, u = blockIdx.x + g * gridDim.x; u < n_units; i += G, u += G * gridDim.x) {
        const int s = i % C::NST, n = i / C::NST;
        const int m = u / H, h = u - m * H;
        const size_t hb = (size_t)h * DK;
        const float4 wq = __ldg(w4 + hb + ct), wk = __ldg(w4 + D + hb + ct), wv = __ldg(w4 + 2 * D + hb + ct);
        const float beta = __ldg(a.beta + u);
        const int hp = (i / G) & 1;  // this head's v and row-entry buffers
        float *vbh = vb + hp * DK, *rowh = rowd + hp * 4 * DK;

        // the stage's refill was issued, then its bytes landed (a thread whose
        // wait gives up reads no further data and writes nothing; the group
        // leaves together at barrier 1)
        const bool landed = (n == 0 || ptx::mbar_wait(&issued[s], (n - 1) & 1, ptx::kWaitBudget)) &&
                            ptx::mbar_wait(&full[s], n & 1, ptx::kWaitBudget);
        if (!landed) raise_error(4u);
        const unsigned char *st = smem + s * C::STAGE;
        const TS *Ss = reinterpret_cast<const TS *>(st);
        const float *al = reinterpret_cast<const float *>(st + C::A_OFF);
        const TX *xs = reinterpret_cast<const TX *>(st + C::X_OFF);
        const TX *cs = reinterpret_cast<const TX *>(st + C::C_OFF);

        // (a) this thread's 16 x 8 state values, packed
        uint4 sp[C::RPT];
#pragma unroll
        for (int p = 0; p < C::RPT; ++p)
            sp[p] = *reinterpret_cast<const uint4 *>(Ss + (p * C::RGROUPS + rg) * DK + strip * C::VEC);

        // (b) conv + SiLU of channel ct of q, k and v; the row entry of key
        // channel ct; warp partials of k.k, q.q, q.k
        const size_t cbase = (size_t)m * 9 * D + hb;
        float qv = 0.f, kv = 0.f, vv = 0.f;
        if (landed) {
            qv = conv_stage(wq, cs, xs, 0, ct, cache + cbase + ct, D);
            kv = conv_stage(wk, cs, xs, 1, ct, cache + cbase + 3 * D + ct, D);
            vv = conv_stage(wv, cs, xs, 2, ct, cache + cbase + 6 * D + ct, D);
        }
        const float ar = al[ct];
        *reinterpret_cast<float2 *>(rowh + 2 * ct) = make_float2(ar * kv, ar * qv);
        *reinterpret_cast<float2 *>(rowh + 2 * DK + 2 * ct) = make_float2(ar, kv);
        vbh[ct] = vv;
        float nk = kv * kv, nq = qv * qv, nb = qv * kv;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            nk += __shfl_xor_sync(0xffffffffu, nk, off);
            nq += __shfl_xor_sync(0xffffffffu, nq, off);
            nb += __shfl_xor_sync(0xffffffffu, nb, off);
        }
        if (lane == 0) {
            nrm[4 * cwarp] = nk;
            nrm[4 * cwarp + 1] = nq;
            nrm[4 * cwarp + 2] = nb;
        }
        // barrier 1: stage read; rows, v, norm partials visible; every wait succeeded
        if (!ptx::named_bar_and(bar_id, C::GT, landed)) break;
        if (ct == 0) {
            const int ur = blockIdx.x + (i + C::NST) * gridDim.x;  // refill with head i + NST
            if (ur < n_units) {
                load_head<TS, TX, 2, false>(smem + s * C::STAGE, &full[s], a, mp, ur, pol);
                fills[s] = fills[s] + 1u;
                ptx::mbar_arrive(&issued[s]);
            }
        }
        float sk = 0.f, sq = 0.f, sb = 0.f;
#pragma unroll
        for (int w = 0; w < C::CWARPS; ++w) {
            sk += nrm[4 * w];
            sq += nrm[4 * w + 1];
            sb += nrm[4 * w + 2];
        }
        const float rk = 1.0f / sqrtf(sk + kL2Eps), rq = 1.0f / sqrtf(sq + kL2Eps);

        // (c) column sums u = (alpha k).s and w = (alpha q).s over this thread's rows
        float2 u2[4], w2[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) u2[c] = w2[c] = make_float2(0.f, 0.f);
#pragma unroll
        for (int p = 0; p < C::RPT; ++p) {
            const float2 rw = *reinterpret_cast<const float2 *>(rowh + 2 * (p * C::RGROUPS + rg));
            float f[8];
            Strip<TS>::unpack(sp[p], f);
            const float2 ka = make_float2(rw.x, rw.x), qa = make_float2(rw.y, rw.y);
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const float2 s2 = make_float2(f[2 * c], f[2 * c + 1]);
                u2[c] = __ffma2_rn(ka, s2, u2[c]);
                w2[c] = __ffma2_rn(qa, s2, w2[c]);
            }
        }
#pragma unroll
        for (int c = 0; c < 4; ++c) {  // the warp's two row groups
            u2[c].x += __shfl_xor_sync(0xffffffffu, u2[c].x, 16);
            u2[c].y += __shfl_xor_sync(0xffffffffu, u2[c].y, 16);
            w2[c].x += __shfl_xor_sync(0xffffffffu, w2[c].x, 16);
            w2[c].y += __shfl_xor_sync(0xffffffffu, w2[c].y, 16);
        }
        if (sub == 0) {
            float4 *ru = reinterpret_cast<float4 *>(red + cwarp * DK + strip * C::VEC);
            float4 *rw4 = reinterpret_cast<float4 *>(redw + cwarp * DK + strip * C::VEC);
            ru[0] = make_float4(u2[0].x, u2[0].y, u2[1].x, u2[1].y);
            ru[1] = make_float4(u2[2].x, u2[2].y, u2[3].x, u2[3].y);
            rw4[0] = make_float4(w2[0].x, w2[0].y, w2[1].x, w2[1].y);
            rw4[1] = make_float4(w2[2].x, w2[2].y, w2[3].x, w2[3].y);
        }
        ptx::named_bar_sync(bar_id, C::GT);  // barrier 2: partial column sums

        // (d) column ct: d = beta (v - u) (published as rk d) and o
        {
            float ut = 0.f, wt = 0.f;
#pragma unroll
            for (int w = 0; w < C::CWARPS; ++w) {
                ut += red[w * DK + ct];
                wt += redw[w * DK + ct];
            }
            const float dj = rk * (beta * (vbh[ct] - rk * ut));
            db[ct] = dj;
            a.o[(size_t)u * DK + ct] = a.scale * rq * fmaf(dj, sb, wt);
        }
        ptx::named_bar_sync(bar_id, C::GT);  // barrier 3: d published

        // (e) S' = alpha s + k (rk d), rounded once to BF16, streamed out
        float dd[8];
        {
            const float4 d0 = reinterpret_cast<const float4 *>(db + strip * C::VEC)[0];
            const float4 d1 = reinterpret_cast<const float4 *>(db + strip * C::VEC)[1];
            dd[0] = d0.x; dd[1] = d0.y; dd[2] = d0.z; dd[3] = d0.w;
            dd[4] = d1.x; dd[5] = d1.y; dd[6] = d1.z; dd[7] = d1.w;
        }
        TS *Sg = static_cast<TS *>(a.state) + (size_t)u * DK * DK + strip * C::VEC;
#pragma unroll
        for (int p = 0; p < C::RPT; ++p) {
            const int row = p * C::RGROUPS + rg;
            const float2 rw = *reinterpret_cast<const float2 *>(rowh + 2 * DK + 2 * row);
            // widened again here rather than kept from the column sums (an opaque
            // copy of the packed words, so the compiler does not keep 128 widened
            // values live across the barriers instead)
            uint4 pk;
            asm volatile("mov.b32 %0, %4;\n\tmov.b32 %1, %5;\n\tmov.b32 %2, %6;\n\tmov.b32 %3, %7;"
                         : "=r"(pk.x), "=r"(pk.y), "=r"(pk.z), "=r"(pk.w)
                         : "r"(sp[p].x), "r"(sp[p].y), "r"(sp[p].z), "r"(sp[p].w));
            float f[8], nv[8];
            Strip<TS>::unpack(pk, f);
            const float2 a2 = make_float2(rw.x, rw.x), k2 = make_float2(rw.y, rw.y);
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const float2 s2 = __fmul2_rn(a2, make_float2(f[2 * c], f[2 * c + 1]));
                const float2 n2 = __ffma2_rn(k2, make_float2(dd[2 * c], dd[2 * c + 1]), s2);
                nv[2 * c] = n2.x;
                nv[2 * c + 1] = n2.y;
            }
            __stcs(reinterpret_cast<uint4 *>(Sg + (size_t)row * DK), Strip<TS>::pack(nv));
        }
    }

    // Exit, as above: once all groups are here no thread issues another bulk
    // copy; the latest fill of every stage has landed before the CTA goes.
    __syncthreads();
    if (tid == 0) {
        for (int s = 0; s < C::NST; ++s) {
            const uint32_t f = fills[s];
            if (f > 0) ptx::mbar_wait(&full[s], (f - 1) & 1, ptx::kDrainBudget);
        }
    }
}

template <typename TS, typename TX, int G, bool GATE, bool NORM>
cudaError_t launch_stream_typed(const DecodeArgs &a, cudaStream_t stream) {
    using C = Cfg<TS, TX, G>;
    auto kernel = kda_decode_stream_kernel<TS, TX, G, GATE, NORM>;
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    DecMaps mp;
    e = make_decode_maps<TX>(&mp, a, sizeof(TS) == 2 || a.M * a.H <= kTensorInputsMaxHeadsF32);
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
    return cudaLaunchKernelEx(&cfg, kernel, a, mp);
}

template <typename TX>
cudaError_t launch_packed_typed(const DecodeArgs &a, cudaStream_t stream) {
    using C = PCfg<TX>;
    auto kernel = kda_decode_packed_kernel<TX>;
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    DecMaps mp;
    e = make_decode_maps<TX>(&mp, a, true);
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
    return cudaLaunchKernelEx(&cfg, kernel, a, mp);
}

template <typename TS, typename TX>
cudaError_t launch_groups(const DecodeArgs &a, int groups, cudaStream_t stream) {
    if (groups == 1) return launch_stream_typed<TS, TX, 1, false, false>(a, stream);
    if (groups == 2) return launch_stream_typed<TS, TX, 2, false, false>(a, stream);
    if constexpr (sizeof(TS) == 2) {
        if (groups == 4) return launch_packed_typed<TX>(a, stream);
    }
    return cudaErrorNotSupported;
}

template <typename TS, typename TX>
cudaError_t launch_fused(const DecodeArgs &a, cudaStream_t stream) {
    if (a.out_gate) return launch_stream_typed<TS, TX, 2, true, true>(a, stream);
    return launch_stream_typed<TS, TX, 2, true, false>(a, stream);
}

}  // namespace

cudaError_t launch_decode_stream(const DecodeArgs &a, int x_dtype, int state_dtype, int groups,
                                 cudaStream_t stream) {
    const bool xb = x_dtype == KDA_BF16, sb = state_dtype == KDA_BF16;
    if (sb && xb) return launch_groups<__nv_bfloat16, __nv_bfloat16>(a, groups, stream);
    if (sb) return launch_groups<__nv_bfloat16, float>(a, groups, stream);
    if (xb) return launch_groups<float, __nv_bfloat16>(a, groups, stream);
    return launch_groups<float, float>(a, groups, stream);
}

cudaError_t launch_decode_stream_fused(const DecodeArgs &a, int x_dtype, int state_dtype,
                                       cudaStream_t stream) {
    const bool xb = x_dtype == KDA_BF16, sb = state_dtype == KDA_BF16;
    if (sb && xb) return launch_fused<__nv_bfloat16, __nv_bfloat16>(a, stream);
    if (sb) return launch_fused<__nv_bfloat16, float>(a, stream);
    if (xb) return launch_fused<float, __nv_bfloat16>(a, stream);
    return launch_fused<float, float>(a, stream);
}

cudaError_t read_stream_error(unsigned int *code) {
    return cudaMemcpyFromSymbol(code, g_stream_error, sizeof(unsigned int));
}

cudaError_t clear_stream_error() {
    const unsigned int zero = 0;
    return cudaMemcpyToSymbol(g_stream_error, &zero, sizeof(unsigned int));
}

}  // namespace kda
