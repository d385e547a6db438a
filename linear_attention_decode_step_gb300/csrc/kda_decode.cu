// Fused KDA decode step for sm_103a: short conv + SiLU, L2 norm of q and k,
// the gated delta rule and the readout, in one HBM read + write pass over
// the recurrent state.
//
// What one step computes per stream and head ("GLM-5.3 deep dive", section
// 8.2.3 Eq. 1 in the four-step order of section 8.2.6). Value column j of
// S is self-contained:
//     s_i  = alpha_i S[i][j]                 fade
//     u_j  = sum_i k_i s_i                   predict
//     w_j  = sum_i q_i s_i                   (read of the faded state)
//     d_j  = beta (v_j - u_j)                correct
//     S'[i][j] = s_i + k_i d_j
//     o_j  = scale (w_j + d_j (k . q))       read: S'^T q, expanded
// The last line is S'^T q written without a second pass over S'; the same
// identity appears in "At the 262k cap the DSA indexer costs 12x the sparse
// MLA it selects for", section "KDA decode step" (o = w + d (k . q)).
//
// Work split. A head's 128 value columns are cut into NS slices of CB
// columns; one CTA owns one (stream, head, slice) and the NS CTAs of a head
// form a thread-block cluster. Each thread owns a 16-byte strip of VEC
// columns in RPT rows: state loads and stores are 128-bit, a warp touches
// whole 32-byte sectors, and every state element is read once and written
// once. The column sums u and w are reduced in registers, then with warp
// shuffles over the lanes that share a strip, then across warps: each warp
// stores its partial sums as contiguous [warp][column] rows, CB column
// threads add them, form d and o, and publish d for the state update.
//
// Conv and normalisation. q and k are needed in full by every slice, but
// each CTA convolves only its own CB channels of q, k and v, so exactly one
// CTA reads and rewrites every conv-cache channel (no cross-CTA race on the
// cache). The CTA pushes its raw q, k values and its partial sums of q^2,
// k^2 and q.k into every peer's shared memory (DSMEM), then one cluster
// barrier publishes them. All CTAs of a head then hold identical q, k and
// norms, summed in the same order.
//
// The state loads are issued first, before the conv, so the HBM latency of
// the big read overlaps the small conv work. Launched with programmatic
// stream serialisation: each CTA waits for the preceding grid
// (griddepcontrol.wait) before its first global access and lets the next
// launch start placing CTAs right away, which hides the launch gap between
// consecutive layers (what dominates at a few streams).

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/kda.h"
#include "kda_internal.cuh"
#include "kda_ptx.cuh"

namespace kda {
namespace {

constexpr int DK = kHeadDim;
constexpr float kL2Eps = 1e-6f;

// ---------------------------------------------------------------- storage
template <typename TS> struct Strip;

template <> struct Strip<float> {
    static constexpr int VEC = 4;
    __device__ __forceinline__ static void unpack(const uint4 &r, float (&f)[VEC]) {
        f[0] = __uint_as_float(r.x); f[1] = __uint_as_float(r.y);
        f[2] = __uint_as_float(r.z); f[3] = __uint_as_float(r.w);
    }
    __device__ __forceinline__ static uint4 pack(const float (&f)[VEC]) {
        return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]),
                          __float_as_uint(f[2]), __float_as_uint(f[3]));
    }
};

__device__ __forceinline__ uint32_t bf16x2_rn(float lo, float hi) {
    __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&p);
}

template <> struct Strip<__nv_bfloat16> {
    static constexpr int VEC = 8;
    __device__ __forceinline__ static void unpack(const uint4 &r, float (&f)[VEC]) {
        const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            f[2 * e] = __uint_as_float(w[e] << 16);
            f[2 * e + 1] = __uint_as_float(w[e] & 0xffff0000u);
        }
    }
    __device__ __forceinline__ static uint4 pack(const float (&f)[VEC]) {
        return make_uint4(bf16x2_rn(f[0], f[1]), bf16x2_rn(f[2], f[3]),
                          bf16x2_rn(f[4], f[5]), bf16x2_rn(f[6], f[7]));
    }
};

// conv input / cache element (FP32 or BF16), widened exactly
__device__ __forceinline__ float widen(float v) { return v; }
__device__ __forceinline__ float widen(__nv_bfloat16 v) { return __bfloat162float(v); }

// ---------------------------------------------------------------- cluster
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t peer_addr(const void *local, uint32_t rank) {
    uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(local)), r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
    return r;
}
__device__ __forceinline__ void st_peer(uint32_t addr, float v) {
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}
// Split arrive / wait of the start-up barrier: a CTA may write into a peer's
// shared memory only once every CTA of the cluster is running.
__device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
    asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_barrier() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Short conv (kernel 4) + SiLU of one channel; rewrites its cache taps.
template <typename TX>
__device__ __forceinline__ float conv_silu(const TX *__restrict__ x, const float *__restrict__ w,
                                           TX *__restrict__ cache, int m, int X, size_t D,
                                           size_t ch) {
    const float4 wv = __ldg(reinterpret_cast<const float4 *>(w) + (size_t)X * D + ch);
    TX *c = cache + ((size_t)m * 3 + X) * 3 * D + ch;
    const TX c0 = c[0], c1 = c[D], c2 = c[2 * D];
    const TX xt = x[((size_t)m * 3 + X) * D + ch];
    const float pre = wv.x * widen(c0) + wv.y * widen(c1) + wv.z * widen(c2) + wv.w * widen(xt);
    c[0] = c1;
    c[D] = c2;
    c[2 * D] = xt;
    return pre / (1.0f + expf(-pre));
}

template <typename TS, typename TX, int CB, int NT>
__global__ void __launch_bounds__(NT) kda_decode_kernel(const DecodeArgs a) {
    constexpr int NS = DK / CB;               // slices (CTAs) per head = cluster size
    constexpr int VEC = Strip<TS>::VEC;       // columns per 16-byte strip
    constexpr int LPR = CB / VEC;             // lanes covering one row of the slice
    static_assert(LPR >= 1 && LPR <= 32 && 32 % LPR == 0, "bad strip split");
    constexpr int RPW = 32 / LPR;             // rows per warp per pass
    constexpr int NW = NT / 32;
    constexpr int RPP = NW * RPW;             // rows per pass of the CTA
    static_assert(DK % RPP == 0, "rows must split evenly");
    constexpr int RPT = DK / RPP;             // rows per thread
    constexpr int WPC = (CB + 31) / 32;       // warps holding conv partial sums
    static_assert(NT >= 2 * CB, "conv needs 2*CB threads");

    __shared__ float s_q[DK];
    __shared__ float s_k[DK];
    __shared__ float s_part[NS * WPC][4];
    __shared__ float s_v[CB];
    __shared__ __align__(16) float s_ru[NW][CB];
    __shared__ __align__(16) float s_rw[NW][CB];
    __shared__ __align__(16) float s_d[CB];

    const int slice = static_cast<int>(cluster_rank());
    const int h = blockIdx.y, m = blockIdx.z;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int cg = lane % LPR, rw = lane / LPR;
    const size_t head = (size_t)m * a.H + h;
    const size_t D = (size_t)a.H * DK;

    ptx::grid_dependency_wait();  // the previous grid's writes are visible from here on
    ptx::launch_dependents();

    // 1. issue the state loads (the HBM stream) and the per-row decays
    TS *Sg = static_cast<TS *>(a.state) + head * DK * DK + slice * CB + cg * VEC;
    uint4 raw[RPT];
    float al[RPT];
#pragma unroll
    for (int p = 0; p < RPT; ++p) {
        const int row = p * RPP + warp * RPW + rw;
        raw[p] = __ldcs(reinterpret_cast<const uint4 *>(Sg + (size_t)row * DK));
    }
#pragma unroll
    for (int p = 0; p < RPT; ++p) al[p] = __ldg(a.alpha + head * DK + p * RPP + warp * RPW + rw);
    const float beta = __ldg(a.beta + head);
    cluster_arrive_relaxed();

    // 2. conv + SiLU of this slice's channels of q, k (threads < CB) and v
    const TX *x = static_cast<const TX *>(a.x);
    TX *cache = static_cast<TX *>(a.cache);
    const size_t ch0 = (size_t)h * DK + slice * CB;
    float pq = 0.f, pk = 0.f, pqk = 0.f;
    float yq = 0.f, yk = 0.f;
    if (tid < CB) {
        yq = conv_silu(x, a.conv_w, cache, m, 0, D, ch0 + tid);
        yk = conv_silu(x, a.conv_w, cache, m, 1, D, ch0 + tid);
        pq = yq * yq;
        pk = yk * yk;
        pqk = yq * yk;
    } else if (tid < 2 * CB) {
        s_v[tid - CB] = conv_silu(x, a.conv_w, cache, m, 2, D, ch0 + tid - CB);
    }
    if (warp < WPC) {
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            pq += __shfl_xor_sync(0xffffffffu, pq, off);
            pk += __shfl_xor_sync(0xffffffffu, pk, off);
            pqk += __shfl_xor_sync(0xffffffffu, pqk, off);
        }
    }
    cluster_wait();  // every peer is running: DSMEM stores are allowed now
    if (tid < CB) {
#pragma unroll
        for (int r = 0; r < NS; ++r) {
            st_peer(peer_addr(&s_q[slice * CB + tid], r), yq);
            st_peer(peer_addr(&s_k[slice * CB + tid], r), yk);
        }
    }
    if (warp < WPC) {
        if (lane == 0) {
#pragma unroll
            for (int r = 0; r < NS; ++r) {
                st_peer(peer_addr(&s_part[slice * WPC + warp][0], r), pq);
                st_peer(peer_addr(&s_part[slice * WPC + warp][1], r), pk);
                st_peer(peer_addr(&s_part[slice * WPC + warp][2], r), pqk);
            }
        }
    }
    cluster_barrier();  // peers' q, k and partial sums (and local v) visible

    // 3. L2 norms of q and k, and k.q of the normalised vectors
    float sq = 0.f, sk = 0.f, sqk = 0.f;
#pragma unroll
    for (int i = 0; i < NS * WPC; ++i) {
        sq += s_part[i][0];
        sk += s_part[i][1];
        sqk += s_part[i][2];
    }
    const float rq = 1.0f / sqrtf(sq + kL2Eps);
    const float rk = 1.0f / sqrtf(sk + kL2Eps);
    const float kq = sqk * rq * rk;

    // 4. fade, then the column sums u = k.s and w = q.s over this thread's rows
    float st[RPT][VEC], kr[RPT];
    float u[VEC], w[VEC];
#pragma unroll
    for (int c = 0; c < VEC; ++c) u[c] = w[c] = 0.f;
#pragma unroll
    for (int p = 0; p < RPT; ++p) {
        const int row = p * RPP + warp * RPW + rw;
        kr[p] = s_k[row] * rk;
        const float qr = s_q[row] * rq;
        Strip<TS>::unpack(raw[p], st[p]);
#pragma unroll
        for (int c = 0; c < VEC; ++c) {
            st[p][c] *= al[p];
            u[c] = fmaf(kr[p], st[p][c], u[c]);
            w[c] = fmaf(qr, st[p][c], w[c]);
        }
    }
#pragma unroll
    for (int off = LPR; off < 32; off <<= 1) {
#pragma unroll
        for (int c = 0; c < VEC; ++c) {
            u[c] += __shfl_xor_sync(0xffffffffu, u[c], off);
            w[c] += __shfl_xor_sync(0xffffffffu, w[c], off);
        }
    }
    if (rw == 0) {
#pragma unroll
        for (int e = 0; e < VEC / 4; ++e) {
            reinterpret_cast<float4 *>(&s_ru[warp][cg * VEC])[e] =
                make_float4(u[4 * e], u[4 * e + 1], u[4 * e + 2], u[4 * e + 3]);
            reinterpret_cast<float4 *>(&s_rw[warp][cg * VEC])[e] =
                make_float4(w[4 * e], w[4 * e + 1], w[4 * e + 2], w[4 * e + 3]);
        }
    }
    __syncthreads();

    // 5. column threads: d = beta (v - u) and the readout o = scale (w + d (k.q))
    if (tid < CB) {
        float ut = 0.f, wt = 0.f;
#pragma unroll
        for (int ww = 0; ww < NW; ++ww) {
            ut += s_ru[ww][tid];
            wt += s_rw[ww][tid];
        }
        const float d = beta * (s_v[tid] - ut);
        s_d[tid] = d;
        a.o[head * DK + slice * CB + tid] = a.scale * fmaf(d, kq, wt);
    }
    __syncthreads();

    // 6. correct: S' = s + k d; 128-bit streaming stores
    float dcol[VEC];
#pragma unroll
    for (int e = 0; e < VEC / 4; ++e) {
        const float4 d4 = reinterpret_cast<const float4 *>(&s_d[cg * VEC])[e];
        dcol[4 * e] = d4.x;
        dcol[4 * e + 1] = d4.y;
        dcol[4 * e + 2] = d4.z;
        dcol[4 * e + 3] = d4.w;
    }
#pragma unroll
    for (int p = 0; p < RPT; ++p) {
        const int row = p * RPP + warp * RPW + rw;
        float nv[VEC];
#pragma unroll
        for (int c = 0; c < VEC; ++c) nv[c] = fmaf(kr[p], dcol[c], st[p][c]);
        __stcs(reinterpret_cast<uint4 *>(Sg + (size_t)row * DK), Strip<TS>::pack(nv));
    }
}

template <typename TS, typename TX, int CB, int NT>
cudaError_t launch_tile(const DecodeArgs &a, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(DK / CB, a.H, a.M);
    cfg.blockDim = dim3(NT, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = DK / CB;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kda_decode_kernel<TS, TX, CB, NT>, a);
}

template <typename TS, typename TX>
cudaError_t launch_typed(const DecodeArgs &a, int columns, int threads, cudaStream_t s) {
#define KDA_TILE(CB, NT) \
    if (columns == CB && threads == NT) return launch_tile<TS, TX, CB, NT>(a, s);
    KDA_TILE(16, 64)
    KDA_TILE(32, 64)
    KDA_TILE(32, 128)
    KDA_TILE(64, 128)
    KDA_TILE(64, 256)
    KDA_TILE(128, 256)
#undef KDA_TILE
    return cudaErrorNotSupported;
}

}  // namespace

cudaError_t launch_decode(const DecodeArgs &a, int x_dtype, int state_dtype, int columns,
                          int threads, cudaStream_t stream) {
    const bool xb = x_dtype == KDA_BF16, sb = state_dtype == KDA_BF16;
    if (sb && xb) return launch_typed<__nv_bfloat16, __nv_bfloat16>(a, columns, threads, stream);
    if (sb) return launch_typed<__nv_bfloat16, float>(a, columns, threads, stream);
    if (xb) return launch_typed<float, __nv_bfloat16>(a, columns, threads, stream);
    return launch_typed<float, float>(a, columns, threads, stream);
}

void default_decode_config(int M, int H, int state_dtype, int *kernel, int *columns,
                           int *threads) {
    // The streaming kernel is ahead at every M measured (1 to 64 streams x 64
    // heads, FP32 and BF16 state); the cluster kernel stays selectable.
    (void)M;
    (void)H;
    (void)state_dtype;
    *kernel = KDA_DECODE_STREAM;
    *columns = 32;
    *threads = 128;
}

}  // namespace kda
