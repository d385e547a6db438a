// C ABI of the KDA library (declared and documented in include/kda.h):
// host-side argument checks, then one kernel launch on the caller's stream.
// Nothing here allocates memory or synchronises the device.

#include <cuda_runtime.h>

#include <cmath>
#include <cstddef>
#include <cstdint>

#include "../../include/kda.h"
#include "kda_internal.cuh"

namespace {

thread_local int g_last_cuda_error = 0;

kda_status cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return KDA_OK;
    g_last_cuda_error = static_cast<int>(e);
    return KDA_ERR_CUDA;
}

// most (stream, head) units one call may cover (2^30; far beyond any GPU's memory)
constexpr long long kMaxUnits = 1LL << 30;

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool valid_dtype(int t) { return t == KDA_F32 || t == KDA_BF16; }

size_t dtype_bytes(int t) { return t == KDA_BF16 ? 2u : 4u; }

// [a, a + na) and [b, b + nb) overlap
bool overlap(const void *a, size_t na, const void *b, size_t nb) {
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

// A buffer as the byte range a call touches (p may be null for an absent
// optional input).
struct Span {
    const void *p;
    size_t n;
};

// Every buffer a call writes is disjoint from every other one it writes and
// from every buffer it reads.
bool writes_disjoint(const Span *outs, int n_out, const Span *ins, int n_in) {
    for (int i = 0; i < n_out; ++i) {
        for (int j = i + 1; j < n_out; ++j)
            if (overlap(outs[i].p, outs[i].n, outs[j].p, outs[j].n)) return false;
        for (int j = 0; j < n_in; ++j)
            if (ins[j].p && overlap(outs[i].p, outs[i].n, ins[j].p, ins[j].n)) return false;
    }
    return true;
}

kda_status check_decode(const void *x, int x_dtype, const float *conv_w, void *conv_cache,
                        int cache_dtype, const float *alpha, const float *beta, void *state,
                        int state_dtype, float *o, int M, int H, int dk, int dv, int T = 1) {
    if (!x || !conv_w || !conv_cache || !alpha || !beta || !state || !o)
        return KDA_ERR_INVALID_ARG;
    if (M <= 0 || H <= 0 || dk <= 0 || dv <= 0 || T <= 0) return KDA_ERR_INVALID_ARG;
    if (!valid_dtype(x_dtype) || !valid_dtype(cache_dtype) || !valid_dtype(state_dtype))
        return KDA_ERR_INVALID_ARG;
    if (dk != kda::kHeadDim || dv != kda::kHeadDim) return KDA_ERR_UNSUPPORTED;
    if (cache_dtype != x_dtype) return KDA_ERR_UNSUPPORTED;
    // the kernels count (stream, head) units in 32-bit integers
    if (M > 65535 || H > 65535 || (long long)M * H > kMaxUnits) return KDA_ERR_UNSUPPORTED;
    if (!aligned16(x) || !aligned16(conv_w) || !aligned16(conv_cache) || !aligned16(alpha) ||
        !aligned16(beta) || !aligned16(state) || !aligned16(o))
        return KDA_ERR_ALIGNMENT;
    const size_t D = (size_t)H * dk;
    const Span outs[3] = {{o, (size_t)M * T * H * dv * sizeof(float)},
                          {state, (size_t)M * H * dk * dv * dtype_bytes(state_dtype)},
                          {conv_cache, (size_t)M * 9 * D * dtype_bytes(cache_dtype)}};
    const Span ins[4] = {{x, (size_t)M * T * 3 * D * dtype_bytes(x_dtype)},
                         {conv_w, (size_t)3 * D * 4 * sizeof(float)},
                         {alpha, (size_t)M * T * H * dk * sizeof(float)},
                         {beta, (size_t)M * T * H * sizeof(float)}};
    if (!writes_disjoint(outs, 3, ins, 4)) return KDA_ERR_INVALID_ARG;
    return KDA_OK;
}

kda_status check_prefill(const void *q, const void *k, const void *v, int qkv_dtype,
                         const float *alpha, const float *beta, const float *state,
                         const float *o, int M, int T, int H, int dk, int dv, int chunk) {
    if (!q || !k || !v || !alpha || !beta || !state || !o) return KDA_ERR_INVALID_ARG;
    if (M <= 0 || T <= 0 || H <= 0 || dk <= 0 || dv <= 0 || chunk <= 0)
        return KDA_ERR_INVALID_ARG;
    if (!valid_dtype(qkv_dtype)) return KDA_ERR_INVALID_ARG;
    if (dk != kda::kHeadDim || dv != kda::kHeadDim || chunk != 64) return KDA_ERR_UNSUPPORTED;
    // the kernels count (stream, head) units in 32-bit integers
    if (M > 65535 || H > 65535 || (long long)M * H > kMaxUnits) return KDA_ERR_UNSUPPORTED;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(alpha) ||
        !aligned16(beta) || !aligned16(state) || !aligned16(o))
        return KDA_ERR_ALIGNMENT;
    const size_t tok = (size_t)M * T * H;
    const size_t n_qkv = tok * dk * dtype_bytes(qkv_dtype);
    const Span outs[2] = {{o, tok * dv * 4}, {state, (size_t)M * H * dk * dv * 4}};
    const Span ins[5] = {{q, n_qkv}, {k, n_qkv}, {v, n_qkv}, {alpha, tok * dk * 4},
                         {beta, tok * 4}};
    if (!writes_disjoint(outs, 2, ins, 5)) return KDA_ERR_INVALID_ARG;
    return KDA_OK;
}

}  // namespace

extern "C" {

const char *kda_status_string(int status) {
    switch (status) {
        case KDA_OK: return "KDA_OK";
        case KDA_ERR_INVALID_ARG: return "KDA_ERR_INVALID_ARG";
        case KDA_ERR_UNSUPPORTED: return "KDA_ERR_UNSUPPORTED";
        case KDA_ERR_ALIGNMENT: return "KDA_ERR_ALIGNMENT";
        case KDA_ERR_CUDA: return "KDA_ERR_CUDA";
        case KDA_ERR_TIMEOUT: return "KDA_ERR_TIMEOUT";
        default: return "KDA_ERR_UNKNOWN";
    }
}

int kda_last_cuda_error(void) { return g_last_cuda_error; }

int kda_version(void) { return 100; }

kda_status kda_conv_step(const void *x, int x_dtype, const float *conv_w, void *conv_cache,
                         int cache_dtype, float *y, int M, int D, void *stream) {
    if (!x || !conv_w || !conv_cache || !y) return KDA_ERR_INVALID_ARG;
    if (M <= 0 || D <= 0) return KDA_ERR_INVALID_ARG;
    if (!valid_dtype(x_dtype) || !valid_dtype(cache_dtype)) return KDA_ERR_INVALID_ARG;
    if (cache_dtype != x_dtype) return KDA_ERR_UNSUPPORTED;
    if (!aligned16(x) || !aligned16(conv_w) || !aligned16(conv_cache) || !aligned16(y))
        return KDA_ERR_ALIGNMENT;
    const size_t b = dtype_bytes(x_dtype);
    const Span outs[2] = {{y, (size_t)M * 3 * D * sizeof(float)},
                          {conv_cache, (size_t)M * 9 * D * b}};
    const Span ins[2] = {{x, (size_t)M * 3 * D * b}, {conv_w, (size_t)3 * D * 4 * sizeof(float)}};
    if (!writes_disjoint(outs, 2, ins, 2)) return KDA_ERR_INVALID_ARG;
    return cuda_status(kda::launch_conv(x, x_dtype, conv_w, conv_cache, y, M, D,
                                        static_cast<cudaStream_t>(stream)));
}

kda_status kda_decode_step_config(const void *x, int x_dtype, const float *conv_w,
                                  void *conv_cache, int cache_dtype, const float *alpha,
                                  const float *beta, void *state, int state_dtype, float scale,
                                  float *o, int M, int H, int dk, int dv, int kernel,
                                  int columns, int threads, void *stream) {
    const kda_status st = check_decode(x, x_dtype, conv_w, conv_cache, cache_dtype, alpha, beta,
                                       state, state_dtype, o, M, H, dk, dv);
    if (st != KDA_OK) return st;
    const bool explicit_kernel = kernel != KDA_DECODE_AUTO;
    if (!explicit_kernel) kda::default_decode_config(M, H, state_dtype, &kernel, &columns, &threads);
    kda::DecodeArgs a = {};
    a.x = x;
    a.conv_w = conv_w;
    a.cache = conv_cache;
    a.alpha = alpha;
    a.beta = beta;
    a.state = state;
    a.o = o;
    a.M = M;
    a.H = H;
    a.scale = scale;
    const long long heads = (long long)M * H;
    a.l2_prefetch = state_dtype == KDA_F32 && heads >= kda::kL2PrefetchMinHeads &&
                            heads <= kda::kL2PrefetchMaxHeads
                        ? kda::kL2PrefetchMid
                        : kda::kDefaultL2Prefetch;
    // BF16 state: four groups of four warps with the state packed in registers
    int groups = state_dtype == KDA_BF16 ? kda::kDefaultGroupsBf16 : kda::kDefaultGroups;
    if (explicit_kernel && kernel == KDA_DECODE_STREAM) {
        if (columns < 0 || columns > 16) return KDA_ERR_UNSUPPORTED;
        a.l2_prefetch = columns;
        if (threads != 0) groups = threads;
    }
    cudaError_t e;
    if (kernel == KDA_DECODE_CLUSTER)
        e = kda::launch_decode(a, x_dtype, state_dtype, columns, threads,
                               static_cast<cudaStream_t>(stream));
    else if (kernel == KDA_DECODE_STREAM)
        e = kda::launch_decode_stream(a, x_dtype, state_dtype, groups,
                                      static_cast<cudaStream_t>(stream));
    else
        return KDA_ERR_INVALID_ARG;
    if (e == cudaErrorNotSupported) return KDA_ERR_UNSUPPORTED;
    return cuda_status(e);
}

kda_status kda_decode_step(const void *x, int x_dtype, const float *conv_w, void *conv_cache,
                           int cache_dtype, const float *alpha, const float *beta, void *state,
                           int state_dtype, float scale, float *o, int M, int H, int dk, int dv,
                           void *stream) {
    return kda_decode_step_config(x, x_dtype, conv_w, conv_cache, cache_dtype, alpha, beta, state,
                                  state_dtype, scale, o, M, H, dk, dv, KDA_DECODE_AUTO, 0, 0,
                                  stream);
}

kda_status kda_chunk_prefill_config(const void *q, const void *k, const void *v, int qkv_dtype,
                                    const float *alpha, const float *beta, float *state,
                                    float *o, float scale, int M, int T, int H, int dk, int dv,
                                    int chunk, int kernel, void *stream) {
    const kda_status st =
        check_prefill(q, k, v, qkv_dtype, alpha, beta, state, o, M, T, H, dk, dv, chunk);
    if (st != KDA_OK) return st;
    kda::PrefillArgs a = {};
    a.q = q;
    a.k = k;
    a.v = v;
    a.alpha = alpha;
    a.beta = beta;
    a.state = state;
    a.o = o;
    a.M = M;
    a.T = T;
    a.H = H;
    a.scale = scale;
    if (kernel == KDA_PREFILL_AUTO) kernel = KDA_PREFILL_TC;
    if (kernel == KDA_PREFILL_SIMT)
        return cuda_status(
            kda::launch_prefill_simt(a, qkv_dtype, static_cast<cudaStream_t>(stream)));
    if (kernel == KDA_PREFILL_TC)
        return cuda_status(kda::launch_prefill_tc(a, qkv_dtype, static_cast<cudaStream_t>(stream)));
    return KDA_ERR_INVALID_ARG;
}

kda_status kda_chunk_prefill(const void *q, const void *k, const void *v, int qkv_dtype,
                             const float *alpha, const float *beta, float *state, float *o,
                             float scale, int M, int T, int H, int dk, int dv, int chunk,
                             void *stream) {
    return kda_chunk_prefill_config(q, k, v, qkv_dtype, alpha, beta, state, o, scale, M, T, H, dk,
                                    dv, chunk, KDA_PREFILL_AUTO, stream);
}

kda_status kda_prefill_layer(const void *x, int x_dtype, const float *conv_w, void *conv_cache,
                             int cache_dtype, const float *gate_f, const float *A_log,
                             const float *dt_bias, float gate_lower_bound, const float *beta,
                             float *state, float scale, const float *out_gate,
                             const float *norm_weight, float norm_eps, float *y, int M, int T, int H,
                             int dk, int dv, int chunk, void *stream) {
    if (!x || !conv_w || !conv_cache || !gate_f || !A_log || !dt_bias || !beta || !state || !y ||
        (out_gate && !norm_weight))
        return KDA_ERR_INVALID_ARG;
    if (M <= 0 || T <= 0 || H <= 0 || dk <= 0 || dv <= 0 || chunk <= 0) return KDA_ERR_INVALID_ARG;
    if (!valid_dtype(x_dtype) || !valid_dtype(cache_dtype)) return KDA_ERR_INVALID_ARG;
    if (dk != kda::kHeadDim || dv != kda::kHeadDim || chunk != 64) return KDA_ERR_UNSUPPORTED;
    if (cache_dtype != x_dtype) return KDA_ERR_UNSUPPORTED;
    // the kernels count (stream, head) units in 32-bit integers
    if (M > 65535 || H > 65535 || (long long)M * H > kMaxUnits) return KDA_ERR_UNSUPPORTED;
    if (!aligned16(x) || !aligned16(conv_w) || !aligned16(conv_cache) || !aligned16(gate_f) ||
        !aligned16(A_log) || !aligned16(dt_bias) || !aligned16(beta) || !aligned16(state) ||
        !aligned16(y) || (out_gate && !aligned16(out_gate)) ||
        (norm_weight && !aligned16(norm_weight)))
        return KDA_ERR_ALIGNMENT;
    const size_t D = (size_t)H * dk, tok = (size_t)M * T * H;
    const Span outs[3] = {{y, tok * dv * 4},
                          {state, (size_t)M * H * dk * dv * 4},
                          {conv_cache, (size_t)M * 9 * D * dtype_bytes(cache_dtype)}};
    const Span ins[8] = {{x, (size_t)M * T * 3 * D * dtype_bytes(x_dtype)},
                         {conv_w, 3 * D * 4 * sizeof(float)},
                         {gate_f, tok * dk * 4},
                         {A_log, (size_t)H * sizeof(float)},
                         {dt_bias, D * sizeof(float)},
                         {beta, tok * 4},
                         {out_gate, tok * dv * 4},
                         {norm_weight, (size_t)dv * sizeof(float)}};
    if (!writes_disjoint(outs, 3, ins, 8)) return KDA_ERR_INVALID_ARG;
    kda::PrefillArgs a = {};
    a.q = x;
    a.alpha = gate_f;
    a.beta = beta;
    a.state = state;
    a.o = y;
    a.M = M;
    a.T = T;
    a.H = H;
    a.scale = scale;
    a.conv_w = conv_w;
    a.cache = conv_cache;
    a.A_log = A_log;
    a.dt_bias = dt_bias;
    a.gate_lb = gate_lower_bound;
    a.out_gate = out_gate;
    a.norm_w = norm_weight;
    a.norm_eps = norm_eps;
    return cuda_status(kda::launch_prefill_layer(a, x_dtype, static_cast<cudaStream_t>(stream)));
}

kda_status kda_decode_step_fused(const void *x, int x_dtype, const float *conv_w,
                                 void *conv_cache, int cache_dtype, const float *gate_f,
                                 const float *A_log, const float *dt_bias, float gate_lower_bound,
                                 const float *beta, void *state, int state_dtype, float scale,
                                 const float *out_gate, const float *norm_weight, float norm_eps,
                                 float *y, int M, int H, int dk, int dv, void *stream) {
    if (!A_log || !dt_bias || (out_gate && !norm_weight)) return KDA_ERR_INVALID_ARG;
    kda_status st = check_decode(x, x_dtype, conv_w, conv_cache, cache_dtype, gate_f, beta, state,
                                 state_dtype, y, M, H, dk, dv);
    if (st != KDA_OK) return st;
    if (!aligned16(A_log) || !aligned16(dt_bias) || (out_gate && !aligned16(out_gate)) ||
        (norm_weight && !aligned16(norm_weight)))
        return KDA_ERR_ALIGNMENT;
    // beyond check_decode: the written buffers against the gate and norm inputs
    const size_t D = (size_t)H * dk;
    const Span outs[3] = {{y, (size_t)M * H * dv * sizeof(float)},
                          {state, (size_t)M * H * dk * dv * dtype_bytes(state_dtype)},
                          {conv_cache, (size_t)M * 9 * D * dtype_bytes(cache_dtype)}};
    const Span ins[4] = {{A_log, (size_t)H * sizeof(float)},
                         {dt_bias, D * sizeof(float)},
                         {out_gate, (size_t)M * H * dv * sizeof(float)},
                         {norm_weight, (size_t)dv * sizeof(float)}};
    if (!writes_disjoint(outs, 3, ins, 4)) return KDA_ERR_INVALID_ARG;
    kda::DecodeArgs a = {};
    a.x = x;
    a.conv_w = conv_w;
    a.cache = conv_cache;
    a.alpha = gate_f;
    a.beta = beta;
    a.state = state;
    a.o = y;
    a.M = M;
    a.H = H;
    a.scale = scale;
    a.l2_prefetch = kda::kDefaultL2Prefetch;
    a.A_log = A_log;
    a.dt_bias = dt_bias;
    a.gate_lb = gate_lower_bound;
    a.out_gate = out_gate;
    a.norm_w = norm_weight;
    a.norm_eps = norm_eps;
    return cuda_status(kda::launch_decode_stream_fused(a, x_dtype, state_dtype,
                                                       static_cast<cudaStream_t>(stream)));
}

kda_status kda_decode_tokens(const void *x, int x_dtype, const float *conv_w, void *conv_cache,
                             int cache_dtype, const float *alpha, const float *beta, void *state,
                             int state_dtype, float scale, float *o, int M, int T, int H, int dk,
                             int dv, void *stream) {
    const kda_status st = check_decode(x, x_dtype, conv_w, conv_cache, cache_dtype, alpha, beta,
                                       state, state_dtype, o, M, H, dk, dv, T);
    if (st != KDA_OK) return st;
    kda::DecodeArgs a = {};
    a.x = x;
    a.conv_w = conv_w;
    a.cache = conv_cache;
    a.alpha = alpha;
    a.beta = beta;
    a.state = state;
    a.o = o;
    a.M = M;
    a.H = H;
    a.scale = scale;
    return cuda_status(kda::launch_decode_tokens(a, T, x_dtype, state_dtype,
                                                 static_cast<cudaStream_t>(stream)));
}

kda_status kda_device_error(void *stream) {
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_status(e);
    // all three words are read before any is cleared, so a failed read loses
    // nothing; then the words that were set are cleared
    unsigned int ws = 0, wp = 0, wt = 0;
    e = kda::read_stream_error(&ws);
    if (e == cudaSuccess) e = kda::read_prefill_error(&wp);
    if (e == cudaSuccess) e = kda::read_tokens_error(&wt);
    if (e != cudaSuccess) return cuda_status(e);
    if (ws) e = kda::clear_stream_error();
    if (e == cudaSuccess && wp) e = kda::clear_prefill_error();
    if (e == cudaSuccess && wt) e = kda::clear_tokens_error();
    if (e != cudaSuccess) return cuda_status(e);
    // a wait that gave up takes precedence over the prefill's alignment report
    if (ws || wt || (wp & ~kda::kPrefillErrMisaligned)) return KDA_ERR_TIMEOUT;
    if (wp & kda::kPrefillErrMisaligned) return KDA_ERR_ALIGNMENT;
    return KDA_OK;
}

}  // extern "C"
