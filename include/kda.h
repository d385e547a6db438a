/*
 * kda.h — C ABI of the GB300 (sm_103a) Kimi Delta Attention library.
 *
 * What it computes. Per stream m and head h, one decode step of a KDA layer:
 *   1. short convolution, kernel 4 (three cached taps), followed by SiLU, on
 *      each channel of the pre-conv q, k and v
 *      ("GLM-5.3 deep dive", section 8.2.4, steps 2 and 6; channel layout
 *      from "At the 262k cap the DSA indexer costs 12x the sparse MLA it
 *      selects for", section "Geometry": depthwise, weight [8192, 1, 4]);
 *   2. L2 normalisation of q and k: x / sqrt(sum x^2 + 1e-6)
 *      ("GLM-5.3 deep dive", section 8.2.6, implementation notes);
 *   3. the gated delta rule ("GLM-5.3 deep dive", section 8.2.3, Eq. 1)
 *         S <- (I - beta k k^T) Diag(alpha) S + beta k v^T,
 *      taken in the four-step order of section 8.2.6 (fade, predict,
 *      correct), on a dk x dv state;
 *   4. the readout o = scale * S^T q from the updated state (Eq. 1 with
 *      scale = 1; fla's default is 1 / sqrt(dk)).
 * The chunked prefill computes the same recurrence over T tokens of
 * post-conv q, k, v in the chunkwise WY / UT form of section 8.2.5 (Eq. 6-9).
 *
 * Conventions shared by every entry point.
 *   - Every buffer argument is a DEVICE pointer, owned by the caller. The
 *     library allocates nothing and keeps no pointer after the call returns.
 *   - Arrays are dense, row-major (C order), with the layouts stated per
 *     argument. D = H * d is the number of channels of one of q, k, v.
 *   - Every buffer pointer must be 16-byte aligned.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream). Work is enqueued on it; calls return without waiting.
 *   - Arguments are checked on the host before anything is launched. On any
 *     error status other than KDA_ERR_CUDA no buffer has been touched.
 *   - KDA_ERR_CUDA means a CUDA runtime call failed (for example the launch);
 *     kda_last_cuda_error() gives the cudaError_t value, per host thread.
 *   - No exceptions cross this boundary. There is no CPU fallback: every step
 *     of the computation runs in this library's kernels.
 *   - The entry points are thread-safe; they keep no mutable global state
 *     other than the per-thread last CUDA error and, on each device, the
 *     device error word that bounded waits set (see kda_device_error).
 */
#ifndef KDA_GB300_H
#define KDA_GB300_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    KDA_OK = 0,
    KDA_ERR_INVALID_ARG = 1, /* null pointer, non-positive size, overlapping outputs */
    KDA_ERR_UNSUPPORTED = 2, /* valid request this library does not implement (e.g. dk != 128) */
    KDA_ERR_ALIGNMENT = 3,   /* a buffer pointer is not 16-byte aligned */
    KDA_ERR_CUDA = 4,        /* a CUDA runtime call failed; see kda_last_cuda_error() */
    KDA_ERR_TIMEOUT = 5      /* a bounded device-side wait gave up */
} kda_status;

typedef enum {
    KDA_F32 = 0,  /* IEEE binary32 */
    KDA_BF16 = 1  /* bfloat16; values are widened exactly, stores round to nearest even */
} kda_dtype;

/* Human-readable name of a status code. Never NULL; static storage. */
const char *kda_status_string(int status);

/* cudaError_t of the last failed CUDA call made by this host thread inside
 * the library (0 if none). */
int kda_last_cuda_error(void);

/* Library ABI version (major * 100 + minor). */
int kda_version(void);

/*
 * kda_conv_step — short convolution + SiLU for one token, q, k and v at once.
 * ("GLM-5.3 deep dive", section 8.2.4, step 2; kernel 4, no bias.)
 *
 *   x           [M, 3, D]    pre-conv q, k, v of this token (x_dtype)
 *   conv_w      [3, D, 4]    FP32 weights; [.][c][3] multiplies the current
 *                            token, [.][c][0] the oldest cached one
 *   conv_cache  [M, 3, 3, D] the three previous inputs per channel, tap 0
 *                            oldest (cache_dtype, must equal x_dtype).
 *                            Updated in place to (tap1, tap2, x).
 *   y           [M, 3, D]    FP32 output: SiLU(w . [cache, x])
 *   M >= 1 streams, D >= 1 channels per tensor.
 * y and conv_cache (the buffers the call writes) must not overlap each other,
 * x or conv_w; an overlap returns KDA_ERR_INVALID_ARG.
 */
kda_status kda_conv_step(const void *x, int x_dtype, const float *conv_w,
                         void *conv_cache, int cache_dtype, float *y,
                         int M, int D, void *stream);

/*
 * kda_decode_step — one fused KDA decode step for M streams (conv + SiLU,
 * L2 norm of q and k, Eq. 1 update, readout), one launch.
 *
 *   x           [M, 3, H*dk] pre-conv q, k, v of this token (x_dtype)
 *   conv_w      [3, H*dk, 4] FP32 conv weights (as in kda_conv_step)
 *   conv_cache  [M, 3, 3, H*dk] conv cache (cache_dtype == x_dtype), in place
 *   alpha       [M, H, dk]   FP32 per-key-channel decay, linear space (0, 1]
 *   beta        [M, H]       FP32 write strength per head
 *   state       [M, H, dk, dv] recurrent state S[i][j] (i: key channel,
 *                            j: value channel), state_dtype; read and
 *                            written in place. With BF16 storage the
 *                            arithmetic is FP32 and the readout uses the
 *                            unrounded updated state; only the store rounds.
 *   scale       multiplies the readout (1.0 reproduces Eq. 1)
 *   o           [M, H, dv]   FP32 output
 *   dk = dv = 128 (other sizes return KDA_ERR_UNSUPPORTED); 1 <= M, H <= 65535
 *   and M * H <= 2^30 (KDA_ERR_UNSUPPORTED beyond).
 * The buffers the call writes (o, state, conv_cache) must not overlap each
 * other or any input; an overlap returns KDA_ERR_INVALID_ARG.
 * The streaming kernel reads x and the conv cache by tiled tensor copies
 * through maps encoded on the host at each call (cuTensorMapEncodeTiled via
 * the runtime's driver entry point), with BF16 state and, with FP32 state,
 * up to 1024 heads; a driver without that entry point returns
 * KDA_ERR_UNSUPPORTED before any launch. Under CUDA-graph capture the maps
 * are part of the captured launch.
 */
kda_status kda_decode_step(const void *x, int x_dtype, const float *conv_w,
                           void *conv_cache, int cache_dtype,
                           const float *alpha, const float *beta,
                           void *state, int state_dtype, float scale,
                           float *o, int M, int H, int dk, int dv, void *stream);

/*
 * kda_decode_step_fused — kda_decode_step with the layer's neighbouring steps
 * fused in: the KDA forget gate in front and, optionally, the gated RMSNorm
 * on the output ("GLM-5.3 deep dive", sections 8.2.3 and 8.2.4 step 7).
 *
 *   gate_f      [M, H, dk]  FP32 raw forget-gate input f (replaces alpha):
 *                           alpha = exp(lb * sigmoid(exp(A_log[h]) * (f + dt_bias[h*dk + i])))
 *   A_log       [H]         FP32
 *   dt_bias     [H * dk]    FP32
 *   gate_lower_bound        lb (-5 in GLM-5.3-Flash)
 *   out_gate    [M, H, dv]  FP32 output-gate input, or NULL for no norm
 *   norm_weight [dv]        FP32 RMSNorm weight (required with out_gate)
 *   norm_eps                RMSNorm eps (1e-5 in GLM-5.3-Flash)
 *   y           [M, H, dv]  FP32 output: o, or with out_gate
 *                           o / sqrt(mean(o^2) + norm_eps) * norm_weight * sigmoid(out_gate)
 * All other arguments, layouts and checks as kda_decode_step; the buffers the
 * call writes (y, state, conv_cache) must not overlap each other or any
 * input, the gate and norm inputs included.
 */
kda_status kda_decode_step_fused(const void *x, int x_dtype, const float *conv_w,
                                 void *conv_cache, int cache_dtype,
                                 const float *gate_f, const float *A_log, const float *dt_bias,
                                 float gate_lower_bound, const float *beta,
                                 void *state, int state_dtype, float scale,
                                 const float *out_gate, const float *norm_weight, float norm_eps,
                                 float *y, int M, int H, int dk, int dv, void *stream);

/*
 * kda_decode_tokens — T consecutive decode steps of one KDA layer for M
 * streams in one launch: token t = 0 .. T-1 goes through exactly the steps of
 * kda_decode_step, seeing the conv cache and state the previous token left
 * (the fused-recurrent mode of "GLM-5.3 deep dive" section 8.2.5, for a few
 * tokens at once, e.g. verifying drafted tokens). Each head's state and conv
 * cache are read from HBM once and written once per call.
 *
 *   x           [M, T, 3, H*dk] pre-conv q, k, v of the T tokens (x_dtype)
 *   conv_w      [3, H*dk, 4]    as kda_decode_step
 *   conv_cache  [M, 3, 3, H*dk] in place; afterwards it holds the last three
 *                               inputs of the sequence (cache, x_0 .. x_{T-1})
 *   alpha       [M, T, H, dk]   FP32 per-token decay, linear space
 *   beta        [M, T, H]       FP32
 *   state       [M, H, dk, dv]  in place. The state stays FP32 across the T
 *                               tokens; with BF16 storage it is rounded once,
 *                               when stored at the end of the call.
 *   o           [M, T, H, dv]   FP32 outputs of every token
 *   T >= 1 (state traffic is amortised over T; the arithmetic grows with T,
 *   so for long inputs the chunked prefill is the faster path). Calls of 3
 *   or more tokens regroup the recurrence into chunks of up to 8 tokens
 *   (section 8.2.4's WY form, FP32 throughout): results agree with the
 *   token-by-token order to FP32 rounding, and two calls split at a multiple
 *   of 8 tokens reproduce one call bit for bit.
 * Other arguments, checks and errors as kda_decode_step (sizes scale with T).
 * The chunked kernel stages x, alpha and the conv cache by tiled tensor
 * copies through maps encoded at each call (with BF16 x), and the
 * token-by-token kernel the conv cache (BF16 state, or FP32 state from 1024
 * heads); a map the driver rejects returns KDA_ERR_CUDA before any launch.
 */
kda_status kda_decode_tokens(const void *x, int x_dtype, const float *conv_w,
                             void *conv_cache, int cache_dtype,
                             const float *alpha, const float *beta,
                             void *state, int state_dtype, float scale,
                             float *o, int M, int T, int H, int dk, int dv, void *stream);

/* Decode kernels selectable through kda_decode_step_config. */
typedef enum {
    KDA_DECODE_AUTO = 0,    /* the library picks (what kda_decode_step does) */
    KDA_DECODE_CLUSTER = 1, /* one CTA per (stream, head, column slice); the slices of a
                               head form a thread-block cluster sharing q and k */
    KDA_DECODE_STREAM = 2   /* persistent: one CTA per SM streams whole heads through a
                               ring of shared-memory stages filled by bulk copies */
} kda_decode_kernel;

/*
 * kda_decode_step_config — kda_decode_step with an explicit kernel and work
 * split, for tuning and tests. With KDA_DECODE_CLUSTER each head's dv value
 * columns are split into slices of `columns` (16, 32, 64 or 128), one CTA of
 * `threads` threads each. With KDA_DECODE_STREAM, `columns` is the number of
 * heads (0-16) whose state is prefetched into L2 ahead of the shared-memory
 * ring (kda_decode_step uses 2 with FP32 state from 768 to 2048 heads, else
 * 0) and `threads` the number of consumer groups per CTA (1 or 2, or 4
 * with BF16 state: four groups of four warps holding the state packed; 0
 * picks the default: 2 for FP32 state, 4 for BF16). With `threads` = 4 the
 * L2 prefetch count is ignored.
 * Unsupported combinations return KDA_ERR_UNSUPPORTED. Same arguments,
 * layouts and results as kda_decode_step.
 */
kda_status kda_decode_step_config(const void *x, int x_dtype, const float *conv_w,
                                  void *conv_cache, int cache_dtype,
                                  const float *alpha, const float *beta,
                                  void *state, int state_dtype, float scale,
                                  float *o, int M, int H, int dk, int dv,
                                  int kernel, int columns, int threads, void *stream);

/* Prefill kernels selectable through kda_chunk_prefill_config. */
typedef enum {
    KDA_PREFILL_AUTO = 0,  /* the library picks (what kda_chunk_prefill does) */
    KDA_PREFILL_SIMT = 1,  /* CUDA-core chunk kernel: one CTA per (stream, head, 64 value
                              columns) walks the sequence chunk by chunk */
    KDA_PREFILL_TC = 2     /* tensor-core chunk kernel (tcgen05, TF32 operands, FP32
                              accumulation): one CTA per (stream, head), state kept in
                              tensor memory across its chunks; with more (stream, head)
                              pairs than SMs each sequence is cut into pieces of
                              consecutive chunks run in rounds of kernel launches, the
                              state passed between pieces in place (bit-identical) */
} kda_prefill_kernel;

/*
 * kda_chunk_prefill — the KDA recurrence over T tokens of post-conv q, k, v,
 * in the chunkwise WY / UT form ("GLM-5.3 deep dive", section 8.2.5, Eq. 6-9):
 * per (stream, head) the same result as T consecutive steps of steps 2-4 of
 * kda_decode_step (L2 norm of q and k, Eq. 1 update, readout), without the
 * convolution.
 *
 *   q, k, v  [M, T, H, dk]  post-conv inputs (qkv_dtype); q and k are
 *                           L2-normalised inside (eps 1e-6), v is not
 *   alpha    [M, T, H, dk]  FP32 per-key-channel decay, linear space (0, 1]
 *   beta     [M, T, H]      FP32 write strength
 *   state    [M, H, dk, dv] FP32, the state before the first token on entry
 *                           and after the last token on return (in place)
 *   o        [M, T, H, dv]  FP32 output, o_t = scale * S_t^T q_t
 *   chunk    tokens per chunk: 64 (other values return KDA_ERR_UNSUPPORTED)
 *   dk = dv = 128; 1 <= M, H <= 65535, M * H <= 2^30; T >= 1 (a ragged last
 *   chunk is fine).
 * Numerical domain: every per-token log(alpha) above about -5.4 (the model's
 * gate keeps it above -5), so that decay factors over a 16-token block stay
 * inside FP32.
 * o must not overlap any input or the state; the state must not overlap any
 * input.
 * The tensor-core path may issue several launches on `stream` (rounds of
 * pieces, see kda_prefill_kernel); they are stream-ordered and capturable in
 * a CUDA graph like a single launch.
 * The tensor-core kernel moves q, k, alpha, v and o by tiled tensor copies
 * through maps encoded on the host at each call (cuTensorMapEncodeTiled via
 * the runtime's driver entry point): a map the driver rejects (a stride of
 * 2^40 bytes or more, i.e. T * H * 256 * element size beyond that) returns
 * KDA_ERR_CUDA with kda_last_cuda_error() = cudaErrorInvalidValue, and a
 * driver without the entry point cudaErrorNotSupported, before any launch.
 */
kda_status kda_chunk_prefill(const void *q, const void *k, const void *v, int qkv_dtype,
                             const float *alpha, const float *beta, float *state, float *o,
                             float scale, int M, int T, int H, int dk, int dv, int chunk,
                             void *stream);

/*
 * kda_prefill_layer — a KDA layer over a prompt of T tokens for M streams on
 * the tensor cores (one launch, or rounds of pieces as kda_chunk_prefill):
 * the short conv + SiLU of the pre-conv q, k, v
 * with the conv cache as left context, the forget gate from its raw input
 * (in log space), L2 norm of q and k, the chunked recurrence ("GLM-5.3 deep
 * dive" sections 8.2.3 - 8.2.5) and, optionally, the gated RMSNorm on every
 * output (8.2.4 step 7). The result equals T calls of kda_decode_step_fused
 * within the prefill's tolerance (the conv's SiLU is evaluated through a
 * hardware tanh, relative error about 2^-11; products are TF32).
 *
 *   x           [M, T, 3, H*dk]  pre-conv q, k, v of the T tokens (x_dtype)
 *   conv_w      [3, H*dk, 4]     FP32 conv weights (as kda_conv_step)
 *   conv_cache  [M, 3, 3, H*dk]  in place; afterwards it holds the last three
 *                                inputs of (cache, x_0 .. x_{T-1})
 *   gate_f      [M, T, H, dk]    FP32 raw forget-gate input:
 *                                log alpha = lb * sigmoid(exp(A_log[h]) * (f + dt_bias[h*dk + i]))
 *   A_log [H], dt_bias [H * dk], gate_lower_bound (lb, -5 in GLM-5.3-Flash)
 *   beta        [M, T, H]        FP32
 *   state       [M, H, dk, dv]   FP32, in place
 *   out_gate    [M, T, H, dv]    FP32 output-gate input, or NULL for no norm
 *   norm_weight [dv], norm_eps   RMSNorm weight and eps (with out_gate)
 *   y           [M, T, H, dv]    FP32 output (o, or its gated RMSNorm)
 *   dk = dv = 128, chunk = 64 (KDA_ERR_UNSUPPORTED otherwise); cache_dtype ==
 *   x_dtype. The tensor-core arithmetic is TF32 with FP32 accumulation, as in
 *   kda_chunk_prefill, whose decay domain it shares (the gate keeps per-token
 *   log alpha above lb).
 * y, state and conv_cache must not overlap each other or any input.
 */
kda_status kda_prefill_layer(const void *x, int x_dtype, const float *conv_w,
                             void *conv_cache, int cache_dtype,
                             const float *gate_f, const float *A_log, const float *dt_bias,
                             float gate_lower_bound, const float *beta, float *state,
                             float scale, const float *out_gate, const float *norm_weight,
                             float norm_eps, float *y, int M, int T, int H, int dk, int dv,
                             int chunk, void *stream);

/* kda_chunk_prefill with an explicit kernel (kda_prefill_kernel). */
kda_status kda_chunk_prefill_config(const void *q, const void *k, const void *v, int qkv_dtype,
                                    const float *alpha, const float *beta, float *state,
                                    float *o, float scale, int M, int T, int H, int dk, int dv,
                                    int chunk, int kernel, void *stream);

/*
 * kda_device_error — waits for `stream` (cudaStream_t as void*, NULL = legacy
 * default stream), then reads the library's device error words (one per
 * kernel family) and clears those that were set. Returns, in this order of
 * precedence: KDA_ERR_CUDA if the wait, a read or a clear failed (a failed
 * read clears nothing); KDA_ERR_TIMEOUT if a kernel gave up a bounded
 * device-side wait since the words were last cleared (its outputs are then
 * incomplete); KDA_ERR_ALIGNMENT if the tensor-core prefill found its dynamic
 * shared memory not 1024-byte aligned (it then returns without computing; the
 * swizzled tensor copies need that alignment); KDA_OK otherwise.
 * The words are per device, shared by every stream and every caller of the
 * library in the process: callers that share a device and want their own
 * errors must serialise their calls of kda_device_error with their launches.
 */
kda_status kda_device_error(void *stream);

#ifdef __cplusplus
}
#endif

#endif /* KDA_GB300_H */
