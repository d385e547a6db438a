// Internal declarations shared by the library's translation units (not part
// of the public ABI; the public surface is include/kda.h).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace kda {

constexpr int kHeadDim = 128;  // dk = dv handled by the decode and prefill kernels
constexpr int kDefaultL2Prefetch = 0;  // streaming decode: heads prefetched into L2 ahead
// kda_decode_step with FP32 state prefetches two heads into L2 beyond the
// ring from 768 to 2048 heads (measured on the 34-layer stack at 64 heads:
// M = 12 / 16 / 24 / 32 1.5 / 3.1 / 2.6 / 1.2 % faster; equal or slower at
// M <= 8 and M >= 40, and for the fused step and BF16 state)
constexpr int kL2PrefetchMid = 2, kL2PrefetchMinHeads = 768, kL2PrefetchMaxHeads = 2048;
constexpr int kDefaultGroups = 2;      // streaming decode: consumer groups per CTA (FP32 state)
constexpr int kDefaultGroupsBf16 = 4;  // BF16 state: four groups of four warps, state packed

// Arguments of one fused decode step (layouts as documented in kda.h).
struct DecodeArgs {
    const void *x;         // [M, 3, H*128] pre-conv q, k, v
    const float *conv_w;   // [3, H*128, 4]
    void *cache;           // [M, 3, 3, H*128]
    const float *alpha;    // [M, H, 128]
    const float *beta;     // [M, H]
    void *state;           // [M, H, 128, 128]
    float *o;              // [M, H, 128]
    int M, H;
    float scale;
    int l2_prefetch;       // streaming kernel: heads prefetched into L2 beyond the ring
    // fused forget gate: alpha holds the raw gate input f; alpha = exp(lb sigmoid(e^A (f + b)))
    const float *A_log;    // [H]
    const float *dt_bias;  // [H*128]
    float gate_lb;
    // fused gated RMSNorm on o: y = o / sqrt(mean o^2 + eps) * w * sigmoid(out_gate)
    const float *out_gate; // [M, H, 128]
    const float *norm_w;   // [128]
    float norm_eps;
};

// Arguments of one chunked prefill (layouts as documented in kda.h).
struct PrefillArgs {
    const void *q, *k, *v;  // [M, T, H, 128] post-conv (qkv dtype); the layer form: q = pre-conv x [M, T, 3, H*128]
    const float *alpha;     // [M, T, H, 128]; the layer form: raw forget-gate input f
    const float *beta;      // [M, T, H]
    float *state;           // [M, H, 128, 128] in / out
    float *o;               // [M, T, H, 128]
    int M, T, H;
    float scale;
    // the layer form (conv + SiLU, gate and optional gated RMSNorm fused in)
    const float *conv_w;    // [3, H*128, 4]
    void *cache;            // [M, 3, 3, H*128] (qkv dtype), in / out
    const float *A_log;     // [H]
    const float *dt_bias;   // [H*128]
    float gate_lb;
    const float *out_gate;  // [M, T, H, 128] or null (no norm)
    const float *norm_w;    // [128]
    float norm_eps;
};

// Encodes a tiled tensor map over a dense row-major tensor whose dims are
// listed innermost first (dims[0] contiguous; strides follow from the dims),
// with the given box, zero fill outside the tensor, optionally the 128-byte
// swizzle, and L2 promotion of the requests to 0: none, 1: 128 bytes,
// 2: 256 bytes. cudaErrorNotSupported if the driver lacks the encoder,
// cudaErrorInvalidValue if it rejects the map.
cudaError_t make_tensor_map(CUtensorMap *map, const void *base, bool bf16, int rank,
                            const uint64_t *dims, const uint32_t *box, bool swizzle128,
                            int l2_promotion = 2);

// Chunked prefill on CUDA cores (64-token chunks, 16-token blocks).
cudaError_t launch_prefill_simt(const PrefillArgs &a, int qkv_dtype, cudaStream_t stream);

// Chunked prefill on the tensor cores (tcgen05, TF32 operands, state in TMEM).
cudaError_t launch_prefill_tc(const PrefillArgs &a, int qkv_dtype, cudaStream_t stream);

// The tensor-core prefill of a whole KDA layer over a prompt: conv + SiLU of
// the pre-conv x with the cache as left context (cache updated), the forget
// gate from its raw input, the chunked recurrence and, if a.out_gate is set,
// the gated RMSNorm on every output.
cudaError_t launch_prefill_layer(const PrefillArgs &a, int x_dtype, cudaStream_t stream);

// Reads / clears the tensor-core prefill's device error word.
cudaError_t read_prefill_error(unsigned int *code);
cudaError_t clear_prefill_error();
// Bit of the prefill's error word set when its dynamic shared memory is not
// 1024-byte aligned (every other bit marks a bounded wait that gave up).
constexpr unsigned int kPrefillErrMisaligned = 64u;

// Launches the decode kernel for the given storage types and work split.
// Returns cudaErrorNotSupported (without launching) when no kernel is
// instantiated for (columns, threads).
cudaError_t launch_decode(const DecodeArgs &a, int x_dtype, int state_dtype,
                          int columns, int threads, cudaStream_t stream);

// Persistent streaming decode kernel (one CTA per SM, bulk-copy stages,
// `groups` = 1 or 2 consumer groups of 16 / 8 warps, or for BF16 state 4
// groups of 4 warps with the state packed in registers).
// cudaErrorNotSupported for other groups.
cudaError_t launch_decode_stream(const DecodeArgs &a, int x_dtype, int state_dtype, int groups,
                                 cudaStream_t stream);

// Streaming decode kernel with the forget gate fused in front (a.alpha is the
// raw gate input) and, if a.out_gate is set, the gated RMSNorm fused behind.
cudaError_t launch_decode_stream_fused(const DecodeArgs &a, int x_dtype, int state_dtype,
                                       cudaStream_t stream);

// T consecutive decode steps in one launch (x [M, T, 3, H*128], alpha
// [M, T, H, 128], beta [M, T, H], o [M, T, H, 128]; state and conv cache read
// once and written once).
cudaError_t launch_decode_tokens(const DecodeArgs &a, int T, int x_dtype, int state_dtype,
                                 cudaStream_t stream);

// Picks the decode kernel (KDA_DECODE_CLUSTER or KDA_DECODE_STREAM) and, for
// the cluster kernel, its work split (columns per CTA, threads per CTA).
void default_decode_config(int M, int H, int state_dtype, int *kernel, int *columns,
                           int *threads);

// Reads / clears the streaming kernel's device error word.
cudaError_t read_stream_error(unsigned int *code);
cudaError_t clear_stream_error();

// Reads / clears the multi-token decode kernel's device error word.
cudaError_t read_tokens_error(unsigned int *code);
cudaError_t clear_tokens_error();

// Standalone short conv + SiLU for one token.
cudaError_t launch_conv(const void *x, int x_dtype, const float *conv_w, void *cache,
                        float *y, int M, int D, cudaStream_t stream);

}  // namespace kda
