// Standalone short convolution (kernel 4, three cached taps) + SiLU for one
// token over q, k and v ("GLM-5.3 deep dive", section 8.2.4, step 2;
// depthwise conv with weight [8192, 1, 4] per tensor, "At the 262k cap the
// DSA indexer costs 12x the sparse MLA it selects for", section "Geometry").
//
// One thread per channel: y = SiLU(w0 c0 + w1 c1 + w2 c2 + w3 x) with c0 the
// oldest cached input, then the cache shifts to (c1, c2, x). The fused decode
// kernel carries its own copy of this per-channel step; this entry point
// serves callers that want the convolved q, k, v themselves.

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "../../include/kda.h"
#include "kda_internal.cuh"

namespace kda {
namespace {

__device__ __forceinline__ float widen(float v) { return v; }
__device__ __forceinline__ float widen(__nv_bfloat16 v) { return __bfloat162float(v); }

template <typename TX>
__global__ void __launch_bounds__(256) kda_conv_kernel(const TX *__restrict__ x,
                                                       const float *__restrict__ w,
                                                       TX *__restrict__ cache,
                                                       float *__restrict__ y, int M, int D) {
    const size_t n = (size_t)M * 3 * D;
    for (size_t e = blockIdx.x * (size_t)blockDim.x + threadIdx.x; e < n;
         e += (size_t)gridDim.x * blockDim.x) {
        const size_t c = e % D;            // channel
        const size_t mX = e / D;           // m * 3 + X
        const size_t X = mX % 3;
        const float4 wv = __ldg(reinterpret_cast<const float4 *>(w) + X * D + c);
        TX *cc = cache + mX * 3 * D + c;
        const TX c0 = cc[0], c1 = cc[D], c2 = cc[2 * D];
        const TX xt = x[e];
        const float pre = wv.x * widen(c0) + wv.y * widen(c1) + wv.z * widen(c2) + wv.w * widen(xt);
        cc[0] = c1;
        cc[D] = c2;
        cc[2 * D] = xt;
        y[e] = pre / (1.0f + expf(-pre));
    }
}

}  // namespace

cudaError_t launch_conv(const void *x, int x_dtype, const float *conv_w, void *cache, float *y,
                        int M, int D, cudaStream_t stream) {
    int dev = 0, sms = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (err != cudaSuccess) return err;
    const size_t n = (size_t)M * 3 * D;
    size_t blocks = (n + 255) / 256;
    const size_t cap = (size_t)sms * 8;  // grid-stride beyond 8 CTAs per SM
    if (blocks > cap) blocks = cap;
    if (x_dtype == KDA_BF16)
        kda_conv_kernel<__nv_bfloat16><<<(unsigned)blocks, 256, 0, stream>>>(
            static_cast<const __nv_bfloat16 *>(x), conv_w, static_cast<__nv_bfloat16 *>(cache), y,
            M, D);
    else
        kda_conv_kernel<float><<<(unsigned)blocks, 256, 0, stream>>>(
            static_cast<const float *>(x), conv_w, static_cast<float *>(cache), y, M, D);
    return cudaGetLastError();
}

}  // namespace kda
