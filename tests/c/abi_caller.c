/*
 * A plain C99 caller of the KDA library: compiled with gcc against
 * include/kda.h (no C++ and no CUDA headers) and linked with libkda_gb300.so.
 * It exercises only the host side of the boundary: the diagnostics and the
 * argument checks that return before anything is launched, so it runs on a
 * machine without a GPU. Fake device addresses are 16-byte aligned, far
 * apart and never dereferenced.
 *
 * Prints "abi_caller: ok" and exits 0 when every check holds; otherwise
 * prints the failing check and exits 1.
 */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "kda.h"

static int failures = 0;

#define CHECK(cond)                                                        \
    do {                                                                   \
        if (!(cond)) {                                                     \
            fprintf(stderr, "abi_caller: line %d: %s\n", __LINE__, #cond); \
            ++failures;                                                    \
        }                                                                  \
    } while (0)

#define GAP ((uintptr_t)1 << 34)
#define BASE ((uintptr_t)1 << 40)

static void *addr(int slot) { return (void *)(BASE + (uintptr_t)slot * GAP); }
static float *faddr(int slot) { return (float *)addr(slot); }

static kda_status decode(void *x, const float *w, void *cache, const float *alpha,
                         const float *beta, void *state, float *o, int M, int H, int dk, int dv,
                         int x_dtype, int cache_dtype, int state_dtype) {
    return kda_decode_step(x, x_dtype, w, cache, cache_dtype, alpha, beta, state, state_dtype,
                           1.0f, o, M, H, dk, dv, NULL);
}

int main(void) {
    /* diagnostics */
    CHECK(kda_version() >= 100);
    CHECK(strcmp(kda_status_string(KDA_OK), "KDA_OK") == 0);
    CHECK(strcmp(kda_status_string(KDA_ERR_TIMEOUT), "KDA_ERR_TIMEOUT") == 0);
    CHECK(kda_status_string(12345) != NULL);
    CHECK(kda_last_cuda_error() == 0);

    /* decode step: each host-side rejection, in the header's terms */
    void *x = addr(0), *cache = addr(2), *state = addr(5);
    const float *w = faddr(1), *alpha = faddr(3), *beta = faddr(4);
    float *o = faddr(6);
    CHECK(decode(NULL, w, cache, alpha, beta, state, o, 4, 64, 128, 128, KDA_BF16, KDA_BF16,
                 KDA_F32) == KDA_ERR_INVALID_ARG);
    CHECK(decode(x, w, cache, alpha, beta, state, o, 0, 64, 128, 128, KDA_BF16, KDA_BF16,
                 KDA_F32) == KDA_ERR_INVALID_ARG);
    CHECK(decode(x, w, cache, alpha, beta, state, o, 4, 64, 64, 128, KDA_BF16, KDA_BF16,
                 KDA_F32) == KDA_ERR_UNSUPPORTED);
    CHECK(decode(x, w, cache, alpha, beta, state, o, 4, 64, 128, 128, KDA_BF16, KDA_F32,
                 KDA_F32) == KDA_ERR_UNSUPPORTED);
    CHECK(decode(x, w, cache, alpha, beta, state, o, 4, 64, 128, 128, 9, 9,
                 KDA_F32) == KDA_ERR_INVALID_ARG);
    CHECK(decode((char *)x + 8, w, cache, alpha, beta, state, o, 4, 64, 128, 128, KDA_BF16,
                 KDA_BF16, KDA_F32) == KDA_ERR_ALIGNMENT);
    CHECK(decode(x, w, cache, alpha, beta, state, (float *)((char *)state + 4096), 4, 64, 128,
                 128, KDA_BF16, KDA_BF16, KDA_F32) == KDA_ERR_INVALID_ARG);

    /* conv step */
    CHECK(kda_conv_step(x, KDA_BF16, w, cache, KDA_BF16, o, 0, 8192, NULL) ==
          KDA_ERR_INVALID_ARG);
    CHECK(kda_conv_step(x, KDA_BF16, w, cache, KDA_BF16, NULL, 2, 8192, NULL) ==
          KDA_ERR_INVALID_ARG);

    /* multi-token decode */
    CHECK(kda_decode_tokens(x, KDA_BF16, w, cache, KDA_BF16, alpha, beta, state, KDA_F32, 1.0f,
                            o, 4, 0, 64, 128, 128, NULL) == KDA_ERR_INVALID_ARG);

    /* chunked prefill: chunk other than 64, empty prompt, misaligned state */
    const void *q = addr(0), *k = addr(7), *v = addr(8);
    float *S = faddr(5), *O = faddr(6);
    CHECK(kda_chunk_prefill(q, k, v, KDA_BF16, alpha, beta, S, O, 1.0f, 4, 4096, 64, 128, 128,
                            32, NULL) == KDA_ERR_UNSUPPORTED);
    CHECK(kda_chunk_prefill(q, k, v, KDA_BF16, alpha, beta, S, O, 1.0f, 4, 0, 64, 128, 128, 64,
                            NULL) == KDA_ERR_INVALID_ARG);
    CHECK(kda_chunk_prefill(q, k, v, KDA_BF16, alpha, beta, (float *)((char *)S + 4), O, 1.0f,
                            4, 4096, 64, 128, 128, 64, NULL) == KDA_ERR_ALIGNMENT);

    /* prefill of a whole layer */
    CHECK(kda_prefill_layer(x, KDA_BF16, w, cache, KDA_BF16, alpha, faddr(9), faddr(10), -5.0f,
                            beta, S, 1.0f, NULL, NULL, 1e-5f, O, 4, 4096, 64, 128, 256, 64,
                            NULL) == KDA_ERR_UNSUPPORTED);

    /* a rejected call leaves no CUDA error behind */
    CHECK(kda_last_cuda_error() == 0);

    if (failures) return 1;
    printf("abi_caller: ok\n");
    return 0;
}
