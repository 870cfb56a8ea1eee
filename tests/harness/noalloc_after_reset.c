/*
 * noalloc_after_reset.c -- a plain C host program (no PyTorch) that calls
 * dit_attn_fwd_masked_noalloc, resets the device with cudaDeviceReset, and
 * calls it again on the same inputs.  The library's scratch array lives in its
 * own module: after the reset the runtime loads the module into a new primary
 * context, where the array has a new device address, so the second call is
 * right only if the library looks the address up again for the new context.
 * Prints "OK" and exits 0 when the two results are bit-identical, finite, and
 * the watchdog status is clean both times.
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime.h>

#include "dit_attn.h"

enum { B = 1, N = 640, H = 2, D = 128, KVL = 600 };
#define W (4 * ((KVL + 127) / 128)) /* mask words per row */

static uint32_t lcg(uint64_t* s) {
    *s = *s * 6364136223846793005ull + 1442695040888963407ull;
    return (uint32_t)(*s >> 33);
}

/* A float in [-2, 2) rounded down to bf16 (the upper 16 bits). */
static uint16_t rand_bf16(uint64_t* s) {
    float f = ((float)(lcg(s) & 0xffffff) / 16777216.0f) * 4.0f - 2.0f;
    uint32_t u;
    memcpy(&u, &f, 4);
    return (uint16_t)(u >> 16);
}

#define CHECK(x)                                                              \
    do {                                                                      \
        cudaError_t e_ = (x);                                                 \
        if (e_ != cudaSuccess) {                                              \
            fprintf(stderr, "%s: %s\n", #x, cudaGetErrorString(e_));          \
            return 1;                                                         \
        }                                                                     \
    } while (0)

/* One masked no-alloc call on fresh device buffers; O and LSE copied to host. */
static int run_once(const uint16_t* hq, const uint32_t* hmask, float* ho, float* hl) {
    const size_t n_qkv = (size_t)B * N * H * D;
    void *q, *k, *v, *out, *lse, *mask;
    CHECK(cudaMalloc(&q, n_qkv * 2));
    CHECK(cudaMalloc(&k, n_qkv * 2));
    CHECK(cudaMalloc(&v, n_qkv * 2));
    CHECK(cudaMalloc(&out, n_qkv * 4));
    CHECK(cudaMalloc(&lse, (size_t)B * H * N * 4));
    CHECK(cudaMalloc(&mask, (size_t)B * KVL * W * 4));
    CHECK(cudaMemcpy(q, hq, n_qkv * 2, cudaMemcpyHostToDevice));
    CHECK(cudaMemcpy(k, hq + n_qkv, n_qkv * 2, cudaMemcpyHostToDevice));
    CHECK(cudaMemcpy(v, hq + 2 * n_qkv, n_qkv * 2, cudaMemcpyHostToDevice));
    CHECK(cudaMemcpy(mask, hmask, (size_t)B * KVL * W * 4, cudaMemcpyHostToDevice));
    const dit_strides4_t s = {(int64_t)N * H * D, (int64_t)H * D, D, 1};
    const dit_attn_strides_t st = {s, s, s, s};
    dit_status_t rc = dit_attn_fwd_masked_noalloc(q, k, v, &st, B, N, N, H, D, KVL, (const uint32_t*)mask, 0, W,
                                                  KVL, 1.0f / sqrtf((float)D), out, DIT_F32, (float*)lse, NULL);
    if (rc != DIT_OK) {
        fprintf(stderr, "dit_attn_fwd_masked_noalloc: %s\n", dit_status_string(rc));
        return 1;
    }
    uint32_t info[4];
    rc = dit_check_watchdog(NULL, info);
    if (rc != DIT_OK) {
        fprintf(stderr, "watchdog: %s (%u %u %u %u)\n", dit_status_string(rc), info[0], info[1], info[2], info[3]);
        return 1;
    }
    CHECK(cudaMemcpy(ho, out, n_qkv * 4, cudaMemcpyDeviceToHost));
    CHECK(cudaMemcpy(hl, lse, (size_t)B * H * N * 4, cudaMemcpyDeviceToHost));
    CHECK(cudaFree(q));
    CHECK(cudaFree(k));
    CHECK(cudaFree(v));
    CHECK(cudaFree(out));
    CHECK(cudaFree(lse));
    CHECK(cudaFree(mask));
    return 0;
}

int main(void) {
    const size_t n_qkv = (size_t)B * N * H * D;
    uint16_t* hq = (uint16_t*)malloc(3 * n_qkv * 2);
    uint32_t* hmask = (uint32_t*)calloc((size_t)B * KVL * W, 4);
    float *o1 = (float*)malloc(n_qkv * 4), *o2 = (float*)malloc(n_qkv * 4);
    float *l1 = (float*)malloc((size_t)B * H * N * 4), *l2 = (float*)malloc((size_t)B * H * N * 4);
    if (!hq || !hmask || !o1 || !o2 || !l1 || !l2) return 1;
    uint64_t seed = 12345;
    for (size_t i = 0; i < 3 * n_qkv; ++i) hq[i] = rand_bf16(&seed);
    /* rows attend a 100-key band around themselves plus every 7th key */
    for (int i = 0; i < KVL; ++i)
        for (int j = 0; j < KVL; ++j)
            if ((j / 100 == i / 100) || j % 7 == 0) hmask[(size_t)i * W + j / 32] |= 1u << (j & 31);
    CHECK(cudaSetDevice(0));
    if (run_once(hq, hmask, o1, l1)) return 1;
    CHECK(cudaDeviceReset());        /* a new primary context on the next call */
    CHECK(cudaSetDevice(0));
    if (run_once(hq, hmask, o2, l2)) return 1;
    for (size_t i = 0; i < n_qkv; ++i)
        if (!isfinite(o1[i])) {
            fprintf(stderr, "non-finite O at %zu\n", i);
            return 1;
        }
    if (memcmp(o1, o2, n_qkv * 4) != 0 || memcmp(l1, l2, (size_t)B * H * N * 4) != 0) {
        fprintf(stderr, "results differ after the device reset\n");
        return 1;
    }
    printf("OK\n");
    return 0;
}
