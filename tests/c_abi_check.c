/*
 * c_abi_check.c -- the library used from plain C through include/attn.h only
 * (no Python, no torch): device buffers from the CUDA runtime, one causal GQA
 * prefill through attn_fwd and one paged decode step through
 * attn_decode_paged, each compared with a double-precision reference
 * computed here on the host from the definition (softmax of the scaled scores
 * over the visible keys, bottom-right causal alignment, kv head h / (Hq/Hkv)).
 * Exits 0 when every output element agrees within |a - b| <= 4e-3 + 8e-3 |b|
 * and every prefill log-sum-exp within 1e-3.
 *
 * Built and run by tests/test_c_abi_program.py:
 *   gcc -std=c11 -O2 c_abi_check.c -I include -I $CUDA/include -L <pkg> -lattn -L $CUDA/lib64 -lcudart -lm
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "attn.h"

static uint32_t rng_state = 12345u;
static float urand(void) { /* xorshift32 in [-1, 1) */
    rng_state ^= rng_state << 13;
    rng_state ^= rng_state >> 17;
    rng_state ^= rng_state << 5;
    return (float)(rng_state >> 8) / 8388608.0f - 1.0f;
}
static uint16_t to_bf16(float x) { /* round to nearest even (finite inputs) */
    uint32_t u;
    memcpy(&u, &x, 4);
    u += 0x7fffu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}
static double from_bf16(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

#define CHECK_CUDA(x)                                                         \
    do {                                                                      \
        if ((x) != cudaSuccess) {                                             \
            fprintf(stderr, "CUDA error at %s:%d\n", __FILE__, __LINE__);    \
            return 2;                                                         \
        }                                                                     \
    } while (0)
#define CHECK_ATTN(x)                                                                        \
    do {                                                                                     \
        attn_status_t st_ = (x);                                                             \
        if (st_ != ATTN_OK) {                                                                \
            fprintf(stderr, "%s failed: %s\n", #x, attn_status_string(st_));                 \
            return 3;                                                                        \
        }                                                                                    \
    } while (0)

static int within(double got, double want) { return fabs(got - want) <= 4e-3 + 8e-3 * fabs(want); }

static uint16_t *fill(size_t n) {
    uint16_t *h = (uint16_t *)malloc(n * 2);
    for (size_t i = 0; i < n; ++i) h[i] = to_bf16(urand());
    return h;
}

int main(void) {
    printf("attn_version %d\n", attn_version());
    /* ---- prefill: B=2, Hq=8, Hkv=2, S=300, causal, BSHD */
    const int B = 2, Hq = 8, Hkv = 2, S = 300, D = 128;
    const size_t nq = (size_t)B * S * Hq * D, nk = (size_t)B * S * Hkv * D;
    uint16_t *hq = fill(nq), *hk = fill(nk), *hv = fill(nk);
    void *q, *k, *v, *o1;
    float *l1;
    CHECK_CUDA(cudaMalloc(&q, nq * 2));
    CHECK_CUDA(cudaMalloc(&k, nk * 2));
    CHECK_CUDA(cudaMalloc(&v, nk * 2));
    CHECK_CUDA(cudaMalloc(&o1, nq * 2));
    CHECK_CUDA(cudaMalloc((void **)&l1, (size_t)B * Hq * S * 4));
    CHECK_CUDA(cudaMemcpy(q, hq, nq * 2, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(k, hk, nk * 2, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(v, hv, nk * 2, cudaMemcpyHostToDevice));
    const float scale = 0.08838834764831845f;
    CHECK_ATTN(attn_fwd(q, k, v, o1, l1, B, Hq, Hkv, S, S, D, ATTN_LAYOUT_BSHD, 1, scale, NULL));
    int site = 0;
    CHECK_ATTN(attn_get_device_status(NULL, &site));
    uint16_t *ho1 = (uint16_t *)malloc(nq * 2);
    float *hl1 = (float *)malloc((size_t)B * Hq * S * 4);
    CHECK_CUDA(cudaMemcpy(ho1, o1, nq * 2, cudaMemcpyDeviceToHost));
    CHECK_CUDA(cudaMemcpy(hl1, l1, (size_t)B * Hq * S * 4, cudaMemcpyDeviceToHost));
    size_t bad = 0, bad_lse = 0;
    double *sc = (double *)malloc(sizeof(double) * 512);
    for (int b = 0; b < B; ++b)
        for (int i = 0; i < S; ++i)
            for (int h = 0; h < Hq; ++h) {
                /* row (b, i, h) of a BSHD tensor; causal, Sq == Sk: keys 0 .. i */
                const int g = h / (Hq / Hkv);
                const size_t qrow = (((size_t)b * S + i) * Hq + h) * D;
                double m = -INFINITY, l = 0.0, o[128] = {0};
                for (int j = 0; j <= i; ++j) {
                    const size_t krow = (((size_t)b * S + j) * Hkv + g) * D;
                    double s = 0.0;
                    for (int c = 0; c < D; ++c) s += from_bf16(hq[qrow + c]) * from_bf16(hk[krow + c]);
                    sc[j] = s * scale;
                    if (sc[j] > m) m = sc[j];
                }
                for (int j = 0; j <= i; ++j) {
                    const size_t vrow = (((size_t)b * S + j) * Hkv + g) * D;
                    const double w = exp(sc[j] - m);
                    l += w;
                    for (int c = 0; c < D; ++c) o[c] += w * from_bf16(hv[vrow + c]);
                }
                for (int c = 0; c < D; ++c)
                    if (!within(from_bf16(ho1[qrow + c]), o[c] / l)) ++bad;
                if (fabs((double)hl1[((size_t)b * Hq + h) * S + i] - (m + log(l))) > 1e-3) ++bad_lse;
            }
    printf("prefill: %zu of %zu elements differ from the host reference (lse: %zu rows)\n", bad, nq, bad_lse);
    if (bad || bad_lse) return 1;

    /* ---- paged decode: 3 sequences, Hq=8, Hkv=2, 16-token pages in reverse order */
    const int DB = 3, PS = 16, MAXB = 8;
    const int lens[3] = {1, 37, 128};
    int npages = 0, table[3 * 8];
    for (int b = 0; b < DB; ++b)
        for (int pg = 0; pg < MAXB; ++pg) table[b * MAXB + pg] = pg < (lens[b] + PS - 1) / PS ? npages++ : -1;
    for (int i = 0; i < DB * MAXB; ++i) /* physical pages in reverse order */
        if (table[i] >= 0) table[i] = npages - 1 - table[i];
    const size_t npool = (size_t)npages * PS * Hkv * D, ndq = (size_t)DB * Hq * D;
    uint16_t *hkp = fill(npool), *hvp = fill(npool), *hdq = fill(ndq);
    void *kp, *vp, *dq, *dout, *ws;
    int32_t *dtable, *dlens;
    float *dlse;
    const size_t wsb = attn_decode_workspace_bytes(DB, Hq, D, MAXB);
    CHECK_CUDA(cudaMalloc(&kp, npool * 2));
    CHECK_CUDA(cudaMalloc(&vp, npool * 2));
    CHECK_CUDA(cudaMalloc(&dq, ndq * 2));
    CHECK_CUDA(cudaMalloc(&dout, ndq * 2));
    CHECK_CUDA(cudaMalloc((void **)&dlse, (size_t)DB * Hq * 4));
    CHECK_CUDA(cudaMalloc((void **)&dtable, sizeof table));
    CHECK_CUDA(cudaMalloc((void **)&dlens, sizeof lens));
    CHECK_CUDA(cudaMalloc(&ws, wsb));
    CHECK_CUDA(cudaMemcpy(kp, hkp, npool * 2, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(vp, hvp, npool * 2, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(dq, hdq, ndq * 2, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(dtable, table, sizeof table, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(dlens, lens, sizeof lens, cudaMemcpyHostToDevice));
    CHECK_ATTN(attn_decode_paged(dq, kp, vp, dtable, dlens, dout, dlse, DB, Hq, Hkv, D, PS, npages, MAXB, scale, ws,
                                 wsb, NULL));
    CHECK_ATTN(attn_get_device_status(NULL, &site));
    uint16_t *hdo = (uint16_t *)malloc(ndq * 2);
    CHECK_CUDA(cudaMemcpy(hdo, dout, ndq * 2, cudaMemcpyDeviceToHost));
    bad = 0;
    for (int b = 0; b < DB; ++b)
        for (int h = 0; h < Hq; ++h) {
            const int g = h / (Hq / Hkv);
            double m = -INFINITY, l = 0.0, o[128] = {0};
            for (int t = 0; t < lens[b]; ++t) {
                const size_t row = ((size_t)(table[b * MAXB + t / PS] * PS + t % PS) * Hkv + g) * D;
                double s = 0.0;
                for (int c = 0; c < D; ++c) s += from_bf16(hdq[((size_t)b * Hq + h) * D + c]) * from_bf16(hkp[row + c]);
                sc[t] = s * scale;
                if (sc[t] > m) m = sc[t];
            }
            for (int t = 0; t < lens[b]; ++t) {
                const size_t row = ((size_t)(table[b * MAXB + t / PS] * PS + t % PS) * Hkv + g) * D;
                const double w = exp(sc[t] - m);
                l += w;
                for (int c = 0; c < D; ++c) o[c] += w * from_bf16(hvp[row + c]);
            }
            for (int c = 0; c < D; ++c)
                if (!within(from_bf16(hdo[((size_t)b * Hq + h) * D + c]), o[c] / l)) ++bad;
        }
    printf("decode: %zu of %zu elements differ from the host reference\n", bad, ndq);
    return bad ? 1 : 0;
}
