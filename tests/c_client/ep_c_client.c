/* A plain C99 client of the library: no Python, no torch.  It sizes and
 * creates a handle, runs the layout, a bf16 dispatch and a combine with the
 * receive rows as the expert outputs, and checks the result against the
 * closed form of that chain computed on the host:
 *   out[n][h] = bf16( sum over valid k of w[n][k] * x[n][h] )
 * accumulated in float32 in slot order (each product rounded, then added),
 * which the combine's fused multiply-add may differ from by a few units in
 * the last place; the check allows 2 bf16 ulp plus the float32 bound.
 * Exit status 0 on success. */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "ep_layout.h"

#define CHECK_CUDA(x) do { if ((x) != cudaSuccess) { fprintf(stderr, "cuda error at %d\n", __LINE__); return 2; } } while (0)
#define CHECK_EP(x) do { ep_status s_ = (x); if (s_ != EP_OK) { fprintf(stderr, "%s at %d\n", ep_status_string(s_), __LINE__); return 3; } } while (0)

static uint32_t lcg(uint32_t* s) { *s = *s * 1664525u + 1013904223u; return *s >> 8; }

static uint16_t bf16_of(float f) {   /* round to nearest even; inputs are finite */
    uint32_t u; memcpy(&u, &f, 4);
    u += 0x7fffu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}
static float f_of(uint16_t b) { uint32_t u = (uint32_t)b << 16; float f; memcpy(&f, &u, 4); return f; }

int main(void) {
    const int R = 4, T = 96, H = 512, E = 16, K = 4;
    const int64_t N = (int64_t)R * T;
    ep_params p = {R, T, H, E, K, 1, 0};
    CHECK_EP(ep_params_validate(&p));
    size_t ws_bytes = 0;
    CHECK_EP(ep_layout_workspace_size(&p, &ws_bytes));

    /* host inputs: distinct experts per token, one in eight slots empty */
    int64_t* topk = (int64_t*)malloc(sizeof(int64_t) * N * K);
    float* w = (float*)malloc(sizeof(float) * N * K);
    uint16_t* x = (uint16_t*)malloc(2 * (size_t)N * H);
    uint16_t* out = (uint16_t*)malloc(2 * (size_t)N * H);
    uint32_t seed = 12345u;
    for (int64_t n = 0; n < N; ++n) {
        int base = (int)(lcg(&seed) % E);
        for (int k = 0; k < K; ++k) {
            topk[n * K + k] = (lcg(&seed) % 8 == 0) ? -1 : (base + 3 * k) % E;
            w[n * K + k] = (float)(lcg(&seed) % 1000) / 1000.0f;
        }
        for (int h = 0; h < H; ++h) x[n * H + h] = bf16_of((float)((int)(lcg(&seed) % 2001) - 1000) / 250.0f);
    }

    void *ws, *d_topk, *d_w, *d_x, *d_out, *d_recv;
    int64_t cap = N * K;
    CHECK_CUDA(cudaMalloc(&ws, ws_bytes));
    CHECK_CUDA(cudaMalloc(&d_topk, sizeof(int64_t) * N * K));
    CHECK_CUDA(cudaMalloc(&d_w, sizeof(float) * N * K));
    CHECK_CUDA(cudaMalloc(&d_x, 2 * (size_t)N * H));
    CHECK_CUDA(cudaMalloc(&d_out, 2 * (size_t)N * H));
    CHECK_CUDA(cudaMalloc(&d_recv, 2 * (size_t)cap * H));
    CHECK_CUDA(cudaMemcpy(d_topk, topk, sizeof(int64_t) * N * K, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(d_w, w, sizeof(float) * N * K, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(d_x, x, 2 * (size_t)N * H, cudaMemcpyHostToDevice));

    ep_handle* h = NULL;
    CHECK_EP(ep_handle_create(&p, ws, ws_bytes, &h));
    CHECK_EP(ep_layout(h, (const int64_t*)d_topk, NULL));
    int64_t* rank_base = (int64_t*)malloc(sizeof(int64_t) * (R + 1));
    CHECK_EP(ep_handle_recv_rows(h, rank_base, NULL));
    CHECK_EP(ep_dispatch(h, d_x, EP_QUANT_NONE, d_recv, NULL, cap, NULL));
    CHECK_EP(ep_combine(h, d_recv, cap, (const float*)d_w, NULL, 0, d_out, NULL));
    CHECK_EP(ep_handle_status(h, NULL));
    CHECK_CUDA(cudaMemcpy(out, d_out, 2 * (size_t)N * H, cudaMemcpyDeviceToHost));

    int64_t valid = 0;
    for (int64_t i = 0; i < N * K; ++i) valid += topk[i] >= 0;
    if (rank_base[R] != valid) { fprintf(stderr, "rows %lld != valid %lld\n", (long long)rank_base[R], (long long)valid); return 4; }

    int bad = 0;
    for (int64_t n = 0; n < N && bad < 5; ++n)
        for (int hh = 0; hh < H; ++hh) {
            float acc = 0.0f, mag = 0.0f;
            float xv = f_of(x[n * H + hh]);
            for (int k = 0; k < K; ++k)
                if (topk[n * K + k] >= 0) {
                    float prod = w[n * K + k] * xv;
                    acc = acc + prod;
                    mag += fabsf(prod);
                }
            float got = f_of(out[n * H + hh]);
            int ex; frexpf(acc, &ex);
            float ulp = ldexpf(1.0f, ex - 8);
            float bound = 2.0f * ulp + (2.0f * K + 2.0f) * ldexpf(1.0f, -24) * mag + ldexpf(1.0f, -126);
            if (fabsf(got - acc) > bound + ulp) {
                fprintf(stderr, "token %lld h %d: got %g want %g\n", (long long)n, hh, got, acc);
                ++bad;
            }
        }
    ep_handle_destroy(h);
    cudaFree(ws); cudaFree(d_topk); cudaFree(d_w); cudaFree(d_x); cudaFree(d_out); cudaFree(d_recv);
    free(topk); free(w); free(x); free(out); free(rank_base);
    if (bad) return 5;
    printf("c client ok: %lld rows\n", (long long)valid);
    return 0;
}
