/* A small DiT stack driven through the C ABI alone (no Python, no torch):
 * layout query, packing, device buffers and streams from the CUDA runtime,
 * registration, streamed forwards, statistics, slot verification, graphs,
 * teardown.  Prints "c abi ok" and exits 0 when every check holds. */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "dlo.h"

#define NB 3
#define D 256
#define HEADS 4
#define FFN 512
#define TOKENS 96

#define CHECK(cond, ...)                                  \
    do {                                                  \
        if (!(cond)) {                                    \
            fprintf(stderr, "check failed (%s:%d): ", __FILE__, __LINE__); \
            fprintf(stderr, __VA_ARGS__);                 \
            fprintf(stderr, "\n");                        \
            exit(1);                                      \
        }                                                 \
    } while (0)
#define DLO(call) CHECK((call) == DLO_OK, "%s: %s", #call, dlo_last_error(ctx))
#define CU(call) CHECK((call) == cudaSuccess, "%s", #call)

static uint32_t rng = 12345u;
static float uniform(void) { /* [-1, 1) */
    rng = rng * 1664525u + 1013904223u;
    return (float)(rng >> 8) / 8388608.0f - 1.0f;
}

static uint16_t to_bf16(float f) { /* round to nearest even (finite inputs) */
    uint32_t u;
    memcpy(&u, &f, 4);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

static float from_bf16(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* one forward; returns the output as bf16 bits in host memory */
static void forward(dlo_ctx* ctx, const void* dx, const void* dc, void* dy, uint16_t* out, size_t n) {
    DLO(dlo_forward(ctx, dx, dc, NULL, 1, TOKENS, 0, dy));
    DLO(dlo_wait(ctx, 60000));
    CU(cudaMemcpy(out, dy, n * 2, cudaMemcpyDeviceToHost));
}

int main(void) {
    dlo_ctx* ctx = NULL;
    dlo_desc d;
    memset(&d, 0, sizeof(d));
    d.abi_version = DLO_ABI_VERSION;
    d.block_kind = DLO_BLOCK_DIT;
    d.wdtype = DLO_W_BF16;
    d.n_blocks = NB;
    d.hidden = D;
    d.heads = HEADS;
    d.head_dim = D / HEADS;
    d.ffn = FFN;
    d.cond_dim = D;
    d.max_batch = 1;
    d.max_tokens = TOKENS;
    d.eps = 1e-6f;
    d.staging = DLO_STAGE_MEMCPY;

    /* layout and packing: every caller-supplied tensor N(0-ish) * 0.02 */
    const size_t bb = dlo_block_bytes(&d);
    const size_t ws = dlo_workspace_bytes(&d);
    CHECK(bb > 0 && ws > 0, "sizes %zu %zu", bb, ws);
    int count = 0;
    DLO(dlo_block_layout(&d, NULL, 0, &count));
    CHECK(count > 0, "layout count %d", count);
    dlo_tensor_info* info = (dlo_tensor_info*)calloc((size_t)count, sizeof(dlo_tensor_info));
    DLO(dlo_block_layout(&d, info, count, &count));
    void* host[NB];
    for (int b = 0; b < NB; ++b) {
        CU(cudaHostAlloc(&host[b], bb, cudaHostAllocDefault));
        const float** src = (const float**)calloc((size_t)count, sizeof(float*));
        for (int i = 0; i < count; ++i) {
            if (!info[i].source) continue;
            const size_t n = (size_t)info[i].shape[0] * (size_t)(info[i].ndim > 1 ? info[i].shape[1] : 1);
            float* t = (float*)malloc(n * sizeof(float));
            for (size_t j = 0; j < n; ++j) t[j] = 0.02f * uniform();
            src[i] = t;
        }
        DLO(dlo_pack_block(&d, src, count, host[b], bb));
        for (int i = 0; i < count; ++i) free((void*)src[i]);
        free(src);
    }

    /* device buffers and streams owned by the caller */
    void *slot0, *slot1, *wsp, *dx, *dc, *dy;
    cudaStream_t cs, xs;
    CU(cudaMalloc(&slot0, bb));
    CU(cudaMalloc(&slot1, bb));
    CU(cudaMalloc(&wsp, ws));
    const size_t nx = (size_t)TOKENS * D;
    CU(cudaMalloc(&dx, nx * 2));
    CU(cudaMalloc(&dy, nx * 2));
    CU(cudaMalloc(&dc, (size_t)D * 2));
    CU(cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking));
    CU(cudaStreamCreateWithFlags(&xs, cudaStreamNonBlocking));
    uint16_t* hx = (uint16_t*)malloc(nx * 2);
    uint16_t hc[D];
    for (size_t i = 0; i < nx; ++i) hx[i] = to_bf16(uniform());
    for (int i = 0; i < D; ++i) hc[i] = to_bf16(uniform());
    CU(cudaMemcpy(dx, hx, nx * 2, cudaMemcpyHostToDevice));
    CU(cudaMemcpy(dc, hc, (size_t)D * 2, cudaMemcpyHostToDevice));

    DLO(dlo_create(&d, 0, slot0, slot1, bb, wsp, ws, (void*)cs, (void*)xs, &ctx));
    DLO(dlo_register_host_blocks(ctx, NB, (const void* const*)host, bb, DLO_HOST_PINNED));

    uint16_t* y1 = (uint16_t*)malloc(nx * 2);
    uint16_t* y2 = (uint16_t*)malloc(nx * 2);
    uint16_t* y3 = (uint16_t*)malloc(nx * 2);
    forward(ctx, dx, dc, dy, y1, nx);
    forward(ctx, dx, dc, dy, y2, nx);
    CHECK(memcmp(y1, y2, nx * 2) == 0, "same input, different output");
    double diff = 0.0, norm = 0.0;
    for (size_t i = 0; i < nx; ++i) {
        const float a = from_bf16(y1[i]), x = from_bf16(hx[i]);
        CHECK(isfinite(a), "non-finite output at %zu", i);
        diff += (double)(a - x) * (a - x);
        norm += (double)x * x;
    }
    CHECK(diff > 0.0 && diff < norm, "the stack's update looks wrong: %g vs %g", diff, norm);

    dlo_stats st;
    DLO(dlo_get_stats(ctx, &st));
    CHECK(st.forwards == 2 && st.streamed_execs == 2 * NB, "forwards %llu execs %llu", st.forwards,
          st.streamed_execs);
    CHECK(st.stagings == 1 + 2 * NB && st.staged_bytes == st.stagings * bb, "stagings %llu bytes %llu",
          st.stagings, st.staged_bytes);
    CHECK(dlo_verify_slot(ctx, 0, -1) == DLO_OK && dlo_verify_slot(ctx, 1, -1) == DLO_OK, "slot bytes");
    CHECK(dlo_verify_slot(ctx, 0, st.slot_block[1]) == DLO_EMISMATCH || st.slot_block[0] == st.slot_block[1],
          "verify_slot did not notice a different block");

    /* whole-forward graphs give the same bits */
    DLO(dlo_set_graphs(ctx, 1));
    for (int r = 0; r < 3; ++r) {
        forward(ctx, dx, dc, dy, y3, nx);
        CHECK(memcmp(y1, y3, nx * 2) == 0, "graph forward %d differs", r);
    }
    DLO(dlo_get_stats(ctx, &st));
    CHECK(st.graph_launches >= 1, "no graph launch");

    /* errors come back as codes, the context stays usable */
    CHECK(dlo_forward(ctx, dx, dc, NULL, 1, TOKENS + 1, 0, dy) == DLO_EINVAL, "tokens > max accepted");
    forward(ctx, dx, dc, dy, y3, nx);
    CHECK(memcmp(y1, y3, nx * 2) == 0, "forward after a rejected call differs");

    DLO(dlo_destroy(ctx));
    ctx = NULL;
    for (int b = 0; b < NB; ++b) CU(cudaFreeHost(host[b]));
    CU(cudaFree(slot0));
    CU(cudaFree(slot1));
    CU(cudaFree(wsp));
    CU(cudaFree(dx));
    CU(cudaFree(dy));
    CU(cudaFree(dc));
    CU(cudaStreamDestroy(cs));
    CU(cudaStreamDestroy(xs));
    free(info);
    free(hx);
    free(y1);
    free(y2);
    free(y3);
    printf("c abi ok: %d blocks of %zu bytes, %llu stagings\n", NB, bb, st.stagings);
    return 0;
}
