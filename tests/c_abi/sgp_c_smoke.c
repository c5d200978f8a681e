/*
 * A plain C consumer of libsgp: no Python, no PyTorch.  It allocates one small decode layer's
 * weights, KV cache and activations with the CUDA runtime, runs the layer temporally
 * (sgp_layer_temporal) and as a two-stage spatial pipeline (sgp_pipeline_create / run /
 * sync), and checks that both return SGP_OK, that the output is finite and not constant, and
 * that the two outputs are bit-identical, as the header promises.
 *
 * Build (the GPU test does this):
 *   gcc -std=c11 -O2 -I include -I $CUDA/include sgp_c_smoke.c -L <dir of libsgp.so> -lsgp \
 *       -L $CUDA/lib64 -lcudart -Wl,-rpath,<dir of libsgp.so> -o sgp_c_smoke
 * Prints "c abi ok" and exits 0 on success; prints the failing step and exits 1 otherwise.
 */
#include <cuda_runtime_api.h>
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "sgp.h"

enum { H = 256, NQ = 4, NKV = 1, D = 64, E = 8, K = 2, EL = 8, I = 256, T = 8, CAP = 128 };

static uint32_t g_state = 12345u;
/* uniform in [-1, 1) from a 32-bit linear congruential generator */
static float next_uniform(void) {
    g_state = g_state * 1664525u + 1013904223u;
    return (float)(g_state >> 8) / (float)(1u << 23) - 1.0f;
}

/* float -> bfloat16 bits, round to nearest even (finite inputs only) */
static uint16_t to_bf16(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

static float from_bf16(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

static int fail(const char* what, const char* detail) {
    printf("FAIL %s: %s\n", what, detail ? detail : "");
    return 1;
}

#define CUDA_OK(call)                                                      \
    do {                                                                   \
        cudaError_t e_ = (call);                                           \
        if (e_ != cudaSuccess) return fail(#call, cudaGetErrorString(e_)); \
    } while (0)

#define SGP_OK_OR_FAIL(call)                                                          \
    do {                                                                              \
        int s_ = (call);                                                              \
        if (s_ != SGP_OK) {                                                           \
            printf("FAIL %s: %s (%s)\n", #call, sgp_status_string(s_), sgp_last_error()); \
            return 1;                                                                 \
        }                                                                             \
    } while (0)

/* a device bf16 tensor of n values drawn as scale * U[-1, 1) (+ offset) */
static int upload_bf16(void** dev, size_t n, float scale, float offset) {
    uint16_t* h = (uint16_t*)malloc(n * sizeof(uint16_t));
    if (!h) return fail("malloc", NULL);
    for (size_t i = 0; i < n; ++i) h[i] = to_bf16(offset + scale * next_uniform());
    cudaError_t e = cudaMalloc(dev, n * sizeof(uint16_t));
    if (e == cudaSuccess) e = cudaMemcpy(*dev, h, n * sizeof(uint16_t), cudaMemcpyHostToDevice);
    free(h);
    if (e != cudaSuccess) return fail("upload", cudaGetErrorString(e));
    return 0;
}

int main(void) {
    sgp_device_info info;
    SGP_OK_OR_FAIL(sgp_device_info_get(&info));

    sgp_dims d;
    memset(&d, 0, sizeof(d));
    d.hidden = H;
    d.n_q_heads = NQ;
    d.n_kv_heads = NKV;
    d.head_dim = D;
    d.n_experts = E;
    d.top_k = K;
    d.n_local_experts = EL;
    d.inter = I;
    d.rms_eps = 1e-5f;
    d.slot_map = 0;
    d.path = SGP_PATH_AUTO;
    d.gemv_max_tokens = 2;

    void *g_attn, *w_qkv, *w_o, *g_mlp, *w_router, *w_gate_up, *w_down, *kc, *vc, *x;
    if (upload_bf16(&g_attn, H, 0.02f, 1.0f) || upload_bf16(&w_qkv, (size_t)(NQ + 2 * NKV) * D * H, 0.035f, 0.f) ||
        upload_bf16(&w_o, (size_t)H * NQ * D, 0.035f, 0.f) || upload_bf16(&g_mlp, H, 0.02f, 1.0f) ||
        upload_bf16(&w_router, (size_t)E * H, 0.035f, 0.f) ||
        upload_bf16(&w_gate_up, (size_t)EL * 2 * I * H, 0.035f, 0.f) ||
        upload_bf16(&w_down, (size_t)EL * H * I, 0.035f, 0.f) ||
        upload_bf16(&kc, (size_t)T * NKV * CAP * D, 1.0f, 0.f) ||
        upload_bf16(&vc, (size_t)T * NKV * CAP * D, 1.0f, 0.f) ||
        upload_bf16(&x, (size_t)T * H, 1.0f, 0.f))
        return 1;

    int32_t kv_len_h[T];
    for (int t = 0; t < T; ++t) kv_len_h[t] = 1 + (t * 37) % CAP;  /* 1 .. 128, ragged */
    int32_t* kv_len;
    CUDA_OK(cudaMalloc((void**)&kv_len, sizeof(kv_len_h)));
    CUDA_OK(cudaMemcpy(kv_len, kv_len_h, sizeof(kv_len_h), cudaMemcpyHostToDevice));

    sgp_layer layer;
    memset(&layer, 0, sizeof(layer));
    layer.g_attn = g_attn;
    layer.w_qkv = w_qkv;
    layer.w_o = w_o;
    layer.g_mlp = g_mlp;
    layer.w_router = w_router;
    layer.router_bias = NULL;
    layer.w_gate_up = w_gate_up;
    layer.w_down = w_down;
    layer.k_cache = kc;
    layer.v_cache = vc;
    layer.kv_cap = CAP;
    layer.window = 0;

    /* temporal */
    const size_t ws_bytes = sgp_workspace_bytes(&d, T, CAP);
    if (ws_bytes == 0) return fail("sgp_workspace_bytes", "0");
    void *ws, *out_t, *out_p;
    CUDA_OK(cudaMalloc(&ws, ws_bytes));
    CUDA_OK(cudaMemset(ws, 0, ws_bytes));
    CUDA_OK(cudaMalloc(&out_t, (size_t)T * H * 2));
    CUDA_OK(cudaMalloc(&out_p, (size_t)T * H * 2));
    SGP_OK_OR_FAIL(sgp_layer_temporal(&d, &layer, kv_len, x, out_t, T, NULL, NULL, ws, ws_bytes,
                                      NULL, NULL));
    SGP_OK_OR_FAIL(sgp_status_from_workspace(ws, NULL));

    /* two-stage pipeline: the smallest legal pool for stage A, the rest for stage B */
    const int a = info.sm_alignment > 0 ? info.sm_alignment : 1;
    int pa = info.sm_min_partition > a ? info.sm_min_partition : a;
    pa = ((pa + a - 1) / a) * a;
    int split[2] = {pa, ((info.sm_count - pa) / a) * a};
    if (split[1] < pa) return fail("split", "GPU too small for two pools");
    sgp_pipeline* p = NULL;
    SGP_OK_OR_FAIL(sgp_pipeline_create(&d, split, 2, T / 2, T, CAP, NULL, &p));
    SGP_OK_OR_FAIL(sgp_pipeline_run(p, &layer, 1, kv_len, x, out_p, T, NULL, NULL, NULL));
    SGP_OK_OR_FAIL(sgp_pipeline_sync(p));
    sgp_pipeline_destroy(p);

    uint16_t ht[T * H], hp[T * H];
    CUDA_OK(cudaMemcpy(ht, out_t, sizeof(ht), cudaMemcpyDeviceToHost));
    CUDA_OK(cudaMemcpy(hp, out_p, sizeof(hp), cudaMemcpyDeviceToHost));
    float lo = INFINITY, hi = -INFINITY;
    for (int i = 0; i < T * H; ++i) {
        const float v = from_bf16(ht[i]);
        if (!isfinite(v)) return fail("output", "not finite");
        if (v < lo) lo = v;
        if (v > hi) hi = v;
    }
    if (!(hi > lo)) return fail("output", "constant");
    if (memcmp(ht, hp, sizeof(ht)) != 0) return fail("pipelined output", "differs from temporal");

    cudaFree(g_attn);
    cudaFree(w_qkv);
    cudaFree(w_o);
    cudaFree(g_mlp);
    cudaFree(w_router);
    cudaFree(w_gate_up);
    cudaFree(w_down);
    cudaFree(kc);
    cudaFree(vc);
    cudaFree(x);
    cudaFree(kv_len);
    cudaFree(ws);
    cudaFree(out_t);
    cudaFree(out_p);
    printf("c abi ok: %d x %d output in [%g, %g], pipeline %d | %d bit-identical to temporal\n", T,
           H, lo, hi, split[0], split[1]);
    return 0;
}
