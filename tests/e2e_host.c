/*
 * The bench's end-to-end decode step driven from plain C through the
 * library's C ABI (include/kvq.h) and the CUDA runtime, with no Python in
 * the loop.  Per step, as bench.py's e2e leg does through the Python
 * binding: one pinned host -> device copy of the step's inputs (the new
 * cell's K and V, the query, its position and the context length, packed
 * back to back), kvq_append + kvq_decode_attn on an FP16 cache and on an
 * int8 cache, one device -> host copy of both outputs into pinned memory,
 * and a stream synchronize.  The difference between the two legs' times
 * is the cost of the binding and the Python around it.
 *
 * Geometry of the gqa32k decode workload ([kv-q8 PR], "Summary": the
 * decode of the next token over a 32K-cell context): batch 1, 32 query
 * heads, 8 KV heads, head_dim 128, block size 256 (a shuffled block
 * table), 32768 prefilled cells, step j appends cell 32768 + j and decodes
 * over 32769 + j cells; `layers` caches of each format are rotated (step s
 * uses layer s % layers).  Inputs are seeded values of the same shapes;
 * the timing does not depend on them.
 *
 * usage: e2e_host <steps> <warmup> <layers> [device]
 * prints one line of name-value pairs: ms_per_step, h2d_bytes, d2h_bytes,
 * and the host microseconds per step spent enqueueing the two copies, in
 * the four library calls and waiting in the synchronize; exit status 0 on
 * success, 1 on any CUDA or library error (with a message on stderr).
 */
#define _POSIX_C_SOURCE 199309L /* clock_gettime in strict C */

#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>
#include <time.h>

#include <cuda_runtime.h>

#include "kvq.h"

enum { N_KV = 8, N_Q = 32, HD = 128, BS = 256, L0 = 32768, STEPS_PER_LAYER = 64 };

#define CK(x)                                                                        \
    do {                                                                             \
        cudaError_t e_ = (x);                                                        \
        if (e_ != cudaSuccess) {                                                     \
            fprintf(stderr, "%s:%d %s: %s\n", __FILE__, __LINE__, #x,                \
                    cudaGetErrorString(e_));                                         \
            exit(1);                                                                 \
        }                                                                            \
    } while (0)

#define KV(x)                                                                        \
    do {                                                                             \
        kvq_status s_ = (x);                                                         \
        if (s_ != KVQ_OK) {                                                          \
            fprintf(stderr, "%s:%d %s: %s\n", __FILE__, __LINE__, #x,                \
                    kvq_status_string(s_));                                          \
            exit(1);                                                                 \
        }                                                                            \
    } while (0)

/* splitmix64: seeded 64-bit values */
static uint64_t mix_state = 0x243f6a8885a308d3ull;
static uint64_t next_u64(void) {
    uint64_t z = (mix_state += 0x9e3779b97f4a7c15ull);
    z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ull;
    z = (z ^ (z >> 27)) * 0x94d049bb133111ebull;
    return z ^ (z >> 31);
}
/* roughly N(0, 1): a centred sum of four uniforms, scaled */
static float next_value(void) {
    float s = 0.f;
    for (int i = 0; i < 4; ++i) s += (float)(next_u64() >> 40) * (1.0f / 16777216.0f);
    return (s - 2.0f) * 1.7320508f;
}

static double now_s(void) {
    struct timespec ts;
    clock_gettime(CLOCK_MONOTONIC, &ts);
    return (double)ts.tv_sec + 1e-9 * (double)ts.tv_nsec;
}

typedef struct {
    kvq_cache cache;
    void *ws;
    size_t ws_bytes;
} layer_t;

static void make_layer(layer_t *ly, int fmt, int n_blocks) {
    const size_t cells = (size_t)n_blocks * N_KV * BS;
    const size_t esz = fmt == KVQ_F16 ? 2 : 1;
    memset(ly, 0, sizeof(*ly));
    ly->cache.fmt = fmt;
    ly->cache.n_kv_heads = N_KV;
    ly->cache.head_dim = HD;
    ly->cache.block_size = BS;
    ly->cache.n_blocks = n_blocks;
    CK(cudaMalloc(&ly->cache.k_data, cells * HD * esz));
    CK(cudaMalloc(&ly->cache.v_data, cells * HD * esz));
    if (fmt == KVQ_Q8) {
        CK(cudaMalloc(&ly->cache.k_scales, cells * (HD / KVQ_GROUP) * 2));
        CK(cudaMalloc(&ly->cache.v_scales, cells * (HD / KVQ_GROUP) * 2));
    }
}

int main(int argc, char **argv) {
    if (argc != 4 && argc != 5) {
        fprintf(stderr, "usage: %s <steps> <warmup> <layers> [device]\n", argv[0]);
        return 1;
    }
    const int K = atoi(argv[1]), W = atoi(argv[2]), LAYERS = atoi(argv[3]);
    if (K <= 0 || W < 0 || LAYERS <= 0) return 1;
    CK(cudaSetDevice(argc == 5 ? atoi(argv[4]) : 0));
    const int cap = L0 + STEPS_PER_LAYER;
    const int n_blocks = (cap + BS - 1) / BS;
    const float sm_scale = 1.0f / sqrtf((float)HD);

    /* shuffled block table (Fisher-Yates over the seeded generator) */
    int32_t *table = (int32_t *)malloc(sizeof(int32_t) * n_blocks);
    for (int i = 0; i < n_blocks; ++i) table[i] = i;
    for (int i = n_blocks - 1; i > 0; --i) {
        const int j = (int)(next_u64() % (uint64_t)(i + 1));
        const int32_t t = table[i];
        table[i] = table[j];
        table[j] = t;
    }
    int32_t *d_table;
    CK(cudaMalloc((void **)&d_table, sizeof(int32_t) * n_blocks));
    CK(cudaMemcpy(d_table, table, sizeof(int32_t) * n_blocks, cudaMemcpyHostToDevice));

    /* prefill rows, shared by every layer */
    const size_t row = (size_t)N_KV * HD;
    float *h_pre = (float *)malloc(sizeof(float) * row * L0);
    float *d_pk, *d_pv;
    int32_t *d_seq, *d_pos;
    CK(cudaMalloc((void **)&d_pk, sizeof(float) * row * L0));
    CK(cudaMalloc((void **)&d_pv, sizeof(float) * row * L0));
    for (size_t i = 0; i < row * L0; ++i) h_pre[i] = next_value();
    CK(cudaMemcpy(d_pk, h_pre, sizeof(float) * row * L0, cudaMemcpyHostToDevice));
    for (size_t i = 0; i < row * L0; ++i) h_pre[i] = next_value();
    CK(cudaMemcpy(d_pv, h_pre, sizeof(float) * row * L0, cudaMemcpyHostToDevice));
    free(h_pre);
    int32_t *h_pos = (int32_t *)malloc(sizeof(int32_t) * L0);
    for (int i = 0; i < L0; ++i) h_pos[i] = i;
    CK(cudaMalloc((void **)&d_seq, sizeof(int32_t) * L0));
    CK(cudaMalloc((void **)&d_pos, sizeof(int32_t) * L0));
    CK(cudaMemset(d_seq, 0, sizeof(int32_t) * L0));
    CK(cudaMemcpy(d_pos, h_pos, sizeof(int32_t) * L0, cudaMemcpyHostToDevice));
    free(h_pos);

    cudaStream_t st;
    CK(cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking));

    /* the layers: [layer][0] FP16, [layer][1] int8 */
    layer_t *lay = (layer_t *)calloc((size_t)LAYERS * 2, sizeof(layer_t));
    for (int l = 0; l < LAYERS; ++l)
        for (int f = 0; f < 2; ++f) {
            layer_t *ly = &lay[l * 2 + f];
            make_layer(ly, f == 0 ? KVQ_F16 : KVQ_Q8, n_blocks);
            ly->ws_bytes = kvq_decode_workspace_bytes(&ly->cache, 1, 1, N_Q, cap);
            if (ly->ws_bytes == 0) {
                fprintf(stderr, "kvq_decode_workspace_bytes returned 0\n");
                return 1;
            }
            CK(cudaMalloc(&ly->ws, ly->ws_bytes));
            KV(kvq_append(&ly->cache, d_pk, d_pv, L0, d_seq, d_pos, d_table, 1, n_blocks, st));
        }
    CK(cudaStreamSynchronize(st));

    /* per-step inputs, packed: k, v, q, pos, ctx, each from a 64-word boundary */
    const int o_k = 0, o_v = o_k + (int)row, o_q = o_v + (int)row, o_pos = o_q + N_Q * HD,
              o_ctx = o_pos + 64, words = o_ctx + 64;
    float *h_in;
    CK(cudaMallocHost((void **)&h_in, sizeof(float) * (size_t)words * STEPS_PER_LAYER));
    for (int j = 0; j < STEPS_PER_LAYER; ++j) {
        float *p = h_in + (size_t)j * words;
        for (int i = 0; i < words; ++i) p[i] = 0.f;
        for (int i = 0; i < (int)row; ++i) p[o_k + i] = next_value();
        for (int i = 0; i < (int)row; ++i) p[o_v + i] = next_value();
        for (int i = 0; i < N_Q * HD; ++i) p[o_q + i] = next_value();
        const int32_t pos = L0 + j, ctx = L0 + j + 1;
        memcpy(p + o_pos, &pos, 4);
        memcpy(p + o_ctx, &ctx, 4);
    }
    float *d_in, *d_out, *h_out;
    CK(cudaMalloc((void **)&d_in, sizeof(float) * words));
    CK(cudaMalloc((void **)&d_out, sizeof(float) * 2 * N_Q * HD));
    CK(cudaMallocHost((void **)&h_out, sizeof(float) * 2 * N_Q * HD));
    const int32_t *d_tpos = (const int32_t *)(d_in + o_pos);
    const int32_t *d_ctx = (const int32_t *)(d_in + o_ctx);

    /* host seconds spent in: the copies' enqueue, the library calls, the
       synchronize (over the timed steps) */
    double t0 = 0.0, t_copy = 0.0, t_lib = 0.0, t_sync = 0.0;
    for (int s = 0; s < W + K; ++s) {
        if (s == W) {
            CK(cudaStreamSynchronize(st));
            t0 = now_s();
            t_copy = t_lib = t_sync = 0.0;
        }
        const int i = s < W ? s : s - W;
        const int j = (i / LAYERS) % STEPS_PER_LAYER;
        double ta = now_s();
        CK(cudaMemcpyAsync(d_in, h_in + (size_t)j * words, sizeof(float) * words,
                           cudaMemcpyHostToDevice, st));
        double tb = now_s();
        t_copy += tb - ta;
        for (int f = 0; f < 2; ++f) {
            layer_t *ly = &lay[(i % LAYERS) * 2 + f];
            KV(kvq_append(&ly->cache, d_in + o_k, d_in + o_v, 1, d_seq, d_tpos, d_table, 1, n_blocks,
                          st));
            KV(kvq_decode_attn(&ly->cache, d_in + o_q, 1, 1, N_Q, d_ctx, cap, d_table, n_blocks,
                               sm_scale, d_out + (size_t)f * N_Q * HD, ly->ws, ly->ws_bytes, st));
        }
        ta = now_s();
        t_lib += ta - tb;
        CK(cudaMemcpyAsync(h_out, d_out, sizeof(float) * 2 * N_Q * HD, cudaMemcpyDeviceToHost, st));
        tb = now_s();
        t_copy += tb - ta;
        CK(cudaStreamSynchronize(st));
        t_sync += now_s() - tb;
    }
    const double dt = now_s() - t0;
    for (int i = 0; i < 2 * N_Q * HD; ++i)
        if (!(h_out[i] == h_out[i])) {
            fprintf(stderr, "NaN in the decode output\n");
            return 1;
        }
    printf("ms_per_step %.6f h2d_bytes %d d2h_bytes %d copy_enqueue_us %.3f library_calls_us %.3f "
           "sync_wait_us %.3f\n",
           dt / K * 1e3, (int)(sizeof(float) * words), (int)(sizeof(float) * 2 * N_Q * HD),
           t_copy / K * 1e6, t_lib / K * 1e6, t_sync / K * 1e6);
    return 0;
}
