/*
 * c_abi_roundtrip.c -- the C ABI of libep_gb300.so used from plain C (no
 * Python, no torch): a layout, a bf16 dispatch and a combine of identity
 * experts on a small routing, checked on the host against what the
 * operations' definitions fix, plus the error path of a bad configuration.
 *
 * Checks (N = 96 tokens of 4 logical ranks x 32, 32 experts, top-4,
 * alignment 4, hidden 1024):
 *   - sum of num_unaligned_recv_tokens_per_expert = N*K (no masked ids);
 *   - psum_num_recv_tokens_per_expert is the exclusive prefix sum of the counts
 *     rounded up to the alignment and its last entry equals num_recv_tokens;
 *   - every (t, k) has its own receive row, inside its expert's segment;
 *   - recv_x[dst_slot[t][k]] equals x[t] byte for byte;
 *   - with unit weights, combine of the received rows gives bf16(4 * x[t]),
 *     which is exact (a power-of-two scale of a bf16 value);
 *   - ep_handle_create of an invalid configuration returns EP_EINVAL with a
 *     message and no handle.
 * Prints "ok" and returns 0 on success; any failure prints what failed and
 * returns 1.
 */
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "ep_gb300.h"

#define W 4
#define T 32
#define EPR 8
#define E (W * EPR)
#define K 4
#define A 4
#define H 1024
#define N 96

static int failures = 0;

#define CHECK(cond, ...)                 \
    do {                                 \
        if (!(cond)) {                   \
            printf("FAIL: " __VA_ARGS__); \
            printf("\n");                \
            failures++;                  \
        }                                \
    } while (0)

#define CUDA(call)                                                              \
    do {                                                                        \
        cudaError_t e_ = (call);                                                \
        if (e_ != cudaSuccess) {                                                \
            printf("CUDA error %s at %s\n", cudaGetErrorString(e_), #call);    \
            return 1;                                                           \
        }                                                                       \
    } while (0)

#define EP(call)                                                                \
    do {                                                                        \
        int rc_ = (call);                                                       \
        if (rc_ != EP_OK) {                                                     \
            printf("ep error %d at %s: %s\n", rc_, #call, ep_last_error());     \
            return 1;                                                           \
        }                                                                       \
    } while (0)

/* xorshift64 for the inputs (seeded, no library generator) */
static uint64_t rng = 0x9E3779B97F4A7C15ull;
static uint64_t next_u64(void) {
    rng ^= rng << 13;
    rng ^= rng >> 7;
    rng ^= rng << 17;
    return rng;
}

static int32_t fetch_field(ep_handle_t h, int field, int32_t *dst, int64_t max_elems) {
    void *p = NULL;
    int64_t n = 0;
    if (ep_handle_get(h, field, &p, &n) != EP_OK || n > max_elems) return -1;
    if (n > 0 && cudaMemcpy(dst, p, (size_t)n * 4, cudaMemcpyDeviceToHost) != cudaSuccess) return -1;
    return (int32_t)n;
}

int main(void) {
    /* an invalid configuration is rejected on the host, with a message */
    ep_cfg_t bad = {0, H, T, EPR, K, A, EP_BF16, 1, 0};
    ep_handle_t hb = (ep_handle_t)0x1;
    CHECK(ep_handle_create(&bad, &hb) == EP_EINVAL, "bad cfg not rejected");
    CHECK(hb == NULL, "bad cfg left a handle");
    CHECK(strlen(ep_last_error()) > 0, "no message for the bad cfg");

    ep_cfg_t cfg = {W, H, T, EPR, K, A, EP_BF16, 1, 0};
    const int64_t rcap = ep_recv_capacity(&cfg);
    CHECK(rcap == (int64_t)W * T * K + (int64_t)E * (A - 1), "capacity %lld", (long long)rcap);

    /* inputs: K distinct experts per token, finite normal bf16 values */
    static int64_t topk[N * K];
    static uint16_t x[N * H];
    static float w[N * K];
    for (int t = 0; t < N; ++t)
        for (int k = 0; k < K; ++k) {
            int64_t e;
            int dup;
            do {
                e = (int64_t)(next_u64() % E);
                dup = 0;
                for (int j = 0; j < k; ++j) dup |= topk[t * K + j] == e;
            } while (dup);
            topk[t * K + k] = e;
            w[t * K + k] = 1.0f;
        }
    for (int i = 0; i < N * H; ++i) {
        const uint64_t r = next_u64();
        const uint16_t sign = (uint16_t)((r & 1u) << 15);
        const uint16_t expo = (uint16_t)(120 + (r >> 1) % 15);  /* 2^-7 .. 2^7 */
        const uint16_t mant = (uint16_t)((r >> 8) & 0x7F);
        x[i] = (uint16_t)(sign | (expo << 7) | mant);
    }

    int64_t *d_topk;
    uint16_t *d_x, *d_recv, *d_out;
    float *d_w;
    CUDA(cudaMalloc((void **)&d_topk, sizeof topk));
    CUDA(cudaMalloc((void **)&d_x, sizeof x));
    CUDA(cudaMalloc((void **)&d_w, sizeof w));
    CUDA(cudaMalloc((void **)&d_recv, (size_t)rcap * H * 2));
    CUDA(cudaMalloc((void **)&d_out, sizeof x));
    CUDA(cudaMemcpy(d_topk, topk, sizeof topk, cudaMemcpyHostToDevice));
    CUDA(cudaMemcpy(d_x, x, sizeof x, cudaMemcpyHostToDevice));
    CUDA(cudaMemcpy(d_w, w, sizeof w, cudaMemcpyHostToDevice));
    cudaStream_t s;
    CUDA(cudaStreamCreate(&s));

    ep_handle_t h = NULL;
    EP(ep_handle_create(&cfg, &h));
    EP(ep_layout(h, d_topk, N, (ep_stream_t)s));
    EP(ep_dispatch(h, d_x, d_recv, NULL, (ep_stream_t)s));
    EP(ep_combine(h, d_recv, d_w, d_out, (ep_stream_t)s));
    CUDA(cudaStreamSynchronize(s));
    int32_t dev_err = -1;
    EP(ep_handle_status(h, &dev_err));
    CHECK(dev_err == 0, "device error word %d", dev_err);

    /* layout fields */
    static int32_t cnt[E], psum[E + 1], num_recv[1], slot[N * K];
    CHECK(fetch_field(h, EP_FIELD_NUM_UNALIGNED_PER_EXPERT, cnt, E) == E, "cnt field");
    CHECK(fetch_field(h, EP_FIELD_PSUM_PER_EXPERT, psum, E + 1) == E + 1, "psum field");
    CHECK(fetch_field(h, EP_FIELD_NUM_RECV, num_recv, 1) == 1, "num_recv field");
    CHECK(fetch_field(h, EP_FIELD_DST_SLOT, slot, N * K) == N * K, "dst_slot field");
    int64_t total = 0;
    CHECK(psum[0] == 0, "psum[0] = %d", psum[0]);
    for (int e = 0; e < E; ++e) {
        total += cnt[e];
        CHECK(psum[e + 1] - psum[e] == (cnt[e] + A - 1) / A * A, "segment of expert %d", e);
    }
    CHECK(total == N * K, "sum of counts %lld", (long long)total);
    CHECK(num_recv[0] == psum[E], "num_recv %d vs psum[E] %d", num_recv[0], psum[E]);
    char *seen = calloc((size_t)rcap, 1);
    for (int i = 0; i < N * K; ++i) {
        const int e = (int)topk[i], d = slot[i];
        CHECK(d >= psum[e] && d < psum[e] + cnt[e], "row %d of (%d, %d) outside expert %d", d,
              i / K, i % K, e);
        if (d >= 0 && d < rcap) {
            CHECK(!seen[d], "row %d used twice", d);
            seen[d] = 1;
        }
    }
    free(seen);

    /* dispatched rows and the identity round trip */
    uint16_t *recv = malloc((size_t)rcap * H * 2), *out = malloc(sizeof x);
    CUDA(cudaMemcpy(recv, d_recv, (size_t)rcap * H * 2, cudaMemcpyDeviceToHost));
    CUDA(cudaMemcpy(out, d_out, sizeof x, cudaMemcpyDeviceToHost));
    int bad_rows = 0, bad_out = 0;
    for (int i = 0; i < N * K; ++i) {
        const int d = slot[i];
        if (d >= 0 && d < rcap)
            bad_rows += memcmp(recv + (size_t)d * H, x + (size_t)(i / K) * H, H * 2) != 0;
    }
    for (int i = 0; i < N * H; ++i)
        bad_out += out[i] != (uint16_t)(x[i] + (2u << 7));  /* 4 * x: exponent + 2 */
    CHECK(bad_rows == 0, "%d received rows differ from their token", bad_rows);
    CHECK(bad_out == 0, "%d combined values differ from 4 * x", bad_out);
    free(recv);
    free(out);

    char name[128];
    EP(ep_handle_variant(h, 1, name, (int32_t)sizeof name));
    CHECK(strcmp(name, "ep_dispatch_bf16_h1024_k4") == 0, "dispatch variant %s", name);
    ep_handle_free(h);
    cudaFree(d_topk);
    cudaFree(d_x);
    cudaFree(d_w);
    cudaFree(d_recv);
    cudaFree(d_out);
    cudaStreamDestroy(s);
    if (failures) return 1;
    printf("ok\n");
    return 0;
}
