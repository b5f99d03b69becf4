/*
 * ep_oracle.c -- plain, slow, single-threaded CPU oracle for the MoE
 * expert-parallel layout / dispatch / combine path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, includes
 * or calls this file; only the test-suite, the smoke check and the benchmark's
 * CPU-baseline leg load it.  It shares no code, header, table or constant
 * generator with the CUDA implementation.
 *
 * Sources followed (cited by page title and section):
 *   [DEEPEP-ARCH]  "DeepEP overall architecture analysis" (backyes.github.io,
 *                  deepepv2 07_deep_ep_00_overall_architecture): the EPHandle
 *                  class listing (expert_alignment, psum_num_recv_tokens_per_*,
 *                  num_unaligned_recv_tokens_per_expert, recv_src_metadata
 *                  [num_recv_tokens, topk+2], dst_buffer_slot_idx) and the
 *                  "Dispatch data flow" / "Combine data flow" figures
 *                  (notify warps count per rank / expert; dispatch copies token
 *                  data + scale factors; combine reduces weighted by
 *                  topk_weights).
 *   [MORI-V2]      "MORI JIT v2" (rocm.github.io/mori, MORI_JIT_V2_DESIGN):
 *                  §3.2 the EpCfg field list (worldSize, hiddenDim,
 *                  maxTokPerRank, numExpertPerRank, numExpertPerToken,
 *                  useWeights), §3.5 validity rules, §3.7 "dtype is a transport
 *                  property" (dispatch moves bytes, combine reduces).
 *   [MORI-ARCH]    "MORI JIT Architecture" (rocm.github.io/mori,
 *                  MORI_JIT_ARCHITECTURE), the dtype table: torch
 *                  float8_e4m3fn is the OCP e4m3 ("fp8_ocp") format.
 *
 * Readings of points the pages leave open (each is also listed in the design
 * notes of the repository):
 *   - rows of one expert are ordered by the flat index t*K+k (a stable
 *     counting sort by expert id);
 *   - prefix sums are exclusive with E+1 (resp. W+1) entries, the last one
 *     being the number of receive rows R;
 *   - every expert segment is padded up to a multiple of expert_alignment A;
 *   - recv_src_metadata row = {t / T, t mod T, dst_slot[t][0..K-1]}; rows that
 *     receive no token (padding, and everything from R to the capacity) are -1;
 *   - topk_idx == -1 is a masked entry (no slot, slot value -1); any other
 *     value outside [0, E) is skipped and raises error bit 1;
 *   - FP8: s = amax/448 (fp32 division), q = e4m3(x/s) with round-to-nearest-
 *     even and saturation to +-448, one scale per (row, 128-channel group);
 *     a group with amax == 0 gets s = 0 and all-zero bytes;
 *   - combine: acc = +0.0f, then acc = fmaf(w[t][k], y[slot], acc) for
 *     k = 0..K-1 ascending (acc = acc + y without weights), masked k skipped,
 *     then one round-to-nearest-even to bf16.
 *
 * Build: gcc -O2 -std=c99 -ffp-contract=off (no fast-math): every float
 * operation below is a single IEEE-754 binary32 operation.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <math.h>

/* ------------------------------------------------------------------ bf16 */

/* bf16 -> fp32 is exact: the bf16 bits are the high half of the fp32 bits. */
float oracle_bf16_to_f32(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* fp32 -> bf16, round to nearest, ties to even; NaN -> quiet NaN 0x7FC0
 * (sign kept). Written from the definition: keep the high 16 bits, add one
 * unit in the last kept place when the dropped half is above 0x8000, or equal
 * to 0x8000 with an odd kept part. */
uint16_t oracle_f32_to_bf16(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if (isnan(f))
        return (uint16_t)(((u >> 16) & 0x8000u) | 0x7FC0u);
    uint32_t hi = u >> 16;
    uint32_t lo = u & 0xFFFFu;
    if (lo > 0x8000u || (lo == 0x8000u && (hi & 1u)))
        hi += 1u; /* a carry into the exponent is the correct rounding, up to inf */
    return (uint16_t)hi;
}

/* ------------------------------------------------------------------ e4m3 */

/* OCP FP8 e4m3 ("fn"): 1 sign bit, 4 exponent bits with bias 7, 3 mantissa
 * bits; no infinities; 0x7F / 0xFF are NaN; largest finite value 448. */
double oracle_e4m3_decode(uint8_t c)
{
    int sign = (c >> 7) & 1;
    int e = (c >> 3) & 0xF;
    int m = c & 0x7;
    double v;
    if (e == 0xF && m == 0x7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m, -9);               /* subnormal: m/8 * 2^(1-7) */
    else
        v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return sign ? -v : v;
}

/* Sorted table of the 127 finite non-negative e4m3 values (codes 0x00..0x7E,
 * which are monotone in value). */
static double e4m3_pos_table[127];
static int e4m3_table_ready = 0;

static void e4m3_init_table(void)
{
    if (e4m3_table_ready)
        return;
    for (int c = 0; c < 127; ++c)
        e4m3_pos_table[c] = oracle_e4m3_decode((uint8_t)c);
    e4m3_table_ready = 1;
}

/* fp32 -> e4m3 with round-to-nearest-even and saturation to +-448 ("satfinite").
 * Plain definition: pick the nearest of the finite magnitudes; on an exact tie
 * pick the one whose code is even (even mantissa); magnitudes above 448,
 * including infinity, give 448; NaN gives 0x7F. */
uint8_t oracle_e4m3_encode(float v)
{
    e4m3_init_table();
    if (isnan(v))
        return 0x7F;
    uint8_t sign = signbit(v) ? 0x80 : 0x00;
    double a = fabs((double)v);
    if (a >= 448.0)
        return (uint8_t)(sign | 0x7E);
    /* largest code c with table[c] <= a (binary search, table[0] = 0 <= a) */
    int lo = 0, hi = 126;
    while (lo < hi) {
        int mid = (lo + hi + 1) / 2;
        if (e4m3_pos_table[mid] <= a)
            lo = mid;
        else
            hi = mid - 1;
    }
    int c = lo;
    if (e4m3_pos_table[c] != a) {               /* c < 126 here since a < 448 */
        double dlo = a - e4m3_pos_table[c];     /* exact in binary64 */
        double dhi = e4m3_pos_table[c + 1] - a;
        if (dhi < dlo || (dhi == dlo && ((c + 1) % 2 == 0)))
            c = c + 1;
    }
    return (uint8_t)(sign | (uint8_t)c);
}

/* Quantise one token row of H bf16 values (H a multiple of 128) into e4m3
 * bytes q[H] and one fp32 scale per 128-channel group, scales[H/128]. */
void oracle_quant_fp8_row(int H, const uint16_t *x, uint8_t *q, float *scales)
{
    for (int g = 0; g < H / 128; ++g) {
        float amax = 0.0f;
        for (int j = 0; j < 128; ++j) {
            float a = fabsf(oracle_bf16_to_f32(x[g * 128 + j]));
            if (a > amax)
                amax = a;
        }
        if (amax == 0.0f) {
            scales[g] = 0.0f;
            for (int j = 0; j < 128; ++j)
                q[g * 128 + j] = 0x00;
            continue;
        }
        float s = amax / 448.0f;
        scales[g] = s;
        for (int j = 0; j < 128; ++j) {
            float xf = oracle_bf16_to_f32(x[g * 128 + j]);
            float r = xf / s;
            q[g * 128 + j] = oracle_e4m3_encode(r);
        }
    }
}

/* ---------------------------------------------------------------- layout */

/* Number of rows the receive buffer must hold for any routing of up to
 * max_tokens tokens: every (t,k) gets a row, and each of the E expert
 * segments can add at most A-1 padding rows. */
int64_t oracle_recv_capacity(int max_tokens, int K, int E, int A)
{
    return (int64_t)max_tokens * K + (int64_t)E * (A - 1);
}

/* Layout of N tokens with top-K expert ids topk_idx[N][K] (int64, row-major)
 * over E = W*Epr experts; rank r owns experts [r*Epr, (r+1)*Epr).
 * Outputs (caller-allocated):
 *   cnt[E]            number of (t,k) entries routed to each expert
 *                     (num_unaligned_recv_tokens_per_expert)
 *   tok_per_rank[W]   number of tokens with at least one expert on rank r
 *   psum_expert[E+1]  exclusive prefix sum of the aligned counts
 *   psum_rank[W+1]    psum_expert at each rank's first expert
 *   dst_slot[N][K]    receive row of each (t,k), -1 when skipped
 *   meta[rcap][K+2]   recv_src_metadata, -1 rows where nothing is received
 *   num_recv[1]       R = psum_expert[E]
 *   err[1]            bit 0 set when an id outside [-1, E) was seen
 * Returns 0, or -1 when R would exceed rcap (cannot happen when rcap is
 * oracle_recv_capacity(N or more, ...)). */
int oracle_layout(int W, int T, int Epr, int K, int A,
                  const int64_t *topk_idx, int N,
                  int32_t *cnt, int32_t *tok_per_rank,
                  int32_t *psum_expert, int32_t *psum_rank,
                  int32_t *dst_slot, int32_t *meta, int64_t rcap,
                  int32_t *num_recv, int32_t *err)
{
    const int E = W * Epr;
    *err = 0;
    for (int e = 0; e < E; ++e)
        cnt[e] = 0;
    for (int r = 0; r < W; ++r)
        tok_per_rank[r] = 0;

    /* histogram per expert and, per token, the set of ranks it touches */
    char *touched = (char *)calloc((size_t)(W > 0 ? W : 1), 1);
    for (int t = 0; t < N; ++t) {
        memset(touched, 0, (size_t)W);
        for (int k = 0; k < K; ++k) {
            int64_t e = topk_idx[(int64_t)t * K + k];
            if (e == -1)
                continue;
            if (e < -1 || e >= E) {
                *err |= 1;
                continue;
            }
            cnt[e] += 1;
            touched[e / Epr] = 1;
        }
        for (int r = 0; r < W; ++r)
            tok_per_rank[r] += touched[r];
    }
    free(touched);

    /* exclusive prefix sums of the counts padded to a multiple of A */
    psum_expert[0] = 0;
    for (int e = 0; e < E; ++e) {
        int32_t padded = ((cnt[e] + A - 1) / A) * A;
        psum_expert[e + 1] = psum_expert[e] + padded;
    }
    for (int r = 0; r <= W; ++r)
        psum_rank[r] = psum_expert[r * Epr];
    *num_recv = psum_expert[E];
    if ((int64_t)psum_expert[E] > rcap)
        return -1;

    /* slots: a running cursor per expert, walking (t,k) in row-major order */
    int32_t *cursor = (int32_t *)malloc(sizeof(int32_t) * (size_t)(E > 0 ? E : 1));
    for (int e = 0; e < E; ++e)
        cursor[e] = psum_expert[e];
    for (int t = 0; t < N; ++t) {
        for (int k = 0; k < K; ++k) {
            int64_t e = topk_idx[(int64_t)t * K + k];
            int64_t i = (int64_t)t * K + k;
            if (e < 0 || e >= E) {
                dst_slot[i] = -1;
                continue;
            }
            dst_slot[i] = cursor[e];
            cursor[e] += 1;
        }
    }
    free(cursor);

    /* recv_src_metadata: -1 everywhere, then one row per received (t,k) */
    for (int64_t i = 0; i < rcap * (K + 2); ++i)
        meta[i] = -1;
    for (int t = 0; t < N; ++t) {
        for (int k = 0; k < K; ++k) {
            int32_t s = dst_slot[(int64_t)t * K + k];
            if (s < 0)
                continue;
            int32_t *row = meta + (int64_t)s * (K + 2);
            row[0] = t / T;
            row[1] = t % T;
            for (int j = 0; j < K; ++j)
                row[2 + j] = dst_slot[(int64_t)t * K + j];
        }
    }
    return 0;
}

/* -------------------------------------------------------------- dispatch */

/* recv_x[dst_slot[t][k]][:] = x[t][:] for every received (t,k); bf16 rows of
 * H elements are moved as bytes ("dtype is a transport property"). Rows no
 * (t,k) maps to are left untouched. */
void oracle_dispatch_bf16(int N, int H, int K, const uint16_t *x,
                          const int32_t *dst_slot, uint16_t *recv_x)
{
    for (int t = 0; t < N; ++t)
        for (int k = 0; k < K; ++k) {
            int32_t s = dst_slot[(int64_t)t * K + k];
            if (s < 0)
                continue;
            memcpy(recv_x + (int64_t)s * H, x + (int64_t)t * H, sizeof(uint16_t) * (size_t)H);
        }
}

/* FP8 dispatch: each token row is quantised once (oracle_quant_fp8_row) and
 * the same bytes and scales are written to each of its destination rows:
 * recv_x[s][H] e4m3, recv_scales[s][H/128] fp32. */
void oracle_dispatch_fp8(int N, int H, int K, const uint16_t *x,
                         const int32_t *dst_slot, uint8_t *recv_x, float *recv_scales)
{
    const int G = H / 128;
    uint8_t *q = (uint8_t *)malloc((size_t)H);
    float *sc = (float *)malloc(sizeof(float) * (size_t)G);
    for (int t = 0; t < N; ++t) {
        oracle_quant_fp8_row(H, x + (int64_t)t * H, q, sc);
        for (int k = 0; k < K; ++k) {
            int32_t s = dst_slot[(int64_t)t * K + k];
            if (s < 0)
                continue;
            memcpy(recv_x + (int64_t)s * H, q, (size_t)H);
            memcpy(recv_scales + (int64_t)s * G, sc, sizeof(float) * (size_t)G);
        }
    }
    free(q);
    free(sc);
}

/* --------------------------------------------------------------- combine */

/* out[t][c] = bf16_rn( fold over k = 0..K-1 ascending of
 *                      acc = fmaf(w[t][k], y[dst_slot[t][k]][c], acc) ), acc = +0.0f.
 * w == NULL means no weights: acc = acc + y. Masked (t,k) are skipped. */
void oracle_combine(int N, int H, int K, const uint16_t *y, const int32_t *dst_slot,
                    const float *w, uint16_t *out)
{
    for (int t = 0; t < N; ++t) {
        for (int c = 0; c < H; ++c) {
            float acc = 0.0f;
            for (int k = 0; k < K; ++k) {
                int32_t s = dst_slot[(int64_t)t * K + k];
                if (s < 0)
                    continue;
                float v = oracle_bf16_to_f32(y[(int64_t)s * H + c]);
                if (w)
                    acc = fmaf(w[(int64_t)t * K + k], v, acc);
                else
                    acc = acc + v;
            }
            out[(int64_t)t * H + c] = oracle_f32_to_bf16(acc);
        }
    }
}

/* ------------------------------------------------------- array helpers */

/* Element-wise forms of the scalar routines above, for the tests. */
void oracle_e4m3_encode_array(int64_t n, const float *v, uint8_t *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_e4m3_encode(v[i]);
}

void oracle_e4m3_decode_array(int64_t n, const uint8_t *c, double *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_e4m3_decode(c[i]);
}

void oracle_f32_to_bf16_array(int64_t n, const float *v, uint16_t *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_f32_to_bf16(v[i]);
}

/* ------------------------------------------------- transport and routing */

/* Dispatch of an opaque payload: recv[dst_slot[t][k]] = x[t] as row_bytes raw
 * bytes.  This is how the pages treat the narrow and wide transports ("MORI
 * JIT v2" §3.7: Fp32, Fp8 and Fp4x2 payloads are moved, never computed on;
 * an Fp4x2 row of H channels is H/2 bytes). */
void oracle_dispatch_bytes(int N, int64_t row_bytes, int K, const uint8_t *x,
                           const int32_t *dst_slot, uint8_t *recv)
{
    for (int t = 0; t < N; ++t)
        for (int k = 0; k < K; ++k) {
            int32_t s = dst_slot[(int64_t)t * K + k];
            if (s < 0)
                continue;
            memcpy(recv + (int64_t)s * row_bytes, x + (int64_t)t * row_bytes, (size_t)row_bytes);
        }
}

/* Routing that travels with each received row (the dispatch copy epilogue of
 * "DeepEP overall architecture analysis" fills recv_topk_idx and
 * recv_topk_weights): the row of (t, k) carries the expert it was sent to and
 * the token's weight for that expert.  Rows nothing maps to are untouched. */
void oracle_forward_routing(int N, int K, const int64_t *topk_idx, const float *w,
                            const int32_t *dst_slot, float *recv_w, int32_t *recv_idx)
{
    for (int t = 0; t < N; ++t)
        for (int k = 0; k < K; ++k) {
            int64_t i = (int64_t)t * K + k;
            int32_t s = dst_slot[i];
            if (s < 0)
                continue;
            if (recv_w)
                recv_w[s] = w[i];
            if (recv_idx)
                recv_idx[s] = (int32_t)topk_idx[i];
        }
}

/* Combine with an optional bias and an fp32 or bf16 output ("Combine data
 * flow": reduce weighted by topk_weights, "+ bias", write back).  The fold is
 * oracle_combine's; the bias (bf16 [N][H], may be NULL) is then added with one
 * fp32 addition; the sum is stored as fp32 (out_f32) or rounded once to bf16
 * (out_bf16).  Exactly one of out_bf16 / out_f32 is non-NULL. */
void oracle_combine_ex(int N, int H, int K, const uint16_t *y, const int32_t *dst_slot,
                       const float *w, const uint16_t *bias, uint16_t *out_bf16, float *out_f32)
{
    for (int t = 0; t < N; ++t) {
        for (int c = 0; c < H; ++c) {
            float acc = 0.0f;
            for (int k = 0; k < K; ++k) {
                int32_t s = dst_slot[(int64_t)t * K + k];
                if (s < 0)
                    continue;
                float v = oracle_bf16_to_f32(y[(int64_t)s * H + c]);
                if (w)
                    acc = fmaf(w[(int64_t)t * K + k], v, acc);
                else
                    acc = acc + v;
            }
            if (bias)
                acc = acc + oracle_bf16_to_f32(bias[(int64_t)t * H + c]);
            if (out_f32)
                out_f32[(int64_t)t * H + c] = acc;
            else
                out_bf16[(int64_t)t * H + c] = oracle_f32_to_bf16(acc);
        }
    }
}

/* ------------------------------------------------------ non-expand layout */

/* Receive rows for the non-expand layout (EPHandle do_expand = false in
 * "DeepEP overall architecture analysis"): every token is received once by
 * each rank that owns one of its experts, so at most min(K, W) rows per token.
 * Reading of the pages, which name the mode only: one row per (token,
 * destination rank); no expert alignment applies (the rows are not grouped by
 * expert). */
int64_t oracle_recv_capacity_nonexpand(int max_tokens, int K, int W)
{
    return (int64_t)max_tokens * (K < W ? K : W);
}

/* Non-expand layout.  Same arguments and outputs as oracle_layout, with these
 * differences (the expert counts cnt / psum_expert are computed as there: they
 * are what the receiving ranks' expert computation needs):
 *   psum_rank[W+1]    exclusive prefix sum of tok_per_rank (no alignment)
 *   num_recv[1]       R = psum_rank[W], the number of (token, rank) rows
 *   rows              rank r owns rows [psum_rank[r], psum_rank[r+1]); its
 *                     tokens appear once each, in ascending token order
 *   dst_slot[N][K]    the row that carries (t,k): the row of t on the rank of
 *                     expert topk_idx[t][k]; -1 when skipped.  Entries of one
 *                     token whose experts share a rank share the row.
 *   send_slot[N][K]   the distinct rows of t in ascending order (= ascending
 *                     rank), then -1: the rows dispatch writes and combine reads
 *   meta[rcap][K+2]   {t / T, t mod T, dst_slot[t][0..K-1]} per row, -1 rows
 *                     where nothing is received
 * Returns 0, or -1 when R would exceed rcap. */
int oracle_layout_nonexpand(int W, int T, int Epr, int K, int A,
                            const int64_t *topk_idx, int N,
                            int32_t *cnt, int32_t *tok_per_rank,
                            int32_t *psum_expert, int32_t *psum_rank,
                            int32_t *dst_slot, int32_t *send_slot, int32_t *meta, int64_t rcap,
                            int32_t *num_recv, int32_t *err)
{
    const int E = W * Epr;
    *err = 0;
    for (int e = 0; e < E; ++e)
        cnt[e] = 0;
    for (int r = 0; r < W; ++r)
        tok_per_rank[r] = 0;

    /* per token: which ranks it touches; per expert: how many entries */
    char *touched = (char *)calloc((size_t)N * (size_t)(W > 0 ? W : 1) + 1, 1);
    for (int t = 0; t < N; ++t) {
        for (int k = 0; k < K; ++k) {
            int64_t e = topk_idx[(int64_t)t * K + k];
            if (e == -1)
                continue;
            if (e < -1 || e >= E) {
                *err |= 1;
                continue;
            }
            cnt[e] += 1;
            touched[(size_t)t * W + (size_t)(e / Epr)] = 1;
        }
        for (int r = 0; r < W; ++r)
            tok_per_rank[r] += touched[(size_t)t * W + r];
    }

    psum_expert[0] = 0;
    for (int e = 0; e < E; ++e) {
        int32_t padded = ((cnt[e] + A - 1) / A) * A;
        psum_expert[e + 1] = psum_expert[e] + padded;
    }
    psum_rank[0] = 0;
    for (int r = 0; r < W; ++r)
        psum_rank[r + 1] = psum_rank[r] + tok_per_rank[r];
    *num_recv = psum_rank[W];
    if ((int64_t)psum_rank[W] > rcap) {
        free(touched);
        return -1;
    }

    /* rows: a running cursor per rank, walking the tokens in order and, for
     * each token, its ranks in ascending order */
    int32_t *cursor = (int32_t *)malloc(sizeof(int32_t) * (size_t)(W > 0 ? W : 1));
    int32_t *row_of = (int32_t *)malloc(sizeof(int32_t) * (size_t)(W > 0 ? W : 1));
    for (int r = 0; r < W; ++r)
        cursor[r] = psum_rank[r];
    for (int t = 0; t < N; ++t) {
        int j = 0;
        for (int r = 0; r < W; ++r) {
            row_of[r] = -1;
            if (touched[(size_t)t * W + r]) {
                row_of[r] = cursor[r];
                cursor[r] += 1;
                send_slot[(int64_t)t * K + j] = row_of[r];
                j += 1;
            }
        }
        for (; j < K; ++j)
            send_slot[(int64_t)t * K + j] = -1;
        for (int k = 0; k < K; ++k) {
            int64_t e = topk_idx[(int64_t)t * K + k];
            dst_slot[(int64_t)t * K + k] = (e < 0 || e >= E) ? -1 : row_of[e / Epr];
        }
    }
    free(row_of);
    free(cursor);
    free(touched);

    for (int64_t i = 0; i < rcap * (K + 2); ++i)
        meta[i] = -1;
    for (int t = 0; t < N; ++t) {
        for (int j = 0; j < K; ++j) {
            int32_t s = send_slot[(int64_t)t * K + j];
            if (s < 0)
                break;
            int32_t *row = meta + (int64_t)s * (K + 2);
            row[0] = t / T;
            row[1] = t % T;
            for (int k = 0; k < K; ++k)
                row[2 + k] = dst_slot[(int64_t)t * K + k];
        }
    }
    return 0;
}

/* Routing forwarded with the non-expand rows (the copy epilogue's
 * recv_topk_idx / recv_topk_weights, one K-wide row per received row): for each
 * row s of token t and each k,
 *   recv_idx[s][k] = topk_idx[t][k] and recv_w[s][k] = w[t][k]  when (t,k) is carried by s,
 *   recv_idx[s][k] = -1             and recv_w[s][k] = 0.0f     otherwise.
 * Rows that receive nothing are untouched; either output may be NULL. */
void oracle_forward_routing_nonexpand(int N, int K, const int64_t *topk_idx, const float *w,
                                      const int32_t *dst_slot, const int32_t *send_slot,
                                      float *recv_w, int32_t *recv_idx)
{
    for (int t = 0; t < N; ++t)
        for (int j = 0; j < K; ++j) {
            int32_t s = send_slot[(int64_t)t * K + j];
            if (s < 0)
                break;
            for (int k = 0; k < K; ++k) {
                int64_t i = (int64_t)t * K + k;
                int mine = dst_slot[i] == s;
                if (recv_w)
                    recv_w[(int64_t)s * K + k] = mine ? w[i] : 0.0f;
                if (recv_idx)
                    recv_idx[(int64_t)s * K + k] = mine ? (int32_t)topk_idx[i] : -1;
            }
        }
}
