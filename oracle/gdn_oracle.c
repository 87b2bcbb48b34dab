/*
 * gdn_oracle.c -- plain, slow, fp64 CPU reference of paged Gated Delta-Rule
 * (GDN) prefill and decode.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path loads this library:
 * only the tests, the smoke check and the benchmark's CPU-baseline leg do.  It
 * shares no source, header, table or helper with the CUDA library.
 *
 * What it follows ("flashinfer.gdn_paged", docs.flashinfer.ai/api/gdn_paged.html):
 *   - intro: one caller-owned pool state_pool[num_pages, H, V, K]; page j of a
 *     sequence holds the recurrent state after the last token of that page.
 *   - "Page table": sequence b owns page_indices[page_indptr[b]:page_indptr[b+1]]
 *     and has (num_pages_b - 1) * page_size + last_page_len[b] tokens after the
 *     call; its new tokens are the last ones, the ones before are its prefix.
 *   - prefill bullets: read the page holding the last prefix token (zero state
 *     for an empty prefix); store the state at every page boundary the new
 *     tokens cross and the final state to the last page; never write a page
 *     that ends at or before the prefix.  Zero-length sequences write nothing.
 *   - decode paragraph: one token; lpl == 1 reads the previous page and writes
 *     the new one, otherwise the last page is updated in place.
 *   - "Slot arguments of chunk_gated_delta_rule": separate read / final / and
 *     checkpoint rows, -1 = zero state (read) or skip (write); checkpoints at
 *     absolute positions where (prefix_lens[i] + n) % N == 0.
 *
 * The pages name the method but print no formula for it.  The formula used is
 * the standard gated delta rule on a V x K state S:
 *     S_t = exp(g_t) S_{t-1} + beta_t (v_t - exp(g_t) S_{t-1} k_t) k_t^T
 *     o_t = scale * S_t q_t
 * computed token by token in fp64, which is the plain definition: chunking is
 * only a faster route to the same value.
 *
 * Slots are derived by walking token positions with counters (no division),
 * a different route from the closed forms the CUDA library uses.
 *
 * Conventions: q, k are [T, H, K] and v is [T, H, V], as raw bf16 bits
 * (uint16) converted exactly to fp64; g, beta are [T, H] fp32; the output o is
 * [T, H, V] fp64; every pool row is a dense [H, V, K] block at row * row_stride
 * elements, of fp32 or (the _st entry points with state_bf16 = 1) of bf16 bits.
 * Stores round the fp64 state to the nearest fp32 or bf16 value, ties to even;
 * loads convert exactly.
 */
#include <fenv.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

static double bf16_bits_to_double(uint16_t h)
{
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* The bf16 value nearest to x, ties to even, as bits: 8 significant bits, the
 * exponent range of fp32 (quantum 2^-133 below 2^-126), +-inf past the largest
 * finite value.  Rounds x itself, not an fp32 copy of it. */
uint16_t oracle_double_to_bf16(double x)
{
    if (isnan(x)) return (uint16_t)0x7FC0;
    double r = x;
    if (x != 0.0 && !isinf(x)) {
        int e;
        frexp(fabs(x), &e); /* |x| = m 2^e, m in [0.5, 1) */
        int qexp = e - 8;   /* the quantum of an 8-bit significand */
        if (qexp < -133) qexp = -133;
        r = ldexp(nearbyint(ldexp(x, -qexp)), qexp); /* default mode: nearest, ties to even */
    }
    float f = (float)r; /* exact: r has at most 8 significant bits (or overflows to inf) */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(u >> 16);
}

/* ------------------------------------------------------------------------- */
/* Page walking ("Page table" section).                                      */
/* ------------------------------------------------------------------------- */

/* Walk the positions 0 .. upto-1 of one sequence, filling pages of page_size
 * tokens in list order.  Returns the slot (0-based index in the sequence's page
 * list) of the page holding position upto-1, and, through *pages_closed, the
 * number of pages that became full at or before that position. */
static int32_t walk_pages(int64_t upto, int32_t page_size, int64_t *pages_closed)
{
    int32_t slot = 0;
    int64_t fill = 0, closed = 0;
    for (int64_t p = 0; p < upto; ++p) {
        if (fill == page_size) { /* previous page is full: open the next one */
            ++slot;
            fill = 0;
        }
        ++fill;
        if (fill == page_size) ++closed;
    }
    if (pages_closed) *pages_closed = closed;
    return slot;
}

/* Prefill rows of every sequence (the rows that the paged prefill call derives
 * from a page table; "Page table" section and the prefill bullets):
 *   state_indices[b]        page holding the last prefix token, -1 if no prefix
 *   output_state_indices[b] last page, -1 for a zero-length sequence
 *   checkpoint_cu_starts[b] index into page_indices of the first page that ends
 *                           after the prefix (page_indptr[b] + number of pages
 *                           that are full at or before the prefix end)
 *   prefix_lens[b]          tokens before the new ones
 * Returns 0, or -1 if a sequence owns no page, has a last page holding no
 * token or more than page_size tokens, or has more new tokens than tokens. */
int oracle_prefill_slots(int32_t num_seqs, const int32_t *cu_seqlens,
                         const int32_t *page_indptr, const int32_t *page_indices,
                         const int32_t *last_page_len, int32_t page_size,
                         int32_t *state_indices, int32_t *output_state_indices,
                         int32_t *checkpoint_cu_starts, int32_t *prefix_lens)
{
    for (int32_t b = 0; b < num_seqs; ++b) {
        int64_t npages = (int64_t)page_indptr[b + 1] - page_indptr[b];
        if (npages < 1) return -1;
        /* a last page holds at least one token and at most a page of them */
        if (last_page_len[b] < 1 || last_page_len[b] > page_size) return -1;
        int64_t new_tokens = (int64_t)cu_seqlens[b + 1] - cu_seqlens[b];
        int64_t total = (npages - 1) * page_size + last_page_len[b];
        int64_t prefix = total - new_tokens;
        if (prefix < 0 || new_tokens < 0) return -1;
        const int32_t *pages = page_indices + page_indptr[b];

        int64_t closed_before = 0;
        if (prefix > 0) {
            int32_t slot = walk_pages(prefix, page_size, &closed_before);
            state_indices[b] = pages[slot];
        } else {
            state_indices[b] = -1;
        }
        if (new_tokens > 0) {
            int32_t slot = walk_pages(total, page_size, NULL);
            output_state_indices[b] = pages[slot];
        } else {
            output_state_indices[b] = -1;
        }
        checkpoint_cu_starts[b] = (int32_t)(page_indptr[b] + closed_before);
        prefix_lens[b] = (int32_t)prefix;
    }
    return 0;
}

/* Decode rows (decode paragraph): the decoded token is the last of the
 * sequence's tokens; the state before it is the one after the token before
 * it, held by the page of that token (-1 = zero state when there is no such
 * token, which is outside the call's contract).  The new state goes to the
 * page holding the decoded token. */
int oracle_decode_slots(int32_t batch, const int32_t *page_indptr,
                        const int32_t *page_indices, const int32_t *last_page_len,
                        int32_t page_size, int32_t *initial_state_indices,
                        int32_t *output_state_indices)
{
    for (int32_t b = 0; b < batch; ++b) {
        int64_t npages = (int64_t)page_indptr[b + 1] - page_indptr[b];
        if (npages < 1) return -1;
        if (last_page_len[b] < 1 || last_page_len[b] > page_size) return -1;
        int64_t total = (npages - 1) * page_size + last_page_len[b];
        const int32_t *pages = page_indices + page_indptr[b];
        initial_state_indices[b] = total >= 2 ? pages[walk_pages(total - 1, page_size, NULL)] : -1;
        output_state_indices[b] = pages[walk_pages(total, page_size, NULL)];
    }
    return 0;
}

/* ------------------------------------------------------------------------- */
/* The recurrence.                                                           */
/* ------------------------------------------------------------------------- */

/* One token on the V x K state S (row-major, S[i*K + j]):
 *   e = exp(g);  u = S k;  S <- e S + beta (v - e u) k^T;  o = scale S q. */
static void gdn_token(double *S, int32_t K, int32_t V, const double *q, const double *k,
                      const double *v, double g, double beta, double scale, double *o,
                      double *u)
{
    double e = exp(g);
    for (int32_t i = 0; i < V; ++i) {
        double acc = 0.0;
        for (int32_t j = 0; j < K; ++j) acc += S[(int64_t)i * K + j] * k[j];
        u[i] = acc;
    }
    for (int32_t i = 0; i < V; ++i) {
        double d = beta * (v[i] - e * u[i]);
        for (int32_t j = 0; j < K; ++j)
            S[(int64_t)i * K + j] = e * S[(int64_t)i * K + j] + d * k[j];
    }
    for (int32_t i = 0; i < V; ++i) {
        double acc = 0.0;
        for (int32_t j = 0; j < K; ++j) acc += S[(int64_t)i * K + j] * q[j];
        o[i] = scale * acc;
    }
}

static void load_state(double *S, const void *pool, int bf16, int64_t row, int64_t row_stride,
                       int32_t h, int32_t K, int32_t V)
{
    int64_t off = row * row_stride + (int64_t)h * V * K;
    if (bf16) {
        const uint16_t *src = (const uint16_t *)pool + off;
        for (int64_t i = 0; i < (int64_t)V * K; ++i) S[i] = bf16_bits_to_double(src[i]);
    } else {
        const float *src = (const float *)pool + off;
        for (int64_t i = 0; i < (int64_t)V * K; ++i) S[i] = (double)src[i];
    }
}

static void store_state(const double *S, void *pool, int bf16, int64_t row, int64_t row_stride,
                        int32_t h, int32_t K, int32_t V)
{
    int64_t off = row * row_stride + (int64_t)h * V * K;
    if (bf16) {
        uint16_t *dst = (uint16_t *)pool + off;
        for (int64_t i = 0; i < (int64_t)V * K; ++i) dst[i] = oracle_double_to_bf16(S[i]);
    } else {
        float *dst = (float *)pool + off;
        for (int64_t i = 0; i < (int64_t)V * K; ++i) dst[i] = (float)S[i];
    }
}

static void mark(uint8_t *flags, int64_t row)
{
    if (!flags) return;
#pragma omp atomic write
    flags[row] = 1;
}

/* General prefill with slot arguments ("Slot arguments of
 * chunk_gated_delta_rule").  One chain per (sequence b, head h):
 *   - start from row state_indices[b] of initial_state, or from literal zeros
 *     if there is no read row or it is -1 (a pool row is never scaled by 0);
 *   - run the new tokens cu_seqlens[b] .. cu_seqlens[b+1]-1 in order;
 *   - after new token n (1-based) with (prefix_lens[b] + n) % N == 0, store the
 *     state to row checkpoint_state_indices[checkpoint_cu_starts[b] + j] of
 *     state_checkpoints, j counting this call's checkpoints of b from 0, unless
 *     that row is -1;
 *   - after the last token store the state to row output_state_indices[b] of
 *     output_state unless it is -1;
 *   - a zero-length sequence reads and writes nothing.
 * Checkpoint arguments may be NULL (no checkpoints); prefix_lens NULL means 0.
 * chain_mask (optional, [num_seqs * H]) selects the chains to compute; output
 * rows of skipped chains are left as they are.  out_written / ckpt_written
 * (optional) get a 1 for every row stored.  state_bf16 selects bf16 pools
 * (row_stride then counts bf16 elements). */
int oracle_chunk_gdn_st(int32_t num_seqs, const int32_t *cu_seqlens, int32_t H, int32_t K,
                        int32_t V, double scale, const uint16_t *q, const uint16_t *k,
                        const uint16_t *v, const float *g, const float *beta, double *o,
                        const void *initial_state, const int32_t *state_indices,
                        void *output_state, const int32_t *output_state_indices,
                        void *state_checkpoints, const int32_t *checkpoint_state_indices,
                        const int32_t *checkpoint_cu_starts, const int32_t *prefix_lens,
                        int32_t N, int64_t row_stride, const uint8_t *chain_mask,
                        uint8_t *out_written, uint8_t *ckpt_written, int32_t state_bf16)
{
    if (fegetround() != FE_TONEAREST) return -3;
    int use_ckpt = state_checkpoints && checkpoint_state_indices && checkpoint_cu_starts;
    if (use_ckpt && N <= 0) return -1;
    int64_t nchains = (int64_t)num_seqs * H;
    int failed = 0;

#pragma omp parallel
    {
        double *S = (double *)malloc(sizeof(double) * (size_t)V * K);
        double *qd = (double *)malloc(sizeof(double) * (size_t)K);
        double *kd = (double *)malloc(sizeof(double) * (size_t)K);
        double *vd = (double *)malloc(sizeof(double) * (size_t)V);
        double *u = (double *)malloc(sizeof(double) * (size_t)V);
        if (!S || !qd || !kd || !vd || !u) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(dynamic, 1)
        for (int64_t c = 0; c < nchains; ++c) {
            if (failed) continue;
            int32_t b = (int32_t)(c / H), h = (int32_t)(c % H);
            if (chain_mask && !chain_mask[c]) continue;
            int64_t t0 = cu_seqlens[b], len = (int64_t)cu_seqlens[b + 1] - cu_seqlens[b];
            if (len <= 0) continue;
            int64_t prefix = prefix_lens ? prefix_lens[b] : 0;

            memset(S, 0, sizeof(double) * (size_t)V * K);
            if (initial_state && state_indices && state_indices[b] >= 0)
                load_state(S, initial_state, state_bf16, state_indices[b], row_stride, h, K, V);

            int64_t j = 0; /* checkpoints taken so far by this call */
            for (int64_t n = 1; n <= len; ++n) {
                int64_t t = t0 + n - 1;
                for (int32_t x = 0; x < K; ++x) {
                    qd[x] = bf16_bits_to_double(q[(t * H + h) * K + x]);
                    kd[x] = bf16_bits_to_double(k[(t * H + h) * K + x]);
                }
                for (int32_t x = 0; x < V; ++x) vd[x] = bf16_bits_to_double(v[(t * H + h) * V + x]);
                gdn_token(S, K, V, qd, kd, vd, (double)g[t * H + h], (double)beta[t * H + h],
                          scale, o + (t * H + h) * V, u);
                if (use_ckpt && (prefix + n) % N == 0) {
                    int32_t row = checkpoint_state_indices[checkpoint_cu_starts[b] + j];
                    ++j;
                    if (row >= 0) {
                        store_state(S, state_checkpoints, state_bf16, row, row_stride, h, K, V);
                        mark(ckpt_written, row);
                    }
                }
            }
            if (output_state && output_state_indices && output_state_indices[b] >= 0) {
                store_state(S, output_state, state_bf16, output_state_indices[b], row_stride, h, K, V);
                mark(out_written, output_state_indices[b]);
            }
        }
        free(S);
        free(qd);
        free(kd);
        free(vd);
        free(u);
    }
    return failed ? -2 : 0;
}

int oracle_chunk_gdn(int32_t num_seqs, const int32_t *cu_seqlens, int32_t H, int32_t K,
                     int32_t V, double scale, const uint16_t *q, const uint16_t *k,
                     const uint16_t *v, const float *g, const float *beta, double *o,
                     const float *initial_state, const int32_t *state_indices,
                     float *output_state, const int32_t *output_state_indices,
                     float *state_checkpoints, const int32_t *checkpoint_state_indices,
                     const int32_t *checkpoint_cu_starts, const int32_t *prefix_lens,
                     int32_t N, int64_t row_stride, const uint8_t *chain_mask,
                     uint8_t *out_written, uint8_t *ckpt_written)
{
    return oracle_chunk_gdn_st(num_seqs, cu_seqlens, H, K, V, scale, q, k, v, g, beta, o,
                               initial_state, state_indices, output_state, output_state_indices,
                               state_checkpoints, checkpoint_state_indices, checkpoint_cu_starts,
                               prefix_lens, N, row_stride, chain_mask, out_written, ckpt_written, 0);
}

/* Single-token decode (decode paragraph): for every (b, h), read row
 * initial_state_indices[b] (-1 = zero state), apply one token and store the new
 * state to row output_state_indices[b] (in place when the two are equal).
 * q, k are [B, H, K], v [B, H, V], g and beta [B, H], o [B, H, V].  state_bf16
 * selects a bf16 pool. */
int oracle_decode_st(int32_t batch, int32_t H, int32_t K, int32_t V, double scale,
                     const uint16_t *q, const uint16_t *k, const uint16_t *v, const float *g,
                     const float *beta, double *o, void *pool, int64_t row_stride,
                     const int32_t *initial_state_indices, const int32_t *output_state_indices,
                     const uint8_t *chain_mask, uint8_t *written, int32_t state_bf16)
{
    if (fegetround() != FE_TONEAREST) return -3;
    int64_t nchains = (int64_t)batch * H;
    int failed = 0;
#pragma omp parallel
    {
        double *S = (double *)malloc(sizeof(double) * (size_t)V * K);
        double *qd = (double *)malloc(sizeof(double) * (size_t)K);
        double *kd = (double *)malloc(sizeof(double) * (size_t)K);
        double *vd = (double *)malloc(sizeof(double) * (size_t)V);
        double *u = (double *)malloc(sizeof(double) * (size_t)V);
        if (!S || !qd || !kd || !vd || !u) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(dynamic, 16)
        for (int64_t c = 0; c < nchains; ++c) {
            if (failed) continue;
            int32_t b = (int32_t)(c / H), h = (int32_t)(c % H);
            if (chain_mask && !chain_mask[c]) continue;
            memset(S, 0, sizeof(double) * (size_t)V * K);
            if (initial_state_indices[b] >= 0)
                load_state(S, pool, state_bf16, initial_state_indices[b], row_stride, h, K, V);
            for (int32_t x = 0; x < K; ++x) {
                qd[x] = bf16_bits_to_double(q[c * K + x]);
                kd[x] = bf16_bits_to_double(k[c * K + x]);
            }
            for (int32_t x = 0; x < V; ++x) vd[x] = bf16_bits_to_double(v[c * V + x]);
            gdn_token(S, K, V, qd, kd, vd, (double)g[c], (double)beta[c], scale, o + c * V, u);
            if (output_state_indices[b] >= 0) {
                store_state(S, pool, state_bf16, output_state_indices[b], row_stride, h, K, V);
                mark(written, output_state_indices[b]);
            }
        }
        free(S);
        free(qd);
        free(kd);
        free(vd);
        free(u);
    }
    return failed ? -2 : 0;
}

int oracle_decode(int32_t batch, int32_t H, int32_t K, int32_t V, double scale,
                  const uint16_t *q, const uint16_t *k, const uint16_t *v, const float *g,
                  const float *beta, double *o, float *pool, int64_t row_stride,
                  const int32_t *initial_state_indices, const int32_t *output_state_indices,
                  const uint8_t *chain_mask, uint8_t *written)
{
    return oracle_decode_st(batch, H, K, V, scale, q, k, v, g, beta, o, pool, row_stride,
                            initial_state_indices, output_state_indices, chain_mask, written, 0);
}
