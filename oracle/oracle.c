/*
 * oracle.c -- plain, slow, single-threaded CPU oracle for the sparse paged
 * decode path.  TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the
 * benchmark's CPU-baseline leg may call it; the product path never does.
 *
 * It shares no code with the CUDA library: its own E4M3 and BF16 decoders,
 * its own loops, fp64 arithmetic throughout.  Every function writes out the
 * plain definition of what it computes; nothing is blocked, fused or
 * reordered beyond that definition.
 *
 * Sources (page title -- section):
 *   "Kernel ABI" -- Attention block slots: attention.decode,
 *                   attention.msa_block_score, attention.msa_prefill_block_score
 *   "Kernel ABI" -- Attention block slots: attention.sdpa (GQA expansion rule)
 *   "MiniMax-M3 decode through the ATOM kernel library" -- Supported experiment
 *                   (FP8 caches, block size 128) and the paragraph after it
 *                   (static scalar K/V scales)
 *   "Slot contract" -- 3. Correctness uses trusted high-precision ground truth
 *
 * Readings where the pages leave a step open (each one is listed in the
 * design notes):
 *   - block score = max over the valid tokens tau of a block of
 *     (q_idx . k_idx[tau]) * idx_scale; a block with no valid token scores -inf;
 *   - token tau of a request is valid iff tau < seq_len of that query token,
 *     its block lies inside the page table and its page id lies in the pool;
 *   - top-k keeps the K largest candidate cells (not NaN, not -inf), in
 *     descending score order, ties to the lower block id, pads with -1;
 *   - a selection is a set of block ids: negative ids, ids >= the page-table
 *     capacity and repeats select nothing more;
 *   - q head g reads kv head g / (Hq / Hkv);
 *   - a query token with no valid key writes zeros;
 *   - dense attention's causal flag aligns the T query tokens with the last
 *     T of the S keys (query t reads keys j <= t + S - T).
 *
 * Parity pins: every function below is pinned by the "not gpu" tests
 * (brute force with numpy / torch fp64 SDPA, closed forms, invariants,
 * hand-worked fixtures, and planted-mistake runs of a mutated copy).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* element types of the raw buffers handed to the oracle */
enum { OR_F32 = 0, OR_BF16 = 1, OR_F16 = 2, OR_E4M3 = 3, OR_I32 = 4 };

/* ---------------------------------------------------------------- decoders */

/* OCP FP8 E4M3 ("e4m3fn"): 1 sign bit, 4 exponent bits (bias 7), 3 mantissa
 * bits; exponent 0 is subnormal (m/8 * 2^-6); S.1111.111 is NaN; no infinity;
 * the largest finite magnitude is 1.75 * 2^8 = 448. */
double oracle_e4m3_value(uint8_t code)
{
    int sign = code >> 7;
    int expo = (code >> 3) & 0xF;
    int mant = code & 0x7;
    double mag;
    if (expo == 0xF && mant == 0x7)
        return NAN;
    if (expo == 0)
        mag = ldexp((double)mant / 8.0, -6);
    else
        mag = ldexp(1.0 + (double)mant / 8.0, expo - 7);
    return sign ? -mag : mag;
}

/* bfloat16 is the upper half of an IEEE binary32 word. */
double oracle_bf16_value(uint16_t bits)
{
    uint32_t word = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &word, sizeof f);
    return (double)f;
}

/* IEEE binary16: 1 sign, 5 exponent bits (bias 15), 10 mantissa bits. */
double oracle_f16_value(uint16_t bits)
{
    int sign = bits >> 15;
    int expo = (bits >> 10) & 0x1F;
    int mant = bits & 0x3FF;
    double mag;
    if (expo == 0x1F)
        mag = mant ? NAN : INFINITY;
    else if (expo == 0)
        mag = ldexp((double)mant / 1024.0, -14);
    else
        mag = ldexp(1.0 + (double)mant / 1024.0, expo - 15);
    return sign ? -mag : mag;
}

static double load(const void *base, int dtype, int64_t i)
{
    switch (dtype) {
    case OR_F32:  return (double)((const float *)base)[i];
    case OR_BF16: return oracle_bf16_value(((const uint16_t *)base)[i]);
    case OR_F16:  return oracle_f16_value(((const uint16_t *)base)[i]);
    case OR_E4M3: return oracle_e4m3_value(((const uint8_t *)base)[i]);
    default:      return NAN;
    }
}

/* ------------------------------------------------------- paged addressing */

/* Number of leading logical tokens of query token t that can be read at all:
 * seq_len clipped to [0, NB * block_size]; 0 when the token's request row is
 * outside the page table. */
static int64_t token_limit(const int32_t *req_idx, const int32_t *seq_lens,
                           int64_t t, int64_t R, int64_t NB, int64_t bs)
{
    int64_t r = req_idx[t];
    int64_t L = seq_lens[t];
    if (r < 0 || r >= R || L <= 0)
        return 0;
    if (L > NB * bs)
        L = NB * bs;
    return L;
}

/* Page id holding logical block b of request row r, or -1 when it lies
 * outside the pool of n_pages pages. */
static int64_t page_of(const int32_t *block_table, int64_t NB, int64_t r,
                       int64_t b, int64_t n_pages)
{
    int64_t p = block_table[r * NB + b];
    return (p >= 0 && p < n_pages) ? p : -1;
}

/* ------------------------------------------------------------ block score */

/*
 * "Kernel ABI" -- attention.msa_block_score: a score sheet of per-request
 * block-max scores over the paged index cache.
 *
 *   scores[h][t][b] = max over valid tau in block b of
 *                     (sum_d q_idx[t][h][d] * k_idx[slot(tau)][0][d]) * idx_scale
 *
 * with slot(tau) = block_size * block_table[r][tau / block_size] + tau % block_size,
 * r = req_idx[t]; -inf where block b holds no valid token.  The index cache
 * has a single key head shared by the Hi query index heads ("index_k_cache:
 * paged (slots, 1, D)" in attention.msa_prefill_block_score).
 *
 * Layouts (contiguous): q_idx [T][Hi][Di], k_idx [n_slots][1][Di],
 * block_table [R][NB], req_idx [T], seq_lens [T], scores [Hi][T][NB].
 */
int oracle_block_score(const void *q_idx, int q_dtype, int64_t T, int64_t Hi, int64_t Di,
                       const void *k_idx, int k_dtype, int64_t n_slots,
                       const int32_t *block_table, int64_t R, int64_t NB,
                       const int32_t *req_idx, const int32_t *seq_lens,
                       double idx_scale, int64_t block_size, double *scores)
{
    int64_t n_pages = n_slots / block_size;
    for (int64_t h = 0; h < Hi; ++h) {
        for (int64_t t = 0; t < T; ++t) {
            int64_t L = token_limit(req_idx, seq_lens, t, R, NB, block_size);
            int64_t r = req_idx[t];
            for (int64_t b = 0; b < NB; ++b) {
                double best = -INFINITY;
                int64_t page = (b * block_size < L) ? page_of(block_table, NB, r, b, n_pages) : -1;
                if (page >= 0) {
                    for (int64_t i = 0; i < block_size; ++i) {
                        int64_t tau = b * block_size + i;
                        if (tau >= L)
                            break;
                        int64_t slot = page * block_size + i;
                        double dot = 0.0;
                        for (int64_t d = 0; d < Di; ++d)
                            dot += load(q_idx, q_dtype, (t * Hi + h) * Di + d) *
                                   load(k_idx, k_dtype, slot * Di + d);
                        double s = dot * idx_scale;
                        if (s > best)
                            best = s;
                    }
                }
                scores[(h * T + t) * NB + b] = best;
            }
        }
    }
    return 0;
}

/* ------------------------------------------------------------------ top-k */

typedef struct { double score; int32_t block; } cell_t;

/* descending score, ties to the lower block id */
static int cell_order(const void *pa, const void *pb)
{
    const cell_t *a = (const cell_t *)pa, *b = (const cell_t *)pb;
    if (a->score > b->score) return -1;
    if (a->score < b->score) return 1;
    return (a->block > b->block) - (a->block < b->block);
}

/*
 * "Kernel ABI" -- attention.decode ("topk_idx: (Hkv,B,K) block IDs", "-1
 * entries ... are excluded") and attention.msa_prefill_block_score ("unused
 * output cells must be -1"): per row, the K highest-scoring candidate blocks
 * in descending order, ties to the lower block id, padded with -1.
 * A candidate is a cell that is neither NaN nor -inf.
 *
 * Layouts (contiguous): scores [rows][NB], topk [rows][K].
 */
int oracle_select_topk(const double *scores, int64_t rows, int64_t NB, int64_t K, int32_t *topk)
{
    cell_t *cells = (cell_t *)malloc(sizeof(cell_t) * (size_t)(NB > 0 ? NB : 1));
    if (!cells)
        return -1;
    for (int64_t row = 0; row < rows; ++row) {
        int64_t n = 0;
        for (int64_t b = 0; b < NB; ++b) {
            double s = scores[row * NB + b];
            if (!isnan(s) && s != -INFINITY) {
                cells[n].score = s;
                cells[n].block = (int32_t)b;
                ++n;
            }
        }
        qsort(cells, (size_t)n, sizeof(cell_t), cell_order);
        for (int64_t k = 0; k < K; ++k)
            topk[row * K + k] = (k < n) ? cells[k].block : -1;
    }
    free(cells);
    return 0;
}

/* -------------------------------------------------------------- attention */

/*
 * "Kernel ABI" -- attention.decode: paged GQA decode attention of each query
 * row over exactly the supplied non-negative block ids; -1 entries and tokens
 * at or beyond seq_lens are excluded.  K/V are FP8-E4M3 with static scalar
 * scales ("MiniMax-M3 decode through the ATOM kernel library").  GQA: Hq is
 * divisible by Hkv ("attention.sdpa"); q head g reads kv head g / (Hq/Hkv).
 *
 * For query token t and q head g, over the selected valid tokens tau taken in
 * ascending block id, then ascending position:
 *   z_tau  = sm_scale * k_scale * sum_d q[t][g][d] * e4m3(k8[slot(tau)][h][d])
 *   out[t][g][d] = sum_tau exp(z_tau - max z) * v_scale * e4m3(v8[slot(tau)][h][d])
 *                  / sum_tau exp(z_tau - max z)
 * (two passes: the maximum first, then both sums).  No valid token -> 0.
 *
 * topk == NULL selects every block (dense paged decode, the degenerate case).
 * kv_dtype is OR_E4M3 for the FP8 caches of the ATOM run or OR_BF16 for a
 * dense BF16 cache ("Kernel ABI" -- attention.decode: the commissioned cache
 * is dense BF16); the scales multiply the decoded values either way (1.0
 * for a BF16 cache stored unscaled).
 * Layouts (contiguous): q [T][Hq][D], k8/v8 [n_slots][Hkv][D] (E4M3 bytes or BF16),
 * block_table [R][NB], req_idx [T], seq_lens [T], topk [Hkv][T][K],
 * out [T][Hq][D].
 */
int oracle_paged_attention(const void *q, int q_dtype, int64_t T, int64_t Hq, int64_t D,
                           const void *k8, const void *v8, int kv_dtype, int64_t n_slots, int64_t Hkv,
                           const int32_t *block_table, int64_t R, int64_t NB,
                           const int32_t *req_idx, const int32_t *seq_lens,
                           const int32_t *topk, int64_t K,
                           double sm_scale, double k_scale, double v_scale,
                           int64_t block_size, double *out)
{
    int64_t n_pages = n_slots / block_size;
    int64_t G = Hq / Hkv;
    int64_t max_tokens = NB * block_size;
    char *selected = (char *)malloc((size_t)(NB > 0 ? NB : 1));
    int64_t *slots = (int64_t *)malloc(sizeof(int64_t) * (size_t)(max_tokens > 0 ? max_tokens : 1));
    double *z = (double *)malloc(sizeof(double) * (size_t)(max_tokens > 0 ? max_tokens : 1));
    if (!selected || !slots || !z) {
        free(selected); free(slots); free(z);
        return -1;
    }
    for (int64_t t = 0; t < T; ++t) {
        int64_t L = token_limit(req_idx, seq_lens, t, R, NB, block_size);
        int64_t r = req_idx[t];
        for (int64_t g = 0; g < Hq; ++g) {
            int64_t h = g / G;

            /* the selected block set of (kv head h, token t) */
            for (int64_t b = 0; b < NB; ++b)
                selected[b] = (topk == NULL);
            if (topk != NULL) {
                for (int64_t k = 0; k < K; ++k) {
                    int64_t b = topk[(h * T + t) * K + k];
                    if (b >= 0 && b < NB)
                        selected[b] = 1;
                }
            }

            /* the valid tokens, ascending block id then position */
            int64_t n = 0;
            for (int64_t b = 0; b < NB && L > 0; ++b) {
                if (!selected[b] || b * block_size >= L)
                    continue;
                int64_t page = page_of(block_table, NB, r, b, n_pages);
                if (page < 0)
                    continue;
                for (int64_t i = 0; i < block_size && b * block_size + i < L; ++i)
                    slots[n++] = page * block_size + i;
            }

            double *o = out + (t * Hq + g) * D;
            if (n == 0) {
                for (int64_t d = 0; d < D; ++d)
                    o[d] = 0.0;
                continue;
            }

            /* pass 1: logits and their maximum */
            double zmax = -INFINITY;
            for (int64_t j = 0; j < n; ++j) {
                double dot = 0.0;
                for (int64_t d = 0; d < D; ++d)
                    dot += load(q, q_dtype, (t * Hq + g) * D + d) *
                           load(k8, kv_dtype, (slots[j] * Hkv + h) * D + d);
                z[j] = sm_scale * k_scale * dot;
                if (z[j] > zmax)
                    zmax = z[j];
            }

            /* pass 2: normaliser and weighted sum of values */
            double l = 0.0;
            for (int64_t d = 0; d < D; ++d)
                o[d] = 0.0;
            for (int64_t j = 0; j < n; ++j) {
                double w = exp(z[j] - zmax);
                l += w;
                for (int64_t d = 0; d < D; ++d)
                    o[d] += w * v_scale * load(v8, kv_dtype, (slots[j] * Hkv + h) * D + d);
            }
            for (int64_t d = 0; d < D; ++d)
                o[d] /= l;
        }
    }
    free(selected);
    free(slots);
    free(z);
    return 0;
}

/* --------------------------------------------------- dense GQA attention */

/*
 * "Kernel ABI" -- attention.sdpa: scaled dot-product attention of T query
 * tokens over S keys, with GQA expansion (Hq divisible by Hkv; q head g reads
 * kv head g / (Hq / Hkv)) and a causal flag.
 *
 * Causal reading (the page gives the flag, not its alignment): the T query
 * tokens are the last T positions of the S-key sequence, so query token t may
 * read key j iff j <= t + (S - T).  For T == S this is the usual
 * lower-triangular mask; a query token with no readable key (t + S - T < 0)
 * writes zeros.  Without the flag every query token reads all S keys.
 *
 *   z_j  = sm_scale * sum_d q[t][g][d] * k[j][h][d]
 *   out[t][g][d] = sum_j exp(z_j - max z) * v[j][h][d] / sum_j exp(z_j - max z)
 *
 * over the readable keys in ascending j (two passes: the maximum first, then
 * both sums).  q, k and v share one element type.
 * Layouts (contiguous): q [T][Hq][D], k/v [S][Hkv][D], out [T][Hq][D].
 */
int oracle_sdpa(const void *q, const void *k, const void *v, int dtype,
                int64_t T, int64_t S, int64_t Hq, int64_t Hkv, int64_t D,
                double sm_scale, int causal, double *out)
{
    int64_t G = Hq / Hkv;
    double *z = (double *)malloc(sizeof(double) * (size_t)(S > 0 ? S : 1));
    if (!z)
        return -1;
    for (int64_t t = 0; t < T; ++t) {
        /* number of readable keys: 0 .. n-1 */
        int64_t n = S;
        if (causal) {
            n = t + (S - T) + 1;
            if (n < 0)
                n = 0;
            if (n > S)
                n = S;
        }
        for (int64_t g = 0; g < Hq; ++g) {
            int64_t kvh = g / G;
            double *o = out + (t * Hq + g) * D;
            for (int64_t d = 0; d < D; ++d)
                o[d] = 0.0;
            if (n == 0)
                continue;

            /* pass 1: logits and their maximum */
            double zmax = -INFINITY;
            for (int64_t j = 0; j < n; ++j) {
                double dot = 0.0;
                for (int64_t d = 0; d < D; ++d)
                    dot += load(q, dtype, (t * Hq + g) * D + d) * load(k, dtype, (j * Hkv + kvh) * D + d);
                z[j] = sm_scale * dot;
                if (z[j] > zmax)
                    zmax = z[j];
            }

            /* pass 2: normaliser and weighted sum of values */
            double l = 0.0;
            for (int64_t j = 0; j < n; ++j) {
                double w = exp(z[j] - zmax);
                l += w;
                for (int64_t d = 0; d < D; ++d)
                    o[d] += w * load(v, dtype, (j * Hkv + kvh) * D + d);
            }
            for (int64_t d = 0; d < D; ++d)
                o[d] /= l;
        }
    }
    free(z);
    return 0;
}

/* ------------------------------------ prefill score-to-selection (V2) */

/*
 * "Kernel ABI" -- attention.msa_prefill_block_score: one call that scores and
 * selects for a ragged batch of prefill chunks over a paged index cache, per
 * query head and per query block of block_size_q tokens.
 *
 * Sequence b owns query tokens cu_seqlens[b] .. cu_seqlens[b+1]-1 (its chunk,
 * whose first token sits at position prefix_lens[b]), seq_lens[b] keys in
 * total, and output rows cu_seqblocks_q[b] + qb for its query blocks qb.
 * Its keys are read through row slot_ids[b] of the page table.
 *
 * Readings (the page states the rule, not the formulas):
 *   - visibility: query block qb sees the keys at positions up to and
 *     including prefix_lens[b] + qb * block_size_q (its first token's own
 *     position), so L = prefix_lens[b] + qb * block_size_q + 1 keys, clipped
 *     to seq_lens[b] and to the page table; key block kb is visible iff
 *     kb * block_size < L (nvis = ceil(L / block_size) blocks);
 *   - score: the block-max of the decode score sheet taken over the query
 *     block as well: max over the block's tokens t and the keys tau < L of
 *     key block kb of (q[t][h] . k[slot(tau)]) * scale; -inf if none;
 *   - policy: the first init_blocks and the last local_blocks visible blocks
 *     are always selected and come first, in ascending id; the remaining
 *     cells are filled with the other visible candidate blocks (score neither
 *     NaN nor -inf) in descending score, ties to the lower id; then -1.
 *     Ids are logical block ids of the request's key sequence.
 * Rows that no sequence owns are all -1.  With block_size_q = 1 and no
 * init/local blocks a row is exactly the decode top-k of one query token
 * whose seq_len is its position + 1.
 *
 * Layouts (contiguous): q [total_q][Hi][Di], k [n_slots][1][Di],
 * block_table [R][NB], slot_ids/seq_lens/prefix_lens [B],
 * cu_seqlens/cu_seqblocks_q [B+1], out [Hi][n_rows][topk];
 * scores (optional) [Hi][n_rows][NB] receives the block scores (-inf for
 * blocks that are not visible).
 */
int oracle_prefill_topk(const void *q, int q_dtype, int64_t total_q, int64_t Hi, int64_t Di,
                        const void *k, int k_dtype, int64_t n_slots,
                        const int32_t *block_table, int64_t R, int64_t NB,
                        const int32_t *slot_ids, const int32_t *cu_seqlens, const int32_t *seq_lens,
                        const int32_t *prefix_lens, const int32_t *cu_seqblocks_q, int64_t B,
                        int64_t block_size_q, int64_t init_blocks, int64_t local_blocks,
                        double scale, int64_t block_size, int64_t n_rows, int64_t topk,
                        int32_t *out, double *scores)
{
    int64_t n_pages = n_slots / block_size;
    double *s = (double *)malloc(sizeof(double) * (size_t)(NB > 0 ? NB : 1));
    char *forced = (char *)malloc((size_t)(NB > 0 ? NB : 1));
    cell_t *cells = (cell_t *)malloc(sizeof(cell_t) * (size_t)(NB > 0 ? NB : 1));
    if (!s || !forced || !cells) {
        free(s); free(forced); free(cells);
        return -1;
    }
    for (int64_t i = 0; i < Hi * n_rows * topk; ++i)
        out[i] = -1;
    if (scores)
        for (int64_t i = 0; i < Hi * n_rows * NB; ++i)
            scores[i] = -INFINITY;

    for (int64_t b = 0; b < B; ++b) {
        int64_t r = slot_ids[b];
        for (int64_t qb = 0; qb < (int64_t)cu_seqblocks_q[b + 1] - cu_seqblocks_q[b]; ++qb) {
            int64_t row = cu_seqblocks_q[b] + qb;
            if (row < 0 || row >= n_rows)
                continue;

            /* visible keys and blocks */
            int64_t L = (int64_t)prefix_lens[b] + qb * block_size_q + 1;
            if (L > seq_lens[b])
                L = seq_lens[b];
            if (L > NB * block_size)
                L = NB * block_size;
            if (r < 0 || r >= R || L < 0)
                L = 0;
            int64_t nvis = (L + block_size - 1) / block_size;

            /* the query block's tokens */
            int64_t t0 = (int64_t)cu_seqlens[b] + qb * block_size_q;
            int64_t t1 = t0 + block_size_q;
            if (t1 > cu_seqlens[b + 1])
                t1 = cu_seqlens[b + 1];
            if (t0 < 0)
                t0 = 0;
            if (t1 > total_q)
                t1 = total_q;

            for (int64_t h = 0; h < Hi; ++h) {
                /* block scores */
                for (int64_t kb = 0; kb < NB; ++kb) {
                    double best = -INFINITY;
                    int64_t page = kb < nvis ? page_of(block_table, NB, r, kb, n_pages) : -1;
                    for (int64_t t = t0; t < t1 && page >= 0; ++t) {
                        for (int64_t tau = kb * block_size; tau < (kb + 1) * block_size && tau < L; ++tau) {
                            int64_t slot = page * block_size + (tau - kb * block_size);
                            double dot = 0.0;
                            for (int64_t d = 0; d < Di; ++d)
                                dot += load(q, q_dtype, (t * Hi + h) * Di + d) * load(k, k_dtype, slot * Di + d);
                            double v = dot * scale;
                            if (v > best)
                                best = v;
                        }
                    }
                    s[kb] = best;
                    if (scores)
                        scores[(h * n_rows + row) * NB + kb] = best;
                }

                /* policy blocks first, ascending id */
                int32_t *o = out + (h * n_rows + row) * topk;
                int64_t n = 0;
                for (int64_t kb = 0; kb < NB; ++kb) {
                    forced[kb] = kb < nvis && (kb < init_blocks || kb >= nvis - local_blocks);
                    if (forced[kb] && n < topk)
                        o[n++] = (int32_t)kb;
                }

                /* then the best of the other visible candidates */
                int64_t m = 0;
                for (int64_t kb = 0; kb < nvis; ++kb) {
                    if (forced[kb] || isnan(s[kb]) || s[kb] == -INFINITY)
                        continue;
                    cells[m].score = s[kb];
                    cells[m].block = (int32_t)kb;
                    ++m;
                }
                qsort(cells, (size_t)m, sizeof(cell_t), cell_order);
                for (int64_t j = 0; j < m && n < topk; ++j)
                    o[n++] = cells[j].block;
            }
        }
    }
    free(s);
    free(forced);
    free(cells);
    return 0;
}
