/*
 * pa_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * The plain, slow, fp64 CPU oracle for paged-attention decode.  Only the
 * tests, the smoke check and the CPU-baseline leg of the benchmark load it;
 * the product library never does, and the two share no code, header, table
 * or helper.  Every loop below is the textbook definition written out, with
 * no blocking, fusion or reordering beyond what the definition states.
 *
 * Passages followed (page: project_6 commit cd0d9e1, "qwen3_6_scripts"):
 *   [gather]   the prefix-prefill rewrite's pre-gather of all context K/V:
 *              logical block j of a sequence is the physical cache block
 *              named by entry j of its block-table row.
 *   [v1/v2]    the forward_decode heuristic: the single-pass path (V1) and
 *              the partitioned path (V2) are two schedules of one attention
 *              result for the single decode query.
 *   [phase 1]  the V2 description, phase 1: every (sequence, head,
 *              partition) computes its scaled logits, their softmax and the
 *              weighted V sum, and keeps three partial results: the partial
 *              output, the exp-sum and the maximum logit.
 *   [prefill]  the prefix-prefill rewrite: a chunk of new tokens attends to
 *              the whole cached context of its sequence (gathered once) and,
 *              causally, to the chunk itself.
 *   [phase 2]  the V2 description, phase 2: the maximum over partitions is
 *              taken, each partition is weighted by exp(its max - that
 *              maximum) times its exp-sum, and the output is the weighted
 *              mean of the partial outputs.
 *
 * Readings where the pages are silent (each one is listed in the design
 * notes): query head h reads KV head h / (Hq/Hkv); max_logits are maxima of
 * the *scaled* logits scale*q.k; exp_sums are taken relative to the
 * partition's own max; the partial output is normalised by its own exp-sum
 * (this is what makes the phase-2 weight, which multiplies by the exp-sum,
 * correct); the partition count is ceil(L/P); a sequence with L = 0
 * produces a zero output.
 *
 * Layouts (all row-major, element offsets):
 *   query        [S][Hq][d]                 16-bit float bit patterns
 *   key/value    [num_blocks][bs][Hkv][d]   16-bit float bit patterns
 *   block_tables [S][max_blocks]            int32
 *   seq_lens     [S]                        int32
 *   out          [S][Hq][d]                 double
 *   tmp_out      [S][Hq][NP][d]             double
 *   exp_sums, max_logits [S][Hq][NP]        double
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_F16 0
#define ORACLE_BF16 1

#define ORACLE_OK 0
#define ORACLE_BAD_ARGS (-1)
#define ORACLE_BAD_TABLE (-2)
#define ORACLE_NO_MEMORY (-3)

/* Exact widening of one IEEE binary16 or bfloat16 bit pattern to double. */
double oracle_half_bits_to_f64(uint16_t h, int dtype)
{
    if (dtype == ORACLE_BF16) {
        /* bfloat16 is the top half of an IEEE binary32 word. */
        uint32_t w = ((uint32_t)h) << 16;
        float f;
        memcpy(&f, &w, sizeof f);
        return (double)f;
    }
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int m = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24);              /* subnormal: m * 2^-24 */
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(m | 0x400), e - 25); /* (1 + m/1024) * 2^(e-15) */
    return sign ? -v : v;
}

void oracle_bits_to_f64(const uint16_t *in, double *out, int64_t n, int dtype)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_half_bits_to_f64(in[i], dtype);
}

/* Offset of element (block, row, kv head, dim) in a cache. */
static int64_t cache_off(int64_t b, int o, int kvh, int i, int bs, int Hkv, int d)
{
    return ((b * bs + o) * (int64_t)Hkv + kvh) * d + i;
}

/* Physical block holding token t of sequence s, or -1 if the table entry is
 * outside the cache. [gather] */
static int64_t phys_block(const int32_t *bt, int s, int t, int bs, int max_blocks,
                          int num_blocks)
{
    int64_t b = bt[(int64_t)s * max_blocks + t / bs];
    if (b < 0 || b >= num_blocks)
        return -1;
    return b;
}

static int check_lengths(const int32_t *seq_lens, int S, int bs, int max_blocks)
{
    for (int s = 0; s < S; ++s)
        if (seq_lens[s] < 0 || (int64_t)seq_lens[s] > (int64_t)max_blocks * bs)
            return ORACLE_BAD_ARGS;
    return ORACLE_OK;
}

static int check_dims(int S, int Hq, int Hkv, int d, int bs, int num_blocks,
                      int max_blocks)
{
    if (S < 0 || Hq <= 0 || Hkv <= 0 || d <= 0 || bs <= 0 || num_blocks < 0 ||
        max_blocks < 0 || Hq % Hkv != 0)
        return ORACLE_BAD_ARGS;
    return ORACLE_OK;
}

/* x[t - t0] = scale * sum_i qrow[i] * k_t[i] for t in [t0, t1) of sequence s,
 * and the query row widened once into qd[d]. */
static int scaled_logits(double *x, double *qd, const uint16_t *qrow, const uint16_t *kc,
                         const int32_t *bt, int s, int kvh, int t0, int t1, int Hkv, int d,
                         int bs, int num_blocks, int max_blocks, double scale, int dtype)
{
    for (int i = 0; i < d; ++i)
        qd[i] = oracle_half_bits_to_f64(qrow[i], dtype);
    for (int t = t0; t < t1; ++t) {
        int64_t b = phys_block(bt, s, t, bs, max_blocks, num_blocks);
        if (b < 0)
            return ORACLE_BAD_TABLE;
        int64_t base = cache_off(b, t % bs, kvh, 0, bs, Hkv, d);
        double acc = 0.0;
        for (int i = 0; i < d; ++i)
            acc += qd[i] * oracle_half_bits_to_f64(kc[base + i], dtype);
        x[t - t0] = scale * acc;
    }
    return ORACLE_OK;
}

/* Softmax-weighted V sum over tokens [t0, t1) given their logits x:
 *   m = max x,  l = sum exp(x - m),  o = sum exp(x - m) v_t / l.          */
static void softmax_v(double *o, double *m_out, double *l_out, const double *x,
                      const uint16_t *vc, const int32_t *bt, int s, int kvh, int t0,
                      int t1, int Hkv, int d, int bs, int num_blocks, int max_blocks,
                      int dtype)
{
    double m = -INFINITY;
    for (int t = t0; t < t1; ++t)
        if (x[t - t0] > m)
            m = x[t - t0];
    double l = 0.0;
    for (int i = 0; i < d; ++i)
        o[i] = 0.0;
    for (int t = t0; t < t1; ++t) {
        double p = exp(x[t - t0] - m);
        l += p;
        int64_t b = phys_block(bt, s, t, bs, max_blocks, num_blocks);
        int64_t base = cache_off(b, t % bs, kvh, 0, bs, Hkv, d);
        for (int i = 0; i < d; ++i)
            o[i] += p * oracle_half_bits_to_f64(vc[base + i], dtype);
    }
    for (int i = 0; i < d; ++i)
        o[i] /= l;
    *m_out = m;
    *l_out = l;
}

/*
 * Single-pass decode [v1/v2]: for every sequence s and query head h,
 *   out[s][h] = softmax_t(scale * q[s][h] . k_t) weighted sum of v_t,
 * t over the sequence's L = seq_lens[s] tokens, K/V read through the table.
 */
int oracle_attention(double *out, const uint16_t *q, const uint16_t *kc,
                     const uint16_t *vc, const int32_t *bt, const int32_t *seq_lens,
                     int S, int Hq, int Hkv, int d, int bs, int num_blocks,
                     int max_blocks, float scale, int dtype)
{
    int rc = check_dims(S, Hq, Hkv, d, bs, num_blocks, max_blocks);
    if (rc == ORACLE_OK)
        rc = check_lengths(seq_lens, S, bs, max_blocks);
    if (rc != ORACLE_OK)
        return rc;
    int g = Hq / Hkv;
    int status = ORACLE_OK;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t u = 0; u < (int64_t)S * Hq; ++u) {
        int s = (int)(u / Hq), h = (int)(u % Hq);
        int L = seq_lens[s];
        double *o = out + u * d;
        if (L == 0) {
            for (int i = 0; i < d; ++i)
                o[i] = 0.0;
            continue;
        }
        double *x = (double *)malloc(sizeof(double) * (size_t)L);
        double *qd = (double *)malloc(sizeof(double) * (size_t)d);
        if (!x || !qd) {
            free(x);
            free(qd);
#pragma omp atomic write
            status = ORACLE_NO_MEMORY;
            continue;
        }
        int kvh = h / g;
        int r = scaled_logits(x, qd, q + ((int64_t)s * Hq + h) * d, kc, bt, s, kvh, 0, L,
                              Hkv, d, bs, num_blocks, max_blocks, (double)scale, dtype);
        if (r == ORACLE_OK) {
            double m, l;
            softmax_v(o, &m, &l, x, vc, bt, s, kvh, 0, L, Hkv, d, bs, num_blocks,
                      max_blocks, dtype);
        } else {
#pragma omp atomic write
            status = r;
        }
        free(x);
        free(qd);
    }
    return status;
}

/*
 * Phase 1 [phase 1]: for each partition p < ceil(L/P) of tokens
 * [p*P, min((p+1)*P, L)):
 *   max_logits[s][h][p] = m_p = max of the scaled logits,
 *   exp_sums[s][h][p]   = l_p = sum exp(x_t - m_p),
 *   tmp_out[s][h][p]    = sum exp(x_t - m_p) v_t / l_p.
 * Slots p >= ceil(L/P) are left as the caller filled them.
 */
int oracle_partials(double *tmp_out, double *exp_sums, double *max_logits,
                    const uint16_t *q, const uint16_t *kc, const uint16_t *vc,
                    const int32_t *bt, const int32_t *seq_lens, int S, int Hq, int Hkv,
                    int d, int bs, int num_blocks, int max_blocks, float scale,
                    int P, int NP, int dtype)
{
    int rc = check_dims(S, Hq, Hkv, d, bs, num_blocks, max_blocks);
    if (rc == ORACLE_OK)
        rc = check_lengths(seq_lens, S, bs, max_blocks);
    if (rc != ORACLE_OK)
        return rc;
    if (P <= 0 || NP < 0)
        return ORACLE_BAD_ARGS;
    for (int s = 0; s < S; ++s)
        if ((seq_lens[s] + (int64_t)P - 1) / P > NP)
            return ORACLE_BAD_ARGS;
    int g = Hq / Hkv;
    int status = ORACLE_OK;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t u = 0; u < (int64_t)S * Hq; ++u) {
        int s = (int)(u / Hq), h = (int)(u % Hq);
        int L = seq_lens[s];
        int n = (int)((L + (int64_t)P - 1) / P);
        int kvh = h / g;
        double *x = (double *)malloc(sizeof(double) * (size_t)P);
        double *qd = (double *)malloc(sizeof(double) * (size_t)d);
        if (!x || !qd) {
            free(x);
            free(qd);
#pragma omp atomic write
            status = ORACLE_NO_MEMORY;
            continue;
        }
        for (int p = 0; p < n; ++p) {
            int t0 = p * P;
            int t1 = (t0 + P < L) ? t0 + P : L;
            int r = scaled_logits(x, qd, q + ((int64_t)s * Hq + h) * d, kc, bt, s, kvh, t0,
                                  t1, Hkv, d, bs, num_blocks, max_blocks, (double)scale,
                                  dtype);
            if (r != ORACLE_OK) {
#pragma omp atomic write
                status = r;
                break;
            }
            int64_t slot = u * NP + p;
            softmax_v(tmp_out + slot * d, &max_logits[slot], &exp_sums[slot], x, vc,
                      bt, s, kvh, t0, t1, Hkv, d, bs, num_blocks, max_blocks, dtype);
        }
        free(x);
        free(qd);
    }
    return status;
}

/*
 * Phase 2 [phase 2]: with n = ceil(L/P) partitions,
 *   M = max_p m_p,  w_p = exp(m_p - M) * l_p,
 *   out = sum_p (w_p / sum_q w_q) * tmp_out_p.
 * A sequence with no partition (L = 0) gets a zero output.
 */
int oracle_lse_merge(double *out, const double *tmp_out, const double *exp_sums,
                     const double *max_logits, const int32_t *seq_lens, int S, int Hq,
                     int d, int P, int NP)
{
    if (S < 0 || Hq <= 0 || d <= 0 || P <= 0 || NP < 0)
        return ORACLE_BAD_ARGS;
    for (int s = 0; s < S; ++s)
        if (seq_lens[s] < 0 || (seq_lens[s] + (int64_t)P - 1) / P > NP)
            return ORACLE_BAD_ARGS;
    for (int64_t u = 0; u < (int64_t)S * Hq; ++u) {
        int s = (int)(u / Hq);
        int n = (int)((seq_lens[s] + (int64_t)P - 1) / P);
        double *o = out + u * d;
        for (int i = 0; i < d; ++i)
            o[i] = 0.0;
        if (n == 0)
            continue;
        double M = -INFINITY;
        for (int p = 0; p < n; ++p)
            if (max_logits[u * NP + p] > M)
                M = max_logits[u * NP + p];
        double total = 0.0;
        for (int p = 0; p < n; ++p) {
            double w = exp(max_logits[u * NP + p] - M) * exp_sums[u * NP + p];
            total += w;
            for (int i = 0; i < d; ++i)
                o[i] += w * tmp_out[(u * NP + p) * d + i];
        }
        for (int i = 0; i < d; ++i)
            o[i] /= total;
    }
    return ORACLE_OK;
}

/*
 * Prefix prefill [prefill]: sequence s holds L = seq_lens[s] tokens in the
 * cache, the last n_s = q_start[s+1] - q_start[s] of which are new; query row
 * r = q_start[s] + i (i < n_s) sits at position p = L - n_s + i and attends
 * to the cache tokens 0..p of its sequence (the whole prefix, and the chunk
 * causally):
 *   out[r][h] = softmax_{t<=p}(scale * query[r][h] . k_t) weighted sum of v_t.
 * query / out are [q_start[S]][Hq][d].  With n_s = 1 for every sequence this
 * is the decode of oracle_attention.
 */
int oracle_prefill(double *out, const uint16_t *q, const uint16_t *kc, const uint16_t *vc,
                   const int32_t *bt, const int32_t *seq_lens, const int32_t *q_start, int S,
                   int Hq, int Hkv, int d, int bs, int num_blocks, int max_blocks, float scale,
                   int dtype)
{
    int rc = check_dims(S, Hq, Hkv, d, bs, num_blocks, max_blocks);
    if (rc == ORACLE_OK)
        rc = check_lengths(seq_lens, S, bs, max_blocks);
    if (rc != ORACLE_OK)
        return rc;
    if (q_start[0] != 0)
        return ORACLE_BAD_ARGS;
    for (int s = 0; s < S; ++s) {
        int n = q_start[s + 1] - q_start[s];
        if (n < 0 || n > seq_lens[s])
            return ORACLE_BAD_ARGS;
    }
    int g = Hq / Hkv;
    int status = ORACLE_OK;
    int64_t rows = q_start[S];
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t u = 0; u < rows * Hq; ++u) {
        int64_t r = u / Hq;
        int h = (int)(u % Hq);
        int s = 0;
        while (q_start[s + 1] <= r)
            ++s;
        int L = seq_lens[s];
        int n = q_start[s + 1] - q_start[s];
        int p = L - n + (int)(r - q_start[s]);
        double *o = out + u * d;
        double *x = (double *)malloc(sizeof(double) * (size_t)(p + 1));
        double *qd = (double *)malloc(sizeof(double) * (size_t)d);
        if (!x || !qd) {
            free(x);
            free(qd);
#pragma omp atomic write
            status = ORACLE_NO_MEMORY;
            continue;
        }
        int kvh = h / g;
        int rr = scaled_logits(x, qd, q + (r * Hq + h) * d, kc, bt, s, kvh, 0, p + 1, Hkv, d, bs,
                               num_blocks, max_blocks, (double)scale, dtype);
        if (rr == ORACLE_OK) {
            double m, l;
            softmax_v(o, &m, &l, x, vc, bt, s, kvh, 0, p + 1, Hkv, d, bs, num_blocks,
                      max_blocks, dtype);
        } else {
#pragma omp atomic write
            status = rr;
        }
        free(x);
        free(qd);
    }
    return status;
}

/*
 * [gather]: dense copies k_dense[s][t][kvh][:] = key_cache[b][t % bs][kvh][:]
 * with b = block_tables[s][t / bs], for t < L; rows t >= L are untouched.
 * Bit patterns are copied unchanged.
 */
int oracle_gather(uint16_t *k_dense, uint16_t *v_dense, const uint16_t *kc,
                  const uint16_t *vc, const int32_t *bt, const int32_t *seq_lens, int S,
                  int Hkv, int d, int bs, int num_blocks, int max_blocks, int max_len)
{
    int rc = check_dims(S, Hkv, Hkv, d, bs, num_blocks, max_blocks);
    if (rc == ORACLE_OK)
        rc = check_lengths(seq_lens, S, bs, max_blocks);
    if (rc != ORACLE_OK)
        return rc;
    for (int s = 0; s < S; ++s) {
        if (seq_lens[s] > max_len)
            return ORACLE_BAD_ARGS;
        for (int t = 0; t < seq_lens[s]; ++t) {
            int64_t b = phys_block(bt, s, t, bs, max_blocks, num_blocks);
            if (b < 0)
                return ORACLE_BAD_TABLE;
            for (int kvh = 0; kvh < Hkv; ++kvh) {
                int64_t src = cache_off(b, t % bs, kvh, 0, bs, Hkv, d);
                int64_t dst = (((int64_t)s * max_len + t) * Hkv + kvh) * d;
                memcpy(k_dense + dst, kc + src, sizeof(uint16_t) * (size_t)d);
                memcpy(v_dense + dst, vc + src, sizeof(uint16_t) * (size_t)d);
            }
        }
    }
    return ORACLE_OK;
}

/*
 * MoE routing and token regrouping (page: project_6 commit cd0d9e1,
 * "qwen3_6_scripts", the MoE prefill rewrite: 256 experts x top_k = 8; flatten
 * the T x K token-expert pairs, sort them by expert id so that each expert's
 * tokens are contiguous, gather the hidden rows in that order, and scatter the
 * per-pair expert outputs back with index_add_; page: commit 490ff98,
 * "Dockerfile", the _moe_C topk_softmax router kernel).
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *   [router]  p = softmax over all E experts of the token's logits; the k
 *             experts with the largest logits are chosen (softmax is
 *             monotonic, so these are the k largest p), ties going to the
 *             lower expert index, in descending order; the weights are their
 *             p, divided by the sum of the k chosen p when `renormalize`.
 *   [sort]    the sort is stable: within one expert, pairs keep the order of
 *             their flat index t*K + k.
 *   [scatter] index_add_ accumulates w[t][k] * y[pair] into token t's row: the
 *             routing weight is applied in the scatter-back.
 */

/* [router] weights [T][k] (fp64), ids [T][k]; logits [T][E] already widened. */
int oracle_topk_softmax(double *weights, int32_t *ids, const double *logits, int T, int E,
                        int k, int renormalize)
{
    if (T < 0 || E <= 0 || k <= 0 || k > E)
        return ORACLE_BAD_ARGS;
    char *taken = (char *)malloc((size_t)E);
    if (!taken)
        return ORACLE_NO_MEMORY;
    for (int t = 0; t < T; ++t) {
        const double *x = logits + (int64_t)t * E;
        double m = -INFINITY;
        for (int e = 0; e < E; ++e)
            if (x[e] > m)
                m = x[e];
        double z = 0.0;
        for (int e = 0; e < E; ++e)
            z += exp(x[e] - m);
        memset(taken, 0, (size_t)E);
        double sel = 0.0;
        for (int j = 0; j < k; ++j) {
            int best = -1;
            for (int e = 0; e < E; ++e)
                if (!taken[e] && (best < 0 || x[e] > x[best]))
                    best = e;
            taken[best] = 1;
            ids[(int64_t)t * k + j] = best;
            weights[(int64_t)t * k + j] = exp(x[best] - m) / z;
            sel += weights[(int64_t)t * k + j];
        }
        if (renormalize)
            for (int j = 0; j < k; ++j)
                weights[(int64_t)t * k + j] /= sel;
    }
    free(taken);
    return ORACLE_OK;
}

/* [sort] sorted_pairs [P]: the flat pair indices in expert order (stable);
 * offsets [E+1]: first sorted position of each expert, offsets[E] = P;
 * pair_pos [P]: sorted position of each pair (the inverse permutation). */
int oracle_moe_sort(int32_t *sorted_pairs, int32_t *offsets, int32_t *pair_pos,
                    const int32_t *expert_ids, int P, int E)
{
    if (P < 0 || E <= 0)
        return ORACLE_BAD_ARGS;
    for (int p = 0; p < P; ++p)
        if (expert_ids[p] < 0 || expert_ids[p] >= E)
            return ORACLE_BAD_TABLE;
    int r = 0;
    for (int e = 0; e < E; ++e) {
        offsets[e] = r;
        for (int p = 0; p < P; ++p)
            if (expert_ids[p] == e) {
                sorted_pairs[r] = p;
                pair_pos[p] = r;
                ++r;
            }
    }
    offsets[E] = r;
    return ORACLE_OK;
}

/* [gather] out [P][H]: row r is hidden row sorted_pairs[r] / K (bit copy). */
int oracle_moe_gather(uint16_t *out, const uint16_t *hidden, const int32_t *sorted_pairs,
                      int P, int K, int T, int H)
{
    if (P < 0 || K <= 0 || T < 0 || H <= 0)
        return ORACLE_BAD_ARGS;
    for (int r = 0; r < P; ++r) {
        int t = sorted_pairs[r] / K;
        if (sorted_pairs[r] < 0 || t >= T)
            return ORACLE_BAD_TABLE;
        memcpy(out + (int64_t)r * H, hidden + (int64_t)t * H, (size_t)H * sizeof(uint16_t));
    }
    return ORACLE_OK;
}

/* [scatter] out [T][H] (fp64) = sum_k weights[t][k] * y[pair_pos[t*K + k]];
 * y [P][H] holds the per-pair rows in sorted order (16-bit bit patterns). */
int oracle_moe_scatter(double *out, const uint16_t *y, const int32_t *pair_pos,
                       const double *weights, int T, int K, int P, int H, int dtype)
{
    if (T < 0 || K <= 0 || P != T * K || H <= 0)
        return ORACLE_BAD_ARGS;
    for (int t = 0; t < T; ++t) {
        double *o = out + (int64_t)t * H;
        for (int i = 0; i < H; ++i)
            o[i] = 0.0;
        for (int k = 0; k < K; ++k) {
            int r = pair_pos[(int64_t)t * K + k];
            if (r < 0 || r >= P)
                return ORACLE_BAD_TABLE;
            double w = weights[(int64_t)t * K + k];
            const uint16_t *row = y + (int64_t)r * H;
            for (int i = 0; i < H; ++i)
                o[i] += w * oracle_half_bits_to_f64(row[i], dtype);
        }
    }
    return ORACLE_OK;
}
