/*
 * fa_oracle.c -- plain, slow, fp64 CPU oracle for exact attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may include, link
 * or call this file: only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg use it.  It shares no code, header, table or helper with
 * the CUDA library; the two meet only through the seeded inputs.
 *
 * Sources (cited by page title and section):
 *   [EXPL]  "FlashAttention: Fast and Memory-Efficient Exact Attention with
 *           IO-Awareness" -- paper explainer page (xyznot.com).
 *   [MATH]  "Mathematical Properties Behind FlashAttention - Streaming
 *           Transformations for Memory-Efficient Computation" (blog).
 *   [BLOG]  core.today blog post "flash-attention" (online-softmax pseudocode).
 *
 * What is computed (the plain definition; [EXPL] "Problem and motivation":
 * S = Q K^T, P = softmax(S), O = P V).  For one (batch b, head h) and query
 * row i, the allowed key set is
 *     A_i = { j : (!causal || j <= i) && j < kv_len[b]
 *                 && block_mask[i / blk][j / blk] != 0 }
 * (masking is fused into the kernel per [EXPL] "Key ideas", kernel fusion;
 * the block mask is the block-sparse extension, [EXPL] "Extension:
 * Block-Sparse FlashAttention").  Then
 *     s_ij = scale * <q_i, k_j>,   m_i = max_j s_ij,
 *     l_i  = sum_j exp(s_ij - m_i), P_ij = exp(s_ij - m_i) / l_i,
 *     o_i  = sum_j P_ij v_j,        lse_i = m_i + ln l_i     (natural log).
 * A row with an empty A_i gets o_i = 0 and lse_i = -inf.
 *
 * Backward (textbook; the pages state only that S and P are recomputed from
 * Q, K, V, O and the statistics, [EXPL] "Key ideas", recomputation):
 *     dV = P^T dO,  dP = dO V^T,  D_i = <dO_i, o_i>,  dS = P o (dP - D),
 *     dQ = scale * dS K,  dK = scale * dS^T Q.
 *
 * Dropout (fused into the kernels per [EXPL] "Key ideas", kernel fusion; the
 * pages give no formula, so the standard one is used): with a keep mask Z and
 * keep scale c = 1 / (1 - p8/256),
 *     o_i = sum_j P_ij Z_ij c v_j  (lse from P, before dropout),
 *     dV_j = sum_i P_ij Z_ij c dO_i,  dS_ij = P_ij (Z_ij c dP_ij - D_i),
 * with D_i = <dO_i, o_i> of the dropped-out o.  Z is drawn from a
 * counter-based generator, the 32-bit PCG hash of Jarzynski and Olano
 * ("Hash Functions for GPU Rendering", JCGT 9(3), 2020), keyed by the seed
 * and the head and counted by the 2x2 block (i/2, j/2); see keep() below.
 *
 * Everything is in double precision, with plain loops and no blocking,
 * fusion or reordering beyond the definitions above.  Threads (pthreads)
 * split independent rows only; each row's arithmetic is sequential.
 *
 * Layout: Q, K, V, dO, O, dQ, dK, dV are [B, H, N, d] row-major doubles;
 * lse is [B, H, N].  fa_oracle_fwd_qk allows a query length Nq different
 * from the key length Nk (Q, O [B, H, Nq, d]; K, V [B, H, Nk, d]; no block
 * mask there): the same definition, row by row.  Its causal mask is aligned
 * to the bottom right: query i keeps key j iff j <= i + (Nk - Nq), so the
 * last query sees every key and Nq == Nk is the top-left rule above (the
 * pages fix only the square case; this is the reading for a query block
 * that continues a longer key sequence).  kv_len is int32[B] (NULL = N;
 * values clamped to [0, N]); block_mask is uint8[nb * nb], nb = ceil(N / blk),
 * one mask shared by every (b, h) (NULL = all ones).
 *
 * fa_oracle_fwd_stats also returns the two row statistics the pages keep in
 * HBM ([EXPL] "Method": the running max m and the exponential sum l of each
 * row): m_i = max_j s_ij and l_i = sum_j exp(s_ij - m_i) over A_i
 * (-inf and 0 for an empty row).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    const double *q, *k, *v, *dout;
    int B, H, N, d;
    int Nk;             /* key rows (= N except in fa_oracle_fwd_qk) */
    double scale;
    int causal;
    int causal_off;     /* causal keeps j <= i + causal_off (Nk - Nq in fa_oracle_fwd_qk) */
    const int32_t *kv_len;
    const uint8_t *block_mask;
    int blk, nb;
    int p8;             /* dropout threshold in 1/256 units; 0 = no dropout */
    uint64_t seed;
    double keep_scale;  /* 256 / (256 - p8) */
} problem;

static void problem_init(problem *p, const double *q, const double *k, const double *v,
                         const double *dout, int B, int H, int N, int d, double scale,
                         int causal, const int32_t *kv_len, const uint8_t *block_mask,
                         int blk) {
    p->q = q; p->k = k; p->v = v; p->dout = dout;
    p->B = B; p->H = H; p->N = N; p->d = d;
    p->Nk = N;
    p->scale = scale; p->causal = causal;
    p->causal_off = 0;
    p->kv_len = kv_len; p->block_mask = block_mask;
    p->blk = blk > 0 ? blk : 128;
    p->nb = (N + p->blk - 1) / p->blk;
    p->p8 = 0;
    p->seed = 0;
    p->keep_scale = 1.0;
}

static void problem_dropout(problem *p, int p8, uint64_t seed) {
    p->p8 = p8;
    p->seed = seed;
    p->keep_scale = 256.0 / (256.0 - (double)p8);
}

/* The PCG hash: one LCG step of the 32-bit PCG generator followed by its
 * RXS-M-XS output permutation (Jarzynski and Olano, JCGT 2020, "pcg"). */
static uint32_t pcg_hash(uint32_t x) {
    const uint32_t state = x * 747796405u + 2891336453u;
    const uint32_t word = ((state >> ((state >> 28) + 4u)) ^ state) * 277803737u;
    return (word >> 22) ^ word;
}

/* Dropout keep mask Z for (head bh, query i, key j): one 32-bit hash per 2x2
 * block of the head, keyed by the seed and the head; the block's four
 * elements take its four bytes.  Kept when the byte is >= p8. */
static int keep(uint64_t seed, int p8, int bh, int i, int j) {
    const uint32_t k0 = pcg_hash((uint32_t)(seed & 0xffffffffu));
    const uint32_t k1 = pcg_hash(k0 ^ (uint32_t)(seed >> 32));
    const uint32_t kb = pcg_hash(k1 ^ (uint32_t)bh);
    const uint32_t ctr = ((uint32_t)(i >> 1) << 16) | (uint32_t)(j >> 1);
    const uint32_t r = pcg_hash(kb ^ ctr);
    const int byte = ((i & 1) << 1) | (j & 1);
    const int u = (int)((r >> (8 * byte)) & 0xffu);
    return u >= p8;
}

/* Z_ij * keep_scale (1 when there is no dropout). */
static double drop_factor(const problem *p, int bh, int i, int j) {
    if (p->p8 == 0) return 1.0;
    return keep(p->seed, p->p8, bh, i, j) ? p->keep_scale : 0.0;
}

/* Key bound of batch b: kv_len[b] clamped to [0, Nk]. */
static int key_bound(const problem *p, int b) {
    if (!p->kv_len) return p->Nk;
    int L = p->kv_len[b];
    if (L < 0) L = 0;
    if (L > p->Nk) L = p->Nk;
    return L;
}

/* Is key j in A_i for batch b? */
static int allowed(const problem *p, int b, int i, int j) {
    if (p->causal && j > i + p->causal_off) return 0;
    if (j >= key_bound(p, b)) return 0;
    if (p->block_mask && !p->block_mask[(size_t)(i / p->blk) * p->nb + (size_t)(j / p->blk)])
        return 0;
    return 1;
}

static const double *row_of(const double *t, const problem *p, int bh, int i) {
    return t + ((size_t)bh * p->N + (size_t)i) * p->d;
}

/* Row j of K or V (Nk rows per head). */
static const double *key_row(const double *t, const problem *p, int bh, int j) {
    return t + ((size_t)bh * p->Nk + (size_t)j) * p->d;
}

static double dot(const double *a, const double *b, int d) {
    double s = 0.0;
    for (int c = 0; c < d; ++c) s += a[c] * b[c];
    return s;
}

/*
 * Forward for one query row: fills s[0..N) (only allowed entries are
 * meaningful), returns m and l through pointers, o[0..d) and lse.
 * Returns the number of allowed keys.
 */
static int forward_row(const problem *p, int bh, int i, double *s, double *m_out,
                       double *l_out, double *o, double *lse) {
    const int b = bh / p->H, d = p->d;
    const double *qi = row_of(p->q, p, bh, i);
    int count = 0;
    double m = -INFINITY;
    /* 1. scores on the allowed set */
    for (int j = 0; j < p->Nk; ++j) {
        if (!allowed(p, b, i, j)) continue;
        s[j] = p->scale * dot(qi, key_row(p->k, p, bh, j), d);
        if (s[j] > m) m = s[j];
        ++count;
    }
    for (int c = 0; c < d; ++c) o[c] = 0.0;
    if (count == 0) {
        *m_out = -INFINITY; *l_out = 0.0; *lse = -INFINITY;
        return 0;
    }
    /* 2.-3. max-shifted exponential sum */
    double l = 0.0;
    for (int j = 0; j < p->Nk; ++j)
        if (allowed(p, b, i, j)) l += exp(s[j] - m);
    /* 4.-5. normalised probabilities (dropped out and rescaled) times V */
    for (int j = 0; j < p->Nk; ++j) {
        if (!allowed(p, b, i, j)) continue;
        const double pij = exp(s[j] - m) / l * drop_factor(p, bh, i, j);
        const double *vj = key_row(p->v, p, bh, j);
        for (int c = 0; c < d; ++c) o[c] += pij * vj[c];
    }
    *m_out = m; *l_out = l;
    /* 6. log-sum-exp in natural log */
    *lse = m + log(l);
    return count;
}

/* ---------------------------------------------------------------- threads */

typedef struct {
    void (*fn)(void *ctx, int64_t item, double *scratch);
    void *ctx;
    int64_t begin, end;
    size_t scratch_len;
    int failed;
} worker_arg;

static void *worker_main(void *varg) {
    worker_arg *a = (worker_arg *)varg;
    double *scratch = NULL;
    if (a->scratch_len) {
        scratch = (double *)malloc(a->scratch_len * sizeof(double));
        if (!scratch) { a->failed = 1; return NULL; }
    }
    for (int64_t it = a->begin; it < a->end; ++it) a->fn(a->ctx, it, scratch);
    free(scratch);
    return NULL;
}

/* Runs fn(ctx, item, scratch) for item in [0, n) over nthreads threads. */
static int parallel_for(int64_t n, int nthreads, size_t scratch_len,
                        void (*fn)(void *, int64_t, double *), void *ctx) {
    if (n <= 0) return 0;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    if ((int64_t)nthreads > n) nthreads = (int)n;
    pthread_t tids[256];
    worker_arg args[256];
    int started = 0, rc = 0;
    for (int t = 0; t < nthreads; ++t) {
        args[t].fn = fn; args[t].ctx = ctx;
        args[t].begin = n * t / nthreads;
        args[t].end = n * (t + 1) / nthreads;
        args[t].scratch_len = scratch_len;
        args[t].failed = 0;
    }
    for (int t = 1; t < nthreads; ++t) {
        if (pthread_create(&tids[t], NULL, worker_main, &args[t]) != 0) { rc = -2; break; }
        started = t;
    }
    worker_main(&args[0]);
    for (int t = 1; t <= started; ++t) pthread_join(tids[t], NULL);
    if (rc == 0 && started != nthreads - 1) rc = -2;
    for (int t = 0; t < nthreads; ++t)
        if (args[t].failed) rc = -3;
    if (rc == -2) {
        /* thread creation failed part-way: finish the missing ranges here */
        for (int t = started + 1; t < nthreads; ++t) worker_main(&args[t]);
        rc = 0;
        for (int t = 0; t < nthreads; ++t)
            if (args[t].failed) rc = -3;
    }
    return rc;
}

/* ---------------------------------------------------------------- forward */

typedef struct {
    const problem *p;
    const int64_t *rows; /* global row ids bh * N + i, or NULL = all */
    double *o, *lse;
    double *m, *l;       /* optional row statistics */
} fwd_ctx;

static void fwd_item(void *vctx, int64_t item, double *s) {
    fwd_ctx *c = (fwd_ctx *)vctx;
    const problem *p = c->p;
    const int64_t g = c->rows ? c->rows[item] : item;
    const int bh = (int)(g / p->N), i = (int)(g % p->N);
    double m, l;
    forward_row(p, bh, i, s, &m, &l, c->o + (size_t)item * p->d, c->lse + item);
    if (c->m) c->m[item] = m;
    if (c->l) c->l[item] = l;
}

/*
 * Forward on selected rows.  rows[r] = bh * N + i selects query row i of
 * head bh (NULL selects every row, in order).  o is [nrows, d], lse [nrows].
 * Returns 0 on success, a negative value on bad arguments / no memory.
 */
int fa_oracle_fwd_dropout(const double *q, const double *k, const double *v, int B, int H,
                          int N, int d, double scale, int causal, const int32_t *kv_len,
                          const uint8_t *block_mask, int blk, int p8, uint64_t seed,
                          const int64_t *rows, int64_t nrows, double *o, double *lse,
                          int nthreads) {
    if (!q || !k || !v || !o || !lse || B < 1 || H < 1 || N < 1 || d < 1) return -1;
    if (p8 < 0 || p8 > 255) return -1;
    problem p;
    problem_init(&p, q, k, v, NULL, B, H, N, d, scale, causal, kv_len, block_mask, blk);
    problem_dropout(&p, p8, seed);
    const int64_t total = (int64_t)B * H * N;
    if (!rows) nrows = total;
    for (int64_t r = 0; rows && r < nrows; ++r)
        if (rows[r] < 0 || rows[r] >= total) return -1;
    fwd_ctx c = {&p, rows, o, lse, NULL, NULL};
    return parallel_for(nrows, nthreads, (size_t)N, fwd_item, &c);
}

/* fa_oracle_fwd plus the row statistics m [nrows] and l [nrows]. */
int fa_oracle_fwd_stats(const double *q, const double *k, const double *v, int B, int H,
                        int N, int d, double scale, int causal, const int32_t *kv_len,
                        const uint8_t *block_mask, int blk, const int64_t *rows, int64_t nrows,
                        double *o, double *lse, double *m, double *l, int nthreads) {
    if (!q || !k || !v || !o || !lse || !m || !l || B < 1 || H < 1 || N < 1 || d < 1) return -1;
    problem p;
    problem_init(&p, q, k, v, NULL, B, H, N, d, scale, causal, kv_len, block_mask, blk);
    const int64_t total = (int64_t)B * H * N;
    if (!rows) nrows = total;
    for (int64_t r = 0; rows && r < nrows; ++r)
        if (rows[r] < 0 || rows[r] >= total) return -1;
    fwd_ctx c = {&p, rows, o, lse, m, l};
    return parallel_for(nrows, nthreads, (size_t)N, fwd_item, &c);
}

int fa_oracle_fwd(const double *q, const double *k, const double *v, int B, int H, int N,
                  int d, double scale, int causal, const int32_t *kv_len,
                  const uint8_t *block_mask, int blk, const int64_t *rows, int64_t nrows,
                  double *o, double *lse, int nthreads) {
    return fa_oracle_fwd_dropout(q, k, v, B, H, N, d, scale, causal, kv_len, block_mask, blk, 0,
                                 0, rows, nrows, o, lse, nthreads);
}

/*
 * Forward with a query length Nq and a key length Nk (no block mask; kv_len
 * clamped to [0, Nk]; causal aligned to the bottom right, see the top of the
 * file): q [B, H, Nq, d], k and v [B, H, Nk, d]; rows as in fa_oracle_fwd
 * with ids bh * Nq + i; o [nrows, d], lse [nrows].
 */
int fa_oracle_fwd_qk(const double *q, const double *k, const double *v, int B, int H, int Nq,
                     int Nk, int d, double scale, int causal, const int32_t *kv_len,
                     const int64_t *rows, int64_t nrows, double *o, double *lse, int nthreads) {
    if (!q || !k || !v || !o || !lse || B < 1 || H < 1 || Nq < 1 || Nk < 1 || d < 1) return -1;
    problem p;
    problem_init(&p, q, k, v, NULL, B, H, Nq, d, scale, causal, kv_len, NULL, 128);
    p.Nk = Nk;
    p.causal_off = Nk - Nq;
    const int64_t total = (int64_t)B * H * Nq;
    if (!rows) nrows = total;
    for (int64_t r = 0; rows && r < nrows; ++r)
        if (rows[r] < 0 || rows[r] >= total) return -1;
    fwd_ctx cx = {&p, rows, o, lse, NULL, NULL};
    return parallel_for(nrows, nthreads, (size_t)Nk, fwd_item, &cx);
}

/* The dropout keep mask Z_ij (1 kept, 0 dropped) of head bh. */
int fa_oracle_keep(uint64_t seed, int p8, int bh, int i, int j) {
    return keep(seed, p8, bh, i, j);
}

/*
 * Dense probabilities of one head (tiny problems only): P[i * N + j] =
 * exp(s_ij - m_i) / l_i on the allowed set, exactly 0 elsewhere.
 */
int fa_oracle_probs(const double *q, const double *k, int B, int H, int N, int d,
                    double scale, int causal, const int32_t *kv_len,
                    const uint8_t *block_mask, int blk, int bh, double *P) {
    if (!q || !k || !P || bh < 0 || bh >= B * H || d < 1 || N < 1) return -1;
    problem p;
    /* V is not read by this routine; pass Q as a placeholder */
    problem_init(&p, q, k, q, NULL, B, H, N, d, scale, causal, kv_len, block_mask, blk);
    const int b = bh / H;
    double *s = (double *)malloc((size_t)N * sizeof(double));
    if (!s) return -3;
    for (int i = 0; i < N; ++i) {
        double m = -INFINITY;
        int count = 0;
        for (int j = 0; j < N; ++j) {
            P[(size_t)i * N + j] = 0.0;
            if (!allowed(&p, b, i, j)) continue;
            s[j] = scale * dot(row_of(q, &p, bh, i), row_of(k, &p, bh, j), d);
            if (s[j] > m) m = s[j];
            ++count;
        }
        if (!count) continue;
        double l = 0.0;
        for (int j = 0; j < N; ++j)
            if (allowed(&p, b, i, j)) l += exp(s[j] - m);
        for (int j = 0; j < N; ++j)
            if (allowed(&p, b, i, j)) P[(size_t)i * N + j] = exp(s[j] - m) / l;
    }
    free(s);
    return 0;
}

/* ------------------------------------------------------- tiled forward */

/*
 * The pages' tiled forward, in their order and notation ([EXPL] "Method",
 * online softmax tracking and steps 1-4; [MATH] section 7, stateful
 * streaming computation; [BLOG] online-softmax pseudocode).  Query rows are
 * taken in blocks of Br and key/value rows in blocks of Bc.  For block pair
 * (i, j):
 *   1. S_ij = scale * Q_i K_j^T on the allowed entries (others excluded),
 *   2. mt_ij = rowmax(S_ij), Pt_ij = exp(S_ij - mt_ij), lt_ij = rowsum(Pt_ij),
 *   3. m_new = max(m, mt_ij),
 *      l_new = exp(m - m_new) l + exp(mt_ij - m_new) lt_ij,
 *   4. O_i <- diag(l_new)^-1 (diag(l) exp(m - m_new) O_i
 *                             + exp(mt_ij - m_new) Pt_ij V_j),
 * and finally lse = m + ln l.  This is not used as the reference for the
 * GPU; its only job is to pin, by testing, that the streaming merge equals
 * the one-shot definition above for every block split.
 */
int fa_oracle_fwd_tiled(const double *q, const double *k, const double *v, int B, int H,
                        int N, int d, double scale, int causal, const int32_t *kv_len,
                        const uint8_t *block_mask, int blk, int Br, int Bc, double *o,
                        double *lse) {
    if (!q || !k || !v || !o || !lse || Br < 1 || Bc < 1 || d < 1 || N < 1) return -1;
    problem p;
    problem_init(&p, q, k, v, NULL, B, H, N, d, scale, causal, kv_len, block_mask, blk);
    double *S = (double *)malloc((size_t)Br * Bc * sizeof(double));
    double *Pt = (double *)malloc((size_t)Br * Bc * sizeof(double));
    double *mrow = (double *)malloc((size_t)Br * sizeof(double));
    double *lrow = (double *)malloc((size_t)Br * sizeof(double));
    double *Oi = (double *)malloc((size_t)Br * d * sizeof(double));
    if (!S || !Pt || !mrow || !lrow || !Oi) {
        free(S); free(Pt); free(mrow); free(lrow); free(Oi);
        return -3;
    }
    for (int bh = 0; bh < B * H; ++bh) {
        const int b = bh / H;
        for (int i0 = 0; i0 < N; i0 += Br) {
            const int nr = (N - i0 < Br) ? N - i0 : Br;
            /* initialise the state: m = -inf, l = 0, O = 0 */
            for (int r = 0; r < nr; ++r) {
                mrow[r] = -INFINITY; lrow[r] = 0.0;
                for (int c = 0; c < d; ++c) Oi[(size_t)r * d + c] = 0.0;
            }
            for (int j0 = 0; j0 < N; j0 += Bc) {
                const int nc = (N - j0 < Bc) ? N - j0 : Bc;
                for (int r = 0; r < nr; ++r) {
                    const int i = i0 + r;
                    /* step 1 */
                    double mt = -INFINITY;
                    for (int cc = 0; cc < nc; ++cc) {
                        const int j = j0 + cc;
                        if (!allowed(&p, b, i, j)) { S[r * Bc + cc] = -INFINITY; continue; }
                        S[r * Bc + cc] = scale * dot(row_of(q, &p, bh, i), row_of(k, &p, bh, j), d);
                        if (S[r * Bc + cc] > mt) mt = S[r * Bc + cc];
                    }
                    if (mt == -INFINITY) continue; /* nothing allowed in this block */
                    /* step 2 */
                    double lt = 0.0;
                    for (int cc = 0; cc < nc; ++cc) {
                        Pt[r * Bc + cc] = (S[r * Bc + cc] == -INFINITY) ? 0.0 : exp(S[r * Bc + cc] - mt);
                        lt += Pt[r * Bc + cc];
                    }
                    /* step 3 */
                    const double m_old = mrow[r], l_old = lrow[r];
                    const double m_new = (m_old > mt) ? m_old : mt;
                    const double a_old = (m_old == -INFINITY) ? 0.0 : exp(m_old - m_new);
                    const double a_new = exp(mt - m_new);
                    const double l_new = a_old * l_old + a_new * lt;
                    /* step 4 */
                    for (int c = 0; c < d; ++c) {
                        double pv = 0.0;
                        for (int cc = 0; cc < nc; ++cc)
                            pv += Pt[r * Bc + cc] * row_of(v, &p, bh, j0 + cc)[c];
                        Oi[(size_t)r * d + c] =
                            (l_old * a_old * Oi[(size_t)r * d + c] + a_new * pv) / l_new;
                    }
                    mrow[r] = m_new; lrow[r] = l_new;
                }
            }
            for (int r = 0; r < nr; ++r) {
                const size_t g = (size_t)bh * N + (size_t)(i0 + r);
                for (int c = 0; c < d; ++c) o[g * d + c] = Oi[(size_t)r * d + c];
                lse[g] = (lrow[r] > 0.0) ? mrow[r] + log(lrow[r]) : -INFINITY;
            }
        }
    }
    free(S); free(Pt); free(mrow); free(lrow); free(Oi);
    return 0;
}

/* ---------------------------------------------------------------- backward */

typedef struct {
    const problem *p;
    /* per-row forward statistics of the rows the key gradients need */
    const int64_t *fwd_rows;  /* sorted global rows with stats below */
    int64_t nfwd;
    double *fm, *fl, *fo, *fD; /* m, l, o[d], D = <dO, o> per fwd row */
    const int64_t *q_rows;
    double *dq;
    const int64_t *k_rows;
    double *dk, *dv;
    const int64_t *row_index; /* global row -> index in fwd_rows, or -1 */
} bwd_ctx;

/* Statistics (m, l, o, D) for one forward row. */
static void stats_item(void *vctx, int64_t item, double *s) {
    bwd_ctx *c = (bwd_ctx *)vctx;
    const problem *p = c->p;
    const int64_t g = c->fwd_rows[item];
    const int bh = (int)(g / p->N), i = (int)(g % p->N);
    double lse;
    double *o = c->fo + (size_t)item * p->d;
    forward_row(p, bh, i, s, &c->fm[item], &c->fl[item], o, &lse);
    c->fD[item] = dot(row_of(p->dout, p, bh, i), o, p->d);
}

/* dQ_i = scale * sum_j dS_ij k_j, dS_ij = P_ij (dP_ij - D_i), dP_ij = <dO_i, v_j>. */
static void dq_item(void *vctx, int64_t item, double *s) {
    bwd_ctx *c = (bwd_ctx *)vctx;
    const problem *p = c->p;
    const int64_t g = c->q_rows ? c->q_rows[item] : item;
    const int bh = (int)(g / p->N), i = (int)(g % p->N), b = bh / p->H, d = p->d;
    const int64_t fi = c->row_index[g];
    double *dq = c->dq + (size_t)item * d;
    for (int cc = 0; cc < d; ++cc) dq[cc] = 0.0;
    const double m = c->fm[fi], l = c->fl[fi], D = c->fD[fi];
    if (l <= 0.0) return;
    const double *qi = row_of(p->q, p, bh, i), *doi = row_of(p->dout, p, bh, i);
    (void)s;
    for (int j = 0; j < p->Nk; ++j) {
        if (!allowed(p, b, i, j)) continue;
        const double sij = p->scale * dot(qi, key_row(p->k, p, bh, j), d);
        const double pij = exp(sij - m) / l;
        const double dpij = dot(doi, key_row(p->v, p, bh, j), d);
        const double dsij = pij * (drop_factor(p, bh, i, j) * dpij - D);
        const double *kj = key_row(p->k, p, bh, j);
        for (int cc = 0; cc < d; ++cc) dq[cc] += p->scale * dsij * kj[cc];
    }
}

/* dV_j = sum_i P_ij dO_i ; dK_j = scale * sum_i dS_ij q_i. */
static void dkdv_item(void *vctx, int64_t item, double *s) {
    bwd_ctx *c = (bwd_ctx *)vctx;
    const problem *p = c->p;
    const int64_t g = c->k_rows ? c->k_rows[item] : item;
    const int bh = (int)(g / p->Nk), j = (int)(g % p->Nk), b = bh / p->H, d = p->d;
    double *dk = c->dk + (size_t)item * d, *dv = c->dv + (size_t)item * d;
    for (int cc = 0; cc < d; ++cc) { dk[cc] = 0.0; dv[cc] = 0.0; }
    const double *kj = key_row(p->k, p, bh, j), *vj = key_row(p->v, p, bh, j);
    (void)s;
    for (int i = 0; i < p->N; ++i) {
        if (!allowed(p, b, i, j)) continue;
        const int64_t fi = c->row_index[(int64_t)bh * p->N + i];
        const double m = c->fm[fi], l = c->fl[fi], D = c->fD[fi];
        const double *qi = row_of(p->q, p, bh, i), *doi = row_of(p->dout, p, bh, i);
        const double sij = p->scale * dot(qi, kj, d);
        const double pij = exp(sij - m) / l;
        const double dpij = dot(doi, vj, d);
        const double zc = drop_factor(p, bh, i, j);
        const double dsij = pij * (zc * dpij - D);
        for (int cc = 0; cc < d; ++cc) {
            dv[cc] += pij * zc * doi[cc];
            dk[cc] += p->scale * dsij * qi[cc];
        }
    }
}

/*
 * The backward of the problem with N query rows and Nk key rows (causal kept
 * j <= i + Nk - N, the bottom-right rule, which is the top-left one when
 * N = Nk); q_rows are global query rows bh * N + i, k_rows global key rows
 * bh * Nk + j.
 */
static int bwd_general(const double *q, const double *k, const double *v, const double *dout,
                       int B, int H, int N, int Nk, int d, double scale, int causal,
                       const int32_t *kv_len, const uint8_t *block_mask, int blk, int p8,
                       uint64_t seed, const int64_t *q_rows, int64_t nq, const int64_t *k_rows,
                       int64_t nk, double *dq, double *dk, double *dv, int nthreads) {
    if (!q || !k || !v || !dout || B < 1 || H < 1 || N < 1 || Nk < 1 || d < 1) return -1;
    if (p8 < 0 || p8 > 255) return -1;
    if ((nq != 0 || !q_rows) && !dq) return -1;
    if ((nk != 0 || !k_rows) && (!dk || !dv)) return -1;
    problem p;
    problem_init(&p, q, k, v, dout, B, H, N, d, scale, causal, kv_len, block_mask, blk);
    p.Nk = Nk;
    p.causal_off = Nk - N;
    problem_dropout(&p, p8, seed);
    const int64_t total = (int64_t)B * H * N, total_k = (int64_t)B * H * Nk;
    if (!q_rows) nq = total;
    if (!k_rows) nk = total_k;
    for (int64_t r = 0; q_rows && r < nq; ++r)
        if (q_rows[r] < 0 || q_rows[r] >= total) return -1;
    for (int64_t r = 0; k_rows && r < nk; ++r)
        if (k_rows[r] < 0 || k_rows[r] >= total_k) return -1;

    /* mark the query rows whose forward statistics are needed */
    uint8_t *need = (uint8_t *)calloc((size_t)total, 1);
    int64_t *row_index = (int64_t *)malloc((size_t)total * sizeof(int64_t));
    if (!need || !row_index) { free(need); free(row_index); return -3; }
    for (int64_t r = 0; r < nq; ++r) need[q_rows ? q_rows[r] : r] = 1;
    /* key-side needs: every query row of the head that attends to a selected key */
    uint8_t *key_sel = (uint8_t *)calloc((size_t)total_k, 1);
    if (!key_sel) { free(need); free(row_index); return -3; }
    for (int64_t r = 0; r < nk; ++r) key_sel[k_rows ? k_rows[r] : r] = 1;
    int *sel = (int *)malloc((size_t)Nk * sizeof(int));
    if (!sel) { free(need); free(row_index); free(key_sel); return -3; }
    for (int bh = 0; bh < B * H; ++bh) {
        const int b = bh / H;
        int nsel = 0;
        for (int j = 0; j < Nk; ++j)
            if (key_sel[(size_t)bh * Nk + j]) sel[nsel++] = j;
        if (!nsel) continue;
        for (int i = 0; i < N; ++i) {
            if (need[(size_t)bh * N + i]) continue;
            for (int t = 0; t < nsel; ++t)
                if (allowed(&p, b, i, sel[t])) {
                    need[(size_t)bh * N + i] = 1;
                    break;
                }
        }
    }
    free(sel);
    free(key_sel);
    int64_t nfwd = 0;
    for (int64_t g = 0; g < total; ++g) row_index[g] = need[g] ? nfwd++ : -1;
    int64_t *fwd_rows = (int64_t *)malloc((size_t)(nfwd ? nfwd : 1) * sizeof(int64_t));
    double *fm = (double *)malloc((size_t)(nfwd ? nfwd : 1) * sizeof(double));
    double *fl = (double *)malloc((size_t)(nfwd ? nfwd : 1) * sizeof(double));
    double *fD = (double *)malloc((size_t)(nfwd ? nfwd : 1) * sizeof(double));
    double *fo = (double *)malloc((size_t)(nfwd ? nfwd : 1) * d * sizeof(double));
    int rc = 0;
    if (!fwd_rows || !fm || !fl || !fD || !fo) { rc = -3; goto done; }
    for (int64_t g = 0; g < total; ++g)
        if (need[g]) fwd_rows[row_index[g]] = g;
    {
        bwd_ctx c;
        memset(&c, 0, sizeof c);
        c.p = &p; c.fwd_rows = fwd_rows; c.nfwd = nfwd;
        c.fm = fm; c.fl = fl; c.fo = fo; c.fD = fD;
        c.q_rows = q_rows; c.dq = dq; c.k_rows = k_rows; c.dk = dk; c.dv = dv;
        c.row_index = row_index;
        rc = parallel_for(nfwd, nthreads, (size_t)Nk, stats_item, &c);
        if (rc == 0) rc = parallel_for(nq, nthreads, 0, dq_item, &c);
        if (rc == 0) rc = parallel_for(nk, nthreads, 0, dkdv_item, &c);
    }
done:
    free(need); free(row_index); free(fwd_rows); free(fm); free(fl); free(fD); free(fo);
    return rc;
}

/*
 * Backward on selected rows.  q_rows (global bh * N + i, NULL = all) select
 * the dQ rows written to dq [nq, d]; k_rows (global bh * N + j, NULL = all)
 * select the key rows whose dK, dV go to dk, dv [nk, d].  The forward
 * statistics are recomputed here from the definition for exactly the query
 * rows that are needed (the dQ rows, plus every row that attends to one of
 * the selected keys).
 */
int fa_oracle_bwd_dropout(const double *q, const double *k, const double *v,
                          const double *dout, int B, int H, int N, int d, double scale,
                          int causal, const int32_t *kv_len, const uint8_t *block_mask, int blk,
                          int p8, uint64_t seed, const int64_t *q_rows, int64_t nq,
                          const int64_t *k_rows, int64_t nk, double *dq, double *dk,
                          double *dv, int nthreads) {
    return bwd_general(q, k, v, dout, B, H, N, N, d, scale, causal, kv_len, block_mask, blk, p8,
                       seed, q_rows, nq, k_rows, nk, dq, dk, dv, nthreads);
}

/*
 * Backward with Nq query rows and Nk key rows (no block mask, no dropout;
 * causal aligned to the bottom right as in fa_oracle_fwd_qk): q, dout
 * [B, H, Nq, d]; k, v [B, H, Nk, d]; q_rows are bh * Nq + i, k_rows
 * bh * Nk + j.
 */
int fa_oracle_bwd_qk(const double *q, const double *k, const double *v, const double *dout,
                     int B, int H, int Nq, int Nk, int d, double scale, int causal,
                     const int32_t *kv_len, const int64_t *q_rows, int64_t nq,
                     const int64_t *k_rows, int64_t nk, double *dq, double *dk, double *dv,
                     int nthreads) {
    return bwd_general(q, k, v, dout, B, H, Nq, Nk, d, scale, causal, kv_len, NULL, 128, 0, 0,
                       q_rows, nq, k_rows, nk, dq, dk, dv, nthreads);
}

int fa_oracle_bwd(const double *q, const double *k, const double *v, const double *dout,
                  int B, int H, int N, int d, double scale, int causal,
                  const int32_t *kv_len, const uint8_t *block_mask, int blk,
                  const int64_t *q_rows, int64_t nq, const int64_t *k_rows, int64_t nk,
                  double *dq, double *dk, double *dv, int nthreads) {
    return fa_oracle_bwd_dropout(q, k, v, dout, B, H, N, d, scale, causal, kv_len, block_mask,
                                 blk, 0, 0, q_rows, nq, k_rows, nk, dq, dk, dv, nthreads);
}
