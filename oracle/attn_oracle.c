/*
 * Exact scaled-dot-product attention: plain fp64 CPU oracle.
 *
 * TEST INFRASTRUCTURE. Only the test suite, the smoke check and the CPU-baseline
 * leg of the benchmark may load this file's library. The product path (the CUDA
 * library and its Python binding) never calls it, shares no code with it and
 * never falls back to it.
 *
 * Everything here is written for a reader checking it against the pages by eye:
 * no tiling beyond what a function's definition states, no fusion, no reordering.
 * All arithmetic is in double precision. Inputs are double arrays (callers pass
 * the bf16 values the GPU sees, widened exactly to double).
 *
 * Pages cited (by title and section):
 *   [MAK]  "Modern attention kernels" (blog.ecitis.org)
 *   [FAV]  "Flash attention" (understandingdata.com, AI engineering visualised)
 *   [IOA]  "Flash attention and IO-aware attention" (aigrafen.se)
 *   [AK]   "Attention kernels" (inference.tusharamrit.in)
 *
 * Layouts (row-major, contiguous):
 *   q, o : [B][Hq][Nq][d]      k, v : [B][Hkv][Nk][d]      lse : [B][Hq][Nq]
 *   FP8 variant: 8-bit E4M3 codes, V transposed (see oracle_attn_fwd_fp8)
 *   paged caches : [num_blocks][Hkv][block_size][d]
 *   block_table  : int32 [num_seqs][max_blocks_per_seq]
 *
 * Readings taken where the pages are silent:
 *   - causal alignment is bottom-right: row i may see key j iff j <= i + (Nk - Nq);
 *   - window w >= 0 adds the left limit j >= i + (Nk - Nq) - w (w < 0: no limit);
 *   - query head h reads kv head h / (Hq / Hkv) (contiguous groups);
 *   - a row with no allowed key has O = 0 and lse = -inf;
 *   - lse is the natural log of the sum of exp over the scaled scores.
 *
 * Every function returns 0 on success and a negative value on invalid arguments.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_OK 0
#define ORACLE_EINVAL (-1)
#define ORACLE_ENOMEM (-2)
#define ORACLE_EBOUNDS (-3)

/* ------------------------------------------------------------------------- */
/* Mask: which keys a query row may attend.                                   */
/* [MAK] "Kernel structure": causal attention keeps keys up to the diagonal;   */
/* local attention limits how far left a row may look.                         */
/* ------------------------------------------------------------------------- */
static int key_allowed(long i, long j, long Nq, long Nk, int causal, int window)
{
    long diag = i + (Nk - Nq);
    if (j < 0 || j >= Nk) return 0;
    if (causal && j > diag) return 0;
    if (window >= 0 && j < diag - (long)window) return 0;
    return 1;
}

static double dot(const double* a, const double* b, int d)
{
    double s = 0.0;
    for (int t = 0; t < d; ++t) s += a[t] * b[t];
    return s;
}

static int check_dims(int B, int Hq, int Hkv, int Nq, int Nk, int d)
{
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Nq < 0 || Nk < 0 || d <= 0) return ORACLE_EINVAL;
    if (Hq % Hkv != 0) return ORACLE_EINVAL;
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------- */
/* One query row, materialised.                                                */
/* [MAK] "Standard attention materializes quadratic state": S = Q K^T / sqrt d, */
/*   P = softmax(S), O = P V  (here with an explicit scale argument).          */
/* [AK] safe softmax: m = max(x), l = sum exp(x - m), y = exp(x - m) / l.       */
/* The whole score row s[] and probability row p[] are formed before O.        */
/* ------------------------------------------------------------------------- */
static void attend_row_materialised(const double* qi, const double* kh, const double* vh,
                                    long i, long Nq, long Nk, int d, double scale,
                                    int causal, int window,
                                    double* s, double* p, double* oi, double* lse_i)
{
    /* scores S_ij (masked entries are -inf) */
    double m = -INFINITY;
    for (long j = 0; j < Nk; ++j) {
        if (key_allowed(i, j, Nq, Nk, causal, window))
            s[j] = scale * dot(qi, kh + j * d, d);
        else
            s[j] = -INFINITY;
        if (s[j] > m) m = s[j];
    }
    for (int t = 0; t < d; ++t) oi[t] = 0.0;
    if (m == -INFINITY) {            /* empty row */
        *lse_i = -INFINITY;
        return;
    }
    /* safe softmax: subtract the row max, exponentiate, divide by the sum */
    double l = 0.0;
    for (long j = 0; j < Nk; ++j) {
        p[j] = (s[j] == -INFINITY) ? 0.0 : exp(s[j] - m);
        l += p[j];
    }
    for (long j = 0; j < Nk; ++j) p[j] /= l;
    /* O = P V */
    for (long j = 0; j < Nk; ++j) {
        if (p[j] == 0.0) continue;
        const double* vj = vh + j * d;
        for (int t = 0; t < d; ++t) oi[t] += p[j] * vj[t];
    }
    *lse_i = m + log(l);
}

/* Materialised attention for a list of (b, hq, i) rows.
 * rows: int64 [nrows][3]; o_rows: [nrows][d]; lse_rows: [nrows]. */
int oracle_attn_fwd_rows(const double* q, const double* k, const double* v,
                         int B, int Hq, int Hkv, int Nq, int Nk, int d,
                         double scale, int causal, int window,
                         const int64_t* rows, int64_t nrows,
                         double* o_rows, double* lse_rows)
{
    if (check_dims(B, Hq, Hkv, Nq, Nk, d)) return ORACLE_EINVAL;
    int G = Hq / Hkv;
    for (int64_t r = 0; r < nrows; ++r) {
        if (rows[3 * r] < 0 || rows[3 * r] >= B || rows[3 * r + 1] < 0 || rows[3 * r + 1] >= Hq ||
            rows[3 * r + 2] < 0 || rows[3 * r + 2] >= Nq)
            return ORACLE_EINVAL;
    }
    int err = ORACLE_OK;
#pragma omp parallel
    {
        double* s = (double*)malloc(sizeof(double) * (size_t)(Nk > 0 ? Nk : 1));
        double* p = (double*)malloc(sizeof(double) * (size_t)(Nk > 0 ? Nk : 1));
        if (!s || !p) {
#pragma omp atomic write
            err = ORACLE_ENOMEM;
        } else {
#pragma omp for schedule(dynamic, 16)
            for (int64_t r = 0; r < nrows; ++r) {
                long b = (long)rows[3 * r], h = (long)rows[3 * r + 1], i = (long)rows[3 * r + 2];
                long hk = h / G;  /* contiguous query-head groups share one kv head */
                const double* qi = q + (((b * Hq + h) * (long)Nq + i) * d);
                const double* kh = k + ((b * Hkv + hk) * (long)Nk * d);
                const double* vh = v + ((b * Hkv + hk) * (long)Nk * d);
                attend_row_materialised(qi, kh, vh, i, Nq, Nk, d, scale, causal, window,
                                        s, p, o_rows + r * d, lse_rows + r);
            }
        }
        free(s);
        free(p);
    }
    return err;
}

/* Materialised attention over every row. */
int oracle_attn_fwd(const double* q, const double* k, const double* v, double* o, double* lse,
                    int B, int Hq, int Hkv, int Nq, int Nk, int d,
                    double scale, int causal, int window)
{
    if (check_dims(B, Hq, Hkv, Nq, Nk, d)) return ORACLE_EINVAL;
    int64_t nrows = (int64_t)B * Hq * Nq;
    int64_t* rows = (int64_t*)malloc(sizeof(int64_t) * 3 * (size_t)(nrows > 0 ? nrows : 1));
    if (!rows) return ORACLE_ENOMEM;
    int64_t r = 0;
    for (int b = 0; b < B; ++b)
        for (int h = 0; h < Hq; ++h)
            for (int i = 0; i < Nq; ++i) {
                rows[3 * r] = b; rows[3 * r + 1] = h; rows[3 * r + 2] = i; ++r;
            }
    int rc = oracle_attn_fwd_rows(q, k, v, B, Hq, Hkv, Nq, Nk, d, scale, causal, window,
                                  rows, nrows, o, lse);
    free(rows);
    return rc;
}

/* ------------------------------------------------------------------------- */
/* Blocked online-softmax variant.                                             */
/* [IOA] code listing (blocked online-softmax function): the query block is    */
/*   the outer loop; for every key/value block the running max m, running sum  */
/*   l and running output o are corrected by exp(m - m_new) and extended.      */
/* [MAK] "Online softmax makes tiling exact": m' = max(m, m_b),                */
/*   l' = e^{m-m'} l + sum_j e^{s_j - m'},  o' = e^{m-m'} o + sum_j e^{s_j-m'} v_j, */
/*   and after the final tile the output is o / l.                             */
/* Reading for the -inf start state: while nothing has been seen (m = -inf)    */
/*   the correction factor is 0, not e^{-inf - (-inf)}.                        */
/* ------------------------------------------------------------------------- */
int oracle_attn_fwd_blocked(const double* q, const double* k, const double* v, double* o, double* lse,
                            int B, int Hq, int Hkv, int Nq, int Nk, int d,
                            double scale, int causal, int window, int block_r, int block_c)
{
    if (check_dims(B, Hq, Hkv, Nq, Nk, d) || block_r <= 0 || block_c <= 0) return ORACLE_EINVAL;
    int G = Hq / Hkv;
    long n_rblocks = (Nq + block_r - 1) / block_r;
    int err = ORACLE_OK;
#pragma omp parallel
    {
        double* m = (double*)malloc(sizeof(double) * (size_t)block_r);
        double* l = (double*)malloc(sizeof(double) * (size_t)block_r);
        double* acc = (double*)malloc(sizeof(double) * (size_t)block_r * d);
        double* s = (double*)malloc(sizeof(double) * (size_t)block_c);
        if (!m || !l || !acc || !s) {
#pragma omp atomic write
            err = ORACLE_ENOMEM;
        } else {
#pragma omp for schedule(dynamic, 1) collapse(2)
            for (long bh = 0; bh < (long)B * Hq; ++bh) {
                for (long rb = 0; rb < n_rblocks; ++rb) {
                    long b = bh / Hq, h = bh % Hq, hk = h / G;
                    const double* kh = k + ((b * Hkv + hk) * (long)Nk * d);
                    const double* vh = v + ((b * Hkv + hk) * (long)Nk * d);
                    long i0 = rb * block_r;
                    long i1 = i0 + block_r < Nq ? i0 + block_r : Nq;
                    /* initialise the running state of this query block */
                    for (long i = i0; i < i1; ++i) {
                        m[i - i0] = -INFINITY;
                        l[i - i0] = 0.0;
                        for (int t = 0; t < d; ++t) acc[(i - i0) * d + t] = 0.0;
                    }
                    /* sweep the key/value blocks */
                    for (long j0 = 0; j0 < Nk; j0 += block_c) {
                        long j1 = j0 + block_c < Nk ? j0 + block_c : Nk;
                        for (long i = i0; i < i1; ++i) {
                            const double* qi = q + (((b * Hq + h) * (long)Nq + i) * d);
                            double* oi = acc + (i - i0) * d;
                            double m_b = -INFINITY;
                            for (long j = j0; j < j1; ++j) {
                                s[j - j0] = key_allowed(i, j, Nq, Nk, causal, window)
                                                ? scale * dot(qi, kh + j * d, d) : -INFINITY;
                                if (s[j - j0] > m_b) m_b = s[j - j0];
                            }
                            double m_old = m[i - i0];
                            double m_new = m_b > m_old ? m_b : m_old;
                            if (m_new == -INFINITY) continue;   /* nothing allowed so far */
                            double corr = (m_old == -INFINITY) ? 0.0 : exp(m_old - m_new);
                            double lsum = 0.0;
                            for (int t = 0; t < d; ++t) oi[t] *= corr;
                            for (long j = j0; j < j1; ++j) {
                                if (s[j - j0] == -INFINITY) continue;
                                double pj = exp(s[j - j0] - m_new);
                                lsum += pj;
                                const double* vj = vh + j * d;
                                for (int t = 0; t < d; ++t) oi[t] += pj * vj[t];
                            }
                            l[i - i0] = corr * l[i - i0] + lsum;
                            m[i - i0] = m_new;
                        }
                    }
                    /* deferred normalisation: divide by l once, after the last tile */
                    for (long i = i0; i < i1; ++i) {
                        double* oo = o + (((b * Hq + h) * (long)Nq + i) * d);
                        double li = l[i - i0];
                        for (int t = 0; t < d; ++t) oo[t] = li > 0.0 ? acc[(i - i0) * d + t] / li : 0.0;
                        lse[(b * Hq + h) * (long)Nq + i] = li > 0.0 ? m[i - i0] + log(li) : -INFINITY;
                    }
                }
            }
        }
        free(m); free(l); free(acc); free(s);
    }
    return err;
}

/* ------------------------------------------------------------------------- */
/* Split-KV variant with the two-partial merge.                                */
/* [AK] FlashDecoding: the keys of a row are cut into chunks; each chunk gives */
/*   a partial output O_c together with that chunk's m_c and l_c; these are   */
/*   merged with the same rescaling:                                           */
/*     m = max_c m_c,  l = sum_c l_c e^{m_c - m},                              */
/*     O = sum_c O_c (l_c e^{m_c - m} / l).                                    */
/* Each chunk is a materialised safe softmax over its own keys.                */
/* ------------------------------------------------------------------------- */
int oracle_attn_fwd_split(const double* q, const double* k, const double* v, double* o, double* lse,
                          int B, int Hq, int Hkv, int Nq, int Nk, int d,
                          double scale, int causal, int window, int chunk)
{
    if (check_dims(B, Hq, Hkv, Nq, Nk, d) || chunk <= 0) return ORACLE_EINVAL;
    int G = Hq / Hkv;
    long n_chunks = (Nk + chunk - 1) / chunk;
    int err = ORACLE_OK;
#pragma omp parallel
    {
        double* mc = (double*)malloc(sizeof(double) * (size_t)(n_chunks > 0 ? n_chunks : 1));
        double* lc = (double*)malloc(sizeof(double) * (size_t)(n_chunks > 0 ? n_chunks : 1));
        double* oc = (double*)malloc(sizeof(double) * (size_t)(n_chunks > 0 ? n_chunks : 1) * d);
        double* s = (double*)malloc(sizeof(double) * (size_t)chunk);
        if (!mc || !lc || !oc || !s) {
#pragma omp atomic write
            err = ORACLE_ENOMEM;
        } else {
#pragma omp for schedule(dynamic, 16)
            for (long row = 0; row < (long)B * Hq * Nq; ++row) {
                long b = row / ((long)Hq * Nq), h = (row / Nq) % Hq, i = row % Nq, hk = h / G;
                const double* qi = q + row * d;
                const double* kh = k + ((b * Hkv + hk) * (long)Nk * d);
                const double* vh = v + ((b * Hkv + hk) * (long)Nk * d);
                /* one partial per chunk */
                for (long c = 0; c < n_chunks; ++c) {
                    long j0 = c * chunk, j1 = j0 + chunk < Nk ? j0 + chunk : Nk;
                    double m = -INFINITY;
                    for (long j = j0; j < j1; ++j) {
                        s[j - j0] = key_allowed(i, j, Nq, Nk, causal, window)
                                        ? scale * dot(qi, kh + j * d, d) : -INFINITY;
                        if (s[j - j0] > m) m = s[j - j0];
                    }
                    double* o_c = oc + c * d;
                    for (int t = 0; t < d; ++t) o_c[t] = 0.0;
                    mc[c] = m;
                    lc[c] = 0.0;
                    if (m == -INFINITY) continue;
                    for (long j = j0; j < j1; ++j) {
                        if (s[j - j0] == -INFINITY) continue;
                        double pj = exp(s[j - j0] - m);
                        lc[c] += pj;
                        for (int t = 0; t < d; ++t) o_c[t] += pj * vh[j * d + t];
                    }
                    for (int t = 0; t < d; ++t) o_c[t] /= lc[c];   /* normalised partial O_c */
                }
                /* merge */
                double M = -INFINITY;
                for (long c = 0; c < n_chunks; ++c) if (mc[c] > M) M = mc[c];
                double* oo = o + row * d;
                for (int t = 0; t < d; ++t) oo[t] = 0.0;
                if (M == -INFINITY) { lse[row] = -INFINITY; continue; }
                double L = 0.0;
                for (long c = 0; c < n_chunks; ++c)
                    if (mc[c] != -INFINITY) L += lc[c] * exp(mc[c] - M);
                for (long c = 0; c < n_chunks; ++c) {
                    if (mc[c] == -INFINITY) continue;
                    double w = lc[c] * exp(mc[c] - M) / L;
                    for (int t = 0; t < d; ++t) oo[t] += w * oc[c * d + t];
                }
                lse[row] = M + log(L);
            }
        }
        free(mc); free(lc); free(oc); free(s);
    }
    return err;
}

/* ------------------------------------------------------------------------- */
/* One-query decode over a paged KV cache.                                     */
/* [MAK] "Paged attention changes addressing": for token position t of a       */
/*   sequence, logical block = t / block_size, offset = t % block_size,        */
/*   physical = block_table[sequence, logical block],                          */
/*   address = cache_base + physical * block_stride + offset * token_stride.   */
/* Cache layout [num_blocks][Hkv][block_size][d]: block_stride = Hkv*bs*d,     */
/*   token_stride = d, and kv head h adds h*bs*d.                              */
/* [AK] GQA: query head h reads kv head h / (Hq / Hkv).                         */
/* The single query of sequence s attends keys 0 .. seq_lens[s]-1, materialised. */
/* q, o: [num_seqs][Hq][d]; lse: [num_seqs][Hq].                               */
/* ------------------------------------------------------------------------- */
int oracle_attn_decode(const double* q, const double* k_cache, const double* v_cache,
                       const int32_t* block_table, const int32_t* seq_lens,
                       double* o, double* lse,
                       int num_seqs, int Hq, int Hkv, int d, int block_size,
                       int max_blocks_per_seq, int num_blocks, double scale)
{
    if (num_seqs < 0 || Hq <= 0 || Hkv <= 0 || d <= 0 || block_size <= 0 ||
        max_blocks_per_seq < 0 || num_blocks < 0 || Hq % Hkv != 0)
        return ORACLE_EINVAL;
    for (int sq = 0; sq < num_seqs; ++sq) {
        long L = seq_lens[sq];
        if (L < 0 || L > (long)max_blocks_per_seq * block_size) return ORACLE_EINVAL;
        for (long lb = 0; lb < (L + block_size - 1) / block_size; ++lb) {
            int32_t phys = block_table[(long)sq * max_blocks_per_seq + lb];
            if (phys < 0 || phys >= num_blocks) return ORACLE_EBOUNDS;
        }
    }
    int G = Hq / Hkv;
    long block_stride = (long)Hkv * block_size * d;
    long token_stride = d;
    long max_L = 0;
    for (int sq = 0; sq < num_seqs; ++sq) if (seq_lens[sq] > max_L) max_L = seq_lens[sq];
    int err = ORACLE_OK;
#pragma omp parallel
    {
        double* s = (double*)malloc(sizeof(double) * (size_t)(max_L > 0 ? max_L : 1));
        const double** vrow = (const double**)malloc(sizeof(double*) * (size_t)(max_L > 0 ? max_L : 1));
        if (!s || !vrow) {
#pragma omp atomic write
            err = ORACLE_ENOMEM;
        } else {
#pragma omp for schedule(dynamic, 1) collapse(2)
            for (long sq = 0; sq < num_seqs; ++sq) {
                for (long h = 0; h < Hq; ++h) {
                    long hk = h / G;
                    long L = seq_lens[sq];
                    const double* qh = q + (sq * Hq + h) * d;
                    double m = -INFINITY;
                    for (long t = 0; t < L; ++t) {
                        long logical = t / block_size;
                        long offset = t % block_size;
                        long physical = block_table[sq * max_blocks_per_seq + logical];
                        long addr = physical * block_stride + hk * (long)block_size * d + offset * token_stride;
                        s[t] = scale * dot(qh, k_cache + addr, d);
                        vrow[t] = v_cache + addr;
                        if (s[t] > m) m = s[t];
                    }
                    double* oh = o + (sq * Hq + h) * d;
                    for (int c = 0; c < d; ++c) oh[c] = 0.0;
                    if (L == 0) { lse[sq * Hq + h] = -INFINITY; continue; }
                    double l = 0.0;
                    for (long t = 0; t < L; ++t) { s[t] = exp(s[t] - m); l += s[t]; }
                    for (long t = 0; t < L; ++t) {
                        double pt = s[t] / l;
                        for (int c = 0; c < d; ++c) oh[c] += pt * vrow[t][c];
                    }
                    lse[sq * Hq + h] = m + log(l);
                }
            }
        }
        free(s);
        free((void*)vrow);
    }
    return err;
}

/* ------------------------------------------------------------------------- */
/* Block-sparse prefill.                                                        */
/* [MAK] "Kernel structure": an arbitrary sparse mask needs an index telling   */
/*   the kernel which blocks exist; [MAK] (the table of attention variants):   */
/*   sparse attention visits only the selected score blocks.                  */
/* Reading: a CSR index over (query block of block_q rows, key block of         */
/* block_k keys): row_ptr[n_qblk + 1], col_idx[nnz], shared by every batch     */
/* entry and head. Query row i may attend key j when the block pair            */
/* (i / block_q, j / block_k) is listed AND the causal / window mask of the    */
/* dense functions allows it. Materialised per row, like the plain definition. */
/* ------------------------------------------------------------------------- */
static int block_listed(const int32_t* row_ptr, const int32_t* col_idx, long qb, long kb)
{
    for (long e = row_ptr[qb]; e < row_ptr[qb + 1]; ++e)
        if (col_idx[e] == kb) return 1;
    return 0;
}

int oracle_attn_fwd_blocksparse(const double* q, const double* k, const double* v, double* o, double* lse,
                                int B, int Hq, int Hkv, int Nq, int Nk, int d, double scale, int causal, int window,
                                const int32_t* row_ptr, const int32_t* col_idx, int block_q, int block_k)
{
    if (check_dims(B, Hq, Hkv, Nq, Nk, d) || block_q <= 0 || block_k <= 0) return ORACLE_EINVAL;
    long n_qblk = (Nq + block_q - 1) / block_q, n_kblk = (Nk + block_k - 1) / block_k;
    if (row_ptr[0] != 0) return ORACLE_EINVAL;
    for (long qb = 0; qb < n_qblk; ++qb) {
        if (row_ptr[qb + 1] < row_ptr[qb]) return ORACLE_EINVAL;
        for (long e = row_ptr[qb]; e < row_ptr[qb + 1]; ++e)
            if (col_idx[e] < 0 || col_idx[e] >= n_kblk) return ORACLE_EBOUNDS;
    }
    int G = Hq / Hkv;
    int err = ORACLE_OK;
#pragma omp parallel
    {
        double* s = (double*)malloc(sizeof(double) * (size_t)(Nk > 0 ? Nk : 1));
        double* p = (double*)malloc(sizeof(double) * (size_t)(Nk > 0 ? Nk : 1));
        if (!s || !p) {
#pragma omp atomic write
            err = ORACLE_ENOMEM;
        } else {
#pragma omp for schedule(dynamic, 16) collapse(2)
            for (long bh = 0; bh < (long)B * Hq; ++bh) {
                for (long i = 0; i < Nq; ++i) {
                    long b = bh / Hq, h = bh % Hq, hk = h / G;
                    const double* qi = q + ((bh * (long)Nq + i) * d);
                    const double* kh = k + ((b * Hkv + hk) * (long)Nk * d);
                    const double* vh = v + ((b * Hkv + hk) * (long)Nk * d);
                    double* oi = o + ((bh * (long)Nq + i) * d);
                    /* scores of the allowed keys, -inf elsewhere */
                    double m = -INFINITY;
                    for (long j = 0; j < Nk; ++j) {
                        if (key_allowed(i, j, Nq, Nk, causal, window) &&
                            block_listed(row_ptr, col_idx, i / block_q, j / block_k))
                            s[j] = dot(qi, kh + j * d, d) * scale;
                        else
                            s[j] = -INFINITY;
                        if (s[j] > m) m = s[j];
                    }
                    for (int t = 0; t < d; ++t) oi[t] = 0.0;
                    if (m == -INFINITY) {
                        lse[bh * (long)Nq + i] = -INFINITY;
                        continue;
                    }
                    double l = 0.0;
                    for (long j = 0; j < Nk; ++j) {
                        p[j] = (s[j] == -INFINITY) ? 0.0 : exp(s[j] - m);
                        l += p[j];
                    }
                    for (long j = 0; j < Nk; ++j) {
                        if (p[j] == 0.0) continue;
                        for (int t = 0; t < d; ++t) oi[t] += (p[j] / l) * vh[j * d + t];
                    }
                    lse[bh * (long)Nq + i] = m + log(l);
                }
            }
        }
        free(s);
        free(p);
    }
    return err;
}

/* ------------------------------------------------------------------------- */
/* Prefill of several sequences against a paged cache (chunked prefill).       */
/* [MAK] "Paged attention changes addressing": token t of a sequence sits in   */
/*   logical block t / block_size at offset t % block_size; the block table    */
/*   gives the physical block, and the address is base + physical *            */
/*   block_stride + offset * token_stride (the same formula as decode above).  */
/* Reading for several new queries: sequence s holds kv_lens[s] tokens in the  */
/*   cache, the last q_lens[s] of which are its new queries, so query row i    */
/*   sits at position kv_len - q_len + i (the bottom-right causal alignment of */
/*   the prefill functions, with Nq = q_len and Nk = kv_len).                  */
/* Each (sequence, kv head) gathers its keys and values into contiguous rows   */
/* with that formula and hands every new query row to the materialised row     */
/* routine above. q, o: [S][Hq][max_q][d]; lse: [S][Hq][max_q]; rows i >=      */
/* q_lens[s] are neither read nor written.                                     */
/* ------------------------------------------------------------------------- */
int oracle_attn_prefill_paged(const double* q, const double* k_cache, const double* v_cache,
                              const int32_t* block_table, const int32_t* q_lens, const int32_t* kv_lens,
                              double* o, double* lse,
                              int num_seqs, int Hq, int Hkv, int d, int block_size,
                              int max_blocks_per_seq, int num_blocks, int max_q,
                              double scale, int causal, int window)
{
    if (num_seqs < 0 || Hq <= 0 || Hkv <= 0 || d <= 0 || block_size <= 0 || max_q < 0 ||
        max_blocks_per_seq < 0 || num_blocks < 0 || Hq % Hkv != 0)
        return ORACLE_EINVAL;
    long max_kv = 0;
    for (int sq = 0; sq < num_seqs; ++sq) {
        long qn = q_lens[sq], kn = kv_lens[sq];
        if (qn < 0 || qn > max_q || kn < qn || kn > (long)max_blocks_per_seq * block_size) return ORACLE_EINVAL;
        for (long lb = 0; lb < (kn + block_size - 1) / block_size; ++lb) {
            int32_t phys = block_table[(long)sq * max_blocks_per_seq + lb];
            if (phys < 0 || phys >= num_blocks) return ORACLE_EBOUNDS;
        }
        if (kn > max_kv) max_kv = kn;
    }
    int G = Hq / Hkv;
    long block_stride = (long)Hkv * block_size * d;
    long token_stride = d;
    int err = ORACLE_OK;
#pragma omp parallel
    {
        size_t n = (size_t)(max_kv > 0 ? max_kv : 1);
        double* kh = (double*)malloc(sizeof(double) * n * (size_t)d);
        double* vh = (double*)malloc(sizeof(double) * n * (size_t)d);
        double* sr = (double*)malloc(sizeof(double) * n);
        double* pr = (double*)malloc(sizeof(double) * n);
        if (!kh || !vh || !sr || !pr) {
#pragma omp atomic write
            err = ORACLE_ENOMEM;
        } else {
#pragma omp for schedule(dynamic, 1) collapse(2)
            for (long sq = 0; sq < num_seqs; ++sq) {
                for (long h = 0; h < Hq; ++h) {
                    long hk = h / G;
                    long qn = q_lens[sq], kn = kv_lens[sq];
                    for (long t = 0; t < kn; ++t) {
                        long blk = t / block_size, off = t % block_size;
                        long phys = block_table[sq * max_blocks_per_seq + blk];
                        long addr = phys * block_stride + off * token_stride + hk * (long)block_size * d;
                        for (int c = 0; c < d; ++c) {
                            kh[t * d + c] = k_cache[addr + c];
                            vh[t * d + c] = v_cache[addr + c];
                        }
                    }
                    for (long i = 0; i < qn; ++i) {
                        long row = (sq * Hq + h) * (long)max_q + i;
                        attend_row_materialised(q + row * d, kh, vh, i, qn, kn, d, scale, causal, window,
                                                sr, pr, o + row * d, lse + row);
                    }
                }
            }
        }
        free(kh);
        free(vh);
        free(sr);
        free(pr);
    }
    return err;
}

/* ------------------------------------------------------------------------- */
/* Backward pass, materialised.                                                */
/* [MAK] "Backward pass recomputes scores" and [IOA] (backward paragraph): the  */
/*   gradients are formed from the same scores; here every row's score and     */
/*   probability rows are materialised again from Q, K, V (no saved P).        */
/* Chain rule of O = softmax(S) V with S = scale * Q K^T, for an upstream dO:   */
/*   dV_j  = sum_i P_ij dO_i                                                   */
/*   dP_ij = dO_i . v_j                                                        */
/*   dS_ij = P_ij (dP_ij - sum_k P_ik dP_ik)      (softmax Jacobian)            */
/*   dQ_i  = scale * sum_j dS_ij k_j,   dK_j = scale * sum_i dS_ij q_i          */
/* Masked pairs have P_ij = 0 and contribute nothing. With GQA, a kv head's     */
/* dK, dV sum over the query heads that read it.                               */
/* dout, dq: [B][Hq][Nq][d]; dk, dv: [B][Hkv][Nk][d].                           */
/* ------------------------------------------------------------------------- */
int oracle_attn_bwd(const double* q, const double* k, const double* v, const double* dout,
                    double* dq, double* dk, double* dv,
                    int B, int Hq, int Hkv, int Nq, int Nk, int d,
                    double scale, int causal, int window)
{
    if (check_dims(B, Hq, Hkv, Nq, Nk, d)) return ORACLE_EINVAL;
    int G = Hq / Hkv;
    memset(dq, 0, sizeof(double) * (size_t)B * Hq * Nq * d);
    memset(dk, 0, sizeof(double) * (size_t)B * Hkv * Nk * d);
    memset(dv, 0, sizeof(double) * (size_t)B * Hkv * Nk * d);
    int err = ORACLE_OK;
#pragma omp parallel
    {
        double* s = (double*)malloc(sizeof(double) * (size_t)(Nk > 0 ? Nk : 1));
        double* p = (double*)malloc(sizeof(double) * (size_t)(Nk > 0 ? Nk : 1));
        double* dp = (double*)malloc(sizeof(double) * (size_t)(Nk > 0 ? Nk : 1));
        if (!s || !p || !dp) {
#pragma omp atomic write
            err = ORACLE_ENOMEM;
        } else {
            /* one (batch, kv head) per iteration: its dK, dV are written by one thread */
#pragma omp for schedule(dynamic, 1)
            for (long bk = 0; bk < (long)B * Hkv; ++bk) {
                long b = bk / Hkv, hk = bk % Hkv;
                const double* kh = k + (bk * (long)Nk * d);
                const double* vh = v + (bk * (long)Nk * d);
                double* dkh = dk + (bk * (long)Nk * d);
                double* dvh = dv + (bk * (long)Nk * d);
                for (long h = hk * G; h < (hk + 1) * G; ++h) {
                    for (long i = 0; i < Nq; ++i) {
                        const double* qi = q + (((b * Hq + h) * (long)Nq + i) * d);
                        const double* doi = dout + (((b * Hq + h) * (long)Nq + i) * d);
                        double* dqi = dq + (((b * Hq + h) * (long)Nq + i) * d);
                        /* probability row, exactly as in the forward */
                        double m = -INFINITY;
                        for (long j = 0; j < Nk; ++j) {
                            s[j] = key_allowed(i, j, Nq, Nk, causal, window) ? scale * dot(qi, kh + j * d, d)
                                                                             : -INFINITY;
                            if (s[j] > m) m = s[j];
                        }
                        if (m == -INFINITY) continue;  /* empty row: no gradient flows */
                        double l = 0.0;
                        for (long j = 0; j < Nk; ++j) {
                            p[j] = (s[j] == -INFINITY) ? 0.0 : exp(s[j] - m);
                            l += p[j];
                        }
                        for (long j = 0; j < Nk; ++j) p[j] /= l;
                        /* dP row and the row term sum_k P_ik dP_ik */
                        double row = 0.0;
                        for (long j = 0; j < Nk; ++j) {
                            dp[j] = (p[j] == 0.0) ? 0.0 : dot(doi, vh + j * d, d);
                            row += p[j] * dp[j];
                        }
                        for (long j = 0; j < Nk; ++j) {
                            if (p[j] == 0.0) continue;
                            double ds = p[j] * (dp[j] - row);
                            const double* kj = kh + j * d;
                            double* dkj = dkh + j * d;
                            double* dvj = dvh + j * d;
                            for (int t = 0; t < d; ++t) {
                                dvj[t] += p[j] * doi[t];
                                dqi[t] += scale * ds * kj[t];
                                dkj[t] += scale * ds * qi[t];
                            }
                        }
                    }
                }
            }
        }
        free(s);
        free(p);
        free(dp);
    }
    return err;
}

/* ------------------------------------------------------------------------- */
/* FP8 (E4M3) inputs.                                                          */
/* [AK] the FlashAttention-3 paragraph lists FP8 operands among the Hopper-era  */
/*   additions; the attention computed is still the plain definition above,    */
/*   applied to the real values that the 8-bit codes and per-tensor scales      */
/*   denote.                                                                    */
/* The E4M3 code (the OCP 8-bit floating-point format, E4M3 variant): bit 7 is  */
/*   the sign, bits 6..3 the exponent with bias 7, bits 2..0 the mantissa.      */
/*   Exponent field 0 is subnormal: value = mantissa / 8 * 2^-6. Exponent 15    */
/*   with mantissa 7 is NaN; there is no infinity (exponent 15 with mantissa    */
/*   0..6 is an ordinary number, up to 448).                                    */
/* Layouts: q8 [B][Hq][Nq][d], k8 [B][Hkv][Nk][d], vt8 [B][Hkv][d][Nk] (V given */
/*   transposed: element (j, t) of head h's V is vt8[h][t][j]).                 */
/* ------------------------------------------------------------------------- */
double oracle_e4m3_value(uint8_t code)
{
    const int negative = (code >> 7) & 1;
    const int exponent = (code >> 3) & 15;
    const int mantissa = code & 7;
    double magnitude;
    if (exponent == 15 && mantissa == 7) return NAN;
    if (exponent == 0)
        magnitude = ldexp((double)mantissa / 8.0, -6);
    else
        magnitude = ldexp(1.0 + (double)mantissa / 8.0, exponent - 7);
    return negative ? -magnitude : magnitude;
}

int oracle_e4m3_decode(const uint8_t* codes, double* out, int64_t n)
{
    if (n < 0) return ORACLE_EINVAL;
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_e4m3_value(codes[i]);
    return ORACLE_OK;
}

int oracle_attn_fwd_fp8(const uint8_t* q8, const uint8_t* k8, const uint8_t* vt8, double* o, double* lse,
                        int B, int Hq, int Hkv, int Nq, int Nk, int d, double scale,
                        double q_descale, double k_descale, double v_descale, int causal, int window)
{
    if (check_dims(B, Hq, Hkv, Nq, Nk, d)) return ORACLE_EINVAL;
    const int64_t nq = (int64_t)B * Hq * Nq * d;
    const int64_t nk = (int64_t)B * Hkv * Nk * d;
    double* q = (double*)malloc(sizeof(double) * (size_t)(nq > 0 ? nq : 1));
    double* k = (double*)malloc(sizeof(double) * (size_t)(nk > 0 ? nk : 1));
    double* v = (double*)malloc(sizeof(double) * (size_t)(nk > 0 ? nk : 1));
    if (!q || !k || !v) {
        free(q); free(k); free(v);
        return ORACLE_ENOMEM;
    }
    for (int64_t i = 0; i < nq; ++i) q[i] = q_descale * oracle_e4m3_value(q8[i]);
    for (int64_t i = 0; i < nk; ++i) k[i] = k_descale * oracle_e4m3_value(k8[i]);
    /* v[b][h][j][t] = v_descale * value(vt8[b][h][t][j]) */
    for (int64_t bh = 0; bh < (int64_t)B * Hkv; ++bh)
        for (int64_t j = 0; j < Nk; ++j)
            for (int t = 0; t < d; ++t)
                v[(bh * Nk + j) * d + t] = v_descale * oracle_e4m3_value(vt8[(bh * d + t) * Nk + j]);
    const int rc = oracle_attn_fwd(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, d, scale, causal, window);
    free(q); free(k); free(v);
    return rc;
}

/* Number of OpenMP threads the oracle will use (reported beside CPU timings). */
int oracle_num_threads(void)
{
    int n = 1;
#pragma omp parallel
    {
#pragma omp single
        {
#ifdef _OPENMP
            n = omp_get_num_threads();
#endif
        }
    }
    return n;
}
