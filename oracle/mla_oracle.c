/*
 * Oracle for absorbed-MLA speculative-decoding verify attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the bench's
 * CPU-baseline leg may load this library; the product path never does.
 *
 * Plain, slow, fp64 CPU code that states what the verify step computes, one
 * query row (stream b, draft i, head h) at a time, with no tiling, fusion or
 * reordering.  Sources (pages by title):
 *
 *  [MLA]  "The Flash Attention Kernel That Had to Be Built: Designing sm_120
 *         MLA Verify for Blackwell Consumer GPUs", section "What Input
 *         Knowledge Is Required to Understand This Message", paragraph
 *         "Multi-head Latent Attention (MLA)": the cache row is a 512-wide
 *         latent kv_c plus a 64-wide decoupled RoPE key k_pe; the query splits
 *         into an absorbed q_nope and q_pe; the score is the sum of the two
 *         dot products; the latent is also the value.
 *  [MASK] same page, paragraph "Speculative Decoding with DFlash": each draft
 *         query attends to the part of the cache its candidate tree allows;
 *         masked positions are set to -inf before the softmax.
 *  [SOFT] same page, paragraph "Flash Attention Algorithm", and "The Moment of
 *         Truth: Benchmarking a Custom sm_120 Flash Attention Kernel",
 *         section "Input Knowledge Required", paragraph "Online softmax":
 *         softmax over the visible keys, output = weighted sum of values.
 *  [SPLIT] "The Decisive Microbench: When Theory Meets Silicon", section "The
 *         KV-Split Solution": the key range is cut into slices, each slice
 *         keeps an unnormalised accumulator and its statistics, and the
 *         slices are merged with the online-softmax combine.
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *  - scale: an explicit argument (the workloads pass fp32 1/sqrt(192)).
 *  - lse: natural log of sum_t exp(scale * s_t) over visible keys.
 *  - layout: seq_lens[b] = prefix_b + q; the drafts' own cache rows sit at
 *    positions prefix_b .. seq_lens[b]-1; every draft sees the whole prefix.
 *  - mask: uint32 words, LSB first; bit j of row i set <=> draft i sees
 *    draft j; row stride ceil(q/32) words.  Any bit pattern is honoured.
 *  - a row with no visible key: out = 0, lse = -inf.
 *  - rows >= seq_lens[b] are never read.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include "mla_oracle.h"

static double bf16_to_f64(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

typedef struct {
    const uint16_t *q_nope, *q_rope, *kv;
    const int32_t *seq_lens;
    const uint32_t *mask;
    int B, q, H, Smax, Dl, Dr;
    double scale;
    const int32_t *k0, *k1;    /* per-stream key window, NULL = whole range */
    double *out, *lse;         /* full mode */
    double *acc, *m, *l;       /* partial mode */
    int partial;
    long row_begin, row_end;
} job_t;

/* Is key t visible to draft i of stream b?  [MASK] with the layout reading. */
static int visible(const job_t *J, int b, int i, int t)
{
    int S = J->seq_lens[b];
    int prefix = S - J->q;
    if (t < prefix)
        return 1;
    if (t >= S)
        return 0;
    int j = t - prefix;
    int words = (J->q + 31) / 32;
    const uint32_t *row = J->mask + ((size_t)b * J->q + i) * words;
    return (int)((row[j >> 5] >> (j & 31)) & 1u);
}

/* Scaled score of query row (b, i, h) against cache row t.  [MLA] */
static double score(const job_t *J, int b, int i, int h, int t)
{
    const uint16_t *qn = J->q_nope + (((size_t)b * J->q + i) * J->H + h) * J->Dl;
    const uint16_t *qr = J->q_rope + (((size_t)b * J->q + i) * J->H + h) * J->Dr;
    const uint16_t *k = J->kv + ((size_t)b * J->Smax + t) * (size_t)(J->Dl + J->Dr);
    double s = 0.0;
    for (int d = 0; d < J->Dl; ++d)
        s += bf16_to_f64(qn[d]) * bf16_to_f64(k[d]);
    for (int d = 0; d < J->Dr; ++d)
        s += bf16_to_f64(qr[d]) * bf16_to_f64(k[J->Dl + d]);
    return J->scale * s;
}

/* One query row over keys [lo, hi): max, weights, weighted latent sum. */
static void row(const job_t *J, long r, double *sbuf)
{
    int h = (int)(r % J->H);
    int i = (int)((r / J->H) % J->q);
    int b = (int)(r / ((long)J->H * J->q));
    int S = J->seq_lens[b];
    int lo = J->k0 ? J->k0[b] : 0;
    int hi = J->k1 ? J->k1[b] : S;
    if (hi > S)
        hi = S;
    if (lo < 0)
        lo = 0;
    int D = J->Dl + J->Dr;

    /* scores of visible keys; -inf marks a masked key */
    double m = -INFINITY;
    for (int t = lo; t < hi; ++t) {
        if (visible(J, b, i, t)) {
            sbuf[t - lo] = score(J, b, i, h, t);
            if (sbuf[t - lo] > m)
                m = sbuf[t - lo];
        } else {
            sbuf[t - lo] = -INFINITY;
        }
    }
    double *o = J->partial ? J->acc + (size_t)r * J->Dl : J->out + (size_t)r * J->Dl;
    for (int d = 0; d < J->Dl; ++d)
        o[d] = 0.0;
    double l = 0.0;
    if (m != -INFINITY) {
        for (int t = lo; t < hi; ++t) {
            if (sbuf[t - lo] == -INFINITY)
                continue;
            double w = exp(sbuf[t - lo] - m);
            l += w;
            const uint16_t *v = J->kv + ((size_t)b * J->Smax + t) * (size_t)D;
            for (int d = 0; d < J->Dl; ++d)
                o[d] += w * bf16_to_f64(v[d]);
        }
    }
    if (J->partial) {
        J->m[r] = m;
        J->l[r] = l;
        return;
    }
    if (l > 0.0) {
        for (int d = 0; d < J->Dl; ++d)
            o[d] /= l;
        J->lse[r] = m + log(l);
    } else {
        J->lse[r] = -INFINITY;
    }
}

static void *worker(void *arg)
{
    job_t *J = (job_t *)arg;
    double *sbuf = (double *)malloc(sizeof(double) * (size_t)(J->Smax > 0 ? J->Smax : 1));
    if (!sbuf)
        return (void *)1;
    for (long r = J->row_begin; r < J->row_end; ++r)
        row(J, r, sbuf);
    free(sbuf);
    return NULL;
}

static int check(const job_t *J)
{
    if (!J->q_nope || !J->q_rope || !J->kv || !J->seq_lens || !J->mask)
        return MLA_ORACLE_ERR_ARG;
    if (J->B < 0 || J->q < 1 || J->H < 1 || J->Dl < 1 || J->Dr < 0 || J->Smax < 0)
        return MLA_ORACLE_ERR_ARG;
    for (int b = 0; b < J->B; ++b)
        if (J->seq_lens[b] < J->q || J->seq_lens[b] > J->Smax)
            return MLA_ORACLE_ERR_SEQLEN;
    return 0;
}

static int run(job_t *J, long rows_total, int nthreads, long row_offset)
{
    int rc = check(J);
    if (rc)
        return rc;
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > 256)
        nthreads = 256;
    if ((long)nthreads > rows_total)
        nthreads = rows_total > 0 ? (int)rows_total : 1;
    pthread_t th[256];
    job_t jobs[256];
    int joinable[256];
    long per = (rows_total + nthreads - 1) / nthreads;
    int fail = 0;
    for (int k = 0; k < nthreads; ++k) {
        long b = (long)k * per, e = (long)(k + 1) * per;
        jobs[k] = *J;
        jobs[k].row_begin = row_offset + b;
        jobs[k].row_end = row_offset + (e < rows_total ? e : rows_total);
        joinable[k] = 0;
        if (jobs[k].row_begin >= jobs[k].row_end)
            continue;
        if (pthread_create(&th[k], NULL, worker, &jobs[k]) == 0)
            joinable[k] = 1;
        else if (worker(&jobs[k]) != NULL)
            fail = 1;
    }
    for (int k = 0; k < nthreads; ++k) {
        if (joinable[k]) {
            void *ret = NULL;
            pthread_join(th[k], &ret);
            if (ret)
                fail = 1;
        }
    }
    return fail ? MLA_ORACLE_ERR_ALLOC : 0;
}

int mla_oracle_verify_attn(const uint16_t *q_nope, const uint16_t *q_rope, const uint16_t *kv,
                           const int32_t *seq_lens, const uint32_t *tree_mask, int B, int q, int H,
                           int Smax, int Dl, int Dr, double scale, double *out, double *lse,
                           int nthreads)
{
    return mla_oracle_verify_attn_rows(q_nope, q_rope, kv, seq_lens, tree_mask, B, q, H, Smax, Dl,
                                       Dr, scale, 0, (long)B * q * H, out, lse, nthreads);
}

int mla_oracle_verify_attn_rows(const uint16_t *q_nope, const uint16_t *q_rope,
                                const uint16_t *kv, const int32_t *seq_lens,
                                const uint32_t *tree_mask, int B, int q, int H, int Smax, int Dl,
                                int Dr, double scale, long row_begin, long row_count, double *out,
                                double *lse, int nthreads)
{
    job_t J;
    memset(&J, 0, sizeof J);
    J.q_nope = q_nope; J.q_rope = q_rope; J.kv = kv; J.seq_lens = seq_lens; J.mask = tree_mask;
    J.B = B; J.q = q; J.H = H; J.Smax = Smax; J.Dl = Dl; J.Dr = Dr; J.scale = scale;
    J.out = out; J.lse = lse;
    if (!out || !lse || row_begin < 0 || row_begin + row_count > (long)B * q * H)
        return MLA_ORACLE_ERR_ARG;
    /* rows outside [row_begin, row_begin+row_count) are left untouched;
       out/lse are indexed by absolute row number. */
    return run(&J, row_count, nthreads, row_begin);
}

int mla_oracle_partial(const uint16_t *q_nope, const uint16_t *q_rope, const uint16_t *kv,
                       const int32_t *seq_lens, const uint32_t *tree_mask, int B, int q, int H,
                       int Smax, int Dl, int Dr, double scale, const int32_t *k0, const int32_t *k1,
                       double *acc, double *m, double *l, int nthreads)
{
    job_t J;
    memset(&J, 0, sizeof J);
    J.q_nope = q_nope; J.q_rope = q_rope; J.kv = kv; J.seq_lens = seq_lens; J.mask = tree_mask;
    J.B = B; J.q = q; J.H = H; J.Smax = Smax; J.Dl = Dl; J.Dr = Dr; J.scale = scale;
    J.k0 = k0; J.k1 = k1; J.acc = acc; J.m = m; J.l = l; J.partial = 1;
    if (!k0 || !k1 || !acc || !m || !l)
        return MLA_ORACLE_ERR_ARG;
    return run(&J, (long)B * q * H, nthreads, 0);
}

/* Merge nsplit partial states of nrows rows.  [SPLIT]: with M = max_s m_s,
 * w_s = exp(m_s - M), L = sum_s w_s l_s:  out = sum_s w_s acc_s / L,
 * lse = M + ln L.  Splits with l_s = 0 contribute nothing. */
void mla_oracle_combine(const double *acc, const double *m, const double *l, int nsplit,
                        long nrows, int Dl, double *out, double *lse)
{
    for (long r = 0; r < nrows; ++r) {
        double M = -INFINITY;
        for (int s = 0; s < nsplit; ++s)
            if (l[(size_t)s * nrows + r] > 0.0 && m[(size_t)s * nrows + r] > M)
                M = m[(size_t)s * nrows + r];
        double *o = out + (size_t)r * Dl;
        for (int d = 0; d < Dl; ++d)
            o[d] = 0.0;
        if (M == -INFINITY) {
            lse[r] = -INFINITY;
            continue;
        }
        double L = 0.0;
        for (int s = 0; s < nsplit; ++s) {
            double ls = l[(size_t)s * nrows + r];
            if (!(ls > 0.0))
                continue;
            double w = exp(m[(size_t)s * nrows + r] - M);
            L += w * ls;
            const double *a = acc + ((size_t)s * nrows + r) * Dl;
            for (int d = 0; d < Dl; ++d)
                o[d] += w * a[d];
        }
        for (int d = 0; d < Dl; ++d)
            o[d] /= L;
        lse[r] = M + log(L);
    }
}

/* Softmax weights of one query row over all keys [0, Smax): w_t / l, and 0
 * for keys that are not visible.  Used by tests to check sum-to-one and the
 * zero weight of masked keys. */
int mla_oracle_row_weights(const uint16_t *q_nope, const uint16_t *q_rope, const uint16_t *kv,
                           const int32_t *seq_lens, const uint32_t *tree_mask, int B, int q, int H,
                           int Smax, int Dl, int Dr, double scale, int b, int i, int h,
                           double *weights)
{
    job_t J;
    memset(&J, 0, sizeof J);
    J.q_nope = q_nope; J.q_rope = q_rope; J.kv = kv; J.seq_lens = seq_lens; J.mask = tree_mask;
    J.B = B; J.q = q; J.H = H; J.Smax = Smax; J.Dl = Dl; J.Dr = Dr; J.scale = scale;
    int rc = check(&J);
    if (rc)
        return rc;
    if (b < 0 || b >= B || i < 0 || i >= q || h < 0 || h >= H || !weights)
        return MLA_ORACLE_ERR_ARG;
    double m = -INFINITY;
    for (int t = 0; t < Smax; ++t) {
        weights[t] = -INFINITY;
        if (visible(&J, b, i, t)) {
            weights[t] = score(&J, b, i, h, t);
            if (weights[t] > m)
                m = weights[t];
        }
    }
    double l = 0.0;
    for (int t = 0; t < Smax; ++t) {
        weights[t] = (weights[t] == -INFINITY) ? 0.0 : exp(weights[t] - m);
        l += weights[t];
    }
    if (l > 0.0)
        for (int t = 0; t < Smax; ++t)
            weights[t] /= l;
    return 0;
}
