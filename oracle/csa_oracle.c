/*
 * csa_oracle.c -- plain, slow CPU oracle for compressed sparse attention (CSA)
 * decode and its heavily-compressed (HCA) variant.
 *
 * THIS IS TEST INFRASTRUCTURE. Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may call it. It shares no code, header, table or
 * helper with the CUDA library: every number format is decoded here from its
 * bit definition, and every step is the plain definition written out as loops
 * with double-precision accumulation.
 *
 * Sources (web pages of the DSV4 "nvfp4-megamoe-kernel" project):
 *   [AUDIT]   "DSV4 Audit -- Decode Repetition + Precision / Tensor-Core Plan"
 *             (FINAL_STRETCH.md): section A3 (visible range, SWA overlap),
 *             section A4 (inverse RoPE on the attention output),
 *             section B1 (FP8 nope + BF16 rope latent), section B2 (indexer).
 *   [ROADMAP] "ROADMAP -- Stage E and the path to a runnable model"
 *             (archived_plans/NEXT_PRIORITIES_PART_2.md): section E1 (gathers
 *             of selected / all compressed entries and of the SWA window,
 *             FP8 entries with an inverse scale stored alongside), section E6
 *             (FP4 output of the attention with a per-128-element amax),
 *             section E7 (top-k of indexer scores).
 *   [README]  "DSV4 Inference Kernel" (README.md): section Architecture (CSA m=4,
 *             HCA m'=128, one 512-d latent shared by all 128 heads, sink
 *             weights merging sparse and SWA attention).
 *
 * The pages never print formulas. The readings taken here (each one noted at
 * the function that uses it) are the plainest ones the prose supports.
 *
 * Shapes are parameters so that the test suite can pin small special cases;
 * the production shapes are H=128, Dn=448, Dr=64, SB=128, Hi=64, Di=128.
 *
 * Parity pins for every function live in tests/test_oracle_*.py.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Return codes. */
#define ORACLE_OK 0
#define ORACLE_BAD_INDEX 1   /* a selected index outside the cache */
#define ORACLE_BAD_ARG 2
#define ORACLE_NO_MEMORY 3

/* ------------------------------------------------------------------------ */
/* Number formats                                                            */
/* ------------------------------------------------------------------------ */

/* OCP FP8 E4M3 ("e4m3fn"): sign bit 7, exponent bits 6..3 (bias 7), mantissa
 * bits 2..0; no infinities; exponent 15 with mantissa 7 is NaN; exponent 0 is
 * subnormal (mantissa/8 * 2^-6). The pages store the CSA latent's nope dims
 * and the indexer keys in this format ([AUDIT] B1, B2). */
double oracle_e4m3_value(uint8_t code)
{
    int sign = (code >> 7) & 1;
    int expo = (code >> 3) & 15;
    int mant = code & 7;
    double mag;
    if (expo == 15 && mant == 7)
        return NAN;
    if (expo == 0)
        mag = ldexp((double)mant / 8.0, -6);
    else
        mag = ldexp(1.0 + (double)mant / 8.0, expo - 7);
    return sign ? -mag : mag;
}

/* BF16: the high 16 bits of an IEEE binary32. The rope dims and the queries
 * are BF16 ([AUDIT] B1). */
double oracle_bf16_value(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double f32_at(const uint8_t *p)
{
    float f;
    memcpy(&f, p, sizeof f);
    return (double)f;
}

static uint16_t u16_at(const uint8_t *p)
{
    uint16_t v;
    memcpy(&v, p, sizeof v);
    return v;
}

/* ------------------------------------------------------------------------ */
/* a1: causal visibility of compressed blocks                                */
/* ------------------------------------------------------------------------ */

/* [AUDIT] A3, item 1: a decode query sees only compressed blocks strictly
 * before its own, still incomplete, block. With 0-based token position p and
 * m tokens per block, the query's block is floor(p/m), so the visible entries
 * are c = 0 .. floor(p/m)-1. The count is also bounded by the entries that
 * exist (n_comp) and by the cache's per-sequence capacity. */
int oracle_n_visible(int p, int m, int n_comp, int capacity)
{
    int nv;
    if (p < 0 || m <= 0)
        return 0;
    nv = p / m;
    if (nv > n_comp)
        nv = n_comp;
    if (nv > capacity)
        nv = capacity;
    if (nv < 0)
        nv = 0;
    return nv;
}

/* ------------------------------------------------------------------------ */
/* a2: lightning-indexer logits                                              */
/* ------------------------------------------------------------------------ */

/* [AUDIT] B2 names the indexer a "weighted-ReLU MQA logits" score of every
 * query token against every compressed entry (the einsum 'tnd,cd->tnc' over
 * Hi indexer heads), with FP8 keys already in the cache. Reading: per head a
 * dot product of the dequantised FP8 query and key, a ReLU, then a weighted
 * sum over heads with per-token weights:
 *
 *   I[c] = sum_h w[h] * max(0, sum_d (q8[h,d]*sq[h]) * (k8[c,d]*sk[c]))
 *
 * for c < n_vis, and -inf for c >= n_vis (not visible, [AUDIT] A3 item 1).
 * One query token; keys is [Ncap, Di] of one sequence. */
void oracle_indexer_row(const uint8_t *q8, const float *q_scale, const float *w,
                        const uint8_t *k8, const float *k_scale,
                        int Hi, int Di, int n_vis, int Ncap, double *out)
{
    int c, h, d;
    double *qd = (double *)malloc(sizeof(double) * (size_t)Hi * (size_t)Di);
    if (!qd)
        return;
    for (h = 0; h < Hi; ++h)
        for (d = 0; d < Di; ++d)
            qd[(size_t)h * Di + d] = oracle_e4m3_value(q8[(size_t)h * Di + d]) * (double)q_scale[h];
    for (c = 0; c < Ncap; ++c) {
        double acc = 0.0;
        if (c >= n_vis) {
            out[c] = -INFINITY;
            continue;
        }
        for (h = 0; h < Hi; ++h) {
            double dot = 0.0;
            for (d = 0; d < Di; ++d)
                dot += qd[(size_t)h * Di + d] *
                       (oracle_e4m3_value(k8[(size_t)c * Di + d]) * (double)k_scale[c]);
            acc += (double)w[h] * (dot > 0.0 ? dot : 0.0);
        }
        out[c] = acc;
    }
    free(qd);
}

/* Batched driver over flat query rows r = b*T + t in [row_begin, row_end).
 * q8 [B,T,Hi,Di], q_scale/w [B,T,Hi], k8 [B,Ncap,Di], k_scale [B,Ncap],
 * q_pos [B,T], n_comp [B], out [B,T,Ncap]. */
int oracle_indexer_logits(const uint8_t *q8, const float *q_scale, const float *w,
                          const uint8_t *k8, const float *k_scale,
                          const int32_t *q_pos, const int32_t *n_comp,
                          int B, int T, int Ncap, int Hi, int Di, int m,
                          int row_begin, int row_end, double *out)
{
    int r;
    if (B <= 0 || T <= 0 || Ncap < 0 || row_begin < 0 || row_end > B * T)
        return ORACLE_BAD_ARG;
    for (r = row_begin; r < row_end; ++r) {
        int b = r / T;
        int nv = oracle_n_visible(q_pos[r], m, n_comp[b], Ncap);
        oracle_indexer_row(q8 + (size_t)r * Hi * Di, q_scale + (size_t)r * Hi, w + (size_t)r * Hi,
                           k8 + (size_t)b * Ncap * Di, k_scale + (size_t)b * Ncap,
                           Hi, Di, nv, Ncap, out + (size_t)r * Ncap);
    }
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* a3: top-k selection                                                       */
/* ------------------------------------------------------------------------ */

typedef struct {
    double score;
    int32_t index;
} scored_t;

/* Larger score first; equal scores keep the lower index first. */
static int cmp_scored(const void *a, const void *b)
{
    const scored_t *x = (const scored_t *)a, *y = (const scored_t *)b;
    if (x->score > y->score)
        return -1;
    if (x->score < y->score)
        return 1;
    return (x->index > y->index) - (x->index < y->index);
}

/* [AUDIT] B2 / [ROADMAP] E7: top-k of the indexer scores over the causally
 * visible entries. Reading: the min(k, n_vis) entries with the largest scores
 * among c < n_vis, ties going to the lower index; the output is that list in
 * sorted order, padded with -1 to length k. Returns the count. */
int oracle_topk_row(const double *scores, int n_vis, int k, int32_t *idx_out)
{
    int i, cnt = n_vis < k ? n_vis : k;
    scored_t *s;
    if (cnt < 0)
        cnt = 0;
    s = (scored_t *)malloc(sizeof(scored_t) * (size_t)(n_vis > 0 ? n_vis : 1));
    if (!s)
        return -1;
    for (i = 0; i < n_vis; ++i) {
        s[i].score = scores[i];
        s[i].index = i;
    }
    qsort(s, (size_t)(n_vis > 0 ? n_vis : 0), sizeof(scored_t), cmp_scored);
    for (i = 0; i < k; ++i)
        idx_out[i] = i < cnt ? s[i].index : -1;
    free(s);
    return cnt;
}

/* Batched driver. scores [B,T,Ncap] (double), idx_out [B,T,k], cnt_out [B,T]. */
int oracle_topk(const double *scores, const int32_t *q_pos, const int32_t *n_comp,
                int B, int T, int Ncap, int m, int k, int row_begin, int row_end,
                int32_t *idx_out, int32_t *cnt_out)
{
    int r;
    if (k <= 0 || row_begin < 0 || row_end > B * T)
        return ORACLE_BAD_ARG;
    for (r = row_begin; r < row_end; ++r) {
        int b = r / T;
        int nv = oracle_n_visible(q_pos[r], m, n_comp[b], Ncap);
        int c = oracle_topk_row(scores + (size_t)r * Ncap, nv, k, idx_out + (size_t)r * k);
        if (c < 0)
            return ORACLE_NO_MEMORY;
        cnt_out[r] = c;
    }
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* Cache addressing                                                          */
/* ------------------------------------------------------------------------ */

/* A compressed cache is an array of fixed-size records. Logical entry c of
 * sequence b is record b*seq_stride + c, or, with a block table ([README]
 * Architecture: classical paged cache of 128-token pages, i.e. 32 CSA or 1 HCA
 * entries per page), record block_table[b*max_pages + c/page_records] *
 * page_records + c % page_records. Returns NULL outside the cache. */
static const uint8_t *comp_record(const uint8_t *base, int64_t seq_stride,
                                  const int32_t *block_table, int page_records, int max_pages,
                                  int64_t n_records, int seq_capacity, int rec_bytes,
                                  int b, int c)
{
    int64_t rec;
    if (c < 0 || c >= seq_capacity)
        return NULL;
    if (block_table) {
        int page = c / page_records;
        int32_t phys;
        if (page >= max_pages)
            return NULL;
        phys = block_table[(int64_t)b * max_pages + page];
        if (phys < 0)
            return NULL;
        rec = (int64_t)phys * page_records + c % page_records;
    } else {
        rec = (int64_t)b * seq_stride + c;
    }
    if (rec < 0 || rec >= n_records)
        return NULL;
    return base + rec * (int64_t)rec_bytes;
}

/* [AUDIT] A3 item 2 and [ROADMAP] E1: the SWA ring holds the most recent W
 * tokens of a sequence. Reading: the window of a query at position p is
 * positions max(0, p-W+1) .. p (its own token included, oldest first), and
 * position j lives in ring slot j mod R of a per-sequence ring of R slots. */
static int swa_first(int p, int W)
{
    int j0 = p - W + 1;
    return j0 < 0 ? 0 : j0;
}

/* ------------------------------------------------------------------------ */
/* a5: sink-merged attention over one candidate list                         */
/* ------------------------------------------------------------------------ */

/* Dequantise one record ([AUDIT] B1: nope dims FP8 E4M3 with a stored scale,
 * rope dims BF16; [ROADMAP] E1: the "inverse scale stored alongside" is read
 * as the dequantisation multiplier). Record layout: Dn e4m3 bytes, then Dr
 * bf16 values, then ceil(Dn/SB) fp32 scales; scale i covers nope dims
 * [i*SB, min((i+1)*SB, Dn)). */
static void dequant_record(const uint8_t *rec, int Dn, int Dr, int SB, double *x)
{
    int d, r;
    const uint8_t *rope = rec + Dn;
    const uint8_t *scales = rec + Dn + 2 * Dr;
    for (d = 0; d < Dn; ++d)
        x[d] = oracle_e4m3_value(rec[d]) * f32_at(scales + 4 * (d / SB));
    for (r = 0; r < Dr; ++r)
        x[Dn + r] = oracle_bf16_value(u16_at(rope + 2 * r));
}

/* [README] Architecture: one latent per candidate serves as key and value for
 * all H heads, and a per-head sink weight merges the sparse and SWA terms.
 * Reading: the sink is an extra logit in the softmax denominator with no value
 * vector. For head h and candidates j:
 *   z_j = scale * sum_d q[h,d] x_j[d]
 *   M   = max(sink_h, max_j z_j)
 *   den = exp(sink_h - M) + sum_j exp(z_j - M)
 *   o_h = sum_j exp(z_j - M) x_j / den,   lse_h = M + ln(den).
 * No candidates: o = 0 and lse = sink (-inf when sink is -inf).
 * q is [H, Dn+Dr] bf16 bits; cand is n record pointers; out [H, Dn+Dr]. */
int oracle_attention_row(const uint16_t *q, const float *sink, double scale,
                         const uint8_t *const *cand, int n, int H, int Dn, int Dr, int SB,
                         double *out, double *lse)
{
    int D = Dn + Dr, h, j, d;
    double *x, *z, *qd;
    if (n == 0) {
        for (h = 0; h < H; ++h) {
            for (d = 0; d < D; ++d)
                out[(size_t)h * D + d] = 0.0;
            lse[h] = (double)sink[h];
        }
        return ORACLE_OK;
    }
    x = (double *)malloc(sizeof(double) * (size_t)n * D);
    z = (double *)malloc(sizeof(double) * (size_t)n);
    qd = (double *)malloc(sizeof(double) * (size_t)D);
    if (!x || !z || !qd) {
        free(x); free(z); free(qd);
        return ORACLE_NO_MEMORY;
    }
    for (j = 0; j < n; ++j)
        dequant_record(cand[j], Dn, Dr, SB, x + (size_t)j * D);
    for (h = 0; h < H; ++h) {
        double M = (double)sink[h], den;
        for (d = 0; d < D; ++d)
            qd[d] = oracle_bf16_value(q[(size_t)h * D + d]);
        for (j = 0; j < n; ++j) {
            double dot = 0.0;
            for (d = 0; d < D; ++d)
                dot += qd[d] * x[(size_t)j * D + d];
            z[j] = scale * dot;
            if (z[j] > M)
                M = z[j];
        }
        den = exp((double)sink[h] - M);
        for (j = 0; j < n; ++j)
            den += exp(z[j] - M);
        for (d = 0; d < D; ++d) {
            double acc = 0.0;
            for (j = 0; j < n; ++j)
                acc += exp(z[j] - M) * x[(size_t)j * D + d];
            out[(size_t)h * D + d] = acc / den;
        }
        lse[h] = M + log(den);
    }
    free(x); free(z); free(qd);
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* Candidate lists (a4) and the batched CSA / HCA drivers (a5, a6)           */
/* ------------------------------------------------------------------------ */

/* [AUDIT] A3: the decode query attends to [selected compressed entries] ++
 * [SWA window]; a token present in both is seen twice (overlap allowed, no
 * deduplication). The selected list is topk_idx[0 .. cnt-1] in its given
 * order; the window follows, oldest position first. Returns the number of
 * candidates or -1 on an index outside the cache. */
static int csa_candidates(const uint8_t *comp, int64_t seq_stride, const int32_t *block_table,
                          int page_records, int max_pages, int64_t n_records, int seq_capacity,
                          const uint8_t *ring, int R, int W, int rec_bytes,
                          const int32_t *sel, int cnt, int b, int p,
                          const uint8_t **cand)
{
    int i, n = 0, j;
    for (i = 0; i < cnt; ++i) {
        const uint8_t *rec = comp_record(comp, seq_stride, block_table, page_records, max_pages,
                                         n_records, seq_capacity, rec_bytes, b, sel[i]);
        if (!rec)
            return -1;
        cand[n++] = rec;
    }
    if (p >= 0)
        for (j = swa_first(p, W); j <= p; ++j)
            cand[n++] = ring + ((int64_t)b * R + (j % R)) * (int64_t)rec_bytes;
    return n;
}

/* CSA attention for rows r in [row_begin, row_end): q [B,T,H,D] bf16 bits,
 * sink [H], topk_idx [B,T,k], topk_cnt [B,T], ring [B,R,rec], out [B,T,H,D],
 * lse [B,T,H]. */
int oracle_csa_attention(const uint16_t *q, const float *sink, double scale,
                         const uint8_t *comp, int64_t seq_stride, const int32_t *block_table,
                         int page_records, int max_pages, int64_t n_records, int seq_capacity,
                         const uint8_t *ring, int R, int W,
                         const int32_t *topk_idx, const int32_t *topk_cnt, const int32_t *q_pos,
                         int B, int T, int k, int H, int Dn, int Dr, int SB, int rec_bytes,
                         int row_begin, int row_end, double *out, double *lse)
{
    int r, D = Dn + Dr, rc = ORACLE_OK;
    const uint8_t **cand;
    if (row_begin < 0 || row_end > B * T || k < 0 || W < 0 || R < 1)
        return ORACLE_BAD_ARG;
    cand = (const uint8_t **)malloc(sizeof(*cand) * (size_t)(k + W + 1));
    if (!cand)
        return ORACLE_NO_MEMORY;
    for (r = row_begin; r < row_end && rc == ORACLE_OK; ++r) {
        int b = r / T, cnt = topk_cnt[r], n;
        if (cnt < 0 || cnt > k) {
            rc = ORACLE_BAD_ARG;
            break;
        }
        n = csa_candidates(comp, seq_stride, block_table, page_records, max_pages, n_records,
                           seq_capacity, ring, R, W, rec_bytes, topk_idx + (size_t)r * k, cnt,
                           b, q_pos[r], cand);
        if (n < 0) {
            rc = ORACLE_BAD_INDEX;
            break;
        }
        rc = oracle_attention_row(q + (size_t)r * H * D, sink, scale, cand, n, H, Dn, Dr, SB,
                                  out + (size_t)r * H * D, lse + (size_t)r * H);
    }
    free(cand);
    return rc;
}

/* [README] Architecture and [ROADMAP] E1 (gather of all compressed entries):
 * HCA attends to every visible heavily-compressed entry (m' = 128 tokens per
 * entry) plus the SWA window, with no indexer. Candidates = entries
 * 0 .. n_vis-1 ++ the window, n_vis from the same causality rule. */
int oracle_hca_attention(const uint16_t *q, const float *sink, double scale,
                         const uint8_t *comp, int64_t seq_stride, const int32_t *block_table,
                         int page_records, int max_pages, int64_t n_records, int seq_capacity,
                         const int32_t *n_comp, const uint8_t *ring, int R, int W,
                         const int32_t *q_pos, int B, int T, int m_hca,
                         int H, int Dn, int Dr, int SB, int rec_bytes,
                         int row_begin, int row_end, double *out, double *lse)
{
    int r, D = Dn + Dr, rc = ORACLE_OK;
    const uint8_t **cand;
    int32_t *sel;
    if (row_begin < 0 || row_end > B * T || W < 0 || R < 1 || seq_capacity < 0)
        return ORACLE_BAD_ARG;
    cand = (const uint8_t **)malloc(sizeof(*cand) * (size_t)(seq_capacity + W + 1));
    sel = (int32_t *)malloc(sizeof(int32_t) * (size_t)(seq_capacity + 1));
    if (!cand || !sel) {
        free(cand); free(sel);
        return ORACLE_NO_MEMORY;
    }
    for (r = row_begin; r < row_end && rc == ORACLE_OK; ++r) {
        int b = r / T, i, n;
        int nv = oracle_n_visible(q_pos[r], m_hca, n_comp[b], seq_capacity);
        for (i = 0; i < nv; ++i)
            sel[i] = i;
        n = csa_candidates(comp, seq_stride, block_table, page_records, max_pages, n_records,
                           seq_capacity, ring, R, W, rec_bytes, sel, nv, b, q_pos[r], cand);
        if (n < 0) {
            rc = ORACLE_BAD_INDEX;
            break;
        }
        rc = oracle_attention_row(q + (size_t)r * H * D, sink, scale, cand, n, H, Dn, Dr, SB,
                                  out + (size_t)r * H * D, lse + (size_t)r * H);
    }
    free(cand);
    free(sel);
    return rc;
}

/* a4 standalone: the packed candidate records of each query row, byte for
 * byte: kv_out [B,T,k+W,rec] gets the selected records then the window;
 * kv_cnt [B,T] the number written. Slots past the count are not touched. */
int oracle_gather(const uint8_t *comp, int64_t seq_stride, const int32_t *block_table,
                  int page_records, int max_pages, int64_t n_records, int seq_capacity,
                  const uint8_t *ring, int R, int W,
                  const int32_t *topk_idx, const int32_t *topk_cnt, const int32_t *q_pos,
                  int B, int T, int k, int rec_bytes, int row_begin, int row_end,
                  uint8_t *kv_out, int32_t *kv_cnt)
{
    int r, rc = ORACLE_OK;
    const uint8_t **cand;
    if (row_begin < 0 || row_end > B * T || k < 0 || W < 0 || R < 1)
        return ORACLE_BAD_ARG;
    cand = (const uint8_t **)malloc(sizeof(*cand) * (size_t)(k + W + 1));
    if (!cand)
        return ORACLE_NO_MEMORY;
    for (r = row_begin; r < row_end; ++r) {
        int b = r / T, cnt = topk_cnt[r], n, i;
        if (cnt < 0 || cnt > k) {
            rc = ORACLE_BAD_ARG;
            break;
        }
        n = csa_candidates(comp, seq_stride, block_table, page_records, max_pages, n_records,
                           seq_capacity, ring, R, W, rec_bytes, topk_idx + (size_t)r * k, cnt,
                           b, q_pos[r], cand);
        if (n < 0) {
            rc = ORACLE_BAD_INDEX;
            break;
        }
        for (i = 0; i < n; ++i)
            memcpy(kv_out + ((size_t)r * (k + W) + i) * rec_bytes, cand[i], (size_t)rec_bytes);
        kv_cnt[r] = n;
    }
    free(cand);
    return rc;
}

/* ------------------------------------------------------------------------ */
/* Attention output epilogue                                                 */
/* ------------------------------------------------------------------------ */

/* OCP FP4 E2M1 (the low 4 bits of `code`): sign bit 3, exponent bits 2..1
 * (bias 1), mantissa bit 0; exponent 0 is subnormal (mantissa / 2). The
 * magnitudes are 0, 0.5, 1, 1.5, 2, 3, 4, 6; there is no infinity or NaN.
 * [ROADMAP] E6 names E2M1 as the format of the attention's FP4 output. */
double oracle_e2m1_value(uint8_t code)
{
    int sign = (code >> 3) & 1;
    int expo = (code >> 1) & 3;
    int mant = code & 1;
    double mag = expo == 0 ? (double)mant / 2.0 : ldexp(1.0 + (double)mant / 2.0, expo - 1);
    return sign ? -mag : mag;
}

/* The E2M1 code nearest to v: among the eight magnitudes the one closest to
 * |v|, a tie going to the code with mantissa bit 0 (round half to even);
 * magnitudes above 6 give 6 (saturation). The sign bit is v's sign bit, so a
 * negative value that rounds to zero gives the negative-zero code 8. */
uint8_t oracle_e2m1_code(double v)
{
    double a = fabs(v) > 6.0 ? 6.0 : fabs(v), best_d = INFINITY;  /* saturation */
    int c, best = 0;
    for (c = 0; c < 8; ++c) {
        double d = fabs(oracle_e2m1_value((uint8_t)c) - a);
        if (d < best_d || (d == best_d && (c & 1) == 0 && (best & 1) == 1)) {
            best_d = d;
            best = c;
        }
    }
    return (uint8_t)(best | (signbit(v) ? 8 : 0));
}

/* E2M1 quantisation of x[0..n) in blocks of `block` elements (ragged last
 * block) ([ROADMAP] E6: an E2M1 pack with a per-128-element block amax).
 * Reading: block i's multiplier is s_i = amax_i / 6 (the largest E2M1
 * magnitude), 1 for an all-zero block, so that x ~ e2m1 * s_i;
 * codes[d] = the E2M1 code nearest to x[d] / s_i, one code per byte. */
void oracle_e2m1_quantize(const double *x, int n, int block, uint8_t *codes, double *scales)
{
    int b0, d;
    for (b0 = 0; b0 < n; b0 += block) {
        int b1 = b0 + block < n ? b0 + block : n;
        double amax = 0.0, s;
        for (d = b0; d < b1; ++d)
            if (fabs(x[d]) > amax)
                amax = fabs(x[d]);
        s = amax > 0.0 ? amax / 6.0 : 1.0;
        scales[b0 / block] = s;
        for (d = b0; d < b1; ++d)
            codes[d] = oracle_e2m1_code(x[d] / s);
    }
}

/* Inverse RoPE on one attention output row o[0..Dn+Dr) ([AUDIT] A4: the
 * output is rotated by RoPE(-t) at the query position t, turning the absolute
 * positions carried by the summed latents into relative ones). Reading (the
 * pages give no convention): the rope dims are [Dn, Dn+Dr); pair i is
 * (Dn+2i, Dn+2i+1) and turns by t * theta^(-2i/Dr) radians at position t;
 * the inverse turns it back by the same angle:
 *   x' = x cos(a) + y sin(a),  y' = -x sin(a) + y cos(a),  a = t theta^(-2i/Dr).
 * The nope dims are left as they are. */
void oracle_inverse_rope(double *o, int Dn, int Dr, int pos, double theta)
{
    int i;
    for (i = 0; i < Dr / 2; ++i) {
        double a = (double)pos * pow(theta, -2.0 * (double)i / (double)Dr);
        double c = cos(a), s = sin(a);
        double x = o[Dn + 2 * i], y = o[Dn + 2 * i + 1];
        o[Dn + 2 * i] = x * c + y * s;
        o[Dn + 2 * i + 1] = -x * s + y * c;
    }
}
