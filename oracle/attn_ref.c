/*
 * attn_ref.c -- CPU oracle for single-query decode attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file; only the tests, the package smoke check and the CPU
 * baseline leg of the benchmark do.  It shares no code, header or constant
 * with the CUDA library.
 *
 * Everything is plain fp64 on the exact widening of the same bf16 input bits
 * the GPU reads.  Each function follows one passage of the source pages:
 *
 *   oracle_attend       -- the definition S = scale q K^T, P = softmax(S),
 *                          O = P V, with a full (not online) softmax and the
 *                          natural-log log-sum-exp of the scores.  Written
 *                          as in "FlashAttention 与推理算子" (standard
 *                          attention section; its CPU references
 *                          attention_cpu and the paged CPU reference that
 *                          walks the block table), restricted to one query
 *                          row and to a token range [t0, t1).  With
 *                          t0 = 0, t1 = L the result is the attention output;
 *                          a sub-range gives a split's normalised partial
 *                          output and its log-sum-exp (Flash-Decoding
 *                          section of the same page).
 *   oracle_lse_merge    -- the pass-2 merge of "纯手搓 flash decoding sm120"
 *                          section 2: lse_max = max lse_i,
 *                          G = lse_max + ln sum exp(lse_i - lse_max),
 *                          O = sum O_i exp(lse_i - G); segments with
 *                          lse = -inf are skipped (merge exercise of the
 *                          handbook page).
 *   oracle_online_blocks -- the online-softmax recurrence of the handbook's
 *                          FlashAttention section (m, l and O updated block
 *                          by block, O divided by l at the end), for one
 *                          query row with a vector value of width dv.
 *
 * q is bf16 or IEEE fp16 bit patterns (the first page's tensor-map helper
 * accepts either), widened exactly to fp64.  K and V hold the same 16-bit
 * type, or an 8-bit FP8 KV cache ("FlashAttention 与推理算子", the decode
 * kernel checklist: the KV cache is BF16 or FP8, converted to fp32 in
 * registers): OCP FP8 E4M3 or E5M2 codes, each tensor with one
 * dequantisation scale, K_t = k_scale * decode(k8_t) and likewise V.
 *
 * GQA head mapping: query head h reads kv head h / (Hq / Hkv) (consecutive
 * query heads share a kv head).  Paged layout: token t of request b lives
 * in physical page block_table[b][t / P], slot t % P.
 *
 * Several new query tokens per request (q_len > 1): the cache of length L
 * already holds them, and new token i (0-based) sits at position
 * L - q_len + i, so under the causal mask of the handbook's FlashAttention
 * section (query i sees only the keys up to its own position) it attends to
 * tokens [0, L - q_len + i].  q and O are [B, q_len, Hq, D].
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

static double bf16_to_f64(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* IEEE binary16: 1 sign, 5 exponent (bias 15), 10 fraction bits. */
static double f16_to_f64(uint16_t bits)
{
    const int sign = bits >> 15, e = (bits >> 10) & 31, m = bits & 1023;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24);              /* zero or subnormal: m * 2^-24 */
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(m + 1024), e - 25);  /* (1 + m/1024) * 2^(e-15) */
    return sign ? -v : v;
}

/* Element type of q: 0 = bf16, 1 = fp16. */
static double elem_to_f64(uint16_t bits, int dtype)
{
    return dtype ? f16_to_f64(bits) : bf16_to_f64(bits);
}

/* OCP 8-bit floating point, E4M3 ("fn" form): 1 sign, 4 exponent (bias 7),
 * 3 fraction bits; exponent 0 holds zero and the subnormals m * 2^-9; there
 * is no infinity, and S.1111.111 is NaN, so the largest value is 448. */
static double e4m3_to_f64(uint8_t bits)
{
    const int sign = bits >> 7, e = (bits >> 3) & 15, m = bits & 7;
    double v;
    if (e == 0)
        v = ldexp((double)m, -9);
    else if (e == 15 && m == 7)
        v = NAN;
    else
        v = ldexp((double)(m + 8), e - 10);   /* (1 + m/8) * 2^(e-7) */
    return sign ? -v : v;
}

/* OCP 8-bit floating point, E5M2: 1 sign, 5 exponent (bias 15), 2 fraction
 * bits, IEEE-style: subnormals m * 2^-16, infinities and NaNs at
 * exponent 31. */
static double e5m2_to_f64(uint8_t bits)
{
    const int sign = bits >> 7, e = (bits >> 2) & 31, m = bits & 3;
    double v;
    if (e == 0)
        v = ldexp((double)m, -16);
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(m + 4), e - 17);   /* (1 + m/4) * 2^(e-15) */
    return sign ? -v : v;
}

/* K/V element type: 0 = bf16, 1 = fp16, 2 = FP8 E4M3, 3 = FP8 E5M2. */
static int kv_elem_bytes(int kvtype) { return kvtype >= 2 ? 1 : 2; }

/* Element j of a K or V row, before its tensor's dequantisation scale. */
static double kv_elem(const uint8_t *row, int j, int kvtype)
{
    if (kvtype == 2)
        return e4m3_to_f64(row[j]);
    if (kvtype == 3)
        return e5m2_to_f64(row[j]);
    uint16_t bits;
    memcpy(&bits, row + 2 * (int64_t)j, sizeof bits);
    return elem_to_f64(bits, kvtype);
}

/* Where the K (or V) row of logical token t of request b, kv head g lives. */
typedef struct {
    const uint8_t *base;      /* K or V */
    int esize;                /* bytes per element */
    int paged;
    /* contiguous [B, S_max, Hkv, D] */
    int s_max;
    /* paged [num_pages, P, Hkv, D] */
    const int32_t *block_table;
    int max_blocks;
    int page;
    int num_pages;
    int hkv;
    int d;
} kv_view;

/* Returns NULL if the token's page is not a valid physical page. */
static const uint8_t *kv_row(const kv_view *w, int b, int t, int g)
{
    int64_t row;
    if (!w->paged) {
        row = ((int64_t)b * w->s_max + t) * w->hkv + g;
    } else {
        int32_t phys = w->block_table[(int64_t)b * w->max_blocks + t / w->page];
        if (phys < 0 || phys >= w->num_pages)
            return NULL;
        row = ((int64_t)phys * w->page + t % w->page) * w->hkv + g;
    }
    return w->base + row * w->d * w->esize;
}

/*
 * One query row (request b, query head h) against tokens [t0, t1).
 * Writes o[0..d) and *lse.  An empty range gives o = 0, lse = -inf.
 * Returns 0, or -1 when a referenced page is out of range.
 */
static int attend_one(const uint16_t *q, const kv_view *kw, const kv_view *vw,
                      int b, int i_tok, int q_len, int h, int hq, int t0, int t1, double scale,
                      int dtype, int kvtype, double k_scale, double v_scale,
                      double *s /* scratch, >= t1 - t0 */, double *o, double *lse)
{
    const int d = kw->d;
    const int group = hq / kw->hkv;
    const int g = h / group;
    const uint16_t *qrow = q + (((int64_t)b * q_len + i_tok) * hq + h) * d;
    const int n = t1 - t0;

    for (int j = 0; j < d; ++j)
        o[j] = 0.0;
    if (n <= 0) {
        *lse = -INFINITY;
        return 0;
    }

    /* S = scale * q . K_t, K_t = k_scale * (stored row) */
    double mx = -INFINITY;
    for (int i = 0; i < n; ++i) {
        const uint8_t *krow = kv_row(kw, b, t0 + i, g);
        if (!krow)
            return -1;
        double dot = 0.0;
        for (int j = 0; j < d; ++j)
            dot += elem_to_f64(qrow[j], dtype) * (k_scale * kv_elem(krow, j, kvtype));
        s[i] = scale * dot;
        if (s[i] > mx)
            mx = s[i];
    }

    /* P = exp(S - max) / Z ; LSE = max + ln Z */
    double z = 0.0;
    for (int i = 0; i < n; ++i) {
        s[i] = exp(s[i] - mx);
        z += s[i];
    }
    *lse = mx + log(z);

    /* O = sum_t P_t V_t */
    for (int i = 0; i < n; ++i) {
        const uint8_t *vrow = kv_row(vw, b, t0 + i, g);
        if (!vrow)
            return -1;
        const double p = s[i] / z;
        for (int j = 0; j < d; ++j)
            o[j] += p * (v_scale * kv_elem(vrow, j, kvtype));
    }
    return 0;
}

/*
 * dtype: 0 when q holds bf16 bit patterns, 1 for IEEE fp16.  kvtype: the
 * K/V element type (0 bf16, 1 fp16, 2 FP8 E4M3, 3 FP8 E5M2); k_scale and
 * v_scale multiply every decoded K and V element (1 for 16-bit caches).
 * q_len: new query tokens per request (q is [B, q_len, Hq, D]).
 * For each of npairs items (b, r, t0, t1) in `items` (int32, 4 per item),
 * query row r = i * Hq + h is new token i, query head h; t1 < 0 means "to
 * the causal end", the row's visible length max(0, L_b - q_len + i + 1).
 * It computes the attention of that query over tokens [t0, min(t1, L_b)).
 * o is [npairs][d], lse [npairs].
 * page_size == 0 selects the contiguous layout (k, v are [B, S_max, Hkv, D]);
 * otherwise k, v are pages [num_pages, P, Hkv, D] behind block_table.
 * scratch must hold max token count doubles.  Returns 0, or -1 on a bad page
 * or a length outside the layout.
 */
int oracle_attend(const uint16_t *q, const void *k, const void *v,
                  const int32_t *seq_lens, int batch, int hq, int hkv, int d,
                  int s_max, int page_size, const int32_t *block_table,
                  int max_blocks, int num_pages, double scale, int dtype,
                  int kvtype, double k_scale, double v_scale, int q_len,
                  const int32_t *items, int npairs, double *scratch,
                  double *o, double *lse)
{
    if (hkv <= 0 || hq % hkv != 0 || kvtype < 0 || kvtype > 3 || q_len < 1)
        return -1;
    kv_view kw = {(const uint8_t *)k, kv_elem_bytes(kvtype), page_size > 0, s_max, block_table,
                  max_blocks, page_size, num_pages, hkv, d};
    kv_view vw = kw;
    vw.base = (const uint8_t *)v;
    for (int i = 0; i < npairs; ++i) {
        const int b = items[4 * i + 0], r = items[4 * i + 1];
        int t0 = items[4 * i + 2], t1 = items[4 * i + 3];
        if (b < 0 || b >= batch || r < 0 || r >= q_len * hq)
            return -1;
        const int i_tok = r / hq, h = r % hq;
        const int L = seq_lens[b];
        if (L < 0)
            return -1;
        if (page_size == 0 && L > s_max)
            return -1;
        if (page_size > 0 && L > (int64_t)max_blocks * page_size)
            return -1;
        /* causal end of new token i_tok: it sees positions 0 .. L - q_len + i_tok */
        int end = L - q_len + i_tok + 1;
        if (end < 0)
            end = 0;
        if (t1 < 0 || t1 > end)
            t1 = end;
        if (t0 < 0)
            t0 = 0;
        if (attend_one(q, &kw, &vw, b, i_tok, q_len, h, hq, t0, t1, scale, dtype, kvtype, k_scale,
                       v_scale, scratch, o + (int64_t)i * d, lse + i) != 0)
            return -1;
    }
    return 0;
}

/*
 * Merge n partial results (normalised O_i [n][d], natural-log lse_i) into one
 * output o[d] and its log-sum-exp.  Partials with lse = -inf carry no tokens
 * and are skipped; if all are skipped, o = 0 and lse = -inf.
 */
void oracle_lse_merge(const double *o_parts, const double *lse_parts, int n, int d,
                      double *o, double *lse)
{
    double lse_max = -INFINITY;
    for (int i = 0; i < n; ++i)
        if (lse_parts[i] > lse_max)
            lse_max = lse_parts[i];
    for (int j = 0; j < d; ++j)
        o[j] = 0.0;
    if (lse_max == -INFINITY) {
        *lse = -INFINITY;
        return;
    }
    double sum = 0.0;
    for (int i = 0; i < n; ++i)
        if (lse_parts[i] != -INFINITY)
            sum += exp(lse_parts[i] - lse_max);
    const double g = lse_max + log(sum);
    for (int i = 0; i < n; ++i) {
        if (lse_parts[i] == -INFINITY)
            continue;
        const double w = exp(lse_parts[i] - g);
        for (int j = 0; j < d; ++j)
            o[j] += o_parts[(int64_t)i * d + j] * w;
    }
    *lse = g;
}

/*
 * Online softmax over one row of scores s[0..n) with value rows
 * val[n][dv], taken `block` scores at a time.  After block j it records
 * m_j, l_j and the unnormalised O_j (dv values) into m_out[j], l_out[j],
 * o_out[j][dv].  The final output is O_last / l_last, written to o_final.
 * Returns the number of blocks.
 */
int oracle_online_blocks(const double *s, const double *val, int n, int dv, int block,
                         double *m_out, double *l_out, double *o_out, double *o_final)
{
    double m = -INFINITY, l = 0.0;
    double acc[64];
    if (dv > 64 || block <= 0)
        return -1;
    for (int j = 0; j < dv; ++j)
        acc[j] = 0.0;
    int nb = 0;
    for (int b0 = 0; b0 < n; b0 += block, ++nb) {
        const int b1 = b0 + block < n ? b0 + block : n;
        double rowmax = -INFINITY;
        for (int i = b0; i < b1; ++i)
            if (s[i] > rowmax)
                rowmax = s[i];
        const double m_new = m > rowmax ? m : rowmax;
        const double corr = (m == -INFINITY) ? 0.0 : exp(m - m_new);
        double rowsum = 0.0;
        for (int j = 0; j < dv; ++j)
            acc[j] *= corr;
        for (int i = b0; i < b1; ++i) {
            const double p = exp(s[i] - m_new);
            rowsum += p;
            for (int j = 0; j < dv; ++j)
                acc[j] += p * val[(int64_t)i * dv + j];
        }
        l = corr * l + rowsum;
        m = m_new;
        m_out[nb] = m;
        l_out[nb] = l;
        for (int j = 0; j < dv; ++j)
            o_out[(int64_t)nb * dv + j] = acc[j];
    }
    for (int j = 0; j < dv; ++j)
        o_final[j] = (nb > 0) ? acc[j] / l : 0.0;
    return nb;
}
