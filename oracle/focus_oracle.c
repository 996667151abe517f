/*
 * Focus attention oracle -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow CPU restatement of what the Focus inference path computes,
 * used to check the CUDA kernels.  Only the tests, the smoke check and the
 * benchmark's CPU-baseline leg may load it; the product path never does.
 * It shares no code, header, table or helper with the CUDA library.
 *
 * Sources (web summaries of arXiv 2604.03260, "Why Attend to Everything?
 * Focus is the Key"):
 *   [NL]  gist.science/nl, "Technische samenvatting", Methodologie,
 *         Kerncomponenten 1 (centroid system), 3 (attention mechanism),
 *         4 (inference vs training).
 *   [ZH]  gist.science/zh, technical summary, section 2.1 "core
 *         architecture": 2.1.1 token grouping, 2.1.2 gated attention,
 *         2.1.3 inference optimisation (top-k discretisation).
 *   [NL]  Kerncomponenten 2 and [ZH] 2.1.1 also name the Sinkhorn
 *         normalisation of the training-time assignment (oracle_sinkhorn),
 *         and [ZH] 2.1.2 the soft gate of training (oracle_gated_fwd/bwd).
 *
 * Arithmetic: every dot product and softmax sum is accumulated in double;
 * scores and outputs are rounded to float once.  bf16 inputs arrive as raw
 * 16-bit patterns and are widened exactly.
 *
 * Readings taken where the pages are silent (all listed in the design
 * notes): score = (x W_g) . C_c (a plain dot product); the top-k ids are
 * returned in descending score with ties going to the lower centroid id;
 * the local window admits i - j < w; attention is causal (j <= i); the
 * softmax scale defaults to 1/sqrt(d); query head h reads kv head
 * h / (Hq / Hkv).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

static double bf16_bits_to_double(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* -------------------------------------------------------------------------
 * Group assignment, [ZH] 2.1.1 and 2.1.3, [NL] Kerncomponenten 1 and 4:
 * the hidden state is projected into centroid space (z = x W_g), scored
 * against every centroid (s_c = z . C_c), and at inference each token joins
 * its k highest-scoring groups.
 *
 * X      [ntok, hidden]  bf16 bit patterns
 * Wg     [hidden, dg]    float
 * C      [K, dg]         float
 * ids    [ntok, topk]    out: group ids by descending score, ties -> lower id
 * margin [ntok]          out (nullable): smallest gap between consecutive
 *                        scores among the top min(topk+1, K); +inf if K == 1
 * scores [ntok, K]       out (nullable): the float scores
 * ------------------------------------------------------------------------- */
int oracle_assign(const uint16_t *X, const float *Wg, const float *C,
                  int64_t ntok, int hidden, int dg, int K, int topk,
                  int32_t *ids, float *margin, float *scores)
{
    if (!X || !Wg || !C || !ids || ntok < 0 || hidden < 1 || dg < 1 ||
        K < 1 || topk < 1 || topk > K)
        return 1;
    int64_t t;
#pragma omp parallel for schedule(dynamic, 16)
    for (t = 0; t < ntok; ++t) {
        double *z = (double *)malloc(sizeof(double) * (size_t)dg);
        float *s = (float *)malloc(sizeof(float) * (size_t)K);
        char *taken = (char *)calloc((size_t)K, 1);
        const uint16_t *x = X + t * (int64_t)hidden;
        for (int c = 0; c < dg; ++c) z[c] = 0.0;
        for (int h = 0; h < hidden; ++h) {
            double xh = bf16_bits_to_double(x[h]);
            const float *w = Wg + (int64_t)h * dg;
            for (int c = 0; c < dg; ++c) z[c] += xh * (double)w[c];
        }
        for (int g = 0; g < K; ++g) {
            double acc = 0.0;
            const float *cg = C + (int64_t)g * dg;
            for (int c = 0; c < dg; ++c) acc += z[c] * (double)cg[c];
            s[g] = (float)acc;
        }
        if (scores) memcpy(scores + t * (int64_t)K, s, sizeof(float) * (size_t)K);
        /* Selection of the top min(topk+1, K) scores, one at a time: the
         * first strictly larger score wins, so equal scores keep the lower id. */
        int nsel = topk + 1 <= K ? topk + 1 : K;
        float prev = 0.0f, gap = INFINITY;
        for (int r = 0; r < nsel; ++r) {
            int best = -1;
            for (int g = 0; g < K; ++g)
                if (!taken[g] && (best < 0 || s[g] > s[best])) best = g;
            taken[best] = 1;
            if (r < topk) ids[t * topk + r] = best;
            if (r > 0) {
                float dlt = prev - s[best];
                if (dlt < gap) gap = dlt;
            }
            prev = s[best];
        }
        if (margin) margin[t] = gap;
        free(z);
        free(s);
        free(taken);
    }
    return 0;
}

/* -------------------------------------------------------------------------
 * Group lists.  Not on the pages; implied by running attention "within each
 * group" ([ZH] 2.1.3): the members of group g, in ascending token order.
 * Per batch b: offsets[b][g] = number of (token, slot) memberships of groups
 * < g; pos[b][offsets[g] + r] = the r-th smallest token of group g;
 * inv[b][i][s] = the index in pos[b] where (i, ids[b][i][s]) sits.
 * ------------------------------------------------------------------------- */
int oracle_bucket(const int32_t *ids, int B, int n, int K, int topk,
                  int32_t *offsets, int32_t *pos, int32_t *inv)
{
    if (!ids || !offsets || !pos || !inv || B < 1 || n < 0 || K < 1 || topk < 1)
        return 1;
    int32_t *fill = (int32_t *)malloc(sizeof(int32_t) * (size_t)K);
    for (int b = 0; b < B; ++b) {
        const int32_t *idb = ids + (int64_t)b * n * topk;
        int32_t *off = offsets + (int64_t)b * (K + 1);
        int32_t *pb = pos + (int64_t)b * n * topk;
        int32_t *ib = inv + (int64_t)b * n * topk;
        for (int g = 0; g <= K; ++g) off[g] = 0;
        for (int64_t e = 0; e < (int64_t)n * topk; ++e) {
            int g = idb[e];
            if (g < 0 || g >= K) { free(fill); return 1; }
            off[g + 1] += 1;
        }
        for (int g = 0; g < K; ++g) off[g + 1] += off[g];
        for (int g = 0; g < K; ++g) fill[g] = 0;
        for (int i = 0; i < n; ++i)
            for (int s = 0; s < topk; ++s) {
                int g = idb[(int64_t)i * topk + s];
                int32_t r = off[g] + fill[g]++;
                pb[r] = i;
                ib[(int64_t)i * topk + s] = r;
            }
    }
    free(fill);
    return 0;
}

/* Do tokens i and j share at least one of their top-k groups?
 * [ZH] 2.1.2 "only if the two tokens belong to the same group (or share at
 * least one group, see top-k)". */
static int share_group(const int32_t *gi, const int32_t *gj, int topk)
{
    for (int a = 0; a < topk; ++a)
        for (int b = 0; b < topk; ++b)
            if (gi[a] == gj[b]) return 1;
    return 0;
}

/* The allowed-pair rule, [NL] Kerncomponenten 3 and [ZH] 2.1.2, made causal
 * by [ZH] 2.1.3 ("within-group causal attention"): key j is visible to
 * query i iff j <= i and (i - j < window or the two share a group). */
static int allowed(const int32_t *ids_b, int topk, int window, int64_t i, int64_t j)
{
    if (j > i) return 0;
    if (i - j < (int64_t)window) return 1;
    return share_group(ids_b + i * topk, ids_b + j * topk, topk);
}

/* -------------------------------------------------------------------------
 * Exact softmax attention restricted to the allowed pairs, [NL]
 * Kerncomponenten 3 ("scores computed with exact softmax within the allowed
 * pairs").
 *
 * Q [B, n, Hq, d], Kt/V [B, n, Hkv, d]  bf16 bit patterns
 * ids [B, n, topk]
 * rows: nrows flattened query indices b*n + i (NULL: all B*n rows, in order)
 * q_rows_only: if non-zero (and rows given), Q holds only the sampled rows,
 *     [nrows, Hq, d], in the order of `rows`
 * O   [nrows, Hq, d] float out;  LSE [nrows, Hq] float out (natural log),
 *     nullable.  A row with no allowed key cannot occur (j = i is always
 *     allowed because a token shares its own groups).
 * scale <= 0 selects 1/sqrt(d).
 * ------------------------------------------------------------------------- */
int oracle_attention(const uint16_t *Q, const uint16_t *Kt, const uint16_t *V,
                     int B, int n, int Hq, int Hkv, int d, int window, float scale,
                     const int32_t *ids, int topk,
                     const int64_t *rows, int64_t nrows, int q_rows_only,
                     float *O, float *LSE)
{
    if (!Q || !Kt || !V || !ids || !O || B < 1 || n < 1 || Hq < 1 || Hkv < 1 ||
        Hq % Hkv != 0 || d < 1 || window < 0 || topk < 1)
        return 1;
    if (!rows) nrows = (int64_t)B * n;
    const double sc = scale > 0.0f ? (double)scale : 1.0 / sqrt((double)d);
    const int grp = Hq / Hkv;
    int64_t r;
#pragma omp parallel for schedule(dynamic, 1)
    for (r = 0; r < nrows; ++r) {
        int64_t flat = rows ? rows[r] : r;
        int b = (int)(flat / n);
        int64_t i = flat % n;
        const int32_t *ids_b = ids + (int64_t)b * n * topk;
        int64_t *J = (int64_t *)malloc(sizeof(int64_t) * (size_t)(i + 1));
        int64_t nj = 0;
        for (int64_t j = 0; j <= i; ++j)
            if (allowed(ids_b, topk, window, i, j)) J[nj++] = j;
        double *t = (double *)malloc(sizeof(double) * (size_t)(nj ? nj : 1));
        double *acc = (double *)malloc(sizeof(double) * (size_t)d);
        for (int h = 0; h < Hq; ++h) {
            int kvh = h / grp;
            const int64_t qrow = (rows && q_rows_only) ? r : (int64_t)b * n + i;
            const uint16_t *q = Q + (qrow * Hq + h) * d;
            double m = -INFINITY;
            for (int64_t a = 0; a < nj; ++a) {
                const uint16_t *k = Kt + (((int64_t)b * n + J[a]) * Hkv + kvh) * d;
                double dot = 0.0;
                for (int e = 0; e < d; ++e)
                    dot += bf16_bits_to_double(q[e]) * bf16_bits_to_double(k[e]);
                t[a] = sc * dot;
                if (t[a] > m) m = t[a];
            }
            double l = 0.0;
            for (int e = 0; e < d; ++e) acc[e] = 0.0;
            for (int64_t a = 0; a < nj; ++a) {
                double p = exp(t[a] - m);
                l += p;
                const uint16_t *v = V + (((int64_t)b * n + J[a]) * Hkv + kvh) * d;
                for (int e = 0; e < d; ++e) acc[e] += p * bf16_bits_to_double(v[e]);
            }
            float *o = O + (r * Hq + h) * d;
            for (int e = 0; e < d; ++e) o[e] = (float)(acc[e] / l);
            if (LSE) LSE[r * Hq + h] = (float)(m + log(l));
        }
        free(J);
        free(t);
        free(acc);
    }
    return 0;
}

/* -------------------------------------------------------------------------
 * |A_i|: the number of allowed keys of every query row (the work the
 * method does), by direct enumeration of the rule above.
 * rows: nrows flattened query indices b*n + i (NULL: all B*n rows, in order)
 * per_query [nrows] (nullable); the sum over those rows goes to *total.
 * ------------------------------------------------------------------------- */
int oracle_count_pairs(const int32_t *ids, int B, int n, int topk, int window,
                       const int64_t *rows, int64_t nrows,
                       int64_t *per_query, int64_t *total)
{
    if (!ids || !total || B < 1 || n < 0 || topk < 1 || window < 0) return 1;
    if (!rows) nrows = (int64_t)B * n;
    int64_t sum = 0;
    int64_t r;
#pragma omp parallel for schedule(dynamic, 64) reduction(+ : sum)
    for (r = 0; r < nrows; ++r) {
        int64_t flat = rows ? rows[r] : r;
        int b = (int)(flat / n);
        int64_t i = flat % n;
        const int32_t *ids_b = ids + (int64_t)b * n * topk;
        int64_t c = 0;
        for (int64_t j = 0; j <= i; ++j) c += allowed(ids_b, topk, window, i, j);
        if (per_query) per_query[r] = c;
        sum += c;
    }
    *total = sum;
    return 0;
}

/*
 * Sinkhorn normalisation of token-group affinities ([NL] Kerncomponenten 2:
 * balance forced as a hard structural constraint; [ZH] 2.1.1: Sinkhorn in
 * place of softmax, so that every group receives an equal mass of tokens).
 *
 * The pages name the algorithm but not its parameters; the readings taken:
 * kernel A_ic = exp(S_ic / tau); target masses a_i = 1 per token (each
 * token's assignment is a distribution over the K groups) and b_c = n / K
 * per group (equal mass); `iters` rounds of the Sinkhorn-Knopp scaling,
 * each a row update then a column update, in the log domain:
 *     log u_i = log a_i - log sum_c A_ic v_c
 *     log v_c = log b_c - log sum_i A_ic u_i
 * starting from v = 1, and P = diag(u) A diag(v).  Every sequence of the
 * batch is normalised on its own.  Sums are taken as max + log sum exp in
 * double.
 *
 *   S      [B, n, K] float
 *   P      [B, n, K] double out (nullable)
 *   log_u  [B, n]    double out (nullable)
 *   log_v  [B, K]    double out (nullable)
 */
int oracle_sinkhorn(const float *S, int B, int n, int K, double tau, int iters,
                    double *P, double *log_u, double *log_v)
{
    if (B < 1 || n < 1 || K < 1 || !(tau > 0.0) || iters < 1) return 1;
    double *lu = (double *)malloc(sizeof(double) * (size_t)n);
    double *lv = (double *)malloc(sizeof(double) * (size_t)K);
    if (!lu || !lv) {
        free(lu);
        free(lv);
        return 2;
    }
    const double log_a = 0.0, log_b = log((double)n / (double)K);
    for (int b = 0; b < B; ++b) {
        const float *Sb = S + (size_t)b * n * K;
        for (int c = 0; c < K; ++c) lv[c] = 0.0;
        for (int t = 0; t < iters; ++t) {
            /* rows: u_i = a_i / sum_c A_ic v_c */
#pragma omp parallel for schedule(static)
            for (int i = 0; i < n; ++i) {
                double m = -INFINITY;
                for (int c = 0; c < K; ++c) {
                    const double x = (double)Sb[(size_t)i * K + c] / tau + lv[c];
                    if (x > m) m = x;
                }
                double sum = 0.0;
                for (int c = 0; c < K; ++c)
                    sum += exp((double)Sb[(size_t)i * K + c] / tau + lv[c] - m);
                lu[i] = log_a - (m + log(sum));
            }
            /* columns: v_c = b_c / sum_i A_ic u_i */
#pragma omp parallel for schedule(static)
            for (int c = 0; c < K; ++c) {
                double m = -INFINITY;
                for (int i = 0; i < n; ++i) {
                    const double y = (double)Sb[(size_t)i * K + c] / tau + lu[i];
                    if (y > m) m = y;
                }
                double sum = 0.0;
                for (int i = 0; i < n; ++i)
                    sum += exp((double)Sb[(size_t)i * K + c] / tau + lu[i] - m);
                lv[c] = log_b - (m + log(sum));
            }
        }
        if (P)
#pragma omp parallel for schedule(static)
            for (int i = 0; i < n; ++i)
                for (int c = 0; c < K; ++c)
                    P[((size_t)b * n + i) * K + c] =
                        exp((double)Sb[(size_t)i * K + c] / tau + lu[i] + lv[c]);
        if (log_u)
            for (int i = 0; i < n; ++i) log_u[(size_t)b * n + i] = lu[i];
        if (log_v)
            for (int c = 0; c < K; ++c) log_v[(size_t)b * K + c] = lv[c];
    }
    free(lu);
    free(lv);
    return 0;
}

/*
 * Soft-gated attention of training ([ZH] 2.1.2 gated attention; [NL]
 * Kerncomponent 4: during training every pair is computed, with soft
 * gates).  The page prints the score as
 *     s_ij = q_i . k_j * (1_local + (1 - 1_local) * sigma(lambda * a_ij))
 * with a_ij the group affinity of tokens i and j.  Readings taken where the
 * page leaves it open: 1_local = [i - j < w]; a_ij = g_i . g_j, the dot
 * product of the two tokens' soft group assignments (rows of G, e.g. the
 * Sinkhorn-normalised affinities); lambda a scalar; q . k scaled by `scale`
 * (1/sqrt(d) when <= 0) before the gate; causal softmax over j <= i.
 *
 *   Q [B, n, Hq, d], K and V [B, n, Hkv, d] bf16 bits; G [B, n, Kg] float
 *   O [B, n, Hq, d] double out; LSE [B, Hq, n] double out (natural log)
 * oracle_gated_bwd takes dO [B, n, Hq, d] float and returns the gradients
 * of sum(O * dO): dQ [B, n, Hq, d], dK and dV [B, n, Hkv, d], dG [B, n, Kg]
 * (all double, overwritten) and d lambda; dlambda_abs (nullable) receives
 * the sum of the magnitudes of d lambda's per-pair terms, the scale against
 * which a rounded evaluation of that (often cancelling) sum is judged.
 */
static double gated_score(const uint16_t *q, const uint16_t *k, const float *gi,
                          const float *gj, int d, int Kg, double sc, double lambda, int local,
                          double *t_out, double *a_out, double *gate_out)
{
    double dot = 0.0;
    for (int e = 0; e < d; ++e) dot += bf16_bits_to_double(q[e]) * bf16_bits_to_double(k[e]);
    double a = 0.0;
    for (int c = 0; c < Kg; ++c) a += (double)gi[c] * (double)gj[c];
    const double gate = local ? 1.0 : 1.0 / (1.0 + exp(-lambda * a));
    *t_out = sc * dot;
    *a_out = a;
    *gate_out = gate;
    return sc * dot * gate;
}

int oracle_gated_fwd(const uint16_t *Q, const uint16_t *Kt, const uint16_t *V, const float *G,
                     int B, int n, int Hq, int Hkv, int d, int Kg, int window, double lambda,
                     double scale, double *O, double *LSE)
{
    if (!Q || !Kt || !V || !G || !O || B < 1 || n < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv ||
        d < 1 || Kg < 1 || window < 0)
        return 1;
    const double sc = scale > 0.0 ? scale : 1.0 / sqrt((double)d);
    const int grp = Hq / Hkv;
    int bh;
#pragma omp parallel for schedule(dynamic, 1)
    for (bh = 0; bh < B * Hq; ++bh) {
        const int b = bh / Hq, h = bh % Hq, kvh = h / grp;
        double *s = (double *)malloc(sizeof(double) * (size_t)n);
        for (int i = 0; i < n; ++i) {
            const uint16_t *q = Q + (((size_t)b * n + i) * Hq + h) * d;
            const float *gi = G + ((size_t)b * n + i) * Kg;
            double m = -INFINITY;
            for (int j = 0; j <= i; ++j) {
                double t, a, gate;
                s[j] = gated_score(q, Kt + (((size_t)b * n + j) * Hkv + kvh) * d, gi,
                                   G + ((size_t)b * n + j) * Kg, d, Kg, sc, lambda,
                                   i - j < window, &t, &a, &gate);
                if (s[j] > m) m = s[j];
            }
            double l = 0.0;
            double *o = O + (((size_t)b * n + i) * Hq + h) * d;
            for (int e = 0; e < d; ++e) o[e] = 0.0;
            for (int j = 0; j <= i; ++j) {
                const double p = exp(s[j] - m);
                l += p;
                const uint16_t *v = V + (((size_t)b * n + j) * Hkv + kvh) * d;
                for (int e = 0; e < d; ++e) o[e] += p * bf16_bits_to_double(v[e]);
            }
            for (int e = 0; e < d; ++e) o[e] /= l;
            if (LSE) LSE[((size_t)b * Hq + h) * n + i] = m + log(l);
        }
        free(s);
    }
    return 0;
}

int oracle_gated_bwd(const uint16_t *Q, const uint16_t *Kt, const uint16_t *V, const float *G,
                     const float *dO, int B, int n, int Hq, int Hkv, int d, int Kg, int window,
                     double lambda, double scale, double *dQ, double *dK, double *dV,
                     double *dG, double *dlambda, double *dlambda_abs)
{
    if (!Q || !Kt || !V || !G || !dO || !dQ || !dK || !dV || !dG || !dlambda || B < 1 ||
        n < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv || d < 1 || Kg < 1 || window < 0)
        return 1;
    const double sc = scale > 0.0 ? scale : 1.0 / sqrt((double)d);
    const int grp = Hq / Hkv;
    memset(dQ, 0, sizeof(double) * (size_t)B * n * Hq * d);
    memset(dK, 0, sizeof(double) * (size_t)B * n * Hkv * d);
    memset(dV, 0, sizeof(double) * (size_t)B * n * Hkv * d);
    memset(dG, 0, sizeof(double) * (size_t)B * n * Kg);
    double dl = 0.0, dl_abs = 0.0;
    double *s = (double *)malloc(sizeof(double) * (size_t)n);
    double *t = (double *)malloc(sizeof(double) * (size_t)n);
    double *a = (double *)malloc(sizeof(double) * (size_t)n);
    double *gate = (double *)malloc(sizeof(double) * (size_t)n);
    double *dp = (double *)malloc(sizeof(double) * (size_t)n);
    for (int b = 0; b < B; ++b)
        for (int h = 0; h < Hq; ++h) {
            const int kvh = h / grp;
            for (int i = 0; i < n; ++i) {
                const uint16_t *q = Q + (((size_t)b * n + i) * Hq + h) * d;
                const float *gi = G + ((size_t)b * n + i) * Kg;
                const float *go = dO + (((size_t)b * n + i) * Hq + h) * d;
                double m = -INFINITY;
                for (int j = 0; j <= i; ++j) {
                    s[j] = gated_score(q, Kt + (((size_t)b * n + j) * Hkv + kvh) * d, gi,
                                       G + ((size_t)b * n + j) * Kg, d, Kg, sc, lambda,
                                       i - j < window, &t[j], &a[j], &gate[j]);
                    if (s[j] > m) m = s[j];
                }
                double l = 0.0;
                for (int j = 0; j <= i; ++j) l += exp(s[j] - m);
                /* P_ij, dP_ij = dO_i . v_j, D_i = sum_j P_ij dP_ij */
                double D = 0.0;
                for (int j = 0; j <= i; ++j) {
                    const uint16_t *v = V + (((size_t)b * n + j) * Hkv + kvh) * d;
                    double x = 0.0;
                    for (int e = 0; e < d; ++e) x += (double)go[e] * bf16_bits_to_double(v[e]);
                    dp[j] = x;
                    D += exp(s[j] - m) / l * x;
                }
                for (int j = 0; j <= i; ++j) {
                    const double P = exp(s[j] - m) / l;
                    const double ds = P * (dp[j] - D);     /* d sum(O dO) / d s_ij */
                    const double dt = ds * gate[j];
                    const uint16_t *k = Kt + (((size_t)b * n + j) * Hkv + kvh) * d;
                    double *dq = dQ + (((size_t)b * n + i) * Hq + h) * d;
                    double *dk = dK + (((size_t)b * n + j) * Hkv + kvh) * d;
                    double *dv = dV + (((size_t)b * n + j) * Hkv + kvh) * d;
                    for (int e = 0; e < d; ++e) {
                        dq[e] += sc * dt * bf16_bits_to_double(k[e]);
                        dk[e] += sc * dt * bf16_bits_to_double(q[e]);
                        dv[e] += P * (double)go[e];
                    }
                    if (!(i - j < window)) {
                        const double dgate = ds * t[j];
                        const double sp = gate[j] * (1.0 - gate[j]);   /* sigma' */
                        const double da = dgate * lambda * sp;
                        dl += dgate * a[j] * sp;
                        dl_abs += fabs(dgate * a[j] * sp);
                        const float *gj = G + ((size_t)b * n + j) * Kg;
                        double *dgi = dG + ((size_t)b * n + i) * Kg;
                        double *dgj = dG + ((size_t)b * n + j) * Kg;
                        for (int c = 0; c < Kg; ++c) {
                            dgi[c] += da * (double)gj[c];
                            dgj[c] += da * (double)gi[c];
                        }
                    }
                }
            }
        }
    free(s);
    free(t);
    free(a);
    free(gate);
    free(dp);
    *dlambda = dl;
    if (dlambda_abs) *dlambda_abs = dl_abs;
    return 0;
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    extern int omp_get_max_threads(void);
    return omp_get_max_threads();
#else
    return 1;
#endif
}
