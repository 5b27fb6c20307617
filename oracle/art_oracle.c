/*
 * art_oracle.c -- plain fp64 CPU oracle for ART decode attention.
 *
 * TEST INFRASTRUCTURE. Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this library. The product path
 * (the CUDA library) shares no code with it and never calls it.
 *
 * What it computes, per work item (sequence b, KV head g):
 *
 *   Scaled dot-product attention O = softmax(q K^T / sqrt(d)) V
 *   ("ART: Attention Run-time Termination", sec. 3.1, Eq. (1)), evaluated
 *   over the KV blocks of a visit list L in list order, together with the
 *   sequence of partial outputs O^(i), the attention output over only the
 *   first i listed blocks (ART paper, sec. 3.1, the partial outputs of
 *   block-wise attention).
 *
 *   The run-time termination rule (sec. 3.2 probe vector; explainer page
 *   gist.science "2.2 Stabilitaetsbasiertes Terminierungskriterium",
 *   "2.3 Geduld-Mechanismus", "2.4 Integration und Korrektheit"):
 *     x^(i)    = concat over the G query heads of the group of O^(i)_h[probe]
 *                (or over the first probe_heads of them: the paper's probe is
 *                a fragment of one head's output, sec. 3.2)
 *     n_i      = ||x^(i)||_2
 *     d_mag_i  = | n_i - n_{i-1} | / n_{i-1}                      (i >= 2)
 *     d_dir_i  = max(0, 1 - <x^(i), x^(i-1)> / (n_i n_{i-1}))     (i >= 2)
 *     stable_i = d_mag_i < eps_mag  and  d_dir_i < eps_dir
 *                (false if a norm is zero or a value is not finite)
 *     c_1 = 0,  c_i = stable_i ? c_{i-1} + 1 : 0
 *     stop at the first i with c_i >= patience whose prefix L[0..i-1]
 *     contains logical block 0, or at any such i if 0 is not in L;
 *     otherwise process all n listed blocks.
 *   The output is O^(blocks_used).
 *
 * The partial outputs are written out as their plain definition: with one
 * fixed shift M_h (the largest score of head h over the whole list),
 *   O^(i)_h = sum_{t in U_i} e^{s_ht - M_h} v_t / sum_{t in U_i} e^{s_ht - M_h},
 * accumulated as running prefix sums over the listed blocks. There is no
 * online rescaling, blocking or fusion.
 *
 * Layouts (all row-major, element type bf16 bits or fp32):
 *   q        [batch][num_q_heads][head_dim]
 *   k_cache  [num_pages_total][num_kv_heads][page_size][head_dim], v_cache same
 *   block_table [batch][max_pages_per_seq]   physical page of logical page j
 *   seq_lens [batch]
 *   visit_order [batch][num_kv_heads][max_visit] logical ART-block ids,
 *               terminated by the first -1; NULL means 0, 1, ..., T-1
 *   probe_idx [num_probe] head-dim indices
 * Query head h belongs to KV head h / (num_q_heads / num_kv_heads).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

typedef struct {
    int32_t batch, num_q_heads, num_kv_heads, head_dim, page_size, block_size;
    int32_t max_pages_per_seq, max_visit, num_probe, num_pages_total;
    int32_t dtype; /* 0 = bf16 bits (uint16), 1 = fp32 */
} oracle_shape;

enum {
    ORACLE_ITEM_OK = 0,
    ORACLE_ITEM_BAD_VISIT = 1,   /* visit entry outside [0, T)            */
    ORACLE_ITEM_BAD_PAGE = 2,    /* block_table entry outside the pool    */
    ORACLE_ITEM_DUP_VISIT = 3,   /* a block listed twice                  */
};

typedef struct {
    const oracle_shape *sh;
    const void *q, *k, *v;
    const int32_t *block_table, *seq_lens, *visit_order, *probe_idx;
    double eps_mag, eps_dir;
    int32_t patience;
    int32_t probe_heads; /* heads 0 .. probe_heads-1 of the group form the probe */
    int32_t mode; /* 0 = dense (all listed blocks), 1 = ART rule, 2 = forced */
    const int32_t *items;
    const int32_t *forced;
    int32_t num_items;
    double *out;
    int32_t *blocks_used, *item_status;
    double *trace_mag, *trace_dir;
    int32_t next;
    pthread_mutex_t lock;
} job_t;

static double load_elem(const void *base, int dtype, size_t idx)
{
    if (dtype == 1) return (double)((const float *)base)[idx];
    uint32_t bits = (uint32_t)((const uint16_t *)base)[idx] << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/* Physical element offset of (token t, dim e) of KV head g of sequence b. */
static size_t kv_offset(const oracle_shape *sh, int32_t page, int g, int t_in_page, int e)
{
    return (((size_t)page * sh->num_kv_heads + g) * sh->page_size + t_in_page) * sh->head_dim + e;
}

static void run_item(job_t *J, int slot)
{
    const oracle_shape *sh = J->sh;
    const int item = J->items ? J->items[slot] : slot;
    const int b = item / sh->num_kv_heads, g = item % sh->num_kv_heads;
    const int G = sh->num_q_heads / sh->num_kv_heads;
    const int d = sh->head_dim, Bk = sh->block_size, Ps = sh->page_size;
    const int m = sh->num_probe, mx = sh->max_visit;
    const int seq_len = J->seq_lens[b];
    const int T = seq_len > 0 ? (seq_len + Bk - 1) / Bk : 0;
    double *out = J->out + (size_t)slot * G * d;
    double *tmag = J->trace_mag ? J->trace_mag + (size_t)slot * mx : NULL;
    double *tdir = J->trace_dir ? J->trace_dir + (size_t)slot * mx : NULL;

    memset(out, 0, sizeof(double) * G * d);
    if (tmag) for (int i = 0; i < mx; ++i) tmag[i] = NAN;
    if (tdir) for (int i = 0; i < mx; ++i) tdir[i] = NAN;
    J->item_status[slot] = ORACLE_ITEM_OK;
    J->blocks_used[slot] = 0;

    /* Step 1: the visit list. */
    int n = 0;
    int32_t *L = (int32_t *)malloc(sizeof(int32_t) * (size_t)(T > mx ? T : mx) + 4);
    if (J->visit_order) {
        const int32_t *row = J->visit_order + (size_t)item * mx;
        while (n < mx && row[n] != -1) { L[n] = row[n]; ++n; }
    } else {
        for (int c = 0; c < T; ++c) L[c] = c;
        n = T;
    }
    char *seen = (char *)calloc((size_t)T + 1, 1);
    int has0 = 0;
    for (int i = 0; i < n; ++i) {
        if (L[i] < 0 || L[i] >= T) { J->item_status[slot] = ORACLE_ITEM_BAD_VISIT; break; }
        if (seen[L[i]]) { J->item_status[slot] = ORACLE_ITEM_DUP_VISIT; break; }
        seen[L[i]] = 1;
        if (L[i] == 0) has0 = 1;
    }
    free(seen);
    if (J->item_status[slot] != ORACLE_ITEM_OK) { J->blocks_used[slot] = -1; free(L); return; }
    if (n == 0) { free(L); return; }

    /* Step 2: token rows of every listed block, resolved through the table. */
    size_t ntok = 0;
    for (int i = 0; i < n; ++i) {
        int lo = L[i] * Bk, hi = lo + Bk < seq_len ? lo + Bk : seq_len;
        ntok += (size_t)(hi - lo);
    }
    size_t *row_off = (size_t *)malloc(sizeof(size_t) * ntok); /* offset of (t, e=0) */
    int *blk_end = (int *)malloc(sizeof(int) * (size_t)(unsigned)n);            /* tokens in U_i */
    size_t r = 0;
    for (int i = 0; i < n && J->item_status[slot] == ORACLE_ITEM_OK; ++i) {
        int lo = L[i] * Bk, hi = lo + Bk < seq_len ? lo + Bk : seq_len;
        for (int t = lo; t < hi; ++t) {
            int32_t page = J->block_table[(size_t)b * sh->max_pages_per_seq + t / Ps];
            if (page < 0 || page >= sh->num_pages_total) {
                J->item_status[slot] = ORACLE_ITEM_BAD_PAGE;
                break;
            }
            row_off[r++] = kv_offset(sh, page, g, t % Ps, 0);
        }
        blk_end[i] = (int)r;
    }
    if (J->item_status[slot] != ORACLE_ITEM_OK) {
        J->blocks_used[slot] = -1;
        free(row_off); free(blk_end); free(L);
        return;
    }

    /* Step 3: scores s_ht = q_h . k_t / sqrt(d) for every listed token. */
    double *qd = (double *)malloc(sizeof(double) * G * d);
    for (int h = 0; h < G; ++h)
        for (int e = 0; e < d; ++e)
            qd[h * d + e] = load_elem(J->q, sh->dtype,
                                      ((size_t)b * sh->num_q_heads + (size_t)g * G + h) * d + e);
    double *s = (double *)malloc(sizeof(double) * ntok * G);
    const double inv_sqrt_d = 1.0 / sqrt((double)d);
    double *Mh = (double *)malloc(sizeof(double) * G);
    for (int h = 0; h < G; ++h) Mh[h] = -INFINITY;
    double *kv = (double *)malloc(sizeof(double) * d);
    for (size_t t = 0; t < ntok; ++t) {
        for (int e = 0; e < d; ++e) kv[e] = load_elem(J->k, sh->dtype, row_off[t] + e);
        for (int h = 0; h < G; ++h) {
            double acc = 0.0;
            for (int e = 0; e < d; ++e) acc += qd[h * d + e] * kv[e];
            s[t * G + h] = acc * inv_sqrt_d;
            if (s[t * G + h] > Mh[h]) Mh[h] = s[t * G + h];
        }
    }

    /* Steps 4-8: prefix sums at the probe columns, statistics and rule. */
    int bu = n;
    if (J->mode == 2) {
        bu = J->forced[slot];
        if (bu < 0) bu = 0;
        if (bu > n) bu = n;
    } else if (J->mode == 1) {
        double *Z = (double *)calloc((size_t)G, sizeof(double));
        double *Nm = (double *)calloc((size_t)G * m, sizeof(double));
        double *x = (double *)malloc(sizeof(double) * G * m);
        double *xp = (double *)malloc(sizeof(double) * G * m);
        double nprev = 0.0;
        int counter = 0, seen0 = 0;
        bu = n;
        size_t t = 0;
        for (int i = 1; i <= n; ++i) {
            for (; t < (size_t)blk_end[i - 1]; ++t) {
                for (int h = 0; h < G; ++h) {
                    double w = exp(s[t * G + h] - Mh[h]);
                    Z[h] += w;
                    for (int k = 0; k < m; ++k)
                        Nm[h * m + k] += w * load_elem(J->v, sh->dtype, row_off[t] + J->probe_idx[k]);
                }
            }
            if (L[i - 1] == 0) seen0 = 1;
            const int PH = J->probe_heads;
            double nn = 0.0;
            for (int h = 0; h < PH; ++h)
                for (int k = 0; k < m; ++k) {
                    x[h * m + k] = Nm[h * m + k] / Z[h];
                    nn += x[h * m + k] * x[h * m + k];
                }
            nn = sqrt(nn);
            int stable = 0;
            if (i >= 2) {
                double dot = 0.0;
                for (int k = 0; k < PH * m; ++k) dot += x[k] * xp[k];
                double dmag = fabs(nn - nprev) / nprev;
                double ddir = 1.0 - dot / (nn * nprev);
                if (ddir < 0.0) ddir = 0.0;
                if (tmag && i - 1 < mx) tmag[i - 1] = dmag;
                if (tdir && i - 1 < mx) tdir[i - 1] = ddir;
                int ok = nn > 0.0 && nprev > 0.0 && isfinite(nn) && isfinite(nprev) &&
                         isfinite(dmag) && isfinite(ddir);
                stable = ok && dmag < J->eps_mag && ddir < J->eps_dir;
            }
            counter = stable ? counter + 1 : 0;
            if (counter >= J->patience && (seen0 || !has0)) { bu = i; break; }
            memcpy(xp, x, sizeof(double) * G * m);
            nprev = nn;
        }
        free(Z); free(Nm); free(x); free(xp);
    }
    J->blocks_used[slot] = bu;

    /* Step 9: out_h = O^(bu)_h over the full head dimension. */
    if (bu > 0) {
        size_t tend = (size_t)blk_end[bu - 1];
        for (int h = 0; h < G; ++h) {
            double Zh = 0.0;
            double *oh = out + (size_t)h * d;
            for (size_t t = 0; t < tend; ++t) {
                double w = exp(s[t * G + h] - Mh[h]);
                Zh += w;
                for (int e = 0; e < d; ++e) oh[e] += w * load_elem(J->v, sh->dtype, row_off[t] + e);
            }
            for (int e = 0; e < d; ++e) oh[e] /= Zh;
        }
    }
    free(kv); free(Mh); free(s); free(qd); free(row_off); free(blk_end); free(L);
}

static void *worker(void *arg)
{
    job_t *J = (job_t *)arg;
    for (;;) {
        pthread_mutex_lock(&J->lock);
        int slot = J->next++;
        pthread_mutex_unlock(&J->lock);
        if (slot >= J->num_items) break;
        run_item(J, slot);
    }
    return NULL;
}

/*
 * Runs the oracle over num_items work items (items[k] = b * num_kv_heads + g;
 * items == NULL means every item in order). mode: 0 = dense over the whole
 * list, 1 = ART rule, 2 = forced blocks_used (forced[k] per item).
 * Outputs per item slot k: out[k][G][d], blocks_used[k], item_status[k],
 * and (if non-NULL) trace_mag[k][max_visit], trace_dir[k][max_visit]
 * holding d_mag_i / d_dir_i at index i-1 (NaN where undefined or not reached).
 * num_threads <= 0 uses every online core. probe_heads (1..G, or 0 for all G)
 * selects the query heads whose outputs form the probe. Returns the thread
 * count used, or a negative value on a bad argument.
 */
int oracle_art(const oracle_shape *sh, const void *q, const void *k_cache, const void *v_cache,
               const int32_t *block_table, const int32_t *seq_lens, const int32_t *visit_order,
               double eps_mag, double eps_dir, int32_t patience, const int32_t *probe_idx,
               int32_t mode, const int32_t *items, int32_t num_items, const int32_t *forced,
               double *out, int32_t *blocks_used, int32_t *item_status,
               double *trace_mag, double *trace_dir, int32_t num_threads, int32_t probe_heads)
{
    if (!sh || !q || !k_cache || !v_cache || !block_table || !seq_lens || !out || !blocks_used ||
        !item_status)
        return -1;
    if (sh->num_kv_heads <= 0 || sh->num_q_heads % sh->num_kv_heads != 0) return -2;
    if (sh->block_size <= 0 || sh->page_size <= 0 || sh->head_dim <= 0) return -3;
    if (mode == 1 && (patience < 1 || !probe_idx || sh->num_probe <= 0)) return -4;
    if (mode == 2 && !forced) return -5;
    if (sh->dtype != 0 && sh->dtype != 1) return -6;
    if (probe_heads < 0 || probe_heads > sh->num_q_heads / sh->num_kv_heads) return -7;
    if (!items) num_items = sh->batch * sh->num_kv_heads;

    job_t J;
    memset(&J, 0, sizeof J);
    J.sh = sh; J.q = q; J.k = k_cache; J.v = v_cache;
    J.block_table = block_table; J.seq_lens = seq_lens; J.visit_order = visit_order;
    J.probe_idx = probe_idx; J.eps_mag = eps_mag; J.eps_dir = eps_dir; J.patience = patience;
    J.probe_heads = probe_heads > 0 ? probe_heads : sh->num_q_heads / sh->num_kv_heads;
    J.mode = mode; J.items = items; J.forced = forced; J.num_items = num_items;
    J.out = out; J.blocks_used = blocks_used; J.item_status = item_status;
    J.trace_mag = trace_mag; J.trace_dir = trace_dir;
    pthread_mutex_init(&J.lock, NULL);

    int nt = num_threads > 0 ? num_threads : (int)sysconf(_SC_NPROCESSORS_ONLN);
    if (nt < 1) nt = 1;
    if (nt > num_items) nt = num_items > 0 ? num_items : 1;
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * nt);
    for (int i = 0; i < nt; ++i) pthread_create(&th[i], NULL, worker, &J);
    for (int i = 0; i < nt; ++i) pthread_join(th[i], NULL);
    free(th);
    pthread_mutex_destroy(&J.lock);
    return nt;
}
