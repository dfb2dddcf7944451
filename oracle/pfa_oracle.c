/*
 * pfa_oracle.c -- fp64 CPU oracle for chunked causal GQA prefill attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or
 * calls this file; only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg do.  It shares no code, header or constant with the CUDA
 * path under chunked_causal_gqa_gb300/csrc.
 *
 * What it computes is the plain definition of one layer's prefill attention
 * for a chunk of T query tokens at absolute positions start_pos..start_pos+T-1
 * against a KV cache holding L = start_pos + T positions, as the gnosis
 * "Prefill attention -> GPU: handoff" page defines it (section "GPU design",
 * bullets "GQA", "Layout", "Step 1"-"Step 3"; section "What already shipped"
 * for the per-(token, head) loop over the causal range 0..=pos):
 *
 *   group = H / Hkv,  kv head of query head h = h / group      (integer division)
 *   pos   = start_pos + t
 *   visible keys j:  j <= pos, and, when window > 0, j > pos - window
 *                   (the "causal(+windowed)" per-row [lo, hi] band of the
 *                    TensorSharp2 Gemma-4 prefill design, section 5 Option A)
 *   s_j   = scale * sum_d q[t][h][d] * k[kh][j][d]
 *   w_j   = exp(s_j - max_j s_j)
 *   out[t][h][d] = sum_j w_j * v[kh][j][d] / sum_j w_j
 *
 * Layouts (row-major):
 *   q, out : [T][H][D]          (token-major, as the page's batch_q / batch_xb)
 *   k, v   : [Hkv][L][D]        (one contiguous [L x D] block per kv head)
 *
 * The cache-layout entry point reads the same quantities from the strided
 * buffers the gnosis page describes in section "GPU design", "Layout":
 *   q[t][h][d]   at q[t * qkv_dim + h * D + d]       (batch_q rows of qkv_dim)
 *   out[t][h][d] at out[t * qkv_dim + h * D + d]     (batch_xb rows)
 *   k[kh][j][d]  at k[kh * max_seq_len * D + row(j) * D + d]
 * with row(j) = j for a linear cache and row(j) = j mod max_seq_len for a
 * circular one (the sliding-window layers of the TensorSharp2 Gemma-4 prefill
 * design write position pos at index pos % capacity, section 4, R4).
 *
 * Everything is computed in double.  Each (t, h) row is computed by exactly
 * one thread in a fixed serial order, so the result does not depend on the
 * number of threads (the page's rayon split over the flat T x H work set is
 * likewise bit-identical to its serial loop).
 *
 * A second entry point takes a `plant` code that inserts one deliberate,
 * named mistake.  It exists only so the test suite can show that its pins
 * catch each such mistake; the normal entry points always pass 0.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>

enum {
    PLANT_NONE = 0,
    PLANT_MASK_STRICT = 1,      /* causal test j <  pos instead of j <= pos        */
    PLANT_WINDOW_WIDE = 2,      /* window band one key too wide                    */
    PLANT_KV_HEAD_MODULO = 3,   /* kv head h % Hkv instead of h / (H / Hkv)        */
    PLANT_NO_SCALE = 4,         /* scale not applied                               */
    PLANT_NO_MAX_SHIFT = 5,     /* exp(s_j) without subtracting the row maximum    */
    PLANT_KV_STRIDE = 6,        /* kv head block stride taken as T*D, not L*D      */
    PLANT_WINDOW_NARROW = 7,    /* window band one key too narrow                  */
    PLANT_RING_OFFSET = 8,      /* circular cache row (j + 1) mod capacity         */
    PLANT_QKV_STRIDE = 9        /* q rows taken as H*D apart instead of qkv_dim    */
};

typedef struct {
    const double *q, *k, *v;
    double *out;
    int64_t T, start_pos;
    int H, Hkv, D, window;
    double scale;
    int plant;
    /* layout: element strides of q/out rows and of kv heads, circular cache */
    int64_t qkv_dim, max_seq_len;
    int ring;
    /* rows to compute: either all T*H rows (row_t == NULL) or a list */
    const int64_t *row_t;
    const int32_t *row_h;
    int64_t nrows;
    int nthreads, tid;
    int failed;
} job_t;

/* Cache row that holds key position j. */
static int64_t key_row(const job_t *J, int64_t j)
{
    if (!J->ring) return j;
    if (J->plant == PLANT_RING_OFFSET) return (j + 1) % J->max_seq_len;
    return j % J->max_seq_len;
}

/* One output row: out_row[0..D) = attention of query (t, h). */
static int attend_row(const job_t *J, int64_t t, int h, double *out_row, double *s)
{
    const int64_t L = J->start_pos + J->T;
    const int64_t pos = J->start_pos + t;
    const int group = J->H / J->Hkv;
    int kh = h / group;
    if (J->plant == PLANT_KV_HEAD_MODULO) kh = h % J->Hkv;

    /* visible band [lo, hi] */
    int64_t hi = pos;
    int64_t lo = 0;
    if (J->plant == PLANT_MASK_STRICT) hi = pos - 1;
    if (J->window > 0) {
        int64_t w = J->window;
        if (J->plant == PLANT_WINDOW_WIDE) w += 1;
        if (J->plant == PLANT_WINDOW_NARROW) w -= 1;
        lo = pos - w + 1;
        if (lo < 0) lo = 0;
    }
    if (hi >= L) hi = L - 1;
    if (hi < lo) {               /* cannot happen for window >= 1; planted cases only */
        for (int d = 0; d < J->D; ++d) out_row[d] = NAN;
        return 0;
    }

    const int64_t kv_stride = (J->plant == PLANT_KV_STRIDE) ? J->T * (int64_t)J->D
                                                            : J->max_seq_len * (int64_t)J->D;
    const int64_t q_stride = (J->plant == PLANT_QKV_STRIDE) ? (int64_t)J->H * J->D : J->qkv_dim;
    const double *qr = J->q + t * q_stride + h * (int64_t)J->D;
    const double *kb = J->k + kh * kv_stride;
    const double *vb = J->v + kh * kv_stride;
    const double scale = (J->plant == PLANT_NO_SCALE) ? 1.0 : J->scale;

    /* scores */
    double m = -INFINITY;
    for (int64_t j = lo; j <= hi; ++j) {
        const double *kr = kb + key_row(J, j) * J->D;
        double dot = 0.0;
        for (int d = 0; d < J->D; ++d) dot += qr[d] * kr[d];
        s[j - lo] = scale * dot;
        if (s[j - lo] > m) m = s[j - lo];
    }
    if (J->plant == PLANT_NO_MAX_SHIFT) m = 0.0;

    /* softmax weights and weighted sum of V */
    double Z = 0.0;
    for (int d = 0; d < J->D; ++d) out_row[d] = 0.0;
    for (int64_t j = lo; j <= hi; ++j) {
        const double w = exp(s[j - lo] - m);
        Z += w;
        const double *vr = vb + key_row(J, j) * J->D;
        for (int d = 0; d < J->D; ++d) out_row[d] += w * vr[d];
    }
    for (int d = 0; d < J->D; ++d) out_row[d] /= Z;
    return 0;
}

static void *worker(void *arg)
{
    job_t *J = (job_t *)arg;
    const int64_t L = J->start_pos + J->T;
    double *s = (double *)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1));
    if (!s) { J->failed = 1; return NULL; }
    const int64_t total = J->row_t ? J->nrows : J->T * (int64_t)J->H;
    /* static cyclic split of the flat row set */
    for (int64_t r = J->tid; r < total; r += J->nthreads) {
        int64_t t; int h; double *dst;
        if (J->row_t) {
            t = J->row_t[r]; h = J->row_h[r];
            dst = J->out + r * (int64_t)J->D;
        } else {
            t = r / J->H; h = (int)(r % J->H);
            dst = J->out + t * J->qkv_dim + h * (int64_t)J->D;   /* [T][H][D] when qkv_dim = H*D */
        }
        attend_row(J, t, h, dst, s);
    }
    free(s);
    return NULL;
}

static int run(const job_t *proto)
{
    int n = proto->nthreads < 1 ? 1 : proto->nthreads;
    if (n > 1024) n = 1024;
    job_t *jobs = (job_t *)calloc((size_t)n, sizeof(job_t));
    pthread_t *th = (pthread_t *)calloc((size_t)n, sizeof(pthread_t));
    if (!jobs || !th) { free(jobs); free(th); return -8; }
    int rc = 0, started = 0;
    for (int i = 0; i < n; ++i) {
        jobs[i] = *proto;
        jobs[i].nthreads = n;
        jobs[i].tid = i;
        if (n == 1) { worker(&jobs[0]); started = 0; break; }
        if (pthread_create(&th[i], NULL, worker, &jobs[i]) != 0) { rc = -8; break; }
        ++started;
    }
    for (int i = 0; i < started; ++i) pthread_join(th[i], NULL);
    for (int i = 0; i < n; ++i) if (jobs[i].failed) rc = -8;
    free(jobs); free(th);
    return rc;
}

static int check_args(const double *q, const double *k, const double *v, const double *out,
                      int64_t T, int64_t start_pos, int H, int Hkv, int D)
{
    if (!q || !k || !v || !out) return -1;
    if (T < 0 || start_pos < 0 || H <= 0 || Hkv <= 0 || D <= 0) return -2;
    if (H % Hkv != 0) return -2;
    return 0;
}

int pfa_oracle_prefill_attention_planted(const double *q, const double *k, const double *v,
                                         double *out, int64_t T, int64_t start_pos,
                                         int H, int Hkv, int D, int window, double scale,
                                         int nthreads, int plant)
{
    int rc = check_args(q, k, v, out, T, start_pos, H, Hkv, D);
    if (rc) return rc;
    if (T == 0) return 0;
    job_t J = {0};
    J.q = q; J.k = k; J.v = v; J.out = out;
    J.T = T; J.start_pos = start_pos; J.H = H; J.Hkv = Hkv; J.D = D;
    J.window = window; J.scale = scale; J.plant = plant; J.nthreads = nthreads;
    J.qkv_dim = (int64_t)H * D; J.max_seq_len = start_pos + T; J.ring = 0;
    return run(&J);
}

/* Full output: out[T][H][D]. */
int pfa_oracle_prefill_attention(const double *q, const double *k, const double *v,
                                 double *out, int64_t T, int64_t start_pos,
                                 int H, int Hkv, int D, int window, double scale,
                                 int nthreads)
{
    return pfa_oracle_prefill_attention_planted(q, k, v, out, T, start_pos, H, Hkv, D,
                                                window, scale, nthreads, PLANT_NONE);
}

/* Selected rows only: out_rows[r][D] = attention of query (row_t[r], row_h[r]). */
int pfa_oracle_prefill_attention_rows(const double *q, const double *k, const double *v,
                                      int64_t T, int64_t start_pos, int H, int Hkv, int D,
                                      int window, double scale,
                                      const int64_t *row_t, const int32_t *row_h, int64_t nrows,
                                      double *out_rows, int nthreads)
{
    int rc = check_args(q, k, v, out_rows, T, start_pos, H, Hkv, D);
    if (rc) return rc;
    if (!row_t || !row_h) return -1;
    for (int64_t r = 0; r < nrows; ++r)
        if (row_t[r] < 0 || row_t[r] >= T || row_h[r] < 0 || row_h[r] >= H) return -2;
    if (nrows == 0) return 0;
    job_t J = {0};
    J.q = q; J.k = k; J.v = v; J.out = out_rows;
    J.T = T; J.start_pos = start_pos; J.H = H; J.Hkv = Hkv; J.D = D;
    J.window = window; J.scale = scale; J.plant = PLANT_NONE; J.nthreads = nthreads;
    J.qkv_dim = (int64_t)H * D; J.max_seq_len = start_pos + T; J.ring = 0;
    J.row_t = row_t; J.row_h = row_h; J.nrows = nrows;
    return run(&J);
}

/*
 * Cache layout (see the header comment): q and out rows qkv_dim elements
 * apart, max_seq_len rows per kv head, key j in row j (ring == 0, needs
 * max_seq_len >= L) or in row j mod max_seq_len (ring != 0, needs window > 0
 * and max_seq_len >= min(L, window + T - 1): every key some row of the chunk
 * sees is still in the cache).  Only the H*D head elements of each out row
 * are written.
 */
int pfa_oracle_prefill_attention_cache(const double *q, const double *k, const double *v,
                                       double *out, int64_t T, int64_t start_pos,
                                       int H, int Hkv, int D, int window, double scale,
                                       int64_t qkv_dim, int64_t max_seq_len, int ring,
                                       int nthreads, int plant)
{
    int rc = check_args(q, k, v, out, T, start_pos, H, Hkv, D);
    if (rc) return rc;
    const int64_t L = start_pos + T;
    if (qkv_dim < (int64_t)H * D || max_seq_len <= 0) return -2;
    if (!ring && max_seq_len < L) return -2;
    if (ring) {
        if (window <= 0) return -2;
        const int64_t span = (window + T - 1 < L) ? window + T - 1 : L;
        if (max_seq_len < span) return -2;
    }
    if (T == 0) return 0;
    job_t J = {0};
    J.q = q; J.k = k; J.v = v; J.out = out;
    J.T = T; J.start_pos = start_pos; J.H = H; J.Hkv = Hkv; J.D = D;
    J.window = window; J.scale = scale; J.plant = plant; J.nthreads = nthreads;
    J.qkv_dim = qkv_dim; J.max_seq_len = max_seq_len; J.ring = ring ? 1 : 0;
    return run(&J);
}
