/*
 * pkv_oracle.c -- float64 CPU oracle for paged-KV grouped-query decode attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test-suite, the package smoke check and
 * the benchmark's CPU-baseline leg may load this library.  It shares no code,
 * header, table or constant with the CUDA library; the two meet only through
 * the seeded inputs that the trace generator draws.
 *
 * What it follows -- "PersistentKV: Page-Aware Decode Scheduling for
 * Long-Context LLM Serving on Commodity GPUs", technical summary:
 *   - Methodology 1, GQA: G = Hq/Hkv query heads share one KV head.
 *   - Methodology 1, "Layout": attention runs directly on the paged KV cache
 *     through the block table, with no repacking into contiguous tensors.
 *   - Methodology 1, "Sequence splitting": the sequence is cut into S disjoint
 *     ranges, each computing a partial online-softmax state; a separate merge
 *     combines the states exactly.
 *   - Methodology 1, "Row-local bounds": tile counts and split ranges come from
 *     each row's real length N*_i; empty splits write neutral states.
 *   - Methodology 1, "Compact workqueue": a 1D list of only the non-empty
 *     (row, kv-head, split) intervals.
 *   - Results, "Scheduling overhead": launches per step, exact-length buckets
 *     versus the compact workqueue.
 *
 * Readings taken where the pages are silent (each one is listed in the
 * design notes of this repository):
 *   - KV layout: k_cache, v_cache are [num_pages][P][Hkv][d] ("NHD"), fp16.
 *   - Query head h reads KV head floor(h / G).
 *   - Splits are fixed chunks of C tokens from position 0: split j covers
 *     tokens [j*C, min((j+1)*C, N)).  n_i = ceil(N_i / C).
 *   - Partial state of a split: m = max_t s_t, l = sum_t exp(s_t - m),
 *     acc = sum_t exp(s_t - m) V_t.  Neutral state: (-inf, 0, 0).
 *   - A row with N = 0 has o = 0 and lse = -inf.
 *   - Natural exponent; s_t = scale * (q . K_t) with the scale passed in.
 *
 * Everything is computed in double from the exact fp16 input values.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define PKVO_OK 0
#define PKVO_EBADARG (-1)
#define PKVO_EBADPAGE (-2)
#define PKVO_ETOOLONG (-3)
#define PKVO_ENOMEM (-4)

/* ------------------------------------------------------------------ fp16 */

/* IEEE 754-2008 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction
 * bits.  Exponent 0 is zero/subnormal (f * 2^-24), exponent 31 is inf/NaN. */
double pkvo_half_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + f), e - 25);
    return sign ? -v : v;
}

static double g_half[65536];

__attribute__((constructor)) static void pkvo_build_table(void)
{
    for (int i = 0; i < 65536; ++i)
        g_half[i] = pkvo_half_to_double((uint16_t)i);
}

void pkvo_half_array_to_double(const uint16_t *src, double *dst, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        dst[i] = g_half[src[i]];
}

int pkvo_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ------------------------------------------------------------ validation */

static int check_shape(int32_t B, int32_t Hq, int32_t Hkv, int32_t d, int32_t P)
{
    if (B < 0 || Hq <= 0 || Hkv <= 0 || d <= 0 || P <= 0)
        return PKVO_EBADARG;
    if (Hq % Hkv != 0)
        return PKVO_EBADARG;
    return PKVO_OK;
}

/* Every block-table entry that a valid token reaches must name a pool page. */
static int check_table(int32_t B, int32_t P, int32_t num_pages, int32_t bt_stride,
                       const int32_t *bt, const int32_t *seq_lens)
{
    for (int32_t i = 0; i < B; ++i) {
        int64_t N = seq_lens[i];
        if (N < 0)
            return PKVO_EBADARG;
        int64_t npages = (N + P - 1) / P;
        if (npages > bt_stride)
            return PKVO_ETOOLONG;
        for (int64_t p = 0; p < npages; ++p) {
            int32_t page = bt[(int64_t)i * bt_stride + p];
            if (page < 0 || page >= num_pages)
                return PKVO_EBADPAGE;
        }
    }
    return PKVO_OK;
}

/* Element offset of K_t / V_t for row i, kv head g, token t (gather through
 * the block table; logical page t / P, slot t mod P). */
static int64_t kv_offset(const int32_t *bt, int32_t bt_stride, int32_t i, int64_t t,
                         int32_t P, int32_t Hkv, int32_t g, int32_t d)
{
    int64_t page = bt[(int64_t)i * bt_stride + t / P];
    int64_t slot = t % P;
    return ((page * P + slot) * Hkv + g) * (int64_t)d;
}

/* s_t = scale * sum_c q[c] K_t[c] for t in [t0, t1) of row i, query head h. */
static void scores(const uint16_t *q, const uint16_t *k, const int32_t *bt,
                   int32_t i, int32_t h, int32_t Hq, int32_t Hkv, int32_t d, int32_t P,
                   int32_t bt_stride, double scale, int64_t t0, int64_t t1, double *s)
{
    int32_t G = Hq / Hkv;
    int32_t g = h / G;
    const uint16_t *qh = q + ((int64_t)i * Hq + h) * d;
    for (int64_t t = t0; t < t1; ++t) {
        const uint16_t *kt = k + kv_offset(bt, bt_stride, i, t, P, Hkv, g, d);
        double dot = 0.0;
        for (int32_t c = 0; c < d; ++c)
            dot += g_half[qh[c]] * g_half[kt[c]];
        s[t - t0] = scale * dot;
    }
}

/* ----------------------------------------------------- plain attention */

/* o[i,h,:] = softmax_t(s_t) . V_t over t < N_i, lse[i,h] = log sum_t exp(s_t).
 * This is the plain definition; the split/merge method must reach it exactly
 * up to rounding.  nthreads <= 0 uses every OpenMP thread. */
int pkvo_attention(int32_t B, int32_t Hq, int32_t Hkv, int32_t d, int32_t P,
                   int32_t num_pages, int32_t bt_stride, double scale,
                   const uint16_t *q, const uint16_t *k, const uint16_t *v,
                   const int32_t *bt, const int32_t *seq_lens,
                   double *o, double *lse, int32_t nthreads)
{
    int rc = check_shape(B, Hq, Hkv, d, P);
    if (rc)
        return rc;
    rc = check_table(B, P, num_pages, bt_stride, bt, seq_lens);
    if (rc)
        return rc;
    int32_t G = Hq / Hkv;
    int64_t rows = (int64_t)B * Hq;
    int failed = 0;
#ifdef _OPENMP
    int nt = nthreads > 0 ? nthreads : omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(nt)
#endif
    for (int64_t r = 0; r < rows; ++r) {
        int32_t i = (int32_t)(r / Hq), h = (int32_t)(r % Hq), g = h / G;
        int64_t N = seq_lens[i];
        double *out = o + r * d;
        for (int32_t c = 0; c < d; ++c)
            out[c] = 0.0;
        if (N == 0) {
            lse[r] = -INFINITY;
            continue;
        }
        double *s = (double *)malloc(sizeof(double) * (size_t)N);
        if (!s) {
            failed = 1;
            continue;
        }
        scores(q, k, bt, i, h, Hq, Hkv, d, P, bt_stride, scale, 0, N, s);
        double M = -INFINITY;
        for (int64_t t = 0; t < N; ++t)
            if (s[t] > M)
                M = s[t];
        double L = 0.0;
        for (int64_t t = 0; t < N; ++t) {
            double w = exp(s[t] - M);
            L += w;
            const uint16_t *vt = v + kv_offset(bt, bt_stride, i, t, P, Hkv, g, d);
            for (int32_t c = 0; c < d; ++c)
                out[c] += w * g_half[vt[c]];
        }
        for (int32_t c = 0; c < d; ++c)
            out[c] /= L;
        lse[r] = M + log(L);
        free(s);
    }
    return failed ? PKVO_ENOMEM : PKVO_OK;
}

/* ------------------------------------------------------------- the plan */

/* Compact workqueue, enumerated by loops in canonical (row, kv-head, split)
 * order.  n_i = ceil(N_i / C); offsets[i] = n_0 + ... + n_{i-1} (B+1 entries);
 * task = {i, g, j, state_base = (offsets[i] + j) * Hq + g * G}.  Writes at most
 * cap tasks (tasks may be NULL) and returns the task count T. */
int64_t pkvo_plan_compact(int32_t B, int32_t Hq, int32_t Hkv, int32_t C,
                          const int32_t *seq_lens, int32_t *tasks, int64_t cap,
                          int32_t *offsets)
{
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || C <= 0)
        return PKVO_EBADARG;
    int32_t G = Hq / Hkv;
    int64_t T = 0, o = 0;
    for (int32_t i = 0; i < B; ++i) {
        int64_t N = seq_lens[i];
        int64_t n = (N + C - 1) / C;
        if (offsets)
            offsets[i] = (int32_t)o;
        for (int32_t g = 0; g < Hkv; ++g)
            for (int64_t j = 0; j < n; ++j) {
                if (tasks && T < cap) {
                    int32_t *rec = tasks + 4 * T;
                    rec[0] = i;
                    rec[1] = g;
                    rec[2] = (int32_t)j;
                    rec[3] = (int32_t)((o + j) * Hq + (int64_t)g * G);
                }
                ++T;
            }
        o += n;
    }
    if (offsets)
        offsets[B] = (int32_t)o;
    return T;
}

/* Rectangular (length-bucketed) grid: every (i, g, j) with j < S_b, where the
 * bucket S_b * C covers N_max.  state_base = (i * S_b + j) * Hq + g * G.
 * empty[k] = 1 when split j starts at or past N_i (a neutral-state cell). */
int64_t pkvo_plan_rect(int32_t B, int32_t Hq, int32_t Hkv, int32_t C, int32_t S_b,
                       const int32_t *seq_lens, int32_t *tasks, int64_t cap,
                       int32_t *empty)
{
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || C <= 0 || S_b < 0)
        return PKVO_EBADARG;
    int32_t G = Hq / Hkv;
    int64_t T = 0;
    for (int32_t i = 0; i < B; ++i)
        for (int32_t g = 0; g < Hkv; ++g)
            for (int32_t j = 0; j < S_b; ++j) {
                if (T < cap) {
                    if (tasks) {
                        int32_t *rec = tasks + 4 * T;
                        rec[0] = i;
                        rec[1] = g;
                        rec[2] = j;
                        rec[3] = (int32_t)(((int64_t)i * S_b + j) * Hq + (int64_t)g * G);
                    }
                    if (empty)
                        empty[T] = ((int64_t)j * C >= seq_lens[i]) ? 1 : 0;
                }
                ++T;
            }
    return T;
}

/* ------------------------------------------------------ partial states */

/* Per-split partial states in double.  State slot of (row i, split j, head h):
 * compact (rect == 0): (offsets_i + j) * Hq + h for j < n_i;
 * rectangular (rect != 0): (i * S_b + j) * Hq + h for j < S_b, where a split
 * past the row end holds the neutral state (-inf, 0, 0).
 * m, l: [n_slots]; acc: [n_slots * d]. */
int pkvo_partials(int32_t B, int32_t Hq, int32_t Hkv, int32_t d, int32_t P,
                  int32_t num_pages, int32_t bt_stride, double scale,
                  const uint16_t *q, const uint16_t *k, const uint16_t *v,
                  const int32_t *bt, const int32_t *seq_lens, int32_t C,
                  int32_t rect, int32_t S_b, double *m, double *l, double *acc,
                  int64_t n_slots, int32_t nthreads)
{
    int rc = check_shape(B, Hq, Hkv, d, P);
    if (rc)
        return rc;
    if (C <= 0)
        return PKVO_EBADARG;
    rc = check_table(B, P, num_pages, bt_stride, bt, seq_lens);
    if (rc)
        return rc;
    int32_t G = Hq / Hkv;
    int64_t *base = (int64_t *)malloc(sizeof(int64_t) * (size_t)(B + 1));
    if (!base)
        return PKVO_ENOMEM;
    int64_t o = 0;
    for (int32_t i = 0; i < B; ++i) {
        int64_t n = ((int64_t)seq_lens[i] + C - 1) / C;
        if (rect && n > S_b) {
            free(base);
            return PKVO_ETOOLONG;
        }
        base[i] = rect ? (int64_t)i * S_b : o;
        o += n;
    }
    int64_t need = rect ? (int64_t)B * S_b * Hq : o * Hq;
    if (need > n_slots) {
        free(base);
        return PKVO_EBADARG;
    }
    int64_t rows = (int64_t)B * Hq;
    int failed = 0;
#ifdef _OPENMP
    int nt = nthreads > 0 ? nthreads : omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(nt)
#endif
    for (int64_t r = 0; r < rows; ++r) {
        int32_t i = (int32_t)(r / Hq), h = (int32_t)(r % Hq), g = h / G;
        int64_t N = seq_lens[i];
        int64_t nsplit = rect ? S_b : (N + C - 1) / C;
        double *s = (double *)malloc(sizeof(double) * (size_t)C);
        if (!s) {
            failed = 1;
            continue;
        }
        for (int64_t j = 0; j < nsplit; ++j) {
            int64_t slot = (base[i] + j) * Hq + h;
            double *a = acc + slot * d;
            for (int32_t c = 0; c < d; ++c)
                a[c] = 0.0;
            int64_t t0 = j * C, t1 = (j + 1) * C < N ? (j + 1) * C : N;
            if (t0 >= t1) {
                m[slot] = -INFINITY;
                l[slot] = 0.0;
                continue;
            }
            scores(q, k, bt, i, h, Hq, Hkv, d, P, bt_stride, scale, t0, t1, s);
            double mj = -INFINITY;
            for (int64_t t = 0; t < t1 - t0; ++t)
                if (s[t] > mj)
                    mj = s[t];
            double lj = 0.0;
            for (int64_t t = t0; t < t1; ++t) {
                double w = exp(s[t - t0] - mj);
                lj += w;
                const uint16_t *vt = v + kv_offset(bt, bt_stride, i, t, P, Hkv, g, d);
                for (int32_t c = 0; c < d; ++c)
                    a[c] += w * g_half[vt[c]];
            }
            m[slot] = mj;
            l[slot] = lj;
        }
        free(s);
    }
    free(base);
    return failed ? PKVO_ENOMEM : PKVO_OK;
}

/* --------------------------------------------------------------- merge */

/* Exact log-sum-exp merge of the partial states of each (row, head):
 * M = max_j m_j, L = sum_j l_j exp(m_j - M), o = sum_j acc_j exp(m_j - M) / L,
 * lse = M + log L.  States with l = 0 (neutral) are skipped; a row with no
 * non-neutral state gets o = 0, lse = -inf.  Slot indexing as in
 * pkvo_partials. */
int pkvo_merge(int32_t B, int32_t Hq, int32_t d, int32_t C, int32_t rect, int32_t S_b,
               const int32_t *seq_lens, const double *m, const double *l,
               const double *acc, double *o, double *lse)
{
    if (B < 0 || Hq <= 0 || d <= 0 || C <= 0)
        return PKVO_EBADARG;
    int64_t run = 0;
    for (int32_t i = 0; i < B; ++i) {
        int64_t n = ((int64_t)seq_lens[i] + C - 1) / C;
        int64_t base = rect ? (int64_t)i * S_b : run;
        int64_t nvisit = rect ? S_b : n;
        for (int32_t h = 0; h < Hq; ++h) {
            double *out = o + ((int64_t)i * Hq + h) * d;
            double M = -INFINITY;
            for (int64_t j = 0; j < nvisit; ++j) {
                int64_t slot = (base + j) * Hq + h;
                if (l[slot] > 0.0 && m[slot] > M)
                    M = m[slot];
            }
            for (int32_t c = 0; c < d; ++c)
                out[c] = 0.0;
            if (M == -INFINITY) {
                lse[(int64_t)i * Hq + h] = -INFINITY;
                continue;
            }
            double L = 0.0;
            for (int64_t j = 0; j < nvisit; ++j) {
                int64_t slot = (base + j) * Hq + h;
                if (!(l[slot] > 0.0))
                    continue;
                double w = exp(m[slot] - M);
                L += l[slot] * w;
                for (int32_t c = 0; c < d; ++c)
                    out[c] += acc[slot * d + c] * w;
            }
            for (int32_t c = 0; c < d; ++c)
                out[c] /= L;
            lse[(int64_t)i * Hq + h] = M + log(L);
        }
        run += n;
    }
    return PKVO_OK;
}

/* ------------------------------------------------------------ counters */

/* Scheduler-derived counters of one decode step (technical summary,
 * "Results": launches per step and merge-state traffic).
 * path: 0 length-bucketed split (one bucket covering N_max: rectangular grid
 *         B x Hkv x S_b, split + merge launches),
 *       1 compact workqueue (split + merge launches; the plan launch is
 *         counted apart),
 *       2 single pass (one launch, no partial states),
 *       3 exact-length buckets (one split + one merge launch per distinct
 *         non-zero length).
 * Merge-state traffic counts fp32 state bytes, (d + 2) * 4 per state: every
 * state the split kernel writes plus every state the merge reads.  The
 * rectangular grid writes a neutral state for each empty cell; the merge
 * reads only the row-local n_i states of each row. */
typedef struct {
    int64_t attn_launches;
    int64_t plan_launches;
    int64_t tasks;
    int64_t grid_tasks;
    int64_t states_written;
    int64_t states_read;
    int64_t merge_state_bytes;
    int64_t kv_bytes;
} pkvo_counters_t;

int pkvo_counters(int32_t path, int32_t B, int32_t Hq, int32_t Hkv, int32_t d, int32_t C,
                  int32_t S_b, const int32_t *seq_lens, pkvo_counters_t *out)
{
    if (!out || B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || d <= 0 || C <= 0)
        return PKVO_EBADARG;
    memset(out, 0, sizeof(*out));
    int64_t sum_n = 0, sum_tok = 0;
    for (int32_t i = 0; i < B; ++i) {
        sum_n += ((int64_t)seq_lens[i] + C - 1) / C;
        sum_tok += seq_lens[i];
    }
    int64_t state_bytes = (int64_t)(d + 2) * 4;
    out->kv_bytes = sum_tok * Hkv * d * 2 * 2;
    switch (path) {
    case 0:
        out->attn_launches = 2;
        out->tasks = sum_n * Hkv;
        out->grid_tasks = (int64_t)B * Hkv * S_b;
        out->states_written = (int64_t)B * S_b * Hq;
        out->states_read = sum_n * Hq;
        break;
    case 1:
        out->attn_launches = 2;
        out->plan_launches = 1;
        out->tasks = out->grid_tasks = sum_n * Hkv;
        out->states_written = out->states_read = sum_n * Hq;
        break;
    case 2:
        out->attn_launches = 1;
        out->tasks = out->grid_tasks = (int64_t)B * Hkv;
        break;
    case 3: {
        int64_t distinct = 0;
        for (int32_t i = 0; i < B; ++i) {
            if (seq_lens[i] == 0)
                continue;
            int seen = 0;
            for (int32_t k = 0; k < i; ++k)
                if (seq_lens[k] == seq_lens[i])
                    seen = 1;
            distinct += !seen;
        }
        out->attn_launches = 2 * distinct;
        out->tasks = out->grid_tasks = sum_n * Hkv;
        out->states_written = out->states_read = sum_n * Hq;
        break;
    }
    default:
        return PKVO_EBADARG;
    }
    out->merge_state_bytes = (out->states_written + out->states_read) * state_bytes;
    return PKVO_OK;
}
