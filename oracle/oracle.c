/*
 * CPU oracle for the selection step of one speculative-decoding round.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, obviously correct
 * statement of what the GPU path computes.  Only the test suite, the smoke
 * check and the benchmark's CPU-baseline / reference arm load it; the
 * library itself never links, calls or falls back to it.  It shares no code,
 * header, table or helper with the CUDA path.
 *
 * What it computes, and where the rule comes from:
 *
 *   top-k      For each column of V bf16 logits, the k largest values,
 *              largest first, ties going to the smaller row (token) id.
 *              ["A drafter inside the artifact" (Ignis DFlash2 page),
 *              section "How it works", third paragraph: the page's faster
 *              top-k gives the same selection, order and tie-breaking by
 *              row id as the kernel it replaced.]
 *              Written out as the definition: sort all V (value, id) pairs
 *              by value descending, then id ascending, and keep the first k.
 *              Values compare as numbers (bf16 widened exactly to double), so
 *              -0 and +0 are a tie; each output carries its own element's
 *              bit pattern.  NaN is outside the contract and is rejected.
 *
 *   top-k, shortlist   The same over a shortlist column whose local ids map
 *              to vocabulary ids through id_map; ties go to the smaller
 *              vocabulary id, and the output ids are vocabulary ids.
 *              [same page, "How it works", second paragraph: an optional
 *              quantised drafter head restricted to 131,072 token ids.]
 *
 *   verify     Per lane: t[j] = argmax of target column j (j = 0..gamma),
 *              ties to the smaller id; accept the longest prefix of drafts
 *              with drafts[i] == t[i]; commit that prefix plus the target's
 *              own next token t[a]; pad with -1.
 *              [same page, "How it works", first paragraph: a lane keeps
 *              its drafts up to the first the target disagrees with, then
 *              one token chosen by the target.  "Speculative decoding,
 *              measured on my M4 Max", section 1: with greedy decoding the
 *              result is the same text the target would produce alone.]
 *
 * Parity pins (tests/test_oracle_pins.py): brute force against an
 * independent repeated-maximum selector on tiny columns and exhaustively on
 * V <= 6; closed forms (planted peaks, all-ties, 64-level ties by a level
 * scan); k = V against a library lexsort; k = 1 against a library argmax;
 * invariants; planted acceptance lengths; hand-worked examples under
 * tests/golden/.  Every function here is pinned.
 *
 * Build: gcc -O2 -shared -fPIC -pthread oracle.c -o liboracle.so
 */
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_ERR_ARG (-1)
#define ORACLE_ERR_NAN (-2)
#define ORACLE_ERR_NOMEM (-3)

/* bf16 is the upper half of an IEEE binary32: widening is exact. */
static double bf16_value(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static int bf16_is_nan(uint16_t bits)
{
    return (bits & 0x7F80u) == 0x7F80u && (bits & 0x007Fu) != 0;
}

typedef struct {
    double value;   /* the logit as a number */
    int64_t tie;    /* tie-break id: row id, or vocabulary id for a shortlist */
    int64_t row;    /* position in the column */
} entry;

/* Order of the selection: value descending, then tie id ascending. */
static int by_value_desc_then_id(const void *pa, const void *pb)
{
    const entry *a = (const entry *)pa;
    const entry *b = (const entry *)pb;
    if (a->value > b->value) return -1;
    if (a->value < b->value) return 1;
    if (a->tie < b->tie) return -1;
    if (a->tie > b->tie) return 1;
    return 0;
}

/* One column: full sort, keep the first k. */
static int topk_column(const uint16_t *col, int64_t V, int32_t k, const int32_t *id_map,
                       uint16_t *out_vals, int32_t *out_ids)
{
    entry *e = (entry *)malloc((size_t)V * sizeof(entry));
    if (!e) return ORACLE_ERR_NOMEM;
    for (int64_t i = 0; i < V; ++i) {
        if (bf16_is_nan(col[i])) { free(e); return ORACLE_ERR_NAN; }
        e[i].value = bf16_value(col[i]);
        e[i].tie = id_map ? (int64_t)id_map[i] : i;
        e[i].row = i;
    }
    qsort(e, (size_t)V, sizeof(entry), by_value_desc_then_id);
    for (int32_t r = 0; r < k; ++r) {
        out_vals[r] = col[e[r].row];
        out_ids[r] = (int32_t)e[r].tie;
    }
    free(e);
    return ORACLE_OK;
}

/* Greedy argmax: first index attaining the maximum (ties to the smaller id). */
static int argmax_column(const uint16_t *col, int64_t V, int32_t *out)
{
    int64_t best = 0;
    for (int64_t i = 0; i < V; ++i) {
        if (bf16_is_nan(col[i])) return ORACLE_ERR_NAN;
        if (bf16_value(col[i]) > bf16_value(col[best])) best = i;
    }
    *out = (int32_t)best;
    return ORACLE_OK;
}

/* One lane of the greedy verify. */
static void verify_lane(const int32_t *t, const int32_t *drafts, int32_t gamma,
                        int32_t *accept_len, int32_t *commit)
{
    int32_t a = 0;
    while (a < gamma && drafts[a] == t[a]) ++a;
    *accept_len = a;
    for (int32_t j = 0; j <= gamma; ++j) commit[j] = (j <= a) ? t[j] : -1;
}

/* ---- a plain pthread fan-out over independent columns ---------------- */

typedef struct {
    int kind;               /* 0 = top-k, 1 = argmax */
    const uint16_t *data;
    int64_t V;
    int32_t k;
    const int32_t *id_map;
    uint16_t *out_vals;
    int32_t *out_ids;
    int64_t begin, end;     /* column range */
    int status;
} job;

static void *run_job(void *p)
{
    job *j = (job *)p;
    j->status = ORACLE_OK;
    for (int64_t c = j->begin; c < j->end && j->status == ORACLE_OK; ++c) {
        const uint16_t *col = j->data + c * j->V;
        if (j->kind == 0)
            j->status = topk_column(col, j->V, j->k, j->id_map, j->out_vals + c * j->k,
                                    j->out_ids + c * j->k);
        else
            j->status = argmax_column(col, j->V, j->out_ids + c);
    }
    return NULL;
}

static int fan_out(int kind, const uint16_t *data, int64_t cols, int64_t V, int32_t k,
                   const int32_t *id_map, uint16_t *out_vals, int32_t *out_ids, int threads)
{
    if (threads < 1) threads = 1;
    if (threads > 256) threads = 256;
    if ((int64_t)threads > cols) threads = (int)(cols > 0 ? cols : 1);
    job jobs[256];
    pthread_t tid[256];
    for (int t = 0; t < threads; ++t) {
        jobs[t] = (job){kind, data, V, k, id_map, out_vals, out_ids,
                        cols * t / threads, cols * (t + 1) / threads, ORACLE_OK};
    }
    int started = 0;
    for (int t = 1; t < threads; ++t) {
        if (pthread_create(&tid[t], NULL, run_job, &jobs[t]) != 0) break;
        started = t;
    }
    run_job(&jobs[0]);
    for (int t = started + 1; t < threads; ++t) run_job(&jobs[t]);  /* threads that failed to start */
    for (int t = 1; t <= started; ++t) pthread_join(tid[t], NULL);
    for (int t = 0; t < threads; ++t)
        if (jobs[t].status != ORACLE_OK) return jobs[t].status;
    return ORACLE_OK;
}

/* ---- exported entry points ------------------------------------------- */

int oracle_topk(const uint16_t *logits, int64_t cols, int64_t V, int32_t k,
                uint16_t *out_vals, int32_t *out_ids, int threads)
{
    if (cols < 0 || V < 1 || k < 1 || k > V) return ORACLE_ERR_ARG;
    if (cols == 0) return ORACLE_OK;
    if (!logits || !out_vals || !out_ids) return ORACLE_ERR_ARG;
    return fan_out(0, logits, cols, V, k, NULL, out_vals, out_ids, threads);
}

int oracle_topk_mapped(const uint16_t *logits, int64_t cols, int64_t V, int32_t k,
                       const int32_t *id_map, uint16_t *out_vals, int32_t *out_ids, int threads)
{
    if (cols < 0 || V < 1 || k < 1 || k > V || !id_map) return ORACLE_ERR_ARG;
    if (cols == 0) return ORACLE_OK;
    if (!logits || !out_vals || !out_ids) return ORACLE_ERR_ARG;
    return fan_out(0, logits, cols, V, k, id_map, out_vals, out_ids, threads);
}

int oracle_argmax(const uint16_t *logits, int64_t cols, int64_t V, int32_t *out_ids, int threads)
{
    if (cols < 0 || V < 1) return ORACLE_ERR_ARG;
    if (cols == 0) return ORACLE_OK;
    if (!logits || !out_ids) return ORACLE_ERR_ARG;
    return fan_out(1, logits, cols, V, 1, NULL, NULL, out_ids, threads);
}

int oracle_verify(const uint16_t *target_logits, const int32_t *drafts, int64_t lanes,
                  int32_t gamma, int64_t V, int32_t *out_accept_len, int32_t *out_commit_ids,
                  int threads)
{
    if (lanes < 0 || gamma < 1 || V < 1) return ORACLE_ERR_ARG;
    if (lanes == 0) return ORACLE_OK;
    if (!target_logits || !drafts || !out_accept_len || !out_commit_ids) return ORACLE_ERR_ARG;
    int64_t n = lanes * (int64_t)(gamma + 1);
    int32_t *t = (int32_t *)malloc((size_t)n * sizeof(int32_t));
    if (!t) return ORACLE_ERR_NOMEM;
    int st = oracle_argmax(target_logits, n, V, t, threads);
    if (st == ORACLE_OK)
        for (int64_t l = 0; l < lanes; ++l)
            verify_lane(t + l * (gamma + 1), drafts + l * gamma, gamma, out_accept_len + l,
                        out_commit_ids + l * (gamma + 1));
    free(t);
    return st;
}
