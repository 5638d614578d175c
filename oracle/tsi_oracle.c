/*
 * CPU oracle for the DSA lightning-indexer + top-k + IndexShare sparse attention path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or call this
 * file.  Only the tests, the smoke check and the CPU-baseline leg of the benchmark use
 * it.  It shares no code, header, table or constant with the CUDA library.
 *
 * Everything is computed in double precision, one element at a time, in the order the
 * formulas are written.  Stored inputs (fp32, bf16, FP8 e4m3) are decoded exactly to
 * double from their bit patterns.
 *
 * Sources (page title, section):
 *   - Indexer score I[t,s] = sum_j w[t,j] * ReLU(qI[t,j] . kI[s]) over keys s <= t:
 *     "GLM-5.2 技术报告速览", §IndexShare (the unnumbered score equation and the sentence
 *     before it, which restricts keys to s <= t; one index key per position, shared by
 *     all H_I indexer heads).
 *   - Top-k with k = 2048 << L, attention restricted to the chosen keys: same section.
 *     Ties go to the lower key index (deterministic top-k: "GLM-5: from Vibe Coding to Agentic
 *     Engineering" (Chinese translation), §3.2 "DSA RL 要点", asks for a deterministic operator; the lower-index rule is this
 *     build's fixed reading of it).
 *   - Sparse attention over the selected keys, with each layer using its own Q/K/V and
 *     Shared layers reusing only the Full layer's index set: "GLM-5.2 技术报告速览"
 *     §IndexShare; "GLM 5.2: Built for Long Horizon Tasks" §5.2 and the discussion §3
 *     (sparse attention over indices == dense attention under a top-k mask).
 *
 * Parity status: every function here is pinned by the CPU tests (brute force on tiny
 * inputs, closed forms, library special cases, invariants); see tests/test_oracle_pins.py.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { TSIO_F32 = 0, TSIO_BF16 = 1, TSIO_E4M3 = 2 };

/* ---------------------------------------------------------------- decoding ---- */

/* FP8 e4m3 ("fn" variant): 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits,
 * no infinities, S.1111.111 is NaN.  Exponent field 0 is subnormal: m * 2^-9. */
static double decode_e4m3(uint8_t b) {
    int sign = (b >> 7) & 1;
    int e = (b >> 3) & 0xF;
    int m = b & 0x7;
    double v;
    if (e == 0xF && m == 0x7) return NAN;
    if (e == 0)
        v = ldexp((double)m, -9);
    else
        v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return sign ? -v : v;
}

/* bfloat16: the upper 16 bits of an IEEE binary32. */
static double decode_bf16(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double decode_f32(const void* p) {
    float f;
    memcpy(&f, p, sizeof f);
    return (double)f;
}

double tsio_decode(const void* base, int64_t i, int dtype) {
    switch (dtype) {
        case TSIO_F32: return decode_f32((const char*)base + 4 * i);
        case TSIO_BF16: {
            uint16_t b;
            memcpy(&b, (const char*)base + 2 * i, 2);
            return decode_bf16(b);
        }
        case TSIO_E4M3: return decode_e4m3(((const uint8_t*)base)[i]);
        default: return NAN;
    }
}

/* Every stored element of a buffer of n elements, decoded to double. */
void tsio_decode_n(const void* base, int64_t n, int dtype, double* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = tsio_decode(base, i, dtype);
}

static int dtype_ok(int dt) { return dt == TSIO_F32 || dt == TSIO_BF16 || dt == TSIO_E4M3; }

/* Position of query row t of sequence b: the T query rows are the last T of the
 * kv_len[b] cached positions (prefill T == S gives p_t = t, decode T == 1 gives
 * p = kv_len - 1).  kv_len == NULL means every sequence holds S positions. */
static int64_t query_pos(const int32_t* kv_len, int b, int T, int S, int t) {
    int64_t len = kv_len ? (int64_t)kv_len[b] : (int64_t)S;
    if (len > S) len = S;
    if (len < 0) len = 0;
    return len - (int64_t)T + (int64_t)t;
}

/* --------------------------------------------------------- indexer score ---- */

/* I[s] for s = 0..p of one query row:  I[s] = sum_j w[j] * max(0, sum_d q[j][d]*k[s][d]).
 * qrow: the row's H_I x d_I query block, wrow: its H_I gate weights, kseq: the
 * sequence's S x d_I index keys.  Writes p+1 scores; returns p+1 (0 if p < 0). */
static int64_t row_scores(const void* qrow, const void* wrow, const void* kseq, int qk_dtype,
                          int w_dtype, int H_I, int d_I, int64_t p, double* out, double* qd,
                          double* kd) {
    if (p < 0) return 0;
    for (int j = 0; j < H_I; ++j)
        for (int d = 0; d < d_I; ++d) qd[j * d_I + d] = tsio_decode(qrow, (int64_t)j * d_I + d, qk_dtype);
    for (int64_t s = 0; s <= p; ++s) {
        for (int d = 0; d < d_I; ++d) kd[d] = tsio_decode(kseq, s * d_I + d, qk_dtype);
        double I = 0.0;
        for (int j = 0; j < H_I; ++j) {
            double dot = 0.0;
            for (int d = 0; d < d_I; ++d) dot += qd[j * d_I + d] * kd[d];
            double relu = dot > 0.0 ? dot : 0.0;
            I += tsio_decode(wrow, j, w_dtype) * relu;
        }
        out[s] = I;
    }
    return p + 1;
}

typedef struct {
    double score;
    int32_t s;
} scored_t;

/* Rank order: higher score first; equal scores go to the lower key index. */
static int rank_cmp(const void* a, const void* b) {
    const scored_t* x = (const scored_t*)a;
    const scored_t* y = (const scored_t*)b;
    if (x->score > y->score) return -1;
    if (x->score < y->score) return 1;
    return (x->s > y->s) - (x->s < y->s);
}

/* ---------------------------------------------------------- thread helper ---- */

typedef void (*row_fn)(void* ctx, int64_t r);
typedef struct {
    row_fn fn;
    void* ctx;
    int64_t n_rows;
    int n_threads;
    int id;
} worker_t;

static void* worker_main(void* arg) {
    worker_t* w = (worker_t*)arg;
    for (int64_t r = w->id; r < w->n_rows; r += w->n_threads) w->fn(w->ctx, r);
    return NULL;
}

static void run_rows(row_fn fn, void* ctx, int64_t n_rows, int n_threads) {
    if (n_threads < 1) n_threads = 1;
    if (n_threads > 256) n_threads = 256;
    if (n_threads > n_rows) n_threads = (int)(n_rows > 0 ? n_rows : 1);
    pthread_t th[256];
    worker_t ws[256];
    for (int i = 0; i < n_threads; ++i) {
        ws[i].fn = fn;
        ws[i].ctx = ctx;
        ws[i].n_rows = n_rows;
        ws[i].n_threads = n_threads;
        ws[i].id = i;
    }
    for (int i = 1; i < n_threads; ++i) pthread_create(&th[i], NULL, worker_main, &ws[i]);
    worker_main(&ws[0]);
    for (int i = 1; i < n_threads; ++i) pthread_join(th[i], NULL);
}

static size_t dtype_size(int dt) { return dt == TSIO_F32 ? 4 : dt == TSIO_BF16 ? 2 : 1; }

/* ------------------------------------------------------ indexer + top-k ---- */

typedef struct {
    const void* q_rows;   /* [n_rows, H_I, d_I] */
    const void* kI;       /* [B, S, d_I] */
    const void* w_rows;   /* [n_rows, H_I] */
    int qk_dtype, w_dtype;
    int B, T, S, H_I, d_I, topk;
    const int32_t* kv_len;
    const int32_t* row_b;
    const int32_t* row_t;
    int32_t* idx_out;     /* [n_rows, topk] */
    double* score_out;    /* [n_rows, topk] or NULL */
    int status;
} topk_ctx;

static void topk_row(void* vctx, int64_t r) {
    topk_ctx* c = (topk_ctx*)vctx;
    int b = c->row_b[r], t = c->row_t[r];
    int64_t p = query_pos(c->kv_len, b, c->T, c->S, t);
    int32_t* idx = c->idx_out + r * (int64_t)c->topk;
    double* sc = c->score_out ? c->score_out + r * (int64_t)c->topk : NULL;
    int64_t n = p + 1 > 0 ? p + 1 : 0;
    double* scores = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
    scored_t* order = (scored_t*)malloc(sizeof(scored_t) * (size_t)(n > 0 ? n : 1));
    double* qd = (double*)malloc(sizeof(double) * (size_t)c->H_I * c->d_I);
    double* kd = (double*)malloc(sizeof(double) * (size_t)c->d_I);
    if (!scores || !order || !qd || !kd) {
        c->status = 1;
        free(scores); free(order); free(qd); free(kd);
        return;
    }
    const char* qrow = (const char*)c->q_rows + r * (int64_t)c->H_I * c->d_I * dtype_size(c->qk_dtype);
    const char* wrow = (const char*)c->w_rows + r * (int64_t)c->H_I * dtype_size(c->w_dtype);
    const char* kseq = (const char*)c->kI + (int64_t)b * c->S * c->d_I * dtype_size(c->qk_dtype);
    row_scores(qrow, wrow, kseq, c->qk_dtype, c->w_dtype, c->H_I, c->d_I, p, scores, qd, kd);
    for (int64_t s = 0; s < n; ++s) {
        order[s].score = scores[s];
        order[s].s = (int32_t)s;
    }
    qsort(order, (size_t)n, sizeof(scored_t), rank_cmp);
    int64_t keep = n < c->topk ? n : c->topk;
    for (int64_t i = 0; i < c->topk; ++i) {
        idx[i] = i < keep ? order[i].s : -1;
        if (sc) sc[i] = i < keep ? order[i].score : -INFINITY;
    }
    free(scores); free(order); free(qd); free(kd);
}

/* Top-k indices of the indexer score for n_rows query rows.  Query-side tensors are
 * passed compacted to the requested rows; (row_b[r], row_t[r]) locate row r.
 * Returns 0 on success, nonzero on bad arguments or allocation failure. */
int tsio_indexer_topk(const void* q_rows, const void* kI, const void* w_rows, int qk_dtype,
                      int w_dtype, int B, int T, int S, int H_I, int d_I, int topk,
                      const int32_t* kv_len, int64_t n_rows, const int32_t* row_b,
                      const int32_t* row_t, int32_t* idx_out, double* score_out, int n_threads) {
    if (!dtype_ok(qk_dtype) || !dtype_ok(w_dtype) || B < 0 || T < 0 || S < 0 || H_I < 1 ||
        d_I < 1 || topk < 1 || n_rows < 0)
        return 2;
    for (int64_t r = 0; r < n_rows; ++r)
        if (row_b[r] < 0 || row_b[r] >= B || row_t[r] < 0 || row_t[r] >= T) return 2;
    topk_ctx c = {q_rows, kI, w_rows, qk_dtype, w_dtype, B, T, S, H_I, d_I, topk,
                  kv_len, row_b, row_t, idx_out, score_out, 0};
    run_rows(topk_row, &c, n_rows, n_threads);
    return c.status;
}

/* Every score of one query row (s = 0..p).  Returns p+1, or -1 on bad arguments. */
int64_t tsio_indexer_scores(const void* q_row, const void* kseq, const void* w_row, int qk_dtype,
                            int w_dtype, int H_I, int d_I, int64_t p, double* out) {
    if (!dtype_ok(qk_dtype) || !dtype_ok(w_dtype) || H_I < 1 || d_I < 1) return -1;
    double* qd = (double*)malloc(sizeof(double) * (size_t)H_I * d_I);
    double* kd = (double*)malloc(sizeof(double) * (size_t)d_I);
    if (!qd || !kd) {
        free(qd); free(kd);
        return -1;
    }
    int64_t n = row_scores(q_row, w_row, kseq, qk_dtype, w_dtype, H_I, d_I, p, out, qd, kd);
    free(qd); free(kd);
    return n;
}

/* ------------------------------------------------------- sparse attention ---- */

typedef struct {
    const void* q_rows;  /* [n_rows, H, Dqk] */
    const void* k;       /* [B, S, Hkv, Dqk] */
    const void* v;       /* [B, S, Hkv, Dv] or NULL: value = k[..., :Dv] */
    int dtype;
    int B, T, S, H, Hkv, Dqk, Dv;
    double scale;
    const int32_t* idx_rows; /* [n_rows, topk] */
    int topk;
    const int32_t* kv_len;
    const int32_t* row_b;
    const int32_t* row_t;
    double* out;         /* [n_rows, H, Dv] */
    int status;
} attn_ctx;

/* O[h] = sum_{s in S_t} softmax_s(scale * Q[h] . K[s]) V[s], where S_t holds the row's
 * index entries that name a cached position (0 <= s < kv_len[b]); the -1 padding
 * of short rows is not a key.  A row with no key gets O = 0. */
static void attn_row(void* vctx, int64_t r) {
    attn_ctx* c = (attn_ctx*)vctx;
    int b = c->row_b[r];
    int64_t len = c->kv_len ? (int64_t)c->kv_len[b] : (int64_t)c->S;
    if (len > c->S) len = c->S;
    const int32_t* sel = c->idx_rows + r * (int64_t)c->topk;
    size_t es = dtype_size(c->dtype);
    double* z = (double*)malloc(sizeof(double) * (size_t)c->topk);
    int32_t* keys = (int32_t*)malloc(sizeof(int32_t) * (size_t)c->topk);
    double* qd = (double*)malloc(sizeof(double) * (size_t)c->Dqk);
    double* acc = (double*)malloc(sizeof(double) * (size_t)c->Dv);
    if (!z || !keys || !qd || !acc) {
        c->status = 1;
        free(z); free(keys); free(qd); free(acc);
        return;
    }
    int nk = 0;
    for (int i = 0; i < c->topk; ++i)
        if (sel[i] >= 0 && sel[i] < len) keys[nk++] = sel[i];
    int group = c->H / c->Hkv;
    for (int h = 0; h < c->H; ++h) {
        int kvh = h / group;
        const char* qh = (const char*)c->q_rows + ((r * (int64_t)c->H + h) * c->Dqk) * es;
        for (int d = 0; d < c->Dqk; ++d) qd[d] = tsio_decode(qh, d, c->dtype);
        double zmax = -INFINITY;
        for (int i = 0; i < nk; ++i) {
            int64_t krow = (((int64_t)b * c->S + keys[i]) * c->Hkv + kvh) * c->Dqk;
            double dot = 0.0;
            for (int d = 0; d < c->Dqk; ++d) dot += qd[d] * tsio_decode(c->k, krow + d, c->dtype);
            z[i] = c->scale * dot;
            if (z[i] > zmax) zmax = z[i];
        }
        double den = 0.0;
        for (int e = 0; e < c->Dv; ++e) acc[e] = 0.0;
        for (int i = 0; i < nk; ++i) {
            double pexp = exp(z[i] - zmax);
            den += pexp;
            for (int e = 0; e < c->Dv; ++e) {
                double ve;
                if (c->v) {
                    int64_t vrow = (((int64_t)b * c->S + keys[i]) * c->Hkv + kvh) * c->Dv;
                    ve = tsio_decode(c->v, vrow + e, c->dtype);
                } else {
                    int64_t krow = (((int64_t)b * c->S + keys[i]) * c->Hkv + kvh) * c->Dqk;
                    ve = tsio_decode(c->k, krow + e, c->dtype);
                }
                acc[e] += pexp * ve;
            }
        }
        double* o = c->out + (r * (int64_t)c->H + h) * c->Dv;
        for (int e = 0; e < c->Dv; ++e) o[e] = nk > 0 ? acc[e] / den : 0.0;
    }
    free(z); free(keys); free(qd); free(acc);
}

/* Sparse attention of n_rows query rows of one layer over the index sets idx_rows
 * (the Full layer's rows; Shared layers pass the same buffer).  Query rows are passed
 * compacted; keys/values are the full per-sequence caches.  Returns 0 on success. */
int tsio_sparse_attn(const void* q_rows, const void* k, const void* v, int dtype, int B, int T,
                     int S, int H, int Hkv, int Dqk, int Dv, double scale, const int32_t* idx_rows,
                     int topk, const int32_t* kv_len, int64_t n_rows, const int32_t* row_b,
                     const int32_t* row_t, double* out, int n_threads) {
    if (!dtype_ok(dtype) || B < 0 || T < 0 || S < 0 || H < 1 || Hkv < 1 || H % Hkv || Dqk < 1 ||
        Dv < 1 || topk < 1 || n_rows < 0 || (!v && Dv > Dqk))
        return 2;
    for (int64_t r = 0; r < n_rows; ++r)
        if (row_b[r] < 0 || row_b[r] >= B || row_t[r] < 0 || row_t[r] >= T) return 2;
    attn_ctx c = {q_rows, k, v, dtype, B, T, S, H, Hkv, Dqk, Dv, scale, idx_rows, topk,
                  kv_len, row_b, row_t, out, 0};
    run_rows(attn_row, &c, n_rows, n_threads);
    return c.status;
}
