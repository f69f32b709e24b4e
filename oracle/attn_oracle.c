/*
 * ORACLE -- TEST INFRASTRUCTURE ONLY.
 *
 * Plain, slow, float64 CPU definitions of what the Ulysses sequence-parallel
 * attention path computes.  Only the tests, the smoke check and the CPU
 * baseline leg of the benchmark may load this file's library; the CUDA path
 * shares no code with it.
 *
 * Sources (web pages on Ulysses sequence parallelism / context parallelism):
 *  - "Million-Token-Kontexte im Training" (bytewire.ai), section "Ulysses: Die
 *    Sequenz als Verteilungseinheit": the sequence is split along the token
 *    dimension across devices and Q, K, V are exchanged by an all-to-all.
 *  - "Ulysses Sequence Parallelism" (topot.news), section "Как работает
 *    Ulysses": equal parts per device; after the all-to-all each device holds
 *    the full context for its share of the attention.
 *  - "Context Parallelism" (ultralytics.com glossary), section "So funktioniert
 *    Kontextparallelitaet": 32 000 tokens on four devices gives ~8 000 each;
 *    token-local layers run on the local shard; ring attention computes
 *    partial attention per KV block and the result is mathematically equal
 *    to attention over the full sequence.  Its code example (section
 *    "Praktische Anwendung und Kompromisse") fixes the tensor shape
 *    B x H x N x d with the sequence at dimension 2, causal scaled dot
 *    product attention with the default scale, and the loss mean(out^2).
 *
 * Readings taken where the pages are silent (heads split contiguously per
 * rank, query head h uses KV head h / (Hq/Hkv), scale 1/sqrt(d) by default,
 * natural-log LSE, top-left causal alignment j <= i) are stated per function.
 *
 * Every function computes the plain definition directly: no tiling, no online
 * softmax, no reordering beyond a two-pass max/sum for the softmax.
 *
 * Element access: input tensors are given as float32 (dtype 0) or raw bf16
 * bits (dtype 1); both are widened exactly to double.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* helpers                                                                   */

static double elem(const void* base, int dtype, size_t idx) {
    if (dtype == 0) return (double)((const float*)base)[idx];
    uint32_t bits = ((uint32_t)((const uint16_t*)base)[idx]) << 16;
    float f;
    memcpy(&f, &bits, 4);
    return (double)f;
}

typedef void (*work_fn)(void* ctx, long item);

typedef struct {
    work_fn fn;
    void* ctx;
    long n_items;
    long next;
    pthread_mutex_t mu;
} pool_t;

static void* pool_worker(void* arg) {
    pool_t* p = (pool_t*)arg;
    for (;;) {
        pthread_mutex_lock(&p->mu);
        long it = p->next++;
        pthread_mutex_unlock(&p->mu);
        if (it >= p->n_items) break;
        p->fn(p->ctx, it);
    }
    return 0;
}

/* Run fn(ctx, i) for i in [0, n_items) on up to nthreads threads. */
static void parallel_for(work_fn fn, void* ctx, long n_items, int nthreads) {
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 512) nthreads = 512;
    if (n_items < nthreads) nthreads = (int)(n_items > 0 ? n_items : 1);
    pool_t p;
    p.fn = fn;
    p.ctx = ctx;
    p.n_items = n_items;
    p.next = 0;
    pthread_mutex_init(&p.mu, 0);
    pthread_t th[512];
    int created[512];
    for (int t = 1; t < nthreads; ++t) created[t] = pthread_create(&th[t], 0, pool_worker, &p) == 0;
    pool_worker(&p);
    for (int t = 1; t < nthreads; ++t)
        if (created[t]) pthread_join(th[t], 0);
    pthread_mutex_destroy(&p.mu);
}

/* ------------------------------------------------------------------------ */
/* Layout maps (bytewire.ai "Ulysses: Die Sequenz als Verteilungseinheit";
 * topot.news "Как работает Ulysses"; ultralytics.com "So funktioniert").
 *
 * Logical tensor: [B][H][N][d], sequence at dimension 2 (ultralytics.com code
 * example: buffer_seq_dims = 2).
 * Sequence-sharded: rank p holds tokens [p*N/P, (p+1)*N/P) of every head:
 *   [P][B][N/P][H][d].
 * Head-sharded (after the all-to-all): rank r holds all N tokens of heads
 *   [r*H/P, (r+1)*H/P): [P][B][H/P][N][d].
 * Elements are moved as opaque byte strings of size esz.                    */

/* logical [B][H][N][d] -> sequence-sharded [P][B][N/P][H][d] */
int orc_shard_seq(int B, int H, long N, int d, int P, int esz, const void* logical, void* sharded) {
    if (P < 1 || N % P != 0) return 1;
    long Np = N / P;
    const char* src = (const char*)logical;
    char* dst = (char*)sharded;
    for (int b = 0; b < B; ++b)
        for (int h = 0; h < H; ++h)
            for (long n = 0; n < N; ++n)
                for (int c = 0; c < d; ++c) {
                    long p = n / Np, np_ = n % Np;
                    size_t s = ((((size_t)b * H + h) * N + n) * d + c) * (size_t)esz;
                    size_t t = (((((size_t)p * B + b) * Np + np_) * H + h) * d + c) * (size_t)esz;
                    memcpy(dst + t, src + s, (size_t)esz);
                }
    return 0;
}

/* sequence-sharded [P][B][N/P][H][d] -> logical [B][H][N][d] */
int orc_unshard_seq(int B, int H, long N, int d, int P, int esz, const void* sharded, void* logical) {
    if (P < 1 || N % P != 0) return 1;
    long Np = N / P;
    const char* src = (const char*)sharded;
    char* dst = (char*)logical;
    for (int p = 0; p < P; ++p)
        for (int b = 0; b < B; ++b)
            for (long np_ = 0; np_ < Np; ++np_)
                for (int h = 0; h < H; ++h)
                    for (int c = 0; c < d; ++c) {
                        long n = (long)p * Np + np_;
                        size_t s = (((((size_t)p * B + b) * Np + np_) * H + h) * d + c) * (size_t)esz;
                        size_t t = ((((size_t)b * H + h) * N + n) * d + c) * (size_t)esz;
                        memcpy(dst + t, src + s, (size_t)esz);
                    }
    return 0;
}

/* All-to-all seq -> head: dst[r][b][h'][n][:] = src[n/(N/P)][b][n%(N/P)][r*Hx/P+h'][:] */
int orc_seq2head(int B, int Hx, long N, int d, int P, int esz, const void* src_, void* dst_) {
    if (P < 1 || N % P != 0 || Hx % P != 0) return 1;
    long Np = N / P;
    int Hl = Hx / P;
    const char* src = (const char*)src_;
    char* dst = (char*)dst_;
    for (int r = 0; r < P; ++r)
        for (int b = 0; b < B; ++b)
            for (int hl = 0; hl < Hl; ++hl)
                for (long n = 0; n < N; ++n)
                    for (int c = 0; c < d; ++c) {
                        long p = n / Np, np_ = n % Np;
                        int h = r * Hl + hl;
                        size_t t = (((((size_t)r * B + b) * Hl + hl) * N + n) * d + c) * (size_t)esz;
                        size_t s = (((((size_t)p * B + b) * Np + np_) * Hx + h) * d + c) * (size_t)esz;
                        memcpy(dst + t, src + s, (size_t)esz);
                    }
    return 0;
}

/* All-to-all head -> seq (the return trip before token-local layers,
 * ultralytics.com "So funktioniert"):
 * dst[p][b][n'][h][:] = src[h/(Hx/P)][b][h%(Hx/P)][p*N/P+n'][:] */
int orc_head2seq(int B, int Hx, long N, int d, int P, int esz, const void* src_, void* dst_) {
    if (P < 1 || N % P != 0 || Hx % P != 0) return 1;
    long Np = N / P;
    int Hl = Hx / P;
    const char* src = (const char*)src_;
    char* dst = (char*)dst_;
    for (int p = 0; p < P; ++p)
        for (int b = 0; b < B; ++b)
            for (long np_ = 0; np_ < Np; ++np_)
                for (int h = 0; h < Hx; ++h)
                    for (int c = 0; c < d; ++c) {
                        int r = h / Hl, hl = h % Hl;
                        long n = (long)p * Np + np_;
                        size_t t = (((((size_t)p * B + b) * Np + np_) * Hx + h) * d + c) * (size_t)esz;
                        size_t s = (((((size_t)r * B + b) * Hl + hl) * N + n) * d + c) * (size_t)esz;
                        memcpy(dst + t, src + s, (size_t)esz);
                    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Attention forward for selected query rows.
 *
 * Definition (ultralytics.com code example: scaled_dot_product_attention with
 * is_causal=True; exact equivalence with full-sequence attention in "So
 * funktioniert"):
 *   S_ij   = scale * sum_c Q[b,h,i,c] K[b,hk,j,c],   hk = h / (Hq/Hkv)
 *   visible keys: key_lo <= j < key_hi and (if causal) j <= i
 *   LSE_i  = ln sum_{visible j} exp(S_ij)
 *   O_i    = sum_{visible j} exp(S_ij - LSE_i) V[b,hk,j,:]
 * The key range [key_lo, key_hi) gives the partial attention of one KV block
 * (ring attention, "So funktioniert").  No visible key: LSE = -inf, O = 0.
 * Inputs are logical [B][H][N][d].  Outputs: o [B][Hq][nrows][d],
 * lse [B][Hq][nrows] for the query positions rows[0..nrows).               */

typedef struct {
    int B, Hq, Hkv, d, dtype, causal;
    long N, key_lo, key_hi, nrows;
    double scale;
    const void *q, *k, *v;
    const int64_t* rows;
    double *o, *lse;
} fwd_ctx;

static void fwd_item(void* vctx, long item) {
    fwd_ctx* c = (fwd_ctx*)vctx;
    long r = item % c->nrows;
    long bh = item / c->nrows;
    int h = (int)(bh % c->Hq), b = (int)(bh / c->Hq);
    int hk = h / (c->Hq / c->Hkv);
    long i = (long)c->rows[r];
    int d = c->d;
    long jhi = c->key_hi;
    if (c->causal && i + 1 < jhi) jhi = i + 1;
    long jlo = c->key_lo;
    double* orow = c->o + ((size_t)bh * c->nrows + r) * d;
    for (int t = 0; t < d; ++t) orow[t] = 0.0;
    if (jhi <= jlo) {
        c->lse[(size_t)bh * c->nrows + r] = -INFINITY;
        return;
    }
    size_t qbase = (((size_t)b * c->Hq + h) * c->N + i) * d;
    double* s = (double*)malloc(sizeof(double) * (size_t)(jhi - jlo));
    double mx = -INFINITY;
    for (long j = jlo; j < jhi; ++j) {
        size_t kbase = (((size_t)b * c->Hkv + hk) * c->N + j) * d;
        double acc = 0.0;
        for (int t = 0; t < d; ++t) acc += elem(c->q, c->dtype, qbase + t) * elem(c->k, c->dtype, kbase + t);
        s[j - jlo] = c->scale * acc;
        if (s[j - jlo] > mx) mx = s[j - jlo];
    }
    double l = 0.0;
    for (long j = jlo; j < jhi; ++j) l += exp(s[j - jlo] - mx);
    double lse = mx + log(l);
    for (long j = jlo; j < jhi; ++j) {
        double p = exp(s[j - jlo] - lse);
        size_t vbase = (((size_t)b * c->Hkv + hk) * c->N + j) * d;
        for (int t = 0; t < d; ++t) orow[t] += p * elem(c->v, c->dtype, vbase + t);
    }
    c->lse[(size_t)bh * c->nrows + r] = lse;
    free(s);
}

int orc_attn_rows(int B, int Hq, int Hkv, long N, int d, const void* q, const void* k, const void* v,
                  int dtype, int causal, double scale, long key_lo, long key_hi, long nrows,
                  const int64_t* rows, double* o, double* lse, int nthreads) {
    if (Hkv < 1 || Hq % Hkv != 0 || nrows < 0 || key_lo < 0 || key_hi > N) return 1;
    for (long r = 0; r < nrows; ++r)
        if (rows[r] < 0 || rows[r] >= N) return 1;
    fwd_ctx c = {B, Hq, Hkv, d, dtype, causal, N, key_lo, key_hi, nrows, scale, q, k, v, rows, o, lse};
    parallel_for(fwd_item, &c, (long)B * Hq * nrows, nthreads);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Backward, query side: gradient of loss L with dL/dO = dO (the loss of the
 * ultralytics.com code example is mean(out^2), whose dO is 2*O/numel; any dO
 * is accepted here).  For each selected query row i (definitions as above):
 *   P_ij  = exp(S_ij - LSE_i)            (recomputed from the definition)
 *   O_i   = sum_j P_ij V_j,  D_i = dO_i . O_i
 *   dP_ij = dO_i . V_j
 *   dS_ij = P_ij (dP_ij - D_i)
 *   dQ_i  = scale * sum_j dS_ij K_j
 * dO is the full logical [B][Hq][N][d] tensor (only the selected rows are
 * read), float32 or bf16 independently of Q/K/V (dout_dtype).  Output dq
 * [B][Hq][nrows][d].                                      */

typedef struct {
    int B, Hq, Hkv, d, dtype, dout_dtype, causal;
    long N, nrows;
    double scale;
    const void *q, *k, *v, *dout;
    const int64_t* rows;
    double* dq;
} bwdq_ctx;

static void bwdq_item(void* vctx, long item) {
    bwdq_ctx* c = (bwdq_ctx*)vctx;
    long r = item % c->nrows;
    long bh = item / c->nrows;
    int h = (int)(bh % c->Hq), b = (int)(bh / c->Hq);
    int hk = h / (c->Hq / c->Hkv);
    long i = (long)c->rows[r];
    int d = c->d;
    long jhi = c->causal ? i + 1 : c->N;
    size_t qbase = (((size_t)b * c->Hq + h) * c->N + i) * d;
    double* s = (double*)malloc(sizeof(double) * (size_t)jhi);
    double* oi = (double*)calloc((size_t)d, sizeof(double));
    double mx = -INFINITY;
    for (long j = 0; j < jhi; ++j) {
        size_t kbase = (((size_t)b * c->Hkv + hk) * c->N + j) * d;
        double acc = 0.0;
        for (int t = 0; t < d; ++t) acc += elem(c->q, c->dtype, qbase + t) * elem(c->k, c->dtype, kbase + t);
        s[j] = c->scale * acc;
        if (s[j] > mx) mx = s[j];
    }
    double l = 0.0;
    for (long j = 0; j < jhi; ++j) l += exp(s[j] - mx);
    double lse = mx + log(l);
    for (long j = 0; j < jhi; ++j) {
        s[j] = exp(s[j] - lse); /* s now holds P_ij */
        size_t vbase = (((size_t)b * c->Hkv + hk) * c->N + j) * d;
        for (int t = 0; t < d; ++t) oi[t] += s[j] * elem(c->v, c->dtype, vbase + t);
    }
    double Di = 0.0;
    for (int t = 0; t < d; ++t) Di += elem(c->dout, c->dout_dtype, qbase + t) * oi[t];
    double* dqrow = c->dq + ((size_t)bh * c->nrows + r) * d;
    for (int t = 0; t < d; ++t) dqrow[t] = 0.0;
    for (long j = 0; j < jhi; ++j) {
        size_t vbase = (((size_t)b * c->Hkv + hk) * c->N + j) * d;
        double dp = 0.0;
        for (int t = 0; t < d; ++t) dp += elem(c->dout, c->dout_dtype, qbase + t) * elem(c->v, c->dtype, vbase + t);
        double ds = s[j] * (dp - Di);
        for (int t = 0; t < d; ++t) dqrow[t] += c->scale * ds * elem(c->k, c->dtype, vbase + t);
    }
    free(s);
    free(oi);
}

int orc_attn_bwd_q_rows(int B, int Hq, int Hkv, long N, int d, const void* q, const void* k, const void* v,
                        const void* dout, int dtype, int dout_dtype, int causal, double scale, long nrows,
                        const int64_t* rows, double* dq, int nthreads) {
    if (Hkv < 1 || Hq % Hkv != 0 || nrows < 0) return 1;
    for (long r = 0; r < nrows; ++r)
        if (rows[r] < 0 || rows[r] >= N) return 1;
    bwdq_ctx c = {B, Hq, Hkv, d, dtype, dout_dtype, causal, N, nrows, scale, q, k, v, dout, rows, dq};
    parallel_for(bwdq_item, &c, (long)B * Hq * nrows, nthreads);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Backward, key/value side, for selected key rows j of each KV head hk; the
 * sums run over every query head h of the group (h / (Hq/Hkv) == hk) and
 * every query row i that sees key j (i >= j if causal, else all i):
 *   P_ij  = exp(S_ij - LSE_i)
 *   dV_j  = sum_h sum_i P_ij dO_i
 *   dS_ij = P_ij (dO_i . V_j - D_i)
 *   dK_j  = scale * sum_h sum_i dS_ij Q_i
 * lse and dvec are [B][Hq][N] arrays of LSE_i and D_i = dO_i . O_i; only the
 * entries of rows i that see a selected key are read.
 * Outputs dk, dv: [B][Hkv][nrows][d].                                      */

typedef struct {
    int B, Hq, Hkv, d, dtype, dout_dtype, causal;
    long N, nrows;
    double scale;
    const void *q, *k, *v, *dout;
    const double *lse, *dvec;
    const int64_t* rows;
    double *dk, *dv;
} bwdkv_ctx;

static void bwdkv_item(void* vctx, long item) {
    bwdkv_ctx* c = (bwdkv_ctx*)vctx;
    long r = item % c->nrows;
    long bhk = item / c->nrows;
    int hk = (int)(bhk % c->Hkv), b = (int)(bhk / c->Hkv);
    int g = c->Hq / c->Hkv;
    long j = (long)c->rows[r];
    int d = c->d;
    size_t kbase = (((size_t)b * c->Hkv + hk) * c->N + j) * d;
    double* dkrow = c->dk + ((size_t)bhk * c->nrows + r) * d;
    double* dvrow = c->dv + ((size_t)bhk * c->nrows + r) * d;
    for (int t = 0; t < d; ++t) dkrow[t] = dvrow[t] = 0.0;
    for (int h = hk * g; h < (hk + 1) * g; ++h) {
        long ilo = c->causal ? j : 0;
        for (long i = ilo; i < c->N; ++i) {
            size_t qbase = (((size_t)b * c->Hq + h) * c->N + i) * d;
            double acc = 0.0;
            for (int t = 0; t < d; ++t) acc += elem(c->q, c->dtype, qbase + t) * elem(c->k, c->dtype, kbase + t);
            double sij = c->scale * acc;
            double lse_i = c->lse[((size_t)b * c->Hq + h) * c->N + i];
            double pij = exp(sij - lse_i);
            double dp = 0.0;
            for (int t = 0; t < d; ++t) dp += elem(c->dout, c->dout_dtype, qbase + t) * elem(c->v, c->dtype, kbase + t);
            double ds = pij * (dp - c->dvec[((size_t)b * c->Hq + h) * c->N + i]);
            for (int t = 0; t < d; ++t) {
                dvrow[t] += pij * elem(c->dout, c->dout_dtype, qbase + t);
                dkrow[t] += c->scale * ds * elem(c->q, c->dtype, qbase + t);
            }
        }
    }
}

int orc_attn_bwd_kv_rows(int B, int Hq, int Hkv, long N, int d, const void* q, const void* k, const void* v,
                         const void* dout, int dtype, int dout_dtype, int causal, double scale, const double* lse,
                         const double* dvec, long nrows, const int64_t* rows, double* dk, double* dv,
                         int nthreads) {
    if (Hkv < 1 || Hq % Hkv != 0 || nrows < 0) return 1;
    for (long r = 0; r < nrows; ++r)
        if (rows[r] < 0 || rows[r] >= N) return 1;
    bwdkv_ctx c = {B, Hq, Hkv, d, dtype, dout_dtype, causal, N, nrows, scale, q, k, v, dout, lse, dvec, rows, dk, dv};
    parallel_for(bwdkv_item, &c, (long)B * Hkv * nrows, nthreads);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Exact merge of two partial attentions over disjoint key sets (ring
 * attention, ultralytics.com "So funktioniert": partial attention per KV
 * block, equal to full-sequence attention in the end).  With
 * O_x = sum_{j in X} exp(S_j - LSE_x) V_j and LSE_x = ln sum_{j in X} exp(S_j):
 *   LSE = ln(exp(LSE_a) + exp(LSE_b))
 *   O   = exp(LSE_a - LSE) O_a + exp(LSE_b - LSE) O_b
 * An empty partial has LSE = -inf and contributes nothing.                  */
void orc_lse_merge(long rows, int d, const double* o_a, const double* lse_a, const double* o_b,
                   const double* lse_b, double* o, double* lse) {
    for (long r = 0; r < rows; ++r) {
        double la = lse_a[r], lb = lse_b[r];
        if (la == -INFINITY && lb == -INFINITY) {
            lse[r] = -INFINITY;
            for (int t = 0; t < d; ++t) o[(size_t)r * d + t] = 0.0;
            continue;
        }
        double m = la > lb ? la : lb;
        double l = m + log(exp(la - m) + exp(lb - m));
        double wa = exp(la - l), wb = exp(lb - l);
        for (int t = 0; t < d; ++t)
            o[(size_t)r * d + t] = wa * o_a[(size_t)r * d + t] + wb * o_b[(size_t)r * d + t];
        lse[r] = l;
    }
}
