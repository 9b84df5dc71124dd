/*
 * Oracle for MLA verify attention -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, double-precision CPU implementation of what the verify
 * attention of "The Occupancy Epiphany" pages computes: a block of q_len draft
 * queries per stream, H heads, a 576-d absorbed query (512 latent + 64 rope)
 * attending over a page_size=1 latent KV pool whose rows' first 512 dims double
 * as V, with a causal-chain or tree mask among the drafts.  Every output row is
 * computed from the definition, in two passes (scores, then weights), with no
 * tiling, no online softmax and no KV split.  Only tests, the smoke check and
 * the benchmark's CPU-baseline leg may load this library; the CUDA library
 * shares no code with it.
 *
 * Definitions followed (restated, not copied):
 *  - MLA absorbed attention, "latent head dimension is 512" -- "The Occupancy
 *    Probe", section "The Scene: What Came Before": a key row is 576-d
 *    (512 latent + 64 rope), V is the 512-d latent part of the same row.
 *  - verify attention of draft tokens against the whole KV cache with
 *    page_size=1 paging -- "The Occupancy Epiphany: How a CUDA Kernel Designer
 *    Discovered ...", section "Context: The Problem and the Stakes".
 *  - draft tree verification (DDTree) -- "The Occupancy Epiphany: How One
 *    Environment Variable Unlocked 3x Throughput ...", sections "The Broader
 *    Context" and "Assumptions Underlying the Reasoning".
 *  - fp8 latent KV with per-token scales, gathered by top-k indices -- "The
 *    Occupancy Probe", section "The Scene: What Came Before".
 * Readings where the pages are silent (drafts occupy the last q_len keys of a
 * stream, mask[b,t,i] = draft t sees draft i, NULL mask = causal chain, one
 * scale over all 576 dims, natural-log LSE of the scaled scores, empty key set
 * gives out = 0 and lse = -inf) are listed in the design notes.
 *
 * Precision: inputs are decoded exactly (bf16 and e4m3 both embed exactly in
 * double); all arithmetic is IEEE double.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define D_QK 576
#define D_V 512
#define D_ROPE 64

enum { OR_OK = 0, OR_ERR_ARG = -1, OR_ERR_LEN = -2, OR_ERR_SLOT = -3, OR_ERR_NOMEM = -4 };

/* bf16 bit pattern -> double: the bf16 bits are the top half of a float32. */
double oracle_bf16_to_f64(uint16_t bits) {
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* OCP 8-bit floating point, E4M3 ("fn" variant): 1 sign bit, 4 exponent bits with
 * bias 7, 3 mantissa bits; exponent field 0 is subnormal (m * 2^-9); S.1111.111
 * is NaN; there are no infinities, so the largest finite magnitude is
 * 1.75 * 2^8 = 448. */
double oracle_e4m3_to_f64(uint8_t byte) {
    int sign = (byte >> 7) & 1, e = (byte >> 3) & 0xF, m = byte & 7;
    double v;
    if (e == 0xF && m == 7) return NAN;
    if (e == 0) v = ldexp((double)m, -9);
    else v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return sign ? -v : v;
}

void oracle_bf16_to_f64_array(const uint16_t* in, double* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_bf16_to_f64(in[i]);
}

void oracle_e4m3_to_f64_array(const uint8_t* in, double* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_e4m3_to_f64(in[i]);
}

/* ------------------------------------------------------------------------ */
/* Masked softmax attention of one query row over an explicit key list.      */
/* get_key(ctx, j, buf) decodes the j-th listed key (576 dims) into buf;     */
/* out gets the 512 V dims.                                                  */
/* ------------------------------------------------------------------------ */
typedef void (*key_fn)(const void* ctx, int64_t j, double* buf);

static void attend_row(const double* q, key_fn get_key, const void* ctx, int64_t nk,
                       double scale, double* scores, double* kbuf, double* out, double* lse) {
    int64_t j;
    int d;
    for (d = 0; d < D_V; ++d) out[d] = 0.0;
    if (nk == 0) { *lse = -INFINITY; return; }
    /* pass 1: s_j = scale * <q, k_j> over all 576 dims */
    double m = -INFINITY;
    for (j = 0; j < nk; ++j) {
        get_key(ctx, j, kbuf);
        double acc = 0.0;
        for (d = 0; d < D_QK; ++d) acc += q[d] * kbuf[d];
        scores[j] = scale * acc;
        if (scores[j] > m) m = scores[j];
    }
    /* log-sum-exp with the maximum taken out */
    double z = 0.0;
    for (j = 0; j < nk; ++j) z += exp(scores[j] - m);
    double l = m + log(z);
    /* pass 2: out = sum_j softmax_j * v_j, v_j = first 512 dims of key j */
    for (j = 0; j < nk; ++j) {
        double w = exp(scores[j] - l);
        get_key(ctx, j, kbuf);
        for (d = 0; d < D_V; ++d) out[d] += w * kbuf[d];
    }
    *lse = l;
}

/* ------------------------------------------------------------------------ */
/* Verify attention                                                          */
/* ------------------------------------------------------------------------ */
typedef struct {
    const uint16_t* q; const uint16_t* kv; int64_t n_pool;
    const int32_t* slot; int slot_stride; const int32_t* seq_lens; const uint8_t* mask;
    const uint64_t* mask_bits;        /* packed form of the same mask (one word per draft) */
    int B, q_len, H; double scale;
    int64_t key_begin, key_end;       /* keys j restricted to [key_begin, key_end) */
    const int64_t* rows; int64_t n_rows;
    double* out; double* lse;
    int nthreads, tid;
    int status;
} verify_job;

/* Draft t of stream b sees key j (0 <= j < n) iff j is a prefix key, or j is
 * draft i = j - p and mask[b, t, i] = 1 (NULL mask: i <= t).  The packed form
 * holds the same relation as bit i of the 64-bit word mask_bits[b, t]. */
static int visible(const verify_job* J, int b, int t, int64_t j, int64_t p) {
    if (j < p) return 1;
    int64_t i = j - p;
    if (J->mask_bits != NULL) return (int)((J->mask_bits[(int64_t)b * J->q_len + t] >> i) & 1u);
    if (J->mask == NULL) return i <= t;
    return J->mask[((int64_t)b * J->q_len + t) * J->q_len + i] != 0;
}

typedef struct { const uint16_t* kv; const int64_t* list; } bf16_keys;

static void bf16_key(const void* ctx, int64_t j, double* buf) {
    const bf16_keys* K = (const bf16_keys*)ctx;
    const uint16_t* row = K->kv + K->list[j] * D_QK;
    for (int d = 0; d < D_QK; ++d) buf[d] = oracle_bf16_to_f64(row[d]);
}

static void* verify_worker(void* arg) {
    verify_job* J = (verify_job*)arg;
    int64_t cap = J->slot_stride > 0 ? J->slot_stride : 1;
    double* qd = (double*)malloc(sizeof(double) * D_QK);
    double* kbuf = (double*)malloc(sizeof(double) * D_QK);
    double* scores = (double*)malloc(sizeof(double) * cap);
    int64_t* list = (int64_t*)malloc(sizeof(int64_t) * cap);
    if (!qd || !kbuf || !scores || !list) { J->status = OR_ERR_NOMEM; goto done; }
    int64_t total = J->rows ? J->n_rows : (int64_t)J->B * J->q_len * J->H;
    for (int64_t r = J->tid; r < total; r += J->nthreads) {
        int64_t flat = J->rows ? J->rows[r] : r;
        if (flat < 0 || flat >= (int64_t)J->B * J->q_len * J->H) { J->status = OR_ERR_ARG; goto done; }
        int h = (int)(flat % J->H);
        int t = (int)((flat / J->H) % J->q_len);
        int b = (int)(flat / ((int64_t)J->H * J->q_len));
        (void)h;
        int64_t n = J->seq_lens[b];
        if (n < J->q_len || n > J->slot_stride) { J->status = OR_ERR_LEN; goto done; }
        int64_t p = n - J->q_len;
        const uint16_t* qrow = J->q + flat * D_QK;
        for (int d = 0; d < D_QK; ++d) qd[d] = oracle_bf16_to_f64(qrow[d]);
        int64_t nk = 0;
        int64_t j0 = J->key_begin > 0 ? J->key_begin : 0;
        int64_t j1 = J->key_end < n ? J->key_end : n;
        for (int64_t j = j0; j < j1; ++j) {
            if (!visible(J, b, t, j, p)) continue;
            int64_t s = J->slot[(int64_t)b * J->slot_stride + j];
            if (s < 0 || s >= J->n_pool) { J->status = OR_ERR_SLOT; goto done; }
            list[nk++] = s;
        }
        bf16_keys K = { J->kv, list };
        attend_row(qd, bf16_key, &K, nk, J->scale, scores, kbuf, J->out + r * D_V, J->lse + r);
    }
done:
    free(qd); free(kbuf); free(scores); free(list);
    return NULL;
}

static int run_jobs(verify_job* base, int nthreads, void* (*fn)(void*), size_t job_size) {
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    pthread_t th[256];
    int joined[256];
    char* jobs = (char*)malloc(job_size * (size_t)nthreads);
    if (!jobs) return OR_ERR_NOMEM;
    for (int i = 0; i < nthreads; ++i) {
        verify_job* J = (verify_job*)(jobs + job_size * (size_t)i);
        memcpy(J, base, job_size);
        J->nthreads = nthreads; J->tid = i; J->status = OR_OK;
        joined[i] = pthread_create(&th[i], NULL, fn, J) == 0;
        if (!joined[i]) fn(J);          /* no thread available: run this share inline */
    }
    int status = OR_OK;
    for (int i = 0; i < nthreads; ++i) if (joined[i]) pthread_join(th[i], NULL);
    for (int i = 0; i < nthreads; ++i) {
        verify_job* J = (verify_job*)(jobs + job_size * (size_t)i);
        if (J->status != OR_OK) status = J->status;
    }
    free(jobs);
    return status;
}

/*
 * out[r, 0:512], lse[r] for every query row r = (b, t, h) in natural order
 * (rows == NULL), or for the n_rows flat rows listed in `rows` (output row k
 * belongs to rows[k]).  Flat row index = (b * q_len + t) * H + h.
 * Keys are restricted to [key_begin, key_end) (pass 0 and INT64_MAX for all).
 */
int oracle_mla_verify(const uint16_t* q, const uint16_t* kv, int64_t n_pool,
                      const int32_t* slot_table, int slot_stride, const int32_t* seq_lens,
                      const uint8_t* mask, int B, int q_len, int H, double scale,
                      int64_t key_begin, int64_t key_end,
                      const int64_t* rows, int64_t n_rows,
                      double* out, double* lse, int nthreads) {
    if (!q || !kv || !slot_table || !seq_lens || !out || !lse) return OR_ERR_ARG;
    if (B < 0 || q_len < 1 || H < 1 || slot_stride < 0 || n_pool < 0) return OR_ERR_ARG;
    verify_job J;
    memset(&J, 0, sizeof J);
    J.q = q; J.kv = kv; J.n_pool = n_pool; J.slot = slot_table; J.slot_stride = slot_stride;
    J.seq_lens = seq_lens; J.mask = mask; J.B = B; J.q_len = q_len; J.H = H; J.scale = scale;
    J.key_begin = key_begin; J.key_end = key_end; J.rows = rows; J.n_rows = n_rows;
    J.out = out; J.lse = lse;
    return run_jobs(&J, nthreads, verify_worker, sizeof(verify_job));
}

/*
 * The same with the draft mask bit-packed: bit i of mask_bits[b * q_len + t] set
 * means draft t sees draft i (q_len <= 64); NULL means the causal chain.
 * Larger draft trees ("The Occupancy Epiphany: How One Environment Variable
 * Unlocked 3x Throughput ...", sections "The Broader Context" and "Input
 * Knowledge Required": DDTree draft trees) need more than the 8-16 drafts of a
 * chain, and one 64-bit word per draft holds a tree of up to 64 nodes.
 */
int oracle_mla_verify_packed(const uint16_t* q, const uint16_t* kv, int64_t n_pool,
                             const int32_t* slot_table, int slot_stride, const int32_t* seq_lens,
                             const uint64_t* mask_bits, int B, int q_len, int H, double scale,
                             int64_t key_begin, int64_t key_end,
                             const int64_t* rows, int64_t n_rows,
                             double* out, double* lse, int nthreads) {
    if (!q || !kv || !slot_table || !seq_lens || !out || !lse) return OR_ERR_ARG;
    if (B < 0 || q_len < 1 || q_len > 64 || H < 1 || slot_stride < 0 || n_pool < 0) return OR_ERR_ARG;
    verify_job J;
    memset(&J, 0, sizeof J);
    J.q = q; J.kv = kv; J.n_pool = n_pool; J.slot = slot_table; J.slot_stride = slot_stride;
    J.seq_lens = seq_lens; J.mask = NULL; J.mask_bits = mask_bits; J.B = B; J.q_len = q_len; J.H = H;
    J.scale = scale; J.key_begin = key_begin; J.key_end = key_end; J.rows = rows; J.n_rows = n_rows;
    J.out = out; J.lse = lse;
    return run_jobs(&J, nthreads, verify_worker, sizeof(verify_job));
}

/* ------------------------------------------------------------------------ */
/* KV append                                                                 */
/* ------------------------------------------------------------------------ */
/*
 * Before a verify step the q_len draft rows of each stream enter the paged
 * latent cache ("The Occupancy Epiphany: How One Environment Variable ...",
 * section "The Broader Context": KV slots handed out by a paged allocator,
 * possibly scattered): row i of stream b, new_kv[b, i, 0:576], is written to
 * pool row slot_table[b, seq_lens[b] - q_len + i] (the drafts are the last
 * q_len keys of the stream).  All lengths and slots are checked first; on an
 * error nothing is written.
 */
int oracle_kv_append(uint16_t* kv, int64_t n_pool, const int32_t* slot_table, int slot_stride,
                     const int32_t* seq_lens, const uint16_t* new_kv, int B, int q_len) {
    if (!kv || !slot_table || !seq_lens || !new_kv || B < 0 || q_len < 1 || slot_stride < q_len) return OR_ERR_ARG;
    for (int b = 0; b < B; ++b) {
        int64_t n = seq_lens[b];
        if (n < q_len || n > slot_stride) return OR_ERR_LEN;
        for (int i = 0; i < q_len; ++i) {
            int64_t s = slot_table[(int64_t)b * slot_stride + (n - q_len + i)];
            if (s < 0 || s >= n_pool) return OR_ERR_SLOT;
        }
    }
    for (int b = 0; b < B; ++b) {
        int64_t n = seq_lens[b];
        for (int i = 0; i < q_len; ++i) {
            int64_t s = slot_table[(int64_t)b * slot_stride + (n - q_len + i)];
            memcpy(kv + s * D_QK, new_kv + ((int64_t)b * q_len + i) * D_QK, sizeof(uint16_t) * D_QK);
        }
    }
    return OR_OK;
}

/* ------------------------------------------------------------------------ */
/* Combine of KV-split partials (log-sum-exp weighted merge)                 */
/* ------------------------------------------------------------------------ */
/*
 * part_out [n_rows, S, Dv] holds each split's normalised output and part_lse
 * [n_rows, S] its log-sum-exp; a split with no keys has lse = -inf.
 * lse = log(sum_s exp(lse_s)); out = sum_s exp(lse_s - lse) * out_s.
 * A row whose splits are all empty gets out = 0, lse = -inf.
 */
void oracle_mla_combine(const double* part_out, const double* part_lse, int64_t n_rows, int S,
                        int Dv, double* out, double* lse) {
    for (int64_t r = 0; r < n_rows; ++r) {
        const double* pl = part_lse + r * S;
        double m = -INFINITY;
        for (int s = 0; s < S; ++s) if (pl[s] > m) m = pl[s];
        double* o = out + r * Dv;
        for (int d = 0; d < Dv; ++d) o[d] = 0.0;
        if (m == -INFINITY) { lse[r] = -INFINITY; continue; }
        double z = 0.0;
        for (int s = 0; s < S; ++s) z += exp(pl[s] - m);
        double l = m + log(z);
        for (int s = 0; s < S; ++s) {
            double w = exp(pl[s] - l);
            if (w == 0.0) continue;
            const double* po = part_out + (r * S + s) * Dv;
            for (int d = 0; d < Dv; ++d) o[d] += w * po[d];
        }
        lse[r] = l;
    }
}

/* ------------------------------------------------------------------------ */
/* fp8 (e4m3) latent sparse decode, q_len = 1, top-k index lists             */
/* ------------------------------------------------------------------------ */
typedef struct {
    verify_job base;                   /* nthreads / tid / status / rows / out / lse / scale */
    const uint16_t* q; const uint8_t* lat; const float* kscale; const uint16_t* rope;
    int64_t n_pool; const int32_t* topk_slots; int topk; int B; int H;
} sparse_job;

typedef struct { const uint8_t* lat; const float* kscale; const uint16_t* rope; const int32_t* list; } fp8_keys;

/* latent: dequantised e4m3 code times the token's scale; rope: bf16 */
static void fp8_key(const void* ctx, int64_t j, double* buf) {
    const fp8_keys* K = (const fp8_keys*)ctx;
    int64_t s = K->list[j];
    double ts = (double)K->kscale[s];
    for (int d = 0; d < D_V; ++d) buf[d] = oracle_e4m3_to_f64(K->lat[s * D_V + d]) * ts;
    for (int d = 0; d < D_ROPE; ++d) buf[D_V + d] = oracle_bf16_to_f64(K->rope[s * D_ROPE + d]);
}

static void* sparse_worker(void* arg) {
    sparse_job* S = (sparse_job*)arg;
    verify_job* J = &S->base;
    int64_t cap = S->topk > 0 ? S->topk : 1;
    double* qd = (double*)malloc(sizeof(double) * D_QK);
    double* kbuf = (double*)malloc(sizeof(double) * D_QK);
    double* scores = (double*)malloc(sizeof(double) * cap);
    if (!qd || !kbuf || !scores) { J->status = OR_ERR_NOMEM; goto done; }
    int64_t total = J->rows ? J->n_rows : (int64_t)S->B * S->H;
    for (int64_t r = J->tid; r < total; r += J->nthreads) {
        int64_t flat = J->rows ? J->rows[r] : r;
        if (flat < 0 || flat >= (int64_t)S->B * S->H) { J->status = OR_ERR_ARG; goto done; }
        int b = (int)(flat / S->H);
        for (int d = 0; d < D_QK; ++d) qd[d] = oracle_bf16_to_f64(S->q[flat * D_QK + d]);
        const int32_t* list = S->topk_slots + (int64_t)b * S->topk;
        for (int j = 0; j < S->topk; ++j)
            if (list[j] < 0 || list[j] >= S->n_pool) { J->status = OR_ERR_SLOT; goto done; }
        fp8_keys K = { S->lat, S->kscale, S->rope, list };
        attend_row(qd, fp8_key, &K, S->topk, J->scale, scores, kbuf, J->out + r * D_V, J->lse + r);
    }
done:
    free(qd); free(kbuf); free(scores);
    return NULL;
}

/*
 * q [B, H, 576] bf16; kv_lat [n_pool, 512] e4m3 codes; kv_scale [n_pool] f32;
 * kv_rope [n_pool, 64] bf16; topk_slots [B, topk].  Row r = b * H + h.
 */
int oracle_mla_sparse_fp8(const uint16_t* q, const uint8_t* kv_lat, const float* kv_scale,
                          const uint16_t* kv_rope, int64_t n_pool, const int32_t* topk_slots,
                          int topk, int B, int H, double scale,
                          const int64_t* rows, int64_t n_rows,
                          double* out, double* lse, int nthreads) {
    if (!q || !kv_lat || !kv_scale || !kv_rope || !topk_slots || !out || !lse) return OR_ERR_ARG;
    if (B < 0 || H < 1 || topk < 0) return OR_ERR_ARG;
    sparse_job S;
    memset(&S, 0, sizeof S);
    S.base.scale = scale; S.base.rows = rows; S.base.n_rows = n_rows;
    S.base.out = out; S.base.lse = lse;
    S.q = q; S.lat = kv_lat; S.kscale = kv_scale; S.rope = kv_rope; S.n_pool = n_pool;
    S.topk_slots = topk_slots; S.topk = topk; S.B = B; S.H = H;
    return run_jobs(&S.base, nthreads, sparse_worker, sizeof(sparse_job));
}

/*
 * Row scatter of the fp8 cache's append: row i of each source array goes to pool row
 * slots[i] of the matching cache array (latent codes, per-token scale, rope), the rows
 * having been quantised by the caller (the pages fix no quantisation rule).  All
 * slots are checked first; on an error nothing is written.
 */
int oracle_kv_append_rows(uint8_t* dst, int64_t n_pool, int64_t row_bytes, const int32_t* slots,
                          const uint8_t* src, int64_t n_rows) {
    if (!dst || !slots || !src || n_rows < 0 || row_bytes < 1) return OR_ERR_ARG;
    for (int64_t i = 0; i < n_rows; ++i)
        if (slots[i] < 0 || slots[i] >= n_pool) return OR_ERR_SLOT;
    for (int64_t i = 0; i < n_rows; ++i)
        memcpy(dst + (int64_t)slots[i] * row_bytes, src + i * row_bytes, (size_t)row_bytes);
    return OR_OK;
}
