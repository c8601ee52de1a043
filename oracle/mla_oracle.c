/*
 * mla_oracle.c -- plain, slow, fp64 CPU oracle for absorbed-form MLA decode
 * over a paged latent KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or calls
 * this file: only the tests, the package smoke check and the benchmark's
 * CPU-baseline / reference arm do.  It shares no code, header, table or helper
 * with the CUDA library.
 *
 * What it computes (the plain definition; no blocking, fusion or reordering):
 *   For request b, query index i in [0, q_len) and head h, with L = seq_lens[b]
 *   (L counts the q_len new tokens):
 *     V      = L - q_len + 1 + i                       visible tokens (causal)
 *     x_t    = kv_cache[block_table[b, t / page], t % page, 0:576]   t < V
 *     s_t    = softmax_scale * (q_nope . x_t[0:512] + q_pe . x_t[512:576])
 *     m      = max_t s_t ;  Z = sum_t exp(s_t - m) ;  lse = m + ln Z
 *     out    = sum_t exp(s_t - lse) * x_t[0:512]
 *   With an FP8 cache x_t = decode_e4m3(byte) * kv_scale.
 *
 * Sources: vLLM PR #41778 "TOKENSPEED_MLA" summary (DeepSeek-R1 MLA dims
 * qk_nope=128, qk_rope=64 in risk 4; uniform query length; FP8 dequant scale in
 * the implementation breakdown, step 1) and vLLM PR #46819 "Triton MLA attn
 * logits preallocation" summary (split partials of width kv_lora_rank + 1 in
 * the key code excerpt).  The absorbed formula itself (512-d c_kv + 64-d k_pe
 * rows, score = scale*(q_nope.c_kv + q_pe.k_pe), scale = 1/sqrt(192), output
 * sum softmax*c_kv plus per-row LSE) is the benchmark spec's; the pages print
 * no formula.
 *
 * Readings taken where the pages are silent: seq_len includes the q_len new
 * tokens and query i sits at absolute position L - q_len + i; LSE is the
 * natural log; V = c_kv (k_pe is key-only); q_pe/k_pe arrive already rotated;
 * slots past L in the last page are never part of the result.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define KV_LORA 512
#define ROPE 64
#define ROW (KV_LORA + ROPE)

/* bf16 -> double: a bf16 value is the top 16 bits of an IEEE binary32. */
double oracle_bf16_to_double(uint16_t bits) {
    uint32_t w = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &w, sizeof f);
    return (double)f;
}

/* OCP FP8 E4M3 (e4m3fn) -> double, written from the format definition:
 * 1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits, no infinities,
 * S.1111.111 is NaN, exponent field 0 encodes subnormals m * 2^-9. */
double oracle_e4m3_to_double(uint8_t byte) {
    int s = (byte >> 7) & 1;
    int e = (byte >> 3) & 0xF;
    int m = byte & 0x7;
    double v;
    if (e == 0xF && m == 0x7) return NAN;
    if (e == 0)
        v = ldexp((double)m, -9);
    else
        v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return s ? -v : v;
}

/* double -> OCP FP8 E4M3 (e4m3fn) code: round to nearest, ties to even, on the
 * e4m3 grid (spacing 2^(E-3) in binade [2^E, 2^(E+1)) for E >= -6, and the
 * subnormal spacing 2^-9 below 2^-6); magnitudes of 448 and beyond (and
 * infinities) saturate to the largest finite code, NaN gives 0x7F.  The code
 * is found by searching the decoder's table, so encode and decode agree by
 * construction.  Used to quantise an FP8 output with a per-tensor scale. */
uint8_t oracle_e4m3_encode(double x) {
    if (isnan(x)) return 0x7F;
    uint8_t sign = signbit(x) ? 0x80 : 0x00;
    double a = fabs(x);
    if (a >= 448.0) return sign | 0x7E;
    int e2;
    frexp(a, &e2);          /* a = f * 2^e2 with f in [0.5, 1): binade 2^(e2-1) */
    int E = e2 - 1;
    if (E < -6) E = -6;     /* subnormals share the smallest normal binade's spacing */
    double q = ldexp(1.0, E - 3);
    double v = rint(a / q) * q;  /* default rounding mode: nearest, ties to even */
    for (int c = 0; c <= 0x7E; ++c)
        if (oracle_e4m3_to_double((uint8_t)c) == v) return sign | (uint8_t)c;
    return 0x7F;            /* unreachable: every rounded value is on the grid */
}

void oracle_e4m3_encode_array(const double* src, uint8_t* dst, int64_t n) {
    for (int64_t k = 0; k < n; ++k) dst[k] = oracle_e4m3_encode(src[k]);
}

void oracle_bf16_array_to_double(const uint16_t* src, double* dst, int64_t n) {
    for (int64_t k = 0; k < n; ++k) dst[k] = oracle_bf16_to_double(src[k]);
}

void oracle_e4m3_array_to_double(const uint8_t* src, double* dst, int64_t n) {
    for (int64_t k = 0; k < n; ++k) dst[k] = oracle_e4m3_to_double(src[k]);
}

typedef struct {
    int batch, num_heads, q_len, page_size;
    const double* q;            /* [B, q_len, H, 576]: q_nope | q_pe, already decoded */
    const void* kv;             /* [num_pages, page_size, 576] bf16 bits or e4m3 bytes */
    int kv_fp8;
    double kv_scale;            /* applied only when kv_fp8 */
    const int32_t* block_table; /* [B, bt_stride] */
    int bt_stride;
    const int32_t* seq_lens;    /* [B] */
    double softmax_scale;
    const int32_t* reqs;        /* subset of requests to evaluate, or NULL = all */
    int n_reqs;
    /* split form only */
    int num_splits, chunk_tokens;
    double* part;               /* [rows, num_splits, 513] or NULL */
    /* token-range (sequence shard) form only */
    const int32_t* range_lo;    /* [B] first absolute position of the range */
    const int32_t* range_hi;    /* [B] one past the last */
    /* un-absorbed form only */
    const double* q_orig;       /* [B, q_len, H, 128] */
    const double* w_uk;         /* [H, 128, 512] */
    int qk_nope;
    /* outputs */
    double* out;                /* [B, q_len, H, 512] */
    double* lse;                /* [B, q_len, H] */
    int status;
} job_t;

/* One cached latent row x_t, decoded to double. */
static void load_row(const job_t* J, int b, int t, double* x) {
    int page = J->block_table[(int64_t)b * J->bt_stride + t / J->page_size];
    int64_t base = ((int64_t)page * J->page_size + (t % J->page_size)) * ROW;
    if (J->kv_fp8) {
        const uint8_t* p = (const uint8_t*)J->kv + base;
        for (int d = 0; d < ROW; ++d) x[d] = oracle_e4m3_to_double(p[d]) * J->kv_scale;
    } else {
        const uint16_t* p = (const uint16_t*)J->kv + base;
        for (int d = 0; d < ROW; ++d) x[d] = oracle_bf16_to_double(p[d]);
    }
}

/* Absorbed-form score of query row qrow (576 doubles) against token t. */
static double score_absorbed(const job_t* J, const double* qrow, const double* x) {
    double acc_nope = 0.0, acc_pe = 0.0;
    for (int d = 0; d < KV_LORA; ++d) acc_nope += qrow[d] * x[d];
    for (int d = 0; d < ROPE; ++d) acc_pe += qrow[KV_LORA + d] * x[KV_LORA + d];
    return J->softmax_scale * (acc_nope + acc_pe);
}

/* Un-absorbed (explicit MHA) score: K_h,t = W_UK,h . c_kv,t (qk_nope-d) | k_pe,t. */
static double score_unabsorbed(const job_t* J, int h, const double* qo, const double* qpe,
                               const double* x) {
    double acc_nope = 0.0, acc_pe = 0.0;
    const double* W = J->w_uk + (int64_t)h * J->qk_nope * KV_LORA;
    for (int e = 0; e < J->qk_nope; ++e) {
        double k = 0.0;
        for (int d = 0; d < KV_LORA; ++d) k += W[(int64_t)e * KV_LORA + d] * x[d];
        acc_nope += qo[e] * k;
    }
    for (int d = 0; d < ROPE; ++d) acc_pe += qpe[d] * x[KV_LORA + d];
    return J->softmax_scale * (acc_nope + acc_pe);
}

/* Softmax-weighted sum of c_kv over tokens [lo, hi) of request b for one row.
 * Writes o[512] and returns the LSE; an empty range gives o = 0, lse = -inf. */
static double attend_range(const job_t* J, int b, int i, int h, int lo, int hi,
                           double* s, double* x, double* o) {
    int64_t r = ((int64_t)b * J->q_len + i) * J->num_heads + h;
    for (int d = 0; d < KV_LORA; ++d) o[d] = 0.0;
    if (hi <= lo) return -INFINITY;
    for (int t = lo; t < hi; ++t) {
        load_row(J, b, t, x);
        if (J->w_uk)
            s[t - lo] = score_unabsorbed(J, h, J->q_orig + r * J->qk_nope, J->q + r * ROW + KV_LORA, x);
        else
            s[t - lo] = score_absorbed(J, J->q + r * ROW, x);
    }
    double m = -INFINITY;
    for (int t = lo; t < hi; ++t)
        if (s[t - lo] > m) m = s[t - lo];
    double Z = 0.0;
    for (int t = lo; t < hi; ++t) Z += exp(s[t - lo] - m);
    double l = m + log(Z);
    for (int t = lo; t < hi; ++t) {
        double w = exp(s[t - lo] - l);
        load_row(J, b, t, x);
        for (int d = 0; d < KV_LORA; ++d) o[d] += w * x[d];
    }
    return l;
}

/* Token-range form for a sequence-sharded (DCP) cache: row (b, i, h) attends
 * only to the absolute positions [range_lo[b], range_hi[b]) that it may see,
 * i.e. [range_lo[b], min(range_hi[b], V)).  Writes the range's normalised
 * output and LSE as one 513-entry partial (an empty range gives o = 0 and
 * lse = -inf), exactly what one shard contributes before the LSE merge. */
static void range_row(const job_t* J, int b, int i, int h, double* s, double* x, double* part) {
    int L = J->seq_lens[b];
    int V = L - J->q_len + 1 + i;
    int lo = J->range_lo[b];
    int hi = J->range_hi[b] < V ? J->range_hi[b] : V;
    part[KV_LORA] = attend_range(J, b, i, h, lo, hi, s, x, part);
}

typedef struct {
    job_t* J;
    int tid, nthreads;
} worker_t;

static void* worker(void* arg) {
    worker_t* W = (worker_t*)arg;
    job_t* J = W->J;
    int nreq = J->reqs ? J->n_reqs : J->batch;
    int max_L = 0;
    for (int k = 0; k < nreq; ++k) {
        int b = J->reqs ? J->reqs[k] : k;
        if (J->seq_lens[b] > max_L) max_L = J->seq_lens[b];
    }
    double* s = (double*)malloc(sizeof(double) * (size_t)(max_L > 0 ? max_L : 1));
    double* x = (double*)malloc(sizeof(double) * ROW);
    int64_t nrows = (int64_t)nreq * J->q_len * J->num_heads;
    for (int64_t k = W->tid; k < nrows; k += W->nthreads) {
        int h = (int)(k % J->num_heads);
        int i = (int)((k / J->num_heads) % J->q_len);
        int b = (int)(k / ((int64_t)J->num_heads * J->q_len));
        if (J->reqs) b = J->reqs[b];
        int64_t r = ((int64_t)b * J->q_len + i) * J->num_heads + h;
        int L = J->seq_lens[b];
        int V = L - J->q_len + 1 + i;
        if (J->range_lo) {
            range_row(J, b, i, h, s, x, J->part + r * (KV_LORA + 1));
            continue;
        }
        double* out = J->out + r * KV_LORA;
        if (J->num_splits <= 0) {
            J->lse[r] = attend_range(J, b, i, h, 0, V, s, x, out);
            continue;
        }
        /* Split form: every split j covers [j*c, min((j+1)*c, V)); each writes its
         * own normalised partial and LSE, then an LSE-weighted combine merges them. */
        double* part = J->part + r * (int64_t)J->num_splits * (KV_LORA + 1);
        for (int j = 0; j < J->num_splits; ++j) {
            int lo = j * J->chunk_tokens;
            int hi = (j + 1) * J->chunk_tokens;
            if (hi > V) hi = V;
            double* pj = part + (int64_t)j * (KV_LORA + 1);
            pj[KV_LORA] = attend_range(J, b, i, h, lo, hi, s, x, pj);
        }
        double M = -INFINITY;
        for (int j = 0; j < J->num_splits; ++j) {
            double lj = part[(int64_t)j * (KV_LORA + 1) + KV_LORA];
            if (lj > M) M = lj;
        }
        double acc = 0.0;
        for (int j = 0; j < J->num_splits; ++j)
            acc += exp(part[(int64_t)j * (KV_LORA + 1) + KV_LORA] - M);
        double l = M + log(acc);
        for (int d = 0; d < KV_LORA; ++d) out[d] = 0.0;
        for (int j = 0; j < J->num_splits; ++j) {
            const double* pj = part + (int64_t)j * (KV_LORA + 1);
            double w = exp(pj[KV_LORA] - l);
            for (int d = 0; d < KV_LORA; ++d) out[d] += w * pj[d];
        }
        J->lse[r] = l;
    }
    free(s);
    free(x);
    return NULL;
}

/* Checks the arguments every entry point shares; returns 0 when valid. */
static int validate(const job_t* J) {
    if (J->batch < 0 || J->num_heads <= 0 || J->q_len <= 0 || J->page_size <= 0) return 1;
    int nreq = J->reqs ? J->n_reqs : J->batch;
    for (int k = 0; k < nreq; ++k) {
        int b = J->reqs ? J->reqs[k] : k;
        if (b < 0 || b >= J->batch) return 2;
        int L = J->seq_lens[b];
        if (L < J->q_len) return 3;
        int pages = (L + J->page_size - 1) / J->page_size;
        if (pages > J->bt_stride) return 4;
        if (J->range_lo && (J->range_lo[b] < 0 || J->range_hi[b] < J->range_lo[b] || J->range_hi[b] > L))
            return 7;
    }
    return 0;
}

static int run(job_t* J, int num_threads) {
    int err = validate(J);
    if (err) return err;
    if (num_threads < 1) num_threads = 1;
    pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)num_threads);
    worker_t* ws = (worker_t*)malloc(sizeof(worker_t) * (size_t)num_threads);
    for (int k = 0; k < num_threads; ++k) {
        ws[k].J = J;
        ws[k].tid = k;
        ws[k].nthreads = num_threads;
        pthread_create(&th[k], NULL, worker, &ws[k]);
    }
    for (int k = 0; k < num_threads; ++k) pthread_join(th[k], NULL);
    free(th);
    free(ws);
    return 0;
}

/* Single-pass absorbed form. Returns 0 on success, >0 on invalid arguments. */
int oracle_mla_decode(int batch, int num_heads, int q_len, int page_size, const double* q,
                      const void* kv, int kv_fp8, double kv_scale, const int32_t* block_table,
                      int bt_stride, const int32_t* seq_lens, double softmax_scale,
                      const int32_t* reqs, int n_reqs, double* out, double* lse,
                      int num_threads) {
    job_t J;
    memset(&J, 0, sizeof J);
    J.batch = batch; J.num_heads = num_heads; J.q_len = q_len; J.page_size = page_size;
    J.q = q; J.kv = kv; J.kv_fp8 = kv_fp8; J.kv_scale = kv_scale;
    J.block_table = block_table; J.bt_stride = bt_stride; J.seq_lens = seq_lens;
    J.softmax_scale = softmax_scale; J.reqs = reqs; J.n_reqs = n_reqs;
    J.out = out; J.lse = lse;
    return run(&J, num_threads);
}

/* Split form: per-split partials [rows, num_splits, 513] (512 normalised outputs
 * then the split's LSE) followed by the LSE-weighted combine into out/lse. */
int oracle_mla_decode_split(int batch, int num_heads, int q_len, int page_size, const double* q,
                            const void* kv, int kv_fp8, double kv_scale,
                            const int32_t* block_table, int bt_stride, const int32_t* seq_lens,
                            double softmax_scale, int num_splits, int chunk_tokens, double* part,
                            double* out, double* lse, int num_threads) {
    if (num_splits <= 0 || chunk_tokens <= 0) return 5;
    job_t J;
    memset(&J, 0, sizeof J);
    J.batch = batch; J.num_heads = num_heads; J.q_len = q_len; J.page_size = page_size;
    J.q = q; J.kv = kv; J.kv_fp8 = kv_fp8; J.kv_scale = kv_scale;
    J.block_table = block_table; J.bt_stride = bt_stride; J.seq_lens = seq_lens;
    J.softmax_scale = softmax_scale;
    J.num_splits = num_splits; J.chunk_tokens = chunk_tokens; J.part = part;
    J.out = out; J.lse = lse;
    return run(&J, num_threads);
}

/* Un-absorbed MHA form: explicit keys K_h,t = W_UK,h c_kv,t (qk_nope-d) | k_pe,t,
 * queries q_orig (qk_nope-d) | q_pe, values V = c_kv.  q carries q_pe in its
 * last 64 entries (the first 512 are ignored here). */
int oracle_mla_decode_unabsorbed(int batch, int num_heads, int q_len, int page_size,
                                 const double* q_orig, int qk_nope, const double* w_uk,
                                 const double* q, const void* kv, int kv_fp8, double kv_scale,
                                 const int32_t* block_table, int bt_stride,
                                 const int32_t* seq_lens, double softmax_scale, double* out,
                                 double* lse, int num_threads) {
    if (qk_nope <= 0) return 6;
    job_t J;
    memset(&J, 0, sizeof J);
    J.batch = batch; J.num_heads = num_heads; J.q_len = q_len; J.page_size = page_size;
    J.q = q; J.kv = kv; J.kv_fp8 = kv_fp8; J.kv_scale = kv_scale;
    J.block_table = block_table; J.bt_stride = bt_stride; J.seq_lens = seq_lens;
    J.softmax_scale = softmax_scale;
    J.q_orig = q_orig; J.w_uk = w_uk; J.qk_nope = qk_nope;
    J.out = out; J.lse = lse;
    return run(&J, num_threads);
}

/* Token-range form (one sequence shard): part [rows, 513] per row (b, i, h),
 * the normalised output over the visible positions of [range_lo[b],
 * range_hi[b]) followed by that range's LSE. */
int oracle_mla_decode_range(int batch, int num_heads, int q_len, int page_size, const double* q,
                            const void* kv, int kv_fp8, double kv_scale,
                            const int32_t* block_table, int bt_stride, const int32_t* seq_lens,
                            double softmax_scale, const int32_t* range_lo, const int32_t* range_hi,
                            double* part, int num_threads) {
    if (!range_lo || !range_hi || !part) return 8;
    job_t J;
    memset(&J, 0, sizeof J);
    J.batch = batch; J.num_heads = num_heads; J.q_len = q_len; J.page_size = page_size;
    J.q = q; J.kv = kv; J.kv_fp8 = kv_fp8; J.kv_scale = kv_scale;
    J.block_table = block_table; J.bt_stride = bt_stride; J.seq_lens = seq_lens;
    J.softmax_scale = softmax_scale;
    J.range_lo = range_lo; J.range_hi = range_hi; J.part = part;
    return run(&J, num_threads);
}

/* LSE merge of R partials per row: parts [R, rows, 513] (shard-major, the
 * layout an all-gather of per-shard partials produces).  For every row:
 * M = max_s lse_s, lse = M + ln sum_s exp(lse_s - M),
 * out = sum_s exp(lse_s - lse) o_s; rows whose partials are all empty get
 * out = 0 and lse = -inf. */
void oracle_lse_merge(int64_t rows, int num_parts, const double* parts, double* out, double* lse) {
    for (int64_t r = 0; r < rows; ++r) {
        double M = -INFINITY;
        for (int k = 0; k < num_parts; ++k) {
            double lk = parts[((int64_t)k * rows + r) * (KV_LORA + 1) + KV_LORA];
            if (lk > M) M = lk;
        }
        double* o = out + r * KV_LORA;
        for (int d = 0; d < KV_LORA; ++d) o[d] = 0.0;
        if (M == -INFINITY) {
            lse[r] = -INFINITY;
            continue;
        }
        double acc = 0.0;
        for (int k = 0; k < num_parts; ++k)
            acc += exp(parts[((int64_t)k * rows + r) * (KV_LORA + 1) + KV_LORA] - M);
        double l = M + log(acc);
        for (int k = 0; k < num_parts; ++k) {
            const double* pk = parts + ((int64_t)k * rows + r) * (KV_LORA + 1);
            double w = exp(pk[KV_LORA] - l);
            for (int d = 0; d < KV_LORA; ++d) o[d] += w * pk[d];
        }
        lse[r] = l;
    }
}
