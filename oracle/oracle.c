/*
 * oracle.c -- plain, slow, fp64 CPU reference for paged GQA decode attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, includes or
 * calls this file; only the tests, the smoke check and the benchmark's CPU
 * baseline leg do.  It shares no code, header, table or helper with the CUDA
 * path.
 *
 * What it computes (the plain definition; the split-KV method reaches the same
 * result up to floating-point rounding order):
 *
 *   for every sequence b and query head h:
 *     g   = floor(h / (Hq / Hkv))                  contiguous GQA groups
 *     for j in 0 .. L_b-1:
 *       page = block_table[b][j / P],  slot = j mod P
 *       k_j  = K[page, slot, g, :],   v_j = V[page, slot, g, :]   (bf16 -> double, exact)
 *       s_j  = scale * sum_d q[b,h,d] * k_j[d]                     (double)
 *     M   = max_j s_j
 *     Z   = sum_j exp(s_j - M)
 *     out = sum_j exp(s_j - M) * v_j / Z
 *     lse = M + ln Z                                               (natural log)
 *   L_b == 0  ->  out = 0, lse = -inf.
 *
 * Passages followed:
 *   - FlashQuant wiki "CUDA Kernels", flash_attention.cu, "GQA (Grouped Query
 *     Attention) Support": a query head maps to kv head h / (H_Q / H_KV).
 *   - same page, paged_decode.cu, "Page Table Addressing": the logical block
 *     is kv_pos / block_size, the slot kv_pos mod block_size, the physical
 *     block block_table[logical block].
 *   - same page, "Online Softmax": the online recurrence reaches exactly the
 *     softmax above; the oracle writes the softmax out directly instead.
 *   - same page, split_k_reduce.cu, "Algorithm": the merge of per-split
 *     partial states (oracle_merge below), restated for normalised partial
 *     outputs and natural-log LSEs.
 *
 * Readings where the pages are silent: the returned LSE is a natural log;
 * scale is applied to q.k exactly as passed (widened to double); L_b == 0 gives
 * out = 0 and lse = -inf; slots past L_b and table entries past the used pages
 * are never read.
 *
 * Multi-token rows (AstrAI "CUDA Kernels", "Q Scheduling and KV Addressing":
 * a packed [total_q, Hq, D] query tensor with qo_indptr): request b owns query
 * rows qo_indptr[b] .. qo_indptr[b+1]-1, n_b of them, and L_b keys.  Reading:
 * the new tokens are the last n_b positions of the request, so under the causal
 * mask query row i (0-based within the request) sees keys j <= L_b - n_b + i,
 * and without the mask all L_b keys; a row that sees no key gives 0 and -inf.
 * Decode is the case n_b = 1, qo_indptr[b] = b.
 *
 * FP8 KV variant (OASR "Kernel Layer", "FP8 KV variants"): the cache may hold
 * float8 e4m3 codes with one f32 scale per (token, kv head); the key/value used
 * is then code value * scale, exact in double.  The codec (e4m3_value,
 * oracle_e4m3_encode) is written from the format's definition, and the
 * quantiser (oracle_fp8_quantize_rows) picks a power-of-two scale per row.
 *
 * Parallelism: (b, h) outputs are independent; worker threads take them by a
 * fixed stride, so results do not depend on the thread count.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

static double bf16_bits_to_double(uint16_t bits)
{
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/*
 * float8 e4m3, the "fn" variant the pages name (float8_e4m3fn): bit 7 sign,
 * bits 6..3 exponent E with bias 7, bits 2..0 mantissa M, no infinities.
 *   E == 0:            (M / 8) * 2^-6            (subnormal; M == 0 is +-0)
 *   E == 15 && M == 7: NaN
 *   otherwise:         (1 + M / 8) * 2^(E - 7)   (largest finite: 448)
 */
static double e4m3_value(uint8_t code)
{
    const int neg = code >> 7, E = (code >> 3) & 15, M = code & 7;
    if (E == 15 && M == 7) return NAN;
    const double mag = E == 0 ? ldexp((double)M, -9) : ldexp(1.0 + M / 8.0, E - 7);
    return neg ? -mag : mag;
}

double oracle_e4m3_value(uint8_t code) { return e4m3_value(code); }

/*
 * Round to the nearest finite e4m3 value, ties to the even code (the one whose
 * mantissa's last bit is 0), saturating at +-448; NaN gives the NaN code 0x7F.
 * The non-negative finite codes 0x00..0x7E are in increasing order of value,
 * so the neighbours of |x| are found by bisection over the codes.
 */
uint8_t oracle_e4m3_encode(double x)
{
    if (isnan(x)) return 0x7F;
    const uint8_t sign = signbit(x) ? 0x80 : 0x00;
    const double ax = fabs(x);
    int code;
    if (ax >= 448.0) {
        code = 0x7E;
    } else {
        int lo = 0, hi = 0x7E;  /* value(lo) <= ax < value(hi) */
        while (hi - lo > 1) {
            const int mid = (lo + hi) / 2;
            if (e4m3_value((uint8_t)mid) <= ax) lo = mid; else hi = mid;
        }
        const double dlo = ax - e4m3_value((uint8_t)lo), dhi = e4m3_value((uint8_t)hi) - ax;
        if (dlo < dhi) code = lo;
        else if (dhi < dlo) code = hi;
        else code = (lo % 2 == 0) ? lo : hi;
    }
    return (uint8_t)(sign | code);
}

/*
 * Quantise N rows of D bf16 values (one row = one token of one kv head): the
 * row's scale is s = 2^k with k the smallest integer in [-64, 64] such that
 * max_d |x_d| <= 448 * 2^k (NaN values are left out of the maximum), and code_d
 * = encode(x_d / s).  A power of two makes x / s exact and code * s exactly
 * representable in bf16 (OASR "Kernel Layer", "FP8 KV variants": power-of-two
 * scales make the dequantised product exact).  Reading: the pages fix the
 * scale to a power of two but not which one; this is the smallest that does not
 * saturate the row, and the exponent clamp keeps every dequantised value an
 * exact bf16 normal.  An all-zero row gets 2^-64.
 */
void oracle_fp8_quantize_rows(const uint16_t *x, int N, int D, uint8_t *codes, float *scales)
{
    for (int n = 0; n < N; ++n) {
        const uint16_t *row = x + (size_t)n * D;
        double amax = 0.0;
        for (int d = 0; d < D; ++d) {
            const double a = fabs(bf16_bits_to_double(row[d]));
            if (a > amax) amax = a;  /* NaN compares false and is skipped */
        }
        int k = -64;
        while (k < 64 && amax > ldexp(448.0, k)) ++k;
        const double s = ldexp(1.0, k);
        scales[n] = (float)s;
        for (int d = 0; d < D; ++d)
            codes[(size_t)n * D + d] = oracle_e4m3_encode(bf16_bits_to_double(row[d]) / s);
    }
}

typedef struct {
    const uint16_t *q;           /* [B, Hq, D] bf16 bits */
    const uint16_t *k;           /* [num_pages, P, Hkv, D] bf16 bits (bf16 cache) */
    const uint16_t *v;           /* same */
    const uint8_t *k8;           /* [num_pages, P, Hkv, D] e4m3 codes (fp8 cache), else NULL */
    const uint8_t *v8;           /* same */
    const float *k_scale;        /* [num_pages, Hkv, P] f32 per (token, kv head) (fp8 cache) */
    const float *v_scale;        /* same */
    const int32_t *block_table;  /* [B, max_pages] */
    const int32_t *seq_lens;     /* [B] */
    const int32_t *qo_indptr;    /* [B+1] query rows per request, or NULL: one row per request */
    int total_q;                 /* query rows (B when qo_indptr is NULL) */
    int causal;                  /* 1: row i of a request sees keys j <= L - n + i */
    int B, Hq, Hkv, D, P, num_pages, max_pages;
    double scale;
    const int32_t *sel;          /* optional list of flattened row*Hq+h indices */
    int nsel;
    double *out;                 /* [total_q, Hq, D] or [nsel, D] when sel != NULL */
    double *lse;                 /* [total_q, Hq]    or [nsel]    when sel != NULL */
    int nthreads;
    int error;                   /* set to 1 when a used page id is out of range */
} decode_args;

typedef struct {
    decode_args *a;
    int tid;
} worker_arg;

/* Element d of the key (is_v == 0) or value (is_v == 1) of slot `slot` in page
 * `page`, kv head g, as an exact double: a bf16 value, or code value * scale. */
static double kv_elem(const decode_args *a, int is_v, int page, int slot, int g, int d)
{
    const size_t off = (((size_t)page * a->P + slot) * a->Hkv + g) * a->D + d;
    if (!a->k8) return bf16_bits_to_double((is_v ? a->v : a->k)[off]);
    const uint8_t code = (is_v ? a->v8 : a->k8)[off];
    const float s = (is_v ? a->v_scale : a->k_scale)[((size_t)page * a->Hkv + g) * a->P + slot];
    return e4m3_value(code) * (double)s;
}

/* The request that owns query row t (a linear scan of qo_indptr). */
static int request_of(const decode_args *a, int t)
{
    if (!a->qo_indptr) return t;
    for (int b = 0; b < a->B; ++b)
        if (t >= a->qo_indptr[b] && t < a->qo_indptr[b + 1]) return b;
    return -1;
}

/* One output row (query row t, head h): the definition above, written out. */
static int decode_one(const decode_args *a, int t, int h, double *o, double *lse_out)
{
    const int G = a->Hq / a->Hkv;
    const int g = h / G;
    const int b = request_of(a, t);
    const int D = a->D;
    const uint16_t *qh = a->q + ((size_t)t * a->Hq + h) * D;
    if (b < 0) return 1;
    int L = a->seq_lens[b];
    if (a->qo_indptr && a->causal) {
        const int n = a->qo_indptr[b + 1] - a->qo_indptr[b];
        const int i = t - a->qo_indptr[b];
        if (L - n + i + 1 < L) L = L - n + i + 1;  /* keys j <= L - n + i */
    }

    if (L <= 0) {
        for (int d = 0; d < D; ++d) o[d] = 0.0;
        *lse_out = -INFINITY;
        return 0;
    }

    double *s = (double *)malloc(sizeof(double) * (size_t)L);
    int *jpage = (int *)malloc(sizeof(int) * (size_t)L);
    if (!s || !jpage) { free(s); free(jpage); return 1; }

    for (int j = 0; j < L; ++j) {
        const int page = a->block_table[(size_t)b * a->max_pages + j / a->P];
        const int slot = j % a->P;
        if (page < 0 || page >= a->num_pages) { free(s); free(jpage); return 1; }
        double dot = 0.0;
        for (int d = 0; d < D; ++d)
            dot += bf16_bits_to_double(qh[d]) * kv_elem(a, 0, page, slot, g, d);
        s[j] = a->scale * dot;
        jpage[j] = page;
    }

    double M = s[0];
    for (int j = 1; j < L; ++j)
        if (s[j] > M) M = s[j];

    double Z = 0.0;
    for (int j = 0; j < L; ++j) {
        s[j] = exp(s[j] - M);     /* s now holds the unnormalised weights */
        Z += s[j];
    }
    for (int d = 0; d < D; ++d) {
        double acc = 0.0;
        for (int j = 0; j < L; ++j)
            acc += s[j] * kv_elem(a, 1, jpage[j], j % a->P, g, d);
        o[d] = acc / Z;
    }
    *lse_out = M + log(Z);

    free(s);
    free(jpage);
    return 0;
}

static void *decode_worker(void *p)
{
    worker_arg *w = (worker_arg *)p;
    decode_args *a = w->a;
    const int n = a->sel ? a->nsel : a->total_q * a->Hq;
    for (int i = w->tid; i < n; i += a->nthreads) {
        const int flat = a->sel ? a->sel[i] : i;
        const int t = flat / a->Hq, h = flat % a->Hq;
        if (decode_one(a, t, h, a->out + (size_t)i * a->D, a->lse + i))
            a->error = 1;  /* benign race: any writer stores 1 */
    }
    return NULL;
}

static int resolve_threads(int nthreads)
{
    if (nthreads > 0) return nthreads;
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n > 0 ? (int)n : 1;
}

static int run_decode(decode_args *a, int nthreads)
{
    if (a->B < 0 || a->Hq <= 0 || a->Hkv <= 0 || a->D <= 0 || a->P <= 0 || a->Hq % a->Hkv != 0)
        return 2;
    for (int b = 0; b < a->B; ++b)
        if (a->seq_lens[b] > (long)a->max_pages * a->P) return 2;
    if (!a->qo_indptr) {
        a->total_q = a->B;
    } else {
        if (a->qo_indptr[0] != 0 || a->qo_indptr[a->B] != a->total_q) return 2;
        for (int b = 0; b < a->B; ++b)
            if (a->qo_indptr[b + 1] < a->qo_indptr[b]) return 2;
    }
    a->nthreads = resolve_threads(nthreads);

    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)a->nthreads);
    worker_arg *wa = (worker_arg *)malloc(sizeof(worker_arg) * (size_t)a->nthreads);
    if (!th || !wa) { free(th); free(wa); return 2; }
    for (int t = 0; t < a->nthreads; ++t) {
        wa[t].a = a;
        wa[t].tid = t;
        pthread_create(&th[t], NULL, decode_worker, &wa[t]);
    }
    for (int t = 0; t < a->nthreads; ++t) pthread_join(th[t], NULL);
    free(th);
    free(wa);
    return a->error ? 1 : 0;
}

/*
 * oracle_paged_decode: returns 0 on success, 1 if a used block_table entry is
 * outside [0, num_pages), 2 on bad arguments.  `sel` (may be NULL) restricts
 * the computation to the listed flattened (b*Hq + h) rows; outputs are then
 * packed in list order.  nthreads <= 0 means one thread per online core.
 */
int oracle_paged_decode(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                        const int32_t *block_table, const int32_t *seq_lens,
                        int B, int Hq, int Hkv, int D, int P, int num_pages,
                        int max_pages, double scale, const int32_t *sel, int nsel,
                        double *out, double *lse, int nthreads)
{
    decode_args a;
    memset(&a, 0, sizeof a);
    a.q = q; a.k = k; a.v = v; a.block_table = block_table; a.seq_lens = seq_lens;
    a.B = B; a.Hq = Hq; a.Hkv = Hkv; a.D = D; a.P = P;
    a.num_pages = num_pages; a.max_pages = max_pages; a.scale = scale;
    a.sel = sel; a.nsel = nsel; a.out = out; a.lse = lse;
    return run_decode(&a, nthreads);
}

/*
 * oracle_paged_decode_fp8: the same definition over an fp8 cache.  k8, v8 are
 * e4m3 codes [num_pages, P, Hkv, D]; k_scale, v_scale are f32 [num_pages, Hkv, P];
 * key/value element = code value * scale.  Return codes as above.
 */
int oracle_paged_decode_fp8(const uint16_t *q, const uint8_t *k8, const uint8_t *v8,
                            const float *k_scale, const float *v_scale,
                            const int32_t *block_table, const int32_t *seq_lens,
                            int B, int Hq, int Hkv, int D, int P, int num_pages,
                            int max_pages, double scale, const int32_t *sel, int nsel,
                            double *out, double *lse, int nthreads)
{
    decode_args a;
    memset(&a, 0, sizeof a);
    a.q = q; a.k8 = k8; a.v8 = v8; a.k_scale = k_scale; a.v_scale = v_scale;
    a.block_table = block_table; a.seq_lens = seq_lens;
    a.B = B; a.Hq = Hq; a.Hkv = Hkv; a.D = D; a.P = P;
    a.num_pages = num_pages; a.max_pages = max_pages; a.scale = scale;
    a.sel = sel; a.nsel = nsel; a.out = out; a.lse = lse;
    return run_decode(&a, nthreads);
}

/*
 * oracle_paged_prefill: several query rows per request (see the header), over a
 * bf16 cache (k, v non-NULL) or an fp8 one (k8, v8, k_scale, v_scale non-NULL).
 *   q [total_q, Hq, D] bf16 bits; qo_indptr [B+1] with qo_indptr[0] = 0 and
 *   qo_indptr[B] = total_q; out [total_q, Hq, D], lse [total_q, Hq] (or the
 *   selected rows, flattened t*Hq + h).  Return codes as oracle_paged_decode.
 */
int oracle_paged_prefill(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                         const uint8_t *k8, const uint8_t *v8, const float *k_scale, const float *v_scale,
                         const int32_t *qo_indptr, const int32_t *block_table, const int32_t *seq_lens,
                         int B, int Hq, int Hkv, int D, int P, int num_pages, int max_pages, int total_q,
                         double scale, int causal, const int32_t *sel, int nsel,
                         double *out, double *lse, int nthreads)
{
    decode_args a;
    memset(&a, 0, sizeof a);
    a.q = q; a.k = k; a.v = v; a.k8 = k8; a.v8 = v8; a.k_scale = k_scale; a.v_scale = v_scale;
    a.qo_indptr = qo_indptr; a.total_q = total_q; a.causal = causal;
    a.block_table = block_table; a.seq_lens = seq_lens;
    a.B = B; a.Hq = Hq; a.Hkv = Hkv; a.D = D; a.P = P;
    a.num_pages = num_pages; a.max_pages = max_pages; a.scale = scale;
    a.sel = sel; a.nsel = nsel; a.out = out; a.lse = lse;
    if (!qo_indptr) return 2;
    return run_decode(&a, nthreads);
}

/*
 * oracle_merge: combine S per-split partial states of N rows.
 *   partial_out [S, N, D]: each split's softmax-normalised output over its keys
 *   partial_lse [S, N]   : each split's natural-log LSE; -inf marks an empty split
 * For each row:  M = max_s lse_s;  w_s = exp(lse_s - M);  W = sum_s w_s;
 *                out = sum_s w_s * o_s / W;  lse = M + ln W.
 * All splits empty -> out = 0, lse = -inf.
 * (FlashQuant wiki "CUDA Kernels", split_k_reduce.cu, "Algorithm" and
 *  "Numerical Stability": global max, rescaled weights, weighted combination,
 *  guarded normaliser.  Their weight l_s * exp2(m_s - m_final) equals
 *  exp(lse_s - M) once lse_s = ln l_s + m_s ln 2 and M is the natural-log max.)
 */
void oracle_merge(const double *partial_out, const double *partial_lse,
                  int S, int N, int D, double *out, double *lse)
{
    for (int n = 0; n < N; ++n) {
        double M = -INFINITY;
        for (int s = 0; s < S; ++s)
            if (partial_lse[(size_t)s * N + n] > M) M = partial_lse[(size_t)s * N + n];
        double *o = out + (size_t)n * D;
        if (M == -INFINITY) {
            for (int d = 0; d < D; ++d) o[d] = 0.0;
            lse[n] = -INFINITY;
            continue;
        }
        double W = 0.0;
        for (int s = 0; s < S; ++s)
            W += exp(partial_lse[(size_t)s * N + n] - M);
        for (int d = 0; d < D; ++d) {
            double acc = 0.0;
            for (int s = 0; s < S; ++s)
                acc += exp(partial_lse[(size_t)s * N + n] - M) *
                       partial_out[((size_t)s * N + n) * D + d];
            o[d] = acc / W;
        }
        lse[n] = M + log(W);
    }
}

/*
 * oracle_kv_append: write one new key row and value row per (sequence, kv head)
 * into the page pool, at logical key position positions[b]: physical page
 * block_table[b][positions[b] / P], slot positions[b] mod P (the page-table
 * addressing of FlashQuant wiki "CUDA Kernels", paged_decode.cu "Page Table
 * Addressing"; the per-token cache write of Atlas "CUDA Kernel Engineering",
 * "The kernel inventory", KV append).
 *   k_new, v_new [B, Hkv, D] bf16 bits; k_cache, v_cache [num_pages, P, Hkv, D] (updated in place)
 * positions[b] < 0 skips sequence b.  Returns the number of sequences skipped because
 * the position is past max_pages*P or the page id is outside [0, num_pages); their
 * rows are not written.
 */
int oracle_kv_append(const uint16_t *k_new, const uint16_t *v_new, const int32_t *block_table,
                     const int32_t *positions, int B, int Hkv, int D, int P, int num_pages, int max_pages,
                     uint16_t *k_cache, uint16_t *v_cache)
{
    int rejected = 0;
    for (int b = 0; b < B; ++b) {
        const int pos = positions[b];
        if (pos < 0) continue;
        if (pos >= max_pages * P) { ++rejected; continue; }
        const int page = block_table[(size_t)b * max_pages + pos / P];
        if (page < 0 || page >= num_pages) { ++rejected; continue; }
        const int slot = pos % P;
        for (int g = 0; g < Hkv; ++g) {
            const size_t dst = (((size_t)page * P + slot) * Hkv + g) * D;
            const size_t src = ((size_t)b * Hkv + g) * D;
            memcpy(k_cache + dst, k_new + src, sizeof(uint16_t) * (size_t)D);
            memcpy(v_cache + dst, v_new + src, sizeof(uint16_t) * (size_t)D);
        }
    }
    return rejected;
}

/*
 * oracle_kv_append_fp8: the append above into an fp8 cache, quantising on the
 * way (OASR "Kernel Layer", "FP8 KV variants": one quantise-and-scatter launch
 * writes K and V).  Each new (sequence, kv head) row is quantised by
 * oracle_fp8_quantize_rows; its codes go to k8/v8 [num_pages, P, Hkv, D] and its
 * scale to k_scale/v_scale [num_pages, Hkv, P].  Skip and reject rules and the
 * return value are those of oracle_kv_append.
 */
int oracle_kv_append_fp8(const uint16_t *k_new, const uint16_t *v_new, const int32_t *block_table,
                         const int32_t *positions, int B, int Hkv, int D, int P, int num_pages, int max_pages,
                         uint8_t *k8, uint8_t *v8, float *k_scale, float *v_scale)
{
    int rejected = 0;
    for (int b = 0; b < B; ++b) {
        const int pos = positions[b];
        if (pos < 0) continue;
        if (pos >= max_pages * P) { ++rejected; continue; }
        const int page = block_table[(size_t)b * max_pages + pos / P];
        if (page < 0 || page >= num_pages) { ++rejected; continue; }
        const int slot = pos % P;
        for (int g = 0; g < Hkv; ++g) {
            const size_t dst = (((size_t)page * P + slot) * Hkv + g) * D;
            const size_t src = ((size_t)b * Hkv + g) * D;
            const size_t sdst = ((size_t)page * Hkv + g) * P + slot;
            oracle_fp8_quantize_rows(k_new + src, 1, D, k8 + dst, k_scale + sdst);
            oracle_fp8_quantize_rows(v_new + src, 1, D, v8 + dst, v_scale + sdst);
        }
    }
    return rejected;
}
