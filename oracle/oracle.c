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

typedef struct {
    const uint16_t *q;           /* [B, Hq, D] bf16 bits */
    const uint16_t *k;           /* [num_pages, P, Hkv, D] bf16 bits */
    const uint16_t *v;           /* same */
    const int32_t *block_table;  /* [B, max_pages] */
    const int32_t *seq_lens;     /* [B] */
    int B, Hq, Hkv, D, P, num_pages, max_pages;
    double scale;
    const int32_t *sel;          /* optional list of flattened b*Hq+h indices */
    int nsel;
    double *out;                 /* [B, Hq, D] or [nsel, D] when sel != NULL */
    double *lse;                 /* [B, Hq]    or [nsel]    when sel != NULL */
    int nthreads;
    int error;                   /* set to 1 when a used page id is out of range */
} decode_args;

typedef struct {
    decode_args *a;
    int tid;
} worker_arg;

/* One output row: the definition above, written out. */
static int decode_one(const decode_args *a, int b, int h, double *o, double *lse_out)
{
    const int G = a->Hq / a->Hkv;
    const int g = h / G;
    const int L = a->seq_lens[b];
    const int D = a->D;
    const uint16_t *qh = a->q + ((size_t)b * a->Hq + h) * D;

    if (L <= 0) {
        for (int d = 0; d < D; ++d) o[d] = 0.0;
        *lse_out = -INFINITY;
        return 0;
    }

    double *s = (double *)malloc(sizeof(double) * (size_t)L);
    const uint16_t **vrow = (const uint16_t **)malloc(sizeof(*vrow) * (size_t)L);
    if (!s || !vrow) { free(s); free(vrow); return 1; }

    for (int j = 0; j < L; ++j) {
        const int page = a->block_table[(size_t)b * a->max_pages + j / a->P];
        const int slot = j % a->P;
        if (page < 0 || page >= a->num_pages) { free(s); free(vrow); return 1; }
        const size_t row = (((size_t)page * a->P + slot) * a->Hkv + g) * D;
        const uint16_t *kj = a->k + row;
        double dot = 0.0;
        for (int d = 0; d < D; ++d)
            dot += bf16_bits_to_double(qh[d]) * bf16_bits_to_double(kj[d]);
        s[j] = a->scale * dot;
        vrow[j] = a->v + row;
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
            acc += s[j] * bf16_bits_to_double(vrow[j][d]);
        o[d] = acc / Z;
    }
    *lse_out = M + log(Z);

    free(s);
    free(vrow);
    return 0;
}

static void *decode_worker(void *p)
{
    worker_arg *w = (worker_arg *)p;
    decode_args *a = w->a;
    const int n = a->sel ? a->nsel : a->B * a->Hq;
    for (int i = w->tid; i < n; i += a->nthreads) {
        const int flat = a->sel ? a->sel[i] : i;
        const int b = flat / a->Hq, h = flat % a->Hq;
        if (decode_one(a, b, h, a->out + (size_t)i * a->D, a->lse + i))
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
    if (B < 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || P <= 0 || Hq % Hkv != 0)
        return 2;
    for (int b = 0; b < B; ++b)
        if (seq_lens[b] > (long)max_pages * P) return 2;

    decode_args a;
    memset(&a, 0, sizeof a);
    a.q = q; a.k = k; a.v = v; a.block_table = block_table; a.seq_lens = seq_lens;
    a.B = B; a.Hq = Hq; a.Hkv = Hkv; a.D = D; a.P = P;
    a.num_pages = num_pages; a.max_pages = max_pages; a.scale = scale;
    a.sel = sel; a.nsel = nsel; a.out = out; a.lse = lse;
    a.nthreads = resolve_threads(nthreads);

    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)a.nthreads);
    worker_arg *wa = (worker_arg *)malloc(sizeof(worker_arg) * (size_t)a.nthreads);
    if (!th || !wa) { free(th); free(wa); return 2; }
    for (int t = 0; t < a.nthreads; ++t) {
        wa[t].a = &a;
        wa[t].tid = t;
        pthread_create(&th[t], NULL, decode_worker, &wa[t]);
    }
    for (int t = 0; t < a.nthreads; ++t) pthread_join(th[t], NULL);
    free(th);
    free(wa);
    return a.error ? 1 : 0;
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
