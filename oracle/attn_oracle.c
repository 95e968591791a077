/*
 * attn_oracle.c — plain fp64 CPU oracle for the attention forward pass.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the product path may link, load or call this file;
 * only the tests, the package smoke check and the benchmark's CPU-baseline leg use it. It
 * shares no code, header, table or helper with the CUDA library.
 *
 * What it computes (written straight from the definition, no tiling, no online update):
 *   For batch/segment/sequence b, query head h and query row i, with g = h / (Hq / Hkv)
 *   (contiguous GQA groups) and V(i) the keys the mask makes visible to row i:
 *     z_j  = s * sum_c q[b,h,i,c] * k[b,g,j,c]      for j in V(i)  (scores materialised)
 *     M    = max_j z_j
 *     l    = sum_j exp(z_j - M)
 *     O[i] = sum_j exp(z_j - M) * v[b,g,j,:] / l
 *     LSE  = M + ln(l)
 *   Softmax with the max subtracted is the one stated in "Flash MSA Attention Kernel
 *   Implementation Tutorial", section "Understanding Flash MSA Core Mechanics"; the scale s
 *   multiplies the raw dot products as in that page's kernel listing. The oracle takes two
 *   passes over the materialised row (max, then exponent sum) rather than the page's running
 *   update, which reaches the same function.
 *
 * Visible sets (readings of the pages fixed for this build):
 *   NONE       all j < N
 *   CAUSAL     j <= i
 *   SLIDING    i - W < j <= i   (causal, W keys including the query itself; the two-sided
 *              wording of "Optimizing Triton Kernels for Custom Attention Patterns on H100",
 *              Pattern B, is read as this causal window)
 *   DOCUMENT   cu[s] <= j <= i where cu[s] <= i < cu[s+1] (causal inside the query's own
 *              segment; the segment-offset mask of the same page, Pattern A)
 *   PAGED      all j < L_b, key/value j of sequence b read from physical page
 *              table[b][j / page] at slot j % page (the block-table indirection of Pattern C)
 *   DECODE     all j < L_b, key/value j of sequence b read from a dense per-sequence cache
 *              k[b, g, j, :] (the plain attention kernel run on the gathered pages, the
 *              second stage of Pattern C's two-stage path)
 *   SLIDING_BIDIR  i - W <= j <= i + W (Pattern B's plus-or-minus-W neighbourhood taken literally:
 *              W keys on each side of the query plus the query, clipped to [0, N))
 *   DOCUMENT_BIDIR cu[s] <= j < cu[s+1] where cu[s] <= i < cu[s+1] (Pattern A's kernel as
 *              printed: every key of the query's own segment, none outside it)
 *   PREFIX_LM  j <= i or j < P, P = the prefix length passed as the window argument (the
 *              prefix-LM mask the same page lists among masks with exploitable structure:
 *              the first P tokens see each other in both directions, later tokens see
 *              every earlier token)
 *   PAGED_PREFILL  a chunk of Lq_b new query tokens of sequence b whose context (the chunk
 *              included) holds Lk_b >= Lq_b keys in a paged cache: query t of the chunk sits
 *              at position Lk_b - Lq_b + t and sees keys j <= that position, read through
 *              the block table as for PAGED (Pattern C's prefix-caching use of a block
 *              table, with the query block longer than one token). Queries are packed like
 *              DOCUMENT: cu[] holds the chunks' starts, seqlens_k[] the context lengths.
 *
 * Inputs are raw bf16 bit patterns widened exactly to fp64. The fp32 scale is widened too.
 * A row that sees no key (impossible for valid inputs) gets O = 0 and LSE = -inf.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { OR_NONE = 0, OR_CAUSAL = 1, OR_SLIDING = 2, OR_DOCUMENT = 3, OR_PAGED = 4, OR_DECODE = 5,
       OR_SLIDING_BIDIR = 6, OR_DOCUMENT_BIDIR = 7, OR_PREFIX_LM = 8, OR_PAGED_PREFILL = 9 };

/* One query per sequence (PAGED, DECODE). */
static int is_decode(int mask) { return mask == OR_PAGED || mask == OR_DECODE; }

/* Packed query rows described by cu_seqlens (DOCUMENT, DOCUMENT_BIDIR, PAGED_PREFILL). */
static int is_document(int mask) {
    return mask == OR_DOCUMENT || mask == OR_DOCUMENT_BIDIR || mask == OR_PAGED_PREFILL;
}

/* Keys read through a block table. */
static int is_paged(int mask) { return mask == OR_PAGED || mask == OR_PAGED_PREFILL; }

typedef struct {
    const uint16_t *q, *k, *v;
    const double *qd, *kd;  /* when set, Q and K are these fp64 values instead of q / k */
    int B, Hq, Hkv, N, d;
    double s;
    int mask, W;
    const int32_t *cu;
    const int32_t *seqlens_k;
    const int32_t *table;
    int max_pages, page;
} problem_t;

static double widen_bf16(uint16_t bits) {
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Number of query rows, in the flattened order of the O / LSE outputs. */
static int64_t row_count(const problem_t *P) {
    if (is_decode(P->mask)) return (int64_t)P->B * P->Hq;
    if (is_document(P->mask)) return (int64_t)P->Hq * P->N;
    return (int64_t)P->B * P->Hq * P->N;
}

/* Flattened row r -> (b, h, i). For DOCUMENT, b is the segment that holds token i. */
static void row_coords(const problem_t *P, int64_t r, int *b, int *h, int *i) {
    if (is_decode(P->mask)) {
        *b = (int)(r / P->Hq);
        *h = (int)(r % P->Hq);
        *i = 0;
    } else if (is_document(P->mask)) {
        *h = (int)(r / P->N);
        *i = (int)(r % P->N);
        int s = 0;
        while (s + 1 < P->B && P->cu[s + 1] <= *i) s++;
        *b = s;
    } else {
        *b = (int)(r / ((int64_t)P->Hq * P->N));
        *h = (int)((r / P->N) % P->Hq);
        *i = (int)(r % P->N);
    }
}

/* Number of keys row i of batch b can address (before the mask). */
static int key_count(const problem_t *P, int b) {
    if (is_decode(P->mask)) return P->cu[b + 1] - P->cu[b];
    if (P->mask == OR_PAGED_PREFILL) return P->seqlens_k[b];
    return P->N;
}

static int visible(const problem_t *P, int b, int i, int j) {
    switch (P->mask) {
    case OR_NONE: return 1;
    case OR_CAUSAL: return j <= i;
    case OR_SLIDING: return j <= i && j > i - P->W;
    case OR_DOCUMENT: return j <= i && j >= P->cu[b];
    case OR_PAGED:
    case OR_DECODE: return j < P->cu[b + 1] - P->cu[b];
    case OR_SLIDING_BIDIR: return (int64_t)j >= (int64_t)i - P->W && (int64_t)j <= (int64_t)i + P->W;
    case OR_DOCUMENT_BIDIR: return j >= P->cu[b] && j < P->cu[b + 1];
    case OR_PREFIX_LM: return j <= i || j < P->W;
    case OR_PAGED_PREFILL: {
        const int Lq = P->cu[b + 1] - P->cu[b], Lk = P->seqlens_k[b];
        return j < Lk && j <= (i - P->cu[b]) + (Lk - Lq);
    }
    }
    return 0;
}

/* Element offset of query row (b, h, i). */
static size_t query_row(const problem_t *P, int b, int h, int i) {
    if (is_decode(P->mask)) return ((size_t)b * P->Hq + h) * P->d;
    if (is_document(P->mask)) return ((size_t)h * P->N + i) * P->d;
    return (((size_t)b * P->Hq + h) * P->N + i) * P->d;
}

/* Element offset of key / value row j of (b, g) (k and v share the layout). */
static size_t kv_row(const problem_t *P, int b, int g, int j) {
    if (is_paged(P->mask)) {
        int phys = P->table[(size_t)b * P->max_pages + j / P->page];
        return ((((size_t)phys * P->Hkv + g) * P->page) + (size_t)(j % P->page)) * P->d;
    }
    if (is_document(P->mask)) return ((size_t)g * P->N + j) * P->d;
    return (((size_t)b * P->Hkv + g) * P->N + j) * P->d;
}

static double q_at(const problem_t *P, size_t off) {
    return P->qd ? P->qd[off] : widen_bf16(P->q[off]);
}

static double k_at(const problem_t *P, size_t off) {
    return P->kd ? P->kd[off] : widen_bf16(P->k[off]);
}

/* One query row from the definition. z is scratch of key_count() doubles; probs (optional)
 * receives exp(z_j - M) / l for every addressable key (0 where not visible). */
static void attend_row(const problem_t *P, int64_t r, double *z, double *o, double *lse,
                       double *probs) {
    int b, h, i;
    row_coords(P, r, &b, &h, &i);
    const int g = h / (P->Hq / P->Hkv);
    const int nk = key_count(P, b);
    const size_t qr = query_row(P, b, h, i);

    double M = -INFINITY;
    int any = 0;
    for (int j = 0; j < nk; j++) {
        if (!visible(P, b, i, j)) continue;
        const size_t kr = kv_row(P, b, g, j);
        double dot = 0.0;
        for (int c = 0; c < P->d; c++) dot += q_at(P, qr + c) * k_at(P, kr + c);
        z[j] = P->s * dot;
        if (z[j] > M) M = z[j];
        any = 1;
    }
    for (int c = 0; c < P->d; c++) o[c] = 0.0;
    if (!any) {
        *lse = -INFINITY;
        if (probs)
            for (int j = 0; j < nk; j++) probs[j] = 0.0;
        return;
    }
    double l = 0.0;
    for (int j = 0; j < nk; j++)
        if (visible(P, b, i, j)) l += exp(z[j] - M);
    for (int j = 0; j < nk; j++) {
        if (!visible(P, b, i, j)) {
            if (probs) probs[j] = 0.0;
            continue;
        }
        const double e = exp(z[j] - M);
        const uint16_t *vr = P->v + kv_row(P, b, g, j);
        for (int c = 0; c < P->d; c++) o[c] += e * widen_bf16(vr[c]);
        if (probs) probs[j] = e / l;
    }
    for (int c = 0; c < P->d; c++) o[c] /= l;
    *lse = M + log(l);
}

/*
 * Compute O and LSE for the given rows (rows == NULL: every row, in output order).
 * o: nrows x d doubles; lse: nrows doubles; probs (optional): nrows x probs_stride doubles.
 * Returns 0, or -1 for arguments the definition does not cover.
 */
static int oracle_run(const uint16_t *q, const uint16_t *k, const double *qd, const double *kd,
                      const uint16_t *v, int B, int Hq, int Hkv, int N, int d, float scale,
                      int mask_kind, int window, const int32_t *cu_seqlens,
                      const int32_t *seqlens_k, const int32_t *block_table, int max_pages,
                      int page_size, const int64_t *rows, int64_t nrows, double *o, double *lse,
                      double *probs, int64_t probs_stride, int nthreads) {
    problem_t P = {q, k, v, qd, kd, B, Hq, Hkv, N, d, (double)scale, mask_kind, window,
                   cu_seqlens, seqlens_k, block_table, max_pages, page_size};
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || d <= 0 || N < 0) return -1;
    if (mask_kind < OR_NONE || mask_kind > OR_PAGED_PREFILL) return -1;
    if (mask_kind == OR_SLIDING && window < 1) return -1;
    if ((mask_kind == OR_SLIDING_BIDIR || mask_kind == OR_PREFIX_LM) && window < 0) return -1;
    if ((is_document(mask_kind) || is_decode(mask_kind)) && !cu_seqlens) return -1;
    for (int b = 0; mask_kind == OR_DECODE && b < B; b++) {
        const int L = cu_seqlens[b + 1] - cu_seqlens[b];
        if (L < 0 || L > N) return -1;  /* the dense cache holds N keys per sequence */
    }
    if (is_paged(mask_kind) && (!block_table || page_size <= 0)) return -1;
    if (mask_kind == OR_PAGED_PREFILL) {
        if (!seqlens_k || cu_seqlens[0] != 0 || cu_seqlens[B] != N) return -1;
        for (int b = 0; b < B; b++) {
            const int Lq = cu_seqlens[b + 1] - cu_seqlens[b], Lk = seqlens_k[b];
            if (Lq < 0 || Lk < Lq || Lk > max_pages * page_size) return -1;
        }
    }

    const int64_t total = row_count(&P);
    const int64_t n = rows ? nrows : total;
    for (int64_t t = 0; rows && t < n; t++)
        if (rows[t] < 0 || rows[t] >= total) return -1;
    int maxk = is_decode(mask_kind) ? 0 : N;
    for (int b = 0; is_decode(mask_kind) && b < B; b++) {
        int L = cu_seqlens[b + 1] - cu_seqlens[b];
        if (L > maxk) maxk = L;
    }
    for (int b = 0; mask_kind == OR_PAGED_PREFILL && b < B; b++)
        if (seqlens_k[b] > maxk) maxk = seqlens_k[b];
    if (probs && probs_stride < maxk) return -1;

#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
    int failed = 0;
#pragma omp parallel
    {
        double *z = (double *)malloc(sizeof(double) * (size_t)(maxk > 0 ? maxk : 1));
        if (!z) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(dynamic, 4)
        for (int64_t t = 0; t < n; t++) {
            if (!z) continue;
            const int64_t r = rows ? rows[t] : t;
            attend_row(&P, r, z, o + (size_t)t * d, lse + t,
                       probs ? probs + (size_t)t * probs_stride : NULL);
        }
        free(z);
    }
    return failed ? -2 : 0;
}

int oracle_attn(const uint16_t *q, const uint16_t *k, const uint16_t *v, int B, int Hq,
                int Hkv, int N, int d, float scale, int mask_kind, int window,
                const int32_t *cu_seqlens, const int32_t *seqlens_k,
                const int32_t *block_table, int max_pages, int page_size, const int64_t *rows,
                int64_t nrows, double *o, double *lse, double *probs, int64_t probs_stride,
                int nthreads) {
    return oracle_run(q, k, NULL, NULL, v, B, Hq, Hkv, N, d, scale, mask_kind, window,
                      cu_seqlens, seqlens_k, block_table, max_pages, page_size, rows, nrows, o,
                      lse, probs, probs_stride, nthreads);
}

/* The same with Q and K given as fp64 values (the FP8 path passes its dequantized blocks,
 * code value times block scale, which fp64 holds exactly); V stays bf16. */
int oracle_attn_qk_f64(const double *q, const double *k, const uint16_t *v, int B, int Hq,
                       int Hkv, int N, int d, float scale, int mask_kind, int window,
                       const int32_t *cu_seqlens, const int32_t *seqlens_k,
                       const int32_t *block_table, int max_pages, int page_size,
                       const int64_t *rows, int64_t nrows, double *o, double *lse,
                       double *probs, int64_t probs_stride, int nthreads) {
    if (!q || !k) return -1;
    return oracle_run(NULL, NULL, q, k, v, B, Hq, Hkv, N, d, scale, mask_kind, window,
                      cu_seqlens, seqlens_k, block_table, max_pages, page_size, rows, nrows, o,
                      lse, probs, probs_stride, nthreads);
}

/* Number of OpenMP threads a parallel region would use (for reporting the CPU baseline). */
int oracle_max_threads(int nthreads) {
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
    return omp_get_max_threads();
#else
    (void)nthreads;
    return 1;
#endif
}
