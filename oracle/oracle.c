/*
 * oracle.c -- plain, slow fp64 reference for cascade verify and prefix-hit
 * prefill over a paged KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or
 * calls this file; only the tests, the smoke check and the benchmark's CPU
 * baseline do.  It shares no code with the CUDA library.
 *
 * What it computes is the *definition*, not the cascade algorithm:
 *
 *   "Cascade attention" page (zdszero.github.io/cascade_attention.html),
 *   section on the split property of standard attention: for one query q,
 *       o = softmax(q K^T / sqrt(d)) V,   LSE = log sum_j exp(q k_j / sqrt(d)).
 *   The same page states that the two-pass cascade with merge_state is
 *   exactly equal to one full attention, so the oracle is one full masked
 *   attention per (query token, query head), in double precision, with no
 *   split, no tiling and no online softmax.
 *
 * Visible key sets:
 *   - verify (same page, "Topk > 1" section): draft token s of branch k of
 *     request b sees the request's whole prefix (positions 0..L_b-1) and its
 *     own branch's drafts 0..s (its ancestors, itself included -- the tree
 *     attention mask of the KV-cache tutorial, Q14, puts each node in its own
 *     ancestor set).  Pass A is the prefix part alone, Pass B the draft part.
 *   - tree verify (KV-cache tutorial, section 8.2 tip box on tree attention,
 *     and interview question Q14): the draft tokens of request b are the N
 *     nodes of a token tree flattened in BFS order; node i sees the whole
 *     prefix and the tree nodes j with M[i, j] = 1, M being the ancestor mask
 *     (j is i or an ancestor of i).  The mask arrives as one 64-bit row per
 *     node, bit j = M[i, j]; the chain-per-branch case above is the forest of
 *     topk chains.
 *   - prefix-hit prefill ("Causal Attention: why attention scales by 1-h^2
 *     after a KV hit", sections 1-2): suffix query i, at absolute position
 *     H+i, sees keys 0..H+i (the rectangle 0..H-1 plus the triangle H..H+i);
 *     this is the tril(..., diagonal = L_total - L_new) mask of the tutorial's
 *     cached-prefill code (section 6.1).
 *
 * Paged addressing (KV-cache tutorial, sections 5.2-5.3 and the
 * append_token sketch of 6.2): logical position pos of a sequence with block
 * table `tab` is page tab[pos / P], slot pos % P.  The pool is laid out
 * [num_pages, P, H_kv, d]; the KV head of query head h is h / (H_q / H_kv)
 * (repeat_interleave grouping, tutorial section 6.3).
 *
 * Conventions fixed here because the pages leave them open: the 1/sqrt(d)
 * scale applies inside both the softmax and LSE; logs are natural; an empty
 * key set gives o = 0 and lse = -inf.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define ORACLE_OK 0
#define ORACLE_BAD_ARG 1
#define ORACLE_BAD_PAGE 2
#define ORACLE_NO_MEM 3

/* Exact widening of a bf16 bit pattern to double. */
static double bf16_bits_to_double(uint16_t b) {
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/*
 * FP8 E4M3 code to double, from the format's definition (1 sign bit, 4
 * exponent bits with bias 7, 3 mantissa bits; exponent field 0 holds the
 * subnormals m/8 * 2^-6; the all-ones exponent with all-ones mantissa is NaN,
 * and there is no infinity).
 */
static double e4m3_to_double(uint8_t b) {
    int sign = b >> 7, e = (b >> 3) & 15, m = b & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0)
        v = ldexp((double)m, -9);          /* (m/8) * 2^(1-7) */
    else
        v = ldexp(8.0 + (double)m, e - 10); /* (1 + m/8) * 2^(e-7) */
    return sign ? -v : v;
}

/*
 * Where a K or V element comes from: the bf16 pools, or FP8 E4M3 pools whose
 * value is code * scale, with one scale per tensor or one per (KV head,
 * channel) ("FP8 KV", per-tensor / per-channel: KV-cache tutorial, section
 * 4.5).
 */
typedef struct {
    const uint16_t *k16, *v16;        /* bf16 bit patterns, or NULL */
    const uint8_t *k8, *v8;           /* E4M3 codes, or NULL */
    const double *k_scale, *v_scale;  /* E4M3 only */
    int per_channel;                  /* scales indexed [kv_head * d + c], else [0] */
} kv_src_t;

static double kv_elem(const kv_src_t *kv, int is_v, int64_t off, int kv_head, int d, int c) {
    if (kv->k8) {
        const uint8_t *pool = is_v ? kv->v8 : kv->k8;
        const double *sc = is_v ? kv->v_scale : kv->k_scale;
        double scale = kv->per_channel ? sc[(int64_t)kv_head * d + c] : sc[0];
        return e4m3_to_double(pool[off + c]) * scale;
    }
    return bf16_bits_to_double((is_v ? kv->v16 : kv->k16)[off + c]);
}

/*
 * Full attention of one query over an explicit list of key rows.
 * key_off[j] is the element offset of key j's head row inside the K / V
 * pools.  Scores, max, sum and weighted sum are taken in that order, as the
 * softmax definition reads; nothing is blocked or rescaled on the way.
 */
static void attend_one(const double *q, const kv_src_t *kv, int kv_head, const int64_t *key_off,
                       int n_keys, int d, double scale, double *scores, double *o, double *lse) {
    for (int c = 0; c < d; ++c) o[c] = 0.0;
    if (n_keys == 0) {
        *lse = -INFINITY;
        return;
    }
    double m = -INFINITY;
    for (int j = 0; j < n_keys; ++j) {
        double dot = 0.0;
        for (int c = 0; c < d; ++c) dot += q[c] * kv_elem(kv, 0, key_off[j], kv_head, d, c);
        scores[j] = dot * scale;
        if (scores[j] > m) m = scores[j];
    }
    double z = 0.0;
    for (int j = 0; j < n_keys; ++j) {
        double w = exp(scores[j] - m);
        scores[j] = w;
        z += w;
    }
    for (int j = 0; j < n_keys; ++j) {
        double w = scores[j] / z;
        for (int c = 0; c < d; ++c) o[c] += w * kv_elem(kv, 1, key_off[j], kv_head, d, c);
    }
    *lse = m + log(z);
}

/* ------------------------------------------------------------------ */
/* Problem descriptions                                                */
/* ------------------------------------------------------------------ */

enum { KIND_VERIFY = 0, KIND_PREFILL = 1, KIND_TREE = 2 };
/* part: 0 = full visible set, 1 = first piece only (prefix / rectangle),
 *       2 = second piece only (own drafts / causal triangle);
 *       multi-level verify also: 3 = shared prefix only, 4 = own prefix only. */

typedef struct {
    int kind;
    int part;
    const uint16_t *q, *k_pages, *v_pages;
    kv_src_t kv;  /* filled from k_pages / v_pages unless the pools are FP8 */
    int64_t num_pages;
    int H_q, H_kv, d, P;
    double scale;
    /* verify */
    const int32_t *prefix_pt, *draft_pt, *prefix_lens;
    int prefix_stride, draft_stride, B, topk, S;
    /* multi-level verify: one shared prefix per group of group_size requests */
    const int32_t *shared_pt;
    int shared_stride, shared_len, group_size;
    /* tree verify (also uses prefix_pt, prefix_stride, prefix_lens, B, N) */
    const int32_t *tree_pt;
    int tree_stride;
    const uint64_t *masks;
    /* prefill */
    const int32_t *pt;
    int pt_stride, N, H;
    /* rows to evaluate: row = token * H_q + head; NULL = all rows in order */
    const int64_t *rows;
    int64_t n_rows;
    double *o, *lse;
    int max_keys;
    volatile int error;
} problem_t;

static int64_t key_offset(const problem_t *p, const int32_t *table_row, int pos, int kv_head,
                          int *bad) {
    int32_t page = table_row[pos / p->P];
    if (page < 0 || (int64_t)page >= p->num_pages) {
        *bad = 1;
        return 0;
    }
    int slot = pos % p->P;
    return (((int64_t)page * p->P + slot) * p->H_kv + kv_head) * (int64_t)p->d;
}

/* Fill key_off with the visible keys of one (token, head) row; returns count or -1. */
static int visible_keys(const problem_t *p, int64_t token, int head, int64_t *key_off) {
    int group = p->H_q / p->H_kv;
    int kv_head = head / group;
    int n = 0, bad = 0;
    if (p->kind == KIND_VERIFY) {
        int TS = p->topk * p->S;
        int b = (int)(token / TS);
        int i = (int)(token % TS);
        int branch = i / p->S;
        int s = i % p->S;
        /* pieces in key order: the group's shared prefix (multi-level only), the
         * request's own prefix, the branch's own drafts */
        int want_shared = p->part == 0 || p->part == 1 || p->part == 3;
        int want_own = p->part == 0 || p->part == 1 || p->part == 4;
        int want_draft = p->part == 0 || p->part == 2;
        if (p->shared_pt && want_shared) {
            const int32_t *row = p->shared_pt + (int64_t)(b / p->group_size) * p->shared_stride;
            for (int pos = 0; pos < p->shared_len; ++pos)
                key_off[n++] = key_offset(p, row, pos, kv_head, &bad);
        }
        if (want_own) {
            const int32_t *row = p->prefix_pt + (int64_t)b * p->prefix_stride;
            int L = p->prefix_lens[b];
            for (int pos = 0; pos < L; ++pos) key_off[n++] = key_offset(p, row, pos, kv_head, &bad);
        }
        if (want_draft) {
            const int32_t *row = p->draft_pt + ((int64_t)b * p->topk + branch) * p->draft_stride;
            for (int j = 0; j <= s; ++j) key_off[n++] = key_offset(p, row, j, kv_head, &bad);
        }
    } else if (p->kind == KIND_TREE) {
        int b = (int)(token / p->N);
        if (p->part != 2) {
            const int32_t *row = p->prefix_pt + (int64_t)b * p->prefix_stride;
            int L = p->prefix_lens[b];
            for (int pos = 0; pos < L; ++pos) key_off[n++] = key_offset(p, row, pos, kv_head, &bad);
        }
        if (p->part != 1) {
            const int32_t *row = p->tree_pt + (int64_t)b * p->tree_stride;
            uint64_t m = p->masks[token];
            for (int j = 0; j < p->N; ++j)
                if ((m >> j) & 1u) key_off[n++] = key_offset(p, row, j, kv_head, &bad);
        }
    } else {
        int M = p->N - p->H;
        int b = (int)(token / M);
        int i = (int)(token % M);
        const int32_t *row = p->pt + (int64_t)b * p->pt_stride;
        int lo = (p->part == 2) ? p->H : 0;
        int hi = (p->part == 1) ? p->H : p->H + i + 1; /* exclusive */
        for (int pos = lo; pos < hi; ++pos) key_off[n++] = key_offset(p, row, pos, kv_head, &bad);
    }
    return bad ? -1 : n;
}

typedef struct {
    problem_t *p;
    int64_t lo, hi;
} slice_t;

static void *worker(void *arg) {
    slice_t *sl = (slice_t *)arg;
    problem_t *p = sl->p;
    int d = p->d;
    int64_t *key_off = (int64_t *)malloc(sizeof(int64_t) * (size_t)(p->max_keys + 1));
    double *scores = (double *)malloc(sizeof(double) * (size_t)(p->max_keys + 1));
    double *qd = (double *)malloc(sizeof(double) * (size_t)d);
    if (!key_off || !scores || !qd) {
        p->error = ORACLE_NO_MEM;
        free(key_off); free(scores); free(qd);
        return NULL;
    }
    for (int64_t r = sl->lo; r < sl->hi; ++r) {
        int64_t row = p->rows ? p->rows[r] : r;
        int64_t token = row / p->H_q;
        int head = (int)(row % p->H_q);
        const uint16_t *qr = p->q + row * d;
        for (int c = 0; c < d; ++c) qd[c] = bf16_bits_to_double(qr[c]);
        int n = visible_keys(p, token, head, key_off);
        if (n < 0) {
            p->error = ORACLE_BAD_PAGE;
            continue;
        }
        attend_one(qd, &p->kv, head / (p->H_q / p->H_kv), key_off, n, d, p->scale, scores,
                   p->o + r * d, p->lse + r);
    }
    free(key_off); free(scores); free(qd);
    return NULL;
}

static int run_rows(problem_t *p, int n_threads) {
    if (!p->kv.k8) {
        p->kv.k16 = p->k_pages;
        p->kv.v16 = p->v_pages;
    }
    if (n_threads <= 0) {
        long c = sysconf(_SC_NPROCESSORS_ONLN);
        n_threads = c > 0 ? (int)c : 1;
    }
    if (n_threads > 256) n_threads = 256;
    if ((int64_t)n_threads > p->n_rows) n_threads = p->n_rows > 0 ? (int)p->n_rows : 1;
    pthread_t th[256];
    int spawned[256];
    slice_t sl[256];
    for (int t = 0; t < n_threads; ++t) {
        sl[t].p = p;
        sl[t].lo = p->n_rows * t / n_threads;
        sl[t].hi = p->n_rows * (t + 1) / n_threads;
        spawned[t] = n_threads > 1 && pthread_create(&th[t], NULL, worker, &sl[t]) == 0;
        if (!spawned[t]) worker(&sl[t]);
    }
    for (int t = 0; t < n_threads; ++t)
        if (spawned[t]) pthread_join(th[t], NULL);
    return p->error;
}

/* ------------------------------------------------------------------ */
/* Exported entry points                                               */
/* ------------------------------------------------------------------ */

/*
 * Verify attention for rows (token, head).  part 0 = full (prefix + own
 * drafts 0..s), 1 = prefix only (Pass A), 2 = own drafts only (Pass B).
 * o: [n_rows, d] doubles, lse: [n_rows] natural log.
 */
int oracle_verify(const uint16_t *q, const uint16_t *k_pages, const uint16_t *v_pages,
                  int64_t num_pages, const int32_t *prefix_pt, int prefix_stride,
                  const int32_t *draft_pt, int draft_stride, const int32_t *prefix_lens, int B,
                  int topk, int S, int H_q, int H_kv, int d, int P, int part, double scale,
                  const int64_t *rows, int64_t n_rows, double *o, double *lse, int n_threads) {
    if (B < 0 || topk < 1 || S < 1 || H_kv < 1 || H_q % H_kv != 0 || d < 1 || P < 1 ||
        part < 0 || part > 2)
        return ORACLE_BAD_ARG;
    problem_t p;
    memset(&p, 0, sizeof p);
    p.kind = KIND_VERIFY;
    p.part = part;
    p.q = q; p.k_pages = k_pages; p.v_pages = v_pages; p.num_pages = num_pages;
    p.H_q = H_q; p.H_kv = H_kv; p.d = d; p.P = P; p.scale = scale;
    p.prefix_pt = prefix_pt; p.draft_pt = draft_pt; p.prefix_lens = prefix_lens;
    p.prefix_stride = prefix_stride; p.draft_stride = draft_stride;
    p.B = B; p.topk = topk; p.S = S;
    int64_t total_rows = (int64_t)B * topk * S * H_q;
    p.rows = rows;
    p.n_rows = rows ? n_rows : total_rows;
    int maxL = 0;
    for (int b = 0; b < B; ++b) {
        if (prefix_lens[b] < 0) return ORACLE_BAD_ARG;
        if (prefix_lens[b] > maxL) maxL = prefix_lens[b];
    }
    if (rows)
        for (int64_t r = 0; r < n_rows; ++r)
            if (rows[r] < 0 || rows[r] >= total_rows) return ORACLE_BAD_ARG;
    p.max_keys = maxL + S;
    p.o = o; p.lse = lse;
    return run_rows(&p, n_threads);
}

/*
 * Verify over FP8 KV pools ("FP8 KV" of the KV-cache tutorial, section 4.5:
 * per-tensor or per-channel FP8).  k_codes / v_codes are E4M3 codes laid out
 * like the bf16 pools, [num_pages, P, H_kv, d]; element value = decoded code *
 * scale, with k_scale / v_scale of length 1 (per_channel = 0) or H_kv * d
 * (per_channel = 1, index kv_head * d + channel).  Everything else as
 * oracle_verify.
 */
int oracle_verify_fp8(const uint16_t *q, const uint8_t *k_codes, const uint8_t *v_codes,
                      const double *k_scale, const double *v_scale, int per_channel,
                      int64_t num_pages, const int32_t *prefix_pt, int prefix_stride,
                      const int32_t *draft_pt, int draft_stride, const int32_t *prefix_lens,
                      int B, int topk, int S, int H_q, int H_kv, int d, int P, int part,
                      double scale, const int64_t *rows, int64_t n_rows, double *o, double *lse,
                      int n_threads) {
    if (B < 0 || topk < 1 || S < 1 || H_kv < 1 || H_q % H_kv != 0 || d < 1 || P < 1 ||
        part < 0 || part > 2 || !k_codes || !v_codes || !k_scale || !v_scale)
        return ORACLE_BAD_ARG;
    problem_t p;
    memset(&p, 0, sizeof p);
    p.kind = KIND_VERIFY;
    p.part = part;
    p.q = q; p.num_pages = num_pages;
    p.kv.k8 = k_codes; p.kv.v8 = v_codes;
    p.kv.k_scale = k_scale; p.kv.v_scale = v_scale; p.kv.per_channel = per_channel ? 1 : 0;
    p.H_q = H_q; p.H_kv = H_kv; p.d = d; p.P = P; p.scale = scale;
    p.prefix_pt = prefix_pt; p.draft_pt = draft_pt; p.prefix_lens = prefix_lens;
    p.prefix_stride = prefix_stride; p.draft_stride = draft_stride;
    p.B = B; p.topk = topk; p.S = S;
    int64_t total_rows = (int64_t)B * topk * S * H_q;
    p.rows = rows;
    p.n_rows = rows ? n_rows : total_rows;
    int maxL = 0;
    for (int b = 0; b < B; ++b) {
        if (prefix_lens[b] < 0) return ORACLE_BAD_ARG;
        if (prefix_lens[b] > maxL) maxL = prefix_lens[b];
    }
    if (rows)
        for (int64_t r = 0; r < n_rows; ++r)
            if (rows[r] < 0 || rows[r] >= total_rows) return ORACLE_BAD_ARG;
    p.max_keys = maxL + S;
    p.o = o; p.lse = lse;
    return run_rows(&p, n_threads);
}

/* Decode n E4M3 codes to doubles (for checking the decoder). */
void oracle_e4m3_decode(const uint8_t *codes, int64_t n, double *out) {
    for (int64_t i = 0; i < n; ++i) out[i] = e4m3_to_double(codes[i]);
}

/*
 * Multi-level verify (KV-cache tutorial, sections 5.3 and 6.2: requests whose
 * block tables begin with the same physical pages share that prefix).  The
 * B requests form B / group_size groups of consecutive requests; group g's
 * shared prefix is positions 0..shared_len-1 of shared_pt row g.  Request b
 * then has its own prefix (prefix_pt row b, prefix_lens[b] tokens) and its
 * branches' drafts as in oracle_verify.  Draft s of branch k of request b
 * sees the shared prefix, the own prefix and drafts 0..s of its branch.
 * part 0 = all, 1 = shared + own prefix, 2 = drafts, 3 = shared only,
 * 4 = own prefix only.
 */
int oracle_verify_shared(const uint16_t *q, const uint16_t *k_pages, const uint16_t *v_pages,
                         int64_t num_pages, const int32_t *shared_pt, int shared_stride,
                         int shared_len, int group_size, const int32_t *prefix_pt,
                         int prefix_stride, const int32_t *draft_pt, int draft_stride,
                         const int32_t *prefix_lens, int B, int topk, int S, int H_q, int H_kv,
                         int d, int P, int part, double scale, const int64_t *rows,
                         int64_t n_rows, double *o, double *lse, int n_threads) {
    if (B < 0 || topk < 1 || S < 1 || H_kv < 1 || H_q % H_kv != 0 || d < 1 || P < 1 ||
        part < 0 || part > 4 || !shared_pt || shared_len < 0 || group_size < 1 ||
        B % group_size != 0)
        return ORACLE_BAD_ARG;
    problem_t p;
    memset(&p, 0, sizeof p);
    p.kind = KIND_VERIFY;
    p.part = part;
    p.q = q; p.k_pages = k_pages; p.v_pages = v_pages; p.num_pages = num_pages;
    p.H_q = H_q; p.H_kv = H_kv; p.d = d; p.P = P; p.scale = scale;
    p.shared_pt = shared_pt; p.shared_stride = shared_stride; p.shared_len = shared_len;
    p.group_size = group_size;
    p.prefix_pt = prefix_pt; p.draft_pt = draft_pt; p.prefix_lens = prefix_lens;
    p.prefix_stride = prefix_stride; p.draft_stride = draft_stride;
    p.B = B; p.topk = topk; p.S = S;
    int64_t total_rows = (int64_t)B * topk * S * H_q;
    p.rows = rows;
    p.n_rows = rows ? n_rows : total_rows;
    int maxL = 0;
    for (int b = 0; b < B; ++b) {
        if (prefix_lens[b] < 0) return ORACLE_BAD_ARG;
        if (prefix_lens[b] > maxL) maxL = prefix_lens[b];
    }
    if (rows)
        for (int64_t r = 0; r < n_rows; ++r)
            if (rows[r] < 0 || rows[r] >= total_rows) return ORACLE_BAD_ARG;
    p.max_keys = shared_len + maxL + S;
    p.o = o; p.lse = lse;
    return run_rows(&p, n_threads);
}

/*
 * Tree verify for rows (token, head), token = b * N + i the BFS index i of
 * a node of request b's draft tree.  masks[token] bit j set means node i sees
 * tree node j (stored at logical position j of tree_pt row b).  part 0 =
 * prefix + masked tree nodes, 1 = prefix only, 2 = tree nodes only.
 * 1 <= N <= 64; bits at or above N must be clear.
 */
int oracle_tree_verify(const uint16_t *q, const uint16_t *k_pages, const uint16_t *v_pages,
                       int64_t num_pages, const int32_t *prefix_pt, int prefix_stride,
                       const int32_t *tree_pt, int tree_stride, const int32_t *prefix_lens,
                       const uint64_t *masks, int B, int N, int H_q, int H_kv, int d, int P,
                       int part, double scale, const int64_t *rows, int64_t n_rows, double *o,
                       double *lse, int n_threads) {
    if (B < 0 || N < 1 || N > 64 || H_kv < 1 || H_q % H_kv != 0 || d < 1 || P < 1 || part < 0 ||
        part > 2)
        return ORACLE_BAD_ARG;
    problem_t p;
    memset(&p, 0, sizeof p);
    p.kind = KIND_TREE;
    p.part = part;
    p.q = q; p.k_pages = k_pages; p.v_pages = v_pages; p.num_pages = num_pages;
    p.H_q = H_q; p.H_kv = H_kv; p.d = d; p.P = P; p.scale = scale;
    p.prefix_pt = prefix_pt; p.prefix_stride = prefix_stride; p.prefix_lens = prefix_lens;
    p.tree_pt = tree_pt; p.tree_stride = tree_stride; p.masks = masks;
    p.B = B; p.N = N;
    int64_t total_rows = (int64_t)B * N * H_q;
    p.rows = rows;
    p.n_rows = rows ? n_rows : total_rows;
    int maxL = 0;
    for (int b = 0; b < B; ++b) {
        if (prefix_lens[b] < 0) return ORACLE_BAD_ARG;
        if (prefix_lens[b] > maxL) maxL = prefix_lens[b];
    }
    for (int64_t t = 0; t < (int64_t)B * N; ++t)
        if (N < 64 && (masks[t] >> N) != 0) return ORACLE_BAD_ARG;
    if (rows)
        for (int64_t r = 0; r < n_rows; ++r)
            if (rows[r] < 0 || rows[r] >= total_rows) return ORACLE_BAD_ARG;
    p.max_keys = maxL + N;
    p.o = o; p.lse = lse;
    return run_rows(&p, n_threads);
}

/*
 * Prefix-hit prefill: B requests of N tokens, first H cached; queries are the
 * M = N - H suffix tokens (token = b * M + i).  part 0 = keys 0..H+i,
 * 1 = rectangle keys 0..H-1, 2 = triangle keys H..H+i.
 */
int oracle_prefill(const uint16_t *q, const uint16_t *k_pages, const uint16_t *v_pages,
                   int64_t num_pages, const int32_t *pt, int pt_stride, int B, int N, int H,
                   int H_q, int H_kv, int d, int P, int part, double scale, const int64_t *rows,
                   int64_t n_rows, double *o, double *lse, int n_threads) {
    if (B < 0 || N < 0 || H < 0 || H > N || H_kv < 1 || H_q % H_kv != 0 || d < 1 || P < 1 ||
        part < 0 || part > 2)
        return ORACLE_BAD_ARG;
    problem_t p;
    memset(&p, 0, sizeof p);
    p.kind = KIND_PREFILL;
    p.part = part;
    p.q = q; p.k_pages = k_pages; p.v_pages = v_pages; p.num_pages = num_pages;
    p.H_q = H_q; p.H_kv = H_kv; p.d = d; p.P = P; p.scale = scale;
    p.pt = pt; p.pt_stride = pt_stride; p.B = B; p.N = N; p.H = H;
    int64_t total_rows = (int64_t)B * (N - H) * H_q;
    p.rows = rows;
    p.n_rows = rows ? n_rows : total_rows;
    if (rows)
        for (int64_t r = 0; r < n_rows; ++r)
            if (rows[r] < 0 || rows[r] >= total_rows) return ORACLE_BAD_ARG;
    p.max_keys = N;
    p.o = o; p.lse = lse;
    return run_rows(&p, n_threads);
}

/*
 * merge_state, as the cascade page writes it:
 *   LSE = log(e^{LSE_A} + e^{LSE_B}),
 *   o   = e^{LSE_A - LSE} o_A + e^{LSE_B - LSE} o_B.
 * The log-sum is taken about the larger of the two so that exp cannot
 * overflow; two empty parts (both -inf) give o = 0, LSE = -inf.
 */
void oracle_merge_state(const double *o_a, const double *lse_a, const double *o_b,
                        const double *lse_b, int64_t n, int d, double *o, double *lse) {
    for (int64_t r = 0; r < n; ++r) {
        double a = lse_a[r], b = lse_b[r];
        if (isinf(a) && a < 0 && isinf(b) && b < 0) {
            lse[r] = -INFINITY;
            for (int c = 0; c < d; ++c) o[r * d + c] = 0.0;
            continue;
        }
        double m = a > b ? a : b;
        double tot = m + log(exp(a - m) + exp(b - m));
        double wa = exp(a - tot), wb = exp(b - tot);
        lse[r] = tot;
        for (int c = 0; c < d; ++c) o[r * d + c] = wa * o_a[r * d + c] + wb * o_b[r * d + c];
    }
}
