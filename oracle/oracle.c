/*
 * oracle.c -- plain, slow, fp64 CPU oracle for one batched DDTree round.
 *
 * TEST INFRASTRUCTURE. Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg load this library. The CUDA library never
 * calls it, and the two share no source, header, table or helper.
 *
 * Every floating-point step runs in IEEE double. Inputs arrive as fp32 or as
 * raw bf16 bit patterns and are widened exactly. Each function states the
 * passage it follows; pages are named by title and section:
 *
 *   [SPARK]  "SparklingTree: 30-40% faster speculative decoding over DSpark",
 *            section "How is the tree actually created?", Steps 1-4.
 *   [DDTX]   "DDTree Explained: From Block Diffusion to Optimal Diffusion
 *            Draft Trees for Speculative Decoding", sections 2-5.
 *   [TSPK]   "Robot2050/TreeSpark", item 4 (exactness by construction) and
 *            the continuous-batching engine description.
 *
 * Readings where the pages are silent are listed beside the function.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_LMAX 32 /* deepest draft block the oracle accepts */

/* status bits returned by the oracle (0 = clean) */
#define ORC_NAN_SEEN 1
#define ORC_BAD_ARG 2
#define ORC_BAD_PAGE 4

/* exact widening: dtype 0 = fp32, 1 = bf16 bit pattern, 2 = fp64 */
static double widen(const void *base, int dtype, int64_t i)
{
    if (dtype == 0)
        return (double)((const float *)base)[i];
    if (dtype == 2)
        return ((const double *)base)[i];
    uint32_t u = ((uint32_t)((const uint16_t *)base)[i]) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double bf16_to_double(uint16_t b)
{
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* ------------------------------------------------------------------------
 * Step 1 of the round [SPARK, Step 1; DDTX section 3, Lemma 1].
 * For every row (request r, depth d) of the drafter's marginals:
 *   logZ = log sum_v exp(z_v)           (max-shifted, fp64)
 *   the K largest logits, ordered by value descending, equal values by
 *   lower token id first (reading: the pages' top-k leaves ties open),
 *   lp_k = z_{id_k} - logZ.
 * Rows are independent; OpenMP spreads them over host threads.
 * ---------------------------------------------------------------------- */
int orc_topk_logprobs(const void *z, int dtype, int64_t rows, int64_t V, int K,
                      double *lp, int32_t *ids, double *logz_out)
{
    if (K < 1 || (int64_t)K > V)
        return ORC_BAD_ARG;
    int flags = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : flags)
    for (int64_t row = 0; row < rows; ++row) {
        const int64_t off = row * V;
        double m = -INFINITY;
        for (int64_t v = 0; v < V; ++v) {
            double x = widen(z, dtype, off + v);
            if (isnan(x))
                flags |= ORC_NAN_SEEN;
            if (x > m)
                m = x;
        }
        double s = 0.0;
        for (int64_t v = 0; v < V; ++v)
            s += exp(widen(z, dtype, off + v) - m);
        const double logZ = m + log(s);

        /* running top-K by insertion; ids arrive in increasing order, so an
         * equal value never displaces an earlier (lower) id */
        double *tv = (double *)malloc(sizeof(double) * (size_t)K);
        int32_t *ti = (int32_t *)malloc(sizeof(int32_t) * (size_t)K);
        int n = 0;
        for (int64_t v = 0; v < V; ++v) {
            double x = widen(z, dtype, off + v);
            if (n == K && !(x > tv[K - 1]))
                continue;
            int pos = (n < K) ? n : K - 1;
            while (pos > 0 && tv[pos - 1] < x) {
                tv[pos] = tv[pos - 1];
                ti[pos] = ti[pos - 1];
                --pos;
            }
            tv[pos] = x;
            ti[pos] = (int32_t)v;
            if (n < K)
                ++n;
        }
        for (int k = 0; k < K; ++k) {
            lp[row * K + k] = tv[k] - logZ;
            ids[row * K + k] = ti[k];
        }
        if (logz_out)
            logz_out[row] = logZ;
        free(tv);
        free(ti);
    }
    return flags;
}

/* ------------------------------------------------------------------------
 * Step 2: best-first selection of the B most probable prefixes
 * [SPARK, Step 3; DDTX section 4, Algorithm 1; DDTX section 3, Prop. 2].
 *
 * A prefix is a rank tuple rho = (rho_1..rho_d): position i takes the
 * rho_i-th most probable token of row i. Its score is
 *   S(rho) = lp[0][rho_1] + lp[1][rho_2] + ... + lp[d-1][rho_d],
 * accumulated left to right in fp64. The heap pops the entry with the
 * largest S; equal S falls to the lexicographically smaller rank tuple,
 * a tuple before its own extensions (this is how the pages' heap compares
 * its (-score, ranks, ...) records). Each pop becomes node n = pops so far,
 * then pushes the sibling (.., rho_d + 1) when rho_d + 1 < K and the child
 * (.., rho_d, 0) when d < L. The heap starts from the single entry (0,).
 *
 * Reading: the pages update a sibling's score incrementally
 * (score - lp[rank] + lp[rank+1]); here every entry carries its parent's S
 * and scores as parent_S + lp, which is the same number in exact
 * arithmetic and rounds identically on every machine.
 * ---------------------------------------------------------------------- */
typedef struct {
    double S;
    double parent_S;
    int32_t ranks[ORC_LMAX];
    int32_t len; /* depth of the prefix */
    int32_t parent;
} heap_ent;

/* does a pop before b? */
static int ent_before(const heap_ent *a, const heap_ent *b)
{
    if (a->S != b->S)
        return a->S > b->S;
    int n = a->len < b->len ? a->len : b->len;
    for (int i = 0; i < n; ++i)
        if (a->ranks[i] != b->ranks[i])
            return a->ranks[i] < b->ranks[i];
    return a->len < b->len;
}

static void heap_push(heap_ent *h, int *size, const heap_ent *e)
{
    int i = (*size)++;
    h[i] = *e;
    while (i > 0) {
        int p = (i - 1) / 2;
        if (!ent_before(&h[i], &h[p]))
            break;
        heap_ent t = h[i];
        h[i] = h[p];
        h[p] = t;
        i = p;
    }
}

static heap_ent heap_pop(heap_ent *h, int *size)
{
    heap_ent top = h[0];
    h[0] = h[--(*size)];
    int i = 0;
    for (;;) {
        int l = 2 * i + 1, r = l + 1, best = i;
        if (l < *size && ent_before(&h[l], &h[best]))
            best = l;
        if (r < *size && ent_before(&h[r], &h[best]))
            best = r;
        if (best == i)
            break;
        heap_ent t = h[i];
        h[i] = h[best];
        h[best] = t;
        i = best;
    }
    return top;
}

/*
 * lp, ids: [R, L, K]. Outputs per request (P = B + 1 positions):
 *   tree_tokens [R, B]   token of node n at slot n-1, -1 when unused
 *   parents     [R, P]   parents[0] = -1 (root = the bonus token)
 *   depths      [R, P]   depths[0] = 0, nodes are 1-based in depth
 *   node_S      [R, P]   prefix score of each node, node_S[0] = 0
 *   node_ranks  [R, P, L] rank tuple of each node, -1 padded
 *   n_nodes     [R]      number of non-root nodes (< B only when the
 *                        whole prefix space is smaller than B)
 */
int orc_build_tree(const double *lp, const int32_t *ids, int R, int L, int K, int B,
                   int32_t *tree_tokens, int32_t *parents, int32_t *depths,
                   double *node_S, int32_t *node_ranks, int32_t *n_nodes)
{
    if (L < 1 || L > ORC_LMAX || K < 1 || B < 1)
        return ORC_BAD_ARG;
    const int P = B + 1;
#pragma omp parallel for schedule(dynamic, 1)
    for (int r = 0; r < R; ++r) {
        const double *lpr = lp + (int64_t)r * L * K;
        const int32_t *idr = ids + (int64_t)r * L * K;
        int32_t *tok = tree_tokens + (int64_t)r * B;
        int32_t *par = parents + (int64_t)r * P;
        int32_t *dep = depths + (int64_t)r * P;
        double *ns = node_S + (int64_t)r * P;
        int32_t *nr = node_ranks + (int64_t)r * P * L;
        for (int j = 0; j < B; ++j)
            tok[j] = -1;
        for (int j = 0; j < P; ++j) {
            par[j] = -1;
            dep[j] = -1;
            ns[j] = 0.0;
            for (int i = 0; i < L; ++i)
                nr[j * L + i] = -1;
        }
        dep[0] = 0;

        heap_ent *heap = (heap_ent *)malloc(sizeof(heap_ent) * (size_t)(2 * B + 4));
        int size = 0;
        heap_ent first;
        memset(&first, 0, sizeof first);
        first.parent_S = 0.0;
        first.S = 0.0 + lpr[0];
        first.ranks[0] = 0;
        first.len = 1;
        first.parent = 0;
        heap_push(heap, &size, &first);

        int count = 0;
        while (size > 0 && count < B) {
            heap_ent e = heap_pop(heap, &size);
            const int depth = e.len;
            const int rank = e.ranks[depth - 1];
            const int node = count + 1;
            tok[count] = idr[(depth - 1) * K + rank];
            par[node] = e.parent;
            dep[node] = depth;
            ns[node] = e.S;
            for (int i = 0; i < depth; ++i)
                nr[node * L + i] = e.ranks[i];
            ++count;
            if (rank + 1 < K) {
                heap_ent sib = e;
                sib.ranks[depth - 1] = rank + 1;
                sib.S = e.parent_S + lpr[(depth - 1) * K + rank + 1];
                heap_push(heap, &size, &sib);
            }
            if (depth < L) {
                heap_ent ch = e;
                ch.ranks[depth] = 0;
                ch.len = depth + 1;
                ch.parent = node;
                ch.parent_S = e.S;
                ch.S = e.S + lpr[depth * K + 0];
                heap_push(heap, &size, &ch);
            }
        }
        n_nodes[r] = count;
        free(heap);
    }
    return 0;
}

/* ------------------------------------------------------------------------
 * Second, independent construction of the same tree for small inputs: list
 * every prefix of depth 1..L over ranks 0..K-1, score each left to right,
 * sort the whole list by (S descending, rank tuple ascending) with qsort,
 * keep the first B. [DDTX section 3, Prop. 2: the B best prefixes form a
 * prefix-closed tree.] Node n is the n-th prefix of the sorted list; its
 * parent is the node whose tuple drops the last rank. Returns the number of
 * enumerated prefixes, or -1 when that exceeds max_prefixes.
 * ---------------------------------------------------------------------- */
typedef struct {
    double S;
    int32_t ranks[ORC_LMAX];
    int32_t len;
} pref_ent;

static int pref_cmp(const void *pa, const void *pb)
{
    const pref_ent *a = (const pref_ent *)pa, *b = (const pref_ent *)pb;
    if (a->S != b->S)
        return a->S > b->S ? -1 : 1;
    int n = a->len < b->len ? a->len : b->len;
    for (int i = 0; i < n; ++i)
        if (a->ranks[i] != b->ranks[i])
            return a->ranks[i] < b->ranks[i] ? -1 : 1;
    return (a->len > b->len) - (a->len < b->len);
}

int64_t orc_build_tree_bruteforce(const double *lp, const int32_t *ids, int L, int K, int B,
                                  int64_t max_prefixes, int32_t *tree_tokens, int32_t *parents,
                                  int32_t *depths, double *node_S, int32_t *node_ranks,
                                  int32_t *n_nodes)
{
    if (L < 1 || L > ORC_LMAX || K < 1 || B < 1)
        return -1;
    int64_t total = 0, layer = 1;
    for (int d = 1; d <= L; ++d) {
        layer *= K;
        total += layer;
        if (total > max_prefixes)
            return -1;
    }
    pref_ent *all = (pref_ent *)calloc((size_t)total, sizeof(pref_ent));
    int64_t n = 0;
    int32_t digits[ORC_LMAX];
    for (int d = 1; d <= L; ++d) {
        for (int i = 0; i < d; ++i)
            digits[i] = 0;
        for (;;) {
            pref_ent *p = &all[n++];
            p->len = d;
            double S = 0.0;
            for (int i = 0; i < d; ++i) {
                p->ranks[i] = digits[i];
                S = S + lp[i * K + digits[i]];
            }
            p->S = S;
            int i = d - 1;
            while (i >= 0 && ++digits[i] == K) {
                digits[i] = 0;
                --i;
            }
            if (i < 0)
                break;
        }
    }
    qsort(all, (size_t)n, sizeof(pref_ent), pref_cmp);
    const int P = B + 1;
    const int take = (int)(n < B ? n : B);
    for (int j = 0; j < B; ++j)
        tree_tokens[j] = -1;
    for (int j = 0; j < P; ++j) {
        parents[j] = -1;
        depths[j] = -1;
        node_S[j] = 0.0;
        for (int i = 0; i < L; ++i)
            node_ranks[j * L + i] = -1;
    }
    depths[0] = 0;
    for (int j = 0; j < take; ++j) {
        const pref_ent *p = &all[j];
        const int node = j + 1;
        tree_tokens[j] = ids[(p->len - 1) * K + p->ranks[p->len - 1]];
        depths[node] = p->len;
        node_S[node] = p->S;
        for (int i = 0; i < p->len; ++i)
            node_ranks[node * L + i] = p->ranks[i];
        /* parent: the selected prefix equal to this one minus its last rank */
        int parent = -1;
        if (p->len == 1) {
            parent = 0;
        } else {
            for (int q = 0; q < j; ++q) {
                const pref_ent *c = &all[q];
                if (c->len != p->len - 1)
                    continue;
                int same = 1;
                for (int i = 0; i < c->len; ++i)
                    if (c->ranks[i] != p->ranks[i]) {
                        same = 0;
                        break;
                    }
                if (same) {
                    parent = q + 1;
                    break;
                }
            }
        }
        parents[node] = parent; /* -1 here would mean the set is not prefix-closed */
    }
    *n_nodes = take;
    free(all);
    return n;
}

/* ------------------------------------------------------------------------
 * Step 3: ancestor visibility [SPARK, Step 4; DDTX section 5, "ancestor-only
 * tree attention mask"]. Row 0 sees only itself; row i copies its parent's
 * row over columns < i and sets its own column. Rows of unused positions
 * (i > n_nodes) stay empty (reading). Packed as little-endian 32-bit words:
 * bit j of word w is column 32*w + j.
 * ---------------------------------------------------------------------- */
void orc_build_mask(const int32_t *parents, const int32_t *n_nodes, int R, int P, uint32_t *mask)
{
    const int W = (P + 31) / 32;
    unsigned char *vis = (unsigned char *)malloc((size_t)P * (size_t)P);
    for (int r = 0; r < R; ++r) {
        memset(vis, 0, (size_t)P * (size_t)P);
        const int32_t *par = parents + (int64_t)r * P;
        vis[0] = 1;
        for (int i = 1; i <= n_nodes[r] && i < P; ++i) {
            const int p = par[i];
            for (int j = 0; j < i; ++j)
                vis[i * P + j] = vis[p * P + j];
            vis[i * P + i] = 1;
        }
        for (int i = 0; i < P; ++i)
            for (int w = 0; w < W; ++w) {
                uint32_t word = 0;
                for (int b = 0; b < 32; ++b) {
                    const int j = 32 * w + b;
                    if (j < P && vis[i * P + j])
                        word |= (uint32_t)1 << b;
                }
                mask[((int64_t)r * P + i) * W + w] = word;
            }
    }
    free(vis);
}

/* ------------------------------------------------------------------------
 * Step 4: tree attention for one query row [SPARK, Step 4 and "the weird
 * matmul"; DDTX sections 5 and 8 (custom attention mask, Qwen GQA)].
 * Query (r, i, h) attends to every cached token t < ctx_lens[r] of its KV
 * head g = h / (Hq / Hkv), reached through the page table, and to every
 * tree position j whose bit is set in mask row (r, i). Scores are
 * q . k * scale; softmax and the weighted sum of values run in fp64.
 * Layouts (bf16 bit patterns):
 *   q, out  [R, P, Hq, d]          k_tree, v_tree [R, P, Hkv, d]
 *   k_cache, v_cache [pages, page, Hkv, d], block_table [R, max_pages]
 * sel lists n query rows as (r, i, h) triples; out is [n, d] doubles.
 * ---------------------------------------------------------------------- */
int orc_tree_attention_rows(const uint16_t *q, const uint16_t *k_tree, const uint16_t *v_tree,
                            const uint16_t *k_cache, const uint16_t *v_cache,
                            const int32_t *block_table, int max_pages, int64_t num_pages,
                            const int32_t *ctx_lens, const uint32_t *mask, int R, int P, int Hq,
                            int Hkv, int d, int page, double scale, const int32_t *sel, int64_t n,
                            double *out)
{
    if (Hkv < 1 || Hq % Hkv != 0 || d < 1 || page < 1)
        return ORC_BAD_ARG;
    (void)R; /* rows are named by (r, i, h) in sel */
    const int W = (P + 31) / 32;
    const int group = Hq / Hkv;
    int flags = 0;
#pragma omp parallel for schedule(dynamic, 4) reduction(| : flags)
    for (int64_t s = 0; s < n; ++s) {
        const int r = sel[3 * s], i = sel[3 * s + 1], h = sel[3 * s + 2];
        const int g = h / group;
        const int ctx = ctx_lens[r];
        const uint16_t *qrow = q + (((int64_t)r * P + i) * Hq + h) * d;
        const uint32_t *mrow = mask + ((int64_t)r * P + i) * W;
        const int ntree = P;
        double *scores = (double *)malloc(sizeof(double) * (size_t)(ctx + ntree));
        const uint16_t **vrows = (const uint16_t **)malloc(sizeof(void *) * (size_t)(ctx + ntree));
        int cnt = 0;
        double mx = -INFINITY;
        for (int t = 0; t < ctx; ++t) {
            const int32_t pg = block_table[(int64_t)r * max_pages + t / page];
            if (pg < 0 || pg >= num_pages) {
                flags |= ORC_BAD_PAGE;
                continue;
            }
            const int64_t row = ((int64_t)pg * page + t % page) * Hkv + g;
            const uint16_t *krow = k_cache + row * d;
            double dot = 0.0;
            for (int x = 0; x < d; ++x)
                dot += bf16_to_double(qrow[x]) * bf16_to_double(krow[x]);
            scores[cnt] = dot * scale;
            vrows[cnt] = v_cache + row * d;
            if (scores[cnt] > mx)
                mx = scores[cnt];
            ++cnt;
        }
        for (int j = 0; j < ntree; ++j) {
            if (!((mrow[j / 32] >> (j % 32)) & 1u))
                continue;
            const int64_t row = ((int64_t)r * P + j) * Hkv + g;
            const uint16_t *krow = k_tree + row * d;
            double dot = 0.0;
            for (int x = 0; x < d; ++x)
                dot += bf16_to_double(qrow[x]) * bf16_to_double(krow[x]);
            scores[cnt] = dot * scale;
            vrows[cnt] = v_tree + row * d;
            if (scores[cnt] > mx)
                mx = scores[cnt];
            ++cnt;
        }
        double *o = out + s * d;
        for (int x = 0; x < d; ++x)
            o[x] = 0.0;
        double den = 0.0;
        for (int c = 0; c < cnt; ++c) {
            const double p = exp(scores[c] - mx);
            den += p;
            for (int x = 0; x < d; ++x)
                o[x] += p * bf16_to_double(vrows[c][x]);
        }
        for (int x = 0; x < d; ++x)
            o[x] = cnt ? o[x] / den : 0.0;
        free(scores);
        free(vrows);
    }
    return flags;
}

/* ------------------------------------------------------------------------
 * Step 5a: target argmax per tree position [DDTX section 5, verifier walk
 * under the greedy decoding rule; TSPK, vectorised acceptance retrieval].
 * The first index holding the largest value wins; -0 equals +0. A NaN is
 * reported through the status bits (the pages assume finite logits).
 * ---------------------------------------------------------------------- */
int orc_argmax(const void *t, int dtype, int64_t rows, int64_t V, int32_t *out)
{
    int flags = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : flags)
    for (int64_t row = 0; row < rows; ++row) {
        double best = 0.0;
        int32_t arg = -1;
        for (int64_t v = 0; v < V; ++v) {
            const double x = widen(t, dtype, row * V + v);
            if (isnan(x)) {
                flags |= ORC_NAN_SEEN;
                continue;
            }
            if (arg < 0 || x > best) {
                best = x;
                arg = (int32_t)v;
            }
        }
        if (arg < 0)
            arg = 0;
        out[row] = arg;
    }
    return flags;
}

/* ------------------------------------------------------------------------
 * Step 5b: greedy verifier walk [DDTX section 5, "Verifier walk"; TSPK
 * item 4]. Start at the root (the bonus token). At node cur, the target's
 * greedy token is a[cur]; if a child of cur carries that token the child is
 * accepted and the walk moves to it, otherwise a[cur] becomes the new bonus
 * token and the walk ends. Outputs per request:
 *   acc_len    accepted drafts + 1 (the bonus is counted, as the pages'
 *              acceptance length is)
 *   acc_nodes  [R, L] accepted node indices in path order, -1 padded
 *   acc_tokens [R, L+1] accepted tokens then the bonus, -1 padded
 *   bonus      [R]
 * ---------------------------------------------------------------------- */
void orc_walk(const int32_t *a, const int32_t *tree_tokens, const int32_t *parents,
              const int32_t *n_nodes, int R, int B, int L, int32_t *acc_len, int32_t *acc_nodes,
              int32_t *acc_tokens, int32_t *bonus)
{
    const int P = B + 1;
    for (int r = 0; r < R; ++r) {
        const int32_t *ar = a + (int64_t)r * P;
        const int32_t *tok = tree_tokens + (int64_t)r * B;
        const int32_t *par = parents + (int64_t)r * P;
        int32_t *an = acc_nodes + (int64_t)r * L;
        int32_t *at = acc_tokens + (int64_t)r * (L + 1);
        for (int j = 0; j < L; ++j)
            an[j] = -1;
        for (int j = 0; j <= L; ++j)
            at[j] = -1;
        int cur = 0, n = 0;
        for (;;) {
            const int32_t want = ar[cur];
            int found = -1;
            for (int c = 1; c <= n_nodes[r]; ++c)
                if (par[c] == cur && tok[c - 1] == want) {
                    found = c;
                    break;
                }
            if (found < 0 || n >= L) {
                bonus[r] = want;
                break;
            }
            an[n] = found;
            at[n] = want;
            ++n;
            cur = found;
        }
        at[n] = bonus[r];
        acc_len[r] = n + 1;
    }
}

/* ------------------------------------------------------------------------
 * Step 5c: KV compaction to the accepted path [DDTX section 5,
 * "compact_cache keeps only the accepted path's cache"; SPARK, conclusion
 * (the C++ KV compaction kernel)].
 * Reading: this round's tree keys and values are inputs k_tree, v_tree
 * [R, P, Hkv, d]. The root goes to sequence slot ctx, the accepted node at
 * path depth j to slot ctx + j; slot s lives in page block_table[r][s/page]
 * at row s % page. Afterwards ctx_lens[r] grows by acc_len[r].
 * ---------------------------------------------------------------------- */
int orc_compact(uint16_t *k_cache, uint16_t *v_cache, const int32_t *block_table, int max_pages,
                int64_t num_pages, int32_t *ctx_lens, const uint16_t *k_tree,
                const uint16_t *v_tree, const int32_t *acc_nodes, const int32_t *acc_len, int R,
                int P, int L, int Hkv, int d, int page)
{
    int flags = 0;
    const int64_t rowlen = (int64_t)Hkv * d;
    for (int r = 0; r < R; ++r) {
        const int ctx = ctx_lens[r];
        const int n_acc = acc_len[r] - 1;
        for (int j = 0; j <= n_acc; ++j) {
            const int node = (j == 0) ? 0 : acc_nodes[(int64_t)r * L + j - 1];
            const int slot = ctx + j;
            const int pidx = slot / page;
            if (pidx >= max_pages) {
                flags |= ORC_BAD_PAGE;
                continue;
            }
            const int32_t pg = block_table[(int64_t)r * max_pages + pidx];
            if (pg < 0 || pg >= num_pages) {
                flags |= ORC_BAD_PAGE;
                continue;
            }
            const int64_t dst = ((int64_t)pg * page + slot % page) * rowlen;
            const int64_t src = ((int64_t)r * P + node) * rowlen;
            memcpy(k_cache + dst, k_tree + src, sizeof(uint16_t) * (size_t)rowlen);
            memcpy(v_cache + dst, v_tree + src, sizeof(uint16_t) * (size_t)rowlen);
        }
        ctx_lens[r] = ctx + 1 + n_acc;
    }
    return flags;
}

/* number of threads OpenMP will use (1 when built without OpenMP) */
int orc_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ------------------------------------------------------------------------
 * NEXT row 1: the parent-conditioned tree ["Robot2050/TreeSpark", items 1
 * and 2: one backbone pass gives per-depth logits l_d; a first-order Markov
 * head specialises depth d to a parent token, z_d(u) = l_d + W e(t_u);
 * trees grow by per-parent top-k expansion with joint path-score frontier
 * pruning, and are packed to N non-root nodes by global top-N].
 *
 * Readings (the page gives the policy, not its arithmetic):
 *   - a parent's children are the k largest z_d(u) (equal values: lower
 *     token id first); a child's path score is S(u) + lp with
 *     lp = z - logsumexp(z) in fp64, S(root) = 0;
 *   - depth d's candidates are all children of depth d-1's frontier, in
 *     creation order (frontier slot, then child rank); the frontier of
 *     depth d is its F best candidates by (S desc, creation order asc);
 *     depth 1's frontier parent is the root (the anchor token);
 *   - packing takes the N best candidates of all depths by (S desc, depth
 *     asc, creation order asc), which is prefix-closed (lp <= 0, a parent
 *     sorts before its children); node n is the n-th of them.
 *   With k = F = 4 and 7 depths the candidates number 4 + 6 * 16 = 100,
 *   the page's "up to 100 candidates before packing".
 * ---------------------------------------------------------------------- */
typedef struct {
    double S;
    int32_t depth, order, parent_cand, token;
} cond_cand;

static int cond_prune_cmp(const void *pa, const void *pb)
{
    const cond_cand *a = (const cond_cand *)pa, *b = (const cond_cand *)pb;
    if (a->S != b->S)
        return a->S > b->S ? -1 : 1;
    return (a->order > b->order) - (a->order < b->order);
}

static int cond_pack_cmp(const void *pa, const void *pb)
{
    const cond_cand *a = (const cond_cand *)pa, *b = (const cond_cand *)pb;
    if (a->S != b->S)
        return a->S > b->S ? -1 : 1;
    if (a->depth != b->depth)
        return a->depth < b->depth ? -1 : 1;
    return (a->order > b->order) - (a->order < b->order);
}

/* z = l + W e(tok) for one parent, its log-partition and top-k */
static void cond_parent(const void *ell_row, int ell_dtype, const void *W, const void *E, int w_dtype,
                        int64_t V, int H, int tok, int k, double *zbuf, double *lp, int32_t *ids)
{
    double m = -INFINITY;
    for (int64_t v = 0; v < V; ++v) {
        double b = 0.0;
        for (int h = 0; h < H; ++h)
            b += widen(W, w_dtype, v * H + h) * widen(E, w_dtype, (int64_t)tok * H + h);
        const double z = widen(ell_row, ell_dtype, v) + b;
        zbuf[v] = z;
        if (z > m)
            m = z;
    }
    double s = 0.0;
    for (int64_t v = 0; v < V; ++v)
        s += exp(zbuf[v] - m);
    const double logz = m + log(s);
    for (int j = 0; j < k; ++j) {
        ids[j] = -1;
        lp[j] = -INFINITY;
    }
    for (int64_t v = 0; v < V; ++v) {  /* insertion: value desc, lower id first */
        const double z = zbuf[v];
        if (ids[k - 1] >= 0 && !(z > lp[k - 1]))
            continue;
        int j = k - 1;
        while (j > 0 && (ids[j - 1] < 0 || z > lp[j - 1])) {
            lp[j] = lp[j - 1];
            ids[j] = ids[j - 1];
            --j;
        }
        lp[j] = z;
        ids[j] = (int32_t)v;
    }
    for (int j = 0; j < k; ++j)
        lp[j] -= logz;
}

/*
 * ell [R, D, V] (dtype as widen), W and E [V, H] (w_dtype), anchors [R].
 * Outputs (P = N + 1): tree_tokens [R, N], parents / depths [R, P] (root 0,
 * parents[0] = -1), node_S [R, P], n_nodes [R]; optional per-parent lists
 * cand_lp / cand_ids [R, D, F, k] and the parent token of each frontier slot
 * frontier_tok [R, D, F] (-1 where a depth has fewer parents).
 * replay_lp / replay_ids [R, D, F, k], when not NULL, replace the computed
 * per-parent lists (the frontier and packing logic then runs on them).
 */
int orc_cond_tree(const void *ell, int ell_dtype, const void *W, const void *E, int w_dtype,
                  const int32_t *anchors, int R, int D, int64_t V, int H, int k, int F, int N,
                  const double *replay_lp, const int32_t *replay_ids, int32_t *tree_tokens,
                  int32_t *parents, int32_t *depths, double *node_S, int32_t *n_nodes,
                  double *cand_lp, int32_t *cand_ids, int32_t *frontier_tok)
{
    if (R < 1 || D < 1 || V < 1 || k < 1 || k > V || F < 1 || N < 1 || (replay_lp == NULL && H < 1))
        return ORC_BAD_ARG;
    const int P = N + 1;
    const int64_t cmax = (int64_t)k + (int64_t)(D - 1) * F * k;
#pragma omp parallel for schedule(dynamic, 1)
    for (int r = 0; r < R; ++r) {
        cond_cand *cand = (cond_cand *)malloc(sizeof(cond_cand) * (size_t)cmax);
        cond_cand *tmp = (cond_cand *)malloc(sizeof(cond_cand) * (size_t)(F * k + 1));
        int32_t *front = (int32_t *)malloc(sizeof(int32_t) * (size_t)F);  /* candidate index, -1 root */
        double *zbuf = replay_lp ? NULL : (double *)malloc(sizeof(double) * (size_t)V);
        double *lp = (double *)malloc(sizeof(double) * (size_t)k);
        int32_t *ids = (int32_t *)malloc(sizeof(int32_t) * (size_t)k);
        int nf = 1, nc = 0;
        front[0] = -1;
        for (int d = 1; d <= D; ++d) {
            const int first = nc;
            for (int f = 0; f < F; ++f) {
                const int64_t slot = ((int64_t)r * D + (d - 1)) * F + f;
                if (frontier_tok)
                    frontier_tok[slot] = (f < nf) ? (front[f] < 0 ? anchors[r] : cand[front[f]].token) : -1;
                if (f >= nf) {
                    if (cand_lp)
                        for (int j = 0; j < k; ++j) {
                            cand_lp[slot * k + j] = -INFINITY;
                            cand_ids[slot * k + j] = -1;
                        }
                    continue;
                }
                const int u = front[f];
                const int tok = (u < 0) ? anchors[r] : cand[u].token;
                const double Su = (u < 0) ? 0.0 : cand[u].S;
                if (replay_lp) {
                    for (int j = 0; j < k; ++j) {
                        lp[j] = replay_lp[slot * k + j];
                        ids[j] = replay_ids[slot * k + j];
                    }
                } else {
                    const char *row = (const char *)ell +
                                      (((int64_t)r * D + (d - 1)) * V) * (ell_dtype == 1 ? 2 : ell_dtype == 0 ? 4 : 8);
                    cond_parent(row, ell_dtype, W, E, w_dtype, V, H, tok, k, zbuf, lp, ids);
                }
                for (int j = 0; j < k; ++j) {
                    if (cand_lp) {
                        cand_lp[slot * k + j] = lp[j];
                        cand_ids[slot * k + j] = ids[j];
                    }
                    cond_cand *c = &cand[nc];
                    c->S = Su + lp[j];
                    c->depth = d;
                    c->order = nc;
                    c->parent_cand = u;
                    c->token = ids[j];
                    ++nc;
                }
            }
            /* frontier of the next depth: the F best of this depth's candidates */
            const int nd = nc - first;
            memcpy(tmp, cand + first, sizeof(cond_cand) * (size_t)nd);
            qsort(tmp, (size_t)nd, sizeof(cond_cand), cond_prune_cmp);
            nf = nd < F ? nd : F;
            for (int f = 0; f < nf; ++f)
                front[f] = tmp[f].order;
        }
        /* packing: the N best of all candidates */
        cond_cand *all = (cond_cand *)malloc(sizeof(cond_cand) * (size_t)nc);
        memcpy(all, cand, sizeof(cond_cand) * (size_t)nc);
        qsort(all, (size_t)nc, sizeof(cond_cand), cond_pack_cmp);
        const int n = nc < N ? nc : N;
        int32_t *node_of = (int32_t *)malloc(sizeof(int32_t) * (size_t)nc);
        for (int i = 0; i < nc; ++i)
            node_of[i] = -1;
        int32_t *tok = tree_tokens + (int64_t)r * N;
        int32_t *par = parents + (int64_t)r * P;
        int32_t *dep = depths + (int64_t)r * P;
        double *ns = node_S + (int64_t)r * P;
        for (int j = 0; j < N; ++j)
            tok[j] = -1;
        for (int j = 0; j < P; ++j) {
            par[j] = -1;
            dep[j] = -1;
            ns[j] = 0.0;
        }
        dep[0] = 0;
        for (int i = 0; i < n; ++i) {
            const cond_cand *c = &all[i];
            node_of[c->order] = i + 1;
            tok[i] = c->token;
            par[i + 1] = (c->parent_cand < 0) ? 0 : node_of[c->parent_cand];
            dep[i + 1] = c->depth;
            ns[i + 1] = c->S;
        }
        n_nodes[r] = n;
        free(node_of);
        free(all);
        free(ids);
        free(lp);
        free(zbuf);
        free(front);
        free(tmp);
        free(cand);
    }
    return 0;
}

/* One parent's children lists of the parent-conditioned tree, for given
 * (request, depth, parent token) triples: z = l[r, d] + W e(tok), lp = z -
 * logsumexp(z) (fp64), the k largest (equal values: lower id first).
 * lp, ids: [n, k]. */
int orc_cond_parent_lists(const void *ell, int ell_dtype, const void *W, const void *E,
                          int w_dtype, int R, int D, int64_t V, int H, int k, int64_t n,
                          const int32_t *req, const int32_t *depth, const int32_t *tok,
                          double *lp, int32_t *ids)
{
    if (k < 1 || k > V || H < 1)
        return ORC_BAD_ARG;
    const int esz = ell_dtype == 1 ? 2 : ell_dtype == 0 ? 4 : 8;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < n; ++i) {
        double *zbuf = (double *)malloc(sizeof(double) * (size_t)V);
        const char *row = (const char *)ell + (((int64_t)req[i] * D + depth[i]) * V) * esz;
        cond_parent(row, ell_dtype, W, E, w_dtype, V, H, tok[i], k, zbuf, lp + i * k, ids + i * k);
        free(zbuf);
    }
    (void)R;
    return 0;
}

/* ------------------------------------------------------------------------
 * NEXT row 2: the SparklingTree tree built from a table [SPARK, "Building
 * SparklingTree", Steps 1-6, and "Solving the candidate tree construction":
 * a top-C prefilter of every depth's logits, then a precomputed table of the
 * Markov head's conditional rows that the heap only reads; the head of
 * "First order markov model conditioning": a bias B(x_prev, .) =
 * W1[x_prev] W2 on the next position's logits, written here as
 *   z_d(b | a) = l_d[b] + sum_h W[b][h] E[a][h],   W, E [V, H]].
 *
 * Readings (the page gives the mechanism, not its arithmetic):
 *   - prefilter: depth d keeps its C best tokens of l_d (value desc, lower
 *     id first); every node's children are drawn from them;
 *   - table: for depth d and parent candidate a (the anchor at d = 0, else
 *     the a-th kept token of depth d-1),
 *       lp_d(b | a) = z_d(b | a) - log sum_b' exp z_d(b' | a)
 *     over the C kept tokens b' of depth d (the softmax is re-normalised
 *     over what the prefilter kept); rows a >= 1 of depth 0 are -inf;
 *   - heap: Algorithm 1 with a list per parent: a node's children are its
 *     table row ordered by (lp desc, token id asc); the child of rank j
 *     scores S(parent) + lp; pops go by (S desc, rank tuple asc, a prefix
 *     before its extensions); node n is the n-th pop.
 * ---------------------------------------------------------------------- */

/* the C best entries of one logit row: value desc, lower id first */
static void mk_prefilter_row(const void *ell, int dtype, int64_t base, int64_t V, int C,
                             double *val, int32_t *out)
{
    for (int j = 0; j < C; ++j) {
        val[j] = -INFINITY;
        out[j] = -1;
    }
    for (int64_t v = 0; v < V; ++v) {
        const double x = widen(ell, dtype, base + v);
        if (out[C - 1] >= 0 && !(x > val[C - 1]))
            continue;
        int j = C - 1;
        while (j > 0 && (out[j - 1] < 0 || x > val[j - 1])) {
            val[j] = val[j - 1];
            out[j] = out[j - 1];
            --j;
        }
        val[j] = x;
        out[j] = (int32_t)v;
    }
}

/*
 * ell [R, L, V] (dtype as widen), W and E [V, H] (w_dtype), anchors [R].
 * Outputs: cand [R, L, C] the kept tokens of every depth (best first) and
 * tab [R, L, C, C]: tab[r][d][a][b] = lp_d(b | a).
 */
int orc_markov_table(const void *ell, int ell_dtype, const void *W, const void *E, int w_dtype,
                     const int32_t *anchors, int R, int L, int64_t V, int H, int C,
                     int32_t *cand, double *tab)
{
    if (R < 1 || L < 1 || L > ORC_LMAX || C < 1 || C > V || H < 1)
        return ORC_BAD_ARG;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t rd = 0; rd < (int64_t)R * L; ++rd) {
        double *val = (double *)malloc(sizeof(double) * (size_t)C);
        mk_prefilter_row(ell, ell_dtype, rd * V, V, C, val, cand + rd * C);
        free(val);
    }
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t rda = 0; rda < (int64_t)R * L * C; ++rda) {
        const int64_t rd = rda / C;
        const int a = (int)(rda % C);
        const int r = (int)(rd / L), d = (int)(rd % L);
        double *row = tab + rda * C;
        const int parent = (d == 0) ? (a == 0 ? anchors[r] : -1)
                                    : cand[((int64_t)r * L + d - 1) * C + a];
        if (parent < 0 || parent >= V) {
            for (int b = 0; b < C; ++b)
                row[b] = -INFINITY;
            continue;
        }
        double m = -INFINITY;
        for (int b = 0; b < C; ++b) {
            const int tok = cand[rd * C + b];
            double bias = 0.0;
            for (int h = 0; h < H; ++h)
                bias += widen(W, w_dtype, (int64_t)tok * H + h) * widen(E, w_dtype, (int64_t)parent * H + h);
            row[b] = widen(ell, ell_dtype, rd * V + tok) + bias;
            if (row[b] > m)
                m = row[b];
        }
        double s = 0.0;
        for (int b = 0; b < C; ++b)
            s += exp(row[b] - m);
        const double logz = m + log(s);
        for (int b = 0; b < C; ++b)
            row[b] -= logz;
    }
    return 0;
}

/* order of one table row: candidate indices by (lp desc, token id asc) */
static void mk_sort_row(const double *row, const int32_t *toks, int C, int32_t *order)
{
    for (int j = 0; j < C; ++j) {
        int32_t b = j;
        int i = j;
        while (i > 0) {
            const int32_t c = order[i - 1];
            const int before = row[b] > row[c] || (row[b] == row[c] && toks[b] < toks[c]);
            if (!before)
                break;
            order[i] = c;
            --i;
        }
        order[i] = b;
    }
}

/*
 * cand [R, L, C], tab [R, L, C, C] (lp, fp64; the GPU's fp32 values widen
 * exactly). Outputs per request (P = B + 1): tree_tokens [R, B],
 * parents / depths [R, P] (root 0, parents[0] = -1, depth 0), node_S [R, P],
 * node_cand [R, P] (each node's index into its depth's kept tokens, -1 for
 * the root) and n_nodes [R].
 */
int orc_markov_tree(const int32_t *cand, const double *tab, int R, int L, int C, int B,
                    int32_t *tree_tokens, int32_t *parents, int32_t *depths, double *node_S,
                    int32_t *node_cand, int32_t *n_nodes)
{
    if (R < 1 || L < 1 || L > ORC_LMAX || C < 1 || B < 1)
        return ORC_BAD_ARG;
    const int P = B + 1;
#pragma omp parallel for schedule(dynamic, 1)
    for (int r = 0; r < R; ++r) {
        int32_t *tok = tree_tokens + (int64_t)r * B;
        int32_t *par = parents + (int64_t)r * P;
        int32_t *dep = depths + (int64_t)r * P;
        double *ns = node_S + (int64_t)r * P;
        int32_t *nc = node_cand + (int64_t)r * P;
        for (int j = 0; j < B; ++j)
            tok[j] = -1;
        for (int j = 0; j < P; ++j) {
            par[j] = -1;
            dep[j] = -1;
            ns[j] = 0.0;
            nc[j] = -1;
        }
        dep[0] = 0;
        /* each node's children: its row and that row's order */
        const double **rows = (const double **)malloc(sizeof(double *) * (size_t)P);
        int32_t *order = (int32_t *)malloc(sizeof(int32_t) * (size_t)P * C);
        heap_ent *heap = (heap_ent *)malloc(sizeof(heap_ent) * (size_t)(2 * B + 4));
        int size = 0, count = 0;
        /* the root's children: depth 0, parent candidate 0 (the anchor) */
        rows[0] = tab + (((int64_t)r * L + 0) * C + 0) * C;
        mk_sort_row(rows[0], cand + ((int64_t)r * L + 0) * C, C, order);
        if (rows[0][order[0]] > -INFINITY) {
            heap_ent e;
            memset(&e, 0, sizeof e);
            e.parent_S = 0.0;
            e.S = rows[0][order[0]];
            e.ranks[0] = 0;
            e.len = 1;
            e.parent = 0;
            heap_push(heap, &size, &e);
        }
        while (size > 0 && count < B) {
            heap_ent e = heap_pop(heap, &size);
            const int depth = e.len, j = e.ranks[depth - 1], pn = e.parent;
            const int b = order[(int64_t)pn * C + j];
            const int node = count + 1;
            tok[count] = cand[((int64_t)r * L + depth - 1) * C + b];
            par[node] = pn;
            dep[node] = depth;
            ns[node] = e.S;
            nc[node] = b;
            ++count;
            if (j + 1 < C) {
                const double lp = rows[pn][order[(int64_t)pn * C + j + 1]];
                if (lp > -INFINITY) {
                    heap_ent s = e;
                    s.ranks[depth - 1] = j + 1;
                    s.S = e.parent_S + lp;
                    heap_push(heap, &size, &s);
                }
            }
            if (depth < L) {
                rows[node] = tab + (((int64_t)r * L + depth) * C + b) * C;
                mk_sort_row(rows[node], cand + ((int64_t)r * L + depth) * C, C,
                            order + (int64_t)node * C);
                const double lp = rows[node][order[(int64_t)node * C]];
                if (lp > -INFINITY) {
                    heap_ent c = e;
                    c.ranks[depth] = 0;
                    c.len = depth + 1;
                    c.parent = node;
                    c.parent_S = e.S;
                    c.S = e.S + lp;
                    heap_push(heap, &size, &c);
                }
            }
        }
        n_nodes[r] = count;
        free(heap);
        free(order);
        free(rows);
    }
    return 0;
}

/*
 * Second, independent construction for one request of a small table: list
 * every prefix of depth 1..L over every rank, score it left to right through
 * the per-parent orders, sort the whole list by (S desc, rank tuple asc,
 * shorter first) and keep the first B [DDTX section 3, Prop. 2, with each
 * parent's own list]. Returns the number of prefixes, or -1 above
 * max_prefixes.
 */
int64_t orc_markov_tree_bruteforce(const int32_t *cand, const double *tab, int L, int C, int B,
                                   int64_t max_prefixes, int32_t *tree_tokens, int32_t *parents,
                                   int32_t *depths, double *node_S, int32_t *n_nodes)
{
    if (L < 1 || L > ORC_LMAX || C < 1 || B < 1)
        return -1;
    int64_t total = 0, layer = 1;
    for (int d = 1; d <= L; ++d) {
        layer *= C;
        total += layer;
        if (total > max_prefixes)
            return -1;
    }
    /* the order of every row of the table */
    int32_t *order = (int32_t *)malloc(sizeof(int32_t) * (size_t)L * C * C);
    for (int d = 0; d < L; ++d)
        for (int a = 0; a < C; ++a)
            mk_sort_row(tab + ((int64_t)d * C + a) * C, cand + (int64_t)d * C, C,
                        order + ((int64_t)d * C + a) * C);
    pref_ent *all = (pref_ent *)calloc((size_t)total, sizeof(pref_ent));
    int32_t *last_b = (int32_t *)calloc((size_t)total, sizeof(int32_t));
    int64_t n = 0;
    int32_t digits[ORC_LMAX];
    for (int d = 1; d <= L; ++d) {
        for (int i = 0; i < d; ++i)
            digits[i] = 0;
        for (;;) {
            double S = 0.0;
            int a = 0, b = -1, ok = 1;
            for (int i = 0; i < d; ++i) {
                b = order[((int64_t)i * C + a) * C + digits[i]];
                const double lp = tab[((int64_t)i * C + a) * C + b];
                if (!(lp > -INFINITY)) {
                    ok = 0;
                    break;
                }
                S = S + lp;
                a = b;
            }
            if (ok) {
                pref_ent *p = &all[n];
                p->len = d;
                p->S = S;
                for (int i = 0; i < d; ++i)
                    p->ranks[i] = digits[i];
                last_b[n] = cand[(int64_t)(d - 1) * C + b];
                ++n;
            }
            int i = d - 1;
            while (i >= 0 && ++digits[i] == C) {
                digits[i] = 0;
                --i;
            }
            if (i < 0)
                break;
        }
    }
    /* sort indices by the prefix order, keeping each prefix's token */
    int64_t *idx = (int64_t *)malloc(sizeof(int64_t) * (size_t)(n > 0 ? n : 1));
    pref_ent *sorted = (pref_ent *)malloc(sizeof(pref_ent) * (size_t)(n > 0 ? n : 1));
    for (int64_t i = 0; i < n; ++i)
        idx[i] = i;
    /* insertion sort: n is small here */
    for (int64_t i = 1; i < n; ++i) {
        const int64_t x = idx[i];
        int64_t j = i;
        while (j > 0 && pref_cmp(&all[x], &all[idx[j - 1]]) < 0) {
            idx[j] = idx[j - 1];
            --j;
        }
        idx[j] = x;
    }
    for (int64_t i = 0; i < n; ++i)
        sorted[i] = all[idx[i]];
    const int P = B + 1;
    const int take = (int)(n < B ? n : B);
    for (int j = 0; j < B; ++j)
        tree_tokens[j] = -1;
    for (int j = 0; j < P; ++j) {
        parents[j] = -1;
        depths[j] = -1;
        node_S[j] = 0.0;
    }
    depths[0] = 0;
    for (int j = 0; j < take; ++j) {
        const pref_ent *p = &sorted[j];
        const int node = j + 1;
        tree_tokens[j] = last_b[idx[j]];
        depths[node] = p->len;
        node_S[node] = p->S;
        int parent = -1;
        if (p->len == 1) {
            parent = 0;
        } else {
            for (int q = 0; q < j; ++q) {
                const pref_ent *c = &sorted[q];
                if (c->len != p->len - 1)
                    continue;
                int same = 1;
                for (int i = 0; i < c->len; ++i)
                    if (c->ranks[i] != p->ranks[i]) {
                        same = 0;
                        break;
                    }
                if (same) {
                    parent = q + 1;
                    break;
                }
            }
        }
        parents[node] = parent;
    }
    *n_nodes = take;
    free(sorted);
    free(idx);
    free(last_b);
    free(all);
    free(order);
    return n;
}

/* ------------------------------------------------------------------------
 * NEXT row 3: stochastic verification of a drafted chain at temperature 1
 * ["DSpark Speculative Decoding Explained: Block Drafting and Confidence
 * Checks", the probability rule and its toy: keep the k-th guess x_k with
 * probability min(1, p_k(x_k) / q_k(x_k)); at the first rejected guess draw a
 * replacement from the leftover max(0, p_k - q_k) and drop the rest; if every
 * guess survives, draw a bonus token from the target's next distribution].
 *
 * The random numbers are inputs: u[k] decides guess k (kept iff
 * u[k] < min(1, p/q)); r draws the replacement or bonus token by inverse CDF
 * over the vocabulary in index order: the first index whose running sum of
 * weights exceeds r times their total (the rule of a cumulative-weights
 * bisection). Sums run left to right in fp64.
 *
 * orc_verify_chain: p [L+1, V] and q [L, V] as explicit probabilities (rows
 * need not be normalised: weights), one request. Writes the committed tokens
 * to out[0..n) and returns n (accepted guesses + 1).
 * ---------------------------------------------------------------------- */
static int draw_index(const double *w, int64_t V, double r)
{
    double total = 0.0;
    for (int64_t v = 0; v < V; ++v)
        total += w[v];
    const double x = r * total;
    double cum = 0.0;
    int64_t last = -1;
    for (int64_t v = 0; v < V; ++v) {
        cum += w[v];
        if (w[v] > 0.0)
            last = v;
        if (cum > x)
            return (int)v;
    }
    return (int)last; /* only when rounding left x at the total */
}

int orc_verify_chain(const double *p, const double *q, const int32_t *tokens, const double *u,
                     double r, int L, int64_t V, int32_t *out)
{
    if (L < 0 || V < 1)
        return -1;
    double *w = (double *)malloc(sizeof(double) * (size_t)V);
    int n = 0;
    for (int k = 0; k < L; ++k) {
        const int x = tokens[k];
        const double pk = p[(int64_t)k * V + x], qk = q[(int64_t)k * V + x];
        const double a = (qk > 0.0) ? (pk / qk < 1.0 ? pk / qk : 1.0) : 1.0;
        if (u[k] < a) {
            out[n++] = x;
            continue;
        }
        for (int64_t v = 0; v < V; ++v) {
            const double d = p[(int64_t)k * V + v] - q[(int64_t)k * V + v];
            w[v] = d > 0.0 ? d : 0.0;
        }
        out[n++] = draw_index(w, V, r);
        free(w);
        return n;
    }
    out[n++] = draw_index(p + (int64_t)L * V, V, r);
    free(w);
    return n;
}

/*
 * The same rule on logits, for R requests: draft [R, L, V] and target
 * [R, L+1, V] (dtype as widen), softmax at temperature 1 in fp64, tokens
 * [R, L], u [R, L], r [R]. Outputs acc_len [R] (accepted guesses + 1) and
 * acc_tokens [R, L+1] (-1 past acc_len).
 * n_guess [R] (may be NULL: L each): request i verifies only its first
 * n_guess[i] guesses (clamped to [0, L]; the prefix a scheduler kept), so
 * when all of those survive the bonus comes from target row n_guess[i].
 */
int orc_accept_stochastic(const void *draft, const void *target, int dtype, const int32_t *tokens,
                          const double *u, const double *r, int R, int L, int64_t V,
                          const int32_t *n_guess, int32_t *acc_len, int32_t *acc_tokens)
{
    if (R < 1 || L < 0 || V < 1)
        return ORC_BAD_ARG;
#pragma omp parallel for schedule(dynamic, 1)
    for (int i = 0; i < R; ++i) {
        double *p = (double *)malloc(sizeof(double) * (size_t)(L + 1) * V);
        double *q = (double *)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1) * V);
        for (int k = 0; k <= L; ++k) {
            const int64_t base = ((int64_t)i * (L + 1) + k) * V;
            double m = -INFINITY;
            for (int64_t v = 0; v < V; ++v) {
                const double z = widen(target, dtype, base + v);
                if (z > m)
                    m = z;
            }
            double s = 0.0;
            for (int64_t v = 0; v < V; ++v) {
                p[(int64_t)k * V + v] = exp(widen(target, dtype, base + v) - m);
                s += p[(int64_t)k * V + v];
            }
            for (int64_t v = 0; v < V; ++v)
                p[(int64_t)k * V + v] /= s;
        }
        for (int k = 0; k < L; ++k) {
            const int64_t base = ((int64_t)i * L + k) * V;
            double m = -INFINITY;
            for (int64_t v = 0; v < V; ++v) {
                const double z = widen(draft, dtype, base + v);
                if (z > m)
                    m = z;
            }
            double s = 0.0;
            for (int64_t v = 0; v < V; ++v) {
                q[(int64_t)k * V + v] = exp(widen(draft, dtype, base + v) - m);
                s += q[(int64_t)k * V + v];
            }
            for (int64_t v = 0; v < V; ++v)
                q[(int64_t)k * V + v] /= s;
        }
        int32_t *out = acc_tokens + (int64_t)i * (L + 1);
        for (int k = 0; k <= L; ++k)
            out[k] = -1;
        int n = n_guess ? n_guess[i] : L;
        n = n < 0 ? 0 : (n > L ? L : n);
        /* the first n guesses: target rows 0..n, draft rows 0..n-1 */
        acc_len[i] = orc_verify_chain(p, q, tokens + (int64_t)i * L, u + (int64_t)i * L, r[i], n, V,
                                      out);
        free(q);
        free(p);
    }
    return 0;
}

/* ------------------------------------------------------------------------
 * The hardware-aware prefix scheduler ["DSpark Speculative Decoding
 * Explained: Block Drafting and Confidence Checks", sections "Survival
 * probability" and "Picking the budget"; the DSpark speculative-decoder
 * post, "Hardware aware prefix scheduler"] (NEXT row 4).
 *
 * conf [R, L]: the chance that guess k of request r survives, given that the
 * guesses before it did. Values outside [0, 1] are clamped; NaN counts as 0
 * and is reported. The survival of slot (r, k) is the product conf[r][0] *
 * ... * conf[r][k], taken in that order in fp64; it cannot rise along a
 * block. Slots are ranked by survival, descending; equal survivals go by
 * position, then request, ascending.
 *
 * Verifying the n best slots (n = 0 .. R*L) is expected to commit R + (their
 * survivals' sum) tokens -- one guaranteed token per request -- at a step
 * cost of cost[n] milliseconds. The chosen n maximises tokens per
 * millisecond; the smallest such n wins a tie, and an n whose cost is not
 * positive (or NaN) is never chosen (n = 0 when none is valid).
 *
 * Outputs: n_keep [R] (request r keeps its first n_keep[r] guesses; the
 * ranking makes the chosen slots a prefix of every block), *n_total, and
 * stats [2] = (the best tokens per ms, the expected tokens); stats may be
 * NULL. Returns ORC_NAN_SEEN when a confidence was NaN.
 * ---------------------------------------------------------------------- */
typedef struct {
    double s;
    int k, r;
} sched_slot;

static int sched_cmp(const void *pa, const void *pb)
{
    const sched_slot *a = (const sched_slot *)pa, *b = (const sched_slot *)pb;
    if (a->s != b->s)
        return a->s > b->s ? -1 : 1;
    if (a->k != b->k)
        return a->k < b->k ? -1 : 1;
    return a->r < b->r ? -1 : (a->r > b->r ? 1 : 0);
}

static double sched_conf(double c, int *nan_seen)
{
    if (c != c) {
        *nan_seen = 1;
        return 0.0;
    }
    return c < 0.0 ? 0.0 : (c > 1.0 ? 1.0 : c);
}

static int sched_cost_ok(double c) { return c == c && c > 0.0; }

int orc_schedule_prefix(const double *conf, int R, int L, const double *cost, int32_t *n_keep,
                        int32_t *n_total, double *stats)
{
    if (R < 0 || L < 1)
        return ORC_BAD_ARG;
    const int N = R * L;
    int nan_seen = 0;
    sched_slot *slots = (sched_slot *)malloc(sizeof(sched_slot) * (size_t)(N > 0 ? N : 1));
    for (int r = 0; r < R; ++r) {
        double s = 1.0;
        for (int k = 0; k < L; ++k) {
            s = s * sched_conf(conf[(int64_t)r * L + k], &nan_seen);
            slots[r * L + k].s = s;
            slots[r * L + k].k = k;
            slots[r * L + k].r = r;
        }
    }
    qsort(slots, (size_t)N, sizeof(sched_slot), sched_cmp);
    /* tokens per ms for every n, the sum growing one slot at a time */
    int best_n = 0;
    double best = -INFINITY, best_tokens = (double)R, sum = 0.0;
    for (int n = 0; n <= N; ++n) {
        if (n > 0)
            sum += slots[n - 1].s;
        if (!sched_cost_ok(cost[n]))
            continue;
        const double theta = ((double)R + sum) / cost[n];
        if (theta > best) {
            best = theta;
            best_n = n;
            best_tokens = (double)R + sum;
        }
    }
    for (int r = 0; r < R; ++r)
        n_keep[r] = 0;
    for (int j = 0; j < best_n; ++j)
        n_keep[slots[j].r] += 1;
    *n_total = best_n;
    if (stats) {
        stats[0] = best == -INFINITY ? 0.0 : best;
        stats[1] = best_tokens;
    }
    free(slots);
    return nan_seen ? ORC_NAN_SEEN : 0;
}

/* Brute force for the pins: the best tokens per ms over EVERY subset of the
 * R*L slots (not only prefixes, no ranking), for R*L <= 20. */
double orc_schedule_bruteforce(const double *conf, int R, int L, const double *cost)
{
    const int N = R * L;
    if (N > 20 || N < 0)
        return NAN;
    double s[20];
    int nan_seen = 0;
    for (int r = 0; r < R; ++r) {
        double p = 1.0;
        for (int k = 0; k < L; ++k) {
            p = p * sched_conf(conf[r * L + k], &nan_seen);
            s[r * L + k] = p;
        }
    }
    double best = -INFINITY;
    for (uint32_t m = 0; m < (1u << N); ++m) {
        double tokens = (double)R;
        int n = 0;
        for (int j = 0; j < N; ++j)
            if (m & (1u << j)) {
                tokens += s[j];
                ++n;
            }
        if (sched_cost_ok(cost[n]) && tokens / cost[n] > best)
            best = tokens / cost[n];
    }
    return best == -INFINITY ? 0.0 : best;
}
