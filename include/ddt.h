/*
 * ddt.h -- C ABI of the GB300 (sm_103a) batched draft-tree round.
 *
 * One round, for R in-flight requests that each hold a block drafter's
 * per-depth marginals, runs
 *   a1 ddt_topk_logprobs   per-depth log-softmax + top-K over the vocabulary
 *   a2 ddt_build_tree      best-first selection of the B most probable prefixes
 *   a3 ddt_build_mask      ancestor bitmask of every tree position
 *   a4 ddt_tree_attention  paged GQA attention of the tree queries
 *   a5 ddt_target_argmax   greedy target token at every tree position
 *   a6 ddt_walk            greedy acceptance walk down the tree
 *   a7 ddt_compact         KV of the accepted path written into the cache
 * and ddt_round chains a1..a7 (ddt_accept chains a5..a7) on one stream
 * with no host synchronisation.
 *
 * Further entry points (declared after the round's):
 *   ddt_build_tree_conditioned / ddt_round_conditioned
 *       TreeSpark's parent-conditioned tree (Markov bias per parent,
 *       per-parent top-k, frontier pruning, top-N packing), and its round
 *   ddt_markov_table / ddt_build_tree_markov / ddt_round_markov
 *       SparklingTree's top-C prefilter, Markov table and the heap over it
 *   ddt_accept_stochastic
 *       stochastic verification of drafted chains at temperature 1, of
 *       every guess or of a per-request prefix
 *   ddt_schedule_prefix
 *       the hardware-aware prefix scheduler (guesses to verify per request;
 *       its output is ddt_accept_stochastic's prefix lengths)
 *   ddt_topk_logprobs_noalloc
 *       a1 without a context
 *
 * Pages the operations follow (title and section):
 *   "SparklingTree: 30-40% faster speculative decoding over DSpark",
 *       "How is the tree actually created?", Steps 1-4.
 *   "DDTree Explained: From Block Diffusion to Optimal Diffusion Draft Trees
 *       for Speculative Decoding", sections 3 (Prop. 1, Prop. 2, Lemma 1),
 *       4 (Algorithm 1) and 5 (implementation highlights).
 *   "Robot2050/TreeSpark", item 4 and the continuous-batching engine
 *       (device-side masks, vectorised acceptance, ragged-batch KV); items
 *       1 and 2 for the parent-conditioned tree.
 *   "SparklingTree ...", "First order markov model conditioning",
 *       "Building SparklingTree" and "Solving the candidate tree
 *       construction" for the table tree.
 *   "DSpark Speculative Decoding Explained: Block Drafting and Confidence
 *       Checks", the probability rule (stochastic verification), "Survival
 *       probability" and "Picking the budget" (the scheduler).
 *
 * Conventions shared by every call
 *   - Pointers are DEVICE pointers unless stated. The caller owns every
 *     input and output buffer; a context owns only its workspace.
 *   - bf16 tensors are passed as uint16_t* holding raw bf16 bit patterns.
 *   - Logit tensors (draft, target) are bf16 or fp32 as the context's
 *     config says; their pointers are const void*.
 *   - All tensors are dense row-major with the shapes given below; no
 *     strides are accepted. Vectorised paths need 16-byte-aligned base
 *     pointers; every other pointer needs its element's alignment (4 bytes
 *     for i32 and f32, 8 for f64). Unaligned ones are rejected with
 *     DDT_EINVAL.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream). Every
 *     call only enqueues work on it and returns; none synchronises the host
 *     except ddt_device_status. One context must not be used by two streams
 *     at once (its workspace is shared by its calls).
 *   - Shape and argument errors return DDT_EINVAL (or DDT_EUNSUPPORTED)
 *     synchronously and enqueue nothing. Launch failures return DDT_ECUDA.
 *     Data errors found on the device (NaN logits, page ids out of range,
 *     malformed parents) never trap: they set bits of a device status word
 *     read with ddt_device_status, and the kernels skip the bad access.
 *
 * Notation: R requests (R <= R_max), L draft depths, V vocabulary, B budget
 * of non-root tree nodes, K = min(B, V) kept per depth (the config may ask
 * for another K <= V), P = B + 1 tree positions (position 0 is the root, the
 * round's bonus token), W = ceil(P / 32) mask words, Hq query heads, Hkv KV
 * heads (Hq % Hkv == 0), d head dimension, page_size tokens per KV page.
 */
#ifndef DDT_H
#define DDT_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum ddt_status {
    DDT_OK = 0,
    DDT_EINVAL = 1,       /* bad shape, dtype, pointer or alignment; nothing enqueued */
    DDT_EUNSUPPORTED = 2, /* valid request outside what this build implements */
    DDT_ECUDA = 3,        /* a CUDA runtime call failed (see ddt_last_cuda_error) */
    DDT_ENOMEM = 4        /* workspace allocation failed in ddt_create */
} ddt_status;

typedef enum ddt_dtype { DDT_BF16 = 0, DDT_F32 = 1 } ddt_dtype;

/* bits of the device status word (ddt_device_status) */
#define DDT_DEV_NAN_LOGITS 0x1 /* a NaN reached top-K or argmax */
#define DDT_DEV_BAD_PAGE 0x2   /* a block-table entry was outside [0, num_pages) */
#define DDT_DEV_BAD_TREE 0x4   /* parents/n_nodes/acc arrays out of range */
#define DDT_DEV_TIMEOUT 0x8    /* a bounded on-device wait gave up (the kernel wound down) */

typedef struct ddt_config {
    int32_t R_max;             /* most requests a call may carry (1..2048) */
    int32_t L;                 /* draft depths per request (1..18) */
    int32_t V;                 /* vocabulary size (at most 64 chunks of a1: 1048576 bf16,
                                  524288 fp32 draft logits) */
    int32_t B;                 /* non-root tree nodes (1..127) */
    int32_t K;                 /* per-depth top-K; 0 selects min(B, V) */
    int32_t Hq, Hkv, d;        /* attention heads and head dim (d = 128 or 64); a4 needs
                                  Hq / Hkv in {1, 2, 4, 8, 16} */
    int32_t page_size;         /* tokens per KV page: a power of two, at least 16 */
    int32_t max_pages_per_req; /* row length of block_table */
    int64_t num_pages;         /* pages in the KV pool (bounds checks); at most
                                  (2^31 - 1) / page_size, since a4 addresses the
                                  pool's token rows with 32-bit coordinates */
    int32_t draft_dtype;       /* ddt_dtype of draft logits */
    int32_t target_dtype;      /* ddt_dtype of target logits */
    /* parent-conditioned tree (ddt_build_tree_conditioned); 0 = not used */
    int32_t markov_dim;        /* H of the Markov head W, E [V, H]: 64..256, multiple of 64 */
    int32_t frontier;          /* F: parents kept per depth (1..8); F * K <= 32 */
    /* SparklingTree table tree (ddt_markov_table, ddt_build_tree_markov); 0 =
     * not used. C: tokens kept per depth by the prefilter, 1..128 and <= V;
     * needs markov_dim > 0 and bf16 draft logits. */
    int32_t prefilter;
} ddt_config;

typedef struct ddt_ctx ddt_ctx; /* opaque */

/* Validate cfg, pick the current CUDA device, allocate the workspace
 * (ddt_workspace_bytes) and return a context in *out. DDT_EINVAL for a bad
 * config, DDT_ENOMEM if the workspace cannot be allocated. */
ddt_status ddt_create(const ddt_config *cfg, ddt_ctx **out);

/* Free the workspace and the context (waits for nothing: the caller makes
 * sure no enqueued call still runs). NULL is ignored. */
void ddt_destroy(ddt_ctx *ctx);

/* Device bytes a context with this config allocates (0 for a bad config). */
size_t ddt_workspace_bytes(const ddt_config *cfg);

/* a1 -- "SparklingTree ...", Step 1; "DDTree Explained ...", Lemma 1.
 * draft_logits [R, L, V] (draft_dtype). For each (request, depth) row:
 * logZ = log sum_v exp(z_v); the K largest logits in order value
 * descending, equal values by lower token id; top_lp = z - logZ (fp32),
 * top_ids their token ids. Outputs top_lp [R, L, K] f32, top_ids [R, L, K]
 * i32. NaN logits set DDT_DEV_NAN_LOGITS. */
ddt_status ddt_topk_logprobs(ddt_ctx *ctx, const void *draft_logits, int32_t R, float *top_lp,
                             int32_t *top_ids, void *stream);

/* a2 -- "DDTree Explained ...", section 4, Algorithm 1; "SparklingTree ...",
 * Step 3. From top_lp/top_ids [R, L, K], pops the B prefixes with the
 * largest S (the fp64 sum of their per-depth log-probs, parent score plus
 * own log-prob); equal S goes to the lexicographically smaller rank tuple.
 * Node n (1..B) is the n-th pop. Outputs:
 *   tree_tokens [R, B]  token of node n at index n-1 (-1 if unused)
 *   parents     [R, P]  parent node of node n; parents[0] = -1
 *   depths      [R, P]  depth of node n (1..L); depths[0] = 0; -1 if unused
 *   n_nodes     [R]     nodes built (B unless the prefix space is smaller)
 * mask (may be NULL): when given, the a3 ancestor mask is written as well
 * ([R, P, W] u32, same contents as ddt_build_mask). */
ddt_status ddt_build_tree(ddt_ctx *ctx, const float *top_lp, const int32_t *top_ids, int32_t R,
                          int32_t *tree_tokens, int32_t *parents, int32_t *depths,
                          int32_t *n_nodes, uint32_t *mask, void *stream);

/* a3 -- "SparklingTree ...", Step 4; "DDTree Explained ...", section 5.
 * mask [R, P, W] u32: bit j of word w of row (r, i) is set iff position
 * 32w + j is the root, an ancestor of i, or i itself. Rows past n_nodes are
 * zero. Bad parents set DDT_DEV_BAD_TREE. */
ddt_status ddt_build_mask(ddt_ctx *ctx, const int32_t *parents, const int32_t *n_nodes,
                          int32_t R, uint32_t *mask, void *stream);

/* a4 -- "SparklingTree ...", Step 4 and the verification discussion;
 * "DDTree Explained ...", sections 5 and 8 (ancestor-only mask, GQA).
 * Query row (r, i, h) attends, with scale 1/sqrt(d), to the ctx_lens[r]
 * cached tokens of KV head h / (Hq / Hkv) and to the tree positions set in
 * mask row (r, i); softmax in fp32, bf16 inputs, fp32 accumulation, fp32
 * output (a bf16 output alone would round values in [2, 4) by up to 0.0078).
 *   q               [R, P, Hq, d] bf16;  out [R, P, Hq, d] f32
 *   k_tree, v_tree  [R, P, Hkv, d] bf16 (this round's tree keys/values)
 *   k_cache,v_cache [num_pages, page_size, Hkv, d] bf16
 *   block_table     [R, max_pages_per_req] i32: page of token t is
 *                   block_table[r][t / page_size], row t % page_size
 *   ctx_lens        [R] i32, mask [R, P, W] u32
 * Page ids out of range set DDT_DEV_BAD_PAGE and are read as zeros. One
 * tcgen05 tensor-core kernel serves d = 64 and d = 128. Keys and values are
 * read in blocks of 16 tokens, so the rows of a request's last page past
 * ctx_lens are read and masked out: they must hold finite values (zeros, or
 * earlier rounds' keys and values). */
ddt_status ddt_tree_attention(ddt_ctx *ctx, const uint16_t *q, const uint16_t *k_tree,
                              const uint16_t *v_tree, const uint16_t *k_cache,
                              const uint16_t *v_cache, const int32_t *block_table,
                              const int32_t *ctx_lens, const uint32_t *mask, int32_t R,
                              float *out, void *stream);

/* a5 -- "DDTree Explained ...", section 5 (verifier walk under greedy
 * decoding); "Robot2050/TreeSpark" (vectorised acceptance).
 * target_logits [R, P, V] (target_dtype) -> argmax_out [R, P] i32, the first
 * index of each row's maximum (-0 equals +0). NaN sets DDT_DEV_NAN_LOGITS. */
ddt_status ddt_target_argmax(ddt_ctx *ctx, const void *target_logits, int32_t R,
                             int32_t *argmax_out, void *stream);

/* a6 -- "DDTree Explained ...", section 5, verifier walk; "Robot2050/
 * TreeSpark" item 4. From the root, while a child of the current node
 * carries the target's token argmax[r][cur], accept it and move there;
 * the first unmatched argmax is the new bonus token. Outputs
 *   acc_len    [R]       accepted drafts + 1 (the bonus counts)
 *   acc_nodes  [R, L]    accepted node indices, -1 padded
 *   acc_tokens [R, L+1]  accepted tokens then the bonus, -1 padded
 *   bonus      [R] */
ddt_status ddt_walk(ddt_ctx *ctx, const int32_t *argmax, const int32_t *tree_tokens,
                    const int32_t *parents, const int32_t *n_nodes, int32_t R, int32_t *acc_len,
                    int32_t *acc_nodes, int32_t *acc_tokens, int32_t *bonus, void *stream);

/* a7 -- "DDTree Explained ...", section 5 (compact_cache keeps only the
 * accepted path). Writes the root's tree K/V to sequence slot ctx_lens[r]
 * and the accepted node at path depth j to slot ctx_lens[r] + j, through
 * block_table, then adds acc_len[r] to ctx_lens[r] (in place). The page
 * table must already cover the new slots; entries out of range set
 * DDT_DEV_BAD_PAGE and the row is skipped. */
ddt_status ddt_compact(ddt_ctx *ctx, uint16_t *k_cache, uint16_t *v_cache,
                       const int32_t *block_table, int32_t *ctx_lens, const uint16_t *k_tree,
                       const uint16_t *v_tree, const int32_t *acc_nodes, const int32_t *acc_len,
                       int32_t R, void *stream);

/* a5..a7 in one call. argmax_out may be NULL. */
ddt_status ddt_accept(ddt_ctx *ctx, const void *target_logits, const int32_t *tree_tokens,
                      const int32_t *parents, const int32_t *n_nodes, int32_t R,
                      int32_t *argmax_out, int32_t *acc_len, int32_t *acc_nodes,
                      int32_t *acc_tokens, int32_t *bonus, uint16_t *k_cache, uint16_t *v_cache,
                      const int32_t *block_table, const uint16_t *k_tree, const uint16_t *v_tree,
                      int32_t *ctx_lens, void *stream);

/* Parent-conditioned tree ("Robot2050/TreeSpark", items 1 and 2): a
 * backbone's per-depth logits l_d (draft_logits [R, L, V], bf16) specialised
 * to each parent token t_u by a first-order Markov head,
 *     z_d(u) = l_d + W e(t_u),        W, E: [V, H] bf16 (H = markov_dim),
 * the K best children of every parent (log-probs of z_d(u); equal values:
 * lower token id first), the F best children of a depth by path score
 * S = S(parent) + lp (fp64; S(root) = 0) as the next depth's parents
 * (frontier), and the B best candidates of all depths by (S desc, depth asc,
 * creation order asc) packed as nodes 1..B -- a prefix-closed tree, written
 * in the layout of ddt_build_tree (root 0 = the anchor token, anchors [R]).
 * The config's L is the number of depths, K the children per parent (<= 8),
 * B the node budget; R * F <= 128.
 * Optional outputs (NULL to skip): cand_lp / cand_ids [R, L, F, K] fp32 /
 * int32, the children lists of each depth's frontier slots (-inf / -1 past
 * the frontier), and frontier_tok [R, L, F], the parent token of each slot.
 * mask [R, P, W] (optional) as in ddt_build_tree. DDT_EUNSUPPORTED if the
 * context was not created for this tree (markov_dim == 0) or the limits are
 * exceeded. */
ddt_status ddt_build_tree_conditioned(ddt_ctx *ctx, const void *draft_logits, const uint16_t *W,
                                      const uint16_t *E, const int32_t *anchors, int32_t R,
                                      float *cand_lp, int32_t *cand_ids, int32_t *frontier_tok,
                                      int32_t *tree_tokens, int32_t *parents, int32_t *depths,
                                      int32_t *n_nodes, uint32_t *mask, void *stream);

/* Everything one round reads and writes (shapes as above). */
typedef struct ddt_round_args {
    int32_t R;
    const void *draft_logits;  /* [R, L, V] */
    const void *target_logits; /* [R, P, V] */
    const uint16_t *q;         /* [R, P, Hq, d] */
    const uint16_t *k_tree;    /* [R, P, Hkv, d] */
    const uint16_t *v_tree;    /* [R, P, Hkv, d] */
    uint16_t *k_cache;         /* [num_pages, page_size, Hkv, d], compacted in place */
    uint16_t *v_cache;
    const int32_t *block_table; /* [R, max_pages_per_req] */
    int32_t *ctx_lens;          /* [R], grows by acc_len */
    float *top_lp;              /* [R, L, K] */
    int32_t *top_ids;           /* [R, L, K] */
    int32_t *tree_tokens;       /* [R, B] */
    int32_t *parents;           /* [R, P] */
    int32_t *depths;            /* [R, P] */
    int32_t *n_nodes;           /* [R] */
    uint32_t *mask;             /* [R, P, W] */
    float *attn_out;            /* [R, P, Hq, d] f32 */
    int32_t *target_argmax;     /* [R, P], may be NULL */
    int32_t *acc_len;           /* [R] */
    int32_t *acc_nodes;         /* [R, L] */
    int32_t *acc_tokens;        /* [R, L+1] */
    int32_t *bonus;             /* [R] */
    /* Optional timing hooks (cudaEvent_t, may be NULL): recorded on the
     * round's stream immediately before and after the a4 launch. */
    void *att_event_begin;
    void *att_event_end;
} ddt_round_args;

/* a1..a7 with no host synchronisation. All work is ordered after what was
 * already enqueued on `stream`, and everything later on `stream` is ordered
 * after the whole round. Inside, a1..a3 run on a highest-priority stream of
 * the context's own and a5 (which needs only the target logits) on a
 * lowest-priority one, concurrently; a4 waits for both on `stream`, then
 * a6/a7 follow there. */
ddt_status ddt_round(ddt_ctx *ctx, const ddt_round_args *args, void *stream);

/* The parent-conditioned round -- "Robot2050/TreeSpark", items 1 and 2 (the
 * tree from one backbone pass with a first-order Markov head), then the same
 * verification as ddt_round: the tree and its mask come from
 * ddt_build_tree_conditioned on args->draft_logits (the backbone's per-depth
 * logits l_d [R, L, V], bf16) with the head W, E [V, markov_dim] bf16 and the
 * roots anchors [R] (the bonus tokens); a4..a7 follow as in ddt_round, with
 * a5 beside the tree on a lowest-priority stream. args->top_lp and
 * args->top_ids are not used (may be NULL); the tree has cfg.B nodes at
 * most. Requires markov_dim > 0 (else DDT_EUNSUPPORTED); argument errors as
 * for ddt_round and ddt_build_tree_conditioned. */
ddt_status ddt_round_conditioned(ddt_ctx *ctx, const ddt_round_args *args, const uint16_t *W,
                                 const uint16_t *E, const int32_t *anchors, void *stream);

/* NEXT row 2 -- "SparklingTree: 30-40% faster speculative decoding over
 * DSpark", sections "Solving the candidate tree construction" (a top-k
 * prefilter of every position's logits on the GPU, then a precomputed table
 * of the Markov model's conditional rows that the tree loop only reads) and
 * "Building SparklingTree" (the heap loop), with the Markov head of "First
 * order markov model conditioning" (a bias W1[x_prev] W2 on the next
 * position's logits, here z_d(b | a) = l_d[b] + W[b] . E[a]).
 *
 * ddt_markov_table: for every request r and depth d, cand_ids[r, d, :] are
 * the C = cfg.prefilter largest draft_logits[r, d, :] (bf16 [R, L, V]; value
 * descending, lower id first). tab_lp[r, d, a, b] (f32 [R, L, C, C]) is
 * log-softmax over b of l_d[cand b] + W[cand b] . E[parent a], where parent a
 * is anchors[r] at d = 0 (row a = 0; rows a >= 1 are -inf) and the a-th kept
 * token of depth d - 1 otherwise; the softmax runs over the C kept tokens.
 * W, E: [V, markov_dim] bf16, 16-byte aligned; anchors [R] int32. The
 * products run on the tensor cores (bf16 in, fp32 accumulation). */
ddt_status ddt_markov_table(ddt_ctx *ctx, const void *draft_logits, const uint16_t *W,
                            const uint16_t *E, const int32_t *anchors, int32_t R,
                            int32_t *cand_ids, float *tab_lp, void *stream);

/* ddt_build_tree_markov: Algorithm 1 over the table: a node's children are
 * its row of tab_lp (the root's: row 0 of depth 0; a node with candidate
 * index b at depth d: row b of depth d) in order of (lp descending, token id
 * ascending); a child scores S(parent) + lp in fp64; pops go by (S
 * descending, rank tuple ascending, a prefix before its extensions); node n
 * is the n-th pop. Outputs as ddt_build_tree (tree_tokens [R, B], parents /
 * depths [R, P], n_nodes [R]) and, when mask is not NULL, the ancestor mask
 * [R, P, W] of ddt_build_mask. */
ddt_status ddt_build_tree_markov(ddt_ctx *ctx, const int32_t *cand_ids, const float *tab_lp,
                                 int32_t R, int32_t *tree_tokens, int32_t *parents,
                                 int32_t *depths, int32_t *n_nodes, uint32_t *mask, void *stream);

/* The SparklingTree round: ddt_markov_table into the context's workspace,
 * ddt_build_tree_markov (with the mask), then a4..a7 as in ddt_round, with a5
 * beside the tree on a lowest-priority stream. args->draft_logits are the
 * drafter's per-depth logits; args->top_lp / top_ids are not used. */
ddt_status ddt_round_markov(ddt_ctx *ctx, const ddt_round_args *args, const uint16_t *W,
                            const uint16_t *E, const int32_t *anchors, void *stream);

/* Stochastic verification of a drafted chain at temperature 1 -- "DSpark
 * Speculative Decoding Explained: Block Drafting and Confidence Checks", the
 * probability rule (keep guess k with probability min(1, p_k(x_k) /
 * q_k(x_k)); at the first rejection draw the replacement from max(0, p_k -
 * q_k); when all L guesses survive draw a bonus token from p_L). p and q are
 * the softmax of the target's and the drafter's logits (computed here).
 *   draft_logits  [R, L, V] draft_dtype, device, rows contiguous
 *   target_logits [R, L+1, V] target_dtype, device
 *   draft_tokens  [R, L] i32, the guesses x_0..x_{L-1}
 *   u             [R, L] f32 in [0, 1): guess k is kept iff u[k] < min(1, p/q)
 *                 (q(x) = 0 counts as ratio 1)
 *   r             [R] f32 in [0, 1): the replacement or bonus token is the
 *                 first index (ascending) whose running sum of weights
 *                 exceeds r times the weights' total
 *   n_guess       [R] i32, device, or NULL (L for every request): request i
 *                 verifies only its first n = n_guess[i] guesses (the prefix
 *                 ddt_schedule_prefix kept), so when all n survive the bonus
 *                 comes from target row n. Draft rows k >= n and target rows
 *                 k > n are not read. A value outside [0, L] is clamped into
 *                 it and sets DDT_DEV_BAD_TREE.
 * Outputs: acc_len [R] (kept guesses + 1) and acc_tokens [R, L+1] (the kept
 * guesses, then the drawn token, then -1). The draw is -1 only when every
 * weight is zero (p <= q everywhere after rounding). Guesses outside [0, V)
 * set DDT_DEV_BAD_TREE and count as rejected; NaN logits set
 * DDT_DEV_NAN_LOGITS. Two kernels are enqueued on `stream`, the second as a
 * programmatic dependent launch; calls on one context must not overlap. */
ddt_status ddt_accept_stochastic(ddt_ctx *ctx, const void *draft_logits,
                                 const void *target_logits, const int32_t *draft_tokens,
                                 const float *u, const float *r, int32_t R, int32_t *acc_len,
                                 int32_t *acc_tokens, const int32_t *n_guess, void *stream);

/* The hardware-aware prefix scheduler -- "DSpark Speculative Decoding
 * Explained: Block Drafting and Confidence Checks", sections "Survival
 * probability" and "Picking the budget"; the DSpark post, "Hardware aware
 * prefix scheduler". Decides how many drafted guesses of each request to
 * verify in the next step.
 *   conf    [R, L] f32, device: conf[r][k] is the chance that guess k of
 *           request r survives given that guesses 0..k-1 did. Values are
 *           clamped to [0, 1]; NaN counts as 0 and sets DDT_DEV_NAN_LOGITS.
 *   cost_ms [R*L + 1] f32, device: the step's cost in ms when n guesses are
 *           verified besides the R guaranteed tokens, n = 0..R*L (a table
 *           measured beforehand). An n whose cost is not positive (or NaN)
 *           is never chosen.
 * The survival of slot (r, k) is conf[r][0] * ... * conf[r][k] (fp64). The
 * slots of all requests are ranked by survival, descending (ties: lower k,
 * then lower r first), and n is chosen to maximise (R + the n best
 * survivals' sum) / cost_ms[n] -- expected committed tokens per ms; the
 * smallest n wins a tie, and n = 0 when no cost is valid.
 * Outputs (device): n_keep [R] i32, the guesses request r verifies (always
 * a prefix of its block; it may be passed as ddt_accept_stochastic's n_guess
 * without leaving the device); n_total [1] i32 (may be NULL), the chosen n;
 * stats [2] f64 (may be NULL): the best tokens per ms and the expected
 * committed tokens. Requires R * L <= DDT_SCHED_MAX_SLOTS (else
 * DDT_EUNSUPPORTED). One kernel is enqueued on `stream`: while (R * L) * R
 * <= 2^23, a grid that counts every slot's rank, whose last CTA to finish
 * picks the budget; beyond that, one CTA that sorts the slots. */
#define DDT_SCHED_MAX_SLOTS 8192
ddt_status ddt_schedule_prefix(ddt_ctx *ctx, const float *conf, int32_t R, const float *cost_ms,
                               int32_t *n_keep, int32_t *n_total, double *stats, void *stream);

/* Wait for the context's device to finish all enqueued work, copy the
 * device status word to *host_out (DDT_DEV_* bits) and clear it. */
ddt_status ddt_device_status(ddt_ctx *ctx, int32_t *host_out);

/* Test-only failure detection for the a4 kernel's bounded waits. The pages
 * have no counterpart; the call exists so that a test can drive the timeout
 * path on a GPU without a fault.
 *
 * Arms the context's next a4 launch (ddt_tree_attention, or the attention of
 * one of the round entry points), once: every CTA of that launch starts with
 * one bounded wait on an on-chip barrier that nothing arrives at, limited to
 * wait_cycles SM clock cycles. The wait runs out before the CTA has issued
 * any copy or MMA; the CTA then raises DDT_DEV_TIMEOUT in the device status
 * word, skips its work (the attention output of that launch is undefined),
 * frees its tensor memory and returns. The context stays usable and the next
 * launch is normal. wait_cycles <= 0 disarms. The setting is host state of
 * the context, read and cleared when the next a4 launch is enqueued. */
ddt_status ddt_debug_arm_attention_timeout(ddt_ctx *ctx, int64_t wait_cycles);

/* a1 without a context, for callers that cannot allocate device memory.
 * The pages have no counterpart to this entry point.
 *
 * Who needs it: code that must not call cudaMalloc -- for example a hook or
 * plugin inside a serving engine that owns all device memory and hands its
 * extensions no workspace, or a latency-critical loop that may not risk the
 * device-wide synchronisation an allocation can cause. ddt_create allocates
 * a workspace, so such callers cannot use ddt_topk_logprobs.
 *
 * Same operation, layouts and kernel as ddt_topk_logprobs, for `rows`
 * independent rows of V logits (draft_logits [rows, V], draft_dtype BF16 or
 * F32; top_lp, top_ids [rows, K]). Its scratch (each warp's (max, sum of
 * exp), each 64-logit group's max, each warp's best group keys, a status
 * word) is one fixed array in the library's device memory, about 24 MB, which
 * every GPU that loads libddt.so keeps until the process exits. No call
 * allocates or frees device memory.
 *
 * Limits (DDT_EUNSUPPORTED beyond them, nothing enqueued), with
 * chunks = ceil(V / 16384) for bf16 and ceil(V / 8192) for fp32:
 *   rows <= DDT_NOALLOC_MAX_ROWS, rows * chunks <= DDT_NOALLOC_MAX_ROW_CHUNKS,
 *   chunks * K <= 2048, chunks <= 64, 1 <= K <= min(127, V). Bad pointers or
 *   dtype: DDT_EINVAL.
 * Set-up: every call looks up the array's device address in the calling
 * thread's current CUDA context, so any context works (the primary one, one
 * made with cuCtxCreate, a new one after a device reset). The first call in
 * a context may load the library's module into it, which is not allowed
 * while a stream is being captured: make that first call before any
 * capture. Every call writes the scratch it reads (on `stream`) before
 * reading it, but all calls share the one array: calls that can overlap on
 * the GPU (other streams, other threads) race and corrupt each other's
 * results. NaN logits are not reported by this entry point. */
#define DDT_NOALLOC_MAX_ROWS 4096
#define DDT_NOALLOC_MAX_ROW_CHUNKS 32768
ddt_status ddt_topk_logprobs_noalloc(const void *draft_logits, int32_t draft_dtype, int32_t rows,
                                     int32_t V, int32_t K, float *top_lp, int32_t *top_ids,
                                     void *stream);

/* Static text for a status code. */
const char *ddt_strerror(ddt_status status);

/* The CUDA error code behind the most recent DDT_ECUDA of this thread. */
int32_t ddt_last_cuda_error(void);

#ifdef __cplusplus
}
#endif

#endif /* DDT_H */
