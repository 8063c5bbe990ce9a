// ddt_internal.h -- context layout and kernel launchers shared by the
// translation units of libddt.so. Not part of the public ABI.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "ddt.h"

// ---------------------------------------------------------------- limits
constexpr int DDT_MAX_L = 18;    // rank tuples pack 18 fields of 7 bits into 128 bits
constexpr int DDT_MAX_K = 127;   // rank + 1 must fit a 7-bit field
constexpr int DDT_MAX_B = 127;   // frontier of <= B entries in 4 slots per lane
constexpr int DDT_MAX_P = 128;   // tree positions (B + 1)

// a1: one CTA of TOPK_THREADS reads one chunk of TOPK_THREADS *
// TOPK_VEC_PER_THREAD 16-byte vectors of a row
constexpr int TOPK_THREADS = 256;
constexpr int TOPK_VEC_PER_THREAD = 8;   // 16-byte vectors per thread (one group)
constexpr int TOPK_CTAS_PER_SM = 5;
constexpr int TOPK_MAX_CHUNKS = 64;      // a row's group keys fit 32 KB of shared memory
constexpr int TOPK_CAND_CAP = 2048;      // limit on chunks x K per row

// a5: same chunking as a1
constexpr int AMAX_THREADS = 256;
constexpr int AMAX_VEC_PER_THREAD = 8;

// a4: rows of one partial output (128 main rows plus up to 16 tail rows) and
// the most CTAs of the attention grid (two partial slots each)
constexpr int ATT_ROWS = 144;
constexpr int ATT_MAX_CTAS = 256;
constexpr int ATT_MAX_CTX = 262144;  // tokens of context per request

// parent-conditioned tree: most CTAs of its per-depth GEMM (partials per CTA)
constexpr int CG_GRID_MAX = 256;
constexpr int CG_NP_MAX = 128;  // parents of one depth of the conditioned tree (R * F)

struct ddt_ctx {
    ddt_config cfg;  // with K resolved
    int device;
    int num_sms;
    size_t ws_bytes;
    char *ws;                // one allocation, carved below
    cudaStream_t hi;         // ddt_round: a1..a3 on a highest-priority stream,
    cudaStream_t side;       //   a5 beside them on a lowest-priority one
    cudaEvent_t ev_fork, ev_tree, ev_join, ev_walk;
    int32_t *status;         // device status word
    int64_t debug_att_wait;  // > 0: the next attention launch starts with a wait that runs out (test only)
    // a1 partials
    int tk_nch;              // chunks per row
    uint16_t *tk_gkey;       // [R_max * L, nch * TOPK_THREADS] each group's max (ordered key)
    uint16_t *tk_wtop;       // [R_max * L, nch * TOPK_THREADS / 32, Q] each warp's Q largest keys
    float2 *tk_ms;           // [R_max * L, nch * TOPK_THREADS / 32] each warp's (max, sum of exp)
    // a5 partials
    int am_nch;
    float *am_val;           // [R_max * P, nch]
    int32_t *am_idx;         // [R_max * P, nch]
    // a4 partials of the runs that share boundaries split (two slots per CTA)
    int att_max_items;       // 2 * ATT_MAX_CTAS
    float *att_part_o;       // [max_items, ATT_ROWS, d]
    float2 *att_part_ml;     // [max_items, ATT_ROWS]
    // parent-conditioned tree (markov_dim > 0)
    int cg_grid;             // CTAs of the per-depth GEMM
    float2 *cg_part_ms;      // [R_max * F, cg_grid] (max, sum of exp)
    uint64_t *cg_part_top;   // [R_max * F, cg_grid, 8] top-k keys
    int32_t *cg_fr_tok, *cg_fr_cand, *cg_fr_n;  // [R_max, F], [R_max, F], [R_max]
    double *cg_fr_S;         // [R_max, F]
    double *cg_c_S;          // [R_max, Cmax] candidate scores
    int32_t *cg_c_meta;      // [R_max, Cmax, 3] depth, parent candidate, token
    uint32_t *cg_thr;        // [L, CG_NP_MAX] per-parent lower bounds of the k-th child (value keys)
    float *cg_seed_lp;       // [R_max, L, K] the seeds' log-probs (written by top-K, not read)
    int32_t *cg_seed_ids;    // [R_max, L, K] the draft's top-K columns per depth: bound seeds
    // SparklingTree table tree (prefilter > 0)
    int32_t *mk_cand;        // [R_max, L, C] kept tokens (ddt_round_markov)
    float *mk_tab;           // [R_max, L, C, C] the table (ddt_round_markov)
    // stochastic chain verification
    int sv_nch_d, sv_nch_t, sv_nch_w;  // chunks per draft row, target row, drawn row
    float2 *sv_part_d;       // [R_max * L, sv_nch_d] (max, sum of exp)
    float2 *sv_part_t;       // [R_max * (L + 1), sv_nch_t]
    unsigned *sv_cnt;        // [R_max] arrival counters of the draw (self-resetting)
    float *sv_part_w;        // [R_max, sv_nch_w] chunk totals of the draw's weights
    // prefix scheduler (rank-counting grid)
    uint64_t *ps_rk;         // [DDT_SCHED_MAX_SLOTS] survival bits in ranking order
    int32_t *ps_rid;         // [DDT_SCHED_MAX_SLOTS] their tie ids
    unsigned *ps_arrive;     // arrival counter (self-resetting)
};

// launchers (return the cudaGetLastError of the launch)
cudaError_t launch_topk(const ddt_ctx *c, const void *z, int R, float *top_lp, int32_t *top_ids,
                        cudaStream_t s);
cudaError_t launch_build_tree(const ddt_ctx *c, const float *top_lp, const int32_t *top_ids, int R,
                              int32_t *tree_tokens, int32_t *parents, int32_t *depths,
                              int32_t *n_nodes, uint32_t *mask, cudaStream_t s);
cudaError_t launch_build_mask(const ddt_ctx *c, const int32_t *parents, const int32_t *n_nodes,
                              int R, uint32_t *mask, cudaStream_t s);
cudaError_t launch_argmax_partials(const ddt_ctx *c, const void *t, int R, cudaStream_t s);
cudaError_t launch_argmax_finish(const ddt_ctx *c, int R, int32_t *argmax_out, cudaStream_t s);
cudaError_t launch_walk_compact(const ddt_ctx *c, const int32_t *argmax, bool argmax_from_partials,
                                int32_t *argmax_out, const int32_t *tree_tokens,
                                const int32_t *parents, const int32_t *n_nodes, int R,
                                int32_t *acc_len, int32_t *acc_nodes, int32_t *acc_tokens,
                                int32_t *bonus, bool do_walk, bool do_compact, uint16_t *k_cache,
                                uint16_t *v_cache, const int32_t *block_table, int32_t *ctx_lens,
                                const uint16_t *k_tree, const uint16_t *v_tree, bool advance_ctx,
                                cudaStream_t s);
cudaError_t launch_ctx_advance(int R, int32_t *ctx_lens, const int32_t *acc_len, cudaStream_t s);
cudaError_t launch_attention(ddt_ctx *c, const uint16_t *q, const uint16_t *k_tree,
                             const uint16_t *v_tree, const uint16_t *k_cache,
                             const uint16_t *v_cache, const int32_t *block_table,
                             const int32_t *ctx_lens, const uint32_t *mask, int R, float *out,
                             cudaStream_t s);

// a4 on tcgen05 (attention_tc.cu): the shapes it takes (head dim 64 or 128,
// G = Hq / Hkv dividing 16, pages of a power-of-two multiple of 16 tokens)
bool attention_tc_supported(const ddt_config &cfg);
void attention_tc_rows(const ddt_config &cfg, int *n_main, int *tail_rows, int *rowgroups);

// the parent-conditioned tree (cond_tree.cu)
bool cond_tree_supported(const ddt_config &cfg);
int cond_tree_cmax(const ddt_config &cfg);
cudaError_t launch_cond_tree(const ddt_ctx *c, const uint16_t *ell, const uint16_t *W,
                             const uint16_t *E, const int32_t *anchors, int R, float *cand_lp,
                             int32_t *cand_ids, int32_t *frontier_tok, int32_t *tree_tokens,
                             int32_t *parents, int32_t *depths, int32_t *n_nodes, uint32_t *mask,
                             cudaStream_t s);

// the SparklingTree table tree (markov.cu)
bool markov_supported(const ddt_config &cfg);
cudaError_t launch_markov_table(const ddt_ctx *c, const uint16_t *ell, const uint16_t *W,
                                const uint16_t *E, const int32_t *anchors, int R, int32_t *cand,
                                float *tab, cudaStream_t s);
cudaError_t launch_markov_tree(const ddt_ctx *c, const int32_t *cand, const float *tab, int R,
                               int32_t *tree_tokens, int32_t *parents, int32_t *depths,
                               int32_t *n_nodes, uint32_t *mask, cudaStream_t s);

// stochastic verification of a chain (stochastic.cu)
int stochastic_chunk_elems(int dtype);
int stochastic_draw_chunks(int V);
cudaError_t launch_accept_stochastic(const ddt_ctx *c, const void *draft, const void *target,
                                     const int32_t *tokens, const float *u, const float *r, int R,
                                     const int32_t *n_guess, int32_t *acc_len, int32_t *acc_tokens,
                                     cudaStream_t s);

// the hardware-aware prefix scheduler (sched.cu)
int schedule_smem_bytes(int R, int L);
cudaError_t launch_schedule_prefix(const ddt_ctx *c, const float *conf, int R, const float *cost,
                                   int32_t *n_keep, int32_t *n_total, double *stats,
                                   cudaStream_t s);

// a1 with caller-supplied scratch (used by the allocation-free entry point)
cudaError_t launch_topk_scratch(const void *z, int dtype, int rows, int V, int K, int nch,
                                int num_sms, uint16_t *gkey, uint16_t *wtop, float2 *part_ms,
                                float *top_lp, int32_t *top_ids, int32_t *status, cudaStream_t s);
// keys each warp of a1 keeps for the row threshold (Q)
int topk_warp_keys(int nch, int K);

// records the CUDA error reported by ddt_last_cuda_error (this thread)
void ddt_note_cuda_error(int e);

// sizes used by both the workspace carve-up and the launchers
int topk_chunk_elems(int dtype);
int amax_chunk_elems(int dtype);
