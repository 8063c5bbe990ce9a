// api.cu -- the extern "C" boundary of libddt.so: argument validation,
// workspace layout and the launch sequence of a round. Every check that can
// be made on the host is made here, before anything is enqueued.
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include "ddt_internal.h"

namespace {

thread_local int g_last_cuda_error = 0;

ddt_status cuda_fail(cudaError_t e)
{
    g_last_cuda_error = (int)e;
    return DDT_ECUDA;
}

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// resolve K and check every field; fills *out with the resolved config
ddt_status check_config(const ddt_config *in, ddt_config *out)
{
    if (in == nullptr)
        return DDT_EINVAL;
    ddt_config c = *in;
    if (c.K == 0)
        c.K = c.B < c.V ? c.B : c.V;
    if (c.R_max < 1 || c.L < 1 || c.V < 1 || c.B < 1 || c.K < 1 || c.K > c.V)
        return DDT_EINVAL;
    if (c.Hq < 1 || c.Hkv < 1 || c.Hq % c.Hkv != 0 || c.page_size < 1 ||
        c.max_pages_per_req < 1 || c.num_pages < 1)
        return DDT_EINVAL;
    if ((c.draft_dtype != DDT_BF16 && c.draft_dtype != DDT_F32) ||
        (c.target_dtype != DDT_BF16 && c.target_dtype != DDT_F32))
        return DDT_EINVAL;
    if (c.L > DDT_MAX_L || c.K > DDT_MAX_K || c.B > DDT_MAX_B)
        return DDT_EUNSUPPORTED;
    if (c.d != 64 && c.d != 128)
        return DDT_EUNSUPPORTED;
    if (!attention_tc_supported(c))
        return DDT_EUNSUPPORTED;  // the tcgen05 attention kernel cannot take this shape
    if (c.Hkv > 255)
        return DDT_EUNSUPPORTED;
    const int nch = (c.V + topk_chunk_elems(c.draft_dtype) - 1) / topk_chunk_elems(c.draft_dtype);
    if ((int64_t)nch * c.K > TOPK_CAND_CAP || nch > TOPK_MAX_CHUNKS)
        return DDT_EUNSUPPORTED;
    const int64_t max_ctx = (int64_t)c.max_pages_per_req * c.page_size;
    if (max_ctx > ATT_MAX_CTX || c.R_max > 2048)
        return DDT_EUNSUPPORTED;
    // the pool's token rows are TMA row coordinates (signed 32-bit) in a4
    if (c.num_pages > (int64_t)0x7FFFFFFF / c.page_size)
        return DDT_EUNSUPPORTED;
    if (c.markov_dim < 0 || c.frontier < 0 || c.prefilter < 0)
        return DDT_EINVAL;
    if ((c.frontier > 0 || c.prefilter > 0) && c.markov_dim == 0)
        return DDT_EINVAL;
    if (c.markov_dim > 0 && c.frontier == 0 && c.prefilter == 0)
        return DDT_EINVAL;
    if (c.markov_dim > 0 && c.draft_dtype != DDT_BF16)
        return DDT_EUNSUPPORTED;
    if (c.frontier > 0 && !cond_tree_supported(c))
        return DDT_EUNSUPPORTED;
    if (c.prefilter > 0 && (c.prefilter > c.V || !markov_supported(c)))
        return DDT_EUNSUPPORTED;
    *out = c;
    return DDT_OK;
}

struct Layout {
    size_t status, tk_gkey, tk_wtop, tk_ms, am_val, am_idx, att_part_o, att_part_ml, cg_part_ms, cg_part_top, cg_fr_tok, cg_fr_cand,
        cg_fr_n, cg_fr_S, cg_c_S, cg_c_meta, cg_thr, cg_seed_lp, cg_seed_ids, mk_cand, mk_tab,
        sv_part_d, sv_part_t, sv_cnt, sv_part_w, ps_rk, ps_rid, ps_arrive, total;
    int tk_nch, am_nch, max_items, sv_nch_d, sv_nch_t, sv_nch_w;
};

Layout layout_for(const ddt_config &c)
{
    Layout L;
    const int P = c.B + 1, G = c.Hq / c.Hkv;
    L.tk_nch = (c.V + topk_chunk_elems(c.draft_dtype) - 1) / topk_chunk_elems(c.draft_dtype);
    L.am_nch = (c.V + amax_chunk_elems(c.target_dtype) - 1) / amax_chunk_elems(c.target_dtype);
    L.max_items = 2 * ATT_MAX_CTAS;
    const size_t rows_d = (size_t)c.R_max * c.L, rows_t = (size_t)c.R_max * P;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t at = off;
        off = align_up(off + bytes, 256);
        return at;
    };
    L.status = take(sizeof(int32_t));
    L.tk_gkey = take(rows_d * L.tk_nch * TOPK_THREADS * sizeof(uint16_t));
    L.tk_wtop = take(rows_d * L.tk_nch * (TOPK_THREADS / 32) * topk_warp_keys(L.tk_nch, c.K) *
                     sizeof(uint16_t));
    L.tk_ms = take(rows_d * L.tk_nch * (TOPK_THREADS / 32) * sizeof(float2));
    L.am_val = take(rows_t * L.am_nch * sizeof(float));
    L.am_idx = take(rows_t * L.am_nch * sizeof(int32_t));
    L.att_part_o = take((size_t)L.max_items * ATT_ROWS * c.d * sizeof(float));
    L.att_part_ml = take((size_t)L.max_items * ATT_ROWS * sizeof(float2));
    // parent-conditioned tree (sized for up to CG_GRID_MAX CTAs of its GEMM)
    const size_t np = c.markov_dim > 0 ? (size_t)c.R_max * c.frontier : 0;
    const size_t cmax = c.markov_dim > 0 ? (size_t)cond_tree_cmax(c) : 0;
    const size_t nfr = c.markov_dim > 0 ? (size_t)c.R_max * c.frontier : 0;
    L.cg_part_ms = take(np * CG_GRID_MAX * sizeof(float2));
    L.cg_part_top = take(np * CG_GRID_MAX * 8 * sizeof(uint64_t));
    L.cg_fr_tok = take(nfr * sizeof(int32_t));
    L.cg_fr_cand = take(nfr * sizeof(int32_t));
    L.cg_fr_n = take((c.markov_dim > 0 ? (size_t)c.R_max : 0) * sizeof(int32_t));
    L.cg_fr_S = take(nfr * sizeof(double));
    L.cg_c_S = take((size_t)(c.markov_dim > 0 ? c.R_max : 0) * cmax * sizeof(double));
    L.cg_c_meta = take((size_t)(c.markov_dim > 0 ? c.R_max : 0) * cmax * 3 * sizeof(int32_t));
    L.cg_thr = take((c.markov_dim > 0 ? (size_t)c.L * CG_NP_MAX : 0) * sizeof(uint32_t));
    const size_t nseed = c.markov_dim > 0 ? (size_t)c.R_max * c.L * c.K : 0;
    L.cg_seed_lp = take(nseed * sizeof(float));
    L.cg_seed_ids = take(nseed * sizeof(int32_t));
    // SparklingTree table tree: the round's kept tokens and table
    const size_t mrows = c.prefilter > 0 ? (size_t)c.R_max * c.L : 0;
    const size_t C = (size_t)c.prefilter;
    L.mk_cand = take(mrows * C * sizeof(int32_t));
    L.mk_tab = take(mrows * C * C * sizeof(float));
    // stochastic chain verification: chunk pairs of the L draft and L + 1
    // target rows, the draw's chunk totals, an arrival counter per request
    L.sv_nch_d = (c.V + stochastic_chunk_elems(c.draft_dtype) - 1) /
                 stochastic_chunk_elems(c.draft_dtype);
    L.sv_nch_t = (c.V + stochastic_chunk_elems(c.target_dtype) - 1) /
                 stochastic_chunk_elems(c.target_dtype);
    L.sv_nch_w = stochastic_draw_chunks(c.V);
    L.sv_part_d = take((size_t)c.R_max * c.L * L.sv_nch_d * sizeof(float2));
    L.sv_part_t = take((size_t)c.R_max * (c.L + 1) * L.sv_nch_t * sizeof(float2));
    L.sv_cnt = take((size_t)c.R_max * sizeof(unsigned));
    L.sv_part_w = take((size_t)c.R_max * L.sv_nch_w * sizeof(float));
    // prefix scheduler: the ranking of up to DDT_SCHED_MAX_SLOTS slots
    L.ps_rk = take((size_t)DDT_SCHED_MAX_SLOTS * sizeof(uint64_t));
    L.ps_rid = take((size_t)DDT_SCHED_MAX_SLOTS * sizeof(int32_t));
    L.ps_arrive = take(sizeof(unsigned));
    L.total = off;
    return L;
}

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }
bool aligned4(const void *p) { return ((uintptr_t)p & 3u) == 0; }
bool aligned8(const void *p) { return ((uintptr_t)p & 7u) == 0; }

ddt_status check_R(const ddt_ctx *ctx, int32_t R)
{
    if (ctx == nullptr || R < 0 || R > ctx->cfg.R_max)
        return DDT_EINVAL;
    return DDT_OK;
}

ddt_status set_device(const ddt_ctx *ctx)
{
    int cur = -1;
    cudaError_t e = cudaGetDevice(&cur);
    if (e != cudaSuccess)
        return cuda_fail(e);
    if (cur != ctx->device) {
        e = cudaSetDevice(ctx->device);
        if (e != cudaSuccess)
            return cuda_fail(e);
    }
    return DDT_OK;
}

#define DDT_TRY(expr)                                                                              \
    do {                                                                                           \
        cudaError_t _e = (expr);                                                                   \
        if (_e != cudaSuccess)                                                                     \
            return cuda_fail(_e);                                                                  \
    } while (0)

#define DDT_CHECK(cond)                                                                            \
    do {                                                                                           \
        if (!(cond))                                                                               \
            return DDT_EINVAL;                                                                     \
    } while (0)

ddt_status chk_topk(const ddt_ctx *c, const void *z, const float *lp, const int32_t *ids)
{
    DDT_CHECK(z && lp && ids && aligned16(z) && aligned4(lp) && aligned4(ids));
    (void)c;
    return DDT_OK;
}

ddt_status chk_tree(const float *lp, const int32_t *ids, const int32_t *tok, const int32_t *par,
                    const int32_t *dep, const int32_t *nn)
{
    DDT_CHECK(lp && ids && tok && par && dep && nn);
    DDT_CHECK(aligned4(lp) && aligned4(ids) && aligned4(tok) && aligned4(par) && aligned4(dep) &&
              aligned4(nn));
    return DDT_OK;
}

ddt_status chk_attn(const uint16_t *q, const uint16_t *kt, const uint16_t *vt, const uint16_t *kc,
                    const uint16_t *vc, const int32_t *bt, const int32_t *cl, const uint32_t *mask,
                    const float *out)
{
    DDT_CHECK(q && kt && vt && kc && vc && bt && cl && mask && out);
    DDT_CHECK(aligned16(q) && aligned16(kt) && aligned16(vt) && aligned16(kc) && aligned16(vc) &&
              aligned16(out) && aligned4(bt) && aligned4(cl) && aligned4(mask));
    return DDT_OK;
}

ddt_status chk_walk(const int32_t *tok, const int32_t *par, const int32_t *nn, const int32_t *al,
                    const int32_t *an, const int32_t *at, const int32_t *bo)
{
    DDT_CHECK(tok && par && nn && al && an && at && bo);
    DDT_CHECK(aligned4(tok) && aligned4(par) && aligned4(nn) && aligned4(al) && aligned4(an) &&
              aligned4(at) && aligned4(bo));
    return DDT_OK;
}

ddt_status chk_compact(const uint16_t *kc, const uint16_t *vc, const int32_t *bt,
                       const int32_t *cl, const uint16_t *kt, const uint16_t *vt)
{
    DDT_CHECK(kc && vc && bt && cl && kt && vt);
    DDT_CHECK(aligned16(kc) && aligned16(vc) && aligned16(kt) && aligned16(vt) && aligned4(bt) &&
              aligned4(cl));
    return DDT_OK;
}

}  // namespace

extern "C" {

size_t ddt_workspace_bytes(const ddt_config *cfg)
{
    ddt_config c;
    if (check_config(cfg, &c) != DDT_OK)
        return 0;
    return layout_for(c).total;
}

ddt_status ddt_create(const ddt_config *cfg, ddt_ctx **out)
{
    if (out == nullptr)
        return DDT_EINVAL;
    *out = nullptr;
    ddt_config c;
    const ddt_status st = check_config(cfg, &c);
    if (st != DDT_OK)
        return st;
    ddt_ctx *ctx = (ddt_ctx *)calloc(1, sizeof(ddt_ctx));
    if (ctx == nullptr)
        return DDT_ENOMEM;
    ctx->cfg = c;
    cudaError_t e = cudaGetDevice(&ctx->device);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&ctx->num_sms, cudaDevAttrMultiProcessorCount, ctx->device);
    if (e != cudaSuccess) {
        free(ctx);
        return cuda_fail(e);
    }
    const Layout L = layout_for(c);
    e = cudaMalloc((void **)&ctx->ws, L.total);
    if (e != cudaSuccess) {
        free(ctx);
        g_last_cuda_error = (int)e;
        return DDT_ENOMEM;
    }
    e = cudaMemset(ctx->ws, 0, L.total);
    if (e == cudaSuccess)
        e = cudaDeviceSynchronize();
    if (e != cudaSuccess) {
        cudaFree(ctx->ws);
        free(ctx);
        return cuda_fail(e);
    }
    ctx->ws_bytes = L.total;
    char *w = ctx->ws;
    ctx->status = (int32_t *)(w + L.status);
    ctx->tk_nch = L.tk_nch;
    ctx->tk_gkey = (uint16_t *)(w + L.tk_gkey);
    ctx->tk_wtop = (uint16_t *)(w + L.tk_wtop);
    ctx->tk_ms = (float2 *)(w + L.tk_ms);
    ctx->am_nch = L.am_nch;
    ctx->am_val = (float *)(w + L.am_val);
    ctx->am_idx = (int32_t *)(w + L.am_idx);
    ctx->att_max_items = L.max_items;
    ctx->att_part_o = (float *)(w + L.att_part_o);
    ctx->att_part_ml = (float2 *)(w + L.att_part_ml);
    ctx->cg_grid = ctx->num_sms < CG_GRID_MAX ? ctx->num_sms : CG_GRID_MAX;
    ctx->cg_part_ms = (float2 *)(w + L.cg_part_ms);
    ctx->cg_part_top = (uint64_t *)(w + L.cg_part_top);
    ctx->cg_fr_tok = (int32_t *)(w + L.cg_fr_tok);
    ctx->cg_fr_cand = (int32_t *)(w + L.cg_fr_cand);
    ctx->cg_fr_n = (int32_t *)(w + L.cg_fr_n);
    ctx->cg_fr_S = (double *)(w + L.cg_fr_S);
    ctx->cg_c_S = (double *)(w + L.cg_c_S);
    ctx->cg_c_meta = (int32_t *)(w + L.cg_c_meta);
    ctx->cg_thr = (uint32_t *)(w + L.cg_thr);
    ctx->cg_seed_lp = (float *)(w + L.cg_seed_lp);
    ctx->cg_seed_ids = (int32_t *)(w + L.cg_seed_ids);
    ctx->mk_cand = (int32_t *)(w + L.mk_cand);
    ctx->mk_tab = (float *)(w + L.mk_tab);
    ctx->sv_nch_d = L.sv_nch_d;
    ctx->sv_nch_t = L.sv_nch_t;
    ctx->sv_nch_w = L.sv_nch_w;
    ctx->sv_part_d = (float2 *)(w + L.sv_part_d);
    ctx->sv_part_t = (float2 *)(w + L.sv_part_t);
    ctx->sv_cnt = (unsigned *)(w + L.sv_cnt);
    ctx->sv_part_w = (float *)(w + L.sv_part_w);
    ctx->ps_rk = (uint64_t *)(w + L.ps_rk);
    ctx->ps_rid = (int32_t *)(w + L.ps_rid);
    ctx->ps_arrive = (unsigned *)(w + L.ps_arrive);
    // ddt_round's streams: a1..a3 at the highest priority, a5 at the lowest, so
    // that a5's CTAs only fill what a1..a3 leave idle
    int prio_least = 0, prio_greatest = 0;
    e = cudaDeviceGetStreamPriorityRange(&prio_least, &prio_greatest);
    if (e == cudaSuccess)
        e = cudaStreamCreateWithPriority(&ctx->hi, cudaStreamNonBlocking, prio_greatest);
    if (e == cudaSuccess)
        e = cudaStreamCreateWithPriority(&ctx->side, cudaStreamNonBlocking, prio_least);
    if (e == cudaSuccess)
        e = cudaEventCreateWithFlags(&ctx->ev_fork, cudaEventDisableTiming);
    if (e == cudaSuccess)
        e = cudaEventCreateWithFlags(&ctx->ev_tree, cudaEventDisableTiming);
    if (e == cudaSuccess)
        e = cudaEventCreateWithFlags(&ctx->ev_join, cudaEventDisableTiming);
    if (e == cudaSuccess)
        e = cudaEventCreateWithFlags(&ctx->ev_walk, cudaEventDisableTiming);
    if (e != cudaSuccess) {
        if (ctx->ev_join)
            cudaEventDestroy(ctx->ev_join);
        if (ctx->ev_tree)
            cudaEventDestroy(ctx->ev_tree);
        if (ctx->ev_fork)
            cudaEventDestroy(ctx->ev_fork);
        if (ctx->side)
            cudaStreamDestroy(ctx->side);
        if (ctx->hi)
            cudaStreamDestroy(ctx->hi);
        cudaFree(ctx->ws);
        free(ctx);
        return cuda_fail(e);
    }
    *out = ctx;
    return DDT_OK;
}

void ddt_destroy(ddt_ctx *ctx)
{
    if (ctx == nullptr)
        return;
    int cur = -1;
    cudaGetDevice(&cur);
    cudaSetDevice(ctx->device);
    cudaStreamSynchronize(ctx->side);
    cudaStreamSynchronize(ctx->hi);
    cudaEventDestroy(ctx->ev_walk);
    cudaEventDestroy(ctx->ev_join);
    cudaEventDestroy(ctx->ev_tree);
    cudaEventDestroy(ctx->ev_fork);
    cudaStreamDestroy(ctx->side);
    cudaStreamDestroy(ctx->hi);
    cudaFree(ctx->ws);
    if (cur >= 0)
        cudaSetDevice(cur);
    free(ctx);
}

ddt_status ddt_topk_logprobs(ddt_ctx *ctx, const void *draft_logits, int32_t R, float *top_lp,
                             int32_t *top_ids, void *stream)
{
    ddt_status st = check_R(ctx, R);
    if (st != DDT_OK)
        return st;
    if (R == 0)
        return DDT_OK;
    if ((st = chk_topk(ctx, draft_logits, top_lp, top_ids)) != DDT_OK)
        return st;
    if ((st = set_device(ctx)) != DDT_OK)
        return st;
    DDT_TRY(launch_topk(ctx, draft_logits, R, top_lp, top_ids, (cudaStream_t)stream));
    return DDT_OK;
}

ddt_status ddt_build_tree(ddt_ctx *ctx, const float *top_lp, const int32_t *top_ids, int32_t R,
                          int32_t *tree_tokens, int32_t *parents, int32_t *depths,
                          int32_t *n_nodes, uint32_t *mask, void *stream)
{
    ddt_status st = check_R(ctx, R);
    if (st != DDT_OK)
        return st;
    if (R == 0)
        return DDT_OK;
    if ((st = chk_tree(top_lp, top_ids, tree_tokens, parents, depths, n_nodes)) != DDT_OK)
        return st;
    if (mask != nullptr && !aligned4(mask))
        return DDT_EINVAL;
    if ((st = set_device(ctx)) != DDT_OK)
        return st;
    DDT_TRY(launch_build_tree(ctx, top_lp, top_ids, R, tree_tokens, parents, depths, n_nodes, mask,
                              (cudaStream_t)stream));
    return DDT_OK;
}

ddt_status ddt_build_tree_conditioned(ddt_ctx *ctx, const void *draft_logits, const uint16_t *W,
                                      const uint16_t *E, const int32_t *anchors, int32_t R,
                                      float *cand_lp, int32_t *cand_ids, int32_t *frontier_tok,
                                      int32_t *tree_tokens, int32_t *parents, int32_t *depths,
                                      int32_t *n_nodes, uint32_t *mask, void *stream)
{
    ddt_status st = check_R(ctx, R);
    if (st != DDT_OK)
        return st;
    if (ctx->cfg.markov_dim <= 0 || ctx->cfg.frontier <= 0)
        return DDT_EUNSUPPORTED;
    if (R == 0)
        return DDT_OK;
    DDT_CHECK(draft_logits && W && E && anchors && tree_tokens && parents && depths && n_nodes);
    DDT_CHECK(aligned16(W) && aligned16(E) && aligned4(anchors) && aligned4(tree_tokens) &&
              aligned4(parents) && aligned4(depths) && aligned4(n_nodes));
    DDT_CHECK((cand_lp == nullptr) == (cand_ids == nullptr));
    DDT_CHECK(!cand_lp || (aligned4(cand_lp) && aligned4(cand_ids)));
    DDT_CHECK(!frontier_tok || aligned4(frontier_tok));
    DDT_CHECK(!mask || aligned4(mask));
    if (R * ctx->cfg.frontier > 128)
        return DDT_EUNSUPPORTED;
    if ((st = set_device(ctx)) != DDT_OK)
        return st;
    DDT_TRY(launch_cond_tree(ctx, (const uint16_t *)draft_logits, W, E, anchors, R, cand_lp,
                             cand_ids, frontier_tok, tree_tokens, parents, depths, n_nodes, mask,
                             (cudaStream_t)stream));
    return DDT_OK;
}

ddt_status ddt_build_mask(ddt_ctx *ctx, const int32_t *parents, const int32_t *n_nodes, int32_t R,
                          uint32_t *mask, void *stream)
{
    ddt_status st = check_R(ctx, R);
    if (st != DDT_OK)
        return st;
    if (R == 0)
        return DDT_OK;
    if (!parents || !n_nodes || !mask || !aligned4(parents) || !aligned4(n_nodes) || !aligned4(mask))
        return DDT_EINVAL;
    if ((st = set_device(ctx)) != DDT_OK)
        return st;
    DDT_TRY(launch_build_mask(ctx, parents, n_nodes, R, mask, (cudaStream_t)stream));
    return DDT_OK;
}

ddt_status ddt_tree_attention(ddt_ctx *ctx, const uint16_t *q, const uint16_t *k_tree,
                              const uint16_t *v_tree, const uint16_t *k_cache,
                              const uint16_t *v_cache, const int32_t *block_table,
                              const int32_t *ctx_lens, const uint32_t *mask, int32_t R,
                              float *out, void *stream)
{
    ddt_status st = check_R(ctx, R);
    if (st != DDT_OK)
        return st;
    if (R == 0)
        return DDT_OK;
    if ((st = chk_attn(q, k_tree, v_tree, k_cache, v_cache, block_table, ctx_lens, mask, out)) !=
        DDT_OK)
        return st;
    if ((st = set_device(ctx)) != DDT_OK)
        return st;
    DDT_TRY(launch_attention(ctx, q, k_tree, v_tree, k_cache, v_cache, block_table, ctx_lens, mask,
                             R, out, (cudaStream_t)stream));
    return DDT_OK;
}

ddt_status ddt_target_argmax(ddt_ctx *ctx, const void *target_logits, int32_t R,
                             int32_t *argmax_out, void *stream)
{
    ddt_status st = check_R(ctx, R);
    if (st != DDT_OK)
        return st;
    if (R == 0)
        return DDT_OK;
    if (!target_logits || !argmax_out || !aligned16(target_logits) || !aligned4(argmax_out))
        return DDT_EINVAL;
    if ((st = set_device(ctx)) != DDT_OK)
        return st;
    DDT_TRY(launch_argmax_partials(ctx, target_logits, R, (cudaStream_t)stream));
    DDT_TRY(launch_argmax_finish(ctx, R, argmax_out, (cudaStream_t)stream));
    return DDT_OK;
}

ddt_status ddt_walk(ddt_ctx *ctx, const int32_t *argmax, const int32_t *tree_tokens,
                    const int32_t *parents, const int32_t *n_nodes, int32_t R, int32_t *acc_len,
                    int32_t *acc_nodes, int32_t *acc_tokens, int32_t *bonus, void *stream)
{
    ddt_status st = check_R(ctx, R);
    if (st != DDT_OK)
        return st;
    if (R == 0)
        return DDT_OK;
    if (!argmax || !aligned4(argmax) ||
        (st = chk_walk(tree_tokens, parents, n_nodes, acc_len, acc_nodes, acc_tokens, bonus)) !=
            DDT_OK)
        return DDT_EINVAL;
    if ((st = set_device(ctx)) != DDT_OK)
        return st;
    DDT_TRY(launch_walk_compact(ctx, argmax, false, nullptr, tree_tokens, parents, n_nodes, R,
                                acc_len, acc_nodes, acc_tokens, bonus, true, false, nullptr,
                                nullptr, nullptr, nullptr, nullptr, nullptr, false,
                                (cudaStream_t)stream));
    return DDT_OK;
}

ddt_status ddt_compact(ddt_ctx *ctx, uint16_t *k_cache, uint16_t *v_cache,
                       const int32_t *block_table, int32_t *ctx_lens, const uint16_t *k_tree,
                       const uint16_t *v_tree, const int32_t *acc_nodes, const int32_t *acc_len,
                       int32_t R, void *stream)
{
    ddt_status st = check_R(ctx, R);
    if (st != DDT_OK)
        return st;
    if (R == 0)
        return DDT_OK;
    if (!acc_nodes || !acc_len || !aligned4(acc_nodes) || !aligned4(acc_len) ||
        (st = chk_compact(k_cache, v_cache, block_table, ctx_lens, k_tree, v_tree)) != DDT_OK)
        return DDT_EINVAL;
    if ((st = set_device(ctx)) != DDT_OK)
        return st;
    DDT_TRY(launch_walk_compact(ctx, nullptr, false, nullptr, nullptr, nullptr, nullptr, R,
                                const_cast<int32_t *>(acc_len), const_cast<int32_t *>(acc_nodes),
                                nullptr, nullptr, false, true, k_cache, v_cache, block_table,
                                ctx_lens, k_tree, v_tree, true, (cudaStream_t)stream));
    return DDT_OK;
}

ddt_status ddt_accept(ddt_ctx *ctx, const void *target_logits, const int32_t *tree_tokens,
                      const int32_t *parents, const int32_t *n_nodes, int32_t R,
                      int32_t *argmax_out, int32_t *acc_len, int32_t *acc_nodes,
                      int32_t *acc_tokens, int32_t *bonus, uint16_t *k_cache, uint16_t *v_cache,
                      const int32_t *block_table, const uint16_t *k_tree, const uint16_t *v_tree,
                      int32_t *ctx_lens, void *stream)
{
    ddt_status st = check_R(ctx, R);
    if (st != DDT_OK)
        return st;
    if (R == 0)
        return DDT_OK;
    if (!target_logits || !aligned16(target_logits) || (argmax_out && !aligned4(argmax_out)))
        return DDT_EINVAL;
    if ((st = chk_walk(tree_tokens, parents, n_nodes, acc_len, acc_nodes, acc_tokens, bonus)) !=
            DDT_OK ||
        (st = chk_compact(k_cache, v_cache, block_table, ctx_lens, k_tree, v_tree)) != DDT_OK)
        return DDT_EINVAL;
    if ((st = set_device(ctx)) != DDT_OK)
        return st;
    cudaStream_t s = (cudaStream_t)stream;
    DDT_TRY(launch_argmax_partials(ctx, target_logits, R, s));
    DDT_TRY(launch_walk_compact(ctx, nullptr, true, argmax_out, tree_tokens, parents, n_nodes, R,
                                acc_len, acc_nodes, acc_tokens, bonus, true, true, k_cache, v_cache,
                                block_table, ctx_lens, k_tree, v_tree, true, s));
    return DDT_OK;
}

ddt_status ddt_accept_stochastic(ddt_ctx *ctx, const void *draft_logits,
                                 const void *target_logits, const int32_t *draft_tokens,
                                 const float *u, const float *r, int32_t R, int32_t *acc_len,
                                 int32_t *acc_tokens, const int32_t *n_guess, void *stream)
{
    ddt_status st = check_R(ctx, R);
    if (st != DDT_OK)
        return st;
    if (R == 0)
        return DDT_OK;
    if (!draft_logits || !target_logits || !draft_tokens || !u || !r || !acc_len || !acc_tokens)
        return DDT_EINVAL;
    DDT_CHECK(aligned4(draft_tokens) && aligned4(u) && aligned4(r) && aligned4(acc_len) &&
              aligned4(acc_tokens) && (!n_guess || aligned4(n_guess)));
    if ((st = set_device(ctx)) != DDT_OK)
        return st;
    DDT_TRY(launch_accept_stochastic(ctx, draft_logits, target_logits, draft_tokens, u, r, R,
                                     n_guess, acc_len, acc_tokens, (cudaStream_t)stream));
    return DDT_OK;
}

ddt_status ddt_schedule_prefix(ddt_ctx *ctx, const float *conf, int32_t R, const float *cost_ms,
                               int32_t *n_keep, int32_t *n_total, double *stats, void *stream)
{
    ddt_status st = check_R(ctx, R);
    if (st != DDT_OK)
        return st;
    if (R == 0)
        return DDT_OK;
    if (!conf || !cost_ms || !n_keep)
        return DDT_EINVAL;
    DDT_CHECK(aligned4(conf) && aligned4(cost_ms) && aligned4(n_keep) &&
              (!n_total || aligned4(n_total)) && (!stats || aligned8(stats)));
    if ((int64_t)R * ctx->cfg.L > DDT_SCHED_MAX_SLOTS)
        return DDT_EUNSUPPORTED;
    if ((st = set_device(ctx)) != DDT_OK)
        return st;
    DDT_TRY(launch_schedule_prefix(ctx, conf, R, cost_ms, n_keep, n_total, stats,
                                   (cudaStream_t)stream));
    return DDT_OK;
}

// a4 on `s` once the tree (ev_tree) and a5 (ev_join) are done; beside it, on
// the side stream, a6 and a7's row copies (they need a5 and the tree; the
// rows they write lie past each request's context, which a4 reads only
// masked); the context lengths advance on `s` after both, since a4 reads them
static ddt_status round_verify(ddt_ctx *ctx, const ddt_round_args *a, cudaStream_t s)
{
    const int32_t R = a->R;
    DDT_TRY(cudaStreamWaitEvent(s, ctx->ev_tree, 0));
    DDT_TRY(cudaStreamWaitEvent(s, ctx->ev_join, 0));
    if (a->att_event_begin)
        DDT_TRY(cudaEventRecord((cudaEvent_t)a->att_event_begin, s));
    DDT_TRY(launch_attention(ctx, a->q, a->k_tree, a->v_tree, a->k_cache, a->v_cache,
                             a->block_table, a->ctx_lens, a->mask, R, a->attn_out, s));
    if (a->att_event_end)
        DDT_TRY(cudaEventRecord((cudaEvent_t)a->att_event_end, s));
    DDT_TRY(cudaStreamWaitEvent(ctx->side, ctx->ev_tree, 0));
    DDT_TRY(launch_walk_compact(ctx, nullptr, true, a->target_argmax, a->tree_tokens, a->parents,
                                a->n_nodes, R, a->acc_len, a->acc_nodes, a->acc_tokens, a->bonus,
                                true, true, a->k_cache, a->v_cache, a->block_table, a->ctx_lens,
                                a->k_tree, a->v_tree, false, ctx->side));
    DDT_TRY(cudaEventRecord(ctx->ev_walk, ctx->side));
    DDT_TRY(cudaStreamWaitEvent(s, ctx->ev_walk, 0));
    DDT_TRY(launch_ctx_advance(R, a->ctx_lens, a->acc_len, s));
    return DDT_OK;
}

ddt_status ddt_round(ddt_ctx *ctx, const ddt_round_args *a, void *stream)
{
    if (a == nullptr)
        return DDT_EINVAL;
    const int32_t R = a->R;
    ddt_status st = check_R(ctx, R);
    if (st != DDT_OK)
        return st;
    if (R == 0)
        return DDT_OK;
    if ((st = chk_topk(ctx, a->draft_logits, a->top_lp, a->top_ids)) != DDT_OK ||
        (st = chk_tree(a->top_lp, a->top_ids, a->tree_tokens, a->parents, a->depths,
                       a->n_nodes)) != DDT_OK ||
        (st = chk_attn(a->q, a->k_tree, a->v_tree, a->k_cache, a->v_cache, a->block_table,
                       a->ctx_lens, a->mask, a->attn_out)) != DDT_OK ||
        (st = chk_walk(a->tree_tokens, a->parents, a->n_nodes, a->acc_len, a->acc_nodes,
                       a->acc_tokens, a->bonus)) != DDT_OK)
        return st;
    if (!a->target_logits || !aligned16(a->target_logits) ||
        (a->target_argmax && !aligned4(a->target_argmax)))
        return DDT_EINVAL;
    if ((st = set_device(ctx)) != DDT_OK)
        return st;
    cudaStream_t s = (cudaStream_t)stream;
    // a1..a3 on the highest-priority stream, a5 on the lowest beside them (the
    // tree kernel leaves most SMs idle); both join `s` before a4
    DDT_TRY(cudaEventRecord(ctx->ev_fork, s));
    DDT_TRY(cudaStreamWaitEvent(ctx->hi, ctx->ev_fork, 0));
    DDT_TRY(cudaStreamWaitEvent(ctx->side, ctx->ev_fork, 0));
    DDT_TRY(launch_topk(ctx, a->draft_logits, R, a->top_lp, a->top_ids, ctx->hi));
    DDT_TRY(launch_argmax_partials(ctx, a->target_logits, R, ctx->side));
    DDT_TRY(cudaEventRecord(ctx->ev_join, ctx->side));
    DDT_TRY(launch_build_tree(ctx, a->top_lp, a->top_ids, R, a->tree_tokens, a->parents,
                              a->depths, a->n_nodes, a->mask, ctx->hi));
    DDT_TRY(cudaEventRecord(ctx->ev_tree, ctx->hi));
    return round_verify(ctx, a, s);
}

ddt_status ddt_round_conditioned(ddt_ctx *ctx, const ddt_round_args *a, const uint16_t *W,
                                 const uint16_t *E, const int32_t *anchors, void *stream)
{
    if (a == nullptr)
        return DDT_EINVAL;
    const int32_t R = a->R;
    ddt_status st = check_R(ctx, R);
    if (st != DDT_OK)
        return st;
    if (ctx->cfg.markov_dim <= 0 || ctx->cfg.frontier <= 0)
        return DDT_EUNSUPPORTED;
    if (R == 0)
        return DDT_OK;
    DDT_CHECK(a->draft_logits && aligned16(a->draft_logits) && W && E && anchors &&
              aligned16(W) && aligned16(E) && aligned4(anchors));
    DDT_CHECK(a->tree_tokens && a->parents && a->depths && a->n_nodes && aligned4(a->tree_tokens) &&
              aligned4(a->parents) && aligned4(a->depths) && aligned4(a->n_nodes));
    if ((st = chk_attn(a->q, a->k_tree, a->v_tree, a->k_cache, a->v_cache, a->block_table,
                       a->ctx_lens, a->mask, a->attn_out)) != DDT_OK ||
        (st = chk_walk(a->tree_tokens, a->parents, a->n_nodes, a->acc_len, a->acc_nodes,
                       a->acc_tokens, a->bonus)) != DDT_OK)
        return st;
    if (!a->target_logits || !aligned16(a->target_logits) ||
        (a->target_argmax && !aligned4(a->target_argmax)))
        return DDT_EINVAL;
    if (R * ctx->cfg.frontier > CG_NP_MAX)
        return DDT_EUNSUPPORTED;
    if ((st = set_device(ctx)) != DDT_OK)
        return st;
    cudaStream_t s = (cudaStream_t)stream;
    // the conditioned tree (with its mask) on the highest-priority stream, a5
    // beside it on the lowest; both join `s` before a4
    DDT_TRY(cudaEventRecord(ctx->ev_fork, s));
    DDT_TRY(cudaStreamWaitEvent(ctx->hi, ctx->ev_fork, 0));
    DDT_TRY(cudaStreamWaitEvent(ctx->side, ctx->ev_fork, 0));
    DDT_TRY(launch_argmax_partials(ctx, a->target_logits, R, ctx->side));
    DDT_TRY(cudaEventRecord(ctx->ev_join, ctx->side));
    DDT_TRY(launch_cond_tree(ctx, (const uint16_t *)a->draft_logits, W, E, anchors, R, nullptr,
                             nullptr, nullptr, a->tree_tokens, a->parents, a->depths, a->n_nodes,
                             a->mask, ctx->hi));
    DDT_TRY(cudaEventRecord(ctx->ev_tree, ctx->hi));
    return round_verify(ctx, a, s);
}

ddt_status ddt_markov_table(ddt_ctx *ctx, const void *draft_logits, const uint16_t *W,
                            const uint16_t *E, const int32_t *anchors, int32_t R,
                            int32_t *cand_ids, float *tab_lp, void *stream)
{
    ddt_status st = check_R(ctx, R);
    if (st != DDT_OK)
        return st;
    if (ctx->cfg.prefilter <= 0)
        return DDT_EUNSUPPORTED;
    if (R == 0)
        return DDT_OK;
    DDT_CHECK(draft_logits && W && E && anchors && cand_ids && tab_lp);
    DDT_CHECK(aligned16(draft_logits) && aligned16(W) && aligned16(E) && aligned4(anchors) &&
              aligned4(cand_ids) && aligned16(tab_lp));
    if ((st = set_device(ctx)) != DDT_OK)
        return st;
    DDT_TRY(launch_markov_table(ctx, (const uint16_t *)draft_logits, W, E, anchors, R, cand_ids,
                                tab_lp, (cudaStream_t)stream));
    return DDT_OK;
}

ddt_status ddt_build_tree_markov(ddt_ctx *ctx, const int32_t *cand_ids, const float *tab_lp,
                                 int32_t R, int32_t *tree_tokens, int32_t *parents,
                                 int32_t *depths, int32_t *n_nodes, uint32_t *mask, void *stream)
{
    ddt_status st = check_R(ctx, R);
    if (st != DDT_OK)
        return st;
    if (ctx->cfg.prefilter <= 0)
        return DDT_EUNSUPPORTED;
    if (R == 0)
        return DDT_OK;
    DDT_CHECK(cand_ids && tab_lp && tree_tokens && parents && depths && n_nodes);
    DDT_CHECK(aligned4(cand_ids) && aligned16(tab_lp) && aligned4(tree_tokens) &&
              aligned4(parents) && aligned4(depths) && aligned4(n_nodes));
    DDT_CHECK(!mask || aligned4(mask));
    if ((st = set_device(ctx)) != DDT_OK)
        return st;
    DDT_TRY(launch_markov_tree(ctx, cand_ids, tab_lp, R, tree_tokens, parents, depths, n_nodes,
                               mask, (cudaStream_t)stream));
    return DDT_OK;
}

ddt_status ddt_round_markov(ddt_ctx *ctx, const ddt_round_args *a, const uint16_t *W,
                            const uint16_t *E, const int32_t *anchors, void *stream)
{
    if (a == nullptr)
        return DDT_EINVAL;
    const int32_t R = a->R;
    ddt_status st = check_R(ctx, R);
    if (st != DDT_OK)
        return st;
    if (ctx->cfg.prefilter <= 0)
        return DDT_EUNSUPPORTED;
    if (R == 0)
        return DDT_OK;
    DDT_CHECK(a->draft_logits && aligned16(a->draft_logits) && W && E && anchors &&
              aligned16(W) && aligned16(E) && aligned4(anchors));
    DDT_CHECK(a->tree_tokens && a->parents && a->depths && a->n_nodes && aligned4(a->tree_tokens) &&
              aligned4(a->parents) && aligned4(a->depths) && aligned4(a->n_nodes));
    if ((st = chk_attn(a->q, a->k_tree, a->v_tree, a->k_cache, a->v_cache, a->block_table,
                       a->ctx_lens, a->mask, a->attn_out)) != DDT_OK ||
        (st = chk_walk(a->tree_tokens, a->parents, a->n_nodes, a->acc_len, a->acc_nodes,
                       a->acc_tokens, a->bonus)) != DDT_OK)
        return st;
    if (!a->target_logits || !aligned16(a->target_logits) ||
        (a->target_argmax && !aligned4(a->target_argmax)))
        return DDT_EINVAL;
    if ((st = set_device(ctx)) != DDT_OK)
        return st;
    cudaStream_t s = (cudaStream_t)stream;
    // the table and its tree (with the mask) on the highest-priority stream,
    // a5 beside them on the lowest; both join `s` before a4
    DDT_TRY(cudaEventRecord(ctx->ev_fork, s));
    DDT_TRY(cudaStreamWaitEvent(ctx->hi, ctx->ev_fork, 0));
    DDT_TRY(cudaStreamWaitEvent(ctx->side, ctx->ev_fork, 0));
    DDT_TRY(launch_markov_table(ctx, (const uint16_t *)a->draft_logits, W, E, anchors, R,
                                ctx->mk_cand, ctx->mk_tab, ctx->hi));
    DDT_TRY(launch_argmax_partials(ctx, a->target_logits, R, ctx->side));
    DDT_TRY(cudaEventRecord(ctx->ev_join, ctx->side));
    DDT_TRY(launch_markov_tree(ctx, ctx->mk_cand, ctx->mk_tab, R, a->tree_tokens, a->parents,
                               a->depths, a->n_nodes, a->mask, ctx->hi));
    DDT_TRY(cudaEventRecord(ctx->ev_tree, ctx->hi));
    return round_verify(ctx, a, s);
}

ddt_status ddt_device_status(ddt_ctx *ctx, int32_t *host_out)
{
    if (ctx == nullptr || host_out == nullptr)
        return DDT_EINVAL;
    ddt_status st = set_device(ctx);
    if (st != DDT_OK)
        return st;
    DDT_TRY(cudaDeviceSynchronize());
    DDT_TRY(cudaMemcpy(host_out, ctx->status, sizeof(int32_t), cudaMemcpyDeviceToHost));
    DDT_TRY(cudaMemset(ctx->status, 0, sizeof(int32_t)));
    DDT_TRY(cudaDeviceSynchronize());
    return DDT_OK;
}

ddt_status ddt_debug_arm_attention_timeout(ddt_ctx *ctx, int64_t wait_cycles)
{
    if (ctx == nullptr)
        return DDT_EINVAL;
    ctx->debug_att_wait = wait_cycles > 0 ? wait_cycles : 0;
    return DDT_OK;
}

const char *ddt_strerror(ddt_status status)
{
    switch (status) {
    case DDT_OK:
        return "ok";
    case DDT_EINVAL:
        return "invalid argument";
    case DDT_EUNSUPPORTED:
        return "unsupported configuration";
    case DDT_ECUDA:
        return "CUDA runtime error";
    case DDT_ENOMEM:
        return "out of device memory";
    }
    return "unknown status";
}

int32_t ddt_last_cuda_error(void) { return (int32_t)g_last_cuda_error; }

}  // extern "C"

void ddt_note_cuda_error(int e) { g_last_cuda_error = e; }
