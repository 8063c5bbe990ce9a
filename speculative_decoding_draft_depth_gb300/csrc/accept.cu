// accept.cu -- a5 target argmax, a6 greedy acceptance walk, a7 KV compaction.
//
// a5/a6 follow "DDTree Explained ...", section 5 (verifier walk: from the
// bonus token, take the target's decoding rule -- greedy here -- and match
// it against the children, step by step; return the accepted path and a
// new bonus token) and "Robot2050/TreeSpark" (vectorised acceptance over
// all in-flight trees; greedy tree verification reproduces autoregressive
// greedy output). a7 follows the same section's compact_cache (keep only
// the accepted path's KV).
//
// a5 is HBM-bound: one CTA per (chunk, row) of the [R, P, V] target logits,
// 8 x 16-byte vectors per thread; the chunk's max comes from packed bf16x2
// maxima and warp reductions, and only the threads holding it look at single
// elements. Per-chunk (max, first index) pairs are reduced per row by the
// walk kernel (or the finish kernel).
#include <stdint.h>

#include "ddt_device.cuh"
#include "ddt_internal.h"

namespace {

constexpr int NV = AMAX_VEC_PER_THREAD;
constexpr int IDX_NONE = 0x7FFFFFFF;

DDT_DEVINL uint32_t bmax2_nan(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// combine two partial (max, first index) results
DDT_DEVINL void amax_merge(float &best, int &bi, float ob, int oi)
{
    if (oi == IDX_NONE)
        return;
    if (bi == IDX_NONE || ob > best || (ob == best && oi < bi)) {
        best = ob;
        bi = oi;
    }
}

DDT_DEVINL uint32_t bmax2(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// order-preserving map of a float to uint32 (-0 == +0; NaN must be excluded first)
DDT_DEVINL uint32_t fkey(float x)
{
    const uint32_t b = __float_as_uint(x + 0.0f);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
DDT_DEVINL float fkey_inv(uint32_t k)
{
    return (k & 0x80000000u) ? __uint_as_float(k & 0x7FFFFFFFu) : __uint_as_float(~k);
}

// One CTA per (chunk, row). The chunk's max is found without looking at single
// elements (packed bf16x2 max per thread, one warp reduction, one CTA step);
// only the threads that hold it scan their own elements, in index order, for
// its first occurrence. NaN elements are skipped (and flagged).
template <bool BF16, bool ALIGNED>
__global__ void __launch_bounds__(AMAX_THREADS, 5)
argmax_chunk_kernel(const void *__restrict__ t, int V, int nch, float *__restrict__ am_val,
                    int32_t *__restrict__ am_idx, int32_t *__restrict__ status)
{
    constexpr int VE = BF16 ? 8 : 4;
    constexpr int CH = AMAX_THREADS * NV * VE;
    constexpr uint32_t FILL = BF16 ? 0xFF80FF80u : 0xFF800000u;  // -inf
    const int chunk = blockIdx.x, row = blockIdx.y, tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    const int c0 = chunk * CH;
    const int cn = min(CH, V - c0);
    const char *rowp = (const char *)t + (int64_t)row * V * (BF16 ? 2 : 4);

    uint4 raw[NV];
#pragma unroll
    for (int j = 0; j < NV; ++j) {
        const int e0 = (j * AMAX_THREADS + tid) * VE;
        if (ALIGNED && e0 < cn) {
            raw[j] = ldg_stream(rowp + (int64_t)(c0 + e0) * (BF16 ? 2 : 4));
        } else {
            uint32_t w[4] = {FILL, FILL, FILL, FILL};
            if (!ALIGNED)
                for (int e = 0; e < VE; ++e)
                    if (e0 + e < cn) {
                        if (BF16) {
                            const uint32_t h = __ldg((const unsigned short *)rowp + c0 + e0 + e);
                            w[e >> 1] = (e & 1) ? ((w[e >> 1] & 0xFFFFu) | (h << 16))
                                                : ((w[e >> 1] & 0xFFFF0000u) | h);
                        } else {
                            w[e] = __float_as_uint(__ldg((const float *)rowp + c0 + e0 + e));
                        }
                    }
            raw[j] = make_uint4(w[0], w[1], w[2], w[3]);
        }
    }

    // ---- this thread's max (NaN ignored) and whether it holds a NaN
    float m;
    bool nan;
    if (BF16) {
        uint32_t mx = FILL, mn = FILL;
#pragma unroll
        for (int j = 0; j < NV; ++j) {
            mx = bmax2(mx, bmax2(bmax2(raw[j].x, raw[j].y), bmax2(raw[j].z, raw[j].w)));
            mn = bmax2_nan(mn, bmax2_nan(bmax2_nan(raw[j].x, raw[j].y), bmax2_nan(raw[j].z, raw[j].w)));
        }
        m = fmaxf(bf16lo(mx), bf16hi(mx));
        nan = (bf16lo(mn) != bf16lo(mn)) || (bf16hi(mn) != bf16hi(mn));
    } else {
        m = DDT_NEG_INF;
        nan = false;
#pragma unroll
        for (int j = 0; j < NV; ++j) {
            const float x0 = __uint_as_float(raw[j].x), x1 = __uint_as_float(raw[j].y);
            const float x2 = __uint_as_float(raw[j].z), x3 = __uint_as_float(raw[j].w);
            m = fmaxf(m, fmaxf(fmaxf(x0, x1), fmaxf(x2, x3)));
            nan |= (x0 != x0) | (x1 != x1) | (x2 != x2) | (x3 != x3);
        }
    }
    if (m != m)
        m = DDT_NEG_INF;  // every element NaN

    // ---- the chunk's max
    __shared__ uint32_t s_k[AMAX_THREADS / 32];
    __shared__ int s_i[AMAX_THREADS / 32];
    const uint32_t key = fkey(m);
    const uint32_t wk = __reduce_max_sync(0xFFFFFFFFu, key);
    if (lane == 0)
        s_k[warp] = wk;
    const int any_nan = __syncthreads_or(nan ? 1 : 0);
    uint32_t bk = s_k[0];
#pragma unroll
    for (int w = 1; w < AMAX_THREADS / 32; ++w)
        bk = max(bk, s_k[w]);
    const float M = fkey_inv(bk);

    // ---- its first occurrence: only threads whose max equals it look
    int fi = IDX_NONE;
    if (key == bk) {
#pragma unroll
        for (int j = 0; j < NV; ++j) {
            const int e0 = (j * AMAX_THREADS + tid) * VE;
            const uint32_t w[4] = {raw[j].x, raw[j].y, raw[j].z, raw[j].w};
#pragma unroll
            for (int e = 0; e < VE; ++e) {
                const float x = BF16 ? ((e & 1) ? bf16hi(w[e >> 1]) : bf16lo(w[e >> 1]))
                                     : __uint_as_float(w[e]);
                if (fi == IDX_NONE && x == M && e0 + e < cn)
                    fi = c0 + e0 + e;
            }
        }
    }
    fi = __reduce_min_sync(0xFFFFFFFFu, fi);
    if (lane == 0)
        s_i[warp] = fi;
    __syncthreads();
    if (tid == 0) {
        int i = s_i[0];
#pragma unroll
        for (int w = 1; w < AMAX_THREADS / 32; ++w)
            i = min(i, s_i[w]);
        am_val[(int64_t)row * nch + chunk] = M;
        am_idx[(int64_t)row * nch + chunk] = i;
        if (any_nan)
            set_status(status, DDT_DEV_NAN_LOGITS);
    }
}

DDT_DEVINL int reduce_partials(const float *am_val, const int32_t *am_idx, int64_t row, int nch)
{
    float b = DDT_NEG_INF;
    int i = IDX_NONE;
    for (int c = 0; c < nch; ++c)
        amax_merge(b, i, am_val[row * nch + c], am_idx[row * nch + c]);
    return (i == IDX_NONE) ? 0 : i;
}

__global__ void argmax_finish_kernel(const float *__restrict__ am_val,
                                     const int32_t *__restrict__ am_idx, int rows, int nch,
                                     int32_t *__restrict__ out)
{
    const int row = blockIdx.x * blockDim.x + threadIdx.x;
    if (row < rows)
        out[row] = reduce_partials(am_val, am_idx, row, nch);
}

// one CTA per request: argmax reduction, greedy walk, KV compaction
__global__ void __launch_bounds__(128)
walk_compact_kernel(const int32_t *__restrict__ argmax, const float *__restrict__ am_val,
                    const int32_t *__restrict__ am_idx, int nch, int32_t *__restrict__ argmax_out,
                    const int32_t *__restrict__ tree_tokens, const int32_t *__restrict__ parents,
                    const int32_t *__restrict__ n_nodes, int B, int L,
                    int32_t *__restrict__ acc_len, int32_t *__restrict__ acc_nodes,
                    int32_t *__restrict__ acc_tokens, int32_t *__restrict__ bonus, int do_walk,
                    int do_compact, uint16_t *__restrict__ k_cache, uint16_t *__restrict__ v_cache,
                    const int32_t *__restrict__ block_table, int max_pages, int64_t num_pages,
                    int page, int32_t *__restrict__ ctx_lens, const uint16_t *__restrict__ k_tree,
                    const uint16_t *__restrict__ v_tree, int rowlen, int advance_ctx,
                    int32_t *__restrict__ status)
{
    const int r = blockIdx.x, tid = threadIdx.x;
    const int P = B + 1;
    __shared__ int s_a[DDT_MAX_P];
    __shared__ int s_par[DDT_MAX_P];
    __shared__ int s_tok[DDT_MAX_B];
    __shared__ int s_accn[DDT_MAX_L];
    __shared__ int s_nacc, s_ctx, s_bad;

    if (tid == 0) {
        s_bad = 0;
        s_nacc = 0;
    }
    __syncthreads();
    if (do_walk) {
        for (int i = tid; i < P; i += blockDim.x) {
            const int64_t row = (int64_t)r * P + i;
            const int a = (argmax != nullptr) ? argmax[row] : reduce_partials(am_val, am_idx, row, nch);
            s_a[i] = a;
            if (argmax_out != nullptr)
                argmax_out[row] = a;
            s_par[i] = parents[row];
            if (i < B)
                s_tok[i] = tree_tokens[(int64_t)r * B + i];
        }
        __syncthreads();
        if (tid < 32) {
            const int lane = tid;
            int n = n_nodes[r];
            if (n < 0 || n > B) {
                if (lane == 0)
                    s_bad = 1;
                n = (n < 0) ? 0 : B;
            }
            int cur = 0, nacc = 0;
            for (int step = 0; step < L; ++step) {
                const int want = s_a[cur];
                int found = -1;
                for (int base = 1; base <= n && found < 0; base += 32) {
                    const int c = base + lane;
                    const bool m = (c <= n) && s_par[c] == cur && s_tok[c - 1] == want;
                    const unsigned bal = __ballot_sync(0xFFFFFFFFu, m);
                    if (bal)
                        found = base + __ffs(bal) - 1;
                }
                if (found < 0)
                    break;
                if (lane == 0)
                    s_accn[nacc] = found;
                ++nacc;
                cur = found;
            }
            __syncwarp();
            const int bon = s_a[cur];
            for (int j = lane; j <= L; j += 32) {
                if (j < L)
                    acc_nodes[(int64_t)r * L + j] = (j < nacc) ? s_accn[j] : -1;
                int tokv = -1;
                if (j < nacc)
                    tokv = s_tok[s_accn[j] - 1];
                else if (j == nacc)
                    tokv = bon;
                acc_tokens[(int64_t)r * (L + 1) + j] = tokv;
            }
            if (lane == 0) {
                acc_len[r] = nacc + 1;
                bonus[r] = bon;
                s_nacc = nacc;
            }
        }
    } else if (tid == 0) {
        int nacc = acc_len[r] - 1;
        if (nacc < 0 || nacc > L) {
            s_bad = 1;
            nacc = (nacc < 0) ? 0 : L;
        }
        for (int j = 0; j < nacc; ++j) {
            int node = acc_nodes[(int64_t)r * L + j];
            if (node < 1 || node >= P) {
                s_bad = 1;
                node = 0;
            }
            s_accn[j] = node;
        }
        s_nacc = nacc;
    }
    if (do_compact && tid == 0)
        s_ctx = ctx_lens[r];
    __syncthreads();
    if (tid == 0 && s_bad)
        set_status(status, DDT_DEV_BAD_TREE);
    if (!do_compact)
        return;

    const int nacc = s_nacc, ctx = s_ctx;
    const int vecs = rowlen / 8;  // 16-byte vectors per row
    for (int j = 0; j <= nacc; ++j) {
        const int node = (j == 0) ? 0 : s_accn[j - 1];
        const int slot = ctx + j;
        const int pidx = slot / page;
        int pg = -1;
        if (slot >= 0 && pidx < max_pages)
            pg = block_table[(int64_t)r * max_pages + pidx];
        if (pg < 0 || pg >= num_pages) {
            if (tid == 0)
                set_status(status, DDT_DEV_BAD_PAGE);
            continue;
        }
        const int64_t dst = ((int64_t)pg * page + slot % page) * rowlen;
        const int64_t src = ((int64_t)r * P + node) * rowlen;
        for (int v = tid; v < vecs; v += blockDim.x) {
            reinterpret_cast<uint4 *>(k_cache + dst)[v] = reinterpret_cast<const uint4 *>(k_tree + src)[v];
            reinterpret_cast<uint4 *>(v_cache + dst)[v] = reinterpret_cast<const uint4 *>(v_tree + src)[v];
        }
    }
    __syncthreads();
    if (tid == 0 && advance_ctx)
        ctx_lens[r] = ctx + nacc + 1;
}

// the context lengths after compaction: ctx_lens[r] += acc_len[r] (the root
// and the accepted nodes were copied to slots ctx .. ctx + acc_len - 1)
__global__ void ctx_advance_kernel(int32_t *__restrict__ ctx_lens,
                                   const int32_t *__restrict__ acc_len, int R)
{
    const int r = blockIdx.x * blockDim.x + threadIdx.x;
    if (r < R)
        ctx_lens[r] += acc_len[r];
}

}  // namespace

int amax_chunk_elems(int dtype)
{
    return AMAX_THREADS * NV * (dtype == DDT_BF16 ? 8 : 4);
}

cudaError_t launch_argmax_partials(const ddt_ctx *c, const void *t, int R, cudaStream_t s)
{
    const ddt_config &cfg = c->cfg;
    const int rows = R * (cfg.B + 1);
    dim3 grid(c->am_nch, rows);
    const bool bf16 = cfg.target_dtype == DDT_BF16;
    const int esz = bf16 ? 2 : 4;
    const bool aligned = ((int64_t)cfg.V * esz) % 16 == 0 && ((uintptr_t)t % 16) == 0;
    if (bf16) {
        if (aligned)
            argmax_chunk_kernel<true, true><<<grid, AMAX_THREADS, 0, s>>>(t, cfg.V, c->am_nch, c->am_val, c->am_idx, c->status);
        else
            argmax_chunk_kernel<true, false><<<grid, AMAX_THREADS, 0, s>>>(t, cfg.V, c->am_nch, c->am_val, c->am_idx, c->status);
    } else {
        if (aligned)
            argmax_chunk_kernel<false, true><<<grid, AMAX_THREADS, 0, s>>>(t, cfg.V, c->am_nch, c->am_val, c->am_idx, c->status);
        else
            argmax_chunk_kernel<false, false><<<grid, AMAX_THREADS, 0, s>>>(t, cfg.V, c->am_nch, c->am_val, c->am_idx, c->status);
    }
    return cudaGetLastError();
}

cudaError_t launch_argmax_finish(const ddt_ctx *c, int R, int32_t *argmax_out, cudaStream_t s)
{
    const int rows = R * (c->cfg.B + 1);
    argmax_finish_kernel<<<(rows + 127) / 128, 128, 0, s>>>(c->am_val, c->am_idx, rows, c->am_nch,
                                                            argmax_out);
    return cudaGetLastError();
}

cudaError_t launch_walk_compact(const ddt_ctx *c, const int32_t *argmax, bool argmax_from_partials,
                                int32_t *argmax_out, const int32_t *tree_tokens,
                                const int32_t *parents, const int32_t *n_nodes, int R,
                                int32_t *acc_len, int32_t *acc_nodes, int32_t *acc_tokens,
                                int32_t *bonus, bool do_walk, bool do_compact, uint16_t *k_cache,
                                uint16_t *v_cache, const int32_t *block_table, int32_t *ctx_lens,
                                const uint16_t *k_tree, const uint16_t *v_tree, bool advance_ctx,
                                cudaStream_t s)
{
    const ddt_config &cfg = c->cfg;
    walk_compact_kernel<<<R, 128, 0, s>>>(
        argmax_from_partials ? nullptr : argmax, c->am_val, c->am_idx, c->am_nch, argmax_out,
        tree_tokens, parents, n_nodes, cfg.B, cfg.L, acc_len, acc_nodes, acc_tokens, bonus,
        do_walk ? 1 : 0, do_compact ? 1 : 0, k_cache, v_cache, block_table, cfg.max_pages_per_req,
        cfg.num_pages, cfg.page_size, ctx_lens, k_tree, v_tree, cfg.Hkv * cfg.d,
        advance_ctx ? 1 : 0, c->status);
    return cudaGetLastError();
}

cudaError_t launch_ctx_advance(int R, int32_t *ctx_lens, const int32_t *acc_len, cudaStream_t s)
{
    ctx_advance_kernel<<<(R + 127) / 128, 128, 0, s>>>(ctx_lens, acc_len, R);
    return cudaGetLastError();
}
