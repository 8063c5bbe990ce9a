// stochastic.cu -- stochastic verification of a drafted chain at temperature
// 1 ("DSpark Speculative Decoding Explained: Block Drafting and Confidence
// Checks", the probability rule): guess x_k is kept with probability
// min(1, p_k(x_k) / q_k(x_k)); the first rejected guess is replaced by a draw
// from max(0, p_k - q_k) and the guesses after it are dropped; when every
// guess survives, a bonus token is drawn from p_L. The uniforms are inputs:
// u[k] decides guess k (kept iff u[k] < min(1, p/q)); r draws by inverse CDF
// over the vocabulary in index order (the first index whose running sum of
// weights exceeds r times their total). With per-request guess counts (the
// prefix a scheduler kept), request i verifies only its first n_i guesses;
// when all of them survive, the bonus comes from p_{n_i}.
//
// Design (HBM-bound: every logit is read once, the drawn row once more):
//  * sv_rows_kernel: one CTA per (request, row, chunk of 32 KB); each
//    thread keeps 8 vectors of 16 bytes in registers and the CTA reduces
//    them to the chunk's (max, sum of exp), stores the pair and exits.
//  * sv_rows_counted_kernel (given guess counts): the same per-chunk work on
//    a grid of a few waves, each CTA over a contiguous range of only the
//    used rows' chunks (draft rows k < n_i, target rows k <= n_i).
//  * sv_draw_kernel (a dependent launch): one CTA per (request, 8192 tokens
//    of the drawn row). Every CTA of a request first takes the request's
//    decisions itself -- the log-partitions of its used rows from the
//    pairs (staged in shared memory, or a warp per row when they do not
//    fit), the guesses' log-probs, the n_i decisions in one
//    warp (a ballot finds the first rejection k*) -- the same loads in the
//    same order, so all agree; the request's first CTA writes the committed
//    prefix and the length. Then each sums the draw's weights of its chunk
//    of row k*; the last CTA of the request (an arrival counter) adds the
//    chunk totals in index order, finds the chunk that holds r * total,
//    re-reads that chunk in index order (32 consecutive weights per thread,
//    a block scan) and picks the first index whose running sum exceeds it.
#include <cuda_runtime.h>
#include <algorithm>
#include <math.h>
#include <stdint.h>

#include "ddt_device.cuh"
#include "ddt_internal.h"
#include "logit_vec.cuh"

namespace {

constexpr int SV_THREADS = 256;
constexpr int SV_NV = 8;                   // 16-byte vectors per thread in the row pass
constexpr int SV_WPT = 32;                 // weights per thread in the draw
constexpr int SV_WCH = SV_THREADS * SV_WPT;  // weights per CTA of the draw (8192)
constexpr int SV_DEC_PAIRS = 1024;           // chunk pairs a request's decision stages in smem
constexpr int SV_ROW_WAVES = 2;  // counted row pass: CTAs = SMs x 5 resident x this

// ---------------------------------------------------------------- row pass
// (max, sum of exp(x - max)) of one chunk of a row, for the whole CTA; the
// result is valid in thread 0
template <typename T, bool ALIGNED>
DDT_DEVINL void chunk_ms(const T *__restrict__ zrow, int c0, int cn, float &M, float &S,
                         float *s_m, float *s_s)
{
    constexpr int VE = Elem<T>::VE;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    uint4 raw[SV_NV];
#pragma unroll
    for (int j = 0; j < SV_NV; ++j) {
        const int e0 = (j * SV_THREADS + tid) * VE;
        if (ALIGNED) {
            if (e0 < cn)
                raw[j] = ldg_stream(zrow + c0 + e0);
            else
                raw[j] = make_uint4(Elem<T>::NEG_INF_FILL, Elem<T>::NEG_INF_FILL,
                                    Elem<T>::NEG_INF_FILL, Elem<T>::NEG_INF_FILL);
        } else {
            raw[j] = load_scalar<T>(zrow + c0 + e0, e0 < cn ? min(VE, cn - e0) : 0);
        }
    }
    float m = DDT_NEG_INF;
#pragma unroll
    for (int j = 0; j < SV_NV; ++j)
        m = fmaxf(m, vec_max<T>(raw[j]));
    float s = 0.f;
    if (m != DDT_NEG_INF) {
        const float nb = -m * DDT_LOG2E;
        if constexpr (sizeof(T) == 2) {
            const uint64_t c2 = f2pack(DDT_LOG2E, DDT_LOG2E), b2 = f2pack(nb, nb);
            uint64_t acc0 = f2pack(0.f, 0.f), acc1 = acc0;
#pragma unroll
            for (int j = 0; j < SV_NV; ++j) {
                acc0 = f2add(acc0, exp_pair(raw[j].x, c2, b2));
                acc1 = f2add(acc1, exp_pair(raw[j].y, c2, b2));
                acc0 = f2add(acc0, exp_pair(raw[j].z, c2, b2));
                acc1 = f2add(acc1, exp_pair(raw[j].w, c2, b2));
            }
            float a0, a1, a2, a3;
            f2unpack(acc0, a0, a1);
            f2unpack(acc1, a2, a3);
            s = (a0 + a1) + (a2 + a3);
        } else {
#pragma unroll
            for (int j = 0; j < SV_NV; ++j)
#pragma unroll
                for (int e = 0; e < VE; ++e)
                    s += ex2(fmaf(Elem<T>::get(raw[j], e), DDT_LOG2E, nb));
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float mo = __shfl_xor_sync(0xFFFFFFFFu, m, o);
        const float so = __shfl_xor_sync(0xFFFFFFFFu, s, o);
        ms_combine(m, s, mo, so);
    }
    if (lane == 0) {
        s_m[warp] = m;
        s_s[warp] = s;
    }
    __syncthreads();
    if (tid == 0) {
        M = s_m[0];
        S = s_s[0];
        for (int w = 1; w < SV_THREADS / 32; ++w)
            ms_combine(M, S, s_m[w], s_s[w]);
    }
}

// the guesses request i verifies: n_guess[i] clamped to [0, L], or L
DDT_DEVINL int guesses_of(const int32_t *n_guess, int i, int L)
{
    if (n_guess == nullptr)
        return L;
    const int n = n_guess[i];
    return n < 0 ? 0 : (n > L ? L : n);
}

// one logit of a row (the guess's), as fp32
template <typename T>
DDT_DEVINL float logit_at(const T *row, int x)
{
    if constexpr (sizeof(T) == 2)
        return bf16_to_f32(row[x]);
    else
        return row[x];
}

struct RowsArgs {
    const void *draft;        // [R, L, V] draft logits
    const void *target;       // [R, L + 1, V] target logits
    float2 *part_d, *part_t;  // chunk (max, sum) pairs of the draft / target rows
    const int32_t *n_guess;   // [R] guesses verified per request, or nullptr (L)
    int32_t *status;
    int L, V, nch_d, nch_t;
    bool al_d, al_t;          // 16-byte aligned rows
};

// one item of the row pass: chunk c of draft row k (isd) or target row k of
// request i; thread 0 stores the chunk's (max, sum) pair
template <typename TD, typename TT>
DDT_DEVINL void row_item(const RowsArgs &a, int i, bool isd, int k, int c, float *s_m,
                         float *s_s)
{
    const int L = a.L, V = a.V;
    float M = 0.f, S = 0.f;
    float2 *slot;
    if (isd) {  // a draft row
        const int row = i * L + k;
        constexpr int CH = SV_THREADS * SV_NV * Elem<TD>::VE;
        const TD *z = static_cast<const TD *>(a.draft) + (int64_t)row * V;
        if (a.al_d)
            chunk_ms<TD, true>(z, c * CH, min(CH, V - c * CH), M, S, s_m, s_s);
        else
            chunk_ms<TD, false>(z, c * CH, min(CH, V - c * CH), M, S, s_m, s_s);
        slot = a.part_d + (int64_t)row * a.nch_d + c;
    } else {  // a target row
        const int row = i * (L + 1) + k;
        constexpr int CH = SV_THREADS * SV_NV * Elem<TT>::VE;
        const TT *z = static_cast<const TT *>(a.target) + (int64_t)row * V;
        if (a.al_t)
            chunk_ms<TT, true>(z, c * CH, min(CH, V - c * CH), M, S, s_m, s_s);
        else
            chunk_ms<TT, false>(z, c * CH, min(CH, V - c * CH), M, S, s_m, s_s);
        slot = a.part_t + (int64_t)row * a.nch_t + c;
    }
    if (threadIdx.x == 0) {
        if (M != M || S != S)
            set_status(a.status, DDT_DEV_NAN_LOGITS);
        *slot = make_float2(M, S);
    }
}

// grid: R * (L * nch_d + (L + 1) * nch_t) CTAs, request-major; each stores
// its chunk's (max, sum) pair and exits (the decisions are taken by the
// draw kernel, which waits for this whole grid)
template <typename TD, typename TT>
__global__ void __launch_bounds__(SV_THREADS, 5)  // 48 registers: five CTAs per SM
sv_rows_kernel(RowsArgs a)
{
    const int L = a.L;
    const int per = L * a.nch_d + (L + 1) * a.nch_t;
    const int i = blockIdx.x / per, j = blockIdx.x % per;
    __shared__ float s_m[SV_THREADS / 32], s_s[SV_THREADS / 32];
    pdl_trigger();

    // which row (k) and chunk (c); rows past the request's verified guesses
    // are never read, so their CTAs do nothing
    const bool isd = j < L * a.nch_d;
    const int jj = isd ? j : j - L * a.nch_d, nch = isd ? a.nch_d : a.nch_t;
    const int k = jj / nch;
    const int n = guesses_of(a.n_guess, i, L);
    if (isd ? k >= n : k > n)
        return;
    row_item<TD, TT>(a, i, isd, k, jj - k * nch, s_m, s_s);
}

// The row pass for given guess counts: only the items of the rows the
// requests verify (n_i * nch_d + (n_i + 1) * nch_t for request i), numbered
// request-major, draft rows before target rows. Each CTA first turns the
// counts into every request's first item (in shared memory: s_first [R + 1],
// then s_n [R]), then takes a contiguous range of the items: a binary search
// finds its first item's request, and the rest follow in order. No CTA is launched only to find its row unused.
template <typename TD, typename TT>
__global__ void __launch_bounds__(SV_THREADS, 5)
sv_rows_counted_kernel(RowsArgs a, int R)
{
    extern __shared__ int s_dyn[];
    int *s_first = s_dyn, *s_n = s_dyn + R + 1;
    __shared__ float s_m[SV_THREADS / 32], s_s[SV_THREADS / 32];
    __shared__ int s_wsum[SV_THREADS / 32];
    pdl_trigger();
    const int L = a.L, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    // each thread sums a contiguous run of requests, then a block scan
    const int run = (R + SV_THREADS - 1) / SV_THREADS;
    const int r0 = min(R, tid * run), r1 = min(R, r0 + run);
    int own = 0;
    for (int i = r0; i < r1; ++i) {
        const int n = guesses_of(a.n_guess, i, L);
        s_n[i] = n;
        own += n * a.nch_d + (n + 1) * a.nch_t;
    }
    int incl = own;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o)
            incl += v;
    }
    if (lane == 31)
        s_wsum[warp] = incl;
    __syncthreads();
    int first = incl - own;
    for (int w = 0; w < warp; ++w)
        first += s_wsum[w];
    for (int i = r0; i < r1; ++i) {
        s_first[i] = first;
        first += s_n[i] * a.nch_d + (s_n[i] + 1) * a.nch_t;
    }
    if (tid == SV_THREADS - 1)  // its run ends at R: first is the total
        s_first[R] = first;
    __syncthreads();

    const int total = s_first[R];
    const int span = (total + gridDim.x - 1) / gridDim.x;
    int q = blockIdx.x * span;
    const int qe = min(total, q + span);
    if (q >= qe)
        return;
    // the first item's request: the last i with s_first[i] <= q (every
    // request has at least one item, target row 0)
    int i = 0, hi = R - 1;
    while (i < hi) {
        const int mid = (i + hi + 1) >> 1;
        if (s_first[mid] <= q)
            i = mid;
        else
            hi = mid - 1;
    }
    int n = s_n[i], j = q - s_first[i];  // j: the item within request i
    for (int left = qe - q;;) {
        const int nd = n * a.nch_d;
        const bool isd = j < nd;
        const int jj = isd ? j : j - nd, nch = isd ? a.nch_d : a.nch_t;
        const int k = jj / nch;
        row_item<TD, TT>(a, i, isd, k, jj - k * nch, s_m, s_s);
        if (--left == 0)
            break;
        __syncthreads();  // s_m / s_s are reused by the next item
        if (++j == nd + (n + 1) * a.nch_t) {  // past request i's last item
            ++i;  // items remain: request i exists
            n = s_n[i];
            j = 0;
        }
    }
}

// ---------------------------------------------------------------- the draw
struct DrawArgs {
    const void *draft, *target;
    const int32_t *tokens;          // [R, L] the guesses
    const float *u;                 // [R, L] acceptance uniforms
    const float *r;                 // [R] draw uniforms
    const float2 *part_d, *part_t;  // from sv_rows_kernel
    const int32_t *n_guess;         // [R] guesses verified per request, or nullptr (L)
    float *part_w;                  // [R, nchw] chunk totals of the weights
    unsigned *cnt;                  // [R] arrivals (self-resetting)
    int32_t *acc_len;               // [R]
    int32_t *acc_tokens;            // [R, L + 1]
    int32_t *status;
    int L, V, nchw, nch_d, nch_t;
    bool al_d, al_t;  // (host side: selects the kernel)
};

// Request i's decisions, taken by every CTA of the draw that works on it (the
// same loads in the same order, so each gets the same answer): the
// log-partitions of its 2L + 1 rows from the chunk pairs (a warp per row,
// lanes over chunks), the guesses' log-probs, then the L decisions in warp 0
// (kept iff u < min(1, p/q); a ballot finds the first rejection k*). The CTA
// with `writer` set also stores the length and every committed token but the
// drawn one. Returns k*; s_lse[t] holds the log-partition of row t (draft rows
// 0..L-1, then target rows 0..L). Only the rows the request verifies are
// touched: draft rows k < n and target rows k <= n, n = its guess count.
template <typename TD, typename TT>
__device__ __noinline__ int decide(const DrawArgs &a, int i, bool writer, float *s_lse,
                                   float *s_lz, int *s_ks, float2 *s_pairs)
{
    const int L = a.L, V = a.V;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const TD *zd = static_cast<const TD *>(a.draft) + (int64_t)i * L * V;
    const TT *zt = static_cast<const TT *>(a.target) + (int64_t)i * (L + 1) * V;
    const int nd = L * a.nch_d, nt = (L + 1) * a.nch_t;
    const int n = guesses_of(a.n_guess, i, L);
    // row t (as in s_lse) is one the request verifies
    auto used = [&](int t) { return t < L ? t < n : t - L <= n; };
    if (nd + nt <= SV_DEC_PAIRS) {
        // every pair of the request and the guess logits at once (one round
        // trip), then a thread per row merges its pairs from shared memory
        const float2 *pd = a.part_d + (int64_t)i * nd, *pt = a.part_t + (int64_t)i * nt;
        const int ud = n * a.nch_d, ut = (n + 1) * a.nch_t;  // pairs of the used rows
        for (int q = tid; q < nd + nt; q += SV_THREADS)
            if (q < nd ? q < ud : q - nd < ut)
                s_pairs[q] = q < nd ? __ldcg(pd + q) : __ldcg(pt + (q - nd));
        for (int q = tid; q < 2 * L; q += SV_THREADS) {
            const int k = q < L ? q : q - L;
            float zx = 0.f;
            if (k < n) {
                const int x = a.tokens[(int64_t)i * L + k];
                if (x >= 0 && x < V)
                    zx = q < L ? logit_at(zd + (int64_t)k * V, x)
                               : logit_at(zt + (int64_t)k * V, x);
            }
            s_lz[q] = zx;
        }
        __syncthreads();
        if (tid < 2 * L + 1 && used(tid)) {
            const int t = tid;
            const float2 *pp = t < L ? s_pairs + t * a.nch_d : s_pairs + nd + (t - L) * a.nch_t;
            const int nch = t < L ? a.nch_d : a.nch_t;
            float m = DDT_NEG_INF, sm = 0.f;
            for (int c = 0; c < nch; ++c)
                ms_combine(m, sm, pp[c].x, pp[c].y);
            const float lse = m + logf(sm);
            s_lse[t] = lse;
            if (t < 2 * L)
                s_lz[t] -= lse;
        }
    } else {
        for (int t = warp; t < 2 * L + 1; t += SV_THREADS / 32) {
            if (!used(t))
                continue;
            const bool isd = t < L;
            const int k = isd ? t : t - L;
            const int nch = isd ? a.nch_d : a.nch_t;
            const float2 *part = isd ? a.part_d + ((int64_t)i * L + k) * nch
                                     : a.part_t + ((int64_t)i * (L + 1) + k) * nch;
            float zx = 0.f;  // the guess's logit, loaded beside the pairs
            if (lane == 0 && k < n) {
                const int x = a.tokens[(int64_t)i * L + k];
                if (x >= 0 && x < V)
                    zx = isd ? logit_at(zd + (int64_t)k * V, x) : logit_at(zt + (int64_t)k * V, x);
            }
            float m = DDT_NEG_INF, sm = 0.f;
            for (int c = lane; c < nch; c += 32) {
                const float2 p = __ldcg(part + c);
                ms_combine(m, sm, p.x, p.y);
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const float mo = __shfl_xor_sync(0xFFFFFFFFu, m, o);
                const float so = __shfl_xor_sync(0xFFFFFFFFu, sm, o);
                ms_combine(m, sm, mo, so);
            }
            if (lane == 0) {
                const float lse = m + logf(sm);
                s_lse[t] = lse;
                s_lz[t] = zx - lse;
            }
        }
    }
    __syncthreads();
    if (warp == 0) {
        if (writer && lane == 0 && a.n_guess != nullptr && n != a.n_guess[i])
            set_status(a.status, DDT_DEV_BAD_TREE);
        bool keep = false;
        if (lane < n) {
            const int x = a.tokens[(int64_t)i * L + lane];
            const bool ok = x >= 0 && x < V;
            if (!ok && writer)
                set_status(a.status, DDT_DEV_BAD_TREE);
            // min(1, p/q) from the two log-probs; q = 0 gives +inf (or NaN
            // when p = 0 too), which fminf takes to 1
            const float ratio = fminf(1.f, expf(s_lz[L + lane] - s_lz[lane]));
            keep = ok && a.u[(int64_t)i * L + lane] < ratio;
        }
        const unsigned kept = __ballot_sync(0xFFFFFFFFu, keep);
        const int ks = __ffs(~kept) - 1;  // lanes >= n never keep: ks <= n
        if (lane == 0)
            *s_ks = ks;
        if (writer) {
            if (lane == 0)
                a.acc_len[i] = ks + 1;
            for (int t = lane; t <= L; t += 32)
                if (t != ks)
                    a.acc_tokens[(int64_t)i * (L + 1) + t] =
                        t < ks ? a.tokens[(int64_t)i * L + t] : -1;
        }
    }
    __syncthreads();
    return *s_ks;
}

// one group of 8 consecutive logits (v0 a multiple of 8) as raw 16-byte
// vectors: one for bf16, two for fp32; -inf past V
template <typename T> struct Grp {
    static constexpr int NU = sizeof(T) / 2;  // 16-byte vectors per group
    static constexpr int VE = Elem<T>::VE;
    uint4 u[NU];
    DDT_DEVINL float at(int e) const { return Elem<T>::get(u[e / VE], e % VE); }
};

template <typename T, bool AL>
DDT_DEVINL void ld_group(const T *__restrict__ row, int v0, int V, Grp<T> &g)
{
    constexpr int NU = Grp<T>::NU, VE = Grp<T>::VE;
    if (AL && v0 + 8 <= V) {
#pragma unroll
        for (int k = 0; k < NU; ++k)
            g.u[k] = __ldcg(reinterpret_cast<const uint4 *>(row + v0) + k);
    } else {
#pragma unroll
        for (int k = 0; k < NU; ++k) {
            const int n = V - (v0 + k * VE);
            g.u[k] = load_scalar<T>(row + v0 + k * VE, n <= 0 ? 0 : (n < VE ? n : VE));
        }
    }
}

// the draw's weight of one token: p - q clipped at 0 after a rejection,
// p alone for the bonus draw; p = 2^(z log2 e - log Z log2 e) on the MUFU unit
DDT_DEVINL float draw_weight(float zt, float zd, float bt, float bd, bool leftover)
{
    const float p = ex2(fmaf(zt, DDT_LOG2E, bt));
    if (!leftover)
        return p;
    const float q = ex2(fmaf(zd, DDT_LOG2E, bd));
    return p > q ? p - q : 0.f;
}

constexpr int SV_G = SV_WPT / 8;  // groups of 8 weights per thread
constexpr int SV_GH = 4;          // groups loaded at once (registers)

// sum of the draw's weights of tokens v0 .. v0 + SV_WPT - 1 (in index order)
template <typename TD, typename TT, bool AD, bool AT>
DDT_DEVINL float thread_sum(const TT *zt, const TD *zd, int v0, int V, float bt, float bd,
                            bool leftover)
{
    float s = 0.f;
#pragma unroll
    for (int h = 0; h < SV_G; h += SV_GH) {
        Grp<TT> gt[SV_GH];
        Grp<TD> gd[SV_GH];
#pragma unroll
        for (int g = 0; g < SV_GH; ++g)
            ld_group<TT, AT>(zt, v0 + (h + g) * 8, V, gt[g]);
        if (leftover) {
#pragma unroll
            for (int g = 0; g < SV_GH; ++g)
                ld_group<TD, AD>(zd, v0 + (h + g) * 8, V, gd[g]);
        }
#pragma unroll
        for (int g = 0; g < SV_GH; ++g)
#pragma unroll
            for (int e = 0; e < 8; ++e)
                s += draw_weight(gt[g].at(e), leftover ? gd[g].at(e) : 0.f, bt, bd, leftover);
    }
    return s;
}

// tokens v0 .. v0 + SV_WPT - 1 with running sum `cum` before them: the first positive
// weight whose running sum exceeds x, else (x = +inf) the last positive one
template <typename TD, typename TT, bool AD, bool AT>
__device__ __noinline__ int fine_search(const TT *zt, const TD *zd, int v0, int V, float bt,
                                        float bd, bool leftover, float cum, float x)
{
    int last = -1;
    for (int g = 0; g < SV_G; ++g) {
        Grp<TT> gt;
        Grp<TD> gd;
        ld_group<TT, AT>(zt, v0 + g * 8, V, gt);
        if (leftover)
            ld_group<TD, AD>(zd, v0 + g * 8, V, gd);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const float w = draw_weight(gt.at(e), leftover ? gd.at(e) : 0.f, bt, bd, leftover);
            cum += w;
            if (w > 0.f) {
                last = v0 + g * 8 + e;
                if (cum > x)
                    return last;
            }
        }
    }
    return last;
}

template <typename TD, typename TT, bool AD, bool AT>
DDT_DEVINL void draw_body(const DrawArgs &a, int i, int c)
{
    const int L = a.L, V = a.V;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    __shared__ float s_w[SV_THREADS / 32];
    __shared__ int s_last, s_chunk, s_pick, s_ks;
    __shared__ float s_x;
    __shared__ float s_lse[2 * DDT_MAX_L + 1], s_lz[2 * DDT_MAX_L + 1];
    __shared__ float2 s_pairs[SV_DEC_PAIRS];

    const int ks = decide<TD, TT>(a, i, c == 0, s_lse, s_lz, &s_ks, s_pairs);
    // a rejection draws from the leftover; all verified guesses kept, the
    // bonus from target row ks
    const bool leftover = ks < guesses_of(a.n_guess, i, L);
    const float bt = -s_lse[L + ks] * DDT_LOG2E;
    const float bd = leftover ? -s_lse[ks] * DDT_LOG2E : 0.f;
    const TT *zt = static_cast<const TT *>(a.target) + ((int64_t)i * (L + 1) + ks) * V;
    const TD *zd = static_cast<const TD *>(a.draft) + ((int64_t)i * L + (leftover ? ks : 0)) * V;

    // ---- this chunk's total: the loads of SV_GH groups issued before their
    // arithmetic; groups of 8 tokens interleaved across threads (coalesced)
    float t = 0.f;
#pragma unroll
    for (int h = 0; h < SV_G; h += SV_GH) {
        Grp<TT> gt[SV_GH];
        Grp<TD> gd[SV_GH];
#pragma unroll
        for (int g = 0; g < SV_GH; ++g)
            ld_group<TT, AT>(zt, c * SV_WCH + ((h + g) * SV_THREADS + tid) * 8, V, gt[g]);
        if (leftover) {
#pragma unroll
            for (int g = 0; g < SV_GH; ++g)
                ld_group<TD, AD>(zd, c * SV_WCH + ((h + g) * SV_THREADS + tid) * 8, V, gd[g]);
        }
#pragma unroll
        for (int g = 0; g < SV_GH; ++g)
#pragma unroll
            for (int e = 0; e < 8; ++e)
                t += draw_weight(gt[g].at(e), leftover ? gd[g].at(e) : 0.f, bt, bd, leftover);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        t += __shfl_xor_sync(0xFFFFFFFFu, t, o);
    if (lane == 0)
        s_w[warp] = t;
    __syncthreads();
    if (tid == 0) {
        float ct = 0.f;
        for (int w = 0; w < SV_THREADS / 32; ++w)
            ct += s_w[w];
        a.part_w[(int64_t)i * a.nchw + c] = ct;
        __threadfence();
        const unsigned prev = atomicAdd(&a.cnt[i], 1u);
        s_last = (prev == (unsigned)a.nchw - 1u);
        if (s_last)
            a.cnt[i] = 0u;
    }
    __syncthreads();
    if (!s_last)
        return;
    __threadfence();

    // ---- the request's last CTA. Warp 0: the weights' total W (fp64), then
    // the first chunk whose running total (fp64, index order) exceeds r * W
    if (warp == 0) {
        const float *pw = a.part_w + (int64_t)i * a.nchw;
        double W = 0.0;
        int lastpos = -1;
        for (int b = 0; b < a.nchw; b += 32) {
            const float tk = (b + lane < a.nchw) ? __ldcg(pw + b + lane) : 0.f;
            double s = tk;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1)
                s += __shfl_xor_sync(0xFFFFFFFFu, s, o);
            W += s;
            const unsigned pos = __ballot_sync(0xFFFFFFFFu, tk > 0.f);
            if (pos)
                lastpos = b + 31 - __clz(pos);
        }
        const double x = (double)a.r[i] * W;
        double run = 0.0;
        int found = -1;
        float xin = 0.f;
        for (int b = 0; b < a.nchw && found < 0; b += 32) {
            const float tk = (b + lane < a.nchw) ? __ldcg(pw + b + lane) : 0.f;
            double incl = tk;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const double y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
                if (lane >= o)
                    incl += y;
            }
            incl += run;
            const unsigned hit = __ballot_sync(0xFFFFFFFFu, incl > x);
            if (hit) {
                const int l = __ffs(hit) - 1;
                found = b + l;
                xin = (float)(x - __shfl_sync(0xFFFFFFFFu, incl - (double)tk, l));
            }
            run = __shfl_sync(0xFFFFFFFFu, incl, 31);
        }
        if (lane == 0) {
            if (found < 0) {  // x at the total (rounding, or no weight at all)
                s_chunk = lastpos;
                s_x = __builtin_huge_valf();
            } else {
                s_chunk = found;
                s_x = xin;
            }
            s_pick = 0x7FFFFFFF;
        }
    }
    __syncthreads();
    const int ch = s_chunk;
    int tok = -1;
    if (ch >= 0) {
        // SV_WPT consecutive weights per thread (index order): each thread's sum,
        // an exclusive scan over threads, then the first thread whose range
        // reaches x re-reads its SV_WPT tokens and finds the crossing one
        const float xin = s_x;
        const int v0 = ch * SV_WCH + tid * SV_WPT;
        const float st = thread_sum<TD, TT, AD, AT>(zt, zd, v0, V, bt, bd, leftover);
        float incl = st;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
            if (lane >= o)
                incl += y;
        }
        if (lane == 31)
            s_w[warp] = incl;
        __syncthreads();
        float cum = incl - st;
        for (int q = 0; q < warp; ++q)
            cum += s_w[q];
        if (st > 0.f && cum + st > xin)
            atomicMin(&s_pick, tid);
        __syncthreads();
        int who = s_pick;
        const bool crossed = who != 0x7FFFFFFF;
        if (!crossed) {  // rounding left x past the chunk's sum: its last weight
            __syncthreads();
            if (tid == 0)
                s_pick = -1;
            __syncthreads();
            if (st > 0.f)
                atomicMax(&s_pick, tid);
            __syncthreads();
            who = s_pick;
        }
        __syncthreads();
        if (tid == who)
            s_pick = fine_search<TD, TT, AD, AT>(zt, zd, v0, V, bt, bd, leftover, cum,
                                                crossed ? xin : __builtin_huge_valf());
        __syncthreads();
        tok = who >= 0 ? s_pick : -1;
    }
    if (tid == 0)
        a.acc_tokens[(int64_t)i * (L + 1) + ks] = tok;
}

// grid (nchw, R): one CTA per (chunk of the drawn row, request); AL: both
// logit tensors have 16-byte aligned rows
template <typename TD, typename TT, bool AL>
__global__ void __launch_bounds__(SV_THREADS, sizeof(TD) + sizeof(TT) == 8 ? 3 : 4)
sv_draw_kernel(DrawArgs a)
{
    pdl_wait();  // the chunk pairs come from sv_rows_kernel
    draw_body<TD, TT, AL, AL>(a, blockIdx.y, blockIdx.x);
}

}  // namespace

int stochastic_chunk_elems(int dtype)
{
    return SV_THREADS * SV_NV * (dtype == DDT_BF16 ? 8 : 4);
}

int stochastic_draw_chunks(int V)
{
    return (V + SV_WCH - 1) / SV_WCH;
}

cudaError_t launch_accept_stochastic(const ddt_ctx *c, const void *draft, const void *target,
                                     const int32_t *tokens, const float *u, const float *r, int R,
                                     const int32_t *n_guess, int32_t *acc_len, int32_t *acc_tokens,
                                     cudaStream_t s)
{
    const ddt_config &cfg = c->cfg;
    const int L = cfg.L, V = cfg.V;
    const int esd = cfg.draft_dtype == DDT_BF16 ? 2 : 4, est = cfg.target_dtype == DDT_BF16 ? 2 : 4;
    RowsArgs ra;
    ra.draft = draft;
    ra.target = target;
    ra.part_d = c->sv_part_d;
    ra.part_t = c->sv_part_t;
    ra.n_guess = n_guess;
    ra.status = c->status;
    ra.L = L;
    ra.V = V;
    ra.nch_d = c->sv_nch_d;
    ra.nch_t = c->sv_nch_t;
    ra.al_d = ((int64_t)V * esd) % 16 == 0 && ((uintptr_t)draft % 16) == 0;
    ra.al_t = ((int64_t)V * est) % 16 == 0 && ((uintptr_t)target % 16) == 0;
    const int64_t nrows = (int64_t)R * (L * ra.nch_d + (L + 1) * ra.nch_t);
    if (nrows > 0x7FFFFFFF)
        return cudaErrorInvalidConfiguration;
    const bool bd = cfg.draft_dtype == DDT_BF16, bt = cfg.target_dtype == DDT_BF16;
    if (n_guess != nullptr) {
        // only the used rows' items, over a grid of a few waves; R <= R_max
        // <= 2048 keeps the (2R + 1) ints of shared memory within 16 KB
        const unsigned grid = (unsigned)std::min<int64_t>(nrows, (int64_t)c->num_sms * 5 * SV_ROW_WAVES);
        const size_t sm = (size_t)(2 * R + 1) * sizeof(int);
        if (bd && bt)
            sv_rows_counted_kernel<uint16_t, uint16_t><<<grid, SV_THREADS, sm, s>>>(ra, R);
        else if (bd)
            sv_rows_counted_kernel<uint16_t, float><<<grid, SV_THREADS, sm, s>>>(ra, R);
        else if (bt)
            sv_rows_counted_kernel<float, uint16_t><<<grid, SV_THREADS, sm, s>>>(ra, R);
        else
            sv_rows_counted_kernel<float, float><<<grid, SV_THREADS, sm, s>>>(ra, R);
    } else if (bd && bt)
        sv_rows_kernel<uint16_t, uint16_t><<<(unsigned)nrows, SV_THREADS, 0, s>>>(ra);
    else if (bd)
        sv_rows_kernel<uint16_t, float><<<(unsigned)nrows, SV_THREADS, 0, s>>>(ra);
    else if (bt)
        sv_rows_kernel<float, uint16_t><<<(unsigned)nrows, SV_THREADS, 0, s>>>(ra);
    else
        sv_rows_kernel<float, float><<<(unsigned)nrows, SV_THREADS, 0, s>>>(ra);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return e;

    DrawArgs da;
    da.draft = draft;
    da.target = target;
    da.tokens = tokens;
    da.u = u;
    da.r = r;
    da.part_d = c->sv_part_d;
    da.part_t = c->sv_part_t;
    da.n_guess = n_guess;
    da.part_w = c->sv_part_w;
    da.cnt = c->sv_cnt;
    da.acc_len = acc_len;
    da.acc_tokens = acc_tokens;
    da.status = c->status;
    da.L = L;
    da.V = V;
    da.nchw = c->sv_nch_w;
    da.nch_d = c->sv_nch_d;
    da.nch_t = c->sv_nch_t;
    da.al_d = ra.al_d;
    da.al_t = ra.al_t;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3((unsigned)da.nchw, (unsigned)R);
    lc.blockDim = dim3(SV_THREADS);
    lc.dynamicSmemBytes = 0;
    lc.stream = s;
    lc.attrs = attr;
    lc.numAttrs = 1;
    const bool al = da.al_d && da.al_t;
    if (bd && bt)
        e = al ? cudaLaunchKernelEx(&lc, sv_draw_kernel<uint16_t, uint16_t, true>, da)
               : cudaLaunchKernelEx(&lc, sv_draw_kernel<uint16_t, uint16_t, false>, da);
    else if (bd)
        e = al ? cudaLaunchKernelEx(&lc, sv_draw_kernel<uint16_t, float, true>, da)
               : cudaLaunchKernelEx(&lc, sv_draw_kernel<uint16_t, float, false>, da);
    else if (bt)
        e = al ? cudaLaunchKernelEx(&lc, sv_draw_kernel<float, uint16_t, true>, da)
               : cudaLaunchKernelEx(&lc, sv_draw_kernel<float, uint16_t, false>, da);
    else
        e = al ? cudaLaunchKernelEx(&lc, sv_draw_kernel<float, float, true>, da)
               : cudaLaunchKernelEx(&lc, sv_draw_kernel<float, float, false>, da);
    return e != cudaSuccess ? e : cudaGetLastError();
}
