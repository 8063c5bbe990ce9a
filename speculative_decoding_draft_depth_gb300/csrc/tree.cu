// tree.cu -- a2 best-first prefix selection and a3 ancestor masks.
//
// a2 follows "DDTree Explained ...", section 4 (Algorithm 1: index prefixes
// by rank tuples, pop the most probable, push its sibling (.., rho_d + 1)
// and child (.., rho_d, 0)) and "SparklingTree ...", Step 3 (the heap loop
// with its node numbering, parents and depths). One warp per request:
//  * The frontier (at most B + 1 entries) lives in registers, 4 slots per
//    lane. A pop is a warp-wide arg-best over (S, rank tuple): larger S
//    first, equal S to the lexicographically smaller tuple. S is compared as
//    an order-preserving 64-bit integer key, by two 32-bit warp max
//    reductions; the tuple's four words are reduced only when scores tie.
//  * S is fp64: parent's S plus the entry's own fp32 log-prob, the same
//    additions in the same order on every machine.
//  * A rank tuple packs (rank + 1) into 7-bit fields, most significant
//    first, in a 128-bit (hi, lo) pair; unsigned comparison of the pair is
//    the lexicographic order with a prefix before its extensions.
// a3 follows "SparklingTree ...", Step 4 (a node sees what its parent sees
// plus itself) and "DDTree Explained ...", section 5 (ancestor-only mask).
#include <stdint.h>

#include "ddt_device.cuh"
#include "ddt_internal.h"

namespace {

// Frontier slots per lane (a template parameter of the kernel): each pop
// frees its entry's slot or reuses it for the sibling and adds at most one
// child, so before the i-th pop at most i entries are live and B entries in
// total fit 32 * ceil(B / 32) slots.

DDT_DEVINL void field_or(uint64_t &hi, uint64_t &lo, int i, uint64_t val)
{
    const int sh = 121 - 7 * i;  // bit offset of field i's least significant bit
    if (sh >= 64) {
        hi |= val << (sh - 64);
    } else if (sh + 7 <= 64) {
        lo |= val << sh;
    } else {
        hi |= val >> (64 - sh);
        lo |= val << sh;
    }
}

DDT_DEVINL void field_clear(uint64_t &hi, uint64_t &lo, int i)
{
    uint64_t mh = 0, ml = 0;
    field_or(mh, ml, i, 0x7Full);
    hi &= ~mh;
    lo &= ~ml;
}

// order-preserving map of a (non-NaN) double to uint64; never 0 for a real value
DDT_DEVINL uint64_t skey(double x)
{
    const uint64_t b = (uint64_t)__double_as_longlong(x + 0.0);
    return (b >> 63) ? ~b : (b | 0x8000000000000000ull);
}
DDT_DEVINL double skey_inv(uint64_t k)
{
    return __longlong_as_double((long long)((k >> 63) ? (k & 0x7FFFFFFFFFFFFFFFull) : ~k));
}

// does (ka, ha, la) pop before (kb, hb, lb)? larger score key, then smaller tuple
DDT_DEVINL bool pops_before(uint64_t ka, uint64_t ha, uint64_t la, uint64_t kb, uint64_t hb,
                            uint64_t lb)
{
    return ka > kb || (ka == kb && (ha < hb || (ha == hb && la < lb)));
}

// the lanes whose value v is the warp maximum, among the lanes in cand
DDT_DEVINL unsigned keep_max(unsigned cand, uint32_t v, int lane)
{
    const uint32_t m = __reduce_max_sync(0xFFFFFFFFu, ((cand >> lane) & 1u) ? v : 0u);
    return cand & __ballot_sync(0xFFFFFFFFu, v == m);
}

template <int SLOTS>
__global__ void __launch_bounds__(32)
build_tree_kernel(const float *__restrict__ top_lp, const int32_t *__restrict__ top_ids, int L,
                  int K, int B, int32_t *__restrict__ tree_tokens, int32_t *__restrict__ parents,
                  int32_t *__restrict__ depths, int32_t *__restrict__ n_nodes,
                  uint32_t *__restrict__ mask)
{
    const int r = blockIdx.x, lane = threadIdx.x;
    const int P = B + 1, W = (P + 31) >> 5;
    __shared__ float s_lp[DDT_MAX_L * DDT_MAX_K];
    __shared__ int s_ids[DDT_MAX_L * DDT_MAX_K];
    __shared__ int s_tok[DDT_MAX_B];
    __shared__ int s_par[DDT_MAX_P];
    __shared__ int s_dep[DDT_MAX_P];

    for (int i = lane; i < L * K; i += 32) {
        s_lp[i] = top_lp[(int64_t)r * L * K + i];
        s_ids[i] = top_ids[(int64_t)r * L * K + i];
    }
    for (int i = lane; i < P; i += 32) {
        s_par[i] = -1;
        s_dep[i] = (i == 0) ? 0 : -1;
        if (i < B)
            s_tok[i] = -1;
    }
    __syncwarp();

    // frontier slots (registers): score key (S = skey_inv(sk)), the parent's score
    // key, rank tuple, parent node, depth and rank of the entry's last field; an
    // empty slot has key 0
    uint64_t sk[SLOTS], pk[SLOTS], kh[SLOTS], kl[SLOTS];
    int par[SLOTS], dep[SLOTS], rnk[SLOTS];
#pragma unroll
    for (int f = 0; f < SLOTS; ++f) {
        sk[f] = pk[f] = kh[f] = kl[f] = 0;
        par[f] = dep[f] = rnk[f] = 0;
    }
    if (lane == 0) {  // the single first entry: rank tuple (0,)
        pk[0] = skey(0.0);
        sk[0] = skey(0.0 + (double)s_lp[0]);
        field_or(kh[0], kl[0], 0, 1);
        dep[0] = 1;
    }

    int count = 0;
    while (count < B) {
        // lane-local best slot
        int bf = 0;
        uint64_t bk = sk[0], bh = kh[0], bl = kl[0];
        int bpar = par[0], bdep = dep[0], brnk = rnk[0];
#pragma unroll
        for (int f = 1; f < SLOTS; ++f)
            if (pops_before(sk[f], kh[f], kl[f], bk, bh, bl)) {
                bf = f;
                bk = sk[f];
                bh = kh[f];
                bl = kl[f];
                bpar = par[f];
                bdep = dep[f];
                brnk = rnk[f];
            }
        // warp arg-best: score key high then low word; the rank tuple only on a tie
        unsigned cand = __ballot_sync(0xFFFFFFFFu, bk != 0);
        if (cand == 0u)
            break;  // the whole prefix space is smaller than B
        cand = keep_max(cand, (uint32_t)(bk >> 32), lane);
        cand = keep_max(cand, (uint32_t)bk, lane);
        if (__popc(cand) > 1) {
            cand = keep_max(cand, ~(uint32_t)(bh >> 32), lane);
            cand = keep_max(cand, ~(uint32_t)bh, lane);
            cand = keep_max(cand, ~(uint32_t)(bl >> 32), lane);
            cand = keep_max(cand, ~(uint32_t)bl, lane);
        }
        const int wl = __ffs(cand) - 1;
        // the winner's fields, to every lane
        const uint64_t wk = __shfl_sync(0xFFFFFFFFu, bk, wl);
        const uint64_t wh = __shfl_sync(0xFFFFFFFFu, bh, wl);
        const uint64_t wlo = __shfl_sync(0xFFFFFFFFu, bl, wl);
        const int wpar = __shfl_sync(0xFFFFFFFFu, bpar, wl);
        const int wdep = __shfl_sync(0xFFFFFFFFu, bdep, wl);
        const int wrnk = __shfl_sync(0xFFFFFFFFu, brnk, wl);
        const double wS = skey_inv(wk);

        const int node = count + 1;
        if (lane == 0) {
            s_tok[count] = s_ids[(wdep - 1) * K + wrnk];
            s_par[node] = wpar;
            s_dep[node] = wdep;
        }
        ++count;
        if (count == B)
            break;
        // the popped entry's slot: freed, or reused by its sibling (.., rho_d + 1),
        // whose score is its parent's score plus the next rank's log-prob
        if (lane == wl) {
#pragma unroll
            for (int f = 0; f < SLOTS; ++f)
                if (f == bf) {
                    if (wrnk + 1 < K) {
                        sk[f] = skey(skey_inv(pk[f]) + (double)s_lp[(wdep - 1) * K + wrnk + 1]);
                        field_clear(kh[f], kl[f], wdep - 1);
                        field_or(kh[f], kl[f], wdep - 1, (uint64_t)(wrnk + 2));
                        rnk[f] = wrnk + 1;
                    } else {
                        sk[f] = 0;
                    }
                }
        }
        // child (.., rho_d, 0) goes to the lowest lane with a free slot
        if (wdep < L) {
            unsigned freeslots = 0;
#pragma unroll
            for (int f = 0; f < SLOTS; ++f)
                freeslots |= (sk[f] == 0) ? (1u << f) : 0u;
            const unsigned lanes = __ballot_sync(0xFFFFFFFFu, freeslots != 0u);
            const int tl = __ffs(lanes) - 1;
            if (lane == tl) {
                const int f0 = __ffs(freeslots) - 1;
#pragma unroll
                for (int f = 0; f < SLOTS; ++f)
                    if (f == f0) {
                        sk[f] = skey(wS + (double)s_lp[wdep * K + 0]);
                        pk[f] = wk;
                        kh[f] = wh;
                        kl[f] = wlo;
                        field_or(kh[f], kl[f], wdep, 1ull);
                        par[f] = node;
                        dep[f] = wdep + 1;
                        rnk[f] = 0;
                    }
            }
        }
    }
    __syncwarp();

    for (int i = lane; i < B; i += 32)
        tree_tokens[(int64_t)r * B + i] = s_tok[i];
    for (int i = lane; i < P; i += 32) {
        parents[(int64_t)r * P + i] = s_par[i];
        depths[(int64_t)r * P + i] = s_dep[i];
    }
    if (lane == 0)
        n_nodes[r] = count;
    if (mask != nullptr) {
        for (int i = lane; i < P; i += 32) {
            uint32_t words[4] = {0u, 0u, 0u, 0u};
            if (i <= count) {
                int cur = i;
                for (int step = 0; step <= DDT_MAX_L + 1 && cur >= 0; ++step) {
                    words[cur >> 5] |= 1u << (cur & 31);
                    cur = s_par[cur];
                }
            }
            for (int w = 0; w < W; ++w)
                mask[((int64_t)r * P + i) * W + w] = words[w];
        }
    }
}

// a3 on its own: validates the parent array while it walks it
__global__ void __launch_bounds__(128)
build_mask_kernel(const int32_t *__restrict__ parents, const int32_t *__restrict__ n_nodes, int P,
                  uint32_t *__restrict__ mask, int32_t *__restrict__ status)
{
    const int r = blockIdx.x;
    const int W = (P + 31) >> 5;
    __shared__ int s_par[DDT_MAX_P];
    __shared__ int s_bad;
    if (threadIdx.x == 0)
        s_bad = 0;
    int n = n_nodes[r];
    const bool bad_n = (n < 0 || n > P - 1);
    if (bad_n)
        n = (n < 0) ? 0 : P - 1;
    __syncthreads();
    for (int i = threadIdx.x; i < P; i += blockDim.x) {
        const int p = parents[(int64_t)r * P + i];
        s_par[i] = p;
        if (i >= 1 && i <= n && (p < 0 || p >= i))
            s_bad = 1;
    }
    __syncthreads();
    if (threadIdx.x == 0 && (s_bad || bad_n))
        set_status(status, DDT_DEV_BAD_TREE);
    const bool ok = !s_bad;
    for (int i = threadIdx.x; i < P; i += blockDim.x) {
        uint32_t words[4] = {0u, 0u, 0u, 0u};
        if (ok && i <= n) {
            int cur = i;
            for (int step = 0; step < P && cur >= 0; ++step) {
                words[cur >> 5] |= 1u << (cur & 31);
                cur = (cur == 0) ? -1 : s_par[cur];
            }
        }
        for (int w = 0; w < W; ++w)
            mask[((int64_t)r * P + i) * W + w] = words[w];
    }
}

}  // namespace

cudaError_t launch_build_tree(const ddt_ctx *c, const float *top_lp, const int32_t *top_ids, int R,
                              int32_t *tree_tokens, int32_t *parents, int32_t *depths,
                              int32_t *n_nodes, uint32_t *mask, cudaStream_t s)
{
    const ddt_config &cfg = c->cfg;
    const int slots = (cfg.B + 31) / 32;  // 1..4 (B <= 127)
    if (slots <= 1)
        build_tree_kernel<1><<<R, 32, 0, s>>>(top_lp, top_ids, cfg.L, cfg.K, cfg.B, tree_tokens, parents,
                                              depths, n_nodes, mask);
    else if (slots == 2)
        build_tree_kernel<2><<<R, 32, 0, s>>>(top_lp, top_ids, cfg.L, cfg.K, cfg.B, tree_tokens, parents,
                                              depths, n_nodes, mask);
    else if (slots == 3)
        build_tree_kernel<3><<<R, 32, 0, s>>>(top_lp, top_ids, cfg.L, cfg.K, cfg.B, tree_tokens, parents,
                                              depths, n_nodes, mask);
    else
        build_tree_kernel<4><<<R, 32, 0, s>>>(top_lp, top_ids, cfg.L, cfg.K, cfg.B, tree_tokens, parents,
                                              depths, n_nodes, mask);
    return cudaGetLastError();
}

cudaError_t launch_build_mask(const ddt_ctx *c, const int32_t *parents, const int32_t *n_nodes,
                              int R, uint32_t *mask, cudaStream_t s)
{
    build_mask_kernel<<<R, 128, 0, s>>>(parents, n_nodes, c->cfg.B + 1, mask, c->status);
    return cudaGetLastError();
}
