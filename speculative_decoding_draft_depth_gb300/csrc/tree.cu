// tree.cu -- a2 best-first prefix selection and a3 ancestor masks.
//
// a2 follows "DDTree Explained ...", section 4 (Algorithm 1: index prefixes
// by rank tuples, pop the most probable, push its sibling (.., rho_d + 1)
// and child (.., rho_d, 0)) and "SparklingTree ...", Step 3 (the heap loop
// with its node numbering, parents and depths). One warp per request:
//  * The frontier (at most B entries) lives in registers, 4 slots per lane.
//    A pop is a warp-wide arg-best by xor-shuffles over (S, rank tuple):
//    larger S first, equal S to the lexicographically smaller tuple.
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

constexpr int SLOTS = 4;  // frontier slots per lane: 128 >= B entries

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

// does (Sa, ha, la) pop before (Sb, hb, lb)?
DDT_DEVINL bool pops_before(double Sa, uint64_t ha, uint64_t la, double Sb, uint64_t hb,
                            uint64_t lb)
{
    if (Sa != Sb)
        return Sa > Sb;
    if (ha != hb)
        return ha < hb;
    return la < lb;
}

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

    // frontier slots (registers)
    double S[SLOTS], pS[SLOTS];
    uint64_t kh[SLOTS], kl[SLOTS];
    int par[SLOTS], dep[SLOTS], rnk[SLOTS];
    unsigned valid = 0;
#pragma unroll
    for (int f = 0; f < SLOTS; ++f) {
        S[f] = pS[f] = 0.0;
        kh[f] = kl[f] = 0;
        par[f] = dep[f] = rnk[f] = 0;
    }
    if (lane == 0) {  // the single first entry: rank tuple (0,)
        valid = 1u;
        pS[0] = 0.0;
        S[0] = 0.0 + (double)s_lp[0];
        field_or(kh[0], kl[0], 0, 1);
        par[0] = 0;
        dep[0] = 1;
        rnk[0] = 0;
    }

    int count = 0;
    while (count < B) {
        // lane-local best slot
        int bf = -1;
        double bS = -__builtin_huge_val();
        uint64_t bh = ~0ull, bl = ~0ull;
#pragma unroll
        for (int f = 0; f < SLOTS; ++f)
            if (((valid >> f) & 1u) && (bf < 0 || pops_before(S[f], kh[f], kl[f], bS, bh, bl))) {
                bf = f;
                bS = S[f];
                bh = kh[f];
                bl = kl[f];
            }
        int who = (bf < 0) ? -1 : (lane * SLOTS + bf);
        // warp arg-best
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const double oS = __shfl_xor_sync(0xFFFFFFFFu, bS, off);
            const uint64_t oh = __shfl_xor_sync(0xFFFFFFFFu, bh, off);
            const uint64_t ol = __shfl_xor_sync(0xFFFFFFFFu, bl, off);
            const int ow = __shfl_xor_sync(0xFFFFFFFFu, who, off);
            const bool take = (ow >= 0) && (who < 0 || pops_before(oS, oh, ol, bS, bh, bl));
            if (take) {
                bS = oS;
                bh = oh;
                bl = ol;
                who = ow;
            }
        }
        if (who < 0)
            break;  // the whole prefix space is smaller than B
        const int wl = who / SLOTS, wf = who % SLOTS;
        // broadcast the winner's remaining fields
        double mypS = pS[0];
        int mypar = par[0], mydep = dep[0], myrnk = rnk[0];
#pragma unroll
        for (int f = 1; f < SLOTS; ++f)
            if (wf == f) {
                mypS = pS[f];
                mypar = par[f];
                mydep = dep[f];
                myrnk = rnk[f];
            }
        const double wpS = __shfl_sync(0xFFFFFFFFu, mypS, wl);
        const int wpar = __shfl_sync(0xFFFFFFFFu, mypar, wl);
        const int wdep = __shfl_sync(0xFFFFFFFFu, mydep, wl);
        const int wrnk = __shfl_sync(0xFFFFFFFFu, myrnk, wl);

        const int node = count + 1;
        if (lane == 0) {
            s_tok[count] = s_ids[(wdep - 1) * K + wrnk];
            s_par[node] = wpar;
            s_dep[node] = wdep;
        }
        ++count;
        if (lane == wl)
            valid &= ~(1u << wf);
        if (count == B)
            break;

        // sibling (.., rho_d + 1) takes the freed slot
        if (wrnk + 1 < K && lane == wl) {
#pragma unroll
            for (int f = 0; f < SLOTS; ++f)
                if (f == wf) {
                    S[f] = wpS + (double)s_lp[(wdep - 1) * K + wrnk + 1];
                    pS[f] = wpS;
                    kh[f] = bh;
                    kl[f] = bl;
                    field_clear(kh[f], kl[f], wdep - 1);
                    field_or(kh[f], kl[f], wdep - 1, (uint64_t)(wrnk + 2));
                    par[f] = wpar;
                    dep[f] = wdep;
                    rnk[f] = wrnk + 1;
                    valid |= 1u << f;
                }
        }
        // child (.., rho_d, 0) goes to the lowest lane with a free slot
        if (wdep < L) {
            const unsigned freeslots = (~valid) & ((1u << SLOTS) - 1u);
            const unsigned lanes = __ballot_sync(0xFFFFFFFFu, freeslots != 0u);
            const int tl = __ffs(lanes) - 1;
            if (lane == tl) {
                const int f0 = __ffs(freeslots) - 1;
#pragma unroll
                for (int f = 0; f < SLOTS; ++f)
                    if (f == f0) {
                        S[f] = bS + (double)s_lp[wdep * K + 0];
                        pS[f] = bS;
                        kh[f] = bh;
                        kl[f] = bl;
                        field_or(kh[f], kl[f], wdep, 1ull);
                        par[f] = node;
                        dep[f] = wdep + 1;
                        rnk[f] = 0;
                        valid |= 1u << f;
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
    build_tree_kernel<<<R, 32, 0, s>>>(top_lp, top_ids, cfg.L, cfg.K, cfg.B, tree_tokens, parents,
                                       depths, n_nodes, mask);
    return cudaGetLastError();
}

cudaError_t launch_build_mask(const ddt_ctx *c, const int32_t *parents, const int32_t *n_nodes,
                              int R, uint32_t *mask, cudaStream_t s)
{
    build_mask_kernel<<<R, 128, 0, s>>>(parents, n_nodes, c->cfg.B + 1, mask, c->status);
    return cudaGetLastError();
}
