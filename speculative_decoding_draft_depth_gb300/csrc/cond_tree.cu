// cond_tree.cu -- the parent-conditioned draft tree ("Robot2050/TreeSpark",
// items 1 and 2): one backbone pass gives per-depth logits l_d [R, L, V]; a
// first-order Markov head specialises depth d to a parent token,
//   z_d(u) = l_d + W e(t_u),          W, E: [V, H] bf16,
// each parent keeps its k best children (log-softmax of z_d(u)), the F best
// children of a depth by joint path score become the next depth's parents,
// and the N best candidates of all depths are packed into the tree (prefix-
// closed: lp <= 0, and a parent sorts before its children).
//
// Per depth, two kernels:
//  * cg_gemm_kernel: the Markov bias of every frontier parent of every
//    request at once, as a tcgen05 GEMM: M = 128 vocabulary rows of W per
//    tile (TMA, 128-byte swizzle, two stages), N = the parents' gathered
//    embedding rows (up to 128, K-major in shared memory), K = H; fp32
//    accumulators in TMEM. The epilogue adds l_d and keeps, per parent, a
//    running (max, sum of exp) and top-k over the CTA's tiles; persistent
//    CTAs stride over the vocabulary and write one partial per parent.
//  * cg_merge_kernel: one CTA per request merges the partials of its
//    parents (log-partition in fp64, top-k by 64-bit keys), writes the
//    per-parent lists, scores the children (S = S_parent + lp in fp64),
//    records them as candidates and keeps the F best as the next frontier.
// Then cg_pack_kernel ranks all candidates of a request and writes the tree
// and its ancestor mask.
#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "ddt_device.cuh"
#include "ddt_internal.h"
#include "tc_ptx.cuh"

namespace {

constexpr int CG_THREADS = 128;  // four warps: TMEM lane quarters = vocabulary rows
constexpr int CG_TILE = 128;     // vocabulary rows per tile (M)
constexpr int CG_MAXK = 8;       // children per parent
constexpr int CG_MAXNP = 128;    // parents per depth (N of the MMA)
constexpr int CG_MAXF = 8;       // frontier width
constexpr int CG_MAXG = CG_MAXNP / 32;
constexpr long long CG_WAIT = 4000000000LL;

// ---------------------------------------------------------------- keys
// order-preserving map of a (non-NaN) float to uint32
DDT_DEVINL uint32_t fkey(float x)
{
    const uint32_t b = __float_as_uint(x + 0.0f);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
DDT_DEVINL float fkey_inv(uint32_t k)
{
    return (k & 0x80000000u) ? __uint_as_float(k & 0x7FFFFFFFu) : __uint_as_float(~k);
}
// candidate key: value order high, complemented id low (lower id wins a tie)
DDT_DEVINL uint64_t vkey(float v, int id) { return ((uint64_t)fkey(v) << 32) | (uint32_t)~(uint32_t)id; }

struct GemmArgs {
    const uint16_t *E;       // [V, H] bf16
    const uint16_t *ell;     // [R, L, V] bf16
    const int32_t *fr_tok;   // [R, F] frontier tokens (-1: none)
    float2 *part_ms;         // [NPmax, grid] (max, sum of exp)
    uint64_t *part_top;      // [NPmax, grid, CG_MAXK] (value key, id) packed as vkey
    int R, L, V, H, d, Fd, F, NP, NPpad, k;
    int32_t *status;
};

// per-thread running state of one parent column over the rows it scans
struct ColState {
    float m, s;
    float tv[CG_MAXK];
    int ti[CG_MAXK];
};

DDT_DEVINL void col_reset(ColState &c)
{
    c.m = DDT_NEG_INF;
    c.s = 0.f;
#pragma unroll
    for (int j = 0; j < CG_MAXK; ++j) {
        c.tv[j] = DDT_NEG_INF;
        c.ti[j] = -1;
    }
}

DDT_DEVINL void col_add(ColState &c, int k, float x, int id)
{
    if (x == DDT_NEG_INF)
        return;
    if (x > c.m) {
        c.s = c.s * ex2((c.m - x) * DDT_LOG2E) + 1.f;  // 0 * ex2(-inf) = 0 on the first value
        c.m = x;
    } else {
        c.s += ex2((x - c.m) * DDT_LOG2E);
    }
    // descending top-k, equal values keep the earlier (lower) id
    if (c.ti[k - 1] >= 0 && !(x > c.tv[k - 1]))
        return;
    float v = x;
    int id2 = id;
#pragma unroll
    for (int j = 0; j < CG_MAXK; ++j) {
        if (j < k) {
            const bool take = (c.ti[j] < 0) || (v > c.tv[j]);
            if (take) {
                const float tv = c.tv[j];
                const int ti = c.ti[j];
                c.tv[j] = v;
                c.ti[j] = id2;
                v = tv;
                id2 = ti;
            }
        }
    }
}

// wind-down wait for this CTA's own copies and MMAs (bounded, no status)
DDT_DEVINL void cg_drain(uint32_t bar, uint32_t parity)
{
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity))
        if (clock64() - t0 > 200000000LL)
            return;
}

DDT_DEVINL bool cg_wait(uint32_t bar, uint32_t parity, int32_t *status)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity))
        if (clock64() - t0 > CG_WAIT) {
            atomicOr(status, DDT_DEV_TIMEOUT);
            return false;
        }
    return true;
}

__global__ void __launch_bounds__(CG_THREADS, 1)
cg_gemm_kernel(const __grid_constant__ CUtensorMap tm_w, const GemmArgs a)
{
    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw = (uint32_t)__cvta_generic_to_shared(smem_raw);
    const uint32_t sb = (raw + 1023u) & ~1023u;
    unsigned char *sgen = smem_raw + (sb - raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nblk = a.H / 64;                     // 64-column K blocks
    const uint32_t WST = (uint32_t)nblk * 16384u;  // one W tile
    const uint32_t SM_W = 0, SM_E = 2 * WST;
    const uint32_t EBLK = (uint32_t)a.NPpad * 128u;
    const uint32_t SM_Z = SM_E + (uint32_t)nblk * EBLK;  // [32 columns][CG_TILE + 1] floats
    const uint32_t SM_BAR = SM_Z + 32 * (CG_TILE + 1) * 4;
    const uint32_t bar = sb + SM_BAR;  // [0, 8]: W stages full, [16]: MMA done, [24]: TMEM address
    float *zt = reinterpret_cast<float *>(sgen + SM_Z);
    const int ntiles = (a.V + CG_TILE - 1) / CG_TILE;
    const int ng = a.NPpad / 32;
    uint32_t tcols = 32;
    while ((int)tcols < a.NPpad)
        tcols <<= 1;

    if (tid == 0) {
        mbar_init(bar + 0, 1);
        mbar_init(bar + 8, 1);
        mbar_init(bar + 16, 1);
        mbar_init(bar + 32, 1);
        fence_mbar_init();
        prefetch_tmap(&tm_w);
    }
    if (warp == 0) {
        tmem_alloc(bar + 24, tcols);
        tmem_relinquish();
    }
    // the parents' embedding rows, K-major with the 128-byte swizzle (zero rows pad to NPpad)
    for (int i = tid; i < a.NPpad * (a.H / 8); i += CG_THREADS) {
        const int p = i / (a.H / 8), c = i % (a.H / 8);
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (p < a.NP) {
            const int r = p / a.Fd, f = p % a.Fd;
            const int tok = a.fr_tok[r * a.F + f];
            if (tok >= 0 && tok < a.V)
                v = __ldg(reinterpret_cast<const uint4 *>(a.E + (int64_t)tok * a.H) + c);
        }
        const int blk = c >> 3, ch = c & 7;
        *reinterpret_cast<uint4 *>(sgen + SM_E + blk * EBLK + p * 128 + ((ch ^ (p & 7)) << 4)) = v;
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(sgen + SM_BAR + 24);
    const uint32_t idesc = idesc_bf16(128, a.NPpad, false, false);

    int loads[2] = {0, 0};  // TMA loads issued per stage (thread 0)
    auto load_tile = [&](int tile, int s) {
        ++loads[s];
        mbar_arrive_expect_tx(bar + 8 * s, WST);
        for (int b = 0; b < nblk; ++b)
            tma_load_2d(sb + SM_W + s * WST + b * 16384u, &tm_w, b * 64, tile * CG_TILE, bar + 8 * s);
    };

    ColState st[CG_MAXG];
#pragma unroll
    for (int g = 0; g < CG_MAXG; ++g)
        col_reset(st[g]);
    // the scan after each tile: lane = column (within a group of 32), warp = row quarter

    int i = 0;
    if (tid == 0) {
        if ((int)blockIdx.x < ntiles)
            load_tile(blockIdx.x, 0);
        if ((int)blockIdx.x + (int)gridDim.x < ntiles)
            load_tile(blockIdx.x + gridDim.x, 1);
    }
    bool ok = true;
    for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++i) {
        const int s = i & 1;
        if (tid == 0) {
            ok = cg_wait(bar + 8 * s, (i >> 1) & 1, a.status);
            if (ok) {
                tc_fence_after();
                const uint64_t dA0 = sdesc_sw128(sb + SM_W + s * WST, 16, 1024);
                const uint64_t dB0 = sdesc_sw128(sb + SM_E, 16, 1024);
                for (int kk = 0; kk < a.H / 16; ++kk) {
                    const int b = kk >> 2, w = kk & 3;
                    mma_bf16(tmem, dA0 + ((b * 16384u + w * 32u) >> 4), dB0 + ((b * EBLK + w * 32u) >> 4),
                             idesc, kk > 0 ? 1u : 0u);
                }
                mma_commit(bar + 16);
            }
        }
        ok = __syncthreads_and(ok ? 1 : 0) != 0;
        if (!ok)
            break;
        if (!cg_wait(bar + 16, i & 1, a.status)) {
            ok = false;
        }
        ok = __syncthreads_and(ok ? 1 : 0) != 0;
        if (!ok)
            break;
        tc_fence_after();
        // the stage is consumed: refill it with the tile after next
        if (tid == 0 && tile + 2 * (int)gridDim.x < ntiles)
            load_tile(tile + 2 * gridDim.x, s);
        const int v = tile * CG_TILE + tid;  // this thread's TMEM lane = vocabulary row
#pragma unroll
        for (int g = 0; g < CG_MAXG; ++g) {
            if (g < ng) {
                uint32_t acc[32];
                tmem_ld16(tmem + ((uint32_t)(warp * 32) << 16) + 32u * g, acc);
                tmem_ld16(tmem + ((uint32_t)(warp * 32) << 16) + 32u * g + 16u, acc + 16);
                tmem_wait_ld();
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    const int p = 32 * g + c;
                    float z = DDT_NEG_INF;
                    if (p < a.NP && v < a.V) {
                        const int r = p / a.Fd;
                        z = __uint_as_float(acc[c]) +
                            bf16_to_f32(__ldg(a.ell + ((int64_t)r * a.L + a.d) * a.V + v));
                    }
                    zt[c * (CG_TILE + 1) + tid] = z;
                }
                __syncthreads();
                if (32 * g + lane < a.NP)
                    for (int j = 0; j < 32; ++j) {
                        const int row = warp * 32 + j;
                        col_add(st[g], a.k, zt[lane * (CG_TILE + 1) + row], tile * CG_TILE + row);
                    }
                __syncthreads();
            }
        }
        tc_fence_before();
    }
    // the CTA's partial per parent: warp 0 combines the four row quarters
    // (warps) of each column, passed through shared memory
    float *xm = zt;                                        // [4 warps][32] max
    float *xs = zt + 128;                                  // [4 warps][32] sum
    uint64_t *xt = reinterpret_cast<uint64_t *>(zt + 256); // [4 warps][32][CG_MAXK] keys
    for (int g = 0; g < CG_MAXG; ++g) {
        if (g >= ng)
            break;
        __syncthreads();
        {
#pragma unroll
            for (int gg = 0; gg < CG_MAXG; ++gg)
                if (gg == g) {
                    xm[warp * 32 + lane] = st[gg].m;
                    xs[warp * 32 + lane] = st[gg].s;
#pragma unroll
                    for (int j = 0; j < CG_MAXK; ++j)
                        xt[(warp * 32 + lane) * CG_MAXK + j] =
                            (j < a.k && st[gg].ti[j] >= 0) ? vkey(st[gg].tv[j], st[gg].ti[j]) : 0ull;
                }
        }
        __syncthreads();
        const int p = 32 * g + lane;
        if (warp == 0 && p < a.NP) {
            float M = DDT_NEG_INF;
#pragma unroll
            for (int w = 0; w < 4; ++w)
                M = fmaxf(M, xm[w * 32 + lane]);
            float S = 0.f;
#pragma unroll
            for (int w = 0; w < 4; ++w) {
                const float mw = xm[w * 32 + lane];
                if (mw != DDT_NEG_INF)
                    S += xs[w * 32 + lane] * ex2((mw - M) * DDT_LOG2E);
            }
            // top-k of the four descending lists
            uint64_t best[CG_MAXK];
#pragma unroll
            for (int j = 0; j < CG_MAXK; ++j)
                best[j] = 0ull;
            for (int w = 0; w < 4; ++w)
                for (int j = 0; j < a.k; ++j) {
                    uint64_t x = xt[(w * 32 + lane) * CG_MAXK + j];
#pragma unroll
                    for (int t = 0; t < CG_MAXK; ++t)
                        if (t < a.k && x > best[t]) {
                            const uint64_t y = best[t];
                            best[t] = x;
                            x = y;
                        }
                }
            const int64_t slot = (int64_t)p * gridDim.x + blockIdx.x;
            a.part_ms[slot] = make_float2(M, S);
#pragma unroll
            for (int j = 0; j < CG_MAXK; ++j)
                if (j < a.k)
                    a.part_top[slot * CG_MAXK + j] = best[j];
        }
    }
    // wind down: every copy and MMA this CTA started has finished (bounded)
    if (tid == 0) {
        mma_commit(bar + 32);
        cg_drain(bar + 32, 0);
        for (int s2 = 0; s2 < 2; ++s2)
            if (loads[s2] > 0)
                cg_drain(bar + 8 * s2, (loads[s2] - 1) & 1);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, tcols);
    }
}

struct MergeArgs {
    const float2 *part_ms;
    const uint64_t *part_top;
    int32_t *fr_tok;          // [R, F] in: this depth's parents; out: the next depth's
    int32_t *fr_cand;         // [R, F] candidate index of each frontier parent (-1: root)
    double *fr_S;             // [R, F]
    int32_t *fr_n;            // [R]
    double *c_S;              // [R, Cmax] candidate score
    int32_t *c_meta;          // [R, Cmax, 3]: depth, parent candidate, token
    float *cand_lp;           // [R, L, F, k] (optional)
    int32_t *cand_ids;        // [R, L, F, k] (optional)
    int32_t *frontier_tok;    // [R, L, F] (optional): parents of every depth
    int R, L, d, Fd, F, k, grid, Cmax, base;
};

// one CTA per request; warp f merges frontier parent f
__global__ void __launch_bounds__(32 * CG_MAXF)
cg_merge_kernel(const MergeArgs a)
{
    const int r = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    __shared__ float s_lp[CG_MAXF][CG_MAXK];
    __shared__ int s_id[CG_MAXF][CG_MAXK];
    const int nfr = a.fr_n[r];
    if (warp < a.Fd) {
        const int f = warp;
        const bool live = f < nfr;
        const int p = r * a.Fd + f;
        double logz = 0.0;
        uint64_t mine[CG_MAXK];
#pragma unroll
        for (int j = 0; j < CG_MAXK; ++j)
            mine[j] = 0ull;
        if (live) {
            // log-partition over the CTAs' (max, sum) pairs
            float M = DDT_NEG_INF;
            for (int c = lane; c < a.grid; c += 32)
                M = fmaxf(M, a.part_ms[(int64_t)p * a.grid + c].x);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1)
                M = fmaxf(M, __shfl_xor_sync(0xFFFFFFFFu, M, o));
            float S = 0.f;
            for (int c = lane; c < a.grid; c += 32) {
                const float2 ms = a.part_ms[(int64_t)p * a.grid + c];
                if (ms.x != DDT_NEG_INF)
                    S += ms.y * ex2((ms.x - M) * DDT_LOG2E);
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1)
                S += __shfl_xor_sync(0xFFFFFFFFu, S, o);
            logz = (double)M + log((double)S);
            // this lane's best k of its CTAs' lists, then k warp-wide extractions
            for (int c = lane; c < a.grid; c += 32)
                for (int j = 0; j < a.k; ++j) {
                    uint64_t x = a.part_top[((int64_t)p * a.grid + c) * CG_MAXK + j];
                    if (x == 0ull)
                        break;
#pragma unroll
                    for (int t = 0; t < CG_MAXK; ++t)
                        if (t < a.k && x > mine[t]) {
                            const uint64_t y = mine[t];
                            mine[t] = x;
                            x = y;
                        }
                }
        }
        int head = 0;
        for (int j = 0; j < a.k; ++j) {
            uint64_t cur = 0ull;
#pragma unroll
            for (int t = 0; t < CG_MAXK; ++t)
                if (t == head)
                    cur = mine[t];
            const uint32_t hi = (uint32_t)(cur >> 32), lo = (uint32_t)cur;
            const uint32_t mhi = __reduce_max_sync(0xFFFFFFFFu, hi);
            const uint32_t mlo = __reduce_max_sync(0xFFFFFFFFu, hi == mhi ? lo : 0u);
            const unsigned who = __ballot_sync(0xFFFFFFFFu, hi == mhi && lo == mlo && cur != 0ull);
            if (lane == 0) {
                if (who != 0u && live) {
                    const uint64_t w = ((uint64_t)mhi << 32) | mlo;
                    s_lp[f][j] = (float)((double)fkey_inv((uint32_t)(w >> 32)) - logz);
                    s_id[f][j] = (int)~(uint32_t)w;
                } else {
                    s_lp[f][j] = DDT_NEG_INF;
                    s_id[f][j] = -1;
                }
            }
            if (who != 0u && lane == __ffs(who) - 1)
                ++head;
        }
    }
    __syncthreads();
    if (warp == 0) {
        // this depth's candidates in creation order (frontier slot, child rank)
        // (every slot of the depth is written; a missing parent's slots get token -1)
        const int nd = nfr * a.k;
        double Sc = -INFINITY;
        int tok = -1, par = -1, ord = a.base + lane;
        const bool have = lane < nd;
        if (have) {
            const int f = lane / a.k, j = lane % a.k;
            tok = s_id[f][j];
            Sc = a.fr_S[r * a.F + f] + (double)s_lp[f][j];
            par = a.fr_cand[r * a.F + f];
            if (tok < 0)
                Sc = -INFINITY;
        }
        if (lane < a.Fd * a.k) {
            a.c_S[(int64_t)r * a.Cmax + ord] = Sc;
            int32_t *meta = a.c_meta + ((int64_t)r * a.Cmax + ord) * 3;
            meta[0] = a.d + 1;
            meta[1] = par;
            meta[2] = tok;
        }
        // the next frontier: the F best by (S desc, creation order asc)
        int rank = 0;
        for (int o = 0; o < nd; ++o) {
            const double So = __shfl_sync(0xFFFFFFFFu, Sc, o);
            if (have && (So > Sc || (So == Sc && o < lane)))
                ++rank;
        }
        const int nnext = nd < a.F ? nd : a.F;
        if (have && rank < nnext) {
            a.fr_tok[r * a.F + rank] = tok;
            a.fr_cand[r * a.F + rank] = ord;
            a.fr_S[r * a.F + rank] = Sc;
        }
        if (lane == 0)
            a.fr_n[r] = nnext;
        // outputs: this depth's lists; the next depth's parents
        if (a.cand_lp != nullptr)
            for (int i = lane; i < a.F * a.k; i += 32) {
                const int f = i / a.k, j = i % a.k;
                const int64_t o = (((int64_t)r * a.L + a.d) * a.F + f) * a.k + j;
                a.cand_lp[o] = (f < nfr) ? s_lp[f][j] : DDT_NEG_INF;
                a.cand_ids[o] = (f < nfr) ? s_id[f][j] : -1;
            }
        __syncwarp();
        if (a.frontier_tok != nullptr && a.d + 1 < a.L)
            for (int f = lane; f < a.F; f += 32)
                a.frontier_tok[((int64_t)r * a.L + a.d + 1) * a.F + f] =
                    (f < nnext) ? a.fr_tok[r * a.F + f] : -1;
    }
}

// the root of every request as the only parent of depth 1
__global__ void cg_init_kernel(const int32_t *anchors, int R, int L, int F, int32_t *fr_tok,
                               int32_t *fr_cand, double *fr_S, int32_t *fr_n, int32_t *frontier_tok)
{
    const int r = blockIdx.x * blockDim.x + threadIdx.x;
    if (r >= R)
        return;
    for (int f = 0; f < F; ++f) {
        fr_tok[r * F + f] = (f == 0) ? anchors[r] : -1;
        fr_cand[r * F + f] = -1;
        fr_S[r * F + f] = 0.0;
        if (frontier_tok != nullptr)
            frontier_tok[((int64_t)r * L) * F + f] = (f == 0) ? anchors[r] : -1;
    }
    fr_n[r] = 1;
}

struct PackArgs {
    const double *c_S;
    const int32_t *c_meta;
    int32_t *tree_tokens, *parents, *depths, *n_nodes;
    uint32_t *mask;
    int C, Cmax, N;
};

// one CTA per request: the N best candidates by (S desc, depth asc, order asc)
__global__ void __launch_bounds__(256)
cg_pack_kernel(const PackArgs a)
{
    const int r = blockIdx.x;
    const int P = a.N + 1, W = (P + 31) >> 5;
    __shared__ double s_S[1024];
    __shared__ int s_dep[1024], s_node[1024];
    __shared__ int s_par[DDT_MAX_P];
    const int C = a.C;
    for (int i = threadIdx.x; i < C; i += blockDim.x) {
        s_S[i] = a.c_S[(int64_t)r * a.Cmax + i];
        s_dep[i] = a.c_meta[((int64_t)r * a.Cmax + i) * 3];
        s_node[i] = -1;
    }
    for (int i = threadIdx.x; i < P; i += blockDim.x) {
        a.parents[(int64_t)r * P + i] = -1;
        a.depths[(int64_t)r * P + i] = (i == 0) ? 0 : -1;
        s_par[i] = -1;
        if (i < a.N)
            a.tree_tokens[(int64_t)r * a.N + i] = -1;
    }
    __shared__ int s_count;
    if (threadIdx.x == 0)
        s_count = 0;
    __syncthreads();
    // rank of every real candidate; the N best become nodes 1..N
    for (int i = threadIdx.x; i < C; i += blockDim.x) {
        if (a.c_meta[((int64_t)r * a.Cmax + i) * 3 + 2] < 0)
            continue;  // an empty slot
        const double Si = s_S[i];
        int rank = 0;
        for (int o = 0; o < C; ++o) {
            if (a.c_meta[((int64_t)r * a.Cmax + o) * 3 + 2] < 0)
                continue;
            const double So = s_S[o];
            if (So > Si || (So == Si && (s_dep[o] < s_dep[i] || (s_dep[o] == s_dep[i] && o < i))))
                ++rank;
        }
        if (rank < a.N) {
            s_node[i] = rank + 1;
            atomicAdd(&s_count, 1);
        }
    }
    __syncthreads();
    for (int i = threadIdx.x; i < C; i += blockDim.x) {
        const int node = s_node[i];
        if (node < 0)
            continue;
        const int32_t *meta = a.c_meta + ((int64_t)r * a.Cmax + i) * 3;
        const int pc = meta[1];
        const int pn = (pc < 0) ? 0 : s_node[pc];
        a.tree_tokens[(int64_t)r * a.N + node - 1] = meta[2];
        a.parents[(int64_t)r * P + node] = pn;
        a.depths[(int64_t)r * P + node] = meta[0];
        s_par[node] = pn;
    }
    __syncthreads();
    const int n = s_count;
    if (threadIdx.x == 0)
        a.n_nodes[r] = n;
    if (a.mask != nullptr)
        for (int i = threadIdx.x; i < P; i += blockDim.x) {
            uint32_t words[4] = {0u, 0u, 0u, 0u};
            if (i <= n) {
                int cur = i;
                for (int step = 0; step <= DDT_MAX_L + 1 && cur >= 0; ++step) {
                    words[cur >> 5] |= 1u << (cur & 31);
                    cur = (cur == 0) ? -1 : s_par[cur];
                }
            }
            for (int w = 0; w < W; ++w)
                a.mask[((int64_t)r * P + i) * W + w] = words[w];
        }
}

// ---------------------------------------------------------------- host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    if (fn == nullptr) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (EncodeTiledFn)p;
    }
    return fn;
}

size_t gemm_smem(int H, int NPpad)
{
    const size_t nblk = (size_t)H / 64;
    // W stages, the parents' rows, the transpose (32 x (CG_TILE + 1) floats), barriers,
    // and the slack for 1024-byte alignment
    return 2 * nblk * 16384 + nblk * (size_t)NPpad * 128 + 32 * (CG_TILE + 1) * 4 + 64 + 1024;
}

}  // namespace

int cond_tree_cmax(const ddt_config &cfg)
{
    return cfg.K + (cfg.L - 1) * cfg.frontier * cfg.K;
}

bool cond_tree_supported(const ddt_config &cfg)
{
    const int H = cfg.markov_dim, F = cfg.frontier;
    return H >= 64 && H <= 256 && H % 64 == 0 && F >= 1 && F <= CG_MAXF && cfg.K >= 1 &&
           cfg.K <= CG_MAXK && cfg.R_max * F <= CG_MAXNP && F * cfg.K <= 32 &&
           cond_tree_cmax(cfg) <= 1024 && cfg.B + 1 <= DDT_MAX_P && cfg.L <= DDT_MAX_L &&
           encode_fn() != nullptr;
}

cudaError_t launch_cond_tree(const ddt_ctx *c, const uint16_t *ell, const uint16_t *W,
                             const uint16_t *E, const int32_t *anchors, int R, float *cand_lp,
                             int32_t *cand_ids, int32_t *frontier_tok, int32_t *tree_tokens,
                             int32_t *parents, int32_t *depths, int32_t *n_nodes, uint32_t *mask,
                             cudaStream_t s)
{
    const ddt_config &cfg = c->cfg;
    const int H = cfg.markov_dim, F = cfg.frontier, K = cfg.K, L = cfg.L, V = cfg.V;
    CUtensorMap tm;
    {
        const cuuint64_t dims[2] = {(cuuint64_t)H, (cuuint64_t)V};
        const cuuint64_t strides[1] = {(cuuint64_t)H * 2};
        const cuuint32_t box[2] = {64, CG_TILE};
        const cuuint32_t es[2] = {1, 1};
        if (encode_fn()(&tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t *>(W), dims,
                        strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    const int grid = c->cg_grid;
    cg_init_kernel<<<(R + 127) / 128, 128, 0, s>>>(anchors, R, L, F, c->cg_fr_tok, c->cg_fr_cand,
                                                    c->cg_fr_S, c->cg_fr_n, frontier_tok);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return e;
    int base = 0;
    for (int d = 0; d < L; ++d) {
        const int Fd = (d == 0) ? 1 : F;
        GemmArgs g;
        g.E = E;
        g.ell = ell;
        g.fr_tok = c->cg_fr_tok;
        g.part_ms = c->cg_part_ms;
        g.part_top = c->cg_part_top;
        g.R = R;
        g.L = L;
        g.V = V;
        g.H = H;
        g.d = d;
        g.Fd = Fd;
        g.F = F;
        g.NP = R * Fd;
        g.NPpad = (g.NP + 31) / 32 * 32;
        g.k = K;
        g.status = c->status;
        const size_t smem = gemm_smem(H, g.NPpad);
        static size_t attr_set = 0;
        if (smem > attr_set) {
            e = cudaFuncSetAttribute(cg_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)gemm_smem(256, CG_MAXNP));
            if (e != cudaSuccess)
                return e;
            attr_set = gemm_smem(256, CG_MAXNP);
        }
        cg_gemm_kernel<<<grid, CG_THREADS, smem, s>>>(tm, g);
        if ((e = cudaGetLastError()) != cudaSuccess)
            return e;
        MergeArgs m;
        m.part_ms = c->cg_part_ms;
        m.part_top = c->cg_part_top;
        m.fr_tok = c->cg_fr_tok;
        m.fr_cand = c->cg_fr_cand;
        m.fr_S = c->cg_fr_S;
        m.fr_n = c->cg_fr_n;
        m.c_S = c->cg_c_S;
        m.c_meta = c->cg_c_meta;
        m.cand_lp = cand_lp;
        m.cand_ids = cand_ids;
        m.frontier_tok = frontier_tok;
        m.R = R;
        m.L = L;
        m.d = d;
        m.Fd = Fd;
        m.F = F;
        m.k = K;
        m.grid = grid;
        m.Cmax = cond_tree_cmax(cfg);
        m.base = base;
        cg_merge_kernel<<<R, 32 * CG_MAXF, 0, s>>>(m);
        if ((e = cudaGetLastError()) != cudaSuccess)
            return e;
        base += Fd * K;
    }
    PackArgs pk;
    pk.c_S = c->cg_c_S;
    pk.c_meta = c->cg_c_meta;
    pk.tree_tokens = tree_tokens;
    pk.parents = parents;
    pk.depths = depths;
    pk.n_nodes = n_nodes;
    pk.mask = mask;
    pk.C = base;
    pk.Cmax = cond_tree_cmax(cfg);
    pk.N = cfg.B;
    cg_pack_kernel<<<R, 256, 0, s>>>(pk);
    return cudaGetLastError();
}
