// markov.cu -- the SparklingTree table tree ("SparklingTree: 30-40% faster
// speculative decoding over DSpark", sections "Solving the candidate tree
// construction" and "Building SparklingTree"; the Markov head of "First
// order markov model conditioning": a bias W1[x_prev] W2 on the next
// position's logits, written z_d(b | a) = l_d[b] + W[b] . E[a]).
//
//  * The prefilter keeps every depth's C best draft tokens: a1's kernels with
//    K = C.
//  * mk_table_kernel: one CTA per (request, depth). The parents' E rows
//    (the anchor at depth 0, else depth d-1's kept tokens) and the children's
//    W rows (depth d's kept tokens) are gathered by cp.async into 128-byte
//    swizzled K-major tiles. One tcgen05 MMA chain gives the 128 x 128 bias
//    block in TMEM (M = parents, N = children, K = H, fp32 accumulation).
//    The epilogue adds l_d, takes each parent row's log-softmax over the
//    kept children, and writes the rows out through shared memory.
//  * mk_tree_kernel: one warp per request runs Algorithm 1 with a list per
//    parent. A node's children are its table row in order of (lp desc,
//    token asc); instead of sorting a row, each push takes the largest key
//    below the previous child's key with a warp-wide scan of the row. Rows
//    of expanded nodes stay in shared memory for their later sibling
//    pushes.
#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "ddt_device.cuh"
#include "ddt_internal.h"
#include "tc_ptx.cuh"

namespace {

constexpr int MK_THREADS = 128;  // table kernel: 4 warps = the 4 TMEM lane quarters (parent rows)
constexpr int MK_N = 128;        // children per tile (N of the MMA)
constexpr int MK_CMAX = 128;     // largest prefilter width
constexpr int MK_TROW = MK_N + 1;  // row stride of the staged table (floats, bank-conflict free)
constexpr long long MK_WAIT = 4000000000LL;

// order-preserving map of a (non-NaN) float to uint32
DDT_DEVINL uint32_t mk_fkey(float x)
{
    const uint32_t b = __float_as_uint(x + 0.0f);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
DDT_DEVINL float mk_fkey_inv(uint32_t k)
{
    return (k & 0x80000000u) ? __uint_as_float(k & 0x7FFFFFFFu) : __uint_as_float(~k);
}

DDT_DEVINL bool mk_wait(uint32_t bar, uint32_t parity, int32_t *status)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity))
        if (clock64() - t0 > MK_WAIT) {
            atomicOr(status, DDT_DEV_TIMEOUT);
            return false;
        }
    return true;
}

struct TableArgs {
    const uint16_t *ell;     // [R, L, V] bf16
    const uint16_t *W, *E;   // [V, H] bf16
    const int32_t *anchors;  // [R]
    const int32_t *cand;     // [R, L, C]
    float *tab;              // [R, L, C, C]
    int R, L, V, H, C;
    int32_t *status;
};

// shared memory of the table kernel (offsets from a 1024-byte aligned base):
// A and B operand tiles, then (after the MMA) the staged table over both
struct TableSmem {
    uint32_t a, b, lv, bar, total;
};
__host__ __device__ inline TableSmem table_layout(int H)
{
    TableSmem S;
    const uint32_t nblk = (uint32_t)H / 64;
    S.a = 0;
    S.b = nblk * 16384u;
    uint32_t end = 2 * nblk * 16384u;
    const uint32_t stage = (uint32_t)MK_CMAX * MK_TROW * 4u;
    if (end < stage)
        end = stage;
    S.lv = (end + 15u) & ~15u;  // l of the kept children: [128] floats
    S.bar = S.lv + 4u * MK_N;   // [0]: MMA done, [8]: TMEM address
    S.total = S.bar + 16;
    return S;
}

__global__ void __launch_bounds__(MK_THREADS, 1)
mk_table_kernel(const TableArgs a)
{
    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw = (uint32_t)__cvta_generic_to_shared(smem_raw);
    const uint32_t sb = (raw + 1023u) & ~1023u;
    unsigned char *sgen = smem_raw + (sb - raw);
    const TableSmem S = table_layout(a.H);
    const int rd = blockIdx.x, r = rd / a.L, d = rd - r * a.L;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t bar = sb + S.bar;
    float *s_l = reinterpret_cast<float *>(sgen + S.lv);

    if (tid == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(bar + 8, MK_N);
        tmem_relinquish();
    }
    // A: the parents' E rows; B: the kept children's W rows (zero rows pad to 128)
    const int32_t *cd = a.cand + (int64_t)rd * a.C;
    const int32_t *cp = a.cand + (int64_t)(rd - (d > 0 ? 1 : 0)) * a.C;
    const int per = a.H / 8;  // 16-byte chunks per row
    for (int i = tid; i < MK_N * per; i += MK_THREADS) {
        const int p = i / per, c = i - p * per;
        const uint32_t off = (uint32_t)(c >> 3) * 16384u + (uint32_t)p * 128u + ((uint32_t)((c & 7) ^ (p & 7)) << 4);
        int pt = -1, ct = -1;
        if (d == 0)
            pt = (p == 0) ? a.anchors[r] : -1;
        else if (p < a.C)
            pt = cp[p];
        if (p < a.C)
            ct = cd[p];
        const bool pok = pt >= 0 && pt < a.V, cok = ct >= 0 && ct < a.V;
        cp_async_16(sb + S.a + off, pok ? (const void *)(a.E + (int64_t)pt * a.H + c * 8) : (const void *)a.E,
                    pok ? 16u : 0u);
        cp_async_16(sb + S.b + off, cok ? (const void *)(a.W + (int64_t)ct * a.H + c * 8) : (const void *)a.W,
                    cok ? 16u : 0u);
    }
    for (int b = tid; b < MK_N; b += MK_THREADS) {
        const int ct = (b < a.C) ? cd[b] : -1;
        s_l[b] = (ct >= 0 && ct < a.V) ? bf16_to_f32(a.ell[(int64_t)rd * a.V + ct]) : DDT_NEG_INF;
    }
    cp_async_wait_all();
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(sgen + S.bar + 8);
    if (tid == 0) {
        const uint32_t idesc = idesc_bf16(128, MK_N, false, false);
        const uint64_t dA = sdesc_sw128(sb + S.a, 16, 1024), dB = sdesc_sw128(sb + S.b, 16, 1024);
        for (int kk = 0; kk < a.H / 16; ++kk) {
            const uint32_t off = ((uint32_t)(kk >> 2) * 16384u + (uint32_t)(kk & 3) * 32u) >> 4;
            mma_bf16(tmem, dA + off, dB + off, idesc, kk > 0 ? 1u : 0u);
        }
        mma_commit(bar);
    }
    const bool ok = __syncthreads_and(mk_wait(bar, 0, a.status) ? 1 : 0) != 0;
    tc_fence_after();
    // thread = parent row (its TMEM lane): max, then the sum of exp, then lp
    const uint32_t ta = tmem + ((uint32_t)(warp * 32) << 16);
    float m = DDT_NEG_INF, ssum = 0.f;
    if (ok) {
#pragma unroll 1
        for (int c0 = 0; c0 < MK_N; c0 += 32) {
            uint32_t acc[32];
            tmem_ld16(ta + c0, acc);
            tmem_ld16(ta + c0 + 16, acc + 16);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 32; ++j)
                m = fmaxf(m, __uint_as_float(acc[j]) + s_l[c0 + j]);
        }
        const float nb = -m * DDT_LOG2E;
#pragma unroll 1
        for (int c0 = 0; c0 < MK_N; c0 += 32) {
            uint32_t acc[32];
            tmem_ld16(ta + c0, acc);
            tmem_ld16(ta + c0 + 16, acc + 16);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 32; ++j)
                ssum += ex2(fmaf(__uint_as_float(acc[j]) + s_l[c0 + j], DDT_LOG2E, nb));
        }
    }
    const float lse = m + logf(ssum);
    // rows that hold a table row: the anchor's at depth 0, every kept parent's after
    const bool valid = (d == 0) ? (tid == 0) : (tid < a.C);
    float *T = reinterpret_cast<float *>(sgen);  // [128][MK_TROW], over the operand tiles
    if (ok) {
#pragma unroll 1
        for (int c0 = 0; c0 < MK_N; c0 += 32) {
            uint32_t acc[32];
            tmem_ld16(ta + c0, acc);
            tmem_ld16(ta + c0 + 16, acc + 16);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 32; ++j)
                T[tid * MK_TROW + c0 + j] = valid ? (__uint_as_float(acc[j]) + s_l[c0 + j]) - lse : DDT_NEG_INF;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (ok) {
        float *dst = a.tab + (int64_t)rd * a.C * a.C;
        for (int row = warp; row < a.C; row += MK_THREADS / 32)
            for (int b = lane; b < a.C; b += 32)
                dst[(int64_t)row * a.C + b] = T[row * MK_TROW + b];
    }
    if (!ok && tid == 0) {  // a wait gave up: let the MMA finish before the TMEM goes (bounded)
        const long long t0 = clock64();
        while (!mbar_try_wait(bar, 0) && clock64() - t0 < 200000000LL) {
        }
    }
    __syncthreads();
    if (warp == 0)
        tmem_dealloc(tmem, MK_N);
}

// ---------------------------------------------------------------- the tree
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
    uint64_t b = (uint64_t)__double_as_longlong(x);
    if (b == 0x8000000000000000ull)
        b = 0ull;  // -0 sorts as +0
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

// a child's key in its parent's row: lp high (order-preserving), the
// complemented token low (equal lp: the lower token first); 0 = none
DDT_DEVINL uint64_t child_key(float lp, int tok)
{
    return (lp == DDT_NEG_INF) ? 0ull : (((uint64_t)mk_fkey(lp) << 32) | (uint32_t)~(uint32_t)tok);
}

// the warp's largest key below `bound` among a lane's keys k[0..3]; the
// winning column to every lane (-1: none)
DDT_DEVINL uint64_t warp_best_below(const uint64_t *k, uint64_t bound, int lane, int &col)
{
    uint64_t best = 0ull;
    int bc = -1;
#pragma unroll
    for (int i = 0; i < 4; ++i)
        if (k[i] < bound && k[i] > best) {
            best = k[i];
            bc = lane + 32 * i;
        }
    const uint32_t mh = __reduce_max_sync(0xFFFFFFFFu, (uint32_t)(best >> 32));
    const uint32_t ml = __reduce_max_sync(0xFFFFFFFFu, (uint32_t)(best >> 32) == mh ? (uint32_t)best : 0u);
    const uint64_t w = ((uint64_t)mh << 32) | ml;
    const unsigned who = __ballot_sync(0xFFFFFFFFu, best == w && best != 0ull);
    col = (who != 0u) ? __shfl_sync(0xFFFFFFFFu, bc, __ffs(who) - 1) : -1;
    return (who != 0u) ? w : 0ull;
}

constexpr int SLOTS = 4;  // frontier slots per lane: 128 >= B entries

struct TreeArgs {
    const int32_t *cand;  // [R, L, C]
    const float *tab;     // [R, L, C, C]
    int L, C, B;
    int32_t *tree_tokens, *parents, *depths, *n_nodes;
    uint32_t *mask;
};

__global__ void __launch_bounds__(32)
mk_tree_kernel(const TreeArgs a)
{
    const int r = blockIdx.x, lane = threadIdx.x;
    const int L = a.L, C = a.C, B = a.B, P = B + 1, W = (P + 31) >> 5;
    extern __shared__ __align__(16) unsigned char mk_smem[];
    int *s_cand = reinterpret_cast<int *>(mk_smem);          // [L][C] kept tokens
    float *s_rows = reinterpret_cast<float *>(s_cand + L * C);  // [P][C] node n's children row
    int *s_tok = reinterpret_cast<int *>(s_rows + P * C);     // [B]
    int *s_par = s_tok + B;                                    // [P]
    int *s_dep = s_par + P;                                    // [P]
    const int32_t *cr = a.cand + (int64_t)r * L * C;
    const float *tr = a.tab + (int64_t)r * L * C * C;
    for (int i = lane; i < L * C; i += 32)
        s_cand[i] = cr[i];
    for (int i = lane; i < P; i += 32) {
        s_par[i] = -1;
        s_dep[i] = (i == 0) ? 0 : -1;
        if (i < B)
            s_tok[i] = -1;
    }
    __syncwarp();

    // frontier slots (registers): score key, the parent's score key, rank
    // tuple, the entry's key in its parent's row and its column there, parent
    // node, depth and rank; an empty slot has score key 0
    uint64_t sk[SLOTS], pk[SLOTS], kh[SLOTS], kl[SLOTS], ck[SLOTS];
    int cb[SLOTS], par[SLOTS], dep[SLOTS], rnk[SLOTS];
#pragma unroll
    for (int f = 0; f < SLOTS; ++f) {
        sk[f] = pk[f] = kh[f] = kl[f] = ck[f] = 0;
        cb[f] = par[f] = dep[f] = rnk[f] = 0;
    }
    const int kmax = B < C ? B : C;  // ranks at or above B can never enter the tree

    // a row into shared memory (row n) and its keys
    auto load_row = [&](const float *src, int n, const int *toks, uint64_t *k) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int b = lane + 32 * i;
            float lp = DDT_NEG_INF;
            if (b < C) {
                lp = src[b];
                s_rows[n * C + b] = lp;
            }
            k[i] = (b < C) ? child_key(lp, toks[b]) : 0ull;
        }
    };
    auto row_keys = [&](int n, const int *toks, uint64_t *k) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int b = lane + 32 * i;
            k[i] = (b < C) ? child_key(s_rows[n * C + b], toks[b]) : 0ull;
        }
    };

    {  // the root's row (depth 0, row 0: the anchor) and its first child
        uint64_t k[4];
        load_row(tr, 0, s_cand, k);
        int col;
        const uint64_t w = warp_best_below(k, ~0ull, lane, col);
        if (w != 0ull && lane == 0) {
            pk[0] = skey(0.0);
            sk[0] = skey(0.0 + (double)mk_fkey_inv((uint32_t)(w >> 32)));
            field_or(kh[0], kl[0], 0, 1);
            ck[0] = w;
            cb[0] = col;
            dep[0] = 1;
        }
    }

    int count = 0;
    while (count < B) {
        // lane-local best slot
        int bf = 0;
        uint64_t bk = sk[0], bh = kh[0], bl = kl[0], bck = ck[0];
        int bpar = par[0], bdep = dep[0], brnk = rnk[0], bcb = cb[0];
#pragma unroll
        for (int f = 1; f < SLOTS; ++f)
            if (pops_before(sk[f], kh[f], kl[f], bk, bh, bl)) {
                bf = f;
                bk = sk[f];
                bh = kh[f];
                bl = kl[f];
                bck = ck[f];
                bpar = par[f];
                bdep = dep[f];
                brnk = rnk[f];
                bcb = cb[f];
            }
        // warp arg-best: score key high then low word; the rank tuple only on a tie
        unsigned cand = __ballot_sync(0xFFFFFFFFu, bk != 0);
        if (cand == 0u)
            break;  // every prefix is already in the tree
        cand = keep_max(cand, (uint32_t)(bk >> 32), lane);
        cand = keep_max(cand, (uint32_t)bk, lane);
        if (__popc(cand) > 1) {
            cand = keep_max(cand, ~(uint32_t)(bh >> 32), lane);
            cand = keep_max(cand, ~(uint32_t)bh, lane);
            cand = keep_max(cand, ~(uint32_t)(bl >> 32), lane);
            cand = keep_max(cand, ~(uint32_t)bl, lane);
        }
        const int wl = __ffs(cand) - 1;
        const uint64_t wk = __shfl_sync(0xFFFFFFFFu, bk, wl);
        const uint64_t wh = __shfl_sync(0xFFFFFFFFu, bh, wl);
        const uint64_t wlo = __shfl_sync(0xFFFFFFFFu, bl, wl);
        const uint64_t wck = __shfl_sync(0xFFFFFFFFu, bck, wl);
        const int wpar = __shfl_sync(0xFFFFFFFFu, bpar, wl);
        const int wdep = __shfl_sync(0xFFFFFFFFu, bdep, wl);
        const int wrnk = __shfl_sync(0xFFFFFFFFu, brnk, wl);
        const int wcb = __shfl_sync(0xFFFFFFFFu, bcb, wl);
        const double wS = skey_inv(wk);

        const int node = count + 1;
        if (lane == 0) {
            s_tok[count] = s_cand[(wdep - 1) * C + wcb];
            s_par[node] = wpar;
            s_dep[node] = wdep;
        }
        ++count;
        if (count == B)
            break;
        // the next child of the same parent: the largest key of the parent's
        // row below the popped one's; it reuses the popped slot
        uint64_t sib = 0ull;
        int scol = -1;
        if (wrnk + 1 < kmax) {
            uint64_t k[4];
            row_keys(wpar, s_cand + (wdep - 1) * C, k);
            sib = warp_best_below(k, wck, lane, scol);
        }
        if (lane == wl) {
#pragma unroll
            for (int f = 0; f < SLOTS; ++f)
                if (f == bf) {
                    if (sib != 0ull) {
                        sk[f] = skey(skey_inv(pk[f]) + (double)mk_fkey_inv((uint32_t)(sib >> 32)));
                        field_clear(kh[f], kl[f], wdep - 1);
                        field_or(kh[f], kl[f], wdep - 1, (uint64_t)(wrnk + 2));
                        rnk[f] = wrnk + 1;
                        ck[f] = sib;
                        cb[f] = scol;
                    } else {
                        sk[f] = 0;
                    }
                }
        }
        // the first child: the best of the popped node's own row (depth wdep,
        // row wcb), loaded now and kept for the node's later children
        if (wdep < L) {
            uint64_t k[4];
            load_row(tr + ((int64_t)wdep * C + wcb) * C, node, s_cand + wdep * C, k);
            int ccol;
            const uint64_t chk = warp_best_below(k, ~0ull, lane, ccol);
            if (chk != 0ull) {
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
                            sk[f] = skey(wS + (double)mk_fkey_inv((uint32_t)(chk >> 32)));
                            pk[f] = wk;
                            kh[f] = wh;
                            kl[f] = wlo;
                            field_or(kh[f], kl[f], wdep, 1ull);
                            ck[f] = chk;
                            cb[f] = ccol;
                            par[f] = node;
                            dep[f] = wdep + 1;
                            rnk[f] = 0;
                        }
                }
            }
        }
        __syncwarp();
    }
    __syncwarp();

    for (int i = lane; i < B; i += 32)
        a.tree_tokens[(int64_t)r * B + i] = s_tok[i];
    for (int i = lane; i < P; i += 32) {
        a.parents[(int64_t)r * P + i] = s_par[i];
        a.depths[(int64_t)r * P + i] = s_dep[i];
    }
    if (lane == 0)
        a.n_nodes[r] = count;
    if (a.mask != nullptr) {
        for (int i = lane; i < P; i += 32) {
            uint32_t words[4] = {0u, 0u, 0u, 0u};
            if (i <= count) {
                int cur = i;
                for (int step = 0; step <= DDT_MAX_L + 1 && cur >= 0; ++step) {
#pragma unroll
                    for (int w = 0; w < 4; ++w)
                        if (w == (cur >> 5))
                            words[w] |= 1u << (cur & 31);
                    cur = s_par[cur];
                }
            }
#pragma unroll
            for (int w = 0; w < 4; ++w)
                if (w < W)
                    a.mask[((int64_t)r * P + i) * W + w] = words[w];
        }
    }
}

size_t table_smem(int H)
{
    return (size_t)table_layout(H).total + 1024;  // + the slack for 1024-byte alignment
}

size_t tree_smem(int L, int C, int B)
{
    const int P = B + 1;
    return (size_t)L * C * 4 + (size_t)P * C * 4 + (size_t)(B + 2 * P) * 4;
}

}  // namespace

bool markov_supported(const ddt_config &cfg)
{
    const int H = cfg.markov_dim, C = cfg.prefilter;
    return H >= 64 && H <= 256 && H % 64 == 0 && C >= 1 && C <= MK_CMAX && cfg.B + 1 <= DDT_MAX_P &&
           cfg.L <= DDT_MAX_L && tree_smem(cfg.L, C, cfg.B) <= 200 * 1024 &&
           (int64_t)((cfg.V + topk_chunk_elems(cfg.draft_dtype) - 1) / topk_chunk_elems(cfg.draft_dtype)) * C <=
               TOPK_CAND_CAP;
}

cudaError_t launch_markov_table(const ddt_ctx *c, const uint16_t *ell, const uint16_t *W,
                                const uint16_t *E, const int32_t *anchors, int R, int32_t *cand,
                                float *tab, cudaStream_t s)
{
    const ddt_config &cfg = c->cfg;
    const int C = cfg.prefilter, L = cfg.L;
    // the prefilter: a1's kernels with K = C (their log-probs are not used)
    cudaError_t e = launch_topk_scratch(ell, DDT_BF16, R * L, cfg.V, C, c->mk_nch, c->mk_tk_val,
                                        c->mk_tk_idx, c->mk_tk_ms, c->mk_tk_cnt, c->mk_tk_lp, cand,
                                        c->status, s);
    if (e != cudaSuccess)
        return e;
    static size_t attr = 0;
    const size_t smem = table_smem(cfg.markov_dim);
    if (attr < table_smem(256)) {
        if ((e = cudaFuncSetAttribute(mk_table_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)table_smem(256))) != cudaSuccess)
            return e;
        attr = table_smem(256);
    }
    TableArgs a;
    a.ell = ell;
    a.W = W;
    a.E = E;
    a.anchors = anchors;
    a.cand = cand;
    a.tab = tab;
    a.R = R;
    a.L = L;
    a.V = cfg.V;
    a.H = cfg.markov_dim;
    a.C = C;
    a.status = c->status;
    mk_table_kernel<<<R * L, MK_THREADS, smem, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_markov_tree(const ddt_ctx *c, const int32_t *cand, const float *tab, int R,
                               int32_t *tree_tokens, int32_t *parents, int32_t *depths,
                               int32_t *n_nodes, uint32_t *mask, cudaStream_t s)
{
    const ddt_config &cfg = c->cfg;
    const size_t smem = tree_smem(cfg.L, cfg.prefilter, cfg.B);
    static size_t attr = 0;
    cudaError_t e;
    if (attr < 200 * 1024) {
        if ((e = cudaFuncSetAttribute(mk_tree_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      200 * 1024)) != cudaSuccess)
            return e;
        attr = 200 * 1024;
    }
    TreeArgs a;
    a.cand = cand;
    a.tab = tab;
    a.L = cfg.L;
    a.C = cfg.prefilter;
    a.B = cfg.B;
    a.tree_tokens = tree_tokens;
    a.parents = parents;
    a.depths = depths;
    a.n_nodes = n_nodes;
    a.mask = mask;
    mk_tree_kernel<<<R, 32, smem, s>>>(a);
    return cudaGetLastError();
}
