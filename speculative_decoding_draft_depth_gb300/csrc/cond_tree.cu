// cond_tree.cu -- the parent-conditioned draft tree ("Robot2050/TreeSpark",
// items 1 and 2): one backbone pass gives per-depth logits l_d [R, L, V]; a
// first-order Markov head specialises depth d to a parent token,
//   z_d(u) = l_d + W e(t_u),          W, E: [V, H] bf16,
// each parent keeps its k best children (log-softmax of z_d(u)), the F best
// children of a depth by joint path score become the next depth's parents,
// and the N best candidates of all depths are packed into the tree (prefix-
// closed: lp <= 0, and a parent sorts before its children).
//
// Per depth, two kernels, chained by programmatic dependent launch so that a
// kernel's prologue overlaps the previous kernel's tail:
//  * cg_gemm_kernel: the Markov bias of every frontier parent of every
//    request at once, as a tcgen05 GEMM with the parents in the TMEM lanes:
//    M = the parents' gathered embedding rows (up to 128, K-major in shared
//    memory), N = 128 vocabulary rows of W per tile (TMA, 128-byte swizzle,
//    two stages), K = H; fp32 accumulators in TMEM, double-buffered. Warp
//    roles: a TMA producer, an MMA issuer and eight epilogue warps; an
//    epilogue thread owns one parent (its TMEM lane) and streams a slice of
//    each tile's columns, adding l_d and keeping a running (max, sum of exp)
//    and top-k. Persistent CTAs stride over the vocabulary and write one
//    partial per parent.
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

constexpr int CG_EPI = 8;                      // epilogue warps: CG_EPI / 4 per TMEM lane quarter
constexpr int CG_NH = CG_EPI / 4;              // column slices of a tile
constexpr int CG_THREADS = 32 * (CG_EPI + 2);  // + TMA producer + MMA issuer
constexpr int CG_PROD = CG_EPI, CG_MMA = CG_EPI + 1;  // warp indices of the two roles
constexpr int CG_TILE = 128;                   // vocabulary columns per tile (N)
constexpr int CG_SLICE = CG_TILE / CG_NH;      // columns of a tile per epilogue warp
constexpr int CG_MAXK = 8;                     // children per parent
constexpr int CG_MAXNP = 128;                  // parents per depth (M: TMEM lanes)
constexpr int CG_MAXF = 8;                     // frontier width
constexpr int CG_TMEM_COLS = 2 * CG_TILE;      // two accumulator buffers
constexpr int CG_LROW = CG_TILE * 2 + 16;      // one l row of a tile in shared memory (padded)
constexpr int CG_LRMAX = 48;                   // requests whose l tiles are staged (more: direct loads)
constexpr long long CG_WAIT = 4000000000LL;
static_assert(CG_SLICE % 32 == 0, "epilogue slices are whole 32-column chunks");

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
// order-preserving map of a (non-NaN) double to uint64: path scores compare
// as integers (fp64 compares run on the narrow fp64 pipe)
DDT_DEVINL uint64_t dkey(double x)
{
    uint64_t b = (uint64_t)__double_as_longlong(x);
    if (b == (1ull << 63))
        b = 0ull;  // -0 sorts as +0
    return (b >> 63) ? ~b : (b | (1ull << 63));
}

struct GemmArgs {
    const uint16_t *W;        // [V, H] bf16 (the tiles come through the tensor map)
    const uint16_t *E;        // [V, H] bf16
    const uint16_t *ell;      // [R, L, V] bf16
    const int32_t *fr_tok;    // [R, F] frontier tokens (-1: none)
    const int32_t *anchors;   // [R] the roots: the parents of depth 1
    float2 *part_ms;          // [NP, grid] (max, sum of exp)
    uint64_t *part_top;       // [NP, grid, CG_MAXK] value keys
    int R, L, V, H, d, Fd, F, NP, k;
    int lsm;                  // l tiles staged in shared memory by bulk copies (else direct loads)
    int vec;                  // l rows are 16-byte aligned (V % 8 == 0, aligned base)
    uint32_t *thr;            // [CG_MAXNP] this depth's per-parent bounds (value keys, 0: none)
    const int32_t *seeds;     // [R, L, k] the draft's own k best columns of each depth
    int srows;                // seed rows staged (R * k; 0 when they do not fit: no seeds)
    int32_t *status;
};

// per-thread running state of one parent over the columns it scans
struct ColState {
    float m;       // running max
    uint64_t s2;   // two partial sums of exp(z - m), packed
    float kth;     // the k-th largest value kept (-inf while fewer than k)
    float lb;      // just below a bound that k values of this parent (grid-wide) reach
    float tv[CG_MAXK];
    int ti[CG_MAXK];
};

DDT_DEVINL void col_reset(ColState &c)
{
    c.m = DDT_NEG_INF;
    c.s2 = f2pack(0.f, 0.f);
    c.kth = DDT_NEG_INF;
    c.lb = DDT_NEG_INF;
#pragma unroll
    for (int j = 0; j < CG_MAXK; ++j) {
        c.tv[j] = DDT_NEG_INF;
        c.ti[j] = -1;
    }
}

// insert x (id) into the descending top-k; equal values keep the earlier
// (lower) id, which a thread sees first. Every list index is static so that
// the state stays in registers.
DDT_DEVINL void col_insert(ColState &c, int k, float x, int id)
{
    float v = x;
    int i2 = id;
#pragma unroll
    for (int j = 0; j < CG_MAXK; ++j) {
        if (j < k) {
            const bool take = (c.ti[j] < 0) || (v > c.tv[j]);
            if (take) {
                const float tv = c.tv[j];
                const int ti = c.ti[j];
                c.tv[j] = v;
                c.ti[j] = i2;
                v = tv;
                i2 = ti;
            }
        }
    }
    float kth = __builtin_huge_valf();
#pragma unroll
    for (int j = 0; j < CG_MAXK; ++j)
        if (j < k)
            kth = fminf(kth, c.tv[j]);
    c.kth = kth;
}

// 32 consecutive columns v0.. of one parent: z = accumulator + l (bf16),
// the first nvalid of them real. A value enters the top-k only above both the
// thread's own k-th value and the borrowed bound (values below a value that k
// others reach cannot be among the k best).
DDT_DEVINL void col_scan32(ColState &c, int k, const uint32_t *acc, const uint4 *lv, int v0, int nvalid)
{
    float z[32];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const uint32_t w[4] = {lv[q].x, lv[q].y, lv[q].z, lv[q].w};
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            const int j = 8 * q + 2 * t;
            f2unpack(f2add(f2pack(__uint_as_float(acc[j]), __uint_as_float(acc[j + 1])),
                           f2pack(bf16lo(w[t]), bf16hi(w[t]))),
                     z[j], z[j + 1]);
        }
    }
    if (nvalid < 32) {
#pragma unroll
        for (int j = 0; j < 32; ++j)
            if (j >= nvalid)
                z[j] = DDT_NEG_INF;
    }
    float mx[8];
#pragma unroll
    for (int j = 0; j < 8; ++j)
        mx[j] = fmaxf(fmaxf(z[j], z[j + 8]), fmaxf(z[j + 16], z[j + 24]));
#pragma unroll
    for (int j = 0; j < 4; ++j)
        mx[j] = fmaxf(mx[j], mx[j + 4]);
    const float m = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
    if (m == DDT_NEG_INF)
        return;
    if (m > c.m) {
        const float sc = ex2((c.m - m) * DDT_LOG2E);  // 0 on the first real value
        float s0, s1;
        f2unpack(c.s2, s0, s1);
        c.s2 = f2pack(s0 * sc, s1 * sc);
        c.m = m;
    }
    const float nb = -c.m * DDT_LOG2E;
    const uint64_t c2 = f2pack(DDT_LOG2E, DDT_LOG2E), b2 = f2pack(nb, nb);
    uint64_t e0 = f2pack(0.f, 0.f), e1 = e0;
#pragma unroll
    for (int j = 0; j < 32; j += 4) {
        float t0, t1, t2, t3;
        f2unpack(f2fma(f2pack(z[j], z[j + 1]), c2, b2), t0, t1);
        f2unpack(f2fma(f2pack(z[j + 2], z[j + 3]), c2, b2), t2, t3);
        e0 = f2add(e0, f2pack(ex2(t0), ex2(t1)));
        e1 = f2add(e1, f2pack(ex2(t2), ex2(t3)));
    }
    c.s2 = f2add(c.s2, f2add(e0, e1));
    if (m > fmaxf(c.kth, c.lb)) {
        // the columns above the k-th kept value: a few are taken in column
        // order, each picked from z by a tournament on the bits of its index
        // (static register indices, no local memory)
        const float th = fmaxf(c.kth, c.lb);
        uint32_t msk = 0u;
#pragma unroll
        for (int j = 0; j < 32; ++j)
            msk |= (z[j] > th ? 1u : 0u) << j;
        if (__popc(msk) > 2) {
            // many (a thread's first chunk): at most k extractions of the
            // chunk's largest remaining value, lowest column first on ties
            for (int it = 0; it < k; ++it) {
                float t16[16];
#pragma unroll
                for (int t = 0; t < 16; ++t)
                    t16[t] = fmaxf(z[t], z[t + 16]);
#pragma unroll
                for (int t = 0; t < 8; ++t)
                    t16[t] = fmaxf(t16[t], t16[t + 8]);
#pragma unroll
                for (int t = 0; t < 4; ++t)
                    t16[t] = fmaxf(t16[t], t16[t + 4]);
                const float mv = fmaxf(fmaxf(t16[0], t16[1]), fmaxf(t16[2], t16[3]));
                if (!(mv > fmaxf(c.kth, c.lb)))
                    break;
                uint32_t eq = 0u;
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    eq |= (z[j] == mv ? 1u : 0u) << j;
                const int jm = __ffs(eq) - 1;
                col_insert(c, k, mv, v0 + jm);
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    if (j == jm)
                        z[j] = DDT_NEG_INF;
            }
            msk = 0u;
        }
        while (msk != 0u) {
            const int j = __ffs(msk) - 1;
            msk &= msk - 1u;
            float s16[16], s8[8], s4[4], s2[2];
#pragma unroll
            for (int t = 0; t < 16; ++t)
                s16[t] = (j & 16) ? z[t + 16] : z[t];
#pragma unroll
            for (int t = 0; t < 8; ++t)
                s8[t] = (j & 8) ? s16[t + 8] : s16[t];
#pragma unroll
            for (int t = 0; t < 4; ++t)
                s4[t] = (j & 4) ? s8[t + 4] : s8[t];
#pragma unroll
            for (int t = 0; t < 2; ++t)
                s2[t] = (j & 2) ? s4[t + 2] : s4[t];
            const float x = (j & 1) ? s2[1] : s2[0];
            if (x > fmaxf(c.kth, c.lb))  // the threshold rises as values go in
                col_insert(c, k, x, v0 + j);
        }
    }
}

// the 32 l values of columns v0.. of one row (bf16, zero past nvalid)
DDT_DEVINL void load_l32(const uint16_t *row, int v0, int nvalid, bool vec, uint4 *lv)
{
    if (vec && nvalid >= 32) {
        const uint4 *p = reinterpret_cast<const uint4 *>(row + v0);
#pragma unroll
        for (int q = 0; q < 4; ++q)
            lv[q] = __ldg(p + q);
    } else {
        uint32_t w[16];
#pragma unroll
        for (int t = 0; t < 16; ++t) {
            const uint32_t lo = (2 * t < nvalid) ? (uint32_t)__ldg(row + v0 + 2 * t) : 0u;
            const uint32_t hi = (2 * t + 1 < nvalid) ? (uint32_t)__ldg(row + v0 + 2 * t + 1) : 0u;
            w[t] = lo | (hi << 16);
        }
#pragma unroll
        for (int q = 0; q < 4; ++q)
            lv[q] = make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
    }
}

DDT_DEVINL uint32_t ld_relaxed_u32(const uint32_t *p)
{
    uint32_t v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
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

// shared-memory layout of the GEMM (offsets from a 1024-byte aligned base)
struct GemmSmem {
    uint32_t a, w, wst, l, lst, seed, sw, sl, tok, bar, total;
};
// H: the embedding width; lrows: requests whose l tiles are staged (0: none);
// srows: bound seed rows staged (0: none)
__host__ __device__ inline GemmSmem gemm_layout(int H, int lrows, int srows)
{
    GemmSmem L;
    const uint32_t nblk = (uint32_t)H / 64;
    L.a = 0;                        // parents' rows: [nblk][128 rows][128 B]
    L.wst = nblk * 16384u;          // one W tile: [nblk][128 rows][128 B]
    L.w = L.a + nblk * 16384u;      // two W stages (after the main loop: the exchange)
    L.lst = ((uint32_t)lrows * CG_LROW + 127u) & ~127u;
    L.l = L.w + 2 * L.wst;          // two l stages: [requests][CG_LROW bytes]
    L.seed = L.l + 2 * L.lst;       // the seeds' values: [CG_MAXK][128 parents] floats
    L.sw = L.seed + 4 * CG_MAXK * CG_MAXNP;   // seed rows W[v]: [srows][H * 2 + 16 bytes]
    L.sl = L.sw + (uint32_t)srows * (H * 2 + 16);  // seed values l[v]: [srows] floats
    L.tok = L.sl + (((uint32_t)srows * 4 + 15u) & ~15u);  // the parents' tokens
    L.bar = L.tok + 4 * CG_MAXNP;
    L.total = L.bar + 128;
    return L;
}
// barrier offsets within the barrier block
constexpr uint32_t GB_WFULL = 0, GB_WEMPTY = 16, GB_AFULL = 32, GB_AEMPTY = 48, GB_LFULL = 64,
                   GB_FIN = 80, GB_TMEM = 88;
// exchange record of one parent between the column slices: top-k keys, max, sum
constexpr uint32_t CG_XREC = CG_MAXK * 8 + 8;
static_assert((CG_NH - 1) * CG_MAXNP * CG_XREC <= 2 * 16384, "exchange fits the W stages");

__global__ void __launch_bounds__(CG_THREADS, 1)
cg_gemm_kernel(const __grid_constant__ CUtensorMap tm_w, const GemmArgs a)
{
    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw = (uint32_t)__cvta_generic_to_shared(smem_raw);
    const uint32_t sb = (raw + 1023u) & ~1023u;
    unsigned char *sgen = smem_raw + (sb - raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const GemmSmem S = gemm_layout(a.H, a.lsm ? a.R : 0, a.srows);
    const uint32_t bar = sb + S.bar;
    const int ntiles = (a.V + CG_TILE - 1) / CG_TILE;
    const int nmine = ((int)blockIdx.x < ntiles) ? (ntiles - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
    const int nblk = a.H / 64;

    if (tid == 0) {
        for (int s = 0; s < 2; ++s) {
            mbar_init(bar + GB_WFULL + 8 * s, 1);
            mbar_init(bar + GB_WEMPTY + 8 * s, 1);
            mbar_init(bar + GB_AFULL + 8 * s, 1);
            mbar_init(bar + GB_AEMPTY + 8 * s, CG_EPI);
            mbar_init(bar + GB_LFULL + 8 * s, 1);
        }
        mbar_init(bar + GB_FIN, 1);
        fence_mbar_init();
    }
    if (warp == CG_MMA) {
        tmem_alloc(bar + GB_TMEM, CG_TMEM_COLS);
        tmem_relinquish();
    }
    __syncthreads();

    // W and l are inputs of the whole call: the first tiles load before the
    // wait for the previous kernel of the chain. W is read once per depth, so
    // its lines are kept in L2 ahead of other traffic.
    int loads0 = 0, loads1 = 0, lloads0 = 0, lloads1 = 0;  // loads issued per stage (producer lane)
    const uint64_t keep = policy_evict_last();
    auto load_tile = [&](int i) {
        const int s = i & 1;
        const int tile = (int)blockIdx.x + i * (int)gridDim.x;
        if (s == 0)
            ++loads0;
        else
            ++loads1;
        const uint32_t fb = bar + GB_WFULL + 8 * s;
        mbar_arrive_expect_tx(fb, S.wst);
        for (int b = 0; b < nblk; ++b)
            tma_load_2d_hint(sb + S.w + s * S.wst + b * 16384u, &tm_w, b * 64, tile * CG_TILE, fb, keep);
    };
    // the tile's columns of every request's l_d row (a multiple of 16 bytes: V % 8 == 0)
    auto load_l = [&](int i) {
        const int s = i & 1;
        const int v0 = ((int)blockIdx.x + i * (int)gridDim.x) * CG_TILE;
        const int ncol = (a.V - v0 < CG_TILE) ? a.V - v0 : CG_TILE;
        if (s == 0)
            ++lloads0;
        else
            ++lloads1;
        const uint32_t fb = bar + GB_LFULL + 8 * s;
        mbar_arrive_expect_tx(fb, (uint32_t)(ncol * 2 * a.R));
        for (int r = 0; r < a.R; ++r)
            bulk_load(sb + S.l + s * S.lst + r * CG_LROW, a.ell + ((int64_t)r * a.L + a.d) * a.V + v0,
                      (uint32_t)(ncol * 2), fb);
    };
    if (warp == CG_PROD && lane == 0) {
        prefetch_tmap(&tm_w);
        for (int i = 0; i < 2 && i < nmine; ++i) {
            load_tile(i);
            if (a.lsm)
                load_l(i);
        }
    }
    // the bound seeds' rows W[v] and values l[v]: inputs of the call, like W,
    // staged before the wait (rows [R * k][H * 2 + 16 bytes], values [R * k])
    const int nrow = a.srows;  // seed rows (request, j); 0: no seeds staged
    if (warp < CG_EPI && nrow > 0) {
        const int per = a.H / 8;
        for (int i = tid; i < nrow * per; i += 32 * CG_EPI) {
            const int sr = i / per, c = i - sr * per;
            const int rr = sr / a.k, j = sr - rr * a.k;
            const int v = a.seeds[((int64_t)rr * a.L + a.d) * a.k + j];
            const bool okv = v >= 0 && v < a.V;
            cp_async_16(sb + S.sw + sr * (a.H * 2 + 16) + c * 16,
                        okv ? (const void *)(a.W + (int64_t)v * a.H + c * 8) : (const void *)a.W,
                        okv ? 16u : 0u);
            if (c == 0)
                reinterpret_cast<float *>(sgen + S.sl)[sr] =
                    okv ? bf16_to_f32(a.ell[((int64_t)rr * a.L + a.d) * a.V + v]) : DDT_NEG_INF;
        }
    }
    pdl_wait();
    // the parents' embedding rows, K-major with the 128-byte swizzle (zero rows
    // pad to 128), gathered by asynchronous copies once the tokens are known
    int *s_tok = reinterpret_cast<int *>(sgen + S.tok);
    for (int p = tid; p < CG_MAXNP; p += CG_THREADS) {
        int tok = -1;
        if (p < a.NP) {
            const int r = p / a.Fd, f = p % a.Fd;
            tok = (a.d == 0) ? a.anchors[r] : a.fr_tok[r * a.F + f];
        }
        s_tok[p] = (tok >= 0 && tok < a.V) ? tok : -1;
    }
    __syncthreads();
    for (int i = tid; i < CG_MAXNP * (a.H / 8); i += CG_THREADS) {
        const int p = i / (a.H / 8), c = i % (a.H / 8);
        const int tok = s_tok[p];
        const int blk = c >> 3, ch = c & 7;
        cp_async_16(sb + S.a + blk * 16384 + p * 128 + ((ch ^ (p & 7)) << 4),
                    (tok >= 0) ? (const void *)(a.E + (int64_t)tok * a.H + c * 8) : (const void *)a.E,
                    (tok >= 0) ? 16u : 0u);
    }
    cp_async_wait_all();
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(sgen + S.bar + GB_TMEM);

    bool ok = true;
    ColState st;
    col_reset(st);
    const int q = warp & 3, h = warp >> 2;   // epilogue: lane quarter, column slice
    const int p = 32 * q + lane;             // this thread's parent (TMEM lane)
    // seeds of the bound: z of each parent at its request's k best draft
    // columns, less a margin far above the rounding difference between this
    // sum and the tensor cores' (the epilogue warps, while the first tiles
    // load and multiply)
    const float *zs = reinterpret_cast<const float *>(sgen + S.seed);  // [CG_MAXK][128]
    if (warp < CG_EPI) {
        // a thread per (parent, seed): a compact loop over shared memory (this
        // runs once per CTA, so its code is kept small)
        for (int t = tid; t < a.NP * a.k && nrow > 0; t += 32 * CG_EPI) {
            const int pp = t / a.k, j = t - pp * a.k, sr = (pp / a.Fd) * a.k + j;
            const float lv = reinterpret_cast<const float *>(sgen + S.sl)[sr];
            const unsigned char *wrow = sgen + S.sw + sr * (a.H * 2 + 16);
            uint64_t dot2 = f2pack(0.f, 0.f), abs2 = dot2;
#pragma unroll 1
            for (int c = 0; c < a.H / 8; ++c) {
                const uint4 w = *reinterpret_cast<const uint4 *>(wrow + c * 16);
                const uint4 e = *reinterpret_cast<const uint4 *>(sgen + S.a + (c >> 3) * 16384 + pp * 128 +
                                                                 (((c & 7) ^ (pp & 7)) << 4));
                const uint32_t ww[4] = {w.x, w.y, w.z, w.w}, ee[4] = {e.x, e.y, e.z, e.w};
#pragma unroll
                for (int t2 = 0; t2 < 4; ++t2) {
                    dot2 = f2fma(f2pack(bf16lo(ww[t2]), bf16hi(ww[t2])), f2pack(bf16lo(ee[t2]), bf16hi(ee[t2])),
                                 dot2);
                    const uint32_t wa = ww[t2] & 0x7FFF7FFFu, ea = ee[t2] & 0x7FFF7FFFu;
                    abs2 = f2fma(f2pack(bf16lo(wa), bf16hi(wa)), f2pack(bf16lo(ea), bf16hi(ea)), abs2);
                }
            }
            float d0, d1, a0, a1;
            f2unpack(dot2, d0, d1);
            f2unpack(abs2, a0, a1);
            const float z = lv + (d0 + d1);
            reinterpret_cast<float *>(sgen + S.seed)[j * CG_MAXNP + pp] =
                (lv != DDT_NEG_INF) ? z - 1e-3f * (1.f + fabsf(z) + (a0 + a1)) : DDT_NEG_INF;
        }
        asm volatile("bar.sync 1, %0;" ::"r"(CG_EPI * 32) : "memory");
        // k values of the parent reach the smallest seed: values below it are
        // not among the k best
        if (p < a.NP && nrow > 0) {
            float B = __builtin_huge_valf();
            for (int j = 0; j < a.k; ++j)
                B = fminf(B, zs[j * CG_MAXNP + p]);
            if (B != DDT_NEG_INF) {
                st.lb = nextafterf(B, DDT_NEG_INF);
                if (blockIdx.x == 0 && h == 0)
                    atomicMax(a.thr + p, fkey(B));
            }
        }
    }
    if (warp == CG_PROD) {
        if (lane == 0)
            for (int i = 2; i < nmine; ++i) {
                if (!cg_wait(bar + GB_WEMPTY + 8 * (i & 1), ((i >> 1) - 1) & 1, a.status)) {
                    ok = false;
                    break;
                }
                load_tile(i);
                // the l stage is free once the epilogue has read tile i - 2
                if (a.lsm) {
                    if (!cg_wait(bar + GB_AEMPTY + 8 * (i & 1), ((i >> 1) - 1) & 1, a.status)) {
                        ok = false;
                        break;
                    }
                    load_l(i);
                }
            }
        // every load issued has landed (consumed already, unless a wait gave up)
        if (lane == 0) {
            if (loads0 > 0)
                cg_drain(bar + GB_WFULL, (loads0 - 1) & 1);
            if (loads1 > 0)
                cg_drain(bar + GB_WFULL + 8, (loads1 - 1) & 1);
            if (lloads0 > 0)
                cg_drain(bar + GB_LFULL, (lloads0 - 1) & 1);
            if (lloads1 > 0)
                cg_drain(bar + GB_LFULL + 8, (lloads1 - 1) & 1);
        }
    } else if (warp == CG_MMA) {
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16(128, CG_TILE, false, false);
            const uint64_t dA = sdesc_sw128(sb + S.a, 16, 1024);
            for (int i = 0; i < nmine; ++i) {
                const int s = i & 1;
                if (!cg_wait(bar + GB_WFULL + 8 * s, (i >> 1) & 1, a.status)) {
                    ok = false;
                    break;
                }
                if (i >= 2 && !cg_wait(bar + GB_AEMPTY + 8 * s, ((i >> 1) - 1) & 1, a.status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint64_t dB = sdesc_sw128(sb + S.w + s * S.wst, 16, 1024);
                for (int kk = 0; kk < a.H / 16; ++kk) {
                    const uint32_t off = ((kk >> 2) * 16384u + (kk & 3) * 32u) >> 4;
                    mma_bf16(tmem + s * CG_TILE, dA + off, dB + off, idesc, kk > 0 ? 1u : 0u);
                }
                mma_commit(bar + GB_WEMPTY + 8 * s);
                mma_commit(bar + GB_AFULL + 8 * s);
            }
            mma_commit(bar + GB_FIN);
            cg_drain(bar + GB_FIN, 0);
        }
    } else if (32 * q < a.NP) {
        // epilogue: 32-column chunks u of this warp's slices, l loaded one chunk ahead
        const bool live = p < a.NP;
        const int r = live ? p / a.Fd : 0;
        const uint16_t *row = a.ell + ((int64_t)r * a.L + a.d) * a.V;
        constexpr int CPT = CG_SLICE / 32;  // chunks per tile
        const int nu = nmine * CPT;
        auto chunk_v0 = [&](int u) {
            const int tile = (int)blockIdx.x + (u / CPT) * (int)gridDim.x;
            return tile * CG_TILE + h * CG_SLICE + (u % CPT) * 32;
        };
        const bool lsm = a.lsm != 0;
        uint32_t thr_ld = 0u;
        uint4 lnext[4];
        if (!lsm && nu > 0 && live)
            load_l32(row, chunk_v0(0), a.V - chunk_v0(0), a.vec != 0, lnext);
        for (int u = 0; u < nu; ++u) {
            const int i = u / CPT, b = i & 1, sub = u % CPT;
            const int v0 = chunk_v0(u);
            if (sub == 0) {
                if (!cg_wait(bar + GB_AFULL + 8 * b, (i >> 1) & 1, a.status))
                    ok = false;
                if (ok && lsm && !cg_wait(bar + GB_LFULL + 8 * b, (i >> 1) & 1, a.status))
                    ok = false;
                if (!__all_sync(0xFFFFFFFFu, ok ? 1 : 0)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
            }
            // the grid-wide bound published so far (loaded a chunk ahead)
            if (live) {
                if (thr_ld != 0u)
                    st.lb = fmaxf(st.lb, nextafterf(fkey_inv(thr_ld), DDT_NEG_INF));
                thr_ld = ld_relaxed_u32(a.thr + p);
            }
            uint4 lcur[4];
            if (lsm) {
                if (live) {
                    const uint4 *ls = reinterpret_cast<const uint4 *>(
                        sgen + S.l + b * S.lst + r * CG_LROW + (h * CG_SLICE + sub * 32) * 2);
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        lcur[j] = ls[j];
                }
            } else {
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    lcur[j] = lnext[j];
                if (u + 1 < nu && live)
                    load_l32(row, chunk_v0(u + 1), a.V - chunk_v0(u + 1), a.vec != 0, lnext);
            }
            uint32_t acc[32];
            const uint32_t ta = tmem + ((uint32_t)(32 * q) << 16) + b * CG_TILE + h * CG_SLICE + sub * 32;
            tmem_ld16(ta, acc);
            tmem_ld16(ta + 16, acc + 16);
            tmem_wait_ld();
            if (sub == CPT - 1) {
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(bar + GB_AEMPTY + 8 * b);
            }
            if (live)
                col_scan32(st, a.k, acc, lcur, v0, a.V - v0);
            // publish this thread's k-th value (k values of the parent reach
            // it) after its first two chunks and once more later
            if (live && (u == 0 || u == 1 || u == 7) && st.kth != DDT_NEG_INF)
                atomicMax(a.thr + p, fkey(st.kth));
        }
    } else {
        // a lane quarter with no parent: release the accumulators (and l stages) only
        for (int i = 0; i < nmine; ++i) {
            const int b = i & 1;
            if (!cg_wait(bar + GB_AFULL + 8 * b, (i >> 1) & 1, a.status))
                ok = false;
            if (ok && a.lsm && !cg_wait(bar + GB_LFULL + 8 * b, (i >> 1) & 1, a.status))
                ok = false;
            if (!__all_sync(0xFFFFFFFFu, ok ? 1 : 0)) {
                ok = false;
                break;
            }
            if (lane == 0)
                mbar_arrive(bar + GB_AEMPTY + 8 * b);
        }
    }
    pdl_trigger();
    // every role is done: the MMAs have completed and the W stages are free
    const bool all_ok = __syncthreads_and(ok ? 1 : 0) != 0;
    if (all_ok && warp < CG_EPI) {
        unsigned char *xr = sgen + S.w;  // [CG_NH - 1][128 parents] exchange records
        if (h > 0) {
            unsigned char *rec = xr + ((h - 1) * CG_MAXNP + p) * CG_XREC;
            uint64_t *keys = reinterpret_cast<uint64_t *>(rec);
#pragma unroll
            for (int j = 0; j < CG_MAXK; ++j)
                keys[j] = (st.ti[j] >= 0) ? vkey(st.tv[j], st.ti[j]) : 0ull;
            float s0, s1;
            f2unpack(st.s2, s0, s1);
            reinterpret_cast<float *>(rec + CG_MAXK * 8)[0] = st.m;
            reinterpret_cast<float *>(rec + CG_MAXK * 8)[1] = s0 + s1;
        }
        asm volatile("bar.sync 1, %0;" ::"r"(CG_EPI * 32) : "memory");
        if (h == 0 && p < a.NP) {
            uint64_t best[CG_MAXK];
#pragma unroll
            for (int j = 0; j < CG_MAXK; ++j)
                best[j] = (j < a.k && st.ti[j] >= 0) ? vkey(st.tv[j], st.ti[j]) : 0ull;
            float s0, s1;
            f2unpack(st.s2, s0, s1);
            float M = st.m, Ssum = s0 + s1;
            for (int hh = 1; hh < CG_NH; ++hh) {
                const unsigned char *rec = xr + ((hh - 1) * CG_MAXNP + p) * CG_XREC;
                const float mo = reinterpret_cast<const float *>(rec + CG_MAXK * 8)[0];
                const float so = reinterpret_cast<const float *>(rec + CG_MAXK * 8)[1];
                if (mo != DDT_NEG_INF) {
                    if (mo > M) {
                        Ssum = Ssum * ex2((M - mo) * DDT_LOG2E) + so;
                        M = mo;
                    } else {
                        Ssum += so * ex2((mo - M) * DDT_LOG2E);
                    }
                }
                const uint64_t *keys = reinterpret_cast<const uint64_t *>(rec);
#pragma unroll
                for (int j = 0; j < CG_MAXK; ++j) {
                    uint64_t x = (j < a.k) ? keys[j] : 0ull;
#pragma unroll
                    for (int t = 0; t < CG_MAXK; ++t)
                        if (t < a.k && x > best[t]) {
                            const uint64_t y = best[t];
                            best[t] = x;
                            x = y;
                        }
                }
            }
            const int64_t slot = (int64_t)p * gridDim.x + blockIdx.x;
            // the CTA's k-th value bounds the parent's k-th from below: the
            // merge then only ranks the few list entries at or above it
            if (a.k >= 1) {
                uint64_t kk = ~0ull;  // the smallest of the k (0 while fewer than k)
#pragma unroll
                for (int j = 0; j < CG_MAXK; ++j)
                    if (j < a.k)
                        kk = best[j] < kk ? best[j] : kk;
                if (kk != 0ull)
                    atomicMax(a.thr + p, (uint32_t)(kk >> 32));
            }
            a.part_ms[slot] = make_float2(M, Ssum);
#pragma unroll
            for (int j = 0; j < CG_MAXK; ++j)
                if (j < a.k)
                    a.part_top[slot * CG_MAXK + j] = best[j];
        }
    }
    __syncthreads();
    if (warp == CG_MMA)
        tmem_dealloc(tmem, CG_TMEM_COLS);
}

struct MergeArgs {
    const float2 *part_ms;
    const uint64_t *part_top;
    const int32_t *anchors;   // [R] the roots (depth 0)
    int32_t *fr_tok;          // [R, F] in: this depth's parents; out: the next depth's
    int32_t *fr_cand;         // [R, F] candidate index of each frontier parent (-1: root)
    double *fr_S;             // [R, F]
    int32_t *fr_n;            // [R]
    double *c_S;              // [R, Cmax] candidate score
    int32_t *c_meta;          // [R, Cmax, 3]: depth, parent candidate, token
    float *cand_lp;           // [R, L, F, k] (optional)
    int32_t *cand_ids;        // [R, L, F, k] (optional)
    int32_t *frontier_tok;    // [R, L, F] (optional): parents of every depth
    const uint32_t *thr;      // [Fd * R] the GEMM's per-parent bounds (value keys, 0: none)
    int R, L, d, Fd, F, k, grid, Cmax, base;
};

constexpr int CG_SLOTS = CG_GRID_MAX / 32;  // partials per lane

// one CTA per request; warp f merges frontier parent f
__global__ void __launch_bounds__(32 * CG_MAXF)
cg_merge_kernel(const MergeArgs a)
{
    pdl_trigger();
    pdl_wait();
    const int r = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    __shared__ float s_lp[CG_MAXF][CG_MAXK];
    __shared__ int s_id[CG_MAXF][CG_MAXK];
    extern __shared__ __align__(16) uint64_t s_keys[];  // [Fd][grid][kp] the parents' CTA lists
    __shared__ uint64_t s_cand[CG_MAXF][32];
    const int kp = (a.k + 1) & ~1;        // list stride: whole 16-byte pairs
    // the frontier's records, loaded ahead of their use (warp 0: the
    // candidates of this depth, one lane per parent slot and child rank)
    double fS = 0.0;
    int fcand = -1;
    if (warp == 0 && a.d > 0 && lane < a.Fd * a.k) {
        fS = a.fr_S[r * a.F + lane / a.k];
        fcand = a.fr_cand[r * a.F + lane / a.k];
    }
    const int nfr = (a.d == 0) ? 1 : a.fr_n[r];
    if (warp < a.Fd) {
        const int f = warp;
        const int p = r * a.Fd + f;
        // this parent's CTA lists (descending, kp keys each) into shared
        // memory by asynchronous copies, all in flight at once (the partials
        // of every parent slot exist: a missing parent's come from a zero
        // embedding, so nothing waits for nfr)
        uint64_t *ks = s_keys + (size_t)f * a.grid * kp;
        {
            const uint64_t *src = a.part_top + (int64_t)p * a.grid * CG_MAXK;
            const int per = kp / 2;  // 16-byte pairs per list
            for (int i = lane; i < a.grid * per; i += 32) {
                const int c = i / per, jj = i - c * per;
                cp_async_16((uint32_t)__cvta_generic_to_shared(ks + (size_t)c * kp + 2 * jj),
                            src + (int64_t)c * CG_MAXK + 2 * jj, 16u);
            }
        }
        const uint32_t bnd = a.thr[p];  // k values of the parent reach it (0: none published)
        // log-partition over the CTAs' (max, sum) pairs, all loads at once
        float M = DDT_NEG_INF, logS = 0.f;
        {
            float2 ms[CG_SLOTS];
#pragma unroll
            for (int t = 0; t < CG_SLOTS; ++t) {
                const int c = lane + 32 * t;
                ms[t] = (c < a.grid) ? a.part_ms[(int64_t)p * a.grid + c] : make_float2(DDT_NEG_INF, 0.f);
            }
#pragma unroll
            for (int t = 0; t < CG_SLOTS; ++t)
                M = fmaxf(M, ms[t].x);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1)
                M = fmaxf(M, __shfl_xor_sync(0xFFFFFFFFu, M, o));
            float S = 0.f;
#pragma unroll
            for (int t = 0; t < CG_SLOTS; ++t)
                if (ms[t].x != DDT_NEG_INF)
                    S += ms[t].y * ex2((ms[t].x - M) * DDT_LOG2E);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1)
                S += __shfl_xor_sync(0xFFFFFFFFu, S, o);
            logS = logf(S);  // lp = (z - M) - log S, in fp32 like the lists it ranks
        }
        cp_async_wait_all();
        __syncwarp();
        const bool live = f < nfr;
        // the candidates: keys at or above the bound (the k best are among
        // them); few once the GEMM's threads have published their bounds
        const uint64_t kb = (uint64_t)bnd << 32;
        int mine = 0;  // this lane's list entries at or above the bound
        if (bnd != 0u)
            for (int c = lane; c < a.grid; c += 32)
                for (int j = 0; j < a.k; ++j) {
                    const uint64_t x = ks[(size_t)c * kp + j];
                    if (x == 0ull || x < kb)
                        break;
                    ++mine;
                }
        int incl = mine;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
            if (lane >= o)
                incl += y;
        }
        const int nc = (bnd != 0u) ? __shfl_sync(0xFFFFFFFFu, incl, 31) : 1 << 30;
        if (nc <= 32 && mine > 0) {
            int at = incl - mine;
            for (int c = lane; c < a.grid; c += 32)
                for (int j = 0; j < a.k; ++j) {
                    const uint64_t x = ks[(size_t)c * kp + j];
                    if (x == 0ull || x < kb)
                        break;
                    s_cand[f][at++] = x;
                }
        }
        __syncwarp();
        if (nc >= a.k && nc <= 32) {
            // rank of each candidate among the others (keys are unique)
            const uint64_t x = (lane < nc) ? s_cand[f][lane] : 0ull;
            int rank = 0;
            for (int o = 0; o < nc; ++o)
                rank += (s_cand[f][o] > x) ? 1 : 0;
            if (live && lane < nc && rank < a.k) {
                s_lp[f][rank] = (fkey_inv((uint32_t)(x >> 32)) - M) - logS;
                s_id[f][rank] = (int)~(uint32_t)x;
            }
            if (!live && lane < a.k) {
                s_lp[f][lane] = DDT_NEG_INF;
                s_id[f][lane] = -1;
            }
        } else {
            // k rounds: every lane offers the best head of its lists, the
            // warp's best is taken and its list advances
            int pos[CG_SLOTS];
#pragma unroll
            for (int t = 0; t < CG_SLOTS; ++t)
                pos[t] = 0;
            for (int j = 0; j < a.k; ++j) {
                uint64_t cur = 0ull;
                int bt = -1;
                if (live)
#pragma unroll
                    for (int t = 0; t < CG_SLOTS; ++t) {
                        const int c = lane + 32 * t;
                        if (c < a.grid && pos[t] < a.k) {
                            const uint64_t hk = ks[(size_t)c * kp + pos[t]];
                            if (hk > cur) {
                                cur = hk;
                                bt = t;
                            }
                        }
                    }
                const uint32_t hi = (uint32_t)(cur >> 32), lo = (uint32_t)cur;
                const uint32_t mhi = __reduce_max_sync(0xFFFFFFFFu, hi);
                const uint32_t mlo = __reduce_max_sync(0xFFFFFFFFu, hi == mhi ? lo : 0u);
                const unsigned who = __ballot_sync(0xFFFFFFFFu, hi == mhi && lo == mlo && cur != 0ull);
                if (lane == 0) {
                    if (who != 0u && live) {
                        const uint64_t w = ((uint64_t)mhi << 32) | mlo;
                        s_lp[f][j] = (fkey_inv((uint32_t)(w >> 32)) - M) - logS;
                        s_id[f][j] = (int)~(uint32_t)w;
                    } else {
                        s_lp[f][j] = DDT_NEG_INF;
                        s_id[f][j] = -1;
                    }
                }
                if (who != 0u && lane == __ffs(who) - 1)
#pragma unroll
                    for (int t = 0; t < CG_SLOTS; ++t)
                        if (t == bt)
                            ++pos[t];
            }
        }
    }
    __syncthreads();
    if (warp == 0) {
        // this depth's candidates in creation order (frontier slot, child rank)
        // (every slot of the depth is written; a missing parent's slots get token -1)
        const int nd = nfr * a.k;
        double Sc = -INFINITY;
        uint64_t kc = 0ull;
        int tok = -1, par = -1, ord = a.base + lane;
        const bool have = lane < nd;
        if (have) {
            const int f = lane / a.k, j = lane % a.k;
            tok = s_id[f][j];
            Sc = fS + (double)s_lp[f][j];
            par = fcand;
            if (tok < 0)
                Sc = -INFINITY;
        }
        kc = dkey(Sc);
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
            const uint64_t ko = __shfl_sync(0xFFFFFFFFu, kc, o);
            if (have && (ko > kc || (ko == kc && o < lane)))
                ++rank;
        }
        const int nnext = nd < a.F ? nd : a.F;
        __syncwarp();
        if (have && rank < nnext) {
            a.fr_tok[r * a.F + rank] = tok;
            a.fr_cand[r * a.F + rank] = ord;
            a.fr_S[r * a.F + rank] = Sc;
        }
        if (lane == 0)
            a.fr_n[r] = nnext;
        // outputs: this depth's lists; the parents of this depth and the next
        if (a.cand_lp != nullptr)
            for (int i = lane; i < a.F * a.k; i += 32) {
                const int f = i / a.k, j = i % a.k;
                const int64_t o = (((int64_t)r * a.L + a.d) * a.F + f) * a.k + j;
                a.cand_lp[o] = (f < nfr) ? s_lp[f][j] : DDT_NEG_INF;
                a.cand_ids[o] = (f < nfr) ? s_id[f][j] : -1;
            }
        if (a.frontier_tok != nullptr) {
            if (a.d == 0)
                for (int f = lane; f < a.F; f += 32)
                    a.frontier_tok[((int64_t)r * a.L) * a.F + f] = (f == 0) ? a.anchors[r] : -1;
            if (a.d + 1 < a.L) {
                int32_t *nx = a.frontier_tok + ((int64_t)r * a.L + a.d + 1) * a.F;
                if (have && rank < nnext)
                    nx[rank] = tok;
                for (int f = nnext + lane; f < a.F; f += 32)
                    nx[f] = -1;
            }
        }
    }
}

struct PackArgs {
    const double *c_S;
    const int32_t *c_meta;
    int32_t *tree_tokens, *parents, *depths, *n_nodes;
    uint32_t *mask;
    int C, Cmax, N;
};

constexpr int CG_CMAX = 1024;

// one CTA per request: the N best candidates by (S desc, depth asc, order asc)
__global__ void __launch_bounds__(256)
cg_pack_kernel(const PackArgs a)
{
    pdl_wait();
    const int r = blockIdx.x;
    const int P = a.N + 1, W = (P + 31) >> 5;
    __shared__ uint64_t s_key[CG_CMAX];  // path scores as order-preserving integers
    __shared__ int s_dep[CG_CMAX], s_node[CG_CMAX], s_pc[CG_CMAX], s_tok[CG_CMAX];
    __shared__ int s_par[DDT_MAX_P];
    __shared__ int s_count;
    const int C = a.C;
    for (int i = threadIdx.x; i < C; i += blockDim.x) {
        const int32_t *meta = a.c_meta + ((int64_t)r * a.Cmax + i) * 3;
        s_key[i] = dkey(a.c_S[(int64_t)r * a.Cmax + i]);
        s_dep[i] = meta[0];
        s_pc[i] = meta[1];
        s_tok[i] = meta[2];
        s_node[i] = -1;
    }
    for (int i = threadIdx.x; i < P; i += blockDim.x) {
        a.parents[(int64_t)r * P + i] = -1;
        a.depths[(int64_t)r * P + i] = (i == 0) ? 0 : -1;
        s_par[i] = -1;
        if (i < a.N)
            a.tree_tokens[(int64_t)r * a.N + i] = -1;
    }
    if (threadIdx.x == 0)
        s_count = 0;
    __syncthreads();
    // rank of every real candidate; the N best become nodes 1..N
    for (int i = threadIdx.x; i < C; i += blockDim.x) {
        if (s_tok[i] < 0)
            continue;  // an empty slot
        const uint64_t ki = s_key[i];
        const int di = s_dep[i];
        int rank = 0;
        for (int o = 0; o < C; ++o) {
            if (s_tok[o] < 0)
                continue;
            const uint64_t ko = s_key[o];
            if (ko > ki || (ko == ki && (s_dep[o] < di || (s_dep[o] == di && o < i))))
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
        const int pc = s_pc[i];
        const int pn = (pc < 0) ? 0 : s_node[pc];
        a.tree_tokens[(int64_t)r * a.N + node - 1] = s_tok[i];
        a.parents[(int64_t)r * P + node] = pn;
        a.depths[(int64_t)r * P + node] = s_dep[i];
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
#pragma unroll
                    for (int w = 0; w < 4; ++w)
                        if (w == (cur >> 5))
                            words[w] |= 1u << (cur & 31);
                    cur = (cur == 0) ? -1 : s_par[cur];
                }
            }
#pragma unroll
            for (int w = 0; w < 4; ++w)
                if (w < W)
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

// the merge's staged lists: [Fd][grid][k rounded up to even] keys
size_t merge_smem(int Fd, int grid, int k)
{
    return (size_t)Fd * grid * ((k + 1) & ~1) * sizeof(uint64_t);
}

size_t gemm_smem(int H, int lrows, int srows)
{
    return (size_t)gemm_layout(H, lrows, srows).total + 1024;  // + the slack for 1024-byte alignment
}
constexpr size_t CG_SMEM_MAX = 232448;  // opt-in shared memory per block

// a launch that may start while the previous kernel of the stream finishes
// (the kernel itself waits for it with griddepcontrol.wait)
cudaLaunchConfig_t pdl_config(dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              cudaLaunchAttribute *attr, bool pdl)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cfg;
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
           cond_tree_cmax(cfg) <= CG_CMAX && cfg.B + 1 <= DDT_MAX_P && cfg.L <= DDT_MAX_L &&
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
    static size_t attr_set = 0;
    cudaError_t e;
    if (attr_set < CG_SMEM_MAX) {
        e = cudaFuncSetAttribute(cg_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)CG_SMEM_MAX);
        if (e != cudaSuccess)
            return e;
        attr_set = CG_SMEM_MAX;
    }
    static size_t mattr_set = 0;
    if (mattr_set < merge_smem(CG_MAXF, CG_GRID_MAX, CG_MAXK)) {
        e = cudaFuncSetAttribute(cg_merge_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)merge_smem(CG_MAXF, CG_GRID_MAX, CG_MAXK));
        if (e != cudaSuccess)
            return e;
        mattr_set = merge_smem(CG_MAXF, CG_GRID_MAX, CG_MAXK);
    }
    const int vec = (V % 8 == 0 && ((uintptr_t)ell & 15u) == 0) ? 1 : 0;
    // no bounds yet at any depth (the first GEMM is ordered after this as usual)
    if ((e = cudaMemsetAsync(c->cg_thr, 0, (size_t)L * CG_NP_MAX * sizeof(uint32_t), s)) != cudaSuccess)
        return e;
    const int lsm = (vec && R <= CG_LRMAX) ? 1 : 0;
    // bound seeds when their rows fit in shared memory beside the rest
    const int srows = (gemm_smem(H, lsm ? R : 0, R * K) <= CG_SMEM_MAX) ? R * K : 0;
    // the draft's own k best columns of every depth seed the bounds
    if ((e = launch_topk(c, ell, R, c->cg_seed_lp, c->cg_seed_ids, s)) != cudaSuccess)
        return e;
    int base = 0;
    cudaLaunchAttribute attr[1];
    for (int d = 0; d < L; ++d) {
        const int Fd = (d == 0) ? 1 : F;
        GemmArgs g;
        g.W = W;
        g.E = E;
        g.ell = ell;
        g.fr_tok = c->cg_fr_tok;
        g.anchors = anchors;
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
        g.k = K;
        g.vec = vec;
        g.lsm = lsm;
        g.thr = c->cg_thr + (size_t)d * CG_NP_MAX;
        g.seeds = c->cg_seed_ids;
        g.srows = srows;
        g.status = c->status;
        // the first kernel of the call waits for the stream as usual
        cudaLaunchConfig_t lc = pdl_config(dim3(grid), dim3(CG_THREADS), gemm_smem(H, lsm ? R : 0, srows), s, attr, d > 0);
        if ((e = cudaLaunchKernelEx(&lc, cg_gemm_kernel, tm, g)) != cudaSuccess)
            return e;
        MergeArgs m;
        m.part_ms = c->cg_part_ms;
        m.part_top = c->cg_part_top;
        m.anchors = anchors;
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
        m.thr = c->cg_thr + (size_t)d * CG_NP_MAX;
        lc = pdl_config(dim3(R), dim3(32 * CG_MAXF), merge_smem(Fd, grid, K), s, attr, true);
        if ((e = cudaLaunchKernelEx(&lc, cg_merge_kernel, m)) != cudaSuccess)
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
    cudaLaunchConfig_t lc = pdl_config(dim3(R), dim3(256), 0, s, attr, true);
    return cudaLaunchKernelEx(&lc, cg_pack_kernel, pk);
}
