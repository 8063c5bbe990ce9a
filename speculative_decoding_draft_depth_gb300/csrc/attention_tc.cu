// attention_tc.cu -- a4 on the 5th-generation tensor cores (tcgen05 + TMEM
// + TMA), for head dim 128.
//
// Same operation as attention.cu ("SparklingTree ...", Step 4 and the
// verification discussion; "DDTree Explained ...", sections 5 and 8): every
// tree query row attends to its request's cached context through the page
// table plus the tree positions its ancestor mask allows.
//
// Work items = (request r, KV head g, context chunk s, row group). A plan
// kernel picks the chunk length from the batch's total work (long chunks when
// there is plenty of work, so that few (r, g) pairs are split), and sorts the
// items by size, largest first; persistent CTAs take items from a global
// counter in that order.
//
// Inside a CTA (one per SM), for one item:
//  * main rows: 128 query rows = 128/G positions x G heads (row = pos*G+h);
//    S = Q K^T with the rows in TMEM lanes (fp32), two S buffers.
//  * tail rows (at most TQ, e.g. the 33rd position of a 32-node tree): the
//    transposed products S_t^T = K Q_t^T (M = 128 tokens, N = 16) and
//    O_t^T += V^T P_t^T (M = 128 = d, N = 16): an eighth of the main MMA work
//    instead of a second 128-row tile.
//  * the softmax writes P (bf16) back over its own S columns in TMEM and the
//    P V product reads its A operand straight from TMEM, so P never touches
//    shared memory and a tile's softmax does not wait for the previous P V.
//  * K and V tiles of 128 tokens arrive by TMA in two 2-deep rings, one box
//    per 16-token page run and d-half (16 rows of 128 B, 128-byte swizzle),
//    issued by 8 lanes of the loader warp at once; Q is double-buffered.
//  * warps 0-15: main-row softmax and epilogue, four warps per TMEM lane
//    quarter, each on 32 of the 128 columns; warps 16-19: tail-row softmax;
//    warp 20: item fetch, Q and K loads; warp 21: V loads; warp 22: TMEM
//    owner and MMA issuer, which polls its barriers and issues whichever of
//    the next Q K^T and the next P V is ready.
//  * softmax in the base-2 domain with a lazily updated reference max: O and
//    l are rescaled only when a row's max grows by more than 2^8. A tile's
//    exponentials are computed against the current reference before the four
//    column-quarter maxima of the row are exchanged, and recomputed in the
//    rare case the exchange shows that the reference must move.
//  * every wait is bounded; on timeout the CTA raises DDT_DEV_TIMEOUT in the
//    status word, waits (bounded) for its own copies and MMAs in flight,
//    frees its TMEM and returns.
#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "ddt_device.cuh"
#include "ddt_internal.h"
#include "tc_ptx.cuh"

namespace {

constexpr int TILE = 128;
constexpr int NMAIN = 512;                // main-row softmax threads (warps 0-15)
constexpr int NTAILT = 128;               // tail-row softmax threads (warps 16-19)
constexpr int NSOFT = NMAIN + NTAILT;
constexpr int W_TAIL0 = 16, W_KPROD = 20, W_VPROD = 21, W_MMA = 22;
constexpr int NTHREADS = 23 * 32;
constexpr int NRING = 4;                  // fetched-item ring
constexpr int RING_CONSUMERS = 1 + 1 + 16 + 4;  // V loader, MMA, main warps, tail warps
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t TM_S = 0;     // two S buffers (P overwrites their first columns)
constexpr uint32_t TM_O = 256;   // O main: 128 columns
constexpr uint32_t TM_ST = 384;  // two S tail buffers: 384..399, 400..415
constexpr uint32_t TM_OT = 416;  // O tail: 416..431
constexpr float TAU = 8.0f;      // lazy-rescale threshold (log2 units)
constexpr long long WAIT_LIMIT = 4000000000LL;   // cycles (about 2 s)
constexpr long long DRAIN_LIMIT = 200000000LL;   // cycles, for the wind-down waits
constexpr int PLAN_BINS = 2048;

// shared memory (offsets from a 1024-byte aligned base)
constexpr uint32_t QSLOT = 36864;              // main 2 x 16 KB d-halves + tail 2 x 2 KB
constexpr uint32_t SM_Q = 0;                   // 2 slots
constexpr uint32_t SM_K = SM_Q + 2 * QSLOT;    // 2 slots x 32 KB (2 x 16 KB d-halves)
constexpr uint32_t SM_V = SM_K + 65536;        // 2 slots x 32 KB
constexpr uint32_t SM_PT = SM_V + 65536;       // 2 buffers x (2 x 2 KB token halves of P_t^T)
constexpr uint32_t SM_BAR = SM_PT + 8192;
constexpr uint32_t SM_TOTAL = SM_BAR + 10240;
constexpr uint32_t SM_ALLOC = SM_TOTAL + 1024;

// mbarriers and scratch inside SM_BAR
// Two-slot barriers ([2], indexed by tile parity) are the ones whose producer can
// run a full tile ahead of the consumer; a single barrier would then complete two
// phases before the consumer looks, and a parity wait cannot tell them apart.
constexpr uint32_t B_QFULL = 0, B_QEMPTY = 16, B_KFULL = 32, B_KEMPTY = 48, B_VFULL = 64,
                   B_VEMPTY = 80, B_SFULL = 96, B_STFULL = 112,
                   B_PFULL = 128,   // [2] main P of a tile in TMEM (512 arrivals)
                   B_ODONE = 144,
                   B_PTFULL = 152,  // [2] tail P of a tail tile in shared memory (128 arrivals)
                   B_OTDONE = 168, B_FINAL = 176,
                   B_RFULL = 184,   // [NRING] item ring entry written
                   B_REMPTY = 216,  // [NRING] item ring entry read by every consumer
                   B_XBAR = 248,    // [4 lane quarters][2] row-max exchange (128 arrivals)
                   B_TBAR = 312,    // [2] tail column-max exchange (128 arrivals)
                   B_LBAR = 328,    // [4 lane quarters] row-sum exchange (128 arrivals)
                   B_TLBAR = 360,   // tail-sum exchange (128 arrivals)
                   B_IBAR = 368,    // all softmax threads, split-item combine (640 arrivals)
                   B_TMEM = 376, B_ABORT = 380, B_LAST = 384,
                   B_RING = 400,    // [NRING] ints: item indices
                   B_RED = 512,     // 2 x [4 warps][16] floats: tail column max
                   B_SUM = 1024,    // 2 x [4 warps][16] floats: tail sums
                   B_XMAX = 1536,   // 2 x [4 column quarters][128 rows] floats: row max
                   B_XL = 5632;     // 2 x [4 column quarters][128 rows] floats: row sum

constexpr uint32_t IDESC_QK = idesc_bf16(128, 128, false, false);
constexpr uint32_t IDESC_QKT = idesc_bf16(128, 16, false, false);
constexpr uint32_t IDESC_PV = idesc_bf16(128, 128, false, true);
constexpr uint32_t IDESC_PVT = idesc_bf16(128, 16, true, false);

struct TcArgs {
    const int4 *items;
    int32_t *meta;             // [0] item count, [1] work counter
    const int32_t *rg_base;
    const int32_t *block_table;
    const int32_t *ctx_lens;
    const uint32_t *mask;
    float *out;
    float *part_o;
    float2 *part_ml;
    unsigned *rg_cnt;
    int32_t *status;
    int P, Hq, Hkv, G, g_shift, W, page_shift, max_pages, RG, n_main, tail_rows;
    int64_t num_pages;
    float scale_log2;
};

struct Item {
    int r, g, rg, s, ns, t0, t1, ntile_ctx, ntiles;
    bool last, has_tail;
};

DDT_DEVINL void decode_item(const TcArgs &a, int idx, Item &it)
{
    const int4 w = a.items[idx];
    it.r = w.x & 0xFFF;
    it.ns = w.x >> 12;
    it.g = w.y & 0xFF;
    it.rg = (w.y >> 8) & 0xFF;
    it.s = w.y >> 16;
    it.t0 = w.z;
    it.t1 = w.w;
    it.last = (it.s == it.ns - 1);
    it.ntile_ctx = (it.t1 > it.t0) ? (it.t1 - it.t0 + TILE - 1) / TILE : 0;
    it.ntiles = it.ntile_ctx + (it.last ? 1 : 0);
    it.has_tail = (it.rg == 0 && a.tail_rows > 0);
}

// bounded mbarrier wait; false (and the abort flag raised) on timeout
DDT_DEVINL bool wait_bar(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                         int32_t *status)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (*abort_flag)
            return false;
        if (clock64() - t0 > WAIT_LIMIT) {
            *abort_flag = 1;
            atomicOr(status, DDT_DEV_TIMEOUT);
            return false;
        }
    }
    return true;
}

// wind-down wait for work this thread itself started (ignores the abort flag)
DDT_DEVINL void drain_bar(uint32_t bar, uint32_t parity)
{
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity))
        if (clock64() - t0 > DRAIN_LIMIT)
            return;
}

// the same, with one verdict for the whole (converged) warp, so that the warp
// stays together for the warp-collective TMEM accesses that follow
DDT_DEVINL bool wait_warp(uint32_t bar, uint32_t parity, volatile int *abort_flag, int32_t *status)
{
    return __all_sync(0xFFFFFFFFu, wait_bar(bar, parity, abort_flag, status));
}

// group exchange point: every member arrives once per phase, then waits for the phase
DDT_DEVINL bool gsync(uint32_t bar, uint32_t parity, volatile int *abort_flag, int32_t *status)
{
    mbar_arrive(bar);
    return wait_warp(bar, parity, abort_flag, status);
}

// k-th fetched item index of this CTA (-1: no more); lane 0 of a consumer
// warp frees the ring entry once every lane has the value
DDT_DEVINL bool ring_get(uint32_t bar, const volatile int *ring, int k, int lane, bool release,
                         volatile int *abort_flag, int32_t *status, int &idx)
{
    const int slot = k & (NRING - 1);
    if (!wait_warp(bar + B_RFULL + 8 * slot, (k / NRING) & 1, abort_flag, status))
        return false;
    int v = 0;
    if (lane == 0) {
        v = ring[slot];
        if (release)
            mbar_arrive(bar + B_REMPTY + 8 * slot);
    }
    idx = __shfl_sync(0xFFFFFFFFu, v, 0);
    return true;
}

DDT_DEVINL float warp_max(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    return v;
}
DDT_DEVINL float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}

// row of the 128-row K or V cache tensor for 16-token group u of tile j
// (lanes 0-7 of a loader warp, one group each); -16 = wholly out of range,
// which the TMA fills with zeros
DDT_DEVINL int group_row(const TcArgs &a, const Item &it, int j, int u)
{
    if (j < it.ntile_ctx) {
        const int t16 = it.t0 + j * TILE + 16 * u;  // never straddles a page (page % 16 == 0)
        if (t16 >= it.t1)
            return -16;
        const int pg = __ldg(&a.block_table[(int64_t)it.r * a.max_pages + (t16 >> a.page_shift)]);
        if (pg < 0 || pg >= a.num_pages) {
            atomicOr(a.status, DDT_DEV_BAD_PAGE);
            return -16;
        }
        return (pg << a.page_shift) + (t16 & ((1 << a.page_shift) - 1));
    }
    return it.r * a.P + 16 * u;  // the tree tile: rows of k_tree / v_tree
}

// whole loader warp: the 16 boxes of one K or V tile into dst, completing on fb
DDT_DEVINL void load_tile(const TcArgs &a, const Item &it, int j, int lane, uint32_t dst,
                          const void *map_c, const void *map_t, uint32_t fb)
{
    const int z = (lane < 8) ? group_row(a, it, j, lane) : 0;
    if (lane == 0)
        mbar_arrive_expect_tx(fb, 32768u);
    __syncwarp();
    if (lane < 8) {
        const void *m = (j < it.ntile_ctx) ? map_c : map_t;
        tma_load_3d(dst + lane * 2048, m, 0, it.g, z, fb);
        tma_load_3d(dst + 16384 + lane * 2048, m, 64, it.g, z, fb);
    }
}

// exponentials of this thread's 32 scores against reference m (log2 units),
// packed to bf16 pairs; returns their sum
DDT_DEVINL float exps32(const uint32_t *sv, float scale, float m, uint32_t *pw)
{
    float r0 = 0.f, r1 = 0.f, r2 = 0.f, r3 = 0.f;
#pragma unroll
    for (int e = 0; e < 16; e += 2) {
        const float p0 = ex2(fmaf(__uint_as_float(sv[2 * e]), scale, -m));
        const float p1 = ex2(fmaf(__uint_as_float(sv[2 * e + 1]), scale, -m));
        const float p2 = ex2(fmaf(__uint_as_float(sv[2 * e + 2]), scale, -m));
        const float p3 = ex2(fmaf(__uint_as_float(sv[2 * e + 3]), scale, -m));
        pw[e] = pack_bf16x2(p0, p1);
        pw[e + 1] = pack_bf16x2(p2, p3);
        r0 += p0;
        r1 += p1;
        r2 += p2;
        r3 += p3;
    }
    return (r0 + r1) + (r2 + r3);
}

// a finished split item: all softmax threads publish their partials, the CTA that
// arrives last for its (r, g, row group) combines every chunk into the output
DDT_DEVINL void split_combine(const TcArgs &a, const Item &it, unsigned char *sgen, uint32_t bar,
                              int &ib, volatile int *abort_flag, int tid, int PG)
{
    __threadfence();
    if (!gsync(bar + B_IBAR, ib++ & 1, abort_flag, a.status))
        return;
    int *s_last = reinterpret_cast<int *>(sgen + SM_BAR + B_LAST);
    const int rg_slot = (it.r * a.Hkv + it.g) * a.RG + it.rg;
    if (tid == 0)
        *s_last = (atomicAdd(&a.rg_cnt[rg_slot], 1u) == (unsigned)(it.ns - 1));
    if (!gsync(bar + B_IBAR, ib++ & 1, abort_flag, a.status))
        return;
    if (*reinterpret_cast<volatile int *>(s_last) == 0)
        return;
    __threadfence();
    const int first = a.rg_base[rg_slot];
    const int stride = a.Hkv * a.RG;
    const int nrows = TILE + (it.has_tail ? a.tail_rows : 0);
    // pass 1: per row, the common reference and the total weight
    float2 *fac = reinterpret_cast<float2 *>(sgen + SM_BAR + B_XMAX);  // [nrows] (M, 1/L)
    if (tid < nrows) {
        float M = DDT_NEG_INF;
        for (int s = 0; s < it.ns; ++s)
            M = fmaxf(M, __ldcg(&a.part_ml[(int64_t)(first + s * stride) * ATT_ROWS + tid]).x);
        const float base = (M == DDT_NEG_INF) ? 0.f : M;
        float Ls = 0.f;
        for (int s = 0; s < it.ns; ++s) {
            const float2 ml = __ldcg(&a.part_ml[(int64_t)(first + s * stride) * ATT_ROWS + tid]);
            Ls += (ml.x == DDT_NEG_INF) ? 0.f : ml.y * ex2(ml.x - base);
        }
        fac[tid] = make_float2(base, Ls > 0.f ? 1.f / Ls : 0.f);
    }
    if (!gsync(bar + B_IBAR, ib++ & 1, abort_flag, a.status))
        return;
    // pass 2: every (row, d) element
    const int d = tid & 127;
    for (int rho = tid >> 7; rho < nrows; rho += NSOFT / 128) {
        const int gr2 = (rho < TILE) ? it.rg * TILE + rho : a.n_main * TILE + (rho - TILE);
        if (gr2 >= PG)
            continue;
        const float2 f = fac[rho];
        float x = 0.f;
        for (int s = 0; s < it.ns; ++s) {
            const int64_t ir = (int64_t)(first + s * stride) * ATT_ROWS + rho;
            const float m = __ldcg(&a.part_ml[ir]).x;
            if (m != DDT_NEG_INF)
                x += __ldcg(&a.part_o[ir * 128 + d]) * ex2(m - f.x);
        }
        const int i2 = gr2 >> a.g_shift, h2 = gr2 & (a.G - 1);
        a.out[(((int64_t)it.r * a.P + i2) * a.Hq + it.g * a.G + h2) * 128 + d] = x * f.y;
    }
    if (tid == 0)
        a.rg_cnt[rg_slot] = 0u;
    // the fac scratch is reused by the next item's row-max exchange
    gsync(bar + B_IBAR, ib++ & 1, abort_flag, a.status);
}

template <int TQ>
__global__ void __launch_bounds__(NTHREADS, 1)
att_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_qt,
              const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
              const __grid_constant__ CUtensorMap tm_kt, const __grid_constant__ CUtensorMap tm_vt,
              const TcArgs a)
{
    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw = (uint32_t)__cvta_generic_to_shared(smem_raw);
    const uint32_t sb = (raw + 1023u) & ~1023u;  // 1024-aligned base (shared address)
    unsigned char *sgen = smem_raw + (sb - raw);  // same base, generic pointer
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sgen + SM_BAR + B_ABORT);
    volatile int *ring = reinterpret_cast<volatile int *>(sgen + SM_BAR + B_RING);
    const uint32_t bar = sb + SM_BAR;

    if (tid == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar + B_QFULL + 8 * i, 1);
            mbar_init(bar + B_QEMPTY + 8 * i, 1);
            mbar_init(bar + B_KFULL + 8 * i, 1);
            mbar_init(bar + B_KEMPTY + 8 * i, 1);
            mbar_init(bar + B_VFULL + 8 * i, 1);
            mbar_init(bar + B_VEMPTY + 8 * i, 1);
            mbar_init(bar + B_SFULL + 8 * i, 1);
            mbar_init(bar + B_STFULL + 8 * i, 1);
            mbar_init(bar + B_TBAR + 8 * i, NTAILT);
            mbar_init(bar + B_PFULL + 8 * i, NMAIN);
            mbar_init(bar + B_PTFULL + 8 * i, NTAILT);
        }
        for (int i = 0; i < NRING; ++i) {
            mbar_init(bar + B_RFULL + 8 * i, 1);
            mbar_init(bar + B_REMPTY + 8 * i, RING_CONSUMERS);
        }
        for (int i = 0; i < 8; ++i)
            mbar_init(bar + B_XBAR + 8 * i, 128);
        for (int i = 0; i < 4; ++i)
            mbar_init(bar + B_LBAR + 8 * i, 128);
        mbar_init(bar + B_TLBAR, NTAILT);
        mbar_init(bar + B_IBAR, NSOFT);
        mbar_init(bar + B_ODONE, 1);
        mbar_init(bar + B_OTDONE, 1);
        mbar_init(bar + B_FINAL, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == W_MMA) {
        tmem_alloc(bar + B_TMEM, TMEM_COLS);
        tmem_relinquish();
    }
    // P tail rows past the tail stay zero for the whole kernel
    for (int i = tid; i < 8192 / 16; i += NTHREADS)
        reinterpret_cast<uint4 *>(sgen + SM_PT)[i] = make_uint4(0u, 0u, 0u, 0u);
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(sgen + SM_BAR + B_TMEM);
    const int PG = a.P * a.G;
    const int pos_per_main = TILE >> a.g_shift;

    if (warp == W_KPROD) {
        // ============================================================ fetch, Q and K loads
        if (lane == 0) {
            prefetch_tmap(&tm_q);
            prefetch_tmap(&tm_qt);
            prefetch_tmap(&tm_k);
            prefetch_tmap(&tm_kt);
        }
        const int count = a.meta[0];
        int kn = 0;
        bool ok = true;
        for (int k = 0; ok; ++k) {
            // fetch the next item into ring slot k
            const int slot = k & (NRING - 1);
            if (k >= NRING &&
                !wait_warp(bar + B_REMPTY + 8 * slot, ((k / NRING) - 1) & 1, abort_flag, a.status))
                break;
            int idx = 0;
            if (lane == 0) {
                idx = atomicAdd(&a.meta[1], 1);
                if (idx >= count)
                    idx = -1;
                ring[slot] = idx;
                mbar_arrive(bar + B_RFULL + 8 * slot);
            }
            idx = __shfl_sync(0xFFFFFFFFu, idx, 0);
            if (idx < 0)
                break;
            Item it;
            decode_item(a, idx, it);
            // Q of item k into slot k & 1
            const int qs = k & 1;
            if (k >= 2 && !wait_warp(bar + B_QEMPTY + 8 * qs, ((k >> 1) - 1) & 1, abort_flag, a.status))
                break;
            if (lane == 0) {
                const uint32_t qb = sb + SM_Q + qs * QSLOT, fb = bar + B_QFULL + 8 * qs;
                mbar_arrive_expect_tx(fb, 32768u + (it.has_tail ? 4096u : 0u));
                const int zq = it.r * a.P + it.rg * pos_per_main;
                tma_load_3d(qb, &tm_q, 0, it.g * a.G, zq, fb);
                tma_load_3d(qb + 16384, &tm_q, 64, it.g * a.G, zq, fb);
                if (it.has_tail) {
                    const int zt = it.r * a.P + a.n_main * pos_per_main;
                    tma_load_3d(qb + 32768, &tm_qt, 0, it.g * a.G, zt, fb);
                    tma_load_3d(qb + 34816, &tm_qt, 64, it.g * a.G, zt, fb);
                }
            }
            for (int j = 0; j < it.ntiles; ++j, ++kn) {
                const int sl = kn & 1;
                if (kn >= 2 &&
                    !wait_warp(bar + B_KEMPTY + 8 * sl, ((kn - 2) >> 1) & 1, abort_flag, a.status)) {
                    ok = false;
                    break;
                }
                load_tile(a, it, j, lane, sb + SM_K + sl * 32768u, &tm_k, &tm_kt, bar + B_KFULL + 8 * sl);
            }
        }
        // wind down: the last K tiles this warp issued have landed
        for (int m = kn - 2; m < kn; ++m)
            if (m >= 0)
                drain_bar(bar + B_KFULL + 8 * (m & 1), (m >> 1) & 1);
    } else if (warp == W_VPROD) {
        // ============================================================ V loads
        if (lane == 0) {
            prefetch_tmap(&tm_v);
            prefetch_tmap(&tm_vt);
        }
        int vn = 0;
        bool ok = true;
        for (int k = 0; ok; ++k) {
            int idx;
            if (!ring_get(bar, ring, k, lane, true, abort_flag, a.status, idx) || idx < 0)
                break;
            Item it;
            decode_item(a, idx, it);
            for (int j = 0; j < it.ntiles; ++j, ++vn) {
                const int sl = vn & 1;
                if (vn >= 2 &&
                    !wait_warp(bar + B_VEMPTY + 8 * sl, ((vn - 2) >> 1) & 1, abort_flag, a.status)) {
                    ok = false;
                    break;
                }
                load_tile(a, it, j, lane, sb + SM_V + sl * 32768u, &tm_v, &tm_vt, bar + B_VFULL + 8 * sl);
            }
        }
        for (int m = vn - 2; m < vn; ++m)
            if (m >= 0)
                drain_bar(bar + B_VFULL + 8 * (m & 1), (m >> 1) & 1);
    } else if (warp == W_MMA) {
        // ============================================================ MMA issuer
        if (lane == 0) {
            const uint64_t dK0 = sdesc_sw128(sb + SM_K, 16, 1024);
            const uint64_t dV0 = sdesc_sw128(sb + SM_V, 16384, 1024);
            const uint64_t dQ0 = sdesc_sw128(sb + SM_Q, 16, 1024);
            const uint64_t dPT0 = sdesc_sw128(sb + SM_PT, 16, 1024);
            // Q K^T cursor
            int qk_k = 0, qk_j = 0, qk_n = 0, qt_n = 0;
            int qk_state = 0;  // 0: needs an item, 1: has one, 2: no more items
            Item qi;
            // P V cursor
            int pv_k = 0, pv_j = 0, pv_n = 0, pt_n = 0;
            int pv_state = 0;
            Item pi;
            long long idle_since = clock64();
            bool failed = false;
            while (pv_state != 2) {
                bool progress = false;
                if (*abort_flag) {
                    failed = true;
                    break;
                }
                // ---- next item for either cursor, once its ring entry is there
                if (qk_state == 0) {
                    const int slot = qk_k & (NRING - 1);
                    if (mbar_test_wait(bar + B_RFULL + 8 * slot, (qk_k / NRING) & 1)) {
                        const int idx = ring[slot];
                        if (idx < 0) {
                            qk_state = 2;
                        } else {
                            decode_item(a, idx, qi);
                            qk_state = 1;
                            qk_j = 0;
                        }
                        progress = true;
                    }
                }
                if (pv_state == 0) {
                    const int slot = pv_k & (NRING - 1);
                    if (mbar_test_wait(bar + B_RFULL + 8 * slot, (pv_k / NRING) & 1)) {
                        const int idx = ring[slot];
                        mbar_arrive(bar + B_REMPTY + 8 * slot);
                        if (idx < 0) {
                            pv_state = 2;
                        } else {
                            decode_item(a, idx, pi);
                            pv_state = 1;
                            pv_j = 0;
                        }
                        progress = true;
                    }
                }
                // ---- Q K^T of tile qk_n: its K has landed and S buffer qk_n & 1 is free
                //      (P V of tile qk_n - 2 has been issued)
                if (qk_state == 1 && qk_n <= pv_n + 1) {
                    const int sl = qk_n & 1, qs = qk_k & 1;
                    if ((qk_j > 0 || mbar_test_wait(bar + B_QFULL + 8 * qs, (qk_k >> 1) & 1)) &&
                        mbar_test_wait(bar + B_KFULL + 8 * sl, (qk_n >> 1) & 1)) {
                        tc_fence_after();
                        const uint64_t dK = dK0 + sl * (32768u >> 4);
                        const uint64_t dQ = dQ0 + qs * (QSLOT >> 4);
                        const uint32_t s_t = tmem + TM_S + 128u * sl;
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk) {
                            const uint32_t off = ((kk >> 2) * 16384u + (kk & 3) * 32u) >> 4;
                            mma_bf16(s_t, dQ + off, dK + off, IDESC_QK, kk > 0 ? 1u : 0u);
                        }
                        mma_commit(bar + B_SFULL + 8 * sl);
                        if (qi.has_tail) {
                            const uint32_t st_t = tmem + TM_ST + 16u * (qt_n & 1);
                            const uint64_t dQT = dQ + (32768u >> 4);
#pragma unroll
                            for (int kk = 0; kk < 8; ++kk) {
                                const uint32_t off = ((kk >> 2) * 16384u + (kk & 3) * 32u) >> 4;
                                const uint32_t offq = ((kk >> 2) * 2048u + (kk & 3) * 32u) >> 4;
                                mma_bf16(st_t, dK + off, dQT + offq, IDESC_QKT, kk > 0 ? 1u : 0u);
                            }
                            mma_commit(bar + B_STFULL + 8 * (qt_n & 1));
                            ++qt_n;
                        }
                        mma_commit(bar + B_KEMPTY + 8 * sl);
                        ++qk_n;
                        if (++qk_j == qi.ntiles) {
                            mma_commit(bar + B_QEMPTY + 8 * qs);
                            ++qk_k;
                            qk_state = 0;
                        }
                        progress = true;
                    }
                }
                // ---- P V of tile pv_n: its P (and tail P) and V are ready
                if (pv_state == 1 && pv_n < qk_n) {
                    const int sl = pv_n & 1;
                    if (mbar_test_wait(bar + B_PFULL + 8 * sl, (pv_n >> 1) & 1) &&
                        mbar_test_wait(bar + B_VFULL + 8 * sl, (pv_n >> 1) & 1) &&
                        (!pi.has_tail ||
                         mbar_test_wait(bar + B_PTFULL + 8 * (pt_n & 1), (pt_n >> 1) & 1))) {
                        tc_fence_after();
                        const uint64_t dV = dV0 + sl * (32768u >> 4);
                        const uint32_t p_t = tmem + TM_S + 128u * sl;
#pragma unroll
                        for (int kt = 0; kt < 8; ++kt) {
                            const uint32_t acc = (pv_j > 0 || kt > 0) ? 1u : 0u;
                            mma_bf16_ts(tmem + TM_O, p_t + 32u * (kt >> 1) + 8u * (kt & 1),
                                        dV + kt * (2048u >> 4), IDESC_PV, acc);
                        }
                        mma_commit(bar + B_ODONE);
                        if (pi.has_tail) {
                            const uint64_t dPT = dPT0 + (pt_n & 1) * (4096u >> 4);
#pragma unroll
                            for (int kt = 0; kt < 8; ++kt) {
                                const uint32_t acc = (pv_j > 0 || kt > 0) ? 1u : 0u;
                                const uint32_t offp = ((kt >> 2) * 2048u + (kt & 3) * 32u) >> 4;
                                mma_bf16(tmem + TM_OT, dV + kt * (2048u >> 4), dPT + offp, IDESC_PVT, acc);
                            }
                            mma_commit(bar + B_OTDONE);
                            ++pt_n;
                        }
                        mma_commit(bar + B_VEMPTY + 8 * sl);
                        ++pv_n;
                        if (++pv_j == pi.ntiles) {
                            ++pv_k;
                            pv_state = 0;
                        }
                        progress = true;
                    }
                }
                if (progress) {
                    idle_since = clock64();
                } else if (clock64() - idle_since > WAIT_LIMIT) {
                    *abort_flag = 1;
                    atomicOr(a.status, DDT_DEV_TIMEOUT);
                    failed = true;
                    break;
                }
            }
            (void)failed;
            // wind down: every MMA issued here has completed
            mma_commit(bar + B_FINAL);
            drain_bar(bar + B_FINAL, 0);
        }
        __syncwarp();
    } else if (warp < W_TAIL0) {
        // ============================================================ main-row softmax
        const int qw = warp & 3, cq = warp >> 2;  // lane quarter, column quarter
        const int row = qw * 32 + lane;           // TMEM lane = main row
        const uint32_t lane_addr = (uint32_t)(qw * 32) << 16;
        const uint32_t col0 = 32u * cq;
        float *xmax = reinterpret_cast<float *>(sgen + SM_BAR + B_XMAX);
        float *xl = reinterpret_cast<float *>(sgen + SM_BAR + B_XL);
        int n = 0, ib = 0;
        bool alive = true;
        for (int k = 0; alive; ++k) {
            int idx;
            if (!ring_get(bar, ring, k, lane, true, abort_flag, a.status, idx) || idx < 0)
                break;
            Item it;
            decode_item(a, idx, it);
            const int gr = it.rg * TILE + row;
            const bool row_ok = gr < PG;
            const int pos = gr >> a.g_shift, hl = gr & (a.G - 1);
            uint32_t mk = 0u;  // this thread's 32 tree columns of the ancestor mask
            if (it.last && row_ok && (int)col0 < a.P)
                mk = __ldg(&a.mask[((int64_t)it.r * a.P + pos) * a.W + (col0 >> 5)]);
            float m_used = DDT_NEG_INF, l = 0.f;  // l: this column quarter's share of the row sum

            for (int j = 0; j < it.ntiles; ++j, ++n) {
                const int sl = n & 1;
                if (!wait_warp(bar + B_SFULL + 8 * sl, (n >> 1) & 1, abort_flag, a.status)) {
                    alive = false;
                    break;
                }
                tc_fence_after();
                const uint32_t s_addr = tmem + lane_addr + TM_S + 128u * sl + col0;
                uint32_t sv[32];
                tmem_ld16(s_addr, sv);
                tmem_ld16(s_addr + 16u, sv + 16);
                tmem_wait_ld();

                const bool is_ctx = j < it.ntile_ctx;
                const int lim = is_ctx ? min(TILE, it.t1 - (it.t0 + j * TILE)) : 0;
                // ---- masked max of this quarter of the row (raw scores)
                float m4[4] = {DDT_NEG_INF, DDT_NEG_INF, DDT_NEG_INF, DDT_NEG_INF};
                if (is_ctx && lim == TILE) {
#pragma unroll
                    for (int c = 0; c < 32; ++c)
                        m4[c & 3] = fmaxf(m4[c & 3], __uint_as_float(sv[c]));
                } else {
#pragma unroll
                    for (int c = 0; c < 32; ++c) {
                        const int cc = (int)col0 + c;
                        const bool ok = is_ctx ? (cc < lim) : (cc < a.P && ((mk >> c) & 1u));
                        if (!ok)
                            sv[c] = __float_as_uint(DDT_NEG_INF);
                        m4[c & 3] = fmaxf(m4[c & 3], __uint_as_float(sv[c]));
                    }
                }
                float *xb = xmax + (n & 1) * 512;
                xb[cq * 128 + row] = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
                const uint32_t xbar = bar + B_XBAR + 8 * (qw * 2 + (n & 1));
                mbar_arrive(xbar);

                // ---- exponentials against the current reference, while the other
                //      quarters of the row publish their maxima
                uint32_t pw[16];
                float rs = 0.f;
                bool have = false;
                if (m_used != DDT_NEG_INF) {
                    rs = exps32(sv, a.scale_log2, m_used, pw);
                    have = true;
                }
                if (!wait_warp(xbar, (n >> 1) & 1, abort_flag, a.status)) {
                    alive = false;
                    break;
                }
                const float mx = fmaxf(fmaxf(xb[row], xb[128 + row]), fmaxf(xb[256 + row], xb[384 + row]));
                const float mcand = mx * a.scale_log2;
                float alpha = 1.f;
                const bool need = mcand > m_used + TAU;  // identical in the four warps of a row
                if (need) {
                    alpha = ex2(m_used - mcand);  // 0 while m_used is -inf
                    m_used = mcand;
                    have = false;
                }
                if (!have) {
                    if (m_used != DDT_NEG_INF) {
                        rs = exps32(sv, a.scale_log2, m_used, pw);
                    } else {
#pragma unroll
                        for (int e = 0; e < 16; ++e)
                            pw[e] = 0u;
                        rs = 0.f;
                    }
                }
                l = l * alpha + rs;

                // ---- O rescale (rare): P V of the previous tile must have completed
                if (__any_sync(0xFFFFFFFFu, need && j > 0)) {
                    if (!wait_warp(bar + B_ODONE, (n - 1) & 1, abort_flag, a.status)) {
                        alive = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll 1
                    for (int c = 0; c < 2; ++c) {
                        uint32_t ov[16];
                        tmem_ld16(tmem + lane_addr + TM_O + col0 + 16u * c, ov);
                        tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 16; ++e)
                            ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
                        tmem_st16(tmem + lane_addr + TM_O + col0 + 16u * c, ov);
                    }
                }
                // ---- P over this warp's own S columns
                tmem_st16(s_addr, pw);
                tmem_wait_st();
                // the item's last tile: P V of the tile before it has completed (keeps the
                // epilogue's wait on the last P V unambiguous)
                if (j == it.ntiles - 1 && j > 0 &&
                    !wait_warp(bar + B_ODONE, (n - 1) & 1, abort_flag, a.status)) {
                    alive = false;
                    break;
                }
                tc_fence_before();
                mbar_arrive(bar + B_PFULL + 8 * sl);
            }
            if (!alive)
                break;

            // ---- epilogue: full row sum, O row quarter -> output or partial
            if (it.ntiles > 0 && !wait_warp(bar + B_ODONE, (n - 1) & 1, abort_flag, a.status))
                break;
            tc_fence_after();
            float *xlb = xl + (k & 1) * 512;
            xlb[cq * 128 + row] = l;
            if (!gsync(bar + B_LBAR + 8 * qw, k & 1, abort_flag, a.status))
                break;
            const float lrow = (xlb[row] + xlb[128 + row]) + (xlb[256 + row] + xlb[384 + row]);
            const bool single = (it.ns == 1);
            const int nat = single ? 0 : __ldg(&a.rg_base[(it.r * a.Hkv + it.g) * a.RG + it.rg]) +
                                             it.s * a.Hkv * a.RG;
            const int64_t item_row0 = (int64_t)nat * ATT_ROWS;
            const float inv = (lrow > 0.f) ? 1.f / lrow : 0.f;
            float *dst = a.out + (((int64_t)it.r * a.P + pos) * a.Hq + it.g * a.G + hl) * 128 + col0;
            float *pdst = a.part_o + (item_row0 + row) * 128 + col0;
#pragma unroll 1
            for (int c = 0; c < 2; ++c) {
                uint32_t ov[16];
                if (it.ntiles > 0) {
                    tmem_ld16(tmem + lane_addr + TM_O + col0 + 16u * c, ov);
                    tmem_wait_ld();
                } else {
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        ov[e] = 0u;
                }
                if (single) {
                    if (row_ok) {
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            reinterpret_cast<float4 *>(dst + 16 * c)[e] = make_float4(
                                __uint_as_float(ov[4 * e]) * inv, __uint_as_float(ov[4 * e + 1]) * inv,
                                __uint_as_float(ov[4 * e + 2]) * inv, __uint_as_float(ov[4 * e + 3]) * inv);
                    }
                } else {
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        reinterpret_cast<uint4 *>(pdst + 16 * c)[e] =
                            make_uint4(ov[4 * e], ov[4 * e + 1], ov[4 * e + 2], ov[4 * e + 3]);
                }
            }
            if (!single && cq == 0)
                a.part_ml[item_row0 + row] = make_float2(m_used, lrow);
            tc_fence_before();
            if (!single)
                split_combine(a, it, sgen, bar, ib, abort_flag, tid, PG);
        }
    } else {
        // ============================================================ tail-row softmax
        const int tq = warp - W_TAIL0;       // lane quarter
        const int row = tq * 32 + lane;      // TMEM lane = tail token (S_t^T) = head-dim index (O_t^T)
        const int ttid = tid - NMAIN;        // 0..127
        const uint32_t lane_addr = (uint32_t)(tq * 32) << 16;
        float *red = reinterpret_cast<float *>(sgen + SM_BAR + B_RED);
        float *sums = reinterpret_cast<float *>(sgen + SM_BAR + B_SUM);
        int nt = 0, tail_items = 0, ib = 0;
        bool alive = true;
        for (int k = 0; alive; ++k) {
            int idx;
            if (!ring_get(bar, ring, k, lane, true, abort_flag, a.status, idx) || idx < 0)
                break;
            Item it;
            decode_item(a, idx, it);
            const int tail = it.has_tail ? a.tail_rows : 0;
            if (tail == 0) {
                if (it.ns != 1)
                    split_combine(a, it, sgen, bar, ib, abort_flag, ttid + NMAIN, PG);
                continue;
            }
            const int tail_pos0 = a.n_main * pos_per_main;
            uint32_t tail_bits = 0;  // bit q: this thread's tree position is visible to tail row q
            if (it.last && row < a.P)
                for (int q = 0; q < tail; ++q) {
                    const uint32_t wd =
                        __ldg(&a.mask[((int64_t)it.r * a.P + tail_pos0 + (q >> a.g_shift)) * a.W + (row >> 5)]);
                    tail_bits |= ((wd >> (row & 31)) & 1u) << q;
                }
            float mt[TQ], lt[TQ];
#pragma unroll
            for (int q = 0; q < TQ; ++q) {
                mt[q] = DDT_NEG_INF;
                lt[q] = 0.f;
            }
            for (int j = 0; j < it.ntiles; ++j, ++nt) {
                if (!wait_warp(bar + B_STFULL + 8 * (nt & 1), (nt >> 1) & 1, abort_flag, a.status)) {
                    alive = false;
                    break;
                }
                tc_fence_after();
                uint32_t tv[16];
                tmem_ld16(tmem + lane_addr + TM_ST + 16u * (nt & 1), tv);
                tmem_wait_ld();
                const bool is_ctx = j < it.ntile_ctx;
                const int lim = is_ctx ? min(TILE, it.t1 - (it.t0 + j * TILE)) : 0;
                const bool tok_ok_ctx = is_ctx && row < lim;
                float *rb = red + (nt & 1) * 64;
#pragma unroll
                for (int q = 0; q < TQ; ++q) {
                    const bool ok = q < tail && (is_ctx ? tok_ok_ctx : ((tail_bits >> q) & 1u) != 0u);
                    if (!ok)
                        tv[q] = __float_as_uint(DDT_NEG_INF);
                    const float tm = warp_max(__uint_as_float(tv[q]));
                    if (lane == 0)
                        rb[tq * 16 + q] = tm;
                }
                if (!gsync(bar + B_TBAR + 8 * (nt & 1), (nt >> 1) & 1, abort_flag, a.status)) {
                    alive = false;
                    break;
                }
                float at[TQ];
                bool need_t = false;
                uint32_t pt16[TQ];
#pragma unroll
                for (int q = 0; q < TQ; ++q) {
                    at[q] = 1.f;
                    const float cm = fmaxf(fmaxf(rb[q], rb[16 + q]), fmaxf(rb[32 + q], rb[48 + q]));
                    if (q < tail) {
                        const float mc = cm * a.scale_log2;
                        if (mc > mt[q] + TAU) {
                            at[q] = ex2(mt[q] - mc);
                            mt[q] = mc;
                            need_t = true;
                        }
                    }
                    const float p = (q < tail && mt[q] != DDT_NEG_INF)
                                        ? ex2(fmaf(__uint_as_float(tv[q]), a.scale_log2, -mt[q]))
                                        : 0.f;
                    lt[q] = lt[q] * at[q] + p;
                    pt16[q] = pack_bf16x2(p, 0.f) & 0xFFFFu;
                }
                // O_t rescale (rare): P V of the previous tail tile must have completed
                if (__any_sync(0xFFFFFFFFu, need_t && j > 0)) {
                    if (!wait_warp(bar + B_OTDONE, (nt - 1) & 1, abort_flag, a.status)) {
                        alive = false;
                        break;
                    }
                    tc_fence_after();
                    uint32_t ov[16];
                    tmem_ld16(tmem + lane_addr + TM_OT, ov);
                    tmem_wait_ld();
#pragma unroll
                    for (int q = 0; q < TQ; ++q)
                        ov[q] = __float_as_uint(__uint_as_float(ov[q]) * at[q]);
                    tmem_st16(tmem + lane_addr + TM_OT, ov);
                    tmem_wait_st();
                }
                // P_t^T (K-major: row q, this thread's token column) into buffer nt & 1
                unsigned char *ptb = sgen + SM_PT + (nt & 1) * 4096;
                const int th = row >> 6, tch = (row & 63) >> 3;
#pragma unroll
                for (int q = 0; q < TQ; ++q)
                    if (q < tail)
                        *reinterpret_cast<uint16_t *>(ptb + th * 2048 + q * 128 + ((tch ^ (q & 7)) << 4) +
                                                      (row & 7) * 2) = (uint16_t)pt16[q];
                fence_proxy_async_smem();
                if (j == it.ntiles - 1 && j > 0 &&
                    !wait_warp(bar + B_OTDONE, (nt - 1) & 1, abort_flag, a.status)) {
                    alive = false;
                    break;
                }
                tc_fence_before();
                mbar_arrive(bar + B_PTFULL + 8 * (nt & 1));
            }
            if (!alive)
                break;
            // ---- tail epilogue
            if (it.ntiles > 0 && !wait_warp(bar + B_OTDONE, (nt - 1) & 1, abort_flag, a.status))
                break;
            tc_fence_after();
            float *sb2 = sums + (tail_items & 1) * 64;
#pragma unroll
            for (int q = 0; q < TQ; ++q) {
                const float sm = warp_sum(lt[q]);
                if (lane == 0)
                    sb2[tq * 16 + q] = sm;
            }
            if (!gsync(bar + B_TLBAR, tail_items & 1, abort_flag, a.status))
                break;
            ++tail_items;
            const bool single = (it.ns == 1);
            const int nat = single ? 0 : __ldg(&a.rg_base[(it.r * a.Hkv + it.g) * a.RG + it.rg]) +
                                             it.s * a.Hkv * a.RG;
            const int64_t item_row0 = (int64_t)nat * ATT_ROWS;
            uint32_t ov[16];
            if (it.ntiles > 0) {
                tmem_ld16(tmem + lane_addr + TM_OT, ov);
                tmem_wait_ld();
            } else {
#pragma unroll
                for (int q = 0; q < 16; ++q)
                    ov[q] = 0u;
            }
#pragma unroll
            for (int q = 0; q < TQ; ++q) {
                if (q >= tail)
                    continue;
                const float ltot = sb2[q] + sb2[16 + q] + sb2[32 + q] + sb2[48 + q];
                const int tgr = a.n_main * TILE + q;
                const int tpos = tgr >> a.g_shift, thl = tgr & (a.G - 1);
                if (single) {
                    const float inv = (ltot > 0.f) ? 1.f / ltot : 0.f;
                    a.out[(((int64_t)it.r * a.P + tpos) * a.Hq + it.g * a.G + thl) * 128 + row] =
                        __uint_as_float(ov[q]) * inv;
                } else {
                    a.part_o[(item_row0 + TILE + q) * 128 + row] = __uint_as_float(ov[q]);
                    if (row == 0)
                        a.part_ml[item_row0 + TILE + q] = make_float2(mt[q], ltot);
                }
            }
            tc_fence_before();
            if (!single)
                split_combine(a, it, sgen, bar, ib, abort_flag, ttid + NMAIN, PG);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == W_MMA) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

// block-wide exclusive scan of arr[0..n) in place (blockDim.x == 1024); returns the total
__device__ int block_excl_scan(int *arr, int n, int *s_wsum, int *s_carry)
{
    const int tid = threadIdx.x, nth = blockDim.x;
    if (tid == 0)
        *s_carry = 0;
    __syncthreads();
    for (int base = 0; base < n; base += nth) {
        const int i = base + tid;
        const int v = (i < n) ? arr[i] : 0;
        int x = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xFFFFFFFFu, x, o);
            if ((tid & 31) >= o)
                x += y;
        }
        if ((tid & 31) == 31)
            s_wsum[tid >> 5] = x;
        __syncthreads();
        if (tid < 32) {
            int w = (tid < nth / 32) ? s_wsum[tid] : 0;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xFFFFFFFFu, w, o);
                if (tid >= o)
                    w += y;
            }
            s_wsum[tid] = w;  // inclusive prefix of the warp totals
        }
        __syncthreads();
        const int excl = *s_carry + x - v + ((tid >> 5) > 0 ? s_wsum[(tid >> 5) - 1] : 0);
        if (i < n)
            arr[i] = excl;
        __syncthreads();
        if (tid == 0)
            *s_carry += s_wsum[nth / 32 - 1];
        __syncthreads();
    }
    return *s_carry;
}

// ---------------------------------------------------------------- plan
// One CTA. Chooses the chunk length C (tiles) from the batch's total work,
// cuts every (r, g, row group) context into ns = ceil(tiles / C) near-equal
// chunks of whole tiles (the last one also carries the tree tile), and writes
// the items sorted by size, largest first (order within a size is free).
// meta[0] = item count, meta[1] = 0 (the work counter).
__global__ void att_tc_plan_kernel(const int32_t *__restrict__ ctx_lens, int R, int Hkv, int RG,
                                   int max_ctx, int cap, int num_sms, int4 *__restrict__ items,
                                   int32_t *__restrict__ rg_base, int32_t *__restrict__ meta,
                                   int32_t *__restrict__ status)
{
    extern __shared__ int sp[];
    int *s_ctx = sp, *s_ns = sp + R, *s_len = sp + 2 * R, *s_off = sp + 3 * R;
    int *s_hist = sp + 4 * R;                 // PLAN_BINS
    __shared__ long long s_total;
    __shared__ int s_wsum[32];
    __shared__ int s_count;
    const int tid = threadIdx.x, nth = blockDim.x;
    const int per_req = Hkv * RG;
    if (tid == 0)
        s_total = 0;
    for (int i = tid; i < PLAN_BINS; i += nth)
        s_hist[i] = 0;
    __syncthreads();
    long long mine = 0;
    for (int r = tid; r < R; r += nth) {
        int c = ctx_lens[r];
        if (c < 0 || c > max_ctx) {
            set_status(status, DDT_DEV_BAD_PAGE);
            c = c < 0 ? 0 : max_ctx;
        }
        s_ctx[r] = c;
        mine += (long long)((c + TILE - 1) / TILE + 1) * per_req;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        mine += __shfl_xor_sync(0xFFFFFFFFu, mine, o);
    if ((tid & 31) == 0 && mine != 0)
        atomicAdd((unsigned long long *)&s_total, (unsigned long long)mine);
    __syncthreads();
    const long long T = s_total;
    const long long npairs = (long long)R * per_req;
    long long C = (T + 2LL * num_sms - 1) / (2LL * num_sms);
    if (C < 4)
        C = 4;
    const long long room = (long long)cap - npairs;
    if (room > 0) {
        const long long cmin = (T + room - 1) / room;
        if (C < cmin)
            C = cmin;
    } else {
        C = 1LL << 30;  // one chunk per pair
    }
    for (int r = tid; r < R; r += nth) {
        const int tiles = (s_ctx[r] + TILE - 1) / TILE;
        const int ns = tiles > 0 ? (int)((tiles + C - 1) / C) : 1;
        s_ns[r] = ns;
        s_len[r] = tiles > 0 ? (tiles + ns - 1) / ns : 0;
    }
    __syncthreads();
    // item offsets: exclusive scan of ns * per_req over r
    for (int r = tid; r < R; r += nth)
        s_off[r] = s_ns[r] * per_req;
    __syncthreads();
    const int n_items = block_excl_scan(s_off, R, s_wsum, &s_count);
    // sizes -> histogram (largest first)
    for (int i0 = 0; i0 < n_items; i0 += nth) {
        const int i = i0 + tid;
        int bin = -1;
        if (i < n_items) {
            int lo = 0, hi = R - 1;  // last r with s_off[r] <= i
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (s_off[mid] <= i)
                    lo = mid;
                else
                    hi = mid - 1;
            }
            const int r = lo, rem = i - s_off[r], s = rem / per_req;
            const int ctx = s_ctx[r], len = s_len[r] * TILE;
            const int t0 = min(ctx, s * len), t1 = min(ctx, (s + 1) * len);
            const int size = (t1 - t0 + TILE - 1) / TILE + (s == s_ns[r] - 1 ? 1 : 0);
            bin = PLAN_BINS - 1 - min(size, PLAN_BINS - 1);
        }
        const unsigned same = __match_any_sync(0xFFFFFFFFu, bin);
        if (bin >= 0 && (tid & 31) == __ffs(same) - 1)
            atomicAdd(&s_hist[bin], __popc(same));
    }
    __syncthreads();
    block_excl_scan(s_hist, PLAN_BINS, s_wsum, &s_count);
    for (int i0 = 0; i0 < n_items; i0 += nth) {
        const int i = i0 + tid;
        int bin = -1, r = 0, s = 0, g = 0, rg = 0, ns = 0, t0 = 0, t1 = 0;
        if (i < n_items) {
            int lo = 0, hi = R - 1;
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (s_off[mid] <= i)
                    lo = mid;
                else
                    hi = mid - 1;
            }
            r = lo;
            const int rem = i - s_off[r];
            s = rem / per_req;
            g = (rem / RG) % Hkv;
            rg = rem % RG;
            const int ctx = s_ctx[r], len = s_len[r] * TILE;
            ns = s_ns[r];
            t0 = min(ctx, s * len);
            t1 = min(ctx, (s + 1) * len);
            const int size = (t1 - t0 + TILE - 1) / TILE + (s == ns - 1 ? 1 : 0);
            bin = PLAN_BINS - 1 - min(size, PLAN_BINS - 1);
        }
        const unsigned same = __match_any_sync(0xFFFFFFFFu, bin);
        const int leader = __ffs(same) - 1;
        int base = 0;
        if (bin >= 0 && (tid & 31) == leader)
            base = atomicAdd(&s_hist[bin], __popc(same));
        base = __shfl_sync(0xFFFFFFFFu, base, leader);
        if (bin >= 0) {
            const int at = base + __popc(same & ((1u << (tid & 31)) - 1u));
            items[at] = make_int4(r | (ns << 12), g | (rg << 8) | (s << 16), t0, t1);
            if (s == 0)
                rg_base[((int64_t)r * Hkv + g) * RG + rg] = s_off[r] + g * RG + rg;
        }
    }
    if (tid == 0) {
        meta[0] = n_items;
        meta[1] = 0;
    }
}

// ------------------------------------------------------------------ host side
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

// 3-D bf16 map: (d = 128, heads, rows) with a (64, bh, brows) box, 128-byte swizzle
bool make_map(CUtensorMap *m, const void *base, int heads, int64_t rows, int bh, int brows)
{
    EncodeTiledFn f = encode_fn();
    if (f == nullptr)
        return false;
    const cuuint64_t dims[3] = {128, (cuuint64_t)heads, (cuuint64_t)rows};
    const cuuint64_t strides[2] = {256, (cuuint64_t)heads * 256};
    const cuuint32_t box[3] = {64, (cuuint32_t)bh, (cuuint32_t)brows};
    const cuuint32_t es[3] = {1, 1, 1};
    return f(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box,
             es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int TQ>
cudaError_t launch_tq(const ddt_ctx *c, const CUtensorMap &tq, const CUtensorMap &tqt,
                      const CUtensorMap &tk, const CUtensorMap &tv, const CUtensorMap &tkt,
                      const CUtensorMap &tvt, const TcArgs &a, cudaStream_t s)
{
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(att_tc_kernel<TQ>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)SM_ALLOC);
        if (e != cudaSuccess)
            return e;
        attr_set = true;
    }
    att_tc_kernel<TQ><<<c->num_sms, NTHREADS, SM_ALLOC, s>>>(tq, tqt, tk, tv, tkt, tvt, a);
    return cudaGetLastError();
}

}  // namespace

bool attention_tc_supported(const ddt_config &cfg)
{
    const int G = cfg.Hq / cfg.Hkv;
    const int pg = cfg.page_size;
    return cfg.d == 128 && pg >= 16 && (pg & (pg - 1)) == 0 && G >= 1 && G <= 16 &&
           (16 % G) == 0 && cfg.R_max < 4096 && encode_fn() != nullptr;
}

void attention_tc_rows(const ddt_config &cfg, int *n_main, int *tail_rows, int *rowgroups)
{
    const int PG = (cfg.B + 1) * (cfg.Hq / cfg.Hkv);
    int nm = PG / TILE, tail = PG - nm * TILE;
    if (tail > 16) {
        ++nm;
        tail = 0;
    }
    if (nm == 0) {
        nm = 1;
        tail = 0;
    }
    *n_main = nm;
    *tail_rows = tail;
    *rowgroups = nm;
}

cudaError_t launch_attention_tc(const ddt_ctx *c, const uint16_t *q, const uint16_t *k_tree,
                                const uint16_t *v_tree, const uint16_t *k_cache,
                                const uint16_t *v_cache, const int32_t *block_table,
                                const int32_t *ctx_lens, const uint32_t *mask, int R,
                                float *out, cudaStream_t s)
{
    const ddt_config &cfg = c->cfg;
    const int P = cfg.B + 1, G = cfg.Hq / cfg.Hkv;
    int n_main, tail, RG;
    attention_tc_rows(cfg, &n_main, &tail, &RG);
    CUtensorMap tq, tqt, tk, tv, tkt, tvt;
    const int64_t rowsq = (int64_t)R * P, rowsc = cfg.num_pages * cfg.page_size;
    if (!make_map(&tq, q, cfg.Hq, rowsq, G, TILE / G) ||
        !make_map(&tqt, q, cfg.Hq, rowsq, G, 16 / G) ||
        !make_map(&tk, k_cache, cfg.Hkv, rowsc, 1, 16) ||
        !make_map(&tv, v_cache, cfg.Hkv, rowsc, 1, 16) ||
        !make_map(&tkt, k_tree, cfg.Hkv, rowsq, 1, 16) ||
        !make_map(&tvt, v_tree, cfg.Hkv, rowsq, 1, 16))
        return cudaErrorInvalidValue;
    const int max_ctx = cfg.max_pages_per_req * cfg.page_size;
    const size_t plan_smem = (size_t)(4 * R + PLAN_BINS) * sizeof(int);
    att_tc_plan_kernel<<<1, 1024, plan_smem, s>>>(ctx_lens, R, cfg.Hkv, RG, max_ctx,
                                                  c->att_max_items, c->num_sms, c->att_items,
                                                  c->att_rg_base, c->att_meta, c->status);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return e;
    TcArgs a;
    a.items = c->att_items;
    a.meta = c->att_meta;
    a.rg_base = c->att_rg_base;
    a.block_table = block_table;
    a.ctx_lens = ctx_lens;
    a.mask = mask;
    a.out = out;
    a.part_o = c->att_part_o;
    a.part_ml = c->att_part_ml;
    a.rg_cnt = c->att_rg_cnt;
    a.status = c->status;
    a.P = P;
    a.Hq = cfg.Hq;
    a.Hkv = cfg.Hkv;
    a.G = G;
    a.g_shift = 0;
    while ((1 << a.g_shift) < G)
        ++a.g_shift;
    a.W = (P + 31) / 32;
    a.page_shift = 0;
    while ((1 << a.page_shift) < cfg.page_size)
        ++a.page_shift;
    a.max_pages = cfg.max_pages_per_req;
    a.RG = RG;
    a.n_main = n_main;
    a.tail_rows = tail;
    a.num_pages = cfg.num_pages;
    a.scale_log2 = 1.4426950408889634f / sqrtf(128.0f);
    if (tail <= 4)
        return launch_tq<4>(c, tq, tqt, tk, tv, tkt, tvt, a, s);
    return launch_tq<16>(c, tq, tqt, tk, tv, tkt, tvt, a, s);
}
