// attention_tc.cu -- a4 on the 5th-generation tensor cores (tcgen05 + TMEM
// + TMA), for head dims D = 128 and 64 (one kernel, D a template argument:
// half the K-steps of Q K^T, N = D for P V, one 64-wide box per tile row).
//
// "SparklingTree ...", Step 4 and the verification discussion; "DDTree
// Explained ...", sections 5 and 8 (ancestor-only tree mask over a GQA target
// with a custom attention mask): every tree query row attends to its
// request's cached context through the page table plus the tree positions its
// ancestor mask allows.
//
// Work split: for one KV head, every (request r, row group) pair is a run of
// tiles (its ceil(ctx_r / 128) context tiles, then the tree tile); laid end to
// end they form one sequence of T tiles, the same for every head. The CTAs
// form NG groups of Hkv, CTA c = grp * Hkv + g taking head g of tiles
// [T grp / NG, T (grp + 1) / NG): equal shares, computed by each CTA from
// ctx_lens (no plan kernel), and the Hkv CTAs of a group read the same
// tokens' cache rows at about the same time. A pair cut by a share boundary
// leaves per-CTA partials (two slots per CTA: its first and its last
// segment), combined after the main kernel by att_combine_kernel.
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
//  * K and V tiles of 128 tokens arrive by TMA in a 2-deep K ring and a
//    3-deep V ring (a V slot frees only after its P V), one box per 16-token
//    page run and d-half (16 rows of 128 B, 128-byte swizzle), issued by 8
//    lanes of the loader warp at once.
//  * warps 0-15: main-row softmax and epilogue, four warps per TMEM lane
//    quarter, each on 32 of the 128 columns; warps 16-19: tail-row softmax;
//    warp 20: walks the CTA's share and loads Q and K; warp 21: V loads; warp 22: TMEM
//    owner and MMA issuer of the main rows, which polls its barriers and issues
//    whichever of the next Q K^T and the next P V is ready; warp 23: the same
//    for the tail rows' products (a second issuing thread on another scheduler:
//    the issue of the main and the tail MMAs overlaps, and a K / V / Q slot
//    frees once both issuers have released it).
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
constexpr int W_TAIL0 = 16, W_KPROD = 20, W_VPROD = 21, W_MMA = 22, W_MMAT = 23;
constexpr int NTHREADS = 24 * 32;
constexpr int NRING = 4;                  // ring of segments handed from the walker to the other roles
constexpr int RING_CONSUMERS = 1 + 2 + 16 + 4;  // V loader, two MMA issuers, main warps, tail warps
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t TM_S = 0;     // two S buffers (P overwrites their first columns)
constexpr uint32_t TM_O = 256;   // O main: 128 columns
constexpr uint32_t TM_ST = 384;  // two S tail buffers: 384..399, 400..415
constexpr uint32_t TM_OT = 416;  // O tail: 416..431
constexpr float TAU = 8.0f;      // lazy-rescale threshold (log2 units)
constexpr long long WAIT_LIMIT = 4000000000LL;   // cycles (about 2 s)
constexpr long long DRAIN_LIMIT = 200000000LL;   // cycles, for the wind-down waits

// shared memory (offsets from a 1024-byte aligned base)
constexpr int NQ = 1;                          // Q slots
constexpr int NKS = 2;                         // K ring stages
constexpr int NVS = 3;                         // V ring stages
constexpr uint32_t QSLOT = 36864;              // main 2 x 16 KB d-halves + tail 2 x 2 KB
constexpr uint32_t SM_Q = 0;                   // NQ slots
constexpr uint32_t SM_K = SM_Q + NQ * QSLOT;   // NKS slots x 32 KB (2 x 16 KB d-halves)
constexpr uint32_t SM_V = SM_K + NKS * 32768;  // NVS slots x 32 KB
constexpr uint32_t SM_PT = SM_V + NVS * 32768; // 2 buffers x (2 x 2 KB token halves of P_t^T)
constexpr uint32_t SM_BAR = SM_PT + 8192;
constexpr uint32_t SM_TOTAL = SM_BAR + 10240;
constexpr uint32_t SM_ALLOC = SM_TOTAL + 1024;

// mbarriers and scratch inside SM_BAR
// Two-slot barriers ([2], indexed by tile parity) are the ones whose producer can
// run a full tile ahead of the consumer; a single barrier would then complete two
// phases before the consumer looks, and a parity wait cannot tell them apart.
constexpr uint32_t B_QFULL = 0, B_QEMPTY = 16,
                   B_KFULL = 32,    // [NKS <= 3]
                   B_KEMPTY = 56,   // [NKS <= 3]
                   B_VFULL = 80,    // [NVS <= 3]
                   B_VEMPTY = 104,  // [NVS <= 3]
                   B_SFULL = 128, B_STFULL = 144,
                   B_PFULL = 160,   // [2] main P of a tile in TMEM (512 arrivals)
                   B_ODONE = 176,
                   B_PTFULL = 184,  // [2] tail P of a tail tile in shared memory (128 arrivals)
                   B_OTDONE = 200, B_FINAL = 208,
                   B_RFULL = 216,   // [NRING] item ring entry written
                   B_REMPTY = 248,  // [NRING] item ring entry read by every consumer
                   B_XBAR = 280,    // [4 lane quarters][2] row-max exchange (128 arrivals)
                   B_TBAR = 344,    // [2] tail column-max exchange (128 arrivals)
                   B_LBAR = 360,    // [4 lane quarters] row-sum exchange (128 arrivals)
                   B_TLBAR = 392,   // tail-sum exchange (128 arrivals)
                   B_TMEM = 400, B_ABORT = 404,
                   B_RING = 416,    // [NRING][4] ints: segments (x = -1: end of the share)
                   B_TOTAL = 480,   // int: T, the batch's total tiles
                   B_FINALT = 488,  // the tail issuer's wind-down
                   B_DEBUG = 496,   // a barrier nothing arrives at (the armed test wait)
                   B_RED = 512,     // 2 x [4 warps][16] floats: tail column max
                   B_SUM = 1024,    // 2 x [4 warps][16] floats: tail sums
                   B_XMAX = 1536,   // 2 x [4 column quarters][128 rows] floats: row max
                   B_XL = 5632;     // 2 x [4 column quarters][128 rows] floats: row sum

constexpr uint32_t IDESC_QK = idesc_bf16(128, 128, false, false);
constexpr uint32_t IDESC_QKT = idesc_bf16(128, 16, false, false);
template <int D>
constexpr uint32_t IDESC_PV = idesc_bf16(128, D, false, true);
constexpr uint32_t IDESC_PVT = idesc_bf16(128, 16, true, false);

struct TcArgs {
    const int32_t *block_table;
    const int32_t *ctx_lens;
    const uint32_t *mask;
    float *out;
    float *part_o;
    float2 *part_ml;
    int32_t *status;
    int R, P, Hq, Hkv, G, g_shift, W, page_shift, max_pages, RG, n_main, tail_rows, max_ctx;
    int64_t num_pages;
    float scale_log2;
    long long debug_wait;  // > 0 (tests only): start with a wait that runs out after this many cycles
};

struct Item {
    int r, g, rg, ps, t0, t1, ntile_ctx, ntiles;
    bool last, has_tail, single;
};

// a segment: x = r | g << 12 | rg << 20 | last << 24 | single << 25 (single: the
// whole pair lies in this CTA's share), y = the pair's first tile in the
// batch sequence, z, w = the segment's context tokens [t0, t1)
DDT_DEVINL void decode_item(const TcArgs &a, int x, int y, int z, int w, Item &it)
{
    it.r = x & 0xFFF;
    it.g = (x >> 12) & 0xFF;
    it.rg = (x >> 20) & 0xF;
    it.last = ((x >> 24) & 1) != 0;
    it.single = ((x >> 25) & 1) != 0;
    it.ps = y;
    it.t0 = z;
    it.t1 = w;
    it.ntile_ctx = (it.t1 > it.t0) ? (it.t1 - it.t0 + TILE - 1) / TILE : 0;
    it.ntiles = it.ntile_ctx + (it.last ? 1 : 0);
    it.has_tail = (it.rg == 0 && a.tail_rows > 0);
}

// tiles of one (request r, row group) pair of a head: context tiles, then the tree tile
DDT_DEVINL int pair_tiles(const TcArgs &a, int r)
{
    const int c = min(max(__ldg(&a.ctx_lens[r]), 0), a.max_ctx);
    return (c + TILE - 1) / TILE + 1;
}
// first tile of group grp's share (of NG), and the group whose share holds tile t
DDT_DEVINL long long share_start(long long T, int grp, int NG) { return T * grp / NG; }
DDT_DEVINL int share_of(long long t, long long T, int NG) { return (int)(((t + 1) * NG + T - 1) / T - 1); }
// partial slot of the segment that group grp's CTA for head g holds of a pair
// starting at tile ps: that CTA's first segment (the pair began at or before
// its share) or its last one
DDT_DEVINL int part_slot(long long ps, long long T, int grp, int NG, int g, int Hkv)
{
    const int c = grp * Hkv + g;
    return (ps <= share_start(T, grp, NG)) ? 2 * c : 2 * c + 1;
}

// bounded mbarrier wait; false (and the abort flag raised) on timeout
DDT_DEVINL bool wait_bar_for(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                             int32_t *status, long long limit)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (*abort_flag)
            return false;
        if (clock64() - t0 > limit) {
            *abort_flag = 1;
            atomicOr(status, DDT_DEV_TIMEOUT);
            return false;
        }
    }
    return true;
}

DDT_DEVINL bool wait_bar(uint32_t bar, uint32_t parity, volatile int *abort_flag, int32_t *status)
{
    return wait_bar_for(bar, parity, abort_flag, status, WAIT_LIMIT);
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

// k-th segment of this CTA's share (false: end of the share, or abort); lane 0
// of a consumer warp frees the ring entry once every lane has the value
DDT_DEVINL bool ring_get(const TcArgs &a, uint32_t bar, const volatile int *ring, int k, int lane,
                         volatile int *abort_flag, Item &it)
{
    const int slot = k & (NRING - 1);
    if (!wait_warp(bar + B_RFULL + 8 * slot, (k / NRING) & 1, abort_flag, a.status))
        return false;
    int v0 = 0, v1 = 0, v2 = 0, v3 = 0;
    if (lane == 0) {
        v0 = ring[4 * slot];
        v1 = ring[4 * slot + 1];
        v2 = ring[4 * slot + 2];
        v3 = ring[4 * slot + 3];
        mbar_arrive(bar + B_REMPTY + 8 * slot);
    }
    v0 = __shfl_sync(0xFFFFFFFFu, v0, 0);
    if (v0 < 0)
        return false;
    v1 = __shfl_sync(0xFFFFFFFFu, v1, 0);
    v2 = __shfl_sync(0xFFFFFFFFu, v2, 0);
    v3 = __shfl_sync(0xFFFFFFFFu, v3, 0);
    decode_item(a, v0, v1, v2, v3, it);
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

// whole loader warp: the 8 * D / 64 boxes of one K or V tile into dst,
// completing on fb; z = group_row(...) of this lane, looked up before the wait
// for the slot so that the page-table load overlaps it
template <int D>
DDT_DEVINL void load_tile(const Item &it, int j, int lane, int z, uint32_t dst,
                          const void *map_c, const void *map_t, uint32_t fb)
{
    if (lane == 0)
        mbar_arrive_expect_tx(fb, 16384u * (D / 64));
    __syncwarp();
    if (lane < 8) {
        const void *m = (j < it.ntile_ctx) ? map_c : map_t;
        tma_load_3d(dst + lane * 2048, m, 0, it.g, z, fb);
        if (D == 128)
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

template <int TQ, int D>
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
            mbar_init(bar + B_QEMPTY + 8 * i, 2);  // both issuers


            mbar_init(bar + B_SFULL + 8 * i, 1);
            mbar_init(bar + B_STFULL + 8 * i, 1);
            mbar_init(bar + B_TBAR + 8 * i, NTAILT);
            mbar_init(bar + B_PFULL + 8 * i, NMAIN);
            mbar_init(bar + B_PTFULL + 8 * i, NTAILT);
        }
        for (int i = 0; i < NKS; ++i) {
            mbar_init(bar + B_KFULL + 8 * i, 1);
            mbar_init(bar + B_KEMPTY + 8 * i, 2);  // both issuers
        }
        for (int i = 0; i < NVS; ++i) {
            mbar_init(bar + B_VFULL + 8 * i, 1);
            mbar_init(bar + B_VEMPTY + 8 * i, 2);  // both issuers
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
        mbar_init(bar + B_ODONE, 1);
        mbar_init(bar + B_OTDONE, 1);
        mbar_init(bar + B_FINAL, 1);
        mbar_init(bar + B_FINALT, 1);
        mbar_init(bar + B_DEBUG, 1);
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
    if (a.debug_wait > 0) {
        // armed by a test: a bounded wait on a barrier nothing arrives at, before
        // any copy or MMA is issued; it runs out, and every role is skipped
        if (tid == 0)
            wait_bar_for(bar + B_DEBUG, 0, abort_flag, a.status, a.debug_wait);
        __syncthreads();
    }
    const bool run = (*abort_flag == 0);

    if (!run) {
        // nothing issued: straight to the wind-down
    } else if (warp == W_KPROD) {
        // ============================================================ share walk, Q and K loads
        if (lane == 0) {
            prefetch_tmap(&tm_q);
            prefetch_tmap(&tm_qt);
            prefetch_tmap(&tm_k);
            prefetch_tmap(&tm_kt);
        }
        // ---- T, and the pair holding this CTA's first tile: each lane sums the
        //      tiles of a contiguous run of requests, then one warp scan
        const int PR = a.RG;  // pairs per request, for one head
        const int NG = gridDim.x / a.Hkv, grp = blockIdx.x / a.Hkv, head = blockIdx.x % a.Hkv;
        const int per_lane = (a.R + 31) / 32;
        long long mine = 0;
        for (int i = 0; i < per_lane; ++i) {
            const int r = lane * per_lane + i;
            if (r < a.R)
                mine += (long long)pair_tiles(a, r) * PR;
        }
        long long incl = mine;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const long long y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
            if (lane >= o)
                incl += y;
        }
        const long long T = __shfl_sync(0xFFFFFFFFu, incl, 31);
        const long long lo = share_start(T, grp, NG), hi = share_start(T, grp + 1, NG);
        const long long excl = incl - mine;
        const unsigned holder = __ballot_sync(0xFFFFFFFFu, lo < hi && excl <= lo && lo < excl + mine);
        int wr = 0;             // walker state (lane 0): request, its first tile, pair, tile in pair
        long long req_off = 0;
        if (holder != 0 && lane == __ffs(holder) - 1) {
            long long acc = excl;
            for (int i = 0; i < per_lane; ++i) {
                const int r = lane * per_lane + i;
                const long long span = (long long)pair_tiles(a, r) * PR;
                if (lo < acc + span) {
                    wr = r;
                    req_off = acc;
                    break;
                }
                acc += span;
            }
        }
        if (holder != 0) {
            wr = __shfl_sync(0xFFFFFFFFu, wr, __ffs(holder) - 1);
            req_off = __shfl_sync(0xFFFFFFFFu, req_off, __ffs(holder) - 1);
        }
        if (lane == 0)
            *reinterpret_cast<volatile int *>(sgen + SM_BAR + B_TOTAL) = (int)T;
        if (blockIdx.x == 0)  // out-of-range context lengths are clamped, and reported
            for (int r = lane; r < a.R; r += 32) {
                const int c = __ldg(&a.ctx_lens[r]);
                if (c < 0 || c > a.max_ctx)
                    atomicOr(a.status, DDT_DEV_BAD_PAGE);
            }
        int wtp = (holder != 0) ? pair_tiles(a, wr) : 1;
        int wctx = (holder != 0) ? min(max(__ldg(&a.ctx_lens[wr]), 0), a.max_ctx) : 0;
        int wp = (holder != 0) ? (int)((lo - req_off) / wtp) : 0;
        int wa = (holder != 0) ? (int)((lo - req_off) % wtp) : 0;
        long long cur = (holder != 0) ? lo : hi;

        int kn = 0;
        bool ok = true;
        for (int k = 0; ok; ++k) {
            // the next segment of the share into ring slot k
            const int slot = k & (NRING - 1);
            if (k >= NRING &&
                !wait_warp(bar + B_REMPTY + 8 * slot, ((k / NRING) - 1) & 1, abort_flag, a.status))
                break;
            int ix = -1, iy = 0, iz = 0, iw = 0;
            if (cur < hi) {
                const long long ps = req_off + (long long)wp * wtp;
                const int b = (int)min((long long)wtp, wa + (hi - cur));
                const bool last = (b == wtp), single = (ps >= lo && ps + wtp <= hi);
                ix = wr | (head << 12) | (wp << 20) | ((last ? 1 : 0) << 24) | ((single ? 1 : 0) << 25);
                iy = (int)ps;
                iz = min(wa * TILE, wctx);
                iw = min(b * TILE, wctx);
                cur += b - wa;
                wa = 0;
                if (++wp == PR && cur < hi) {  // next request
                    wp = 0;
                    req_off += (long long)wtp * PR;
                    ++wr;
                    wtp = pair_tiles(a, wr);
                    wctx = min(max(__ldg(&a.ctx_lens[wr]), 0), a.max_ctx);
                }
            }
            if (lane == 0) {
                ring[4 * slot] = ix;
                ring[4 * slot + 1] = iy;
                ring[4 * slot + 2] = iz;
                ring[4 * slot + 3] = iw;
                mbar_arrive(bar + B_RFULL + 8 * slot);
            }
            if (ix < 0)
                break;
            Item it;
            decode_item(a, ix, iy, iz, iw, it);
            // Q of item k into slot k % NQ
            const int qs = k % NQ;
            if (k >= NQ && !wait_warp(bar + B_QEMPTY + 8 * qs, ((k / NQ) - 1) & 1, abort_flag, a.status))
                break;
            if (lane == 0) {
                const uint32_t qb = sb + SM_Q + qs * QSLOT, fb = bar + B_QFULL + 8 * qs;
                mbar_arrive_expect_tx(fb, (16384u + (it.has_tail ? 2048u : 0u)) * (D / 64));
                const int zq = it.r * a.P + it.rg * pos_per_main;
                tma_load_3d(qb, &tm_q, 0, it.g * a.G, zq, fb);
                if (D == 128)
                    tma_load_3d(qb + 16384, &tm_q, 64, it.g * a.G, zq, fb);
                if (it.has_tail) {
                    const int zt = it.r * a.P + a.n_main * pos_per_main;
                    tma_load_3d(qb + 32768, &tm_qt, 0, it.g * a.G, zt, fb);
                    if (D == 128)
                        tma_load_3d(qb + 34816, &tm_qt, 64, it.g * a.G, zt, fb);
                }
            }
            for (int j = 0; j < it.ntiles; ++j, ++kn) {
                const int sl = kn % NKS;
                const int z = (lane < 8) ? group_row(a, it, j, lane) : 0;
                if (kn >= NKS &&
                    !wait_warp(bar + B_KEMPTY + 8 * sl, ((kn / NKS) - 1) & 1, abort_flag, a.status)) {
                    ok = false;
                    break;
                }
                load_tile<D>(it, j, lane, z, sb + SM_K + sl * 32768u, &tm_k, &tm_kt, bar + B_KFULL + 8 * sl);
            }
        }
        // wind down: the last K tiles this warp issued have landed
        for (int m = kn - NKS; m < kn; ++m)
            if (m >= 0)
                drain_bar(bar + B_KFULL + 8 * (m % NKS), (m / NKS) & 1);
    } else if (warp == W_VPROD) {
        // ============================================================ V loads
        if (lane == 0) {
            prefetch_tmap(&tm_v);
            prefetch_tmap(&tm_vt);
        }
        int vn = 0;
        bool ok = true;
        for (int k = 0; ok; ++k) {
            Item it;
            if (!ring_get(a, bar, ring, k, lane, abort_flag, it))
                break;
            for (int j = 0; j < it.ntiles; ++j, ++vn) {
                const int sl = vn % NVS;
                const int z = (lane < 8) ? group_row(a, it, j, lane) : 0;
                if (vn >= NVS &&
                    !wait_warp(bar + B_VEMPTY + 8 * sl, ((vn / NVS) - 1) & 1, abort_flag, a.status)) {
                    ok = false;
                    break;
                }
                load_tile<D>(it, j, lane, z, sb + SM_V + sl * 32768u, &tm_v, &tm_vt, bar + B_VFULL + 8 * sl);
            }
        }
        for (int m = vn - NVS; m < vn; ++m)
            if (m >= 0)
                drain_bar(bar + B_VFULL + 8 * (m % NVS), (m / NVS) & 1);
    } else if (warp == W_MMA || warp == W_MMAT) {
        // ============================================================ MMA issuers
        // (warp W_MMA: the main rows' products; warp W_MMAT: the tail rows'.
        // Both walk every tile of the share; the tail issuer releases the
        // slots of tiles without tail rows by a plain arrival, after the slot's
        // fill it waited for, so its arrivals never run a phase ahead.)
        if (lane == 0) {
            const bool tailw = (warp == W_MMAT);
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
                        const int x = ring[4 * slot];
                        if (x < 0) {
                            qk_state = 2;
                        } else {
                            decode_item(a, x, ring[4 * slot + 1], ring[4 * slot + 2], ring[4 * slot + 3], qi);
                            qk_state = 1;
                            qk_j = 0;
                        }
                        progress = true;
                    }
                }
                if (pv_state == 0) {
                    const int slot = pv_k & (NRING - 1);
                    if (mbar_test_wait(bar + B_RFULL + 8 * slot, (pv_k / NRING) & 1)) {
                        const int x = ring[4 * slot];
                        if (x >= 0)
                            decode_item(a, x, ring[4 * slot + 1], ring[4 * slot + 2], ring[4 * slot + 3], pi);
                        mbar_arrive(bar + B_REMPTY + 8 * slot);
                        if (x < 0) {
                            pv_state = 2;
                        } else {
                            pv_state = 1;
                            pv_j = 0;
                        }
                        progress = true;
                    }
                }
                // ---- Q K^T of tile qk_n: its K has landed and S buffer qk_n & 1 is free
                //      (P V of tile qk_n - 2 has been issued)
                if (qk_state == 1 && qk_n <= pv_n + 1) {
                    const int sl = qk_n & 1, ks = qk_n % NKS, qs = qk_k % NQ;
                    if ((qk_j > 0 || mbar_test_wait(bar + B_QFULL + 8 * qs, (qk_k / NQ) & 1)) &&
                        mbar_test_wait(bar + B_KFULL + 8 * ks, (qk_n / NKS) & 1)) {
                        tc_fence_after();
                        const uint64_t dK = dK0 + ks * (32768u >> 4);
                        const uint64_t dQ = dQ0 + qs * (QSLOT >> 4);
                        const uint32_t s_t = tmem + TM_S + 128u * sl;
                        if (!tailw) {
#pragma unroll
                            for (int kk = 0; kk < D / 16; ++kk) {
                                const uint32_t off = ((kk >> 2) * 16384u + (kk & 3) * 32u) >> 4;
                                mma_bf16(s_t, dQ + off, dK + off, IDESC_QK, kk > 0 ? 1u : 0u);
                            }
                            mma_commit(bar + B_SFULL + 8 * sl);
                        } else if (qi.has_tail) {
                            const uint32_t st_t = tmem + TM_ST + 16u * (qt_n & 1);
                            const uint64_t dQT = dQ + (32768u >> 4);
#pragma unroll
                            for (int kk = 0; kk < D / 16; ++kk) {
                                const uint32_t off = ((kk >> 2) * 16384u + (kk & 3) * 32u) >> 4;
                                const uint32_t offq = ((kk >> 2) * 2048u + (kk & 3) * 32u) >> 4;
                                mma_bf16(st_t, dK + off, dQT + offq, IDESC_QKT, kk > 0 ? 1u : 0u);
                            }
                            mma_commit(bar + B_STFULL + 8 * (qt_n & 1));
                            ++qt_n;
                        }
                        // the K slot (and at the item's end the Q slot) is free once
                        // these MMAs completed; the tail issuer with nothing to do
                        // here releases it at once
                        const bool issued = !tailw || qi.has_tail;
                        if (issued)
                            mma_commit(bar + B_KEMPTY + 8 * ks);
                        else
                            mbar_arrive(bar + B_KEMPTY + 8 * ks);
                        ++qk_n;
                        if (++qk_j == qi.ntiles) {
                            if (issued)
                                mma_commit(bar + B_QEMPTY + 8 * qs);
                            else
                                mbar_arrive(bar + B_QEMPTY + 8 * qs);
                            ++qk_k;
                            qk_state = 0;
                        }
                        progress = true;
                    }
                }
                // ---- P V of tile pv_n: its P (and tail P) and V are ready
                if (pv_state == 1 && pv_n < qk_n) {
                    const int sl = pv_n & 1, vs = pv_n % NVS;
                    const bool ready =
                        tailw ? (mbar_test_wait(bar + B_VFULL + 8 * vs, (pv_n / NVS) & 1) &&
                                 (!pi.has_tail ||
                                  mbar_test_wait(bar + B_PTFULL + 8 * (pt_n & 1), (pt_n >> 1) & 1)))
                              : (mbar_test_wait(bar + B_PFULL + 8 * sl, (pv_n >> 1) & 1) &&
                                 mbar_test_wait(bar + B_VFULL + 8 * vs, (pv_n / NVS) & 1));
                    if (ready) {
                        tc_fence_after();
                        const uint64_t dV = dV0 + vs * (32768u >> 4);
                        const uint32_t p_t = tmem + TM_S + 128u * sl;
                        if (!tailw) {
#pragma unroll
                            for (int kt = 0; kt < 8; ++kt) {
                                const uint32_t acc = (pv_j > 0 || kt > 0) ? 1u : 0u;
                                mma_bf16_ts(tmem + TM_O, p_t + 32u * (kt >> 1) + 8u * (kt & 1),
                                            dV + kt * (2048u >> 4), IDESC_PV<D>, acc);
                            }
                            mma_commit(bar + B_ODONE);
                        } else if (pi.has_tail) {
                            // O_t^T has M = 128 lanes; for D = 64 the upper 64 read the
                            // stage's unused half (in bounds) and are never read back
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
                        if (!tailw || pi.has_tail)
                            mma_commit(bar + B_VEMPTY + 8 * vs);
                        else
                            mbar_arrive(bar + B_VEMPTY + 8 * vs);
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
            const uint32_t fin = bar + (tailw ? B_FINALT : B_FINAL);
            mma_commit(fin);
            drain_bar(fin, 0);
        }
        __syncwarp();
    } else if (warp < W_TAIL0) {
        // ============================================================ main-row softmax
        const int qw = warp & 3, cq = warp >> 2;  // lane quarter, column quarter
        const int row = qw * 32 + lane;           // TMEM lane = main row
        const uint32_t lane_addr = (uint32_t)(qw * 32) << 16;
        const uint32_t col0 = 32u * cq;       // this warp's S columns (tokens)
        const uint32_t ocol0 = (D / 4) * cq;  // this warp's O columns (head dim)
        float *xmax = reinterpret_cast<float *>(sgen + SM_BAR + B_XMAX);
        float *xl = reinterpret_cast<float *>(sgen + SM_BAR + B_XL);
        int n = 0;
        bool alive = true;
        for (int k = 0; alive; ++k) {
            Item it;
            if (!ring_get(a, bar, ring, k, lane, abort_flag, it))
                break;
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
                    for (int c = 0; c < D / 64; ++c) {
                        uint32_t ov[16];
                        tmem_ld16(tmem + lane_addr + TM_O + ocol0 + 16u * c, ov);
                        tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 16; ++e)
                            ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
                        tmem_st16(tmem + lane_addr + TM_O + ocol0 + 16u * c, ov);
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
            const bool single = it.single;
            const int nat = single ? 0 : part_slot(it.ps, *reinterpret_cast<volatile int *>(sgen + SM_BAR + B_TOTAL),
                                                   blockIdx.x / a.Hkv, gridDim.x / a.Hkv, it.g, a.Hkv);
            const int64_t item_row0 = (int64_t)nat * ATT_ROWS;
            const float inv = (lrow > 0.f) ? 1.f / lrow : 0.f;
            float *dst = a.out + (((int64_t)it.r * a.P + pos) * a.Hq + it.g * a.G + hl) * D + ocol0;
            float *pdst = a.part_o + (item_row0 + row) * D + ocol0;
#pragma unroll 1
            for (int c = 0; c < D / 64; ++c) {
                uint32_t ov[16];
                if (it.ntiles > 0) {
                    tmem_ld16(tmem + lane_addr + TM_O + ocol0 + 16u * c, ov);
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
        }
    } else {
        // ============================================================ tail-row softmax
        const int tq = warp - W_TAIL0;       // lane quarter
        const int row = tq * 32 + lane;      // TMEM lane = tail token (S_t^T) = head-dim index (O_t^T)
        const uint32_t lane_addr = (uint32_t)(tq * 32) << 16;
        float *red = reinterpret_cast<float *>(sgen + SM_BAR + B_RED);
        float *sums = reinterpret_cast<float *>(sgen + SM_BAR + B_SUM);
        int nt = 0, tail_items = 0;
        bool alive = true;
        for (int k = 0; alive; ++k) {
            Item it;
            if (!ring_get(a, bar, ring, k, lane, abort_flag, it))
                break;
            const int tail = it.has_tail ? a.tail_rows : 0;
            if (tail == 0)
                continue;
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
            const bool single = it.single;
            const int nat = single ? 0 : part_slot(it.ps, *reinterpret_cast<volatile int *>(sgen + SM_BAR + B_TOTAL),
                                                   blockIdx.x / a.Hkv, gridDim.x / a.Hkv, it.g, a.Hkv);
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
                if (q >= tail || row >= D)  // lanes past D hold no output (D = 64)
                    continue;
                const float ltot = sb2[q] + sb2[16 + q] + sb2[32 + q] + sb2[48 + q];
                const int tgr = a.n_main * TILE + q;
                const int tpos = tgr >> a.g_shift, thl = tgr & (a.G - 1);
                if (single) {
                    const float inv = (ltot > 0.f) ? 1.f / ltot : 0.f;
                    a.out[(((int64_t)it.r * a.P + tpos) * a.Hq + it.g * a.G + thl) * D + row] =
                        __uint_as_float(ov[q]) * inv;
                } else {
                    a.part_o[(item_row0 + TILE + q) * D + row] = __uint_as_float(ov[q]);
                    if (row == 0)
                        a.part_ml[item_row0 + TILE + q] = make_float2(mt[q], ltot);
                }
            }
            tc_fence_before();
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == W_MMA) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}


// ---------------------------------------------------------------- split combine
// After the main kernel: one CTA per (share boundary, KV head). A boundary
// that falls inside a (request, row group) run of tiles split that run; the
// CTAs of the boundaries that cut a run combine its partials (one per share
// that holds a segment of it) into the output rows, each taking an equal
// block of the rows (a short run cut once: one CTA; a long run over many
// shares, as with one request: many CTAs).
constexpr int CB_THREADS = 512;
constexpr int CB_SEGS = 16;  // segment weights held per combine pass

template <int D>
__global__ void __launch_bounds__(CB_THREADS)
att_combine_kernel(const TcArgs a, int NG)
{
    __shared__ float s_fac[CB_SEGS * ATT_ROWS];
    __shared__ float s_M[ATT_ROWS], s_inv[ATT_ROWS];
    __shared__ int s_slots[512];
    __shared__ long long s_ps, s_T;
    __shared__ int s_r, s_rg, s_go, s_ns, s_j, s_nb;
    const int tid = threadIdx.x, lane = tid & 31;
    const int bnd = blockIdx.x / a.Hkv + 1, g = blockIdx.x % a.Hkv;
    if (tid < 32) {
        // T, and the run holding the boundary's first tile
        const int per_lane = (a.R + 31) / 32;
        long long mine = 0;
        for (int i = 0; i < per_lane; ++i) {
            const int r = lane * per_lane + i;
            if (r < a.R)
                mine += (long long)pair_tiles(a, r) * a.RG;
        }
        long long incl = mine;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const long long y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
            if (lane >= o)
                incl += y;
        }
        const long long T = __shfl_sync(0xFFFFFFFFu, incl, 31);
        const long long t = share_start(T, bnd, NG), excl = incl - mine;
        const unsigned holder = __ballot_sync(0xFFFFFFFFu, t < T && excl <= t && t < excl + mine);
        if (tid == 0)
            s_go = 0;
        if (holder != 0 && lane == __ffs(holder) - 1) {
            long long acc = excl;
            for (int i = 0; i < per_lane; ++i) {
                const int r = lane * per_lane + i;
                const long long tp = pair_tiles(a, r), span = tp * a.RG;
                if (t < acc + span) {
                    const int rg = (int)((t - acc) / tp);
                    const long long ps = acc + rg * tp;
                    s_r = r;
                    s_rg = rg;
                    s_ps = ps;
                    s_T = T;
                    // cut inside the run: boundary j of the nb that cut it
                    const int c0 = share_of(ps, T, NG);
                    s_go = (t > ps) ? 1 : 0;
                    s_j = bnd - c0 - 1;
                    s_nb = share_of(ps + tp - 1, T, NG) - c0;
                    break;
                }
                acc += span;
            }
        }
    }
    __syncthreads();
    if (!s_go)
        return;
    // launched as a programmatic dependent of the main kernel: its partials are
    // read only after it has completed (the lookup above reads inputs only)
    pdl_wait();
    const long long T = s_T, ps = s_ps, pe = ps + pair_tiles(a, s_r);
    const int r = s_r, rg = s_rg;
    if (tid == 0) {
        const int c0 = share_of(ps, T, NG), c1 = share_of(pe - 1, T, NG);
        int ns = 0;
        if (T >= NG) {
            // every share holds tiles: the first segment of every share after
            // c0, and of c0 only when the run starts its share
            const bool first = (ps == share_start(T, c0, NG));
            for (int c = c0; c <= c1; ++c)
                s_slots[ns++] = 2 * (c * a.Hkv + g) + ((c == c0 && !first) ? 1 : 0);
        } else {
            for (int c = c0; c <= c1; ++c)
                if (share_start(T, c, NG) < share_start(T, c + 1, NG))
                    s_slots[ns++] = part_slot(ps, T, c, NG, g, a.Hkv);
        }
        s_ns = ns;
    }
    __syncthreads();
    const int ns = s_ns;
    const int PG = a.P * a.G;
    const int nrows = TILE + ((rg == 0 && a.tail_rows > 0) ? a.tail_rows : 0);
    // this CTA's block of the run's rows
    const int rlo = (int)((long long)s_j * nrows / s_nb), rhi = (int)((long long)(s_j + 1) * nrows / s_nb);
    const int nlr = rhi - rlo;
    // per row: the largest m and the total weight over every segment, CB_SEGS
    // segments' (m, l) loaded at once and merged into a running pair
    if (tid < nlr) {
        const int row = rlo + tid;
        float M = DDT_NEG_INF, Ls = 0.f;
        for (int b0 = 0; b0 < ns; b0 += CB_SEGS) {
            float2 ml[CB_SEGS];
#pragma unroll
            for (int s = 0; s < CB_SEGS; ++s)
                ml[s] = (b0 + s < ns) ? __ldcg(&a.part_ml[(int64_t)s_slots[b0 + s] * ATT_ROWS + row])
                                      : make_float2(DDT_NEG_INF, 0.f);
            float Mn = M;
#pragma unroll
            for (int s = 0; s < CB_SEGS; ++s)
                Mn = fmaxf(Mn, ml[s].x);
            float Lb = 0.f;
#pragma unroll
            for (int s = 0; s < CB_SEGS; ++s)
                Lb += (ml[s].x == DDT_NEG_INF) ? 0.f : ml[s].y * ex2(ml[s].x - Mn);
            Ls = ((M == DDT_NEG_INF) ? 0.f : Ls * ex2(M - Mn)) + Lb;
            M = Mn;
        }
        s_M[tid] = M;
        s_inv[tid] = (Ls > 0.f) ? 1.f / Ls : 0.f;
    }
    __syncthreads();
    for (int s0 = 0; s0 < ns; s0 += CB_SEGS) {
        const int sn = min(CB_SEGS, ns - s0);
        // per row: every segment's weight exp2(m_s - M) / L
        if (tid < nlr) {
            const int row = rlo + tid;
            const float M = s_M[tid], inv = s_inv[tid];
            float2 ml[CB_SEGS];
#pragma unroll
            for (int s = 0; s < CB_SEGS; ++s)
                ml[s] = (s < sn) ? __ldcg(&a.part_ml[(int64_t)s_slots[s0 + s] * ATT_ROWS + row])
                                 : make_float2(DDT_NEG_INF, 0.f);
#pragma unroll
            for (int s = 0; s < CB_SEGS; ++s)
                if (s < sn)
                    s_fac[s * ATT_ROWS + tid] = (ml[s].x == DDT_NEG_INF) ? 0.f : ex2(ml[s].x - M) * inv;
        }
        __syncthreads();
        // every (row, 4 columns): independent float4 loads, several in flight
        constexpr int C4 = D / 4;  // float4 per row
        constexpr int PER = (ATT_ROWS * C4 + CB_THREADS - 1) / CB_THREADS;
        float4 acc[PER];
#pragma unroll
        for (int u = 0; u < PER; ++u)
            acc[u] = make_float4(0.f, 0.f, 0.f, 0.f);
        // four segments at a time: their loads are independent and in flight together
        for (int s = 0; s < sn; s += 4) {
            const float4 *po[4];
#pragma unroll
            for (int q = 0; q < 4; ++q)
                po[q] = reinterpret_cast<const float4 *>(
                    a.part_o + (int64_t)s_slots[s0 + min(s + q, sn - 1)] * ATT_ROWS * D);
#pragma unroll
            for (int u = 0; u < PER; ++u) {
                const int e = tid + u * CB_THREADS, lr = e / C4;
                if (lr < nlr) {
                    const int off = (rlo + lr) * C4 + e % C4;
                    float4 v[4];
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        v[q] = __ldcg(po[q] + off);
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const float f = (s + q < sn) ? s_fac[(s + q) * ATT_ROWS + lr] : 0.f;
                        acc[u].x += v[q].x * f;
                        acc[u].y += v[q].y * f;
                        acc[u].z += v[q].z * f;
                        acc[u].w += v[q].w * f;
                    }
                }
            }
        }
#pragma unroll
        for (int u = 0; u < PER; ++u) {
            const int e = tid + u * CB_THREADS, lr = e / C4, d4 = (e % C4) * 4;
            if (lr >= nlr)
                continue;
            const int rho = rlo + lr;
            const int gr2 = (rho < TILE) ? rg * TILE + rho : a.n_main * TILE + (rho - TILE);
            if (gr2 >= PG)
                continue;
            const int i2 = gr2 >> a.g_shift, h2 = gr2 & (a.G - 1);
            float4 *dst = reinterpret_cast<float4 *>(
                a.out + (((int64_t)r * a.P + i2) * a.Hq + g * a.G + h2) * D + d4);
            if (s0 == 0) {
                *dst = acc[u];
            } else {
                float4 o = *dst;
                o.x += acc[u].x;
                o.y += acc[u].y;
                o.z += acc[u].z;
                o.w += acc[u].w;
                *dst = o;
            }
        }
        __syncthreads();
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

// 3-D bf16 map: (d, heads, rows) with a (64, bh, brows) box, 128-byte swizzle
bool make_map(CUtensorMap *m, const void *base, int d, int heads, int64_t rows, int bh, int brows)
{
    EncodeTiledFn f = encode_fn();
    if (f == nullptr)
        return false;
    const cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)heads, (cuuint64_t)rows};
    const cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)heads * d * 2};
    const cuuint32_t box[3] = {64, (cuuint32_t)bh, (cuuint32_t)brows};
    const cuuint32_t es[3] = {1, 1, 1};
    return f(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box,
             es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int TQ, int D>
cudaError_t launch_tq(int grid, const CUtensorMap &tq, const CUtensorMap &tqt,
                      const CUtensorMap &tk, const CUtensorMap &tv, const CUtensorMap &tkt,
                      const CUtensorMap &tvt, const TcArgs &a, cudaStream_t s)
{
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(att_tc_kernel<TQ, D>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)SM_ALLOC);
        if (e != cudaSuccess)
            return e;
        attr_set = true;
    }
    att_tc_kernel<TQ, D><<<grid, NTHREADS, SM_ALLOC, s>>>(tq, tqt, tk, tv, tkt, tvt, a);
    return cudaGetLastError();
}

}  // namespace

bool attention_tc_supported(const ddt_config &cfg)
{
    const int G = cfg.Hq / cfg.Hkv;
    const int pg = cfg.page_size;
    // (the tensor-map encoder is looked up at launch; a missing driver entry
    // point makes the launch fail with a CUDA error)
    if (!((cfg.d == 128 || cfg.d == 64) && pg >= 16 && (pg & (pg - 1)) == 0 && G >= 1 && G <= 16 &&
          (16 % G) == 0 && cfg.R_max < 4096 && cfg.Hkv < 256))
        return false;
    int nm, tail, RG;
    attention_tc_rows(cfg, &nm, &tail, &RG);
    // the batch's tile count (and every tile index) must fit in 31 bits
    const long long max_ctx = (long long)cfg.max_pages_per_req * cfg.page_size;
    const long long tmax = (long long)cfg.R_max * cfg.Hkv * RG * ((max_ctx + TILE - 1) / TILE + 1);
    return RG <= 16 && tmax < (1LL << 31);
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

cudaError_t launch_attention(ddt_ctx *c, const uint16_t *q, const uint16_t *k_tree,
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
    const int d = cfg.d;
    if (!make_map(&tq, q, d, cfg.Hq, rowsq, G, TILE / G) ||
        !make_map(&tqt, q, d, cfg.Hq, rowsq, G, 16 / G) ||
        !make_map(&tk, k_cache, d, cfg.Hkv, rowsc, 1, 16) ||
        !make_map(&tv, v_cache, d, cfg.Hkv, rowsc, 1, 16) ||
        !make_map(&tkt, k_tree, d, cfg.Hkv, rowsq, 1, 16) ||
        !make_map(&tvt, v_tree, d, cfg.Hkv, rowsq, 1, 16))
        return cudaErrorInvalidValue;
    TcArgs a;
    a.block_table = block_table;
    a.ctx_lens = ctx_lens;
    a.mask = mask;
    a.out = out;
    a.part_o = c->att_part_o;
    a.part_ml = c->att_part_ml;
    a.status = c->status;
    a.R = R;
    a.max_ctx = cfg.max_pages_per_req * cfg.page_size;
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
    a.scale_log2 = 1.4426950408889634f / sqrtf((float)d);
    a.debug_wait = c->debug_att_wait;  // one-shot test setting
    c->debug_att_wait = 0;
    // groups of Hkv CTAs (one per KV head), two partial slots per CTA
    int groups = c->num_sms / cfg.Hkv;
    if (groups < 1)
        groups = 1;
    while (groups > 1 && groups * cfg.Hkv * 2 > c->att_max_items)
        --groups;
    const int grid = groups * cfg.Hkv;
    cudaError_t e;
    if (d == 128)
        e = (tail <= 4) ? launch_tq<4, 128>(grid, tq, tqt, tk, tv, tkt, tvt, a, s)
                        : launch_tq<16, 128>(grid, tq, tqt, tk, tv, tkt, tvt, a, s);
    else
        e = (tail <= 4) ? launch_tq<4, 64>(grid, tq, tqt, tk, tv, tkt, tvt, a, s)
                        : launch_tq<16, 64>(grid, tq, tqt, tk, tv, tkt, tvt, a, s);
    if (e != cudaSuccess || groups == 1)
        return e;
    // the merge of split runs, a programmatic dependent of the main kernel (its
    // launch is staged while the main kernel's last CTAs finish)
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3((groups - 1) * cfg.Hkv);
    lc.blockDim = dim3(CB_THREADS);
    lc.dynamicSmemBytes = 0;
    lc.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    lc.attrs = at;
    lc.numAttrs = 1;
    if (d == 128)
        return cudaLaunchKernelEx(&lc, att_combine_kernel<128>, a, groups);
    return cudaLaunchKernelEx(&lc, att_combine_kernel<64>, a, groups);
}
