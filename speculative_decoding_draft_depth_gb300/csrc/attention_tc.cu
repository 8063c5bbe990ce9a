// attention_tc.cu -- a4 on the 5th-generation tensor cores (tcgen05 + TMEM
// + TMA), for head dim 128.
//
// Same operation as attention.cu ("SparklingTree ...", Step 4 and the
// verification discussion; "DDTree Explained ...", sections 5 and 8): every
// tree query row attends to its request's cached context through the page
// table plus the tree positions its ancestor mask allows.
//
// One work item = (request r, KV head g, context chunk, row group):
//  * main rows: 128 query rows = 128/G positions x G heads (row = pos*G+h);
//    S = Q K^T with the rows in TMEM lanes.
//  * tail rows (at most TQ, e.g. the 33rd position of a 32-node tree): the
//    transposed products S_t^T = K Q_t^T (M = 128 tokens, N = 16) and
//    O_t^T += V^T P_t^T (M = 128 = d, N = 16); an eighth of the main MMA
//    work instead of doubling it with padding rows.
//  * K and V tiles of 128 tokens arrive by TMA, one box per 16-token page
//    run and d-half (16 rows of 128 B, 128-byte swizzle), located through the
//    item's page list staged in shared memory; two separate 2-deep rings, each
//    fed by its own loader thread: a K slot is refilled as soon as its Q K^T
//    is done, a V slot as soon as its P V is done. Q comes by TMA per item.
//  * warps 0-15 run the softmax and the epilogue, four warps per TMEM lane
//    quarter, each on 32 of the 128 columns (enough warps per scheduler to
//    hide the MUFU and TMEM latencies); warp 16 loads Q and K, warp 17 loads
//    V, warp 18 owns TMEM and issues the MMAs. Softmax runs in the base-2
//    domain with a lazily updated reference max (O and l are rescaled only
//    when a row's max grows by more than 2^8).
//  * Every mbarrier wait is bounded; on timeout the CTA raises
//    DDT_DEV_TIMEOUT in the status word and winds down.
#include <cuda.h>
#include <stdint.h>

#include "ddt_device.cuh"
#include "ddt_internal.h"
#include "tc_ptx.cuh"

namespace {

constexpr int TILE = 128;
constexpr int NSOFT = 512;               // softmax threads (16 warps)
constexpr int NTHREADS = NSOFT + 96;     // + K loader, V loader, MMA issuer
constexpr int W_KPROD = 16, W_VPROD = 17, W_MMA = 18;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t TM_S = 0;     // two S buffers: columns 0..127, 128..255
constexpr uint32_t TM_O = 256;   // O main: 128 columns
constexpr uint32_t TM_ST = 384;  // two S tail buffers: 384..399, 400..415
constexpr uint32_t TM_OT = 416;  // O tail: 416..431
constexpr float TAU = 8.0f;      // lazy-rescale threshold (log2 units)
constexpr long long WAIT_LIMIT = 4000000000LL;  // cycles (about 2 s)

// shared memory (offsets from a 1024-byte aligned base)
constexpr uint32_t SM_Q = 0;                  // 2 x 16 KB d-halves, [128 rows][128 B]
constexpr uint32_t SM_QT = 32768;             // 2 x 2 KB d-halves, [16 rows][128 B]
constexpr uint32_t SM_K = 36864;              // 2 slots x 32 KB (2 x 16 KB d-halves)
constexpr uint32_t SM_V = SM_K + 65536;       // 2 slots x 32 KB
constexpr uint32_t SM_P = SM_V + 65536;       // 32 KB: 2 x 16 KB token halves [128][64]
constexpr uint32_t SM_PT = SM_P + 32768;      // 2 x 2 KB token halves of P_t^T [16][64]
constexpr uint32_t SM_BAR = SM_PT + 4096;
constexpr uint32_t SM_TOTAL = SM_BAR + 10240;
constexpr uint32_t SM_ALLOC = SM_TOTAL + 1024;

// barrier / scalar slots inside SM_BAR
constexpr uint32_t B_QFULL = 0, B_QEMPTY = 8, B_KFULL = 16, B_KEMPTY = 32, B_VFULL = 48,
                   B_VEMPTY = 64, B_SFULL = 80, B_PFULL = 96, B_ODONE = 104, B_TMEM = 128,
                   B_ABORT = 132, B_LAST = 136,
                   B_RED = 256,    // 2 x [4 warps][16] floats: tail column max
                   B_SUM = 768,    // [4 warps][16] floats: tail sums
                   B_XMAX = 1024,  // 2 x [4 column quarters][128 rows] floats: row max
                   B_XL = 5120,    // [4 column quarters][128 rows] floats: row sum
                   B_PGK = 7168,   // page list of the K loader's item (256 ints)
                   B_PGV = 8192;   // page list of the V loader's item (256 ints)
constexpr int MAX_ITEM_PAGES = 256;

constexpr uint32_t IDESC_QK = idesc_bf16(128, 128, false, false);
constexpr uint32_t IDESC_QKT = idesc_bf16(128, 16, false, false);
constexpr uint32_t IDESC_PV = idesc_bf16(128, 128, false, true);
constexpr uint32_t IDESC_PVT = idesc_bf16(128, 16, true, false);

struct TcArgs {
    const int4 *items;
    const int32_t *meta;
    const int32_t *rg_base;
    const int32_t *block_table;
    const int32_t *ctx_lens;
    const uint32_t *mask;
    float *out;
    float *part_o;
    float2 *part_ml;
    unsigned *rg_cnt;
    int32_t *status;
    int P, Hq, Hkv, G, W, page, max_pages, RG, n_main, tail_rows;
    int64_t num_pages;
    float scale_log2;
};

struct Item {
    int idx, r, g, rg, s, t0, t1, ns, ntile_ctx, ntiles;
    bool last, has_tail;
};

DDT_DEVINL bool get_item(const TcArgs &a, int k, Item &it)
{
    const int count = a.meta[0];
    const int G = gridDim.x;
    const int base = k * G;
    if (base >= count)
        return false;
    const int pos = (k & 1) ? (G - 1 - (int)blockIdx.x) : (int)blockIdx.x;
    const int idx = base + pos;
    if (idx >= count)
        return false;
    const int4 w = a.items[idx];
    it.idx = idx;
    it.r = w.x;
    it.g = w.y & 0xFF;
    it.rg = (w.y >> 8) & 0xFF;
    it.s = w.y >> 16;
    it.t0 = w.z;
    it.t1 = w.w;
    const int ctx = min(max(a.ctx_lens[it.r], 0), a.max_pages * a.page);
    it.ns = max(1, (ctx + ATT_CHUNK - 1) / ATT_CHUNK);
    it.last = (it.s == it.ns - 1);
    it.ntile_ctx = (it.t1 > it.t0) ? (it.t1 - it.t0 + TILE - 1) / TILE : 0;
    it.ntiles = it.ntile_ctx + (it.last ? 1 : 0);
    it.has_tail = (it.rg == 0 && a.tail_rows > 0);
    return true;
}

// next item (from k + 1 on) that has tiles; false when the CTA's list ends
DDT_DEVINL bool next_item_with_tiles(const TcArgs &a, int &k, Item &it)
{
    for (++k;; ++k) {
        if (!get_item(a, k, it))
            return false;
        if (it.ntiles > 0)
            return true;
    }
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
// named barriers: 1 = warps 0-3 (tail work), 2 + q = the four warps of lane quarter q
DDT_DEVINL void tail_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }
DDT_DEVINL void quarter_bar(int q) { asm volatile("bar.sync %0, 128;" ::"r"(2 + q) : "memory"); }

// the same answer in all sixteen softmax warps: true iff every thread says true
// (keeps the softmax warps together when a bounded wait gives up)
DDT_DEVINL bool softmax_all(bool v)
{
    uint32_t r;
    asm volatile(
        "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.and.pred q, 6, 512, p;\n"
        " selp.u32 %0, 1, 0, q;\n}\n"
        : "=r"(r)
        : "r"((uint32_t)v)
        : "memory");
    return r != 0;
}

// the item's page ids covering [t0, t1), staged once per item (whole loader warp)
DDT_DEVINL void stage_pages(const TcArgs &a, const Item &it, int *s_pages, int lane)
{
    __syncwarp();  // the previous item's boxes are all issued
    if (it.t1 > it.t0) {
        const int p0 = it.t0 / a.page, np = min((it.t1 - 1) / a.page - p0 + 1, MAX_ITEM_PAGES);
        for (int i = lane; i < np; i += 32)
            s_pages[i] = __ldg(&a.block_table[(int64_t)it.r * a.max_pages + p0 + i]);
    }
    __syncwarp();
}

// the 16 TMA boxes (16 tokens x one d-half each) of one K or V tile (thread 0 of a loader)
DDT_DEVINL void load_kv_tile(const TcArgs &a, const Item &it, int j, uint32_t dst, const void *map_c,
                             const void *map_t, uint32_t fb, const int *s_pages)
{
    if (j < it.ntile_ctx) {
        const int ts = it.t0 + j * TILE;
        const int p0 = it.t0 / a.page;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int t16 = ts + 16 * u;  // 16 tokens never straddle a page (page % 16 == 0)
            int z = -16;  // wholly outside the tensor: TMA fills zeros
            if (t16 < it.t1) {
                const int pg = s_pages[t16 / a.page - p0];
                if (pg >= 0 && pg < a.num_pages)
                    z = pg * a.page + t16 % a.page;
                else
                    atomicOr(a.status, DDT_DEV_BAD_PAGE);
            }
            tma_load_3d(dst + u * 2048, map_c, 0, it.g, z, fb);
            tma_load_3d(dst + 16384 + u * 2048, map_c, 64, it.g, z, fb);
        }
    } else {
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int z = it.r * a.P + 16 * u;
            tma_load_3d(dst + u * 2048, map_t, 0, it.g, z, fb);
            tma_load_3d(dst + 16384 + u * 2048, map_t, 64, it.g, z, fb);
        }
    }
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
    const uint32_t bar = sb + SM_BAR;

    if (tid == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar + B_KFULL + 8 * i, 1);
            mbar_init(bar + B_KEMPTY + 8 * i, 1);
            mbar_init(bar + B_VFULL + 8 * i, 1);
            mbar_init(bar + B_VEMPTY + 8 * i, 1);
            mbar_init(bar + B_SFULL + 8 * i, 1);
        }
        mbar_init(bar + B_QFULL, 1);
        mbar_init(bar + B_QEMPTY, 1);
        mbar_init(bar + B_PFULL, NSOFT);
        mbar_init(bar + B_ODONE, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == W_MMA) {
        tmem_alloc(bar + B_TMEM, TMEM_COLS);
        tmem_relinquish();
    }
    // P tail rows past the tail stay zero for the whole kernel
    for (int i = tid; i < 4096 / 16; i += NTHREADS)
        reinterpret_cast<uint4 *>(sgen + SM_PT)[i] = make_uint4(0u, 0u, 0u, 0u);
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(sgen + SM_BAR + B_TMEM);
    const int PG = a.P * a.G;
    const int pos_per_main = TILE / a.G;

    if (warp == W_KPROD) {
        // ============================================================ Q and K loads
        int *s_pages = reinterpret_cast<int *>(sgen + SM_BAR + B_PGK);
        if (lane == 0) {
            prefetch_tmap(&tm_q);
            prefetch_tmap(&tm_qt);
            prefetch_tmap(&tm_k);
            prefetch_tmap(&tm_kt);
        }
        int kn = 0, q_n = 0, k = -1;
        Item it;
        bool ok = true;
        while (ok && next_item_with_tiles(a, k, it)) {
            if (q_n > 0 && !wait_bar(bar + B_QEMPTY, (q_n - 1) & 1, abort_flag, a.status))
                break;
            if (lane == 0) {
                mbar_arrive_expect_tx(bar + B_QFULL, 32768u + (it.has_tail ? 4096u : 0u));
                const int zq = it.r * a.P + it.rg * pos_per_main;
                tma_load_3d(sb + SM_Q, &tm_q, 0, it.g * a.G, zq, bar + B_QFULL);
                tma_load_3d(sb + SM_Q + 16384, &tm_q, 64, it.g * a.G, zq, bar + B_QFULL);
                if (it.has_tail) {
                    const int zt = it.r * a.P + a.n_main * pos_per_main;
                    tma_load_3d(sb + SM_QT, &tm_qt, 0, it.g * a.G, zt, bar + B_QFULL);
                    tma_load_3d(sb + SM_QT + 2048, &tm_qt, 64, it.g * a.G, zt, bar + B_QFULL);
                }
            }
            ++q_n;
            stage_pages(a, it, s_pages, lane);
            for (int j = 0; j < it.ntiles; ++j, ++kn) {
                const int sl = kn & 1;
                if (kn >= 2 &&
                    !wait_bar(bar + B_KEMPTY + 8 * sl, ((kn - 2) >> 1) & 1, abort_flag, a.status)) {
                    ok = false;
                    break;
                }
                if (lane == 0) {
                    mbar_arrive_expect_tx(bar + B_KFULL + 8 * sl, 32768u);
                    load_kv_tile(a, it, j, sb + SM_K + sl * 32768u, &tm_k, &tm_kt,
                                 bar + B_KFULL + 8 * sl, s_pages);
                }
            }
        }
    } else if (warp == W_VPROD) {
        // ============================================================ V loads
        int *s_pages = reinterpret_cast<int *>(sgen + SM_BAR + B_PGV);
        if (lane == 0) {
            prefetch_tmap(&tm_v);
            prefetch_tmap(&tm_vt);
        }
        int vn = 0, k = -1;
        Item it;
        bool ok = true;
        while (ok && next_item_with_tiles(a, k, it)) {
            stage_pages(a, it, s_pages, lane);
            for (int j = 0; j < it.ntiles; ++j, ++vn) {
                const int sl = vn & 1;
                if (vn >= 2 &&
                    !wait_bar(bar + B_VEMPTY + 8 * sl, ((vn - 2) >> 1) & 1, abort_flag, a.status)) {
                    ok = false;
                    break;
                }
                if (lane == 0) {
                    mbar_arrive_expect_tx(bar + B_VFULL + 8 * sl, 32768u);
                    load_kv_tile(a, it, j, sb + SM_V + sl * 32768u, &tm_v, &tm_vt,
                                 bar + B_VFULL + 8 * sl, s_pages);
                }
            }
        }
    } else if (warp == W_MMA) {
        // ============================================================ MMA issuer
        if (lane == 0) {
            int qk_n = 0, pv_n = 0, q_n = 0;
            // two cursors over the (item, tile) sequence: Q K^T runs one tile ahead of P V
            Item qi, pi;
            int qk_k = -1, qk_j = 0, pv_k = -1, pv_j = 0;
            bool qk_ok = next_item_with_tiles(a, qk_k, qi);
            bool pv_ok = next_item_with_tiles(a, pv_k, pi);
            // descriptors of every operand base; a K step adds its byte offset >> 4
            const uint64_t dQ = sdesc_sw128(sb + SM_Q, 16, 1024);
            const uint64_t dQT = sdesc_sw128(sb + SM_QT, 16, 1024);
            const uint64_t dP = sdesc_sw128(sb + SM_P, 16, 1024);
            const uint64_t dPT = sdesc_sw128(sb + SM_PT, 16, 1024);
            const uint64_t dK0 = sdesc_sw128(sb + SM_K, 16, 1024);
            const uint64_t dV0 = sdesc_sw128(sb + SM_V, 16384, 1024);

            auto issue_qk = [&]() -> bool {
                if (qk_j == 0 && !wait_bar(bar + B_QFULL, q_n & 1, abort_flag, a.status))
                    return false;
                const int sl = qk_n & 1;
                if (!wait_bar(bar + B_KFULL + 8 * sl, (qk_n >> 1) & 1, abort_flag, a.status))
                    return false;
                tc_fence_after();
                const uint64_t dK = dK0 + sl * (32768u >> 4);
                const uint32_t s_t = tmem + TM_S + 128u * sl;
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t off = ((kk >> 2) * 16384u + (kk & 3) * 32u) >> 4;
                    mma_bf16(s_t, dQ + off, dK + off, IDESC_QK, kk > 0 ? 1u : 0u);
                }
                if (qi.has_tail) {
                    const uint32_t st_t = tmem + TM_ST + 16u * sl;
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const uint32_t off = ((kk >> 2) * 16384u + (kk & 3) * 32u) >> 4;
                        const uint32_t offq = ((kk >> 2) * 2048u + (kk & 3) * 32u) >> 4;
                        mma_bf16(st_t, dK + off, dQT + offq, IDESC_QKT, kk > 0 ? 1u : 0u);
                    }
                }
                mma_commit(bar + B_SFULL + 8 * sl);
                mma_commit(bar + B_KEMPTY + 8 * sl);
                ++qk_n;
                if (++qk_j == qi.ntiles) {
                    mma_commit(bar + B_QEMPTY);
                    ++q_n;
                    qk_j = 0;
                    qk_ok = next_item_with_tiles(a, qk_k, qi);
                }
                return true;
            };

            bool alive = !qk_ok || issue_qk();
            while (alive && pv_ok) {
                if (qk_ok && !issue_qk())
                    break;
                const int sl = pv_n & 1;
                if (!wait_bar(bar + B_PFULL, pv_n & 1, abort_flag, a.status) ||
                    !wait_bar(bar + B_VFULL + 8 * sl, (pv_n >> 1) & 1, abort_flag, a.status))
                    break;
                tc_fence_after();
                const uint64_t dV = dV0 + sl * (32768u >> 4);
#pragma unroll
                for (int kt = 0; kt < 8; ++kt) {
                    const uint32_t acc = (pv_j > 0 || kt > 0) ? 1u : 0u;
                    const uint32_t offp = ((kt >> 2) * 16384u + (kt & 3) * 32u) >> 4;
                    mma_bf16(tmem + TM_O, dP + offp, dV + kt * (2048u >> 4), IDESC_PV, acc);
                }
                if (pi.has_tail) {
#pragma unroll
                    for (int kt = 0; kt < 8; ++kt) {
                        const uint32_t acc = (pv_j > 0 || kt > 0) ? 1u : 0u;
                        const uint32_t offp = ((kt >> 2) * 2048u + (kt & 3) * 32u) >> 4;
                        mma_bf16(tmem + TM_OT, dV + kt * (2048u >> 4), dPT + offp, IDESC_PVT, acc);
                    }
                }
                mma_commit(bar + B_VEMPTY + 8 * sl);
                mma_commit(bar + B_ODONE);
                ++pv_n;
                if (++pv_j == pi.ntiles) {
                    pv_j = 0;
                    pv_ok = next_item_with_tiles(a, pv_k, pi);
                }
            }
        }
    } else {
        // ============================================================ softmax warps
        const int qw = warp & 3, cq = warp >> 2;  // lane quarter, column quarter
        const int row = qw * 32 + lane;  // TMEM lane = main row = tail token = head-dim index
        const uint32_t lane_addr = (uint32_t)(qw * 32) << 16;
        const uint32_t col0 = 32u * cq;
        const bool tail_warp = (cq == 0);
        float *red = reinterpret_cast<float *>(sgen + SM_BAR + B_RED);
        float *sums = reinterpret_cast<float *>(sgen + SM_BAR + B_SUM);
        float *xmax = reinterpret_cast<float *>(sgen + SM_BAR + B_XMAX);
        float *xl = reinterpret_cast<float *>(sgen + SM_BAR + B_XL);
        int n = 0, od_n = 0;
        Item it;
        for (int k = 0; get_item(a, k, it); ++k) {
            if (!softmax_all(*abort_flag == 0))
                break;
            const int gr = it.rg * TILE + row;
            const bool row_ok = gr < PG;
            const int pos = gr / a.G, hl = gr % a.G;
            const int tail = it.has_tail ? a.tail_rows : 0;
            const int tail_pos0 = a.n_main * pos_per_main;
            // this thread's 32 tree columns of the mask (only the last chunk has the tree tile)
            uint32_t mk = 0u;
            uint32_t tail_bits = 0;  // bit q: this thread's tree position is visible to tail row q
            if (it.last) {
                if (row_ok && (int)col0 < a.P)
                    mk = a.mask[((int64_t)it.r * a.P + pos) * a.W + (col0 >> 5)];
                if (tail_warp && row < a.P)
                    for (int q = 0; q < tail; ++q) {
                        const uint32_t wd =
                            a.mask[((int64_t)it.r * a.P + tail_pos0 + q / a.G) * a.W + (row >> 5)];
                        tail_bits |= ((wd >> (row & 31)) & 1u) << q;
                    }
            }
            float m_used = DDT_NEG_INF, l = 0.f;  // l: this column quarter's share of the row sum
            float mt[TQ], lt[TQ];
#pragma unroll
            for (int q = 0; q < TQ; ++q) {
                mt[q] = DDT_NEG_INF;
                lt[q] = 0.f;
            }
            bool o_valid = false;

            for (int j = 0; j < it.ntiles; ++j, ++n) {
                const int sl = n & 1;
                if (!softmax_all(wait_bar(bar + B_SFULL + 8 * sl, (n >> 1) & 1, abort_flag, a.status)))
                    break;
                tc_fence_after();
                uint32_t sv[32];
                tmem_ld16(tmem + lane_addr + TM_S + 128u * sl + col0, sv);
                tmem_ld16(tmem + lane_addr + TM_S + 128u * sl + col0 + 16u, sv + 16);
                uint32_t tv[16];
                if (tail && tail_warp)
                    tmem_ld16(tmem + lane_addr + TM_ST + 16u * sl, tv);
                tmem_wait_ld();

                const bool is_ctx = j < it.ntile_ctx;
                const int ts = it.t0 + j * TILE;
                const int lim = is_ctx ? min(TILE, it.t1 - ts) : 0;
                // ---- masked max of this quarter of the row (raw scores), 4 chains
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
                // ---- tail column maxima (warps 0-3; this thread = token `row`)
                float tmx[TQ];
                if (tail && tail_warp) {
                    const bool tok_ok_ctx = is_ctx && row < lim;
#pragma unroll
                    for (int q = 0; q < TQ; ++q) {
                        const bool ok = q < tail && (is_ctx ? tok_ok_ctx : ((tail_bits >> q) & 1u) != 0u);
                        if (!ok)
                            tv[q] = __float_as_uint(DDT_NEG_INF);
                        tmx[q] = warp_max(__uint_as_float(tv[q]));
                    }
                    float *rb = red + (n & 1) * 64;
                    if (lane == 0)
#pragma unroll
                        for (int q = 0; q < TQ; ++q)
                            rb[qw * 16 + q] = tmx[q];
                    tail_bar();
#pragma unroll
                    for (int q = 0; q < TQ; ++q)
                        tmx[q] = fmaxf(fmaxf(rb[q], rb[16 + q]), fmaxf(rb[32 + q], rb[48 + q]));
                }
                quarter_bar(qw);
                const float mx = fmaxf(fmaxf(xb[row], xb[128 + row]), fmaxf(xb[256 + row], xb[384 + row]));

                // ---- lazy rescale decisions (identical in the four warps of a row)
                const float mcand = mx * a.scale_log2;
                float alpha = 1.f;
                bool need = false;
                if (mcand > m_used + TAU) {
                    alpha = ex2(m_used - mcand);  // 0 while m_used is -inf
                    m_used = mcand;
                    need = true;
                }
                float at[TQ];
                bool need_t = false;
#pragma unroll
                for (int q = 0; q < TQ; ++q) {
                    at[q] = 1.f;
                    if (tail && tail_warp && q < tail) {
                        const float mc = tmx[q] * a.scale_log2;
                        if (mc > mt[q] + TAU) {
                            at[q] = ex2(mt[q] - mc);
                            mt[q] = mc;
                            need_t = true;
                        }
                    }
                }

                // ---- P of this quarter row (registers) and the tail column, before any wait
                const bool live = (m_used != DDT_NEG_INF);
                uint32_t pw[16];
                float rs[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const float p0 = live ? ex2(__uint_as_float(sv[2 * e]) * a.scale_log2 - m_used) : 0.f;
                    const float p1 = live ? ex2(__uint_as_float(sv[2 * e + 1]) * a.scale_log2 - m_used) : 0.f;
                    rs[e & 3] += p0 + p1;
                    pw[e] = pack_bf16x2(p0, p1);
                }
                l = l * alpha + ((rs[0] + rs[1]) + (rs[2] + rs[3]));
                uint16_t pt16[TQ];
                if (tail && tail_warp) {
#pragma unroll
                    for (int q = 0; q < TQ; ++q) {
                        const float p = (q < tail && mt[q] != DDT_NEG_INF)
                                            ? ex2(__uint_as_float(tv[q]) * a.scale_log2 - mt[q])
                                            : 0.f;
                        lt[q] = lt[q] * at[q] + p;
                        pt16[q] = (uint16_t)(pack_bf16x2(p, 0.f) & 0xFFFFu);
                    }
                }

                // ---- P V of the previous tile must be done before O or P is touched
                bool ok = true;
                while (od_n < n) {
                    if (!wait_bar(bar + B_ODONE, od_n & 1, abort_flag, a.status)) {
                        ok = false;
                        break;
                    }
                    ++od_n;
                }
                if (!softmax_all(ok))
                    break;
                tc_fence_after();
                if (o_valid && need) {
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
                if (o_valid && need_t) {
                    uint32_t ov[16];
                    tmem_ld16(tmem + lane_addr + TM_OT, ov);
                    tmem_wait_ld();
#pragma unroll
                    for (int q = 0; q < TQ; ++q)
                        ov[q] = __float_as_uint(__uint_as_float(ov[q]) * at[q]);
                    tmem_st16(tmem + lane_addr + TM_OT, ov);
                }
                tmem_wait_st();

                // ---- store P (K-major, 128-byte swizzle) and the tail column P_t^T [q][token]
                unsigned char *prow = sgen + SM_P + (cq >> 1) * 16384 + row * 128;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int ch = (cq & 1) * 4 + i;
                    *reinterpret_cast<uint4 *>(prow + ((ch ^ (row & 7)) << 4)) =
                        make_uint4(pw[4 * i], pw[4 * i + 1], pw[4 * i + 2], pw[4 * i + 3]);
                }
                if (tail && tail_warp) {
                    const int th = row >> 6, tch = (row & 63) >> 3;
#pragma unroll
                    for (int q = 0; q < TQ; ++q)
                        if (q < tail)
                            *reinterpret_cast<uint16_t *>(sgen + SM_PT + th * 2048 + q * 128 +
                                                          ((tch ^ (q & 7)) << 4) + (row & 7) * 2) = pt16[q];
                }
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(bar + B_PFULL);
                o_valid = true;
            }
            if (!softmax_all(*abort_flag == 0))
                break;

            // ============================================================ epilogue
            if (it.ntiles > 0) {
                bool ok = true;
                while (od_n < n) {
                    if (!wait_bar(bar + B_ODONE, od_n & 1, abort_flag, a.status)) {
                        ok = false;
                        break;
                    }
                    ++od_n;
                }
                if (!softmax_all(ok))
                    break;
                tc_fence_after();
            }
            // full row sum from the four column quarters
            xl[cq * 128 + row] = l;
            quarter_bar(qw);
            const float lrow = (xl[row] + xl[128 + row]) + (xl[256 + row] + xl[384 + row]);
            // tail sums across the 128 tokens
            float ltot[TQ];
            if (tail && tail_warp) {
#pragma unroll
                for (int q = 0; q < TQ; ++q) {
                    const float s = warp_sum(lt[q]);
                    if (lane == 0)
                        sums[qw * 16 + q] = s;
                }
                tail_bar();
#pragma unroll
                for (int q = 0; q < TQ; ++q)
                    ltot[q] = sums[q] + sums[16 + q] + sums[32 + q] + sums[48 + q];
            }
            const bool single = (it.ns == 1);
            const int64_t item_row0 = (int64_t)it.idx * ATT_ROWS;
            {  // this quarter of the main row
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
            }
            if (tail && tail_warp) {  // tail rows (this thread = head-dim index `row`)
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
                    const int tgr = a.n_main * TILE + q;
                    const int tpos = tgr / a.G, thl = tgr % a.G;
                    if (single) {
                        const float inv = (ltot[q] > 0.f) ? 1.f / ltot[q] : 0.f;
                        a.out[(((int64_t)it.r * a.P + tpos) * a.Hq + it.g * a.G + thl) * 128 + row] =
                            __uint_as_float(ov[q]) * inv;
                    } else {
                        a.part_o[(item_row0 + TILE + q) * 128 + row] = __uint_as_float(ov[q]);
                        if (row == 0)
                            a.part_ml[item_row0 + TILE + q] = make_float2(mt[q], ltot[q]);
                    }
                }
            }
            tc_fence_before();
            if (single)
                continue;

            // ---- split item: the last of its (r, g, group) chunks combines
            __threadfence();
            softmax_all(true);
            int *s_last = reinterpret_cast<int *>(sgen + SM_BAR + B_LAST);
            const int rg_slot = (it.r * a.Hkv + it.g) * a.RG + it.rg;
            if (tid == 0)
                *s_last = (atomicAdd(&a.rg_cnt[rg_slot], 1u) == (unsigned)(it.ns - 1));
            softmax_all(true);
            const bool last_arrival = *s_last != 0;
            softmax_all(true);
            if (!last_arrival)
                continue;
            __threadfence();
            const int first = a.rg_base[rg_slot];
            const int stride = a.Hkv * a.RG;
            const int nrows = TILE + (it.has_tail ? a.tail_rows : 0);
            const int d = tid & 127;
            for (int rho = tid >> 7; rho < nrows; rho += NSOFT / 128) {
                const int gr2 = (rho < TILE) ? it.rg * TILE + rho : a.n_main * TILE + (rho - TILE);
                if (gr2 >= PG)
                    continue;
                float M = DDT_NEG_INF;
                for (int s = 0; s < it.ns; ++s)
                    M = fmaxf(M, __ldcg(&a.part_ml[(int64_t)(first + s * stride) * ATT_ROWS + rho]).x);
                const float base = (M == DDT_NEG_INF) ? 0.f : M;
                float Ls = 0.f, x = 0.f;
                for (int s = 0; s < it.ns; ++s) {
                    const int64_t ir = (int64_t)(first + s * stride) * ATT_ROWS + rho;
                    const float2 ml = __ldcg(&a.part_ml[ir]);
                    const float f = (ml.x == DDT_NEG_INF) ? 0.f : ex2(ml.x - base);
                    Ls += ml.y * f;
                    x += __ldcg(&a.part_o[ir * 128 + d]) * f;
                }
                const int i2 = gr2 / a.G, h2 = gr2 % a.G;
                a.out[(((int64_t)it.r * a.P + i2) * a.Hq + it.g * a.G + h2) * 128 + d] =
                    Ls > 0.f ? x / Ls : 0.f;
            }
            if (tid == 0)
                a.rg_cnt[rg_slot] = 0u;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == W_MMA) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
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
    return cfg.d == 128 && cfg.page_size % 16 == 0 && G >= 1 && G <= 16 && (16 % G) == 0 &&
           encode_fn() != nullptr;
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
    cudaError_t e = launch_att_plan(c, ctx_lens, R, RG, max_ctx, s);
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
    a.W = (P + 31) / 32;
    a.page = cfg.page_size;
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
