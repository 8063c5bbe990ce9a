// sched.cu -- the hardware-aware prefix scheduler ("DSpark Speculative
// Decoding Explained: Block Drafting and Confidence Checks", sections
// "Survival probability" and "Picking the budget"; the DSpark post's
// "Hardware aware prefix scheduler").
//
// conf [R, L] holds the chance that guess k of request r survives given that
// the earlier ones did; the survival of slot (r, k) is their running product.
// Every slot of every request is ranked by survival (descending; equal
// survivals by position, then request, ascending). Verifying the n best
// slots is expected to commit R + (their survivals' sum) tokens at a step
// cost of cost[n] ms; the scheduler keeps the n with the most tokens per ms
// (the smallest n on ties; an n with a cost that is not positive is never
// kept). Survival cannot rise along a block, so the kept slots are a prefix
// of every request's block.
//
// Up to 8192 slots. GB300's fp64 pipe is narrow, so fp64 does only the
// products, the running sums and the budget comparisons. The steps:
//  * survivals as fp64 products in position order (the same products, bit
//    for bit, as a sequential reference);
//  * the ranking, one of two ways by size: up to 2^23 slot-request pairs, a
//    grid counts every slot's rank by binary searches (ps_rank_kernel);
//    beyond that, one CTA of 1024 threads runs a bitonic sort of (survival
//    bits as an integer, position * R + request) pairs, in registers,
//    shuffles and shared memory by stride (ps_schedule_kernel);
//  * expected tokens for every n: each of 256 threads sums a contiguous run
//    of the ranked survivals and a block scan gives the runs' offsets;
//    budgets are compared by cross-multiplying tokens and costs, and a
//    reduction finds the best n;
//  * kept slots counted per request with shared-memory atomics.
#include <cuda_runtime.h>
#include <stdint.h>

#include "ddt_device.cuh"
#include "ddt_internal.h"

namespace {

constexpr int PS_THREADS = 1024;
constexpr int PS_WARPS = PS_THREADS / 32;
constexpr int64_t PS_RANK_WORK = 1 << 23;  // slot-request pairs for the rank-counting grid

// Ranking keys: a survival s >= 0 as its fp64 bit pattern (the integer
// order of the bits is the order of the values), with the slot's
// position * R + request breaking ties. Slot a ranks before slot b when
// its survival is larger, or equal with a smaller tie id.
DDT_DEVINL bool ranks_before(uint64_t ka, int ia, uint64_t kb, int ib)
{
    return ka > kb || (ka == kb && ia < ib);
}

// (tokens T, cost c, n): T/c larger wins (compared as T_a c_b > T_b c_a),
// then the smaller n
DDT_DEVINL void best_merge(double &T, double &C, int &n, double T2, double C2, int n2)
{
    const double lhs = T2 * C, rhs = T * C2;
    if (n2 != 0x7FFFFFFF && (n == 0x7FFFFFFF || lhs > rhs || (lhs == rhs && n2 < n))) {
        T = T2;
        C = C2;
        n = n2;
    }
}

DDT_DEVINL bool cost_ok(float c) { return c == c && c > 0.f; }

// Survivals of every slot into keys[r * L + k] (fp64 products in position
// order, as bits) and zeroed per-request counters. The confidences are
// first read by all threads at once (coalesced) and held, clamped, in the
// key array; each request's thread then runs its products in place.
DDT_DEVINL void ps_survivals(const float *__restrict__ conf, int R, int L, uint64_t *keys,
                             int *s_cnt, int32_t *status)
{
    const int N = R * L;
    for (int j = threadIdx.x; j < N; j += PS_THREADS) {
        float c = conf[j];
        if (c != c) {
            if (status)
                set_status(status, DDT_DEV_NAN_LOGITS);
            c = 0.f;
        }
        keys[j] = (uint64_t)__float_as_uint(fminf(fmaxf(c, 0.f), 1.f));
    }
    __syncthreads();
    for (int r = threadIdx.x; r < R; r += PS_THREADS) {
        double sv = 1.0;
        for (int k = 0; k < L; ++k) {
            sv = sv * (double)__uint_as_float((uint32_t)keys[r * L + k]);
            keys[r * L + k] = (uint64_t)__double_as_longlong(sv);
        }
        s_cnt[r] = 0;
    }
}

// The ranked slots (survival bits rk, tie ids rid, in ranking order, N of
// them) to the chosen budget and the kept guesses per request. s_cnt: R
// zeroed counters in shared memory. All PS_THREADS threads call it; the fp64
// work (the running sums and the budget comparisons) stays on PS_FP64
// threads, because GB300's fp64 pipe is narrow: every lane-op counts.
constexpr int PS_FP64 = 256;
constexpr int PS_FP64_WARPS = PS_FP64 / 32;

DDT_DEVINL void ps_budget_and_keep(const uint64_t *s_key, const int *s_id, int *s_cnt, int R,
                                   int N, const float *__restrict__ cost,
                                   int32_t *__restrict__ n_keep, int32_t *__restrict__ n_total,
                                   double *__restrict__ stats)
{
    __shared__ double s_wsum[PS_FP64_WARPS];
    __shared__ double s_bT[PS_FP64_WARPS], s_bC[PS_FP64_WARPS];
    __shared__ int s_bn[PS_FP64_WARPS];
    __shared__ int s_nstar;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const bool fp = tid < PS_FP64;
    // expected tokens for every n: fp thread t owns n = j + 1 for j in a
    // contiguous run [j0, j1) of the ranking (thread 0 also owns n = 0)
    const int seg = (N + PS_FP64 - 1) / PS_FP64;
    const int j0 = fp ? min(N, tid * seg) : N, j1 = fp ? min(N, j0 + seg) : N;
    double run = 0.0, incl = 0.0;
    if (fp) {
        for (int j = j0; j < j1; ++j)
            run += __longlong_as_double((long long)s_key[j]);
        incl = run;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const double y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
            if (lane >= o)
                incl += y;
        }
        if (lane == 31)
            s_wsum[warp] = incl;
    }
    __syncthreads();
    if (warp == 0) {
        const double own = lane < PS_FP64_WARPS ? s_wsum[lane] : 0.0;
        double w = own;
#pragma unroll
        for (int o = 1; o < PS_FP64_WARPS; o <<= 1) {
            const double y = __shfl_up_sync(0xFFFFFFFFu, w, o);
            if (lane >= o)
                w += y;
        }
        if (lane < PS_FP64_WARPS)
            s_wsum[lane] = w - own;  // exclusive over warps
    }
    __syncthreads();
    const double Rd = (double)R;
    double bT = Rd, bC = 1.0;
    int bn = 0x7FFFFFFF;
    if (fp) {
        double P = s_wsum[warp] + (incl - run);
        if (tid == 0 && cost_ok(cost[0]))
            best_merge(bT, bC, bn, Rd, (double)cost[0], 0);
        for (int j = j0; j < j1; ++j) {
            P += __longlong_as_double((long long)s_key[j]);
            const float c = cost[j + 1];
            if (cost_ok(c))
                best_merge(bT, bC, bn, Rd + P, (double)c, j + 1);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const double T2 = __shfl_xor_sync(0xFFFFFFFFu, bT, o);
            const double C2 = __shfl_xor_sync(0xFFFFFFFFu, bC, o);
            const int n2 = __shfl_xor_sync(0xFFFFFFFFu, bn, o);
            best_merge(bT, bC, bn, T2, C2, n2);
        }
        if (lane == 0) {
            s_bT[warp] = bT;
            s_bC[warp] = bC;
            s_bn[warp] = bn;
        }
    }
    __syncthreads();
    if (warp == 0) {
        if (lane < PS_FP64_WARPS) {
            bT = s_bT[lane];
            bC = s_bC[lane];
            bn = s_bn[lane];
        } else {
            bn = 0x7FFFFFFF;
        }
#pragma unroll
        for (int o = PS_FP64_WARPS / 2; o > 0; o >>= 1) {
            const double T2 = __shfl_xor_sync(0xFFFFFFFFu, bT, o);
            const double C2 = __shfl_xor_sync(0xFFFFFFFFu, bC, o);
            const int n2 = __shfl_xor_sync(0xFFFFFFFFu, bn, o);
            best_merge(bT, bC, bn, T2, C2, n2);
        }
        if (lane == 0) {
            double theta = bT / bC;
            if (bn == 0x7FFFFFFF) {  // no n has a valid cost: verify nothing
                bn = 0;
                theta = 0.0;
                bT = Rd;
            }
            s_nstar = bn;
            if (n_total)
                *n_total = bn;
            if (stats) {
                stats[0] = theta;
                stats[1] = bT;
            }
        }
    }
    __syncthreads();

    // kept slots per request (a prefix of each block)
    const int nstar = s_nstar;
    for (int j = tid; j < nstar; j += PS_THREADS)
        atomicAdd(&s_cnt[s_id[j] % R], 1);
    __syncthreads();
    for (int r = tid; r < R; r += PS_THREADS)
        n_keep[r] = s_cnt[r];
}


// one bitonic pass whose partners are registers q and q ^ QS of this thread
template <int EPT, int QS>
DDT_DEVINL void reg_pass(uint64_t (&key)[EPT], int (&id)[EPT], int size, int tid)
{
#pragma unroll
    for (int q = 0; q < EPT; ++q) {
        const int q2 = q ^ QS;
        if (q2 > q && q2 < EPT) {
            const int i = q * PS_THREADS + tid;
            const bool sw = (i & size) == 0 ? ranks_before(key[q2], id[q2], key[q], id[q])
                                            : ranks_before(key[q], id[q], key[q2], id[q2]);
            if (sw) {
                const uint64_t tk = key[q];
                key[q] = key[q2];
                key[q2] = tk;
                const int ti = id[q];
                id[q] = id[q2];
                id[q2] = ti;
            }
        }
    }
}

// EPT ranking slots per thread: slot q * 1024 + tid lives in register q
// during the sort, so strides >= 1024 are swaps within a thread, strides
// < 32 are shuffles within a warp, and only 32 <= stride < 1024 goes
// through shared memory.
template <int EPT>
__global__ void __launch_bounds__(PS_THREADS, 1)
ps_schedule_kernel(const float *__restrict__ conf, const float *__restrict__ cost, int R, int L,
                   int32_t *__restrict__ n_keep, int32_t *__restrict__ n_total,
                   double *__restrict__ stats, int32_t *__restrict__ status)
{
    constexpr int NP = EPT * PS_THREADS;
    extern __shared__ __align__(16) uint8_t ps_smem[];
    uint64_t *s_key = reinterpret_cast<uint64_t *>(ps_smem);  // [NP]
    int *s_id = reinterpret_cast<int *>(s_key + NP);           // [NP]
    int *s_cnt = s_id + NP;                                     // [R]
    const int N = R * L;
    const int tid = threadIdx.x;

    // ---- survivals, request by request in position order (fp64 products)
    ps_survivals(conf, R, L, s_key, s_cnt, status);
    for (int j = tid; j < N; j += PS_THREADS)
        s_id[j] = (j % L) * R + j / L;
    __syncthreads();
    uint64_t key[EPT];
    int id[EPT];
#pragma unroll
    for (int q = 0; q < EPT; ++q) {
        const int i = q * PS_THREADS + tid;
        key[q] = i < N ? s_key[i] : 0ull;  // padding: below every survival ...
        id[q] = i < N ? s_id[i] : 0x7FFFFFFF;  // ... and after it on ties
    }

    // ---- bitonic sort into ranking order
    bool in_smem = false;
    for (int size = 2; size <= NP; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            if (stride >= PS_THREADS) {  // partner in register q ^ (stride / 1024)
                const int qs = stride / PS_THREADS;
                if (qs == 1)
                    reg_pass<EPT, 1>(key, id, size, tid);
                else if (qs == 2)
                    reg_pass<EPT, 2>(key, id, size, tid);
                else
                    reg_pass<EPT, 4>(key, id, size, tid);
            } else if (stride >= 32) {  // partner in another warp: shared memory
                if (!in_smem) {
                    __syncthreads();  // earlier readers are done
#pragma unroll
                    for (int q = 0; q < EPT; ++q) {
                        s_key[q * PS_THREADS + tid] = key[q];
                        s_id[q * PS_THREADS + tid] = id[q];
                    }
                    __syncthreads();
                    in_smem = true;
                }
                for (int p = tid; p < NP / 2; p += PS_THREADS) {
                    const int lo = 2 * p - (p & (stride - 1));
                    const int hi = lo + stride;
                    const uint64_t a = s_key[lo], b = s_key[hi];
                    const int ia = s_id[lo], ib = s_id[hi];
                    const bool sw = (lo & size) == 0 ? ranks_before(b, ib, a, ia)
                                                     : ranks_before(a, ia, b, ib);
                    if (sw) {
                        s_key[lo] = b;
                        s_key[hi] = a;
                        s_id[lo] = ib;
                        s_id[hi] = ia;
                    }
                }
                __syncthreads();
            } else {  // partner in this warp: shuffles
                if (in_smem) {
#pragma unroll
                    for (int q = 0; q < EPT; ++q) {
                        key[q] = s_key[q * PS_THREADS + tid];
                        id[q] = s_id[q * PS_THREADS + tid];
                    }
                    in_smem = false;
                }
#pragma unroll
                for (int q = 0; q < EPT; ++q) {
                    const int i = q * PS_THREADS + tid;
                    const uint64_t ok = __shfl_xor_sync(0xFFFFFFFFu, key[q], stride);
                    const int oi = __shfl_xor_sync(0xFFFFFFFFu, id[q], stride);
                    const bool lower = (i & stride) == 0;
                    const bool asc = (i & size) == 0;
                    // the lower index of an ascending pair keeps the slot that
                    // ranks first; every other combination keeps the other one
                    const bool mine_first = ranks_before(key[q], id[q], ok, oi);
                    const bool keep_mine = (lower == asc) ? mine_first : !mine_first;
                    if (!keep_mine) {
                        key[q] = ok;
                        id[q] = oi;
                    }
                }
            }
        }
    }
    // the ranking, in shared memory, for contiguous runs per thread
    __syncthreads();
    if (!in_smem) {
#pragma unroll
        for (int q = 0; q < EPT; ++q) {
            s_key[q * PS_THREADS + tid] = key[q];
            s_id[q * PS_THREADS + tid] = id[q];
        }
    }
    __syncthreads();

    ps_budget_and_keep(s_key, s_id, s_cnt, R, N, cost, n_keep, n_total, stats);
}

// Up to PS_RANK_WORK slot-request pairs: each request's survivals already
// fall along its block, so a slot's rank is the number of slots of each
// request that rank before it -- one binary search per request. One warp
// per slot (its lanes split the requests), 32 slots per CTA, as many CTAs
// as that takes: every CTA rebuilds the survival table in shared memory,
// scatters its slots' keys to their ranks in the workspace, and the last
// CTA to finish (an arrival counter) reads the ranking back and picks the
// budget.
__global__ void __launch_bounds__(PS_THREADS, 1)
ps_rank_kernel(const float *__restrict__ conf, const float *__restrict__ cost, int R, int L,
               uint64_t *__restrict__ ws_rk, int *__restrict__ ws_rid, unsigned *ws_arrive,
               int32_t *__restrict__ n_keep, int32_t *__restrict__ n_total,
               double *__restrict__ stats, int32_t *__restrict__ status)
{
    extern __shared__ __align__(16) uint8_t ps_smem[];
    const int N = R * L;
    uint64_t *s_key = reinterpret_cast<uint64_t *>(ps_smem);  // [N] by request, position
    int *s_rid = reinterpret_cast<int *>(s_key + N);           // [N] (the last CTA)
    int *s_cnt = s_rid + N;                                     // [R]
    __shared__ bool s_last;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    ps_survivals(conf, R, L, s_key, s_cnt, blockIdx.x == 0 ? status : nullptr);
    __syncthreads();
    const int j = blockIdx.x * PS_WARPS + warp;
    if (j < N) {
        const int r = j / L, k = j - r * L;
        const uint64_t key = s_key[j];
        const int id = k * R + r;
        int rank = 0;
        for (int r2 = lane; r2 < R; r2 += 32) {
            const uint64_t *row = s_key + r2 * L;
            int lo = 0, hi = L;  // slots of r2 that rank before (r, k): a prefix
            while (lo < hi) {
                const int mid = (lo + hi) >> 1;
                if (ranks_before(row[mid], mid * R + r2, key, id))
                    lo = mid + 1;
                else
                    hi = mid;
            }
            rank += lo;
        }
        rank = __reduce_add_sync(0xFFFFFFFFu, rank);
        if (lane == 0) {
            ws_rk[rank] = key;
            ws_rid[rank] = id;
        }
    }
    __syncthreads();
    if (tid == 0) {
        __threadfence();
        const unsigned prev = atomicAdd(ws_arrive, 1u);
        s_last = prev == gridDim.x - 1;
        if (s_last) {
            *ws_arrive = 0u;  // every arrival of this call is in: ready for the next
            __threadfence();
        }
    }
    __syncthreads();
    if (!s_last)
        return;
    for (int q = tid; q < N; q += PS_THREADS) {  // the ranking, over this CTA's survivals
        s_key[q] = __ldcg(ws_rk + q);
        s_rid[q] = __ldcg(ws_rid + q);
    }
    for (int r = tid; r < R; r += PS_THREADS)
        s_cnt[r] = 0;
    __syncthreads();
    ps_budget_and_keep(s_key, s_rid, s_cnt, R, N, cost, n_keep, n_total, stats);
}

}  // namespace

int schedule_smem_bytes(int R, int L)
{
    int NP = PS_THREADS;
    while (NP < R * L)
        NP <<= 1;
    return NP * (int)(sizeof(uint64_t) + sizeof(int)) + R * (int)sizeof(int);
}

template <int EPT>
cudaError_t launch_ps(const ddt_ctx *c, const float *conf, int R, const float *cost,
                      int32_t *n_keep, int32_t *n_total, double *stats, cudaStream_t s)
{
    static bool attr_set = false;  // the same value on every device
    if (!attr_set) {
        const cudaError_t e =
            cudaFuncSetAttribute(ps_schedule_kernel<EPT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 EPT * PS_THREADS * 12 + 4 * EPT * PS_THREADS);
        if (e != cudaSuccess)
            return e;
        attr_set = true;
    }
    ps_schedule_kernel<EPT><<<1, PS_THREADS, schedule_smem_bytes(R, c->cfg.L), s>>>(
        conf, cost, R, c->cfg.L, n_keep, n_total, stats, c->status);
    return cudaGetLastError();
}

cudaError_t launch_schedule_prefix(const ddt_ctx *c, const float *conf, int R, const float *cost,
                                   int32_t *n_keep, int32_t *n_total, double *stats,
                                   cudaStream_t s)
{
    const int N = R * c->cfg.L;
    if ((int64_t)N * R <= PS_RANK_WORK) {
        static bool attr_set = false;  // the same value on every device
        if (!attr_set) {
            const cudaError_t e =
                cudaFuncSetAttribute(ps_rank_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     DDT_SCHED_MAX_SLOTS * 12 + 4 * DDT_SCHED_MAX_SLOTS);
            if (e != cudaSuccess)
                return e;
            attr_set = true;
        }
        const int grid = (N + PS_WARPS - 1) / PS_WARPS;
        ps_rank_kernel<<<grid, PS_THREADS, N * 12 + 4 * R, s>>>(
            conf, cost, R, c->cfg.L, c->ps_rk, c->ps_rid, c->ps_arrive, n_keep, n_total, stats,
            c->status);
        return cudaGetLastError();
    }
    // past 2^23 pairs there are more than 4096 slots (R <= 2048): 8 per thread
    return launch_ps<8>(c, conf, R, cost, n_keep, n_total, stats, s);
}
