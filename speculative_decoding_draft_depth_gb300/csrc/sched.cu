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
// One CTA of 1024 threads and up to 8192 slots, all in shared memory:
//  * survivals as fp64 products in position order (the same products, bit
//    for bit, as a sequential reference);
//  * a bitonic sort of (survival, position * R + request) pairs;
//  * tokens per ms for every n: each thread sums a contiguous run of the
//    ranked survivals, a block scan gives the runs' offsets, and a block
//    reduction finds the best n;
//  * kept slots counted per request with shared-memory atomics.
#include <cuda_runtime.h>
#include <stdint.h>

#include "ddt_device.cuh"
#include "ddt_internal.h"

namespace {

constexpr int PS_THREADS = 1024;
constexpr int PS_WARPS = PS_THREADS / 32;

// slot a goes before slot b in the ranking
DDT_DEVINL bool ranks_before(double sa, int ia, double sb, int ib)
{
    return sa > sb || (sa == sb && ia < ib);
}

// (tokens per ms, n, tokens): the larger ratio wins, then the smaller n
DDT_DEVINL void best_merge(double &th, int &n, double &tok, double th2, int n2, double tok2)
{
    if (th2 > th || (th2 == th && n2 < n)) {
        th = th2;
        n = n2;
        tok = tok2;
    }
}

DDT_DEVINL bool cost_ok(float c) { return c == c && c > 0.f; }

__global__ void __launch_bounds__(PS_THREADS, 1)
ps_schedule_kernel(const float *__restrict__ conf, const float *__restrict__ cost, int R, int L,
                   int NP, int32_t *__restrict__ n_keep, int32_t *__restrict__ n_total,
                   double *__restrict__ stats, int32_t *__restrict__ status)
{
    extern __shared__ __align__(16) uint8_t ps_smem[];
    double *s_s = reinterpret_cast<double *>(ps_smem);  // [NP] survivals, then ranked
    int *s_i = reinterpret_cast<int *>(s_s + NP);       // [NP] position * R + request
    int *s_cnt = s_i + NP;                              // [R] kept slots per request
    __shared__ double s_wsum[PS_WARPS];
    __shared__ double s_bth[PS_WARPS], s_btok[PS_WARPS];
    __shared__ int s_bn[PS_WARPS];
    __shared__ int s_nstar;
    const int N = R * L;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    // ---- survivals, request by request in position order
    for (int r = tid; r < R; r += PS_THREADS) {
        double s = 1.0;
        for (int k = 0; k < L; ++k) {
            float c = conf[(int64_t)r * L + k];
            if (c != c) {
                set_status(status, DDT_DEV_NAN_LOGITS);
                c = 0.f;
            }
            c = fminf(fmaxf(c, 0.f), 1.f);
            s = s * (double)c;
            s_s[r * L + k] = s;
            s_i[r * L + k] = k * R + r;
        }
        s_cnt[r] = 0;
    }
    for (int j = N + tid; j < NP; j += PS_THREADS) {  // padding sorts last
        s_s[j] = -1.0;
        s_i[j] = 0x7FFFFFFF;
    }
    __syncthreads();

    // ---- bitonic sort into ranking order
    for (int size = 2; size <= NP; size <<= 1)
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            for (int p = tid; p < NP / 2; p += PS_THREADS) {
                const int lo = 2 * p - (p & (stride - 1));
                const int hi = lo + stride;
                const double a = s_s[lo], b = s_s[hi];
                const int ia = s_i[lo], ib = s_i[hi];
                const bool swap = (lo & size) == 0 ? ranks_before(b, ib, a, ia)
                                                   : ranks_before(a, ia, b, ib);
                if (swap) {
                    s_s[lo] = b;
                    s_s[hi] = a;
                    s_i[lo] = ib;
                    s_i[hi] = ia;
                }
            }
            __syncthreads();
        }

    // ---- tokens per ms for every n: thread t owns n = j + 1 for j in a
    // contiguous run [j0, j1) of the ranking (thread 0 also owns n = 0)
    const int seg = (N + PS_THREADS - 1) / PS_THREADS;
    const int j0 = min(N, tid * seg), j1 = min(N, j0 + seg);
    double run = 0.0;
    for (int j = j0; j < j1; ++j)
        run += s_s[j];
    // exclusive block scan of the runs' sums
    double incl = run;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const double y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o)
            incl += y;
    }
    if (lane == 31)
        s_wsum[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        double w = s_wsum[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const double y = __shfl_up_sync(0xFFFFFFFFu, w, o);
            if (lane >= o)
                w += y;
        }
        s_wsum[lane] = w - s_wsum[lane];  // exclusive over warps
    }
    __syncthreads();
    double P = s_wsum[warp] + (incl - run);
    const double Rd = (double)R;
    double bth = -__builtin_huge_val(), btok = Rd;
    int bn = 0x7FFFFFFF;
    if (tid == 0 && cost_ok(cost[0])) {
        bth = Rd / (double)cost[0];
        bn = 0;
    }
    for (int j = j0; j < j1; ++j) {
        P += s_s[j];
        const float c = cost[j + 1];
        if (cost_ok(c)) {
            const double th = (Rd + P) / (double)c;
            if (th > bth) {  // n grows along the run: ties keep the smaller n
                bth = th;
                bn = j + 1;
                btok = Rd + P;
            }
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const double th2 = __shfl_xor_sync(0xFFFFFFFFu, bth, o);
        const int n2 = __shfl_xor_sync(0xFFFFFFFFu, bn, o);
        const double tok2 = __shfl_xor_sync(0xFFFFFFFFu, btok, o);
        best_merge(bth, bn, btok, th2, n2, tok2);
    }
    if (lane == 0) {
        s_bth[warp] = bth;
        s_bn[warp] = bn;
        s_btok[warp] = btok;
    }
    __syncthreads();
    if (tid == 0) {
        for (int w = 1; w < PS_WARPS; ++w)
            best_merge(bth, bn, btok, s_bth[w], s_bn[w], s_btok[w]);
        if (bn == 0x7FFFFFFF) {  // no n has a valid cost: verify nothing
            bn = 0;
            bth = 0.0;
            btok = Rd;
        }
        s_nstar = bn;
        if (n_total)
            *n_total = bn;
        if (stats) {
            stats[0] = bth;
            stats[1] = btok;
        }
    }
    __syncthreads();

    // ---- kept slots per request (a prefix of each block)
    const int nstar = s_nstar;
    for (int j = tid; j < nstar; j += PS_THREADS)
        atomicAdd(&s_cnt[s_i[j] % R], 1);
    __syncthreads();
    for (int r = tid; r < R; r += PS_THREADS)
        n_keep[r] = s_cnt[r];
}

}  // namespace

int schedule_smem_bytes(int R, int L)
{
    int NP = 1;
    while (NP < R * L)
        NP <<= 1;
    return NP * (int)(sizeof(double) + sizeof(int)) + R * (int)sizeof(int);
}

cudaError_t launch_schedule_prefix(const ddt_ctx *c, const float *conf, int R, const float *cost,
                                   int32_t *n_keep, int32_t *n_total, double *stats,
                                   cudaStream_t s)
{
    const int L = c->cfg.L;
    int NP = 1;
    while (NP < R * L)
        NP <<= 1;
    const int smem = schedule_smem_bytes(R, L);
    static bool attr_set = false;  // the same value on every device
    if (!attr_set) {
        // the largest layout: DDT_SCHED_MAX_SLOTS slots, as many requests
        const cudaError_t e = cudaFuncSetAttribute(
            ps_schedule_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
            schedule_smem_bytes(DDT_SCHED_MAX_SLOTS, 1));
        if (e != cudaSuccess)
            return e;
        attr_set = true;
    }
    ps_schedule_kernel<<<1, PS_THREADS, smem, s>>>(conf, cost, R, L, NP, n_keep, n_total, stats,
                                                    c->status);
    return cudaGetLastError();
}
