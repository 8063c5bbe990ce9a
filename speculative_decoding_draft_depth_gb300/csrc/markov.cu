// markov.cu -- the SparklingTree table tree ("SparklingTree: 30-40% faster
// speculative decoding over DSpark", sections "Solving the candidate tree
// construction" and "Building SparklingTree"; the Markov head of "First
// order markov model conditioning": a bias W1[x_prev] W2 on the next
// position's logits, written z_d(b | a) = l_d[b] + W[b] . E[a]).
//
//  * mk_prefilter_kernel keeps every depth's C best draft tokens: a lower
//    bound from per-thread maxima, then the few values above it, ranked.
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

// ---------------------------------------------------------------- prefilter
// One CTA per (request, depth) row of bf16 logits. Pass 1: every thread's
// max and the positions of its four best 8-value vectors; the C-th largest of
// the 256 maxima is a value that C elements reach, so no element below it is
// among the C best. Pass 2 re-reads only the vectors that reach it (a few per
// row) and collects their elements at or above it; a rank count sorts them
// by (value desc, id asc). Rows with more survivors than the buffer holds
// (heavy ties) take an exact bitwise search instead.
constexpr int PF_THREADS = 256;
constexpr int PF_CAP = 2048;

DDT_DEVINL uint32_t bmax2(uint32_t a, uint32_t b)
{
    uint32_t r;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}
DDT_DEVINL float vmax8(const uint4 &v)
{
    const uint32_t w = bmax2(bmax2(v.x, v.y), bmax2(v.z, v.w));
    return fmaxf(bf16lo(w), bf16hi(w));
}
DDT_DEVINL float elem8(const uint4 &v, int e)
{
    const uint32_t w = (e < 2) ? v.x : (e < 4) ? v.y : (e < 6) ? v.z : v.w;
    return (e & 1) ? bf16hi(w) : bf16lo(w);
}
// candidate key: ordered value high, complemented id low (lower id wins a tie)
DDT_DEVINL uint64_t pf_key(float v, int id) { return ((uint64_t)mk_fkey(v) << 32) | (uint32_t)~(uint32_t)id; }

DDT_DEVINL int pf_block_sum(int v, int *s_acc)
{
    __syncthreads();
    if (threadIdx.x == 0)
        *s_acc = 0;
    __syncthreads();
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    if ((threadIdx.x & 31) == 0)
        atomicAdd(s_acc, v);
    __syncthreads();
    return *s_acc;
}

__device__ void prefilter_row(const uint16_t *__restrict__ z, int V, int C, int vec,
                              int32_t *__restrict__ out, uint32_t *s_tmax, uint64_t *s_key,
                              uint32_t *s_t_, int *s_n_, int *s_acc_)
{
    const int tid = threadIdx.x, lane = tid & 31;
    uint32_t &s_t = *s_t_;
    int &s_n = *s_n_;
    int &s_acc = *s_acc_;
    const int nvec = vec ? V / 8 : 0;
    const uint4 *zv = reinterpret_cast<const uint4 *>(z);
    // pass 1: this thread's max (NaN never wins), and its four best vectors
    float tv[4] = {DDT_NEG_INF, DDT_NEG_INF, DDT_NEG_INF, DDT_NEG_INF};
    int ti[4] = {-1, -1, -1, -1};
    constexpr int PF_BATCH = 4;  // vectors in flight per thread
    for (int i0 = tid; i0 < nvec; i0 += PF_BATCH * PF_THREADS) {
        float vm[PF_BATCH];
#pragma unroll
        for (int u = 0; u < PF_BATCH; ++u) {
            const int i = i0 + u * PF_THREADS;
            vm[u] = (i < nvec) ? vmax8(__ldg(zv + i)) : DDT_NEG_INF;
        }
#pragma unroll
        for (int u = 0; u < PF_BATCH; ++u) {
            float x = vm[u];
            if (x > tv[3]) {
                int xi = i0 + u * PF_THREADS;
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    if (x > tv[q]) {
                        const float t = tv[q];
                        const int w = ti[q];
                        tv[q] = x;
                        ti[q] = xi;
                        x = t;
                        xi = w;
                    }
            }
        }
    }
    float m = tv[0];
    for (int i = nvec * 8 + tid; i < V; i += PF_THREADS)
        m = fmaxf(m, bf16_to_f32(z[i]));
    // the C-th largest of the 256 maxima: each warp sorts its 32 (descending,
    // bitonic over the lanes), then each thread's rank is its place in its
    // own warp's list plus a binary search in each other warp's
    const uint32_t mk = mk_fkey(m);
    uint32_t sv = mk;
#pragma unroll
    for (int k2 = 2; k2 <= 32; k2 <<= 1)
#pragma unroll
        for (int j = k2 >> 1; j > 0; j >>= 1) {
            const uint32_t o = __shfl_xor_sync(0xFFFFFFFFu, sv, j);
            const bool up = ((lane & k2) == 0) != ((lane & j) != 0);  // keep the larger
            sv = up ? (sv > o ? sv : o) : (sv < o ? sv : o);
        }
    s_tmax[tid] = sv;  // warp w's maxima, descending, at [32 w, 32 w + 32)
    if (tid == 0)
        s_n = 0;
    __syncthreads();
    {
        const int w0 = tid >> 5;
        const uint32_t x = s_tmax[tid];
        int rank = lane;  // equal values: the earlier position in the sorted lists first
        for (int w = 0; w < PF_THREADS / 32; ++w) {
            if (w == w0)
                continue;
            const uint32_t *l = s_tmax + 32 * w;
            int lo = 0, hi = 32;  // entries of list w before x
            while (lo < hi) {
                const int mid = (lo + hi) >> 1;
                if (l[mid] > x || (l[mid] == x && w < w0))
                    lo = mid + 1;
                else
                    hi = mid;
            }
            rank += lo;
        }
        if (rank == C - 1)
            s_t = x;
    }
    __syncthreads();
    const float T = mk_fkey_inv(s_t);
    // pass 2: the elements at or above T. Only vectors whose max reaches T
    // hold them: a thread re-reads its best vectors that do, or all of its
    // vectors when even its fourth best does (more may)
    auto take = [&](int i) {
        const uint4 v = __ldg(zv + i);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const float x = elem8(v, e);
            if (x >= T) {
                const int base = atomicAdd(&s_n, 1);
                if (base < PF_CAP)
                    s_key[base] = pf_key(x, i * 8 + e);
            }
        }
    };
    if (tv[3] >= T) {
#pragma unroll 1
        for (int i = tid; i < nvec; i += PF_THREADS)
            if (vmax8(__ldg(zv + i)) >= T)
                take(i);
    } else {
#pragma unroll
        for (int q = 0; q < 4; ++q)
            if (tv[q] >= T)
                take(ti[q]);
    }
    for (int i = nvec * 8 + tid; i < V; i += PF_THREADS) {
        const float x = bf16_to_f32(z[i]);
        if (x >= T) {
            const int base = atomicAdd(&s_n, 1);
            if (base < PF_CAP)
                s_key[base] = pf_key(x, i);
        }
    }
    __syncthreads();
    int n = s_n;
    if (n > PF_CAP) {
        // exact: the C-th largest key by bits, then every key above it
        uint64_t t = 0;
        for (int b = 63; b >= 0; --b) {
            const uint64_t cb = t | (1ull << b);
            int c = 0;
#pragma unroll 1
            for (int i = tid; i < V; i += PF_THREADS) {
                const float x = bf16_to_f32(z[i]);
                c += (x == x && pf_key(x, i) >= cb) ? 1 : 0;
            }
            if (pf_block_sum(c, &s_acc) >= C)
                t = cb;
        }
        if (tid == 0)
            s_n = 0;
        __syncthreads();
#pragma unroll 1
        for (int i = tid; i < V; i += PF_THREADS) {
            const float x = bf16_to_f32(z[i]);
            if (x == x && pf_key(x, i) >= t)
                s_key[atomicAdd(&s_n, 1)] = pf_key(x, i);  // exactly C of them
        }
        __syncthreads();
        n = s_n;
    }
    // ranks: four threads per survivor, each counting a quarter of the others
    for (int i0 = 0; i0 < n; i0 += PF_THREADS / 4) {
        const int i = i0 + (tid >> 2);
        const bool have = i < n;
        const uint64_t ki = have ? s_key[i] : 0ull;
        int rk = 0;
        if (have) {
#pragma unroll 4
            for (int j = tid & 3; j < n; j += 4)
                rk += (s_key[j] > ki) ? 1 : 0;
        }
        rk += __shfl_xor_sync(0xFFFFFFFFu, rk, 1);
        rk += __shfl_xor_sync(0xFFFFFFFFu, rk, 2);
        if (have && (tid & 3) == 0 && rk < C)
            out[rk] = (int)~(uint32_t)ki;
    }
}

__global__ void __launch_bounds__(PF_THREADS, 7)  // 7 CTAs per SM: every row in one wave
mk_prefilter_kernel(const uint16_t *__restrict__ ell, int rows, int V, int C, int vec,
                    int32_t *__restrict__ cand)
{
    __shared__ uint32_t s_tmax[PF_THREADS];
    __shared__ uint64_t s_key[PF_CAP];
    __shared__ uint32_t s_t;
    __shared__ int s_n, s_acc;
    for (int row = blockIdx.x; row < rows; row += gridDim.x) {
        prefilter_row(ell + (int64_t)row * V, V, C, vec, cand + (int64_t)row * C, s_tmax, s_key,
                      &s_t, &s_n, &s_acc);
        __syncthreads();
    }
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
// the operand tiles of one half of H (A then B, two 64-column blocks each),
// reused for the staged table once the last MMA has completed; small enough
// for three CTAs per SM
constexpr uint32_t MK_HALF = 2 * 16384u;  // one operand tile of 128 rows x 128 columns of H
struct TableSmem {
    uint32_t a, b, lv, bar, total;
};
__host__ __device__ inline TableSmem table_layout(int H)
{
    (void)H;
    TableSmem S;
    S.a = 0;
    S.b = MK_HALF;
    S.lv = 2 * MK_HALF;         // l of the kept children: [128] floats
    S.bar = S.lv + 4u * MK_N;   // [0]: MMA done, [8]: TMEM address
    S.total = S.bar + 16;
    return S;
}

__global__ void __launch_bounds__(MK_THREADS)
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
    const int32_t *cd = a.cand + (int64_t)rd * a.C;
    const int32_t *cp = a.cand + (int64_t)(rd - (d > 0 ? 1 : 0)) * a.C;
    // this thread's rows: the parents' E rows (A) and the kept children's W
    // rows (B), zero past the kept ones
    int pt[MK_N / MK_THREADS], ct[MK_N / MK_THREADS];
    (void)pt;
    for (int b = tid; b < MK_N; b += MK_THREADS) {
        const int c = (b < a.C) ? cd[b] : -1;
        s_l[b] = (c >= 0 && c < a.V) ? bf16_to_f32(a.ell[(int64_t)rd * a.V + c]) : DDT_NEG_INF;
    }
    for (int u = 0; u < MK_N / MK_THREADS; ++u) {
        const int p = tid + u * MK_THREADS;
        int t = -1;
        if (d == 0)
            t = (p == 0) ? a.anchors[r] : -1;
        else if (p < a.C)
            t = cp[p];
        pt[u] = (t >= 0 && t < a.V) ? t : -1;
        const int c = (p < a.C) ? cd[p] : -1;
        ct[u] = (c >= 0 && c < a.V) ? c : -1;
    }
    const int nblk = a.H / 64, nhalf = (nblk + 1) / 2;
    bool ok = true;
    __syncthreads();  // the barrier is initialised
    for (int hf = 0; hf < nhalf; ++hf) {
        const int b0 = 2 * hf, nb = (nblk - b0 < 2) ? nblk - b0 : 2;
        // gather this half: row p = this thread's rows, 16-byte chunks of 8 values
        for (int u = 0; u < MK_N / MK_THREADS; ++u) {
            const int p = tid + u * MK_THREADS;
            for (int c = 0; c < nb * 8; ++c) {
                const uint32_t off = (uint32_t)(c >> 3) * 16384u + (uint32_t)p * 128u +
                                     ((uint32_t)((c & 7) ^ (p & 7)) << 4);
                const int h = (b0 * 8 + c) * 8;  // first of the chunk's 8 values of H
                cp_async_16(sb + S.a + off,
                            pt[u] >= 0 ? (const void *)(a.E + (int64_t)pt[u] * a.H + h) : (const void *)a.E,
                            pt[u] >= 0 ? 16u : 0u);
                cp_async_16(sb + S.b + off,
                            ct[u] >= 0 ? (const void *)(a.W + (int64_t)ct[u] * a.H + h) : (const void *)a.W,
                            ct[u] >= 0 ? 16u : 0u);
            }
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
            for (int kk = 0; kk < nb * 4; ++kk) {
                const uint32_t off = ((uint32_t)(kk >> 2) * 16384u + (uint32_t)(kk & 3) * 32u) >> 4;
                mma_bf16(tmem, dA + off, dB + off, idesc, (hf > 0 || kk > 0) ? 1u : 0u);
            }
            mma_commit(bar);
        }
        // the tiles are free (and the sum complete after the last half) once the MMAs are done
        ok = __syncthreads_and((ok && mk_wait(bar, hf & 1, a.status)) ? 1 : 0) != 0;
        tc_fence_after();
        if (!ok)
            break;
    }
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(sgen + S.bar + 8);
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
    // the staged table over the operand tiles: row a, column b at a * 128 +
    // (b ^ (a & 31)) (conflict-free both when a thread writes its row and when
    // a warp reads one)
    float *T = reinterpret_cast<float *>(sgen);
    if (ok) {
#pragma unroll 1
        for (int c0 = 0; c0 < MK_N; c0 += 32) {
            uint32_t acc[32];
            tmem_ld16(ta + c0, acc);
            tmem_ld16(ta + c0 + 16, acc + 16);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 32; ++j)
                T[tid * MK_N + ((c0 + j) ^ (tid & 31))] =
                    valid ? (__uint_as_float(acc[j]) + s_l[c0 + j]) - lse : DDT_NEG_INF;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (ok) {
        float *dst = a.tab + (int64_t)rd * a.C * a.C;
        for (int row = warp; row < a.C; row += MK_THREADS / 32)
            for (int b = lane; b < a.C; b += 32)
                dst[(int64_t)row * a.C + b] = T[row * MK_N + (b ^ (row & 31))];
    }
    if (!ok && tid == 0) {  // a wait gave up: let the MMAs finish before the TMEM goes (bounded)
        const long long t0 = clock64();
        while (!mbar_try_wait(bar, (nhalf - 1) & 1) && clock64() - t0 < 200000000LL) {
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

// frontier slots per lane: a template parameter, ceil(B / 32) (each pop adds
// at most one entry, so B entries fit)

DDT_DEVINL void prefetch_l1(const void *p)
{
    asm volatile("prefetch.global.L1 [%0];" ::"l"(p));
}

struct TreeArgs {
    const int32_t *cand;  // [R, L, C]
    const float *tab;     // [R, L, C, C]
    int L, C, B;
    int32_t *tree_tokens, *parents, *depths, *n_nodes;
    uint32_t *mask;
};

template <int SLOTS>
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
        // the popped node's own row (its children), requested first: the
        // sibling's scan below runs while it is in flight
        float rv[4];
        if (wdep < L) {
            const float *src = tr + ((int64_t)wdep * C + wcb) * C;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int b = lane + 32 * i;
                rv[i] = (b < C) ? src[b] : DDT_NEG_INF;
            }
        }
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
        // a pushed entry's own row is warmed into L1 now, for when it is popped
        if (sib != 0ull && wdep < L && lane < 4 && lane * 32 < C)
            prefetch_l1(tr + ((int64_t)wdep * C + scol) * C + lane * 32);
        if (wdep < L) {
            uint64_t k[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int b = lane + 32 * i;
                if (b < C)
                    s_rows[node * C + b] = rv[i];
                k[i] = (b < C) ? child_key(rv[i], s_cand[wdep * C + b]) : 0ull;
            }
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
                if (wdep + 1 < L && lane < 4 && lane * 32 < C)
                    prefetch_l1(tr + ((int64_t)(wdep + 1) * C + ccol) * C + lane * 32);
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
           cfg.L <= DDT_MAX_L && tree_smem(cfg.L, C, cfg.B) <= 200 * 1024;
}

cudaError_t launch_markov_table(const ddt_ctx *c, const uint16_t *ell, const uint16_t *W,
                                const uint16_t *E, const int32_t *anchors, int R, int32_t *cand,
                                float *tab, cudaStream_t s)
{
    const ddt_config &cfg = c->cfg;
    const int C = cfg.prefilter, L = cfg.L;
    // the prefilter: each row's C best tokens
    const int vec = (cfg.V % 8 == 0 && ((uintptr_t)ell & 15u) == 0) ? 1 : 0;
    mk_prefilter_kernel<<<R * L, PF_THREADS, 0, s>>>(ell, R * L, cfg.V, C, vec, cand);
    cudaError_t e = cudaGetLastError();
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
    static bool attr = false;
    cudaError_t e;
    if (!attr) {
        if ((e = cudaFuncSetAttribute(mk_tree_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      200 * 1024)) != cudaSuccess ||
            (e = cudaFuncSetAttribute(mk_tree_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      200 * 1024)) != cudaSuccess ||
            (e = cudaFuncSetAttribute(mk_tree_kernel<3>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      200 * 1024)) != cudaSuccess ||
            (e = cudaFuncSetAttribute(mk_tree_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      200 * 1024)) != cudaSuccess)
            return e;
        attr = true;
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
    const int slots = (cfg.B + 31) / 32;  // 1..4 (B <= 127)
    if (slots <= 1)
        mk_tree_kernel<1><<<R, 32, smem, s>>>(a);
    else if (slots == 2)
        mk_tree_kernel<2><<<R, 32, smem, s>>>(a);
    else if (slots == 3)
        mk_tree_kernel<3><<<R, 32, smem, s>>>(a);
    else
        mk_tree_kernel<4><<<R, 32, smem, s>>>(a);
    return cudaGetLastError();
}
