// topk.cu -- a1: per-depth log-softmax and top-K over the vocabulary.
//
// "SparklingTree: 30-40% faster speculative decoding over DSpark", Step 1
// (top-K of each depth row of the drafter's marginals and the row's
// logsumexp; log-probs are logits minus logsumexp) and "DDTree Explained
// ...", section 3, Lemma 1 (K = min(B, |V|) keeps the optimal tree).
//
// Two kernels, HBM-bound: each logit is read from HBM once.
//  * Streaming (topk_chunk_kernel): a row of V logits is cut into chunks of
//    TOPK_THREADS * 8 vectors of 16 bytes; one CTA per (chunk, row), each
//    thread holding its 8 vectors (a "group" of 64 bf16 or 32 fp32 logits) in
//    registers. Pass 1 takes the group's max (bf16 pairs), pass 2 sums
//    exp2((x - max) * log2 e) on packed fp32 pairs and the MUFU unit. Each
//    group's max is stored as a 16-bit ordered key (one 2-byte word per 64
//    bf16 logits) and each warp's (max, sum of exp) pair beside it; the
//    kernel has no barrier and no shared memory, so five CTAs share an SM and
//    retire as soon as their loads land. Each CTA's first thread asks the copy
//    engine to bring the chunk of the CTA one wave later into L2 (a bulk
//    prefetch), so most register loads hit L2.
//  * Selection (topk_select_kernel), one CTA per row, launched as a
//    programmatic dependent of the streaming kernel: every group max is a
//    distinct element of the row, so the K-th largest group max T has at
//    least K elements at or above it and no element of the row's top-K lies
//    below it. T is found exactly by a two-round radix select (8 bits per
//    round) over the row's group keys (bf16 values are 16 bits; for fp32 the
//    16 high bits give the bin's lower edge, still a valid bound). Only the
//    groups whose max reaches T (about K of them) are re-read, mostly from
//    L2; their elements >= T become keys (ordered value above complemented
//    token id: a larger value, then a lower id, wins), ranked by counting,
//    for each key, the keys larger than it. logZ comes from the warps' (max,
//    sum) pairs with the final step in fp64; lp = z - logZ.
//  * Flat or heavily tied rows (more candidates than the buffers hold) take
//    an exact fallback over the whole row: four radix rounds over the 32-bit
//    ordered values find the K-th value t, then the elements above t and the
//    lowest-index ties at t, in index order.
#include <stdint.h>

#include "ddt_device.cuh"
#include "ddt_internal.h"
#include "logit_vec.cuh"

namespace {

constexpr int NV = TOPK_VEC_PER_THREAD;
static_assert(TOPK_THREADS == 256, "one histogram bin per thread");
constexpr int NWARP = TOPK_THREADS / 32;
constexpr int GRP_CAP = 256;   // candidate groups of a row (more: the exact fallback)
constexpr int KEY_CAP = 256;   // candidate elements of a row (more: the exact fallback)

// total ordering key of a float (-0 == +0); larger float -> larger key
DDT_DEVINL uint32_t okey(float x)
{
    const uint32_t b = __float_as_uint(x + 0.0f);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
DDT_DEVINL float okey_val(uint32_t h)
{
    return (h & 0x80000000u) ? __uint_as_float(h & 0x7FFFFFFFu) : __uint_as_float(~h);
}

// key: ordered value in the high word, complemented token id in the low word
// (a lower id wins a tie); a larger key beats a smaller one, 0 beats nothing
DDT_DEVINL uint64_t make_key(float v, int idx)
{
    return ((uint64_t)okey(v) << 32) | (uint32_t)~(uint32_t)idx;
}
DDT_DEVINL float key_val(uint64_t k) { return okey_val((uint32_t)(k >> 32)); }
DDT_DEVINL int key_idx(uint64_t k) { return (int)~(uint32_t)k; }

// number of keys among kv[0 .. n2) (n2 even) larger than ki
DDT_DEVINL int count_beating(const uint64_t *kv, int n2, uint64_t ki)
{
    int r = 0;
    const ulonglong2 *p = reinterpret_cast<const ulonglong2 *>(kv);
#pragma unroll 4
    for (int j = 0; j < n2 / 2; ++j) {
        const ulonglong2 q = p[j];
        r += (q.x > ki) + (q.y > ki);
    }
    return r;
}

// one element as fp32 (the exact fallback's re-read)
template <typename T>
DDT_DEVINL float load_one(const T *p, int i)
{
    if constexpr (sizeof(T) == 2)
        return bf16_to_f32(__ldg(reinterpret_cast<const unsigned short *>(p) + i));
    else
        return __ldg(reinterpret_cast<const float *>(p) + i);
}

DDT_DEVINL int block_sum(int v, int *s_acc)
{
    // s_acc must be zero on entry; returns the CTA-wide sum to every thread
    v = __reduce_add_sync(0xFFFFFFFFu, v);
    if ((threadIdx.x & 31) == 0)
        atomicAdd(s_acc, v);
    __syncthreads();
    const int total = *s_acc;
    __syncthreads();
    if (threadIdx.x == 0)
        *s_acc = 0;
    __syncthreads();
    return total;
}

// One warp: the bin b of a 256-bin histogram (counts of keys by one byte,
// larger byte = larger key) that holds the k-th largest key, and the number of
// keys in bins above b. Lane l holds bins 8l .. 8l+7.
DDT_DEVINL void radix_pick(const int *hist, int k, int lane, int *s_bin, int *s_above)
{
    int c[8];
    int tot = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        c[i] = hist[8 * lane + i];
        tot += c[i];
    }
    int above = tot;  // keys in this lane's bins and above, then above only
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_down_sync(0xFFFFFFFFu, above, o);
        if (lane + o < 32)
            above += y;
    }
    above -= tot;
#pragma unroll
    for (int i = 7; i >= 0; --i) {
        if (above < k && above + c[i] >= k) {
            *s_bin = 8 * lane + i;
            *s_above = above;
        }
        above += c[i];
    }
}

// The row's n (max, sum of exp) pairs -> log-partition, by one warp: every
// lane loads its pairs first (one round trip), combines them, then the warp
// combines the lanes; log of the sum in fp32, the final addition in fp64.
// The pairs are another kernel's writes, read through L2.
DDT_DEVINL double row_logz(const float2 *ms, int n, int lane, int32_t *status)
{
    constexpr int PER = 16;  // pairs per lane held at once
    float M = DDT_NEG_INF, S = 0.f;
    for (int b = 0; b < n; b += 32 * PER) {
        float2 p[PER];
#pragma unroll
        for (int q = 0; q < PER; ++q) {
            const int i = b + q * 32 + lane;
            p[q] = (i < n) ? __ldcg(ms + i) : make_float2(DDT_NEG_INF, 0.f);
        }
#pragma unroll
        for (int q = 0; q < PER; ++q)
            ms_combine(M, S, p[q].x, p[q].y);
    }
    float wm = M;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        wm = fmaxf(wm, __shfl_xor_sync(0xFFFFFFFFu, wm, off));
    float t = (M != DDT_NEG_INF) ? S * ex2((M - wm) * DDT_LOG2E) : (S != S ? S : 0.f);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        t += __shfl_xor_sync(0xFFFFFFFFu, t, off);
    if (lane == 0 && t != t)
        set_status(status, DDT_DEV_NAN_LOGITS);
    return (double)wm + (double)logf(t);
}

struct SelectSmem {
    int hist[2][256];
    uint64_t key[KEY_CAP + 2];
    int grp[GRP_CAP];
    int bin, above, ngrp, nkey, acc;
    float thr;
    double lz;
};

// two radix rounds on the keys k(i), i < n (a 16-bit ordered key per item):
// the 16-bit key of the k-th largest item (every thread gets it). Most keys of a realistic row share one or two high bytes,
// so in the first round the lanes of a warp add to each bin they share once
// (a ballot loop over the warp's distinct bins); the low bytes of the second
// round are spread out, and each lane adds alone.
template <typename KeyAt>
DDT_DEVINL uint32_t radix_select16(SelectSmem &sm, int n, int k, KeyAt key_at)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    sm.hist[0][tid] = 0;
    sm.hist[1][tid] = 0;
    __syncthreads();
    for (int i0 = 0; i0 < n; i0 += TOPK_THREADS) {  // every lane takes part in the ballots
        const int i = i0 + tid;
        const uint32_t bin = (i < n) ? (key_at(i) >> 8) : 0xFFFFu;
        unsigned todo = __ballot_sync(0xFFFFFFFFu, i < n);
        while (todo) {
            const uint32_t b = __shfl_sync(0xFFFFFFFFu, bin, __ffs(todo) - 1);
            const unsigned same = __ballot_sync(0xFFFFFFFFu, bin == b) & todo;
            if (lane == __ffs(same) - 1)
                atomicAdd(&sm.hist[0][b], __popc(same));
            todo &= ~same;
        }
    }
    __syncthreads();
    if (warp == 0)
        radix_pick(sm.hist[0], k, lane, &sm.bin, &sm.above);
    __syncthreads();
    const uint32_t b1 = (uint32_t)sm.bin;
    const int k1 = k - sm.above;
    for (int i = tid; i < n; i += TOPK_THREADS) {
        const uint32_t kk = key_at(i);
        if ((kk >> 8) == b1)
            atomicAdd(&sm.hist[1][kk & 0xFFu], 1);
    }
    __syncthreads();
    if (warp == 0)
        radix_pick(sm.hist[1], k1, lane, &sm.bin, &sm.above);
    __syncthreads();
    return (b1 << 8) | (uint32_t)sm.bin;
}

// Exact fallback for flat or tied rows: the row's top-K keys into sm.key
// (returns their count, min(K, real elements)). Four radix rounds over the
// ordered 32-bit values (each a pass over the row) give the K-th largest value
// key t; the elements above t are collected in one pass, the ties at t in
// index order until K keys are held.
template <typename T>
DDT_DEVINL int exact_row_topk(const T *zrow, int V, int K, SelectSmem &sm)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0)
        sm.acc = 0;
    __syncthreads();
    uint32_t prefix = 0, pmask = 0;
    int k = K;
    int real = 0;  // non-NaN elements (counted in the first round)
    for (int round = 0; round < 4; ++round) {
        const int sh = 24 - 8 * round;
        sm.hist[0][tid] = 0;
        __syncthreads();
        int cnt = 0;
        for (int i = tid; i < V; i += TOPK_THREADS) {
            const float x = load_one(zrow, i);
            if (x == x) {
                ++cnt;
                const uint32_t kx = okey(x);
                if ((kx & pmask) == prefix)
                    atomicAdd(&sm.hist[0][(kx >> sh) & 0xFFu], 1);
            }
        }
        if (round == 0)
            real = block_sum(cnt, &sm.acc);
        if (real < K) {
            k = real;  // fewer than K real elements: take them all
            if (k == 0)
                return 0;
        }
        __syncthreads();
        if (warp == 0)
            radix_pick(sm.hist[0], k, lane, &sm.bin, &sm.above);
        __syncthreads();
        prefix |= (uint32_t)sm.bin << sh;
        pmask |= 0xFFu << sh;
        k -= sm.above;
        __syncthreads();
    }
    const uint32_t t = prefix;  // the K-th largest value key; k ties at t are needed
    const int keep = (real < K) ? real : K;
    if (tid == 0)
        sm.nkey = 0;
    __syncthreads();
    for (int i = tid; i < V; i += TOPK_THREADS) {
        const float x = load_one(zrow, i);
        if (x == x && okey(x) > t) {
            const int pos = atomicAdd(&sm.nkey, 1);
            sm.key[pos] = make_key(x, i);  // fewer than K of them
        }
    }
    __syncthreads();
    // the ties at t, lowest indices first, 256 elements at a time
    for (int b0 = 0; b0 < V; b0 += TOPK_THREADS) {
        if (sm.nkey >= keep)
            break;  // (read after a barrier: uniform)
        const int i = b0 + tid;
        float x = 0.f;
        bool tie = false;
        if (i < V) {
            x = load_one(zrow, i);
            tie = x == x && okey(x) == t;
        }
        const unsigned bal = __ballot_sync(0xFFFFFFFFu, tie);
        if (lane == 0)
            sm.hist[1][warp] = __popc(bal);
        __syncthreads();
        int before = 0;
        for (int w = 0; w < warp; ++w)
            before += sm.hist[1][w];
        before += __popc(bal & ((1u << lane) - 1u));
        const int base = sm.nkey;
        __syncthreads();
        if (tie && base + before < keep)
            sm.key[base + before] = make_key(x, i);
        if (tid == 0) {
            int tot = 0;
            for (int w = 0; w < NWARP; ++w)
                tot += sm.hist[1][w];
            sm.nkey = min(keep, base + tot);
        }
        __syncthreads();
    }
    return sm.nkey;
}

template <typename T, bool ALIGNED>
__global__ void __launch_bounds__(TOPK_THREADS, TOPK_CTAS_PER_SM)
topk_chunk_kernel(const T *__restrict__ z, int V, int nch, int Q, int pf_dist,
                  uint16_t *__restrict__ gkey, uint16_t *__restrict__ wtop,
                  float2 *__restrict__ part_ms)
{
    constexpr int VE = Elem<T>::VE;
    constexpr int CH = TOPK_THREADS * NV * VE;
    const int chunk = blockIdx.x, row = blockIdx.y;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const T *zrow = z + (int64_t)row * V;
    const int c0 = chunk * CH;
    const int cn = min(CH, V - c0);

    // ---- the chunk of the CTA about one wave later into L2 (CTAs start in
    // order of their linear index), so that its loads hit L2
    const int slot = row * nch + chunk;  // rows * chunks < 2^31 (R_max * L * 64)
    if (ALIGNED && tid == 0 && pf_dist > 0) {
        const int b2 = slot + pf_dist;
        if (b2 < (int)gridDim.y * nch) {
            const int r2 = b2 / nch, c2 = b2 - r2 * nch;
            const int n2 = min(CH, V - c2 * CH);
            prefetch_l2(z + (int64_t)r2 * V + c2 * CH, (uint32_t)(n2 * sizeof(T)));
        }
    }
    // ---- this thread's group (coalesced: consecutive threads, consecutive 16 B)
    uint4 raw[NV];
#pragma unroll
    for (int j = 0; j < NV; ++j) {
        const int e0 = (j * TOPK_THREADS + tid) * VE;
        if (ALIGNED) {
            if (e0 < cn)
                raw[j] = ldg_stream(zrow + c0 + e0);
            else
                raw[j] = make_uint4(Elem<T>::NEG_INF_FILL, Elem<T>::NEG_INF_FILL,
                                    Elem<T>::NEG_INF_FILL, Elem<T>::NEG_INF_FILL);
        } else {
            raw[j] = load_scalar<T>(zrow + c0 + e0, e0 < cn ? min(VE, cn - e0) : 0);
        }
    }
    // ---- pass 1: the group max (never NaN: the max instructions drop NaN operands)
    float m;
    if constexpr (sizeof(T) == 2) {
        uint32_t M2 = 0xFF80FF80u;
#pragma unroll
        for (int j = 0; j < NV; ++j)
            M2 = bf16x2_max(M2, bf16x2_max(bf16x2_max(raw[j].x, raw[j].y),
                                           bf16x2_max(raw[j].z, raw[j].w)));
        m = fmaxf(bf16lo(M2), bf16hi(M2));
    } else {
        m = DDT_NEG_INF;
#pragma unroll
        for (int j = 0; j < NV; ++j)
            m = fmaxf(m, vec_max<T>(raw[j]));
    }
    // ---- the group's key
    const uint32_t mk = okey(m) >> 16;
    gkey[slot * TOPK_THREADS + tid] = (uint16_t)mk;
    // ---- pass 2: sum of exp relative to the group max
    float s = 0.f;
    if (m != DDT_NEG_INF) {
        const float nb = -m * DDT_LOG2E;
        if constexpr (sizeof(T) == 2) {
            const uint64_t c2 = f2pack(DDT_LOG2E, DDT_LOG2E), b2 = f2pack(nb, nb);
            uint64_t acc0 = f2pack(0.f, 0.f), acc1 = acc0;
#pragma unroll
            for (int j = 0; j < NV; ++j) {
                acc0 = f2add(acc0, exp_pair(raw[j].x, c2, b2));
                acc1 = f2add(acc1, exp_pair(raw[j].y, c2, b2));
                acc0 = f2add(acc0, exp_pair(raw[j].z, c2, b2));
                acc1 = f2add(acc1, exp_pair(raw[j].w, c2, b2));
            }
            float a0, a1, a2, a3;
            f2unpack(acc0, a0, a1);
            f2unpack(acc1, a2, a3);
            s = (a0 + a1) + (a2 + a3);
        } else {
#pragma unroll
            for (int j = 0; j < NV; ++j)
#pragma unroll
                for (int e = 0; e < VE; ++e)
                    s += ex2(fmaf(Elem<T>::get(raw[j], e), DDT_LOG2E, nb));
        }
    }
    // ---- the warp's Q largest group keys (one per lane q < Q, found by
    // removing the warp's largest key Q - 1 times)
    {
        uint32_t k = mk, mine = 0;
        for (int q = 0; q < Q; ++q) {
            const uint32_t top = __reduce_max_sync(0xFFFFFFFFu, k);
            if (lane == q)
                mine = top;
            const unsigned holders = __ballot_sync(0xFFFFFFFFu, k == top);
            if (lane == __ffs(holders) - 1)
                k = 0;  // below every real key
        }
        if (lane < Q)
            wtop[(slot * NWARP + warp) * Q + lane] = (uint16_t)mine;
    }
    // ---- the warp's (max, sum of exp); no barrier anywhere in this kernel
    float mm = m;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        mm = fmaxf(mm, __shfl_xor_sync(0xFFFFFFFFu, mm, off));
    float ss = (m != DDT_NEG_INF) ? s * ex2((m - mm) * DDT_LOG2E) : (s != s ? s : 0.f);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        ss += __shfl_xor_sync(0xFFFFFFFFu, ss, off);
    if (lane == 0)
        part_ms[slot * NWARP + warp] = make_float2(mm, ss);
}

// One CTA per row, after the chunk kernel (programmatic dependent launch).
// The row's warp top-Q keys and all its group keys are staged in shared
// memory with one round of 16-byte loads. T is the K-th largest of the warps'
// top-Q keys: a subset of the group maxima, so T is a valid bound, and with Q
// chosen so that the subset holds at least 2K keys it almost always equals the
// K-th largest group max. The candidate groups are every group whose key
// reaches T.
template <typename T, bool ALIGNED>
__global__ void __launch_bounds__(TOPK_THREADS)
topk_select_kernel(const T *__restrict__ z, int V, int K, int nch, int Q,
                   const uint16_t *__restrict__ gkey, const uint16_t *__restrict__ wtop,
                   const float2 *__restrict__ part_ms, float *__restrict__ top_lp,
                   int32_t *__restrict__ top_ids, int32_t *__restrict__ status)
{
    constexpr int VE = Elem<T>::VE;
    constexpr int CH = TOPK_THREADS * NV * VE;
    const int row = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const T *zrow = z + (int64_t)row * V;
    const int G = nch * TOPK_THREADS;  // groups of the row
    const int NT = nch * NWARP * Q;    // warp top-Q keys of the row
    __shared__ SelectSmem sm;
    extern __shared__ uint4 s_dyn[];   // [G / 8] group keys, then [NT] top-Q keys
    const uint16_t *gk = reinterpret_cast<const uint16_t *>(s_dyn);
    uint16_t *tq = reinterpret_cast<uint16_t *>(s_dyn + G / 8);
    pdl_wait();  // the chunk kernel's keys and (max, sum) pairs are visible

    // ---- stage the keys (one round of loads), logZ by the last warp meanwhile
    const uint4 *rk4 = reinterpret_cast<const uint4 *>(gkey + (int64_t)row * G);
    for (int i = tid; i < G / 8; i += TOPK_THREADS)
        s_dyn[i] = __ldcg(rk4 + i);
    const uint16_t *rt = wtop + (int64_t)row * NT;
    for (int i = tid; i < NT; i += TOPK_THREADS)
        tq[i] = __ldcg(rt + i);
    if (warp == NWARP - 1) {
        const double lz = row_logz(part_ms + (int64_t)row * nch * NWARP, nch * NWARP, lane, status);
        if (lane == 0)
            sm.lz = lz;
    }
    if (tid == 0) {
        sm.ngrp = 0;
        sm.nkey = 0;
    }
    __syncthreads();

    // ---- T: the K-th largest of the warps' top-Q keys
    const uint32_t t16 = radix_select16(sm, NT, K, [&](int i) { return (uint32_t)tq[i]; });
    float thr;
    if constexpr (sizeof(T) == 2) {
        // the K-th largest of those group maxima itself (a bf16 value)
        thr = __uint_as_float(((t16 & 0x8000u) ? (t16 & 0x7FFFu) : (~t16 & 0xFFFFu)) << 16);
    } else {
        // the lowest value of its 16-bit bin (the -inf bin's lowest is -inf)
        thr = okey_val(t16 << 16);
        if (thr != thr)
            thr = DDT_NEG_INF;
    }
    // ---- candidate groups: every group whose key reaches T (8 keys at a time)
    const uint32_t t2 = t16 | (t16 << 16);
    for (int i = tid; i < G / 8; i += TOPK_THREADS) {
        const uint4 q = s_dyn[i];
        const uint32_t c[4] = {__vcmpgeu2(q.x, t2), __vcmpgeu2(q.y, t2), __vcmpgeu2(q.z, t2),
                               __vcmpgeu2(q.w, t2)};
        if ((c[0] | c[1] | c[2] | c[3]) != 0u) {
#pragma unroll
            for (int h = 0; h < 8; ++h) {
                if ((c[h >> 1] >> (16 * (h & 1))) & 1u) {
                    const int pos = atomicAdd(&sm.ngrp, 1);
                    if (pos < GRP_CAP)
                        sm.grp[pos] = 8 * i + h;
                }
            }
        }
    }
    __syncthreads();
    const int ngrp = sm.ngrp;
    // ---- their elements >= T, one 16-byte vector per thread (re-read, mostly from L2)
    if (ngrp <= GRP_CAP) {
        for (int it = tid; it < ngrp * NV; it += TOPK_THREADS) {
            const int g = sm.grp[it / NV], j = it % NV;
            const int e0 = (g / TOPK_THREADS) * CH + (j * TOPK_THREADS + g % TOPK_THREADS) * VE;
            if (e0 >= V)
                continue;
            const uint4 r = ALIGNED ? __ldg(reinterpret_cast<const uint4 *>(zrow + e0))
                                    : load_scalar<T>(zrow + e0, min(VE, V - e0));
            uint32_t hit = 0;
#pragma unroll
            for (int e = 0; e < VE; ++e)
                hit |= (Elem<T>::get(r, e) >= thr && e0 + e < V) ? (1u << e) : 0u;
            if (hit) {
                int pos = atomicAdd(&sm.nkey, __popc(hit));
                while (hit) {
                    const int e = __ffs(hit) - 1;
                    hit &= hit - 1;
                    if (pos < KEY_CAP)
                        sm.key[pos] = make_key(Elem<T>::get(r, e), e0 + e);
                    ++pos;
                }
            }
        }
    }
    __syncthreads();
    int nk = sm.nkey;
    if (ngrp > GRP_CAP || nk > KEY_CAP) {
        __syncthreads();
        nk = exact_row_topk<T>(zrow, V, K, sm);
    }
    // ---- ranks by counting
    if (tid == 0 && (nk & 1))
        sm.key[nk] = 0ull;  // pads an odd count (a zero key beats nothing)
    __syncthreads();
    const double logz = sm.lz;
    float *olp = top_lp + (int64_t)row * K;
    int32_t *oid = top_ids + (int64_t)row * K;
    const int n2 = (nk + 1) & ~1;
    for (int i = tid; i < nk; i += TOPK_THREADS) {
        const uint64_t ki = sm.key[i];
        const int rank = count_beating(sm.key, n2, ki);
        if (rank < K) {
            olp[rank] = (float)((double)key_val(ki) - logz);
            oid[rank] = key_idx(ki);
        }
    }
    for (int r = nk + tid; r < K; r += TOPK_THREADS) {  // fewer than K elements: padding
        olp[r] = DDT_NEG_INF;
        oid[r] = -1;
    }
}

template <typename T>
cudaError_t launch_chunks(const void *z, int rows, int V, int K, int nch, int num_sms,
                          uint16_t *gkey, uint16_t *wtop, float2 *part_ms, float *top_lp,
                          int32_t *top_ids, int32_t *status, cudaStream_t s)
{
    const bool aligned = ((int64_t)V * (int64_t)sizeof(T)) % 16 == 0 && ((uintptr_t)z % 16) == 0;
    const int pf = TOPK_CTAS_PER_SM * num_sms;  // one wave of resident CTAs
    const int Q = topk_warp_keys(nch, K);
    dim3 grid(nch, rows);
    if (aligned)
        topk_chunk_kernel<T, true><<<grid, TOPK_THREADS, 0, s>>>((const T *)z, V, nch, Q, pf,
                                                                  gkey, wtop, part_ms);
    else
        topk_chunk_kernel<T, false><<<grid, TOPK_THREADS, 0, s>>>((const T *)z, V, nch, Q, pf,
                                                                   gkey, wtop, part_ms);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return e;
    // the row selection, launched while the chunks finish; it waits for them
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3(rows);
    lc.blockDim = dim3(TOPK_THREADS);
    lc.dynamicSmemBytes = (size_t)nch * TOPK_THREADS * sizeof(uint16_t) +
                          (size_t)nch * NWARP * Q * sizeof(uint16_t);
    lc.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    lc.attrs = attr;
    lc.numAttrs = 1;
    const T *zt = (const T *)z;
    const uint16_t *gk = gkey, *wt = wtop;
    const float2 *pm = part_ms;
    e = aligned ? cudaLaunchKernelEx(&lc, topk_select_kernel<T, true>, zt, V, K, nch, Q, gk, wt,
                                     pm, top_lp, top_ids, status)
                : cudaLaunchKernelEx(&lc, topk_select_kernel<T, false>, zt, V, K, nch, Q, gk, wt,
                                     pm, top_lp, top_ids, status);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

int topk_chunk_elems(int dtype)
{
    return TOPK_THREADS * NV * (dtype == DDT_BF16 ? 8 : 4);
}

int topk_warp_keys(int nch, int K)
{
    // at least 4 per warp, and the row's warps together hold at least 2K keys
    const int per = (K + NWARP * nch - 1) / (NWARP * nch);
    const int q = 2 * per > 4 ? 2 * per : 4;
    return q < 32 ? q : 32;
}

cudaError_t launch_topk_scratch(const void *z, int dtype, int rows, int V, int K, int nch,
                                int num_sms, uint16_t *gkey, uint16_t *wtop, float2 *part_ms,
                                float *top_lp, int32_t *top_ids, int32_t *status, cudaStream_t s)
{
    if (rows == 0)
        return cudaSuccess;
    if (dtype == DDT_BF16)
        return launch_chunks<uint16_t>(z, rows, V, K, nch, num_sms, gkey, wtop, part_ms, top_lp,
                                       top_ids, status, s);
    return launch_chunks<float>(z, rows, V, K, nch, num_sms, gkey, wtop, part_ms, top_lp, top_ids,
                                status, s);
}

cudaError_t launch_topk(const ddt_ctx *c, const void *z, int R, float *top_lp, int32_t *top_ids,
                        cudaStream_t s)
{
    const ddt_config &cfg = c->cfg;
    return launch_topk_scratch(z, cfg.draft_dtype, R * cfg.L, cfg.V, cfg.K, c->tk_nch, c->num_sms,
                               c->tk_gkey, c->tk_wtop, c->tk_ms, top_lp, top_ids, c->status, s);
}
