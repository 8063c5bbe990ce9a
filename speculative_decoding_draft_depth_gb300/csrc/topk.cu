// topk.cu -- a1: per-depth log-softmax and top-K over the vocabulary.
//
// "SparklingTree: 30-40% faster speculative decoding over DSpark", Step 1
// (top-K of each depth row of the drafter's marginals and the row's
// logsumexp; log-probs are logits minus logsumexp) and "DDTree Explained
// ...", section 3, Lemma 1 (K = min(B, |V|) keeps the optimal tree).
//
// Design (HBM-bound: each logit is read once):
//  * A row of V logits is cut into chunks of TOPK_THREADS * 8 vectors of
//    16 bytes; one CTA per (chunk, row). Each thread keeps its 8 vectors in
//    registers: pass 1 takes its max, pass 2 sums exp2((x - max) * log2 e)
//    on the MUFU unit; the CTA combines (max, sum) pairs with shuffles.
//  * Candidate filter: every lane's max is a distinct element of the chunk,
//    so if each of the 8 warps finds its ceil(K/8)-th largest lane max, the
//    smallest of those, T0, has at least K chunk elements >= T0 and no
//    element of the chunk's top-K lies below it. Only threads whose max is
//    >= T0 scan their registers; survivors go to a shared buffer.
//  * The exact order (value desc, token id asc) is decided by counting, for
//    each survivor, how many survivors beat it. If the filter lets through
//    too many (flat or heavily tied rows), an exact bitwise search over the
//    ordered 32-bit keys and the chunk-local index picks exactly K.
//  * A merge kernel (one warp per row) combines the per-chunk sorted lists
//    (bitonic merges for K <= 32, binary-search ranks above) and the
//    per-chunk (max, sum) pairs into logZ (final step in fp64), then writes
//    lp = z - logZ. A row that fits one chunk is finished by its chunk CTA.
#include <stdint.h>

#include "ddt_device.cuh"
#include "ddt_internal.h"
#include "logit_vec.cuh"

namespace {

constexpr int NV = TOPK_VEC_PER_THREAD;
constexpr int SELECT_MAX = 512;  // above this many survivors, use the exact search
constexpr int VEC_CAP = 512;     // staged candidate vectors (more: the exact search)
constexpr int IDX_PAD = 0x7FFFFFFF;  // id of a padding entry in a chunk list

// total ordering key of a finite float (-0 == +0); larger float -> larger key
DDT_DEVINL uint32_t okey(float x)
{
    const uint32_t b = __float_as_uint(x + 0.0f);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// candidate key: ordered value in the high word, complemented token id in the
// low word (a lower id wins a tie); a larger key beats a smaller one
DDT_DEVINL uint64_t make_key(float v, int idx)
{
    return ((uint64_t)okey(v) << 32) | (uint32_t)~(uint32_t)idx;
}
DDT_DEVINL float key_val(uint64_t k)
{
    const uint32_t h = (uint32_t)(k >> 32);
    return (h & 0x80000000u) ? __uint_as_float(h & 0x7FFFFFFFu) : __uint_as_float(~h);
}
DDT_DEVINL int key_idx(uint64_t k) { return (int)~(uint32_t)k; }

// exclusive prefix sum over the lanes of a warp
DDT_DEVINL int warp_excl_scan(int v, int lane)
{
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xFFFFFFFFu, x, o);
        if (lane >= o)
            x += y;
    }
    return x - v;
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

template <typename T, bool ALIGNED>
__global__ void __launch_bounds__(TOPK_THREADS, 4)
topk_chunk_kernel(const T *__restrict__ z, int V, int K, int nch, float *__restrict__ part_val,
                  int32_t *__restrict__ part_idx, float2 *__restrict__ part_ms,
                  float *__restrict__ top_lp,
                  int32_t *__restrict__ top_ids, int32_t *__restrict__ status)
{
    constexpr int VE = Elem<T>::VE;
    constexpr int CH = TOPK_THREADS * NV * VE;
    const int chunk = blockIdx.x, row = blockIdx.y;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const T *zrow = z + (int64_t)row * V;
    const int c0 = chunk * CH;
    const int cn = min(CH, V - c0);

    __shared__ uint64_t s_key[TOPK_CAND_CAP];
    __shared__ float s_wm[TOPK_THREADS / 32], s_ws[TOPK_THREADS / 32], s_wt[TOPK_THREADS / 32];
    __shared__ uint4 s_vec[VEC_CAP];
    __shared__ int s_vbase[VEC_CAP];
    __shared__ int s_count, s_acc, s_nvec;
    __shared__ double s_logz;
    __shared__ uint32_t s_lmax[TOPK_THREADS];  // lane max keys (K > 32)
    __shared__ uint32_t s_t0;

    // ---- load this thread's vectors (coalesced: consecutive threads, consecutive 16 B)
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
    if (tid == 0) {
        s_count = 0;
        s_acc = 0;
        s_nvec = 0;
    }

    // ---- pass 1: thread max; pass 2: sum of exp relative to it
    float m = DDT_NEG_INF;
#pragma unroll
    for (int j = 0; j < NV; ++j)
        m = fmaxf(m, vec_max<T>(raw[j]));
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
    const float lane_max = m;

    // ---- K > 32: the threshold is the K-th largest lane max of the CTA (each of
    // those K lanes holds a value at or above it); its rank by counting
    if (K > 32) {
        const uint32_t mk = okey(lane_max == lane_max ? lane_max : DDT_NEG_INF);
        s_lmax[tid] = mk;
        __syncthreads();
        int rank = 0;
#pragma unroll 8
        for (int t = 0; t < TOPK_THREADS; ++t) {
            const uint32_t o = s_lmax[t];
            rank += (o > mk || (o == mk && t < tid)) ? 1 : 0;
        }
        if (rank == K - 1)
            s_t0 = mk;
    }
    // ---- per-warp quota threshold: the ceil(K/8)-th largest lane max, found by
    // removing the warp's largest lane max (one lane at a time) quota - 1 times
    const int quota = (K + (TOPK_THREADS / 32) - 1) / (TOPK_THREADS / 32);
    uint32_t key = okey(lane_max == lane_max ? lane_max : DDT_NEG_INF);
    uint32_t top = __reduce_max_sync(0xFFFFFFFFu, key);
    for (int q = 1; q < quota; ++q) {
        const uint32_t holders = __ballot_sync(0xFFFFFFFFu, key == top);
        if (lane == __ffs(holders) - 1)
            key = 0u;
        top = __reduce_max_sync(0xFFFFFFFFu, key);
    }
    const float warp_t = (top & 0x80000000u) ? __uint_as_float(top & 0x7FFFFFFFu)
                                             : __uint_as_float(~top);

    // ---- CTA (max, sum): warp max by one reduction, sums rescaled to it
    const uint32_t wkey = __reduce_max_sync(0xFFFFFFFFu, okey(m == m ? m : DDT_NEG_INF));
    const float mm = (wkey & 0x80000000u) ? __uint_as_float(wkey & 0x7FFFFFFFu)
                                          : __uint_as_float(~wkey);
    float ss = (m != DDT_NEG_INF && m == m) ? s * ex2((m - mm) * DDT_LOG2E) : (s != s ? s : 0.f);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        ss += __shfl_xor_sync(0xFFFFFFFFu, ss, off);
    if (lane == 0) {
        s_wm[warp] = mm;
        s_ws[warp] = ss;
        s_wt[warp] = warp_t;
    }
    __syncthreads();
    float T0 = s_wt[0];
#pragma unroll
    for (int w = 1; w < TOPK_THREADS / 32; ++w)
        T0 = fminf(T0, s_wt[w]);
    if (K > 32) {
        const uint32_t t0 = s_t0;
        T0 = (t0 & 0x80000000u) ? __uint_as_float(t0 & 0x7FFFFFFFu) : __uint_as_float(~t0);
    }
    float cm = DDT_NEG_INF, cs = 0.f;  // the chunk's (max, sum): thread 0 only
    if (tid == 0) {
        cm = s_wm[0];
        cs = s_ws[0];
        for (int w = 1; w < TOPK_THREADS / 32; ++w)
            ms_combine(cm, cs, s_wm[w], s_ws[w]);
    }

    // ---- survivors of the filter: vectors holding a value >= T0 are staged in
    // shared memory (one atomic per warp), then expanded element by element by
    // the whole CTA; survivors are kept as 64-bit keys (value order, then
    // lower token id), so that "beats" is one unsigned compare
    {
        int cnt = 0;
        if (lane_max >= T0) {
#pragma unroll
            for (int j = 0; j < NV; ++j)
                cnt += (vec_max<T>(raw[j]) >= T0) ? 1 : 0;
        }
        int base = warp_excl_scan(cnt, lane);
        const int wtot = __shfl_sync(0xFFFFFFFFu, base + cnt, 31);
        int wbase = 0;
        if (lane == 31 && wtot > 0)
            wbase = atomicAdd(&s_nvec, wtot);
        base += __shfl_sync(0xFFFFFFFFu, wbase, 31);
        if (cnt > 0) {
#pragma unroll
            for (int j = 0; j < NV; ++j) {
                if (vec_max<T>(raw[j]) >= T0) {
                    if (base < VEC_CAP) {
                        s_vec[base] = raw[j];
                        s_vbase[base] = (j * TOPK_THREADS + tid) * VE;
                    }
                    ++base;
                }
            }
        }
    }
    __syncthreads();
    const int nvec = s_nvec;
    if (nvec <= VEC_CAP) {
        for (int v0 = 0; v0 < nvec; v0 += TOPK_THREADS) {
            const int v = v0 + tid;
            uint4 r = make_uint4(Elem<T>::NEG_INF_FILL, Elem<T>::NEG_INF_FILL, Elem<T>::NEG_INF_FILL,
                                 Elem<T>::NEG_INF_FILL);
            int e0 = 0;
            if (v < nvec) {
                r = s_vec[v];
                e0 = s_vbase[v];
            }
            uint32_t hit = 0;
#pragma unroll
            for (int e = 0; e < VE; ++e)
                hit |= (Elem<T>::get(r, e) >= T0 && e0 + e < cn) ? (1u << e) : 0u;
            const int cnt = __popc(hit);
            int base = warp_excl_scan(cnt, lane);
            const int wtot = __shfl_sync(0xFFFFFFFFu, base + cnt, 31);
            int wbase = 0;
            if (lane == 31 && wtot > 0)
                wbase = atomicAdd(&s_count, wtot);
            base += __shfl_sync(0xFFFFFFFFu, wbase, 31);
            while (hit) {
                const int e = __ffs(hit) - 1;
                hit &= hit - 1;
                if (base < TOPK_CAND_CAP)
                    s_key[base] = make_key(Elem<T>::get(r, e), c0 + e0 + e);
                ++base;
            }
        }
    }
    __syncthreads();
    int n = (nvec <= VEC_CAP) ? s_count : SELECT_MAX + 1;

    if (n > SELECT_MAX) {
        // ---- exact fallback (flat or heavily tied chunks): re-read the chunk
        // from global memory, find the K-th largest key t bit by bit, then
        // the lowest-index ties at t
        __syncthreads();
        const T *cz = zrow + c0;
        uint32_t t = 0;
        for (int b = 31; b >= 0; --b) {
            const uint32_t cand = t | (1u << b);
            int c = 0;
#pragma unroll 1
            for (int li = tid; li < cn; li += TOPK_THREADS) {
                const float x = load_one(cz, li);
                c += (x == x && okey(x) >= cand) ? 1 : 0;
            }
            if (block_sum(c, &s_acc) >= K)
                t = cand;
        }
        int gt = 0;
#pragma unroll 1
        for (int li = tid; li < cn; li += TOPK_THREADS) {
            const float x = load_one(cz, li);
            gt += (x == x && okey(x) > t) ? 1 : 0;
        }
        const int need = K - block_sum(gt, &s_acc);
        int I = 0;  // largest I with #(ties at chunk-local index < I) < need
        for (int b = 15; b >= 0; --b) {
            const int cand = I | (1 << b);
            int c = 0;
#pragma unroll 1
            for (int li = tid; li < cn && li < cand; li += TOPK_THREADS) {
                const float x = load_one(cz, li);
                c += (x == x && okey(x) == t) ? 1 : 0;
            }
            if (block_sum(c, &s_acc) < need)
                I = cand;
        }
        if (tid == 0)
            s_count = 0;
        __syncthreads();
#pragma unroll 1
        for (int li = tid; li < cn; li += TOPK_THREADS) {
            const float x = load_one(cz, li);
            if (x == x) {
                const uint32_t kx = okey(x);
                if (kx > t || (kx == t && li <= I)) {
                    const int pos = atomicAdd(&s_count, 1);
                    s_key[pos] = make_key(x, c0 + li);
                }
            }
        }
        __syncthreads();
        n = s_count;
    }

    // ---- exact ranks of the survivors -> this chunk's sorted top-K
    const bool single = (nch == 1);
    float *pv = part_val + ((int64_t)row * nch + chunk) * K;
    int32_t *pi = part_idx + ((int64_t)row * nch + chunk) * K;
    if (single && tid == 0) {
        if (cs != cs)
            set_status(status, DDT_DEV_NAN_LOGITS);
        s_logz = (double)cm + log((double)cs);
    }
    __syncthreads();
    // four threads per survivor, each counting a quarter of the survivors that beat it
    for (int i0 = 0; i0 < n; i0 += TOPK_THREADS / 4) {
        const int i = i0 + (tid >> 2);
        const bool have = i < n;
        const uint64_t ki = have ? s_key[i] : 0ull;
        int rank = 0;
        if (have) {
#pragma unroll 4
            for (int jx = tid & 3; jx < n; jx += 4)
                rank += (s_key[jx] > ki) ? 1 : 0;
        }
        rank += __shfl_xor_sync(0xFFFFFFFFu, rank, 1);
        rank += __shfl_xor_sync(0xFFFFFFFFu, rank, 2);
        if (have && (tid & 3) == 0 && rank < K) {
            const float vi = key_val(ki);
            const int ii = key_idx(ki);
            if (single) {
                top_lp[(int64_t)row * K + rank] = (float)((double)vi - s_logz);
                top_ids[(int64_t)row * K + rank] = ii;
            } else {
                pv[rank] = vi;
                pi[rank] = ii;
            }
        }
    }
    for (int rank = n + tid; rank < K; rank += TOPK_THREADS) {
        if (single) {
            top_lp[(int64_t)row * K + rank] = DDT_NEG_INF;
            top_ids[(int64_t)row * K + rank] = -1;
        } else {
            pv[rank] = DDT_NEG_INF;
            pi[rank] = IDX_PAD;
        }
    }
    if (!single && tid == 0)
        part_ms[(int64_t)row * nch + chunk] = make_float2(cm, cs);
}

// ---------------------------------------------------------------- row merge
// One warp per row: the row's log-partition from the chunks' (max, sum) pairs
// (final step in fp64), and its top-K from the chunks' sorted lists.
// K <= 32: the running top-32 (one key per lane, descending) absorbs each
// list by a bitonic merge (max against the reversed list, then five
// half-cleaner steps). K > 32: every entry's rank by binary search in the
// other lists.
DDT_DEVINL uint64_t shfl_xor64(uint64_t v, int m)
{
    const uint32_t lo = __shfl_xor_sync(0xFFFFFFFFu, (uint32_t)v, m);
    const uint32_t hi = __shfl_xor_sync(0xFFFFFFFFu, (uint32_t)(v >> 32), m);
    return ((uint64_t)hi << 32) | lo;
}

constexpr int MERGE_LISTS = 16;  // chunk lists a warp stages in shared memory

__global__ void __launch_bounds__(256)
topk_merge_kernel(const float *__restrict__ part_val, const int32_t *__restrict__ part_idx,
                  const float2 *__restrict__ part_ms, int rows, int nch, int K,
                  float *__restrict__ top_lp, int32_t *__restrict__ top_ids,
                  int32_t *__restrict__ status)
{
    __shared__ uint64_t s_merge[8 * MERGE_LISTS * 32];
    const int lane = threadIdx.x & 31;
    const int row = blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
    if (row >= rows)
        return;
    // ---- log-partition
    float M = DDT_NEG_INF, S = 0.f;
    for (int c0 = 0; c0 < nch; c0 += 32) {
        const int c = c0 + lane;
        float2 ms = make_float2(DDT_NEG_INF, 0.f);
        if (c < nch)
            ms = part_ms[(int64_t)row * nch + c];
        float wm = ms.x;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
            wm = fmaxf(wm, __shfl_xor_sync(0xFFFFFFFFu, wm, off));
        float t = (ms.x != DDT_NEG_INF) ? ms.y * ex2((ms.x - wm) * DDT_LOG2E) : (ms.y != ms.y ? ms.y : 0.f);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
            t += __shfl_xor_sync(0xFFFFFFFFu, t, off);
        ms_combine(M, S, wm, t);
    }
    if (lane == 0 && S != S)
        set_status(status, DDT_DEV_NAN_LOGITS);
    const double logz = (double)M + log((double)S);
    const float *rv = part_val + (int64_t)row * nch * K;
    const int32_t *ri = part_idx + (int64_t)row * nch * K;
    float *olp = top_lp + (int64_t)row * K;
    int32_t *oid = top_ids + (int64_t)row * K;

    if (K <= 32 && nch <= MERGE_LISTS) {
        // the row's lists into shared memory first (one round of loads), then
        // absorb them one by one
        uint64_t *sk = s_merge + (threadIdx.x >> 5) * MERGE_LISTS * 32;
        for (int i = lane; i < nch * 32; i += 32) {
            const int b = i >> 5, e = i & 31;
            sk[i] = (e < K) ? make_key(rv[b * K + e], ri[b * K + e]) : 0ull;
        }
        __syncwarp();
        uint64_t cur = sk[lane];
        for (int b = 1; b < nch; ++b) {
            const uint64_t o = sk[b * 32 + 31 - lane];  // the list reversed: ascending
            cur = cur > o ? cur : o;
#pragma unroll
            for (int j = 16; j > 0; j >>= 1) {
                const uint64_t p = shfl_xor64(cur, j);
                cur = (lane & j) ? (cur < p ? cur : p) : (cur > p ? cur : p);
            }
        }
        if (lane < K) {
            const int id = key_idx(cur);
            const bool pad = (cur == 0ull) || id == IDX_PAD;
            olp[lane] = pad ? DDT_NEG_INF : (float)((double)key_val(cur) - logz);
            oid[lane] = pad ? -1 : id;
        }
    } else {
        for (int r = lane; r < K; r += 32) {  // unfilled ranks: padding
            olp[r] = DDT_NEG_INF;
            oid[r] = -1;
        }
        __syncwarp();
        for (int i = lane; i < nch * K; i += 32) {
            const int a = i / K, rho = i - a * K;
            const uint64_t ki = make_key(rv[i], ri[i]);
            if (key_idx(ki) == IDX_PAD)
                continue;
            int rank = rho;
            for (int b = 0; b < nch && rank < K; ++b) {
                if (b == a)
                    continue;
                int lo = 0, hi = K;  // entries of list b that beat entry i
                while (lo < hi) {
                    const int mid = (lo + hi) >> 1;
                    if (make_key(rv[b * K + mid], ri[b * K + mid]) > ki)
                        lo = mid + 1;
                    else
                        hi = mid;
                }
                rank += lo;
            }
            if (rank < K) {
                olp[rank] = (float)((double)key_val(ki) - logz);
                oid[rank] = key_idx(ki);
            }
        }
    }
}

}  // namespace

namespace {
// rows with K > 32: one CTA per row, the chunk lists staged in shared memory;
// every entry's rank is its rank in its own list plus, per other list, the
// number of entries that beat it (a binary search)
constexpr int WIDE_THREADS = 256;

__global__ void __launch_bounds__(WIDE_THREADS)
topk_merge_wide_kernel(const float *__restrict__ part_val, const int32_t *__restrict__ part_idx,
                       const float2 *__restrict__ part_ms, int nch, int K,
                       float *__restrict__ top_lp, int32_t *__restrict__ top_ids,
                       int32_t *__restrict__ status)
{
    extern __shared__ uint64_t s_keys[];  // [nch * K]
    __shared__ double s_lz;
    __shared__ int s_nreal;
    const int row = blockIdx.x, tid = threadIdx.x;
    const int n = nch * K;
    const float *rv = part_val + (int64_t)row * n;
    const int32_t *ri = part_idx + (int64_t)row * n;
    if (tid == 0)
        s_nreal = 0;
    __syncthreads();
    int real = 0;
    for (int i = tid; i < n; i += WIDE_THREADS) {
        const int id = ri[i];
        s_keys[i] = (id == IDX_PAD) ? 0ull : make_key(rv[i], id);
        real += (id == IDX_PAD) ? 0 : 1;
    }
    if (tid < 32) {  // log-partition over the chunks' (max, sum) pairs
        float M = DDT_NEG_INF, S = 0.f;
        for (int c0 = 0; c0 < nch; c0 += 32) {
            const int c = c0 + tid;
            float2 ms = make_float2(DDT_NEG_INF, 0.f);
            if (c < nch)
                ms = part_ms[(int64_t)row * nch + c];
            float wm = ms.x;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1)
                wm = fmaxf(wm, __shfl_xor_sync(0xFFFFFFFFu, wm, off));
            float t = (ms.x != DDT_NEG_INF) ? ms.y * ex2((ms.x - wm) * DDT_LOG2E)
                                            : (ms.y != ms.y ? ms.y : 0.f);
#pragma unroll
            for (int off = 16; off > 0; off >>= 1)
                t += __shfl_xor_sync(0xFFFFFFFFu, t, off);
            ms_combine(M, S, wm, t);
        }
        if (tid == 0) {
            if (S != S)
                set_status(status, DDT_DEV_NAN_LOGITS);
            s_lz = (double)M + log((double)S);
        }
    }
    atomicAdd(&s_nreal, real);
    __syncthreads();
    const double logz = s_lz;
    float *olp = top_lp + (int64_t)row * K;
    int32_t *oid = top_ids + (int64_t)row * K;
    const int filled = s_nreal < K ? s_nreal : K;
    for (int r = filled + tid; r < K; r += WIDE_THREADS) {  // unfilled ranks: padding
        olp[r] = DDT_NEG_INF;
        oid[r] = -1;
    }
    for (int i = tid; i < n; i += WIDE_THREADS) {
        const uint64_t ki = s_keys[i];
        if (ki == 0ull)
            continue;
        const int a = i / K, rho = i - a * K;
        int rank = rho;
        for (int b = 0; b < nch && rank < K; ++b) {
            if (b == a)
                continue;
            const uint64_t *lb = s_keys + b * K;
            int lo = 0, hi = K;  // entries of list b that beat entry i (lists descend; pads are 0)
            while (lo < hi) {
                const int mid = (lo + hi) >> 1;
                if (lb[mid] > ki)
                    lo = mid + 1;
                else
                    hi = mid;
            }
            rank += lo;
        }
        if (rank < K) {
            olp[rank] = (float)((double)key_val(ki) - logz);
            oid[rank] = key_idx(ki);
        }
    }
}
}  // namespace

namespace {
cudaError_t launch_merge(int rows, int V, int K, int nch, const float *part_val,
                         const int32_t *part_idx, const float2 *part_ms, float *top_lp,
                         int32_t *top_ids, int32_t *status, cudaStream_t s)
{
    (void)V;
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || nch == 1 || rows == 0)
        return e;
    if (K > 32) {
        const size_t smem = (size_t)nch * K * sizeof(uint64_t);
        if (smem > 48 * 1024) {
            static size_t attr = 0;
            if (attr < smem) {
                if ((e = cudaFuncSetAttribute(topk_merge_wide_kernel,
                                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                                              (int)smem)) != cudaSuccess)
                    return e;
                attr = smem;
            }
        }
        topk_merge_wide_kernel<<<rows, WIDE_THREADS, smem, s>>>(part_val, part_idx, part_ms, nch,
                                                                K, top_lp, top_ids, status);
        return cudaGetLastError();
    }
    topk_merge_kernel<<<(rows + 7) / 8, 256, 0, s>>>(part_val, part_idx, part_ms, rows, nch, K,
                                                     top_lp, top_ids, status);
    return cudaGetLastError();
}
}  // namespace

int topk_chunk_elems(int dtype)
{
    return TOPK_THREADS * NV * (dtype == DDT_BF16 ? 8 : 4);
}

cudaError_t launch_topk(const ddt_ctx *c, const void *z, int R, float *top_lp, int32_t *top_ids,
                        cudaStream_t s)
{
    const ddt_config &cfg = c->cfg;
    const int rows = R * cfg.L;
    dim3 grid(c->tk_nch, rows);
    const bool bf16 = cfg.draft_dtype == DDT_BF16;
    const int esz = bf16 ? 2 : 4;
    const bool aligned = ((int64_t)cfg.V * esz) % 16 == 0 && ((uintptr_t)z % 16) == 0;
    if (bf16) {
        if (aligned)
            topk_chunk_kernel<uint16_t, true><<<grid, TOPK_THREADS, 0, s>>>(
                (const uint16_t *)z, cfg.V, cfg.K, c->tk_nch, c->tk_val, c->tk_idx, c->tk_ms,
                top_lp, top_ids, c->status);
        else
            topk_chunk_kernel<uint16_t, false><<<grid, TOPK_THREADS, 0, s>>>(
                (const uint16_t *)z, cfg.V, cfg.K, c->tk_nch, c->tk_val, c->tk_idx, c->tk_ms,
                top_lp, top_ids, c->status);
    } else {
        if (aligned)
            topk_chunk_kernel<float, true><<<grid, TOPK_THREADS, 0, s>>>(
                (const float *)z, cfg.V, cfg.K, c->tk_nch, c->tk_val, c->tk_idx, c->tk_ms,
                top_lp, top_ids, c->status);
        else
            topk_chunk_kernel<float, false><<<grid, TOPK_THREADS, 0, s>>>(
                (const float *)z, cfg.V, cfg.K, c->tk_nch, c->tk_val, c->tk_idx, c->tk_ms,
                top_lp, top_ids, c->status);
    }
    return launch_merge(rows, cfg.V, cfg.K, c->tk_nch, c->tk_val, c->tk_idx, c->tk_ms, top_lp,
                        top_ids, c->status, s);
}

cudaError_t launch_topk_scratch(const void *z, int dtype, int rows, int V, int K, int nch,
                                float *part_val, int32_t *part_idx, float2 *part_ms,
                                unsigned *cnt, float *top_lp, int32_t *top_ids, int32_t *status,
                                cudaStream_t s)
{
    dim3 grid(nch, rows);
    const bool bf16 = dtype == DDT_BF16;
    const int esz = bf16 ? 2 : 4;
    const bool aligned = ((int64_t)V * esz) % 16 == 0 && ((uintptr_t)z % 16) == 0;
    if (bf16) {
        if (aligned)
            topk_chunk_kernel<uint16_t, true><<<grid, TOPK_THREADS, 0, s>>>(
                (const uint16_t *)z, V, K, nch, part_val, part_idx, part_ms, top_lp, top_ids,
                status);
        else
            topk_chunk_kernel<uint16_t, false><<<grid, TOPK_THREADS, 0, s>>>(
                (const uint16_t *)z, V, K, nch, part_val, part_idx, part_ms, top_lp, top_ids,
                status);
    } else {
        if (aligned)
            topk_chunk_kernel<float, true><<<grid, TOPK_THREADS, 0, s>>>(
                (const float *)z, V, K, nch, part_val, part_idx, part_ms, top_lp, top_ids,
                status);
        else
            topk_chunk_kernel<float, false><<<grid, TOPK_THREADS, 0, s>>>(
                (const float *)z, V, K, nch, part_val, part_idx, part_ms, top_lp, top_ids,
                status);
    }
    return launch_merge(rows, V, K, nch, part_val, part_idx, part_ms, top_lp, top_ids, status, s);
}
