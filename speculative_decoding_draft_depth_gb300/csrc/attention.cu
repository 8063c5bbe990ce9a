// attention.cu -- a4: paged GQA attention of the tree queries under the
// ancestor mask.
//
// "SparklingTree ...", Step 4 and the verification discussion (the target
// attends to the context plus each node's ancestors in one masked pass) and
// "DDTree Explained ...", sections 5 and 8 (ancestor-only tree mask over a
// GQA target with a custom attention mask).
//
// Work decomposition (one GPU, HBM-bound on the paged KV read):
//  * Rows of one (request r, KV head g): the G = Hq/Hkv query heads of every
//    tree position, row = position * G + head, in groups of 144 rows (nine
//    m16 tiles, one warp each). Every row of a group shares the group's K/V
//    stream, so each cached K/V byte is read once per row group.
//  * A plan kernel splits each request's context into ceil(ctx/4096) nearly
//    equal chunks, orders requests by context length (longest first) and
//    writes the work list; a persistent grid pulls items with an atomic
//    counter. The last chunk of a (r, g, group) also covers the tree keys,
//    masked per row by the ancestor bitmask.
//  * K/V tiles of 64 tokens stream through a 3-stage cp.async pipeline,
//    gathered page by page through the block table, XOR-swizzled in shared
//    memory; QK^T and PV run on bf16 mma.sync with fp32 accumulation and an
//    online (running max, running sum) softmax in the base-2 domain.
//  * Chunks of a split (r, g, group) leave unnormalised partial outputs with
//    their (max, sum); the CTA that finishes last combines them.
#include <stdint.h>

#include "ddt_device.cuh"
#include "ddt_internal.h"

namespace {

constexpr int BN = ATT_BLOCK_N;
constexpr int MAX_SPLITS = 64;

DDT_DEVINL uint32_t smem_u32(const void *p)
{
    return (uint32_t)__cvta_generic_to_shared(p);
}

DDT_DEVINL void cp_async16(uint32_t dst, const void *src, int src_bytes)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(src_bytes));
}
DDT_DEVINL void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
DDT_DEVINL void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N)); }

DDT_DEVINL void ldsm_x4(uint32_t addr, uint32_t &a, uint32_t &b, uint32_t &c, uint32_t &d)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(a), "=r"(b), "=r"(c), "=r"(d)
                 : "r"(addr));
}
DDT_DEVINL void ldsm_x4_t(uint32_t addr, uint32_t &a, uint32_t &b, uint32_t &c, uint32_t &d)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(a), "=r"(b), "=r"(c), "=r"(d)
                 : "r"(addr));
}

DDT_DEVINL void mma16816(float *c, const uint32_t *a, uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// byte offset of 16-byte chunk c of row t in a swizzled tile with CPR chunks per row
template <int CPR>
DDT_DEVINL uint32_t swz(int t, int c)
{
    return (uint32_t)(t * CPR * 16 + ((c ^ (t & 7)) * 16));
}

// ---------------------------------------------------------------- plan
__global__ void att_plan_kernel(const int32_t *__restrict__ ctx_lens, int R, int Hkv, int RG,
                                int max_ctx, int4 *__restrict__ items,
                                int32_t *__restrict__ rg_base, int32_t *__restrict__ meta,
                                int32_t *__restrict__ status)
{
    extern __shared__ int sp[];
    int *s_ctx = sp, *s_ns = sp + R, *s_ord = sp + 2 * R, *s_off = sp + 3 * R;
    for (int r = threadIdx.x; r < R; r += blockDim.x) {
        int c = ctx_lens[r];
        if (c < 0 || c > max_ctx) {
            set_status(status, DDT_DEV_BAD_PAGE);
            c = c < 0 ? 0 : max_ctx;
        }
        s_ctx[r] = c;
        s_ns[r] = max(1, (c + ATT_CHUNK - 1) / ATT_CHUNK);
    }
    __syncthreads();
    for (int r = threadIdx.x; r < R; r += blockDim.x) {
        int rank = 0;
        for (int q = 0; q < R; ++q)
            rank += (s_ctx[q] > s_ctx[r] || (s_ctx[q] == s_ctx[r] && q < r)) ? 1 : 0;
        s_ord[rank] = r;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        int off = 0;
        for (int k = 0; k < R; ++k) {
            const int r = s_ord[k];
            s_off[r] = off;
            off += s_ns[r] * Hkv * RG;
        }
        meta[0] = off;
        meta[1] = 0;
    }
    __syncthreads();
    for (int r = threadIdx.x; r < R; r += blockDim.x) {
        const int ns = s_ns[r], ctx = s_ctx[r], base = s_off[r];
        const int len = ((ctx + ns - 1) / ns + 127) / 128 * 128;  // chunks start on 128-token tiles
        for (int s = 0; s < ns; ++s) {
            const int t0 = min(ctx, s * len), t1 = min(ctx, (s + 1) * len);
            for (int g = 0; g < Hkv; ++g)
                for (int rg = 0; rg < RG; ++rg) {
                    const int idx = base + (s * Hkv + g) * RG + rg;
                    items[idx] = make_int4(r, g | (rg << 8) | (s << 16), t0, t1);
                }
        }
        for (int g = 0; g < Hkv; ++g)
            for (int rg = 0; rg < RG; ++rg)
                rg_base[((int64_t)r * Hkv + g) * RG + rg] = base + g * RG + rg;
    }
}

// ---------------------------------------------------------------- attention
template <int D>
struct AttSmem {
    static constexpr int CPR = D / 8;                    // 16-byte chunks per row
    static constexpr int ROWB = D * 2;                   // bytes per row
    static constexpr int Q_BYTES = ATT_ROWS * ROWB;
    static constexpr int KV_BYTES = BN * ROWB;           // one of K or V, one stage
    static constexpr int STAGE_BYTES = 2 * KV_BYTES;
    static constexpr int FAC_BYTES = MAX_SPLITS * ATT_ROWS * 4;
    static constexpr int TOTAL = Q_BYTES + ATT_STAGES * STAGE_BYTES + FAC_BYTES + 64;
};

struct AttArgs {
    const uint16_t *q, *k_tree, *v_tree, *k_cache, *v_cache;
    const int32_t *block_table, *ctx_lens;
    const uint32_t *mask;
    float *out;
    const int4 *items;
    const int32_t *rg_base;
    int32_t *meta;
    unsigned *rg_cnt;
    float *part_o;
    float2 *part_ml;
    int32_t *status;
    int R, P, Hq, Hkv, G, W, page, max_pages, RG;
    int64_t num_pages;
    float scale_log2;  // log2(e) / sqrt(d)
};

template <int D>
__global__ void __launch_bounds__(ATT_THREADS, 1) att_mma_kernel(AttArgs a)
{
    using SM = AttSmem<D>;
    constexpr int CPR = SM::CPR;
    constexpr int KSTEPS = D / 16;
    constexpr int DTILES = D / 8;
    extern __shared__ __align__(128) unsigned char smem[];
    unsigned char *sQ = smem;
    unsigned char *sKV = smem + SM::Q_BYTES;
    float *sFac = reinterpret_cast<float *>(smem + SM::Q_BYTES + ATT_STAGES * SM::STAGE_BYTES);
    __shared__ int s_item, s_last;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int rowsPerHead = a.P * a.G;

    for (;;) {
        if (tid == 0)
            s_item = atomicAdd(&a.meta[1], 1);
        __syncthreads();
        const int item = s_item;
        if (item >= a.meta[0])
            break;
        const int4 it = a.items[item];
        const int r = it.x, g = it.y & 0xFF, rgi = (it.y >> 8) & 0xFF, sidx = it.y >> 16;
        const int t0 = it.z, t1 = it.w;
        const int ctx = min(max(a.ctx_lens[r], 0), a.max_pages * a.page);
        const int ns = max(1, (ctx + ATT_CHUNK - 1) / ATT_CHUNK);
        const bool last_split = (sidx == ns - 1);
        const int row0 = rgi * ATT_ROWS;
        const int nb_ctx = (t1 - t0 + BN - 1) / BN;
        const int nb_tree = last_split ? (a.P + BN - 1) / BN : 0;
        const int nb = nb_ctx + nb_tree;

        // ---- Q tile (cp.async, group 0)
        for (int c = tid; c < ATT_ROWS * CPR; c += ATT_THREADS) {
            const int rho = c / CPR, ch = c % CPR;
            const int gr = row0 + rho;
            const uint16_t *src = a.q;
            int bytes = 0;
            if (gr < rowsPerHead) {
                const int i = gr / a.G, hl = gr % a.G;
                src = a.q + (((int64_t)r * a.P + i) * a.Hq + g * a.G + hl) * D + ch * 8;
                bytes = 16;
            }
            cp_async16(smem_u32(sQ + swz<CPR>(rho, ch)), src, bytes);
        }

        auto load_block = [&](int b, int stage) {
            unsigned char *sK = sKV + stage * SM::STAGE_BYTES;
            unsigned char *sV = sK + SM::KV_BYTES;
            const bool tree = (b >= nb_ctx);
            const int base_t = tree ? (b - nb_ctx) * BN : t0 + b * BN;
            for (int c = tid; c < BN * CPR; c += ATT_THREADS) {
                const int row = c / CPR, ch = c % CPR;
                const uint16_t *ks = a.k_cache, *vs = a.v_cache;
                int bytes = 0;
                if (tree) {
                    const int j = base_t + row;
                    if (j < a.P) {
                        const int64_t off = (((int64_t)r * a.P + j) * a.Hkv + g) * D + ch * 8;
                        ks = a.k_tree + off;
                        vs = a.v_tree + off;
                        bytes = 16;
                    }
                } else {
                    const int t = base_t + row;
                    if (t < t1) {
                        const int pg = a.block_table[(int64_t)r * a.max_pages + t / a.page];
                        if (pg >= 0 && pg < a.num_pages) {
                            const int64_t off = (((int64_t)pg * a.page + t % a.page) * a.Hkv + g) * D + ch * 8;
                            ks = a.k_cache + off;
                            vs = a.v_cache + off;
                            bytes = 16;
                        } else if (ch == 0) {
                            set_status(a.status, DDT_DEV_BAD_PAGE);
                        }
                    }
                }
                cp_async16(smem_u32(sK + swz<CPR>(row, ch)), ks, bytes);
                cp_async16(smem_u32(sV + swz<CPR>(row, ch)), vs, bytes);
            }
        };

        // prologue: Q + first stages
        load_block(0, 0);
        cp_async_commit();
        for (int st = 1; st < ATT_STAGES - 1; ++st) {
            if (st < nb)
                load_block(st, st);
            cp_async_commit();
        }

        // this warp's rows and their mask words
        const int rho0 = warp * 16 + (lane >> 2), rho1 = rho0 + 8;
        const int gr0 = row0 + rho0, gr1 = row0 + rho1;
        const int i0 = gr0 / a.G, i1 = gr1 / a.G;
        uint32_t mk0[4] = {0u, 0u, 0u, 0u}, mk1[4] = {0u, 0u, 0u, 0u};
        if (nb_tree > 0) {
            for (int w = 0; w < a.W; ++w) {
                if (gr0 < rowsPerHead)
                    mk0[w] = a.mask[((int64_t)r * a.P + i0) * a.W + w];
                if (gr1 < rowsPerHead)
                    mk1[w] = a.mask[((int64_t)r * a.P + i1) * a.W + w];
            }
        }

        float o[DTILES][4];
#pragma unroll
        for (int i = 0; i < DTILES; ++i)
            o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
        float m0 = DDT_NEG_INF, m1 = DDT_NEG_INF, l0 = 0.f, l1 = 0.f;
        uint32_t qa[KSTEPS][4];

        for (int b = 0; b < nb; ++b) {
            cp_async_wait<ATT_STAGES - 2>();
            __syncthreads();
            {
                const int nxt = b + ATT_STAGES - 1;
                if (nxt < nb)
                    load_block(nxt, nxt % ATT_STAGES);
                cp_async_commit();
            }
            if (b == 0) {
#pragma unroll
                for (int kk = 0; kk < KSTEPS; ++kk) {
                    const int mi = lane >> 3;
                    const int row = warp * 16 + (mi & 1) * 8 + (lane & 7);
                    const int ch = kk * 2 + (mi >> 1);
                    ldsm_x4(smem_u32(sQ + swz<CPR>(row, ch)), qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3]);
                }
            }
            const unsigned char *sK = sKV + (b % ATT_STAGES) * SM::STAGE_BYTES;
            const unsigned char *sV = sK + SM::KV_BYTES;

            float sc[BN / 8][4];
#pragma unroll
            for (int i = 0; i < BN / 8; ++i)
                sc[i][0] = sc[i][1] = sc[i][2] = sc[i][3] = 0.f;
#pragma unroll
            for (int kk = 0; kk < KSTEPS; ++kk)
#pragma unroll
                for (int np = 0; np < BN / 16; ++np) {
                    const int mi = lane >> 3;
                    const int tok = np * 16 + (mi >> 1) * 8 + (lane & 7);
                    const int ch = kk * 2 + (mi & 1);
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4(smem_u32(sK + swz<CPR>(tok, ch)), b0, b1, b2, b3);
                    mma16816(sc[2 * np], qa[kk], b0, b1);
                    mma16816(sc[2 * np + 1], qa[kk], b2, b3);
                }

            // mask + scale into the log2 domain
            const bool tree = (b >= nb_ctx);
            const int base_t = tree ? (b - nb_ctx) * BN : t0 + b * BN;
            float mx0 = DDT_NEG_INF, mx1 = DDT_NEG_INF;
#pragma unroll
            for (int nt = 0; nt < BN / 8; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int tk = nt * 8 + (lane & 3) * 2 + e;
                    bool ok0, ok1;
                    if (tree) {
                        const int j = base_t + tk;
                        ok0 = j < a.P && ((mk0[j >> 5] >> (j & 31)) & 1u);
                        ok1 = j < a.P && ((mk1[j >> 5] >> (j & 31)) & 1u);
                    } else {
                        ok0 = ok1 = (base_t + tk < t1);
                    }
                    sc[nt][e] = ok0 ? sc[nt][e] * a.scale_log2 : DDT_NEG_INF;
                    sc[nt][2 + e] = ok1 ? sc[nt][2 + e] * a.scale_log2 : DDT_NEG_INF;
                    mx0 = fmaxf(mx0, sc[nt][e]);
                    mx1 = fmaxf(mx1, sc[nt][2 + e]);
                }
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xFFFFFFFFu, mx0, 1));
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xFFFFFFFFu, mx0, 2));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xFFFFFFFFu, mx1, 1));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xFFFFFFFFu, mx1, 2));
            const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
            const float base0 = (mn0 == DDT_NEG_INF) ? 0.f : mn0;
            const float base1 = (mn1 == DDT_NEG_INF) ? 0.f : mn1;
            const float al0 = ex2(m0 - base0), al1 = ex2(m1 - base1);
            m0 = mn0;
            m1 = mn1;
            float rs0 = 0.f, rs1 = 0.f;
            uint32_t pa[BN / 16][4];
#pragma unroll
            for (int nt = 0; nt < BN / 8; ++nt) {
                const float p0 = ex2(sc[nt][0] - base0), p1 = ex2(sc[nt][1] - base0);
                const float p2 = ex2(sc[nt][2] - base1), p3 = ex2(sc[nt][3] - base1);
                rs0 += p0 + p1;
                rs1 += p2 + p3;
                pa[nt >> 1][(nt & 1) * 2 + 0] = pack_bf16x2(p0, p1);
                pa[nt >> 1][(nt & 1) * 2 + 1] = pack_bf16x2(p2, p3);
            }
            l0 = l0 * al0 + rs0;
            l1 = l1 * al1 + rs1;
#pragma unroll
            for (int dn = 0; dn < DTILES; ++dn) {
                o[dn][0] *= al0;
                o[dn][1] *= al0;
                o[dn][2] *= al1;
                o[dn][3] *= al1;
            }
#pragma unroll
            for (int kt = 0; kt < BN / 16; ++kt)
#pragma unroll
                for (int dp = 0; dp < DTILES / 2; ++dp) {
                    const int mi = lane >> 3;
                    const int tok = kt * 16 + (mi & 1) * 8 + (lane & 7);
                    const int ch = dp * 2 + (mi >> 1);
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4_t(smem_u32(sV + swz<CPR>(tok, ch)), b0, b1, b2, b3);
                    mma16816(o[2 * dp], pa[kt], b0, b1);
                    mma16816(o[2 * dp + 1], pa[kt], b2, b3);
                }
        }
        cp_async_wait<0>();

        l0 += __shfl_xor_sync(0xFFFFFFFFu, l0, 1);
        l0 += __shfl_xor_sync(0xFFFFFFFFu, l0, 2);
        l1 += __shfl_xor_sync(0xFFFFFFFFu, l1, 1);
        l1 += __shfl_xor_sync(0xFFFFFFFFu, l1, 2);

        const int rg_slot = (r * a.Hkv + g) * a.RG + rgi;
        if (ns == 1) {
            const float inv0 = (l0 > 0.f) ? 1.f / l0 : 0.f, inv1 = (l1 > 0.f) ? 1.f / l1 : 0.f;
#pragma unroll
            for (int dn = 0; dn < DTILES; ++dn) {
                const int col = dn * 8 + (lane & 3) * 2;
                if (gr0 < rowsPerHead) {
                    float *dst = a.out + (((int64_t)r * a.P + i0) * a.Hq + g * a.G + gr0 % a.G) * D + col;
                    *reinterpret_cast<float2 *>(dst) = make_float2(o[dn][0] * inv0, o[dn][1] * inv0);
                }
                if (gr1 < rowsPerHead) {
                    float *dst = a.out + (((int64_t)r * a.P + i1) * a.Hq + g * a.G + gr1 % a.G) * D + col;
                    *reinterpret_cast<float2 *>(dst) = make_float2(o[dn][2] * inv1, o[dn][3] * inv1);
                }
            }
            __syncthreads();  // smem reuse by the next item
            continue;
        }

        // ---- partial result of this split
        float *po = a.part_o + (int64_t)item * ATT_ROWS * D;
#pragma unroll
        for (int dn = 0; dn < DTILES; ++dn) {
            const int col = dn * 8 + (lane & 3) * 2;
            *reinterpret_cast<float2 *>(po + rho0 * D + col) = make_float2(o[dn][0], o[dn][1]);
            *reinterpret_cast<float2 *>(po + rho1 * D + col) = make_float2(o[dn][2], o[dn][3]);
        }
        if ((lane & 3) == 0) {
            a.part_ml[(int64_t)item * ATT_ROWS + rho0] = make_float2(m0, l0);
            a.part_ml[(int64_t)item * ATT_ROWS + rho1] = make_float2(m1, l1);
        }
        __threadfence();
        __syncthreads();
        if (tid == 0)
            s_last = (atomicAdd(&a.rg_cnt[rg_slot], 1u) == (unsigned)(ns - 1));
        __syncthreads();
        if (!s_last)
            continue;
        __threadfence();

        // ---- combine the ns partials of this (r, g, row group)
        const int first = a.rg_base[rg_slot];
        const int stride = a.Hkv * a.RG;  // item distance between consecutive splits
        for (int rho = tid; rho < ATT_ROWS; rho += ATT_THREADS) {
            float M = DDT_NEG_INF;
            for (int s = 0; s < ns; ++s)
                M = fmaxf(M, __ldcg(&a.part_ml[(int64_t)(first + s * stride) * ATT_ROWS + rho]).x);
            const float base = (M == DDT_NEG_INF) ? 0.f : M;
            float Ls = 0.f;
            for (int s = 0; s < ns; ++s) {
                const float2 ml = __ldcg(&a.part_ml[(int64_t)(first + s * stride) * ATT_ROWS + rho]);
                const float f = ex2(ml.x - base);
                sFac[s * ATT_ROWS + rho] = f;
                Ls += ml.y * f;
            }
            const float inv = (Ls > 0.f) ? 1.f / Ls : 0.f;
            for (int s = 0; s < ns; ++s)
                sFac[s * ATT_ROWS + rho] *= inv;
        }
        __syncthreads();
        for (int e = tid; e < ATT_ROWS * (D / 2); e += ATT_THREADS) {
            const int rho = e / (D / 2), col = (e % (D / 2)) * 2;
            const int gr = row0 + rho;
            if (gr >= rowsPerHead)
                continue;
            float x0 = 0.f, x1 = 0.f;
            for (int s = 0; s < ns; ++s) {
                const float f = sFac[s * ATT_ROWS + rho];
                const float2 v = __ldcg(reinterpret_cast<const float2 *>(
                    a.part_o + ((int64_t)(first + s * stride) * ATT_ROWS + rho) * D + col));
                x0 += v.x * f;
                x1 += v.y * f;
            }
            const int i = gr / a.G, hl = gr % a.G;
            float *dst = a.out + (((int64_t)r * a.P + i) * a.Hq + g * a.G + hl) * D + col;
            *reinterpret_cast<float2 *>(dst) = make_float2(x0, x1);
        }
        if (tid == 0)
            a.rg_cnt[rg_slot] = 0u;
        __syncthreads();
    }
}

}  // namespace

cudaError_t launch_att_plan(const ddt_ctx *c, const int32_t *ctx_lens, int R, int RG, int max_ctx,
                            cudaStream_t s)
{
    att_plan_kernel<<<1, 256, 4 * R * sizeof(int), s>>>(ctx_lens, R, c->cfg.Hkv, RG, max_ctx,
                                                        c->att_items, c->att_rg_base, c->att_meta,
                                                        c->status);
    return cudaGetLastError();
}

cudaError_t launch_attention(const ddt_ctx *c, const uint16_t *q, const uint16_t *k_tree,
                             const uint16_t *v_tree, const uint16_t *k_cache,
                             const uint16_t *v_cache, const int32_t *block_table,
                             const int32_t *ctx_lens, const uint32_t *mask, int R, float *out,
                             cudaStream_t s)
{
    const ddt_config &cfg = c->cfg;
    if (c->att_use_tc)
        return launch_attention_tc(c, q, k_tree, v_tree, k_cache, v_cache, block_table, ctx_lens,
                                   mask, R, out, s);
    const int P = cfg.B + 1, G = cfg.Hq / cfg.Hkv;
    const int max_ctx = cfg.max_pages_per_req * cfg.page_size;
    const int RG = (P * G + ATT_ROWS - 1) / ATT_ROWS;
    cudaError_t e = launch_att_plan(c, ctx_lens, R, RG, max_ctx, s);
    if (e != cudaSuccess)
        return e;
    AttArgs a;
    a.q = q;
    a.k_tree = k_tree;
    a.v_tree = v_tree;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.block_table = block_table;
    a.ctx_lens = ctx_lens;
    a.mask = mask;
    a.out = out;
    a.items = c->att_items;
    a.rg_base = c->att_rg_base;
    a.meta = c->att_meta;
    a.rg_cnt = c->att_rg_cnt;
    a.part_o = c->att_part_o;
    a.part_ml = c->att_part_ml;
    a.status = c->status;
    a.R = R;
    a.P = P;
    a.Hq = cfg.Hq;
    a.Hkv = cfg.Hkv;
    a.G = G;
    a.W = (P + 31) / 32;
    a.page = cfg.page_size;
    a.max_pages = cfg.max_pages_per_req;
    a.RG = RG;
    a.num_pages = cfg.num_pages;
    a.scale_log2 = 1.4426950408889634f / sqrtf((float)cfg.d);
    if (cfg.d == 128) {
        const int smem = AttSmem<128>::TOTAL;
        cudaFuncSetAttribute(att_mma_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        att_mma_kernel<128><<<c->att_grid, ATT_THREADS, smem, s>>>(a);
    } else {
        const int smem = AttSmem<64>::TOTAL;
        cudaFuncSetAttribute(att_mma_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        att_mma_kernel<64><<<c->att_grid, ATT_THREADS, smem, s>>>(a);
    }
    return cudaGetLastError();
}
