// logit_vec.cuh -- 16-byte vectors of logits (8 bf16 or 4 fp32 values):
// element access, the vector's max, a scalar gather for unaligned rows and
// tails, exp pairs on packed fp32, and the (max, sum of exp) merge. Used by
// the kernels that stream logit rows (top-K, stochastic verification).
#pragma once

#include <stdint.h>

#include "ddt_device.cuh"

// 2^(x * log2 e - m * log2 e) for the two bf16 values of w (c2 = {log2 e, log2 e},
// b2 = {-m log2 e, -m log2 e}), as a packed pair
DDT_DEVINL uint64_t exp_pair(uint32_t w, uint64_t c2, uint64_t b2)
{
    float t0, t1;
    f2unpack(f2fma(f2pack(bf16lo(w), bf16hi(w)), c2, b2), t0, t1);
    return f2pack(ex2(t0), ex2(t1));
}

template <typename T> struct Elem;
template <> struct Elem<uint16_t> {
    static constexpr int VE = 8;
    static constexpr uint32_t NEG_INF_FILL = 0xFF80FF80u;
    DDT_DEVINL static float get(const uint4 &v, int e)
    {
        const uint32_t w = (e < 2) ? v.x : (e < 4) ? v.y : (e < 6) ? v.z : v.w;
        return (e & 1) ? bf16hi(w) : bf16lo(w);
    }
};
template <> struct Elem<float> {
    static constexpr int VE = 4;
    static constexpr uint32_t NEG_INF_FILL = 0xFF800000u;
    DDT_DEVINL static float get(const uint4 &v, int e)
    {
        const uint32_t w = (e == 0) ? v.x : (e == 1) ? v.y : (e == 2) ? v.z : v.w;
        return __uint_as_float(w);
    }
};

// max of one vector's elements (NaN ignored unless all are NaN)
DDT_DEVINL uint32_t bf16x2_max(uint32_t a, uint32_t b)
{
    uint32_t r;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}
template <typename T>
DDT_DEVINL float vec_max(const uint4 &v)
{
    if constexpr (sizeof(T) == 2) {
        const uint32_t w = bf16x2_max(bf16x2_max(v.x, v.y), bf16x2_max(v.z, v.w));
        return fmaxf(bf16lo(w), bf16hi(w));
    } else {
        return fmaxf(fmaxf(__uint_as_float(v.x), __uint_as_float(v.y)),
                     fmaxf(__uint_as_float(v.z), __uint_as_float(v.w)));
    }
}

// scalar gather of one vector's worth of elements (unaligned rows / tails)
template <typename T>
DDT_DEVINL uint4 load_scalar(const T *p, int valid)
{
    uint32_t w[4] = {Elem<T>::NEG_INF_FILL, Elem<T>::NEG_INF_FILL, Elem<T>::NEG_INF_FILL,
                     Elem<T>::NEG_INF_FILL};
    if constexpr (sizeof(T) == 2) {
        for (int e = 0; e < 8; ++e)
            if (e < valid) {
                const uint32_t b = (uint32_t)__ldg(reinterpret_cast<const unsigned short *>(p) + e);
                if (e & 1)
                    w[e >> 1] = (w[e >> 1] & 0x0000FFFFu) | (b << 16);
                else
                    w[e >> 1] = (w[e >> 1] & 0xFFFF0000u) | b;
            }
    } else {
        for (int e = 0; e < 4; ++e)
            if (e < valid)
                w[e] = __float_as_uint(__ldg(reinterpret_cast<const float *>(p) + e));
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// merge two (max, sum-of-exp) pairs
DDT_DEVINL void ms_combine(float &m, float &s, float mo, float so)
{
    const float M = fmaxf(m, mo);
    float r = 0.f;
    if (m != DDT_NEG_INF)
        r += s * ex2((m - M) * DDT_LOG2E);
    if (mo != DDT_NEG_INF)
        r += so * ex2((mo - M) * DDT_LOG2E);
    m = M;
    s = r;
}
