// ddt_device.cuh -- small device helpers shared by the kernels of libddt.so.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#define DDT_DEVINL __device__ __forceinline__

constexpr float DDT_LOG2E = 1.4426950408889634f;
constexpr float DDT_NEG_INF = -__builtin_huge_valf();

// bf16 bit patterns -> fp32 (exact)
DDT_DEVINL float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
DDT_DEVINL float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
DDT_DEVINL float bf16_to_f32(uint16_t b) { return __uint_as_float(((uint32_t)b) << 16); }

// fp32 -> bf16 pair (round to nearest even), lo in the low half
DDT_DEVINL uint32_t pack_bf16x2(float lo, float hi)
{
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// hardware base-2 exponential (MUFU), flush-to-zero
DDT_DEVINL float ex2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// packed fp32 pairs (two lanes of one 64-bit register)
DDT_DEVINL uint64_t f2pack(float lo, float hi)
{
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
DDT_DEVINL void f2unpack(uint64_t v, float &lo, float &hi)
{
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
DDT_DEVINL uint64_t f2fma(uint64_t a, uint64_t b, uint64_t c)
{
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}
DDT_DEVINL uint64_t f2add(uint64_t a, uint64_t b)
{
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
// programmatic dependent launch: wait until the grids this one depends on
// have completed and their writes are visible; let the next grid start its
// prologue (no-ops for a grid launched without the attribute)
DDT_DEVINL void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
DDT_DEVINL void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// streaming 16-byte global load that does not allocate in L1
DDT_DEVINL uint4 ldg_stream(const void *p)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// ask the copy engine to bring [p, p + bytes) into L2 (p 16-byte aligned,
// bytes a multiple of 16); nothing waits for it
DDT_DEVINL void prefetch_l2(const void *p, uint32_t bytes)
{
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

DDT_DEVINL void set_status(int32_t *status, int bits)
{
    atomicOr(status, bits);
}

// (value, index) ordering used by top-K: larger value first, then lower index
DDT_DEVINL bool beats(float va, int ia, float vb, int ib)
{
    return va > vb || (va == vb && ia < ib);
}
