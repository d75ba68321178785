// la_tc_common.cuh -- device helpers shared by the tensor-core kernels:
// global-memory ordering, named barriers, packed fp32 / bf16 arithmetic, the
// bf16 hi/lo split that carries fp32 operands into bf16 MMAs, and the elu+1
// feature map on 128-byte swizzled bf16 tiles.
#pragma once

#include <stdint.h>

#include "la_sm100.cuh"

namespace la {
namespace tcc {

using namespace sm100;

__device__ __forceinline__ uint64_t globaltimer()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void st_release(unsigned* p, unsigned v)
{
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ unsigned ld_acquire(const unsigned* p)
{
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Drop a 128-byte L2 line without writing it back (scratch read for the last
// time).
__device__ __forceinline__ void l2_discard(const void* ptr)
{
    asm volatile("discard.global.L2 [%0], 128;" ::"l"(ptr) : "memory");
}

__device__ __forceinline__ void named_bar(int id, int count)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// A thread group waits through one leader; bar.red hands every thread the
// same verdict, so the group never splits on an abort.
__device__ __forceinline__ bool group_ok(int ok, int barid, int count)
{
    int res;
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %1, 0;\n\t"
        "bar.red.and.pred p, %2, %3, p;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(res)
        : "r"(ok), "r"(barid), "r"(count)
        : "memory");
    return res != 0;
}

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Packed fp32 pair arithmetic (two lanes of work per instruction).
__device__ __forceinline__ float2 sub2(float2 a, float2 b)
{
    float2 r;
    asm("{\n\t.reg .b64 x, y, z;\n\tmov.b64 x, {%2, %3};\n\tmov.b64 y, {%4, %5};\n\t"
        "sub.rn.f32x2 z, x, y;\n\tmov.b64 {%0, %1}, z;\n\t}"
        : "=f"(r.x), "=f"(r.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return r;
}

// split two fp32 into packed bf16 hi and lo parts (hi + lo = x to ~2^-17)
__device__ __forceinline__ void split2(float a, float b, uint32_t& hi, uint32_t& lo)
{
    hi = pack_bf16x2(a, b);
    const float2 r = sub2(make_float2(a, b), make_float2(bf_lo(hi), bf_hi(hi)));
    lo = pack_bf16x2(r.x, r.y);
}

__device__ __forceinline__ float2 mul2(float2 a, float2 b)
{
    float2 r;
    asm("{\n\t.reg .b64 x, y, z;\n\tmov.b64 x, {%2, %3};\n\tmov.b64 y, {%4, %5};\n\t"
        "mul.rn.f32x2 z, x, y;\n\tmov.b64 {%0, %1}, z;\n\t}"
        : "=f"(r.x), "=f"(r.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return r;
}

__device__ __forceinline__ float ex2(float t)
{
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(t));
    return r;
}

// elu(x)+1 on two packed bf16: max(x,0) + exp(min(x,0)), with
// exp(u) = 2^(u log2 e) on the hardware base-2 exponential.  For every
// element one of the two terms is exactly 0 or 1, so the packed bf16 sum of
// max(x,0) and the rounded exponential is the fp32 value rounded once.
__device__ __forceinline__ uint32_t phi2(uint32_t w)
{
    uint32_t mn, mx, r;
    asm("min.bf16x2 %0, %1, %2;" : "=r"(mn) : "r"(w), "r"(0u));
    asm("max.bf16x2 %0, %1, %2;" : "=r"(mx) : "r"(w), "r"(0u));
    const float2 t = mul2(make_float2(bf_lo(mn), bf_hi(mn)),
                          make_float2(1.4426950408889634f, 1.4426950408889634f));
    const uint32_t e = pack_bf16x2(ex2(t.x), ex2(t.y));
    asm("add.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(mx), "r"(e));
    return r;
}

// Feature map in place on a 128 x 64 bf16 tile (128-byte swizzle) by 128
// threads; rows >= valid become zero.
__device__ __forceinline__ void phi_tile(unsigned char* tile, int t, int valid, bool elu)
{
    const int cc = t & 7, r0 = t >> 3;
#pragma unroll 2
    for (int mm = 0; mm < 8; mm += 2) {
        uint4 x[2];
#pragma unroll
        for (int u = 0; u < 2; ++u)
            x[u] = *reinterpret_cast<const uint4*>(tile + sw128_off(r0 + 16 * (mm + u), cc));
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int r = r0 + 16 * (mm + u);
            if (r >= valid)
                x[u] = make_uint4(0, 0, 0, 0);
            else if (elu)
                x[u] = make_uint4(phi2(x[u].x), phi2(x[u].y), phi2(x[u].z), phi2(x[u].w));
            if (r >= valid || elu)
                *reinterpret_cast<uint4*>(tile + sw128_off(r, cc)) = x[u];
        }
    }
}

}  // namespace tcc
}  // namespace la
