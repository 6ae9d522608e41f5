// ct_device.cuh -- small device helpers shared by the kernel translation units.
#pragma once

#include <stdint.h>

namespace ct {

// bf16 is carried as its 16-bit pattern; widening to fp32 is exact (the
// pattern is the upper half of the fp32 pattern).
typedef unsigned short bf16_t;

__device__ __forceinline__ float to_float(float v) { return v; }
__device__ __forceinline__ float to_float(bf16_t v) { return __uint_as_float((uint32_t)v << 16); }

__device__ __forceinline__ float ldg(const float *p) { return __ldg(p); }
__device__ __forceinline__ bf16_t ldg(const bf16_t *p) { return __ldg(p); }

// Fused epilogue of [l2_p26]: t = v + a; t * hardswish(t) with
// hardswish(t) = t * clamp(t + 3, 0, 6) / 6, evaluated in fp32; the division
// by 6 is a multiplication by the fp32 value of 1/6 (within 1 ulp of the
// quotient, and a third of the instructions of an IEEE division).
__device__ __forceinline__ float add_hswish(float v, float a)
{
    const float t = v + a;
    const float c = fminf(fmaxf(t + 3.f, 0.f), 6.f);
    const float hs = (t * c) * (1.f / 6.f);
    return t * hs;
}

}  // namespace ct
