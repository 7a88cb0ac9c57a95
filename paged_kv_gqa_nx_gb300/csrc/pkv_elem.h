// pkv_elem.h -- storage elements of the K/V pool: f32 (the pages' format) or
// bf16 (an addition of this library: every row rounded once, to nearest even,
// when it is written; read back exactly and widened to f32 for the math).
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

namespace pkv {

using bf16 = __nv_bfloat16;

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(bf16 x) { return __bfloat162float(x); }

__device__ __forceinline__ void store1(float *p, float x) { *p = x; }
__device__ __forceinline__ void store1(bf16 *p, float x) { *p = __float2bfloat16_rn(x); }

// Four consecutive elements as a float4: shared or global memory, 16-byte
// (f32) or 8-byte (bf16) aligned.
__device__ __forceinline__ float4 load4(const float *p) { return *reinterpret_cast<const float4 *>(p); }
__device__ __forceinline__ float4 bf16x4_to_f32(uint2 u) {
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.x));
    const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.y));
    return make_float4(a.x, a.y, b.x, b.y);
}
__device__ __forceinline__ float4 load4(const bf16 *p) {
    return bf16x4_to_f32(*reinterpret_cast<const uint2 *>(p));
}

// The same through the read-only path (data that no thread of the launch writes).
__device__ __forceinline__ float4 ldg4(const float *p) { return __ldg(reinterpret_cast<const float4 *>(p)); }
__device__ __forceinline__ float4 ldg4(const bf16 *p) {
    return bf16x4_to_f32(__ldg(reinterpret_cast<const uint2 *>(p)));
}
__device__ __forceinline__ float ldg1(const float *p) { return __ldg(p); }
__device__ __forceinline__ float ldg1(const bf16 *p) {
    return __bfloat162float(__ushort_as_bfloat16(__ldg(reinterpret_cast<const unsigned short *>(p))));
}

// Store four f32 values (rounded to nearest even for bf16).
__device__ __forceinline__ void store4(float *p, float4 v) { *reinterpret_cast<float4 *>(p) = v; }
__device__ __forceinline__ void store4(bf16 *p, float4 v) {
    const __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y);
    const __nv_bfloat162 b = __floats2bfloat162_rn(v.z, v.w);
    uint2 u;
    u.x = *reinterpret_cast<const uint32_t *>(&a);
    u.y = *reinterpret_cast<const uint32_t *>(&b);
    *reinterpret_cast<uint2 *>(p) = u;
}

}  // namespace pkv
