// pkv_elem.h -- storage elements of the K/V pool: f32 (the pages' format),
// bf16 or fp8 e4m3 (additions of this library: every row rounded once, to
// nearest even, when it is written; read back exactly and widened to f32 for
// the math).  An fp8 pool stores e4m3(x / scale), saturated to +-448, with a
// power-of-two scale; callers divide by the scale before a store and apply it
// after a load (where it costs nothing: the queries and the output).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_fp16.h>
#include <cstdint>

namespace pkv {

using bf16 = __nv_bfloat16;
using fp8 = __nv_fp8_e4m3;

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(bf16 x) { return __bfloat162float(x); }
__device__ __forceinline__ float fp8_bits_to_f32(unsigned int b) {
    return __half2float(__half(__nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(b), __NV_E4M3)));
}
__device__ __forceinline__ float to_f32(fp8 x) { return fp8_bits_to_f32(x.__x); }

__device__ __forceinline__ void store1(float *p, float x) { *p = x; }
__device__ __forceinline__ void store1(bf16 *p, float x) { *p = __float2bfloat16_rn(x); }
__device__ __forceinline__ void store1(fp8 *p, float x) {
    p->__x = __nv_cvt_float_to_fp8(x, __NV_SATFINITE, __NV_E4M3);
}

// Four consecutive elements as a float4: shared or global memory, 16-byte
// (f32), 8-byte (bf16) or 4-byte (fp8) aligned; the first element in the
// lowest address.
__device__ __forceinline__ float4 load4(const float *p) { return *reinterpret_cast<const float4 *>(p); }
__device__ __forceinline__ float4 bf16x4_to_f32(uint2 u) {
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.x));
    const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.y));
    return make_float4(a.x, a.y, b.x, b.y);
}
__device__ __forceinline__ float4 load4(const bf16 *p) {
    return bf16x4_to_f32(*reinterpret_cast<const uint2 *>(p));
}
__device__ __forceinline__ float4 fp8x4_to_f32(unsigned int u) {
    const __half2 a(__nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(u & 0xffffu), __NV_E4M3));
    const __half2 b(__nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(u >> 16), __NV_E4M3));
    const float2 fa = __half22float2(a), fb = __half22float2(b);
    return make_float4(fa.x, fa.y, fb.x, fb.y);
}
__device__ __forceinline__ float4 load4(const fp8 *p) {
    return fp8x4_to_f32(*reinterpret_cast<const unsigned int *>(p));
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
__device__ __forceinline__ float4 ldg4(const fp8 *p) {
    return fp8x4_to_f32(__ldg(reinterpret_cast<const unsigned int *>(p)));
}
__device__ __forceinline__ float ldg1(const fp8 *p) {
    return fp8_bits_to_f32(__ldg(reinterpret_cast<const unsigned char *>(p)));
}

// Store four f32 values (rounded to nearest even for bf16, and saturated for fp8).
__device__ __forceinline__ void store4(float *p, float4 v) { *reinterpret_cast<float4 *>(p) = v; }
__device__ __forceinline__ void store4(fp8 *p, float4 v) {
    const unsigned int a = __nv_cvt_float2_to_fp8x2(make_float2(v.x, v.y), __NV_SATFINITE, __NV_E4M3);
    const unsigned int b = __nv_cvt_float2_to_fp8x2(make_float2(v.z, v.w), __NV_SATFINITE, __NV_E4M3);
    *reinterpret_cast<unsigned int *>(p) = a | (b << 16);
}
__device__ __forceinline__ void store4(bf16 *p, float4 v) {
    const __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y);
    const __nv_bfloat162 b = __floats2bfloat162_rn(v.z, v.w);
    uint2 u;
    u.x = *reinterpret_cast<const uint32_t *>(&a);
    u.y = *reinterpret_cast<const uint32_t *>(&b);
    *reinterpret_cast<uint2 *>(p) = u;
}

}  // namespace pkv
