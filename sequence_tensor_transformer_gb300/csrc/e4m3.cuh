// Row-wise E4M3 quantisation helpers shared by the quantiser and the fused
// prologue: a row with maximum magnitude amax gets the power-of-two scale
// 2^e, e the least integer >= -126 with amax <= 448 * 2^e, and codes
// RNE_E4M3(v * 2^-e) (exact products, so the decision is the bf16 value's).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <stdint.h>

namespace sptp {

// With amax = 1.m * 2^E (normal) and 448 = 1.75 * 2^8: e = E - 8, plus one
// when 1.m > 1.75; zero and subnormal maxima give the floor -126.
__device__ __forceinline__ int e4m3_row_exponent(float amax) {
    const uint32_t u = __float_as_uint(amax);
    const int biased = static_cast<int>(u >> 23);  // amax >= 0
    const int e = biased - 127 - 8 + ((u & 0x7FFFFFu) > 0x600000u ? 1 : 0);
    return biased == 0 ? -126 : max(e, -126);
}

// 2^e for -126 <= e <= 127, built from its exponent field
__device__ __forceinline__ float pow2f(int e) { return __uint_as_float(static_cast<uint32_t>(127 + e) << 23); }

// max |.| of 8 bf16 packed in a 16-byte vector
__device__ __forceinline__ float absmax_bf16x8(const uint4 v) {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
    __nv_bfloat162 m = __habs2(h[0]);
    m = __hmax2(m, __habs2(h[1]));
    m = __hmax2(m, __habs2(h[2]));
    m = __hmax2(m, __habs2(h[3]));
    return fmaxf(__low2float(m), __high2float(m));
}

// 8 bf16 -> 8 E4M3 bytes (element order kept), each times inv (a power of two)
__device__ __forceinline__ uint2 e4m3_quant8(const uint4 v, float inv) {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
    uint32_t w[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const float2 a = __bfloat1622float2(h[2 * i]);
        const float2 b = __bfloat1622float2(h[2 * i + 1]);
        const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(a.x * inv, a.y * inv), __NV_SATFINITE, __NV_E4M3);
        const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(b.x * inv, b.y * inv), __NV_SATFINITE, __NV_E4M3);
        w[i] = (lo & 0xFFFFu) | (hi << 16);
    }
    return make_uint2(w[0], w[1]);
}

}  // namespace sptp
