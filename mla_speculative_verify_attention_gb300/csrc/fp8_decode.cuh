// OCP FP8 E4M3 ("fn" variant) -> bf16 for the fp8 key path.
//
// An e4m3 byte s.eeee.mmm has value (-1)^s 2^(e-7) (1 + m/8) for e > 0, (-1)^s 2^-6 (m/8)
// for e = 0, and is NaN for eeee.mmm = 1111.111 (there are no infinities).  Every such
// value is an fp16 and a bf16 value, so the hardware conversion e4m3x2 -> f16x2, the
// widening to fp32 and the rounding to bf16 are all exact (NaN stays NaN, -0 stays -0).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <stdint.h>

namespace mla {

// Sixteen e4m3 codes (byte i of raw = code i) -> sixteen bf16 values, codes 0..7 in lo
// and 8..15 in hi (element i of a uint4 holds bf16 2i in its low half, 2i + 1 in its high).
__device__ __forceinline__ void e4m3x16_to_bf16(const uint4& raw, uint4& lo, uint4& hi) {
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
    uint32_t o[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
#pragma unroll
        for (int hlf = 0; hlf < 2; ++hlf) {
            const __nv_fp8x2_storage_t pair = (__nv_fp8x2_storage_t)(w[i] >> (16 * hlf));
            const __half2 h = __half2(__nv_cvt_fp8x2_to_halfraw2(pair, __NV_E4M3));
            const float2 f = __half22float2(h);
            const __nv_bfloat162 b = __floats2bfloat162_rn(f.x, f.y);
            o[2 * i + hlf] = *reinterpret_cast<const uint32_t*>(&b);
        }
    }
    lo = make_uint4(o[0], o[1], o[2], o[3]);
    hi = make_uint4(o[4], o[5], o[6], o[7]);
}

// The same sixteen codes times the key's scale s (fp32): each value is the fp32 product
// code * s rounded to the nearest bf16, ties to even.  The code (at most 4 significant
// bits) and s are exact in fp32, so the product is exact to fp32 rounding (2^-24) and the
// bf16 result is within a relative 2^-8 (half a bf16 ulp) of the dequantised value s * code.
__device__ __forceinline__ void e4m3x16_to_bf16_scaled(const uint4& raw, float s, uint4& lo, uint4& hi) {
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
    uint32_t o[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
#pragma unroll
        for (int hlf = 0; hlf < 2; ++hlf) {
            const __nv_fp8x2_storage_t pair = (__nv_fp8x2_storage_t)(w[i] >> (16 * hlf));
            const __half2 h = __half2(__nv_cvt_fp8x2_to_halfraw2(pair, __NV_E4M3));
            const float2 f = __half22float2(h);
            const __nv_bfloat162 b = __floats2bfloat162_rn(f.x * s, f.y * s);
            o[2 * i + hlf] = *reinterpret_cast<const uint32_t*>(&b);
        }
    }
    lo = make_uint4(o[0], o[1], o[2], o[3]);
    hi = make_uint4(o[4], o[5], o[6], o[7]);
}

}  // namespace mla
