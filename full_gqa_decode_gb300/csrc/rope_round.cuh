// The written key of a rotary pair, rounded once to bf16.
//
// Neox-style partial RoPE (vllm_omni/edge/spark_export.py, `_rope`) rotates the
// pair (x1, x2) of a new key by the angle of its position:
//     y1 = x1 c - x2 s,   y2 = x2 c + x1 s,
// with x1, x2 bf16 and c, s the fp32 table values.  The stored key is the exact
// value rounded once to nearest-even bf16, so it is reproducible bit for bit.
// Both outputs have the form a c - b s ((a, b) = (x1, x2), then (x2, -x1)).
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

namespace hd {

// One round-to-nearest-even of a double to bf16, through round-to-odd binary32
// (Boldo & Melquiond, IEEE TC 2008): the odd-rounded binary32 keeps enough bits
// that rounding it to bf16 equals rounding the double directly.
__device__ __forceinline__ float f64_to_bf16_value(double x) {
    float t = __double2float_rz(x);
    if ((double)t != x && isfinite(t)) t = __uint_as_float(__float_as_uint(t) | 1u);
    return __bfloat162float(__float2bfloat16_rn(t));
}

// bf16_rne(a c - b s) for bf16 a, b and fp32 c, s, exactly.  The products are
// exact in binary64 (8 + 24 significant bits) and the difference is rounded
// once there.  The fast path evaluates y = fma(a, c, -RN32(b s)) in binary32:
// |y - (a c - b s)| <= ulp(y)/2 + ulp(b s)/2.  The bf16 roundings of all values
// that share y's upper 16 bits break at a single point, the midpoint whose lower
// 16 bits are 0x8000, so when y lies farther than that bound from it, y and the
// exact value round to the same bf16.  Values near the midpoint (ties among
// them), zero, subnormal, infinite or NaN results, and heavy cancellation (the
// bound over 2^13 units) take the binary64 path.
__device__ __forceinline__ float rotated_bf16(float a, float c, float b, float s) {
    const float q = b * s;
    const float y = fmaf(a, c, -q);
    const uint32_t yb = __float_as_uint(y), qb = __float_as_uint(q);
    const int ey = (int)((yb >> 23) & 0xFFu);
    const int eq = max((int)((qb >> 23) & 0xFFu), 1);   // subnormal q: the smallest binade's spacing
    const int d = eq - ey;
    if (ey != 0 && ey != 255 && d <= 13) {
        const int bound = 2 + (d > 0 ? (1 << d) : 1);     // > ulp(y)/2 + ulp(q)/2 in units of ulp(y)
        if (abs((int)(yb & 0xFFFFu) - 0x8000) > bound) return __bfloat162float(__float2bfloat16_rn(y));
    }
    return f64_to_bf16_value(__dsub_rn(__dmul_rn((double)a, (double)c), __dmul_rn((double)b, (double)s)));
}

}  // namespace hd
