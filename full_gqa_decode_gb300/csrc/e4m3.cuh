// OCP FP8 E4M3 ("e4m3fn") on the device: sign, 4 exponent bits (bias 7),
// 3 mantissa bits, no infinities, S.1111.111 = NaN, largest finite 448,
// subnormals m * 2^-9.  Used for the FP8 KV cache: an entry is stored as
// e4m3(x / scale) with one scale per kv head, and read as code * scale.
#pragma once

#include <cstdint>

namespace hd {

// Nearest-even rounding of a double to E4M3, saturating at +-448 (also for
// infinities); NaN gives the NaN code.  |x| is split into its binade 2^e: in
// [2^-6, 448] the E4M3 quantum is 2^(e-3), so rint(|x| / 2^(e-3)) is the
// significand 8..16 (16 carries into the next binade); below 2^-6 the
// quantum is 2^-9 and rint(|x| * 2^9) is already the code (8 = smallest
// normal).  Both scalings are exact.
__device__ __forceinline__ uint8_t e4m3_from_f64(double x) {
    const unsigned long long bits = static_cast<unsigned long long>(__double_as_longlong(x));
    const uint8_t sign = (bits >> 63) ? 0x80 : 0x00;
    const double a = fabs(x);
    if (a != a) return 0x7F;
    if (a > 448.0) return sign | 0x7E;
    if (a < 0.015625) return sign | static_cast<uint8_t>(rint(a * 512.0));   // 2^-6, 2^9
    int e = static_cast<int>((bits >> 52) & 0x7FF) - 1023;                   // a is normal here
    int q = static_cast<int>(rint(ldexp(a, 3 - e)));
    if (q == 16) {
        q = 8;
        ++e;
    }
    return sign | static_cast<uint8_t>(((e + 7) << 3) | (q - 8));
}

// Exact value of an E4M3 code as a float.
__device__ __forceinline__ float e4m3_to_f32(uint8_t code) {
    const int e = (code >> 3) & 15, m = code & 7;
    float v;
    if (e == 15 && m == 7) {
        v = __int_as_float(0x7FC00000);
    } else if (e == 0) {
        v = static_cast<float>(m) * 0.001953125f;                              // m * 2^-9
    } else {
        v = __int_as_float(((e - 7 + 127) << 23) | (m << 20));                 // (1 + m/8) * 2^(e-7)
    }
    return (code & 0x80) ? -v : v;
}

// Two E4M3 codes (low byte first) to an f16x2 register, low half first.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint16_t pair) {
    uint32_t r;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(pair));
    return r;
}

}  // namespace hd
