// OCP FP8 E4M3 ("e4m3fn") on the device: sign, 4 exponent bits (bias 7),
// 3 mantissa bits, no infinities, S.1111.111 = NaN, largest finite 448,
// subnormals m * 2^-9.  Used for the FP8 KV cache: an entry is stored as
// e4m3(x / scale) with one scale per kv head, and read as code * scale.
#pragma once

#include <cstdint>

namespace hd {

// Nearest-even rounding of a double to E4M3, saturating at +-448 (also for
// infinities); NaN gives the NaN code.  Integer arithmetic on the binary64
// fields: a value in binade 2^e (e >= -6) keeps 3 fraction bits, below 2^-6
// the quantum is 2^-9; the dropped bits decide the rounding (above half: up;
// exactly half: to the even significand).  A carry into the next binade is
// the next code; code 8 (2^-6) follows the largest subnormal naturally.
__device__ __forceinline__ uint8_t e4m3_from_f64(double x) {
    const unsigned long long bits = static_cast<unsigned long long>(__double_as_longlong(x));
    const uint8_t sign = (bits >> 63) ? 0x80 : 0x00;
    const unsigned long long mag = bits & 0x7FFFFFFFFFFFFFFFull;
    if (mag > 0x7FF0000000000000ull) return 0x7F;                 // NaN
    if (mag > 0x407C000000000000ull) return sign | 0x7E;          // above 448 = 1.75 * 2^8, or infinite
    const int e = static_cast<int>(mag >> 52) - 1023;             // binary64 subnormals: tiny, round to 0
    const int shift = e >= -6 ? 49 : 43 - e;                      // dropped low bits of the 53-bit significand
    if (shift > 63) return sign;
    const unsigned long long m = (1ull << 52) | (mag & ((1ull << 52) - 1));
    unsigned long long k = m >> shift;
    const unsigned long long rem = m & ((1ull << shift) - 1), half = 1ull << (shift - 1);
    if (rem > half || (rem == half && (k & 1))) ++k;
    if (e < -6) return sign | static_cast<uint8_t>(k);            // k * 2^-9, k <= 8
    int E = e;
    if (k == 16) {                                                // rounded up into the next binade
        k = 8;
        ++E;
    }
    return sign | static_cast<uint8_t>(((E + 7) << 3) | static_cast<int>(k - 8));
}

// e4m3_from_f64(fl64(y / s)) -- the code of the quotient rounded once to
// binary64 -- without a binary64 division in the common case.  The quotient
// is first taken in binary32 (y and s rounded to binary32, then a correctly
// rounded division: relative error below 2^-23).  Its E4M3 rounding is the
// same as the exact quotient's unless the exact quotient lies within that
// error of an E4M3 midpoint; a binary32 quotient whose distance to a midpoint
// is below 2^-18 quanta (the error is at most 2^-19 quanta) takes the exact
// binary64 division instead.  s must be a binary32 value.
__device__ __forceinline__ uint8_t e4m3_quotient(double y, double s) {
    const float qf = __fdiv_rn(__double2float_rn(y), __double2float_rn(s));
    const unsigned u = __float_as_uint(qf) & 0x7FFFFFFFu;
    bool near = false;
    if (u >= 0x3C800000u && u < 0x43E00000u) {          // [2^-6, 448): a quantum is 2^20 binary32 ulps
        near = (u & 0xFFFFFu) - 0x7FFFCu <= 8u;         // within 4 ulps (2^-18 quanta) of a midpoint
    } else if (u >= 0x39800000u && u < 0x3C800000u) {   // [2^-12, 2^-6): quantum 2^-9
        const float t = __uint_as_float(u) * 512.f;     // the value in quanta (exact)
        near = fabsf(t - truncf(t) - 0.5f) <= 3.814697265625e-06f;   // 2^-18
    }
    return near ? e4m3_from_f64(__ddiv_rn(y, s)) : e4m3_from_f64((double)qf);   // NaN, 0 and saturation pass through
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
