// E4M3 quantisation quotients by reciprocal (quantisers that are bound by
// their IEEE divisions use it; tests/test_e4m3_quotient.py checks the rule).
#pragma once
#include "common.cuh"

namespace moe {

// The quotient x / s of a quantisation, for its E4M3 code, as q0 = fl(x * r) with
// r = e4m3_recip(s), where that cannot change the code. q0 lies within about 3 units
// in the last place of fl(x / s) (r and the product each round by at most half a unit,
// the quotient by half a unit), and the code of a float changes only where it crosses
// a midpoint between two E4M3 values. The IEEE division is taken instead
//   - for |q0| >= 2^-6 (E4M3 normals, 3 fraction bits) when the low 20 fp32 fraction
//     bits read within 8 of 0x80000 (q0 within 8 units of a midpoint);
//   - for 2^-11 <= |q0| < 2^-6: E4M3's subnormal steps and the midpoint 2^-10 between
//     0 and the smallest subnormal;
//   - when r is 0.
// Below 2^-11 both codes are the zero of x's sign. So the code is that of
// __fdiv_rn(x, s) for every x.
__device__ __forceinline__ float e4m3_quotient(float x, float s, float r) {
    const float q0 = x * r;
    const uint32_t bits = __float_as_uint(q0) & 0x7fffffffu;
    const uint32_t E = bits >> 23;
    const bool slow =
        r == 0.0f || (E >= 116u && E < 121u) || (E >= 121u && (bits & 0xfffffu) - 0x7fff8u <= 16u);
    return slow ? __fdiv_rn(x, s) : q0;
}
// 1 / s rounded to nearest, or 0 where e4m3_quotient must divide: a scale below the
// smallest normal float (its reciprocal would not be within half a unit) or infinite.
__device__ __forceinline__ float e4m3_recip(float s) { return s >= 0x1p-126f ? __frcp_rn(s) : 0.0f; }

}  // namespace moe
