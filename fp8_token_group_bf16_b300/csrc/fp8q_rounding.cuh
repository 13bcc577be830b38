// The correctly rounded division of a group's maximum by 448 in two
// instructions.  It returns exactly what the IEEE division returns (round to
// nearest even); the tests compare it with the oracle's IEEE division over
// every fp32 significand.  It replaces the general IEEE division (about ten
// instructions with special-case handling) on the path from a group's last
// value to its first code, which every lane of the group waits on: 13.9 us
// against 14.35 us for rms_norm_per_block_quant at T = 4096, H = 5120.
//
// Method: N. Brisebarre, J.-M. Muller, S. K. Raina, "Accelerating correctly
// rounded floating-point division when the divisor is known in advance",
// IEEE Trans. Computers 53(8), 2004: with zh = RN(1/448) and
// zl = RN(1/448 - zh), q = RN(a zh + RN(a zl)), one multiply and one fused
// multiply-add.  Their method is correct for some divisors and not others;
// for 448 it was checked with exact integer arithmetic over all 2^23
// significands of a (the result scales exactly with a's exponent while a zl
// stays normal), and the GPU tests repeat that check on the device.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace fp8q {

// RN(1/448) and RN(1/448 - RN(1/448)).  1/448 = (8/7) 2^-9 and 8/7 =
// 1.001001001..._2, so the 24-bit significand rounds up (0x924925) and the
// remainder is negative.
constexpr float kInv448Hi = 0x1.24924ap-9f;
constexpr float kInv448Lo = -0x1.b6db6ep-34f;

// RN32(a / 448) for finite a >= 1e-30.  Below 2^-60, a zl would leave the
// normal range, so the quotient is formed at a 2^64 and scaled back (both
// scalings exact: the quotient stays above 2^-110).
__device__ __forceinline__ float div448_rn(float a)
{
    const bool tiny = a < 0x1p-60f;
    const float as = tiny ? __fmul_rn(a, 0x1p64f) : a;
    const float q = __fmaf_rn(as, kInv448Hi, __fmul_rn(as, kInv448Lo));
    return tiny ? __fmul_rn(q, 0x1p-64f) : q;
}

}  // namespace fp8q
