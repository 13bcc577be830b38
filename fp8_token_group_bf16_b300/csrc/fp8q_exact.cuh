// Error-free transformations of sums (Knuth's TwoSum; Dekker's Fast2Sum is
// written out where it is used): for floating-point a and b the rounding error
// of RN(a + b) is itself a floating-point number, obtained exactly from a few
// further additions.  The row sum of squares of rms_norm_per_block_quant is
// formed this way, so that the fp32 value it rounds to is the sum of the
// squares rounded once, whatever order the GPU adds them in.
#pragma once

#include <cuda_runtime.h>

namespace fp8q {

// s + e == a + b exactly, s = RN(a + b) (TwoSum: six additions, any a, b).
// Once a sum overflows, s = +inf stays +inf (all summands are >= 0) and e may
// be NaN; the final rounding looks at s alone in that case.
__device__ __forceinline__ void two_sum(float a, float b, float &s, float &e)
{
    s = __fadd_rn(a, b);
    const float bb = __fsub_rn(s, a);
    e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}

// (hi, lo) += (h2, l2): the high parts summed without error, the low parts
// (already tiny next to the high parts) summed plainly.
__device__ __forceinline__ void pair_add(float &hi, float &lo, float h2, float l2)
{
    float s, e;
    two_sum(hi, h2, s, e);
    lo = __fadd_rn(__fadd_rn(lo, l2), e);
    hi = s;
}

}  // namespace fp8q
