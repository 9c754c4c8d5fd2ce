// kivi_divm.h -- correctly rounded fp32 division by the code range
// M = 2^b - 1 (b = 2, 4, 8), the divisor of every group scale.
//
// Method of Brisebarre, Muller and Raina, "Accelerating correctly rounded
// floating-point division when the divisor is known in advance" (IEEE
// Transactions on Computers 53(8), 2004): with zh = RN(1/M) and
// zl = RN(1/M - zh), q = RN(x zh + RN(x zl)) -- one multiply and one fused
// multiply-add -- equals the IEEE quotient RN(x / M) for the x it is checked
// on.  A group's range x = RN(max - min) of two fp16 values is 0 or lies in
// [2^-24, 131008]; tests/test_divm.py checks the identity for every fp32 x in
// [2^-24, 2^17] and each M by exhaustion (0 maps to 0 trivially).  Plain
// C++: included by the CUDA kernels and by that test.
#pragma once

namespace kivi {

template <int BITS>
struct DivM;
template <>
struct DivM<2> {  // M = 3
    static constexpr float M = 3.0f, hi = 0x1.555556p-2f, lo = -0x1.555556p-27f;
};
template <>
struct DivM<4> {  // M = 15
    static constexpr float M = 15.0f, hi = 0x1.111112p-4f, lo = -0x1.dddddep-29f;
};
template <>
struct DivM<8> {  // M = 255
    static constexpr float M = 255.0f, hi = 0x1.010102p-8f, lo = -0x1.fdfdfep-33f;
};

}  // namespace kivi
