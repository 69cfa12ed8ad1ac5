// 2^x on the fused multiply-add pipes instead of the special-function unit.
//
// The IO-Aware Algorithms page names the special-function unit's exponential
// throughput as the resource FlashAttention-4 is bound by on Blackwell: every
// score of the online softmax needs one exp2.  Evaluating a share of them with
// plain FMAs moves that work onto pipes the softmax uses less.
//
// Method (Cody-Waite range reduction followed by a polynomial):
//   x  <- max(x, -127)               masked scores (-inf) and underflow
//   j  =  x + 1.5 * 2^23             rounds x to the nearest integer n, held in
//                                    the low mantissa bits of j (|x| < 2^22)
//   n  =  j - 1.5 * 2^23             exact
//   f  =  x - n                      exact, |f| <= 1/2
//   p  =  1 + f (c1 + f (c2 + ...))  minimax fit of 2^f on [-1/2, 1/2] in
//                                    relative error, with p(0) = 1 exactly
//   2^x = p * 2^n                    by adding n to p's exponent field: the
//                                    bits of j shifted left by 23 are n << 23
//                                    (the constant's own bits shift out)
// x = -127 gives exactly +0 (f = 0, p = 1, exponent field 127 - 127), so a
// masked score contributes nothing; x in (-127, -126) gives a denormal below
// 2^-126.  x = 0 gives exactly 1.
//
// The coefficients are this project's own linear-programming minimax fits
// (fit_exp2_poly.py next to this file prints them), rounded to fp32.  Largest
// relative error of the fp32 evaluation over [-126, 64]: degree 4, 2.9e-6;
// degree 5, 1.6e-7 (tests/test_exp2_poly.py checks it against the C library's
// exp2 on the host, which evaluates the same operations in the same order).
#pragma once

#include <cstdint>
#include <cstring>

#ifndef ELS_EXP2_POLY_DEGREE
#define ELS_EXP2_POLY_DEGREE 4
#endif

#if defined(__CUDACC__)
#define ELS_HD __host__ __device__ __forceinline__
#else
#define ELS_HD inline
#endif

namespace elsattn {

constexpr float kExp2RoundMagic = 12582912.0f;  // 1.5 * 2^23
constexpr float kExp2PolyMin = -127.0f;

#if ELS_EXP2_POLY_DEGREE < 3 || ELS_EXP2_POLY_DEGREE > 5
#error "ELS_EXP2_POLY_DEGREE must be 3, 4 or 5"
#endif
constexpr int kExp2PolyDegree = ELS_EXP2_POLY_DEGREE;

// Coefficient c_{k+1} of the degree-kExp2PolyDegree fit (c_0 = 1).
ELS_HD constexpr float exp2_poly_c(int k) {
#if ELS_EXP2_POLY_DEGREE == 3
    return k == 0 ? 0x1.62f5fap-1f : k == 1 ? 0x1.f00c4cp-3f : 0x1.c2a216p-5f;
#elif ELS_EXP2_POLY_DEGREE == 4
    return k == 0 ? 0x1.62e12ep-1f : k == 1 ? 0x1.ec036cp-3f : k == 2 ? 0x1.c9fc30p-5f : 0x1.3a05f8p-7f;
#else
    return k == 0 ? 0x1.62e42ap-1f
         : k == 1 ? 0x1.ebf9aep-3f
         : k == 2 ? 0x1.c6b64ep-5f
         : k == 3 ? 0x1.3cee66p-7f
                  : 0x1.5c10d4p-10f;
#endif
}

ELS_HD uint32_t exp2_poly_bits(float v) {
#if defined(__CUDA_ARCH__)
    return __float_as_uint(v);
#else
    uint32_t u;
    std::memcpy(&u, &v, sizeof u);
    return u;
#endif
}

ELS_HD float exp2_poly_float(uint32_t u) {
#if defined(__CUDA_ARCH__)
    return __uint_as_float(u);
#else
    float v;
    std::memcpy(&v, &u, sizeof v);
    return v;
#endif
}

// Scalar reference, one operation per step in the order above; the packed
// device version below rounds lane by lane exactly as this does.
ELS_HD float exp2_poly(float x) {
    x = x > kExp2PolyMin ? x : kExp2PolyMin;
    const float j = x + kExp2RoundMagic;
    const float n = j - kExp2RoundMagic;
    const float f = x - n;
    float p = exp2_poly_c(kExp2PolyDegree - 1);
    for (int k = kExp2PolyDegree - 2; k >= 0; --k) p = fmaf(p, f, exp2_poly_c(k));
    p = fmaf(p, f, 1.0f);
    return exp2_poly_float(exp2_poly_bits(p) + (exp2_poly_bits(j) << 23));
}

#if defined(__CUDACC__)
// Two lanes at once: (y0, y1) = (2^x0, 2^x1), with the fp32 arithmetic on
// packed f32x2 instructions (add.rn / fma.rn per lane, as the scalar form).
__device__ __forceinline__ void exp2_poly2(float& y0, float& y1, float x0, float x1) {
    x0 = fmaxf(x0, kExp2PolyMin);
    x1 = fmaxf(x1, kExp2PolyMin);
    uint64_t x, j, n, f, p;
    asm("mov.b64 %0, {%1, %2};" : "=l"(x) : "f"(x0), "f"(x1));
    const float m = kExp2RoundMagic;
    asm("{\n\t.reg .b64 c;\n\tmov.b64 c, {%2, %2};\n\tadd.rn.f32x2 %0, %1, c;\n\t}" : "=l"(j) : "l"(x), "f"(m));
    asm("{\n\t.reg .b64 c;\n\tmov.b64 c, {%2, %2};\n\tsub.rn.f32x2 %0, %1, c;\n\t}" : "=l"(n) : "l"(j), "f"(m));
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(f) : "l"(x), "l"(n));
    const float top = exp2_poly_c(kExp2PolyDegree - 1);
    asm("mov.b64 %0, {%1, %1};" : "=l"(p) : "f"(top));
#pragma unroll
    for (int k = kExp2PolyDegree - 2; k >= 0; --k) {
        const float c = exp2_poly_c(k);
        asm("{\n\t.reg .b64 c;\n\tmov.b64 c, {%3, %3};\n\tfma.rn.f32x2 %0, %1, %2, c;\n\t}"
            : "=l"(p) : "l"(p), "l"(f), "f"(c));
    }
    const float one = 1.0f;
    asm("{\n\t.reg .b64 c;\n\tmov.b64 c, {%3, %3};\n\tfma.rn.f32x2 %0, %1, %2, c;\n\t}"
        : "=l"(p) : "l"(p), "l"(f), "f"(one));
    uint32_t p0, p1, j0, j1;
    asm("mov.b64 {%0, %1}, %2;" : "=r"(p0), "=r"(p1) : "l"(p));
    asm("mov.b64 {%0, %1}, %2;" : "=r"(j0), "=r"(j1) : "l"(j));
    y0 = __uint_as_float(p0 + (j0 << 23));
    y1 = __uint_as_float(p1 + (j1 << 23));
}
#endif

}  // namespace elsattn

#undef ELS_HD
