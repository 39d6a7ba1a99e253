// The canonical confidence key of the unmask/commit step ("Nemotron-Labs-
// TwoTower", Section 2.2, Algorithm 2, confidence), shared by the commit
// kernels: per logit l of a row with maximum m, the fixed-point term
// rint(2^40 * e(RN32(l - m))) of an fp32 exponential e defined for this
// purpose (Cody and Waite range reduction, then the degree-7 Taylor
// polynomial of exp, all with round-to-nearest fused multiply-adds):
//   x < -30 -> term 0
//   n = nearest integer (ties to even) to the exact product x * log2(e)
//   r = fma(-n, C1, x), r = fma(-n, C2, r)     C1 = RN32(ln 2), C2 = RN32(ln 2 - C1)
//   p = c7; p = fma(p, r, c_j), j = 6..0       c_j = RN32(1 / j!)
//   term = rint(p * 2^(n + 40))
// The term is formed without any float-to-64-bit conversion (those run on the
// FP64 pipe, which is narrow on this part): the polynomial carries the 2^40
// factor in its coefficients (exact power-of-two scaling), 2^n is added to the
// exponent field, and rint splits into a multiple of 2^20 plus a remainder,
// both read out of the bits of exact fp32 sums. The arithmetic runs on packed
// f32x2 pairs (each half rounded exactly like the scalar operation).
// Also: the (value, index) encoding whose maximum is the row maximum with the
// lowest index among equal values (the greedy prediction).
#pragma once

#include <cstdint>

namespace tt {
namespace key {

// RN32(1/ln 2), RN32(ln 2), RN32(ln 2 - RN32(ln 2)); 2^40 * RN32(1/j!)
constexpr float kLog2e = 0x1.715476p+0f;
constexpr float kLn2Hi = 0x1.62e430p-1f;
constexpr float kLn2Lo = -0x1.05c610p-29f;
constexpr float kC0 = 0x1.000000p+40f;
constexpr float kC2 = 0x1.000000p+39f;
constexpr float kC3 = 0x1.555556p+37f;
constexpr float kC4 = 0x1.555556p+35f;
constexpr float kC5 = 0x1.111112p+33f;
constexpr float kC6 = 0x1.6c16c2p+30f;
constexpr float kC7 = 0x1.a01a02p+27f;
constexpr float kMagic23 = 0x1.8p+23f;  // fp32 sums in [2^23, 2^24) have ulp 1
constexpr float kMagic43 = 0x1.8p+43f;  // ... in [2^43, 2^44) have ulp 2^20
constexpr unsigned kMagic23Bits = 0x4B400000u;
constexpr unsigned kMagic43Bits = 0x55400000u;

// Packed fp32 pairs: one f32x2 instruction does the same round-to-nearest
// operation on both halves, halving the issue slots of the term arithmetic.
using f2 = unsigned long long;

__device__ __forceinline__ f2 pk(float a, float b) {
    f2 r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}
__device__ __forceinline__ void upk(f2 r, float& a, float& b) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}
__device__ __forceinline__ f2 dup(float c) { return pk(c, c); }
__device__ __forceinline__ f2 ffma2(f2 a, f2 b, f2 c) {
    f2 d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ f2 fadd2(f2 a, f2 b) {
    f2 d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ f2 fsub2(f2 a, f2 b) {
    f2 d;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// Adds the fixed-point terms of x0, x1 (RN32(l - m) clamped below at -31;
// terms below -28.4 round to 0 either way) to the accumulators:
//   sum of terms = (hi - cnt * kMagic43Bits) * 2^20 + (lo - cnt * kMagic23Bits)
// (mod 2^32 each), with cnt the number of terms added; the constant offsets
// are taken out once at the end.
__device__ __forceinline__ void add_terms(f2 x, unsigned& hi, unsigned& lo) {
    const f2 nb = ffma2(x, dup(kLog2e), dup(kMagic23));  // 1.5*2^23 + n
    const f2 n = fsub2(nb, dup(kMagic23));
    f2 r = ffma2(n, dup(-kLn2Hi), x);
    r = ffma2(n, dup(-kLn2Lo), r);
    f2 p = ffma2(dup(kC7), r, dup(kC6));
    p = ffma2(p, r, dup(kC5));
    p = ffma2(p, r, dup(kC4));
    p = ffma2(p, r, dup(kC3));
    p = ffma2(p, r, dup(kC2));
    p = ffma2(p, r, dup(kC0));
    p = ffma2(p, r, dup(kC0));  // 2^40 * p(r), in [2^39.5, 2^40.5]
    float p0, p1, nb0, nb1;
    upk(p, p0, p1);
    upk(nb, nb0, nb1);
    // y = p * 2^n: add n to the exponent field; (bits(nb) << 23) == (n << 23) mod 2^32.
    const f2 y = pk(__uint_as_float(__float_as_uint(p0) + (__float_as_uint(nb0) << 23)),
                    __uint_as_float(__float_as_uint(p1) + (__float_as_uint(nb1) << 23)));
    const f2 a = fadd2(y, dup(kMagic43));               // 1.5*2^43 + 2^20 * round(y / 2^20)
    const f2 rem = fsub2(y, fsub2(a, dup(kMagic43)));   // exact, |rem| <= 2^19
    const f2 b = fadd2(rem, dup(kMagic23));             // 1.5*2^23 + rint(rem)
    float a0, a1, b0, b1;
    upk(a, a0, a1);
    upk(b, b0, b1);
    hi += __float_as_uint(a0) + __float_as_uint(a1);
    lo += __float_as_uint(b0) + __float_as_uint(b1);
}

// (value, index) as one orderable 64-bit word: a larger value wins, equal
// values go to the lower index. -0.0 is folded into +0.0 first (they compare
// equal). 0 is below every encoded pair.
__device__ __forceinline__ unsigned long long enc_argmax(float v, int i) {
    unsigned u = __float_as_uint(v + 0.0f);
    u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    return (static_cast<unsigned long long>(u) << 32) | (0xFFFFFFFFu - static_cast<unsigned>(i));
}
__device__ __forceinline__ float dec_value(unsigned long long e) {
    unsigned u = static_cast<unsigned>(e >> 32);
    u = (u & 0x80000000u) ? (u & 0x7FFFFFFFu) : ~u;
    return __uint_as_float(u);
}
__device__ __forceinline__ int dec_index(unsigned long long e) {
    return static_cast<int>(0xFFFFFFFFu - static_cast<unsigned>(e));
}

}  // namespace key
}  // namespace tt
