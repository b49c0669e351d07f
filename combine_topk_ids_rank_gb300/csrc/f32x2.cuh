// f32x2.cuh -- paired binary32 arithmetic (PTX .f32x2, sm_100 family): one
// instruction performs the same IEEE operation, round-to-nearest-even, on
// two independent fp32 lanes held in a 64-bit register pair.  Each lane's
// result is bit-identical to the scalar add.rn / mul.rn / fma.rn.f32 of
// that lane (no flush to zero; measured on 2^20 random and special pairs).
// Unlike the scalar forms with an explicit rounding mode, a paired multiply
// whose result feeds a paired add was measured to be contracted into one
// fused multiply-add (one rounding instead of two): where both roundings
// matter, form the products with scalar multiplies.
#pragma once

#include <cstdint>

namespace moe {
namespace x2 {

using f2 = unsigned long long;  // (low lane, high lane)

__device__ __forceinline__ f2 pack(float lo, float hi) {
    f2 r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}

__device__ __forceinline__ void unpack(f2 v, float &lo, float &hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}

__device__ __forceinline__ f2 add(f2 a, f2 b) {
    f2 d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

__device__ __forceinline__ f2 mul(f2 a, f2 b) {
    f2 d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// a * b + c with one rounding per lane
__device__ __forceinline__ f2 fma(f2 a, f2 b, f2 c) {
    f2 d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

// The two bf16 halves of a 32-bit word as binary32 (exact): low half in the
// low lane.
__device__ __forceinline__ f2 bf16x2(uint32_t w) {
    return pack(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

}  // namespace x2
}  // namespace moe
