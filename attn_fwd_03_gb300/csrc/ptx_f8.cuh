// ptx_f8.cuh — 8-bit floating-point (E4M3) pieces of the tcgen05 kernels: the
// kind::f8f6f4 instruction descriptor and MMAs, and packing of fp32 values into
// E4M3 codes. Shared by the FP8 forward kernels.
#pragma once
#include <cstdint>

#include "ptx.cuh"

namespace attn {
namespace ptx_f8 {

// Instruction descriptor of kind::f8f6f4 with E4M3 A and B (format code 0) and fp32 D:
//   [4,6) D format (1 = f32)   [7,10) A format   [10,13) B format
//   [15] A major (0 = K, 1 = MN)   [16] B major   [17,23) N >> 3   [24,29) M >> 4
__host__ __device__ constexpr uint32_t idesc_e4m3(int M, int N, bool a_mn, bool b_mn) {
    return (1u << 4) | ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) | ((uint32_t)(N >> 3) << 17) |
           ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma_f8_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void mma_f8_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n\t}\n" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Four floats -> four E4M3 codes (round to nearest even, saturating), x0 in the lowest
// byte. The paired convert puts its first source in the upper byte.
__device__ __forceinline__ uint32_t pack_e4m3x4(float x0, float x1, float x2, float x3) {
    uint16_t lo, hi;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(x1), "f"(x0));
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(x3), "f"(x2));
    return (uint32_t)lo | ((uint32_t)hi << 16);
}

// E4M3 rounding of x (0 <= x <= 448) as a float.
__device__ __forceinline__ float round_e4m3(float x) {
    uint16_t c;
    uint32_t h;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %1;" : "=h"(c) : "f"(x));
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"(c));
    return ptx::unpack_h16<true>(h).x;
}

// ptx::o_divisor for P rounded to E4M3.
__device__ __forceinline__ float o_divisor_e4m3(float l, float m_row, float m_ref) {
    if (!(l > 0.f)) return 0.f;
    const float pm = ptx::ex2(m_row - m_ref);
    return l + (round_e4m3(pm) - pm);
}

}  // namespace ptx_f8
}  // namespace attn
