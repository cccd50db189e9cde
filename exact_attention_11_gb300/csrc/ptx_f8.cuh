// ptx_f8.cuh -- 8-bit (E4M3) helpers for sm_103a: tcgen05 MMAs of
// kind::f8f6f4 and fp32 -> E4M3 conversion.  Shared-memory descriptors use
// the same 128-byte-swizzle format as the 16-bit path (see ptx.cuh); only the
// instruction kind and the operand type fields differ.
#pragma once

#include <cstdint>

#include "ptx.cuh"

namespace fattn {

// Instruction descriptor, kind::f8f6f4: A and B E4M3 (type fields 0), both
// K-major, fp32 accumulator (bit 4); N >> 3 at bit 17, M >> 4 at bit 24.
__host__ __device__ constexpr uint32_t idesc_e4m3_f32(int M, int N) {
  return (1u << 4) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

// D (+)= A B with A and B in shared memory (descriptor low words; high word
// kSdescHi1024).  One MMA covers K = 32 (32 bytes of each operand row).
__device__ __forceinline__ void mma_f8_ss_lo(uint32_t d_tmem, uint32_t a_lo, uint32_t b_lo,
                                             uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .b64 da, db;\n .reg .pred p;\n mov.b64 da, {%1, %5};\n mov.b64 db, {%2, %5};\n"
      " setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], da, db, %3, p;\n}\n" ::"r"(d_tmem),
      "r"(a_lo), "r"(b_lo), "r"(idesc), "r"(accumulate), "r"(kSdescHi1024)
      : "memory");
}

// Four fp32 values -> four E4M3 codes in one word (x0 in the lowest byte),
// each rounded to nearest even and saturated to +-448.
__device__ __forceinline__ uint32_t pack_e4m3x4(float x0, float x1, float x2, float x3) {
  uint32_t r;
  asm("{\n .reg .b16 lo, hi;\n"
      " cvt.rn.satfinite.e4m3x2.f32 lo, %2, %1;\n"
      " cvt.rn.satfinite.e4m3x2.f32 hi, %4, %3;\n"
      " mov.b32 %0, {lo, hi};\n}\n"
      : "=r"(r)
      : "f"(x0), "f"(x1), "f"(x2), "f"(x3));
  return r;
}

}  // namespace fattn
