// NVFP4 format helpers shared by the quantiser and the GEMM epilogue: the
// fp32 tensor scale S = 2688 / amax (2688 = 6 * 448, the E2M1 and E4M3
// maxima; 1 for an all-zero tensor; capped at the largest finite fp32), E4M3
// scale bytes decoded to fp32, and E2M1 pair conversion.  This is the NVFP4
// recipe the Megatron Core MoE summary names for Blackwell (technical summary
// 2.5), read as the format's own definition: E2M1 elements, one E4M3 scale per
// 16 values along the contraction, one fp32 scale per tensor.
#pragma once
#include <cstdint>
#include <cfloat>

namespace moe {

__device__ __forceinline__ float nv4_tensor_scale(float amax) {
  if (!(amax > 0.f)) return 1.0f;
  const float s = 2688.0f / amax;
  return s <= FLT_MAX ? s : FLT_MAX;
}

// Value of an unsigned E4M3 byte (bias 7; subnormals m * 2^-9), exact in fp32.
// 0x7F (NaN) never occurs: the quantiser saturates to 448.
__device__ __forceinline__ float e4m3_to_f32(uint32_t b) {
  const uint32_t e = (b >> 3) & 15u, m = b & 7u;
  return e == 0 ? static_cast<float>(m) * 0.001953125f : __uint_as_float(((e + 120u) << 23) | (m << 20));
}

// Two values to E2M1 (round to nearest even, saturating to +-6): lo in bits
// 3..0, hi in bits 7..4 -- the element with the lower index in the low nibble.
__device__ __forceinline__ uint32_t cvt_e2m1x2(float lo, float hi) {
  uint32_t r;
  asm("{\n .reg .b8 t;\n cvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n cvt.u32.u8 %0, t;\n}\n"
      : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

}  // namespace moe
