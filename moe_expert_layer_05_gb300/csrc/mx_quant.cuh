// MXFP8 block quantisation on the device, shared by the standalone quantisers
// and the GEMM epilogues that emit quantised outputs: OCP Microscaling v1.0
// with FP8 E4M3 elements -- a block of 32 values shares the E8M0 scale
// X = 2^(floor(log2 amax) - 8) (2^-127 for an all-zero block), each value is
// stored as e4m3(v / X) rounded to nearest even and saturated to +-448.
//
// Scale tiles: one 512-byte tile per 128 rows x 4 blocks (128 columns);
// inside a tile the scale of row r, block b sits at byte
// (r % 32) * 16 + (r / 32) * 4 + b -- the order the tensor cores' scale-factor
// copy (tcgen05.cp 32x128b, broadcast to the four lane quarters) consumes.
#pragma once
#include <cstdint>

namespace moe {

__device__ __forceinline__ uint16_t cvt_e4m3x2(float lo, float hi) {
  uint16_t d;
  // d[15:8] = e4m3(first source), d[7:0] = e4m3(second source)
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(d) : "f"(hi), "f"(lo));
  return d;
}

// E8M0 exponent of a block whose largest magnitude is amax.
__device__ __forceinline__ int mx_exponent(float amax) {
  if (!(amax > 0.f)) return -127;
  int e = ilogbf(amax) - 8;
  return e < -127 ? -127 : (e > 127 ? 127 : e);
}

// 2^-e as a float, e in [-127, 127] (2^-127 is subnormal).  Multiplying by a
// power of two is exact except where the product is subnormal, and there it
// rounds once to nearest even, exactly like scaling by 2^-e.
__device__ __forceinline__ float pow2_neg(int e) {
  return e < 127 ? __int_as_float((127 - e) << 23) : __int_as_float(0x00400000);
}

__device__ __forceinline__ size_t mx_sf_offset(int r, int b, int tiles_per_row) {
  return (static_cast<size_t>(r >> 7) * tiles_per_row + (b >> 2)) * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4 +
         (b & 3);
}

// The same with the rows taken in groups of `group` (128, or 224 for the B
// operand of 224-wide GEMM tiles): group g starts a new tile row, its rows
// 0..127 fill tile row 2g and rows 128..223 the first 96 rows of tile row
// 2g + 1 (the other 32 rows of that tile are never read).
__device__ __forceinline__ size_t mx_sf_offset_g(int r, int b, int tiles_per_row, int group) {
  if (group == 128) return mx_sf_offset(r, b, tiles_per_row);
  const int g = r / group, i = r - g * group;
  const int tr = 2 * g + (i >> 7), rr = i & 127;
  return (static_cast<size_t>(tr) * tiles_per_row + (b >> 2)) * 512 + (rr & 31) * 16 + ((rr >> 5) & 3) * 4 + (b & 3);
}

// max(a, |b|, |c|) in one three-input maximum
__device__ __forceinline__ float max_abs2(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(fabsf(b)), "f"(fabsf(c)));
  return d;
}

// The largest magnitude of 32 values (exact: a maximum rounds nothing).
__device__ __forceinline__ float amax32(const float (&v)[32]) {
  float amax = 0.f;
  #pragma unroll
  for (int i = 0; i < 16; ++i) amax = max_abs2(amax, v[2 * i], v[2 * i + 1]);
  return amax;
}

// (a * s, b * s), each rounded to nearest as a plain fp32 product, in one
// packed two-lane multiply
__device__ __forceinline__ void mul2(float a, float b, float s, float& x, float& y) {
  asm("{\n\t.reg .b64 p, q, r;\n\t"
      "mov.b64 p, {%2, %3};\n\t"
      "mov.b64 q, {%4, %4};\n\t"
      "mul.rn.f32x2 r, p, q;\n\t"
      "mov.b64 {%0, %1}, r;\n\t}"
      : "=f"(x), "=f"(y)
      : "f"(a), "f"(b), "f"(s));
}

// Pack 32 values (scaled by sc) into 8 words of E4M3 codes, value i in byte i.
__device__ __forceinline__ void e4m3_pack32(const float (&v)[32], float sc, uint32_t (&w)[8]) {
  #pragma unroll
  for (int i = 0; i < 8; ++i) {
    float a, b, c, d;
    mul2(v[4 * i + 0], v[4 * i + 1], sc, a, b);
    mul2(v[4 * i + 2], v[4 * i + 3], sc, c, d);
    w[i] = static_cast<uint32_t>(cvt_e4m3x2(a, b)) | (static_cast<uint32_t>(cvt_e4m3x2(c, d)) << 16);
  }
}

// Quantise 32 values held by this thread; writes 32 code bytes and returns the scale byte.
__device__ __forceinline__ uint8_t quantize32(const float (&v)[32], uint8_t* dst) {
  const int e = mx_exponent(amax32(v));
  uint32_t w[8];
  e4m3_pack32(v, pow2_neg(e), w);
  uint4* d = reinterpret_cast<uint4*>(dst);
  d[0] = make_uint4(w[0], w[1], w[2], w[3]);
  d[1] = make_uint4(w[4], w[5], w[6], w[7]);
  return static_cast<uint8_t>(e + 127);
}

// Four values to four E4M3 codes, value i in byte i.
__device__ __forceinline__ uint32_t e4m3_pack4(float a, float b, float c, float d) {
  return static_cast<uint32_t>(cvt_e4m3x2(a, b)) | (static_cast<uint32_t>(cvt_e4m3x2(c, d)) << 16);
}

}  // namespace moe
