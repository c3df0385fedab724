// NVFP4 quantisation: every block of 16 consecutive values along the
// contraction shares one unsigned E4M3 scale, and the tensor has one fp32
// scale S = 2688 / amax.  With d = fp32(amax_b / 6):
//   s    = e4m3(fp32(d * S))        (round to nearest even, saturated to 448)
//   r    = fp32(S / s)              (0 when s is 0; capped at the largest fp32)
//   code = e2m1(fp32(v * r))        (round to nearest even, saturated to +-6)
// so that v ~ e2m1(code) * s / S.  This is the NVFP4 recipe the Megatron Core
// MoE summary names for Blackwell (technical summary 2.5), read as the
// format's own definition; every decision is taken in fp32 in this order.
//
// Codes: two per byte, the lower-indexed element in the low nibble.  Scales:
// one 512-byte tile per 128 rows x 64 columns (4 blocks), tile (i, j) of a
// [R, C] matrix at byte (i * (C/64) + j) * 512; inside it the scale of row r,
// block b at (r % 32) * 16 + (r / 32 % 4) * 4 + b % 4 -- the order in which
// the tensor cores read the scales of one MMA of K = 64.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "internal.h"
#include "nvfp4.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

__device__ __forceinline__ uint32_t cvt_e4m3(float v) {
  uint16_t d;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(d) : "f"(0.0f), "f"(v));   // low byte: e4m3(v)
  return d & 0xFFu;
}

__device__ __forceinline__ size_t sf_offset16(long long r, int b, int tiles_per_row) {
  return (static_cast<size_t>(r >> 7) * tiles_per_row + (b >> 2)) * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4 +
         (b & 3);
}

// Output row of input row r for an expert's [gate; up] rows interleaved in
// 128-row blocks (gate 0..127, up 0..127, gate 128..255, ...); half == 0: identity.
__device__ __forceinline__ long long gate_up_row16(long long r, int half) {
  if (half == 0) return r;
  const long long g = r / (2 * half);
  const int j = static_cast<int>(r % (2 * half));
  const int up = j >= half ? 1 : 0;
  const int jj = j - up * half;
  return g * 2 * half + (jj / 128) * 256 + up * 128 + (jj % 128);
}

// Largest |v| of a bf16 tensor [rows, cols] -> *out (as fp32 bits; *out is
// zeroed by the launcher first).  row_src != nullptr: rows with row_src < 0
// (padding of the expert-ordered buffers) are skipped; rows_end != nullptr:
// only rows below *rows_end count (the expert-ordered buffers' used rows).
__global__ void __launch_bounds__(256) amax_bf16_kernel(const uint4* __restrict__ src, long long nvec,
                                                        int vec_per_row, const int32_t* __restrict__ row_src,
                                                        const int32_t* __restrict__ rows_end,
                                                        unsigned* __restrict__ out) {
  pdl_entry();
  float m = 0.f;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  if (rows_end != nullptr) {
    const long long e = static_cast<long long>(__ldg(rows_end)) * vec_per_row;
    if (e < nvec) nvec = e > 0 ? e : 0;
  }
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < nvec; i += stride) {
    if (row_src != nullptr && __ldg(row_src + i / vec_per_row) < 0) continue;
    const uint4 u = __ldg(src + i);
    m = fmaxf(m, fmaxf(fmaxf(fabsf(bf16_lo(u.x)), fabsf(bf16_hi(u.x))), fmaxf(fabsf(bf16_lo(u.y)), fabsf(bf16_hi(u.y)))));
    m = fmaxf(m, fmaxf(fmaxf(fabsf(bf16_lo(u.z)), fabsf(bf16_hi(u.z))), fmaxf(fabsf(bf16_lo(u.w)), fabsf(bf16_hi(u.w)))));
  }
  #pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  __shared__ float part[8];
  if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < static_cast<int>(blockDim.x >> 5); ++w) m = fmaxf(m, part[w]);
    atomicMax(out, __float_as_uint(m));      // non-negative floats order as their bit patterns
  }
}

// One block of 16 values (two 16-byte loads of bf16) -> eight code bytes
// (w[0], w[1]) and the scale byte, with the tensor scale S.
__device__ __forceinline__ uint32_t quantize16(const uint4* p, float S, uint32_t (&w)[2]) {
  const uint4 u0 = __ldg(p), u1 = __ldg(p + 1);
  const float v[16] = {bf16_lo(u0.x), bf16_hi(u0.x), bf16_lo(u0.y), bf16_hi(u0.y),
                       bf16_lo(u0.z), bf16_hi(u0.z), bf16_lo(u0.w), bf16_hi(u0.w),
                       bf16_lo(u1.x), bf16_hi(u1.x), bf16_lo(u1.y), bf16_hi(u1.y),
                       bf16_lo(u1.z), bf16_hi(u1.z), bf16_lo(u1.w), bf16_hi(u1.w)};
  float amax_b = 0.f;
  #pragma unroll
  for (int j = 0; j < 16; ++j) amax_b = fmaxf(amax_b, fabsf(v[j]));
  const float d = amax_b / 6.0f;
  const uint32_t s = cvt_e4m3(d * S);
  const float sv = e4m3_to_f32(s);
  float rr = sv > 0.f ? S / sv : 0.f;
  if (!(rr <= FLT_MAX)) rr = FLT_MAX;
  w[0] = w[1] = 0u;
  #pragma unroll
  for (int j = 0; j < 8; ++j) w[j >> 2] |= cvt_e2m1x2(v[2 * j] * rr, v[2 * j + 1] * rr) << (8 * (j & 3));
  return s;
}

// Blocks of 16 along each row: src [rows, cols] bf16 -> codes [rows, cols/2]
// bytes, scale tiles.  One thread per block: two 16-byte loads, one 8-byte
// store of codes, one scale byte.
__global__ void __launch_bounds__(256) quantize_rows_nv4_kernel(const uint4* __restrict__ src, long long rows,
                                                                int cols, int half, const float* __restrict__ amax_p,
                                                                uint8_t* __restrict__ codes,
                                                                uint8_t* __restrict__ sf) {
  pdl_entry();
  const int nb = cols / 16;
  const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= rows * nb) return;
  const long long r_in = i / nb;
  const long long r = gate_up_row16(r_in, half);
  const int b = static_cast<int>(i - r_in * nb);
  uint32_t w[2];
  const uint32_t s = quantize16(src + 2 * i, nv4_tensor_scale(__ldg(amax_p)), w);
  *reinterpret_cast<uint2*>(codes + r * (cols / 2) + b * 8) = make_uint2(w[0], w[1]);
  sf[sf_offset16(r, b, cols / 64)] = static_cast<uint8_t>(s);
}

// Token rows of x [T, H] quantised straight into expert order: block b of
// token t goes to each of its k padded rows (slot_row), and to row t of the
// token-order copy when one is asked for (the shared expert reads it).  The
// codes of a row do not depend on where the row goes (blocks lie along H).
__global__ void __launch_bounds__(256) quantize_gather_nv4_kernel(const uint4* __restrict__ src, int T, int H,
                                                                  const int32_t* __restrict__ slot_row, int k,
                                                                  const float* __restrict__ amax_p,
                                                                  uint8_t* __restrict__ codes_perm,
                                                                  uint8_t* __restrict__ sf_perm,
                                                                  uint8_t* __restrict__ codes_tok,
                                                                  uint8_t* __restrict__ sf_tok) {
  pdl_entry();
  const int nb = H / 16;
  const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= static_cast<long long>(T) * nb) return;
  const int t = static_cast<int>(i / nb);
  const int b = static_cast<int>(i - static_cast<long long>(t) * nb);
  uint32_t w[2];
  const uint32_t s = quantize16(src + 2 * i, nv4_tensor_scale(__ldg(amax_p)), w);
  const uint2 c = make_uint2(w[0], w[1]);
  for (int j = 0; j < k; ++j) {
    const int r = __ldg(slot_row + static_cast<long long>(t) * k + j);
    if (r < 0) continue;
    *reinterpret_cast<uint2*>(codes_perm + static_cast<long long>(r) * (H / 2) + b * 8) = c;
    sf_perm[sf_offset16(r, b, H / 64)] = static_cast<uint8_t>(s);
  }
  if (codes_tok != nullptr) {
    *reinterpret_cast<uint2*>(codes_tok + static_cast<long long>(t) * (H / 2) + b * 8) = c;
    sf_tok[sf_offset16(t, b, H / 64)] = static_cast<uint8_t>(s);
  }
}

}  // namespace

cudaError_t launch_amax_bf16(const void* src, long long rows, int cols, const int32_t* row_src,
                             const int32_t* rows_end, float* amax, cudaStream_t st) {
  cudaError_t e = cudaMemsetAsync(amax, 0, sizeof(float), st);
  if (e != cudaSuccess || rows == 0) return e;
  const long long nvec = rows * (cols / 8);
  long long blocks = (nvec + 255) / 256;
  const long long cap = 4LL * num_sms();
  if (blocks > cap) blocks = cap;
  launch_k(amax_bf16_kernel, static_cast<unsigned>(blocks), 256, 0, st, static_cast<const uint4*>(src), nvec, cols / 8,
                                                                   row_src, rows_end, reinterpret_cast<unsigned*>(amax));
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_quantize_rows_nv4(const void* src, long long rows, int cols, int gate_up_half,
                                     const float* amax, uint8_t* codes, uint8_t* sf, cudaStream_t st) {
  const long long n = rows * (cols / 16);
  if (n == 0) return cudaSuccess;
  launch_k(quantize_rows_nv4_kernel, static_cast<unsigned>((n + 255) / 256), 256, 0, st, 
      static_cast<const uint4*>(src), rows, cols, gate_up_half, amax, codes, sf);
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_quantize_gather_nv4(const void* x, int T, int H, const int32_t* slot_row, int k,
                                      const float* amax, uint8_t* codes_perm, uint8_t* sf_perm, uint8_t* codes_tok,
                                      uint8_t* sf_tok, cudaStream_t st) {
  const long long n = static_cast<long long>(T) * (H / 16);
  if (n == 0) return cudaSuccess;
  launch_k(quantize_gather_nv4_kernel, static_cast<unsigned>((n + 255) / 256), 256, 0, st, 
      static_cast<const uint4*>(x), T, H, slot_row, k, amax, codes_perm, sf_perm, codes_tok, sf_tok);
  count_launches(1);
  return cudaGetLastError();
}


}  // namespace moe
