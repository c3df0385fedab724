// MXFP8 quantisation (OCP Microscaling v1.0 with FP8 E4M3 elements): every
// block of 32 consecutive values along the contraction dimension shares one
// E8M0 scale X = 2^(floor(log2 amax) - 8), and each value is stored as
// e4m3(v / X), rounded to nearest even and saturated to +-448.  This is the
// MXFP8 recipe the Megatron Core MoE summary names for Blackwell (technical
// summary 2.5); the block size and element type are the MX format's.
//
// Scales are written in the tiled order the tensor cores' scale-factor copy
// (tcgen05.cp 32x128b, broadcast to the four lane quarters) consumes: one
// 512-byte tile per 128 rows x 4 blocks (128 columns); inside a tile the scale
// of row r, block b sits at byte (r % 32) * 16 + (r / 32) * 4 + b.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "internal.h"
#include "mx_quant.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

// Output row of input row r when the rows come in groups of 2*half (an
// expert's [gate; up] projection) and are interleaved in 128-row blocks:
// gate 0..127, up 0..127, gate 128..255, up 128..255, ...  half == 0: identity.
__device__ __forceinline__ long long gate_up_row(long long r, int half) {
  if (half == 0) return r;
  const long long g = r / (2 * half);
  const int j = static_cast<int>(r % (2 * half));
  const int up = j >= half ? 1 : 0;
  const int jj = j - up * half;
  return g * 2 * half + (jj / 128) * 256 + up * 128 + (jj % 128);
}

// Blocks along the row: src [rows, cols] bf16 -> codes [rows, cols], scales
// tiled.  One thread per 32-value block: four 16-byte loads, two 16-byte
// stores of codes, one scale byte.
__global__ void __launch_bounds__(256) quantize_rows_kernel(const uint4* __restrict__ src, long long rows, int cols,
                                                            int half, int group, const int32_t* __restrict__ row_limit,
                                                            uint8_t* __restrict__ codes, uint8_t* __restrict__ sf) {
  const int nb = cols / 32;
  const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= rows * nb) return;
  const long long r_in = i / nb;
  if (row_limit != nullptr && r_in >= __ldg(row_limit)) return;   // rows past the last expert: never read
  const long long r = gate_up_row(r_in, half);
  const int b = static_cast<int>(i - r_in * nb);
  const uint4* p = src + i * 4;
  uint4 u[4];
  #pragma unroll
  for (int q = 0; q < 4; ++q) u[q] = __ldg(p + q);
  float v[32];
  #pragma unroll
  for (int q = 0; q < 4; ++q) {
    v[8 * q + 0] = bf16_lo(u[q].x); v[8 * q + 1] = bf16_hi(u[q].x);
    v[8 * q + 2] = bf16_lo(u[q].y); v[8 * q + 3] = bf16_hi(u[q].y);
    v[8 * q + 4] = bf16_lo(u[q].z); v[8 * q + 5] = bf16_hi(u[q].z);
    v[8 * q + 6] = bf16_lo(u[q].w); v[8 * q + 7] = bf16_hi(u[q].w);
  }
  const uint8_t s = quantize32(v, codes + r * cols + b * 32);
  sf[mx_sf_offset_g(static_cast<int>(r), b, cols / 128, group)] = s;
}

// Blocks along the column, output transposed: src [rows, cols] bf16 ->
// codes [cols, rows] (row c of the output = column c of the input), scales
// tiled over the [cols, rows] output.  batch: independent matrices one after
// another (expert weights).  A block reads a 128-row x 64-column tile with
// 16-byte loads into shared memory; thread (c, q) quantises rows 32q..32q+31
// of column c.  The four threads of a column sit next to each other in a warp,
// so their 32-byte pieces of one output row form a full 128-byte line.
// Shared memory: element (r, c) in 16-byte chunk (c / 8) ^ (r / 32) of row r,
// so the four row blocks read by one warp fall in different banks.
// row_map (nullable, batch 1 only): input row r is src row row_map[r], or a
// zero row where row_map[r] is outside [0, src_rows) -- the expert-ordered
// rows read straight from token order through row_src, padding rows zero.
__global__ void __launch_bounds__(256) quantize_cols_kernel(const __nv_bfloat16* __restrict__ src, int rows,
                                                            int cols, const int32_t* __restrict__ row_map,
                                                            int src_rows, int group,
                                                            const int32_t* __restrict__ row_limit,
                                                            uint8_t* __restrict__ codes, uint8_t* __restrict__ sf) {
  __shared__ uint4 tile[128][8];           // 128 rows x 64 bf16
  const int rb = blockIdx.x;               // block of 128 input rows
  if (row_limit != nullptr && rb * 128 >= __ldg(row_limit)) return;   // past the last expert: never read
  const int c0 = blockIdx.y * 64;
  const long long mat = blockIdx.z;
  const __nv_bfloat16* base = src + mat * rows * cols + static_cast<long long>(rb) * 128 * cols + c0;
  #pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int i = threadIdx.x + 256 * k;   // 16-byte piece i: row i / 8, chunk i % 8
    const int r = i >> 3, j = i & 7;
    uint4 v;
    if (row_map != nullptr) {
      const int t = row_map[rb * 128 + r];
      v = (t >= 0 && t < src_rows)
              ? __ldg(reinterpret_cast<const uint4*>(src + static_cast<long long>(t) * cols + c0) + j)
              : make_uint4(0, 0, 0, 0);
    } else {
      v = __ldg(reinterpret_cast<const uint4*>(base + static_cast<long long>(r) * cols) + j);
    }
    tile[r][j ^ (r >> 5)] = v;
  }
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int cl = warp * 8 + (lane >> 2);   // column inside the tile
  const int q = lane & 3;                  // block of 32 rows inside the tile
  const __nv_bfloat16* t = reinterpret_cast<const __nv_bfloat16*>(&tile[0][0]);
  float v[32];
  #pragma unroll
  for (int i = 0; i < 32; ++i) {
    const int r = 32 * q + i;
    v[i] = __bfloat162float(t[r * 64 + (((cl >> 3) ^ q) << 3) + (cl & 7)]);
  }
  const int c = c0 + cl;
  uint8_t* out = codes + mat * rows * cols + static_cast<long long>(c) * rows + rb * 128 + 32 * q;
  const uint8_t e = quantize32(v, out);
  // scale bytes of one matrix: its output rows (the input columns) in groups
  const long long mat_sf = static_cast<long long>(group == 128 ? cols / 128 : 2 * (cols / group)) * rows * 4;
  sf[mat * mat_sf + mx_sf_offset_g(c, rb * 4 + q, rows / 128, group)] = e;
}

// Padding rows of expert e's segment: zero codes and the scale of an
// all-zero block (byte 0), as quantising zero rows would give.
__device__ __forceinline__ void zero_pad_rows_mx(const int32_t* __restrict__ counts,
                                                 const int32_t* __restrict__ poffsets, int e, int H,
                                                 uint4* __restrict__ codes, uint8_t* __restrict__ sf) {
  const int r0 = poffsets[e] + counts[e], r1 = poffsets[e + 1];
  const int nv = H / 16, nb = H / 32;
  const long long n = static_cast<long long>(r1 - r0) * nv;
  uint4* base = codes + static_cast<long long>(r0) * nv;
  for (long long i = threadIdx.x; i < n; i += blockDim.x) base[i] = make_uint4(0, 0, 0, 0);
  const long long m = static_cast<long long>(r1 - r0) * nb;
  for (long long i = threadIdx.x; i < m; i += blockDim.x)
    sf[mx_sf_offset(r0 + static_cast<int>(i / nb), static_cast<int>(i % nb), H / 128)] = 0;
}

// Token-order quantised rows (codes [T, H] and their scale tiles) -> expert
// order: the same permutation as the bf16 gather, on codes and scales.  Row
// blocks of 32 lie along H, so a row's codes do not depend on where it goes.
// Blocks 0 .. E_pad - 1 zero the padding rows of expert `block` in the same
// launch (first, so they overlap the gathers rather than trail them).
__global__ void __launch_bounds__(128) gather_rows_mx_kernel(const uint4* __restrict__ codes_tok,
                                                             const uint8_t* __restrict__ sf_tok,
                                                             const int32_t* __restrict__ slot_row, int E_pad, int k,
                                                             int H, const int32_t* __restrict__ counts,
                                                             const int32_t* __restrict__ poffsets,
                                                             uint4* __restrict__ codes_perm,
                                                             uint8_t* __restrict__ sf_perm) {
  if (static_cast<int>(blockIdx.x) < E_pad) {
    zero_pad_rows_mx(counts, poffsets, blockIdx.x, H, codes_perm, sf_perm);
    return;
  }
  const int t = blockIdx.x - E_pad;
  __shared__ int s_rows[kMaxK];
  if (threadIdx.x < k) s_rows[threadIdx.x] = slot_row[static_cast<long long>(t) * k + threadIdx.x];
  __syncthreads();
  const int nv = H / 16;
  for (int v = threadIdx.x; v < nv; v += blockDim.x) {
    const uint4 c = __ldg(codes_tok + static_cast<long long>(t) * nv + v);
    for (int i = 0; i < k; ++i) {
      const int r = s_rows[i];
      if (r >= 0) codes_perm[static_cast<long long>(r) * nv + v] = c;
    }
  }
  const int nb = H / 32, tiles = H / 128;
  for (int b = threadIdx.x; b < nb; b += blockDim.x) {
    const uint8_t e = sf_tok[mx_sf_offset(t, b, tiles)];
    for (int i = 0; i < k; ++i) {
      const int r = s_rows[i];
      if (r >= 0) sf_perm[mx_sf_offset(r, b, tiles)] = e;
    }
  }
}

}  // namespace

cudaError_t launch_quantize_rows(const void* src, long long rows, int cols, int gate_up_half, uint8_t* codes,
                                 uint8_t* sf, cudaStream_t st, int group, const int32_t* row_limit) {
  const long long n = rows * (cols / 32);
  if (n == 0) return cudaSuccess;
  quantize_rows_kernel<<<static_cast<unsigned>((n + 255) / 256), 256, 0, st>>>(
      static_cast<const uint4*>(src), rows, cols, gate_up_half, group, row_limit, codes, sf);
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_quantize_cols(const void* src, int batch, int rows, int cols, uint8_t* codes, uint8_t* sf,
                                 cudaStream_t st, int group, const int32_t* row_limit) {
  if (batch == 0 || rows == 0 || cols == 0) return cudaSuccess;
  dim3 grid(rows / 128, cols / 64, batch);   // rows % 128 == 0 and cols % 128 == 0 (checked by the callers)
  quantize_cols_kernel<<<grid, 256, 0, st>>>(static_cast<const __nv_bfloat16*>(src), rows, cols, nullptr, 0, group,
                                             row_limit, codes, sf);
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_quantize_cols_gather(const void* src, int src_rows, const int32_t* row_map, int rows, int cols,
                                        uint8_t* codes, uint8_t* sf, cudaStream_t st, int group,
                                        const int32_t* row_limit) {
  if (rows == 0 || cols == 0) return cudaSuccess;
  dim3 grid(rows / 128, cols / 64, 1);
  quantize_cols_kernel<<<grid, 256, 0, st>>>(static_cast<const __nv_bfloat16*>(src), rows, cols, row_map, src_rows,
                                             group, row_limit, codes, sf);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace moe

namespace moe {
cudaError_t launch_gather_rows_mx(const uint8_t* codes_tok, const uint8_t* sf_tok, const int32_t* slot_row, int T,
                                  int k, int H, uint8_t* codes_perm, uint8_t* sf_perm, cudaStream_t st,
                                  const int32_t* counts, const int32_t* poffsets, int E_pad) {
  if (T + E_pad == 0) return cudaSuccess;
  gather_rows_mx_kernel<<<T + E_pad, 128, 0, st>>>(reinterpret_cast<const uint4*>(codes_tok), sf_tok, slot_row,
                                                   E_pad, k, H, counts, poffsets,
                                                   reinterpret_cast<uint4*>(codes_perm), sf_perm);
  count_launches(1);
  return cudaGetLastError();
}
}  // namespace moe
