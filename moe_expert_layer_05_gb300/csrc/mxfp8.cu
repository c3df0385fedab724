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
  pdl_entry();
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
// another (expert weights).  Tiles of 128 rows x 64 columns; thread (c, q)
// quantises rows 32q..32q+31 of column c.  The four threads of a column sit
// next to each other in a warp, so their 32-byte pieces of one output row form
// a full 128-byte line.  Shared memory: element (r, c) in 16-byte chunk
// (c / 8) ^ (r / 32) of row r, so the four row blocks read by one warp fall in
// different banks.
// Persistent: a block walks tiles blockIdx.x, + gridDim.x, ... (row blocks
// fastest, then column blocks, then matrices, so the blocks in flight share
// one 64-column slice of the source), quantising one tile while the next
// one's rows land in the other half of a double buffer (cp.async, 16-byte
// pieces, zero-filled for zero rows) and the row indices of the one after are
// read.  The tile walk steps without divisions (with 64-bit divisions per tile
// the kernel was slower than the one-shot version it replaced).
// row_map (nullable, batch 1 only): input row r is src row row_map[r], or a
// zero row where row_map[r] is outside [0, src_rows) -- the expert-ordered
// rows read straight from token order through row_src, padding rows zero.
// row_limit (nullable): row blocks from row_limit[0] on are neither read nor
// written (rows past the last expert).
template <int GROUP>
__global__ void __launch_bounds__(256) quantize_cols_kernel(const __nv_bfloat16* __restrict__ src, int batch,
                                                            int rows, int cols,
                                                            const int32_t* __restrict__ row_map, int src_rows,
                                                            const int32_t* __restrict__ row_limit,
                                                            uint8_t* __restrict__ codes, uint8_t* __restrict__ sf) {
  pdl_entry();
  __shared__ uint4 tile[2][128 * 8];       // two 128-row x 64-column tiles
  int nrb = rows / 128;
  if (row_limit != nullptr) nrb = min(nrb, (__ldg(row_limit) + 127) / 128);
  const int ncb = cols / 64;
  const int total = nrb * ncb * batch;
  const int G = static_cast<int>(gridDim.x);
  int t = static_cast<int>(blockIdx.x);
  if (t >= total) return;
  const int j = threadIdx.x & 7, r0 = threadIdx.x >> 3;   // pieces: rows r0 + 32 k, chunk j
  const int lim = row_map != nullptr ? src_rows : rows;
  int idx[4];
  auto rows_of = [&](int rb) {
    #pragma unroll
    for (int k = 0; k < 4; ++k)
      idx[k] = row_map != nullptr ? __ldg(row_map + rb * 128 + r0 + 32 * k) : rb * 128 + r0 + 32 * k;
  };
  auto issue = [&](int rb, int cb, int mat, int buf) {
    const __nv_bfloat16* m = src + static_cast<long long>(mat) * rows * cols + cb * 64 + 8 * j;
    #pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int r = r0 + 32 * k;
      const bool ok = idx[k] >= 0 && idx[k] < lim;
      cp_async_16(smem_u32(&tile[buf][r * 8 + (j ^ (r >> 5))]), ok ? m + static_cast<long long>(idx[k]) * cols : src,
                  ok ? 16u : 0u);
    }
  };
  const int g_cb = G / nrb, g_rb = G - g_cb * nrb;   // one step of G tiles: column blocks and rows blocks
  auto advance = [&](int& rb, int& cb, int& mat) {
    rb += g_rb;
    cb += g_cb;
    if (rb >= nrb) { rb -= nrb; ++cb; }
    if (batch > 1) { mat += cb / ncb; cb %= ncb; }   // (batch 1: t < total keeps cb < ncb)
  };
  int rb = t % nrb, cb = (t / nrb) % ncb, mat = t / (nrb * ncb);
  rows_of(rb);
  issue(rb, cb, mat, 0);
  cp_async_commit();
  int rbn = rb, cbn = cb, matn = mat;
  advance(rbn, cbn, matn);
  if (t + G < total) rows_of(rbn);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int cl = warp * 8 + (lane >> 2);   // column inside the tile
  const int q = lane & 3;                  // block of 32 rows inside the tile
  // scale bytes of one matrix: its output rows (the input columns) in groups
  const long long mat_sf = static_cast<long long>(GROUP == 128 ? cols / 128 : 2 * (cols / GROUP)) * rows * 4;
  for (int buf = 0; t < total; t += G, buf ^= 1) {
    if (t + G < total) issue(rbn, cbn, matn, buf ^ 1);
    cp_async_commit();
    int rb2 = rbn, cb2 = cbn, mat2 = matn;
    advance(rb2, cb2, mat2);
    if (t + 2 * G < total) rows_of(rb2);   // (read while this tile is quantised)
    cp_async_wait<1>();                    // this thread's pieces of tile t have landed
    __syncthreads();
    const __nv_bfloat16* tb = reinterpret_cast<const __nv_bfloat16*>(&tile[buf][0]);
    float v[32];
    #pragma unroll
    for (int i = 0; i < 32; ++i) {
      const int r = 32 * q + i;
      v[i] = __bfloat162float(tb[r * 64 + (((cl >> 3) ^ q) << 3) + (cl & 7)]);
    }
    __syncthreads();                       // the buffer may be refilled (two tiles on)
    const int c = cb * 64 + cl;
    uint8_t* out = codes + static_cast<long long>(mat) * rows * cols + static_cast<long long>(c) * rows + rb * 128 +
                   32 * q;
    const uint8_t e = quantize32(v, out);
    sf[mat * mat_sf + mx_sf_offset_g(c, rb * 4 + q, rows / 128, GROUP)] = e;
    rb = rbn; cb = cbn; mat = matn;
    rbn = rb2; cbn = cb2; matn = mat2;
  }
}

// Padding rows of expert e's segment: zero codes and the scale of an
// all-zero block (byte 0), as quantising zero rows would give.
__device__ __forceinline__ void zero_pad_rows_mx(const int32_t* __restrict__ counts,
                                                 const int32_t* __restrict__ poffsets, int e, int H,
                                                 uint4* __restrict__ codes, uint8_t* __restrict__ sf) {
  const int r0 = poffsets[e] + counts[e], r1 = poffsets[e + 1];
  const int nv = H / 16;
  const long long n = static_cast<long long>(r1 - r0) * nv;
  uint4* base = codes + static_cast<long long>(r0) * nv;
  for (long long i = threadIdx.x; i < n; i += blockDim.x) base[i] = make_uint4(0, 0, 0, 0);
  const int tiles = H / 128;                  // a row's four scales of a tile: one 32-bit word
  const long long m = static_cast<long long>(r1 - r0) * tiles;
  for (long long i = threadIdx.x; i < m; i += blockDim.x)
    *reinterpret_cast<uint32_t*>(sf + mx_sf_offset(r0 + static_cast<int>(i / tiles),
                                                   4 * static_cast<int>(i % tiles), tiles)) = 0u;
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
  pdl_entry();
  if (static_cast<int>(blockIdx.x) < E_pad) {
    zero_pad_rows_mx(counts, poffsets, blockIdx.x, H, codes_perm, sf_perm);
    return;
  }
  const int t = blockIdx.x - E_pad;
  __shared__ int s_rows[kMaxK];
  if (threadIdx.x < k) s_rows[threadIdx.x] = slot_row[static_cast<long long>(t) * k + threadIdx.x];
  __syncthreads();
  const int nv = H / 16;
  const uint4* src = codes_tok + static_cast<long long>(t) * nv;
  for (int v0 = threadIdx.x; v0 < nv; v0 += 4 * blockDim.x) {
    uint4 c[4];                                    // four 16-byte loads in flight before the stores
    #pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int v = v0 + u * blockDim.x;
      if (v < nv) c[u] = __ldg(src + v);
    }
    for (int i = 0; i < k; ++i) {
      const int r = s_rows[i];
      if (r < 0) continue;
      uint4* dst = codes_perm + static_cast<long long>(r) * nv;
      #pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int v = v0 + u * blockDim.x;
        if (v < nv) dst[v] = c[u];
      }
    }
  }
  // scales: a row's four blocks of one 128-column tile are four adjacent
  // bytes in the tiled layout, so they move as one 32-bit word
  const int tiles = H / 128;
  for (int j = threadIdx.x; j < tiles; j += blockDim.x) {
    const uint32_t w = *reinterpret_cast<const uint32_t*>(sf_tok + mx_sf_offset(t, 4 * j, tiles));
    for (int i = 0; i < k; ++i) {
      const int r = s_rows[i];
      if (r >= 0) *reinterpret_cast<uint32_t*>(sf_perm + mx_sf_offset(r, 4 * j, tiles)) = w;
    }
  }
}

}  // namespace

cudaError_t launch_quantize_rows(const void* src, long long rows, int cols, int gate_up_half, uint8_t* codes,
                                 uint8_t* sf, cudaStream_t st, int group, const int32_t* row_limit) {
  const long long n = rows * (cols / 32);
  if (n == 0) return cudaSuccess;
  launch_k(quantize_rows_kernel, static_cast<unsigned>((n + 255) / 256), 256, 0, st, 
      static_cast<const uint4*>(src), rows, cols, gate_up_half, group, row_limit, codes, sf);
  count_launches(1);
  return cudaGetLastError();
}

namespace {
// The persistent column quantiser with as many blocks as are resident on the
// GPU at once, at most one per tile; the scale grouping (128 or 224 rows) is
// a template argument so that its row-group division is a constant one.
template <int GROUP>
cudaError_t launch_cols(const void* src, int batch, int rows, int cols, const int32_t* row_map, int src_rows,
                        const int32_t* row_limit, uint8_t* codes, uint8_t* sf, cudaStream_t st) {
  const long long tiles = static_cast<long long>(batch) * (rows / 128) * (cols / 64);
  if (tiles > 0x7fffffffLL) return cudaErrorInvalidValue;
  static int per_sm = 0;
  if (per_sm == 0 &&
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, quantize_cols_kernel<GROUP>, 256, 0) != cudaSuccess)
    per_sm = 1;
  const long long cap = static_cast<long long>(per_sm < 1 ? 1 : per_sm) * num_sms();
  launch_k(quantize_cols_kernel<GROUP>, static_cast<unsigned>(tiles < cap ? tiles : cap), 256, 0, st, 
      static_cast<const __nv_bfloat16*>(src), batch, rows, cols, row_map, src_rows, row_limit, codes, sf);
  count_launches(1);
  return cudaGetLastError();
}
}  // namespace

cudaError_t launch_quantize_cols(const void* src, int batch, int rows, int cols, uint8_t* codes, uint8_t* sf,
                                 cudaStream_t st, int group, const int32_t* row_limit) {
  if (batch == 0 || rows == 0 || cols == 0) return cudaSuccess;
  // rows % 128 == 0 and cols % 128 == 0 (checked by the callers)
  if (group == kMxScaleGroup224)
    return launch_cols<kMxScaleGroup224>(src, batch, rows, cols, nullptr, 0, row_limit, codes, sf, st);
  if (group != 128) return cudaErrorInvalidValue;
  return launch_cols<128>(src, batch, rows, cols, nullptr, 0, row_limit, codes, sf, st);
}

cudaError_t launch_quantize_cols_gather(const void* src, int src_rows, const int32_t* row_map, int rows, int cols,
                                        uint8_t* codes, uint8_t* sf, cudaStream_t st, int group,
                                        const int32_t* row_limit) {
  if (rows == 0 || cols == 0) return cudaSuccess;
  if (group == kMxScaleGroup224)
    return launch_cols<kMxScaleGroup224>(src, 1, rows, cols, row_map, src_rows, row_limit, codes, sf, st);
  if (group != 128) return cudaErrorInvalidValue;
  return launch_cols<128>(src, 1, rows, cols, row_map, src_rows, row_limit, codes, sf, st);
}

}  // namespace moe

namespace moe {
cudaError_t launch_gather_rows_mx(const uint8_t* codes_tok, const uint8_t* sf_tok, const int32_t* slot_row, int T,
                                  int k, int H, uint8_t* codes_perm, uint8_t* sf_perm, cudaStream_t st,
                                  const int32_t* counts, const int32_t* poffsets, int E_pad) {
  if (T + E_pad == 0) return cudaSuccess;
  launch_k(gather_rows_mx_kernel, T + E_pad, 128, 0, st, reinterpret_cast<const uint4*>(codes_tok), sf_tok, slot_row,
                                                   E_pad, k, H, counts, poffsets,
                                                   reinterpret_cast<uint4*>(codes_perm), sf_perm);
  count_launches(1);
  return cudaGetLastError();
}
}  // namespace moe
