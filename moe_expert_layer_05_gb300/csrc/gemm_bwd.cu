// Backward GEMM launchers: data gradients through fc2 (with the SwiGLU
// backward epilogue that recomputes silu(a)*b from the saved fc1 output) and
// fc1, and the weight gradients whose contraction runs over each expert's
// rows (ragged K, read from device offsets).
#include <cuda.h>
#include <cuda_runtime.h>

#include "gemm_common.h"

namespace moe {

namespace {
template <int BN>
cudaError_t dgrad_fc2_bn(const void* dy_perm, int rows_alloc, int H, const void* w2, int E, int F,
                         const int32_t* poffsets, int dense_rows, const void* z, const float* row_gate, void* dz,
                         float* dgate_part, int* status, cudaStream_t st) {
  // B[n=f, k=h] = W2_e[h, f]: W2 seen as [E*H rows, F cols], N contiguous (MN-major).
  // N = 256: 256 x 256 tiles on CTA pairs (half of A and of B per SM, six
  // stages, double-buffered accumulators).  N = 128: 256-row tiles on one CTA,
  // two MMAs sharing each B k-block.
  constexpr bool PAIR = (BN == 256);
  CUtensorMap ta, tb;
  if (!make_tmap_bf16(&ta, dy_perm, H, rows_alloc, 64, PAIR ? 128 : 256) ||
      !make_tmap_bf16(&tb, w2, F, static_cast<uint64_t>(E) * H, 64, 64))
    return cudaErrorInvalidValue;
  GemmParams p = gemm_params_zero();
  p.poffsets = poffsets;
  p.E = E;
  p.m_rows = dense_rows;
  p.k_len = H;
  p.n_tiles = F / BN;
  p.b_rows_per_group = H;
  p.c = dz;
  p.ldc = 2 * F;
  p.half_cols = F;
  p.aux = static_cast<const __nv_bfloat16*>(z);
  p.ld_aux = 2 * F;
  p.row_gate = row_gate;
  p.dgate_part = dgate_part;
  p.rows_cap = rows_alloc;
  p.status = status;
  CUtensorMap tc;
  if (!make_tmap_out_bf16(&tc, dz, 2 * F, rows_alloc)) return cudaErrorInvalidValue;
  if (poffsets != nullptr) {
    using C = GemmCfg<BN, false, true, Sched::kRoutedM, Epi::kSwigluBwd, false, !PAIR, PAIR>;
    const int upper = (rows_alloc / 128) * p.n_tiles;
    if constexpr (PAIR) return launch_gemm_pair<C>(ta, tb, tc, tc, p, upper, st);
    else return launch_gemm<C>(ta, tb, tc, tc, p, upper < num_sms() ? upper : num_sms(), st);
  }
  using C = GemmCfg<BN, false, true, Sched::kDenseM, Epi::kSwigluBwd, false, !PAIR, PAIR>;
  const int tiles = ((dense_rows + C::TILE_M - 1) / C::TILE_M) * p.n_tiles;
  if constexpr (PAIR) return launch_gemm_pair<C>(ta, tb, tc, tc, p, tiles, st);
  else return launch_gemm<C>(ta, tb, tc, tc, p, tiles < num_sms() ? tiles : num_sms(), st);
}
}  // namespace

// dgate_part gets one partial sum per 128 columns of dh whatever the tile width.
cudaError_t gemm_dgrad_fc2(const void* dy_perm, int rows_alloc, int H, const void* w2, int E, int F,
                           const int32_t* poffsets, int dense_rows, const void* z, const float* row_gate,
                           void* dz, float* dgate_part, int* status, cudaStream_t st) {
  if (F % 256 == 0)
    return dgrad_fc2_bn<256>(dy_perm, rows_alloc, H, w2, E, F, poffsets, dense_rows, z, row_gate, dz, dgate_part,
                             status, st);
  return dgrad_fc2_bn<128>(dy_perm, rows_alloc, H, w2, E, F, poffsets, dense_rows, z, row_gate, dz, dgate_part,
                           status, st);
}

namespace {
template <int BN>
cudaError_t dgrad_fc1_bn(const void* dz, int rows_alloc, int F, const void* w1, int E, int H,
                         const int32_t* poffsets, int dense_rows, void* dx_perm, int* status, cudaStream_t st) {
  // B[n=h, k=j] = W1_e[j, h]: W1 seen as [E*2F rows, H cols] (MN-major).
  constexpr bool M256 = (BN == 256);     // 256-row tiles where two MMAs can share a 256-wide B k-block
  CUtensorMap ta, tb;
  if (!make_tmap_bf16(&ta, dz, 2 * F, rows_alloc, 64, M256 ? 256 : 128) ||
      !make_tmap_bf16(&tb, w1, H, static_cast<uint64_t>(E) * 2 * F, 64, 64))
    return cudaErrorInvalidValue;
  GemmParams p = gemm_params_zero();
  p.poffsets = poffsets;
  p.E = E;
  p.m_rows = dense_rows;
  p.k_len = 2 * F;
  p.n_tiles = H / BN;
  p.b_rows_per_group = 2 * F;
  p.c = dx_perm;
  p.ldc = H;
  p.rows_cap = rows_alloc;
  p.status = status;
  CUtensorMap tc;
  if (!make_tmap_out_bf16(&tc, dx_perm, H, rows_alloc)) return cudaErrorInvalidValue;
  if (poffsets != nullptr) {
    using C = GemmCfg<BN, false, true, Sched::kRoutedM, Epi::kStoreBf16, false, M256>;
    const int upper = (rows_alloc / 128) * p.n_tiles;
    return launch_gemm<C>(ta, tb, tc, tc, p, upper < num_sms() ? upper : num_sms(), st);
  }
  using C = GemmCfg<BN, false, true, Sched::kDenseM, Epi::kStoreBf16, false, M256>;
  const int tiles = ((dense_rows + C::TILE_M - 1) / C::TILE_M) * p.n_tiles;
  return launch_gemm<C>(ta, tb, tc, tc, p, tiles < num_sms() ? tiles : num_sms(), st);
}

template <int BN>
cudaError_t wgrad_bn(const void* a, int M, const void* b, int N, int rows_alloc, int E, const int32_t* poffsets,
                     int dense_rows, float* dw, int* status, cudaStream_t st) {
  // A[m, k] = a[k_row0 + k, m], B[n, k] = b[k_row0 + k, n]: both MN-major.
  CUtensorMap ta, tb;
  // boxes of 64 columns x BK rows (BK = 128 on CTA pairs, 64 otherwise)
  constexpr bool PAIR_K = (BN == 256);
  CUtensorMap ta2, tb2;
  if (!make_tmap_bf16(&ta, a, M, rows_alloc, 64, 64) || !make_tmap_bf16(&tb, b, N, rows_alloc, 64, 64) ||
      !make_tmap_bf16(&ta2, a, M, rows_alloc, 64, PAIR_K ? 128 : 64) ||
      !make_tmap_bf16(&tb2, b, N, rows_alloc, 64, PAIR_K ? 128 : 64))
    return cudaErrorInvalidValue;
  GemmParams p = gemm_params_zero();
  p.poffsets = poffsets;
  p.E = (poffsets != nullptr) ? E : 1;
  p.m_rows = M;
  p.k_len = dense_rows;
  p.m_tiles_w = M / 128;
  p.n_tiles = N / BN;
  p.c = dw;
  p.ldc = N;
  p.c_group_stride = static_cast<long long>(M) * N;
  p.rows_cap = rows_alloc;
  p.status = status;
  CUtensorMap tc;
  if (!make_tmap_out_f32(&tc, dw, N, static_cast<uint64_t>(p.E) * M)) return cudaErrorInvalidValue;
  if constexpr (BN == 256) {
    if (M % 256 == 0) {
      // 256 x 256 tiles on CTA pairs: each SM loads half of A and half of B
      // per k-block, so the loads keep up with the MMAs and the fp32 stores
      // (the bulk of the traffic) set the pace.
      using C = GemmCfg<BN, true, true, Sched::kRoutedK, Epi::kStoreF32, false, false, true>;
      p.m_tiles_w = M / 256;
      return launch_gemm_pair<C>(ta2, tb2, tc, tc, p, p.E * p.m_tiles_w * p.n_tiles, st);
    }
  }
  using C = GemmCfg<BN, true, true, Sched::kRoutedK, Epi::kStoreF32>;
  const int tiles = p.E * p.m_tiles_w * p.n_tiles;
  return launch_gemm<C>(ta, tb, tc, tc, p, tiles < num_sms() ? tiles : num_sms(), st);
}
}  // namespace

cudaError_t gemm_dgrad_fc1(const void* dz, int rows_alloc, int F, const void* w1, int E, int H,
                           const int32_t* poffsets, int dense_rows, void* dx_perm, int* status, cudaStream_t st) {
  if (H % 256 == 0) return dgrad_fc1_bn<256>(dz, rows_alloc, F, w1, E, H, poffsets, dense_rows, dx_perm, status, st);
  return dgrad_fc1_bn<128>(dz, rows_alloc, F, w1, E, H, poffsets, dense_rows, dx_perm, status, st);
}

cudaError_t gemm_wgrad(const void* a, int M, const void* b, int N, int rows_alloc, int E, const int32_t* poffsets,
                       int dense_rows, float* dw, int* status, cudaStream_t st) {
  if (N % 256 == 0) return wgrad_bn<256>(a, M, b, N, rows_alloc, E, poffsets, dense_rows, dw, status, st);
  return wgrad_bn<128>(a, M, b, N, rows_alloc, E, poffsets, dense_rows, dw, status, st);
}

}  // namespace moe
