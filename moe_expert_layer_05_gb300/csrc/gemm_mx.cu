// MXFP8 GEMM launchers: the same persistent tcgen05 kernel with E4M3 operands
// and E8M0 1x32 block scales (tcgen05.mma kind::mxf8f6f4.block_scale), the
// recipe the Megatron Core MoE summary names for the expert GEMMs on
// Blackwell (technical summary 2.5: expert GEMMs and activations in FP8, the
// router and the rest in higher precision).
//
// Every operand is K-major E4M3 with its scale tiles (see mxfp8.cu).  Where the
// contraction runs along the other dimension of a tensor (data gradients
// through the weights, weight gradients over tokens) the operand is a
// transposed quantised copy, so each 32-element block always lies along K.
#include <cuda.h>
#include <cuda_runtime.h>

#include "gemm_common.h"

namespace moe {

namespace {
inline bool make_tmap_u8(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer, uint32_t box_outer) {
  return make_tmap_2d(map, base, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, inner, outer, 128, box_outer);
}

template <class C>
cudaError_t launch_mx(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tc, const CUtensorMap& tc2,
                      const GemmParams& p, int rows_alloc, int dense_rows, cudaStream_t st) {
  int grid;
  if constexpr (C::S == Sched::kRoutedK) {
    grid = p.E * p.m_tiles_w * p.n_tiles;
  } else if (p.poffsets != nullptr) {
    grid = (rows_alloc / 128) * p.n_tiles;
  } else {
    grid = ((dense_rows + 127) / 128) * p.n_tiles;
  }
  return launch_gemm<C>(ta, tb, tc, tc2, p, grid < num_sms() ? grid : num_sms(), st);
}
}  // namespace

cudaError_t gemm_mx_fc1(const void* aq, const void* asf, int rows_alloc, int H, const void* w1q, const void* w1sf,
                        int E, int F, const int32_t* poffsets, int dense_rows, const float* row_gate, void* h,
                        void* z, int* status, cudaStream_t st, const MxOutQ* q) {
  // w1q rows of one expert are [gate 0..127, up 0..127, gate 128..255, up 128..255, ...]
  if (q != nullptr && poffsets == nullptr) return cudaErrorInvalidValue;
  if (h == nullptr && (q == nullptr || q->codes == nullptr)) return cudaErrorInvalidValue;
  CUtensorMap ta, tb;
  if (!make_tmap_u8(&ta, aq, H, rows_alloc, 128) || !make_tmap_u8(&tb, w1q, H, static_cast<uint64_t>(E) * 2 * F, 256))
    return cudaErrorInvalidValue;
  GemmParams p = gemm_params_zero();
  p.poffsets = poffsets;
  p.E = E;
  p.m_rows = dense_rows;
  p.k_len = H;
  p.n_tiles = F / 128;
  p.b_rows_per_group = 2 * F;
  p.c = h;
  p.ldc = F;
  p.c2 = z;
  p.ldc2 = 2 * F;
  p.half_cols = F;
  p.row_gate = row_gate;
  p.rows_cap = rows_alloc;
  p.status = status;
  p.sfa = static_cast<const uint8_t*>(asf);
  p.sfb = static_cast<const uint8_t*>(w1sf);
  p.sfa_tiles_k = H / 128;
  p.sfb_tiles_k = H / 128;
  if (q != nullptr) {                   // (the split SwiGLU epilogue writes them)
    p.q_codes = q->codes;
    p.q_sf = q->sf;
    p.qt_codes = q->codes_t;
    p.qt_sf = q->sf_t;
    p.ld_q = F;
  }
  // 32-column boxes (eight split-column epilogue warps, 2 KB staging); without a
  // bf16 h the map is encoded on the codes buffer and never used
  CUtensorMap tc, tz;
  const void* h_map = h != nullptr ? h : static_cast<const void*>(q->codes);
  if (!make_tmap_out_bf16_32_sw64(&tc, h_map, F, rows_alloc) ||
      (z != nullptr && !make_tmap_out_bf16_32_sw64(&tz, z, 2 * F, rows_alloc)))
    return cudaErrorInvalidValue;
  if (z == nullptr) tz = tc;
  if (poffsets != nullptr)
    return launch_mx<GemmCfg<256, false, false, Sched::kRoutedM, Epi::kSwiglu, true>>(ta, tb, tc, tz, p, rows_alloc,
                                                                                      dense_rows, st);
  return launch_mx<GemmCfg<256, false, false, Sched::kDenseM, Epi::kSwiglu, true>>(ta, tb, tc, tz, p, rows_alloc,
                                                                                   dense_rows, st);
}

namespace {
template <int BN>
cudaError_t mx_nt_bf16_bn(const void* aq, const void* asf, int rows_alloc, int K, const void* bq, const void* bsf,
                          int E, int N, const int32_t* poffsets, int dense_rows, void* c, int* status,
                          cudaStream_t st) {
  CUtensorMap ta, tb;
  if (!make_tmap_u8(&ta, aq, K, rows_alloc, 128) || !make_tmap_u8(&tb, bq, K, static_cast<uint64_t>(E) * N, BN))
    return cudaErrorInvalidValue;
  GemmParams p = gemm_params_zero();
  p.poffsets = poffsets;
  p.E = E;
  p.m_rows = dense_rows;
  p.k_len = K;
  p.n_tiles = N / BN;
  p.b_rows_per_group = N;
  p.c = c;
  p.ldc = N;
  p.rows_cap = rows_alloc;
  p.status = status;
  p.sfa = static_cast<const uint8_t*>(asf);
  p.sfb = static_cast<const uint8_t*>(bsf);
  p.sfa_tiles_k = K / 128;
  p.sfb_tiles_k = K / 128;
  CUtensorMap tc;
  if (!make_tmap_out_bf16(&tc, c, N, rows_alloc)) return cudaErrorInvalidValue;
  if (poffsets != nullptr)
    return launch_mx<GemmCfg<BN, false, false, Sched::kRoutedM, Epi::kStoreBf16, true>>(ta, tb, tc, tc, p, rows_alloc,
                                                                                        dense_rows, st);
  return launch_mx<GemmCfg<BN, false, false, Sched::kDenseM, Epi::kStoreBf16, true>>(ta, tb, tc, tc, p, rows_alloc,
                                                                                     dense_rows, st);
}

// 256 x 224 tiles (routed, N % 224 == 0, B's scale tiles grouped by 224 rows):
// two 128 x 224 MMAs share each B k-block, so a k-block brings 60 KB of
// operands for 256 x 224 x 128 instead of 48 KB for 128 x 256 x 128 -- 29 %
// fewer bytes per flop for the GEMMs whose operand feed sets the pace.
cudaError_t mx_nt_bf16_224(const void* aq, const void* asf, int rows_alloc, int K, const void* bq, const void* bsf,
                           int E, int N, const int32_t* poffsets, void* c, int* status, cudaStream_t st) {
  CUtensorMap ta, tb;
  if (!make_tmap_u8(&ta, aq, K, rows_alloc, 256) || !make_tmap_u8(&tb, bq, K, static_cast<uint64_t>(E) * N, 224))
    return cudaErrorInvalidValue;
  GemmParams p = gemm_params_zero();
  p.poffsets = poffsets;
  p.E = E;
  p.k_len = K;
  p.n_tiles = N / 224;
  p.b_rows_per_group = N;
  p.c = c;
  p.ldc = N;
  p.rows_cap = rows_alloc;
  p.status = status;
  p.sfa = static_cast<const uint8_t*>(asf);
  p.sfb = static_cast<const uint8_t*>(bsf);
  p.sfa_tiles_k = K / 128;
  p.sfb_tiles_k = K / 128;
  CUtensorMap tc, tc2;
  if (!make_tmap_out_bf16(&tc, c, N, rows_alloc) || !make_tmap_out_bf16_32(&tc2, c, N, rows_alloc))
    return cudaErrorInvalidValue;
  return launch_mx<GemmCfg<224, false, false, Sched::kRoutedM, Epi::kStoreBf16, true, true>>(ta, tb, tc, tc2, p,
                                                                                            rows_alloc, 0, st);
}
}  // namespace

// c [rows, N] bf16 = A [rows, K] x B_e [N, K]^T, both E4M3 with scales.
cudaError_t gemm_mx_nt_bf16(const void* aq, const void* asf, int rows_alloc, int K, const void* bq, const void* bsf,
                            int E, int N, const int32_t* poffsets, int dense_rows, void* c, int* status,
                            cudaStream_t st, int b_group) {
  if (b_group == kMxScaleGroup224) {
    if (poffsets == nullptr || N % 224 != 0) return cudaErrorInvalidValue;
    return mx_nt_bf16_224(aq, asf, rows_alloc, K, bq, bsf, E, N, poffsets, c, status, st);
  }
  if (N % 256 == 0)
    return mx_nt_bf16_bn<256>(aq, asf, rows_alloc, K, bq, bsf, E, N, poffsets, dense_rows, c, status, st);
  return mx_nt_bf16_bn<128>(aq, asf, rows_alloc, K, bq, bsf, E, N, poffsets, dense_rows, c, status, st);
}

cudaError_t gemm_mx_fc2_combine(const void* aq, const void* asf, int rows_alloc, int F, const void* bq,
                                const void* bsf, int E, int H, const int32_t* poffsets, void* o,
                                const CombineArgs& cmb, int* status, cudaStream_t st) {
  if (H % 256 != 0 || poffsets == nullptr) return cudaErrorInvalidValue;
  CUtensorMap ta, tb;
  if (!make_tmap_u8(&ta, aq, F, rows_alloc, 128) || !make_tmap_u8(&tb, bq, F, static_cast<uint64_t>(E) * H, 256))
    return cudaErrorInvalidValue;
  GemmParams p = gemm_params_zero();
  p.poffsets = poffsets;
  p.E = E;
  p.k_len = F;
  p.n_tiles = H / 256;
  p.b_rows_per_group = H;
  p.c = o;
  p.ldc = H;
  p.rows_cap = rows_alloc;
  p.status = status;
  p.sfa = static_cast<const uint8_t*>(asf);
  p.sfb = static_cast<const uint8_t*>(bsf);
  p.sfa_tiles_k = F / 128;
  p.sfb_tiles_k = F / 128;
  set_combine(p, cmb);
  CUtensorMap tc;
  if (!make_tmap_out_bf16(&tc, o, H, rows_alloc)) return cudaErrorInvalidValue;
  return launch_mx<GemmCfg<256, false, false, Sched::kRoutedM, Epi::kStoreBf16, true>>(ta, tb, tc, tc, p, rows_alloc,
                                                                                      0, st);
}

#ifndef MOE_MX_DGRAD_FC2_BN
#define MOE_MX_DGRAD_FC2_BN 256
#endif
bool gemm_mx_dgrad_fc2_quantises(int F) { return MOE_MX_DGRAD_FC2_BN == 256 && F % 256 == 0; }

cudaError_t gemm_mx_dgrad_fc2(const void* dyq, const void* dysf, int rows_alloc, int H, const void* w2tq,
                              const void* w2tsf, int E, int F, const int32_t* poffsets, int dense_rows, const void* z,
                              const float* row_gate, void* dz, float* dgate_part, int* status, cudaStream_t st,
                              const MxOutQ* q) {
  if (q != nullptr && (!gemm_mx_dgrad_fc2_quantises(F) || poffsets == nullptr)) return cudaErrorInvalidValue;
  if (q == nullptr && dz == nullptr) return cudaErrorInvalidValue;
  // B_e = W2_e^T [F, H], quantised along H.  256-column tiles where F allows:
  // one accumulator (256 columns beside the scale columns), 48 KB per k-block
  // of 128 x 256 x 128 instead of 32 KB per 128 x 128 x 128.
  const bool wide = MOE_MX_DGRAD_FC2_BN == 256 && F % 256 == 0;
  CUtensorMap ta, tb;
  if (!make_tmap_u8(&ta, dyq, H, rows_alloc, 128) ||
      !make_tmap_u8(&tb, w2tq, H, static_cast<uint64_t>(E) * F, wide ? 256 : 128))
    return cudaErrorInvalidValue;
  GemmParams p = gemm_params_zero();
  p.poffsets = poffsets;
  p.E = E;
  p.m_rows = dense_rows;
  p.k_len = H;
  p.n_tiles = F / 128;
  p.b_rows_per_group = F;
  p.c = dz;
  p.ldc = 2 * F;
  p.half_cols = F;
  p.aux = static_cast<const __nv_bfloat16*>(z);
  p.ld_aux = 2 * F;
  p.row_gate = row_gate;
  p.dgate_part = dgate_part;
  if (q != nullptr) {                   // (the split 256-column epilogue writes them)
    p.q_codes = q->codes;
    p.q_sf = q->sf;
    p.qt_codes = q->codes_t;
    p.qt_sf = q->sf_t;
    p.ld_q = 2 * F;
  }
  p.rows_cap = rows_alloc;
  p.status = status;
  p.sfa = static_cast<const uint8_t*>(dysf);
  p.sfb = static_cast<const uint8_t*>(w2tsf);
  p.sfa_tiles_k = H / 128;
  p.sfb_tiles_k = H / 128;
  CUtensorMap tc, tc32;
  // (no bf16 dz: the maps are encoded on the codes buffer and never used)
  const void* dz_map = dz != nullptr ? dz : (q->codes != nullptr ? static_cast<const void*>(q->codes) : q->codes_t);
  if (!make_tmap_out_bf16(&tc, dz_map, 2 * F, rows_alloc) ||
      !make_tmap_out_bf16_32_sw64(&tc32, dz_map, 2 * F, rows_alloc))
    return cudaErrorInvalidValue;
  if (wide) {
    // (eight epilogue warps storing 32-column chunks through tc32)
    p.n_tiles = F / 256;
    if (poffsets != nullptr)
      return launch_mx<GemmCfg<256, false, false, Sched::kRoutedM, Epi::kSwigluBwd, true>>(ta, tb, tc, tc32, p,
                                                                                           rows_alloc, dense_rows, st);
    return launch_mx<GemmCfg<256, false, false, Sched::kDenseM, Epi::kSwigluBwd, true>>(ta, tb, tc, tc32, p,
                                                                                        rows_alloc, dense_rows, st);
  }
  if (poffsets != nullptr)
    return launch_mx<GemmCfg<128, false, false, Sched::kRoutedM, Epi::kSwigluBwd, true>>(ta, tb, tc, tc, p, rows_alloc,
                                                                                         dense_rows, st);
  return launch_mx<GemmCfg<128, false, false, Sched::kDenseM, Epi::kSwigluBwd, true>>(ta, tb, tc, tc, p, rows_alloc,
                                                                                      dense_rows, st);
}

namespace {
template <int BN>
cudaError_t mx_wgrad_bn(const void* atq, const void* atsf, int M, const void* btq, const void* btsf, int N,
                        int rows_alloc, int E, const int32_t* poffsets, int dense_rows, float* dw, int* status,
                        cudaStream_t st) {
  // A^T [M, rows] and B^T [N, rows], quantised along rows (the contraction)
  CUtensorMap ta, tb;
  if (!make_tmap_u8(&ta, atq, rows_alloc, M, 128) || !make_tmap_u8(&tb, btq, rows_alloc, N, BN))
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
  p.sfa = static_cast<const uint8_t*>(atsf);
  p.sfb = static_cast<const uint8_t*>(btsf);
  p.sfa_tiles_k = rows_alloc / 128;
  p.sfb_tiles_k = rows_alloc / 128;
  CUtensorMap tc;
  if (!make_tmap_out_f32(&tc, dw, N, static_cast<uint64_t>(p.E) * M)) return cudaErrorInvalidValue;
  return launch_mx<GemmCfg<BN, false, false, Sched::kRoutedK, Epi::kStoreF32, true>>(ta, tb, tc, tc, p, rows_alloc,
                                                                                     dense_rows, st);
}
}  // namespace

namespace {
// 256 x 224 weight-gradient tiles (B's scale tiles grouped by 224 rows): two
// 128 x 224 MMAs share each B k-block, 60 KB of operands per k-block for
// 256 x 224 outputs instead of 48 KB for 128 x 256, and eight epilogue warps.
cudaError_t mx_wgrad_224(const void* atq, const void* atsf, int M, const void* btq, const void* btsf, int N,
                         int rows_alloc, int E, const int32_t* poffsets, int dense_rows, float* dw, int* status,
                         cudaStream_t st, bool c_trans) {
  CUtensorMap ta, tb;
  if (!make_tmap_u8(&ta, atq, rows_alloc, M, 256) || !make_tmap_u8(&tb, btq, rows_alloc, N, 224))
    return cudaErrorInvalidValue;
  GemmParams p = gemm_params_zero();
  p.poffsets = poffsets;
  p.E = (poffsets != nullptr) ? E : 1;
  p.m_rows = M;
  p.k_len = dense_rows;
  p.m_tiles_w = M / 256;
  p.n_tiles = N / 224;
  p.c = dw;
  p.ldc = N;
  p.c_group_stride = static_cast<long long>(M) * N;
  p.rows_cap = rows_alloc;
  p.status = status;
  p.sfa = static_cast<const uint8_t*>(atsf);
  p.sfb = static_cast<const uint8_t*>(btsf);
  p.sfa_tiles_k = rows_alloc / 128;
  p.sfb_tiles_k = rows_alloc / 128;
  p.c_trans = c_trans ? 1 : 0;
  CUtensorMap tc;
  const bool map_ok = c_trans ? make_tmap_out_f32(&tc, dw, M, static_cast<uint64_t>(p.E) * N)
                              : make_tmap_out_f32(&tc, dw, N, static_cast<uint64_t>(p.E) * M);
  if (!map_ok) return cudaErrorInvalidValue;
  return launch_mx<GemmCfg<224, false, false, Sched::kRoutedK, Epi::kStoreF32, true, true>>(ta, tb, tc, tc, p,
                                                                                           rows_alloc, dense_rows, st);
}
}  // namespace

cudaError_t gemm_mx_wgrad(const void* atq, const void* atsf, int M, const void* btq, const void* btsf, int N,
                          int rows_alloc, int E, const int32_t* poffsets, int dense_rows, float* dw, int* status,
                          cudaStream_t st, int b_group, bool c_trans) {
  if (b_group == kMxScaleGroup224) {
    if (N % 224 != 0 || M % 256 != 0) return cudaErrorInvalidValue;
    return mx_wgrad_224(atq, atsf, M, btq, btsf, N, rows_alloc, E, poffsets, dense_rows, dw, status, st, c_trans);
  }
  if (c_trans) return cudaErrorInvalidValue;
  if (N % 256 == 0)
    return mx_wgrad_bn<256>(atq, atsf, M, btq, btsf, N, rows_alloc, E, poffsets, dense_rows, dw, status, st);
  return mx_wgrad_bn<128>(atq, atsf, M, btq, btsf, N, rows_alloc, E, poffsets, dense_rows, dw, status, st);
}

// ---------------------------------------------------------------- NVFP4
// The same kernel with E2M1 operands (two codes per byte, so a 128-byte
// K-major row holds 256 elements), one E4M3 scale per 16 along K (four 512-byte
// tiles per k-block and 128 rows), kind::mxf4nvf4 MMAs of K = 64, and the
// tensor scales applied to the accumulator in the epilogue (see nvfp4.cu).

cudaError_t gemm_nv4_fc1(const void* aq, const void* asf, const float* amax_a, int rows_alloc, int H,
                         const void* w1q, const void* w1sf, const float* amax_w, int E, int F,
                         const int32_t* poffsets, int dense_rows, const float* row_gate, void* h, void* z,
                         float* amax_h, int* status, cudaStream_t st) {
  // w1q rows of one expert are [gate 0..127, up 0..127, gate 128..255, up 128..255, ...]
  CUtensorMap ta, tb;
  if (!make_tmap_u8(&ta, aq, H / 2, rows_alloc, 128) ||
      !make_tmap_u8(&tb, w1q, H / 2, static_cast<uint64_t>(E) * 2 * F, 256))
    return cudaErrorInvalidValue;
  GemmParams p = gemm_params_zero();
  p.poffsets = poffsets;
  p.E = E;
  p.m_rows = dense_rows;
  p.k_len = H;
  p.n_tiles = F / 128;
  p.b_rows_per_group = 2 * F;
  p.c = h;
  p.ldc = F;
  p.c2 = z;
  p.ldc2 = 2 * F;
  p.half_cols = F;
  p.row_gate = row_gate;
  p.rows_cap = rows_alloc;
  p.status = status;
  p.sfa = static_cast<const uint8_t*>(asf);
  p.sfb = static_cast<const uint8_t*>(w1sf);
  p.sfa_tiles_k = H / 64;
  p.sfb_tiles_k = H / 64;
  p.amax_a = amax_a;
  p.amax_b = amax_w;
  p.amax_out = reinterpret_cast<unsigned*>(amax_h);
  CUtensorMap tc, tz;
  if (!make_tmap_out_bf16(&tc, h, F, rows_alloc) || (z != nullptr && !make_tmap_out_bf16(&tz, z, 2 * F, rows_alloc)))
    return cudaErrorInvalidValue;
  if (z == nullptr) tz = tc;
  if (poffsets != nullptr)
    return launch_mx<GemmCfg<256, false, false, Sched::kRoutedM, Epi::kSwiglu, 2>>(ta, tb, tc, tz, p, rows_alloc,
                                                                                   dense_rows, st);
  return launch_mx<GemmCfg<256, false, false, Sched::kDenseM, Epi::kSwiglu, 2>>(ta, tb, tc, tz, p, rows_alloc,
                                                                                dense_rows, st);
}

namespace {
template <int BN>
cudaError_t nv4_nt_bf16_bn(const void* aq, const void* asf, const float* amax_a, int rows_alloc, int K,
                           const void* bq, const void* bsf, const float* amax_b, int E, int N,
                           const int32_t* poffsets, int dense_rows, void* c, int* status, cudaStream_t st) {
  CUtensorMap ta, tb;
  if (!make_tmap_u8(&ta, aq, K / 2, rows_alloc, 128) || !make_tmap_u8(&tb, bq, K / 2, static_cast<uint64_t>(E) * N, BN))
    return cudaErrorInvalidValue;
  GemmParams p = gemm_params_zero();
  p.poffsets = poffsets;
  p.E = E;
  p.m_rows = dense_rows;
  p.k_len = K;
  p.n_tiles = N / BN;
  p.b_rows_per_group = N;
  p.c = c;
  p.ldc = N;
  p.rows_cap = rows_alloc;
  p.status = status;
  p.sfa = static_cast<const uint8_t*>(asf);
  p.sfb = static_cast<const uint8_t*>(bsf);
  p.sfa_tiles_k = K / 64;
  p.sfb_tiles_k = K / 64;
  p.amax_a = amax_a;
  p.amax_b = amax_b;
  CUtensorMap tc;
  if (!make_tmap_out_bf16(&tc, c, N, rows_alloc)) return cudaErrorInvalidValue;
  if (poffsets != nullptr)
    return launch_mx<GemmCfg<BN, false, false, Sched::kRoutedM, Epi::kStoreBf16, 2>>(ta, tb, tc, tc, p, rows_alloc,
                                                                                     dense_rows, st);
  return launch_mx<GemmCfg<BN, false, false, Sched::kDenseM, Epi::kStoreBf16, 2>>(ta, tb, tc, tc, p, rows_alloc,
                                                                                  dense_rows, st);
}
}  // namespace

// c [rows, N] bf16 = A [rows, K] x B_e [N, K]^T, both NVFP4.
cudaError_t gemm_nv4_nt_bf16(const void* aq, const void* asf, const float* amax_a, int rows_alloc, int K,
                             const void* bq, const void* bsf, const float* amax_b, int E, int N,
                             const int32_t* poffsets, int dense_rows, void* c, int* status, cudaStream_t st) {
  if (N % 256 == 0)
    return nv4_nt_bf16_bn<256>(aq, asf, amax_a, rows_alloc, K, bq, bsf, amax_b, E, N, poffsets, dense_rows, c, status,
                               st);
  return nv4_nt_bf16_bn<128>(aq, asf, amax_a, rows_alloc, K, bq, bsf, amax_b, E, N, poffsets, dense_rows, c, status,
                             st);
}

}  // namespace moe
