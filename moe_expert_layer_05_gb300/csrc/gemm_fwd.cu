// Forward GEMM launchers: router logits, fc1 with the fused gated-SwiGLU
// epilogue, fc2.  Also the TMA descriptor helper shared with gemm_bwd.cu.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "gemm_common.h"

namespace moe {

namespace {
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}
}  // namespace

bool make_tmap_2d(CUtensorMap* map, const void* base, CUtensorMapDataType dtype, int elem_bytes, uint64_t inner,
                  uint64_t outer, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swizzle) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  if (outer == 0) outer = 1;  // an empty tensor still needs a valid map; no tile reads it
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {inner * static_cast<uint64_t>(elem_bytes)};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, dtype, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

namespace {

template <int BN>
cudaError_t router_bn(const void* x, const void* wr, int T, int H, int E, float* logits, int* status,
                      cudaStream_t st) {
  using C = GemmCfg<BN, false, false, Sched::kDenseM, Epi::kStoreF32>;
  CUtensorMap ta, tb;
  if (!make_tmap_bf16(&ta, x, H, T, 64, 128) || !make_tmap_bf16(&tb, wr, H, E, 64, BN))
    return cudaErrorInvalidValue;
  GemmParams p = gemm_params_zero();
  p.E = 1;
  p.m_rows = T;
  p.k_len = H;
  p.n_tiles = (E + BN - 1) / BN;
  p.b_rows_per_group = 0;
  p.c = logits;
  p.ldc = E;
  p.valid_cols = E;
  p.rows_cap = T;
  p.status = status;
  const int tiles = ((T + 127) / 128) * p.n_tiles;
  return launch_gemm<C>(ta, tb, ta, ta, p, tiles < num_sms() ? tiles : num_sms(), st);   // plain stores
}

}  // namespace

cudaError_t gemm_router(const void* x, const void* wr, int T, int H, int E, float* logits, int* status,
                        cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  if (E <= 16) return router_bn<16>(x, wr, T, H, E, logits, status, st);
  if (E <= 32) return router_bn<32>(x, wr, T, H, E, logits, status, st);
  if (E <= 64) return router_bn<64>(x, wr, T, H, E, logits, status, st);
  // E > 128: two 128-wide N tiles per row block, twice as many CTAs busy as
  // one 256-wide tile (the router has only T/128 row blocks)
  return router_bn<128>(x, wr, T, H, E, logits, status, st);
}

cudaError_t gemm_fc1(const void* a, int rows_alloc, int H, const void* w1, int E, int F, const int32_t* poffsets,
                     int dense_rows, const float* row_gate, void* h, void* z, int* status, cudaStream_t st) {
  CUtensorMap ta, tb;
  if (!make_tmap_bf16(&ta, a, H, rows_alloc, 64, 256) ||
      !make_tmap_bf16(&tb, w1, H, static_cast<uint64_t>(E) * 2 * F, 64, 128))
    return cudaErrorInvalidValue;
  GemmParams p = gemm_params_zero();
  p.poffsets = poffsets;
  p.E = E;
  p.m_rows = dense_rows;
  p.k_len = H;
  p.n_tiles = F / 128;
  p.b_rows_per_group = 2 * F;
  p.b_half_offset = F;
  p.c = h;
  p.ldc = F;
  p.c2 = z;
  p.ldc2 = 2 * F;
  p.half_cols = F;
  p.row_gate = row_gate;
  p.rows_cap = rows_alloc;
  p.status = status;
  CUtensorMap tc, tz;
  if (!make_tmap_out_bf16(&tc, h, F, rows_alloc) || (z != nullptr && !make_tmap_out_bf16(&tz, z, 2 * F, rows_alloc)))
    return cudaErrorInvalidValue;
  if (z == nullptr) tz = tc;
  if (poffsets != nullptr) {
    using C = GemmCfg<256, false, false, Sched::kRoutedM, Epi::kSwiglu, false, true>;
    const int upper = (rows_alloc / 128) * p.n_tiles;
    return launch_gemm<C>(ta, tb, tc, tz, p, upper < num_sms() ? upper : num_sms(), st);
  }
  using C = GemmCfg<256, false, false, Sched::kDenseM, Epi::kSwiglu, false, true>;
  const int tiles = ((dense_rows + 255) / 256) * p.n_tiles;
  return launch_gemm<C>(ta, tb, tc, tz, p, tiles < num_sms() ? tiles : num_sms(), st);
}

cudaError_t gemm_fc1_gather(const void* x, int T, const int32_t* row_src, int rows_alloc, int H, const void* w1,
                            int E, int F, const int32_t* poffsets, const float* row_gate, void* h, void* z, int* status,
                            cudaStream_t st) {
  // A rows are copied by the kernel's producer warp from x [T, H] (token order)
  // through row_src; only W1 goes through TMA
  CUtensorMap tb;
  if (!make_tmap_bf16(&tb, w1, H, static_cast<uint64_t>(E) * 2 * F, 64, 128)) return cudaErrorInvalidValue;
  GemmParams p = gemm_params_zero();
  p.poffsets = poffsets;
  p.E = E;
  p.k_len = H;
  p.n_tiles = F / 128;
  p.b_rows_per_group = 2 * F;
  p.b_half_offset = F;
  p.c = h;
  p.ldc = F;
  p.c2 = z;
  p.ldc2 = 2 * F;
  p.half_cols = F;
  p.row_gate = row_gate;
  p.rows_cap = rows_alloc;
  p.status = status;
  p.a_tok = static_cast<const __nv_bfloat16*>(x);
  p.a_row_src = row_src;
  p.a_rows = T;
  CUtensorMap tc, tz;
  if (!make_tmap_out_bf16(&tc, h, F, rows_alloc) || (z != nullptr && !make_tmap_out_bf16(&tz, z, 2 * F, rows_alloc)))
    return cudaErrorInvalidValue;
  if (z == nullptr) tz = tc;
  using C = GemmCfg<256, false, false, Sched::kRoutedM, Epi::kSwiglu, 0, true, false, true>;
  const int upper = (rows_alloc / 128) * p.n_tiles;
  return launch_gemm<C>(tb, tb, tc, tz, p, upper < num_sms() ? upper : num_sms(), st);
}

namespace {
template <int BN>
cudaError_t fc2_bn(const void* a, int rows_alloc, int F, const void* w2, int E, int H, const int32_t* poffsets,
                   int dense_rows, void* o, int* status, cudaStream_t st) {
  constexpr bool M256 = (BN == 256);     // 256-row tiles where two MMAs can share a 256-wide B k-block
  CUtensorMap ta, tb;
  if (!make_tmap_bf16(&ta, a, F, rows_alloc, 64, M256 ? 256 : 128) ||
      !make_tmap_bf16(&tb, w2, F, static_cast<uint64_t>(E) * H, 64, BN))
    return cudaErrorInvalidValue;
  GemmParams p = gemm_params_zero();
  p.poffsets = poffsets;
  p.E = E;
  p.m_rows = dense_rows;
  p.k_len = F;
  p.n_tiles = H / BN;
  p.b_rows_per_group = H;
  p.c = o;
  p.ldc = H;
  p.rows_cap = rows_alloc;
  p.status = status;
  CUtensorMap tc;
  if (!make_tmap_out_bf16(&tc, o, H, rows_alloc)) return cudaErrorInvalidValue;
  if (poffsets != nullptr) {
    using C = GemmCfg<BN, false, false, Sched::kRoutedM, Epi::kStoreBf16, false, M256>;
    const int upper = (rows_alloc / 128) * p.n_tiles;
    return launch_gemm<C>(ta, tb, tc, tc, p, upper < num_sms() ? upper : num_sms(), st);
  }
  using C = GemmCfg<BN, false, false, Sched::kDenseM, Epi::kStoreBf16, false, M256>;
  const int tiles = ((dense_rows + C::TILE_M - 1) / C::TILE_M) * p.n_tiles;
  return launch_gemm<C>(ta, tb, tc, tc, p, tiles < num_sms() ? tiles : num_sms(), st);
}
}  // namespace

cudaError_t gemm_fc2(const void* a, int rows_alloc, int F, const void* w2, int E, int H, const int32_t* poffsets,
                     int dense_rows, void* o, int* status, cudaStream_t st) {
  if (H % 256 == 0) return fc2_bn<256>(a, rows_alloc, F, w2, E, H, poffsets, dense_rows, o, status, st);
  return fc2_bn<128>(a, rows_alloc, F, w2, E, H, poffsets, dense_rows, o, status, st);
}

cudaError_t gemm_fc2_combine(const void* a, int rows_alloc, int F, const void* w2, int E, int H,
                             const int32_t* poffsets, void* o, const CombineArgs& cmb, int* status, cudaStream_t st) {
  if (H % 256 != 0 || poffsets == nullptr) return cudaErrorInvalidValue;
  CUtensorMap ta, tb;
  if (!make_tmap_bf16(&ta, a, F, rows_alloc, 64, 256) ||
      !make_tmap_bf16(&tb, w2, F, static_cast<uint64_t>(E) * H, 64, 256))
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
  set_combine(p, cmb);
  CUtensorMap tc;
  if (!make_tmap_out_bf16(&tc, o, H, rows_alloc)) return cudaErrorInvalidValue;
  using C = GemmCfg<256, false, false, Sched::kRoutedM, Epi::kStoreBf16, false, true>;
  const int upper = (rows_alloc / 128) * p.n_tiles;
  return launch_gemm<C>(ta, tb, tc, tc, p, upper < num_sms() ? upper : num_sms(), st);
}

}  // namespace moe
