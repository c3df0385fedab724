// Host-side helpers for the tcgen05 GEMM launchers: TMA descriptor encoding
// (through the driver entry point, so the library needs no link-time libcuda)
// and a typed launch wrapper.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

#include "gemm.cuh"
#include "internal.h"

namespace moe {

// Encode a 2-D row-major tensor map (128-byte swizzle unless told otherwise).
// inner = elements per row, outer = rows, box = {box_inner, box_outer} elements.
bool make_tmap_2d(CUtensorMap* map, const void* base, CUtensorMapDataType dtype, int elem_bytes, uint64_t inner,
                  uint64_t outer, uint32_t box_inner, uint32_t box_outer,
                  CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B);

inline bool make_tmap_bf16(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer, uint32_t box_inner,
                           uint32_t box_outer) {
  return make_tmap_2d(map, base, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, inner, outer, box_inner, box_outer);
}

// Per-device, per-kernel launch set-up state (function attributes are per
// device; the cluster occupancy is a property of the device too).
constexpr int kMaxDevices = 64;
inline int current_device() {
  int d = -1;
  return (cudaGetDevice(&d) == cudaSuccess && d >= 0 && d < kMaxDevices) ? d : -1;
}

template <class C>
cudaError_t launch_gemm(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tc, const CUtensorMap& tc2,
                        const GemmParams& p, int grid, cudaStream_t st) {
  static std::atomic<bool> attr_set[kMaxDevices];
  auto kern = grouped_gemm_kernel<C>;
  const int dev = current_device();
  if (dev < 0) return cudaErrorInvalidDevice;
  if (!attr_set[dev].load(std::memory_order_acquire)) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    attr_set[dev].store(true, std::memory_order_release);
  }
  if (grid <= 0) return cudaSuccess;
  GemmParams q = p;
  q.sched = (p.status != nullptr) ? p.status + kSchedCounterWord : nullptr;
  q.wait_ns = gemm_wait_limit_ns();
  launch_k(kern, grid, C::THREADS, C::SMEM_BYTES, st, ta, tb, tc, tc2, q);
  count_launches(1);
  return cudaGetLastError();
}

// Launch of the CTA-pair kernel: clusters of two, as many as can be resident
// at once (queried once per configuration), never more than tiles_upper.
template <class C>
cudaError_t launch_gemm_pair(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tc,
                             const CUtensorMap& tc2, const GemmParams& p, int tiles_upper, cudaStream_t st) {
  static std::atomic<int> max_clusters_of[kMaxDevices];
  auto kern = grouped_gemm_pair_kernel<C>;
  const int dev = current_device();
  if (dev < 0) return cudaErrorInvalidDevice;
  int max_clusters = max_clusters_of[dev].load(std::memory_order_acquire);
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;   // (see launch_k)
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(C::THREADS, 1, 1);
  cfg.dynamicSmemBytes = C::SMEM_BYTES;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;                       // (the occupancy query takes the cluster shape alone)
  if (max_clusters == 0) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    cfg.gridDim = dim3(2 * (num_sms() / 2), 1, 1);
    int n = 0;
    e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
    if (e != cudaSuccess) return e;
    if (n <= 0) return cudaErrorInvalidConfiguration;
    max_clusters = n;
    max_clusters_of[dev].store(n, std::memory_order_release);
  }
  if (tiles_upper <= 0) return cudaSuccess;
  const int clusters = tiles_upper < max_clusters ? tiles_upper : max_clusters;
  cfg.gridDim = dim3(2 * clusters, 1, 1);
  GemmParams q = p;
  q.wait_ns = gemm_wait_limit_ns();
  cfg.numAttrs = 2;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, ta, tb, tc, tc2, q);
  count_launches(1);
  return e;
}

// Output map for the TMA-store epilogue: boxes of 128 bytes x 32 rows, 128B swizzle.
inline bool make_tmap_out_bf16(CUtensorMap* map, const void* base, uint64_t cols, uint64_t rows) {
  return make_tmap_2d(map, base, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, cols, rows, 64, 32);
}
// 32-column bf16 boxes (64-byte rows, no swizzle): the last columns of a 224-wide tile
inline bool make_tmap_out_bf16_32(CUtensorMap* map, const void* base, uint64_t cols, uint64_t rows) {
  return make_tmap_2d(map, base, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, cols, rows, 32, 32, CU_TENSOR_MAP_SWIZZLE_NONE);
}
// 32-column bf16 boxes with 64-byte swizzle (the split SwiGLU-backward epilogue)
inline bool make_tmap_out_bf16_32_sw64(CUtensorMap* map, const void* base, uint64_t cols, uint64_t rows) {
  return make_tmap_2d(map, base, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, cols, rows, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B);
}
inline bool make_tmap_out_f32(CUtensorMap* map, const void* base, uint64_t cols, uint64_t rows) {
  return make_tmap_2d(map, base, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, cols, rows, 32, 32);
}

inline void set_combine(GemmParams& p, const CombineArgs& c) {
  p.cmb_row_src = c.row_src;
  p.cmb_slot_row = c.slot_row;
  p.cmb_k = c.k;
  p.cmb_count = c.count;
  p.cmb_shared = static_cast<const __nv_bfloat16*>(c.shared);
  p.cmb_y = static_cast<__nv_bfloat16*>(c.y);
}

inline GemmParams gemm_params_zero() {
  GemmParams p{};
  p.valid_cols = 1 << 30;
  return p;
}

}  // namespace moe
