// moe_permute_noalloc: the permutation step for callers that cannot allocate
// device memory.
//
// Some callers only ever receive tensor pointers and may not allocate: a
// plugin inside an inference engine that hands its kernels preallocated
// buffers, a host loop whose memory budget is fixed up front, or code that
// must not pay the device-wide synchronisation a cudaMalloc implies.  Such a
// caller cannot provide the workspace that moe_permute needs for its
// per-block histograms.  This entry point keeps that scratch in a fixed array
// of device memory that belongs to the library instead: every GPU that loads
// the library holds it (1 MiB) until the process exits.
//
// The array's name is only a host-side stand-in in host code, so its device
// address is looked up once per device with cudaGetSymbolAddress (with that
// device current) during the first call on that device, and passed to the
// kernels as a plain pointer.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "../../include/moe_gb300.h"
#include "internal.h"

namespace moe {
namespace {

// Scratch for the counting sort: ceil(T / floor(256/k)) * E histogram entries.
constexpr long long kNoAllocScratchInts = 1LL << 18;   // 1 MiB of int32
static __device__ __align__(256) int32_t g_permute_scratch[kNoAllocScratchInts];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
struct ScratchAddr {
  CUcontext ctx = nullptr;     // context the address belongs to
  int32_t* addr = nullptr;
};
ScratchAddr g_scratch[kMaxDevices];

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);

// cuCtxGetCurrent through the runtime's driver entry point (no link-time libcuda).
CtxGetCurrentFn ctx_get_current_fn() {
  static CtxGetCurrentFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CtxGetCurrentFn>(p);
  });
  return fn;
}

// Device address of g_permute_scratch in the current device's current context,
// looked up with cudaGetSymbolAddress the first time this device (in this
// context) calls, then reused.  A different current context on the same
// device (one made with the driver API) gets its own lookup.
int32_t* scratch_on_current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  CUcontext ctx = nullptr;
  CtxGetCurrentFn get_ctx = ctx_get_current_fn();
  if (get_ctx == nullptr || get_ctx(&ctx) != CUDA_SUCCESS) return nullptr;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  ScratchAddr& s = g_scratch[dev];
  if (s.addr == nullptr || ctx == nullptr || s.ctx != ctx) {
    void* p = nullptr;
    // (binds the device's primary context if no context was current yet)
    if (cudaGetSymbolAddress(&p, g_permute_scratch) != cudaSuccess || p == nullptr) return nullptr;
    if (ctx == nullptr && (get_ctx(&ctx) != CUDA_SUCCESS || ctx == nullptr)) return nullptr;
    s.ctx = ctx;
    s.addr = static_cast<int32_t*>(p);
  }
  return s.addr;
}

bool aligned16(const void* p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" moe_status moe_permute_noalloc(const moe_config* cfg, const void* x, const int32_t* topk_idx,
                                          const float* topk_gate, int32_t* counts, int32_t* offsets,
                                          int32_t* poffsets, int32_t* slot_row, int32_t* row_src,
                                          float* row_gate, void* x_perm, int32_t zero_pad, void* stream) {
  if (moe_capacity_rows(cfg) < 0) return MOE_ERR_INVALID_ARG;
  if (!aligned16(counts) || !aligned16(offsets) || !aligned16(poffsets) || !aligned16(row_src) ||
      !aligned16(x_perm))
    return MOE_ERR_INVALID_ARG;
  if (cfg->T > 0 && (!aligned16(x) || !aligned16(topk_idx) || !aligned16(slot_row))) return MOE_ERR_INVALID_ARG;
  if (topk_gate != nullptr && !aligned16(row_gate)) return MOE_ERR_INVALID_ARG;
  const long long tokens_per_chunk = kPairsPerBlock / cfg->k;
  const long long blocks = (cfg->T + tokens_per_chunk - 1) / tokens_per_chunk;
  if (blocks * cfg->E > kNoAllocScratchInts) return MOE_ERR_WORKSPACE;   // beyond the fixed scratch
  if (!device_is_gb300()) return MOE_ERR_UNSUPPORTED;
  int32_t* hist = scratch_on_current_device();
  if (hist == nullptr) return MOE_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // Every histogram entry the scan reads is written by this call first, so
  // nothing left in the array by an earlier call is ever read.
  if (launch_permute_maps(topk_idx, topk_gate, cfg->T, cfg->E, cfg->k, hist, counts, offsets, poffsets, slot_row,
                          row_src, topk_gate != nullptr ? row_gate : nullptr, nullptr, st) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (launch_gather_rows(x, slot_row, cfg->T, cfg->k, cfg->H, x_perm, st) != cudaSuccess) return MOE_ERR_CUDA;
  if (zero_pad && launch_zero_pad_rows(counts, poffsets, cfg->E, cfg->H, x_perm, st) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}
