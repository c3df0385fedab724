// C ABI of the library (declared in include/moe_gb300.h): argument checks on
// the host, buffer layouts, and the fixed launch sequences of the layer's
// forward and backward passes.  No call here allocates device memory,
// synchronises, or reads a device value on the host.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/moe_gb300.h"
#include "internal.h"

namespace moe {

namespace {
struct DevInfo {
  int sms = 0;
  bool gb300 = false;
  bool probed = false;
};
DevInfo g_dev[64];
std::mutex g_dev_mu;

DevInfo& dev_info() {
  int d = 0;
  if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= 64) {
    static DevInfo none;
    return none;
  }
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DevInfo& info = g_dev[d];
  if (!info.probed) {
    int major = 0, minor = 0, sms = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, d);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, d);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, d);
    info.sms = sms > 0 ? sms : 1;
    info.gb300 = (major == 10 && minor == 3);
    info.probed = true;
  }
  return info;
}
}  // namespace

std::atomic<unsigned long long> g_launches{0};
void count_launches(int n) { g_launches.fetch_add(static_cast<unsigned long long>(n), std::memory_order_relaxed); }

int num_sms() { return dev_info().sms; }

namespace {
std::atomic<unsigned long long> g_wait_limit_ns{0};
}  // namespace
unsigned long long gemm_wait_limit_ns() { return g_wait_limit_ns.load(std::memory_order_relaxed); }
bool device_is_gb300() { return dev_info().gb300; }

}  // namespace moe

using namespace moe;

namespace {

constexpr size_t kAlign = 256;
// Whether the layer forward fuses the combine into fc2 (where H % 256 == 0).
// Off: measured on GB300 the fused epilogue costs fc2 more than the separate
// combine kernel takes (DeepSeek-like: 2.17 ms against 1.86 + 0.19 ms), since
// that kernel already streams at the HBM rate.  MOE_GG_FC2_COMBINE offers it.
#ifndef MOE_FUSE_COMBINE
#define MOE_FUSE_COMBINE 0
#endif
constexpr bool kFuseCombine = MOE_FUSE_COMBINE != 0;
constexpr size_t kStatusBytes = 256;   // status word region at the start of the workspace
constexpr size_t kNone = SIZE_MAX;

size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

bool config_ok(const moe_config* c) {
  if (c == nullptr) return false;
  if (c->T < 0 || c->H <= 0 || c->E <= 0 || c->k <= 0 || c->F <= 0 || c->S < 0) return false;
  if (c->k > kMaxK || c->k > c->E || c->E > kMaxE) return false;
  if (c->H % 128 || c->F % 128 || c->S % 128) return false;
  if (c->score != MOE_SCORE_SOFTMAX && c->score != MOE_SCORE_SIGMOID) return false;
  if (c->dtype != MOE_GEMM_BF16 && c->dtype != MOE_GEMM_MXFP8 && c->dtype != MOE_GEMM_NVFP4) return false;
  if (c->dtype != MOE_GEMM_BF16 && c->T % 128 != 0) return false;   // whole 128-row scale tiles
  // NVFP4: 256-element k-blocks along H, F and S
  if (c->dtype == MOE_GEMM_NVFP4 && (c->H % 256 || c->F % 256 || c->S % 256)) return false;
  const long long pairs = static_cast<long long>(c->T) * c->k;
  if (pairs + 128LL * c->E >= (1LL << 31)) return false;
  return true;
}

int cap_rows(const moe_config* c) {
  const long long r = static_cast<long long>(c->T) * c->k + 127LL * c->E;
  return static_cast<int>((r + 127) / 128 * 128);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool dev_ptr_ok(const void* p) { return p != nullptr && aligned16(p); }
bool f32_ptr_ok(const float* p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

moe_status cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

#define MOE_TRY(expr)                                   \
  do {                                                  \
    cudaError_t e_ = (expr);                            \
    if (e_ != cudaSuccess) return MOE_ERR_CUDA;         \
  } while (0)

template <class T>
T* at(void* base, size_t off) {
  return reinterpret_cast<T*>(static_cast<char*>(base) + off);
}

size_t hist_bytes(const moe_config* c) {
  const long long tpb = kPairsPerBlock / c->k;            // tokens per counting-sort chunk
  const long long nb = (c->T + tpb - 1) / tpb;
  return static_cast<size_t>(nb) * c->E * sizeof(int32_t);
}

moe_status compute_layout(const moe_config* c, int with_bwd, moe_act_layout* L) {
  if (!config_ok(c) || L == nullptr) return MOE_ERR_INVALID_ARG;
  const size_t T = c->T, H = c->H, E = c->E, k = c->k, F = c->F, S = c->S;
  const size_t cap = static_cast<size_t>(cap_rows(c));
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align_up(off + (bytes == 0 ? 1 : bytes));
    return o;
  };
  L->cap = static_cast<int32_t>(cap);
  L->backward = with_bwd ? 1 : 0;
  L->logits = take(T * E * 4);
  L->topk_idx = take(T * k * 4);
  L->topk_gate = take(T * k * 4);
  L->counts = take(E * 4);
  L->offsets = take((E + 1) * 4);
  L->poffsets = take((E + 1) * 4);
  L->slot_row = take(T * k * 4);
  L->row_src = take(cap * 4);
  L->row_gate = take(cap * 4);
  L->x_perm = take(cap * H * 2);
  L->z = take(cap * 2 * F * 2);
  L->h = take(cap * F * 2);
  L->o = take(cap * H * 2);
  if (S > 0) {
    L->zs = take(T * 2 * S * 2);
    L->hs = take(T * S * 2);
    L->os = take(T * H * 2);
  } else {
    L->zs = L->hs = L->os = kNone;
  }
  if (with_bwd) {
    L->dy_perm = take(cap * H * 2);
    L->dz = take(cap * 2 * F * 2);
    L->dx_perm = take(cap * H * 2);
    L->dgate_part = take(cap * (F / 128) * 4);
    L->dlogits = take(T * E * 4);
    L->row_dlogit = take(cap * 4);
    if (S > 0) {
      L->dzs = take(T * 2 * S * 2);
      L->dxs = take(T * H * 2);
    } else {
      L->dzs = L->dxs = kNone;
    }
    if (c->dtype == MOE_GEMM_MXFP8) {   // dz^T and h'^T as the weight gradients read them
      L->dz_qt = take(2 * F * cap);
      L->dz_qt_sf = take(2 * F * cap / 32);
      L->h_qt = take(F * cap);
      L->h_qt_sf = take(F * cap / 32);
    } else {
      L->dz_qt = L->dz_qt_sf = L->h_qt = L->h_qt_sf = kNone;
    }
  } else {
    L->dy_perm = L->dz = L->dx_perm = L->dgate_part = L->dlogits = L->row_dlogit = L->dzs = L->dxs = kNone;
    L->dz_qt = L->dz_qt_sf = L->h_qt = L->h_qt_sf = kNone;
  }
  L->total = off;
  return MOE_OK;
}

// ---------------------------------------------------------------- MXFP8 buffers
struct MxBuf {
  size_t q = kNone, sf = kNone;   // E4M3 codes, E8M0 scale tiles (codes / 32 bytes)
};

// The routed fc2 and fc1 data gradient (N = H) run on 256 x 224 tiles when H
// allows: their B operands (W2, W1^T) then keep scale tiles per 224 rows.
// (The fused fc2 + combine keeps 256-wide tiles and W2's 128-row tiles.)
bool mx_b224(const moe_config* c) { return c->H % 224 == 0 && !kFuseCombine; }
// x^T, the B operand of the routed fc1 weight gradient (N = H), likewise.
int mx_xt_group(const moe_config* c) { return c->H % 224 == 0 ? kMxScaleGroup224 : 128; }
// The routed fc2 weight gradient as dW2^T = h'^T-rows x dy^T (M = F, N = H)
// on 256 x 224 tiles stored transposed: dy^T then keeps 224-row scale groups.
bool mx_dw2_trans(const moe_config* c) { return c->H % 224 == 0 && c->F % 256 == 0; }

// Transient quantised activations, placed in the workspace after the
// histograms.  The forward, dgrad and wgrad calls each use their own set; the
// region is the largest of the three.
struct MxWs {
  MxBuf x, h, xs, hs;                             // forward
  MxBuf dy, dz, dys, dzs;                         // dgrad
  MxBuf xT, dyT, dzsT, xsT, dysT, hsT;            // wgrad (transposed: blocks along tokens; dz^T, h'^T in act)
  size_t total = 0;
};

MxWs mx_ws_layout(const moe_config* c) {
  MxWs m;
  const size_t T = c->T, H = c->H, F = c->F, S = c->S, cap = static_cast<size_t>(cap_rows(c));
  size_t off = 0, end = 0;
  auto buf = [&](size_t elems, size_t sf_bytes = 0) {
    MxBuf b;
    b.q = off;
    off = align_up(off + (elems ? elems : 1));
    b.sf = off;
    if (sf_bytes == 0) sf_bytes = elems / 32;
    off = align_up(off + (sf_bytes ? sf_bytes : 1));
    return b;
  };
  auto region = [&]() { end = off > end ? off : end; off = 0; };
  // xs / dys: x and dy quantised per token (fed to the shared expert, and
  // gathered into expert order for the routed experts)
  m.x = buf(cap * H); m.h = buf(cap * F); m.xs = buf(T * H);
  if (S) m.hs = buf(T * S);
  region();
  m.dy = buf(cap * H); m.dz = buf(cap * 2 * F); m.dys = buf(T * H);
  if (S) m.dzs = buf(T * 2 * S);
  region();
  m.dyT = buf(H * cap, mx_scale_bytes(H, cap, mx_dw2_trans(c) ? kMxScaleGroup224 : 128));
  m.xT = buf(H * cap, mx_scale_bytes(H, cap, mx_xt_group(c)));   // rows grouped by 224 for the 256 x 224 tiles
  if (S) { m.dzsT = buf(2 * S * T); m.xsT = buf(H * T); m.dysT = buf(H * T); m.hsT = buf(S * T); }
  region();
  m.total = end;
  return m;
}

// Quantised weights, prepared once by moe_prepare_mxfp8_weights.
struct MxW {
  MxBuf w1, w2, w1t, w2t, s1, s2, s1t, s2t;
  size_t total = 0;
};


MxW mx_weight_layout(const moe_config* c) {
  MxW m;
  const size_t H = c->H, E = c->E, F = c->F, S = c->S;
  const int g = mx_b224(c) ? kMxScaleGroup224 : 128;
  size_t off = 0;
  auto buf = [&](size_t elems, size_t sf_bytes) {
    MxBuf b;
    b.q = off;
    off = align_up(off + elems);
    b.sf = off;
    off = align_up(off + sf_bytes);
    return b;
  };
  m.w1 = buf(E * 2 * F * H, E * 2 * F * H / 32);                 // [E*2F, H], gate/up interleaved (fc1)
  m.w2 = buf(E * H * F, mx_scale_bytes(E * H, F, g));            // [E*H, F]  (fc2)
  m.w1t = buf(E * H * 2 * F, E * mx_scale_bytes(H, 2 * F, g));   // [E, H, 2F] = W1_e^T, blocks along 2F (fc1 dgrad)
  m.w2t = buf(E * F * H, E * F * H / 32);                       // [E, F, H] = W2_e^T, blocks along H (fc2 dgrad)
  if (S) {
    m.s1 = buf(2 * S * H, 2 * S * H / 32); m.s2 = buf(H * S, H * S / 32);
    m.s1t = buf(H * 2 * S, H * 2 * S / 32); m.s2t = buf(S * H, S * H / 32);
  }
  m.total = off;
  return m;
}

size_t mx_ws_base(const moe_config* c) { return kStatusBytes + align_up(hist_bytes(c)); }

// ---------------------------------------------------------------- NVFP4 buffers
// E2M1 codes (elems / 2 bytes) and E4M3 scale tiles (elems / 16 bytes), and
// one fp32 amax per quantised tensor.
struct Nv4Buf {
  size_t q = kNone, sf = kNone;
};

Nv4Buf nv4_buf(size_t& off, size_t elems) {
  Nv4Buf b;
  b.q = off;
  off = align_up(off + (elems / 2 ? elems / 2 : 1));
  b.sf = off;
  off = align_up(off + (elems / 16 ? elems / 16 : 1));
  return b;
}

// Forward activations: x quantised per token (xs) and gathered into expert
// order (x), h (expert order), hs (shared expert); amax slots x, h, hs.
struct Nv4Ws {
  Nv4Buf x, h, xs, hs;
  size_t amax = kNone;
  size_t total = 0;
};

Nv4Ws nv4_ws_layout(const moe_config* c) {
  Nv4Ws m;
  const size_t T = c->T, H = c->H, F = c->F, S = c->S, cap = static_cast<size_t>(cap_rows(c));
  size_t off = 0;
  m.amax = off;
  off = align_up(off + 4 * sizeof(float));
  m.x = nv4_buf(off, cap * H);
  m.h = nv4_buf(off, cap * F);
  m.xs = nv4_buf(off, T * H);
  if (S) m.hs = nv4_buf(off, T * S);
  m.total = off;
  return m;
}

// Weights, prepared once by moe_prepare_nvfp4_weights: w1 (gate/up rows
// interleaved in 128-row blocks), w2, and the shared expert's; amax slots w1,
// w2, s1, s2.
struct Nv4W {
  Nv4Buf w1, w2, s1, s2;
  size_t amax = kNone;
  size_t total = 0;
};

Nv4W nv4_weight_layout(const moe_config* c) {
  Nv4W m;
  const size_t H = c->H, E = c->E, F = c->F, S = c->S;
  size_t off = 0;
  m.amax = off;
  off = align_up(off + 4 * sizeof(float));
  m.w1 = nv4_buf(off, E * 2 * F * H);
  m.w2 = nv4_buf(off, E * H * F);
  if (S) { m.s1 = nv4_buf(off, 2 * S * H); m.s2 = nv4_buf(off, H * S); }
  m.total = off;
  return m;
}

// Counters of the combine fused into fc2 (one int per token and 256-column
// tile of y), after the quantised activations; zero between launches.
size_t combine_count_bytes(const moe_config* c) {
  return c->H % 256 == 0 ? static_cast<size_t>(c->T) * (c->H / 256) * sizeof(int32_t) : 0;
}
size_t combine_count_offset(const moe_config* c) {
  size_t b = kStatusBytes + align_up(hist_bytes(c));
  if (c->dtype == MOE_GEMM_MXFP8) b += mx_ws_layout(c).total;
  if (c->dtype == MOE_GEMM_NVFP4) b += nv4_ws_layout(c).total;
  return b;
}

CombineArgs combine_args(const moe_config* c, const moe_gemm_args* a, void* ws) {
  CombineArgs r;
  r.row_src = a->a_rows;
  r.slot_row = a->slot_row;
  r.k = c->k;
  r.count = at<int32_t>(ws, combine_count_offset(c));
  r.shared = a->aux;
  r.y = a->c2;
  return r;
}

moe_status check_device() { return device_is_gb300() ? MOE_OK : MOE_ERR_UNSUPPORTED; }

int* status_ptr(void* ws) { return static_cast<int*>(ws); }
int32_t* hist_ptr(void* ws) { return at<int32_t>(ws, kStatusBytes); }

}  // namespace

namespace {
// The host-side checks of one grouped-GEMM call that depend on the op and
// the operand type, all before the device check so that a bad argument
// reads as MOE_ERR_INVALID_ARG (or an op the type does not offer as
// MOE_ERR_UNSUPPORTED) on any machine.
moe_status gemm_args_check(const moe_config* cfg, const moe_gemm_args* a, bool dense) {
  const bool fc1 = a->op == MOE_GG_FC1_SWIGLU || a->op == MOE_GG_FC1_SWIGLU_GATHERED;
  if (fc1 && a->c2 != nullptr && !aligned16(a->c2)) return MOE_ERR_INVALID_ARG;
  if (a->op == MOE_GG_DGRAD_FC2 && !dev_ptr_ok(a->aux)) return MOE_ERR_INVALID_ARG;
  if (a->op < MOE_GG_FC1_SWIGLU || a->op > MOE_GG_FC2_COMBINE) return MOE_ERR_INVALID_ARG;
  if (a->op == MOE_GG_FC2_COMBINE) {
    if (dense || cfg->dtype == MOE_GEMM_NVFP4 || cfg->H % 256 != 0) return MOE_ERR_INVALID_ARG;
    if (cfg->T > 0 && (!dev_ptr_ok(a->c2) || !dev_ptr_ok(a->a_rows) || !dev_ptr_ok(a->slot_row)))
      return MOE_ERR_INVALID_ARG;
    if (a->aux != nullptr && !aligned16(a->aux)) return MOE_ERR_INVALID_ARG;
  }
  if (cfg->dtype == MOE_GEMM_BF16) {
    if (a->op == MOE_GG_FC1_SWIGLU_GATHERED && (dense || !dev_ptr_ok(a->a_rows))) return MOE_ERR_INVALID_ARG;
    if (a->q_codes || a->q_scales || a->qt_codes || a->qt_scales) return MOE_ERR_INVALID_ARG;
    return (a->b_scale_group == 0 || a->b_scale_group == 128) ? MOE_OK : MOE_ERR_INVALID_ARG;
  }
  if (a->op == MOE_GG_FC1_SWIGLU_GATHERED) return MOE_ERR_INVALID_ARG;     // bf16 only
  // MXFP8 copies of the output from the epilogue: dz (fc2 data gradient) or h' (fc1)
  const bool want_q = a->q_codes != nullptr || a->q_scales != nullptr;
  const bool want_qt = a->qt_codes != nullptr || a->qt_scales != nullptr;
  if (want_q || want_qt) {
    const bool op_ok = (a->op == MOE_GG_DGRAD_FC2 && gemm_mx_dgrad_fc2_quantises(cfg->F)) ||
                       a->op == MOE_GG_FC1_SWIGLU;
    if (cfg->dtype != MOE_GEMM_MXFP8 || !op_ok || dense) return MOE_ERR_INVALID_ARG;
    if (want_q && (!dev_ptr_ok(a->q_codes) || !dev_ptr_ok(a->q_scales))) return MOE_ERR_INVALID_ARG;
    if (want_qt && (!dev_ptr_ok(a->qt_codes) || !dev_ptr_ok(a->qt_scales))) return MOE_ERR_INVALID_ARG;
  }
  if (!dev_ptr_ok(a->a_scales) || !dev_ptr_ok(a->b_scales)) return MOE_ERR_INVALID_ARG;
  // B's scale tiles grouped by 224 rows: MXFP8 FC2 / DGRAD_FC1 / WGRAD_FC1 (the GEMMs
  // whose N is H) and WGRAD_FC2 with its operands swapped (F % 256 == 0), routed,
  // H % 224 == 0
  if (a->b_scale_group != 0 && a->b_scale_group != 128) {
    if (a->b_scale_group != kMxScaleGroup224 || cfg->dtype != MOE_GEMM_MXFP8 || dense || cfg->H % 224 != 0 ||
        (a->op != MOE_GG_FC2 && a->op != MOE_GG_DGRAD_FC1 && a->op != MOE_GG_WGRAD_FC1 &&
         a->op != MOE_GG_WGRAD_FC2) ||
        (a->op == MOE_GG_WGRAD_FC2 && cfg->F % 256 != 0))
      return MOE_ERR_INVALID_ARG;
  }
  if (dense && a->dense_rows % 128 != 0) return MOE_ERR_INVALID_ARG;
  if (cfg->dtype == MOE_GEMM_NVFP4) {
    if (!f32_ptr_ok(a->a_amax) || !f32_ptr_ok(a->b_amax)) return MOE_ERR_INVALID_ARG;
    if (a->op != MOE_GG_FC1_SWIGLU && a->op != MOE_GG_FC2) return MOE_ERR_UNSUPPORTED;   // forward GEMMs only
  }
  return MOE_OK;
}
}  // namespace

extern "C" {

const char* moe_status_string(moe_status s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported device or shape";
    case MOE_ERR_CUDA: return "CUDA call failed";
    case MOE_ERR_WORKSPACE: return "workspace or activation buffer too small";
    case MOE_ERR_BAD_INDEX: return "expert index out of range";
    case MOE_ERR_TIMEOUT: return "device pipeline wait timed out";
  }
  return "unknown status";
}

int32_t moe_version(void) { return 0x000100; }

void moe_debug_set_wait_limit_ns(uint64_t ns) { g_wait_limit_ns.store(ns, std::memory_order_relaxed); }

uint64_t moe_kernel_launches(void) { return g_launches.load(std::memory_order_relaxed); }

int32_t moe_capacity_rows(const moe_config* cfg) { return config_ok(cfg) ? cap_rows(cfg) : -1; }

moe_status moe_activation_layout(const moe_config* cfg, int32_t with_backward, moe_act_layout* out) {
  return compute_layout(cfg, with_backward, out);
}

size_t moe_workspace_bytes(const moe_config* cfg) {
  if (!config_ok(cfg)) return 0;
  return combine_count_offset(cfg) + align_up(combine_count_bytes(cfg));
}

size_t moe_mxfp8_weights_bytes(const moe_config* cfg) {
  if (!config_ok(cfg)) return 0;
  return mx_weight_layout(cfg).total;
}

moe_status moe_quantize_mxfp8(const void* src, int32_t batch, int32_t rows, int32_t cols, int32_t mode,
                              uint8_t* codes, uint8_t* scales, void* stream) {
  if (batch < 0 || rows < 0 || cols < 0) return MOE_ERR_INVALID_ARG;
  const long long n = static_cast<long long>(batch) * rows * cols;
  if (n == 0) return MOE_OK;
  if (!dev_ptr_ok(src) || !dev_ptr_ok(codes) || !dev_ptr_ok(scales)) return MOE_ERR_INVALID_ARG;
  if (cols % 128 != 0) return MOE_ERR_INVALID_ARG;
  const long long R = static_cast<long long>(batch) * rows;
  bool shape_ok = false;
  switch (mode) {
    case MOE_MX_ROWS: shape_ok = R % 128 == 0; break;
    case MOE_MX_ROWS_GATE_UP: shape_ok = rows % 256 == 0; break;
    case MOE_MX_COLS_T: shape_ok = rows % 128 == 0; break;
    case MOE_MX_ROWS_G224: shape_ok = R % 224 == 0; break;
    case MOE_MX_COLS_T_G224: shape_ok = rows % 128 == 0 && cols % 224 == 0; break;
    default: break;
  }
  if (!shape_ok) return MOE_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (moe_status s = check_device(); s != MOE_OK) return s;
  switch (mode) {
    case MOE_MX_ROWS:
      return cuda_status(launch_quantize_rows(src, R, cols, 0, codes, scales, st));
    case MOE_MX_ROWS_GATE_UP:
      return cuda_status(launch_quantize_rows(src, R, cols, rows / 2, codes, scales, st));
    case MOE_MX_COLS_T:
      return cuda_status(launch_quantize_cols(src, batch, rows, cols, codes, scales, st));
    case MOE_MX_ROWS_G224:
      return cuda_status(launch_quantize_rows(src, R, cols, 0, codes, scales, st, kMxScaleGroup224));
    default:   // MOE_MX_COLS_T_G224
      return cuda_status(launch_quantize_cols(src, batch, rows, cols, codes, scales, st, kMxScaleGroup224));
  }
}

moe_status moe_prepare_mxfp8_weights(const moe_config* cfg, const moe_weights* w, void* mx, size_t mx_bytes,
                                     void* stream) {
  if (!config_ok(cfg) || w == nullptr || !dev_ptr_ok(mx) || !dev_ptr_ok(w->w1) || !dev_ptr_ok(w->w2))
    return MOE_ERR_INVALID_ARG;
  if (cfg->S > 0 && (!dev_ptr_ok(w->w1_shared) || !dev_ptr_ok(w->w2_shared))) return MOE_ERR_INVALID_ARG;
  const MxW L = mx_weight_layout(cfg);
  if (mx_bytes < L.total) return MOE_ERR_WORKSPACE;
  if (moe_status s = check_device(); s != MOE_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int H = cfg->H, E = cfg->E, F = cfg->F, S = cfg->S;
  auto q = [&](const MxBuf& b) { return at<uint8_t>(mx, b.q); };
  auto f = [&](const MxBuf& b) { return at<uint8_t>(mx, b.sf); };
  MOE_TRY(launch_quantize_rows(w->w1, static_cast<long long>(E) * 2 * F, H, F, q(L.w1), f(L.w1), st));
  const int g = mx_b224(cfg) ? kMxScaleGroup224 : 128;
  MOE_TRY(launch_quantize_rows(w->w2, static_cast<long long>(E) * H, F, 0, q(L.w2), f(L.w2), st, g));
  MOE_TRY(launch_quantize_cols(w->w1, E, 2 * F, H, q(L.w1t), f(L.w1t), st, g));
  MOE_TRY(launch_quantize_cols(w->w2, E, H, F, q(L.w2t), f(L.w2t), st));
  if (S > 0) {
    MOE_TRY(launch_quantize_rows(w->w1_shared, 2 * S, H, S, q(L.s1), f(L.s1), st));
    MOE_TRY(launch_quantize_rows(w->w2_shared, H, S, 0, q(L.s2), f(L.s2), st));
    MOE_TRY(launch_quantize_cols(w->w1_shared, 1, 2 * S, H, q(L.s1t), f(L.s1t), st));
    MOE_TRY(launch_quantize_cols(w->w2_shared, 1, H, S, q(L.s2t), f(L.s2t), st));
  }
  return MOE_OK;
}

size_t moe_nvfp4_weights_bytes(const moe_config* cfg) {
  if (!config_ok(cfg) || cfg->dtype != MOE_GEMM_NVFP4) return 0;
  return nv4_weight_layout(cfg).total;
}

moe_status moe_quantize_nvfp4(const void* src, int32_t batch, int32_t rows, int32_t cols, int32_t mode,
                              uint8_t* codes, uint8_t* scales, float* amax, void* stream) {
  if (batch < 0 || rows < 0 || cols < 0) return MOE_ERR_INVALID_ARG;
  if (!f32_ptr_ok(amax)) return MOE_ERR_INVALID_ARG;
  const long long n = static_cast<long long>(batch) * rows * cols;
  if (n > 0 && (!dev_ptr_ok(src) || !dev_ptr_ok(codes) || !dev_ptr_ok(scales))) return MOE_ERR_INVALID_ARG;
  if (cols % 64 != 0) return MOE_ERR_INVALID_ARG;
  if ((static_cast<long long>(batch) * rows) % 128 != 0) return MOE_ERR_INVALID_ARG;
  if (mode == MOE_MX_ROWS_GATE_UP && rows % 256 != 0) return MOE_ERR_INVALID_ARG;
  if (mode != MOE_MX_ROWS && mode != MOE_MX_ROWS_GATE_UP) return MOE_ERR_INVALID_ARG;
  if (moe_status s = check_device(); s != MOE_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const long long R = static_cast<long long>(batch) * rows;
  MOE_TRY(launch_amax_bf16(src, R, cols, nullptr, nullptr, amax, st));
  return cuda_status(
      launch_quantize_rows_nv4(src, R, cols, mode == MOE_MX_ROWS_GATE_UP ? rows / 2 : 0, amax, codes, scales, st));
}

moe_status moe_prepare_nvfp4_weights(const moe_config* cfg, const moe_weights* w, void* buf, size_t bytes,
                                     void* stream) {
  if (!config_ok(cfg) || cfg->dtype != MOE_GEMM_NVFP4 || w == nullptr || !dev_ptr_ok(buf) || !dev_ptr_ok(w->w1) ||
      !dev_ptr_ok(w->w2))
    return MOE_ERR_INVALID_ARG;
  if (cfg->S > 0 && (!dev_ptr_ok(w->w1_shared) || !dev_ptr_ok(w->w2_shared))) return MOE_ERR_INVALID_ARG;
  const Nv4W L = nv4_weight_layout(cfg);
  if (bytes < L.total) return MOE_ERR_WORKSPACE;
  if (moe_status s = check_device(); s != MOE_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const long long H = cfg->H, E = cfg->E, F = cfg->F, S = cfg->S;
  float* amax = at<float>(buf, L.amax);
  auto q = [&](const Nv4Buf& b) { return at<uint8_t>(buf, b.q); };
  auto f = [&](const Nv4Buf& b) { return at<uint8_t>(buf, b.sf); };
  MOE_TRY(launch_amax_bf16(w->w1, E * 2 * F, static_cast<int>(H), nullptr, nullptr, amax + 0, st));
  MOE_TRY(launch_quantize_rows_nv4(w->w1, E * 2 * F, static_cast<int>(H), static_cast<int>(F), amax + 0, q(L.w1),
                                   f(L.w1), st));
  MOE_TRY(launch_amax_bf16(w->w2, E * H, static_cast<int>(F), nullptr, nullptr, amax + 1, st));
  MOE_TRY(launch_quantize_rows_nv4(w->w2, E * H, static_cast<int>(F), 0, amax + 1, q(L.w2), f(L.w2), st));
  if (S > 0) {
    MOE_TRY(launch_amax_bf16(w->w1_shared, 2 * S, static_cast<int>(H), nullptr, nullptr, amax + 2, st));
    MOE_TRY(launch_quantize_rows_nv4(w->w1_shared, 2 * S, static_cast<int>(H), static_cast<int>(S), amax + 2,
                                     q(L.s1), f(L.s1), st));
    MOE_TRY(launch_amax_bf16(w->w2_shared, H, static_cast<int>(S), nullptr, nullptr, amax + 3, st));
    MOE_TRY(launch_quantize_rows_nv4(w->w2_shared, H, static_cast<int>(S), 0, amax + 3, q(L.s2), f(L.s2), st));
  }
  return MOE_OK;
}

moe_status moe_workspace_init(void* ws, size_t ws_bytes, void* stream) {
  if (!dev_ptr_ok(ws) || ws_bytes < kStatusBytes) return MOE_ERR_INVALID_ARG;
  return cuda_status(cudaMemsetAsync(ws, 0, ws_bytes, static_cast<cudaStream_t>(stream)));
}

moe_status moe_read_device_status(const void* ws, int32_t* code, void* stream) {
  if (!dev_ptr_ok(ws) || code == nullptr) return MOE_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  MOE_TRY(cudaStreamSynchronize(st));
  int32_t v = 0;
  MOE_TRY(cudaMemcpy(&v, ws, sizeof(v), cudaMemcpyDeviceToHost));
  *code = v;
  return MOE_OK;
}

moe_status moe_topk_gating(const moe_config* cfg, const float* logits, const float* bias, int32_t* topk_idx,
                           float* topk_gate, void* stream) {
  if (!config_ok(cfg)) return MOE_ERR_INVALID_ARG;
  if (cfg->T > 0 && (!dev_ptr_ok(logits) || !dev_ptr_ok(topk_idx) || !dev_ptr_ok(topk_gate)))
    return MOE_ERR_INVALID_ARG;
  if (moe_status s = check_device(); s != MOE_OK) return s;
  return cuda_status(launch_topk(logits, cfg->score == MOE_SCORE_SIGMOID ? bias : nullptr, cfg->T, cfg->E, cfg->k,
                                 cfg->score, topk_idx, topk_gate, static_cast<cudaStream_t>(stream)));
}

moe_status moe_router_topk(const moe_config* cfg, const void* x, const void* w_router, const float* bias,
                           float* logits, int32_t* topk_idx, float* topk_gate, void* ws, void* stream) {
  if (!config_ok(cfg) || !dev_ptr_ok(ws)) return MOE_ERR_INVALID_ARG;
  if (cfg->T > 0 && (!dev_ptr_ok(x) || !dev_ptr_ok(w_router) || !dev_ptr_ok(logits) || !dev_ptr_ok(topk_idx) ||
                     !dev_ptr_ok(topk_gate)))
    return MOE_ERR_INVALID_ARG;
  if (moe_status s = check_device(); s != MOE_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  MOE_TRY(gemm_router(x, w_router, cfg->T, cfg->H, cfg->E, logits, status_ptr(ws), st));
  return moe_topk_gating(cfg, logits, bias, topk_idx, topk_gate, stream);
}

moe_status moe_permute(const moe_config* cfg, const void* x, const int32_t* topk_idx, const float* topk_gate,
                       int32_t* counts, int32_t* offsets, int32_t* poffsets, int32_t* slot_row, int32_t* row_src,
                       float* row_gate, void* x_perm, int32_t zero_pad, void* ws, void* stream) {
  if (!config_ok(cfg) || !dev_ptr_ok(ws) || !dev_ptr_ok(counts) || !dev_ptr_ok(offsets) || !dev_ptr_ok(poffsets) ||
      !dev_ptr_ok(row_src) || !dev_ptr_ok(x_perm))
    return MOE_ERR_INVALID_ARG;
  if (cfg->T > 0 && (!dev_ptr_ok(x) || !dev_ptr_ok(topk_idx) || !dev_ptr_ok(slot_row))) return MOE_ERR_INVALID_ARG;
  if (topk_gate != nullptr && !dev_ptr_ok(row_gate)) return MOE_ERR_INVALID_ARG;
  if (moe_status s = check_device(); s != MOE_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  MOE_TRY(launch_permute_gather(topk_idx, topk_gate, cfg->T, cfg->E, cfg->k, hist_ptr(ws),
                                status_ptr(ws) + kMapsDoneWord, counts, offsets, poffsets, slot_row, row_src,
                                topk_gate != nullptr ? row_gate : nullptr, x, cfg->H, x_perm, zero_pad ? 1 : 0,
                                status_ptr(ws), st));
  return MOE_OK;
}

moe_status moe_grouped_gemm(const moe_config* cfg, const moe_gemm_args* a, void* ws, void* stream) {
  if (!config_ok(cfg) || a == nullptr || !dev_ptr_ok(ws)) return MOE_ERR_INVALID_ARG;
  // (DGRAD_FC2 writing both MXFP8 copies of dz may leave the bf16 dz out, FC1
  // writing the row copy of h' the bf16 h')
  const bool c_optional = a->c == nullptr && ((a->op == MOE_GG_DGRAD_FC2 && a->q_codes != nullptr &&
                                               a->qt_codes != nullptr) ||
                                              (a->op == MOE_GG_FC1_SWIGLU && a->q_codes != nullptr));
  if (!dev_ptr_ok(a->a) || !dev_ptr_ok(a->b) || (!c_optional && !dev_ptr_ok(a->c))) return MOE_ERR_INVALID_ARG;
  const bool dense = a->dense_rows > 0;
  if (!dense && !dev_ptr_ok(a->poffsets)) return MOE_ERR_INVALID_ARG;
  if (a->dense_rows < 0) return MOE_ERR_INVALID_ARG;
  if (moe_status s = gemm_args_check(cfg, a, dense); s != MOE_OK) return s;
  if (moe_status s = check_device(); s != MOE_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int H = cfg->H;
  const int F = dense ? (cfg->S > 0 ? cfg->S : cfg->F) : cfg->F;
  const int E = dense ? 1 : cfg->E;
  const int rows = dense ? a->dense_rows : cap_rows(cfg);
  const int32_t* po = dense ? nullptr : a->poffsets;
  int* status = status_ptr(ws);
  if (cfg->dtype == MOE_GEMM_NVFP4) {
    if (!dev_ptr_ok(a->a_scales) || !dev_ptr_ok(a->b_scales) || !f32_ptr_ok(a->a_amax) || !f32_ptr_ok(a->b_amax))
      return MOE_ERR_INVALID_ARG;
    if (dense && a->dense_rows % 128 != 0) return MOE_ERR_INVALID_ARG;
    switch (a->op) {
      case MOE_GG_FC1_SWIGLU:
        if (a->c2 != nullptr && !aligned16(a->c2)) return MOE_ERR_INVALID_ARG;
        return cuda_status(gemm_nv4_fc1(a->a, a->a_scales, a->a_amax, rows, H, a->b, a->b_scales, a->b_amax, E, F, po,
                                        a->dense_rows, a->row_gate, a->c, a->c2, nullptr, status, st));
      case MOE_GG_FC2:
        return cuda_status(gemm_nv4_nt_bf16(a->a, a->a_scales, a->a_amax, rows, F, a->b, a->b_scales, a->b_amax, E, H,
                                            po, a->dense_rows, a->c, status, st));
      case MOE_GG_DGRAD_FC2:
      case MOE_GG_DGRAD_FC1:
      case MOE_GG_WGRAD_FC1:
      case MOE_GG_WGRAD_FC2:
        return MOE_ERR_UNSUPPORTED;            // NVFP4: forward GEMMs only
      default:
        return MOE_ERR_INVALID_ARG;
    }
  }
  if (cfg->dtype == MOE_GEMM_MXFP8) {
    if (!dev_ptr_ok(a->a_scales) || !dev_ptr_ok(a->b_scales)) return MOE_ERR_INVALID_ARG;
    if (dense && a->dense_rows % 128 != 0) return MOE_ERR_INVALID_ARG;
    switch (a->op) {
      case MOE_GG_FC1_SWIGLU: {
        if (a->c2 != nullptr && !aligned16(a->c2)) return MOE_ERR_INVALID_ARG;
        const MxOutQ q{static_cast<uint8_t*>(a->q_codes), static_cast<uint8_t*>(a->q_scales),
                       static_cast<uint8_t*>(a->qt_codes), static_cast<uint8_t*>(a->qt_scales)};
        const bool any_q = q.codes != nullptr || q.codes_t != nullptr;
        return cuda_status(gemm_mx_fc1(a->a, a->a_scales, rows, H, a->b, a->b_scales, E, F, po, a->dense_rows,
                                       a->row_gate, a->c, a->c2, status, st, any_q ? &q : nullptr));
      }
      case MOE_GG_FC2:
        return cuda_status(gemm_mx_nt_bf16(a->a, a->a_scales, rows, F, a->b, a->b_scales, E, H, po, a->dense_rows,
                                           a->c, status, st, a->b_scale_group == 0 ? 128 : a->b_scale_group));
      case MOE_GG_FC2_COMBINE:
        return cuda_status(gemm_mx_fc2_combine(a->a, a->a_scales, rows, F, a->b, a->b_scales, E, H, po, a->c,
                                               combine_args(cfg, a, ws), status, st));
      case MOE_GG_DGRAD_FC2: {
        if (!dev_ptr_ok(a->aux)) return MOE_ERR_INVALID_ARG;
        const MxOutQ q{static_cast<uint8_t*>(a->q_codes), static_cast<uint8_t*>(a->q_scales),
                       static_cast<uint8_t*>(a->qt_codes), static_cast<uint8_t*>(a->qt_scales)};
        const bool any_q = q.codes != nullptr || q.codes_t != nullptr;
        return cuda_status(gemm_mx_dgrad_fc2(a->a, a->a_scales, rows, H, a->b, a->b_scales, E, F, po, a->dense_rows,
                                             a->aux, a->row_gate, a->c, a->dgate_part, status, st,
                                             any_q ? &q : nullptr));
      }
      case MOE_GG_DGRAD_FC1:
        return cuda_status(gemm_mx_nt_bf16(a->a, a->a_scales, rows, 2 * F, a->b, a->b_scales, E, H, po,
                                           a->dense_rows, a->c, status, st,
                                           a->b_scale_group == 0 ? 128 : a->b_scale_group));
      case MOE_GG_WGRAD_FC1:
        return cuda_status(gemm_mx_wgrad(a->a, a->a_scales, 2 * F, a->b, a->b_scales, H, rows, E, po, a->dense_rows,
                                         static_cast<float*>(a->c), status, st,
                                         a->b_scale_group == 0 ? 128 : a->b_scale_group));
      case MOE_GG_WGRAD_FC2:
        if (a->b_scale_group == kMxScaleGroup224)   // operands swapped: a = h'^T, b = dy^T; c still [E, H, F]
          return cuda_status(gemm_mx_wgrad(a->a, a->a_scales, F, a->b, a->b_scales, H, rows, E, po, a->dense_rows,
                                           static_cast<float*>(a->c), status, st, kMxScaleGroup224, true));
        return cuda_status(gemm_mx_wgrad(a->a, a->a_scales, H, a->b, a->b_scales, F, rows, E, po, a->dense_rows,
                                         static_cast<float*>(a->c), status, st));
      default:
        return MOE_ERR_INVALID_ARG;
    }
  }
  switch (a->op) {
    case MOE_GG_FC1_SWIGLU:
      if (a->c2 != nullptr && !aligned16(a->c2)) return MOE_ERR_INVALID_ARG;
      return cuda_status(gemm_fc1(a->a, rows, H, a->b, E, F, po, a->dense_rows, a->row_gate, a->c, a->c2, status, st));
    case MOE_GG_FC1_SWIGLU_GATHERED:
      if (dense || !dev_ptr_ok(a->a_rows) || (a->c2 != nullptr && !aligned16(a->c2))) return MOE_ERR_INVALID_ARG;
      if (cfg->F % 128 != 0) return MOE_ERR_INVALID_ARG;
      return cuda_status(gemm_fc1_gather(a->a, cfg->T, a->a_rows, rows, H, a->b, E, F, po, a->row_gate, a->c, a->c2,
                                         status, st));
    case MOE_GG_FC2:
      return cuda_status(gemm_fc2(a->a, rows, F, a->b, E, H, po, a->dense_rows, a->c, status, st));
    case MOE_GG_FC2_COMBINE:
      return cuda_status(gemm_fc2_combine(a->a, rows, F, a->b, E, H, po, a->c, combine_args(cfg, a, ws), status, st));
    case MOE_GG_DGRAD_FC2:
      if (!dev_ptr_ok(a->aux)) return MOE_ERR_INVALID_ARG;
      return cuda_status(gemm_dgrad_fc2(a->a, rows, H, a->b, E, F, po, a->dense_rows, a->aux, a->row_gate, a->c,
                                        a->dgate_part, status, st));
    case MOE_GG_DGRAD_FC1:
      return cuda_status(gemm_dgrad_fc1(a->a, rows, F, a->b, E, H, po, a->dense_rows, a->c, status, st));
    case MOE_GG_WGRAD_FC1:
      return cuda_status(gemm_wgrad(a->a, 2 * F, a->b, H, rows, E, po, a->dense_rows, static_cast<float*>(a->c),
                                    status, st));
    case MOE_GG_WGRAD_FC2:
      return cuda_status(gemm_wgrad(a->a, H, a->b, F, rows, E, po, a->dense_rows, static_cast<float*>(a->c),
                                    status, st));
    default:
      return MOE_ERR_INVALID_ARG;
  }
}

moe_status moe_unpermute(const moe_config* cfg, const void* o_perm, const int32_t* slot_row, const void* shared_out,
                         void* y, void* stream) {
  if (!config_ok(cfg)) return MOE_ERR_INVALID_ARG;
  if (cfg->T > 0 && (!dev_ptr_ok(o_perm) || !dev_ptr_ok(slot_row) || !dev_ptr_ok(y))) return MOE_ERR_INVALID_ARG;
  if (shared_out != nullptr && !aligned16(shared_out)) return MOE_ERR_INVALID_ARG;
  if (moe_status s = check_device(); s != MOE_OK) return s;
  return cuda_status(launch_combine(o_perm, slot_row, shared_out, cfg->T, cfg->k, cfg->H, y,
                                    static_cast<cudaStream_t>(stream)));
}

moe_status moe_layer_forward(const moe_config* cfg, const moe_weights* w, const void* x, void* y, void* act,
                             size_t act_bytes, int32_t with_backward, void* ws, size_t ws_bytes, void* stream) {
  moe_act_layout L;
  if (compute_layout(cfg, with_backward, &L) != MOE_OK || w == nullptr) return MOE_ERR_INVALID_ARG;
  if (!dev_ptr_ok(act) || !dev_ptr_ok(ws) || !dev_ptr_ok(w->w_router) || !dev_ptr_ok(w->w1) || !dev_ptr_ok(w->w2))
    return MOE_ERR_INVALID_ARG;
  if (cfg->T > 0 && (!dev_ptr_ok(x) || !dev_ptr_ok(y))) return MOE_ERR_INVALID_ARG;
  if (cfg->S > 0 && (!dev_ptr_ok(w->w1_shared) || !dev_ptr_ok(w->w2_shared))) return MOE_ERR_INVALID_ARG;
  if (w->router_bias != nullptr && !aligned16(w->router_bias)) return MOE_ERR_INVALID_ARG;
  if (cfg->dtype != MOE_GEMM_BF16 && !dev_ptr_ok(w->mx)) return MOE_ERR_INVALID_ARG;
  if (cfg->dtype == MOE_GEMM_NVFP4 && with_backward) return MOE_ERR_UNSUPPORTED;   // NVFP4: forward only
  if (act_bytes < L.total || ws_bytes < moe_workspace_bytes(cfg)) return MOE_ERR_WORKSPACE;
  if (moe_status s = check_device(); s != MOE_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int T = cfg->T, H = cfg->H, E = cfg->E, k = cfg->k, F = cfg->F, S = cfg->S, cap = L.cap;
  int* status = status_ptr(ws);
  float* logits = at<float>(act, L.logits);
  int32_t* idx = at<int32_t>(act, L.topk_idx);
  float* gate = at<float>(act, L.topk_gate);
  int32_t* counts = at<int32_t>(act, L.counts);
  int32_t* poff = at<int32_t>(act, L.poffsets);
  int32_t* slot_row = at<int32_t>(act, L.slot_row);
  float* row_gate = at<float>(act, L.row_gate);
  void* x_perm = at<void>(act, L.x_perm);
  void* h = at<void>(act, L.h);
  void* o = at<void>(act, L.o);

  // 1-2: router GEMM + top-k gating
  MOE_TRY(gemm_router(x, w->w_router, T, H, E, logits, status, st));
  // 2-4: top-k gating fused with the counting-sort histograms, scan, scatter (sync-free)
  const float* rbias = cfg->score == MOE_SCORE_SIGMOID ? w->router_bias : nullptr;
  if (cfg->dtype == MOE_GEMM_BF16) {
    // the maps and the row copy of x: two launches where the histograms are small
    MOE_TRY(launch_topk_permute_gather(logits, rbias, T, E, k, cfg->score, idx, gate, hist_ptr(ws),
                                       status + kMapsDoneWord, counts, at<int32_t>(act, L.offsets), poff, slot_row,
                                       at<int32_t>(act, L.row_src), row_gate, x, H, x_perm, with_backward ? 1 : 0,
                                       status, st));
  } else {
    // (MXFP8 and NVFP4 layers permute the quantised codes instead and read x
    // through row_src where its rows are needed again; x_perm stays unwritten)
    MOE_TRY(launch_topk_permute_maps(logits, rbias, T, E, k, cfg->score, idx, gate, hist_ptr(ws), counts,
                                     at<int32_t>(act, L.offsets), poff, slot_row, at<int32_t>(act, L.row_src),
                                     row_gate, st));
  }
  // 5-6: grouped expert GEMMs; the gate multiplies the SwiGLU output inside fc1
  void* z = with_backward ? at<void>(act, L.z) : nullptr;
  void* zs = with_backward && S > 0 ? at<void>(act, L.zs) : nullptr;
  const void* shared_out = nullptr;
  // 7 fused into fc2's epilogue where its 256-column tiles cover H: each
  // token's y is summed by the tile that completes it (same bits as the
  // separate combine kernel); otherwise a combine kernel after fc2
  const bool fused_combine = kFuseCombine && H % 256 == 0 && T > 0;
  CombineArgs cmb{};
  if (fused_combine) {
    cmb.row_src = at<int32_t>(act, L.row_src);
    cmb.slot_row = slot_row;
    cmb.k = k;
    cmb.count = at<int32_t>(ws, combine_count_offset(cfg));
    cmb.y = y;
  }
  // (the shared expert's output, when there is one, is set below before fc2)
  auto with_shared = [&]() { cmb.shared = shared_out; };
  if (cfg->dtype == MOE_GEMM_NVFP4) {
    // NVFP4 expert GEMMs (forward): x quantised once per token with the tensor
    // scale of all of x, codes permuted into expert order; h quantised with
    // the tensor scale of its valid rows (row_src >= 0); weights prepared once.
    const Nv4Ws M = nv4_ws_layout(cfg);
    const Nv4W W = nv4_weight_layout(cfg);
    char* mb = static_cast<char*>(ws) + mx_ws_base(cfg);
    auto q = [&](const Nv4Buf& b) { return reinterpret_cast<uint8_t*>(mb + b.q); };
    auto f = [&](const Nv4Buf& b) { return reinterpret_cast<uint8_t*>(mb + b.sf); };
    auto wq = [&](const Nv4Buf& b) { return at<const uint8_t>(const_cast<void*>(w->mx), b.q); };
    auto wf = [&](const Nv4Buf& b) { return at<const uint8_t>(const_cast<void*>(w->mx), b.sf); };
    float* amax = reinterpret_cast<float*>(mb + M.amax);
    const float* wamax = at<const float>(const_cast<void*>(w->mx), W.amax);
    MOE_TRY(launch_amax_bf16(x, T, H, nullptr, nullptr, amax + 0, st));
    // straight into expert order; the token-order copy only for the shared expert
    MOE_TRY(launch_quantize_gather_nv4(x, T, H, slot_row, k, amax + 0, q(M.x), f(M.x), S > 0 ? q(M.xs) : nullptr,
                                       S > 0 ? f(M.xs) : nullptr, st));
    // fc1 writes h' and its amax (padding rows have gate 0, so h' = 0 there;
    // rows past the last expert's segment are never computed)
    MOE_TRY(cudaMemsetAsync(amax + 1, 0, sizeof(float), st));
    MOE_TRY(gemm_nv4_fc1(q(M.x), f(M.x), amax + 0, cap, H, wq(W.w1), wf(W.w1), wamax + 0, E, F, poff, 0, row_gate, h,
                         nullptr, amax + 1, status, st));
    MOE_TRY(launch_quantize_rows_nv4(h, cap, F, 0, amax + 1, q(M.h), f(M.h), st));
    MOE_TRY(gemm_nv4_nt_bf16(q(M.h), f(M.h), amax + 1, cap, F, wq(W.w2), wf(W.w2), wamax + 1, E, H, poff, 0, o, status,
                             st));
    if (S > 0 && T > 0) {
      void* hs = at<void>(act, L.hs);
      MOE_TRY(cudaMemsetAsync(amax + 2, 0, sizeof(float), st));
      MOE_TRY(gemm_nv4_fc1(q(M.xs), f(M.xs), amax + 0, T, H, wq(W.s1), wf(W.s1), wamax + 2, 1, S, nullptr, T, nullptr,
                           hs, nullptr, amax + 2, status, st));
      MOE_TRY(launch_quantize_rows_nv4(hs, T, S, 0, amax + 2, q(M.hs), f(M.hs), st));
      MOE_TRY(gemm_nv4_nt_bf16(q(M.hs), f(M.hs), amax + 2, T, S, wq(W.s2), wf(W.s2), wamax + 3, 1, H, nullptr, T,
                               at<void>(act, L.os), status, st));
      shared_out = at<void>(act, L.os);
    }
  } else if (cfg->dtype == MOE_GEMM_MXFP8) {
    // MXFP8 expert GEMMs: activations quantised (blocks of 32 along K) on the
    // way in, weights prepared once; router, gates and combine stay fp32/bf16.
    const MxWs M = mx_ws_layout(cfg);
    const MxW W = mx_weight_layout(cfg);
    char* mb = static_cast<char*>(ws) + mx_ws_base(cfg);
    auto q = [&](const MxBuf& b) { return reinterpret_cast<uint8_t*>(mb + b.q); };
    auto f = [&](const MxBuf& b) { return reinterpret_cast<uint8_t*>(mb + b.sf); };
    auto wq = [&](const MxBuf& b) { return at<const uint8_t>(const_cast<void*>(w->mx), b.q); };
    auto wf = [&](const MxBuf& b) { return at<const uint8_t>(const_cast<void*>(w->mx), b.sf); };
    // x is quantised once per token and the codes are permuted like x itself
    // (blocks lie along H, so quantising before or after the gather is the same)
    MOE_TRY(launch_quantize_rows(x, T, H, 0, q(M.xs), f(M.xs), st));
    MOE_TRY(launch_gather_rows_mx(q(M.xs), f(M.xs), slot_row, T, k, H, q(M.x), f(M.x), st, counts, poff,
                                  with_backward ? E : 0));
    // the shared expert first: with the combine fused into fc2 its rows must exist
    if (S > 0 && T > 0) {
      MOE_TRY(gemm_mx_fc1(q(M.xs), f(M.xs), T, H, wq(W.s1), wf(W.s1), 1, S, nullptr, T, nullptr, at<void>(act, L.hs),
                          zs, status, st));
      MOE_TRY(launch_quantize_rows(at<void>(act, L.hs), T, S, 0, q(M.hs), f(M.hs), st));
      MOE_TRY(gemm_mx_nt_bf16(q(M.hs), f(M.hs), T, S, wq(W.s2), wf(W.s2), 1, H, nullptr, T, at<void>(act, L.os),
                              status, st));
      shared_out = at<void>(act, L.os);
    }
    // h' only in MXFP8, from fc1's epilogue: the row copy for fc2 (workspace) and,
    // for training, the transposed copy for the fc2 weight gradient (act)
    const MxOutQ hq{q(M.h), f(M.h), with_backward ? at<uint8_t>(act, L.h_qt) : nullptr,
                    with_backward ? at<uint8_t>(act, L.h_qt_sf) : nullptr};
    MOE_TRY(gemm_mx_fc1(q(M.x), f(M.x), cap, H, wq(W.w1), wf(W.w1), E, F, poff, 0, row_gate, nullptr, z, status, st,
                        &hq));
    with_shared();
    if (fused_combine) {
      MOE_TRY(gemm_mx_fc2_combine(q(M.h), f(M.h), cap, F, wq(W.w2), wf(W.w2), E, H, poff, o, cmb, status, st));
      return MOE_OK;
    }
    MOE_TRY(gemm_mx_nt_bf16(q(M.h), f(M.h), cap, F, wq(W.w2), wf(W.w2), E, H, poff, 0, o, status, st,
                            mx_b224(cfg) ? kMxScaleGroup224 : 128));
  } else {
    if (S > 0 && T > 0) {
      MOE_TRY(gemm_fc1(x, T, H, w->w1_shared, 1, S, nullptr, T, nullptr, at<void>(act, L.hs), zs, status, st));
      MOE_TRY(gemm_fc2(at<void>(act, L.hs), T, S, w->w2_shared, 1, H, nullptr, T, at<void>(act, L.os), status, st));
      shared_out = at<void>(act, L.os);
    }
    MOE_TRY(gemm_fc1(x_perm, cap, H, w->w1, E, F, poff, 0, row_gate, h, z, status, st));
    with_shared();
    if (fused_combine) {
      MOE_TRY(gemm_fc2_combine(h, cap, F, w->w2, E, H, poff, o, cmb, status, st));
      return MOE_OK;
    }
    MOE_TRY(gemm_fc2(h, cap, F, w->w2, E, H, poff, 0, o, status, st));
  }
  // 7: unweighted combine
  MOE_TRY(launch_combine(o, slot_row, shared_out, T, k, H, y, st));
  return MOE_OK;
}

moe_status moe_layer_backward_dgrad(const moe_config* cfg, const moe_weights* w, const void* x, const void* dy,
                                    void* dx, float* dgate, void* act, size_t act_bytes, void* ws, size_t ws_bytes,
                                    void* stream) {
  moe_act_layout L;
  if (compute_layout(cfg, 1, &L) != MOE_OK || w == nullptr) return MOE_ERR_INVALID_ARG;
  if (!dev_ptr_ok(act) || !dev_ptr_ok(ws) || !dev_ptr_ok(w->w_router) || !dev_ptr_ok(w->w1) || !dev_ptr_ok(w->w2))
    return MOE_ERR_INVALID_ARG;
  if (cfg->T > 0 && (!dev_ptr_ok(x) || !dev_ptr_ok(dy) || !dev_ptr_ok(dx))) return MOE_ERR_INVALID_ARG;
  if (cfg->S > 0 && (!dev_ptr_ok(w->w1_shared) || !dev_ptr_ok(w->w2_shared))) return MOE_ERR_INVALID_ARG;
  if (dgate != nullptr && !aligned16(dgate)) return MOE_ERR_INVALID_ARG;
  if (cfg->dtype == MOE_GEMM_NVFP4) return MOE_ERR_UNSUPPORTED;   // NVFP4: forward only
  if (cfg->dtype == MOE_GEMM_MXFP8 && !dev_ptr_ok(w->mx)) return MOE_ERR_INVALID_ARG;
  if (act_bytes < L.total || ws_bytes < moe_workspace_bytes(cfg)) return MOE_ERR_WORKSPACE;
  if (moe_status s = check_device(); s != MOE_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int T = cfg->T, H = cfg->H, E = cfg->E, k = cfg->k, F = cfg->F, S = cfg->S, cap = L.cap;
  int* status = status_ptr(ws);
  const int32_t* counts = at<int32_t>(act, L.counts);
  const int32_t* poff = at<int32_t>(act, L.poffsets);
  const int32_t* slot_row = at<int32_t>(act, L.slot_row);
  void* dy_perm = at<void>(act, L.dy_perm);
  void* dz = at<void>(act, L.dz);
  void* dx_perm = at<void>(act, L.dx_perm);
  float* dpart = at<float>(act, L.dgate_part);

  if (cfg->dtype == MOE_GEMM_BF16) {
    MOE_TRY(launch_gather_rows_zero(dy, slot_row, T, k, E, counts, H, dy_perm, st));
  }
  const void* dxs = nullptr;
  if (cfg->dtype == MOE_GEMM_MXFP8) {
    const MxWs M = mx_ws_layout(cfg);
    const MxW W = mx_weight_layout(cfg);
    char* mb = static_cast<char*>(ws) + mx_ws_base(cfg);
    auto q = [&](const MxBuf& b) { return reinterpret_cast<uint8_t*>(mb + b.q); };
    auto f = [&](const MxBuf& b) { return reinterpret_cast<uint8_t*>(mb + b.sf); };
    auto wq = [&](const MxBuf& b) { return at<const uint8_t>(const_cast<void*>(w->mx), b.q); };
    auto wf = [&](const MxBuf& b) { return at<const uint8_t>(const_cast<void*>(w->mx), b.sf); };
    MOE_TRY(launch_quantize_rows(dy, T, H, 0, q(M.dys), f(M.dys), st));
    MOE_TRY(launch_gather_rows_mx(q(M.dys), f(M.dys), slot_row, T, k, H, q(M.dy), f(M.dy), st, counts, poff, E));
    // dz's MXFP8 copies for the fc1 data gradient (rows, workspace) and the fc1
    // weight gradient (transposed, act): from the epilogue where it can, else
    // quantised from the bf16 dz
    uint8_t* dz_qt = at<uint8_t>(act, L.dz_qt);
    uint8_t* dz_qt_sf = at<uint8_t>(act, L.dz_qt_sf);
    const MxOutQ dzq{q(M.dz), f(M.dz), dz_qt, dz_qt_sf};
    const bool fused_q = gemm_mx_dgrad_fc2_quantises(F);
    MOE_TRY(gemm_mx_dgrad_fc2(q(M.dy), f(M.dy), cap, H, wq(W.w2t), wf(W.w2t), E, F, poff, 0, at<void>(act, L.z),
                              at<float>(act, L.row_gate), fused_q ? nullptr : dz, dpart, status, st,
                              fused_q ? &dzq : nullptr));
    if (!fused_q) {
      MOE_TRY(launch_quantize_rows(dz, cap, 2 * F, 0, q(M.dz), f(M.dz), st, 128, poff + E));
      MOE_TRY(launch_quantize_cols(dz, 1, cap, 2 * F, dz_qt, dz_qt_sf, st, 128, poff + E));
    }
    MOE_TRY(gemm_mx_nt_bf16(q(M.dz), f(M.dz), cap, 2 * F, wq(W.w1t), wf(W.w1t), E, H, poff, 0, dx_perm, status, st,
                            mx_b224(cfg) ? kMxScaleGroup224 : 128));
    if (S > 0 && T > 0) {
      MOE_TRY(gemm_mx_dgrad_fc2(q(M.dys), f(M.dys), T, H, wq(W.s2t), wf(W.s2t), 1, S, nullptr, T, at<void>(act, L.zs),
                                nullptr, at<void>(act, L.dzs), nullptr, status, st));
      MOE_TRY(launch_quantize_rows(at<void>(act, L.dzs), T, 2 * S, 0, q(M.dzs), f(M.dzs), st));
      MOE_TRY(gemm_mx_nt_bf16(q(M.dzs), f(M.dzs), T, 2 * S, wq(W.s1t), wf(W.s1t), 1, H, nullptr, T,
                              at<void>(act, L.dxs), status, st));
      dxs = at<void>(act, L.dxs);
    }
  } else {
    MOE_TRY(gemm_dgrad_fc2(dy_perm, cap, H, w->w2, E, F, poff, 0, at<void>(act, L.z), at<float>(act, L.row_gate), dz,
                           dpart, status, st));
    MOE_TRY(gemm_dgrad_fc1(dz, cap, F, w->w1, E, H, poff, 0, dx_perm, status, st));
    if (S > 0 && T > 0) {
      MOE_TRY(gemm_dgrad_fc2(dy, T, H, w->w2_shared, 1, S, nullptr, T, at<void>(act, L.zs), nullptr,
                             at<void>(act, L.dzs), nullptr, status, st));
      MOE_TRY(gemm_dgrad_fc1(at<void>(act, L.dzs), T, S, w->w1_shared, 1, H, nullptr, T, at<void>(act, L.dxs), status,
                             st));
      dxs = at<void>(act, L.dxs);
    }
  }
  MOE_TRY(launch_dgrad_combine(dx_perm, slot_row, at<int32_t>(act, L.topk_idx), at<float>(act, L.topk_gate),
                               at<float>(act, L.logits), dpart, F / 128, w->w_router, dxs, T, E, k, H, cfg->score, dx,
                               dgate, at<float>(act, L.dlogits), at<float>(act, L.row_dlogit), st));
  return MOE_OK;
}

moe_status moe_layer_backward_wgrad(const moe_config* cfg, const moe_weights* w, const void* x, const void* dy,
                                    const moe_grads* g, void* act, size_t act_bytes, void* ws, size_t ws_bytes,
                                    void* stream) {
  moe_act_layout L;
  if (compute_layout(cfg, 1, &L) != MOE_OK || w == nullptr || g == nullptr) return MOE_ERR_INVALID_ARG;
  if (!dev_ptr_ok(act) || !dev_ptr_ok(ws) || !dev_ptr_ok(g->dw_router) || !dev_ptr_ok(g->dw1) ||
      !dev_ptr_ok(g->dw2))
    return MOE_ERR_INVALID_ARG;
  if (cfg->T > 0 && (!dev_ptr_ok(x) || !dev_ptr_ok(dy))) return MOE_ERR_INVALID_ARG;
  if (cfg->S > 0 && (!dev_ptr_ok(g->dw1_shared) || !dev_ptr_ok(g->dw2_shared))) return MOE_ERR_INVALID_ARG;
  if (cfg->dtype == MOE_GEMM_NVFP4) return MOE_ERR_UNSUPPORTED;   // NVFP4: forward only
  if (cfg->dtype == MOE_GEMM_MXFP8 && !dev_ptr_ok(w->mx)) return MOE_ERR_INVALID_ARG;
  if (act_bytes < L.total || ws_bytes < moe_workspace_bytes(cfg)) return MOE_ERR_WORKSPACE;
  if (moe_status s = check_device(); s != MOE_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int T = cfg->T, H = cfg->H, E = cfg->E, F = cfg->F, S = cfg->S, cap = L.cap;
  int* status = status_ptr(ws);
  const int32_t* counts = at<int32_t>(act, L.counts);
  const int32_t* poff = at<int32_t>(act, L.poffsets);
  if (cfg->dtype == MOE_GEMM_MXFP8) {
    // contraction over tokens: transposed copies quantised along the tokens
    const MxWs M = mx_ws_layout(cfg);
    char* mb = static_cast<char*>(ws) + mx_ws_base(cfg);
    auto q = [&](const MxBuf& b) { return reinterpret_cast<uint8_t*>(mb + b.q); };
    auto f = [&](const MxBuf& b) { return reinterpret_cast<uint8_t*>(mb + b.sf); };
    // x and dy in expert order are read straight from token order through row_src
    const int32_t* row_src = at<int32_t>(act, L.row_src);
    // (rows past the last expert's padded end are skipped: no GEMM reads them)
    MOE_TRY(launch_quantize_cols_gather(x, T, row_src, cap, H, q(M.xT), f(M.xT), st, mx_xt_group(cfg), poff + E));
    // dz^T: left in act by the data gradient
    MOE_TRY(gemm_mx_wgrad(at<uint8_t>(act, L.dz_qt), at<uint8_t>(act, L.dz_qt_sf), 2 * F, q(M.xT), f(M.xT), H, cap, E,
                          poff, 0, g->dw1, status, st,
                          mx_xt_group(cfg)));
    // h'^T: left in act by fc1
    if (mx_dw2_trans(cfg)) {
      MOE_TRY(launch_quantize_cols_gather(dy, T, row_src, cap, H, q(M.dyT), f(M.dyT), st, kMxScaleGroup224,
                                          poff + E));
      MOE_TRY(gemm_mx_wgrad(at<uint8_t>(act, L.h_qt), at<uint8_t>(act, L.h_qt_sf), F, q(M.dyT), f(M.dyT), H, cap, E,
                            poff, 0, g->dw2, status, st, kMxScaleGroup224, true));
    } else {
      MOE_TRY(launch_quantize_cols_gather(dy, T, row_src, cap, H, q(M.dyT), f(M.dyT), st, 128, poff + E));
      MOE_TRY(gemm_mx_wgrad(q(M.dyT), f(M.dyT), H, at<uint8_t>(act, L.h_qt), at<uint8_t>(act, L.h_qt_sf), F, cap, E,
                            poff, 0, g->dw2, status, st));
    }
    if (S > 0 && T > 0) {
      MOE_TRY(launch_quantize_cols(at<void>(act, L.dzs), 1, T, 2 * S, q(M.dzsT), f(M.dzsT), st));
      MOE_TRY(launch_quantize_cols(x, 1, T, H, q(M.xsT), f(M.xsT), st));
      MOE_TRY(gemm_mx_wgrad(q(M.dzsT), f(M.dzsT), 2 * S, q(M.xsT), f(M.xsT), H, T, 1, nullptr, T, g->dw1_shared,
                            status, st));
      MOE_TRY(launch_quantize_cols(dy, 1, T, H, q(M.dysT), f(M.dysT), st));
      MOE_TRY(launch_quantize_cols(at<void>(act, L.hs), 1, T, S, q(M.hsT), f(M.hsT), st));
      MOE_TRY(gemm_mx_wgrad(q(M.dysT), f(M.dysT), H, q(M.hsT), f(M.hsT), S, T, 1, nullptr, T, g->dw2_shared, status,
                            st));
    }
  } else {
    MOE_TRY(gemm_wgrad(at<void>(act, L.dz), 2 * F, at<void>(act, L.x_perm), H, cap, E, poff, 0, g->dw1, status, st));
    MOE_TRY(gemm_wgrad(at<void>(act, L.dy_perm), H, at<void>(act, L.h), F, cap, E, poff, 0, g->dw2, status, st));
    if (S > 0 && T > 0) {
      MOE_TRY(gemm_wgrad(at<void>(act, L.dzs), 2 * S, x, H, T, 1, nullptr, T, g->dw1_shared, status, st));
      MOE_TRY(gemm_wgrad(dy, H, at<void>(act, L.hs), S, T, 1, nullptr, T, g->dw2_shared, status, st));
    }
  }
  if (cfg->dtype == MOE_GEMM_MXFP8)
    MOE_TRY(launch_router_wgrad(x, at<int32_t>(act, L.row_src), at<float>(act, L.row_dlogit), counts, poff, E, H,
                                g->dw_router, st));
  else
    MOE_TRY(launch_router_wgrad(at<void>(act, L.x_perm), nullptr, at<float>(act, L.row_dlogit), counts, poff, E, H,
                                g->dw_router, st));
  if (S > 0 && T == 0) {
    MOE_TRY(cudaMemsetAsync(g->dw1_shared, 0, sizeof(float) * 2 * S * H, st));
    MOE_TRY(cudaMemsetAsync(g->dw2_shared, 0, sizeof(float) * S * H, st));
  }
  return MOE_OK;
}

}  // extern "C"
