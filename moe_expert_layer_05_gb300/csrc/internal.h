// Launchers shared between the translation units of the library (not part of
// the public ABI).  All pointers are device pointers; all calls are
// stream-ordered and never synchronise.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

namespace moe {

constexpr int kPadRows = 128;      // expert segments start at multiples of this
constexpr int kPairsPerBlock = 256;  // (token, slot) pairs per counting-sort block
constexpr int kMaxE = 256;
constexpr int kMaxK = 32;
// Int of the workspace's 256-byte status region that counts the finished
// blocks of the permutation's histogram launch (zero between launches).
constexpr int kMapsDoneWord = 40;

int num_sms();
bool device_is_gb300();

// Launch of one of the library's kernels (each begins with pdl_entry()) with
// programmatic stream serialization, so that its launch overlaps the tail of
// the kernel before it in the stream.  Errors are also left for
// cudaGetLastError, as with <<<>>>.
template <class... KArgs, class... Args>
cudaError_t launch_k(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, Args&&... args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}
// Limit of one pipeline wait inside the grouped GEMMs (0: the kernels' 2 s
// default); set through moe_debug_set_wait_limit_ns.
unsigned long long gemm_wait_limit_ns();
// Counts kernel launches issued by the library (process-wide).
void count_launches(int n);

// ------------------------------------------------------------ routing (route.cu)
cudaError_t launch_topk(const float* logits, const float* bias, int T, int E, int k, int score, int32_t* idx,
                        float* gate, cudaStream_t st);
// Counting sort of T*k pairs by expert, in chunks of (256/k)*k pairs.  hist
// is scratch of ceil(T / (256/k)) * E ints.
cudaError_t launch_permute_maps(const int32_t* idx, const float* gate, int T, int E, int k, int32_t* hist,
                                int32_t* counts, int32_t* offsets, int32_t* poffsets, int32_t* slot_row,
                                int32_t* row_src, float* row_gate, int* status, cudaStream_t st);
// Top-k gating of the logits fused with the chunk histograms, then the same
// scan and scatter as launch_permute_maps.
cudaError_t launch_topk_permute_maps(const float* logits, const float* bias, int T, int E, int k, int score,
                                     int32_t* idx, float* gate, int32_t* hist, int32_t* counts, int32_t* offsets,
                                     int32_t* poffsets, int32_t* slot_row, int32_t* row_src, float* row_gate,
                                     cudaStream_t st);
// The same maps plus the row copy of x into x_perm (and, with zero_pad, zeros
// in the segments' padding rows), in two launches where NB * E is small
// (histograms, ranks and the scan in the first; the maps and the copy in the
// second), three otherwise.  done: a workspace int, zero between launches.
cudaError_t launch_permute_gather(const int32_t* idx, const float* gate, int T, int E, int k, int32_t* hist,
                                  int* done, int32_t* counts, int32_t* offsets, int32_t* poffsets, int32_t* slot_row,
                                  int32_t* row_src, float* row_gate, const void* x, int H, void* x_perm, int zero_pad,
                                  int* status, cudaStream_t st);
// Top-k gating fused into the first launch of launch_permute_gather.
cudaError_t launch_topk_permute_gather(const float* logits, const float* bias, int T, int E, int k, int score,
                                       int32_t* idx, float* gate, int32_t* hist, int* done, int32_t* counts,
                                       int32_t* offsets, int32_t* poffsets, int32_t* slot_row, int32_t* row_src,
                                       float* row_gate, const void* x, int H, void* x_perm, int zero_pad,
                                       int* status, cudaStream_t st);
cudaError_t launch_gather_rows(const void* x, const int32_t* slot_row, int T, int k, int H, void* x_perm,
                               cudaStream_t st);
// The row copy of an input whose maps exist (dy), zeroing the segments'
// padding rows in the same launch.
cudaError_t launch_gather_rows_zero(const void* x, const int32_t* slot_row, int T, int k, int E,
                                   const int32_t* counts, int H, void* x_perm, cudaStream_t st);
cudaError_t launch_zero_pad_rows(const int32_t* counts, const int32_t* poffsets, int E, int H, void* buf,
                                 cudaStream_t st);
cudaError_t launch_combine(const void* o_perm, const int32_t* slot_row, const void* shared, int T, int k, int H,
                           void* y, cudaStream_t st);
// Backward per token: dgate from partial sums, router backward (dlogits and
// per-row dlogit), dx = sum of expert rows + router term + shared term.
cudaError_t launch_dgrad_combine(const void* dx_perm, const int32_t* slot_row, const int32_t* topk_idx,
                                 const float* topk_gate, const float* logits, const float* dgate_part,
                                 int n_part, const void* w_router, const void* dx_shared, int T, int E, int k,
                                 int H, int score, void* dx, float* dgate, float* dlogits, float* row_dlogit,
                                 cudaStream_t st);
// dWr[e] = sum over expert e's rows of row_dlogit[r] * x_perm[r]  (fp32);
// with row_src given, x_perm is x in token order, read through row_src.
cudaError_t launch_router_wgrad(const void* x_perm, const int32_t* row_src, const float* row_dlogit,
                                const int32_t* counts, const int32_t* poffsets, int E, int H, float* dw_router,
                                cudaStream_t st);

// ------------------------------------------------------------ GEMMs (gemm_*.cu)
// logits[T,E] (fp32) = x[T,H] * Wr[E,H]^T
cudaError_t gemm_router(const void* x, const void* wr, int T, int H, int E, float* logits, int* status,
                        cudaStream_t st);
// h[cap,F] = g * silu(z_gate) * z_up with z = A[cap,H] * W1_e[2F,H]^T; z saved if non-null.
// poffsets == nullptr: dense, rows = dense_rows, one group.
cudaError_t gemm_fc1(const void* a, int rows_alloc, int H, const void* w1, int E, int F, const int32_t* poffsets,
                     int dense_rows, const float* row_gate, void* h, void* z, int* status, cudaStream_t st);
// fc1 with the permutation fused into its A load: row r of A is x[row_src[r]]
// (zeros where row_src[r] < 0); x [T,H] in token order.
cudaError_t gemm_fc1_gather(const void* x, int T, const int32_t* row_src, int rows_alloc, int H, const void* w1,
                            int E, int F, const int32_t* poffsets, const float* row_gate, void* h, void* z, int* status,
                            cudaStream_t st);
// o[cap,H] = A[cap,F] * W2_e[H,F]^T
cudaError_t gemm_fc2(const void* a, int rows_alloc, int F, const void* w2, int E, int H, const int32_t* poffsets,
                     int dense_rows, void* o, int* status, cudaStream_t st);
// The combine fused into fc2's epilogue: besides o, y[t] = sum_i o[slot_row[t,i]]
// (+ shared[t]) in slot order, fp32, one rounding -- the bits of launch_combine.
// count: [T, H/256] ints, zero before the launch and after it.  H % 256 == 0.
struct CombineArgs {
  const int32_t* row_src;
  const int32_t* slot_row;
  int k;
  int* count;
  const void* shared;   // nullable
  void* y;
};
cudaError_t gemm_fc2_combine(const void* a, int rows_alloc, int F, const void* w2, int E, int H,
                             const int32_t* poffsets, void* o, const CombineArgs& cmb, int* status, cudaStream_t st);
// dz[cap,2F] from dh = A[cap,H] * W2_e ([H,F]) with SwiGLU backward epilogue.
cudaError_t gemm_dgrad_fc2(const void* dy_perm, int rows_alloc, int H, const void* w2, int E, int F,
                           const int32_t* poffsets, int dense_rows, const void* z, const float* row_gate,
                           void* dz, float* dgate_part, int* status, cudaStream_t st);
// dx_perm[cap,H] = dz[cap,2F] * W1_e ([2F,H])
cudaError_t gemm_dgrad_fc1(const void* dz, int rows_alloc, int F, const void* w1, int E, int H,
                           const int32_t* poffsets, int dense_rows, void* dx_perm, int* status, cudaStream_t st);
// dW[e] (fp32 [M,N]) = A_e^T B_e, A [rows, M] bf16, B [rows, N] bf16 over each expert's rows
// (poffsets) or over dense_rows rows (poffsets == nullptr, one group).
cudaError_t gemm_wgrad(const void* a, int M, const void* b, int N, int rows_alloc, int E, const int32_t* poffsets,
                       int dense_rows, float* dw, int* status, cudaStream_t st);

// ------------------------------------------------------------ MXFP8 (mxfp8.cu, gemm_mx.cu)
// row_limit (device, nullable; the quantisers below take it too): rows from
// *row_limit on are skipped -- the capacity rows past the last expert, which
// no GEMM reads.
// Row mode: blocks of 32 along each row; gate_up_half > 0 also interleaves
// the rows of every [gate; up] group of 2*half rows in 128-row blocks.
// group: scale tiles per 128 rows (128), or per group of 224 rows (two tiles
// a group, the second one's last 32 rows unused; rows % 224 == 0): the B
// operand layout of the 224-wide GEMM tiles (kMxScaleGroup224).
cudaError_t launch_quantize_rows(const void* src, long long rows, int cols, int gate_up_half, uint8_t* codes,
                                 uint8_t* sf, cudaStream_t st, int group = 128, const int32_t* row_limit = nullptr);
// Row-quantised token rows -> expert order (codes and scale tiles), and the
// zero codes / scales of the padding rows.
// E_pad > 0: the same launch zeroes the padding rows (codes and scales) of
// experts 0 .. E_pad-1 (counts, poffsets [E+1]).
cudaError_t launch_gather_rows_mx(const uint8_t* codes_tok, const uint8_t* sf_tok, const int32_t* slot_row, int T,
                                  int k, int H, uint8_t* codes_perm, uint8_t* sf_perm, cudaStream_t st,
                                  const int32_t* counts = nullptr, const int32_t* poffsets = nullptr, int E_pad = 0);
// Column mode: batch x [rows, cols] -> batch x [cols, rows], blocks along rows
// (group: as for the row mode, over the output rows; cols % 224 == 0 for 224).
cudaError_t launch_quantize_cols(const void* src, int batch, int rows, int cols, uint8_t* codes, uint8_t* sf,
                                 cudaStream_t st, int group = 128, const int32_t* row_limit = nullptr);
// Scale bytes of a [rows, cols] codes matrix (blocks along cols) with its
// rows' scale tiles in groups of `group` rows.
inline size_t mx_scale_bytes(size_t rows, size_t cols, int group) {
  return group == 128 ? rows * cols / 32 : (rows / group) * 2 * (cols / 128) * 512;
}
constexpr int kMxScaleGroup224 = 224;
// Column mode on rows gathered through row_map: row r of the [rows, cols]
// input is src row row_map[r] (a zero row where it is outside [0, src_rows)).
cudaError_t launch_quantize_cols_gather(const void* src, int src_rows, const int32_t* row_map, int rows, int cols,
                                        uint8_t* codes, uint8_t* sf, cudaStream_t st, int group = 128,
                                        const int32_t* row_limit = nullptr);
// MXFP8 copies of a GEMM output written by its epilogue: codes / sf = rows
// quantised along the row, codes_t / sf_t = quantised along the rows and
// transposed (nullptr: that copy is not written).
struct MxOutQ {
  uint8_t* codes;
  uint8_t* sf;
  uint8_t* codes_t;
  uint8_t* sf_t;
};
// q (nullable; routed only): h''s MXFP8 copies ([cap, F] and [F, cap]) from
// the epilogue; h (bf16) may then be nullptr if q->codes is given.
cudaError_t gemm_mx_fc1(const void* aq, const void* asf, int rows_alloc, int H, const void* w1q, const void* w1sf,
                        int E, int F, const int32_t* poffsets, int dense_rows, const float* row_gate, void* h,
                        void* z, int* status, cudaStream_t st, const MxOutQ* q = nullptr);
// b_group: the row grouping of B's scale tiles (128, or 224: 256 x 224 tiles,
// routed calls with N % 224 == 0).
cudaError_t gemm_mx_nt_bf16(const void* aq, const void* asf, int rows_alloc, int K, const void* bq, const void* bsf,
                            int E, int N, const int32_t* poffsets, int dense_rows, void* c, int* status,
                            cudaStream_t st, int b_group = 128);
// MXFP8 fc2 (N = H, H % 256 == 0) with the combine fused into its epilogue.
cudaError_t gemm_mx_fc2_combine(const void* aq, const void* asf, int rows_alloc, int F, const void* bq,
                                const void* bsf, int E, int H, const int32_t* poffsets, void* o,
                                const CombineArgs& cmb, int* status, cudaStream_t st);
// q (nullable): dz's MXFP8 copies ([cap, 2F] and [2F, cap]) from the epilogue;
// only where gemm_mx_dgrad_fc2_quantises(F).  dz (bf16) may then be nullptr.
bool gemm_mx_dgrad_fc2_quantises(int F);
cudaError_t gemm_mx_dgrad_fc2(const void* dyq, const void* dysf, int rows_alloc, int H, const void* w2tq,
                              const void* w2tsf, int E, int F, const int32_t* poffsets, int dense_rows, const void* z,
                              const float* row_gate, void* dz, float* dgate_part, int* status, cudaStream_t st,
                              const MxOutQ* q = nullptr);
// b_group 224: B's scale tiles grouped by 224 rows (256 x 224 tiles; N % 224 == 0, M % 256 == 0).
// c_trans (b_group 224 only): dw is [E, N, M], the tiles stored transposed.
cudaError_t gemm_mx_wgrad(const void* atq, const void* atsf, int M, const void* btq, const void* btsf, int N,
                          int rows_alloc, int E, const int32_t* poffsets, int dense_rows, float* dw, int* status,
                          cudaStream_t st, int b_group = 128, bool c_trans = false);

// ------------------------------------------------------------ NVFP4 (nvfp4.cu, gemm_mx.cu)
// *amax = max |v| over a bf16 [rows, cols] tensor (rows with row_src < 0 skipped
// when row_src is given, rows from *rows_end on when rows_end is given); zeroes
// *amax first.
cudaError_t launch_amax_bf16(const void* src, long long rows, int cols, const int32_t* row_src,
                             const int32_t* rows_end, float* amax, cudaStream_t st);
// Blocks of 16 along each row with the tensor scale of *amax; codes [rows, cols/2].
cudaError_t launch_quantize_rows_nv4(const void* src, long long rows, int cols, int gate_up_half,
                                     const float* amax, uint8_t* codes, uint8_t* sf, cudaStream_t st);
// x [T,H] quantised straight into its k expert-ordered rows (and into token
// order as well when codes_tok is given).
cudaError_t launch_quantize_gather_nv4(const void* x, int T, int H, const int32_t* slot_row, int k,
                                      const float* amax, uint8_t* codes_perm, uint8_t* sf_perm, uint8_t* codes_tok,
                                      uint8_t* sf_tok, cudaStream_t st);
// NVFP4 GEMMs: A [rows, K] and B_e [N, K] E2M1 codes with scale tiles; amax_a,
// amax_b their tensor amaxes (device).  amax_h (nullable, zeroed by the caller):
// receives max |h'| over the rows fc1 computes.
cudaError_t gemm_nv4_fc1(const void* aq, const void* asf, const float* amax_a, int rows_alloc, int H,
                         const void* w1q, const void* w1sf, const float* amax_w, int E, int F,
                         const int32_t* poffsets, int dense_rows, const float* row_gate, void* h, void* z,
                         float* amax_h, int* status, cudaStream_t st);
cudaError_t gemm_nv4_nt_bf16(const void* aq, const void* asf, const float* amax_a, int rows_alloc, int K,
                             const void* bq, const void* bsf, const float* amax_b, int E, int N,
                             const int32_t* poffsets, int dense_rows, void* c, int* status, cudaStream_t st);

}  // namespace moe
