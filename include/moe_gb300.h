/*
 * moe_gb300.h — C ABI of the single-GPU Mixture-of-Experts expert layer for
 * NVIDIA GB300 (sm_103a).
 *
 * The layer is the one the summary of "Scalable Training of Mixture-of-Experts
 * Models with Megatron Core" describes:
 *   - each token is sent to a few of many experts, the rest stay idle
 *     (Problem, section 1);
 *   - the router stays in high precision (technical summary 2.5, selective
 *     precision);
 *   - routing and permutation create dynamic shapes that must not cost host
 *     synchronisation or many launches (technical summary 1, compute
 *     efficiency wall); the GPU reads the shape information itself
 *     (technical summary 2.4, sync-free kernels);
 *   - all experts run in one grouped GEMM (technical summary 2.4);
 *   - the routing weight is applied before the activation computation so that
 *     backward needs no extra saved tensor (technical summary 2.2,
 *     memory-efficient permutation).
 * The pages give no API; the calls below follow that problem statement.
 *
 * Conventions for every call:
 *   - All tensor arguments are DEVICE pointers owned by the caller, row-major,
 *     16-byte aligned.  The library allocates nothing in these calls.
 *   - bf16 = IEEE bfloat16 (uint16 storage); fp32 = IEEE float.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  No call
 *     synchronises the host or copies device data to the host, except
 *     moe_read_device_status.
 *   - Host-detectable errors return before any launch.  A launch failure
 *     returns MOE_ERR_CUDA.  Errors found on the device (an expert index out
 *     of range, a pipeline wait that timed out) are recorded in the status
 *     word of the workspace; read it with moe_read_device_status.
 *   - Only compute capability 10.3 (GB300) is supported; elsewhere every
 *     compute call returns MOE_ERR_UNSUPPORTED.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = -1,  /* bad size, null pointer, misaligned pointer */
  MOE_ERR_UNSUPPORTED = -2,  /* not a GB300, or a shape outside the limits below */
  MOE_ERR_CUDA = -3,         /* a CUDA runtime / driver call failed */
  MOE_ERR_WORKSPACE = -4,    /* workspace or activation buffer too small */
  MOE_ERR_BAD_INDEX = -5,    /* device: an expert index was outside [0, E) */
  MOE_ERR_TIMEOUT = -6       /* device: a pipeline wait exceeded its limit */
} moe_status;

typedef enum { MOE_SCORE_SOFTMAX = 0, MOE_SCORE_SIGMOID = 1 } moe_score_fn;
typedef enum { MOE_GEMM_BF16 = 0, MOE_GEMM_MXFP8 = 1, MOE_GEMM_NVFP4 = 2 } moe_gemm_dtype;

/* Layer shape.
 *   T tokens, H hidden, E routed experts, k experts per token, F routed expert
 *   SwiGLU width, S shared expert SwiGLU width (0 = no shared expert).
 * Limits: 1 <= k <= 32, k <= E <= 256; H and F multiples of 128; S = 0 or a multiple
 * of 128; 0 <= T and T*k < 2^31 - 128*E.
 * score: softmax scoring selects on the raw logit and normalises exp(logit)
 *   over the chosen k; sigmoid scoring selects on sigmoid(logit) + bias[e]
 *   and normalises sigmoid(logit) over the chosen k.  Equal keys go to the
 *   lower expert id.
 */
typedef struct {
  int32_t T, H, E, k, F, S;
  int32_t score;   /* moe_score_fn */
  int32_t dtype;   /* moe_gemm_dtype; MXFP8 and NVFP4 also need T % 128 == 0, NVFP4
                      H, F, S multiples of 256 (NVFP4 layers run forward only) */
} moe_config;

/* Weights (device, bf16 unless noted).
 *   w_router [E,H]; router_bias [E] fp32 or NULL (selection only);
 *   w1 [E,2F,H]: rows 0..F-1 are the gate projection, rows F..2F-1 the up
 *   projection; w2 [E,H,F]; w1_shared [2S,H], w2_shared [H,S] (NULL if S=0). */
typedef struct {
  const void* w_router;
  const float* router_bias;
  const void* w1;
  const void* w2;
  const void* w1_shared;
  const void* w2_shared;
  /* MOE_GEMM_MXFP8 / MOE_GEMM_NVFP4 only: the buffer moe_prepare_mxfp8_weights
   * or moe_prepare_nvfp4_weights filled from the weights above (NULL for bf16). */
  const void* mx;
} moe_weights;

/* Weight gradients (device, fp32 outputs).  dw_router [E,H], dw1 [E,2F,H],
 * dw2 [E,H,F], dw1_shared [2S,H], dw2_shared [H,S]. */
typedef struct {
  float* dw_router;
  float* dw1;
  float* dw2;
  float* dw1_shared;
  float* dw2_shared;
} moe_grads;

/* Byte offsets of the tensors kept in the activation buffer between the
 * forward and the backward calls.  cap = rows of every expert-ordered buffer;
 * each expert's rows start at a multiple of 128 ("padded offsets").
 * Layout of each field:
 *   logits fp32 [T,E]; topk_idx int32 [T,k] (descending key); topk_gate fp32 [T,k];
 *   counts int32 [E]; offsets int32 [E+1] (compact); poffsets int32 [E+1] (padded);
 *   slot_row int32 [T,k] (padded row of each (token, slot)); row_src int32 [cap]
 *   (token of each padded row, -1 for padding); row_gate fp32 [cap] (0 for padding);
 *   x_perm bf16 [cap,H]; z bf16 [cap,2F] (fc1 output); h bf16 [cap,F] (gate *
 *   SwiGLU output); o bf16 [cap,H] (fc2 output);
 *   zs bf16 [T,2S], hs bf16 [T,S], os bf16 [T,H] (shared expert, if S > 0);
 *   backward only: dy_perm bf16 [cap,H]; dz bf16 [cap,2F] (MXFP8 layers with F %
 *   256 == 0 leave it unwritten: their fc2 data gradient writes dz in MXFP8
 *   only); dx_perm bf16 [cap,H];
 *   dgate_part fp32 [cap, F/128]; dlogits fp32 [T,E]; row_dlogit fp32 [cap];
 *   dzs bf16 [T,2S]; dxs bf16 [T,H];
 *   MXFP8 layers, backward only: dz_qt u8 [2F,cap] (dz quantised along the
 *   rows, 32-row blocks, and transposed: the fc1 weight gradient's A operand,
 *   written by moe_layer_backward_dgrad) and dz_qt_sf its scale tiles (cap/128
 *   tiles per tile row of 128 of the 2F rows); h_qt u8 [F,cap] and h_qt_sf,
 *   h' the same way (the fc2 weight gradient's B operand, written by the
 *   forward).  MXFP8 layers write h' only in MXFP8: h stays unwritten.
 * Fields that do not apply have offset SIZE_MAX. */
typedef struct {
  size_t logits, topk_idx, topk_gate, counts, offsets, poffsets, slot_row, row_src, row_gate;
  size_t x_perm, z, h, o, zs, hs, os;
  size_t dy_perm, dz, dx_perm, dgate_part, dlogits, row_dlogit, dzs, dxs;
  size_t dz_qt, dz_qt_sf, h_qt, h_qt_sf;
  size_t total;          /* bytes the activation buffer needs */
  int32_t cap;           /* rows of the expert-ordered buffers */
  int32_t backward;      /* 1 if the backward fields are present */
} moe_act_layout;

/* Name of a status code (static string). */
const char* moe_status_string(moe_status s);

/* Library version, e.g. 0x000100 for 0.1.0. */
int32_t moe_version(void);

/* Number of CUDA kernels this library has launched in this process so far
 * (all devices, all streams).  Host only; for instrumentation. */
uint64_t moe_kernel_launches(void);

/* Rows of the expert-ordered buffers: the worst case over all routings,
 * T*k + 127*E rounded up to a multiple of 128.  Returns -1 on a bad config. */
int32_t moe_capacity_rows(const moe_config* cfg);

/* Fill `out` with the activation-buffer layout; with_backward = 1 adds the
 * backward fields.  Host only. */
moe_status moe_activation_layout(const moe_config* cfg, int32_t with_backward, moe_act_layout* out);

/* Bytes of scratch workspace every compute call below needs.  Host only.
 * The first 256 bytes of the workspace hold the device status word, the
 * grouped GEMMs' tile counter (ints 32 and 33), which hands out output tiles
 * in order and is back at zero after every GEMM launch, and the permutation's
 * count of finished histogram blocks (int 40, back at zero after each
 * moe_permute / bf16 moe_layer_forward).  Initialise them
 * once with moe_workspace_init before first use.  Calls that share one
 * workspace must not overlap on the GPU (issue them on one stream). */
size_t moe_workspace_bytes(const moe_config* cfg);

/* Zero the whole workspace (the device status word, the GEMM tile counter,
 * the fused combine's counters).  Stream-ordered, does not block. */
moe_status moe_workspace_init(void* ws, size_t ws_bytes, void* stream);

/* For tests of the failure path: every pipeline wait inside the grouped
 * GEMMs launched after this call gives up after `ns` nanoseconds instead of
 * the default 2 s (0 restores the default).  A wait that gives up makes its
 * kernel raise a flag that ends the other waits of its CTA, let every copy and
 * MMA already issued finish (bounded drains), free its TMEM and set
 * MOE_ERR_TIMEOUT in the status word; the outputs of that launch are then
 * incomplete.  Process-wide; not meant for production use.  No counterpart on
 * the pages: a library-side check of the bounded waits. */
void moe_debug_set_wait_limit_ns(uint64_t ns);

/* Synchronise `stream`, then copy the device status word to *code
 * (MOE_OK or the first device error since the last moe_workspace_init).
 * The only call that blocks; keep it out of the hot path. */
moe_status moe_read_device_status(const void* ws, int32_t* code, void* stream);

/* --------------------------------------------------------------------------
 * Step-level calls
 * ----------------------------------------------------------------------- */

/* Router GEMM and top-k gating.
 *   logits[t,e] = sum_h x[t,h] * w_router[e,h]  (bf16 in, fp32 accumulate, fp32 out)
 *   topk_idx[t,:] = the k experts with the largest key (key = logit for softmax,
 *   sigmoid(logit) + bias[e] for sigmoid), by key descending, lower id first on ties;
 *   a NaN key ranks as -infinity (after every finite key);
 *   topk_gate[t,:] = the normalised gates of those experts (fp32, sum to 1).
 * x [T,H] bf16; w_router [E,H] bf16; bias [E] fp32 or NULL.
 * Outputs: logits [T,E] fp32, topk_idx [T,k] int32, topk_gate [T,k] fp32. */
moe_status moe_router_topk(const moe_config* cfg, const void* x, const void* w_router, const float* bias,
                           float* logits, int32_t* topk_idx, float* topk_gate, void* ws, void* stream);

/* Top-k gating of given fp32 logits (the second half of moe_router_topk). */
moe_status moe_topk_gating(const moe_config* cfg, const float* logits, const float* bias, int32_t* topk_idx,
                           float* topk_gate, void* stream);

/* Sync-free permutation into expert-contiguous order (a stable counting sort
 * of the T*k (token, slot) pairs by expert id; inside an expert, ascending
 * token).  Any topk_idx may be given (router replay).  Outputs, all device:
 *   counts [E], offsets [E+1], poffsets [E+1] (segments padded to 128 rows),
 *   slot_row [T,k], row_src [cap] (-1 on padding), row_gate [cap] (topk_gate of
 *   the pair, 0 on padding; topk_gate may be NULL, then row_gate is not written),
 *   x_perm [cap,H] bf16 with x_perm[slot_row[t,i]] = x[t].  zero_pad = 1 also
 *   zeroes the padding rows of x_perm (needed before weight gradients).
 * An index outside [0,E) sets MOE_ERR_BAD_INDEX on the device; that pair is
 * dropped and no out-of-range memory is written. */
moe_status moe_permute(const moe_config* cfg, const void* x, const int32_t* topk_idx, const float* topk_gate,
                       int32_t* counts, int32_t* offsets, int32_t* poffsets, int32_t* slot_row,
                       int32_t* row_src, float* row_gate, void* x_perm, int32_t zero_pad, void* ws,
                       void* stream);

/* moe_permute without a workspace argument, for callers that cannot allocate
 * device memory: for example a plugin that an inference engine hands only
 * preallocated tensors, a host loop whose memory budget is fixed in advance,
 * or code that must not pay the device-wide synchronisation of cudaMalloc.
 * The pages have no counterpart to this call; it exists for such callers.
 *
 * Same arguments, outputs and layouts as moe_permute, minus `ws`.  The
 * counting sort's scratch lives in a 1 MiB array of device memory owned by
 * the library (every GPU that loads the library keeps it until the process
 * exits), so the call allocates nothing: no cudaMalloc, no cudaFree, no
 * allocating library routine.
 * Limit: ceil(T / floor(256/k)) * E <= 262144, i.e. ceil(T*k/256) * E when k
 * divides 256 (e.g. T*k up to 262144 pairs with
 * E = 256); larger shapes return MOE_ERR_WORKSPACE before any launch.
 * The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress, with that device current) and keeps it for that
 * device's current context; make that first call before any stream capture.
 * A call from another context on the same device (made with the driver API)
 * looks the address up again.  Not supported: calling it again after a
 * device reset (cudaDeviceReset) of a device it already ran on in this
 * process, where a new context may reuse the old handle.  All calls share the one array: calls whose
 * work overlaps on the GPU (other streams, other threads) race and must be
 * ordered by the caller.  The array's old contents are never read.
 * Device-side errors are not recorded (there is no status word): a pair with
 * an expert index outside [0,E) is dropped and its slot_row entry is -1. */
moe_status moe_permute_noalloc(const moe_config* cfg, const void* x, const int32_t* topk_idx,
                               const float* topk_gate, int32_t* counts, int32_t* offsets, int32_t* poffsets,
                               int32_t* slot_row, int32_t* row_src, float* row_gate, void* x_perm,
                               int32_t zero_pad, void* stream);

typedef enum {
  /* z = A * W1_e^T, h = g * silu(z[:, :F]) * z[:, F:].  a = x_perm [cap,H],
   * b = w1 [E,2F,H]; c = h [cap,F]; c2 = z [cap,2F] or NULL; row_gate [cap] or NULL (g = 1). */
  MOE_GG_FC1_SWIGLU = 0,
  /* o = A * W2_e^T.  a = h [cap,F], b = w2 [E,H,F]; c = o [cap,H]. */
  MOE_GG_FC2 = 1,
  /* dh = A * W2_e with A = dy_perm [cap,H], b = w2 [E,H,F]; epilogue with saved
   * aux = z [cap,2F]: dz = [g dh b silu'(a), g dh silu(a)] -> c [cap,2F];
   * dgate_part [cap, F/128] = partial sums of <dh, silu(a) b>. */
  MOE_GG_DGRAD_FC2 = 2,
  /* dx_perm = A * W1_e.  a = dz [cap,2F], b = w1 [E,2F,H]; c [cap,H]. */
  MOE_GG_DGRAD_FC1 = 3,
  /* dW1_e = A_e^T B_e over each expert's rows: a = dz [cap,2F], b = x_perm [cap,H];
   * c = dw1 [E,2F,H] fp32 (zero for experts with no rows). */
  MOE_GG_WGRAD_FC1 = 4,
  /* dW2_e = A_e^T B_e: a = dy_perm [cap,H], b = h [cap,F]; c = dw2 [E,H,F] fp32. */
  MOE_GG_WGRAD_FC2 = 5,
  /* FC1_SWIGLU with the permutation fused into the A load (bf16, routed only):
   * a = x [T,H] in token order, a_rows = row_src [cap] (token of each padded
   * row, -1 for padding: a zero row); A row r is x[a_rows[r]].  b, c, c2,
   * row_gate, poffsets as FC1_SWIGLU.  x_perm is neither read nor written. */
  MOE_GG_FC1_SWIGLU_GATHERED = 6,
  /* FC2 with the combine fused into its epilogue (bf16 or MXFP8, routed only,
   * H % 256 == 0): c = o [cap,H] as FC2, and c2 = y [T,H] with
   * y[t] = sum_i o[slot_row[t,i]] (+ aux[t]) summed in slot order in fp32 and
   * rounded once -- the same bits as moe_unpermute.  a_rows = row_src [cap],
   * slot_row [T,k] (rows -1 are skipped), aux = the shared expert's output
   * [T,H] or NULL.  Once a tile's rows of o are stored it counts them per
   * (token, 256 columns) in the workspace; the tile that completes a token's
   * slots sums them, so the order never depends on timing.  The counters must
   * be zero before the call (moe_workspace_init) and are zero after it; after
   * a device error (status word set) call moe_workspace_init again.  A token
   * none of whose slots is valid gets no y row.  Technical summary 2.2 of the
   * Megatron Core MoE summary (memory-efficient permutation: the combine is an
   * unweighted sum because the gate was applied before the activation). */
  MOE_GG_FC2_COMBINE = 7
} moe_gg_op;

/* Arguments of one grouped GEMM.  `poffsets` [E+1] (device) gives each expert's
 * first padded row; the host never reads it.  With dense_rows > 0 the GEMM runs
 * as one group of dense_rows rows instead (shared expert; poffsets ignored;
 * for the WGRAD ops the contraction runs over dense_rows rows and c has one
 * group).  Pass E in cfg as usual; the shapes H, F (or S for dense calls, see
 * moe_grouped_gemm) come from cfg. */
/* MXFP8 (dtype == MOE_GEMM_MXFP8): every operand is E4M3 codes plus E8M0
 * scales (see moe_quantize_mxfp8), K-major, blocks of 32 along the
 * contraction: a and b are codes and a_scales / b_scales their scale tiles.
 *   FC1_SWIGLU: a = x_perm [cap,H]; b = W1 rows gate/up interleaved
 *               (MOE_MX_ROWS_GATE_UP of w1 [E,2F,H]).
 *   FC2:        a = h [cap,F]; b = W2 [E*H,F] (MOE_MX_ROWS, or MOE_MX_ROWS_G224 with
 *               b_scale_group = 224).
 *   DGRAD_FC2:  a = dy_perm [cap,H]; b = W2^T [E,F,H] (MOE_MX_COLS_T of w2); aux = z (bf16).
 *   DGRAD_FC1:  a = dz [cap,2F]; b = W1^T [E,H,2F] (MOE_MX_COLS_T of w1, or MOE_MX_COLS_T_G224
 *               with b_scale_group = 224).
 *   WGRAD_FC1:  a = dz^T [2F,cap], b = x_perm^T [H,cap] (MOE_MX_COLS_T, or MOE_MX_COLS_T_G224
 *               with b_scale_group = 224).
 *   WGRAD_FC2:  a = dy_perm^T [H,cap], b = h^T [F,cap] (MOE_MX_COLS_T); or, with
 *               b_scale_group = 224 (F % 256 == 0), the operands swapped: a = h^T
 *               [F,cap] (MOE_MX_COLS_T), b = dy_perm^T [H,cap] (MOE_MX_COLS_T_G224),
 *               the GEMM computing dW2^T on 256 x 224 tiles and storing them
 *               transposed, so c is dW2 [E,H,F] either way.
 * Dense calls need dense_rows % 128 == 0.
 * NVFP4 (dtype == MOE_GEMM_NVFP4; forward ops only, the others return
 * MOE_ERR_UNSUPPORTED): a and b are E2M1 codes (see moe_quantize_nvfp4),
 * a_scales / b_scales their E4M3 scale tiles and a_amax / b_amax (device, one
 * fp32 each) the tensor amaxes they were quantised with.
 *   FC1_SWIGLU: a = x_perm codes [cap,H/2]; b = W1 codes, gate/up interleaved
 *               (MOE_MX_ROWS_GATE_UP of w1).
 *   FC2:        a = h codes [cap,F/2]; b = W2 codes [E*H,F/2] (MOE_MX_ROWS). */
typedef struct {
  int32_t op;             /* moe_gg_op */
  int32_t dense_rows;     /* 0: routed; >0: one dense group of this many rows */
  const void* a;
  const void* b;
  void* c;
  void* c2;
  const void* aux;
  const float* row_gate;
  float* dgate_part;
  const int32_t* poffsets;
  const void* a_scales;   /* MXFP8 / NVFP4 only */
  const void* b_scales;   /* MXFP8 / NVFP4 only */
  const float* a_amax;    /* NVFP4 only */
  const float* b_amax;    /* NVFP4 only */
  const int32_t* a_rows;  /* FC1_SWIGLU_GATHERED, FC2_COMBINE */
  const int32_t* slot_row;/* FC2_COMBINE only */
  int32_t b_scale_group;  /* MXFP8 FC2 / DGRAD_FC1 / WGRAD_FC1 / WGRAD_FC2 (routed, H % 224 == 0;
                             WGRAD_FC2 also F % 256 == 0, operands swapped as above): 224 when
                             b's scales were written by MOE_MX_ROWS_G224 / MOE_MX_COLS_T_G224 (the
                             GEMM then runs 256 x 224 tiles); 0 (or 128) otherwise and for every
                             other op */
  /* MXFP8 DGRAD_FC2 (routed, F % 256 == 0) and FC1_SWIGLU (routed); NULL
   * pairs: not written.  The output (dz, resp. h') also written in MXFP8 by
   * the epilogue, for the GEMMs that read it next -- q_codes [cap,N] with
   * q_scales (blocks along the row, as MOE_MX_ROWS) and qt_codes [N,cap] with
   * qt_scales (blocks of 32 rows, transposed, as MOE_MX_COLS_T), N = 2F for
   * dz and F for h'; bit-identical to quantising the bf16 output, rows < the
   * last expert's padded end.  c may be NULL (no bf16 output written) for
   * DGRAD_FC2 with both copies requested and for FC1_SWIGLU with the row copy. */
  void* q_codes;
  void* q_scales;
  void* qt_codes;
  void* qt_scales;
} moe_gemm_args;

/* One grouped GEMM on the tensor cores (tcgen05, TMA-fed, persistent).  For
 * dense calls (dense_rows > 0) the expert width is cfg->S if cfg->S > 0, else
 * cfg->F. */
moe_status moe_grouped_gemm(const moe_config* cfg, const moe_gemm_args* args, void* ws, void* stream);

/* Combine: y[t] = sum_i o_perm[slot_row[t,i]] (+ shared_out[t]), summed in
 * fp32 in slot order and rounded to bf16 once.  The gate is already inside
 * o_perm (technical summary 2.2).  o_perm [cap,H] bf16, slot_row [T,k],
 * shared_out [T,H] bf16 or NULL, y [T,H] bf16. */
moe_status moe_unpermute(const moe_config* cfg, const void* o_perm, const int32_t* slot_row,
                         const void* shared_out, void* y, void* stream);

/* --------------------------------------------------------------------------
 * MXFP8 (technical summary 2.5: FP8 expert GEMMs and activations, router
 * and combine kept in higher precision; the MXFP8 recipe on Blackwell).
 * Element type E4M3, one E8M0 scale per block of 32 values along the
 * contraction: X = 2^(floor(log2 amax) - 8) clamped to [2^-127, 2^127]
 * (2^-127 for an all-zero block), code = E4M3(v / X) rounded to nearest even,
 * saturated to +-448.
 * Scale layout ("scale tiles"): for a codes matrix [R, C] (R % 128 == 0,
 * C % 128 == 0) the R*C/32 scale bytes form 512-byte tiles, tile (i, j) covering
 * rows 128i..128i+127 and blocks 4j..4j+3 (columns 128j..128j+127) at byte
 * (i*(C/128) + j)*512; inside a tile the scale of row r, block b is at
 * (r%32)*16 + (r/32)*4 + b.  This is the order the tensor cores' scale-factor
 * copy consumes.
 * ----------------------------------------------------------------------- */

typedef enum {
  MOE_MX_ROWS = 0,          /* src [batch*rows, cols] -> codes [batch*rows, cols], blocks along each row */
  MOE_MX_COLS_T = 1,        /* src batch x [rows, cols] -> codes batch x [cols, rows], blocks along rows
                               (each matrix transposed; scale tiles per matrix) */
  MOE_MX_ROWS_GATE_UP = 2,  /* as ROWS, rows of every [gate; up] matrix of `rows` rows reordered as
                               gate 0..127, up 0..127, gate 128..255, up 128..255, ... (fc1 weights;
                               rows % 256 == 0) */
  MOE_MX_ROWS_G224 = 3,     /* as ROWS, codes identical, but the scale tiles take the rows in groups
                               of 224: group g's rows 0..127 are tile row 2g, its rows 128..223 the
                               first 96 rows of tile row 2g+1 (the other 32 rows of that tile are
                               never written nor read); batch*rows % 224 == 0.  For the B operand of
                               the 256 x 224 GEMM tiles (moe_gemm_args.b_scale_group). */
  MOE_MX_COLS_T_G224 = 4    /* as COLS_T with the output rows (the input columns) grouped by 224 the
                               same way, per matrix; cols % 224 == 0 */
} moe_mx_mode;

/* Quantise a bf16 tensor to MXFP8.  codes: batch*rows*cols bytes; scales:
 * batch*rows*cols/32 bytes (the G224 modes: 8/7 of that, R/224 * 2 tile rows
 * for R grouped rows).  cols % 128 == 0; ROWS: batch*rows % 128 == 0;
 * COLS_T: rows % 128 == 0; ROWS_GATE_UP: rows % 256 == 0; ROWS_G224:
 * batch*rows % 224 == 0; COLS_T_G224: rows % 128 == 0, cols % 224 == 0. */
moe_status moe_quantize_mxfp8(const void* src, int32_t batch, int32_t rows, int32_t cols, int32_t mode,
                              uint8_t* codes, uint8_t* scales, void* stream);

/* Bytes of the quantised-weight buffer an MXFP8 layer needs (moe_weights.mx). */
size_t moe_mxfp8_weights_bytes(const moe_config* cfg);

/* Quantise w1, w2 (and the shared expert) once into `mx`: the fc1/fc2 copies
 * and the transposed copies the data gradients contract over.  Call again
 * after every weight update. */
moe_status moe_prepare_mxfp8_weights(const moe_config* cfg, const moe_weights* w, void* mx, size_t mx_bytes,
                                     void* stream);

/* --------------------------------------------------------------------------
 * NVFP4 (technical summary 2.5 names NVFP4 beside MXFP8 for the expert GEMMs;
 * the format's own definition is taken as the recipe; forward GEMMs only).
 * Element type E2M1 (0, 0.5, 1, 1.5, 2, 3, 4, 6 and negatives), two codes per
 * byte with the lower-indexed element in the low nibble; one unsigned E4M3
 * scale per block of 16 values along the contraction; one fp32 tensor scale
 * S = 2688 / amax (1 if amax == 0).  With d = fp32(amax_b / 6), all in fp32:
 * s = e4m3(d * S) (nearest even, saturated to 448), r = S / s (0 if s == 0),
 * code = e2m1(v * r) (nearest even, saturated to +-6); value = e2m1 * s / S.
 * Scale tiles: for codes of a [R, C] matrix (R % 128 == 0, C % 64 == 0) the
 * R*C/16 scale bytes form 512-byte tiles, tile (i, j) covering rows
 * 128i..128i+127 and blocks 4j..4j+3 (columns 64j..64j+63) at byte
 * (i*(C/64) + j)*512; inside a tile the scale of row r, block b is at
 * (r%32)*16 + (r/32)*4 + b.
 * ----------------------------------------------------------------------- */

/* Quantise a bf16 tensor [batch*rows, cols] to NVFP4 along its rows (mode
 * MOE_MX_ROWS, or MOE_MX_ROWS_GATE_UP as for MXFP8).  Writes the tensor's
 * amax (fp32) to *amax (device) first, then codes (batch*rows*cols/2 bytes)
 * and scales (batch*rows*cols/16 bytes).  cols % 64 == 0, batch*rows % 128 == 0;
 * ROWS_GATE_UP: rows % 256 == 0.  Inputs must be finite. */
moe_status moe_quantize_nvfp4(const void* src, int32_t batch, int32_t rows, int32_t cols, int32_t mode,
                              uint8_t* codes, uint8_t* scales, float* amax, void* stream);

/* Bytes of the quantised-weight buffer an NVFP4 layer needs (moe_weights.mx);
 * 0 unless cfg->dtype == MOE_GEMM_NVFP4. */
size_t moe_nvfp4_weights_bytes(const moe_config* cfg);

/* Quantise w1 (gate/up interleaved), w2 and the shared expert once into the
 * buffer, each with its own tensor amax.  Call again after every weight update. */
moe_status moe_prepare_nvfp4_weights(const moe_config* cfg, const moe_weights* w, void* buf, size_t bytes,
                                     void* stream);

/* --------------------------------------------------------------------------
 * Whole layer
 * ----------------------------------------------------------------------- */

/* Forward: y = sum_i g_i SwiGLU_{e_i}(x) (+ SharedSwiGLU(x)).
 * x [T,H] bf16, y [T,H] bf16.  `act` holds everything backward needs (layout
 * from moe_activation_layout(cfg, with_backward)); with_backward = 1 also
 * zeroes the padding rows.  Fixed number of launches; no host sync.
 * NVFP4 layers: with_backward must be 0 (MOE_ERR_UNSUPPORTED otherwise); x is
 * quantised per token and its codes permuted, so x_perm is left unwritten.
 * MXFP8 layers likewise permute x's quantised codes and leave x_perm (and, in
 * the backward, dy_perm) unwritten: their weight gradients and the router's
 * read x and dy through row_src. 
 * The backward calls return MOE_ERR_UNSUPPORTED for NVFP4 layers. */
moe_status moe_layer_forward(const moe_config* cfg, const moe_weights* w, const void* x, void* y, void* act,
                             size_t act_bytes, int32_t with_backward, void* ws, size_t ws_bytes, void* stream);

/* Backward, data gradients.  Needs `act` from moe_layer_forward(with_backward=1)
 * of the same x.  dy [T,H] bf16 -> dx [T,H] bf16 (through the experts, the
 * shared expert and the router) and dgate [T,k] fp32 (NULL allowed).  Leaves
 * the tensors the weight gradients need in `act`. */
moe_status moe_layer_backward_dgrad(const moe_config* cfg, const moe_weights* w, const void* x, const void* dy,
                                    void* dx, float* dgate, void* act, size_t act_bytes, void* ws,
                                    size_t ws_bytes, void* stream);

/* Backward, weight gradients (fp32, overwritten).  Call after
 * moe_layer_backward_dgrad with the same `act`.  Experts that received no
 * token get zero gradients.  x [T,H] bf16, dy [T,H] bf16. */
moe_status moe_layer_backward_wgrad(const moe_config* cfg, const moe_weights* w, const void* x, const void* dy,
                                    const moe_grads* g, void* act, size_t act_bytes, void* ws, size_t ws_bytes,
                                    void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_H */
