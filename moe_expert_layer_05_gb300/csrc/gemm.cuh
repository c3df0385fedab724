// Persistent grouped GEMM on the 5th-generation tensor cores (tcgen05).
//
// One CTA per SM walks a list of output tiles: 128 x BN, or 256 x BN where two
// 128-row MMAs share each B k-block.  Warp roles:
//   warp 0      TMA producer: takes tile indices from a counter in global
//               memory and streams A and B k-blocks (one 128-B swizzle row:
//               64 bf16, 128 E4M3 or 256 E2M1 values, plus their scale tiles
//               for MXFP8 / NVFP4) into a STAGES-deep shared-memory ring; for
//               the gathered fc1 all 32 lanes copy A rows with cp.async;
//   warp 1      allocates TMEM; one lane issues tcgen05.mma (M=128, N=BN;
//               kind::f16, mxf8f6f4 or mxf4nvf4 block-scaled) into a TMEM
//               accumulator (two where they fit, so the epilogue of one tile
//               overlaps the MMAs of the next);
//   warps 2..   epilogue: tcgen05.ld the finished accumulator (warp w reads
//               TMEM lanes 32*(w%4)..+31, i.e. one output row per thread),
//               apply the fused elementwise step and store through TMA.
// grouped_gemm_pair_kernel at the end of this file runs 256 x 256 tiles on a
// pair of CTAs (a cluster of two) with tcgen05.mma.cta_group::2.
//
// Group shapes never reach the host.  For routed problems the kernel reads
// the padded per-expert row offsets (every expert segment is a whole number of
// 128-row blocks) from device memory and derives its tile list from them: this
// is the grouped GEMM with device-side shapes that the Megatron Core MoE
// summary describes (technical summary 2.4, grouped GEMM and sync-free
// kernels).
#pragma once
#include "nvfp4.cuh"
#include "mx_quant.cuh"
#include "ptx.cuh"

namespace moe {

enum class Sched : int {
  kRoutedM = 0,  // rows grouped by expert (padded offsets on device), K fixed
  kDenseM = 1,   // one group of m_rows rows
  kRoutedK = 2,  // contraction over each expert's rows (weight gradients)
};

enum class Epi : int {
  kStoreF32 = 0,    // fp32 accumulator -> fp32
  kStoreBf16 = 1,   // -> bf16
  kSwiglu = 2,      // z = [gate | up] -> h = g * silu(gate) * up (bf16), z saved (bf16)
  kSwigluBwd = 3,   // dh -> dz = [dgate_in | dup] (bf16) and partial <dh, h> per row
};

struct GemmParams {
  const int* poffsets;     // [E+1] padded row offsets (kRoutedM, kRoutedK); nullptr = one group
  int E;                   // number of groups
  int m_rows;              // kDenseM: rows; kRoutedK: output rows per group
  int k_len;               // contraction length (kRoutedM, kDenseM); kRoutedK without poffsets: rows
  int n_tiles;             // output tiles along N
  int m_tiles_w;           // kRoutedK: output tiles along M per group
  int b_rows_per_group;    // rows of B's 2-D view that belong to one group
  int b_half_offset;       // kSwiglu: row offset of the "up" half inside a group of B
  void* c;                 // primary output
  long long ldc;           // its row stride (elements)
  long long c_group_stride;// kRoutedK: elements between groups of the output
  void* c2;                // kSwiglu: z (nullable)
  long long ldc2;
  int half_cols;           // kSwiglu / kSwigluBwd: F (column offset of the up half in z / dz)
  const __nv_bfloat16* aux;// kSwigluBwd: saved z
  long long ld_aux;
  const float* row_gate;   // per output row gate (nullptr: 1.0)
  float* dgate_part;       // kSwigluBwd: [rows, n_tiles] partial dot products
  int valid_cols;          // kStoreF32: store only columns < valid_cols
  int c_trans;             // kStoreF32, kRoutedK: output stored transposed, element (m, n) of group g
                           // at c[g * c_group_stride + n * m_rows + m]
  int rows_cap;            // rows allocated in the expert-ordered buffers (routed modes)
  // MXFP8 / NVFP4: scale tiles of A and B (512 B per 128 rows x 128 K of
  // E8M0, or x 64 K of E4M3; see mxfp8.cu, nvfp4.cu) and the number of tiles
  // along K in one 128-row band of each.
  const uint8_t* sfa;
  const uint8_t* sfb;
  int sfa_tiles_k;
  int sfb_tiles_k;
  // NVFP4: the tensor amax of A and of B (device); the accumulator is
  // multiplied by 1 / (S_a * S_b) before the epilogue's arithmetic.
  const float* amax_a;
  const float* amax_b;
  // NVFP4 kSwiglu (nullable): atomicMax of |h'| as stored (bf16 values, fp32
  // bit patterns, non-negative so they order as unsigned) -- the tensor amax
  // the NVFP4 quantiser of h' needs, taken without another pass over h'.
  unsigned* amax_out;
  // Gathered A (fc1 with the permutation fused into its A load): row r of the
  // tile is row a_row_src[r] of a_tok [a_rows, k_len] (token order), or zeros
  // where a_row_src[r] < 0 (padding).
  const __nv_bfloat16* a_tok;
  const int32_t* a_row_src;
  int a_rows;
  int* status;             // device status word (first error wins)
  int* sched;              // [0] next tile, [1] CTAs finished: the dynamic schedule (nullptr: static)
  unsigned long long wait_ns;  // limit of a pipeline wait before the kernel gives up (0: kWaitLimitNs)
  // fc2 with the combine fused into its epilogue (kStoreBf16, BN = 256, routed;
  // cmb_y == nullptr: off).  After a tile's rows of o are stored, each row adds
  // one to the counter of (its token, this N tile); the arrival that completes
  // the token's valid slots sums the token's k rows of those columns in slot
  // order (fp32, plus the shared expert's row), writes y once and puts the
  // counter back to zero.
  // MXFP8 copies of the output quantised in the epilogue for the GEMMs that
  // read it next (the split SwiGLU-backward tiles; nullptr: none): q = rows
  // quantised along the row, [rows_cap, ld_q] codes with ld_q / 128 scale
  // tiles per tile row; qt = quantised along the rows (32-row blocks, one per
  // epilogue warp) and transposed, [ld_q, rows_cap] codes with rows_cap / 128
  // scale tiles per tile row.  Bit-identical to the standalone quantisers
  // applied to the bf16 output.
  uint8_t* q_codes;
  uint8_t* q_sf;
  uint8_t* qt_codes;
  uint8_t* qt_sf;
  int ld_q;
  const int32_t* cmb_row_src;      // [rows_cap] token of each row, -1 padding
  const int32_t* cmb_slot_row;     // [T, k] row of each (token, slot), -1 dropped
  int cmb_k;
  int* cmb_count;                  // [T, n_tiles], zero between launches
  const __nv_bfloat16* cmb_shared; // [T, ldc] or nullptr
  __nv_bfloat16* cmb_y;            // [T, ldc]
};

template <int BN_, bool A_MN_, bool B_MN_, Sched S_, Epi EP_, int MX_ = 0, bool M256_ = false,
          bool PAIR_ = false, bool GATHER_ = false>
struct GemmCfg {
  static constexpr int BM = 128;                  // rows of A and D per CTA and MMA
  static constexpr bool M256 = M256_;             // 256-row tiles: two MMAs share each B k-block
  static constexpr bool PAIR = PAIR_;             // 256-row tiles on a CTA pair (cta_group::2)
  static constexpr bool ROWS256 = M256 || PAIR;   // tiles of 256 rows (pairs of 128-row blocks)
  static constexpr int TILE_M = ROWS256 ? 256 : 128;
  static constexpr bool MX = MX_ != 0;            // block-scaled operands: 1 MXFP8, 2 NVFP4
  // A rows gathered by the producer warp from the token-order input with
  // 16-byte cp.async copies (the permutation fused into fc1's A load)
  static constexpr bool GATHER = GATHER_;
  // arrivals that complete a full barrier: the TMA producer's, plus one per
  // gathering lane
  static constexpr int FULL_COUNT = GATHER ? 33 : 1;
  static constexpr bool NV4 = MX_ == 2;           // NVFP4 (E2M1 + E4M3 1x16 scales + tensor scale)
  // Contraction elements per k-block: one 128-byte swizzle row (K-major), or
  // for the weight gradients on CTA pairs (MN-major, short per-expert K) 128
  // token rows, so each TMA box is 16 KB instead of 8 KB.
  static constexpr bool WIDE_K = PAIR_ && (S_ == Sched::kRoutedK);
  static constexpr int BK = NV4 ? 256 : MX ? 128 : (WIDE_K ? 128 : 64);   // elements (128 B K-major rows)
  static constexpr int MN_CHUNK = BK * 128;       // MN-major: bytes of one 64-wide MN chunk (BK rows of 128 B)
  static constexpr int KSTEP = NV4 ? 64 : MX ? 32 : 16;   // K of one MMA instruction (32 bytes)
  static constexpr int BN = BN_;
  static constexpr bool A_MN = A_MN_;
  static constexpr bool B_MN = B_MN_;
  static constexpr Sched S = S_;
  static constexpr Epi EP = EP_;
  static constexpr int ROW_BYTES = NV4 ? BK / 2 : MX ? BK : BK * 2;   // bytes of one A / B row of a k-block
  static constexpr int A_BYTES = (M256 ? 256 : 128) * ROW_BYTES;   // this CTA's A rows of one k-block
  static constexpr int B_BYTES = (PAIR ? BN / 2 : BN) * ROW_BYTES;  // this CTA's B rows (a pair splits N)
  // scale tiles of one k-block: one 512-byte tile per 128 rows (MXFP8), four
  // (one per MMA of K = 64) for NVFP4
  static constexpr int SF_TILES_KB = NV4 ? 4 : 1;
  // scale tiles of A (one per 128 rows of the tile) and of B (one per 128
  // rows, rounded up: a 224-row B tile takes two, from the layout that groups
  // B's rows by 224 -- the tile's rows 128..223 fill 96 rows of the second)
  static constexpr int SFA_TILES = M256 ? 2 : 1;
  static constexpr int SFB_TILES = (BN + 127) / 128;
  static constexpr int SFB_GROUP = (MX && BN % 128 != 0) ? BN : 128;
  static constexpr int SFA_BYTES = MX ? 512 * SF_TILES_KB * SFA_TILES : 0;
  static constexpr int SFB_BYTES = MX ? SFB_TILES * 512 * SF_TILES_KB : 0;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES + SFA_BYTES + SFB_BYTES;
  // Outputs leave through TMA stores staged in shared memory (every epilogue
  // but the router's narrow fp32 logits, whose rows need not be 16-byte sized).
  static constexpr bool TMA_OUT = !(EP == Epi::kStoreF32 && S == Sched::kDenseM);
  // Epilogue warps: four (one per TMEM lane quarter), or eight for 256-row
  // tiles, where the second four write rows 128..255 at the same time.
  // NVFP4 SwiGLU tiles (one accumulator, MMAs fast enough that the MMA warp
  // waits for it): eight warps too, the second four taking the upper half of
  // the h' columns, so the accumulator is read and handed back in half the time.
  // MXFP8 SwiGLU-backward tiles of N = 256 likewise: each warp loads its 128
  // columns of dh into registers and hands the accumulator back at once (the
  // elementwise backward is the long part of that epilogue), then stores dz in
  // 32-column chunks through 2 KB staging buffers, so the ring keeps 4 stages.
  static constexpr bool SPLIT_BWD = MX && !NV4 && EP == Epi::kSwigluBwd && BN == 256;
  // MXFP8 gated-SwiGLU tiles likewise: each warp takes 64 columns of h' (its
  // 64 gate and 64 up accumulator columns), then writes z and h' (or h''s
  // MXFP8 copies) in 32-column chunks through the same 2 KB staging.
  static constexpr bool SPLIT_FWD = MX && !NV4 && EP == Epi::kSwiglu && BN == 256;
  static constexpr bool SPLIT_COLS = (NV4 && EP == Epi::kSwiglu && BN == 256) || SPLIT_BWD || SPLIT_FWD;
  static constexpr int EPI_WARPS = (M256 || SPLIT_COLS) ? 8 : 4;
  // Shared memory (all of it dynamic): the k-block ring, 4 KB staging buffers
  // (32 rows x 128 B, 128B-swizzled) per epilogue warp -- two each, or one
  // where two would cost the ring its fourth stage -- and the bookkeeping
  // (barriers, expert offsets, tile prefix).  The ring starts on a 1024-byte
  // boundary; up to 1 KB of slack is kept for that where it fits, and the
  // kernel checks the base it is given before it touches anything.
  static constexpr int BOOK_BYTES = ROWS256 ? 2432 : 1408;
  static constexpr int SLACK_MIN = ROWS256 ? 0 : 1024;
  static constexpr int SMEM_BUDGET = 232448 - BOOK_BYTES - SLACK_MIN;
  static constexpr int RING_IF_TWO = (SMEM_BUDGET - (TMA_OUT ? EPI_WARPS * 2 * 4096 : 0)) / STAGE_BYTES;
  // Weight gradients are bound by their fp32 stores: each epilogue warp keeps
  // several 4 KB stores in flight (the k-loops are short, so the ring needs
  // few stages).
  // (256 x 224 MXFP8 weight-gradient tiles: eight warps, one buffer each, so
  // the ring keeps three 62 KB stages)
  static constexpr int WGRAD_BUFS = WIDE_K ? 2 : (M256 ? 1 : 4);
  static constexpr int STAGING_BUFS = (S == Sched::kRoutedK && TMA_OUT) ? WGRAD_BUFS
                                      // gate and up chunks side by side; one buffer (the up chunk
                                      // waits in registers) where two would cost the ring a stage
                                      : (EP == Epi::kSwigluBwd) ? ((MX && BN == 256) ? 1 : 2)
                                      : ((TMA_OUT && RING_IF_TWO < 4) ? 1 : 2);
  static constexpr int STAGING_BUF = (SPLIT_BWD || SPLIT_FWD) ? 2048 : 4096;   // bytes of one staging buffer
  static constexpr int STAGING_BYTES = TMA_OUT ? EPI_WARPS * STAGING_BUFS * STAGING_BUF : 0;
  static constexpr int STAGES_RAW = (SMEM_BUDGET - STAGING_BYTES - (MX ? 1024 : 0)) / STAGE_BYTES;
  static constexpr int STAGES = STAGES_RAW > 8 ? 8 : STAGES_RAW;
  // the scale tiles of all stages, padded so the staging buffers after them
  // start on a 1024-byte boundary (the 128-byte swizzle of the TMA stores)
  static constexpr int SF_REGION = (STAGES * (SFA_BYTES + SFB_BYTES) + 1023) / 1024 * 1024;
  static constexpr int SMEM_USED = STAGES * (A_BYTES + B_BYTES) + SF_REGION + STAGING_BYTES + BOOK_BYTES;
  static constexpr int SMEM_BYTES = (SMEM_USED + 1024 <= 232448) ? SMEM_USED + 1024 : 232448;
  // TMEM columns of one stage's scales (4 per 128 rows and scale tile)
  static constexpr int SF_COLS = MX ? SF_TILES_KB * 4 * (SFA_TILES + SFB_TILES) : 0;
  // TMEM accumulators: two (epilogue of tile i overlaps MMAs of tile i+1),
  // or one where two would not fit next to the scales (MXFP8, N=256) or in
  // 512 columns at all (256-row tiles of N=256: 2 x 256 columns per tile).
  static constexpr int ACC_COLS = (M256 ? 2 : 1) * BN;      // a pair: each CTA holds its 128 rows
  static constexpr int ACC_BUFS = ((MX && BN == 256) || 2 * ACC_COLS > 512) ? 1 : 2;
  static constexpr int TMEM_COLS_RAW = ACC_BUFS * ACC_COLS + STAGES * SF_COLS;
  static constexpr int TMEM_COLS = TMEM_COLS_RAW <= 32 ? 32 : TMEM_COLS_RAW <= 64 ? 64
                                   : TMEM_COLS_RAW <= 128 ? 128 : TMEM_COLS_RAW <= 256 ? 256 : 512;
  // Rows of one K-major B box (the SwiGLU tile loads gate and up halves as two boxes).
  // (MXFP8: W1 is stored with gate and up rows interleaved in 128-row blocks, one box.)
  static constexpr int B_BOX_ROWS = ((EP == Epi::kSwiglu && !MX) || PAIR) ? BN / 2 : BN;
  // Columns of the output a tile covers (SwiGLU: half of the accumulator).
  static constexpr int OUT_COLS = (EP == Epi::kSwiglu) ? BN / 2 : BN;
  static constexpr int THREADS = 64 + 32 * EPI_WARPS;
  static constexpr uint32_t IDESC = NV4  ? idesc_nvf4_e2m1(BM, BN)
                                    : MX  ? idesc_mxf8_e4m3(BM, BN)
                                          : idesc_bf16_f32(PAIR ? 256 : BM, BN, A_MN, B_MN);
  static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "N of one MMA");
  static_assert(!B_MN || BN % 64 == 0, "MN-major B is loaded in 64-column chunks");
  static_assert(EP != Epi::kSwiglu || BN == 256, "SwiGLU tile: 128 gate + 128 matching up columns");
  static_assert(!MX || ((BN % 128 == 0 || (BN == 224 && M256)) && !A_MN && !B_MN),
                "MXFP8 operands are K-major, 128-row scale tiles (224-row B tiles: 256 x 224 tiles)");
  static_assert(!NV4 || (S != Sched::kRoutedK && EP != Epi::kSwigluBwd && EP != Epi::kStoreF32),
                "NVFP4: forward GEMMs (bf16 or SwiGLU epilogue)");
  static_assert(TMEM_COLS_RAW <= 512, "TMEM columns");
  static_assert(!M256 || (!A_MN && (MX ? (!NV4 && BN == 224 &&
                                           (S == Sched::kRoutedK ? EP == Epi::kStoreF32 : EP == Epi::kStoreBf16))
                                        : S != Sched::kRoutedK)),
                "256-row tiles: K-major A; bf16 ones row-grouped, MXFP8 ones 256 x 224 (bf16 stores, or fp32 "
                "weight gradients)");
  static_assert(!M256 || TMA_OUT, "256-row tiles store through TMA");
  static_assert(!GATHER || (M256 && !MX && !A_MN && S == Sched::kRoutedM && BK == 64),
                "gathered A: bf16 256-row row-grouped tiles");
  static_assert(!WIDE_K || (A_MN && B_MN), "128-row k-blocks only for MN-major operands");
  static_assert(!PAIR || (!M256 && !MX && TMA_OUT && BN == 256 &&
                          (S == Sched::kRoutedK ? (A_MN && B_MN && EP == Epi::kStoreF32) : !A_MN)),
                "CTA pairs: bf16, N = 256; row-grouped GEMMs with K-major A, or MN-major weight gradients");
  static_assert(SMEM_USED <= SMEM_BYTES && SMEM_BYTES <= 232448, "shared memory per CTA");
  static_assert(STAGES >= 2, "pipeline depth");
  static_assert((STAGES * (A_BYTES + B_BYTES) + SF_REGION) % 1024 == 0, "staging buffers 1024-byte aligned");
};

struct TileInfo {
  int group;     // expert
  int m0;        // first A row (kRoutedM / kDenseM) or first output row (kRoutedK)
  int n;         // N tile index
  int num_kb;    // k-blocks
  int k_row0;    // kRoutedK: first contraction row
  bool half1;    // 256-row tiles: rows m0+128..m0+255 belong to this tile
};

// 256-row tiles of a routed problem: expert e has ceil(blocks_e / 2) row pairs
// (blocks of 128 rows) per N tile; s_tpre[e] = tiles of the experts before e.
__device__ __forceinline__ void build_pair_prefix(const int* s_poff, int E, int n_tiles, int* s_tpre) {
  // one warp: lane l owns a contiguous run of experts
  const int lane = threadIdx.x & 31;
  const int per = (E + 31) / 32;
  const int e0 = lane * per, e1 = min(E, e0 + per);
  int sum = 0;
  for (int e = e0; e < e1; ++e) sum += ((s_poff[e + 1] - s_poff[e]) / 128 + 1) / 2 * n_tiles;
  int inc = sum;
  #pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, inc, d);
    if (lane >= d) inc += v;
  }
  int run = inc - sum;
  for (int e = e0; e < e1; ++e) {
    s_tpre[e] = run;
    run += ((s_poff[e + 1] - s_poff[e]) / 128 + 1) / 2 * n_tiles;
  }
  if (lane == 31) s_tpre[E] = inc;
}

template <class C>
__device__ __forceinline__ int total_tiles(const GemmParams& p, const int* s_poff, const int* s_tpre) {
  if constexpr (C::S == Sched::kRoutedM) {
    if constexpr (C::ROWS256) return s_tpre[p.E];
    return (s_poff[p.E] / C::BM) * p.n_tiles;
  } else if constexpr (C::S == Sched::kDenseM) {
    return ((p.m_rows + C::TILE_M - 1) / C::TILE_M) * p.n_tiles;
  } else {
    return p.E * p.m_tiles_w * p.n_tiles;
  }
}

template <class C>
__device__ __forceinline__ TileInfo decode_tile(const GemmParams& p, const int* s_poff, const int* s_tpre, int t) {
  TileInfo ti;
  ti.half1 = false;
  if constexpr (C::S == Sched::kRoutedM && C::ROWS256) {
    int lo = 0, hi = p.E - 1;          // largest e with s_tpre[e] <= t (a non-empty expert)
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s_tpre[mid] <= t) lo = mid; else hi = mid - 1;
    }
    const int local = t - s_tpre[lo];
    const int mt = ((s_poff[lo + 1] - s_poff[lo]) / 128 + 1) / 2;
    ti.group = lo;
    ti.n = local / mt;                       // n outer: a B panel stays hot in L2
    ti.m0 = s_poff[lo] + (local % mt) * 256;
    ti.half1 = ti.m0 + 128 < s_poff[lo + 1];
    ti.num_kb = p.k_len / C::BK;
    ti.k_row0 = 0;
  } else if constexpr (C::S == Sched::kRoutedM) {
    // largest e with (poff[e]/BM)*n_tiles <= t; empty experts share a prefix
    // with the next one, so the result is always a non-empty expert.
    int lo = 0, hi = p.E - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if ((s_poff[mid] / C::BM) * p.n_tiles <= t) lo = mid; else hi = mid - 1;
    }
    const int local = t - (s_poff[lo] / C::BM) * p.n_tiles;
    const int mt = (s_poff[lo + 1] - s_poff[lo]) / C::BM;
    ti.group = lo;
    ti.n = local / mt;                       // n outer: a B panel stays hot in L2
    ti.m0 = s_poff[lo] + (local % mt) * C::BM;
    ti.num_kb = p.k_len / C::BK;
    ti.k_row0 = 0;
  } else if constexpr (C::S == Sched::kDenseM) {
    const int mb = (p.m_rows + C::TILE_M - 1) / C::TILE_M;
    ti.group = 0;
    ti.n = t / mb;
    ti.m0 = (t % mb) * C::TILE_M;
    ti.half1 = C::ROWS256 && (ti.m0 + 128 < p.m_rows);
    ti.num_kb = p.k_len / C::BK;
    ti.k_row0 = 0;
  } else {
    const int per = p.m_tiles_w * p.n_tiles;
    ti.group = t / per;
    const int r = t % per;
    ti.m0 = (r / p.n_tiles) * (C::ROWS256 ? 256 : C::BM);   // a pair or a 256-row tile covers 256 output rows
    ti.half1 = C::ROWS256;                                  // (both halves always in range)
    ti.n = r % p.n_tiles;
    if (p.poffsets != nullptr) {
      ti.k_row0 = s_poff[ti.group];
      ti.num_kb = (s_poff[ti.group + 1] - s_poff[ti.group]) / C::BK;
    } else {
      ti.k_row0 = 0;
      ti.num_kb = (p.k_len + C::BK - 1) / C::BK;
    }
  }
  return ti;
}

template <class C>
__device__ __forceinline__ void issue_loads(const CUtensorMap* tmA, const CUtensorMap* tmB, const GemmParams& p,
                                            const TileInfo& ti, int kb, uint8_t* a_dst, uint8_t* b_dst,
                                            uint8_t* sf_dst, uint64_t* bar) {
  const int k0 = kb * C::BK;
  if constexpr (C::MX) {
    // K-major E4M3 tiles (128 B per row) plus their 512-byte scale tiles.
    int a_row, b_row, k_col;
    if constexpr (C::S == Sched::kRoutedK) {
      a_row = ti.m0;
      b_row = ti.n * C::BN;
      k_col = ti.k_row0 + k0;
    } else {
      a_row = ti.m0;
      b_row = ti.group * p.b_rows_per_group + ti.n * C::BN;
      k_col = k0;
    }
    // the TMA maps count bytes along K: two E2M1 codes per byte for NVFP4
    const int k_byte = C::NV4 ? k_col / 2 : k_col;
    tma_load_2d(a_dst, tmA, bar, k_byte, a_row);
    tma_load_2d(b_dst, tmB, bar, k_byte, b_row);
    // scale tiles of this k-block: contiguous along K within a 128-row band
    constexpr int TB = 512 * C::SF_TILES_KB;
    const int kt = k_col / (C::NV4 ? 64 : 128);
    bulk_load(sf_dst, p.sfa + ((long long)(a_row / 128) * p.sfa_tiles_k + kt) * 512, TB, bar);
    if constexpr (C::SFA_TILES == 2) {
      // rows 128..255 of a 256-row tile; a tile without them (the last of an
      // expert with an odd number of 128-row blocks) loads its first tile again,
      // so the byte count stays fixed and nothing past the buffer is read
      const int a_tile1 = a_row / 128 + (ti.half1 ? 1 : 0);
      bulk_load(sf_dst + TB, p.sfa + ((long long)a_tile1 * p.sfa_tiles_k + kt) * 512, TB, bar);
    }
    // B rows grouped by SFB_GROUP (128: one tile per 128 rows; 224: two tiles a group)
    const int b_tile0 = (C::SFB_GROUP == 128) ? b_row / 128 : (b_row / C::SFB_GROUP) * C::SFB_TILES;
    #pragma unroll
    for (int i = 0; i < C::SFB_TILES; ++i)
      bulk_load(sf_dst + TB * (C::SFA_TILES + i), p.sfb + ((long long)(b_tile0 + i) * p.sfb_tiles_k + kt) * 512, TB,
                bar);
    return;
  }
  // ---- A (gathered tiles: the producer warp copies A itself)
  if constexpr (C::S == Sched::kRoutedK) {
    // A[m, k] = Abuf[k_row0 + k, m0 + m]  (MN-major, two 64-wide chunks)
    tma_load_2d(a_dst, tmA, bar, ti.m0, ti.k_row0 + k0);
    tma_load_2d(a_dst + 8192, tmA, bar, ti.m0 + 64, ti.k_row0 + k0);
  } else if constexpr (!C::GATHER) {
    tma_load_2d(a_dst, tmA, bar, k0, ti.m0);
  }
  // ---- B
  if constexpr (C::S == Sched::kRoutedK) {
    #pragma unroll
    for (int j = 0; j < C::BN / 64; ++j)
      tma_load_2d(b_dst + j * 8192, tmB, bar, ti.n * C::BN + j * 64, ti.k_row0 + k0);
  } else if constexpr (C::B_MN) {
    // B[n, k] = W[group*K + k, n]   (weights stored [K, N] per group, N contiguous)
    #pragma unroll
    for (int j = 0; j < C::BN / 64; ++j)
      tma_load_2d(b_dst + j * 8192, tmB, bar, ti.n * C::BN + j * 64, ti.group * p.b_rows_per_group + k0);
  } else if constexpr (C::EP == Epi::kSwiglu) {
    const int row = ti.group * p.b_rows_per_group + ti.n * (C::BN / 2);
    tma_load_2d(b_dst, tmB, bar, k0, row);
    tma_load_2d(b_dst + (C::BN / 2) * 128, tmB, bar, k0, row + p.b_half_offset);
  } else {
    tma_load_2d(b_dst, tmB, bar, k0, ti.group * p.b_rows_per_group + ti.n * C::BN);
  }
}

__device__ __forceinline__ bool mbar_wait_drain(uint64_t* bar, uint32_t parity) {
  const unsigned long long t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > kWaitLimitNs / 4) return false;
  }
  return true;
}

template <class C>
__device__ __forceinline__ void epilogue_tile(const GemmParams& p, const TileInfo& ti, uint32_t tmem_acc,
                                              int quarter, int lane) {
  // Plain stores: only the router logits (fp32, N = E columns, rows not
  // necessarily 16-byte sized) leave this way; every other epilogue uses TMA.
  static_assert(C::EP == Epi::kStoreF32 && C::S == Sched::kDenseM, "router epilogue");
  const int row = ti.m0 + quarter * 32 + lane;
  const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
  const bool row_ok = row < p.m_rows;
  float* out = reinterpret_cast<float*>(p.c) + (long long)row * p.ldc;
  #pragma unroll 1
  for (int c0 = 0; c0 < C::BN; c0 += 16) {
    uint32_t v[16];
    tmem_ld_x16(tmem_acc + lane_addr + c0, v);
    tmem_ld_wait(v);
    const int colbase = ti.n * C::BN + c0;
    if (row_ok) {
      #pragma unroll
      for (int j = 0; j < 16; ++j)
        if (colbase + j < p.valid_cols) out[colbase + j] = __uint_as_float(v[j]);
    }
  }
}

// Per-warp staging of output chunks for TMA stores: two 4 KB buffers, each
// 32 rows (one per lane) x 128 bytes in the 128-byte swizzled order (16-byte
// chunk c of row r sits at chunk c ^ (r % 8)), so a warp's 16-byte stores hit
// distinct banks.  Lane 0 issues the stores and owns the bulk groups.
template <int NBUF, int BUF = 4096>
struct Stager {
  uint8_t* buf;
  int cur;
  int lane;

  __device__ __forceinline__ void begin() {   // the buffer about to be filled is no longer read by TMA
    if (lane == 0) bulk_wait_group_read<NBUF - 1>();
    __syncwarp();
  }
  __device__ __forceinline__ void begin_all() {   // every buffer is no longer read by TMA
    if (lane == 0) bulk_wait_group_read<0>();
    __syncwarp();
  }
  __device__ __forceinline__ void put(int c, uint32_t a, uint32_t b, uint32_t cc, uint32_t d) {
    const uint32_t base = smem_u32(buf + cur * BUF);
    st_shared_v4(base + lane * 128 + ((c ^ (lane & 7)) << 4), a, b, cc, d);
  }
  // 16-byte chunk c of this lane's row in a buffer of 64-byte rows without
  // swizzle (for a 32-column bf16 box)
  __device__ __forceinline__ void put_rows64(int c, uint32_t a, uint32_t b, uint32_t cc, uint32_t d) {
    const uint32_t base = smem_u32(buf + cur * BUF);
    st_shared_v4(base + lane * 64 + (c << 4), a, b, cc, d);
  }
  // 16-byte chunk c of this lane's 64-byte row in the 64-byte swizzled order
  // (chunk c of row r at chunk c ^ ((r / 2) % 4)): 32-column bf16 boxes, with
  // eight consecutive lanes' stores in distinct banks
  __device__ __forceinline__ void put_rows64_sw(int c, uint32_t a, uint32_t b, uint32_t cc, uint32_t d) {
    const uint32_t base = smem_u32(buf + cur * BUF);
    st_shared_v4(base + lane * 64 + ((c ^ ((lane >> 1) & 3)) << 4), a, b, cc, d);
  }
  // into the buffer after the current one (two buffers filled in one pass)
  __device__ __forceinline__ void put_next(int c, uint32_t a, uint32_t b, uint32_t cc, uint32_t d) {
    const uint32_t base = smem_u32(buf + (cur ^ 1) * BUF);
    st_shared_v4(base + lane * 128 + ((c ^ (lane & 7)) << 4), a, b, cc, d);
  }
  __device__ __forceinline__ void flush(const CUtensorMap* map, int x, int y) {
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      tma_store_2d(map, buf + cur * BUF, x, y);
      bulk_commit_group();
    }
    cur = (cur + 1 == NBUF) ? 0 : cur + 1;
  }
  __device__ __forceinline__ void drain() {
    if (lane == 0) bulk_wait_group_all();
    __syncwarp();
  }
};

// One 32-column chunk of a bf16 output held by a warp, lane = row y + lane, o
// = the row's 32 values as packed pairs, first column ocol.  The chunk goes
// to the 64-byte-swizzled staging buffer; from there it is stored through tm
// (nullptr: not stored) and, as p asks, quantised: q = this row's 32 values
// as one MX block (from the registers); qt = column ocol + lane's 32 rows as
// one block, transposed (the lane reads its column back from the staging, two
// short loops, so the code stays small).
template <int NBUF, int BUF>
__device__ __forceinline__ void emit_chunk32(const GemmParams& p, Stager<NBUF, BUF>& st, const uint32_t (&o)[16],
                                             int ocol, int y, int lane, const CUtensorMap* tm, bool quant = true) {
  st.begin();
  #pragma unroll
  for (int q = 0; q < 4; ++q) st.put_rows64_sw(q, o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
  const bool want_qt = quant && p.qt_codes != nullptr, want_q = quant && p.q_codes != nullptr;
  const uint32_t sbase = smem_u32(st.buf + st.cur * BUF);
  if (want_qt) {
    uint32_t t[8];
    __syncwarp();                               // every row of the chunk is in the staging
    // element (r, lane): 16-byte chunk lane/8 of row r, swizzled, element lane%8
    const uint32_t col_off = static_cast<uint32_t>((lane & 7) * 2);
    const uint32_t cj = static_cast<uint32_t>(lane >> 3);
    auto elem = [&](int r) {
      const uint32_t a = sbase + r * 64 + ((cj ^ ((r >> 1) & 3)) << 4) + col_off;
      return __uint_as_float(ld_shared_u16(a) << 16);
    };
    float amax = 0.f;
    #pragma unroll 4
    for (int r = 0; r < 32; ++r) amax = fmaxf(amax, fabsf(elem(r)));
    const int et = mx_exponent(amax);
    const float sc = pow2_neg(et);
    #pragma unroll
    for (int r4 = 0; r4 < 8; ++r4)
      t[r4] = e4m3_pack4(elem(4 * r4) * sc, elem(4 * r4 + 1) * sc, elem(4 * r4 + 2) * sc, elem(4 * r4 + 3) * sc);
    // (transposed copy: this lane's column, 32 bytes, straight to its row of qt)
    uint4* dst = reinterpret_cast<uint4*>(p.qt_codes + (long long)(ocol + lane) * p.rows_cap + y);
    dst[0] = make_uint4(t[0], t[1], t[2], t[3]);
    dst[1] = make_uint4(t[4], t[5], t[6], t[7]);
    p.qt_sf[mx_sf_offset(ocol + lane, y >> 5, p.rows_cap >> 7)] = static_cast<uint8_t>(et + 127);
  }
  if (want_q) {
    // (row copy: this lane's 32 bytes straight to its row)
    float v[32];
    #pragma unroll
    for (int i = 0; i < 16; ++i) {
      v[2 * i] = bf16_lo(o[i]);
      v[2 * i + 1] = bf16_hi(o[i]);
    }
    const int eq = mx_exponent(amax32(v));
    uint32_t w[8];
    e4m3_pack32(v, pow2_neg(eq), w);
    uint4* d = reinterpret_cast<uint4*>(p.q_codes + (long long)(y + lane) * p.ld_q + ocol);
    d[0] = make_uint4(w[0], w[1], w[2], w[3]);
    d[1] = make_uint4(w[4], w[5], w[6], w[7]);
    p.q_sf[mx_sf_offset(y + lane, ocol >> 5, p.ld_q >> 7)] = static_cast<uint8_t>(eq + 127);
  }
  if (tm != nullptr) st.flush(tm, ocol, y);     // the bf16 chunk
}

__device__ __forceinline__ void load32(uint32_t taddr, uint32_t (&a)[16], uint32_t (&b)[16]) {
  tmem_ld_x16(taddr, a);
  tmem_ld_x16(taddr + 16, b);
  tmem_ld_wait(a);
  tmem_ld_wait(b);
}

// Factor `al` the epilogue applies to the accumulator before its arithmetic:
// NVFP4 GEMMs multiply the block-scaled codes, so the tensor scales 1/S_a and
// 1/S_b are still owed; 1 otherwise.  Computed once per CTA.
template <class C>
__device__ __forceinline__ float acc_scale(const GemmParams& p) {
  if constexpr (C::NV4) {
    return (1.0f / nv4_tensor_scale(*p.amax_a)) * (1.0f / nv4_tensor_scale(*p.amax_b));
  } else {
    return 1.0f;
  }
}

// |h'| maximum of packed bf16 pairs, folded into a warp maximum and one
// atomicMax per warp (NaN inputs are ignored by fmaxf).
__device__ __forceinline__ float amax_bf16x2(float m, uint32_t w) {
  return fmaxf(m, fmaxf(fabsf(bf16_lo(w)), fabsf(bf16_hi(w))));
}
__device__ __forceinline__ void amax_flush(unsigned* out, float m, int lane) {
  const unsigned u = __reduce_max_sync(0xffffffffu, __float_as_uint(m));
  if (lane == 0) atomicMax(out, u);
}

__device__ __forceinline__ void add8_bf16(float (&acc)[8], const uint4& v) {
  acc[0] += bf16_lo(v.x); acc[1] += bf16_hi(v.x);
  acc[2] += bf16_lo(v.y); acc[3] += bf16_hi(v.y);
  acc[4] += bf16_lo(v.z); acc[5] += bf16_hi(v.z);
  acc[6] += bf16_lo(v.w); acc[7] += bf16_hi(v.w);
}

// The combine fused into fc2's epilogue (GemmParams::cmb_*), for this warp's
// 32 rows (y0 .. y0+31) of N tile n, once their TMA stores have been issued.
// Every row of a tile belongs to a different token (a token picks an expert at
// most once), so a lane's counter is its own.  The sum runs in slot order
// whichever tile arrives last, so y is the same bits on every run.
template <int NBUF>
__device__ __forceinline__ void fused_combine_rows(const GemmParams& p, int y0, int n, int lane,
                                                   Stager<NBUF, 4096>& st) {
  st.drain();                                   // lane 0: this warp's stores of o are complete
  if (lane == 0) fence_proxy_async_global();
  __syncwarp();
  const int r = y0 + lane;
  const int t = (r < p.rows_cap) ? p.cmb_row_src[r] : -1;
  const int k = p.cmb_k;
  bool last = false;
  if (t >= 0) {
    int valid = 0;
    for (int i = 0; i < k; ++i) valid += p.cmb_slot_row[(long long)t * k + i] >= 0 ? 1 : 0;
    __threadfence();                            // o's rows before the count others act on
    last = atomicAdd(p.cmb_count + (long long)t * p.n_tiles + n, 1) + 1 == valid;
  }
  unsigned todo = __ballot_sync(0xffffffffu, last);
  if (todo == 0) return;
  __threadfence();                              // the other tiles' rows after their counts
  const long long ld = p.ldc;
  const int col = n * 256 + 8 * lane;           // 8 columns (16 bytes) per lane
  const __nv_bfloat16* o = static_cast<const __nv_bfloat16*>(p.c);
  while (todo != 0) {
    const int src = __ffs(todo) - 1;
    todo &= todo - 1;
    const int tt = __shfl_sync(0xffffffffu, t, src);
    // lane i < k holds slot i's row; the rows are loaded 8 at a time (all in
    // flight together) and added in slot order
    const int my_row = (lane < k) ? p.cmb_slot_row[(long long)tt * k + lane] : -1;
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    uint4 sv = make_uint4(0, 0, 0, 0);
    if (p.cmb_shared != nullptr) sv = __ldg(reinterpret_cast<const uint4*>(p.cmb_shared + tt * ld + col));
    for (int i0 = 0; i0 < k; i0 += 8) {
      uint4 v[8];
      int rr[8];
      #pragma unroll
      for (int j = 0; j < 8; ++j) {
        rr[j] = __shfl_sync(0xffffffffu, my_row, (i0 + j) & 31);
        if (i0 + j >= k) rr[j] = -1;
        v[j] = rr[j] >= 0 ? __ldcg(reinterpret_cast<const uint4*>(o + rr[j] * ld + col)) : make_uint4(0, 0, 0, 0);
      }
      #pragma unroll
      for (int j = 0; j < 8; ++j)
        if (rr[j] >= 0) add8_bf16(acc, v[j]);
    }
    if (p.cmb_shared != nullptr) add8_bf16(acc, sv);
    *reinterpret_cast<uint4*>(p.cmb_y + tt * ld + col) =
        make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]), pack_bf16x2(acc[4], acc[5]),
                   pack_bf16x2(acc[6], acc[7]));
    if (lane == src) p.cmb_count[(long long)tt * p.n_tiles + n] = 0;   // ready for the next launch
  }
}

// Epilogue with TMA stores.  Rows of the tile: warp quarter q owns rows
// 32q..32q+31, lane = row.  Dense tiles past the last row are clipped by TMA.
template <class C>
__device__ __forceinline__ void epilogue_tile_tma(const GemmParams& p, const TileInfo& ti, uint32_t tmem_acc,
                                                  int quarter, int lane,
                                                  Stager<C::STAGING_BUFS, C::STAGING_BUF>& st,
                                                  const CUtensorMap* tmC,
                                                  const CUtensorMap* tmC2,
                                                  uint64_t* release_bar = nullptr, bool* released = nullptr,
                                                  const float al = 1.0f, const int cpart = 0) {
  const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
  const uint32_t t0 = tmem_acc + lane_addr;
  const bool no_mma = (ti.num_kb == 0);         // empty group (weight gradients): result is zero

  if constexpr (C::EP == Epi::kStoreF32) {      // weight gradients: [group*M + row, col] fp32
    const int y = ti.group * p.m_rows + ti.m0 + quarter * 32;
    if constexpr (C::ACC_BUFS == 1 && C::BN == 256 && C::STAGING_BUFS >= 4) {
      if (release_bar != nullptr) {
        // Single accumulator: columns 0..127 go straight into the four staging
        // buffers (their stores start at once), columns 128..255 into
        // registers; then the accumulator is handed back and the rest stored.
        #pragma unroll 1
        for (int c0 = 0; c0 < 128; c0 += 32) {
          uint32_t a[16], b[16];
          load32(t0 + c0, a, b);
          st.begin();
          #pragma unroll
          for (int j = 0; j < 4; ++j) st.put(j, no_mma ? 0u : a[4 * j], no_mma ? 0u : a[4 * j + 1],
                                            no_mma ? 0u : a[4 * j + 2], no_mma ? 0u : a[4 * j + 3]);
          #pragma unroll
          for (int j = 0; j < 4; ++j) st.put(4 + j, no_mma ? 0u : b[4 * j], no_mma ? 0u : b[4 * j + 1],
                                            no_mma ? 0u : b[4 * j + 2], no_mma ? 0u : b[4 * j + 3]);
          st.flush(tmC, ti.n * C::BN + c0, y);
        }
        uint32_t keep[128];
        #pragma unroll
        for (int h = 0; h < 8; ++h) {
          uint32_t v[16];
          tmem_ld_x16(t0 + 128 + 16 * h, v);
          tmem_ld_wait(v);
          #pragma unroll
          for (int j = 0; j < 16; ++j) keep[16 * h + j] = no_mma ? 0u : v[j];
        }
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(release_bar);
        *released = true;
        #pragma unroll
        for (int c = 0; c < 4; ++c) {
          st.begin();
          #pragma unroll
          for (int j = 0; j < 8; ++j) {
            const uint32_t* w = keep + 32 * c + 4 * j;
            st.put(j, w[0], w[1], w[2], w[3]);
          }
          st.flush(tmC, ti.n * C::BN + 128 + 32 * c, y);
        }
        return;
      }
    }
    if constexpr (C::S == Sched::kRoutedK) {
      if (p.c_trans) {
        // transposed: the 32 x 32 block (rows y.., columns c0..) goes to the
        // staging as 32 rows of one column each (row j = column c0 + j, 128
        // bytes, 16-byte chunks in the 128-byte swizzled order; lane = element
        // within the row, so each store of the warp hits 32 distinct banks)
        // and from there to rows group * N + n0 + c0.. of the [E * N, M] output
        const uint32_t lane_off = static_cast<uint32_t>((lane & 3) * 4);
        const uint32_t lane_chunk = static_cast<uint32_t>(lane >> 2);
        #pragma unroll 1
        for (int c0 = 0; c0 < C::BN; c0 += 32) {
          uint32_t a[16], b[16];
          load32(t0 + c0, a, b);
          st.begin();
          const uint32_t base = smem_u32(st.buf + st.cur * C::STAGING_BUF);
          #pragma unroll
          for (int j = 0; j < 16; ++j)
            st_shared_u32(base + j * 128 + ((lane_chunk ^ (j & 7)) << 4) + lane_off, no_mma ? 0u : a[j]);
          #pragma unroll
          for (int j = 0; j < 16; ++j)
            st_shared_u32(base + (16 + j) * 128 + ((lane_chunk ^ (j & 7)) << 4) + lane_off, no_mma ? 0u : b[j]);
          st.flush(tmC, ti.m0 + quarter * 32, ti.group * p.n_tiles * C::BN + ti.n * C::BN + c0);
        }
        return;
      }
    }
    #pragma unroll 1
    for (int c0 = 0; c0 < C::BN; c0 += 32) {
      uint32_t a[16], b[16];
      load32(t0 + c0, a, b);
      st.begin();
      #pragma unroll
      for (int j = 0; j < 4; ++j) st.put(j, no_mma ? 0u : a[4 * j], no_mma ? 0u : a[4 * j + 1],
                                        no_mma ? 0u : a[4 * j + 2], no_mma ? 0u : a[4 * j + 3]);
      #pragma unroll
      for (int j = 0; j < 4; ++j) st.put(4 + j, no_mma ? 0u : b[4 * j], no_mma ? 0u : b[4 * j + 1],
                                        no_mma ? 0u : b[4 * j + 2], no_mma ? 0u : b[4 * j + 3]);
      st.flush(tmC, ti.n * C::BN + c0, y);
    }
  } else if constexpr (C::EP == Epi::kStoreBf16) {
    const int y = ti.m0 + quarter * 32;
    if constexpr (C::BN == 224) {
      // 256 x 224 tiles (one accumulator): this row's 224 outputs as bf16 pairs
      // in registers, the accumulator handed back, then three 64-column stores
      // through the swizzled staging and the last 32 columns through tmC2
      // (64-byte rows, no swizzle)
      uint32_t pk[112];
      #pragma unroll
      for (int h = 0; h < 14; h += 2) {
        uint32_t v[2][16];
        tmem_ld_x16(t0 + 16 * h, v[0]);
        tmem_ld_x16(t0 + 16 * (h + 1), v[1]);
        tmem_ld_wait(v[0]);
        tmem_ld_wait(v[1]);
        #pragma unroll
        for (int u = 0; u < 2; ++u)
          #pragma unroll
          for (int j = 0; j < 8; ++j)
            pk[8 * (h + u) + j] = pack_bf16x2(__uint_as_float(v[u][2 * j]) * al,
                                              __uint_as_float(v[u][2 * j + 1]) * al);
      }
      tc_fence_before_sync();
      __syncwarp();
      if (release_bar != nullptr) {
        if (lane == 0) mbar_arrive(release_bar);
        *released = true;
      }
      #pragma unroll
      for (int c = 0; c < 3; ++c) {
        st.begin();
        #pragma unroll
        for (int q = 0; q < 8; ++q) {
          const uint32_t* w = pk + 32 * c + 4 * q;
          st.put(q, w[0], w[1], w[2], w[3]);
        }
        st.flush(tmC, ti.n * C::BN + 64 * c, y);
      }
      st.begin();
      #pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint32_t* w = pk + 96 + 4 * q;
        st.put_rows64(q, w[0], w[1], w[2], w[3]);
      }
      st.flush(tmC2, ti.n * C::BN + 192, y);
    } else {
    if constexpr ((C::M256 || C::ACC_BUFS == 1) && C::BN == 256) {
      if (release_bar != nullptr) {
        // (single accumulator) this row's 256 outputs as bf16 pairs in registers, the accumulator
        // handed back to the MMA warp, then the stores
        uint32_t pk[128];
        #pragma unroll
        for (int h = 0; h < 16; h += 2) {
          uint32_t v[2][16];
          tmem_ld_x16(t0 + 16 * h, v[0]);
          tmem_ld_x16(t0 + 16 * (h + 1), v[1]);
          tmem_ld_wait(v[0]);
          tmem_ld_wait(v[1]);
          #pragma unroll
          for (int u = 0; u < 2; ++u)
            #pragma unroll
            for (int j = 0; j < 8; ++j)
              pk[8 * (h + u) + j] = pack_bf16x2(__uint_as_float(v[u][2 * j]) * al,
                                                __uint_as_float(v[u][2 * j + 1]) * al);
        }
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(release_bar);
        *released = true;
        #pragma unroll
        for (int c = 0; c < 4; ++c) {                // 64-column chunks
          st.begin();
          #pragma unroll
          for (int q = 0; q < 8; ++q) {
            const uint32_t* w = pk + 32 * c + 4 * q;
            st.put(q, w[0], w[1], w[2], w[3]);
          }
          st.flush(tmC, ti.n * C::BN + 64 * c, y);
        }
        if constexpr (C::S == Sched::kRoutedM) {
          if (p.cmb_y != nullptr) fused_combine_rows(p, y, ti.n, lane, st);
        }
        return;
      }
    }
    #pragma unroll 1
    for (int c0 = 0; c0 < C::BN; c0 += 64) {
      uint32_t v[4][16];                        // 64 columns in one TMEM round trip
      #pragma unroll
      for (int h = 0; h < 4; ++h) tmem_ld_x16(t0 + c0 + 16 * h, v[h]);
      #pragma unroll
      for (int h = 0; h < 4; ++h) tmem_ld_wait(v[h]);
      st.begin();
      #pragma unroll
      for (int h = 0; h < 4; ++h) {
        uint32_t w[8];
        #pragma unroll
        for (int j = 0; j < 8; ++j)
          w[j] = pack_bf16x2(__uint_as_float(v[h][2 * j]) * al, __uint_as_float(v[h][2 * j + 1]) * al);
        st.put(2 * h, w[0], w[1], w[2], w[3]);
        st.put(2 * h + 1, w[4], w[5], w[6], w[7]);
      }
      st.flush(tmC, ti.n * C::BN + c0, y);
    }
    if constexpr (C::S == Sched::kRoutedM && C::BN == 256) {
      if (p.cmb_y != nullptr) fused_combine_rows(p, y, ti.n, lane, st);
    }
    }
  } else if constexpr (C::EP == Epi::kSwiglu && C::SPLIT_FWD) {
    // gated SwiGLU on 8 warps: this warp's 64 columns of h' (half cpart of the
    // tile's 128) -- its 64 gate and 64 up accumulator columns -- to
    // registers, the accumulator handed back, then per 32 columns:
    // h' = g * silu(a) * b, the saved z chunks (gate, up) and h' itself (bf16
    // through tmC, and/or its MXFP8 copies) through the 2 KB staging
    // (32-column boxes, 64-byte swizzle)
    const int row = ti.m0 + quarter * 32 + lane;
    const bool row_ok = (C::S != Sched::kDenseM) || (row < p.m_rows);
    const float g = (p.row_gate != nullptr && row_ok) ? p.row_gate[row] : 1.0f;
    const int colh = ti.n * (C::BN / 2) + 64 * cpart;
    const int y = ti.m0 + quarter * 32;
    uint32_t ga[64], ua[64];
    #pragma unroll
    for (int h = 0; h < 4; ++h) {
      uint32_t a[16], b[16];
      tmem_ld_x16(t0 + 64 * cpart + 16 * h, a);
      tmem_ld_x16(t0 + C::BN / 2 + 64 * cpart + 16 * h, b);
      tmem_ld_wait(a);
      tmem_ld_wait(b);
      #pragma unroll
      for (int j = 0; j < 16; ++j) {
        ga[16 * h + j] = a[j];
        ua[16 * h + j] = b[j];
      }
    }
    tc_fence_before_sync();
    __syncwarp();
    if (release_bar != nullptr) {
      if (lane == 0) mbar_arrive(release_bar);
      *released = true;
    }
    #pragma unroll
    for (int c = 0; c < 2; ++c) {
      uint32_t hp[16], zg[16], zu[16];
      #pragma unroll
      for (int j = 0; j < 16; ++j) {
        const float a0 = __uint_as_float(ga[32 * c + 2 * j]) * al, a1 = __uint_as_float(ga[32 * c + 2 * j + 1]) * al;
        const float b0 = __uint_as_float(ua[32 * c + 2 * j]) * al, b1 = __uint_as_float(ua[32 * c + 2 * j + 1]) * al;
        hp[j] = pack_bf16x2(g * __fdividef(a0, 1.0f + __expf(-a0)) * b0, g * __fdividef(a1, 1.0f + __expf(-a1)) * b1);
        zg[j] = pack_bf16x2(a0, a1);
        zu[j] = pack_bf16x2(b0, b1);
      }
      if (p.c2 != nullptr) {
        emit_chunk32(p, st, zg, colh + 32 * c, y, lane, tmC2, false);
        emit_chunk32(p, st, zu, p.half_cols + colh + 32 * c, y, lane, tmC2, false);
      }
      emit_chunk32(p, st, hp, colh + 32 * c, y, lane, p.c != nullptr ? tmC : nullptr, true);
    }
  } else if constexpr (C::EP == Epi::kSwiglu) {
    // accumulator columns [0, BN/2) = gate rows of W1, [BN/2, BN) = the matching up rows
    const int row = ti.m0 + quarter * 32 + lane;
    const bool row_ok = (C::S != Sched::kDenseM) || (row < p.m_rows);
    const float g = (p.row_gate != nullptr && row_ok) ? p.row_gate[row] : 1.0f;
    const int col0 = ti.n * (C::BN / 2);
    const int y = ti.m0 + quarter * 32;
    if constexpr (C::BN == 256 && C::ACC_BUFS == 1 && !C::M256) {
      if (p.c2 != nullptr && release_bar != nullptr) {
        // Single accumulator, z saved: h' and both halves of z for this row's
        // 128 columns (64 when the columns are split over two warps) go to
        // registers (bf16 pairs), the accumulator is handed back, then
        // everything is stored.
        constexpr int NQ = C::SPLIT_COLS ? 4 : 8;   // 16-column groups of h' this warp owns
        const int q0 = C::SPLIT_COLS ? 4 * cpart : 0;
        uint32_t hp[8 * NQ], zg[8 * NQ], zu[8 * NQ];
        #pragma unroll
        for (int q = 0; q < NQ; ++q) {
          uint32_t a[16], b[16];
          tmem_ld_x16(t0 + 16 * (q0 + q), a);
          tmem_ld_x16(t0 + C::BN / 2 + 16 * (q0 + q), b);
          tmem_ld_wait(a);
          tmem_ld_wait(b);
          #pragma unroll
          for (int j = 0; j < 8; ++j) {
            const float a0 = __uint_as_float(a[2 * j]) * al, a1 = __uint_as_float(a[2 * j + 1]) * al;
            const float b0 = __uint_as_float(b[2 * j]) * al, b1 = __uint_as_float(b[2 * j + 1]) * al;
            hp[8 * q + j] = pack_bf16x2(g * __fdividef(a0, 1.0f + __expf(-a0)) * b0,
                                        g * __fdividef(a1, 1.0f + __expf(-a1)) * b1);
            zg[8 * q + j] = pack_bf16x2(a0, a1);
            zu[8 * q + j] = pack_bf16x2(b0, b1);
          }
        }
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(release_bar);
        *released = true;
        if constexpr (C::NV4) {
          if (p.amax_out != nullptr) {
            float m = 0.f;
            #pragma unroll
            for (int i = 0; i < 8 * NQ; ++i) m = amax_bf16x2(m, hp[i]);
            amax_flush(p.amax_out, m, lane);
          }
        }
        #pragma unroll
        for (int c = 0; c < NQ / 4; ++c) {          // 64-column chunks: h', z gate, z up
          const int cc = q0 / 4 + c;
          st.begin();
          #pragma unroll
          for (int q = 0; q < 8; ++q) st.put(q, hp[32 * c + 4 * q], hp[32 * c + 4 * q + 1], hp[32 * c + 4 * q + 2],
                                            hp[32 * c + 4 * q + 3]);
          st.flush(tmC, col0 + 64 * cc, y);
          st.begin();
          #pragma unroll
          for (int q = 0; q < 8; ++q) st.put(q, zg[32 * c + 4 * q], zg[32 * c + 4 * q + 1], zg[32 * c + 4 * q + 2],
                                            zg[32 * c + 4 * q + 3]);
          st.flush(tmC2, col0 + 64 * cc, y);
          st.begin();
          #pragma unroll
          for (int q = 0; q < 8; ++q) st.put(q, zu[32 * c + 4 * q], zu[32 * c + 4 * q + 1], zu[32 * c + 4 * q + 2],
                                            zu[32 * c + 4 * q + 3]);
          st.flush(tmC2, p.half_cols + col0 + 64 * cc, y);
        }
        return;
      }
    }
    if constexpr (C::BN == 256) {
      if (p.c2 == nullptr && release_bar != nullptr) {
        // Forward without saved z: compute this row's 128 values of h' into
        // registers, hand the accumulator back to the MMA warp, then store.
        constexpr int NQ = C::SPLIT_COLS ? 4 : 8;   // 16-column groups of h' this warp owns
        const int q0 = C::SPLIT_COLS ? 4 * cpart : 0;
        uint32_t hp[8 * NQ];                        // packed bf16 pairs
        #pragma unroll
        for (int qq = 0; qq < NQ; qq += 2) {
          uint32_t av[2][16], bv[2][16];
          #pragma unroll
          for (int u = 0; u < 2; ++u) {
            tmem_ld_x16(t0 + 16 * (q0 + qq + u), av[u]);
            tmem_ld_x16(t0 + C::BN / 2 + 16 * (q0 + qq + u), bv[u]);
          }
          #pragma unroll
          for (int u = 0; u < 2; ++u) {
            tmem_ld_wait(av[u]);
            tmem_ld_wait(bv[u]);
          }
          #pragma unroll
          for (int u = 0; u < 2; ++u) {
            #pragma unroll
            for (int j = 0; j < 8; ++j) {
              const float a0 = __uint_as_float(av[u][2 * j]) * al, a1 = __uint_as_float(av[u][2 * j + 1]) * al;
              const float b0 = __uint_as_float(bv[u][2 * j]) * al, b1 = __uint_as_float(bv[u][2 * j + 1]) * al;
              hp[8 * (qq + u) + j] = pack_bf16x2(g * __fdividef(a0, 1.0f + __expf(-a0)) * b0,
                                                 g * __fdividef(a1, 1.0f + __expf(-a1)) * b1);
            }
          }
        }
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(release_bar);
        *released = true;
        if constexpr (C::NV4) {
          if (p.amax_out != nullptr) {
            float m = 0.f;
            #pragma unroll
            for (int i = 0; i < 8 * NQ; ++i) m = amax_bf16x2(m, hp[i]);
            amax_flush(p.amax_out, m, lane);
          }
        }
        #pragma unroll
        for (int c = 0; c < NQ / 4; ++c) {          // 64-column chunks
          st.begin();
          #pragma unroll
          for (int q = 0; q < 4; ++q) {
            const uint32_t* w = hp + 8 * (4 * c + q);
            st.put(2 * q, w[0], w[1], w[2], w[3]);
            st.put(2 * q + 1, w[4], w[5], w[6], w[7]);
          }
          st.flush(tmC, col0 + 64 * (q0 / 4 + c), y);
        }
        return;
      }
    }
    float hmax = 0.f;
    #pragma unroll 1
    for (int c0 = 0; c0 < C::BN / 2; c0 += 64) {
      if (C::SPLIT_COLS && c0 != 64 * cpart) continue;   // the other warp of this lane quarter has it
      st.begin();
      #pragma unroll 1
      for (int qq = 0; qq < 4; qq += 2) {
       uint32_t av[2][16], bv[2][16];            // two 16-column groups per TMEM round trip
       #pragma unroll
       for (int u = 0; u < 2; ++u) {
         tmem_ld_x16(t0 + c0 + 16 * (qq + u), av[u]);
         tmem_ld_x16(t0 + C::BN / 2 + c0 + 16 * (qq + u), bv[u]);
       }
       #pragma unroll
       for (int u = 0; u < 2; ++u) {
         tmem_ld_wait(av[u]);
         tmem_ld_wait(bv[u]);
       }
       #pragma unroll
       for (int u = 0; u < 2; ++u) {
        const int q = qq + u;
        const uint32_t* a = av[u];
        const uint32_t* b = bv[u];
        uint32_t hw[8];
        #pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float a0 = __uint_as_float(a[2 * j]) * al, a1 = __uint_as_float(a[2 * j + 1]) * al;
          const float b0 = __uint_as_float(b[2 * j]) * al, b1 = __uint_as_float(b[2 * j + 1]) * al;
          // silu(a) = a / (1 + e^-a) with the fast exponential and divide: their
          // relative error (~1e-6) is far below the bf16 rounding of h
          hw[j] = pack_bf16x2(g * __fdividef(a0, 1.0f + __expf(-a0)) * b0,
                              g * __fdividef(a1, 1.0f + __expf(-a1)) * b1);
        }
        if constexpr (C::NV4) {
          #pragma unroll
          for (int j = 0; j < 8; ++j) hmax = amax_bf16x2(hmax, hw[j]);
        }
        st.put(2 * q, hw[0], hw[1], hw[2], hw[3]);
        st.put(2 * q + 1, hw[4], hw[5], hw[6], hw[7]);
       }
      }
      st.flush(tmC, col0 + c0, y);
      if (p.c2 != nullptr) {                    // z, saved for backward: gate chunk then up chunk
        #pragma unroll 1
        for (int half = 0; half < 2; ++half) {
          st.begin();
          #pragma unroll
          for (int h2 = 0; h2 < 2; ++h2) {
            uint32_t a[16], b[16];
            load32(t0 + half * (C::BN / 2) + c0 + 32 * h2, a, b);
            uint32_t w[16];
            #pragma unroll
            for (int j = 0; j < 8; ++j)
              w[j] = pack_bf16x2(__uint_as_float(a[2 * j]) * al, __uint_as_float(a[2 * j + 1]) * al);
            #pragma unroll
            for (int j = 0; j < 8; ++j)
              w[8 + j] = pack_bf16x2(__uint_as_float(b[2 * j]) * al, __uint_as_float(b[2 * j + 1]) * al);
            #pragma unroll
            for (int j = 0; j < 4; ++j) st.put(4 * h2 + j, w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
          }
          st.flush(tmC2, half * p.half_cols + col0 + c0, y);
        }
      }
    }
    if constexpr (C::NV4) {
      if (p.amax_out != nullptr) amax_flush(p.amax_out, hmax, lane);
    }
  } else if constexpr (C::SPLIT_BWD) {
    // kSwigluBwd on 8 warps: this warp's 128 columns of dh (half cpart of the
    // tile) to registers, the accumulator handed back, then per 32 columns the
    // saved z, the SwiGLU backward and the dz gate and up chunks through the
    // 2 KB staging (tmC2: 32-column boxes, 64-byte swizzle); one partial
    // <dh, silu(a) b> per warp (its 128 columns)
    const int row = ti.m0 + quarter * 32 + lane;
    const bool row_ok = (C::S != Sched::kDenseM) || (row < p.m_rows);
    const float g = (p.row_gate != nullptr && row_ok) ? p.row_gate[row] : 1.0f;
    const int colw = ti.n * C::BN + 128 * cpart;
    const int y = ti.m0 + quarter * 32;
    const int parts = p.n_tiles * (C::BN / 128);
    uint32_t dh[128];
    #pragma unroll
    for (int h = 0; h < 8; h += 2) {
      uint32_t v[2][16];
      tmem_ld_x16(t0 + 128 * cpart + 16 * h, v[0]);
      tmem_ld_x16(t0 + 128 * cpart + 16 * (h + 1), v[1]);
      tmem_ld_wait(v[0]);
      tmem_ld_wait(v[1]);
      #pragma unroll
      for (int u = 0; u < 2; ++u)
        #pragma unroll
        for (int j = 0; j < 16; ++j) dh[16 * (h + u) + j] = no_mma ? 0u : v[u][j];
    }
    tc_fence_before_sync();
    __syncwarp();
    if (release_bar != nullptr) {
      if (lane == 0) mbar_arrive(release_bar);
      *released = true;
    }
    const __nv_bfloat16* zrow = p.aux + (long long)(row_ok ? row : 0) * p.ld_aux + colw;
    float dg = 0.f;
    #pragma unroll
    for (int c = 0; c < 4; ++c) {
      uint4 za[4], zb[4];
      #pragma unroll
      for (int i = 0; i < 4; ++i) {
        za[i] = reinterpret_cast<const uint4*>(zrow + 32 * c)[i];
        zb[i] = reinterpret_cast<const uint4*>(zrow + p.half_cols + 32 * c)[i];
      }
      uint32_t og[16], ou[16];
      #pragma unroll
      for (int j = 0; j < 16; ++j) {
        const uint4& a4 = za[j >> 2];
        const uint4& b4 = zb[j >> 2];
        const uint32_t zaw = (j & 3) == 0 ? a4.x : (j & 3) == 1 ? a4.y : (j & 3) == 2 ? a4.z : a4.w;
        const uint32_t zbw = (j & 3) == 0 ? b4.x : (j & 3) == 1 ? b4.y : (j & 3) == 2 ? b4.z : b4.w;
        float g2[2], u2[2];
        #pragma unroll
        for (int u = 0; u < 2; ++u) {
          const float av = u ? bf16_hi(zaw) : bf16_lo(zaw);
          const float bv = u ? bf16_hi(zbw) : bf16_lo(zbw);
          const float dhv = __uint_as_float(dh[32 * c + 2 * j + u]);
          // sigmoid with the fast exponential and divide (relative error ~1e-6)
          const float sg = __fdividef(1.0f, 1.0f + __expf(-av));
          const float si = av * sg;
          const float dhg = g * dhv;
          dg += dhv * si * bv;
          g2[u] = dhg * bv * sg * (1.0f + av * (1.0f - sg));   // d(gate input)
          u2[u] = dhg * si;                                  // d(up input)
        }
        og[j] = pack_bf16x2(g2[0], g2[1]);
        ou[j] = pack_bf16x2(u2[0], u2[1]);
      }
      const CUtensorMap* tm = (p.c != nullptr) ? tmC2 : nullptr;
      emit_chunk32(p, st, og, colw + 32 * c, y, lane, tm);
      emit_chunk32(p, st, ou, p.half_cols + colw + 32 * c, y, lane, tm);
    }
    if (row_ok && p.dgate_part != nullptr) p.dgate_part[(long long)row * parts + colw / 128] = dg;
  } else {  // kSwigluBwd: dz gate and up chunks of each 64 columns in one pass
    static_assert(C::STAGING_BUFS == 2 || C::STAGING_BUFS == 1, "gate and up chunks: two buffers, or one");
    const int row = ti.m0 + quarter * 32 + lane;
    const bool row_ok = (C::S != Sched::kDenseM) || (row < p.m_rows);
    const float g = (p.row_gate != nullptr && row_ok) ? p.row_gate[row] : 1.0f;
    const int col0 = ti.n * C::BN;
    const __nv_bfloat16* zrow = p.aux + (long long)(row_ok ? row : 0) * p.ld_aux + col0;
    const int y = ti.m0 + quarter * 32;
    const int parts = p.n_tiles * (C::BN / 128);   // partials per row: one per 128 columns of dh
    float dg = 0.f;
    #pragma unroll 1
    for (int c0 = 0; c0 < C::BN; c0 += 64) {
      // this row's saved z for the 64 columns (gate and up), loaded before the TMEM reads
      uint4 za[8], zb[8];
      #pragma unroll
      for (int i = 0; i < 8; ++i) {
        za[i] = reinterpret_cast<const uint4*>(zrow + c0)[i];
        zb[i] = reinterpret_cast<const uint4*>(zrow + p.half_cols + c0)[i];
      }
      st.begin_all();
      uint32_t up_keep[C::STAGING_BUFS == 1 ? 32 : 1];   // one buffer: the up chunk waits here
      #pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint32_t v[16];
        tmem_ld_x16(t0 + c0 + 16 * q, v);
        tmem_ld_wait(v);
        const uint32_t zaw[8] = {za[2 * q].x, za[2 * q].y, za[2 * q].z, za[2 * q].w,
                                 za[2 * q + 1].x, za[2 * q + 1].y, za[2 * q + 1].z, za[2 * q + 1].w};
        const uint32_t zbw[8] = {zb[2 * q].x, zb[2 * q].y, zb[2 * q].z, zb[2 * q].w,
                                 zb[2 * q + 1].x, zb[2 * q + 1].y, zb[2 * q + 1].z, zb[2 * q + 1].w};
        uint32_t og[8], ou[8];
        #pragma unroll
        for (int j = 0; j < 8; ++j) {
          float g2[2], u2[2];
          #pragma unroll
          for (int u = 0; u < 2; ++u) {
            const float av = u ? bf16_hi(zaw[j]) : bf16_lo(zaw[j]);
            const float bv = u ? bf16_hi(zbw[j]) : bf16_lo(zbw[j]);
            const float dh = no_mma ? 0.f : __uint_as_float(v[2 * j + u]);
            // sigmoid with the fast exponential and divide (relative error ~1e-6)
            const float sg = __fdividef(1.0f, 1.0f + __expf(-av));
            const float si = av * sg;
            const float dhg = g * dh;
            dg += dh * si * bv;
            g2[u] = dhg * bv * sg * (1.0f + av * (1.0f - sg));   // d(gate input)
            u2[u] = dhg * si;                                  // d(up input)
          }
          og[j] = pack_bf16x2(g2[0], g2[1]);
          ou[j] = pack_bf16x2(u2[0], u2[1]);
        }
        st.put(2 * q, og[0], og[1], og[2], og[3]);
        st.put(2 * q + 1, og[4], og[5], og[6], og[7]);
        if constexpr (C::STAGING_BUFS == 2) {
          st.put_next(2 * q, ou[0], ou[1], ou[2], ou[3]);
          st.put_next(2 * q + 1, ou[4], ou[5], ou[6], ou[7]);
        } else {
          #pragma unroll
          for (int j = 0; j < 8; ++j) up_keep[8 * q + j] = ou[j];
        }
      }
      st.flush(tmC, col0 + c0, y);                  // gate chunk (current buffer)
      if constexpr (C::STAGING_BUFS == 1) {
        st.begin();                                 // the gate chunk's store has read the buffer
        #pragma unroll
        for (int q = 0; q < 4; ++q) {
          st.put(2 * q, up_keep[8 * q], up_keep[8 * q + 1], up_keep[8 * q + 2], up_keep[8 * q + 3]);
          st.put(2 * q + 1, up_keep[8 * q + 4], up_keep[8 * q + 5], up_keep[8 * q + 6], up_keep[8 * q + 7]);
        }
      }
      st.flush(tmC, p.half_cols + col0 + c0, y);    // up chunk (the next buffer, or the same one again)
      if ((c0 & 127) == 64) {                       // one partial <dh, silu(a) b> per 128 columns
        if (row_ok && p.dgate_part != nullptr) p.dgate_part[(long long)row * parts + (col0 + c0) / 128] = dg;
        dg = 0.f;
      }
    }

  }
}

// Tiles are handed out in index order from a counter in global memory: the
// producer takes the next index with one atomicAdd per tile, so tiles that
// share an expert's weight panel (consecutive indices) start at about the same
// time on different SMs and the panel is read from HBM once, not once per
// tile.  The producer passes each index to the MMA and epilogue warps through
// a small ring in shared memory; -1 ends the list.  The last CTA to finish
// puts the counter back to zero for the next launch.
constexpr int kSchedDepth = 4;

// Barriers and per-launch tables, kept at the end of dynamic shared memory.
template <class C>
struct GemmBook {
  uint64_t sched_full[kSchedDepth];
  uint64_t sched_empty[kSchedDepth];
  uint64_t full_bar[C::STAGES];
  uint64_t empty_bar[C::STAGES];
  uint64_t tfull_bar[C::ACC_BUFS];
  uint64_t tempty_bar[C::ACC_BUFS];
  uint64_t drain_bar;
  uint32_t tmem_slot;
  int abort_flag;
  int bad;
  int sched_tile[kSchedDepth];
  int poff[257];
  int tpre[C::ROWS256 ? 257 : 1];
};

// Called once per CTA after its producer took its last tile index.
__device__ __forceinline__ void sched_finish(int* sched) {
  if (sched == nullptr) return;
  __threadfence();
  if (atomicAdd(sched + 1, 1) == static_cast<int>(gridDim.x) - 1) {
    atomicExch(sched, 0);
    atomicExch(sched + 1, 0);
  }
}

template <class C>
__global__ void __launch_bounds__(C::THREADS, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmC2,
                        const GemmParams p) {
  pdl_wait();
  static_assert(sizeof(GemmBook<C>) <= C::BOOK_BYTES, "bookkeeping size");
  static_assert(!C::PAIR, "CTA-pair tiles run in grouped_gemm_pair_kernel");
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  {
    // the ring needs a 1024-byte aligned base inside the allocation
    const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
    if (pad + C::SMEM_USED > static_cast<uint32_t>(C::SMEM_BYTES)) {
      if (threadIdx.x == 0) {
        set_status(p.status, kErrLaunch);
        sched_finish(p.sched);
      }
      return;
    }
  }
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* a_smem = smem;
  uint8_t* b_smem = smem + C::STAGES * C::A_BYTES;
  uint8_t* sf_smem = b_smem + C::STAGES * C::B_BYTES;   // MXFP8 scale tiles (STAGES x (SFA + SFB))
  uint8_t* stage_smem = sf_smem + C::SF_REGION;   // epilogue staging (1 KB aligned)
  GemmBook<C>& bk = *reinterpret_cast<GemmBook<C>*>(stage_smem + C::STAGING_BYTES);
  uint64_t* full_bar = bk.full_bar;
  uint64_t* empty_bar = bk.empty_bar;
  uint64_t* tfull_bar = bk.tfull_bar;
  uint64_t* tempty_bar = bk.tempty_bar;
  uint64_t& drain_bar = bk.drain_bar;
  uint32_t& tmem_slot = bk.tmem_slot;
  int& abort_flag = bk.abort_flag;
  int& s_bad = bk.bad;
  int* s_poff = bk.poff;
  int* s_tpre = bk.tpre;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full_bar[s], C::FULL_COUNT);
      mbar_init(&empty_bar[s], 1);
    }
    for (int a = 0; a < C::ACC_BUFS; ++a) {
      mbar_init(&tfull_bar[a], 1);
      mbar_init(&tempty_bar[a], C::EPI_WARPS);
    }
    for (int j = 0; j < kSchedDepth; ++j) {
      mbar_init(&bk.sched_full[j], 1);
      mbar_init(&bk.sched_empty[j], 1 + C::EPI_WARPS);   // the MMA thread and every epilogue warp
    }
    mbar_init(&drain_bar, 1);
    abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tensormap(&tmA);
    prefetch_tensormap(&tmB);
  }
  if (threadIdx.x == 0) s_bad = 0;
  __syncthreads();
  if (C::S != Sched::kDenseM && p.poffsets != nullptr) {
    // offsets must be non-decreasing multiples of 128 inside the buffer;
    // anything else is reported and no tile is processed.
    for (int i = threadIdx.x; i <= p.E; i += blockDim.x) {
      const int v = p.poffsets[i];
      s_poff[i] = v;
      const int prev = (i == 0) ? 0 : p.poffsets[i - 1];
      if ((v & (C::BM - 1)) != 0 || v < prev || v > p.rows_cap || (i == 0 && v != 0)) s_bad = 1;
    }
  }
  if (warp == 1) {
    tmem_alloc(&tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = tmem_slot;
  volatile int* abort_ptr = &abort_flag;
  const unsigned long long wait_lim = p.wait_ns != 0 ? p.wait_ns : kWaitLimitNs;

  if (s_bad) {
    if (threadIdx.x == 0) set_status(p.status, kErrBadIndex);
  }
  if constexpr (C::ROWS256 && C::S == Sched::kRoutedM) {
    if (warp == 0 && !s_bad) build_pair_prefix(s_poff, p.E, p.n_tiles, s_tpre);
    __syncthreads();
  }
  const int ntiles = s_bad ? 0 : total_tiles<C>(p, s_poff, s_tpre);

  if (warp == 0) {
    if constexpr (C::GATHER) {
      // -------------------------------- gathering producer (all 32 lanes)
      // Lane 0 runs the schedule and the B TMA loads; every lane copies 8 rows
      // of each A k-block (rows lane + 32 i) from the token-order input with
      // 16-byte cp.async into the 128B-swizzled layout TMA would have written
      // (chunk c of row r at r * 128 + ((c ^ (r % 8)) * 16)).  A stage is
      // signalled once its copies have landed: after the next stage's copies are
      // issued, each lane waits for its older group, fences the writes for the
      // tensor cores' (async) proxy and arrives on the stage's full barrier.
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued_mask = 0, issued_parity = 0;
      int pending = -1;
      bool ok = true;
      int next = 0;
      if (lane == 0) next = (p.sched != nullptr) ? atomicAdd(p.sched, 1) : static_cast<int>(blockIdx.x);
      next = __shfl_sync(0xffffffffu, next, 0);
      const uint32_t a_base = smem_u32(a_smem);
      for (int j = 0; ok; ++j) {
        const int slot = j % kSchedDepth;
        int w = 1;
        if (lane == 0) w = mbar_wait(&bk.sched_empty[slot], ((j / kSchedDepth) & 1) ^ 1u, abort_ptr, wait_lim) ? 1 : 0;
        if (!__shfl_sync(0xffffffffu, w, 0)) { ok = false; break; }
        const int t = (next < ntiles) ? next : -1;
        if (lane == 0) {
          bk.sched_tile[slot] = t;
          mbar_arrive(&bk.sched_full[slot]);
          if (t >= 0) next = (p.sched != nullptr) ? atomicAdd(p.sched, 1) : t + static_cast<int>(gridDim.x);
        }
        if (t < 0) break;
        next = __shfl_sync(0xffffffffu, next, 0);
        const TileInfo ti = decode_tile<C>(p, s_poff, s_tpre, t);
        const __nv_bfloat16* src[8];
        uint32_t live = 0;                   // rows with a token (the rest are zero rows)
        #pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int r = ti.m0 + lane + 32 * i;
          int tok = (r < p.rows_cap) ? p.a_row_src[r] : -1;
          if (tok >= p.a_rows) tok = -1;
          src[i] = p.a_tok + (tok >= 0 ? static_cast<long long>(tok) * p.k_len : 0);
          live |= (tok >= 0 ? 1u : 0u) << i;
        }
        for (int kb = 0; kb < ti.num_kb; ++kb) {
          int e = 1;
          if (lane == 0) e = mbar_wait(&empty_bar[stage], phase ^ 1u, abort_ptr, wait_lim) ? 1 : 0;
          if (!__shfl_sync(0xffffffffu, e, 0)) { ok = false; break; }
          if (lane == 0) {
            mbar_arrive_expect_tx(&full_bar[stage], C::B_BYTES);
            issue_loads<C>(&tmA, &tmB, p, ti, kb, a_smem + stage * C::A_BYTES, b_smem + stage * C::B_BYTES,
                           sf_smem, &full_bar[stage]);
          }
          const int k0 = kb * C::BK;
          const uint32_t dst0 = a_base + stage * C::A_BYTES;
          #pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int r = lane + 32 * i;
            const uint32_t rb = dst0 + r * 128;
            const uint32_t nbytes = ((live >> i) & 1u) ? 16u : 0u;
            #pragma unroll
            for (int c = 0; c < 8; ++c) cp_async_16(rb + ((c ^ (r & 7)) << 4), src[i] + k0 + 8 * c, nbytes);
          }
          cp_async_commit();
          if (pending >= 0) {
            cp_async_wait<1>();
            fence_proxy_async_smem();
            mbar_arrive(&full_bar[pending]);
          }
          pending = stage;
          issued_mask |= 1u << stage;
          issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == C::STAGES) { stage = 0; phase ^= 1u; }
        }
      }
      cp_async_wait<0>();
      fence_proxy_async_smem();
      if (pending >= 0) mbar_arrive(&full_bar[pending]);
      if (lane == 0) {
        sched_finish(p.sched);
        if (!ok) {
          for (int s = 0; s < C::STAGES; ++s)
            if (issued_mask & (1u << s)) mbar_wait_drain(&full_bar[s], (issued_parity >> s) & 1u);
        }
      }
    } else {
    if (lane == 0) {
      // ------------------------------------------------ TMA producer
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued_mask = 0, issued_parity = 0;
      bool ok = true;
      int next = (p.sched != nullptr) ? atomicAdd(p.sched, 1) : static_cast<int>(blockIdx.x);
      for (int j = 0; ok; ++j) {
        const int slot = j % kSchedDepth;
        if (!mbar_wait(&bk.sched_empty[slot], ((j / kSchedDepth) & 1) ^ 1u, abort_ptr, wait_lim)) { ok = false; break; }
        const int t = (next < ntiles) ? next : -1;
        bk.sched_tile[slot] = t;
        mbar_arrive(&bk.sched_full[slot]);
        if (t < 0) break;
        // the next index is reserved now; its value is first needed one tile later
        next = (p.sched != nullptr) ? atomicAdd(p.sched, 1) : t + static_cast<int>(gridDim.x);
        const TileInfo ti = decode_tile<C>(p, s_poff, s_tpre, t);
        for (int kb = 0; kb < ti.num_kb; ++kb) {
          if (!mbar_wait(&empty_bar[stage], phase ^ 1u, abort_ptr, wait_lim)) { ok = false; break; }
          mbar_arrive_expect_tx(&full_bar[stage], C::STAGE_BYTES);
          issue_loads<C>(&tmA, &tmB, p, ti, kb, a_smem + stage * C::A_BYTES, b_smem + stage * C::B_BYTES,
                         sf_smem + stage * (C::SFA_BYTES + C::SFB_BYTES), &full_bar[stage]);
          issued_mask |= 1u << stage;
          issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == C::STAGES) { stage = 0; phase ^= 1u; }
        }
      }
      sched_finish(p.sched);
      if (!ok) {
        // unwinding: let every load still in flight land before the CTA exits
        for (int s = 0; s < C::STAGES; ++s)
          if (issued_mask & (1u << s)) mbar_wait_drain(&full_bar[s], (issued_parity >> s) & 1u);
      }
    }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------ MMA issuer
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true, any = false;
      for (int j = 0; ok; ++j) {
        const int slot = j % kSchedDepth;
        if (!mbar_wait(&bk.sched_full[slot], (j / kSchedDepth) & 1, abort_ptr, wait_lim)) { ok = false; break; }
        const int t = bk.sched_tile[slot];
        mbar_arrive(&bk.sched_empty[slot]);
        if (t < 0) break;
        const TileInfo ti = decode_tile<C>(p, s_poff, s_tpre, t);
        if (!mbar_wait(&tempty_bar[acc], acc_phase ^ 1u, abort_ptr, wait_lim)) { ok = false; break; }
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + acc * C::ACC_COLS;
        for (int kb = 0; kb < ti.num_kb; ++kb) {
          if (!mbar_wait(&full_bar[stage], phase, abort_ptr, wait_lim)) { ok = false; break; }
          tc_fence_after_sync();
          const uint32_t a_addr = smem_u32(a_smem + stage * C::A_BYTES);
          const uint32_t b_addr = smem_u32(b_smem + stage * C::B_BYTES);
          if constexpr (C::NV4) {
            // scale tiles of this stage -> TMEM (tile kk of A: 4 columns; of B: 4 per
            // 128 rows), then 4 MMAs of K = 64; each TMEM cell holds the four E4M3
            // scales of one row for one MMA (16 values each)
            const uint32_t sf_addr = smem_u32(sf_smem + stage * (C::SFA_BYTES + C::SFB_BYTES));
            const uint32_t sfa_t = tmem_base + C::ACC_BUFS * C::ACC_COLS + stage * C::SF_COLS;
            const uint32_t sfb_t = sfa_t + 16;
            #pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              tmem_cp_32x128b_warpx4(sfa_t + 4 * kk, smem_desc_plain16(sf_addr + 512 * kk));
              #pragma unroll
              for (int i = 0; i < C::BN / 128; ++i)
                tmem_cp_32x128b_warpx4(sfb_t + (C::BN / 32) * kk + 4 * i,
                                       smem_desc_plain16(sf_addr + 2048 * (i + 1) + 512 * kk));
            }
            #pragma unroll
            for (int kk = 0; kk < C::BK / C::KSTEP; ++kk) {
              const uint64_t ad = smem_desc_sw128(a_addr + kk * 32, 16, 1024);
              const uint64_t bd = smem_desc_sw128(b_addr + kk * 32, 16, 1024);
              mma_nvf4_ss(d_tmem, ad, bd, C::IDESC, sfa_t + 4 * kk, sfb_t + (C::BN / 32) * kk,
                          (kb | kk) != 0 ? 1u : 0u);
            }
          } else if constexpr (C::MX) {
            // scale tiles of this stage -> TMEM, then 4 MMAs of K=32; MMA kk reads byte kk
            // (256-row tiles: A's two scale tiles in 4 columns each, then B's; the
            // second MMA takes A rows 128..255, 16 KB further on, into the
            // accumulator's second half)
            const uint32_t sf_addr = smem_u32(sf_smem + stage * (C::SFA_BYTES + C::SFB_BYTES));
            const uint32_t sfa_t = tmem_base + C::ACC_BUFS * C::ACC_COLS + stage * C::SF_COLS;
            const uint32_t sfb_t = sfa_t + 4 * C::SFA_TILES;
            #pragma unroll
            for (int i = 0; i < C::SFA_TILES; ++i)
              tmem_cp_32x128b_warpx4(sfa_t + 4 * i, smem_desc_plain16(sf_addr + 512 * i));
            #pragma unroll
            for (int i = 0; i < C::SFB_TILES; ++i)
              tmem_cp_32x128b_warpx4(sfb_t + 4 * i, smem_desc_plain16(sf_addr + 512 * (C::SFA_TILES + i)));
            #pragma unroll
            for (int kk = 0; kk < C::BK / C::KSTEP; ++kk) {
              const uint64_t ad = smem_desc_sw128(a_addr + kk * 32, 16, 1024);
              const uint64_t bd = smem_desc_sw128(b_addr + kk * 32, 16, 1024);
              mma_mxf8_ss(d_tmem, ad, bd, C::IDESC | idesc_sf_ids(kk, kk), sfa_t, sfb_t, (kb | kk) != 0 ? 1u : 0u);
              if constexpr (C::M256) {
                if (ti.half1)
                  mma_mxf8_ss(d_tmem + C::BN, smem_desc_sw128(a_addr + 16384 + kk * 32, 16, 1024), bd,
                              C::IDESC | idesc_sf_ids(kk, kk), sfa_t + 4, sfb_t, (kb | kk) != 0 ? 1u : 0u);
              }
            }
          } else {
            #pragma unroll
            for (int kk = 0; kk < C::BK / C::KSTEP; ++kk) {
              const uint64_t ad = C::A_MN ? smem_desc_sw128(a_addr + kk * 2048, 8192, 1024)
                                          : smem_desc_sw128(a_addr + kk * 32, 16, 1024);
              const uint64_t bd = C::B_MN ? smem_desc_sw128(b_addr + kk * 2048, 8192, 1024)
                                          : smem_desc_sw128(b_addr + kk * 32, 16, 1024);
              mma_bf16_ss(d_tmem, ad, bd, C::IDESC, (kb | kk) != 0 ? 1u : 0u);
              if constexpr (C::M256) {
                // rows 128..255 of the A tile (16 KB further on) against the same B k-block
                if (ti.half1)
                  mma_bf16_ss(d_tmem + C::BN, smem_desc_sw128(a_addr + 16384 + kk * 32, 16, 1024), bd, C::IDESC,
                              (kb | kk) != 0 ? 1u : 0u);
              }
            }
          }
          any = true;
          mma_commit(&empty_bar[stage]);
          if (++stage == C::STAGES) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        mma_commit(&tfull_bar[acc]);
        if (++acc == C::ACC_BUFS) { acc = 0; acc_phase ^= 1u; }
      }
      if (!ok && any) {
        mma_commit(&drain_bar);
        mbar_wait_drain(&drain_bar, 0);
      }
    }
  } else {
    // ---------------------------------------- epilogue (warps 2 .. 1 + EPI_WARPS)
    const int ew = warp - 2;
    const int quarter = warp & 3;          // TMEM lanes a warp may read: 32 * (warp % 4) onwards
    const int part = ew >> 2;              // 256-row tiles: which 128-row half this warp writes
                                           // (split-column tiles: which half of the h' columns)
    int acc = 0;
    uint32_t acc_phase = 0;
    Stager<C::STAGING_BUFS, C::STAGING_BUF> st{stage_smem + ew * (C::STAGING_BUFS * C::STAGING_BUF), 0, lane};
    const float al = acc_scale<C>(p);
    for (int j = 0;; ++j) {
      const int slot = j % kSchedDepth;
      if (!mbar_wait(&bk.sched_full[slot], (j / kSchedDepth) & 1, abort_ptr, wait_lim)) break;
      const int t = bk.sched_tile[slot];
      __syncwarp();
      if (lane == 0) mbar_arrive(&bk.sched_empty[slot]);
      if (t < 0) break;
      const TileInfo ti = decode_tile<C>(p, s_poff, s_tpre, t);
      if (!mbar_wait(&tfull_bar[acc], acc_phase, abort_ptr, wait_lim)) break;
      tc_fence_after_sync();
      bool released = false;                 // accumulator already handed back by the epilogue
      if constexpr (C::M256) {
        if (part == 0 || ti.half1) {
          TileInfo th = ti;
          th.m0 += 128 * part;
          epilogue_tile_tma<C>(p, th, tmem_base + acc * C::ACC_COLS + part * C::BN, quarter, lane, st, &tmC, &tmC2,
                               &tempty_bar[acc], &released, al);
        }
      } else if constexpr (C::TMA_OUT) {
        epilogue_tile_tma<C>(p, ti, tmem_base + acc * C::ACC_COLS, quarter, lane, st, &tmC, &tmC2,
                             &tempty_bar[acc], &released, al, C::SPLIT_COLS ? part : 0);
      } else {
        epilogue_tile<C>(p, ti, tmem_base + acc * C::BN, quarter, lane);
      }
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0 && !released) mbar_arrive(&tempty_bar[acc]);
      if (++acc == C::ACC_BUFS) { acc = 0; acc_phase ^= 1u; }
    }
    if constexpr (C::TMA_OUT) st.drain();     // every TMA store has finished before the CTA exits
  }

  __syncwarp();
  tc_fence_before_sync();
  __syncthreads();
  pdl_launch_next();
  if (threadIdx.x == 0 && abort_flag) set_status(p.status, kErrTimeout);
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
}


// This CTA's share of one k-block of a pair tile: A rows m0 + 128*rank and
// half of the B rows (SwiGLU: rank 0 the gate rows, rank 1 the matching up
// rows), both counted on the even CTA's full barrier.
template <class C>
__device__ __forceinline__ void issue_loads_pair(const CUtensorMap* tmA, const CUtensorMap* tmB, const GemmParams& p,
                                                 const TileInfo& ti, int kb, uint32_t rank, uint8_t* a_dst,
                                                 uint8_t* b_dst, uint32_t bar_cluster_addr) {
  const int k0 = kb * C::BK;
  if constexpr (C::S == Sched::kRoutedK) {
    // A[m, k] = Abuf[k_row0 + k, m0 + 128*rank + m], B[n, k] = Bbuf[k_row0 + k, n*BN + 128*rank + n]:
    // MN-major, two 64-wide chunks each
    const int mr = ti.m0 + 128 * static_cast<int>(rank);
    const int nr = ti.n * C::BN + 128 * static_cast<int>(rank);
    tma_load_2d_pair(a_dst, tmA, bar_cluster_addr, mr, ti.k_row0 + k0);
    tma_load_2d_pair(a_dst + C::MN_CHUNK, tmA, bar_cluster_addr, mr + 64, ti.k_row0 + k0);
    tma_load_2d_pair(b_dst, tmB, bar_cluster_addr, nr, ti.k_row0 + k0);
    tma_load_2d_pair(b_dst + C::MN_CHUNK, tmB, bar_cluster_addr, nr + 64, ti.k_row0 + k0);
    return;
  }
  tma_load_2d_pair(a_dst, tmA, bar_cluster_addr, k0, ti.m0 + 128 * static_cast<int>(rank));
  if constexpr (C::B_MN) {
    // B[n, k] = W[group*K + k, n]: this CTA's 128 columns of N, two 64-wide chunks
    const int nr = ti.n * C::BN + 128 * static_cast<int>(rank);
    tma_load_2d_pair(b_dst, tmB, bar_cluster_addr, nr, ti.group * p.b_rows_per_group + k0);
    tma_load_2d_pair(b_dst + 8192, tmB, bar_cluster_addr, nr + 64, ti.group * p.b_rows_per_group + k0);
    return;
  }
  int b_row;
  if constexpr (C::EP == Epi::kSwiglu)
    b_row = ti.group * p.b_rows_per_group + ti.n * (C::BN / 2) + (rank ? p.b_half_offset : 0);
  else
    b_row = ti.group * p.b_rows_per_group + ti.n * C::BN + static_cast<int>(rank) * (C::BN / 2);
  tma_load_2d_pair(b_dst, tmB, bar_cluster_addr, k0, b_row);
}

// The grouped GEMM on CTA pairs (clusters of two, one CTA per SM): each
// 256 x 256 tile is one chain of tcgen05.mma.cta_group::2 (M = 256, N = 256,
// K = 16) issued by the even CTA.  Each CTA streams 128 rows of A and 128 rows
// of B per k-block (32 KB per 512 MMA cycles), holds its 128 x 256 fp32
// accumulator in its own TMEM -- two of them, so the epilogue of one tile
// overlaps the MMAs of the next -- and writes its own 128 output rows.
//
// Pipeline: full[s] lives in the even CTA and counts both CTAs' TMA bytes;
// the MMA completion of stage s arrives on empty[s] of both CTAs; the
// accumulator completion arrives on tfull of both; both CTAs' epilogue warps
// arrive on the even CTA's tempty.  Waits are bounded as in the one-CTA
// kernel; both CTAs meet in two cluster barriers (after set-up, before TMEM
// is freed), which every path reaches.
template <class C>
__global__ void __launch_bounds__(C::THREADS, 1)
    grouped_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                             const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmC2,
                             const GemmParams p) {
  pdl_wait();
  static_assert(C::PAIR, "pair configuration");
  static_assert(sizeof(GemmBook<C>) <= C::BOOK_BYTES, "bookkeeping size");
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t rank = cluster_ctarank();
  const bool leader = (rank == 0);
  const int cid = static_cast<int>(cluster_id_x());
  const int ncl = static_cast<int>(num_clusters_x());
  {
    const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
    if (pad + C::SMEM_USED > static_cast<uint32_t>(C::SMEM_BYTES)) {
      if (threadIdx.x == 0) set_status(p.status, kErrLaunch);
      cluster_sync();   // the peer meets both cluster barriers whatever it finds
      cluster_sync();
      return;
    }
  }
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* a_smem = smem;
  uint8_t* b_smem = smem + C::STAGES * C::A_BYTES;
  uint8_t* stage_smem = b_smem + C::STAGES * C::B_BYTES;   // epilogue staging (1 KB aligned)
  GemmBook<C>& bk = *reinterpret_cast<GemmBook<C>*>(stage_smem + C::STAGING_BYTES);
  uint64_t* full_bar = bk.full_bar;
  uint64_t* empty_bar = bk.empty_bar;
  uint64_t* tfull_bar = bk.tfull_bar;
  uint64_t* tempty_bar = bk.tempty_bar;
  int* s_poff = bk.poff;
  int* s_tpre = bk.tpre;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full_bar[s], 1);       // even CTA: its producer's arrive + both CTAs' bytes
      mbar_init(&empty_bar[s], 1);
    }
    for (int a = 0; a < C::ACC_BUFS; ++a) {
      mbar_init(&tfull_bar[a], 1);
      mbar_init(&tempty_bar[a], 2 * C::EPI_WARPS);   // even CTA: the epilogue warps of both CTAs
    }
    mbar_init(&bk.drain_bar, 1);
    bk.abort_flag = 0;
    bk.bad = 0;
    fence_mbarrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tensormap(&tmA);
    prefetch_tensormap(&tmB);
  }
  __syncthreads();
  if (C::S != Sched::kDenseM && p.poffsets != nullptr) {
    for (int i = threadIdx.x; i <= p.E; i += blockDim.x) {
      const int v = p.poffsets[i];
      s_poff[i] = v;
      const int prev = (i == 0) ? 0 : p.poffsets[i - 1];
      if ((v & (C::BM - 1)) != 0 || v < prev || v > p.rows_cap || (i == 0 && v != 0)) bk.bad = 1;
    }
  }
  if (warp == 1) {
    tmem_alloc_pair(&bk.tmem_slot, C::TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before_sync();
  __syncthreads();
  cluster_sync();                       // barriers of both CTAs initialised before any cross-CTA signal
  tc_fence_after_sync();
  const uint32_t tmem_base = bk.tmem_slot;
  volatile int* abort_ptr = &bk.abort_flag;
  const unsigned long long wait_lim = p.wait_ns != 0 ? p.wait_ns : kWaitLimitNs;
  const bool bad = bk.bad != 0;          // both CTAs read the same offsets
  if (bad && leader && threadIdx.x == 0) set_status(p.status, kErrBadIndex);
  if constexpr (C::S == Sched::kRoutedM) {
    if (warp == 0 && !bad) build_pair_prefix(s_poff, p.E, p.n_tiles, s_tpre);
    __syncthreads();
  }
  const int ntiles = bad ? 0 : total_tiles<C>(p, s_poff, s_tpre);

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------ TMA producer (both CTAs)
      const uint32_t full_leader = mapa_shared(smem_u32(&full_bar[0]), 0);
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued_mask = 0, issued_parity = 0;
      bool ok = true;
      for (int t = cid; t < ntiles && ok; t += ncl) {
        const TileInfo ti = decode_tile<C>(p, s_poff, s_tpre, t);
        for (int kb = 0; kb < ti.num_kb; ++kb) {
          if (!mbar_wait(&empty_bar[stage], phase ^ 1u, abort_ptr, wait_lim)) { ok = false; break; }
          if (leader) mbar_arrive_expect_tx(&full_bar[stage], 2 * C::STAGE_BYTES);
          issue_loads_pair<C>(&tmA, &tmB, p, ti, kb, rank, a_smem + stage * C::A_BYTES, b_smem + stage * C::B_BYTES,
                              full_leader + 8u * stage);
          issued_mask |= 1u << stage;
          issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == C::STAGES) { stage = 0; phase ^= 1u; }
        }
      }
      if (!ok) {
        if (leader) {
          // unwinding: let every stage still counted on this CTA's barriers land
          for (int s = 0; s < C::STAGES; ++s)
            if (issued_mask & (1u << s)) mbar_wait_drain(&full_bar[s], (issued_parity >> s) & 1u);
        } else {
          // this CTA's loads complete on the peer's barriers: give them time to land
          const unsigned long long t0 = global_timer_ns();
          while (global_timer_ns() - t0 < 200000ull) {
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      // ------------------------------------------------ MMA issuer (even CTA)
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true, any = false;
      for (int t = cid; t < ntiles && ok; t += ncl) {
        const TileInfo ti = decode_tile<C>(p, s_poff, s_tpre, t);
        if (!mbar_wait_cluster(&tempty_bar[acc], acc_phase ^ 1u, abort_ptr, wait_lim)) { ok = false; break; }
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + acc * C::ACC_COLS;
        for (int kb = 0; kb < ti.num_kb; ++kb) {
          if (!mbar_wait(&full_bar[stage], phase, abort_ptr, wait_lim)) { ok = false; break; }
          tc_fence_after_sync();
          const uint32_t a_addr = smem_u32(a_smem + stage * C::A_BYTES);
          const uint32_t b_addr = smem_u32(b_smem + stage * C::B_BYTES);
          #pragma unroll
          for (int kk = 0; kk < C::BK / C::KSTEP; ++kk) {
            const uint64_t ad = C::A_MN ? smem_desc_sw128(a_addr + kk * 2048, C::MN_CHUNK, 1024)
                                        : smem_desc_sw128(a_addr + kk * 32, 16, 1024);
            const uint64_t bd = C::B_MN ? smem_desc_sw128(b_addr + kk * 2048, C::MN_CHUNK, 1024)
                                        : smem_desc_sw128(b_addr + kk * 32, 16, 1024);
            mma_bf16_pair(d_tmem, ad, bd, C::IDESC, (kb | kk) != 0 ? 1u : 0u);
          }
          any = true;
          mma_commit_pair_both(&empty_bar[stage]);
          if (++stage == C::STAGES) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        mma_commit_pair_both(&tfull_bar[acc]);
        if (++acc == C::ACC_BUFS) { acc = 0; acc_phase ^= 1u; }
      }
      if (!ok && any) {
        mma_commit_pair(&bk.drain_bar);
        mbar_wait_drain(&bk.drain_bar, 0);
      }
    }
  } else {
    // -------------------------------------------------- epilogue (warps 2..5 of both CTAs)
    const int quarter = warp & 3;
    const uint32_t tempty_leader = mapa_shared(smem_u32(&tempty_bar[0]), 0);
    int acc = 0;
    uint32_t acc_phase = 0;
    Stager<C::STAGING_BUFS, C::STAGING_BUF> st{stage_smem + (warp - 2) * (C::STAGING_BUFS * C::STAGING_BUF), 0,
                                               lane};
    for (int t = cid; t < ntiles; t += ncl) {
      const TileInfo ti = decode_tile<C>(p, s_poff, s_tpre, t);
      if (!mbar_wait(&tfull_bar[acc], acc_phase, abort_ptr, wait_lim)) break;
      tc_fence_after_sync();
      if (leader || ti.half1) {           // a half tile: the odd CTA's rows are not this expert's
        TileInfo th = ti;
        th.m0 += 128 * static_cast<int>(rank);
        epilogue_tile_tma<C>(p, th, tmem_base + acc * C::ACC_COLS, quarter, lane, st, &tmC, &tmC2);
      }
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(tempty_leader + 8u * acc);
      if (++acc == C::ACC_BUFS) { acc = 0; acc_phase ^= 1u; }
    }
    st.drain();
  }

  __syncwarp();
  tc_fence_before_sync();
  __syncthreads();
  cluster_sync();                       // the peer no longer reads this CTA's memory or signals its barriers
  pdl_launch_next();
  if (threadIdx.x == 0 && bk.abort_flag) set_status(p.status, kErrTimeout);
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc_pair(tmem_base, C::TMEM_COLS);
  }
}

}  // namespace moe
