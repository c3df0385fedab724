// Routing, permutation and combine kernels (CUDA cores, HBM-bound).
//
//  * top-k gating: one warp per token, warp-shuffle arg-max k times;
//  * permutation: a stable counting sort of the T*k (token, slot) pairs by
//    expert, done entirely on the device (per-block histograms and ranks, a
//    scan of the histogram columns, the maps worked out inside the row copy)
//    so the host never sees the expert sizes — the sync-free, dynamic-shape
//    permutation of the Megatron Core MoE summary (technical summary 1 and
//    2.4);
//  * gather / combine: 16-byte vector copies of token rows; the combine is an
//    unweighted fp32 sum because the gate was applied inside the expert
//    (technical summary 2.2, memory-efficient permutation).
#include <cuda_bf16.h>

#include <climits>
#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr unsigned kFull = 0xffffffffu;

// ---------------------------------------------------------------- top-k
struct Cand {
  float key;
  float logit;
  int id;  // INT_MAX = none
};

// Keys are never NaN here (a NaN key is replaced by -inf before ranking), so
// this is a strict total order: key descending, then expert id ascending.
__device__ __forceinline__ bool better(const Cand& a, const Cand& b) {
  if (a.id == INT_MAX) return false;
  if (b.id == INT_MAX) return true;
  return a.key > b.key || (a.key == b.key && a.id < b.id);
}

// A key as an unsigned integer with the same order (-0 taken as +0 first, so
// that keys equal as floats stay equal); 0 lies below every key (-inf maps to
// 0x007FFFFF) and marks an expert that is taken or absent.
__device__ __forceinline__ uint32_t ordered_key(float key) {
  const uint32_t u = __float_as_uint(key + 0.0f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Route one token (the whole warp): lane s < k receives slot s's expert and gate.
// Lane l holds experts l, l + 32, ...  Each slot is one warp maximum of the
// keys and one warp minimum of the ids that reach it (ties go to the lower id),
// the same order as better() on (key, id).
template <int PER_LANE>
__device__ __forceinline__ void topk_one_token(const float* __restrict__ row, const float* __restrict__ bias, int E,
                                               int k, int score, int lane, int& out_id, float& out_gate) {
  uint32_t okey[PER_LANE];
  #pragma unroll
  for (int j = 0; j < PER_LANE; ++j) {
    const int e = lane + 32 * j;
    const float lg = (e < E) ? row[e] : 0.f;
    float key;
    if (score == 0) {
      key = lg;
    } else {
      key = 1.0f / (1.0f + expf(-lg));
      if (bias != nullptr && e < E) key += bias[e];
    }
    if (key != key) key = -INFINITY;   // NaN ranks last: the order stays total
    okey[j] = (e < E) ? ordered_key(key) : 0u;
  }
  int my_id = 0;  // lane s keeps slot s
  for (int s = 0; s < k; ++s) {
    uint32_t bk = 0u;
    int bj = 0;
    #pragma unroll
    for (int j = 0; j < PER_LANE; ++j)   // strict: the lane's lowest id among equal keys
      if (okey[j] > bk) { bk = okey[j]; bj = j; }
    const uint32_t m = __reduce_max_sync(kFull, bk);
    const uint32_t id = __reduce_min_sync(kFull, (bk == m && m != 0u) ? static_cast<uint32_t>(lane + 32 * bj)
                                                                       : 0xFFFFFFFFu);
    if (id != 0xFFFFFFFFu && static_cast<int>(id & 31u) == lane) {
      #pragma unroll
      for (int j = 0; j < PER_LANE; ++j)
        if (j == static_cast<int>(id >> 5)) okey[j] = 0u;
    }
    if (lane == s) my_id = id != 0xFFFFFFFFu ? static_cast<int>(id) : 0;
  }
  const float my_logit = (lane < k) ? row[my_id] : 0.f;
  // gates of the chosen k, normalised over them
  float w;
  if (score == 0) {
    const float lmax = __shfl_sync(kFull, my_logit, 0);   // slot 0 has the largest logit
    w = (lane < k) ? expf(my_logit - lmax) : 0.f;
  } else {
    w = (lane < k) ? 1.0f / (1.0f + expf(-my_logit)) : 0.f;
  }
  float sum = 0.f;                                        // slot order: deterministic
  for (int s = 0; s < k; ++s) sum += __shfl_sync(kFull, w, s);
  out_id = my_id;
  out_gate = w / sum;
}

// Route one token in one thread (few experts: E <= kThreadTopkE): the same
// keys, tie rule, slot order and gate arithmetic as topk_one_token, so the
// result is identical; a warp then routes 32 tokens at once instead of one.
// The slot loop is not unrolled (only the scan over the experts is): the
// kernel's code stays small, which matters because its instructions are
// fetched cold at every step.
constexpr int kThreadTopkE = 16;
__device__ __forceinline__ void topk_one_token_thread(const float* __restrict__ row, const float* __restrict__ bias,
                                                      int E, int k, int score, int32_t* __restrict__ idx_out,
                                                      float* __restrict__ gate_out, int* __restrict__ s_idx_out) {
  float lg[kThreadTopkE], key[kThreadTopkE];
  #pragma unroll
  for (int e = 0; e < kThreadTopkE; ++e) {
    lg[e] = (e < E) ? row[e] : 0.f;
    if (score == 0) {
      key[e] = lg[e];
    } else {
      key[e] = 1.0f / (1.0f + expf(-lg[e]));
      if (bias != nullptr && e < E) key[e] += bias[e];
    }
    if (key[e] != key[e]) key[e] = -INFINITY;   // as in topk_one_token
  }
  // pass 1: the slots in order, their weights summed in slot order
  uint32_t taken = 0;
  float l0 = 0.f, sum = 0.f;
  #pragma unroll 1
  for (int s = 0; s < k; ++s) {
    Cand best{0.f, 0.f, INT_MAX};
    #pragma unroll
    for (int e = 0; e < kThreadTopkE; ++e) {
      Cand c{key[e], lg[e], (e < E && !((taken >> e) & 1u)) ? e : INT_MAX};
      if (better(c, best)) best = c;
    }
    taken |= 1u << best.id;
    if (s == 0) l0 = best.logit;                          // slot 0 has the largest logit
    sum += (score == 0) ? expf(best.logit - l0) : 1.0f / (1.0f + expf(-best.logit));
    idx_out[s] = best.id;
    s_idx_out[s] = best.id;
  }
  // pass 2: each slot's weight again (the same expression on the same logit)
  // over the sum
  #pragma unroll 1
  for (int s = 0; s < k; ++s) {
    const float l = row[s_idx_out[s]];
    gate_out[s] = ((score == 0) ? expf(l - l0) : 1.0f / (1.0f + expf(-l))) / sum;
  }
}

template <int PER_LANE>
__global__ void __launch_bounds__(256) topk_kernel(const float* __restrict__ logits, const float* __restrict__ bias,
                                                   int T, int E, int k, int score, int32_t* __restrict__ idx,
                                                   float* __restrict__ gate) {
  pdl_entry();
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (warp >= T) return;
  int id;
  float g;
  topk_one_token<PER_LANE>(logits + (long long)warp * E, bias, E, k, score, lane, id, g);
  if (lane < k) {
    idx[(long long)warp * k + lane] = id;
    gate[(long long)warp * k + lane] = g;
  }
}

// ---------------------------------------------------------------- counting sort
// The T*k (token, slot) pairs, in token-major order, are cut into chunks of
// pb = (256/k)*k pairs (whole tokens); chunk b is one block of the count and
// scatter kernels.  Stable rank of a pair = number of earlier pairs of the
// same chunk with the same expert (earlier tokens: a token never picks an
// expert twice).
__host__ __device__ constexpr int pairs_per_chunk(int k) { return (kPairsPerBlock / k) * k; }

// e: expert of this thread's pair (-1: none).  s_cnt [8][E], s_tot [E] in
// shared memory.  Returns the stable rank; leaves per-expert totals in s_tot.
__device__ __forceinline__ int block_stable_rank(int e, int E, int* s_cnt, int* s_tot) {
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  for (int i = tid; i < 8 * E; i += blockDim.x) s_cnt[i] = 0;
  __syncthreads();
  const unsigned peers = __match_any_sync(kFull, e);
  const int rank_w = __popc(peers & ((1u << lane) - 1u));
  if (e >= 0 && (__ffs(peers) - 1) == lane) s_cnt[warp * E + e] = __popc(peers);
  __syncthreads();
  for (int x = tid; x < E; x += blockDim.x) {
    int run = 0;
    #pragma unroll
    for (int w = 0; w < 8; ++w) {
      const int c = s_cnt[w * E + x];
      s_cnt[w * E + x] = run;
      run += c;
    }
    s_tot[x] = run;
  }
  __syncthreads();
  return (e >= 0) ? s_cnt[warp * E + e] + rank_w : -1;
}

__device__ __forceinline__ int load_pair_expert(const int32_t* __restrict__ idx, long long npairs, int pb, int E,
                                                int* status) {
  const long long p = (long long)blockIdx.x * pb + threadIdx.x;
  int e = -1;
  if (threadIdx.x < pb && p < npairs) {
    e = idx[p];
    if (e < 0 || e >= E) {
      set_status(status, kErrBadIndex);
      e = -1;
    }
  }
  return e;
}

// One warp scans column col[0..NB) in place (exclusive) and returns its total.
// The loads go through L2 (another block may have written the column).
__device__ __forceinline__ int scan_column(int32_t* __restrict__ col, int NB, int lane) {
  constexpr int kBatch = 8;
  int run = 0;
  for (int b0 = 0; b0 < NB; b0 += 32 * kBatch) {
    int v[kBatch];
    #pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      const int b = b0 + 32 * j + lane;
      v[j] = (b < NB) ? __ldcg(col + b) : 0;
    }
    #pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      int inc = v[j];
      #pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int u = __shfl_up_sync(kFull, inc, d);
        if (lane >= d) inc += u;
      }
      const int b = b0 + 32 * j + lane;
      if (b < NB) col[b] = run + inc - v[j];
      run += __shfl_sync(kFull, inc, 31);
    }
  }
  return run;
}

// ------------------------------------------- permutation in two launches
// The histogram launch (count_rank_kernel, or topk_hist_kernel with MODE 1
// or 2) also leaves each pair's stable rank inside its chunk in slot_row (-1
// for a dropped pair).  The column scan then takes one of three forms: with
// at most 32 chunks and 32 experts none at all (gather_scatter_kernel RAW
// sums the columns it needs itself); with LAST_SCAN (NB * E <=
// kLastScanEntries) the last of the histogram blocks to finish -- found by
// an atomic count of finished blocks, no block waits for another -- scans the
// columns and writes counts; otherwise scan_cols_kernel runs between the two
// launches.  gather_scatter_kernel turns the ranks into rows and copies the
// token rows in the same launch.
constexpr int kLastScanEntries = 8192;
// gather_scatter_kernel: a block per token, warp 0 deriving the expert
// offsets while warp 1 fetches the pairs' maps.  Where all blocks fit on the
// GPU at once (T <= kGsSmallT) two warps, each thread with 8 16-byte loads of
// the row in flight (a 4096-wide bf16 row in one batch); otherwise four
// warps with 4 loads each (measured faster for the larger batches).
constexpr int kGsSmallT = 4864;   // 152 SMs x 32 blocks

template <bool LAST_SCAN>
__device__ __forceinline__ void hist_rank_tail(int e, long long p, bool has_pair, int E, int32_t* __restrict__ hist,
                                               int32_t* __restrict__ slot_row, int* __restrict__ done,
                                               int32_t* __restrict__ counts, int* s_cnt, int* s_tot) {
  const int r = block_stable_rank(e, E, s_cnt, s_tot);
  for (int x = threadIdx.x; x < E; x += blockDim.x) hist[(long long)x * gridDim.x + blockIdx.x] = s_tot[x];
  if (has_pair) slot_row[p] = r;                   // (-1 where e < 0)
  if constexpr (LAST_SCAN) {
    __shared__ int s_last;
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) s_last = (atomicAdd(done, 1) == static_cast<int>(gridDim.x) - 1) ? 1 : 0;
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int x = warp; x < E; x += blockDim.x / 32) {
      const int tot = scan_column(hist + (long long)x * gridDim.x, gridDim.x, lane);
      if (lane == 0) counts[x] = tot;
    }
    if (threadIdx.x == 0) atomicExch(done, 0);   // zero for the next launch
  }
}

__global__ void __launch_bounds__(kPairsPerBlock) count_kernel(const int32_t* __restrict__ idx, long long npairs,
                                                               int pb, int E, int32_t* __restrict__ hist,
                                                               int* status) {
  pdl_entry();
  __shared__ int s_cnt[8 * kMaxE];
  __shared__ int s_tot[kMaxE];
  const int e = load_pair_expert(idx, npairs, pb, E, status);
  block_stable_rank(e, E, s_cnt, s_tot);
  for (int x = threadIdx.x; x < E; x += blockDim.x) hist[(long long)x * gridDim.x + blockIdx.x] = s_tot[x];
}

// Top-k gating fused with the chunk histogram: block b routes the tokens of
// chunk b (one warp per token, as topk_kernel; one thread per token when
// E <= kThreadTopkE) and then counts its pairs.
// MODE 0: the histograms only; 1: also the ranks in slot_row; 2: also the
// last block's column scan (see hist_rank_tail).
template <int PER_LANE, int MODE>
__global__ void __launch_bounds__(kPairsPerBlock) topk_hist_kernel(const float* __restrict__ logits,
                                                                   const float* __restrict__ bias, int T, int E,
                                                                   int k, int score, int32_t* __restrict__ idx,
                                                                   float* __restrict__ gate,
                                                                   int32_t* __restrict__ hist,
                                                                   int32_t* __restrict__ slot_row,
                                                                   int* __restrict__ done,
                                                                   int32_t* __restrict__ counts) {
  pdl_entry();
  constexpr int kStageFloats = 8192;             // logits of the chunk staged in shared memory (32 KB)
  __shared__ int s_idx[kPairsPerBlock];
  __shared__ int s_cnt[8 * kMaxE];
  __shared__ int s_tot[kMaxE];
  __shared__ float s_logit[kStageFloats];
  const int tpb = kPairsPerBlock / k;            // tokens of this chunk
  const int t0 = blockIdx.x * tpb;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // The chunk's logits are one contiguous range: read it with the whole block
  // (many loads in flight) instead of one row at a time per warp.
  const int nt = min(tpb, T - t0);
  const bool staged = nt * E <= kStageFloats;
  if (staged) {
    const float* src = logits + (long long)t0 * E;
    for (int i = threadIdx.x; i < nt * E; i += blockDim.x) s_logit[i] = __ldg(src + i);
    __syncthreads();
  }
  if constexpr (PER_LANE == 0) {
    // few experts (E <= kThreadTopkE): one thread per token
    for (int u = threadIdx.x; u < nt; u += blockDim.x) {
      const long long t = t0 + u;
      topk_one_token_thread(staged ? s_logit + u * E : logits + t * E, bias, E, k, score, idx + t * k, gate + t * k,
                            s_idx + u * k);
    }
  } else {
    for (int u = warp; u < tpb; u += 8) {
      const int t = t0 + u;
      if (t >= T) break;
      int id;
      float g;
      topk_one_token<PER_LANE>(staged ? s_logit + u * E : logits + (long long)t * E, bias, E, k, score, lane, id, g);
      if (lane < k) {
        idx[(long long)t * k + lane] = id;
        gate[(long long)t * k + lane] = g;
        s_idx[u * k + lane] = id;
      }
    }
  }
  __syncthreads();
  const int pb = tpb * k;
  const long long npairs = (long long)T * k;
  const long long p = (long long)blockIdx.x * pb + threadIdx.x;
  const int e = (threadIdx.x < pb && p < npairs) ? s_idx[threadIdx.x] : -1;
  if constexpr (MODE == 0) {
    block_stable_rank(e, E, s_cnt, s_tot);
    for (int x = threadIdx.x; x < E; x += blockDim.x) hist[(long long)x * gridDim.x + blockIdx.x] = s_tot[x];
  } else {
    hist_rank_tail<MODE == 2>(e, p, threadIdx.x < pb && p < npairs, E, hist, slot_row, done, counts, s_cnt, s_tot);
  }
}

// The chunk histograms are laid out per expert: hist[e * NB + b] = pairs of
// chunk b routed to expert e.  One warp per expert scans its column in place:
// hist[e][b] becomes the number of expert-e pairs in the chunks before b, and
// counts[e] the column total.  All of a lane's loads of a batch are issued
// before the first is used.
__global__ void __launch_bounds__(256) scan_cols_kernel(int32_t* __restrict__ hist, int NB, int E,
                                                        int32_t* __restrict__ counts) {
  pdl_entry();
  const int e = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (e >= E) return;
  int32_t* col = hist + (long long)e * NB;
  constexpr int kBatch = 8;
  int run = 0;
  for (int b0 = 0; b0 < NB; b0 += 32 * kBatch) {
    int v[kBatch];
    #pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      const int b = b0 + 32 * j + lane;
      v[j] = (b < NB) ? col[b] : 0;
    }
    #pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      int inc = v[j];
      #pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int u = __shfl_up_sync(kFull, inc, d);
        if (lane >= d) inc += u;
      }
      const int b = b0 + 32 * j + lane;
      if (b < NB) col[b] = run + inc - v[j];
      run += __shfl_sync(kFull, inc, 31);
    }
  }
  if (lane == 0) counts[e] = run;
}

// Exclusive scans over the experts of counts and of counts rounded up to
// whole 128-row blocks, by the first warp of a block, into s_off / s_poff
// (E + 1 entries each).
__device__ __forceinline__ void expert_offsets(const int32_t* __restrict__ counts, int E, int* s_off, int* s_poff) {
  const int tid = threadIdx.x;
  if (tid < 32) {
    const int per_lane = (E + 31) / 32;
    const int e0 = tid * per_lane, e1 = min(E, e0 + per_lane);
    int cs = 0, ps = 0;
    for (int x = e0; x < e1; ++x) {
      const int c = counts[x];
      cs += c;
      ps += (c + kPadRows - 1) / kPadRows * kPadRows;
    }
    int ci = cs, pi = ps;
    #pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int a = __shfl_up_sync(kFull, ci, d), b = __shfl_up_sync(kFull, pi, d);
      if (tid >= d) { ci += a; pi += b; }
    }
    int c_ex = ci - cs, p_ex = pi - ps;
    for (int x = e0; x < e1; ++x) {
      const int c = counts[x];
      s_off[x] = c_ex;
      s_poff[x] = p_ex;
      c_ex += c;
      p_ex += (c + kPadRows - 1) / kPadRows * kPadRows;
    }
    if (tid == 31) { s_off[E] = ci; s_poff[E] = pi; }
  }
}

// Block b: the maps of chunk b's pairs.  Row of a pair = poffsets[e] + pairs
// of expert e in earlier chunks (the scanned column) + its stable rank inside
// the chunk.  Block 0 also writes offsets and poffsets and marks the padding
// rows of every segment (row_src -1, row_gate 0).
__global__ void __launch_bounds__(kPairsPerBlock) scatter_kernel(const int32_t* __restrict__ idx,
                                                                 const float* __restrict__ gate, long long npairs,
                                                                 int pb, int E, int k, int NB,
                                                                 const int32_t* __restrict__ base,
                                                                 const int32_t* __restrict__ counts,
                                                                 int32_t* __restrict__ offsets,
                                                                 int32_t* __restrict__ poffsets,
                                                                 int32_t* __restrict__ slot_row,
                                                                 int32_t* __restrict__ row_src,
                                                                 float* __restrict__ row_gate) {
  pdl_entry();
  __shared__ int s_cnt[8 * kMaxE];
  __shared__ int s_tot[kMaxE];
  __shared__ int s_off[kMaxE + 1];
  __shared__ int s_poff[kMaxE + 1];
  expert_offsets(counts, E, s_off, s_poff);
  const int e = load_pair_expert(idx, npairs, pb, E, nullptr);
  const int r = block_stable_rank(e, E, s_cnt, s_tot);   // (its barriers also publish s_off, s_poff)
  if (blockIdx.x == 0) {
    for (int x = threadIdx.x; x <= E; x += blockDim.x) {
      offsets[x] = s_off[x];
      poffsets[x] = s_poff[x];
    }
    for (int i = threadIdx.x; i < E * kPadRows; i += blockDim.x) {
      const int x = i / kPadRows, j = i % kPadRows;
      const int rr = s_poff[x] + counts[x] + j;
      if (rr < s_poff[x + 1]) {
        row_src[rr] = -1;
        if (row_gate != nullptr) row_gate[rr] = 0.f;
      }
    }
  }
  const long long p = (long long)blockIdx.x * pb + threadIdx.x;
  if (threadIdx.x >= pb || p >= npairs) return;
  if (e < 0) {
    slot_row[p] = -1;
    return;
  }
  const int row = s_poff[e] + base[(long long)e * NB + blockIdx.x] + r;
  slot_row[p] = row;
  row_src[row] = static_cast<int32_t>(p / k);
  if (row_gate != nullptr) row_gate[row] = gate[p];
}

template <bool LAST_SCAN>
__global__ void __launch_bounds__(kPairsPerBlock) count_rank_kernel(const int32_t* __restrict__ idx,
                                                                    long long npairs, int pb, int E,
                                                                    int32_t* __restrict__ hist,
                                                                    int32_t* __restrict__ slot_row,
                                                                    int* __restrict__ done,
                                                                    int32_t* __restrict__ counts, int* status) {
  pdl_entry();
  __shared__ int s_cnt[8 * kMaxE];
  __shared__ int s_tot[kMaxE];
  const int e = load_pair_expert(idx, npairs, pb, E, status);
  const long long p = (long long)blockIdx.x * pb + threadIdx.x;
  hist_rank_tail<LAST_SCAN>(e, p, threadIdx.x < pb && p < npairs, E, hist, slot_row, done, counts, s_cnt, s_tot);
}

// Block t: token t's k pairs get their rows, row = padded
// offset of the expert + its pairs in earlier chunks (the scanned column) +
// the rank the histogram launch left in slot_row; then x[t] is copied to
// them.  Every block derives the expert offsets from counts (E <= 256);
// block 0 also writes offsets, poffsets and marks the padding rows.  Launched
// with max(T, 1) blocks.
// Zero the padding rows of the expert segments, spread over the blocks of a
// row-copy launch: block b takes padding rows b, b + nblocks, ... of the
// concatenation of every expert's padding (s_off / s_poff: the expert
// offsets and padded offsets in shared memory; expert e's padding starts
// after its counts and has s_poff[e+1] - s_poff[e] - (s_off[e+1] - s_off[e])
// rows).
template <int THREADS>
__device__ __forceinline__ void zero_padding_rows(int b, int nblocks, const int* s_off, const int* s_poff, int E,
                                                  int vec_per_row, uint4* __restrict__ buf) {
  const int total = (s_poff[E] - s_off[E]);       // padding rows before expert E
  for (int j = b; j < total; j += nblocks) {
    int lo = 0, hi = E - 1;                       // largest e with padding-before(e) <= j
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s_poff[mid] - s_off[mid] <= j) lo = mid; else hi = mid - 1;
    }
    const int row = s_off[lo + 1] - s_off[lo] + s_poff[lo] + (j - (s_poff[lo] - s_off[lo]));
    uint4* dst = buf + (long long)row * vec_per_row;
    for (int v = threadIdx.x; v < vec_per_row; v += THREADS) dst[v] = make_uint4(0, 0, 0, 0);
  }
}

// RAW (at most 32 chunks and 32 experts): base holds the chunk histograms
// as counted, not scanned, and counts is not written yet; each block sums the
// columns it needs itself (one coalesced load per expert and per pair) and
// block 0 also writes counts -- no scan between the two launches.
template <int kGsThreads, int kGsBatch, bool RAW>
__global__ void __launch_bounds__(kGsThreads) gather_scatter_kernel(
    const uint4* __restrict__ x, const int32_t* __restrict__ idx, const float* __restrict__ gate, int T, int E,
    int k, int NB, int pb, int vec_per_row, const int32_t* __restrict__ base, int32_t* __restrict__ counts,
    int32_t* __restrict__ offsets, int32_t* __restrict__ poffsets, int32_t* __restrict__ slot_row,
    int32_t* __restrict__ row_src, float* __restrict__ row_gate, uint4* __restrict__ x_perm, int zero_pad,
    int* status) {
  pdl_entry();
  __shared__ int s_off[kMaxE + 1];
  __shared__ int s_poff[kMaxE + 1];
  __shared__ int s_rows[kMaxK];
  __shared__ int s_e[kMaxK];
  __shared__ int s_in[kMaxK];
  const int t = blockIdx.x;
  // the first batch of x[t]'s loads is issued before the maps are worked
  // out, and warp 1 fetches the pairs' experts, scanned columns and ranks
  // while warp 0 derives the expert offsets, so the latencies overlap
  const uint4* src = x + (long long)min(t, max(T - 1, 0)) * vec_per_row;
  uint4 val[kGsBatch];
  #pragma unroll
  for (int u = 0; u < kGsBatch; ++u) {
    const int v = threadIdx.x + u * kGsThreads;
    if (t < T && v < vec_per_row) val[u] = __ldg(src + v);
  }
  const int i1 = threadIdx.x - 32;
  if constexpr (RAW) {
    const int lane = threadIdx.x & 31;
    if (threadIdx.x < 32) {
      // warp 0: counts[e] = sum over the chunks of column e (lane e keeps it),
      // then the exclusive scans over the experts
      int col[32];
      #pragma unroll
      for (int e = 0; e < 32; ++e) col[e] = (e < E && lane < NB) ? base[e * NB + lane] : 0;
      int c = 0;
      #pragma unroll
      for (int e = 0; e < 32; ++e) {
        const int tot = __reduce_add_sync(kFull, col[e]);
        if (lane == e) c = tot;
      }
      const int pc = (c + kPadRows - 1) / kPadRows * kPadRows;
      int ci = c, pi = pc;
      #pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int a = __shfl_up_sync(kFull, ci, d), b = __shfl_up_sync(kFull, pi, d);
        if (lane >= d) { ci += a; pi += b; }
      }
      if (lane < E) {
        s_off[lane] = ci - c;
        s_poff[lane] = pi - pc;
      }
      if (lane == 31) {                               // lanes >= E add nothing
        s_off[E] = ci;
        s_poff[E] = pi;
      }
    } else if (threadIdx.x < 64 && t < T) {
      // warp 1: lane i < k holds pair i; pairs of its expert in the chunks
      // before this token's = sum of that column's first `chunk` entries
      const long long p0 = (long long)t * k;
      const int chunk = static_cast<int>(p0 / pb);
      int e = -1, r = 0;
      if (lane < k) {
        e = idx[p0 + lane];
        if (e < 0 || e >= E) e = -1;
        else r = slot_row[p0 + lane];
      }
      int in_e = r;
      for (int g = 0; g < k; g += 8) {
        int v[8];
        #pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int ej = __shfl_sync(kFull, e, (g + j) & 31);
          v[j] = (g + j < k && ej >= 0 && lane < chunk) ? base[ej * NB + lane] : 0;
        }
        #pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int sum = __reduce_add_sync(kFull, v[j]);
          if (lane == g + j) in_e += sum;
        }
      }
      if (lane < k) {
        s_e[lane] = e;
        s_in[lane] = in_e;
      }
    }
  } else {
    if (t < T && i1 >= 0 && i1 < k) {
      const long long p = (long long)t * k + i1;
      int e = idx[p];
      int in_e = 0;                                  // pairs of expert e before this one
      if (e >= 0 && e < E) in_e = base[(long long)e * NB + static_cast<int>(p / pb)] + slot_row[p];
      else e = -1;
      s_e[i1] = e;
      s_in[i1] = in_e;
    }
    expert_offsets(counts, E, s_off, s_poff);
  }
  __syncthreads();
  if (t == 0) {
    for (int i = threadIdx.x; i <= E; i += kGsThreads) {
      offsets[i] = s_off[i];
      poffsets[i] = s_poff[i];
      if (RAW && i < E) counts[i] = s_off[i + 1] - s_off[i];
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int e = warp; e < E; e += kGsThreads / 32) {
      for (int rr = s_poff[e] + (s_off[e + 1] - s_off[e]) + lane; rr < s_poff[e + 1]; rr += 32) {
        row_src[rr] = -1;
        if (row_gate != nullptr) row_gate[rr] = 0.f;
      }
    }
  }
  if (zero_pad) zero_padding_rows<kGsThreads>(t, gridDim.x, s_off, s_poff, E, vec_per_row, x_perm);
  if (t >= T) return;
  if (threadIdx.x < k) {
    const long long p = (long long)t * k + threadIdx.x;
    const int e = s_e[threadIdx.x];
    int row = -1;
    if (e >= 0) {
      const int in_e = s_in[threadIdx.x];
      row = s_poff[e] + in_e;
      if (in_e < 0 || in_e >= s_off[e + 1] - s_off[e]) {
        // only reachable if the histogram launch's results are inconsistent
        // (a workspace not initialised, or shared by overlapping calls)
        set_status(status, kErrBadIndex);
        row = -1;
      } else {
        row_src[row] = t;
        if (row_gate != nullptr) row_gate[row] = gate[p];
      }
    }
    slot_row[p] = row;
    s_rows[threadIdx.x] = row;
  }
  __syncthreads();
  for (int v0 = threadIdx.x; v0 < vec_per_row; v0 += kGsBatch * kGsThreads) {
    if (v0 != threadIdx.x) {
      #pragma unroll
      for (int u = 0; u < kGsBatch; ++u) {
        const int v = v0 + u * kGsThreads;
        if (v < vec_per_row) val[u] = __ldg(src + v);
      }
    }
    for (int i = 0; i < k; ++i) {
      const int r = s_rows[i];
      if (r < 0) continue;
      uint4* dst = x_perm + (long long)r * vec_per_row;
      #pragma unroll
      for (int u = 0; u < kGsBatch; ++u) {
        const int v = v0 + u * kGsThreads;
        if (v < vec_per_row) dst[v] = val[u];
      }
    }
  }
}

// ---------------------------------------------------------------- row copies
// One block per token: read x[t] once, write it to its k rows.  Each thread
// keeps up to 4 16-byte loads in flight before storing.
__global__ void __launch_bounds__(128) gather_kernel(const uint4* __restrict__ x, const int32_t* __restrict__ slot_row,
                                                     int k, int vec_per_row, uint4* __restrict__ x_perm) {
  pdl_entry();
  const int t = blockIdx.x;
  __shared__ int s_rows[kMaxK];
  if (threadIdx.x < k) s_rows[threadIdx.x] = slot_row[(long long)t * k + threadIdx.x];
  __syncthreads();
  const uint4* src = x + (long long)t * vec_per_row;
  for (int v0 = threadIdx.x; v0 < vec_per_row; v0 += 4 * blockDim.x) {
    uint4 val[4];
    #pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int v = v0 + u * blockDim.x;
      if (v < vec_per_row) val[u] = __ldg(src + v);
    }
    for (int i = 0; i < k; ++i) {
      const int r = s_rows[i];
      if (r < 0) continue;
      uint4* dst = x_perm + (long long)r * vec_per_row;
      #pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int v = v0 + u * blockDim.x;
        if (v < vec_per_row) dst[v] = val[u];
      }
    }
  }
}

// The row copy of an input whose maps exist already (dy in the backward),
// with the segments' padding rows zeroed in the same launch (block t copies
// token t and zeroes padding rows t, t + T, ...; every block derives the
// expert offsets from counts).
__global__ void __launch_bounds__(128) gather_zero_kernel(const uint4* __restrict__ x,
                                                          const int32_t* __restrict__ slot_row, int T, int k, int E,
                                                          const int32_t* __restrict__ counts, int vec_per_row,
                                                          uint4* __restrict__ x_perm) {
  pdl_entry();
  __shared__ int s_off[kMaxE + 1];
  __shared__ int s_poff[kMaxE + 1];
  __shared__ int s_rows[kMaxK];
  const int t = blockIdx.x;
  if (t < T && threadIdx.x < k) s_rows[threadIdx.x] = slot_row[(long long)t * k + threadIdx.x];
  expert_offsets(counts, E, s_off, s_poff);
  __syncthreads();
  zero_padding_rows<128>(t, gridDim.x, s_off, s_poff, E, vec_per_row, x_perm);
  if (t >= T) return;
  const uint4* src = x + (long long)t * vec_per_row;
  for (int v0 = threadIdx.x; v0 < vec_per_row; v0 += 4 * blockDim.x) {
    uint4 val[4];
    #pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int v = v0 + u * blockDim.x;
      if (v < vec_per_row) val[u] = __ldg(src + v);
    }
    for (int i = 0; i < k; ++i) {
      const int r = s_rows[i];
      if (r < 0) continue;
      uint4* dst = x_perm + (long long)r * vec_per_row;
      #pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int v = v0 + u * blockDim.x;
        if (v < vec_per_row) dst[v] = val[u];
      }
    }
  }
}

__global__ void zero_pad_kernel(const int32_t* __restrict__ counts, const int32_t* __restrict__ poffsets,
                                int vec_per_row, uint4* __restrict__ buf) {
  pdl_entry();
  const int e = blockIdx.x;
  const int r0 = poffsets[e] + counts[e], r1 = poffsets[e + 1];
  const long long n = (long long)(r1 - r0) * vec_per_row;
  uint4* base = buf + (long long)r0 * vec_per_row;
  for (long long i = threadIdx.x; i < n; i += blockDim.x) base[i] = make_uint4(0, 0, 0, 0);
}

__device__ __forceinline__ void add_bf16x8(float (&acc)[8], const uint4& v) {
  acc[0] += bf16_lo(v.x); acc[1] += bf16_hi(v.x);
  acc[2] += bf16_lo(v.y); acc[3] += bf16_hi(v.y);
  acc[4] += bf16_lo(v.z); acc[5] += bf16_hi(v.z);
  acc[6] += bf16_lo(v.w); acc[7] += bf16_hi(v.w);
}

__device__ __forceinline__ uint4 pack8(const float (&a)[8]) {
  return make_uint4(pack_bf16x2(a[0], a[1]), pack_bf16x2(a[2], a[3]), pack_bf16x2(a[4], a[5]),
                    pack_bf16x2(a[6], a[7]));
}

// y[t] = sum_i o[slot_row[t,i]] (+ shared[t]), fp32 in slot order, one rounding.
// Each thread handles 2 vectors per pass with all k row loads issued first.
__global__ void __launch_bounds__(128) combine_kernel(const uint4* __restrict__ o, const int32_t* __restrict__ slot_row,
                                                      const uint4* __restrict__ shared, int k, int vec_per_row,
                                                      uint4* __restrict__ y) {
  pdl_entry();
  const int t = blockIdx.x;
  __shared__ int s_rows[kMaxK];
  if (threadIdx.x < k) s_rows[threadIdx.x] = slot_row[(long long)t * k + threadIdx.x];
  __syncthreads();
  for (int v0 = threadIdx.x; v0 < vec_per_row; v0 += 2 * blockDim.x) {
    const int v1 = v0 + blockDim.x;
    const bool has1 = v1 < vec_per_row;
    float a0[8] = {0, 0, 0, 0, 0, 0, 0, 0}, a1[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    int i = 0;
    for (; i + 2 <= k; i += 2) {
      const int r0 = s_rows[i], r1 = s_rows[i + 1];
      uint4 p0 = make_uint4(0, 0, 0, 0), p1 = p0, q0 = p0, q1 = p0;
      if (r0 >= 0) { p0 = __ldg(o + (long long)r0 * vec_per_row + v0); if (has1) p1 = __ldg(o + (long long)r0 * vec_per_row + v1); }
      if (r1 >= 0) { q0 = __ldg(o + (long long)r1 * vec_per_row + v0); if (has1) q1 = __ldg(o + (long long)r1 * vec_per_row + v1); }
      add_bf16x8(a0, p0); add_bf16x8(a1, p1);
      add_bf16x8(a0, q0); add_bf16x8(a1, q1);
    }
    for (; i < k; ++i) {
      const int r = s_rows[i];
      if (r < 0) continue;
      add_bf16x8(a0, __ldg(o + (long long)r * vec_per_row + v0));
      if (has1) add_bf16x8(a1, __ldg(o + (long long)r * vec_per_row + v1));
    }
    if (shared != nullptr) {
      add_bf16x8(a0, __ldg(shared + (long long)t * vec_per_row + v0));
      if (has1) add_bf16x8(a1, __ldg(shared + (long long)t * vec_per_row + v1));
    }
    y[(long long)t * vec_per_row + v0] = pack8(a0);
    if (has1) y[(long long)t * vec_per_row + v1] = pack8(a1);
  }
}

// ---------------------------------------------------------------- backward
__global__ void __launch_bounds__(128) dgrad_combine_kernel(
    const uint4* __restrict__ dx_perm, const int32_t* __restrict__ slot_row, const int32_t* __restrict__ topk_idx,
    const float* __restrict__ topk_gate, const float* __restrict__ logits, const float* __restrict__ dgate_part,
    int n_part, const uint4* __restrict__ w_router, const uint4* __restrict__ dx_shared, int E, int k,
    int vec_per_row, int score, uint4* __restrict__ dx, float* __restrict__ dgate, float* __restrict__ dlogits,
    float* __restrict__ row_dlogit) {
  pdl_entry();
  const int t = blockIdx.x;
  __shared__ int s_rows[kMaxK];
  __shared__ int s_ids[kMaxK];
  __shared__ float s_dl[kMaxK];
  const int tid = threadIdx.x;
  if (tid < 32) {
    const int lane = tid;
    int row = -1, id = 0;
    float g = 0.f, dg = 0.f, lg = 0.f;
    if (lane < k) {
      row = slot_row[(long long)t * k + lane];
      id = topk_idx[(long long)t * k + lane];
      g = topk_gate[(long long)t * k + lane];
      lg = logits[(long long)t * E + min(max(id, 0), E - 1)];
      if (row >= 0)
        for (int n = 0; n < n_part; ++n) dg += dgate_part[(long long)row * n_part + n];
    }
    // inner = sum_i g_i dg_i (slot order)
    float inner = 0.f, ssum = 0.f;
    const float sg = 1.0f / (1.0f + expf(-lg));
    for (int s = 0; s < k; ++s) {
      inner += __shfl_sync(kFull, g * dg, s);
      ssum += __shfl_sync(kFull, sg, s);
    }
    float dl;
    if (score == 0) {
      dl = g * (dg - inner);
    } else {
      dl = (dg - inner) / ssum * sg * (1.0f - sg);
    }
    if (lane < k) {
      s_rows[lane] = row;
      s_ids[lane] = id;
      s_dl[lane] = dl;
      if (dgate != nullptr) dgate[(long long)t * k + lane] = dg;
      if (row >= 0 && row_dlogit != nullptr) row_dlogit[row] = dl;
    }
  }
  __syncthreads();
  if (dlogits != nullptr) {
    for (int e = tid; e < E; e += blockDim.x) {
      float v = 0.f;
      for (int i = 0; i < k; ++i)
        if (s_ids[i] == e) v = s_dl[i];
      dlogits[(long long)t * E + e] = v;
    }
  }
  for (int v = tid; v < vec_per_row; v += blockDim.x) {
    float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    for (int i = 0; i < k; ++i) {
      const int r = s_rows[i];
      if (r >= 0) add_bf16x8(acc, __ldg(dx_perm + (long long)r * vec_per_row + v));
    }
    if (w_router != nullptr) {
      for (int i = 0; i < k; ++i) {
        const uint4 wv = __ldg(w_router + (long long)s_ids[i] * vec_per_row + v);
        const float d = s_dl[i];
        acc[0] += d * bf16_lo(wv.x); acc[1] += d * bf16_hi(wv.x);
        acc[2] += d * bf16_lo(wv.y); acc[3] += d * bf16_hi(wv.y);
        acc[4] += d * bf16_lo(wv.z); acc[5] += d * bf16_hi(wv.z);
        acc[6] += d * bf16_lo(wv.w); acc[7] += d * bf16_hi(wv.w);
      }
    }
    if (dx_shared != nullptr) add_bf16x8(acc, __ldg(dx_shared + (long long)t * vec_per_row + v));
    dx[(long long)t * vec_per_row + v] = pack8(acc);
  }
}

// dWr[e] = sum over the rows r of expert e of dl_r * x_perm[r]: grid (E, H/256).
// With row_src given, x_perm is x in token order and row r of expert e is
// x[row_src[r]] (the expert-ordered copy need not exist).
__global__ void __launch_bounds__(256) router_wgrad_kernel(const uint4* __restrict__ x_perm,
                                                           const int32_t* __restrict__ row_src,
                                                           const float* __restrict__ row_dlogit,
                                                           const int32_t* __restrict__ counts,
                                                           const int32_t* __restrict__ poffsets, int vec_per_row,
                                                           float* __restrict__ dw) {
  pdl_entry();
  // Block (e, b): 256 columns of dWr[e] (lane = 8 columns); warp w sums the
  // rows w, w+8, w+16, ... of expert e; the eight partial sums are then added
  // in warp order, so the result does not depend on scheduling.
  __shared__ float part[8][256];
  const int e = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int v = blockIdx.y * 32 + lane;
  const bool active = v < vec_per_row;
  const int r0 = poffsets[e], n = counts[e];
  float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  const uint4* xcol = x_perm + (row_src != nullptr ? 0 : (long long)r0 * vec_per_row) + v;
  // row index within x_perm's view: the expert's row, or its token
  auto xrow = [&](int rr) -> long long { return row_src != nullptr ? (long long)__ldg(row_src + r0 + rr) : rr; };
  int r = warp;
  if (active) {
    for (; r + 24 < n; r += 32) {
      uint4 xv[4];
      float d[4];
      #pragma unroll
      for (int u = 0; u < 4; ++u) {
        xv[u] = __ldg(xcol + xrow(r + 8 * u) * vec_per_row);
        d[u] = __ldg(row_dlogit + r0 + r + 8 * u);
      }
      #pragma unroll
      for (int u = 0; u < 4; ++u) {
        acc[0] += d[u] * bf16_lo(xv[u].x); acc[1] += d[u] * bf16_hi(xv[u].x);
        acc[2] += d[u] * bf16_lo(xv[u].y); acc[3] += d[u] * bf16_hi(xv[u].y);
        acc[4] += d[u] * bf16_lo(xv[u].z); acc[5] += d[u] * bf16_hi(xv[u].z);
        acc[6] += d[u] * bf16_lo(xv[u].w); acc[7] += d[u] * bf16_hi(xv[u].w);
      }
    }
    for (; r < n; r += 8) {
      const uint4 xv = __ldg(xcol + xrow(r) * vec_per_row);
      const float d = __ldg(row_dlogit + r0 + r);
      acc[0] += d * bf16_lo(xv.x); acc[1] += d * bf16_hi(xv.x);
      acc[2] += d * bf16_lo(xv.y); acc[3] += d * bf16_hi(xv.y);
      acc[4] += d * bf16_lo(xv.z); acc[5] += d * bf16_hi(xv.z);
      acc[6] += d * bf16_lo(xv.w); acc[7] += d * bf16_hi(xv.w);
    }
  }
  #pragma unroll
  for (int j = 0; j < 8; ++j) part[warp][lane * 8 + j] = acc[j];
  __syncthreads();
  const int c = threadIdx.x;                     // column of this block's 256
  if (blockIdx.y * 256 + c < vec_per_row * 8) {
    float sum = 0.f;
    #pragma unroll
    for (int w = 0; w < 8; ++w) sum += part[w][c];
    dw[(long long)e * vec_per_row * 8 + blockIdx.y * 256 + c] = sum;
  }
}

}  // namespace

// ---------------------------------------------------------------- launchers
cudaError_t launch_topk(const float* logits, const float* bias, int T, int E, int k, int score, int32_t* idx,
                        float* gate, cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  const int blocks = (T + 7) / 8;
  if (E <= 32) launch_k(topk_kernel<1>, blocks, 256, 0, st, logits, bias, T, E, k, score, idx, gate);
  else if (E <= 64) launch_k(topk_kernel<2>, blocks, 256, 0, st, logits, bias, T, E, k, score, idx, gate);
  else if (E <= 128) launch_k(topk_kernel<4>, blocks, 256, 0, st, logits, bias, T, E, k, score, idx, gate);
  else launch_k(topk_kernel<8>, blocks, 256, 0, st, logits, bias, T, E, k, score, idx, gate);
  count_launches(1);
  return cudaGetLastError();
}

namespace {
int chunks_of(int T, int k) { return (T + kPairsPerBlock / k - 1) / (kPairsPerBlock / k); }

cudaError_t launch_scan_scatter(const int32_t* idx, const float* gate, int T, int E, int k, int32_t* hist,
                                int32_t* counts, int32_t* offsets, int32_t* poffsets, int32_t* slot_row,
                                int32_t* row_src, float* row_gate, cudaStream_t st) {
  const long long npairs = (long long)T * k;
  const int NB = chunks_of(T, k);
  launch_k(scan_cols_kernel, (E + 7) / 8, 256, 0, st, hist, NB, E, counts);
  // (with no tokens one block still writes the offsets)
  launch_k(scatter_kernel, NB > 0 ? NB : 1, kPairsPerBlock, 0, st, idx, gate, npairs, pairs_per_chunk(k), E, k, NB, hist,
                                                             counts, offsets, poffsets, slot_row, row_src,
                                                             gate != nullptr ? row_gate : nullptr);
  count_launches(2);
  return cudaGetLastError();
}
}  // namespace

cudaError_t launch_permute_maps(const int32_t* idx, const float* gate, int T, int E, int k, int32_t* hist,
                                int32_t* counts, int32_t* offsets, int32_t* poffsets, int32_t* slot_row,
                                int32_t* row_src, float* row_gate, int* status, cudaStream_t st) {
  const long long npairs = (long long)T * k;
  const int NB = chunks_of(T, k);
  if (NB > 0) {
    launch_k(count_kernel, NB, kPairsPerBlock, 0, st, idx, npairs, pairs_per_chunk(k), E, hist, status);
    count_launches(1);
  }
  return launch_scan_scatter(idx, gate, T, E, k, hist, counts, offsets, poffsets, slot_row, row_src, row_gate, st);
}

namespace {
template <int MODE>
void topk_hist(const float* logits, const float* bias, int T, int E, int k, int score, int32_t* idx, float* gate,
               int32_t* hist, int32_t* slot_row, int* done, int32_t* counts, int NB, cudaStream_t st) {
  if (E <= kThreadTopkE)
    launch_k(topk_hist_kernel<0, MODE>, NB, kPairsPerBlock, 0, st, logits, bias, T, E, k, score, idx, gate, hist, slot_row,
                                                             done, counts);
  else if (E <= 32)
    launch_k(topk_hist_kernel<1, MODE>, NB, kPairsPerBlock, 0, st, logits, bias, T, E, k, score, idx, gate, hist, slot_row,
                                                             done, counts);
  else if (E <= 64)
    launch_k(topk_hist_kernel<2, MODE>, NB, kPairsPerBlock, 0, st, logits, bias, T, E, k, score, idx, gate, hist, slot_row,
                                                             done, counts);
  else if (E <= 128)
    launch_k(topk_hist_kernel<4, MODE>, NB, kPairsPerBlock, 0, st, logits, bias, T, E, k, score, idx, gate, hist, slot_row,
                                                             done, counts);
  else
    launch_k(topk_hist_kernel<8, MODE>, NB, kPairsPerBlock, 0, st, logits, bias, T, E, k, score, idx, gate, hist, slot_row,
                                                             done, counts);
  count_launches(1);
}

// The second launch (after the histograms and ranks, and scan_cols_kernel
// where the histogram launch did not scan).
// At most 32 chunks and 32 experts: the row copy sums the raw histogram
// columns itself (gather_scatter_kernel RAW), so nothing runs between the
// two launches.
bool raw_histograms(int T, int E, int k) {
  const int NB = chunks_of(T, k);
  return NB >= 1 && NB <= 32 && E <= 32;
}

cudaError_t launch_gather_scatter(const void* x, const int32_t* idx, const float* gate, int T, int E, int k, int H,
                                  const int32_t* hist, int32_t* counts, int32_t* offsets, int32_t* poffsets,
                                  int32_t* slot_row, int32_t* row_src, float* row_gate, void* x_perm, int zero_pad,
                                  int* status, cudaStream_t st) {
  const bool raw = raw_histograms(T, E, k);
  auto kern = raw ? gather_scatter_kernel<64, 8, true>
                  : (T <= kGsSmallT) ? gather_scatter_kernel<64, 8, false> : gather_scatter_kernel<128, 4, false>;
  launch_k(kern, T > 0 ? T : 1, (raw || T <= kGsSmallT) ? 64 : 128, 0, st, 
      static_cast<const uint4*>(x), idx, gate, T, E, k, chunks_of(T, k), pairs_per_chunk(k), H / 8, hist, counts,
      offsets, poffsets, slot_row, row_src, gate != nullptr ? row_gate : nullptr, static_cast<uint4*>(x_perm),
      zero_pad, status);
  count_launches(1);
  return cudaGetLastError();
}
}  // namespace

cudaError_t launch_topk_permute_maps(const float* logits, const float* bias, int T, int E, int k, int score,
                                     int32_t* idx, float* gate, int32_t* hist, int32_t* counts, int32_t* offsets,
                                     int32_t* poffsets, int32_t* slot_row, int32_t* row_src, float* row_gate,
                                     cudaStream_t st) {
  const int NB = chunks_of(T, k);
  if (NB > 0) topk_hist<0>(logits, bias, T, E, k, score, idx, gate, hist, nullptr, nullptr, nullptr, NB, st);
  return launch_scan_scatter(idx, gate, T, E, k, hist, counts, offsets, poffsets, slot_row, row_src, row_gate, st);
}

cudaError_t launch_topk_permute_gather(const float* logits, const float* bias, int T, int E, int k, int score,
                                       int32_t* idx, float* gate, int32_t* hist, int* done, int32_t* counts,
                                       int32_t* offsets, int32_t* poffsets, int32_t* slot_row, int32_t* row_src,
                                       float* row_gate, const void* x, int H, void* x_perm, int zero_pad,
                                       int* status, cudaStream_t st) {
  const int NB = chunks_of(T, k);
  if (raw_histograms(T, E, k)) {
    topk_hist<1>(logits, bias, T, E, k, score, idx, gate, hist, slot_row, done, counts, NB, st);
  } else if (NB > 0) {
    if ((long long)NB * E <= kLastScanEntries) {
      topk_hist<2>(logits, bias, T, E, k, score, idx, gate, hist, slot_row, done, counts, NB, st);
    } else {
      topk_hist<1>(logits, bias, T, E, k, score, idx, gate, hist, slot_row, done, counts, NB, st);
      launch_k(scan_cols_kernel, (E + 7) / 8, 256, 0, st, hist, NB, E, counts);
      count_launches(1);
    }
  } else {
    launch_k(scan_cols_kernel, (E + 7) / 8, 256, 0, st, hist, 0, E, counts);   // counts = 0
    count_launches(1);
  }
  return launch_gather_scatter(x, idx, gate, T, E, k, H, hist, counts, offsets, poffsets, slot_row, row_src, row_gate,
                               x_perm, zero_pad, status, st);
}

cudaError_t launch_permute_gather(const int32_t* idx, const float* gate, int T, int E, int k, int32_t* hist,
                                  int* done, int32_t* counts, int32_t* offsets, int32_t* poffsets, int32_t* slot_row,
                                  int32_t* row_src, float* row_gate, const void* x, int H, void* x_perm, int zero_pad,
                                  int* status, cudaStream_t st) {
  const long long npairs = (long long)T * k;
  const int NB = chunks_of(T, k);
  if (raw_histograms(T, E, k)) {
    launch_k(count_rank_kernel<false>, NB, kPairsPerBlock, 0, st, idx, npairs, pairs_per_chunk(k), E, hist, slot_row, done,
                                                            counts, status);
    count_launches(1);
  } else if (NB > 0) {
    if ((long long)NB * E <= kLastScanEntries) {
      launch_k(count_rank_kernel<true>, NB, kPairsPerBlock, 0, st, idx, npairs, pairs_per_chunk(k), E, hist, slot_row, done,
                                                             counts, status);
      count_launches(1);
    } else {
      launch_k(count_rank_kernel<false>, NB, kPairsPerBlock, 0, st, idx, npairs, pairs_per_chunk(k), E, hist, slot_row,
                                                              done, counts, status);
      launch_k(scan_cols_kernel, (E + 7) / 8, 256, 0, st, hist, NB, E, counts);
      count_launches(2);
    }
  } else {
    launch_k(scan_cols_kernel, (E + 7) / 8, 256, 0, st, hist, 0, E, counts);   // counts = 0
    count_launches(1);
  }
  return launch_gather_scatter(x, idx, gate, T, E, k, H, hist, counts, offsets, poffsets, slot_row, row_src, row_gate,
                               x_perm, zero_pad, status, st);
}

cudaError_t launch_gather_rows(const void* x, const int32_t* slot_row, int T, int k, int H, void* x_perm,
                               cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  launch_k(gather_kernel, T, 128, 0, st, static_cast<const uint4*>(x), slot_row, k, H / 8, static_cast<uint4*>(x_perm));
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_gather_rows_zero(const void* x, const int32_t* slot_row, int T, int k, int E,
                                   const int32_t* counts, int H, void* x_perm, cudaStream_t st) {
  launch_k(gather_zero_kernel, T > 0 ? T : 1, 128, 0, st, static_cast<const uint4*>(x), slot_row, T, k, E, counts,
           H / 8, static_cast<uint4*>(x_perm));
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_zero_pad_rows(const int32_t* counts, const int32_t* poffsets, int E, int H, void* buf,
                                 cudaStream_t st) {
  launch_k(zero_pad_kernel, E, 256, 0, st, counts, poffsets, H / 8, static_cast<uint4*>(buf));
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_combine(const void* o_perm, const int32_t* slot_row, const void* shared, int T, int k, int H,
                           void* y, cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  launch_k(combine_kernel, T, 128, 0, st, static_cast<const uint4*>(o_perm), slot_row, static_cast<const uint4*>(shared),
                                    k, H / 8, static_cast<uint4*>(y));
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_dgrad_combine(const void* dx_perm, const int32_t* slot_row, const int32_t* topk_idx,
                                 const float* topk_gate, const float* logits, const float* dgate_part,
                                 int n_part, const void* w_router, const void* dx_shared, int T, int E, int k,
                                 int H, int score, void* dx, float* dgate, float* dlogits, float* row_dlogit,
                                 cudaStream_t st) {
  if (T == 0) return cudaSuccess;
  launch_k(dgrad_combine_kernel, T, 128, 0, st, 
      static_cast<const uint4*>(dx_perm), slot_row, topk_idx, topk_gate, logits, dgate_part, n_part,
      static_cast<const uint4*>(w_router), static_cast<const uint4*>(dx_shared), E, k, H / 8, score,
      static_cast<uint4*>(dx), dgate, dlogits, row_dlogit);
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_router_wgrad(const void* x_perm, const int32_t* row_src, const float* row_dlogit,
                                const int32_t* counts, const int32_t* poffsets, int E, int H, float* dw_router,
                                cudaStream_t st) {
  const int vpr = H / 8;
  dim3 grid(E, (vpr + 31) / 32);
  launch_k(router_wgrad_kernel, grid, 256, 0, st, static_cast<const uint4*>(x_perm), row_src, row_dlogit, counts, poffsets,
                                            vpr, dw_router);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace moe
