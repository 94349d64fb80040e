// topk_window.cu -- deterministic windowed per-row top-k (the sparse-MLA
// indexer's selection).
//
// Source: "[BI][DSv4] Pin sparse-MLA decode and prefill scheduling under
// batch invariance", commit log: the deterministic per-row top-k commit
// (score descending, exact ties by ascending column, emitted ascending with a
// -1 tail, window-relative coordinates, -0.0 canonicalised to +0.0, a monotone
// int32 key, the exact k-th key found by a search of the key space and one
// ascending pass emitting the keys above it plus the first ties; row bounds
// clamped to [0, num_cols]) and the masked-lane and validity-first ranking
// commits (only in-window columns can be chosen; no key value is reserved).
//
// One CTA of 512 threads per row, up to 8192 columns: thread t holds columns
// t, t+512, ... (coalesced loads) as unsigned keys (the int32 key with its sign
// bit flipped, so unsigned order is key order).  The exact k-th largest key T
// is found by a 4-pass radix select, 8 bits per pass, on a shared-memory
// histogram, one atomic per key.  (Aggregating a warp's equal digits first
// with match.any, or a shuffle-and-vote plateau test, puts a dependent
// instruction in front of every atomic and cost more than the same-bin
// conflicts it saves: 13.2 and 12.0 us per row on GB300 against 9.0 us, and a
// row whose scores are all equal, every key in one bin, takes 9.4 us.)  Then one pass in column order: a chosen column's output slot is
// (keys > T before it) + min(ties before it, budget), from warp ballots and a
// block scan.  Everything is integer counting: the result is a pure function
// of the row.
#include "bimoe_internal.cuh"

namespace bimoe {

constexpr int kTwThreads = 512;
constexpr int kTwWarps = kTwThreads / 32;
constexpr int kTwMaxCols = 8192;
constexpr int kTwVT = kTwMaxCols / kTwThreads;  // columns per thread

__device__ __forceinline__ uint32_t tw_ukey(float v) {
  uint32_t u = __float_as_uint(v);
  if (u == 0x80000000u) u = 0u;           // -0.0 ranks as +0.0
  if (u & 0x80000000u) u ^= 0x7fffffffu;  // the monotone int32 key ...
  return u ^ 0x80000000u;                 // ... in unsigned order
}

__device__ __forceinline__ int64_t tw_clamp(int64_t v, int64_t lo, int64_t hi) {
  return v < lo ? lo : (v > hi ? hi : v);
}

// Exclusive prefix sum of one value per thread over the whole CTA (thread
// order).  Every thread must call it; scratch holds kTwWarps words.
__device__ __forceinline__ uint32_t tw_block_excl_scan(uint32_t v, uint32_t *scratch,
                                                       uint32_t *total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t incl = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const uint32_t o = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += o;
  }
  if (lane == 31) scratch[warp] = incl;
  __syncthreads();
  uint32_t base = 0, all = 0;
#pragma unroll
  for (int w = 0; w < kTwWarps; ++w) {
    const uint32_t s = scratch[w];
    if (w < warp) base += s;
    all += s;
  }
  __syncthreads();  // scratch is reused by the next call
  if (total) *total = all;
  return base + incl - v;
}

__global__ void __launch_bounds__(kTwThreads) topk_window_kernel(
    const float *__restrict__ scores, int64_t ld, const int64_t *__restrict__ row_start,
    const int64_t *__restrict__ row_end, int num_cols, int k, int32_t *__restrict__ out) {
  __shared__ uint32_t hist[256];
  __shared__ uint32_t scratch[kTwWarps];
  __shared__ uint32_t s_digit, s_kk;
  __shared__ uint32_t pre_gt[kTwVT * kTwWarps], pre_tie[kTwVT * kTwWarps];

  griddep_wait();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t row = blockIdx.x;
  const int64_t rs = row_start ? tw_clamp(row_start[row], 0, num_cols) : 0;
  const int64_t re = row_end ? tw_clamp(row_end[row], 0, num_cols) : num_cols;
  const int nvalid = re > rs ? static_cast<int>(re - rs) : 0;
  const float *srow = scores + row * ld;
  int32_t *orow = out + row * static_cast<int64_t>(k);

  if (nvalid <= k) {
    // the whole window is chosen: column c goes to slot c - rs
    for (int p = tid; p < k; p += kTwThreads) orow[p] = p < nvalid ? p : -1;
    return;
  }

  uint32_t key[kTwVT];
  uint32_t valid = 0;  // bit j: column j*512 + tid is in the window
#pragma unroll
  for (int j = 0; j < kTwVT; ++j) {
    const int c = j * kTwThreads + tid;
    key[j] = 0u;
    if (c >= rs && c < re) {
      key[j] = tw_ukey(srow[c]);
      valid |= 1u << j;
    }
  }

  // ---- radix select: T = the k-th largest key, kk = how many of the keys
  // equal to T are chosen (the tie budget)
  uint32_t prefix = 0u, pmask = 0u, kk = static_cast<uint32_t>(k);
#pragma unroll 1
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    if (tid < 256) hist[tid] = 0u;
    __syncthreads();
#pragma unroll
    for (int j = 0; j < kTwVT; ++j) {
      const bool in = ((valid >> j) & 1u) && (key[j] & pmask) == prefix;
      // one atomic per key, results unused, so the 16 of a pass issue back
      // to back (lanes of a warp hitting one bin are merged by the shared
      // memory atomic unit)
      if (in) atomicAdd(&hist[(key[j] >> shift) & 255u], 1u);
    }
    __syncthreads();
    // thread t < 256 holds bin 255 - t: bins in descending digit order
    const uint32_t v = tid < 256 ? hist[255 - tid] : 0u;
    const uint32_t excl = tw_block_excl_scan(v, scratch, nullptr);
    if (tid < 256 && excl < kk && excl + v >= kk) {
      s_digit = 255u - static_cast<uint32_t>(tid);
      s_kk = kk - excl;
    }
    __syncthreads();
    prefix |= s_digit << shift;
    pmask |= 255u << shift;
    kk = s_kk;
  }
  const uint32_t T = prefix, budget = kk;

  // ---- emission in column order (block j, then warp, then lane)
  const uint32_t lt = (1u << lane) - 1u;
#pragma unroll
  for (int j = 0; j < kTwVT; ++j) {
    const bool v_ = (valid >> j) & 1u;
    const uint32_t bg = __ballot_sync(0xffffffffu, v_ && key[j] > T);
    const uint32_t bt = __ballot_sync(0xffffffffu, v_ && key[j] == T);
    if (lane == 0) {
      pre_gt[j * kTwWarps + warp] = __popc(bg);
      pre_tie[j * kTwWarps + warp] = __popc(bt);
    }
  }
  __syncthreads();
  // exclusive prefixes of the kTwVT * kTwWarps = 256 (block, warp) counts
  const uint32_t cg = tid < kTwVT * kTwWarps ? pre_gt[tid] : 0u;
  const uint32_t ct = tid < kTwVT * kTwWarps ? pre_tie[tid] : 0u;
  const uint32_t eg = tw_block_excl_scan(cg, scratch, nullptr);
  const uint32_t et = tw_block_excl_scan(ct, scratch, nullptr);
  if (tid < kTwVT * kTwWarps) {
    pre_gt[tid] = eg;
    pre_tie[tid] = et;
  }
  __syncthreads();
#pragma unroll
  for (int j = 0; j < kTwVT; ++j) {
    const bool v_ = (valid >> j) & 1u;
    const bool gt = v_ && key[j] > T, tie = v_ && key[j] == T;
    const uint32_t bg = __ballot_sync(0xffffffffu, gt);
    const uint32_t bt = __ballot_sync(0xffffffffu, tie);
    const uint32_t gb = pre_gt[j * kTwWarps + warp] + __popc(bg & lt);
    const uint32_t tb = pre_tie[j * kTwWarps + warp] + __popc(bt & lt);
    if (gt || (tie && tb < budget)) {
      const uint32_t pos = gb + min(tb, budget);
      orow[pos] = j * kTwThreads + tid - static_cast<int>(rs);
    }
  }
}

bi_status launch_topk_window(const float *scores, int64_t ld, const int64_t *row_start,
                             const int64_t *row_end, int64_t n_rows, int64_t num_cols, int32_t k,
                             int32_t *out, cudaStream_t stream) {
  return launch_chained(topk_window_kernel, dim3(static_cast<unsigned>(n_rows)), dim3(kTwThreads), 0,
                        stream, 1, scores, ld, row_start, row_end, static_cast<int>(num_cols), k, out);
}

}  // namespace bimoe
