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
// is found by a 3-pass radix select on digits of 11, 11 and 10 bits, on a
// 2048-bin shared-memory histogram, one atomic per key; each thread owns a
// quad of bins for the descending scan, and the next pass's clear rides on
// the scan's own barrier, so a pass costs three barriers.  (Aggregating a
// warp's equal digits first with match.any, or a shuffle-and-vote plateau
// test, puts a dependent instruction in front of every atomic and cost more
// than the same-bin conflicts it saves.)  Then one pass in column order: a
// chosen column's output slot is (keys > T before it) + min(ties before it,
// budget), from warp ballots and one block scan of both counts packed in a
// word.  Everything is integer counting: the result is a pure function
// of the row.
#include "bimoe_internal.cuh"

namespace bimoe {

constexpr int kTwThreads = 512;
constexpr int kTwWarps = kTwThreads / 32;
constexpr int kTwMaxCols = 8192;
constexpr int kTwVT = kTwMaxCols / kTwThreads;  // columns per thread
constexpr int kTwBins = 2048;                  // 11-bit digits
static_assert(kTwThreads * 4 == kTwBins, "one bin quad per thread");

// the score's bits, read as an integer so that no float operation touches them
__device__ __forceinline__ uint32_t tw_ukey(uint32_t u) {
  if (u == 0x80000000u) u = 0u;           // -0.0 ranks as +0.0
  if (u & 0x80000000u) u ^= 0x7fffffffu;  // the monotone int32 key ...
  return u ^ 0x80000000u;                 // ... in unsigned order
}

__device__ __forceinline__ int64_t tw_clamp(int64_t v, int64_t lo, int64_t hi) {
  return v < lo ? lo : (v > hi ? hi : v);
}

// Exclusive prefix sum of one value per thread over the whole CTA (thread
// order).  Every thread must call it; scratch holds kTwWarps words.  There is
// one barrier inside and none at the end: the caller puts a barrier between
// this call's return and the next write of scratch.
__device__ __forceinline__ uint32_t tw_block_excl_scan(uint32_t v, uint32_t *scratch) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t incl = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const uint32_t o = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += o;
  }
  if (lane == 31) scratch[warp] = incl;
  __syncthreads();
  // prefix over the warp totals: lane w < kTwWarps scans total w, and warp w
  // takes the exclusive prefix held by its lane w
  const uint32_t wt = lane < kTwWarps ? scratch[lane] : 0u;
  uint32_t wincl = wt;
#pragma unroll
  for (int off = 1; off < kTwWarps; off <<= 1) {
    const uint32_t o = __shfl_up_sync(0xffffffffu, wincl, off);
    if (lane >= off) wincl += o;
  }
  const uint32_t base = __shfl_sync(0xffffffffu, wincl - wt, warp);
  return base + incl - v;
}

__global__ void __launch_bounds__(kTwThreads) topk_window_kernel(
    const float *__restrict__ scores, int64_t ld, const int64_t *__restrict__ row_start,
    const int64_t *__restrict__ row_end, int num_cols, int k, int32_t *__restrict__ out) {
  __shared__ __align__(16) uint32_t hist[kTwBins];
  __shared__ uint32_t scratch[kTwWarps];
  __shared__ uint32_t s_digit, s_kk;
  // per (column block, warp): keys above T in the low half, ties in the high
  __shared__ uint32_t pre[kTwVT * kTwWarps];

  griddep_wait();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t row = blockIdx.x;
  // the row bounds and the scores are loaded together: every column below
  // num_cols is readable whatever the window, so the score loads do not wait
  // for the bounds
  const int64_t rs_in = row_start ? row_start[row] : 0;
  const int64_t re_in = row_end ? row_end[row] : num_cols;
  const uint32_t *srow = reinterpret_cast<const uint32_t *>(scores + row * ld);
  uint32_t sv[kTwVT];
#pragma unroll
  for (int j = 0; j < kTwVT; ++j) {
    const int c = j * kTwThreads + tid;
    sv[j] = c < num_cols ? srow[c] : 0u;
  }
  const int64_t rs = tw_clamp(rs_in, 0, num_cols);
  const int64_t re = tw_clamp(re_in, 0, num_cols);
  const int nvalid = re > rs ? static_cast<int>(re - rs) : 0;
  int32_t *orow = out + row * static_cast<int64_t>(k);

  if (nvalid <= k) {
    // the whole window is chosen: column c goes to slot c - rs
    for (int p = tid; p < k; p += kTwThreads) orow[p] = p < nvalid ? p : -1;
    return;
  }

  uint4 *hist4 = reinterpret_cast<uint4 *>(hist);
  hist4[tid] = make_uint4(0u, 0u, 0u, 0u);  // kTwThreads * 4 == kTwBins

  uint32_t key[kTwVT];
  uint32_t valid = 0;  // bit j: column j*512 + tid is in the window
#pragma unroll
  for (int j = 0; j < kTwVT; ++j) {
    const int c = j * kTwThreads + tid;
    key[j] = 0u;
    if (c >= rs && c < re) {
      key[j] = tw_ukey(sv[j]);
      valid |= 1u << j;
    }
  }
  __syncthreads();

  // ---- radix select over digits of 11, 11 and 10 bits: T = the k-th largest
  // key, kk = how many of the keys equal to T are chosen (the tie budget)
  uint32_t prefix = 0u, pmask = 0u, kk = static_cast<uint32_t>(k);
#pragma unroll 1
  for (int pass = 0; pass < 3; ++pass) {
    const int shift = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
    const uint32_t dmask = pass == 2 ? 1023u : 2047u;
    const int nq = static_cast<int>(dmask + 1u) / 4;  // bin quads in use
#pragma unroll
    for (int j = 0; j < kTwVT; ++j) {
      const bool in = ((valid >> j) & 1u) && (key[j] & pmask) == prefix;
      // one atomic per key, results unused, so the 16 of a pass issue back
      // to back (lanes of a warp hitting one bin are merged by the shared
      // memory atomic unit)
      if (in) atomicAdd(&hist[(key[j] >> shift) & dmask], 1u);
    }
    __syncthreads();
    // thread t < nq holds the quad of bins 4(nq-1-t) .. 4(nq-1-t)+3, so the
    // threads walk the bins in descending digit order
    const uint4 q = tid < nq ? hist4[nq - 1 - tid] : make_uint4(0u, 0u, 0u, 0u);
    const uint32_t sum = q.x + q.y + q.z + q.w;
    const uint32_t excl = tw_block_excl_scan(sum, scratch);
    // every thread has read its quad (the scan's barrier): clear for the next
    // pass
    if (pass < 2) hist4[tid] = make_uint4(0u, 0u, 0u, 0u);
    if (excl < kk && excl + sum >= kk) {
      const uint32_t top = 4u * static_cast<uint32_t>(nq - 1 - tid) + 3u;
      const uint32_t v[4] = {q.w, q.z, q.y, q.x};
      uint32_t c = excl;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        if (c < kk && c + v[i] >= kk) {
          s_digit = top - static_cast<uint32_t>(i);
          s_kk = kk - c;
        }
        c += v[i];
      }
    }
    __syncthreads();
    prefix |= s_digit << shift;
    pmask |= dmask << shift;
    kk = s_kk;
  }
  const uint32_t T = prefix, budget = kk;

  // ---- emission in column order (block j, then warp, then lane)
  const uint32_t lt = (1u << lane) - 1u;
  uint32_t bgt[kTwVT], btie[kTwVT];  // warp ballots of "key > T" and "key == T"
#pragma unroll
  for (int j = 0; j < kTwVT; ++j) {
    const bool v_ = (valid >> j) & 1u;
    bgt[j] = __ballot_sync(0xffffffffu, v_ && key[j] > T);
    btie[j] = __ballot_sync(0xffffffffu, v_ && key[j] == T);
    if (lane == 0) pre[j * kTwWarps + warp] = __popc(bgt[j]) | (__popc(btie[j]) << 16);
  }
  __syncthreads();
  // exclusive prefixes of the kTwVT * kTwWarps = 256 (block, warp) counts,
  // both halves in one scan: each half's total is at most 8192, so the low
  // half never carries into the high one
  const uint32_t cnt = tid < kTwVT * kTwWarps ? pre[tid] : 0u;
  const uint32_t ex = tw_block_excl_scan(cnt, scratch);
  if (tid < kTwVT * kTwWarps) pre[tid] = ex;
  __syncthreads();
#pragma unroll
  for (int j = 0; j < kTwVT; ++j) {
    const bool gt = (bgt[j] >> lane) & 1u, tie = (btie[j] >> lane) & 1u;
    const uint32_t pw = pre[j * kTwWarps + warp];
    const uint32_t gb = (pw & 0xffffu) + __popc(bgt[j] & lt);
    const uint32_t tb = (pw >> 16) + __popc(btie[j] & lt);
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
