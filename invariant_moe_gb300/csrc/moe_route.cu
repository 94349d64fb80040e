// moe_route.cu -- token permutation by expert, row gather, and the top-k
// combine of the batch-invariant fused-MoE path.
//
// Source: "Batch-invariance generation with vLLM fused-MoE backend at
// improved performance", section "What's included" and the strict-review
// summary (tokens grouped per expert for the grouped GEMMs; the top-k
// contributions reduced with unit weights in a fixed `for t in range(topk)`
// order).
//
// Permutation = stable grouping of the (token, slot) pairs by expert, with
// integer arithmetic only; up to 1024 tokens in one single-CTA launch, beyond
// that in three launches:
//   count   per 256-token block, per-expert pair counts (shared-memory
//           counters: a count does not depend on the order of increments)
//   scan    per expert, exclusive scan over blocks; exclusive scan over
//           experts -> offsets
//   scatter per block, one bit per (expert, token) in shared memory; the rank
//           of a pair inside its expert and block is the popcount of the lower
//           tokens' bits, so positions never depend on thread timing.
// A pair is skipped (and BI_DEVERR_* recorded) when its expert id is outside
// [0,E) or repeats an earlier slot of the same row; the other pairs keep
// their positions.  When asked, the permutation also writes each token's mask
// of valid slots (bit t set: slot t is a pair that the GEMMs compute), so the
// layer's combine sums exactly the valid slots and a skipped pair adds
// nothing.
#include "bimoe_internal.cuh"

namespace bimoe {

constexpr int kTokBlock = 256;

__device__ __forceinline__ bool pair_ok(const int32_t *row_ids, int t, int E, int *err) {
  const int e = row_ids[t];
  if (e < 0 || e >= E) {
    report_error(err, BI_DEVERR_BAD_EXPERT_ID);
    return false;
  }
  for (int u = 0; u < t; ++u)
    if (row_ids[u] == e) {
      report_error(err, BI_DEVERR_REPEATED_EXPERT);
      return false;
    }
  return true;
}

__global__ void __launch_bounds__(kTokBlock) moe_count_kernel(const int32_t *__restrict__ ids,
                                                              int M, int E, int top_k,
                                                              int32_t *__restrict__ blkcnt,
                                                              int *err) {
  griddep_wait();
  extern __shared__ int s_cnt[];
  for (int e = threadIdx.x; e < E; e += blockDim.x) s_cnt[e] = 0;
  __syncthreads();
  const int m = blockIdx.x * kTokBlock + threadIdx.x;
  if (m < M) {
    const int32_t *r = ids + static_cast<size_t>(m) * top_k;
    for (int t = 0; t < top_k; ++t)
      if (pair_ok(r, t, E, err)) atomicAdd(&s_cnt[r[t]], 1);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x)
    blkcnt[static_cast<size_t>(blockIdx.x) * E + e] = s_cnt[e];
}

// One CTA of 1024 threads.  blkoff[b,e] = offsets[e] + pairs of expert e in
// blocks < b; offsets[E] = number of valid pairs.
__global__ void __launch_bounds__(1024) moe_scan_kernel(const int32_t *__restrict__ blkcnt,
                                                        int nblk, int E,
                                                        int32_t *__restrict__ blkoff,
                                                        int32_t *__restrict__ offsets) {
  griddep_wait();
  __shared__ int s_warp[32];
  const int e = threadIdx.x;
  int run = 0;
  if (e < E) {
    for (int b = 0; b < nblk; ++b) {
      const int c = blkcnt[static_cast<size_t>(b) * E + e];
      blkoff[static_cast<size_t>(b) * E + e] = run;
      run += c;
    }
  }
  // exclusive scan of run over e (warp shuffles, then warp totals)
  const int lane = e & 31, w = e >> 5;
  int incl = run;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += v;
  }
  if (lane == 31) s_warp[w] = incl;
  __syncthreads();
  if (w == 0) {
    int v = s_warp[lane];
    int inc2 = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, inc2, off);
      if (lane >= off) inc2 += u;
    }
    s_warp[lane] = inc2 - v;  // exclusive prefix of warp totals
  }
  __syncthreads();
  const int excl = s_warp[w] + incl - run;
  if (e < E) {
    offsets[e] = excl;
    for (int b = 0; b < nblk; ++b) blkoff[static_cast<size_t>(b) * E + e] += excl;
  }
  if (e == E - 1) offsets[E] = excl + run;
}

__global__ void __launch_bounds__(kTokBlock) moe_scatter_kernel(const int32_t *__restrict__ ids,
                                                                int M, int E, int top_k,
                                                                const int32_t *__restrict__ blkoff,
                                                                int32_t *__restrict__ perm,
                                                                uint32_t *__restrict__ slot_mask) {
  griddep_wait();
  constexpr int W = kTokBlock / 32, WP = W + 1;  // odd pitch: conflict-free rank loads
  extern __shared__ uint32_t s_bits[];  // [E][WP]
  for (int i = threadIdx.x; i < E * WP; i += blockDim.x) s_bits[i] = 0u;
  __syncthreads();
  const int lm = threadIdx.x;
  const int m = blockIdx.x * kTokBlock + lm;
  const int32_t *r = ids + static_cast<size_t>(m) * top_k;
  if (m < M)
    for (int t = 0; t < top_k; ++t)
      if (pair_ok(r, t, E, nullptr)) atomicOr(&s_bits[r[t] * WP + (lm >> 5)], 1u << (lm & 31));
  __syncthreads();
  if (m < M) {
    uint32_t ok = 0u;
    for (int t = 0; t < top_k; ++t) {
      if (!pair_ok(r, t, E, nullptr)) continue;
      ok |= 1u << t;
      const int e = r[t];
      int rank = 0;
      for (int w = 0; w < (lm >> 5); ++w) rank += __popc(s_bits[e * WP + w]);
      rank += __popc(s_bits[e * WP + (lm >> 5)] & ((1u << (lm & 31)) - 1u));
      const int pos = blkoff[static_cast<size_t>(blockIdx.x) * E + e] + rank;
      perm[pos] = m * top_k + t;
    }
    if (slot_mask) slot_mask[m] = ok;
  }
}

// Single-CTA permutation for M <= 1024 tokens (one thread per token): the
// count, scan and scatter above in one launch.  The positions are the same:
// inside an expert the pairs are in token order, and a pair's rank is the
// number of lower tokens holding that expert (popcounts of a bit matrix).
constexpr int kSmallPermuteMaxM = 1024;

__device__ __forceinline__ int block_excl_scan_int(int v, int *s_warp, int *total) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int incl = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int u = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += u;
  }
  if (lane == 31) s_warp[w] = incl;
  __syncthreads();
  int base = 0, all = 0;
  for (int i = 0; i < nw; ++i) {
    const int t = s_warp[i];
    if (i < w) base += t;
    all += t;
  }
  *total = all;
  return base + incl - v;
}

__global__ void __launch_bounds__(kSmallPermuteMaxM) moe_permute_small_kernel(
    const int32_t *__restrict__ ids, int M, int E, int top_k, int32_t *__restrict__ offsets,
    int32_t *__restrict__ perm, uint32_t *__restrict__ slot_mask, int *err) {
  griddep_wait_small_release();
  extern __shared__ int s_pm[];
  __shared__ int s_warp[32];
  // bit rows padded to an odd pitch: lanes reading word w of different
  // experts' rows then hit different banks
  const int T = blockDim.x, W = T >> 5, WP = W + 1, tid = threadIdx.x;
  int *s_cnt = s_pm;                                          // [E]
  int *s_off = s_pm + E;                                      // [E]
  uint32_t *s_bits = reinterpret_cast<uint32_t *>(s_pm + 2 * E);  // [E][WP]
  for (int i = tid; i < E * WP; i += T) s_bits[i] = 0u;
  for (int e = tid; e < E; e += T) s_cnt[e] = 0;
  __syncthreads();
  const int m = tid;
  const int32_t *r = ids + static_cast<size_t>(m) * top_k;
  uint32_t ok = 0u;  // bit t: slot t is a valid pair
  if (m < M)
    for (int t = 0; t < top_k; ++t)
      if (pair_ok(r, t, E, err)) {
        ok |= 1u << t;
        atomicAdd(&s_cnt[r[t]], 1);
        atomicOr(&s_bits[r[t] * WP + (m >> 5)], 1u << (m & 31));
      }
  __syncthreads();
  // exclusive scan over experts: thread tid owns experts [tid*c, tid*c + c)
  const int c = (E + T - 1) / T;
  const int e0 = min(E, tid * c), e1 = min(E, e0 + c);
  int local = 0;
  for (int e = e0; e < e1; ++e) local += s_cnt[e];
  int total;
  int run = block_excl_scan_int(local, s_warp, &total);
  for (int e = e0; e < e1; ++e) {
    s_off[e] = run;
    offsets[e] = run;
    run += s_cnt[e];
  }
  if (tid == 0) offsets[E] = total;
  if (slot_mask && m < M) slot_mask[m] = ok;
  __syncthreads();
  for (int t = 0; t < top_k; ++t) {
    if (!((ok >> t) & 1u)) continue;
    const int e = r[t];
    const uint32_t *row = s_bits + e * WP;
    int rank = __popc(row[m >> 5] & ((1u << (m & 31)) - 1u));
    for (int w = 0; w < (m >> 5); ++w) rank += __popc(row[w]);
    perm[s_off[e] + rank] = m * top_k + t;
  }
}

// x_perm[p, :] = x[perm[p] / top_k, :] for p < offsets[E]; one warp per row,
// 16-byte copies.
__global__ void __launch_bounds__(256) moe_gather_kernel(const uint4 *__restrict__ x,
                                                         const int32_t *__restrict__ perm,
                                                         const int32_t *__restrict__ offsets,
                                                         int E, int top_k, int P, int row_vec,
                                                         uint4 *__restrict__ xp, int *err) {
  griddep_wait_small_release();
  const int p = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  const int npos = offsets[E];
  if (p == 0 && lane == 0 && (npos < 0 || npos > P)) report_error(err, BI_DEVERR_BAD_PERMUTATION);
  if (p >= min(npos, P)) return;
  const int pair = perm[p];
  if (static_cast<unsigned>(pair) >= static_cast<unsigned>(P)) {  // not a pair id: no copy
    if (lane == 0) report_error(err, BI_DEVERR_BAD_PERMUTATION);
    return;
  }
  const int m = pair / top_k;
  const uint4 *src = x + static_cast<size_t>(m) * row_vec;
  uint4 *dst = xp + static_cast<size_t>(p) * row_vec;
  for (int c = lane; c < row_vec; c += 32) dst[c] = src[c];
}

// Expert-parallel dispatch: for every permuted position p < offsets[E],
// lid[p] = ids[perm[p]] % experts_per_rank (the expert's index on the rank
// that owns it) and pw[p] = wts[perm[p]]: the routing that travels with the
// gathered token rows.  One thread per position.
__global__ void __launch_bounds__(256) moe_gather_routing_kernel(
    const int32_t *__restrict__ ids, const float *__restrict__ wts, const int32_t *__restrict__ offsets,
    const int32_t *__restrict__ perm, int E, int P, int experts_per_rank, int32_t *__restrict__ lid,
    float *__restrict__ pw, int *err) {
  griddep_wait_small_release();
  const int p = blockIdx.x * blockDim.x + threadIdx.x;
  const int npos = offsets[E];
  if (p == 0 && (npos < 0 || npos > P)) report_error(err, BI_DEVERR_BAD_PERMUTATION);
  if (p >= min(npos, P)) return;
  const int pair = perm[p];
  if (static_cast<unsigned>(pair) >= static_cast<unsigned>(P)) {
    report_error(err, BI_DEVERR_BAD_PERMUTATION);
    return;
  }
  const int e = ids[pair];
  lid[p] = e >= 0 ? e % experts_per_rank : -1;
  pw[p] = wts[pair];
}

// Expert-parallel return: contrib[perm[p], :] = rows[p, :] for p < offsets[E]
// (the contributions computed on the experts' ranks, back in (token, slot)
// order at the tokens' home rank).  One warp per position, 16-byte copies.
__global__ void __launch_bounds__(256) moe_scatter_contrib_kernel(
    const uint4 *__restrict__ rows, const int32_t *__restrict__ offsets, const int32_t *__restrict__ perm,
    int E, int P, int row_vec, uint4 *__restrict__ contrib, int *err) {
  griddep_wait_small_release();
  const int p = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  const int npos = offsets[E];
  if (p == 0 && lane == 0 && (npos < 0 || npos > P)) report_error(err, BI_DEVERR_BAD_PERMUTATION);
  if (p >= min(npos, P)) return;
  const int pair = perm[p];
  if (static_cast<unsigned>(pair) >= static_cast<unsigned>(P)) {
    if (lane == 0) report_error(err, BI_DEVERR_BAD_PERMUTATION);
    return;
  }
  const uint4 *src = rows + static_cast<size_t>(p) * row_vec;
  uint4 *dst = contrib + static_cast<size_t>(pair) * row_vec;
  for (int c = lane; c < row_vec; c += 32) dst[c] = src[c];
}

// out[m, h] = bf16(((c[m,0,h] + c[m,1,h]) + ...) + c[m,k-1,h]), fp32 adds in
// slot order; four consecutive h per thread.  MASK (the layer's own
// permutation wrote slot_mask): only the valid slots are summed, in the same
// order -- the first valid contribution, then each later valid one added; a
// token with no valid slot gets +0; with every slot valid this is the same
// sequence of adds as without a mask.  Every slot's row is loaded whatever
// the mask says (a skipped slot's row holds stale but readable data and is
// selected away), so the loads issue back to back in both forms.
template <bool CONSUME, bool MASK>
__global__ void __launch_bounds__(256) moe_combine_kernel(const float4 *__restrict__ contrib,
                                                          __nv_bfloat16 *__restrict__ out, int M,
                                                          int H4, int top_k,
                                                          const uint32_t *__restrict__ slot_mask) {
  griddep_wait_small_release();
  const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const bool active = idx < static_cast<int64_t>(M) * H4;
  const int64_t m = active ? idx / H4 : 0;
  const int h4 = static_cast<int>(idx % H4);
  const float4 *c = contrib + m * top_k * H4 + h4;
  if (active) {
    float4 s = c[0];
    if (!MASK) {
      for (int t = 1; t < top_k; ++t) {
        const float4 v = c[static_cast<int64_t>(t) * H4];
        s.x = __fadd_rn(s.x, v.x);
        s.y = __fadd_rn(s.y, v.y);
        s.z = __fadd_rn(s.z, v.z);
        s.w = __fadd_rn(s.w, v.w);
      }
    } else {
      const uint32_t valid = slot_mask[m];
      bool any = (valid & 1u) != 0u;
      if (!any) s = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
      for (int t = 1; t < top_k; ++t) {
        const float4 v = c[static_cast<int64_t>(t) * H4];
        const bool vt = ((valid >> t) & 1u) != 0u;
        float4 a;
        a.x = __fadd_rn(s.x, v.x);
        a.y = __fadd_rn(s.y, v.y);
        a.z = __fadd_rn(s.z, v.z);
        a.w = __fadd_rn(s.w, v.w);
        if (!any) a = v;  // the first valid slot starts the sum
        if (vt) s = a;
        any = any || vt;
      }
    }
    __nv_bfloat162 lo = __floats2bfloat162_rn(s.x, s.y);
    __nv_bfloat162 hi = __floats2bfloat162_rn(s.z, s.w);
    uint2 pk;
    pk.x = *reinterpret_cast<uint32_t *>(&lo);
    pk.y = *reinterpret_cast<uint32_t *>(&hi);
    *reinterpret_cast<uint2 *>(out + idx * 4) = pk;
  }
  if (CONSUME) {
    // every contribution line has been read (by the eight lanes that share
    // it, all in this warp): drop it from L2 without a write-back.  The host
    // takes this path only when H is a multiple of 32 and contrib is 128-byte
    // aligned, so lines never straddle two rows.
    __syncwarp();
    if (active && (h4 & 7) == 0)
      for (int t = 0; t < top_k; ++t) discard_l2_line(c + static_cast<int64_t>(t) * H4);
  }
}

// ------------------------------------------------------------------- host --
size_t permute_scratch_bytes(int64_t M, int64_t E) {
  const int64_t nblk = (M + kTokBlock - 1) / kTokBlock;
  const size_t one = static_cast<size_t>(nblk * E) * sizeof(int32_t);
  return 2 * ((one + 255) / 256 * 256);
}

bi_status launch_permute(const int32_t *ids, int32_t *offsets, int32_t *perm, int64_t M,
                         int64_t E, int32_t top_k, void *scratch, cudaStream_t stream,
                         uint32_t *slot_mask) {
  if (M <= kSmallPermuteMaxM) {
    const int T = static_cast<int>((M + 255) / 256 * 256);
    const size_t smem = static_cast<size_t>(E) * (2 * sizeof(int) + (T / 32 + 1) * sizeof(uint32_t));
    if (smem <= 48 * 1024)
      return launch_chained(moe_permute_small_kernel, dim3(1), dim3(T), smem, stream, 1, ids, (int)M,
                            (int)E, top_k, offsets, perm, slot_mask, device_error_word());
  }
  const int nblk = static_cast<int>((M + kTokBlock - 1) / kTokBlock);
  const size_t one = (static_cast<size_t>(nblk) * E * sizeof(int32_t) + 255) / 256 * 256;
  int32_t *blkcnt = static_cast<int32_t *>(scratch);
  int32_t *blkoff = reinterpret_cast<int32_t *>(static_cast<char *>(scratch) + one);
  int *err = device_error_word();
  bi_status st;
  if ((st = launch_chained(moe_count_kernel, dim3(nblk), dim3(kTokBlock), E * sizeof(int), stream, 1,
                           ids, (int)M, (int)E, top_k, blkcnt, err)) != BI_OK)
    return st;
  if ((st = launch_chained(moe_scan_kernel, dim3(1), dim3(1024), 0, stream, 1, blkcnt, nblk, (int)E,
                           blkoff, offsets)) != BI_OK)
    return st;
  return launch_chained(moe_scatter_kernel, dim3(nblk), dim3(kTokBlock),
                        E * (kTokBlock / 32 + 1) * sizeof(uint32_t), stream, 1, ids, (int)M, (int)E,
                        top_k, blkoff, perm, slot_mask);
}

bi_status launch_gather(const void *x, const int32_t *perm, const int32_t *offsets, int64_t P,
                        int64_t H, int64_t E, int32_t top_k, void *xp, cudaStream_t stream) {
  const unsigned blocks = static_cast<unsigned>((P + 7) / 8);
  return launch_chained(moe_gather_kernel, dim3(blocks), dim3(256), 0, stream, 1,
                        static_cast<const uint4 *>(x), perm, offsets, (int)E, top_k, (int)P,
                        (int)(H / 8), static_cast<uint4 *>(xp), device_error_word());
}

bi_status launch_gather_routing(const int32_t *ids, const float *wts, const int32_t *offsets,
                                const int32_t *perm, int64_t P, int64_t E, int64_t experts_per_rank,
                                int32_t *lid, float *pw, cudaStream_t stream) {
  const unsigned blocks = static_cast<unsigned>((P + 255) / 256);
  return launch_chained(moe_gather_routing_kernel, dim3(blocks), dim3(256), 0, stream, 1, ids, wts, offsets,
                        perm, (int)E, (int)P, (int)experts_per_rank, lid, pw, device_error_word());
}

bi_status launch_scatter_contrib(const float *rows, const int32_t *offsets, const int32_t *perm,
                                 int64_t P, int64_t H, int64_t E, float *contrib, cudaStream_t stream) {
  const unsigned blocks = static_cast<unsigned>((P + 7) / 8);
  return launch_chained(moe_scatter_contrib_kernel, dim3(blocks), dim3(256), 0, stream, 1,
                        reinterpret_cast<const uint4 *>(rows), offsets, perm, (int)E, (int)P, (int)(H / 4),
                        reinterpret_cast<uint4 *>(contrib), device_error_word());
}

bi_status launch_combine(const float *contrib, void *out, int64_t M, int64_t H, int32_t top_k,
                         bool consume, cudaStream_t stream, const uint32_t *slot_mask) {
  const int64_t total = M * (H / 4);
  const unsigned blocks = static_cast<unsigned>((total + 255) / 256);
  const float4 *c4 = reinterpret_cast<const float4 *>(contrib);
  __nv_bfloat16 *o = static_cast<__nv_bfloat16 *>(out);
  const bool drop = consume && H % 32 == 0 && reinterpret_cast<uintptr_t>(contrib) % 128 == 0;
  if (drop && slot_mask)
    return launch_chained(moe_combine_kernel<true, true>, dim3(blocks), dim3(256), 0, stream, 1, c4, o, (int)M,
                          (int)(H / 4), top_k, slot_mask);
  if (drop)
    return launch_chained(moe_combine_kernel<true, false>, dim3(blocks), dim3(256), 0, stream, 1, c4, o, (int)M,
                          (int)(H / 4), top_k, slot_mask);
  if (slot_mask)
    return launch_chained(moe_combine_kernel<false, true>, dim3(blocks), dim3(256), 0, stream, 1, c4, o, (int)M,
                          (int)(H / 4), top_k, slot_mask);
  return launch_chained(moe_combine_kernel<false, false>, dim3(blocks), dim3(256), 0, stream, 1, c4, o, (int)M,
                        (int)(H / 4), top_k, slot_mask);
}

}  // namespace bimoe
