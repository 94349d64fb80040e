// topk_warp.cuh -- deterministic top-k of one row by one warp.
//
// Source: "[BI][DSv4] Pin sparse-MLA decode and prefill scheduling under
// batch invariance", commit log, the deterministic per-row top-k commit and
// the sentinel/NaN audit commits that follow it: rank by score descending,
// break exact ties by ascending index, canonicalise -0.0 to +0.0, compare a
// monotone int32 key of the fp32 bits, rank on validity before key (no
// reserved sentinel value), and never resolve ties through shared-memory
// atomics.
//
// The row is held in registers (lane l owns experts l, l+32, ...).  top_k
// rounds; in each round every lane proposes its best untaken expert and two
// warp reductions (redux.sync) pick the warp winner by (valid, key desc,
// index asc).  The result is a pure function of the row's values.
#pragma once

#include "bimoe_internal.cuh"

namespace bimoe {

__device__ __forceinline__ int32_t score_key(float v) {
  uint32_t u = __float_as_uint(v);
  if (u == 0x80000000u) u = 0u;
  if (u & 0x80000000u) u ^= 0x7fffffffu;
  return static_cast<int32_t>(u);
}
__device__ __forceinline__ float key_value(int32_t key) {
  uint32_t u = static_cast<uint32_t>(key);
  if (u & 0x80000000u) u ^= 0x7fffffffu;
  return __uint_as_float(u);
}
// Logistic sigmoid in fp32: 1 / (1 + e^-v).
__device__ __forceinline__ float sigmoid_f32(float v) {
  return __fdiv_rn(1.0f, __fadd_rn(1.0f, expf(-v)));
}

// Selects the top_k (<= 32) of the row's E scores (E <= 32 * VPL), called by
// all 32 lanes of a warp; load(j) returns score j.  Writes ids_row[t],
// wts_row[t] = sigmoid(score) for slots t < top_k and, if probs_row is
// non-null, sigmoid of every score.
template <int VPL, typename Load>
__device__ __forceinline__ void topk_select_warp(Load load, int E, int top_k, int32_t *ids_row,
                                                 float *wts_row, float *probs_row, int lane) {
  int32_t key[VPL];
  uint32_t avail = 0;  // bit i: expert lane + 32 i exists and is not taken
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    const int j = lane + 32 * i;
    if (j < E) {
      const float v = load(j);
      key[i] = score_key(v);
      avail |= 1u << i;
      if (probs_row) probs_row[j] = sigmoid_f32(v);
    } else {
      key[i] = 0;
    }
  }
  // lane t keeps the winner of round t; its sigmoid is taken after the
  // rounds, off the rounds' dependent chain
  int32_t my_id = 0, my_key = 0;
  for (int t = 0; t < top_k; ++t) {
    // best candidate of this lane: ascending index, strictly greater key wins
    int have = 0;
    int32_t bk = 0;
    int bi = 0;
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
      if ((avail >> i) & 1u) {
        if (!have || key[i] > bk) {
          have = 1;
          bk = key[i];
          bi = lane + 32 * i;
        }
      }
    }
    // warp winner in two reductions: the largest key (biased to unsigned
    // order), then, among the lanes holding it, the smallest index (largest
    // bit-inverted index; a real candidate's is never 0, so 0 = none)
    const uint32_t ub = static_cast<uint32_t>(bk) ^ 0x80000000u;
    const uint32_t kmax = __reduce_max_sync(0xffffffffu, have ? ub : 0u);
    const uint32_t inv = __reduce_max_sync(0xffffffffu, (have && ub == kmax) ? ~static_cast<uint32_t>(bi) : 0u);
    const int wi = static_cast<int>(~inv);
    const int32_t wk = static_cast<int32_t>(kmax ^ 0x80000000u);
    // every lane now holds the winner (wk, wi)
    if ((wi & 31) == lane) avail &= ~(1u << (wi >> 5));
    if (lane == t) {
      my_id = wi;
      my_key = wk;
    }
  }
  if (lane < top_k) {
    ids_row[lane] = my_id;
    wts_row[lane] = sigmoid_f32(key_value(my_key));
  }
}

// The selection on a row srow[0..E) in global memory.  L2 = true reads the
// scores with ld.global.cg (they were written by other CTAs of the same
// launch or by the grid this one overlapped with); otherwise through the
// read-only path.
template <int VPL, bool L2>
__device__ __forceinline__ void topk_row_warp(const float *srow, int E, int top_k, int32_t *ids_row,
                                              float *wts_row, float *probs_row, int lane) {
  topk_select_warp<VPL>([&](int j) { return L2 ? __ldcg(srow + j) : __ldg(srow + j); }, E, top_k, ids_row,
                        wts_row, probs_row, lane);
}

// Calls topk_row_warp with the smallest VPL that holds E (E <= 512).
template <bool L2>
__device__ __forceinline__ void topk_row_dispatch(const float *srow, int E, int top_k,
                                                  int32_t *ids_row, float *wts_row,
                                                  float *probs_row, int lane) {
  if (E <= 32) topk_row_warp<1, L2>(srow, E, top_k, ids_row, wts_row, probs_row, lane);
  else if (E <= 64) topk_row_warp<2, L2>(srow, E, top_k, ids_row, wts_row, probs_row, lane);
  else if (E <= 128) topk_row_warp<4, L2>(srow, E, top_k, ids_row, wts_row, probs_row, lane);
  else if (E <= 256) topk_row_warp<8, L2>(srow, E, top_k, ids_row, wts_row, probs_row, lane);
  else topk_row_warp<16, L2>(srow, E, top_k, ids_row, wts_row, probs_row, lane);
}

}  // namespace bimoe
