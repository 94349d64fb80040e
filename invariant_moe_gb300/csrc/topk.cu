// topk.cu -- sigmoid scoring and deterministic top-k expert selection.
//
// Source: "[BI][DSv4] Pin sparse-MLA decode and prefill scheduling under
// batch invariance", commit log, the deterministic per-row top-k commit and
// the sentinel/NaN audit commits that follow it: rank by score descending,
// break exact ties by ascending index, canonicalise -0.0 to +0.0, compare a
// monotone int32 key of the fp32 bits, rank on validity before key (no
// reserved sentinel value), and never resolve ties through shared-memory
// atomics.
//
// One warp per row, the row held in registers (lane l owns experts l, l+32,
// ...).  top_k rounds; in each round every lane proposes its best untaken
// expert and a butterfly of shuffles picks the warp winner by
// (valid, key desc, index asc).  The result is a pure function of the row.
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

template <int VPL>
__global__ void __launch_bounds__(128) topk_kernel(const float *__restrict__ scores,
                                                   int32_t *__restrict__ ids,
                                                   float *__restrict__ wts,
                                                   float *__restrict__ probs, int M, int E,
                                                   int top_k) {
  const int lane = threadIdx.x & 31;
  const int row = blockIdx.x * 4 + (threadIdx.x >> 5);
  if (row >= M) return;  // whole warp leaves together
  const float *srow = scores + static_cast<size_t>(row) * E;
  int32_t key[VPL];
  uint32_t avail = 0;  // bit i: expert lane + 32 i exists and is not taken
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    const int j = lane + 32 * i;
    if (j < E) {
      const float v = srow[j];
      key[i] = score_key(v);
      avail |= 1u << i;
      if (probs) probs[static_cast<size_t>(row) * E + j] = sigmoid_f32(v);
    } else {
      key[i] = 0;
    }
  }
  int32_t my_id = 0;
  float my_w = 0.0f;
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
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const int oh = __shfl_xor_sync(0xffffffffu, have, off);
      const int32_t ok = __shfl_xor_sync(0xffffffffu, bk, off);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
      const bool better = oh && (!have || ok > bk || (ok == bk && oi < bi));
      if (better) {
        have = oh;
        bk = ok;
        bi = oi;
      }
    }
    // every lane now holds the winner (bk, bi)
    if ((bi & 31) == lane) avail &= ~(1u << (bi >> 5));
    if (lane == t) {
      my_id = bi;
      my_w = sigmoid_f32(key_value(bk));
    }
  }
  if (lane < top_k) {
    ids[static_cast<size_t>(row) * top_k + lane] = my_id;
    wts[static_cast<size_t>(row) * top_k + lane] = my_w;
  }
}

bi_status launch_topk(const float *scores, int32_t *ids, float *wts, float *probs, int64_t M,
                      int64_t E, int32_t top_k, cudaStream_t stream) {
  const unsigned blocks = static_cast<unsigned>((M + 3) / 4);
  const int vpl = static_cast<int>((E + 31) / 32);
#define BI_TOPK_CASE(V)                                                                       \
  topk_kernel<V><<<blocks, 128, 0, stream>>>(scores, ids, wts, probs, (int)M, (int)E, top_k); \
  break;
  switch (vpl <= 1 ? 1 : vpl <= 2 ? 2 : vpl <= 4 ? 4 : vpl <= 8 ? 8 : 16) {
    case 1: BI_TOPK_CASE(1)
    case 2: BI_TOPK_CASE(2)
    case 4: BI_TOPK_CASE(4)
    case 8: BI_TOPK_CASE(8)
    default: BI_TOPK_CASE(16)
  }
#undef BI_TOPK_CASE
  BI_CHECK_LAUNCH();
  return BI_OK;
}

}  // namespace bimoe
