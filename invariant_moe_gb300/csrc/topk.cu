// topk.cu -- sigmoid scoring and deterministic top-k expert selection: one
// warp per row running the selection of topk_warp.cuh.
#include "topk_warp.cuh"

namespace bimoe {

template <int VPL>
__global__ void __launch_bounds__(128) topk_kernel(const float *__restrict__ scores,
                                                   int32_t *__restrict__ ids,
                                                   float *__restrict__ wts,
                                                   float *__restrict__ probs, int M, int E,
                                                   int top_k) {
  griddep_wait_small_release();
  const int lane = threadIdx.x & 31;
  const int row = blockIdx.x * 4 + (threadIdx.x >> 5);
  if (row >= M) return;  // whole warp leaves together
  // L2 (ld.global.cg) reads: the scores may come from the grid this one
  // overlapped with (a programmatic dependent launch)
  topk_row_warp<VPL, true>(scores + static_cast<size_t>(row) * E, E, top_k,
                           ids + static_cast<size_t>(row) * top_k,
                           wts + static_cast<size_t>(row) * top_k,
                           probs ? probs + static_cast<size_t>(row) * E : nullptr, lane);
}

bi_status launch_topk(const float *scores, int32_t *ids, float *wts, float *probs, int64_t M,
                      int64_t E, int32_t top_k, cudaStream_t stream) {
  const dim3 grid(static_cast<unsigned>((M + 3) / 4)), block(128);
  const int vpl = static_cast<int>((E + 31) / 32);
  const int Mi = static_cast<int>(M), Ei = static_cast<int>(E);
  switch (vpl <= 1 ? 1 : vpl <= 2 ? 2 : vpl <= 4 ? 4 : vpl <= 8 ? 8 : 16) {
    case 1: return launch_chained(topk_kernel<1>, grid, block, 0, stream, 1, scores, ids, wts, probs, Mi, Ei, top_k);
    case 2: return launch_chained(topk_kernel<2>, grid, block, 0, stream, 1, scores, ids, wts, probs, Mi, Ei, top_k);
    case 4: return launch_chained(topk_kernel<4>, grid, block, 0, stream, 1, scores, ids, wts, probs, Mi, Ei, top_k);
    case 8: return launch_chained(topk_kernel<8>, grid, block, 0, stream, 1, scores, ids, wts, probs, Mi, Ei, top_k);
    default: return launch_chained(topk_kernel<16>, grid, block, 0, stream, 1, scores, ids, wts, probs, Mi, Ei, top_k);
  }
}

}  // namespace bimoe
