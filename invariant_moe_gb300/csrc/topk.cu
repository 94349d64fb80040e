// topk.cu -- sigmoid scoring and deterministic top-k expert selection: one
// warp per row running the selection of topk_warp.cuh.
#include "topk_warp.cuh"

namespace bimoe {

// DEPENDENT: launched as a programmatic dependent of the router grid that
// writes `scores` (bi_router_topk); it waits for that grid before reading.
template <int VPL, bool DEPENDENT>
__global__ void __launch_bounds__(128) topk_kernel(const float *__restrict__ scores,
                                                   int32_t *__restrict__ ids,
                                                   float *__restrict__ wts,
                                                   float *__restrict__ probs, int M, int E,
                                                   int top_k) {
  if (DEPENDENT) griddep_wait();
  const int lane = threadIdx.x & 31;
  const int row = blockIdx.x * 4 + (threadIdx.x >> 5);
  if (row >= M) return;  // whole warp leaves together
  topk_row_warp<VPL, DEPENDENT>(scores + static_cast<size_t>(row) * E, E, top_k,
                            ids + static_cast<size_t>(row) * top_k,
                            wts + static_cast<size_t>(row) * top_k,
                            probs ? probs + static_cast<size_t>(row) * E : nullptr, lane);
}

template <bool DEPENDENT>
static bi_status launch_topk_t(const float *scores, int32_t *ids, float *wts, float *probs,
                               int64_t M, int64_t E, int32_t top_k, cudaStream_t stream) {
  const unsigned blocks = static_cast<unsigned>((M + 3) / 4);
  const int vpl = static_cast<int>((E + 31) / 32);
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cfg.gridDim = dim3(blocks);
  cfg.blockDim = dim3(128);
  cfg.stream = stream;
  if (DEPENDENT) {
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  const int Mi = static_cast<int>(M), Ei = static_cast<int>(E);
  cudaError_t e;
  switch (vpl <= 1 ? 1 : vpl <= 2 ? 2 : vpl <= 4 ? 4 : vpl <= 8 ? 8 : 16) {
    case 1: e = cudaLaunchKernelEx(&cfg, topk_kernel<1, DEPENDENT>, scores, ids, wts, probs, Mi, Ei, top_k); break;
    case 2: e = cudaLaunchKernelEx(&cfg, topk_kernel<2, DEPENDENT>, scores, ids, wts, probs, Mi, Ei, top_k); break;
    case 4: e = cudaLaunchKernelEx(&cfg, topk_kernel<4, DEPENDENT>, scores, ids, wts, probs, Mi, Ei, top_k); break;
    case 8: e = cudaLaunchKernelEx(&cfg, topk_kernel<8, DEPENDENT>, scores, ids, wts, probs, Mi, Ei, top_k); break;
    default: e = cudaLaunchKernelEx(&cfg, topk_kernel<16, DEPENDENT>, scores, ids, wts, probs, Mi, Ei, top_k); break;
  }
  if (e != cudaSuccess) {
    set_error("top-k launch: %s", cudaGetErrorString(e));
    return BI_ERR_CUDA;
  }
  BI_CHECK_LAUNCH();
  return BI_OK;
}

bi_status launch_topk(const float *scores, int32_t *ids, float *wts, float *probs, int64_t M,
                      int64_t E, int32_t top_k, cudaStream_t stream) {
  return launch_topk_t<false>(scores, ids, wts, probs, M, E, top_k, stream);
}

// The selection of bi_router_topk: launched right behind the router grid
// that writes `scores`, overlapping its launch with the router's run.
bi_status launch_topk_dependent(const float *scores, int32_t *ids, float *wts, float *probs,
                                int64_t M, int64_t E, int32_t top_k, cudaStream_t stream) {
  return launch_topk_t<true>(scores, ids, wts, probs, M, E, top_k, stream);
}

}  // namespace bimoe
